// Falcon-3 forward (window-averaged NLMS write over the last W pairs) as a
// column-parallel recurrence on CUDA cores, fp32 arithmetic
// [JC Falcon家族六个变体各管一段 (Falcon-3 window mini-batch); FW Falcon 家族].
//
// Per step t, with the window W(t) of existing pairs j in [t-W+1, t],
// n_t = |W(t)|, e_t the mean key energy over W(t), c_t = beta_t / (eps + e_t) / n_t
// and gamma_t the clamped decay [JC 数学上的稳定阀门:正衰减钳制]:
//   rho_{t,b} = v_{t-b} - gamma_t S_{t-1}^T x_{t-b}        (b = key age, 0..W-1)
//   S_t       = gamma_t S_{t-1} + c_t sum_b x_{t-b} rho_{t,b}^T,   o_t = S_t^T q_t.
// In the chunked form every chunk couples C x W unknowns and its chain of
// chunk states stays sequential, so this path walks the steps directly and
// spends its work where the recurrence is cheapest:
//  - S's value columns evolve independently: a CTA owns one (b, h) and 16
//    columns, 8 lanes per column, each lane 8 (d_k = 64) or 4 (d_k = 32) rows
//    of its column in registers (runs of four rows, 32 rows apart);
//  - the projections z_b = S_{t-1}^T x_{t-b} of the window keys are carried
//    from step to step instead of recomputed (lane b of a column holds z_b):
//      S_t^T x_{t+1-a} = gamma_t z_{a-1} + c_t sum_b (x_{t+1-a} . x_{t-b}) rho_b,
//    with the key Gram band x_j . x_{j-o} (o <= W) formed per block of steps;
//  - the projection of the next step's new key on the state is taken one
//    step ahead, S_{t-1}^T x_{t+1}, so its reduction across lanes is off the
//    step-to-step dependency chain; the output reduction is off it as well.
// Keys, values, queries and gates of a block of steps are staged in shared
// memory; the window keys' rows live in a register ring of W + 1 slots.

#include "common.cuh"

namespace falcon {

namespace {

constexpr int kCols = 16;   // value columns per CTA
constexpr int kLanes = 8;   // lanes per column
constexpr int kThr = kCols * kLanes;

template <int W>
struct ScanDims {
  static constexpr int R = W + 1;           // register ring slots (window + the next key)
  static constexpr int TB = R * (64 / R);   // steps per staged block, a multiple of R
  static constexpr int NX = TB + W;         // staged pairs t0-W+1 .. t0+TB
  static constexpr int NV = TB + W - 1;     // staged values t0-W+1 .. t0+TB-1
};

template <int W, int DK>
struct ScanSmem {
  using D = ScanDims<W>;
  float xs[D::NX][DK];
  float qs[D::TB][DK];
  float vs[D::NV][kCols];
  float gb[D::NX][W + 1];   // gb[i][o] = x_i . x_{i-o}
  float gam[D::TB], cf[D::TB];
  float os[D::TB][kCols];
};

template <typename Tin>
__device__ __forceinline__ float ldw(const void* p, size_t i) {
  return to_f32(reinterpret_cast<const Tin*>(p)[i]);
}

// 8 consecutive elements (16-byte aligned) as fp32
__device__ __forceinline__ void ld8(const __nv_bfloat16* p, float* x) {
  const uint4 raw = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h2[e]);
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
}
__device__ __forceinline__ void ld8(const float* p, float* x) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// row of the key of local pair j (NULL: zero key, the pair does not exist or
// lies past the call)
template <typename Tin>
__device__ __forceinline__ const Tin* key_row(const FwdArgs& a, int b, int h, int j, int64_t pos) {
  if (j >= a.T || pos + j < a.shift) return nullptr;
  if (j >= a.shift) return reinterpret_cast<const Tin*>(a.k) + (((size_t)b * a.T + (j - a.shift)) * a.H + h) * a.dk;
  if (j == 0) return a.kprev_in ? reinterpret_cast<const Tin*>(a.kprev_in) + ((size_t)b * a.H + h) * a.dk : nullptr;
  if (!a.winx_in) return nullptr;
  const int slot = ring_slot(pos + j, a.W - 1);
  return reinterpret_cast<const Tin*>(a.winx_in) + (((size_t)b * a.H + h) * (a.W - 1) + slot) * a.dk;
}

template <typename Tin>
__device__ __forceinline__ const Tin* value_row(const FwdArgs& a, int b, int h, int j, int64_t pos) {
  if (j >= a.T || pos + j < a.shift) return nullptr;
  if (j >= 0) return reinterpret_cast<const Tin*>(a.v) + (((size_t)b * a.T + j) * a.H + h) * a.dv;
  if (!a.winv_in) return nullptr;
  const int slot = ring_slot(pos + j, a.W - 1);
  return reinterpret_cast<const Tin*>(a.winv_in) + (((size_t)b * a.H + h) * (a.W - 1) + slot) * a.dv;
}

// sum over the 8 lanes of a column
__device__ __forceinline__ float col_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  return x;
}

template <typename Tin, int W, int DK>
__global__ void __launch_bounds__(kThr) window_scan_kernel(FwdArgs a) {
  using D = ScanDims<W>;
  using L = ScanSmem<W, DK>;
  constexpr int R = D::R, TB = D::TB, RPT = DK / kLanes;
  extern __shared__ float4 smem_f4[];
  L& sm = *reinterpret_cast<L*>(smem_f4);
  const int tid = threadIdx.x, g = tid / kLanes, ln = tid % kLanes;
  const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
  const int c0 = blockIdx.y * kCols, col = c0 + g;
  const int T = a.T;
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  // this lane's rows of its column: groups of four, 32 rows apart, so that
  // the eight lanes of a column read a 128-byte run of a key row at once
  auto rowof = [&](int k) { return (k / 4) * 32 + ln * 4 + (k % 4); };

  float S[RPT];
#pragma unroll
  for (int k = 0; k < RPT; ++k)
    S[k] = a.S_in ? a.S_in[((size_t)bh * DK + rowof(k)) * a.dv + col] : 0.f;
  float ring[R][RPT];
  float z = 0.f;  // lane b: z_b = S_{t-1}^T x_{t-b}

  for (int t0 = 0; t0 < T; t0 += TB) {
    // ---- stage the block: keys of pairs t0-W+1 .. t0+TB, values, queries
    __syncthreads();  // the previous block's outputs and stage are consumed
    for (int i = tid; i < D::NX * (DK / 8); i += kThr) {
      const int r = i / (DK / 8), e0 = 8 * (i % (DK / 8));
      const Tin* src = key_row<Tin>(a, b, h, t0 - W + 1 + r, pos);
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (src) ld8(src + e0, x);
      *reinterpret_cast<float4*>(&sm.xs[r][e0]) = make_float4(x[0], x[1], x[2], x[3]);
      *reinterpret_cast<float4*>(&sm.xs[r][e0 + 4]) = make_float4(x[4], x[5], x[6], x[7]);
    }
    for (int i = tid; i < D::NV * (kCols / 8); i += kThr) {
      const int r = i / (kCols / 8), e0 = 8 * (i % (kCols / 8));
      const Tin* src = value_row<Tin>(a, b, h, t0 - W + 1 + r, pos);
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (src) ld8(src + c0 + e0, x);
      *reinterpret_cast<float4*>(&sm.vs[r][e0]) = make_float4(x[0], x[1], x[2], x[3]);
      *reinterpret_cast<float4*>(&sm.vs[r][e0 + 4]) = make_float4(x[4], x[5], x[6], x[7]);
    }
    for (int i = tid; i < TB * (DK / 8); i += kThr) {
      const int r = i / (DK / 8), e0 = 8 * (i % (DK / 8));
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (t0 + r < T) ld8(reinterpret_cast<const Tin*>(a.q) + (((size_t)b * T + t0 + r) * a.H + h) * DK + e0, x);
      *reinterpret_cast<float4*>(&sm.qs[r][e0]) = make_float4(x[0], x[1], x[2], x[3]);
      *reinterpret_cast<float4*>(&sm.qs[r][e0 + 4]) = make_float4(x[4], x[5], x[6], x[7]);
    }
    __syncthreads();
    for (int i = tid; i < D::NX * (W + 1); i += kThr) {  // Gram band
      const int r = i / (W + 1), o = i % (W + 1);
      float s = 0.f;
      if (r - o >= 0) {
#pragma unroll 4
        for (int c4 = 0; c4 < DK / 4; ++c4) {
          const int c = 4 * ((c4 + r) % (DK / 4));  // rotated start: rows spread over the banks
          const float4 x = *reinterpret_cast<const float4*>(&sm.xs[r][c]);
          const float4 y = *reinterpret_cast<const float4*>(&sm.xs[r - o][c]);
          s = fmaf(x.x, y.x, s);
          s = fmaf(x.y, y.y, s);
          s = fmaf(x.z, y.z, s);
          s = fmaf(x.w, y.w, s);
        }
      }
      sm.gb[r][o] = s;
    }
    __syncthreads();
    if (tid < TB) {  // gates of step t0 + tid
      const int t = t0 + tid;
      float gam = 1.f, cf = 0.f;
      if (t < T) {
        const size_t gi = ((size_t)b * T + t) * a.H + h;
        gam = fminf(fmaxf(1.f - a.lam[gi], a.eps_gamma), 1.f);
        int n = 0;
        float e = 0.f;
        for (int bb = 0; bb < W; ++bb) {
          const int j = t - bb;
          if (pos + j >= a.shift) {
            ++n;
            e += sm.gb[tid + W - 1 - bb][0];
          }
        }
        if (n > 0) cf = a.beta[gi] / (a.eps + e / (float)n) / (float)n;
      }
      sm.gam[tid] = gam;
      sm.cf[tid] = cf;
    }
    __syncthreads();

    if (t0 == 0) {  // ring <- pairs -W+1 .. 0 (slot = pair mod R); z_b = S_in^T x_{-b}
#pragma unroll
      for (int s = 0; s < R; ++s) {
        const int j = (s == 0) ? 0 : s - R;  // slot 1 is filled by the first step's look-ahead
        if (s != 1) {
#pragma unroll
          for (int k = 0; k < RPT; ++k) ring[s][k] = sm.xs[j + W - 1][rowof(k)];
        }
      }
#pragma unroll
      for (int bb = 0; bb < W; ++bb) {
        const int s = ((-bb) % R + R) % R;
        float p = 0.f;
#pragma unroll
        for (int k = 0; k < RPT; ++k) p = fmaf(S[k], ring[s][k], p);
        p = col_sum(p);
        if (ln == bb) z = p;
      }
    }

    for (int u0 = 0; u0 < TB; u0 += R) {
      if (t0 + u0 >= T) break;
#pragma unroll
      for (int uu = 0; uu < R; ++uu) {
        const int u = u0 + uu, t = t0 + u;
        if (t >= T) break;
        const int sn = (uu + 1) % R;  // slot of pair t + 1
        // next step's key, and its projection on S_{t-1}
#pragma unroll
        for (int k = 0; k < RPT; k += 4) {
          const float4 x4 = *reinterpret_cast<const float4*>(&sm.xs[u + W][rowof(k)]);
          ring[sn][k] = x4.x; ring[sn][k + 1] = x4.y; ring[sn][k + 2] = x4.z; ring[sn][k + 3] = x4.w;
        }
        float P = 0.f;
#pragma unroll
        for (int k = 0; k < RPT; ++k) P = fmaf(S[k], ring[sn][k], P);
        P = col_sum(P);
        const float gam = sm.gam[u], cf = sm.cf[u];
        // residuals of the window pairs (lane b: pair t - b)
        float rho = 0.f;
        if (ln < W) rho = sm.vs[u + W - 1 - ln][g] - gam * z;
        float rh[W];
#pragma unroll
        for (int bb = 0; bb < W; ++bb) rh[bb] = __shfl_sync(0xffffffffu, rho, (tid & 31 & ~7) | bb);
        // state update
#pragma unroll
        for (int k = 0; k < RPT; ++k) {
          float acc = 0.f;
#pragma unroll
          for (int bb = 0; bb < W; ++bb) acc = fmaf(ring[(uu - bb + 2 * R) % R][k], rh[bb], acc);
          S[k] = fmaf(gam, S[k], cf * acc);
        }
        // carried projections for step t + 1: lane a holds S_t^T x_{t+1-a}
        const float zprev = __shfl_up_sync(0xffffffffu, z, 1, kLanes);
        if (ln < W) {
          const int ap = ln - 1;  // age at step t of the key lane ln tracks (-1: pair t + 1)
          float gs = 0.f;
#pragma unroll
          for (int bb = 0; bb < W; ++bb) {
            const int mn = ap < bb ? ap : bb;
            const int off = ap < bb ? bb - ap : ap - bb;
            gs = fmaf(sm.gb[u + W - 1 - mn][off], rh[bb], gs);
          }
          z = (ln == 0 ? gam * P : gam * zprev) + cf * gs;
        }
        // output o_t = S_t^T q_t
        float o = 0.f;
#pragma unroll
        for (int k = 0; k < RPT; k += 4) {
          const float4 q4 = *reinterpret_cast<const float4*>(&sm.qs[u][rowof(k)]);
          o = fmaf(S[k], q4.x, o);
          o = fmaf(S[k + 1], q4.y, o);
          o = fmaf(S[k + 2], q4.z, o);
          o = fmaf(S[k + 3], q4.w, o);
        }
        o = col_sum(o);
        if (ln == 0) sm.os[u][g] = o;
      }
    }
    __syncthreads();
    for (int i = tid; i < TB * kCols; i += kThr) {
      const int r = i / kCols, c = i % kCols;
      if (t0 + r < T)
        reinterpret_cast<Tin*>(a.o)[(((size_t)b * T + t0 + r) * a.H + h) * a.dv + c0 + c] = from_f32<Tin>(sm.os[r][c]);
    }
  }

  // ---- carry out
  if (a.S_out) {
#pragma unroll
    for (int k = 0; k < RPT; ++k) a.S_out[((size_t)bh * DK + rowof(k)) * a.dv + col] = S[k];
  }
  Tin* kpo = reinterpret_cast<Tin*>(a.kprev_out);
  if (blockIdx.y == 0 && kpo) {
    for (int c = tid; c < DK; c += kThr) {
      const float x = (T >= 1) ? ldw<Tin>(a.k, (((size_t)b * T + (T - 1)) * a.H + h) * DK + c)
                               : (a.kprev_in ? ldw<Tin>(a.kprev_in, (size_t)bh * DK + c) : 0.f);
      kpo[(size_t)bh * DK + c] = from_f32<Tin>(x);
    }
  }
  if (blockIdx.y == 0 && a.pos_out && tid == 0) a.pos_out[bh] = pos + T;
  // ring slot s holds the pair p in [pos+T-Wr, pos+T-1] with p = s (mod Wr);
  // a pair that does not exist leaves a zero slot
  const int Wr = a.W - 1;
  Tin* wxo = reinterpret_cast<Tin*>(a.winx_out);
  Tin* wvo = reinterpret_cast<Tin*>(a.winv_out);
  for (int64_t p = pos + T - Wr; p <= pos + T - 1; ++p) {
    const int j = (int)(p - pos);
    const int slot = (int)(((p % Wr) + Wr) % Wr);
    if (blockIdx.y == 0 && wxo) {
      const Tin* src = key_row<Tin>(a, b, h, j, pos);
      for (int c = tid; c < DK; c += kThr)
        wxo[((size_t)bh * Wr + slot) * DK + c] = src ? src[c] : from_f32<Tin>(0.f);
    }
    if (wvo) {
      const Tin* src = value_row<Tin>(a, b, h, j, pos);
      for (int c = tid; c < kCols; c += kThr)
        wvo[((size_t)bh * Wr + slot) * a.dv + c0 + c] = src ? src[c0 + c] : from_f32<Tin>(0.f);
    }
  }
}

template <typename Tin, int W>
int launch_scan_w(const FwdArgs& a) {
  dim3 grid(a.B * a.H, a.dv / kCols);
  auto go = [&](auto kern, size_t smem) {
    if (!set_smem_limit(reinterpret_cast<const void*>(kern), smem)) return FALCON_ERR_CUDA;
    record_event(a, 0);
    kern<<<grid, kThr, smem, a.stream>>>(a);
    record_event(a, 1);
    return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
  };
  if (a.dk == 64) return go(window_scan_kernel<Tin, W, 64>, sizeof(ScanSmem<W, 64>));
  return go(window_scan_kernel<Tin, W, 32>, sizeof(ScanSmem<W, 32>));
}

template <typename Tin>
int launch_scan_t(const FwdArgs& a) {
  switch (a.W) {
    case 2: return launch_scan_w<Tin, 2>(a);
    case 3: return launch_scan_w<Tin, 3>(a);
    case 4: return launch_scan_w<Tin, 4>(a);
    case 5: return launch_scan_w<Tin, 5>(a);
    case 6: return launch_scan_w<Tin, 6>(a);
    case 7: return launch_scan_w<Tin, 7>(a);
    default: return launch_scan_w<Tin, 8>(a);
  }
}

}  // namespace

bool window_scan_supported(const FwdArgs& a) {
  return a.variant == FALCON_3 && a.W >= 2 && a.W <= 8 && (a.dk == 32 || a.dk == 64) && a.dv % kCols == 0;
}

int launch_window_scan(const FwdArgs& a) {
  return a.dtype == FALCON_BF16 ? launch_scan_t<__nv_bfloat16>(a) : launch_scan_t<float>(a);
}

}  // namespace falcon
