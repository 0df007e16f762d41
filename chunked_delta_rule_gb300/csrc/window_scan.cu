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
// spends its work where the recurrence is cheapest.  Two kernels:
//  (a) window_prep_kernel, parallel over (b, h, 64 pairs): the key Gram band
//      x_j . x_{j-o} (o = 0..W) of every pair and the gates (gamma_t, c_t)
//      of every step, into the workspace;
//  (b) window_scan_kernel, one CTA per (b, h) and 16 value columns (S's
//      columns evolve independently), 8 lanes per column, each lane 8
//      (d_k = 64) or 4 (d_k = 32) rows of its column in registers:
//      - the projections z_b = S_{t-1}^T x_{t-b} of the window keys are
//        carried from step to step instead of recomputed (lane b holds z_b):
//          S_t^T x_{t+1-a} = gamma_t z_{a-1} + c_t sum_b (x_{t+1-a} . x_{t-b}) rho_b;
//      - the new key's projection is taken one step ahead, S_{t-1}^T x_{t+1},
//        so its reduction is off the step-to-step dependency chain;
//      - keys, queries, values and the band of a block of steps arrive by
//        cp.async into one of two buffers while the previous block computes;
//        the window keys' rows of a lane live in a register ring of W + 1 slots.

#include "common.cuh"

namespace falcon {

namespace {

constexpr int kCols = 16;   // value columns per CTA
constexpr int kLanes = 8;   // lanes per column
constexpr int kThr = kCols * kLanes;
constexpr int kPrepRows = 64;

__host__ __device__ constexpr int band_stride(int W) { return (W + 3 + 3) / 4 * 4; }  // W+1 band, gamma, c

template <int W>
struct ScanDims {
  static constexpr int R = W + 1;           // register ring slots (window + the next key)
  static constexpr int TB = R * (40 / R);   // steps per staged block, a multiple of R
  static constexpr int NX = TB + W;         // staged pairs t0-W+1 .. t0+TB
  static constexpr int NV = TB + W - 1;     // staged values t0-W+1 .. t0+TB-1
  static constexpr int NBF = band_stride(W);
  static constexpr int WP = (W + 3) / 4 * 4;   // Gram row length, padded for 16-byte loads
};

template <typename Tin, int W, int DK>
struct ScanStage {
  using D = ScanDims<W>;
  Tin xr[D::NX][DK];            // keys of pairs t0-W+1 .. t0+TB (input dtype)
  Tin qr[D::TB][DK];
  Tin vr[D::NV][kCols];
  float band[D::NX][D::NBF];    // x_j . x_{j-o} (o = 0..W), gamma_j, c_j
};

template <typename Tin, int W, int DK>
struct ScanSmem {
  using D = ScanDims<W>;
  ScanStage<Tin, W, DK> st[2];
  float gz[D::TB][kLanes][D::WP];   // per step and lane: Gram of its tracked key with key age b
  float op[D::TB][kCols][kLanes];   // per-lane output partial sums
};

// packed fp32 pairs (two lanes of the FMA pipe per instruction)
__device__ __forceinline__ unsigned long long pk2(float2 v) {
  return (unsigned long long)__float_as_uint(v.x) | ((unsigned long long)__float_as_uint(v.y) << 32);
}
__device__ __forceinline__ float2 upk2(unsigned long long u) {
  return make_float2(__uint_as_float((unsigned)u), __uint_as_float((unsigned)(u >> 32)));
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pk2(a)), "l"(pk2(b)), "l"(pk2(c)));
  return upk2(d);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk2(a)), "l"(pk2(b)));
  return upk2(d);
}

// 16-byte global -> shared copy; src_bytes = 0 fills zeros
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// four consecutive elements as fp32
__device__ __forceinline__ float4 ld4f(const __nv_bfloat16* p) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 ld4f(const float* p) { return *reinterpret_cast<const float4*>(p); }

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

// ---------------------------------------------------------------- (a)
// Band row of pair j (j = -W+1 .. T) at workspace row j + W - 1 of its head.
template <typename Tin, int W, int DK>
__global__ void __launch_bounds__(128) window_prep_kernel(FwdArgs a) {
  constexpr int NBF = band_stride(W), NR = kPrepRows + W;
  __shared__ float xs[NR][DK + 1];
  __shared__ float nrm[NR];
  const int tid = threadIdx.x;
  const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
  const int j0 = -W + 1 + kPrepRows * blockIdx.y;  // first pair of this CTA
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  for (int i = tid; i < NR * DK; i += 128) {  // pairs j0-W .. j0+63
    const int r = i / DK, c = i % DK;
    const Tin* src = key_row<Tin>(a, b, h, j0 - W + r, pos);
    xs[r][c] = src ? to_f32(src[c]) : 0.f;
  }
  __syncthreads();
  for (int r = tid; r < NR; r += 128) {
    float s = 0.f;
    for (int c = 0; c < DK; ++c) s = fmaf(xs[r][c], xs[r][c], s);
    nrm[r] = s;
  }
  __syncthreads();
  float* out = reinterpret_cast<float*>(a.ws) + (size_t)bh * (a.T + W) * NBF;
  for (int i = tid; i < kPrepRows * NBF; i += 128) {
    const int rr = i / NBF, o = i % NBF, j = j0 + rr, r = rr + W;
    if (j > a.T) continue;
    float val = 0.f;
    if (o == 0) {
      val = nrm[r];
    } else if (o <= W) {
      for (int c = 0; c < DK; ++c) val = fmaf(xs[r][c], xs[r - o][c], val);
    } else if (o == W + 1 || o == W + 2) {  // gates of step j
      float gam = 1.f, cf = 0.f;
      if (j >= 0 && j < a.T) {
        const size_t gi = ((size_t)b * a.T + j) * a.H + h;
        gam = fminf(fmaxf(1.f - a.lam[gi], a.eps_gamma), 1.f);
        int n = 0;
        float e = 0.f;
        for (int bb = 0; bb < W; ++bb) {
          if (pos + j - bb >= a.shift) {
            ++n;
            e += nrm[r - bb];
          }
        }
        if (n > 0) cf = a.beta[gi] / (a.eps + e / (float)n) / (float)n;
      }
      val = (o == W + 1) ? gam : cf;
    }
    out[(size_t)(j + W - 1) * NBF + o] = val;
  }
}

// ---------------------------------------------------------------- (b)
template <typename Tin, int W, int DK>
__device__ __forceinline__ void stage_block(const FwdArgs& a, ScanStage<Tin, W, DK>& st, int t0, int b, int h,
                                            int c0, int64_t pos, const float* band_head) {
  using D = ScanDims<W>;
  constexpr int KC = DK * (int)sizeof(Tin) / 16;      // 16-byte chunks per key / query row
  constexpr int VC = kCols * (int)sizeof(Tin) / 16;   // per value row slice
  constexpr int BC = D::NBF / 4;                      // per band row
  constexpr int EC = 16 / (int)sizeof(Tin);           // elements per chunk
  const int tid = threadIdx.x;
  const Tin* dummy = reinterpret_cast<const Tin*>(a.k);
  for (int i = tid; i < D::NX * KC; i += kThr) {
    const int r = i / KC, e0 = EC * (i % KC);
    const Tin* src = key_row<Tin>(a, b, h, t0 - W + 1 + r, pos);
    cp_async16(&st.xr[r][e0], src ? src + e0 : dummy, src ? 16 : 0);
  }
  for (int i = tid; i < D::TB * KC; i += kThr) {
    const int r = i / KC, e0 = EC * (i % KC);
    const bool ok = t0 + r < a.T;
    const Tin* src = reinterpret_cast<const Tin*>(a.q) + (((size_t)b * a.T + (ok ? t0 + r : 0)) * a.H + h) * DK + e0;
    cp_async16(&st.qr[r][e0], src, ok ? 16 : 0);
  }
  for (int i = tid; i < D::NV * VC; i += kThr) {
    const int r = i / VC, e0 = EC * (i % VC);
    const Tin* src = value_row<Tin>(a, b, h, t0 - W + 1 + r, pos);
    cp_async16(&st.vr[r][e0], src ? src + c0 + e0 : dummy, src ? 16 : 0);
  }
  for (int i = tid; i < D::NX * BC; i += kThr) {
    const int r = i / BC, e0 = 4 * (i % BC);
    const bool ok = t0 + r <= a.T + W - 1;  // workspace rows: pairs -W+1 .. T
    cp_async16(&st.band[r][e0], band_head + (size_t)(ok ? t0 + r : 0) * D::NBF + e0, ok ? 16 : 0);
  }
}

template <typename Tin, int W, int DK>
__global__ void __launch_bounds__(kThr) window_scan_kernel(FwdArgs a) {
  using D = ScanDims<W>;
  using L = ScanSmem<Tin, W, DK>;
  constexpr int R = D::R, TB = D::TB, WP = D::WP, RPT = DK / kLanes, P2 = RPT / 2;
  extern __shared__ float4 smem_f4[];
  L& sm = *reinterpret_cast<L*>(smem_f4);
  const int tid = threadIdx.x, g = tid / kLanes, ln = tid % kLanes;
  const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
  const int c0 = blockIdx.y * kCols, col = c0 + g;
  const int T = a.T, NBLK = (T + TB - 1) / TB;
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  const float* band_head = reinterpret_cast<const float*>(a.ws) + (size_t)bh * (T + W) * D::NBF;
  // this lane's rows of its column: runs of four, 32 rows apart, so that the
  // eight lanes of a column read one contiguous stretch of a key row
  auto rowof = [&](int k) { return (k / 4) * 32 + ln * 4 + (k % 4); };

  float2 S[P2];  // rows rowof(2i), rowof(2i + 1)
#pragma unroll
  for (int i = 0; i < P2; ++i)
    S[i] = a.S_in ? make_float2(a.S_in[((size_t)bh * DK + rowof(2 * i)) * a.dv + col],
                                a.S_in[((size_t)bh * DK + rowof(2 * i + 1)) * a.dv + col])
                  : make_float2(0.f, 0.f);
  float2 ring[R][P2];  // window keys (and the next key) on this lane's rows
  float z = 0.f;       // lane b: z_b = S_{t-1}^T x_{t-b}

  if (NBLK > 0) stage_block<Tin, W, DK>(a, sm.st[0], 0, b, h, c0, pos, band_head);
  cp_async_commit();
  if (NBLK > 1) stage_block<Tin, W, DK>(a, sm.st[1], TB, b, h, c0, pos, band_head);
  cp_async_commit();

  for (int n = 0; n < NBLK; ++n) {
    const int t0 = n * TB;
    ScanStage<Tin, W, DK>& st = sm.st[n & 1];
    cp_async_wait1();  // block n's copies (all but the latest group) are done
    __syncthreads();
    for (int i = tid; i < TB * kLanes * WP; i += kThr) {  // per-lane Gram rows
      const int u = i / (kLanes * WP), la = (i / WP) % kLanes, bb = i % WP;
      float gval = 0.f;
      if (la < W && bb < W) {
        const int ap = la - 1;  // age at step u of the key lane la tracks (-1: the next pair)
        const int mn = ap < bb ? ap : bb, off = ap < bb ? bb - ap : ap - bb;
        gval = st.band[u + W - 1 - mn][off];
      }
      sm.gz[u][la][bb] = gval;
    }
    __syncthreads();

    if (n == 0) {  // ring <- pairs -W+1 .. 0 (slot = pair mod R); z_b = S_in^T x_{-b}
#pragma unroll
      for (int s2 = 0; s2 < R; ++s2) {
        const int j = (s2 == 0) ? 0 : s2 - R;  // slot 1 is filled by the first step's look-ahead
        if (s2 != 1) {
#pragma unroll
          for (int i = 0; i < P2; i += 2) {
            const float4 x4 = ld4f(&st.xr[j + W - 1][rowof(2 * i)]);
            ring[s2][i] = make_float2(x4.x, x4.y);
            ring[s2][i + 1] = make_float2(x4.z, x4.w);
          }
        }
      }
#pragma unroll
      for (int bb = 0; bb < W; ++bb) {
        const int s2 = ((-bb) % R + R) % R;
        float2 p2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < P2; ++i) p2 = ffma2(S[i], ring[s2][i], p2);
        const float p = col_sum(p2.x + p2.y);
        if (ln == bb) z = p;
      }
    }

    // ---- the block's steps, R at a time (ring slots static); steps past the
    // end of the call are no-ops (gamma = 1, c = 0, zero keys and values)
    for (int u0 = 0; u0 < TB && t0 + u0 < T; u0 += R) {
#pragma unroll
      for (int uu = 0; uu < R; ++uu) {
        const int u = u0 + uu;
        const int sn = (uu + 1) % R;  // slot of pair t + 1
        // next step's key, and its projection on S_{t-1}
#pragma unroll
        for (int i = 0; i < P2; i += 2) {
          const float4 x4 = ld4f(&st.xr[u + W][rowof(2 * i)]);
          ring[sn][i] = make_float2(x4.x, x4.y);
          ring[sn][i + 1] = make_float2(x4.z, x4.w);
        }
        float2 p2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < P2; ++i) p2 = ffma2(S[i], ring[sn][i], p2);
        const float P = col_sum(p2.x + p2.y);
        const bool live = t0 + u < T;  // gate rows past the call are not in the workspace
        const float gam = live ? st.band[u + W - 1][W + 1] : 1.f;
        const float cf = live ? st.band[u + W - 1][W + 2] : 0.f;
        // scaled residuals c_t rho_b of the window pairs (lane b: pair t - b)
        const float vb = to_f32(st.vr[u + W - 1 - (ln < W ? ln : 0)][g]);
        const float rho = ln < W ? cf * (vb - gam * z) : 0.f;
        float rh[W];
#pragma unroll
        for (int bb = 0; bb < W; ++bb) rh[bb] = __shfl_sync(0xffffffffu, rho, (tid & 31 & ~7) | bb);
        // state update S_t = gamma S_{t-1} + sum_b x_{t-b} (c rho_b)
        const float2 g2 = make_float2(gam, gam);
#pragma unroll
        for (int i = 0; i < P2; ++i) {
          float2 acc = fmul2(g2, S[i]);
#pragma unroll
          for (int bb = 0; bb < W; ++bb)
            acc = ffma2(ring[(uu - bb + 2 * R) % R][i], make_float2(rh[bb], rh[bb]), acc);
          S[i] = acc;
        }
        // carried projections for step t + 1: lane a holds S_t^T x_{t+1-a}
        const float zprev = __shfl_up_sync(0xffffffffu, z, 1, kLanes);
        {
          float gs = 0.f;
#pragma unroll
          for (int b4 = 0; b4 < WP; b4 += 4) {
            const float4 gv = *reinterpret_cast<const float4*>(&sm.gz[u][ln][b4]);
            const float gq[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (b4 + e < W) gs = fmaf(gq[e], rh[b4 + e], gs);
          }
          z = (ln == 0 ? gam * P : gam * zprev) + gs;
        }
        // output o_t = S_t^T q_t: this lane's partial sum
        float2 o2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < P2; i += 2) {
          const float4 q4 = ld4f(&st.qr[u][rowof(2 * i)]);
          o2 = ffma2(S[i], make_float2(q4.x, q4.y), o2);
          o2 = ffma2(S[i + 1], make_float2(q4.z, q4.w), o2);
        }
        sm.op[u][g][ln] = o2.x + o2.y;
      }
    }
    __syncthreads();  // outputs complete, stage n consumed
    if (n + 2 < NBLK) stage_block<Tin, W, DK>(a, st, t0 + 2 * TB, b, h, c0, pos, band_head);
    cp_async_commit();
    for (int i = tid; i < TB * kCols; i += kThr) {
      const int r = i / kCols, c = i % kCols;
      if (t0 + r < T) {
        const float4 lo = *reinterpret_cast<const float4*>(&sm.op[r][c][0]);
        const float4 hi = *reinterpret_cast<const float4*>(&sm.op[r][c][4]);
        const float o = ((lo.x + lo.y) + (lo.z + lo.w)) + ((hi.x + hi.y) + (hi.z + hi.w));
        reinterpret_cast<Tin*>(a.o)[(((size_t)b * T + t0 + r) * a.H + h) * a.dv + c0 + c] = from_f32<Tin>(o);
      }
    }
  }
  cp_async_wait0();

  // ---- carry out
  if (a.S_out) {
#pragma unroll
    for (int i = 0; i < P2; ++i) {
      a.S_out[((size_t)bh * DK + rowof(2 * i)) * a.dv + col] = S[i].x;
      a.S_out[((size_t)bh * DK + rowof(2 * i + 1)) * a.dv + col] = S[i].y;
    }
  }
  Tin* kpo = reinterpret_cast<Tin*>(a.kprev_out);
  if (blockIdx.y == 0 && kpo) {
    for (int c = tid; c < DK; c += kThr) {
      const float x = (T >= 1) ? to_f32(reinterpret_cast<const Tin*>(a.k)[(((size_t)b * T + (T - 1)) * a.H + h) * DK + c])
                               : (a.kprev_in ? to_f32(reinterpret_cast<const Tin*>(a.kprev_in)[(size_t)bh * DK + c]) : 0.f);
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

template <typename Tin, int W, int DK>
int launch_scan_wd(const FwdArgs& a) {
  record_event(a, 0);
  if (a.T > 0)  // an empty call only passes the carry through: no band needed
    window_prep_kernel<Tin, W, DK>
        <<<dim3(a.B * a.H, (a.T + W + kPrepRows - 1) / kPrepRows), 128, 0, a.stream>>>(a);
  record_event(a, 1);
  auto kern = window_scan_kernel<Tin, W, DK>;
  const size_t smem = sizeof(ScanSmem<Tin, W, DK>);
  if (!set_smem_limit(reinterpret_cast<const void*>(kern), smem)) return FALCON_ERR_CUDA;
  kern<<<dim3(a.B * a.H, a.dv / kCols), kThr, smem, a.stream>>>(a);
  record_event(a, 2);
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

template <typename Tin, int W>
int launch_scan_w(const FwdArgs& a) {
  return a.dk == 64 ? launch_scan_wd<Tin, W, 64>(a) : launch_scan_wd<Tin, W, 32>(a);
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

size_t window_scan_ws_bytes(int B, int T, int H, int W) {
  if (T == 0) return 0;
  return align_up((size_t)B * H * (T + W) * band_stride(W) * sizeof(float), 256);
}

int launch_window_scan(const FwdArgs& a) {
  return a.dtype == FALCON_BF16 ? launch_scan_t<__nv_bfloat16>(a) : launch_scan_t<float>(a);
}

}  // namespace falcon
