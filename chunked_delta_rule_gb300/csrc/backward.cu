// Backward of the Falcon forward for the one-pair variants (Falcon-1, 1A, 2,
// 2A), d_k = d_v = D in {32, 64}, bf16 or fp32 inputs, fp32 arithmetic (the
// dispatch at the end sends Falcon-3/3A and d = 128 to the window kernel).
//
// The pages give no gradient formulas; they follow from the update of
// [JC 把记忆更新变成一次梯度下降; FW 三种等价形式] written per step,
//   x = x_t, n = |x|^2, eta = beta / (eps + n) (per channel for 2/2A, zero
//   for a pair that does not exist), gamma = clamp(1 - lambda, eps_gamma, 1),
//   Z = gamma S_{t-1},  delta = eta (.) (v - Z^T x)   (additive: eta (.) v),
//   S_t = Z + x delta^T,  o_t = S_t^T q_t,
// by the chain rule, going back in time with dS (the gradient of S_t):
//   dS += q do^T;  dq = gamma S_{t-1} do + x (delta . do)
//   ddelta = dS^T x;  regression: dr = eta (.) ddelta, dv = dr,
//     deta = r (.) ddelta, dZ = dS - x dr^T, dx = dS delta - gamma S_{t-1} dr;
//   additive: dv = eta (.) ddelta, deta = v (.) ddelta, dZ = dS, dx = dS delta;
//   dbeta = deta / (eps + n) (summed over channels for a scalar beta),
//   dx += 2 dn x with dn = -sum_j deta_j eta_j / (eps + n);
//   dgamma = <dZ, S_{t-1}>, dlambda = -dgamma where the clamp passes it;
//   dS_{t-1} = gamma dZ;  dk of the key x came from gets dx.
// One CTA per (b, h) walks the sequence: a forward pass stores the state at
// every 64-step block start in the workspace; then, block by block from the
// end, the block's states are recomputed into the workspace and the steps
// are reversed.  Each thread owns 16 state elements (one column, every
// RS-th row); reductions over rows go through a partial-sum table, over
// columns through a padded transpose in shared memory.

#include "common.cuh"

namespace falcon {

namespace {

constexpr int kBB = 64;  // steps per recomputed block

struct BwdArgs {
  int B, T, H;
  float eps, eps_gamma;
  int variant, shift;
  const void* q;
  const void* k;
  const void* v;
  const void* dO;
  const float* beta;
  const float* lam;
  const float* S_in;
  const void* kprev_in;
  const int64_t* pos_in;
  const float* dS_final;
  void* dq;
  void* dk;
  void* dv;
  float* dbeta;
  float* dlam;
  float* dS_in;
  void* dk_prev;
  float* ws;  // per (b, h): block-start states [NB][D*D], then the block's states [kBB][D*D]
};

template <typename Tin>
__device__ __forceinline__ float ldf(const void* p, size_t i) {
  return to_f32(reinterpret_cast<const Tin*>(p)[i]);
}
template <typename Tin>
__device__ __forceinline__ void stf(void* p, size_t i, float x) {
  reinterpret_cast<Tin*>(p)[i] = from_f32<Tin>(x);
}

template <int D>
struct BwdSmem {
  static constexpr int NT = D * D / 16, RS = NT / D;
  float xs[D], qs[D], vs[D], dos[D], dd[D], dr[D], deta[D], cA[D], cB[D], cC[D];
  float rv[kBB][D];   // residual v - Z^T x of each step of the block (regression)
  float dl[kBB][D];   // write delta of each step of the block
  float et[kBB][D];   // eta of each step (channel 0 holds the scalar step)
  float gm[kBB], nr[kBB], lm[kBB];
  float part[RS][D];
  float tr[3][D][D + 1];
  float red[NT / 32 + 3];
};

template <typename Tin, int D, bool ADD, bool PERCH>
__global__ void __launch_bounds__(D * D / 16) falcon_bwd_kernel(BwdArgs a) {
  using L = BwdSmem<D>;
  constexpr int NT = L::NT, RS = L::RS;
  extern __shared__ float4 smem_f4[];
  L& sm = *reinterpret_cast<L*>(smem_f4);
  const int tid = threadIdx.x, j = tid % D, rg = tid / D;
  const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
  const int T = a.T, NB = (T + kBB - 1) / kBB;
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  float* ckpt = a.ws + (size_t)bh * (NB + kBB) * D * D;
  float* sts = ckpt + (size_t)NB * D * D;
  auto row = [&](int m) { return rg + RS * m; };
  auto gidx = [&](int t) { return ((size_t)b * T + t) * a.H + h; };

  // key of pair t (x_t): k_{t - shift}, or the carried key for t = 0 (prefix)
  auto load_x = [&](int t) {
    for (int i = tid; i < D; i += NT) {
      float x = 0.f;
      if (t - a.shift >= 0) x = ldf<Tin>(a.k, gidx(t - a.shift) * D + i);
      else if (a.kprev_in) x = ldf<Tin>(a.kprev_in, (size_t)bh * D + i);
      sm.xs[i] = x;
    }
  };
  // sum over the thread's rows and row groups of val (for column j): every thread gets its column's sum
  auto row_reduce = [&](float s) {
    sm.part[rg][j] = s;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int g = 0; g < RS; ++g) tot += sm.part[g][j];
    __syncthreads();
    return tot;
  };
  // one forward step on the register state (optionally recording it for the backward)
  float S[16];
  auto fwd_step = [&](int t, int tl, bool record) {
    load_x(t);
    if (tid < D) sm.vs[tid] = ldf<Tin>(a.v, gidx(t) * D + tid);
    __syncthreads();
    float n = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; ++i) n = fmaf(sm.xs[i], sm.xs[i], n);
    const bool exists = pos + t >= a.shift;
    const float gam = fminf(fmaxf(1.f - a.lam[gidx(t)], a.eps_gamma), 1.f);
    const float bt = PERCH ? a.beta[gidx(t) * D + j] : a.beta[gidx(t)];
    const float eta = exists ? bt / (a.eps + n) : 0.f;
    float delta, r = 0.f;
    if (ADD) {
      delta = eta * sm.vs[j];
    } else {
      float s = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) s = fmaf(sm.xs[row(m)], S[m], s);
      r = sm.vs[j] - gam * row_reduce(s);
      delta = eta * r;
    }
    if (record && rg == 0) {
      sm.rv[tl][j] = r;
      sm.dl[tl][j] = delta;
      sm.et[tl][j] = eta;
      if (j == 0) { sm.gm[tl] = gam; sm.nr[tl] = n; sm.lm[tl] = a.lam[gidx(t)]; }
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) S[m] = fmaf(gam, S[m], sm.xs[row(m)] * delta);
    __syncthreads();
  };

  // ---- pass 1: forward, state at every block start
#pragma unroll
  for (int m = 0; m < 16; ++m) S[m] = a.S_in ? a.S_in[(size_t)bh * D * D + row(m) * D + j] : 0.f;
  for (int blk = 0; blk < NB; ++blk) {
#pragma unroll
    for (int m = 0; m < 16; ++m) ckpt[(size_t)blk * D * D + row(m) * D + j] = S[m];
    const int t1 = min(T, (blk + 1) * kBB);
    for (int t = blk * kBB; t < t1; ++t) fwd_step(t, 0, false);
  }

  // ---- pass 2: backward, block by block from the end
  float dS[16];
#pragma unroll
  for (int m = 0; m < 16; ++m) dS[m] = a.dS_final ? a.dS_final[(size_t)bh * D * D + row(m) * D + j] : 0.f;
  if (a.shift == 1 && T >= 1) {  // the last key is not the x of any pair of this call
    for (int i = tid; i < D; i += NT) stf<Tin>(a.dk, gidx(T - 1) * D + i, 0.f);
  }
  if (a.dk_prev && (a.shift == 0 || T == 0)) {  // the carried key is read by no pair
    for (int i = tid; i < D; i += NT) stf<Tin>(a.dk_prev, (size_t)bh * D + i, 0.f);
  }
  for (int blk = NB - 1; blk >= 0; --blk) {
    const int t0 = blk * kBB, t1 = min(T, t0 + kBB);
#pragma unroll
    for (int m = 0; m < 16; ++m) S[m] = ckpt[(size_t)blk * D * D + row(m) * D + j];
    for (int t = t0; t < t1; ++t) {  // recompute and record the block's states
#pragma unroll
      for (int m = 0; m < 16; ++m) sts[(size_t)(t - t0) * D * D + row(m) * D + j] = S[m];
      fwd_step(t, t - t0, true);
    }
    for (int t = t1 - 1; t >= t0; --t) {
      const int tl = t - t0;
      float Sp[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) Sp[m] = sts[(size_t)tl * D * D + row(m) * D + j];
      load_x(t);
      if (tid < D) {
        sm.qs[tid] = ldf<Tin>(a.q, gidx(t) * D + tid);
        sm.dos[tid] = ldf<Tin>(a.dO, gidx(t) * D + tid);
        sm.vs[tid] = ldf<Tin>(a.v, gidx(t) * D + tid);
      }
      __syncthreads();
      const float gam = sm.gm[tl], n = sm.nr[tl];
      const float eta = sm.et[tl][j], delta = sm.dl[tl][j], dov = sm.dos[j];
      // dS += q do^T, then ddelta = dS^T x
      float s = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        dS[m] = fmaf(sm.qs[row(m)], dov, dS[m]);
        s = fmaf(sm.xs[row(m)], dS[m], s);
      }
      const float ddel = row_reduce(s);
      float drj, dvj, detaj;
      if (ADD) {
        drj = 0.f;
        dvj = eta * ddel;
        detaj = sm.vs[j] * ddel;
      } else {
        drj = eta * ddel;
        dvj = drj;
        detaj = sm.rv[tl][j] * ddel;
      }
      // products reduced over the columns: Sp do, Sp dr, dS delta
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        sm.tr[0][row(m)][j] = Sp[m] * dov;
        sm.tr[1][row(m)][j] = Sp[m] * drj;
        sm.tr[2][row(m)][j] = dS[m] * delta;
      }
      if (rg == 0) {
        sm.dd[j] = delta * dov;      // delta . do (summed below)
        sm.deta[j] = detaj * eta;    // for dn
        sm.dr[j] = detaj;            // deta, for dbeta
      }
      __syncthreads();
      {  // row i = tid % D, column range rg * (D / RS) ... : partial sums, then combine
        const int i = tid % D, c0 = rg * (D / RS);
        float pa = 0.f, pb = 0.f, pc = 0.f;
#pragma unroll 4
        for (int c = c0; c < c0 + D / RS; ++c) {
          pa += sm.tr[0][i][c];
          pb += sm.tr[1][i][c];
          pc += sm.tr[2][i][c];
        }
        __syncthreads();
        sm.tr[0][i][rg] = pa;
        sm.tr[1][i][rg] = pb;
        sm.tr[2][i][rg] = pc;
        __syncthreads();
        if (tid < D) {
          float A = 0.f, Bv = 0.f, C = 0.f;
#pragma unroll
          for (int g = 0; g < RS; ++g) { A += sm.tr[0][tid][g]; Bv += sm.tr[1][tid][g]; C += sm.tr[2][tid][g]; }
          sm.cA[tid] = A;
          sm.cB[tid] = Bv;
          sm.cC[tid] = C;
        }
      }
      // scalars: delta . do, sum_j deta_j eta_j, sum_j deta_j
      float ddo = 0.f, de = 0.f, dsum = 0.f;
      if (tid < 32) {
        for (int c = tid; c < D; c += 32) { ddo += sm.dd[c]; de += sm.deta[c]; dsum += sm.dr[c]; }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          ddo += __shfl_xor_sync(0xffffffffu, ddo, o);
          de += __shfl_xor_sync(0xffffffffu, de, o);
          dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
        }
        if (tid == 0) { sm.red[0] = ddo; sm.red[1] = de; sm.red[2] = dsum; }
      }
      __syncthreads();
      ddo = sm.red[0];
      de = sm.red[1];
      dsum = sm.red[2];
      const bool exists = pos + t >= a.shift;
      const float dn = exists ? -de / (a.eps + n) : 0.f;
      // dq, dx (this pair's key), dv, dbeta
      if (tid < D) {
        const float xi = sm.xs[tid];
        const float dq = gam * sm.cA[tid] + xi * ddo;
        const float dx = sm.cC[tid] - (ADD ? 0.f : gam * sm.cB[tid]) + 2.f * dn * xi;
        stf<Tin>(a.dq, gidx(t) * D + tid, dq);
        if (t - a.shift >= 0) stf<Tin>(a.dk, gidx(t - a.shift) * D + tid, dx);
        else if (a.dk_prev) stf<Tin>(a.dk_prev, (size_t)bh * D + tid, dx);
      }
      if (rg == 0) {
        stf<Tin>(a.dv, gidx(t) * D + j, dvj);
        if (PERCH) a.dbeta[gidx(t) * D + j] = exists ? detaj / (a.eps + n) : 0.f;
      }
      if (!PERCH && tid == 0) a.dbeta[gidx(t)] = exists ? dsum / (a.eps + n) : 0.f;
      // dZ, dgamma = <dZ, S_{t-1}>, dS_{t-1} = gamma dZ
      float g = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float dz = ADD ? dS[m] : fmaf(-sm.xs[row(m)], drj, dS[m]);
        g = fmaf(dz, Sp[m], g);
        dS[m] = gam * dz;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
      if ((tid & 31) == 0) sm.red[3 + (tid >> 5)] = g;
      __syncthreads();
      if (tid == 0) {
        float dg = 0.f;
        for (int w = 0; w < NT / 32; ++w) dg += sm.red[3 + w];
        const float om = 1.f - sm.lm[tl];
        a.dlam[gidx(t)] = (om >= a.eps_gamma && om <= 1.f) ? -dg : 0.f;
      }
      __syncthreads();
    }
  }
  if (a.dS_in) {
#pragma unroll
    for (int m = 0; m < 16; ++m) a.dS_in[(size_t)bh * D * D + row(m) * D + j] = dS[m];
  }
}

template <typename Tin, int D>
int launch_bwd_d(const BwdArgs& a, cudaStream_t stream) {
  const bool add = variant_additive(a.variant), perch = variant_per_channel(a.variant);
  const size_t smem = sizeof(BwdSmem<D>);
  auto go = [&](auto kern) {
    if (!set_smem_limit(reinterpret_cast<const void*>(kern), smem)) return FALCON_ERR_CUDA;
    kern<<<a.B * a.H, D * D / 16, smem, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
  };
  if (add) return perch ? go(falcon_bwd_kernel<Tin, D, true, true>) : go(falcon_bwd_kernel<Tin, D, true, false>);
  return perch ? go(falcon_bwd_kernel<Tin, D, false, true>) : go(falcon_bwd_kernel<Tin, D, false, false>);
}

}  // namespace

// The window kernel (backward_window.cu) takes Falcon-3/3A and d = 128; the
// chunked kernel Falcon-1/1A at d = 64; this file's kernel the rest.
static bool use_window_kernel(int variant, int d) { return variant_windowed(variant) || d == 128; }

size_t backward_ws_bytes(int variant, int B, int T, int H, int d, int window) {
  if (use_window_kernel(variant, d)) return backward_window_ws_bytes(B, T, H, d, effective_window(variant, window));
  if (backward_chunk_supported(variant, d, d, T)) return backward_chunk_ws_bytes(B, T, H);
  const size_t NB = (size_t)(T + kBB - 1) / kBB;
  return (size_t)B * H * (NB + kBB) * d * d * sizeof(float);
}

bool backward_supported(int variant, int dk, int dv, int window) {
  if (use_window_kernel(variant, dk)) return backward_window_supported(variant, dk, dv, window);
  return dk == dv && (dk == 32 || dk == 64);
}

int launch_backward(const FwdArgs& f, const void* dO, const float* dS_final, void* dq, void* dk, void* dv,
                    float* dbeta, float* dlam, float* dS_in, void* dk_prev, void* dwin_x, void* dwin_v) {
  if (use_window_kernel(f.variant, f.dk))
    return launch_backward_window(f, dO, dS_final, dq, dk, dv, dbeta, dlam, dS_in, dk_prev, dwin_x, dwin_v);
  BwdArgs a;
  a.B = f.B; a.T = f.T; a.H = f.H;
  a.eps = f.eps; a.eps_gamma = f.eps_gamma;
  a.variant = f.variant; a.shift = f.shift;
  a.q = f.q; a.k = f.k; a.v = f.v; a.dO = dO; a.beta = f.beta; a.lam = f.lam;
  a.S_in = f.S_in; a.kprev_in = f.kprev_in; a.pos_in = f.pos_in; a.dS_final = dS_final;
  a.dq = dq; a.dk = dk; a.dv = dv; a.dbeta = dbeta; a.dlam = dlam; a.dS_in = dS_in; a.dk_prev = dk_prev;
  if (backward_chunk_supported(f.variant, f.dk, f.dv, f.T))
    return launch_backward_chunk(f, dO, dS_final, dq, dk, dv, dbeta, dlam, dS_in, dk_prev);
  a.ws = reinterpret_cast<float*>(f.ws);
  if (f.dk == 64)
    return f.dtype == FALCON_BF16 ? launch_bwd_d<__nv_bfloat16, 64>(a, f.stream) : launch_bwd_d<float, 64>(a, f.stream);
  return f.dtype == FALCON_BF16 ? launch_bwd_d<__nv_bfloat16, 32>(a, f.stream) : launch_bwd_d<float, 32>(a, f.stream);
}

}  // namespace falcon
