// Masked-parallel form of a fresh sequence, fp32 [FW 三种等价形式 (linear
// attention (phi(Q) phi(K)^T (.) M) V without a denominator); JC
// 三种视角看同一个更新].  A quadratic-cost reference for tests (T <= 1024).
//
// The whole sequence is one block: g_t is the cumulative log of the clamped
// decay over all T steps, M_ts = exp(g_t - g_s) (s <= t), and the write
// coefficients d_{t,a} of window slot a at step t solve the unit
// lower-triangular system
//   d_{t,a} = coef_{t,a} (v_j - sum_{s<t} M_ts sum_b (x_j . x_{j'}) d_{s,b})
// (j / j' = pairs of slots a / b; additive variants drop the sum).  Then
//   o_t = sum_{s<=t} M_ts sum_b (q_t . x_{j'}) d_{s,b},
//   S_T = sum_s M_{T-1,s} sum_b x_{j'} d_{s,b}^T.
// Three launches: (1) per (b, h) prefix/gates and the key Gram matrices in
// the workspace, (2) the forward substitution (sequential in t, parallel in
// slots x channels), (3) outputs and the final state.

#include "common.cuh"

namespace falcon {

namespace {

constexpr int kMpThreads = 256;

struct MpLayout {  // per (b, h) offsets, in floats
  size_t g, coef, Xw, Gk, PQ, Dl, total;
};

__host__ __device__ inline MpLayout mp_layout(int T, int dk, int dv, int W) {
  MpLayout L;
  const size_t NP = (size_t)T + W - 1;
  size_t off = 0;
  auto take = [&](size_t n) { size_t o = off; off += (n + 63) & ~size_t(63); return o; };
  L.g = take(T);
  L.coef = take((size_t)T * W * dv);
  L.Xw = take(NP * dk);
  L.Gk = take(NP * NP);
  L.PQ = take((size_t)T * NP);
  L.Dl = take((size_t)T * W * dv);
  L.total = off;
  return L;
}

template <typename Tin>
__device__ __forceinline__ float ldm(const void* p, size_t i) {
  return to_f32(reinterpret_cast<const Tin*>(p)[i]);
}

// (1a) per (b, h): pairs, cumulative log-decay, coefficients
template <typename Tin>
__global__ void mp_prep_kernel(FwdArgs a, float* ws) {
  const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
  const int T = a.T, dk = a.dk, dv = a.dv, W = a.W;
  const MpLayout L = mp_layout(T, dk, dv, W);
  float* base = ws + (size_t)bh * L.total;
  float* g = base + L.g;
  float* coef = base + L.coef;
  float* Xw = base + L.Xw;
  const int NP = T + W - 1;
  // pair j = i - (W-1): (k_{j-shift}, v_j); in a fresh sequence only j >= shift
  // exists (shift 1: prefix alignment, 0: same-step pairing)
  for (int i = threadIdx.x; i < NP * dk; i += blockDim.x) {
    int p = i / dk, d = i % dk;
    int j = p - (W - 1);
    Xw[i] = (j >= a.shift) ? ldm<Tin>(a.k, (((size_t)b * T + (j - a.shift)) * a.H + h) * dk + d) : 0.f;
  }
  if (threadIdx.x == 0) {
    float acc = 0.f;
    for (int t = 0; t < T; ++t) {
      acc += clamped_log_decay(a.lam[((size_t)b * T + t) * a.H + h], a.eps_gamma);
      g[t] = acc;
    }
  }
  __syncthreads();
  const bool perch = variant_per_channel(a.variant);
  for (int i = threadIdx.x; i < T * dv; i += blockDim.x) {
    int t = i / dv, cc = i % dv;
    float n = 0.f, e = 0.f;
    for (int s = 0; s < W; ++s) {
      int j = t - (W - 1) + s;
      if (j >= a.shift) {
        n += 1.f;
        float nn = 0.f;
        for (int d = 0; d < dk; ++d) { float x = Xw[(size_t)(t + s) * dk + d]; nn += x * x; }
        e += nn;
      }
    }
    float eta = 0.f;
    if (n > 0.f) {
      float bt = perch ? a.beta[(((size_t)b * T + t) * a.H + h) * dv + cc] : a.beta[((size_t)b * T + t) * a.H + h];
      eta = bt / (a.eps + e / n) / n;
    }
    for (int s = 0; s < W; ++s) {
      int j = t - (W - 1) + s;
      coef[((size_t)t * W + s) * dv + cc] = (j >= a.shift) ? eta : 0.f;
    }
  }
}

// (1b) Gram of the pairs' keys and q . x, one thread per entry
template <typename Tin>
__global__ void mp_gram_kernel(FwdArgs a, float* ws) {
  const int bh = blockIdx.y;
  const int b = bh / a.H, h = bh % a.H;
  const int T = a.T, dk = a.dk, W = a.W;
  const MpLayout L = mp_layout(T, dk, a.dv, W);
  float* base = ws + (size_t)bh * L.total;
  const float* Xw = base + L.Xw;
  float* Gk = base + L.Gk;
  float* PQ = base + L.PQ;
  const size_t NP = (size_t)T + W - 1;
  const size_t nG = NP * NP, nP = (size_t)T * NP;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nG + nP;
       i += (size_t)gridDim.x * blockDim.x) {
    if (i < nG) {
      size_t r = i / NP, c = i % NP;
      float acc = 0.f;
      for (int d = 0; d < dk; ++d) acc += Xw[r * dk + d] * Xw[c * dk + d];
      Gk[i] = acc;
    } else {
      size_t k = i - nG, t = k / NP, c = k % NP;
      float acc = 0.f;
      for (int d = 0; d < dk; ++d)
        acc += ldm<Tin>(a.q, (((size_t)b * T + t) * a.H + h) * dk + d) * Xw[c * dk + d];
      PQ[k] = acc;
    }
  }
}

// (2) forward substitution, one CTA per (b, h, 32-channel slice)
template <typename Tin>
__global__ void mp_solve_kernel(FwdArgs a, float* ws) {
  const int bh = blockIdx.y, slice = blockIdx.x;
  const int b = bh / a.H, h = bh % a.H;
  const int T = a.T, dv = a.dv, W = a.W;
  const MpLayout L = mp_layout(T, a.dk, dv, W);
  float* base = ws + (size_t)bh * L.total;
  const float* g = base + L.g;
  const float* coef = base + L.coef;
  const float* Gk = base + L.Gk;
  float* Dl = base + L.Dl;
  const size_t NP = (size_t)T + W - 1;
  const bool additive = variant_additive(a.variant);
  const int c0 = slice * 32;
  for (int t = 0; t < T; ++t) {
    for (int i = threadIdx.x; i < W * 32; i += blockDim.x) {
      int s = i / 32, cc = c0 + i % 32;
      if (cc >= dv) continue;
      int j = t - (W - 1) + s;
      float r = (j >= 0) ? ldm<Tin>(a.v, (((size_t)b * T + j) * a.H + h) * dv + cc) : 0.f;
      if (!additive) {
        const float* grow = Gk + (size_t)(t + s) * NP;
        for (int tp = 0; tp < t; ++tp) {
          float acc = 0.f;
          for (int bb = 0; bb < W; ++bb) acc += grow[tp + bb] * Dl[((size_t)tp * W + bb) * dv + cc];
          r -= expf(g[t] - g[tp]) * acc;
        }
      }
      Dl[((size_t)t * W + s) * dv + cc] = coef[((size_t)t * W + s) * dv + cc] * r;
    }
    __syncthreads();
  }
}

// (3) outputs and the final state, one thread per entry
template <typename Tin>
__global__ void mp_out_kernel(FwdArgs a, float* ws, float* S_final) {
  const int bh = blockIdx.y;
  const int b = bh / a.H, h = bh % a.H;
  const int T = a.T, dk = a.dk, dv = a.dv, W = a.W;
  const MpLayout L = mp_layout(T, dk, dv, W);
  const float* base = ws + (size_t)bh * L.total;
  const float* g = base + L.g;
  const float* Xw = base + L.Xw;
  const float* PQ = base + L.PQ;
  const float* Dl = base + L.Dl;
  const size_t NP = (size_t)T + W - 1;
  const size_t nO = (size_t)T * dv, nS = (size_t)dk * dv;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nO + nS;
       i += (size_t)gridDim.x * blockDim.x) {
    if (i < nO) {
      int t = (int)(i / dv), cc = (int)(i % dv);
      float acc = 0.f;
      for (int s = 0; s <= t; ++s) {
        float inner = 0.f;
        for (int bb = 0; bb < W; ++bb) inner += PQ[(size_t)t * NP + s + bb] * Dl[((size_t)s * W + bb) * dv + cc];
        acc += expf(g[t] - g[s]) * inner;
      }
      reinterpret_cast<Tin*>(a.o)[(((size_t)b * T + t) * a.H + h) * dv + cc] = from_f32<Tin>(acc);
    } else {
      size_t k = i - nO;
      int d = (int)(k / dv), cc = (int)(k % dv);
      float acc = 0.f;
      for (int s = 0; s < T; ++s) {
        float inner = 0.f;
        for (int bb = 0; bb < W; ++bb) inner += Xw[(size_t)(s + bb) * dk + d] * Dl[((size_t)s * W + bb) * dv + cc];
        acc += expf(g[T - 1] - g[s]) * inner;
      }
      S_final[(size_t)bh * dk * dv + k] = acc;
    }
  }
}

template <typename Tin>
int launch_mp(const FwdArgs& a, float* S_final) {
  float* ws = reinterpret_cast<float*>(a.ws);
  const int BH = a.B * a.H;
  mp_prep_kernel<Tin><<<BH, kMpThreads, 0, a.stream>>>(a, ws);
  mp_gram_kernel<Tin><<<dim3(64, BH), kMpThreads, 0, a.stream>>>(a, ws);
  mp_solve_kernel<Tin><<<dim3((a.dv + 31) / 32, BH), kMpThreads, 0, a.stream>>>(a, ws);
  mp_out_kernel<Tin><<<dim3(64, BH), kMpThreads, 0, a.stream>>>(a, ws, S_final);
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace

size_t masked_parallel_ws_bytes(int B, int T, int H, int dk, int dv, int W) {
  return (size_t)B * H * mp_layout(T, dk, dv, W).total * sizeof(float);
}

int launch_masked_parallel(const FwdArgs& a) {
  return a.dtype == FALCON_BF16 ? launch_mp<__nv_bfloat16>(a, a.S_out) : launch_mp<float>(a, a.S_out);
}

}  // namespace falcon
