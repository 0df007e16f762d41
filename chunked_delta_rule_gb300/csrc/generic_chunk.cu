// Portable chunk-parallel forward on CUDA cores (fp32 arithmetic), every
// variant.  It is the fp32-input path and the fallback for shapes the
// tensor-core path does not cover.
//
// Chunked form [FW 三种等价形式; JC 三种视角看同一个更新]: one CTA owns one
// (b, h) pair and a slice of value channels, and walks the sequence in blocks
// of c steps carrying the fp32 state S (dk x dvs) in shared memory.  Inside a
// block the writes are solved all at once from the Gram matrix of the block's
// keys: with Z_s the shrunk state before step s and rho_{s,a} the residual of
// window pair a at step s,
//   rho_{s,a} = v_{j} - Gamma_s (S0^T x_j) - sum_{s'<s} exp(g_s - g_{s'}) sum_b (x_j . x_{j'}) d_{s',b}
//   d_{s,a}   = coef_{s,a} * rho_{s,a}          (coef = eta_s / n_s, zero for missing pairs)
// (j = pair of slot a at step s, j' = pair of slot b at step s').  This is a
// unit lower-triangular system in (s, a) solved by forward substitution; for
// W = 1 it is the WY / TriSolve chunk form of Falcon-1 and the row-scaled
// batched solve of Falcon-2 (eta per channel, L shared)
// [JC Falcon家族六个变体各管一段].  Then
//   o_s   = Gamma_s S0^T q_s + sum_{s'<=s} exp(g_s - g_{s'}) sum_b (q_s . x_{j'}) d_{s',b}
//   S_end = Gamma_end S0 + sum_{s'} exp(g_end - g_{s'}) sum_b x_{j'} d_{s',b}^T
// with g the in-block cumulative log of the clamped decay
// [JC 数学上的稳定阀门:正衰减钳制]; decays are only ever formed as
// exp(g_s - g_s') with s' <= s, so nothing overflows.

#include <algorithm>

#include "common.cuh"

namespace falcon {

namespace {

constexpr int kThreads = 256;

struct GenLayout {
  int NP;  // pairs touched by a block: c + W - 1
  size_t Xw, Vw, Qb, S, XS, QS, Gk, PQ, Dm, Dl, coef, gl, Gam, pval, xn, total;
};

__host__ __device__ inline GenLayout gen_layout(int dk, int dvs, int c, int W) {
  GenLayout L;
  L.NP = c + W - 1;
  size_t off = 0;
  auto take = [&](size_t n) { size_t o = off; off += (n + 3) & ~size_t(3); return o; };
  L.Xw = take((size_t)L.NP * (dk + 1));  // rows padded to dk + 1: no bank conflicts
  L.Vw = take((size_t)L.NP * dvs);
  L.Qb = take((size_t)c * (dk + 1));
  L.S = take((size_t)dk * dvs);
  L.XS = take((size_t)L.NP * dvs);
  L.QS = take((size_t)c * dvs);
  L.Gk = take((size_t)L.NP * L.NP);
  L.PQ = take((size_t)c * L.NP);
  L.Dm = take((size_t)c * c);
  L.Dl = take((size_t)c * W * dvs);
  L.coef = take((size_t)c * dvs);
  L.gl = take((size_t)c);
  L.Gam = take((size_t)c);
  L.pval = take((size_t)L.NP);
  L.xn = take((size_t)L.NP);
  L.total = off;
  return L;
}

template <typename Tin>
__device__ __forceinline__ float ld(const void* p, size_t i) {
  return to_f32(reinterpret_cast<const Tin*>(p)[i]);
}

// Key x_j and value v_j (value columns [c0, c0+ncols)) of local pair j.
template <typename Tin>
__device__ __forceinline__ float pair_key(const FwdArgs& a, int b, int h, int j, int col,
                                          int64_t pos) {
  if (j >= a.shift) return ld<Tin>(a.k, (((size_t)b * a.T + (j - a.shift)) * a.H + h) * a.dk + col);
  if (j == 0) return a.kprev_in ? ld<Tin>(a.kprev_in, ((size_t)b * a.H + h) * a.dk + col) : 0.f;
  if (a.W > 1 && a.winx_in) {
    int slot = ring_slot(pos + j, a.W - 1);
    return ld<Tin>(a.winx_in, (((size_t)b * a.H + h) * (a.W - 1) + slot) * a.dk + col);
  }
  return 0.f;
}

template <typename Tin>
__device__ __forceinline__ float pair_value(const FwdArgs& a, int b, int h, int j, int col,
                                            int64_t pos) {
  if (j >= 0) return ld<Tin>(a.v, (((size_t)b * a.T + j) * a.H + h) * a.dv + col);
  if (a.W > 1 && a.winv_in) {
    int slot = ring_slot(pos + j, a.W - 1);
    return ld<Tin>(a.winv_in, (((size_t)b * a.H + h) * (a.W - 1) + slot) * a.dv + col);
  }
  return 0.f;
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) generic_chunk_kernel(FwdArgs a, int c, int dvs) {
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  const int slice = blockIdx.y;
  const int bh = blockIdx.x;
  const int b = bh / a.H, h = bh % a.H;
  const int c0 = slice * dvs;  // first value channel of this CTA
  const int ncol = min(dvs, a.dv - c0);
  const int tid = threadIdx.x;
  const int dk = a.dk, W = a.W, T = a.T;
  const bool additive = variant_additive(a.variant);
  const bool perch = variant_per_channel(a.variant);
  const GenLayout L = gen_layout(dk, dvs, c, W);
  const int NP = L.NP;
  const int LX = dk + 1;  // padded row stride of Xw and Qb
  float* Xw = sm + L.Xw;
  float* Vw = sm + L.Vw;
  float* Qb = sm + L.Qb;
  float* S = sm + L.S;
  float* XS = sm + L.XS;
  float* QS = sm + L.QS;
  float* Gk = sm + L.Gk;
  float* PQ = sm + L.PQ;
  float* Dm = sm + L.Dm;
  float* Dl = sm + L.Dl;
  float* coef = sm + L.coef;
  float* gl = sm + L.gl;
  float* Gam = sm + L.Gam;
  float* pval = sm + L.pval;
  float* xn = sm + L.xn;

  const int64_t pos = a.pos_in ? a.pos_in[(size_t)b * a.H + h] : 0;

  for (int i = tid; i < dk * dvs; i += kThreads) {
    int r = i / dvs, col = i % dvs;
    S[i] = (a.S_in && col < ncol) ? a.S_in[(((size_t)b * a.H + h) * dk + r) * a.dv + c0 + col] : 0.f;
  }

  for (int s0 = 0; s0 < T; s0 += c) {
    __syncthreads();
    // ---- pairs of the block (slot a of step s0+sigma is pair s0+sigma-W+1+a)
    for (int i = tid; i < NP; i += kThreads) {
      int j = s0 - W + 1 + i;
      pval[i] = (pos + j >= a.shift && j < T) ? 1.f : 0.f;
    }
    for (int i = tid; i < NP * dk; i += kThreads) {
      int kk = i / dk, col = i % dk;
      int j = s0 - W + 1 + kk;
      bool ok = (pos + j >= a.shift) && (j < T);
      Xw[kk * LX + col] = ok ? pair_key<Tin>(a, b, h, j, col, pos) : 0.f;
    }
    for (int i = tid; i < NP * dvs; i += kThreads) {
      int kk = i / dvs, col = i % dvs;
      int j = s0 - W + 1 + kk;
      bool ok = (pos + j >= a.shift) && (j < T) && col < ncol;
      Vw[i] = ok ? pair_value<Tin>(a, b, h, j, c0 + col, pos) : 0.f;
    }
    for (int i = tid; i < c * dk; i += kThreads) {
      int sg = i / dk, col = i % dk;
      int s = s0 + sg;
      Qb[sg * LX + col] = (s < T) ? ld<Tin>(a.q, (((size_t)b * T + s) * a.H + h) * dk + col) : 0.f;
    }
    for (int sg = tid; sg < c; sg += kThreads) {
      int s = s0 + sg;
      gl[sg] = (s < T) ? clamped_log_decay(a.lam[((size_t)b * T + s) * a.H + h], a.eps_gamma) : 0.f;
    }
    __syncthreads();
    if (tid == 0) {  // inclusive cumulative log-decay inside the block
      float acc = 0.f;
      for (int sg = 0; sg < c; ++sg) { acc += gl[sg]; gl[sg] = acc; }
    }
    for (int kk = tid; kk < NP; kk += kThreads) {
      float acc = 0.f;
      for (int d = 0; d < dk; ++d) acc += Xw[kk * LX + d] * Xw[kk * LX + d];
      xn[kk] = acc;
    }
    __syncthreads();
    for (int i = tid; i < c * c; i += kThreads) {
      int r = i / c, q = i % c;
      Dm[i] = (q <= r) ? expf(gl[r] - gl[q]) : 0.f;
    }
    for (int sg = tid; sg < c; sg += kThreads) Gam[sg] = expf(gl[sg]);
    // ---- step coefficients coef = eta / n (window-averaged energy)
    for (int i = tid; i < c * (perch ? dvs : 1); i += kThreads) {
      int sg = perch ? i / dvs : i;
      int col = perch ? i % dvs : 0;
      int s = s0 + sg;
      float n = 0.f, e = 0.f;
      for (int aa = 0; aa < W; ++aa) { n += pval[sg + aa]; e += pval[sg + aa] * xn[sg + aa]; }
      float cf = 0.f;
      if (s < T && n > 0.f && (!perch || col < ncol)) {
        float bt = perch ? a.beta[(((size_t)b * T + s) * a.H + h) * a.dv + c0 + col]
                         : a.beta[((size_t)b * T + s) * a.H + h];
        cf = bt / (a.eps + e / n) / n;
      }
      coef[perch ? sg * dvs + col : sg] = cf;
    }
    // ---- Gram matrices and state products
    if (!additive) {
      for (int i = tid; i < NP * NP; i += kThreads) {
        int r = i / NP, q = i % NP;
        float acc = 0.f;
        for (int d = 0; d < dk; ++d) acc += Xw[r * LX + d] * Xw[q * LX + d];
        Gk[i] = acc;
      }
      for (int i = tid; i < NP * dvs; i += kThreads) {
        int kk = i / dvs, col = i % dvs;
        float acc = 0.f;
        for (int d = 0; d < dk; ++d) acc += Xw[kk * LX + d] * S[d * dvs + col];
        XS[i] = acc;
      }
    }
    for (int i = tid; i < c * NP; i += kThreads) {
      int r = i / NP, q = i % NP;
      float acc = 0.f;
      for (int d = 0; d < dk; ++d) acc += Qb[r * LX + d] * Xw[q * LX + d];
      PQ[i] = acc;
    }
    for (int i = tid; i < c * dvs; i += kThreads) {
      int sg = i / dvs, col = i % dvs;
      float acc = 0.f;
      for (int d = 0; d < dk; ++d) acc += Qb[sg * LX + d] * S[d * dvs + col];
      QS[i] = acc;
    }
    __syncthreads();
    // ---- the writes d_{s,a}
    if (additive) {
      for (int i = tid; i < c * W * dvs; i += kThreads) {
        int sg = i / (W * dvs), rem = i % (W * dvs), aa = rem / dvs, col = rem % dvs;
        float cf = coef[perch ? sg * dvs + col : sg];
        Dl[i] = pval[sg + aa] * cf * Vw[(sg + aa) * dvs + col];
      }
    } else {
      for (int sg = 0; sg < c; ++sg) {
        for (int i = tid; i < W * dvs; i += kThreads) {
          int aa = i / dvs, col = i % dvs;
          int kt = sg + aa;
          float r = Vw[kt * dvs + col] - Gam[sg] * XS[kt * dvs + col];
          for (int sp = 0; sp < sg; ++sp) {
            float acc = 0.f;
            for (int bb = 0; bb < W; ++bb)
              acc += Gk[kt * NP + sp + bb] * Dl[(sp * W + bb) * dvs + col];
            r -= Dm[sg * c + sp] * acc;
          }
          float cf = coef[perch ? sg * dvs + col : sg];
          Dl[(sg * W + aa) * dvs + col] = pval[kt] * cf * r;
        }
        __syncthreads();
      }
    }
    __syncthreads();
    // ---- outputs of the block
    for (int i = tid; i < c * dvs; i += kThreads) {
      int sg = i / dvs, col = i % dvs;
      int s = s0 + sg;
      if (s >= T || col >= ncol) continue;
      float acc = Gam[sg] * QS[i];
      for (int sp = 0; sp <= sg; ++sp) {
        float inner = 0.f;
        for (int bb = 0; bb < W; ++bb) inner += PQ[sg * NP + sp + bb] * Dl[(sp * W + bb) * dvs + col];
        acc += Dm[sg * c + sp] * inner;
      }
      size_t oi = (((size_t)b * T + s) * a.H + h) * a.dv + c0 + col;
      if (a.dtype == FALCON_BF16)
        reinterpret_cast<__nv_bfloat16*>(a.o)[oi] = __float2bfloat16_rn(acc);
      else
        reinterpret_cast<float*>(a.o)[oi] = acc;
    }
    // ---- state at the end of the block
    const float gend = Gam[c - 1];
    for (int i = tid; i < dk * dvs; i += kThreads) {
      int d = i / dvs, col = i % dvs;
      float acc = 0.f;
      for (int sp = 0; sp < c; ++sp) {
        float inner = 0.f;
        for (int bb = 0; bb < W; ++bb) inner += Xw[(sp + bb) * LX + d] * Dl[(sp * W + bb) * dvs + col];
        acc += Dm[(c - 1) * c + sp] * inner;
      }
      S[i] = gend * S[i] + acc;
    }
  }
  __syncthreads();
  // ---- carry out
  if (a.S_out) {
    for (int i = tid; i < dk * dvs; i += kThreads) {
      int r = i / dvs, col = i % dvs;
      if (col < ncol) a.S_out[(((size_t)b * a.H + h) * dk + r) * a.dv + c0 + col] = S[i];
    }
  }
  Tin* kpo = reinterpret_cast<Tin*>(a.kprev_out);
  if (slice == 0 && kpo) {
    for (int col = tid; col < dk; col += kThreads) {
      float x = (T >= 1) ? ld<Tin>(a.k, (((size_t)b * T + (T - 1)) * a.H + h) * dk + col)
                         : (a.kprev_in ? ld<Tin>(a.kprev_in, ((size_t)b * a.H + h) * dk + col) : 0.f);
      kpo[((size_t)b * a.H + h) * dk + col] = from_f32<Tin>(x);
    }
  }
  if (slice == 0 && a.pos_out && tid == 0) a.pos_out[(size_t)b * a.H + h] = pos + T;
  if (W > 1) {
    // slot s holds the pair p in [pos+T-Wr, pos+T-1] with p = s (mod Wr);
    // pairs with p < 1 do not exist and leave a zero slot
    const int Wr = W - 1;
    Tin* wxo = reinterpret_cast<Tin*>(a.winx_out);
    Tin* wvo = reinterpret_cast<Tin*>(a.winv_out);
    for (int64_t p = pos + T - Wr; p <= pos + T - 1; ++p) {
      const int j = (int)(p - pos);
      const int slot = (int)(((p % Wr) + Wr) % Wr);
      const bool ok = p >= a.shift;
      if (slice == 0 && wxo)
        for (int col = tid; col < dk; col += kThreads)
          wxo[(((size_t)b * a.H + h) * Wr + slot) * dk + col] =
              from_f32<Tin>(ok ? pair_key<Tin>(a, b, h, j, col, pos) : 0.f);
      if (wvo)
        for (int col = tid; col < ncol; col += kThreads)
          wvo[(((size_t)b * a.H + h) * Wr + slot) * a.dv + c0 + col] =
              from_f32<Tin>(ok ? pair_value<Tin>(a, b, h, j, c0 + col, pos) : 0.f);
    }
  }
}

inline int pow2_floor(int x) {
  int p = 1;
  while (p * 2 <= x) p *= 2;
  return p;
}

}  // namespace

static int generic_block_steps(int chunk, int W) {
  int c = chunk;
  if (W > 1) c = std::min(chunk, std::max(1, pow2_floor(std::max(1, 128 / W))));
  return c;
}

static int generic_slice(int dv) { return std::min(dv, 32); }

size_t generic_chunk_smem_bytes(int dk, int dvs, int c, int W) {
  return gen_layout(dk, dvs, c, W).total * sizeof(float);
}

int launch_generic_chunk(const FwdArgs& a) {
  const int c = generic_block_steps(a.chunk, a.W);
  const int dvs = generic_slice(a.dv);
  const size_t smem = generic_chunk_smem_bytes(a.dk, dvs, c, a.W);
  if (smem > 227 * 1024) return FALCON_ERR_UNSUPPORTED;
  dim3 grid(a.B * a.H, (a.dv + dvs - 1) / dvs);
  record_event(a, 0);
  if (a.dtype == FALCON_BF16) {
    auto k = generic_chunk_kernel<__nv_bfloat16>;
    if (!set_smem_limit(reinterpret_cast<const void*>(k), smem))
      return FALCON_ERR_CUDA;
    k<<<grid, kThreads, smem, a.stream>>>(a, c, dvs);
  } else {
    auto k = generic_chunk_kernel<float>;
    if (!set_smem_limit(reinterpret_cast<const void*>(k), smem))
      return FALCON_ERR_CUDA;
    k<<<grid, kThreads, smem, a.stream>>>(a, c, dvs);
  }
  record_event(a, 1);
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace falcon
