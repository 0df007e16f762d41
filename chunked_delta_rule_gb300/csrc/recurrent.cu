// Recurrent form, one decode token per (b, h) [FW 三种等价形式 (inference
// form with an O(1) state per step); JC 三种视角看同一个更新].
//
// One CTA per (b, h).  The fp32 state S (dk x dv) is read from HBM once and
// written once: every thread keeps its share of S in registers while the
// CTA forms the window predictions a_j = S^T x_j and c = S^T q (partial sums
// reduced through shared memory), then
//   d_j = coef_j * (v_j - gamma a_j)          (additive variants: coef_j v_j)
//   S'  = gamma S + sum_j x_j d_j^T
//   o   = S'^T q = gamma c + sum_j (x_j . q) d_j
// so o needs no second pass over S.  The carry is updated in place:
// k_prev <- k, the current pair enters ring slot pos mod (W-1), pos += 1.
// The step is memory-bound (HBM traffic ~ 8 dk dv bytes per (b, h)).

#include "common.cuh"

namespace falcon {

namespace {

constexpr int kRecThreads = 256;

template <typename Tin>
__device__ __forceinline__ float ldv(const void* p, size_t i) {
  return to_f32(reinterpret_cast<const Tin*>(p)[i]);
}

template <typename Tin, int EPT>
__global__ void __launch_bounds__(kRecThreads) recurrent_step_kernel(FwdArgs a) {
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  const int bh = blockIdx.x;
  const int b = bh / a.H, h = bh % a.H;
  const int tid = threadIdx.x;
  const int dk = a.dk, dv = a.dv, W = a.W;
  const int RG = kRecThreads / dv;  // row groups (threads sharing one column)
  const int col = tid % dv;
  const int rg = tid / dv;
  const size_t bhi = (size_t)b * a.H + h;
  float* Sg = a.S_out + bhi * dk * dv;  // in place: S_out == S_in

  // issue the state loads first; they are the traffic that matters
  float s[EPT];
#pragma unroll
  for (int i = 0; i < EPT; ++i) s[i] = Sg[(size_t)(rg + RG * i) * dv + col];

  float* xw = sm;                       // [W][dk]
  float* vw = xw + W * dk;              // [W][dv]
  float* qv = vw + W * dv;              // [dk]
  float* pv = qv + dk;                  // [W] pair exists
  float* xq = pv + W;                   // [W] x_j . q
  float* xn = xq + W;                   // [W] ||x_j||^2
  float* cf = xn + W;                   // [dv] coefficient eta/n (per channel) or [1]
  float* red = cf + dv;                 // [RG][W+1][dv] partial sums
  float* dl = red + RG * (W + 1) * dv;  // [W][dv] writes d_j
  float* misc = dl + W * dv;            // gamma

  const int64_t pos = a.pos_out[bhi];
  const int Wr = W - 1;
  // window slot w (oldest first): pair p = pos - (W-1) + w; the newest slot
  // is the current pair (x = k_prev, v = v_t)
  for (int i = tid; i < W * dk; i += kRecThreads) {
    int w = i / dk, d = i % dk;
    int64_t p = pos - Wr + w;
    float x = 0.f;
    if (p >= 1) {
      if (w == Wr) x = ldv<Tin>(a.kprev_out, bhi * dk + d);
      else x = ldv<Tin>(a.winx_out, (bhi * Wr + ring_slot(p, Wr)) * dk + d);
    }
    xw[i] = x;
  }
  for (int i = tid; i < W * dv; i += kRecThreads) {
    int w = i / dv, d = i % dv;
    int64_t p = pos - Wr + w;
    float x = 0.f;
    if (p >= 1) {
      if (w == Wr) x = ldv<Tin>(a.v, bhi * dv + d);
      else x = ldv<Tin>(a.winv_out, (bhi * Wr + ring_slot(p, Wr)) * dv + d);
    }
    vw[i] = x;
  }
  for (int d = tid; d < dk; d += kRecThreads) qv[d] = ldv<Tin>(a.q, bhi * dk + d);
  for (int w = tid; w < W; w += kRecThreads) pv[w] = (pos - Wr + w >= 1) ? 1.f : 0.f;
  __syncthreads();
  // dot products x_j . q and ||x_j||^2: one warp per window slot
  {
    const int warp = tid / 32, lane = tid % 32;
    for (int w = warp; w < W; w += kRecThreads / 32) {
      float aq = 0.f, an = 0.f;
      for (int d = lane; d < dk; d += 32) {
        float x = xw[w * dk + d];
        aq += x * qv[d];
        an += x * x;
      }
      for (int o = 16; o > 0; o >>= 1) {
        aq += __shfl_xor_sync(0xffffffffu, aq, o);
        an += __shfl_xor_sync(0xffffffffu, an, o);
      }
      if (lane == 0) { xq[w] = aq; xn[w] = an; }
    }
  }
  __syncthreads();
  const bool perch = variant_per_channel(a.variant);
  if (tid == 0) misc[0] = fminf(fmaxf(1.0f - a.lam[bhi], a.eps_gamma), 1.0f);
  for (int i = tid; i < (perch ? dv : 1); i += kRecThreads) {
    float n = 0.f, e = 0.f;
    for (int w = 0; w < W; ++w) { n += pv[w]; e += pv[w] * xn[w]; }
    float c = 0.f;
    if (n > 0.f) {
      float bt = perch ? a.beta[bhi * dv + i] : a.beta[bhi];
      c = bt / (a.eps + e / n) / n;
    }
    cf[i] = c;
  }
  // partial predictions over this thread's rows
  const bool additive = variant_additive(a.variant);
  {
    float pc = 0.f;
#pragma unroll
    for (int i = 0; i < EPT; ++i) pc += s[i] * qv[rg + RG * i];
    red[(rg * (W + 1) + W) * dv + col] = pc;
    if (!additive) {
      for (int w = 0; w < W; ++w) {
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < EPT; ++i) p += s[i] * xw[w * dk + rg + RG * i];
        red[(rg * (W + 1) + w) * dv + col] = p;
      }
    }
  }
  __syncthreads();
  const float gamma = misc[0];
  // writes d_j and the output
  for (int i = tid; i < W * dv; i += kRecThreads) {
    int w = i / dv, cc = i % dv;
    float c = cf[perch ? cc : 0] * pv[w];
    float r = vw[i];
    if (!additive) {
      float p = 0.f;
      for (int g = 0; g < RG; ++g) p += red[(g * (W + 1) + w) * dv + cc];
      r -= gamma * p;
    }
    dl[i] = c * r;
  }
  __syncthreads();
  if (tid < dv) {
    float cq = 0.f;
    for (int g = 0; g < RG; ++g) cq += red[(g * (W + 1) + W) * dv + tid];
    float o = gamma * cq;
    for (int w = 0; w < W; ++w) o += xq[w] * dl[w * dv + tid];
    reinterpret_cast<Tin*>(a.o)[bhi * dv + tid] = from_f32<Tin>(o);
  }
  // state update, written back in place
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int r = rg + RG * i;
    float acc = gamma * s[i];
    for (int w = 0; w < W; ++w) acc += xw[w * dk + r] * dl[w * dv + col];
    Sg[(size_t)r * dv + col] = acc;
  }
  // carry: ring push of the current pair, new k_prev, position
  if (Wr > 0) {
    const int slot = ring_slot(pos, Wr);
    const bool ok = pos >= 1;
    for (int d = tid; d < dk; d += kRecThreads)
      reinterpret_cast<Tin*>(a.winx_out)[(bhi * Wr + slot) * dk + d] =
          from_f32<Tin>(ok ? xw[Wr * dk + d] : 0.f);
    for (int d = tid; d < dv; d += kRecThreads)
      reinterpret_cast<Tin*>(a.winv_out)[(bhi * Wr + slot) * dv + d] =
          from_f32<Tin>(ok ? vw[Wr * dv + d] : 0.f);
  }
  for (int d = tid; d < dk; d += kRecThreads)
    reinterpret_cast<Tin*>(a.kprev_out)[bhi * dk + d] =
        reinterpret_cast<const Tin*>(a.k)[bhi * dk + d];
  if (tid == 0) a.pos_out[bhi] = pos + 1;
}

template <typename Tin, int EPT>
int launch_rec(const FwdArgs& a) {
  const int RG = kRecThreads / a.dv;
  const size_t smem = sizeof(float) * ((size_t)a.W * a.dk + (size_t)a.W * a.dv + a.dk + 3 * a.W +
                                       a.dv + (size_t)RG * (a.W + 1) * a.dv + (size_t)a.W * a.dv + 4);
  if (smem > 227 * 1024) return FALCON_ERR_UNSUPPORTED;
  auto k = recurrent_step_kernel<Tin, EPT>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return FALCON_ERR_CUDA;
  k<<<a.B * a.H, kRecThreads, smem, a.stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

template <typename Tin>
int launch_rec_t(const FwdArgs& a) {
  // elements per thread: dk*dv / 256, for d in {16, 32, 64, 128}
  switch (a.dk * a.dv / kRecThreads) {
    case 1: return launch_rec<Tin, 1>(a);
    case 2: return launch_rec<Tin, 2>(a);
    case 4: return launch_rec<Tin, 4>(a);
    case 8: return launch_rec<Tin, 8>(a);
    case 16: return launch_rec<Tin, 16>(a);
    case 32: return launch_rec<Tin, 32>(a);
    case 64: return launch_rec<Tin, 64>(a);
    default: return FALCON_ERR_UNSUPPORTED;
  }
}

}  // namespace

int launch_recurrent_step(const FwdArgs& a) {
  // the thread layout needs dv | 256 and dk*dv >= 256
  if (kRecThreads % a.dv != 0 || a.dk * a.dv < kRecThreads) return FALCON_ERR_UNSUPPORTED;
  return a.dtype == FALCON_BF16 ? launch_rec_t<__nv_bfloat16>(a) : launch_rec_t<float>(a);
}

}  // namespace falcon
