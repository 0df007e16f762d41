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

// Scales of phi (per-token L2 normalisation) of q and k, by the first warp;
// 1 without the prologue flag.
template <typename Tin>
__device__ __forceinline__ void phi_scales(const FwdArgs& a, size_t bhi, int tid, float* out2) {
  if (!(a.prologue & FALCON_PROLOGUE_L2NORM_QK)) {
    if (tid == 0) { out2[0] = 1.f; out2[1] = 1.f; }
    return;
  }
  if (tid < 32) {
    float sq = 0.f, sk = 0.f;
    for (int d = tid; d < a.dk; d += 32) {
      const float q = ldv<Tin>(a.q, bhi * a.dk + d), k = ldv<Tin>(a.k, bhi * a.dk + d);
      sq = fmaf(q, q, sq);
      sk = fmaf(k, k, sk);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    if (tid == 0) {
      out2[0] = 1.f / fmaxf(sqrtf(sq), 1e-12f);
      out2[1] = 1.f / fmaxf(sqrtf(sk), 1e-12f);
    }
  }
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
  phi_scales<Tin>(a, bhi, tid, misc + 1);
  __syncthreads();
  const float sq = misc[1], sk = misc[2];
  // window slot w (oldest first): pair p = pos - (W-1) + w; the newest slot
  // is the current pair (x = k_prev, v = v_t)
  for (int i = tid; i < W * dk; i += kRecThreads) {
    int w = i / dk, d = i % dk;
    int64_t p = pos - Wr + w;
    float x = 0.f;
    if (p >= a.shift) {
      if (w == Wr) x = a.shift ? ldv<Tin>(a.kprev_out, bhi * dk + d) : sk * ldv<Tin>(a.k, bhi * dk + d);
      else x = ldv<Tin>(a.winx_out, (bhi * Wr + ring_slot(p, Wr)) * dk + d);
    }
    xw[i] = x;
  }
  for (int i = tid; i < W * dv; i += kRecThreads) {
    int w = i / dv, d = i % dv;
    int64_t p = pos - Wr + w;
    float x = 0.f;
    if (p >= a.shift) {
      if (w == Wr) x = ldv<Tin>(a.v, bhi * dv + d);
      else x = ldv<Tin>(a.winv_out, (bhi * Wr + ring_slot(p, Wr)) * dv + d);
    }
    vw[i] = x;
  }
  for (int d = tid; d < dk; d += kRecThreads) qv[d] = sq * ldv<Tin>(a.q, bhi * dk + d);
  for (int w = tid; w < W; w += kRecThreads) pv[w] = (pos - Wr + w >= a.shift) ? 1.f : 0.f;
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
  if (tid == 0) misc[0] = gate_gamma(a.lam[bhi], a.eps_gamma, a.prologue);
  for (int i = tid; i < (perch ? dv : 1); i += kRecThreads) {
    float n = 0.f, e = 0.f;
    for (int w = 0; w < W; ++w) { n += pv[w]; e += pv[w] * xn[w]; }
    float c = 0.f;
    if (n > 0.f) {
      float bt = gate_beta(perch ? a.beta[bhi * dv + i] : a.beta[bhi], a.prologue);
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
    const bool ok = pos >= a.shift;
    for (int d = tid; d < dk; d += kRecThreads)
      reinterpret_cast<Tin*>(a.winx_out)[(bhi * Wr + slot) * dk + d] =
          from_f32<Tin>(ok ? xw[Wr * dk + d] : 0.f);
    for (int d = tid; d < dv; d += kRecThreads)
      reinterpret_cast<Tin*>(a.winv_out)[(bhi * Wr + slot) * dv + d] =
          from_f32<Tin>(ok ? vw[Wr * dv + d] : 0.f);
  }
  for (int d = tid; d < dk; d += kRecThreads)
    reinterpret_cast<Tin*>(a.kprev_out)[bhi * dk + d] =
        (a.prologue & FALCON_PROLOGUE_L2NORM_QK) ? from_f32<Tin>(sk * ldv<Tin>(a.k, bhi * dk + d))
                                                  : reinterpret_cast<const Tin*>(a.k)[bhi * dk + d];
  if (tid == 0) a.pos_out[bhi] = pos + 1;
}

// Bandwidth-shaped variant for d_k = d_v in {64, 128}: float4 state
// accesses (every warp moves whole 256/512-byte rows), partial predictions
// reduced with shuffles and one shared-memory pass, two CTA barriers.
// Thread t owns 4 value columns (quad t % NQ) of the rows rg + RGS * i.
// (d = 64: at most 64 registers a thread so that eight CTAs share an SM and
// keep eight states in flight per SM)
template <typename Tin, int D, int NT, int MAXW>
__global__ void __launch_bounds__(NT, D == 64 ? 8 : 1) recurrent_step_vec_kernel(FwdArgs a) {
  constexpr int NQ = D / 4;          // column quads
  constexpr int RGS = NT / NQ;       // row groups
  constexpr int RPT = D / RGS;       // rows per thread
  constexpr int GPW = 32 / NQ;       // row groups inside one warp
  constexpr int NW = NT / 32;
  __shared__ float xw[MAXW][D];      // window keys (oldest first; last = current pair)
  __shared__ float vw[MAXW][D];
  __shared__ float qv[D];
  __shared__ float pv[MAXW], xq[MAXW], xn[MAXW];
  __shared__ float4 red[NW][MAXW + 1][NQ];
  __shared__ float scl[2];
  const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = tid % NQ, rg = tid / NQ;
  const int W = a.W, Wr = W - 1;
  const size_t bhi = (size_t)bh;
  float4* Sg = reinterpret_cast<float4*>(a.S_out + bhi * D * D);
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = Sg[(size_t)(rg + RGS * i) * NQ + cq];

  const int64_t pos = a.pos_out[bhi];
  phi_scales<Tin>(a, bhi, tid, scl);
  __syncthreads();
  const float sq = scl[0], sk = scl[1];
  for (int i = tid; i < W * D; i += NT) {
    const int w = i / D, d = i % D;
    const int64_t p = pos - Wr + w;
    float x = 0.f, v = 0.f;
    if (p >= a.shift) {
      if (w == Wr) {
        x = a.shift ? to_f32(reinterpret_cast<const Tin*>(a.kprev_out)[bhi * D + d])
                    : sk * to_f32(reinterpret_cast<const Tin*>(a.k)[bhi * D + d]);
        v = to_f32(reinterpret_cast<const Tin*>(a.v)[bhi * D + d]);
      } else {
        const size_t o = (bhi * Wr + ring_slot(p, Wr)) * D + d;
        x = to_f32(reinterpret_cast<const Tin*>(a.winx_out)[o]);
        v = to_f32(reinterpret_cast<const Tin*>(a.winv_out)[o]);
      }
    }
    xw[w][d] = x;
    vw[w][d] = v;
  }
  for (int d = tid; d < D; d += NT) qv[d] = sq * to_f32(reinterpret_cast<const Tin*>(a.q)[bhi * D + d]);
  __syncthreads();
  for (int w = warp; w < W; w += NW) {  // x_j . q and ||x_j||^2
    float aq = 0.f, an = 0.f;
    for (int d = lane; d < D; d += 32) {
      const float x = xw[w][d];
      aq += x * qv[d];
      an += x * x;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      aq += __shfl_xor_sync(0xffffffffu, aq, o);
      an += __shfl_xor_sync(0xffffffffu, an, o);
    }
    if (lane == 0) {
      xq[w] = aq;
      xn[w] = an;
      pv[w] = (pos - Wr + w >= a.shift) ? 1.f : 0.f;
    }
  }
  // partial predictions S^T x_j (j < W) and S^T q over this thread's rows
  const bool additive = variant_additive(a.variant);
  for (int w = 0; w <= W; ++w) {
    if (additive && w < W) continue;
    const float* xv = (w < W) ? xw[w] : qv;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const float x = xv[rg + RGS * i];
      acc.x += s[i].x * x; acc.y += s[i].y * x; acc.z += s[i].z * x; acc.w += s[i].w * x;
    }
#pragma unroll
    for (int o = NQ; o < 32; o <<= 1) {
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
    }
    if (lane < NQ) red[warp][w][cq] = acc;
  }
  __syncthreads();
  // every thread forms the writes of its own 4 columns
  const float gamma = gate_gamma(a.lam[bhi], a.eps_gamma, a.prologue);
  const bool perch = variant_per_channel(a.variant);
  float n = 0.f, e = 0.f;
  for (int w = 0; w < W; ++w) { n += pv[w]; e += pv[w] * xn[w]; }
  float4 cf = make_float4(0.f, 0.f, 0.f, 0.f);
  if (n > 0.f) {
    const float den = a.eps + e / n;
    if (perch) {
      float4 bt = reinterpret_cast<const float4*>(a.beta + bhi * D)[cq];
      bt = make_float4(gate_beta(bt.x, a.prologue), gate_beta(bt.y, a.prologue), gate_beta(bt.z, a.prologue),
                       gate_beta(bt.w, a.prologue));
      cf = make_float4(bt.x / den / n, bt.y / den / n, bt.z / den / n, bt.w / den / n);
    } else {
      const float c = gate_beta(a.beta[bhi], a.prologue) / den / n;
      cf = make_float4(c, c, c, c);
    }
  }
  auto total = [&](int w) {
    float4 t = red[0][w][cq];
#pragma unroll
    for (int g = 1; g < NW; ++g) {
      const float4 u = red[g][w][cq];
      t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
    }
    return t;
  };
  float4 dl[MAXW];
  const float4 cqs = total(W);
  float4 o = make_float4(gamma * cqs.x, gamma * cqs.y, gamma * cqs.z, gamma * cqs.w);
#pragma unroll
  for (int w = 0; w < MAXW; ++w) {
    if (w >= W) break;
    const float4 v4 = *reinterpret_cast<const float4*>(&vw[w][4 * cq]);
    float4 r = v4;
    if (!additive) {
      const float4 pr = total(w);
      r = make_float4(v4.x - gamma * pr.x, v4.y - gamma * pr.y, v4.z - gamma * pr.z, v4.w - gamma * pr.w);
    }
    const float m = pv[w];
    dl[w] = make_float4(m * cf.x * r.x, m * cf.y * r.y, m * cf.z * r.z, m * cf.w * r.w);
    const float xqw = xq[w];
    o.x += xqw * dl[w].x; o.y += xqw * dl[w].y; o.z += xqw * dl[w].z; o.w += xqw * dl[w].w;
  }
  if (rg == 0) {
    Tin* op = reinterpret_cast<Tin*>(a.o) + bhi * D + 4 * cq;
    op[0] = from_f32<Tin>(o.x); op[1] = from_f32<Tin>(o.y);
    op[2] = from_f32<Tin>(o.z); op[3] = from_f32<Tin>(o.w);
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + RGS * i;
    float4 acc = make_float4(gamma * s[i].x, gamma * s[i].y, gamma * s[i].z, gamma * s[i].w);
#pragma unroll
    for (int w = 0; w < MAXW; ++w) {
      if (w >= W) break;
      const float x = xw[w][r];
      acc.x += x * dl[w].x; acc.y += x * dl[w].y; acc.z += x * dl[w].z; acc.w += x * dl[w].w;
    }
    Sg[(size_t)r * NQ + cq] = acc;
  }
  if (Wr > 0) {  // ring push of the current pair
    const int slot = ring_slot(pos, Wr);
    const bool ok = pos >= a.shift;
    for (int d = tid; d < D; d += NT) {
      reinterpret_cast<Tin*>(a.winx_out)[(bhi * Wr + slot) * D + d] = from_f32<Tin>(ok ? xw[Wr][d] : 0.f);
      reinterpret_cast<Tin*>(a.winv_out)[(bhi * Wr + slot) * D + d] = from_f32<Tin>(ok ? vw[Wr][d] : 0.f);
    }
  }
  for (int d = tid; d < D; d += NT)
    reinterpret_cast<Tin*>(a.kprev_out)[bhi * D + d] =
        (a.prologue & FALCON_PROLOGUE_L2NORM_QK)
            ? from_f32<Tin>(sk * to_f32(reinterpret_cast<const Tin*>(a.k)[bhi * D + d]))
            : reinterpret_cast<const Tin*>(a.k)[bhi * D + d];
  if (tid == 0) a.pos_out[bhi] = pos + 1;
}

// Column-per-thread variant for d_k = d_v = 64: one CTA of 64 threads per
// (b, h), thread j holding the state's value column S[:, j] in 64 registers.
// Its 64 loads are one 128-byte row slice per warp each (coalesced), issued
// before anything else; S^T x_j and S^T q are then sums over the thread's own
// registers (the window keys and the query broadcast from shared memory), so
// no reduction over the state crosses threads.  The only block-wide step is
// staging the few input rows (one barrier); the dot products of the inputs
// (x_j . q, |x_j|^2, the phi scales) are formed by each warp on its own.
template <typename Tin, int MAXW>
__global__ void __launch_bounds__(64, 8) recurrent_step_col_kernel(FwdArgs a) {
  constexpr int D = 64;
  __shared__ __align__(16) float xw[MAXW][D];  // window keys, oldest first; the last is the current pair
  __shared__ __align__(16) float qv[D];
  __shared__ float kr[D];                      // the current raw key
  const int j = threadIdx.x, lane = j & 31;
  const size_t bhi = blockIdx.x;
  const int W = a.W, Wr = W - 1;
  float* Sg = a.S_out + bhi * D * D + j;  // column j, rows r at r * D (in place)
  float s[D];
#pragma unroll
  for (int r = 0; r < D; ++r) s[r] = Sg[r * D];

  const int64_t pos = a.pos_out[bhi];
  // ring slot of window pair w (global index pos - Wr + w): (pos + w) mod Wr
  const int slot0 = Wr > 0 ? (int)(pos % Wr) : 0;
  const Tin* kin = reinterpret_cast<const Tin*>(a.k) + bhi * D;
  const float qraw = to_f32(reinterpret_cast<const Tin*>(a.q)[bhi * D + j]);
  const float kraw = to_f32(kin[j]);
  float vv[MAXW];  // this column's entry of each window value
  const float vcur = to_f32(reinterpret_cast<const Tin*>(a.v)[bhi * D + j]);  // the current pair's
#pragma unroll
  for (int w = 0; w < MAXW; ++w) {
    if (w >= W) break;
    const int64_t p = pos - Wr + w;
    float x = 0.f, v = 0.f;
    if (p >= a.shift) {
      if (w == Wr) {
        x = a.shift ? to_f32(reinterpret_cast<const Tin*>(a.kprev_out)[bhi * D + j]) : kraw;
        v = vcur;
      } else {
        const int sl = slot0 + w >= Wr ? slot0 + w - Wr : slot0 + w;
        const size_t o = (bhi * Wr + sl) * D + j;
        x = to_f32(reinterpret_cast<const Tin*>(a.winx_out)[o]);
        v = to_f32(reinterpret_cast<const Tin*>(a.winv_out)[o]);
      }
    }
    xw[w][j] = x;
    vv[w] = v;
  }
  qv[j] = qraw;
  kr[j] = kraw;
  __syncthreads();
  // per-warp sums over all 64 entries: lane l takes entries l and l + 32
  auto wsum = [&](float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
  };
  float sq = 1.f, sk = 1.f;  // phi scales (prologue), 1 otherwise
  if (a.prologue & FALCON_PROLOGUE_L2NORM_QK) {
    const float q0 = qv[lane], q1 = qv[lane + 32], k0 = kr[lane], k1 = kr[lane + 32];
    sq = 1.f / fmaxf(sqrtf(wsum(q0 * q0 + q1 * q1)), 1e-12f);
    sk = 1.f / fmaxf(sqrtf(wsum(k0 * k0 + k1 * k1)), 1e-12f);
  }
  // the current key enters the window as phi(k) under same-step pairing
  const float xsc_cur = a.shift ? 1.f : sk;
  // x_w . q for every window slot and the window's total key energy (a
  // slot whose pair does not exist holds a zero key): the partial sums of
  // all slots first, then their warp reductions side by side
  float xq[MAXW], n = 0.f, e = 0.f;
#pragma unroll
  for (int w = 0; w < MAXW; ++w) {
    xq[w] = 0.f;
    if (w < W) {
      const float sc = (w == Wr) ? xsc_cur : 1.f;
      const float x0 = sc * xw[w][lane], x1 = sc * xw[w][lane + 32];
      xq[w] = x0 * qv[lane] + x1 * qv[lane + 32];
      e = fmaf(x0, x0, fmaf(x1, x1, e));
      n += (pos - Wr + w >= a.shift) ? 1.f : 0.f;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int w = 0; w < MAXW; ++w) xq[w] += __shfl_xor_sync(0xffffffffu, xq[w], o);
    e += __shfl_xor_sync(0xffffffffu, e, o);
  }
#pragma unroll
  for (int w = 0; w < MAXW; ++w) xq[w] *= sq;
  const float gamma = gate_gamma(a.lam[bhi], a.eps_gamma, a.prologue);
  float cf = 0.f;  // eta / n for this column
  if (n > 0.f) {
    const float bt = gate_beta(variant_per_channel(a.variant) ? a.beta[bhi * D + j] : a.beta[bhi], a.prologue);
    cf = bt / (a.eps + e / n) / n;
  }
  // S^T q and, for the regression variants, S^T x_w: this column's sums,
  // the window's sums advanced together row by row (independent chains)
  const bool additive = variant_additive(a.variant);
  float c = 0.f, aw[MAXW];
#pragma unroll
  for (int w = 0; w < MAXW; ++w) aw[w] = 0.f;
  const int Wp = additive ? 0 : W;  // window sums needed
#pragma unroll
  for (int r = 0; r < D; r += 4) {
    const float4 q4 = *reinterpret_cast<const float4*>(&qv[r]);
    c = fmaf(s[r], q4.x, c); c = fmaf(s[r + 1], q4.y, c); c = fmaf(s[r + 2], q4.z, c); c = fmaf(s[r + 3], q4.w, c);
#pragma unroll
    for (int w = 0; w < MAXW; ++w) {
      if (w < Wp) {
        const float4 x4 = *reinterpret_cast<const float4*>(&xw[w][r]);
        aw[w] = fmaf(s[r], x4.x, aw[w]); aw[w] = fmaf(s[r + 1], x4.y, aw[w]);
        aw[w] = fmaf(s[r + 2], x4.z, aw[w]); aw[w] = fmaf(s[r + 3], x4.w, aw[w]);
      }
    }
  }
  c *= sq;
  float dl[MAXW];
  float o = gamma * c;
#pragma unroll
  for (int w = 0; w < MAXW; ++w) {
    if (w >= W) break;
    float r_w = vv[w];
    if (!additive) r_w -= gamma * (w == Wr ? aw[w] * xsc_cur : aw[w]);
    const bool ok = pos - Wr + w >= a.shift;
    dl[w] = ok ? cf * r_w : 0.f;
    o = fmaf(xq[w], dl[w], o);
  }
  reinterpret_cast<Tin*>(a.o)[bhi * D + j] = from_f32<Tin>(o);
  // S' = gamma S + sum_w x_w dl_w^T, column j, written back in place (the
  // current key's row sits unscaled in shared memory: its scale goes to dl)
#pragma unroll
  for (int w = 0; w < MAXW; ++w)
    if (w == Wr) dl[w] *= xsc_cur;
#pragma unroll
  for (int r = 0; r < D; r += 4) {
    float4 acc = make_float4(gamma * s[r], gamma * s[r + 1], gamma * s[r + 2], gamma * s[r + 3]);
#pragma unroll
    for (int w = 0; w < MAXW; ++w) {
      if (w >= W) break;
      const float4 x4 = *reinterpret_cast<const float4*>(&xw[w][r]);
      acc.x = fmaf(x4.x, dl[w], acc.x); acc.y = fmaf(x4.y, dl[w], acc.y);
      acc.z = fmaf(x4.z, dl[w], acc.z); acc.w = fmaf(x4.w, dl[w], acc.w);
    }
    Sg[r * D] = acc.x;
    Sg[(r + 1) * D] = acc.y;
    Sg[(r + 2) * D] = acc.z;
    Sg[(r + 3) * D] = acc.w;
  }
  // carry: ring push of the current pair, the new k_prev (phi(k) under the
  // prologue), the position
  const Tin kout = from_f32<Tin>((a.prologue & FALCON_PROLOGUE_L2NORM_QK) ? sk * kraw : kraw);
  if (Wr > 0) {
    const int slot = slot0;
    const bool ok = pos >= a.shift;
    reinterpret_cast<Tin*>(a.winx_out)[(bhi * Wr + slot) * D + j] =
        from_f32<Tin>(ok ? xsc_cur * xw[Wr][j] : 0.f);
    reinterpret_cast<Tin*>(a.winv_out)[(bhi * Wr + slot) * D + j] = from_f32<Tin>(ok ? vcur : 0.f);
  }
  reinterpret_cast<Tin*>(a.kprev_out)[bhi * D + j] =
      (a.prologue & FALCON_PROLOGUE_L2NORM_QK) ? kout : kin[j];
  if (j == 0) a.pos_out[bhi] = pos + 1;
}

template <typename Tin, int EPT>
int launch_rec(const FwdArgs& a) {
  const int RG = kRecThreads / a.dv;
  const size_t smem = sizeof(float) * ((size_t)a.W * a.dk + (size_t)a.W * a.dv + a.dk + 3 * a.W +
                                       a.dv + (size_t)RG * (a.W + 1) * a.dv + (size_t)a.W * a.dv + 4);
  if (smem > 227 * 1024) return FALCON_ERR_UNSUPPORTED;
  auto k = recurrent_step_kernel<Tin, EPT>;
  if (!set_smem_limit(reinterpret_cast<const void*>(k), smem))
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

template <typename Tin, int D, int NT>
int launch_rec_vec(const FwdArgs& a) {
  if (a.W <= 1) {
    recurrent_step_vec_kernel<Tin, D, NT, 1><<<a.B * a.H, NT, 0, a.stream>>>(a);
  } else if (a.W <= 8) {
    recurrent_step_vec_kernel<Tin, D, NT, 8><<<a.B * a.H, NT, 0, a.stream>>>(a);
  } else {
    return -100;  // not covered: the generic kernel takes it
  }
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

template <typename Tin>
int launch_rec_col(const FwdArgs& a) {
  if (a.W <= 1)
    recurrent_step_col_kernel<Tin, 1><<<a.B * a.H, 64, 0, a.stream>>>(a);
  else
    recurrent_step_col_kernel<Tin, 8><<<a.B * a.H, 64, 0, a.stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

int launch_recurrent_step(const FwdArgs& a) {
  if (a.dk == 64 && a.dv == 64 && a.W <= 8)
    return a.dtype == FALCON_BF16 ? launch_rec_col<__nv_bfloat16>(a) : launch_rec_col<float>(a);
  if (a.dk == a.dv && (a.dk == 64 || a.dk == 128) && a.W <= 8) {
    int st;
    if (a.dk == 64)
      st = a.dtype == FALCON_BF16 ? launch_rec_vec<__nv_bfloat16, 64, 128>(a) : launch_rec_vec<float, 64, 128>(a);
    else
      st = a.dtype == FALCON_BF16 ? launch_rec_vec<__nv_bfloat16, 128, 256>(a) : launch_rec_vec<float, 128, 256>(a);
    if (st != -100) return st;
  }
  // the thread layout needs dv | 256 and dk*dv >= 256
  if (kRecThreads % a.dv != 0 || a.dk * a.dv < kRecThreads) return FALCON_ERR_UNSUPPORTED;
  return a.dtype == FALCON_BF16 ? launch_rec_t<__nv_bfloat16>(a) : launch_rec_t<float>(a);
}

}  // namespace falcon
