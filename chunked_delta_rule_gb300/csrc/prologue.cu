// The steps either side of the path [FW 三种等价形式 (phi(Q), phi(K)); JC
// 把记忆更新变成一次梯度下降 (beta, lambda as learned knobs)]:
//  - prologue_kernel: per (b, t, h) row, the feature map phi = per-token L2
//    normalisation of q and k (x / max(|x|, 1e-12), fp32, rounded to the
//    input dtype) and the gates from logits (beta = sigmoid(b),
//    lambda = sigmoid(a), so gamma = 1 - lambda = sigmoid(-a)), written as a
//    dense [B, T, H, .] batch.  For packed sequences (cu_seqlens) it also
//    lays sequence b's tokens at rows (b, 0 .. len_b - 1) and fills the rest
//    with beta = 0, lambda = 0 and zero q, k, v: such a step neither writes
//    nor decays, so the state after T padded steps is the state after len_b
//    (when the kernels after it skip the chunks past a sequence's last, only
//    the padding inside its last chunk is written).
//  - varlen_scatter_kernel: the outputs of the real rows back to the packed
//    layout;
//  - varlen_carry_kernel: the carry fields that depend on where a sequence
//    ends (last key, token count, window ring of the last W - 1 pairs).
// One warp per row; q and k norms by warp reductions.

#include "common.cuh"

namespace falcon {

namespace {

constexpr int kProWarps = 8;

__device__ __forceinline__ float sigmoidf(float x) { return 1.f / (1.f + __expf(-x)); }

template <typename Tin>
__device__ __forceinline__ const Tin* cptr(const void* p) { return reinterpret_cast<const Tin*>(p); }

// row index of token t of sequence b in the input layout, or -1 past its end
__device__ __forceinline__ long long src_row(const ProArgs& a, int b, int t) {
  if (!a.cu) return (long long)b * a.T + t;
  const int s = a.cu[b], e = a.cu[b + 1];
  return t < e - s ? (long long)s + t : -1;
}

template <typename Tin>
__global__ void __launch_bounds__(32 * kProWarps) prologue_kernel(ProArgs a) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kProWarps + (threadIdx.x >> 5);  // (b, t, h)
  const long long nrows = (long long)a.B * a.T * a.H;
  if (row >= nrows) return;
  const int h = (int)(row % a.H);
  const long long bt = row / a.H;
  const int t = (int)(bt % a.T), b = (int)(bt / a.T);
  const long long sr = src_row(a, b, t);
  const size_t dst = (size_t)row;
  Tin* qo = reinterpret_cast<Tin*>(a.qo);
  Tin* ko = reinterpret_cast<Tin*>(a.ko);
  Tin* vo = reinterpret_cast<Tin*>(a.vo);
  const int nb = a.perch ? a.dv : 1;
  if (sr < 0 && a.skip_tail) {  // a chunk past the sequence's last: read by no kernel
    const int len = a.cu[b + 1] - a.cu[b];
    if (t >= (len + 63) / 64 * 64) return;
  }
  if (sr < 0) {  // padding: a step that neither writes nor decays
    for (int i = lane; i < a.dk; i += 32) {
      qo[dst * a.dk + i] = from_f32<Tin>(0.f);
      ko[dst * a.dk + i] = from_f32<Tin>(0.f);
    }
    for (int i = lane; i < a.dv; i += 32) vo[dst * a.dv + i] = from_f32<Tin>(0.f);
    for (int i = lane; i < nb; i += 32) a.bo[dst * nb + i] = 0.f;
    if (lane == 0) a.lo[dst] = 0.f;
    return;
  }
  const size_t srow = (size_t)sr * a.H + h;
  const bool l2 = (a.flags & FALCON_PROLOGUE_L2NORM_QK) != 0;
  const bool logits = (a.flags & FALCON_PROLOGUE_GATE_LOGITS) != 0;
  for (int which = 0; which < 2; ++which) {  // q, then k
    const Tin* src = cptr<Tin>(which == 0 ? a.q : a.k) + srow * a.dk;
    Tin* out = which == 0 ? qo : ko;
    float x[4];
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = lane + 32 * e;
      x[e] = i < a.dk ? to_f32(src[i]) : 0.f;
      ss = fmaf(x[e], x[e], ss);
    }
    float scale = 1.f;
    if (l2) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      scale = 1.f / fmaxf(sqrtf(ss), 1e-12f);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = lane + 32 * e;
      if (i < a.dk) out[dst * a.dk + i] = from_f32<Tin>(x[e] * scale);
    }
  }
  for (int i = lane; i < a.dv; i += 32) vo[dst * a.dv + i] = cptr<Tin>(a.v)[srow * a.dv + i];
  for (int i = lane; i < nb; i += 32) {
    const float bv = a.beta[srow * nb + i];
    a.bo[dst * nb + i] = logits ? sigmoidf(bv) : bv;
  }
  if (lane == 0) {
    const float lv = a.lam[srow];
    a.lo[dst] = logits ? sigmoidf(lv) : lv;
  }
}

// Vectorised form for 16-byte aligned rows: a row of q or k is LPR lanes of
// 16 bytes; a warp takes 32 / LPR rows at a time.
template <typename Tin>
__global__ void __launch_bounds__(32 * kProWarps) prologue_vec_kernel(ProArgs a, int LPR) {
  constexpr int EC = 16 / (int)sizeof(Tin);  // elements per 16 bytes
  const int lane = threadIdx.x & 31, sub = lane % LPR;
  const int rpw = 32 / LPR;
  const long long nrows = (long long)a.B * a.T * a.H;
  const long long row = ((long long)blockIdx.x * kProWarps + (threadIdx.x >> 5)) * rpw + lane / LPR;
  const bool live = row < nrows;
  const int h = live ? (int)(row % a.H) : 0;
  const long long bt = live ? row / a.H : 0;
  const int t = (int)(bt % a.T), b = (int)(bt / a.T);
  const long long sr = live ? src_row(a, b, t) : -1;
  // a row of a chunk past the sequence's last is read by no kernel: not
  // written (the lanes still join the shuffles below)
  const bool put = live && !(sr < 0 && a.skip_tail && t >= (a.cu[b + 1] - a.cu[b] + 63) / 64 * 64);
  const size_t dst = (size_t)row, srow = (size_t)(sr < 0 ? 0 : sr) * a.H + h;
  const bool l2 = (a.flags & FALCON_PROLOGUE_L2NORM_QK) != 0;
  const bool logits = (a.flags & FALCON_PROLOGUE_GATE_LOGITS) != 0;
  const unsigned full = 0xffffffffu;
#pragma unroll
  for (int which = 0; which < 2; ++which) {  // q, then k: one 16-byte piece per lane
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (sr >= 0) raw = *reinterpret_cast<const uint4*>(cptr<Tin>(which == 0 ? a.q : a.k) + srow * a.dk + sub * EC);
    float x[EC];
    const Tin* e = reinterpret_cast<const Tin*>(&raw);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < EC; ++i) {
      x[i] = to_f32(e[i]);
      ss = fmaf(x[i], x[i], ss);
    }
    for (int o = 1; o < LPR; o <<= 1) ss += __shfl_xor_sync(full, ss, o);
    const float scale = l2 ? 1.f / fmaxf(sqrtf(ss), 1e-12f) : 1.f;
    uint4 outv;
    Tin* oe = reinterpret_cast<Tin*>(&outv);
#pragma unroll
    for (int i = 0; i < EC; ++i) oe[i] = from_f32<Tin>(x[i] * scale);
    if (put) *reinterpret_cast<uint4*>(reinterpret_cast<Tin*>(which == 0 ? a.qo : a.ko) + dst * a.dk + sub * EC) = outv;
  }
  if (!put) return;
  const int vc = a.dv / EC;  // 16-byte pieces per value row
  for (int c = sub; c < vc; c += LPR) {
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (sr >= 0) raw = *reinterpret_cast<const uint4*>(cptr<Tin>(a.v) + srow * a.dv + c * EC);
    *reinterpret_cast<uint4*>(reinterpret_cast<Tin*>(a.vo) + dst * a.dv + c * EC) = raw;
  }
  const int nb = a.perch ? a.dv : 1;
  for (int i = sub; i < nb; i += LPR) {
    const float bv = sr >= 0 ? a.beta[srow * nb + i] : 0.f;
    a.bo[dst * nb + i] = (sr >= 0 && logits) ? sigmoidf(bv) : bv;
  }
  if (sub == 0) {
    const float lv = sr >= 0 ? a.lam[srow] : 0.f;
    a.lo[dst] = (sr >= 0 && logits) ? sigmoidf(lv) : lv;
  }
}

// one thread per 16 bytes of a row (rows of both layouts on 16-byte boundaries)
__global__ void __launch_bounds__(256) varlen_scatter16_kernel(ProArgs a, int pieces, const uint4* o_pad, uint4* o) {
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  if (i >= (long long)a.B * a.T * a.H * pieces) return;
  const long long row = i / pieces;
  const int c = (int)(i % pieces);
  const int h = (int)(row % a.H);
  const long long bt = row / a.H;
  const int t = (int)(bt % a.T), b = (int)(bt / a.T);
  const long long sr = src_row(a, b, t);
  if (sr < 0) return;
  o[((size_t)sr * a.H + h) * pieces + c] = o_pad[(size_t)row * pieces + c];
}

template <typename Tin>
__global__ void __launch_bounds__(32 * kProWarps) varlen_scatter_kernel(ProArgs a, const void* o_pad, void* o) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kProWarps + (threadIdx.x >> 5);
  if (row >= (long long)a.B * a.T * a.H) return;
  const int h = (int)(row % a.H);
  const long long bt = row / a.H;
  const int t = (int)(bt % a.T), b = (int)(bt / a.T);
  const long long sr = src_row(a, b, t);
  if (sr < 0) return;
  const Tin* src = cptr<Tin>(o_pad) + (size_t)row * a.dv;
  Tin* dst = reinterpret_cast<Tin*>(o) + ((size_t)sr * a.H + h) * a.dv;
  for (int i = lane; i < a.dv; i += 32) dst[i] = src[i];
}

// per (sequence, head): last key, token count and window ring after the call,
// from the padded batch of the gather or (packed) from the packed rows, whose
// keys then still take phi here
template <typename Tin>
__global__ void __launch_bounds__(128) varlen_carry_kernel(ProArgs a, int packed, int W, int shift,
                                                           const void* kprev_in, const void* winx_in,
                                                           const void* winv_in, const int64_t* pos_in,
                                                           void* kprev_out, void* winx_out, void* winv_out,
                                                           int64_t* pos_out) {
  __shared__ float red[4];
  const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H, tid = threadIdx.x;
  const int len = a.cu[b + 1] - a.cu[b];
  const int64_t pos = pos_in ? pos_in[bh] : 0;
  const Tin* kpad = cptr<Tin>(packed ? a.k : a.ko);
  const Tin* vpad = cptr<Tin>(packed ? a.v : a.vo);
  auto pad_row = [&](int t) { return packed ? ((size_t)a.cu[b] + t) * a.H + h : ((size_t)b * a.T + t) * a.H + h; };
  // phi's scale 1 / max(|x|, 1e-12) of key row t (1 unless the packed rows still need it); every thread calls it
  auto key_scale = [&](int t) {
    if (!packed || !(a.flags & FALCON_PROLOGUE_L2NORM_QK)) return 1.f;
    float ss = 0.f;
    for (int i = tid; i < a.dk; i += 128) {
      const float x = to_f32(kpad[pad_row(t) * a.dk + i]);
      ss = fmaf(x, x, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    const float tot = (red[0] + red[1]) + (red[2] + red[3]);
    __syncthreads();
    return 1.f / fmaxf(sqrtf(tot), 1e-12f);
  };
  if (kprev_out) {
    Tin* kp = reinterpret_cast<Tin*>(kprev_out);
    const float sc = len >= 1 ? key_scale(len - 1) : 1.f;
    for (int i = tid; i < a.dk; i += 128) {
      Tin x = from_f32<Tin>(0.f);
      if (len >= 1) x = from_f32<Tin>(to_f32(kpad[pad_row(len - 1) * a.dk + i]) * sc);
      else if (kprev_in) x = cptr<Tin>(kprev_in)[(size_t)bh * a.dk + i];
      kp[(size_t)bh * a.dk + i] = x;
    }
  }
  if (pos_out && tid == 0) pos_out[bh] = pos + len;
  const int Wr = W - 1;
  if (Wr <= 0) return;
  for (int64_t p = pos + len - Wr; p <= pos + len - 1; ++p) {
    const int j = (int)(p - pos);
    const int slot = (int)(((p % Wr) + Wr) % Wr);  // p may be negative here
    const bool ok = p >= shift;
    if (winx_out) {
      Tin* dst = reinterpret_cast<Tin*>(winx_out) + ((size_t)bh * Wr + slot) * a.dk;
      for (int i = tid; i < a.dk; i += 128) {
        Tin x = from_f32<Tin>(0.f);
        if (ok) {
          if (j >= shift) x = kpad[pad_row(j - shift) * a.dk + i];
          else if (j == 0) x = kprev_in ? cptr<Tin>(kprev_in)[(size_t)bh * a.dk + i] : from_f32<Tin>(0.f);
          else if (winx_in) x = cptr<Tin>(winx_in)[((size_t)bh * Wr + slot) * a.dk + i];
        }
        dst[i] = x;
      }
    }
    if (winv_out) {
      Tin* dst = reinterpret_cast<Tin*>(winv_out) + ((size_t)bh * Wr + slot) * a.dv;
      for (int i = tid; i < a.dv; i += 128) {
        Tin v = from_f32<Tin>(0.f);
        if (ok) {
          if (j >= 0) v = vpad[pad_row(j) * a.dv + i];
          else if (winv_in) v = cptr<Tin>(winv_in)[((size_t)bh * Wr + slot) * a.dv + i];
        }
        dst[i] = v;
      }
    }
  }
}

inline unsigned rows_grid(const ProArgs& a) {
  return (unsigned)(((long long)a.B * a.T * a.H + kProWarps - 1) / kProWarps);
}

}  // namespace

size_t prologue_ws_bytes(int B, int T, int H, int dk, int dv, int dtype, bool perch, bool with_o) {
  const size_t es = dtype == FALCON_BF16 ? 2 : 4, n = (size_t)B * T * H;
  size_t s = align_up(n * dk * es, 256) * 2 + align_up(n * dv * es, 256) * (with_o ? 2 : 1);
  s += align_up(n * (perch ? dv : 1) * 4, 256) + align_up(n * 4, 256);
  return s;
}

void prologue_carve(ProArgs& a, void* base, bool with_o, void** o_pad) {
  const size_t es = a.dtype == FALCON_BF16 ? 2 : 4, n = (size_t)a.B * a.T * a.H;
  uint8_t* p = reinterpret_cast<uint8_t*>(base);
  a.qo = p; p += align_up(n * a.dk * es, 256);
  a.ko = p; p += align_up(n * a.dk * es, 256);
  a.vo = p; p += align_up(n * a.dv * es, 256);
  if (with_o) { *o_pad = p; p += align_up(n * a.dv * es, 256); }
  a.bo = reinterpret_cast<float*>(p); p += align_up(n * (a.perch ? a.dv : 1) * 4, 256);
  a.lo = reinterpret_cast<float*>(p);
}

int launch_prologue(const ProArgs& a, cudaStream_t s) {
  const long long nrows = (long long)a.B * a.T * a.H;
  if (nrows == 0) return FALCON_OK;
  const size_t es = a.dtype == FALCON_BF16 ? 2 : 4;
  const void* ps[3] = {a.q, a.k, a.v};
  bool aligned = true;
  for (const void* x : ps) aligned = aligned && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  const int LPR = (int)(a.dk * es / 16);
  if (aligned && (a.dv * es) % 16 == 0 && LPR >= 1 && LPR <= 32) {
    const long long rows_per_cta = (long long)kProWarps * (32 / LPR);
    const unsigned grid = (unsigned)((nrows + rows_per_cta - 1) / rows_per_cta);
    if (a.dtype == FALCON_BF16) prologue_vec_kernel<__nv_bfloat16><<<grid, 32 * kProWarps, 0, s>>>(a, LPR);
    else prologue_vec_kernel<float><<<grid, 32 * kProWarps, 0, s>>>(a, LPR);
  } else if (a.dtype == FALCON_BF16) {
    prologue_kernel<__nv_bfloat16><<<rows_grid(a), 32 * kProWarps, 0, s>>>(a);
  } else {
    prologue_kernel<float><<<rows_grid(a), 32 * kProWarps, 0, s>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

int launch_varlen_finish(const ProArgs& a, const void* o_pad, void* o, int W, int shift,
                         const falcon_carry_t* ci, falcon_carry_t* co, cudaStream_t s) {
  const size_t row_bytes = (size_t)a.dv * (a.dtype == FALCON_BF16 ? 2 : 4);
  const long long rows = o_pad ? (long long)a.B * a.T * a.H : 0;  // no padded outputs: written in place
  const int packed = o_pad ? 0 : 1;
  if (rows > 0 && row_bytes % 16 == 0 && ((reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(o_pad)) & 15) == 0) {
    const int pieces = (int)(row_bytes / 16);
    const long long n = rows * pieces;
    varlen_scatter16_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, pieces, reinterpret_cast<const uint4*>(o_pad),
                                                                       reinterpret_cast<uint4*>(o));
  } else if (rows > 0) {
    if (a.dtype == FALCON_BF16) varlen_scatter_kernel<__nv_bfloat16><<<rows_grid(a), 32 * kProWarps, 0, s>>>(a, o_pad, o);
    else varlen_scatter_kernel<float><<<rows_grid(a), 32 * kProWarps, 0, s>>>(a, o_pad, o);
  }
  if (co && (co->k_prev || co->pos || co->win_x || co->win_v)) {
    const void* kpi = ci ? ci->k_prev : nullptr;
    const void* wxi = ci && W > 1 ? ci->win_x : nullptr;
    const void* wvi = ci && W > 1 ? ci->win_v : nullptr;
    const int64_t* pi = ci ? ci->pos : nullptr;
    void* wxo = W > 1 ? co->win_x : nullptr;
    void* wvo = W > 1 ? co->win_v : nullptr;
    if (a.dtype == FALCON_BF16)
      varlen_carry_kernel<__nv_bfloat16><<<a.B * a.H, 128, 0, s>>>(a, packed, W, shift, kpi, wxi, wvi, pi, co->k_prev,
                                                                  wxo, wvo, co->pos);
    else
      varlen_carry_kernel<float><<<a.B * a.H, 128, 0, s>>>(a, packed, W, shift, kpi, wxi, wvi, pi, co->k_prev, wxo,
                                                          wvo, co->pos);
  }
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace falcon
