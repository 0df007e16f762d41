// Chunked (WY-form) backward of Falcon-1 / Falcon-1A, d_k = d_v = 64, chunk
// 64, fp32-accurate arithmetic [FW 三种等价形式; JC 三种视角看同一个更新].
//
// Forward of one chunk (rows r, i = 0..63; g the in-chunk cumulative log of
// the clamped decay, Gamma = exp(g), E_r = exp(g_63 - g_r),
// D_ri = exp(g_r - g_i) for i <= r, eta_r = beta_r / (eps + |x_r|^2)):
//   L = D (.) X X^T (i < r),  T = (I + diag(eta) L)^{-1},
//   W = T diag(eta Gamma) X,  U = T diag(eta) V,  Delta = U - W S0
//   (Falcon-1A: Delta = diag(eta) V),
//   O = diag(Gamma) Q S0 + (Q X^T (.) D) Delta,   S1 = Gamma_63 S0 + (diag(E) X)^T Delta.
// Its transpose gives the backward: with dS1 the gradient of the chunk's end
// state,
//   dDelta = (P (.) D)^T dO + diag(E) X dS1,  dR = T^T dDelta  (Falcon-1A: dR = dDelta),
//   dS0 = Gamma_63 dS1 + Q^T diag(Gamma) dO - W^T dDelta,
// a chain over chunks as sequential as the forward's, and per chunk
//   dV = diag(eta) dR,  d eta_r = sum_j dR_rj (V - Gamma X S0 - L Delta)_rj,
//   dQ = diag(Gamma) dO S0^T + dP X,  dP = (dO Delta^T) (.) D,
//   dX = (dG + dG^T) X - diag(eta Gamma) dR S0^T + dP^T Q + diag(E) Delta dS1^T + 2 dn x,
//   dG = -(diag(eta) dR Delta^T) (.) D (i < r),
// and the log-decay gradients from Gamma, E and D (row minus column sums of
// D (.) dD), summed back over the chunk's steps.  With the chunk transition
// A = Gamma_63 I - (diag(E) X)^T W and offset b = (diag(E) X)^T U both chains
// are one product a step: S1 = A S0 + b, dS0 = A^T dS1 + Y.
//
// bf16 inputs, every product on tcgen05 (the sections "on tcgen05" below):
//  (a) bwdc_prep_tc_kernel, per chunk: gates, T, W, U, Y, b, and A as images;
//  (b, c) bwdc_chain_tc_kernel, per (b, h, 32 value columns) and direction
//      (both chains in one launch): chunk start states, end-state gradients;
//  (d) bwdc_grad_tc_kernel, per chunk: every gradient.
// fp32 inputs (tolerance 1e-3, operands not exact in bf16) keep the first
// forms: bwdc_prep_kernel, bwdc_fwd_chain_kernel / bwdc_bwd_chain_kernel
// (two products a step, from W and diag(E) X), bwdc_grad_kernel, whose
// 64 x 64 products read fp32 operands from shared memory and run as
// warp-level m16n8k8 tf32 MMAs with the three-term split of each operand
// (hi + lo), which keeps their error at the level of fp32 accumulation.
// The element-wise work and the reductions stay in fp32 in both forms.

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_util.cuh"

namespace falcon {

namespace {

constexpr int kN = 64;       // chunk rows and head dim
constexpr int LDM = 68;      // fp32 row stride of the shared-memory matrices
constexpr int kThr = 256;     // per-chunk kernels
constexpr int kRows = kN * 16 / kThr;  // product rows per thread (16 column groups of 4)
constexpr int kRowT = kThr / kN;       // threads per row in row sums
static_assert(kRows * (kThr / 16) == kN && (kRows == 2 || kRows == 4), "product tile must cover 64 rows");
static_assert(kRowT * kN == kThr && (kN % kRowT) == 0, "row sums must cover 64 rows");
constexpr int kThrC = 256;    // chain kernels
constexpr size_t kMat = (size_t)kN * kN;
// per chunk: T, W, U, diag(E) X (fp32 inputs) or the chain offset b (bf16
// inputs), Y, the start state, the end-state gradient, and (bf16 inputs) the
// chain transition A as hi | lo bf16 images
enum { M_T = 0, M_W, M_U, M_XT, M_Y, M_S0, M_DS1, M_AC, kMats };
constexpr int kGateVecs = 8;  // per chunk: g, Gamma, E, eta, nrm, exists, (2 spare)
constexpr int NN = 0, TN = 1, NT = 2;

struct CbArgs {
  int B, T, H, NC, shift, additive;
  float eps, eps_gamma;
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
  float* ws;
  uint32_t* status;   // the call's status word (a bounded wait that gave up)
  uint64_t wait_ns;
};

__device__ __forceinline__ float* wsmat(const CbArgs& a, size_t cg, int which) {
  return a.ws + (cg * kMats + which) * kMat;
}
__device__ __forceinline__ float* wsgate(const CbArgs& a, size_t cg) {
  return a.ws + (size_t)a.B * a.H * a.NC * kMats * kMat + cg * kGateVecs * kN;
}

// C (4 x 4 per thread) += op(A) op(B) over K = 64, both operands fp32 in
// shared memory with row stride LDM.  NN: A [M][K], B [K][N]; TN: A [K][M],
// B [K][N]; NT: A [M][K], B [N][K].  Tensor-core m16n8k8 products with the
// three-term tf32 split (a = a_hi + a_lo, a b ~ a_hi b_hi + a_hi b_lo +
// a_lo b_hi), whose error stays at the level of fp32 accumulation.  Warp w
// covers rows 32 (w / 4) .. + 31 and columns 16 (w % 4) .. + 15; thread
// (gid, tig) = (lane / 4, lane % 4) owns rows 32 (w / 4) + gid + 8 i and
// columns 16 (w % 4) + 8 (j / 2) + 2 tig + j % 2.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = tc::to_tf32(x);
  lo = tc::to_tf32(x - __uint_as_float(hi));
}

// AX / BX: that operand holds values exact in tf32 (bf16 inputs as loaded),
// so its low part is zero and the product term that would use it is skipped.
template <int MODE, bool AX = false, bool BX = false>
__device__ __forceinline__ void mm64(float (&acc)[kRows][4], const float* __restrict__ A,
                                     const float* __restrict__ B) {
  static_assert(kRows == 4, "two 16-row tiles of two 8-column tiles per warp");
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int m0 = 32 * (w >> 2), n0 = 16 * (w & 3);
#pragma unroll 2
  for (int k0 = 0; k0 < kN; k0 += 8) {
    uint32_t ah[2][4], al[2][4], bh[2][2], bl[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int m = m0 + 16 * mt + gid;
      float x[4];
      if (MODE == TN) {
        x[0] = A[(k0 + tig) * LDM + m];
        x[1] = A[(k0 + tig) * LDM + m + 8];
        x[2] = A[(k0 + tig + 4) * LDM + m];
        x[3] = A[(k0 + tig + 4) * LDM + m + 8];
      } else {
        x[0] = A[m * LDM + k0 + tig];
        x[1] = A[(m + 8) * LDM + k0 + tig];
        x[2] = A[m * LDM + k0 + tig + 4];
        x[3] = A[(m + 8) * LDM + k0 + tig + 4];
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (AX) ah[mt][e] = __float_as_uint(x[e]);
        else split_tf32(x[e], ah[mt][e], al[mt][e]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int n = n0 + 8 * nt + gid;
      float y[2];
      if (MODE == NT) {
        y[0] = B[n * LDM + k0 + tig];
        y[1] = B[n * LDM + k0 + tig + 4];
      } else {
        y[0] = B[(k0 + tig) * LDM + n];
        y[1] = B[(k0 + tig + 4) * LDM + n];
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if (BX) bh[nt][e] = __float_as_uint(y[e]);
        else split_tf32(y[e], bh[nt][e], bl[nt][e]);
      }
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float c[4] = {acc[2 * mt][2 * nt], acc[2 * mt][2 * nt + 1], acc[2 * mt + 1][2 * nt],
                      acc[2 * mt + 1][2 * nt + 1]};
        if (!AX) tc::mma_tf32_16x8x8(c, al[mt], bh[nt]);
        if (!BX) tc::mma_tf32_16x8x8(c, ah[mt], bl[nt]);
        tc::mma_tf32_16x8x8(c, ah[mt], bh[nt]);
        acc[2 * mt][2 * nt] = c[0];
        acc[2 * mt][2 * nt + 1] = c[1];
        acc[2 * mt + 1][2 * nt] = c[2];
        acc[2 * mt + 1][2 * nt + 1] = c[3];
      }
  }
}

template <int MODE>
__device__ __forceinline__ int out_row(int i) {
  return 32 * (int)(threadIdx.x >> 7) + (int)((threadIdx.x & 31) >> 2) + 8 * i;
}
template <int MODE>
__device__ __forceinline__ int out_col(int j) {
  return 16 * (int)((threadIdx.x >> 5) & 3) + 8 * (j >> 1) + 2 * (int)(threadIdx.x & 3) + (j & 1);
}

__device__ __forceinline__ void zero_acc(float (&acc)[kRows][4]) {
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
}

// sum over the 64 columns of f(r, c), kRowT threads per row; every thread of
// the row's group returns the row's sum (row = tid / kRowT)
template <typename Fn>
__device__ __forceinline__ float row_sum(Fn f) {
  constexpr int NC_ = kN / kRowT;
  const int r = threadIdx.x / kRowT, part = threadIdx.x % kRowT;
  float s = 0.f;
#pragma unroll 4
  for (int c = part * NC_; c < part * NC_ + NC_; ++c) s += f(r, c);
#pragma unroll
  for (int o = 1; o < kRowT; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

template <typename Tin>
__device__ __forceinline__ float ldx(const void* p, size_t i) { return to_f32(reinterpret_cast<const Tin*>(p)[i]); }
template <typename Tin>
__device__ __forceinline__ void stx(void* p, size_t i, float x) { reinterpret_cast<Tin*>(p)[i] = from_f32<Tin>(x); }
// eight consecutive elements p[i .. i + 7] (i a multiple of 8) in 16-byte stores
template <typename Tin>
__device__ __forceinline__ void stx8(void* p, size_t i, const float (&v)[8]) {
  if constexpr (sizeof(Tin) == 2) {
    uint32_t pk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
      pk[e] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(reinterpret_cast<Tin*>(p) + i) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  } else {
    float4* q = reinterpret_cast<float4*>(reinterpret_cast<Tin*>(p) + i);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}
// eight consecutive fp32 values of a shared-memory row
__device__ __forceinline__ void lds8(float (&v)[8], const float* p) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Rows of a chunk into shared memory (zero past the end of the call) in two
// halves, so that a kernel can have the loads of several tiles in flight
// together: fetch_* issues a thread's 16-byte loads into registers, put_rows
// converts them to fp32 rows.
template <typename Tin>
struct RowRaw {
  static constexpr int EC = 16 / (int)sizeof(Tin), PR = kN / EC, PT = kN * PR / kThr;  // per row / thread
  uint4 v[PT];
};
template <typename Tin>
__device__ __forceinline__ void fetch_rows(RowRaw<Tin>& raw, const void* src, const CbArgs& a, int b, int h, int t0) {
  using R = RowRaw<Tin>;
#pragma unroll
  for (int k = 0; k < R::PT; ++k) {
    const int i = threadIdx.x + kThr * k, r = i / R::PR, c = (i % R::PR) * R::EC, t = t0 + r;
    raw.v[k] = t < a.T ? *reinterpret_cast<const uint4*>(reinterpret_cast<const Tin*>(src) +
                                                       (((size_t)b * a.T + t) * a.H + h) * kN + c)
                       : make_uint4(0u, 0u, 0u, 0u);
  }
}
// keys of the chunk's pairs: x_r = k_{t - shift}, the carried key for the
// first pair (prefix), zero where the pair does not exist
template <typename Tin>
__device__ __forceinline__ void fetch_keys(RowRaw<Tin>& raw, const CbArgs& a, int b, int h, int t0, int64_t pos) {
  using R = RowRaw<Tin>;
#pragma unroll
  for (int k = 0; k < R::PT; ++k) {
    const int i = threadIdx.x + kThr * k, r = i / R::PR, c = (i % R::PR) * R::EC, t = t0 + r;
    const Tin* row = nullptr;
    if (t < a.T && pos + t >= a.shift) {
      if (t - a.shift >= 0) row = reinterpret_cast<const Tin*>(a.k) + (((size_t)b * a.T + (t - a.shift)) * a.H + h) * kN;
      else if (a.kprev_in) row = reinterpret_cast<const Tin*>(a.kprev_in) + ((size_t)b * a.H + h) * kN;
    }
    raw.v[k] = row ? *reinterpret_cast<const uint4*>(row + c) : make_uint4(0u, 0u, 0u, 0u);
  }
}
template <typename Tin>
__device__ __forceinline__ void put_rows(float* dst, const RowRaw<Tin>& raw) {
  using R = RowRaw<Tin>;
#pragma unroll
  for (int k = 0; k < R::PT; ++k) {
    const int i = threadIdx.x + kThr * k, r = i / R::PR, c = (i % R::PR) * R::EC;
    const Tin* e = reinterpret_cast<const Tin*>(&raw.v[k]);
#pragma unroll
    for (int q = 0; q < R::EC; q += 4)
      *reinterpret_cast<float4*>(&dst[r * LDM + c + q]) =
          make_float4(to_f32(e[q]), to_f32(e[q + 1]), to_f32(e[q + 2]), to_f32(e[q + 3]));
  }
}
// keys, queries, values and output gradients of the chunk, all loads in flight together
template <typename Tin>
__device__ __forceinline__ void load_inputs(float* X, float* Q, float* V, float* dO, const CbArgs& a, int b, int h,
                                            int t0, int64_t pos) {
  RowRaw<Tin> rx, rq, rv, rd;
  fetch_keys<Tin>(rx, a, b, h, t0, pos);
  fetch_rows<Tin>(rq, a.q, a, b, h, t0);
  fetch_rows<Tin>(rv, a.v, a, b, h, t0);
  fetch_rows<Tin>(rd, a.dO, a, b, h, t0);
  put_rows<Tin>(X, rx);
  put_rows<Tin>(Q, rq);
  put_rows<Tin>(V, rv);
  put_rows<Tin>(dO, rd);
}
__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// a 64 x 64 fp32 workspace matrix into shared memory by cp.async (no wait)
__device__ __forceinline__ void cp_mat(float* dst, const float* src) {
#pragma unroll
  for (int k = 0; k < kN * kN / 4 / kThr; ++k) {
    const int i = threadIdx.x + kThr * k;
    cp16(&dst[(i >> 4) * LDM + (i & 15) * 4], &src[(i >> 4) * kN + (i & 15) * 4]);
  }
}
struct GateSm {
  float g[kN], Gam[kN], E[kN], eta[kN], nrm[kN], ex[kN], gam[kN];
};

// gates of the chunk (needs the keys in X); threads < 64, then a barrier
__device__ void make_gates(GateSm& gs, const float* X, const CbArgs& a, int b, int h, int t0, int64_t pos) {
  const int r = threadIdx.x;
  if (r < kN) {
    const int t = t0 + r;
    float n = 0.f;
#pragma unroll 8
    for (int c = 0; c < kN; ++c) n = fmaf(X[r * LDM + c], X[r * LDM + c], n);
    const bool live = t < a.T, ex = live && pos + t >= a.shift;
    const size_t gi = ((size_t)b * a.T + (live ? t : 0)) * a.H + h;
    gs.nrm[r] = n;
    gs.ex[r] = ex ? 1.f : 0.f;
    gs.eta[r] = ex ? a.beta[gi] / (a.eps + n) : 0.f;
    const float gm = live ? fminf(fmaxf(1.f - a.lam[gi], a.eps_gamma), 1.f) : 1.f;
    gs.gam[r] = gm;
    gs.g[r] = live ? logf(gm) : 0.f;
  }
  __syncthreads();
  if (threadIdx.x < 32) {  // inclusive prefix sum over the 64 rows
    float v0 = gs.g[threadIdx.x], v1 = gs.g[threadIdx.x + 32];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n0 = __shfl_up_sync(0xffffffffu, v0, o), n1 = __shfl_up_sync(0xffffffffu, v1, o);
      if ((int)threadIdx.x >= o) { v0 += n0; v1 += n1; }
    }
    v1 += __shfl_sync(0xffffffffu, v0, 31);
    gs.g[threadIdx.x] = v0;
    gs.g[threadIdx.x + 32] = v1;
  }
  __syncthreads();
  if (r < kN) {
    gs.Gam[r] = __expf(gs.g[r]);
    gs.E[r] = __expf(gs.g[kN - 1] - gs.g[r]);
  }
  __syncthreads();
}

__device__ __forceinline__ float dmask(const GateSm& gs, int r, int i) {  // D_ri (i <= r), else 0
  return i <= r ? __expf(gs.g[r] - gs.g[i]) : 0.f;
}

// ---------------------------------------------------------------- (a)
template <typename Tin>
__global__ void __launch_bounds__(kThr) bwdc_prep_kernel(CbArgs a) {
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  float* X = sm;
  float* Q = X + kN * LDM;
  float* V = Q + kN * LDM;
  float* dO = V + kN * LDM;
  float* M1 = dO + kN * LDM;
  float* Tm = M1 + kN * LDM;
  float* M3 = Tm + kN * LDM;
  float* Wm = M3 + kN * LDM;
  GateSm& gs = *reinterpret_cast<GateSm*>(Wm + kN * LDM);
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0u;  // each call starts with a clear status
  const size_t cg = blockIdx.x;
  const int c = (int)(cg % a.NC), bh = (int)(cg / a.NC), b = bh / a.H, h = bh % a.H, t0 = c * kN;
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  const int tid = threadIdx.x;
  constexpr bool kE = sizeof(Tin) == 2;  // bf16 inputs: X, Q, V, dO exact in tf32
  load_inputs<Tin>(X, Q, V, dO, a, b, h, t0, pos);
  __syncthreads();
  make_gates(gs, X, a, b, h, t0, pos);
  float acc[kRows][4];
  if (!a.additive) {
    // A = diag(eta) (D (.) X X^T), strictly lower
    zero_acc(acc);
    mm64<NT, kE, kE>(acc, X, X);
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = out_row<NT>(i), ci = out_col<NT>(j);
        M1[r * LDM + ci] = ci < r ? gs.eta[r] * __expf(gs.g[r] - gs.g[ci]) * acc[i][j] : 0.f;
      }
    __syncthreads();
    // T = (I + A)^{-1}: thread j < 64 solves column j by forward substitution,
    // the column in registers, the rows of A read as broadcasts
    if (tid < kN) {
      const int j = tid;
      float tcol[kN];
#pragma unroll
      for (int r = 0; r < kN; ++r) {
        float s0 = (r == j) ? 1.f : 0.f, s1 = 0.f;
#pragma unroll
        for (int i = 0; i < r; i += 2) {
          s0 = fmaf(-M1[r * LDM + i], tcol[i], s0);
          if (i + 1 < r) s1 = fmaf(-M1[r * LDM + i + 1], tcol[i + 1], s1);
        }
        tcol[r] = s0 + s1;
      }
#pragma unroll
      for (int r = 0; r < kN; ++r) Tm[r * LDM + j] = tcol[r];
    }
    __syncthreads();
    // W = T diag(eta Gamma) X, U = T diag(eta) V
    for (int i = tid; i < kN * kN; i += kThr) {
      const int r = i / kN, cc = i % kN;
      M3[r * LDM + cc] = gs.eta[r] * gs.Gam[r] * X[r * LDM + cc];
      M1[r * LDM + cc] = gs.eta[r] * V[r * LDM + cc];
    }
    __syncthreads();
    zero_acc(acc);
    mm64<NN>(acc, Tm, M3);
    float* wW = wsmat(a, cg, M_W);
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = out_row<NN>(i), cc = out_col<NN>(j);
        Wm[r * LDM + cc] = acc[i][j];
        wW[r * kN + cc] = acc[i][j];
      }
    zero_acc(acc);
    mm64<NN>(acc, Tm, M1);
    float* wU = wsmat(a, cg, M_U);
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) wU[out_row<NN>(i) * kN + out_col<NN>(j)] = acc[i][j];
    float* wT = wsmat(a, cg, M_T);
    for (int i = tid; i < kN * kN; i += kThr) wT[i] = Tm[(i / kN) * LDM + i % kN];
  } else {
    float* wU = wsmat(a, cg, M_U);
    for (int i = tid; i < kN * kN; i += kThr) wU[i] = gs.eta[i / kN] * V[(i / kN) * LDM + i % kN];
  }
  {  // diag(E) X, gates
    float* wX = wsmat(a, cg, M_XT);
    for (int i = tid; i < kN * kN; i += kThr) wX[i] = gs.E[i / kN] * X[(i / kN) * LDM + i % kN];
    float* gv = wsgate(a, cg);
    if (tid < kN) {
      gv[tid] = gs.g[tid];
      gv[kN + tid] = gs.Gam[tid];
      gv[2 * kN + tid] = gs.E[tid];
      gv[3 * kN + tid] = gs.eta[tid];
      gv[4 * kN + tid] = gs.nrm[tid];
      gv[5 * kN + tid] = gs.ex[tid];
      gv[6 * kN + tid] = gs.gam[tid];
    }
  }
  __syncthreads();
  // Y = Q^T diag(Gamma) dO - W^T (P (.) D)^T dO
  zero_acc(acc);
  mm64<NT, kE, kE>(acc, Q, X);  // P = Q X^T
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = out_row<NT>(i), ci = out_col<NT>(j);
      M1[r * LDM + ci] = dmask(gs, r, ci) * acc[i][j];
    }
  for (int i = tid; i < kN * kN; i += kThr) {
    const int r = i / kN, cc = i % kN;
    M3[r * LDM + cc] = gs.Gam[r] * dO[r * LDM + cc];
  }
  __syncthreads();
  float yacc[kRows][4];
  zero_acc(yacc);
  mm64<TN, kE>(yacc, Q, M3);  // Q^T diag(Gamma) dO
  if (!a.additive) {
    zero_acc(acc);
    mm64<TN, false, kE>(acc, M1, dO);  // Z = (P (.) D)^T dO
    __syncthreads();        // M3 is read by every thread above
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) M3[out_row<TN>(i) * LDM + out_col<TN>(j)] = acc[i][j];
    __syncthreads();
    float wz[kRows][4];
    zero_acc(wz);
    mm64<TN>(wz, Wm, M3);  // W^T Z
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) yacc[i][j] -= wz[i][j];
  }
  float* wY = wsmat(a, cg, M_Y);
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) wY[out_row<TN>(i) * kN + out_col<TN>(j)] = yacc[i][j];
}

// ---------------------------------------------------------------- (b), (c)
// One CTA of 256 threads per (b, h, SC value columns), SC = 16, or 32 when
// the 16-column CTAs would not fit one wave (two CTAs per SM); the S (or dS)
// slice, 64 x SC, in shared memory.  Each chunk step is two 64 x 64 x SC
// products on the tensor cores (three-term tf32 split, as in mm64): warp w
// owns the SC / 16 tiles of 16 x 8 at rows 16 (w / 2), columns from
// (SC / 2) (w % 2).  The next chunk's W, diag(E) X, value slice (U or Y) and
// decay arrive by cp.async into the other of two stages.
template <int SC>
struct ChainStage {
  static constexpr int CPT = SC / 4;  // columns per thread in the row-wise copies
  static constexpr int LDS_ = SC + 8; // row stride of the slices: fragment loads free of bank conflicts
  static constexpr int NTW = SC / 16; // 8-column tiles per warp
  float W[kN * LDM];
  float X[kN * LDM];
  float C[kN * LDS_];   // U (forward) or Y (backward) slice
  float g4[4];          // Gamma of rows 60..63
};
template <int SC>
struct ChainSmem {
  ChainStage<SC> st[2];
  float S[kN * ChainStage<SC>::LDS_];
  float Dl[kN * ChainStage<SC>::LDS_];
};

template <int SC>
__device__ __forceinline__ void chain_stage(const CbArgs& a, ChainStage<SC>& st, size_t cg, int c0, int which_c) {
  constexpr int LDS_ = ChainStage<SC>::LDS_;
  const int tid = threadIdx.x;
  const float* wW = wsmat(a, cg, M_W);
  const float* wX = wsmat(a, cg, M_XT);
  const float* wC = wsmat(a, cg, which_c);
#pragma unroll
  for (int k = 0; k < kN * kN / 4 / kThrC; ++k) {
    const int i = tid + kThrC * k, r = i >> 4, c = (i & 15) * 4;
    if (!a.additive) cp16(&st.W[r * LDM + c], &wW[r * kN + c]);
    cp16(&st.X[r * LDM + c], &wX[r * kN + c]);
  }
#pragma unroll
  for (int k = 0; k < kN * SC / 4 / kThrC; ++k) {
    const int i = tid + kThrC * k, r = i / (SC / 4), c = (i % (SC / 4)) * 4;
    cp16(&st.C[r * LDS_ + c], &wC[r * kN + c0 + c]);
  }
  if (tid == 0) cp16(st.g4, wsgate(a, cg) + kN + kN - 4);
}

// c[j] (this warp's 16 x 8 tiles at rows m0, columns n0 + 8 j) += sgn A B over
// K = 64: A [M][K] at A[m * LDM + k] (AT: A[k * LDM + m]), B [K][SC] at
// B[k * LDS_ + n]; the A fragments serve every tile.  Two accumulators per
// tile over alternate k steps shorten the dependent chain.
template <int SC, bool AT>
__device__ __forceinline__ void tile_mma(float (&c)[SC / 16][4], const float* __restrict__ A,
                                         const float* __restrict__ B, int m0, int n0, float sgn) {
  constexpr int LDS_ = ChainStage<SC>::LDS_, NTW = SC / 16;
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
  float c2[NTW][4] = {};
#pragma unroll
  for (int k0 = 0; k0 < kN; k0 += 8) {
    float x[4];
    if (AT) {
      x[0] = A[(k0 + tig) * LDM + m0 + gid];
      x[1] = A[(k0 + tig) * LDM + m0 + gid + 8];
      x[2] = A[(k0 + tig + 4) * LDM + m0 + gid];
      x[3] = A[(k0 + tig + 4) * LDM + m0 + gid + 8];
    } else {
      x[0] = A[(m0 + gid) * LDM + k0 + tig];
      x[1] = A[(m0 + gid + 8) * LDM + k0 + tig];
      x[2] = A[(m0 + gid) * LDM + k0 + tig + 4];
      x[3] = A[(m0 + gid + 8) * LDM + k0 + tig + 4];
    }
    uint32_t ah[4], al[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_tf32(sgn * x[e], ah[e], al[e]);
#pragma unroll
    for (int j = 0; j < NTW; ++j) {
      uint32_t bh[2], bl[2];
      split_tf32(B[(k0 + tig) * LDS_ + n0 + 8 * j + gid], bh[0], bl[0]);
      split_tf32(B[(k0 + tig + 4) * LDS_ + n0 + 8 * j + gid], bh[1], bl[1]);
      float (&acc)[4] = (k0 & 8) ? c2[j] : c[j];
      tc::mma_tf32_16x8x8(acc, al, bh);
      tc::mma_tf32_16x8x8(acc, ah, bl);
      tc::mma_tf32_16x8x8(acc, ah, bh);
    }
  }
#pragma unroll
  for (int j = 0; j < NTW; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) c[j][e] += c2[j][e];
}
// the tiles' elements of a [64][LDS_] slice: tile j, (row, column) =
// (m0 + gid + 8 (e / 2), n0 + 8 j + 2 tig + e % 2)
template <int SC>
__device__ __forceinline__ void tile_ld(float (&v)[SC / 16][4], const float* p, int m0, int n0) {
  constexpr int LDS_ = ChainStage<SC>::LDS_;
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int j = 0; j < SC / 16; ++j) {
    const float2 a = *reinterpret_cast<const float2*>(&p[(m0 + gid) * LDS_ + n0 + 8 * j + 2 * tig]);
    const float2 b = *reinterpret_cast<const float2*>(&p[(m0 + gid + 8) * LDS_ + n0 + 8 * j + 2 * tig]);
    v[j][0] = a.x; v[j][1] = a.y; v[j][2] = b.x; v[j][3] = b.y;
  }
}
template <int SC>
__device__ __forceinline__ void tile_st(float* p, const float (&v)[SC / 16][4], int m0, int n0) {
  constexpr int LDS_ = ChainStage<SC>::LDS_;
  const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int j = 0; j < SC / 16; ++j) {
    *reinterpret_cast<float2*>(&p[(m0 + gid) * LDS_ + n0 + 8 * j + 2 * tig]) = make_float2(v[j][0], v[j][1]);
    *reinterpret_cast<float2*>(&p[(m0 + gid + 8) * LDS_ + n0 + 8 * j + 2 * tig]) = make_float2(v[j][2], v[j][3]);
  }
}
// CPT consecutive fp32 values of shared-memory row p to global row q (16-byte pieces)
template <int CPT>
__device__ __forceinline__ void copy_row(float* q, const float* p) {
#pragma unroll
  for (int i = 0; i < CPT; i += 4) *reinterpret_cast<float4*>(q + i) = *reinterpret_cast<const float4*>(p + i);
}

template <int SC>
__global__ void __launch_bounds__(kThrC) bwdc_fwd_chain_kernel(CbArgs a) {
  using St = ChainStage<SC>;
  constexpr int CPT = St::CPT, LDS_ = St::LDS_, NTW = St::NTW;
  extern __shared__ float4 smem_f4[];
  ChainSmem<SC>& sm = *reinterpret_cast<ChainSmem<SC>*>(smem_f4);
  const int bh = blockIdx.x, c0 = blockIdx.y * SC, tid = threadIdx.x;
  const int r = tid >> 2, q8 = (tid & 3) * CPT;
  const int m0 = 16 * (tid >> 6), n0 = (SC / 2) * ((tid >> 5) & 1);
  for (int i = tid; i < kN * SC; i += kThrC) {
    const int rr = i / SC, cc = i % SC;
    sm.S[rr * LDS_ + cc] = a.S_in ? a.S_in[((size_t)bh * kN + rr) * kN + c0 + cc] : 0.f;
  }
  chain_stage<SC>(a, sm.st[0], (size_t)bh * a.NC, c0, M_U);
  cp_commit();
  if (a.NC > 1) chain_stage<SC>(a, sm.st[1], (size_t)bh * a.NC + 1, c0, M_U);
  cp_commit();
  for (int c = 0; c < a.NC; ++c) {
    const size_t cg = (size_t)bh * a.NC + c;
    St& st = sm.st[c & 1];
    cp_wait1();
    __syncthreads();
    copy_row<CPT>(&wsmat(a, cg, M_S0)[(size_t)r * kN + c0 + q8], &sm.S[r * LDS_ + q8]);  // chunk start state out
    float d[NTW][4];  // Delta = U - W S  (additive: Delta = U)
    tile_ld<SC>(d, st.C, m0, n0);
    if (!a.additive) tile_mma<SC, false>(d, st.W, sm.S, m0, n0, -1.f);
    tile_st<SC>(sm.Dl, d, m0, n0);
    __syncthreads();
    // S = Gamma_63 S + (diag(E) X)^T Delta   (row of S = key index)
    float v[NTW][4];
    tile_ld<SC>(v, sm.S, m0, n0);
#pragma unroll
    for (int j = 0; j < NTW; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) v[j][e] *= st.g4[3];
    tile_mma<SC, true>(v, st.X, sm.Dl, m0, n0, 1.f);
    __syncthreads();  // every read of S and of this stage is done
    tile_st<SC>(sm.S, v, m0, n0);
    if (c + 2 < a.NC) chain_stage<SC>(a, st, cg + 2, c0, M_U);
    cp_commit();
  }
  cp_wait0();
}

template <int SC>
__global__ void __launch_bounds__(kThrC) bwdc_bwd_chain_kernel(CbArgs a) {
  using St = ChainStage<SC>;
  constexpr int CPT = St::CPT, LDS_ = St::LDS_, NTW = St::NTW;
  extern __shared__ float4 smem_f4[];
  ChainSmem<SC>& sm = *reinterpret_cast<ChainSmem<SC>*>(smem_f4);
  const int bh = blockIdx.x, c0 = blockIdx.y * SC, tid = threadIdx.x;
  const int r = tid >> 2, q8 = (tid & 3) * CPT;
  const int m0 = 16 * (tid >> 6), n0 = (SC / 2) * ((tid >> 5) & 1);
  for (int i = tid; i < kN * SC; i += kThrC) {
    const int rr = i / SC, cc = i % SC;
    sm.S[rr * LDS_ + cc] = a.dS_final ? a.dS_final[((size_t)bh * kN + rr) * kN + c0 + cc] : 0.f;
  }
  const size_t base = (size_t)bh * a.NC;
  chain_stage<SC>(a, sm.st[0], base + a.NC - 1, c0, M_Y);
  cp_commit();
  if (a.NC > 1) chain_stage<SC>(a, sm.st[1], base + a.NC - 2, c0, M_Y);
  cp_commit();
  for (int n = 0; n < a.NC; ++n) {
    const int c = a.NC - 1 - n;
    const size_t cg = base + c;
    St& st = sm.st[n & 1];
    cp_wait1();
    __syncthreads();
    copy_row<CPT>(&wsmat(a, cg, M_DS1)[(size_t)r * kN + c0 + q8], &sm.S[r * LDS_ + q8]);  // end-state gradient out
    if (!a.additive) {  // Z = diag(E) X dS  (row = chunk row)
      float z[NTW][4] = {};
      tile_mma<SC, false>(z, st.X, sm.S, m0, n0, 1.f);
      tile_st<SC>(sm.Dl, z, m0, n0);
    }
    __syncthreads();
    // dS = Gamma_63 dS - W^T Z + Y   (row = key index)
    float v[NTW][4], y[NTW][4];
    tile_ld<SC>(v, sm.S, m0, n0);
    tile_ld<SC>(y, st.C, m0, n0);
#pragma unroll
    for (int j = 0; j < NTW; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) v[j][e] = fmaf(st.g4[3], v[j][e], y[j][e]);
    if (!a.additive) tile_mma<SC, true>(v, st.W, sm.Dl, m0, n0, -1.f);
    __syncthreads();
    tile_st<SC>(sm.S, v, m0, n0);
    if (n + 2 < a.NC) chain_stage<SC>(a, st, base + a.NC - 3 - n, c0, M_Y);
    cp_commit();
  }
  cp_wait0();
  __syncthreads();
  if (a.dS_in)
    for (int i = tid; i < kN * SC; i += kThrC)
      a.dS_in[((size_t)bh * kN + i / SC) * kN + c0 + i % SC] = sm.S[(i / SC) * LDS_ + i % SC];
}

// ---------------------------------------------------------------- (d)
template <typename Tin>
__global__ void __launch_bounds__(kThr) bwdc_grad_kernel(CbArgs a) {
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  float* X = sm;
  float* Q = X + kN * LDM;
  float* V = Q + kN * LDM;
  float* dO = V + kN * LDM;
  float* S0 = dO + kN * LDM;
  float* dS1 = S0 + kN * LDM;
  float* s1 = dS1 + kN * LDM;
  float* s2 = s1 + kN * LDM;
  float* s3 = s2 + kN * LDM;
  float* s4 = s3 + kN * LDM;
  float* s5 = s4 + kN * LDM;
  float* s6 = s5 + kN * LDM;
  GateSm& gs = *reinterpret_cast<GateSm*>(s6 + kN * LDM);
  float* vec = reinterpret_cast<float*>(&gs + 1);  // dGo, dGr, EdE, deta, rowM, colM, dg, misc
  float* dGo = vec;
  float* dGr = vec + kN;
  float* EdE = vec + 2 * kN;
  float* deta = vec + 3 * kN;
  float* rowM = vec + 4 * kN;
  float* colM = vec + 5 * kN;
  float* dgv = vec + 6 * kN;
  const size_t cg = blockIdx.x;
  const int c = (int)(cg % a.NC), bh = (int)(cg / a.NC), b = bh / a.H, h = bh % a.H, t0 = c * kN;
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  const int tid = threadIdx.x;
  const bool reg = !a.additive;
  constexpr bool kE = sizeof(Tin) == 2;  // bf16 inputs: X, Q, V, dO exact in tf32
  {  // the workspace matrices by cp.async, the input rows meanwhile
    cp_mat(S0, wsmat(a, cg, M_S0));
    cp_mat(dS1, wsmat(a, cg, M_DS1));
    if (reg) {
      cp_mat(s1, wsmat(a, cg, M_W));
      cp_mat(s2, wsmat(a, cg, M_U));
    }
    // the gate vectors g, Gamma, E, eta, |x|^2, exists, gamma: GateSm's order
    static_assert(sizeof(GateSm) == 7 * kN * sizeof(float), "gate rows back to back");
    if (tid < (int)(sizeof(GateSm) / 16)) cp16(reinterpret_cast<float*>(&gs) + 4 * tid, wsgate(a, cg) + 4 * tid);
    cp_commit();
    load_inputs<Tin>(X, Q, V, dO, a, b, h, t0, pos);
    cp_wait0();
  }
  __syncthreads();
  float acc[kRows][4];
  // Delta -> s2
  if (reg) {
    zero_acc(acc);
    mm64<NN>(acc, s1, S0);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = out_row<NN>(i), cc = out_col<NN>(j);
        s2[r * LDM + cc] -= acc[i][j];
      }
  } else {
    for (int i = tid; i < kN * kN; i += kThr) {
      const int r = i / kN, cc = i % kN;
      s2[r * LDM + cc] = gs.eta[r] * V[r * LDM + cc];
    }
  }
  // X S0 -> s1 (regression); Q S0 -> s3
  if (reg) {
    zero_acc(acc);
    mm64<NN, kE>(acc, X, S0);
    __syncthreads();  // s1 (W) is consumed
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s1[out_row<NN>(i) * LDM + out_col<NN>(j)] = acc[i][j];
  }
  zero_acc(acc);
  mm64<NN, kE>(acc, Q, S0);
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) s3[out_row<NN>(i) * LDM + out_col<NN>(j)] = acc[i][j];
  __syncthreads();
  {
    const float v = row_sum([&](int r, int cc) { return dO[r * LDM + cc] * s3[r * LDM + cc]; });
    if (tid % kRowT == 0) dGo[tid / kRowT] = v;
  }
  __syncthreads();
  // P (.) D -> s3 (lower incl. diagonal)
  zero_acc(acc);
  mm64<NT, kE, kE>(acc, Q, X);
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = out_row<NT>(i), ci = out_col<NT>(j);
      s3[r * LDM + ci] = dmask(gs, r, ci) * acc[i][j];
    }
  // X dS1 -> s4
  zero_acc(acc);
  mm64<NN, kE>(acc, X, dS1);
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) s4[out_row<NN>(i) * LDM + out_col<NN>(j)] = acc[i][j];
  __syncthreads();
  {
    const float v = row_sum([&](int r, int cc) { return s4[r * LDM + cc] * s2[r * LDM + cc]; });
    if (tid % kRowT == 0) EdE[tid / kRowT] = gs.E[tid / kRowT] * v;
  }
  // dDelta = (P (.) D)^T dO + diag(E) X dS1 -> s5
  zero_acc(acc);
  mm64<TN, false, kE>(acc, s3, dO);
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = out_row<TN>(i), cc = out_col<TN>(j);
      s5[r * LDM + cc] = acc[i][j] + gs.E[r] * s4[r * LDM + cc];
    }
  __syncthreads();
  // dR = T^T dDelta -> s6 (additive: dR = dDelta)
  if (reg) {
    cp_mat(s4, wsmat(a, cg, M_T));
    cp_commit();
    cp_wait0();
    __syncthreads();
    zero_acc(acc);
    mm64<TN>(acc, s4, s5);
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s6[out_row<TN>(i) * LDM + out_col<TN>(j)] = acc[i][j];
  } else {
    for (int i = tid; i < kN * kN; i += kThr) s6[(i / kN) * LDM + i % kN] = s5[(i / kN) * LDM + i % kN];
  }
  __syncthreads();
  // dV, d eta (residual part), dGamma (residual part)
  for (int i = tid; i < kN * kN / 8; i += kThr) {
    const int r = i / (kN / 8), cc = (i % (kN / 8)) * 8, t = t0 + r;
    if (t >= a.T) continue;
    float v8[8];
    lds8(v8, &s6[r * LDM + cc]);
#pragma unroll
    for (int e = 0; e < 8; ++e) v8[e] *= gs.eta[r];
    stx8<Tin>(a.dv, (((size_t)b * a.T + t) * a.H + h) * kN + cc, v8);
  }
  {
    const int r = tid / kRowT;
    float de, dgr = 0.f;
    if (reg) {
      de = row_sum([&](int rr, int cc) { return s6[rr * LDM + cc] * (V[rr * LDM + cc] - gs.Gam[rr] * s1[rr * LDM + cc]); });
      dgr = -gs.eta[r] * row_sum([&](int rr, int cc) { return s6[rr * LDM + cc] * s1[rr * LDM + cc]; });
    } else {
      de = row_sum([&](int rr, int cc) { return s6[rr * LDM + cc] * V[rr * LDM + cc]; });
    }
    if (tid % kRowT == 0) { deta[r] = de; dGr[r] = dgr; }
  }
  __syncthreads();
  // M = D (.) dD -> s5;  dX -> s4
  if (reg) {
    zero_acc(acc);
    mm64<NT>(acc, s6, s2);  // dR Delta^T
    float gacc[kRows][4];
    zero_acc(gacc);
    mm64<NT, kE, kE>(gacc, X, X);   // G
    __syncthreads();        // s4 (T), s5 consumed
    float dea[kRows] = {};
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = out_row<NT>(i), ci = out_col<NT>(j);
        float dg = 0.f, m = 0.f;
        if (ci < r) {
          const float D = __expf(gs.g[r] - gs.g[ci]);
          const float dA = -acc[i][j];
          dea[i] += dA * D * gacc[i][j];          // d eta through A = diag(eta) L
          const float dL = gs.eta[r] * dA;
          dg = dL * D;                              // dG (strictly lower)
          m = D * dL * gacc[i][j];                  // D (.) dD
        }
        s1[r * LDM + ci] = dg;
        s5[r * LDM + ci] = m;
      }
    // d eta: a row's columns sit in the four lanes of one gid and in four
    // warps; reduce over the lanes, then one shared-memory add per warp
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      float v = dea[i];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      if ((tid & 3) == 0) atomicAdd(&deta[out_row<NT>(i)], v);
    }
    __syncthreads();
    zero_acc(acc);
    mm64<NN, false, kE>(acc, s1, X);   // dG X
    mm64<TN, false, kE>(acc, s1, X);   // dG^T X
    float dx2[kRows][4];
    zero_acc(dx2);
    mm64<NT>(dx2, s6, S0);  // dR S0^T (NT layout)
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s4[out_row<NN>(i) * LDM + out_col<NN>(j)] = acc[i][j];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = out_row<NT>(i), cc = out_col<NT>(j);
        s4[r * LDM + cc] -= gs.eta[r] * gs.Gam[r] * dx2[i][j];
      }
  } else {
    for (int i = tid; i < kN * kN; i += kThr) {
      s4[(i / kN) * LDM + i % kN] = 0.f;
      s5[(i / kN) * LDM + i % kN] = 0.f;
    }
  }
  __syncthreads();
  // dO Delta^T -> M += (dO Delta^T) (.) (P (.) D); dP = (dO Delta^T) (.) D -> s1
  zero_acc(acc);
  mm64<NT, kE>(acc, dO, s2);
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = out_row<NT>(i), ci = out_col<NT>(j);
      s5[r * LDM + ci] += acc[i][j] * s3[r * LDM + ci];
      s1[r * LDM + ci] = dmask(gs, r, ci) * acc[i][j];
    }
  __syncthreads();
  // dQ = diag(Gamma) dO S0^T + dP X
  {
    float qa[kRows][4], qb[kRows][4];
    zero_acc(qa);
    mm64<NT, kE>(qa, dO, S0);
    zero_acc(qb);
    mm64<NN, false, kE>(qb, s1, X);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s6[out_row<NT>(i) * LDM + out_col<NT>(j)] = gs.Gam[out_row<NT>(i)] * qa[i][j];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s6[out_row<NN>(i) * LDM + out_col<NN>(j)] += qb[i][j];
  }
  // dX += dP^T Q + diag(E) Delta dS1^T
  zero_acc(acc);
  mm64<TN, false, kE>(acc, s1, Q);
  {
    float xa[kRows][4];
    zero_acc(xa);
    mm64<NT>(xa, s2, dS1);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s4[out_row<TN>(i) * LDM + out_col<TN>(j)] += acc[i][j];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = out_row<NT>(i);
        s4[r * LDM + out_col<NT>(j)] += gs.E[r] * xa[i][j];
      }
  }
  // row and column sums of M, <S0, dS1>
  {
    const float rs = row_sum([&](int r, int cc) { return s5[r * LDM + cc]; });
    const float cs = row_sum([&](int r, int cc) { return s5[cc * LDM + r]; });
    const float sd = row_sum([&](int r, int cc) { return S0[r * LDM + cc] * dS1[r * LDM + cc]; });
    if (tid % kRowT == 0) { rowM[tid / kRowT] = rs; colM[tid / kRowT] = cs; dgv[tid / kRowT] = sd; }
  }
  __syncthreads();
  // outputs: dq, dk (with the norm term), dbeta, dlambda
  for (int i = tid; i < kN * kN / 8; i += kThr) {
    const int r = i / (kN / 8), cc = (i % (kN / 8)) * 8, t = t0 + r;
    if (t >= a.T) continue;
    float v8[8], x8[8];
    lds8(v8, &s6[r * LDM + cc]);
    stx8<Tin>(a.dq, (((size_t)b * a.T + t) * a.H + h) * kN + cc, v8);
    const float dn = gs.ex[r] != 0.f ? -deta[r] * gs.eta[r] / (a.eps + gs.nrm[r]) : 0.f;
    lds8(v8, &s4[r * LDM + cc]);
    lds8(x8, &X[r * LDM + cc]);
#pragma unroll
    for (int e = 0; e < 8; ++e) v8[e] += 2.f * dn * x8[e];
    if (t - a.shift >= 0) stx8<Tin>(a.dk, (((size_t)b * a.T + (t - a.shift)) * a.H + h) * kN + cc, v8);
    else if (a.dk_prev) stx8<Tin>(a.dk_prev, (size_t)bh * kN + cc, v8);
  }
  if (tid < 32) {  // gate gradients: dg_r, then the reverse cumulative sum over the chunk
    const float sdS = [&] {
      float s = 0.f;
      for (int r = tid; r < kN; r += 32) s += dgv[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      return s;
    }();
    float sE = EdE[tid] + EdE[tid + 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sE += __shfl_xor_sync(0xffffffffu, sE, o);
    float d[2];
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      const int r = tid + 32 * hlf;
      float dG = dGo[r] + dGr[r] + (r == kN - 1 ? sdS : 0.f);
      d[hlf] = gs.Gam[r] * dG + rowM[r] - colM[r] - EdE[r] + (r == kN - 1 ? sE : 0.f);
    }
    // reverse inclusive scan: dl_s = sum_{r >= s} dg_r
    float v1 = d[1], v0 = d[0];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n1 = __shfl_down_sync(0xffffffffu, v1, o), n0 = __shfl_down_sync(0xffffffffu, v0, o);
      if (tid + o < 32) { v1 += n1; v0 += n0; }
    }
    v0 += __shfl_sync(0xffffffffu, v1, 0);
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      const int r = tid + 32 * hlf, t = t0 + r;
      if (t >= a.T) continue;
      const size_t gi = ((size_t)b * a.T + t) * a.H + h;
      const float dl = hlf ? v1 : v0;
      const float om = 1.f - a.lam[gi];
      a.dlam[gi] = (om >= a.eps_gamma && om <= 1.f) ? -dl / gs.gam[r] : 0.f;
      a.dbeta[gi] = gs.ex[r] != 0.f ? deta[r] / (a.eps + gs.nrm[r]) : 0.f;
    }
  }
  if (a.shift == 1 && c == a.NC - 1)  // the last key is the x of no pair of this call
    for (int cc = tid; cc < kN; cc += kThr) stx<Tin>(a.dk, (((size_t)b * a.T + (a.T - 1)) * a.H + h) * kN + cc, 0.f);
  if (c == 0 && a.dk_prev && a.shift == 0)
    for (int cc = tid; cc < kN; cc += kThr) stx<Tin>(a.dk_prev, (size_t)bh * kN + cc, 0.f);
}

// ---------------------------------------------------------------- (d) on tcgen05
// The gradient kernel for bf16 inputs, every 64 x 64 x 64 product a chain of
// tcgen05 MMAs (kind::f16, M = N = 64, fp32 accumulators in TMEM).  An fp32
// operand is split into bf16 hi = bf16(x) and lo = bf16(x - hi), 16
// significant bits together, and a b ~ a_hi b_hi + a_hi b_lo + a_lo b_hi
// (the dropped terms are ~2^-16 of |a| |b|); keys, queries and output
// gradients are exact in bf16 and take one image.  Each matrix sits in
// shared memory once, as 64 rows of 64 bf16 with the 128-byte swizzle: the
// same image is a K-major operand where its rows run along M (or N) and an
// MN-major one where they run along K, so transposed products need no
// transposed copy.  A thread owns one row and 16 columns of every 64 x 64
// result (an M = 64 accumulator keeps row 16 q + l in TMEM lane 32 q + l),
// so the element-wise work runs in registers and each result is written
// back as images straight from them.  Thirteen image slots, reused as their
// images die, and four 64-column accumulators: two CTAs share an SM.
namespace gtc {
constexpr int kImg = 64 * 128;
enum {
  I_X = 0, I_Q, I_DO,       // exact inputs
  I_DL, I_S0, I_DS1,        // hi images: Delta (then diag(E) Delta), the start state, the end-state gradient
  I_DLL, I_S0L, I_DS1L,     // their lo images
  I_W, I_WL,                // W; then P (.) D; then dDelta; then dG | dP (one image each)
  I_T, I_TL,                // T; then dR (then -diag(eta Gamma) dR)
  kImgs
};
enum { R_DGO = 0, R_EDE, R_DE, R_DGR, R_DEA, R_ROWM, R_SD, kRed };  // row sums, by column half
struct Tail {
  GateSm gs;
  float red[kRed][2][kN];
  float colM[4][kN];  // column sums of M by row quarter
  uint64_t bar;       // the MMA steps
  uint64_t ld;        // the bulk copies of the workspace's images
  uint32_t tmem;
  int pad;
};
constexpr size_t kSmem = 1024 + (size_t)kImgs * kImg + sizeof(Tail);
static_assert(2 * (kSmem + 1024) <= 228 * 1024, "two CTAs per SM");

// D (+)= op(A) op(B) over K = 64 (M = 64, N columns): the hi x hi term, then
// hi x lo and lo x hi where that operand has a low part.  amn / bmn: the
// image's rows run along K.
__device__ __forceinline__ void terms(uint32_t d, uint32_t ahi, uint32_t alo, bool asp, bool amn, uint32_t bhi,
                                      uint32_t blo, bool bsp, bool bmn, bool accumulate, int N = 64) {
  const uint32_t id = tc::idesc_bf16(64, N, amn, bmn);
  auto dsc = [](uint32_t s, bool mn, int ks) { return mn ? tcu::mndesc(s, ks) : tcu::kdesc<64>(s, ks); };
  uint32_t on = accumulate ? 1u : 0u;
#pragma unroll
  for (int ks = 0; ks < 4; ++ks, on = 1u) tc::umma_bf16(d, dsc(ahi, amn, ks), dsc(bhi, bmn, ks), id, on);
  if (bsp)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) tc::umma_bf16(d, dsc(ahi, amn, ks), dsc(blo, bmn, ks), id, 1u);
  if (asp)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) tc::umma_bf16(d, dsc(alo, amn, ks), dsc(bhi, bmn, ks), id, 1u);
}

// 16 fp32 values of row r, columns c0 .. c0 + 15, into the hi and lo images
__device__ __forceinline__ void put_split(uint8_t* hi, uint8_t* lo, int r, int c0, const float (&v)[16]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x0 = v[8 * j + 2 * e], x1 = v[8 * j + 2 * e + 1];
      const __nv_bfloat162 hv = __floats2bfloat162_rn(x0, x1);
      const float2 hf = __bfloat1622float2(hv);
      const __nv_bfloat162 lv = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
      ph[e] = *reinterpret_cast<const uint32_t*>(&hv);
      pl[e] = *reinterpret_cast<const uint32_t*>(&lv);
    }
    const uint32_t off = tcu::sw128(r, c0 + 8 * j);
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
    *reinterpret_cast<uint4*>(lo + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
  }
}
// The first 1024-byte boundary of a dynamic shared-memory array, as an
// offset from the array itself, so that the compiler keeps the pointers in
// the shared space (shared loads and stores, not generic ones).
__device__ __forceinline__ uint8_t* shared_align1024(uint8_t* raw) {
  return raw + ((1024u - (tc::smem_u32(raw) & 1023u)) & 1023u);
}
// 16 fp32 values of row r, columns c0 .. c0 + 15, into one bf16 image
__device__ __forceinline__ void put_one(uint8_t* im, int r, int c0, const float (&v)[16]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t ph[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) ph[e] = tcu::pack_bf16(v[8 * j + 2 * e], v[8 * j + 2 * e + 1]);
    *reinterpret_cast<uint4*>(im + tcu::sw128(r, c0 + 8 * j)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
  }
}
// 16 values of an exact image's row r from column c0
__device__ __forceinline__ void get_row(float (&v)[16], const uint8_t* im, int r, int c0) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint4 p = *reinterpret_cast<const uint4*>(im + tcu::sw128(r, c0 + 8 * j));
    const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&p);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(e[q]);
      v[8 * j + 2 * q] = f.x;
      v[8 * j + 2 * q + 1] = f.y;
    }
  }
}
__device__ __forceinline__ void ld16(float (&v)[16], const float* p) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 f = reinterpret_cast<const float4*>(p)[k];
    v[4 * k] = f.x; v[4 * k + 1] = f.y; v[4 * k + 2] = f.z; v[4 * k + 3] = f.w;
  }
}
// keys (with the pairing's shift and the carried key), queries and output
// gradients of the chunk as exact bf16 images
__device__ __forceinline__ void load_xqdo(const CbArgs& a, uint8_t* ix, uint8_t* iq, uint8_t* ido, int b, int h,
                                          int t0, int64_t pos, int bh) {
  using Tin = __nv_bfloat16;
  uint4 px[2], pq[2], pd[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = threadIdx.x + kThr * k, r = i >> 3, ch = i & 7, tr = t0 + r;
    const Tin* row = nullptr;
    if (tr < a.T && pos + tr >= a.shift) {
      if (tr - a.shift >= 0) row = reinterpret_cast<const Tin*>(a.k) + (((size_t)b * a.T + (tr - a.shift)) * a.H + h) * kN;
      else if (a.kprev_in) row = reinterpret_cast<const Tin*>(a.kprev_in) + (size_t)bh * kN;
    }
    const size_t gi = (((size_t)b * a.T + tr) * a.H + h) * kN + 8 * ch;
    px[k] = row ? *reinterpret_cast<const uint4*>(row + 8 * ch) : make_uint4(0u, 0u, 0u, 0u);
    pq[k] = tr < a.T ? *reinterpret_cast<const uint4*>(reinterpret_cast<const Tin*>(a.q) + gi) : make_uint4(0u, 0u, 0u, 0u);
    pd[k] = tr < a.T ? *reinterpret_cast<const uint4*>(reinterpret_cast<const Tin*>(a.dO) + gi) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = threadIdx.x + kThr * k, r = i >> 3, ch = i & 7;
    const uint32_t off = (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4));
    *reinterpret_cast<uint4*>(ix + off) = px[k];
    *reinterpret_cast<uint4*>(iq + off) = pq[k];
    *reinterpret_cast<uint4*>(ido + off) = pd[k];
  }
}
// 16 values of row t of a [B, T, H, 64] bf16 tensor from column c0 (zero past T)
__device__ __forceinline__ void load_row16(float (&v)[16], const void* src, const CbArgs& a, int b, int h, int t,
                                           int c0) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint4 p = t < a.T ? *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(src) +
                                                            (((size_t)b * a.T + t) * a.H + h) * kN + c0 + 8 * j)
                            : make_uint4(0u, 0u, 0u, 0u);
    const __nv_bfloat162* e2 = reinterpret_cast<const __nv_bfloat162*>(&p);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(e2[q]);
      v[8 * j + 2 * q] = f.x;
      v[8 * j + 2 * q + 1] = f.y;
    }
  }
}
__device__ __forceinline__ void st16(float* p, const float (&v)[16]) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    reinterpret_cast<float4*>(p)[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}

// Element (r, c) of a 64 x 64 fp32 matrix in shared memory whose 16-byte
// pieces are permuted within each row (piece q at q ^ (r & 7)): eight
// consecutive rows read or written at one column hit different banks.
__device__ __forceinline__ int swz(int r, int c) { return r * kN + ((((c >> 2) ^ (r & 7))) << 2) + (c & 3); }
// the four values (r, c .. c + 3), c a multiple of 4
__device__ __forceinline__ float4 ld4s(const float* m, int r, int c) {
  return *reinterpret_cast<const float4*>(m + swz(r, c));
}
__device__ __forceinline__ void st4s(float* m, int r, int c, float4 v) { *reinterpret_cast<float4*>(m + swz(r, c)) = v; }
}  // namespace gtc

__global__ void __launch_bounds__(kThr, 2) bwdc_grad_tc_kernel(CbArgs a) {
  using namespace gtc;
  extern __shared__ uint8_t gtc_raw[];
  uint8_t* base = shared_align1024(gtc_raw);
  auto img = [&](int i) { return base + (size_t)i * kImg; };
  auto sa = [&](int i) { return tc::smem_u32(base + (size_t)i * kImg); };
  Tail& tl = *reinterpret_cast<Tail*>(base + (size_t)kImgs * kImg);
  GateSm& gs = tl.gs;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int R = 16 * quad + (lane & 15), C0 = 32 * half + 16 * (lane >> 4);  // this thread's row and columns
  const size_t cg = blockIdx.x;
  const int c = (int)(cg % a.NC), bh = (int)(cg / a.NC), b = bh / a.H, h = bh % a.H, t0 = c * kN;
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  const bool reg = !a.additive;
  const int t = t0 + R;
  using Tin = __nv_bfloat16;

  if (warp == 0) {
    tc::tmem_alloc(&tl.tmem, 256);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    tc::mbar_init(&tl.bar, 1);
    tc::mbar_init(&tl.ld, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();  // the barriers are initialised
  // ---- loads, one round: the workspace's images of S0, dS1, W and T by bulk
  // copies, the gates by cp.async, keys, queries, output gradients as
  // images, this thread's U and V
  if (tid == 0) {
    tc::mbar_arrive_expect_tx(&tl.ld, (reg ? 4u : 2u) * 2u * kImg);
    const uint8_t* s0 = reinterpret_cast<const uint8_t*>(wsmat(a, cg, M_S0));
    const uint8_t* ds = reinterpret_cast<const uint8_t*>(wsmat(a, cg, M_DS1));
    tc::bulk_load(img(I_S0), s0, kImg, &tl.ld);
    tc::bulk_load(img(I_S0L), s0 + kImg, kImg, &tl.ld);
    tc::bulk_load(img(I_DS1), ds, kImg, &tl.ld);
    tc::bulk_load(img(I_DS1L), ds + kImg, kImg, &tl.ld);
    if (reg) {
      tc::bulk_load(img(I_W), wsmat(a, cg, M_W), 2 * kImg, &tl.ld);
      tc::bulk_load(img(I_T), wsmat(a, cg, M_T), 2 * kImg, &tl.ld);
    }
  }
  if (tid < (int)(sizeof(GateSm) / 16)) cp16(reinterpret_cast<float*>(&gs) + 4 * tid, wsgate(a, cg) + 4 * tid);
  cp_commit();
  load_xqdo(a, img(I_X), img(I_Q), img(I_DO), b, h, t0, pos, bh);
  float vv[16], u[16];
  load_row16(vv, a.v, a, b, h, t, C0);
  if (reg) ld16(u, wsmat(a, cg, M_U) + R * kN + C0);
  cp_wait0();
  bool ok = tc::mbar_wait(&tl.ld, 0, a.wait_ns);
  ok = !__syncthreads_or(!ok);
  tc::fence_proxy_async();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tl.tmem;
  const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
  auto acc = [&](int s) { return tmem + (uint32_t)(64 * s); };
  auto tld = [&](int s, float (&v)[16]) {
    uint32_t r[16];
    tc::tmem_ld16x2_16(tmem + lane_off + (uint32_t)(64 * s + 32 * half), r);
    tc::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
  };
  // row sums: the two threads of a row in this warp, then one entry per column half
  auto row_part = [&](int which, float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    if (lane < 16) tl.red[which][half][R] = v;
  };
  auto row_sum = [&](int which, int r) { return tl.red[which][0][r] + tl.red[which][1][r]; };
  // a row block of a split image pair, back in fp32 (hi + lo)
  auto get_split = [&](float (&v)[16], int hi, int lo) {
    float l[16];
    get_row(v, img(hi), R, C0);
    get_row(l, img(lo), R, C0);
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] += l[e];
  };
  uint32_t phase = 0;
  // every thread waits for the step's MMAs; all agree on the outcome
  auto wait_step = [&]() {
    const bool mine = tc::mbar_wait(&tl.bar, phase, a.wait_ns);
    phase ^= 1u;
    tc::tc_fence_after();
    ok = !__syncthreads_or(!mine);
    return ok;
  };
  // the images written since the last step are visible to the MMAs, and
  // every accumulator read so far is done
  auto step_barrier = [&]() {
    tc::fence_proxy_async();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
  };
  const float etaR = gs.eta[R], GamR = gs.Gam[R], ER = gs.E[R], gR = gs.g[R];

  do {
    if (!ok) break;
    {  // <S0, dS1> by rows
      float s0[16], ds[16], sd = 0.f;
      get_split(s0, I_S0, I_S0L);
      get_split(ds, I_DS1, I_DS1L);
#pragma unroll
      for (int e = 0; e < 16; ++e) sd = fmaf(s0[e], ds[e], sd);
      row_part(R_SD, sd);
    }
    // ---- step 1: W S0, Q S0, Q X^T, X dS1
    if (tid == 0) {
      if (reg) terms(acc(0), sa(I_W), sa(I_WL), true, false, sa(I_S0), sa(I_S0L), true, true, false);
      terms(acc(1), sa(I_Q), 0, false, false, sa(I_S0), sa(I_S0L), true, true, false);
      terms(acc(2), sa(I_Q), 0, false, false, sa(I_X), 0, false, false, false);
      terms(acc(3), sa(I_X), 0, false, false, sa(I_DS1), sa(I_DS1L), true, true, false);
      tc::umma_commit(&tl.bar);
    }
    if (!wait_step()) break;

    // ---- E1: Delta; dGamma through the output term; P (.) D (into W's slots); E dE
    float dl[16], pv[16];
    if (reg) {
      tld(0, pv);
#pragma unroll
      for (int e = 0; e < 16; ++e) dl[e] = u[e] - pv[e];
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) dl[e] = etaR * vv[e];
    }
    put_split(img(I_DL), img(I_DLL), R, C0, dl);
    {
      float dov[16], s = 0.f;
      get_row(dov, img(I_DO), R, C0);
      tld(1, pv);
#pragma unroll
      for (int e = 0; e < 16; ++e) s = fmaf(dov[e], pv[e], s);
      row_part(R_DGO, s);
    }
    {
      float pd[16];
      tld(2, pv);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int cc = C0 + e;
        pd[e] = cc <= R ? __expf(gR - gs.g[cc]) * pv[e] : 0.f;
      }
      put_split(img(I_W), img(I_WL), R, C0, pd);
    }
    {
      float s = 0.f;
      tld(3, pv);
#pragma unroll
      for (int e = 0; e < 16; ++e) s = fmaf(pv[e], dl[e], s);
      row_part(R_EDE, s);
    }
    step_barrier();

    // ---- step 2: (P (.) D)^T dO, X S0
    if (tid == 0) {
      terms(acc(0), sa(I_W), sa(I_WL), true, true, sa(I_DO), 0, false, true, false);
      if (reg) terms(acc(1), sa(I_X), 0, false, false, sa(I_S0), sa(I_S0L), true, true, false);
      tc::umma_commit(&tl.bar);
    }
    if (!wait_step()) break;
    // ---- E2: dDelta = (P (.) D)^T dO + diag(E) X dS1
    float dd[16];
    {
      float p2[16];
      tld(0, pv);
      tld(3, p2);
#pragma unroll
      for (int e = 0; e < 16; ++e) dd[e] = pv[e] + ER * p2[e];
    }
    if (reg) {
      put_split(img(I_W), img(I_WL), R, C0, dd);  // dDelta (P (.) D is consumed)
      step_barrier();
      // ---- step 3: dR = T^T dDelta; G = X X^T
      if (tid == 0) {
        terms(acc(0), sa(I_T), sa(I_TL), true, true, sa(I_W), sa(I_WL), true, true, false);
        terms(acc(3), sa(I_X), 0, false, false, sa(I_X), 0, false, false, false);
        tc::umma_commit(&tl.bar);
      }
      if (!wait_step()) break;
      tld(0, dd);
    }
    // ---- E3 (dd holds dR): dV, d eta and dGamma through the residual; dR into T's slots
    if (t < a.T) {
      float v8[8];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int e = 0; e < 8; ++e) v8[e] = etaR * dd[8 * j + e];
        stx8<Tin>(a.dv, (((size_t)b * a.T + t) * a.H + h) * kN + C0 + 8 * j, v8);
      }
    }
    {
      float de = 0.f, dgr = 0.f;
      if (reg) {
        tld(1, pv);  // X S0
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          de = fmaf(dd[e], vv[e] - GamR * pv[e], de);
          dgr = fmaf(dd[e], pv[e], dgr);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) de = fmaf(dd[e], vv[e], de);
      }
      row_part(R_DE, de);
      row_part(R_DGR, dgr);
    }
    put_split(img(I_T), img(I_TL), R, C0, dd);
    step_barrier();

    // ---- step 4: dR Delta^T, dO Delta^T
    if (tid == 0) {
      if (reg) terms(acc(0), sa(I_T), sa(I_TL), true, false, sa(I_DL), sa(I_DLL), true, false, false);
      terms(acc(1), sa(I_DO), 0, false, false, sa(I_DL), sa(I_DLL), true, false, false);
      tc::umma_commit(&tl.bar);
    }
    if (!wait_step()) break;
    // ---- E4: dG (A = diag(eta) L), M = D (.) dD, dP; the row scales of
    // step 5's last terms applied to the Delta and dR images in place
    {
      float dod[16], qx[16], dra[16], gg[16], m[16], dp[16], dg[16];
      tld(1, dod);
      tld(2, qx);
      if (reg) {
        tld(0, dra);
        tld(3, gg);
      }
      float dea = 0.f, rm = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int cc = C0 + e;
        const float D = cc <= R ? __expf(gR - gs.g[cc]) : 0.f;
        float me = dod[e] * D * qx[e];  // (dO Delta^T) (.) (P (.) D)
        dp[e] = D * dod[e];
        dg[e] = 0.f;
        if (reg && cc < R) {
          const float dA = -dra[e];
          dea = fmaf(dA * D, gg[e], dea);  // d eta through A = diag(eta) L
          const float dL = etaR * dA;
          dg[e] = dL * D;
          me = fmaf(D * dL, gg[e], me);
        }
        m[e] = me;
        rm += me;
      }
      row_part(R_DEA, dea);
      row_part(R_ROWM, rm);
      // column sums over this quadrant's 16 rows: a reduce-scatter over the
      // half-warp leaves lane l the sum of column C0 + (l & 15)
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
          const float send = up ? m[i] : m[i + o];
          const float keep = up ? m[i + o] : m[i];
          m[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      tl.colM[quad][C0 + (lane & 15)] = m[0];
      // dG and dP feed only dq and dk (bf16 results): one bf16 image each
      put_one(img(I_W), R, C0, dg);
      put_one(img(I_WL), R, C0, dp);
    }
    {
      float v[16];
      get_split(v, I_DL, I_DLL);
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] *= ER;
      put_split(img(I_DL), img(I_DLL), R, C0, v);  // diag(E) Delta
      if (reg) {
        get_split(v, I_T, I_TL);
        const float s = -etaR * GamR;
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] *= s;
        put_split(img(I_T), img(I_TL), R, C0, v);  // -diag(eta Gamma) dR
      }
    }
    step_barrier();

    // ---- step 5: dX = dP^T Q + (dG + dG^T) X + diag(E) Delta dS1^T - diag(eta Gamma) dR S0^T;
    // dP X; dO S0^T
    if (tid == 0) {
      terms(acc(0), sa(I_WL), 0, false, true, sa(I_Q), 0, false, true, false);
      if (reg) {
        terms(acc(0), sa(I_W), 0, false, false, sa(I_X), 0, false, true, true);
        terms(acc(0), sa(I_W), 0, false, true, sa(I_X), 0, false, true, true);
        terms(acc(0), sa(I_T), sa(I_TL), true, false, sa(I_S0), sa(I_S0L), true, false, true);
      }
      terms(acc(0), sa(I_DL), sa(I_DLL), true, false, sa(I_DS1), sa(I_DS1L), true, false, true);
      terms(acc(1), sa(I_WL), 0, false, false, sa(I_X), 0, false, true, false);
      terms(acc(2), sa(I_DO), 0, false, false, sa(I_S0), sa(I_S0L), true, false, false);
      tc::umma_commit(&tl.bar);
    }
    if (!wait_step()) break;
    // ---- E5: dq, dk (the TMEM loads are warp-wide: every lane takes them,
    // only the stores are limited to the call's rows)
    {
      float p1[16], p2[16];
      tld(2, p1);
      tld(1, p2);
#pragma unroll
      for (int e = 0; e < 16; ++e) p1[e] = GamR * p1[e] + p2[e];
      if (t < a.T) {
        stx8<Tin>(a.dq, (((size_t)b * a.T + t) * a.H + h) * kN + C0, *reinterpret_cast<float(*)[8]>(&p1[0]));
        stx8<Tin>(a.dq, (((size_t)b * a.T + t) * a.H + h) * kN + C0 + 8, *reinterpret_cast<float(*)[8]>(&p1[8]));
      }
    }
    {
      const float deta = row_sum(R_DE, R) + row_sum(R_DEA, R);
      const float dn = gs.ex[R] != 0.f ? -deta * etaR / (a.eps + gs.nrm[R]) : 0.f;
      float xr[16], p3[16];
      get_row(xr, img(I_X), R, C0);
      tld(0, p3);
#pragma unroll
      for (int e = 0; e < 16; ++e) p3[e] = fmaf(2.f * dn, xr[e], p3[e]);
      if (t < a.T) {
        Tin* dst = nullptr;
        if (t - a.shift >= 0) dst = reinterpret_cast<Tin*>(a.dk) + (((size_t)b * a.T + (t - a.shift)) * a.H + h) * kN;
        else if (a.dk_prev) dst = reinterpret_cast<Tin*>(a.dk_prev) + (size_t)bh * kN;
        if (dst) {
          stx8<Tin>(dst, C0, *reinterpret_cast<float(*)[8]>(&p3[0]));
          stx8<Tin>(dst, C0 + 8, *reinterpret_cast<float(*)[8]>(&p3[8]));
        }
      }
    }
    if (tid < 32) {  // gate gradients: dg_r, then the reverse cumulative sum over the chunk
      float sdS = row_sum(R_SD, tid) + row_sum(R_SD, tid + 32);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sdS += __shfl_xor_sync(0xffffffffu, sdS, o);
      float ede[2];
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) ede[hlf] = gs.E[tid + 32 * hlf] * row_sum(R_EDE, tid + 32 * hlf);
      float sE = ede[0] + ede[1];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sE += __shfl_xor_sync(0xffffffffu, sE, o);
      float d[2];
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int r = tid + 32 * hlf;
        const float dGr = reg ? -gs.eta[r] * row_sum(R_DGR, r) : 0.f;
        const float colM = tl.colM[0][r] + tl.colM[1][r] + tl.colM[2][r] + tl.colM[3][r];
        const float dG = row_sum(R_DGO, r) + dGr + (r == kN - 1 ? sdS : 0.f);
        d[hlf] = gs.Gam[r] * dG + row_sum(R_ROWM, r) - colM - ede[hlf] + (r == kN - 1 ? sE : 0.f);
      }
      float v1 = d[1], v0 = d[0];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float n1 = __shfl_down_sync(0xffffffffu, v1, o), n0 = __shfl_down_sync(0xffffffffu, v0, o);
        if (tid + o < 32) { v1 += n1; v0 += n0; }
      }
      v0 += __shfl_sync(0xffffffffu, v1, 0);
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int r = tid + 32 * hlf, tr = t0 + r;
        if (tr >= a.T) continue;
        const size_t gi = ((size_t)b * a.T + tr) * a.H + h;
        const float dl_ = hlf ? v1 : v0;
        const float om = 1.f - a.lam[gi];
        a.dlam[gi] = (om >= a.eps_gamma && om <= 1.f) ? -dl_ / gs.gam[r] : 0.f;
        a.dbeta[gi] = gs.ex[r] != 0.f ? (row_sum(R_DE, r) + row_sum(R_DEA, r)) / (a.eps + gs.nrm[r]) : 0.f;
      }
    }
    if (a.shift == 1 && c == a.NC - 1)  // the last key is the x of no pair of this call
      for (int cc = tid; cc < kN; cc += kThr) stx<Tin>(a.dk, (((size_t)b * a.T + (a.T - 1)) * a.H + h) * kN + cc, 0.f);
    if (c == 0 && a.dk_prev && a.shift == 0)
      for (int cc = tid; cc < kN; cc += kThr) stx<Tin>(a.dk_prev, (size_t)bh * kN + cc, 0.f);
  } while (false);
  if (!ok && tid == 0) atomicExch(a.status, tcu::kStatusTimeout);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tl.tmem, 256);
}

// ---------------------------------------------------------------- (a) on tcgen05
// The per-chunk preparation for bf16 inputs with its products on the tensor
// cores, in the images and thread layout of the gradient kernel above:
// A = diag(eta) (D (.) X X^T) and P (.) D from one step of MMAs; T = (I +
// A)^{-1} by forward substitution (a column per thread, as before); then
// W = T diag(eta Gamma) X, U = T diag(eta) V, Q^T diag(Gamma) dO and
// Z = (P (.) D)^T dO in one step, and in a last one W^T Z with the chain's
// transition A = Gamma_63 I - (diag(E) X)^T W (stored as hi | lo images) and
// offset b = (diag(E) X)^T U, so that a chain step is one product (additive:
// A = Gamma_63 I, no product).  Thirteen images and 256 TMEM columns: two
// CTAs share an SM.
namespace ptc {
enum {
  I_X = 0, I_Q, I_DO,
  I_PD, I_PDL,      // P (.) D
  I_M3, I_M3L,      // diag(Gamma) dO
  I_M1, I_M1L,      // diag(eta) V, then W
  I_MX, I_MXL,      // diag(eta Gamma) X, then Z
  I_T, I_TL,        // A as fp32 rows, then T
  kImgs
};
struct Tail {
  GateSm gs;
  float red[2][kN];
  uint64_t bar;
  uint32_t tmem;
  int pad;
};
constexpr size_t kSmem = 1024 + (size_t)kImgs * gtc::kImg + sizeof(Tail);
static_assert(2 * (kSmem + 1024) <= 228 * 1024, "two CTAs per SM");
}  // namespace ptc

__global__ void __launch_bounds__(kThr, 2) bwdc_prep_tc_kernel(CbArgs a) {
  using namespace ptc;
  extern __shared__ uint8_t ptc_raw[];
  uint8_t* base = gtc::shared_align1024(ptc_raw);
  auto img = [&](int i) { return base + (size_t)i * gtc::kImg; };
  auto sa = [&](int i) { return tc::smem_u32(base + (size_t)i * gtc::kImg); };
  Tail& tl = *reinterpret_cast<Tail*>(base + (size_t)kImgs * gtc::kImg);
  GateSm& gs = tl.gs;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int R = 16 * quad + (lane & 15), C0 = 32 * half + 16 * (lane >> 4);
  const size_t cg = blockIdx.x;
  const int c = (int)(cg % a.NC), bh = (int)(cg / a.NC), b = bh / a.H, h = bh % a.H, t0 = c * kN;
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  const bool reg = !a.additive;
  if (blockIdx.x == 0 && tid == 0) *a.status = 0u;  // each call starts with a clear status

  if (warp == 0) {
    tc::tmem_alloc(&tl.tmem, 256);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    tc::mbar_init(&tl.bar, 1);
    tc::fence_mbar_init();
  }
  float beta_r = 0.f, lam_r = 0.f;  // this row's gates (threads < 64), fetched with the inputs
  if (tid < kN && t0 + tid < a.T) {
    const size_t gi = ((size_t)b * a.T + t0 + tid) * a.H + h;
    beta_r = a.beta[gi];
    lam_r = a.lam[gi];
  }
  gtc::load_xqdo(a, img(I_X), img(I_Q), img(I_DO), b, h, t0, pos, bh);
  float vv[16];
  gtc::load_row16(vv, a.v, a, b, h, t0 + R, C0);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tl.tmem;
  const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
  auto acc = [&](int s) { return tmem + (uint32_t)(64 * s); };
  auto tld = [&](int s, float (&v)[16]) {
    uint32_t r[16];
    tc::tmem_ld16x2_16(tmem + lane_off + (uint32_t)(64 * s + 32 * half), r);
    tc::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
  };
  // gates: |x_r|^2 from this thread's 16 columns, summed over the row's four threads
  float xr[16];
  gtc::get_row(xr, img(I_X), R, C0);
  {
    float n = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) n = fmaf(xr[e], xr[e], n);
    n += __shfl_xor_sync(0xffffffffu, n, 16);
    if (lane < 16) tl.red[half][R] = n;
  }
  __syncthreads();
  if (tid < kN) {
    const int r = tid, t = t0 + r;
    const float n = tl.red[0][r] + tl.red[1][r];
    const bool live = t < a.T, ex = live && pos + t >= a.shift;
    gs.nrm[r] = n;
    gs.ex[r] = ex ? 1.f : 0.f;
    gs.eta[r] = ex ? beta_r / (a.eps + n) : 0.f;
    const float gm = live ? fminf(fmaxf(1.f - lam_r, a.eps_gamma), 1.f) : 1.f;
    gs.gam[r] = gm;
    gs.g[r] = live ? logf(gm) : 0.f;
  }
  __syncthreads();
  if (tid < 32) {  // inclusive prefix sum over the 64 rows
    float v0 = gs.g[tid], v1 = gs.g[tid + 32];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n0 = __shfl_up_sync(0xffffffffu, v0, o), n1 = __shfl_up_sync(0xffffffffu, v1, o);
      if (tid >= o) { v0 += n0; v1 += n1; }
    }
    v1 += __shfl_sync(0xffffffffu, v0, 31);
    gs.g[tid] = v0;
    gs.g[tid + 32] = v1;
  }
  __syncthreads();
  if (tid < kN) {
    gs.Gam[tid] = __expf(gs.g[tid]);
    gs.E[tid] = __expf(gs.g[kN - 1] - gs.g[tid]);
  }
  __syncthreads();
  const float etaR = gs.eta[R], GamR = gs.Gam[R], ER = gs.E[R], gR = gs.g[R];
  uint32_t phase = 0;
  bool ok = true;
  auto wait_step = [&]() {
    const bool mine = tc::mbar_wait(&tl.bar, phase, a.wait_ns);
    phase ^= 1u;
    tc::tc_fence_after();
    ok = !__syncthreads_or(!mine);
    return ok;
  };
  auto step_barrier = [&]() {
    tc::fence_proxy_async();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
  };

  do {
    // ---- step 1: X X^T, P = Q X^T
    if (tid == 0) {
      if (reg) gtc::terms(acc(0), sa(I_X), 0, false, false, sa(I_X), 0, false, false, false);
      gtc::terms(acc(1), sa(I_Q), 0, false, false, sa(I_X), 0, false, false, false);
      tc::umma_commit(&tl.bar);
    }
    {  // meanwhile: diag(Gamma) dO as images, the gates into the workspace
      float dov[16], m[16];
      gtc::get_row(dov, img(I_DO), R, C0);
#pragma unroll
      for (int e = 0; e < 16; ++e) m[e] = GamR * dov[e];
      gtc::put_split(img(I_M3), img(I_M3L), R, C0, m);
      float* gv = wsgate(a, cg);
      if (tid < kN) {
        gv[tid] = gs.g[tid];
        gv[kN + tid] = gs.Gam[tid];
        gv[2 * kN + tid] = gs.E[tid];
        gv[3 * kN + tid] = gs.eta[tid];
        gv[4 * kN + tid] = gs.nrm[tid];
        gv[5 * kN + tid] = gs.ex[tid];
        gv[6 * kN + tid] = gs.gam[tid];
      }
    }
    if (!wait_step()) break;
    // ---- E1: P (.) D as images; A = diag(eta) (D (.) X X^T) (strictly lower)
    // as fp32 rows (16-byte pieces permuted, gtc::swz); both accumulators in
    // one TMEM round trip, the decay mask formed once
    {
      uint32_t rp[16], rg[16];
      tc::tmem_ld16x2_16(tmem + lane_off + (uint32_t)(64 * 1 + 32 * half), rp);
      if (reg) tc::tmem_ld16x2_16(tmem + lane_off + (uint32_t)(64 * 0 + 32 * half), rg);
      tc::tmem_wait_ld();
      float p[16], am[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int cc = C0 + e;
        const float D = cc <= R ? __expf(gR - gs.g[cc]) : 0.f;
        p[e] = D * __uint_as_float(rp[e]);
        am[e] = cc < R ? etaR * D * __uint_as_float(rg[e]) : 0.f;
      }
      gtc::put_split(img(I_PD), img(I_PDL), R, C0, p);
      if (reg) {
        float* Aw = reinterpret_cast<float*>(img(I_M1));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          gtc::st4s(Aw, R, C0 + 4 * k, make_float4(am[4 * k], am[4 * k + 1], am[4 * k + 2], am[4 * k + 3]));
      }
    }
    step_barrier();
    if (reg) {
      // T = (I + A)^{-1} by 16 x 16 blocks (A in the slots of diag(eta) V's
      // images, T in those of diag(eta Gamma) X's, both fp32 rows, the images
      // written after): the diagonal blocks by forward substitution (a thread
      // per column), then block diagonal by block diagonal
      //   T_ij = -T_ii G_ij,  G_ij = sum_{k=j}^{i-1} A_ik T_kj  (i > j),
      // the G blocks kept in T's upper blocks, which are zeroed at the end.
      const float* Am = reinterpret_cast<const float*>(img(I_M1));
      float* Tm = reinterpret_cast<float*>(img(I_MX));
      using gtc::swz;
      if (tid < kN) {
        const int o = 16 * (tid >> 4), jj = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float ar[16], sv[4] = {r == jj ? 1.f : 0.f, 0.f, 0.f, 0.f};  // the row's loads first, four chains
#pragma unroll
          for (int i = 0; i < r; ++i) ar[i] = Am[swz(o + r, o + i)];
#pragma unroll
          for (int i = 0; i < r; ++i) sv[i & 3] = fmaf(-ar[i], x[i], sv[i & 3]);
          x[r] = (sv[0] + sv[1]) + (sv[2] + sv[3]);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tm[swz(o + r, o + jj)] = x[r];
      }
      __syncthreads();
      // levels: a thread takes row rr and columns 4 cq .. 4 cq + 3 of a block
      for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;
        const int blk = tid >> 6, rr = (tid >> 2) & 15, cq = tid & 3;
        if (blk < nb) {
          const int j = blk, i = j + d;
          float g[4] = {0.f, 0.f, 0.f, 0.f};
          for (int k = j; k < i; ++k) {
#pragma unroll
            for (int m4 = 0; m4 < 4; ++m4) {
              const float4 a4 = gtc::ld4s(Am, 16 * i + rr, 16 * k + 4 * m4);
              const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
              for (int mm = 0; mm < 4; ++mm) {
                const float4 t4 = gtc::ld4s(Tm, 16 * k + 4 * m4 + mm, 16 * j + 4 * cq);
                g[0] = fmaf(av[mm], t4.x, g[0]);
                g[1] = fmaf(av[mm], t4.y, g[1]);
                g[2] = fmaf(av[mm], t4.z, g[2]);
                g[3] = fmaf(av[mm], t4.w, g[3]);
              }
            }
          }
          gtc::st4s(Tm, rr, 16 * (1 + blk) + 4 * cq, make_float4(g[0], g[1], g[2], g[3]));  // G_ij in upper block (0, 1 + blk)
        }
        __syncthreads();
        if (blk < nb) {
          const int i = blk + d;
          float tv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int m4 = 0; m4 < 4; ++m4) {
            const float4 a4 = gtc::ld4s(Tm, 16 * i + rr, 16 * i + 4 * m4);
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
              const float4 g4 = gtc::ld4s(Tm, 4 * m4 + mm, 16 * (1 + blk) + 4 * cq);
              tv[0] = fmaf(av[mm], g4.x, tv[0]);
              tv[1] = fmaf(av[mm], g4.y, tv[1]);
              tv[2] = fmaf(av[mm], g4.z, tv[2]);
              tv[3] = fmaf(av[mm], g4.w, tv[3]);
            }
          }
          gtc::st4s(Tm, 16 * i + rr, 16 * blk + 4 * cq, make_float4(-tv[0], -tv[1], -tv[2], -tv[3]));
        }
        __syncthreads();
      }
      for (int e = tid; e < 6 * 256; e += kThr) {  // the upper blocks (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
        const int ub = e >> 8, bi = ub < 3 ? 0 : (ub < 5 ? 1 : 2), bj = ub < 3 ? ub + 1 : (ub < 5 ? ub - 1 : 3);
        Tm[swz(16 * bi + ((e >> 4) & 15), 16 * bj + (e & 15))] = 0.f;
      }
      __syncthreads();
      {  // T as images and into the workspace
        float tt[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 f = gtc::ld4s(Tm, R, C0 + 4 * k);
          tt[4 * k] = f.x; tt[4 * k + 1] = f.y; tt[4 * k + 2] = f.z; tt[4 * k + 3] = f.w;
        }
        gtc::put_split(img(I_T), img(I_TL), R, C0, tt);
        uint8_t* gt = reinterpret_cast<uint8_t*>(wsmat(a, cg, M_T));
        gtc::put_split(gt, gt + gtc::kImg, R, C0, tt);
      }
      __syncthreads();  // A and T read: their slots take the scaled operands of step 2
      {
        float m[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) m[e] = etaR * vv[e];
        gtc::put_split(img(I_M1), img(I_M1L), R, C0, m);
#pragma unroll
        for (int e = 0; e < 16; ++e) m[e] = etaR * GamR * xr[e];
        gtc::put_split(img(I_MX), img(I_MXL), R, C0, m);
      }
      step_barrier();
    }
    // ---- step 2: W = T diag(eta Gamma) X, U = T diag(eta) V, Q^T diag(Gamma) dO, Z = (P (.) D)^T dO
    if (tid == 0) {
      if (reg) {
        gtc::terms(acc(0), sa(I_T), sa(I_TL), true, false, sa(I_MX), sa(I_MXL), true, true, false);
        gtc::terms(acc(1), sa(I_T), sa(I_TL), true, false, sa(I_M1), sa(I_M1L), true, true, false);
        gtc::terms(acc(3), sa(I_PD), sa(I_PDL), true, true, sa(I_DO), 0, false, true, false);
      }
      gtc::terms(acc(2), sa(I_Q), 0, false, true, sa(I_M3), sa(I_M3L), true, true, false);
      tc::umma_commit(&tl.bar);
    }
    if (!wait_step()) break;
    // ---- E2: W and U into the workspace; W, U, Z and diag(E) X as images
    {
      float p[16];
      if (reg) {
        tld(0, p);
        {
          uint8_t* gw = reinterpret_cast<uint8_t*>(wsmat(a, cg, M_W));
          gtc::put_split(gw, gw + gtc::kImg, R, C0, p);
        }
        gtc::put_split(img(I_M1), img(I_M1L), R, C0, p);
        tld(1, p);
        gtc::st16(wsmat(a, cg, M_U) + R * kN + C0, p);
        gtc::put_split(img(I_M3), img(I_M3L), R, C0, p);
        tld(3, p);
        gtc::put_split(img(I_MX), img(I_MXL), R, C0, p);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) p[e] = etaR * vv[e];
        gtc::put_split(img(I_M3), img(I_M3L), R, C0, p);
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) p[e] = ER * xr[e];
      gtc::put_split(img(I_T), img(I_TL), R, C0, p);
    }
    step_barrier();
    // ---- step 3: W^T Z, (diag(E) X)^T W, (diag(E) X)^T U
    if (tid == 0) {
      if (reg) {
        gtc::terms(acc(0), sa(I_M1), sa(I_M1L), true, true, sa(I_MX), sa(I_MXL), true, true, false);
        gtc::terms(acc(1), sa(I_T), sa(I_TL), true, true, sa(I_M1), sa(I_M1L), true, true, false);
      }
      gtc::terms(acc(3), sa(I_T), sa(I_TL), true, true, sa(I_M3), sa(I_M3L), true, true, false);
      tc::umma_commit(&tl.bar);
    }
    if (!wait_step()) break;
    // ---- E3: Y = Q^T diag(Gamma) dO - W^T (P (.) D)^T dO; the chain's offset
    // b = (diag(E) X)^T U and transition A = Gamma_63 I - (diag(E) X)^T W
    {
      float y[16], p[16];
      tld(2, y);
      if (reg) {
        tld(0, p);
#pragma unroll
        for (int e = 0; e < 16; ++e) y[e] -= p[e];
      }
      gtc::st16(wsmat(a, cg, M_Y) + R * kN + C0, y);
      tld(3, p);
      gtc::st16(wsmat(a, cg, M_XT) + R * kN + C0, p);
      if (reg) {
        tld(1, p);
        const float g63 = gs.Gam[kN - 1];
#pragma unroll
        for (int e = 0; e < 16; ++e) p[e] = (C0 + e == R ? g63 : 0.f) - p[e];
        uint8_t* ac = reinterpret_cast<uint8_t*>(wsmat(a, cg, M_AC));
        gtc::put_split(ac, ac + gtc::kImg, R, C0, p);
      }
    }
  } while (false);
  if (!ok && tid == 0) atomicExch(a.status, tcu::kStatusTimeout);
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tl.tmem, 256);
}


// ---------------------------------------------------------------- (b), (c) on tcgen05
// The chains for bf16 inputs (one launch, blockIdx.z the direction: the two
// read only the preparation's results), one product per chunk step with the
// transition and offset formed by the preparation:
//   forward   S_{c+1} = A_c S_c + b_c       (S_c out: the chunk's start state),
//   backward  dS_c = A_c^T dS_{c+1} + Y_c   (dS_{c+1} out: its end-state gradient),
// the backward reading the same images MN-major; additive: A_c = Gamma_63 I.
// One CTA of 128 threads per (b, h, 32 value columns); a thread keeps a row
// and 16 columns of the slice in registers (the M = 64 accumulator layout);
// the next chunks' images arrive by bulk copies into a ring of stages.
namespace ctc {
constexpr int kSC = 32, kThr = 128, kNST = 3;
struct Smem {
  uint8_t A[kNST][2 * gtc::kImg];  // hi | lo images of A_c
  uint8_t S[2 * gtc::kImg];        // hi | lo images of the slice (32 of each row's 64 columns)
  uint64_t full[kNST];
  uint64_t done;
  uint32_t tmem;
  int pad;
};
constexpr size_t kSmem = 1024 + sizeof(Smem);
}  // namespace ctc

__global__ void __launch_bounds__(ctc::kThr) bwdc_chain_tc_kernel(CbArgs a) {
  using namespace ctc;
  const bool BWD = blockIdx.z != 0;  // the two chains are independent: one launch runs both
  extern __shared__ uint8_t ctc_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(gtc::shared_align1024(ctc_raw));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x, c0 = blockIdx.y * kSC;
  const int R = 16 * warp + (lane & 15), Cl = 16 * (lane >> 4), C = c0 + Cl;  // row, first column
  const bool reg = !a.additive;
  const size_t base = (size_t)bh * a.NC;
  auto chunk = [&](int n) { return BWD ? a.NC - 1 - n : n; };  // the chunk of step n
  if (warp == 0) {
    tc::tmem_alloc(&sm.tmem, 32);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kNST; ++s) tc::mbar_init(&sm.full[s], 1);
    tc::mbar_init(&sm.done, 1);
    tc::fence_mbar_init();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm.tmem;
  int issued = 0;  // thread 0: transitions requested
  auto issue = [&]() {
    const int s = issued % kNST;
    tc::mbar_arrive_expect_tx(&sm.full[s], 2 * gtc::kImg);
    tc::bulk_load(sm.A[s], wsmat(a, base + chunk(issued), M_AC), 2 * gtc::kImg, &sm.full[s]);
    ++issued;
  };
  if (reg && tid == 0)
    while (issued < kNST && issued < a.NC) issue();
  const int OFF = BWD ? M_Y : M_XT;
  float S[16], off[16];
  const float* init = BWD ? a.dS_final : a.S_in;
  if (init) gtc::ld16(S, init + ((size_t)bh * kN + R) * kN + C);
  else
#pragma unroll
    for (int e = 0; e < 16; ++e) S[e] = 0.f;
  if (a.NC > 0) gtc::ld16(off, wsmat(a, base + chunk(0), OFF) + R * kN + C);
  uint32_t dphase = 0;
  bool ok = true;
  for (int n = 0; n < a.NC; ++n) {
    const size_t cg = base + chunk(n);
    {  // the chunk's state out, as hi | lo images
      uint8_t* gi = reinterpret_cast<uint8_t*>(wsmat(a, cg, BWD ? M_DS1 : M_S0));
      gtc::put_split(gi, gi + gtc::kImg, R, C, S);
    }
    float nxt[16];
    if (n + 1 < a.NC) gtc::ld16(nxt, wsmat(a, base + chunk(n + 1), OFF) + R * kN + C);
    if (reg) {
      gtc::put_split(sm.S, sm.S + gtc::kImg, R, Cl, S);
      tc::fence_proxy_async();
      tc::tc_fence_before();
      __syncthreads();  // the slice's images are written, the last step's TMEM reads are done
      tc::tc_fence_after();
      bool mine = true;
      if (tid == 0) {
        const int s = n % kNST;
        mine = tc::mbar_wait(&sm.full[s], (uint32_t)((n / kNST) & 1), a.wait_ns);
        if (mine) {
          tc::tc_fence_after();
          const uint32_t ah = tc::smem_u32(sm.A[s]), sh = tc::smem_u32(sm.S);
          gtc::terms(tmem, ah, ah + gtc::kImg, true, BWD, sh, sh + gtc::kImg, true, true, false, kSC);
          tc::umma_commit(&sm.done);
        } else {
          tcu::mbar_arrive(&sm.done);  // release the others; the step is abandoned
        }
      }
      mine = tc::mbar_wait(&sm.done, dphase, a.wait_ns) && mine;
      dphase ^= 1u;
      tc::tc_fence_after();
      if (__syncthreads_or(!mine)) {
        ok = false;
        break;
      }
      if (tid == 0 && issued < a.NC) issue();  // the stage read by this step's product is free
      uint32_t r[16];
      tc::tmem_ld16x2_16(tmem + ((uint32_t)(32 * warp) << 16), r);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 16; ++e) S[e] = __uint_as_float(r[e]) + off[e];
    } else {
      const float g63 = wsgate(a, cg)[2 * kN - 1];  // Gamma of the chunk's last row
#pragma unroll
      for (int e = 0; e < 16; ++e) S[e] = fmaf(g63, S[e], off[e]);
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) off[e] = nxt[e];
  }
  if (ok && BWD && a.dS_in) gtc::st16(a.dS_in + ((size_t)bh * kN + R) * kN + C, S);
  if (!ok && tid == 0) {
    atomicExch(a.status, tcu::kStatusTimeout);
    // the copies still in flight land before the CTA leaves (bounded): the
    // last use of each stage
    for (int m = issued - kNST > 0 ? issued - kNST : 0; m < issued; ++m)
      tc::mbar_wait(&sm.full[m % kNST], (uint32_t)((m / kNST) & 1), a.wait_ns);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 32);
}

constexpr size_t prep_smem() { return 8 * kN * LDM * sizeof(float) + sizeof(GateSm) + 4 * kN * sizeof(float); }
constexpr size_t grad_smem() { return 12 * kN * LDM * sizeof(float) + sizeof(GateSm) + 8 * kN * sizeof(float); }

template <int SC>
int launch_chains(const CbArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(ChainSmem<SC>);
  if (!set_smem_limit(reinterpret_cast<const void*>(bwdc_fwd_chain_kernel<SC>), smem) ||
      !set_smem_limit(reinterpret_cast<const void*>(bwdc_bwd_chain_kernel<SC>), smem))
    return FALCON_ERR_CUDA;
  bwdc_fwd_chain_kernel<SC><<<dim3(a.B * a.H, kN / SC), kThrC, smem, s>>>(a);
  bwdc_bwd_chain_kernel<SC><<<dim3(a.B * a.H, kN / SC), kThrC, smem, s>>>(a);
  return FALCON_OK;
}

template <typename Tin>
int launch_bwdc_t(const CbArgs& a, cudaStream_t s) {
  const unsigned nch = (unsigned)(a.B * a.H * a.NC);
  auto prep = bwdc_prep_kernel<float>;
  auto grad = bwdc_grad_kernel<float>;
  if constexpr (sizeof(Tin) == 2) {  // bf16 inputs: the tensor-core kernels
    if (!set_smem_limit(reinterpret_cast<const void*>(bwdc_prep_tc_kernel), ptc::kSmem)) return FALCON_ERR_CUDA;
    bwdc_prep_tc_kernel<<<nch, kThr, ptc::kSmem, s>>>(a);
  } else {
    if (!set_smem_limit(reinterpret_cast<const void*>(prep), prep_smem()) ||
        !set_smem_limit(reinterpret_cast<const void*>(grad), grad_smem()))
      return FALCON_ERR_CUDA;
    prep<<<nch, kThr, prep_smem(), s>>>(a);
  }
  // 16-column chain slices when their CTAs fit one wave at two per SM, else 32
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FALCON_ERR_CUDA;
  if constexpr (sizeof(Tin) == 2) {
    if (!set_smem_limit(reinterpret_cast<const void*>(bwdc_chain_tc_kernel), ctc::kSmem)) return FALCON_ERR_CUDA;
    bwdc_chain_tc_kernel<<<dim3(a.B * a.H, kN / ctc::kSC, 2), ctc::kThr, ctc::kSmem, s>>>(a);
  } else {
    const int st = (long)a.B * a.H * (kN / 16) <= 2L * sms ? launch_chains<16>(a, s) : launch_chains<32>(a, s);
    if (st != FALCON_OK) return st;
  }
  if constexpr (sizeof(Tin) == 2) {
    if (!set_smem_limit(reinterpret_cast<const void*>(bwdc_grad_tc_kernel), gtc::kSmem)) return FALCON_ERR_CUDA;
    bwdc_grad_tc_kernel<<<nch, kThr, gtc::kSmem, s>>>(a);
  } else {
    grad<<<nch, kThr, grad_smem(), s>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace

bool backward_chunk_supported(int variant, int dk, int dv, int T) {
  return (variant == FALCON_1 || variant == FALCON_1A) && dk == 64 && dv == 64 && T >= 1;
}

// a 256-byte block with the status word, then per chunk the matrices, then the gate rows
size_t backward_chunk_ws_bytes(int B, int T, int H) {
  const size_t NC = (size_t)(T + kN - 1) / kN;
  return 256 + (size_t)B * H * NC * (kMats * kMat + kGateVecs * kN) * sizeof(float);
}

int launch_backward_chunk(const FwdArgs& f, const void* dO, const float* dS_final, void* dq, void* dk, void* dv,
                          float* dbeta, float* dlam, float* dS_in, void* dk_prev) {
  CbArgs a;
  a.B = f.B; a.T = f.T; a.H = f.H; a.NC = (f.T + kN - 1) / kN;
  a.shift = f.shift; a.additive = variant_additive(f.variant) ? 1 : 0;
  a.eps = f.eps; a.eps_gamma = f.eps_gamma;
  a.q = f.q; a.k = f.k; a.v = f.v; a.dO = dO; a.beta = f.beta; a.lam = f.lam;
  a.S_in = f.S_in; a.kprev_in = f.kprev_in; a.pos_in = f.pos_in; a.dS_final = dS_final;
  a.dq = dq; a.dk = dk; a.dv = dv; a.dbeta = dbeta; a.dlam = dlam; a.dS_in = dS_in; a.dk_prev = dk_prev;
  a.status = reinterpret_cast<uint32_t*>(f.ws);
  a.ws = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(f.ws) + 256);
  a.wait_ns = wait_limit_ns();
  return f.dtype == FALCON_BF16 ? launch_bwdc_t<__nv_bfloat16>(a, f.stream) : launch_bwdc_t<float>(a, f.stream);
}

}  // namespace falcon
