// Tensor-core chunk forward for Falcon-3 (NLMS regression write averaged over
// a window of the last W pairs), bf16 inputs, fp32 state, chunk 64,
// d_k = d_v = 64, 2 <= W <= 9.
//
// The step [JC Falcon家族六个变体各管一段 (Falcon-3 window mini-batch);
// FW Falcon 家族], with c_t = eta_t / n_t (eta_t from the window-average key
// energy, n_t the existing pairs of the window W(t) of step t) and the
// clamped decay gamma_t [JC 数学上的稳定阀门:正衰减钳制]:
//   S_t = gamma_t S_{t-1} + c_t sum_{p in W(t)} x_p (v_p - gamma_t S_{t-1}^T x_p)^T,  o_t = S_t^T q_t.
// Chunked form used here (a reading of the pages' chunk-parallel form
// [FW 三种等价形式; JC 三种视角看同一个更新] for the window write).  A chunk
// of 64 steps is cut into four sub-chunks of 16 steps; sub-chunk i reads the
// K = 15 + W keys x_{(i,kappa)} (pairs t0 - W + 1 + 16 i + kappa), and every
// write of a step of it lies in their span.  So, from a sub-chunk's start
// state S', S_t = Gamma_tau S' + X_i^T z_tau with z (K x d_v) obeying
//   z_tau = gamma (I - c D_tau G_i) z_{tau-1} + c D_tau (V_i - Gamma_tau X_i S'),
// D_tau selecting the window rows of step tau (existing pairs only) and G_i
// the sub-chunk's key Gram.  Hence z_tau = H_tau V_i - Gamma_tau F~_tau X_i S'
// with two K x K recurrences that do not see the state,
//   F~_tau = (I - c D G) F~_{tau-1} + c D          (no decay: it cancels),
//   H_tau  = gamma (I - c D G) H_{tau-1} + c D,
// and o_t = Gamma_tau q_t^T S' + h_tau^T V_i - Gamma_tau a~_tau^T X_i S' with
// a~ = F~^T X_i q_t, h = H^T X_i q_t.  The four sub-chunks then couple through
// the key-space unknowns w_i = z_16 of each: (I + N) w = [H_i V_i] - [g F~_i X_i] S0
// with N_ij = exp(g_i - g_j) F~_i X_i X_j^T (j < i; g the chunk's cumulative
// log-decay at sub-chunk ends), so with Tf = (I + N)^{-1} bd(exp(g_i) F~_i) and
// Th = (I + N)^{-1} bd(H_i) (96 x 96, block lower triangular) the chunk is
//   S1 = Gamma_last S0 - M S0 + b,   O = Q' S0 + O0,
//   M  = X~^T Tf X_s,  b = X~^T Th V_s,
//   Q' = diag(Gamma) Q - (bd(Gamma a~) + P Tf) X_s,  O0 = (bd(h) + P Th) V_s,
// X_s / V_s the stacked sub-chunk keys / values, X~ their rows scaled by
// exp(g_last - g_j), P_t,(j,.) = exp(g_t - g_j) (X_j q_t - G_ij^T a~_t) (j < i(t)).
// That is the Falcon-1 chain form, so:
//  (a) f3_chunk_kernel, persistent over (b, h, chunk), one CTA per SM:
//      TMA of the stacked keys, values and queries; the key Gram band and
//      X_s Q^T in one tcgen05 product (M = 128, N = 160); the sub-chunk
//      recurrences (F~ and H of a sub-chunk per warp) on the CUDA cores, a
//      lane per column; N, P, X~ and T = (I + N)^{-1} in closed block form
//      (bf16 image); then Z = [X~^T ; P] T (N = 96), [X~^T ; P] [Tf | Th] =
//      Z [bd(exp(g_i) F~_i) | bd(H_i)] (N = 192) and, from its rows plus the
//      block-diagonal terms, [-M ; Q' - Gamma Q] and [b ; O0] by two more
//      products (K = 96); the four tiles leave by one bulk copy.
//  (b) f3_chain_kernel, two CTAs per (b, h), each owning 32 value columns:
//      acc = [-M ; Q'] S0 (one tcgen05 product per chunk, N = 32), then
//      S1 = Gamma_last S0 + b + acc_top on the fp32 state in registers and
//      O = acc_bottom + O0; a producer warp streams the chunk records.
// Every wait is bounded; a timeout is recorded in the workspace status word
// (the chain computes nothing when the first kernel recorded one).

#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_util.cuh"

namespace falcon {

using namespace tc;
using namespace tcu;

namespace {

constexpr int kL = 16;        // steps per sub-chunk
constexpr int kNS = 4;        // sub-chunks per chunk
constexpr int kKP = 24;       // key slots per sub-chunk (15 + W <= 24)
constexpr int kNK = kNS * kKP;  // stacked key-space rows of a chunk (96)
constexpr int kWMax = 9;
constexpr int kGS = 100;      // fp32 row stride of the Gram and X_s Q^T scratch

struct F3Args {
  int B, T, H, W, NC;
  int shift;  // pair t uses key t - shift (1 prefix alignment, 0 same-step)
  float eps, eps_gamma;
  const float* beta;
  const float* lam;
  const int64_t* pos_in;
  const __nv_bfloat16* kprev_in;
  const __nv_bfloat16* winx_in;
  const __nv_bfloat16* winv_in;
  const float* S_in;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  float* S_out;
  __nv_bfloat16* kprev_out;
  __nv_bfloat16* winx_out;
  __nv_bfloat16* winv_out;
  int64_t* pos_out;
  uint32_t* status;
  uint8_t* ws_f3;     // per chunk: [-M ; Q'] | b | O0 | Gamma_last (kF3Rec bytes)
  __nv_bfloat16* o;   // [B, T, H, 64]
  uint64_t wait_ns;   // limit of every bounded wait
  int stall;          // failure-detection test hook: the per-chunk kernel's first CTA waits on
                      // a barrier that nothing completes, and so records a timeout
};

// per chunk in the workspace: [-M ; Q'] (128-row bf16 tile) | b | O0 (64-row
// bf16 tiles, 128B-swizzled) | Gamma_last (first of 64 fp32)
constexpr size_t kF3Rec = 16384 + 8192 + 8192 + 256;

struct F3ChunkSmem {
  // 1024-aligned tiles: stacked keys (96 rows) then queries (64 rows), one
  // K-major B operand of 160 rows; stacked values (96 rows)
  static constexpr size_t XS = 0, QS = 12288, VS = 20480;
  // Gram (96 x 96) and (X_s Q^T)^T (64 x 96) in fp32, later the K-major
  // A tiles -R_F and R_H (128 rows x 96, two 64-column slabs each)
  static constexpr size_t R1 = 32768, GS = R1, XQT = R1 + 96 * kGS * 4, RF = R1, RH = R1 + 32768;
  // in between (Gram and X_s Q^T read, -R_F / R_H not yet written): the
  // bf16 image of T = (I + N)^{-1} (MN-major B, two 96-row atoms) and the
  // K-major A tile Z = [X~^T ; P] T (128 rows x 96, two slabs)
  static constexpr size_t TI = R1, ZT = R1 + 24576;
  // [X~ | P^T] (MN-major A, two 96-row atoms), then the block-diagonal right
  // factor [bd(exp(g_i) F~_i) | bd(H_i)] (MN-major B, three 96-row atoms);
  // the output tiles reuse both once the products read them
  static constexpr size_t AT = 98304, TB = AT + 24576;
  static constexpr size_t OMQ = AT, OB = AT + 16384, OO = AT + 24576, OG = AT + 32768;
  // fp32: F~_i, H_i (24 x 24 each; before them the recurrences' step
  // operands, after them T_20), a~_t, h_t (64 x 24 each), N_ij (6 blocks;
  // before them the recurrences' spare rows and Gram band)
  static constexpr size_t FH = TB + 36864, AH = FH + 8 * 2304, NB = AH + 2 * 64 * 96;
  static constexpr size_t GT = NB + 6 * 2304;
  // gates (fp32 offsets in GT)
  static constexpr int G_C = 0, G_GMA = 64, G_G = 128, G_GAM = 192, G_EX = 256, G_NRM = 352, G_END = 448,
                       G_WS = 452, G_N = 456;
  static constexpr size_t BAR = GT + G_N * 4;
  static constexpr size_t MISC = BAR + 32;
  static constexpr size_t TOTAL = MISC + 16 + 1024;
  static constexpr uint32_t TX = 4 * 3072 * 2 + 8192;
  static constexpr uint32_t NCOLS = 256;
  static_assert(XQT + 64 * kGS * 4 <= RH + 32768 && RH + 32768 == AT, "R1 region");
  static_assert(ZT + 32768 <= AT, "T image and Z inside R1");
  static_assert((4 * 64 + kNS * kKP * 16) * 4 <= 6 * 2304, "spare rows and Gram band inside the N blocks");
  static_assert((128 * kKP + 64 * 12) * 4 <= 8 * 2304, "step operands inside F~ / H's region");
  static_assert(OG + 256 <= FH, "output tiles inside the product operands");
  static_assert(TOTAL <= 232448, "shared memory budget");
};

struct F3ChainSmem {
  static constexpr int NST = 4;                    // chunk records in flight
  static constexpr size_t MQ = 0, BO = 16384, OO = 24576, GO = 32768, STAGE = 33792;
  static constexpr int NB = 4;                     // S0 tiles and TMEM accumulators
  static constexpr size_t SB = NST * STAGE;        // S0 of chunk c in SB + (c % NB) 8192 (MN-major B,
                                                   // this CTA's 32 columns in columns 0..31)
  static constexpr size_t BAR = SB + NB * 8192;
  static constexpr size_t MISC = BAR + 256;
  static constexpr size_t TOTAL = MISC + 16 + 1024;
  static constexpr int kThreads = 160;             // chain 0..1, outputs 2..3, producer 4
  static_assert(STAGE % 1024 == 0 && GO + 256 <= STAGE, "stage layout");
  static_assert(TOTAL <= 232448, "shared memory budget");
};

// Key (x) and value of local pair j of (b, h): j >= shift from the sequence,
// j = 0 (prefix alignment) the carried key with the first value, j < 0 the
// carried window ring.
__device__ __forceinline__ __nv_bfloat16 pair_x(const F3Args& a, int b, int h, int j, int col, int64_t pos) {
  if (j >= a.shift) return a.k[(((size_t)b * a.T + (j - a.shift)) * a.H + h) * 64 + col];
  if (j == 0) return a.kprev_in ? a.kprev_in[((size_t)b * a.H + h) * 64 + col] : __float2bfloat16_rn(0.f);
  if (!a.winx_in || pos + j < a.shift) return __float2bfloat16_rn(0.f);
  const int Wr = a.W - 1;
  return a.winx_in[(((size_t)b * a.H + h) * Wr + ring_slot(pos + j, Wr)) * 64 + col];
}
__device__ __forceinline__ __nv_bfloat16 pair_v(const F3Args& a, int b, int h, int j, int col, int64_t pos) {
  if (j >= 0) return a.v[(((size_t)b * a.T + j) * a.H + h) * 64 + col];
  if (!a.winv_in || pos + j < a.shift) return __float2bfloat16_rn(0.f);
  const int Wr = a.W - 1;
  return a.winv_in[(((size_t)b * a.H + h) * Wr + ring_slot(pos + j, Wr)) * 64 + col];
}

// The sub-chunk's two K x K recurrences, F~ (undecayed) and H, side by side:
// lane j holds column j of both.  Step tau: the window rows tau + r (r < W) take
//   d_r = G[tau + r, :] M_{tau-1},  M_tau = gamma M_{tau-1} + Delta_tau,
//   Delta_tau[tau + r] = -gamma c m_{tau+r} d_r + c m_{tau+r} [j == tau + r]
// (gamma = 1 for F~).  A row that stays in the window needs no new sum over
// the K slots: d_r(tau) = gamma_{tau-1} d_{r+1}(tau - 1) + sum_a G[tau + r][tau - 1 + a]
// Delta_{tau-1}[a]; only the row entering the window takes the full sum, and
// one Gram element feeds both matrices.  The window is handled as kWMax rows
// with the increments of rows past W masked to zero.  The columns are kept in
// rotated order (register k holds row (tau + k) mod kKP at step tau) so that
// the window's rows sit in fixed registers while the steps run as a loop;
// the rotation is a register move per row and step.  After the update,
// outF[t][j] = F~ column j . (X_i q_t) and outH[t][j] = H column j . (X_i q_t);
// lanes past the key slots store into `spare` ([2][32] floats).  The step's
// operands are read as aligned 16-byte rows: `gr` [kL][kKP] the entering
// row's Gram entries in the registers' order, `gb` [kKP][16] the Gram band
// around the diagonal (row rho: G[rho][rho - 8 + o], zero off the block),
// `xqr` [kL][kKP] X_i q_t in that
// order, `scg` [kL][12] the window rows' c m (zero past W) and gamma.  On
// return f / hc hold the columns in row order.
__device__ __forceinline__ void sub_recurrences(const float* __restrict__ gb, const float* __restrict__ gr,
                                                const float* __restrict__ xqr, const float* __restrict__ scg,
                                                int i, int j, float* __restrict__ outF, float* __restrict__ outH,
                                                float* __restrict__ spare, float (&f)[kKP], float (&hc)[kKP]) {
  float fr[kKP], hr[kKP];
#pragma unroll
  for (int k = 0; k < kKP; ++k) {
    fr[k] = 0.f;
    hr[k] = 0.f;
  }
  float pf[kWMax], ph[kWMax], lf[kWMax], lh[kWMax];  // previous step's window sums and increments
#pragma unroll
  for (int r = 0; r < kWMax; ++r) {
    pf[r] = 0.f; ph[r] = 0.f; lf[r] = 0.f; lh[r] = 0.f;
  }
  float gprev = 1.f;
#pragma unroll 1
  for (int tau = 0; tau < kL; ++tau) {
    const int t = kL * i + tau;
    float sc[12];  // the window rows' c m (zero past W), then gamma
#pragma unroll
    for (int q = 0; q < 12; q += 4) {
      const float4 v4 = *reinterpret_cast<const float4*>(scg + t * 12 + q);
      sc[q] = v4.x; sc[q + 1] = v4.y; sc[q + 2] = v4.z; sc[q + 3] = v4.w;
    }
    const float gm = sc[kWMax];
    float df[kWMax], dh[kWMax];
    // rows that stay: carried sums plus last step's increments (side by side);
    // `gb` row rho holds G[rho][rho - 8 + o] at o, so row tau + r needs
    // o = 7 - r + a for the columns tau - 1 + a
#pragma unroll
    for (int r = 0; r < kWMax - 1; ++r) {
      float gv[12];
      const int b0 = (7 - r) / 4;  // first aligned block covering o = 7 - r .. 15 - r
      const float* row = gb + (tau + r) * 16 + 4 * b0;
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const float4 v4 = *reinterpret_cast<const float4*>(row + 4 * q);
        gv[4 * q] = v4.x; gv[4 * q + 1] = v4.y; gv[4 * q + 2] = v4.z; gv[4 * q + 3] = v4.w;
      }
      float af = pf[r + 1], ah = gprev * ph[r + 1];
#pragma unroll
      for (int a = 0; a < kWMax; ++a) {
        const float g = gv[7 - r + a - 4 * b0];
        af = fmaf(g, lf[a], af);
        ah = fmaf(g, lh[a], ah);
      }
      df[r] = af;
      dh[r] = ah;
    }
    {  // the row entering the window: the full sums (register k is row (tau + k) mod kKP,
       // `gr` holds that row's Gram entries in the same order)
      const float* grow = gr + tau * kKP;
      float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
      for (int q = 0; q < kKP; q += 4) {
        const float4 g4 = *reinterpret_cast<const float4*>(grow + q);
        a0 = fmaf(g4.x, fr[q], a0); a1 = fmaf(g4.y, fr[q + 1], a1);
        a0 = fmaf(g4.z, fr[q + 2], a0); a1 = fmaf(g4.w, fr[q + 3], a1);
        b0 = fmaf(g4.x, hr[q], b0); b1 = fmaf(g4.y, hr[q + 1], b1);
        b0 = fmaf(g4.z, hr[q + 2], b0); b1 = fmaf(g4.w, hr[q + 3], b1);
      }
      df[kWMax - 1] = a0 + a1;
      dh[kWMax - 1] = b0 + b1;
    }
#pragma unroll
    for (int k = 0; k < kKP; ++k) hr[k] *= gm;
#pragma unroll
    for (int r = 0; r < kWMax; ++r) {  // the window rows sit in registers 0 .. kWMax - 1
      const float inj = j == tau + r ? sc[r] : 0.f;
      const float incf = fmaf(-sc[r], df[r], inj), inch = fmaf(-gm * sc[r], dh[r], inj);
      fr[r] += incf;
      hr[r] += inch;
      pf[r] = df[r]; ph[r] = dh[r]; lf[r] = incf; lh[r] = inch;
    }
    gprev = gm;
    const float* xq = xqr + t * kKP;  // X_i q_t in the registers' row order
    float s0 = 0.f, s1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
    for (int q = 0; q < kKP; q += 4) {
      const float4 x4 = *reinterpret_cast<const float4*>(xq + q);
      s0 = fmaf(x4.x, fr[q], s0); s1 = fmaf(x4.y, fr[q + 1], s1);
      s0 = fmaf(x4.z, fr[q + 2], s0); s1 = fmaf(x4.w, fr[q + 3], s1);
      u0 = fmaf(x4.x, hr[q], u0); u1 = fmaf(x4.y, hr[q + 1], u1);
      u0 = fmaf(x4.z, hr[q + 2], u0); u1 = fmaf(x4.w, hr[q + 3], u1);
    }
    // lanes past the key slots store into the spare rows: no branch, so the
    // warp stays converged through the steps
    float* of = j < kKP ? outF + t * kKP + j : spare + j;
    float* oh = j < kKP ? outH + t * kKP + j : spare + 32 + j;
    *of = s0 + s1;
    *oh = u0 + u1;
    // rotate: register k takes row (tau + 1 + k) mod kKP
    const float f0 = fr[0], h0 = hr[0];
#pragma unroll
    for (int k = 0; k < kKP - 1; ++k) {
      fr[k] = fr[k + 1];
      hr[k] = hr[k + 1];
    }
    fr[kKP - 1] = f0;
    hr[kKP - 1] = h0;
    __syncwarp();
  }
  // after kL steps register k holds row (kL + k) mod kKP
#pragma unroll
  for (int k = 0; k < kKP; ++k) {
    f[(kL + k) % kKP] = fr[k];
    hc[(kL + k) % kKP] = hr[k];
  }
}

// ======================================================================
// (a) per-chunk operators, every (b, h, chunk) in parallel
// ======================================================================
__global__ void __launch_bounds__(256, 1)
    f3_chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k24,
                    const __grid_constant__ CUtensorMap tm_v24, F3Args a) {
  using L = F3ChunkSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);  // [0] loads, [1] products
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
  float* gt = reinterpret_cast<float*>(sm + L::GT);
  float* GS = reinterpret_cast<float*>(sm + L::GS);
  float* XQT = reinterpret_cast<float*>(sm + L::XQT);
  float* FH = reinterpret_cast<float*>(sm + L::FH);
  float* AHf = reinterpret_cast<float*>(sm + L::AH);  // a~ [64][24], then h [64][24]
  float* NBf = reinterpret_cast<float*>(sm + L::NB);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int W = a.W;
  const int n_items = a.NC * a.B * a.H;  // item = (b, h, chunk), chunk fastest
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0 && tid == 0) atomicExch(a.status, 0u);
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_init(&bar[2], 1);  // the test hook's (never completed)
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, L::NCOLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int quad = warp & 3;
  const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
  auto fail = [&]() {
    *abort_flag = 1;
    atomicExch(a.status, kStatusTimeout);
  };
  // the stacked keys and values of sub-chunk j are the 24 pairs from
  // t0 - W + 1 + 16 j; and the 64 queries (thread 0)
  auto issue_loads = [&](int item) {
    const int c = item % a.NC, bh = item / a.NC, b = bh / a.H, h = bh % a.H;
    const int j0 = c * kC - W + 1;
    mbar_arrive_expect_tx(&bar[0], L::TX);
    for (int j = 0; j < kNS; ++j) {
      tma_load_4d(sm + L::XS + 3072 * j, &tm_k24, &bar[0], 0, h, j0 + 16 * j - a.shift, b);
      tma_load_4d(sm + L::VS + 3072 * j, &tm_v24, &bar[0], 0, h, j0 + 16 * j, b);
    }
    tma_load_4d(sm + L::QS, &tm_q, &bar[0], 0, h, c * kC, b);
  };
  auto gate_in = [&](int item, float& lam, float& beta) {  // step c * 64 + tid
    lam = 0.f;
    beta = 0.f;
    if (tid >= 64 || item >= n_items) return;
    const int c = item % a.NC, bh = item / a.NC, b = bh / a.H, h = bh % a.H;
    const int tg = c * kC + tid;
    if (tg >= a.T) return;
    const size_t gi = ((size_t)b * a.T + tg) * a.H + h;
    lam = a.lam[gi];
    beta = a.beta[gi];
  };
  // loads issued and load phases seen complete (thread 0); products committed
  // (thread 0) and product phases seen complete (every thread)
  int issued = 0, n_loaded = 0, n_commit = 0, n_mma = 0;
  // failure-detection test hook: the first CTA waits, before it loads
  // anything, on a barrier that nothing completes; the bounded wait runs
  // out, the timeout is recorded and the CTA takes no item
  if (a.stall && blockIdx.x == 0 && tid == 0 && !mbar_wait(&bar[2], 0, a.wait_ns)) fail();
  __syncthreads();
  const int first_item = *abort_flag ? n_items : (int)blockIdx.x;
  if (tid == 0 && first_item < n_items) {
    issue_loads(first_item);
    ++issued;
  }
  float lam_n = 0.f, beta_n = 0.f;
  if (first_item < n_items) gate_in(first_item, lam_n, beta_n);
  auto wait_mma = [&]() {
    if (mbar_wait(&bar[1], (uint32_t)(n_mma & 1), a.wait_ns)) ++n_mma;
    else fail();
    tc_fence_after();
  };
  int it = 0;
  for (int item = first_item; item < n_items; item += gridDim.x, ++it) {
    const int c = item % a.NC, bh = item / a.NC, b = bh / a.H, h = bh % a.H;
    const int t0 = c * kC, j0 = t0 - W + 1;
    const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
    const bool step_ok = tid < 64 && t0 + tid < a.T;
    const float lam_c = lam_n, beta = beta_n;
    gate_in(item + gridDim.x, lam_n, beta_n);
    const float ell = step_ok ? clamped_log_decay(lam_c, a.eps_gamma) : 0.f;
    if (mbar_wait(&bar[0], (uint32_t)(it & 1), a.wait_ns)) {
      if (tid == 0) ++n_loaded;
    } else {
      fail();
    }
    if (j0 < a.shift) {  // sub-chunk 0's keys before the sequence: carried key and window ring
      for (int idx = tid; idx < kKP * 64; idx += 256) {
        const int kap = idx >> 6, col = idx & 63, p = j0 + kap;
        if (p < a.shift) {
          *reinterpret_cast<__nv_bfloat16*>(sm + L::XS + sw128(kap, col)) = pair_x(a, b, h, p, col, pos);
          if (p < 0) *reinterpret_cast<__nv_bfloat16*>(sm + L::VS + sw128(kap, col)) = pair_v(a, b, h, p, col, pos);
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    if (__syncthreads_or(*abort_flag)) break;
    tc_fence_after();
    if (tid == 0) {  // [G | (X_s Q^T)] = X_s [X_s ; Q]^T (A rows >= 96 are not read back)
      const uint32_t sX = smem_u32(sm + L::XS);
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tmem, kdesc<128>(sX, ks), kdesc<160>(sX, ks), idesc_bf16(128, 160), ks > 0 ? 1u : 0u);
      umma_commit(&bar[1]);
      ++n_commit;
    }
    // gates meanwhile: key energies and existence of the stacked rows
    if (tid < kNK) {
      const int jb = tid / kKP, kap = tid - kKP * jb, p = j0 + 16 * jb + kap;
      float n = 0.f;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint4 raw = *reinterpret_cast<const uint4*>(sm + L::XS + sw128(tid, 8 * m));
        const __nv_bfloat162* px = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x2 = __bfloat1622float2(px[e]);
          n = fmaf(x2.x, x2.x, n);
          n = fmaf(x2.y, x2.y, n);
        }
      }
      gt[L::G_NRM + tid] = n;
      gt[L::G_EX + tid] = (pos + p >= a.shift && p < a.T && kap < kL + W - 1) ? 1.f : 0.f;
    }
    float g = ell;  // inclusive prefix sum of the log-decay over the chunk
    if (tid < 64) {
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, g, o);
        if (lane >= o) g += n;
      }
      if (lane == 31) gt[L::G_WS + (tid >> 5)] = g;
    }
    __syncthreads();
    if (tid < 64) {  // step t = tid: window statistics and decays
      if ((tid >> 5) == 1) g += gt[L::G_WS];
      const int i = tid >> 4, tau = tid & 15;
      float n = 0.f, e = 0.f;
      for (int r = 0; r < W; ++r) {
        const float ex = gt[L::G_EX + kKP * i + tau + r];
        n += ex;
        e += ex * gt[L::G_NRM + kKP * i + tau + r];
      }
      gt[L::G_C + tid] = (step_ok && n > 0.f) ? beta / (a.eps + e / n) / n : 0.f;
      gt[L::G_GMA + tid] = __expf(ell);
      gt[L::G_G + tid] = g;
      gt[L::G_GAM + tid] = __expf(g);
      if (tau == 15) gt[L::G_END + i] = g;
    }
    wait_mma();
    {  // Gram (columns 0..95) and X_s Q^T (96..159): warp group 0 columns 0..79, group 1 80..159
      const int grp = warp >> 2;
      const int row = 32 * quad + lane;
      if (quad < 3) {
#pragma unroll
        for (int blk = 0; blk < 5; ++blk) {
          const int col0 = 80 * grp + 16 * blk;
          uint32_t r[16];
          tmem_ld16(tmem + lane_off + col0, r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int col = col0 + e;
            if (col < kNK) GS[row * kGS + col] = __uint_as_float(r[e]);
            else XQT[(col - kNK) * kGS + row] = __uint_as_float(r[e]);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    // the recurrences' step operands as aligned rows (in F~ / H's region, free
    // until the recurrences end): per step t = 16 i + tau, the Gram row of key
    // tau + kWMax - 1 and X_i q_t in the rotated order (slot (tau + k) mod kKP
    // at k), and c m of the window rows with gamma
    float* GRr = FH;
    float* XQR = FH + 64 * kKP;
    float* SCg = FH + 128 * kKP;
    for (int u = tid; u < 64 * kKP; u += 256) {
      const int t = u / kKP, k = u - kKP * t, i = t >> 4, tau = t & 15;
      const int col = tau + k >= kKP ? tau + k - kKP : tau + k;
      GRr[u] = GS[(kKP * i + tau + kWMax - 1) * kGS + kKP * i + col];
      XQR[u] = XQT[t * kGS + kKP * i + col];
    }
    float* GBd = NBf + 256;  // after the recurrences' spare rows
    for (int u = tid; u < kNS * kKP * 16; u += 256) {
      const int i = u / (kKP * 16), rem = u - i * kKP * 16, rho = rem >> 4, o = rem & 15, col = rho - 8 + o;
      GBd[u] = (col >= 0 && col < kKP) ? GS[(kKP * i + rho) * kGS + kKP * i + col] : 0.f;
    }
    for (int u = tid; u < 64 * 12; u += 256) {
      const int t = u / 12, r = u - 12 * t, i = t >> 4, tau = t & 15;
      float v = 0.f;
      if (r < W && r < kWMax) v = gt[L::G_C + t] * gt[L::G_EX + kKP * i + tau + r];
      else if (r == kWMax) v = gt[L::G_GMA + t];
      SCg[u] = v;
    }
    __syncthreads();
    if (warp < 4) {  // the recurrences: warp i takes sub-chunk i, F~ and H side by side
      const int i = warp;
      float f[kKP], hc[kKP];
      sub_recurrences(GBd + i * kKP * 16, GRr + kL * i * kKP, XQR, SCg, i, lane, AHf,
                      AHf + 64 * kKP, NBf + i * 64, f, hc);
      named_bar(2, 128);  // every recurrence is done with the step operands in F~ / H's region
      if (lane < kKP) {
#pragma unroll
        for (int k = 0; k < kKP; ++k) {
          FH[i * 576 + k * kKP + lane] = f[k];
          FH[4 * 576 + i * 576 + k * kKP + lane] = hc[k];
        }
      }
    } else {
      // meanwhile, once the previous item's output tiles have left (they
      // overlay these): X~ row (j, kappa) = exp(g_last - g_j) x, and zeroed
      // [Tf | Th] and P^T images
      if (tid == 128) bulk_wait_read0();
      named_bar(1, 128);
      for (int u = tid - 128; u < kNK * 8; u += 128) {
        const int k = u >> 3, dg = u & 7;
        const float sc = __expf(gt[L::G_END + 3] - gt[L::G_END + k / kKP]);
        const uint4 raw = *reinterpret_cast<const uint4*>(sm + L::XS + sw128(k, 8 * dg));
        const __nv_bfloat162* px = reinterpret_cast<const __nv_bfloat162*>(&raw);
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x2 = __bfloat1622float2(px[e]);
          pk[e] = pack_bf16(sc * x2.x, sc * x2.y);
        }
        *reinterpret_cast<uint4*>(sm + L::AT + sw128(k, 8 * dg)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      for (int u = tid - 128; u < 36864 / 16; u += 128)
        *reinterpret_cast<uint4*>(sm + L::TB + 16 * u) = make_uint4(0u, 0u, 0u, 0u);
      for (int u = tid - 128; u < 12288 / 16; u += 128)  // P^T: its nonzero blocks are written below
        *reinterpret_cast<uint4*>(sm + L::AT + 12288 + 16 * u) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    // N_ij = exp(g_i - g_j) F~_i G_ij (j < i) and the nonzero blocks of P^T,
    // in 4 x 4 register tiles (the zero blocks of P^T were written above)
    for (int u = tid; u < 6 * 36 + 6 * 24; u += 256) {
      if (u < 6 * 36) {  // N tile: rows 4 tr.., columns 4 tc.. of pair pi
        const int pi = u / 36, rem = u - 36 * pi, tr = rem / 6, tc = rem - 6 * tr;
        const int i = pi < 1 ? 1 : pi < 3 ? 2 : 3, j = pi - (i * (i - 1)) / 2;
        float acc[4][4] = {};
#pragma unroll
        for (int kk = 0; kk < kKP; kk += 4) {
          float fa[4][4], gb4[4][4];
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const float4 f4 = *reinterpret_cast<const float4*>(FH + i * 576 + (4 * tr + a) * kKP + kk);
            fa[a][0] = f4.x; fa[a][1] = f4.y; fa[a][2] = f4.z; fa[a][3] = f4.w;
            const float4 g4 = *reinterpret_cast<const float4*>(GS + (kKP * i + kk + a) * kGS + kKP * j + 4 * tc);
            gb4[a][0] = g4.x; gb4[a][1] = g4.y; gb4[a][2] = g4.z; gb4[a][3] = g4.w;
          }
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(fa[a][q], gb4[q][b], acc[a][b]);
        }
        const float sc = __expf(gt[L::G_END + i] - gt[L::G_END + j]);
#pragma unroll
        for (int a = 0; a < 4; ++a)
          *reinterpret_cast<float4*>(NBf + pi * 576 + (4 * tr + a) * kKP + 4 * tc) =
              make_float4(sc * acc[a][0], sc * acc[a][1], sc * acc[a][2], sc * acc[a][3]);
      } else {  // P tile: steps 16 i + 4 tt.., keys (j, 4 tk..) of block pair pi
        const int w = u - 6 * 36, pi = w / 24, rem = w - 24 * pi, tt = rem / 6, tk = rem - 6 * tt;
        const int i = pi < 1 ? 1 : pi < 3 ? 2 : 3, j = pi - (i * (i - 1)) / 2;
        const int t0 = kL * i + 4 * tt, k0 = kKP * j + 4 * tk;
        float acc[4][4] = {};  // [step a][key b]: sum_kk a~_t[kk] G[(j, kappa)][(i, kk)]
#pragma unroll
        for (int kk = 0; kk < kKP; kk += 4) {
          float av[4][4], gv[4][4];
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const float4 a4 = *reinterpret_cast<const float4*>(AHf + (t0 + a) * kKP + kk);
            av[a][0] = a4.x; av[a][1] = a4.y; av[a][2] = a4.z; av[a][3] = a4.w;
            const float4 g4 = *reinterpret_cast<const float4*>(GS + (k0 + a) * kGS + kKP * i + kk);
            gv[a][0] = g4.x; gv[a][1] = g4.y; gv[a][2] = g4.z; gv[a][3] = g4.w;
          }
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b)
#pragma unroll
              for (int q = 0; q < 4; ++q) acc[a][b] = fmaf(av[a][q], gv[b][q], acc[a][b]);
        }
        const float gj = gt[L::G_END + j];
        float pv[4][4];  // [key b][step a]
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float e = __expf(gt[L::G_G + t0 + a] - gj);
          const float4 x4 = *reinterpret_cast<const float4*>(XQT + (t0 + a) * kGS + k0);
          pv[0][a] = e * (x4.x - acc[a][0]);
          pv[1][a] = e * (x4.y - acc[a][1]);
          pv[2][a] = e * (x4.z - acc[a][2]);
          pv[3][a] = e * (x4.w - acc[a][3]);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b)  // P^T row (j, kappa), steps t0 .. t0 + 3: one 8-byte store
          *reinterpret_cast<uint2*>(sm + L::AT + 12288 + sw128(k0 + b, t0)) =
              make_uint2(pack_bf16(pv[b][0], pv[b][1]), pack_bf16(pv[b][2], pv[b][3]));
      }
    }
    // the block-diagonal right factor [bd(exp(g_i) F~_i) | bd(H_i)] (bf16
    // image, MN-major B over three atoms; the rest of it was zeroed above)
    auto tb_at = [&](int row, int n) { return sm + L::TB + (n >> 6) * 12288 + sw128(row, n & 63); };
    for (int u = tid; u < kNS * kKP * 6; u += 256) {
      const int i = u / (kKP * 6), rem = u - i * kKP * 6, kap = rem / 6, gsel = rem - 6 * kap;
      const bool hpart = gsel >= 3;
      const int n0 = 8 * (gsel % 3);
      const float* src = FH + (hpart ? 4 * 576 : 0) + i * 576 + kap * kKP + n0;
      const float sc = hpart ? 1.f : __expf(gt[L::G_END + i]);
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pk[e] = pack_bf16(sc * src[2 * e], sc * src[2 * e + 1]);
      *reinterpret_cast<uint4*>(tb_at(kKP * i + kap, (hpart ? kNK : 0) + kKP * i + n0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    __syncthreads();
    // T = (I + N)^{-1}, block lower triangular with identity diagonal blocks:
    // T_{i,i-1} = -N_{i,i-1}, T_20 = -N_20 + N_21 N_10, T_31 = -N_31 + N_32 N_21,
    // then T_30 = -N_30 + N_31 N_10 - N_32 T_20.  bf16 image: MN-major B (rows
    // k, 96 columns over two atoms); T_20 also kept in fp32 (F~ and H are in
    // the image by now, so their scratch is free).
    auto ti_at = [&](int row, int n) { return sm + L::TI + (n >> 6) * 12288 + sw128(row, n & 63); };
    auto nblk = [&](int i, int j) { return NBf + ((i * (i - 1)) / 2 + j) * 576; };
    float* T20 = FH;
    // rows k, columns 8 g .. 8 g + 7 (inside one block), by units of 8
    auto put8 = [&](int k, int n0, const float (&v)[8]) {
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pk[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
      *reinterpret_cast<uint4*>(ti_at(k, n0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    };
    // v = -N_ij[kap][c0..] + A[kap][:] B[:][c0..] (A, B 24 x 24 fp32, row stride kKP)
    auto prod8 = [&](const float* nij, const float* A, const float* Bm, int kap, int c0, float (&v)[8]) {
      const float4 n0 = *reinterpret_cast<const float4*>(nij + kap * kKP + c0);
      const float4 n1 = *reinterpret_cast<const float4*>(nij + kap * kKP + c0 + 4);
      v[0] = -n0.x; v[1] = -n0.y; v[2] = -n0.z; v[3] = -n0.w;
      v[4] = -n1.x; v[5] = -n1.y; v[6] = -n1.z; v[7] = -n1.w;
#pragma unroll
      for (int kk = 0; kk < kKP; kk += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(A + kap * kKP + kk);
        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 b0 = *reinterpret_cast<const float4*>(Bm + (kk + q) * kKP + c0);
          const float4 b1 = *reinterpret_cast<const float4*>(Bm + (kk + q) * kKP + c0 + 4);
          v[0] = fmaf(av[q], b0.x, v[0]); v[1] = fmaf(av[q], b0.y, v[1]);
          v[2] = fmaf(av[q], b0.z, v[2]); v[3] = fmaf(av[q], b0.w, v[3]);
          v[4] = fmaf(av[q], b1.x, v[4]); v[5] = fmaf(av[q], b1.y, v[5]);
          v[6] = fmaf(av[q], b1.z, v[6]); v[7] = fmaf(av[q], b1.w, v[7]);
        }
      }
    };
    // stage A: the two products T_20 and T_31 (144 units), then every other
    // block of the image: identity, -N_{i,i-1}, zero (T_30 below)
    for (int u = tid; u < 2 * kKP * 3 + kNK * 12; u += 256) {
      float v[8];
      if (u < 2 * kKP * 3) {
        const int which = u / (kKP * 3), rem = u - which * kKP * 3, kap = rem / 3, c0 = 8 * (rem - 3 * kap);
        const int bi = which ? 3 : 2, bj = bi - 2;
        prod8(nblk(bi, bj), nblk(bi, bi - 1), nblk(bi - 1, bj), kap, c0, v);
        if (bi == 2) {
          *reinterpret_cast<float4*>(T20 + kap * kKP + c0) = make_float4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<float4*>(T20 + kap * kKP + c0 + 4) = make_float4(v[4], v[5], v[6], v[7]);
        }
        put8(kKP * bi + kap, kKP * bj + c0, v);
      } else {
        const int w = u - 2 * kKP * 3, k = w / 12, g = w - 12 * (w / 12);
        const int bi = k / kKP, kap = k - kKP * bi, n0 = 8 * g, bj = n0 / kKP, c0 = n0 - kKP * bj;
        if (bj == bi - 2 || bj == bi - 3) continue;  // the products (T_30 in stage B)
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
        if (bj == bi) {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = c0 + e == kap ? 1.f : 0.f;
        } else if (bj == bi - 1) {
          const float* nij = nblk(bi, bj) + kap * kKP + c0;
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = -nij[e];
        }
        put8(k, n0, v);
      }
    }
    __syncthreads();
    if (tid < kKP * 3) {  // stage B: T_30 = (-N_30 + N_31 N_10) - N_32 T_20
      const int kap = tid / 3, c0 = 8 * (tid - 3 * kap);
      float v[8], w8[8];
      prod8(nblk(3, 0), nblk(3, 1), nblk(1, 0), kap, c0, v);
      prod8(nblk(3, 0), nblk(3, 2), T20, kap, c0, w8);  // -N_30 + N_32 T_20
      const float* n30 = nblk(3, 0) + kap * kKP + c0;
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = v[e] - (w8[e] + n30[e]);
      put8(3 * kKP + kap, c0, v);
    }
    fence_proxy_async();
    tc_fence_before();
    if (__syncthreads_or(*abort_flag)) break;
    tc_fence_after();
    if (tid == 0) {  // Z = [X~^T ; P] T: A MN-major (two atoms), B MN-major (two atoms, N = 96), K = 96
      const uint32_t sA = smem_u32(sm + L::AT), sT = smem_u32(sm + L::TI);
      for (int ks = 0; ks < kNK / 16; ++ks)
        umma_bf16(tmem, sdesc_mn128_wide(sA + ks * 2048, 12288), sdesc_mn128_wide(sT + ks * 2048, 12288),
                  idesc_bf16(128, kNK, true, true), ks > 0 ? 1u : 0u);
      umma_commit(&bar[1]);
      ++n_commit;
    }
    wait_mma();
    {  // Z rows m as bf16, K-major (K = 96 in two slabs): group 0 columns 0..47, group 1 48..95
      const int grp = warp >> 2, m = 32 * quad + lane;
#pragma unroll
      for (int b16 = 0; b16 < 3; ++b16) {
        const int k0 = 48 * grp + 16 * b16;
        uint32_t r[16];
        tmem_ld16(tmem + lane_off + k0, r);
        tmem_wait_ld();
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {
          const int k = k0 + 8 * h8;
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pk[e] = pack_bf16(__uint_as_float(r[8 * h8 + 2 * e]), __uint_as_float(r[8 * h8 + 2 * e + 1]));
          *reinterpret_cast<uint4*>(sm + L::ZT + (k >> 6) * 16384 + sw128(m, k & 63)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {  // [X~^T ; P] [Tf | Th] = Z [bd | bd]: A K-major, B MN-major (three atoms), K = 96
      const uint32_t sZ = smem_u32(sm + L::ZT), sB = smem_u32(sm + L::TB);
      for (int ks = 0; ks < kNK / 16; ++ks)
        umma_bf16(tmem, kdesc<128>(sZ, ks), sdesc_mn128_wide(sB + ks * 2048, 12288),
                  idesc_bf16(128, 192, false, true), ks > 0 ? 1u : 0u);
      umma_commit(&bar[1]);
      ++n_commit;
    }
    wait_mma();
    {  // rows m: group 0 writes -R_F, group 1 R_H (K-major, K = 96 in two slabs)
      const int grp = warp >> 2, m = 32 * quad + lane;
      const int t = m - 64, ib = t >> 4;
      const float* add = nullptr;
      float asc = 0.f;
      if (m >= 64) {
        add = grp == 0 ? AHf + t * kKP : AHf + 64 * kKP + t * kKP;
        asc = grp == 0 ? gt[L::G_GAM + t] : 1.f;
      }
      uint8_t* tile = sm + (grp == 0 ? L::RF : L::RH);
      const float sg = grp == 0 ? -1.f : 1.f;
#pragma unroll
      for (int blk = 0; blk < 3; ++blk) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + kNK * grp + 32 * blk, r);
        tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int k = 32 * blk + e;
          float x = __uint_as_float(r[e]);
          if (add && k >= kKP * ib && k < kKP * ib + kKP) x = fmaf(asc, add[k - kKP * ib], x);
          v[e] = sg * x;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int k0 = 32 * blk + 8 * q;
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) pk[e] = pack_bf16(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
          *reinterpret_cast<uint4*>(tile + (k0 >> 6) * 16384 + sw128(m, k0 & 63)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && !*abort_flag) {  // [-M ; Q' - Gamma Q] = -R_F X_s, [b ; O0] = R_H V_s
      const uint32_t sF = smem_u32(sm + L::RF), sH = smem_u32(sm + L::RH);
      const uint32_t sX = smem_u32(sm + L::XS), sV = smem_u32(sm + L::VS);
      for (int ks = 0; ks < kNK / 16; ++ks)
        umma_bf16(tmem, kdesc<128>(sF, ks), mndesc(sX, ks), idesc_bf16(128, 64, false, true), ks > 0 ? 1u : 0u);
      for (int ks = 0; ks < kNK / 16; ++ks)
        umma_bf16(tmem + 64, kdesc<128>(sH, ks), mndesc(sV, ks), idesc_bf16(128, 64, false, true), ks > 0 ? 1u : 0u);
      umma_commit(&bar[1]);
      ++n_commit;
    }
    if (!*abort_flag) wait_mma();
    // the query rows the epilogue needs, then the tiles are free for the next item
    const int m = 32 * quad + lane, grp = warp >> 2;
    uint4 qrow[8];
    if (grp == 0 && m >= 64) {
#pragma unroll
      for (int q = 0; q < 8; ++q) qrow[q] = *reinterpret_cast<const uint4*>(sm + L::QS + sw128(m - 64, 8 * q));
    }
    __syncthreads();
    const int next = item + gridDim.x;
    if (tid == 0 && next < n_items && !*abort_flag) {
      issue_loads(next);
      ++issued;
    }
    {
      float d[64];
      tmem_ld64(tmem + lane_off + 64 * grp, d);
      tmem_wait_ld();
      if (grp == 0) {
        if (m >= 64) {
          const float gq = gt[L::G_GAM + m - 64];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const __nv_bfloat162* pq = reinterpret_cast<const __nv_bfloat162*>(&qrow[q]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 q2 = __bfloat1622float2(pq[e]);
              d[8 * q + 2 * e] = fmaf(gq, q2.x, d[8 * q + 2 * e]);
              d[8 * q + 2 * e + 1] = fmaf(gq, q2.y, d[8 * q + 2 * e + 1]);
            }
          }
        }
        store_row64(sm + L::OMQ, m, d);
      } else {
        store_row64(sm + (m < 64 ? L::OB : L::OO), m & 63, d);
      }
      if (tid == 0) reinterpret_cast<float*>(sm + L::OG)[0] = gt[L::G_GAM + 63];
    }
    fence_proxy_async();
    tc_fence_before();
    if (__syncthreads_or(*abort_flag)) break;
    if (tid == 128) {  // the thread that waits for the tiles to leave before they are rewritten
      bulk_store(a.ws_f3 + (size_t)(bh * a.NC + c) * kF3Rec, sm + L::OMQ, (uint32_t)kF3Rec);
      bulk_commit();
    }
  }
  if (tid == 128) bulk_wait0();
  if (tid == 0) {  // loads and a product still in flight complete before the memory goes away
    for (int w = n_loaded; w < issued; ++w) mbar_wait(&bar[0], (uint32_t)(w & 1), a.wait_ns);
    if (n_commit > n_mma) mbar_wait(&bar[1], (uint32_t)(n_mma & 1), a.wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::NCOLS);
  }
}

// ======================================================================
// (b) the chain: acc = [-M ; Q'] S0, S1 = Gamma_last S0 + b + acc_top, O = acc_bottom + O0
// ======================================================================
__global__ void __launch_bounds__(F3ChainSmem::kThreads, 1) f3_chain_kernel(F3Args a) {
  using L = F3ChainSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  constexpr int NST = L::NST, NB = L::NB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* full = bars;              // [NST] record loaded
  uint64_t* empty = bars + NST;       // [NST] chain (64) and outputs (64) done with the record
  uint64_t* mdone = bars + 2 * NST;   // [NB] product of the chunk in TMEM buffer p done
  uint64_t* odone = mdone + NB;       // [NB] outputs read TMEM buffer p (64)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x >> 1, half = blockIdx.x & 1, b = bh / a.H, h = bh % a.H;
  const int c0 = 32 * half;  // this CTA's value columns c0 .. c0 + 31
  const int W = a.W;
  auto stage = [&](int s) { return sm + s * L::STAGE; };
  auto fail = [&]() {
    *abort_flag = 1;
    atomicExch(a.status, kStatusTimeout);
  };
  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 128);
    }
    for (int p = 0; p < NB; ++p) {
      mbar_init(&mdone[p], 1);
      mbar_init(&odone[p], 64);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const bool upstream_failed = *reinterpret_cast<volatile uint32_t*>(a.status) != 0u;
  if (upstream_failed) *abort_flag = 1;
  const int NC = upstream_failed ? 0 : a.NC;
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      int c = 0;
      for (; c < NC; ++c) {
        const int s = c % NST;
        if (c >= NST && !mbar_wait(&empty[s], (uint32_t)(((c - NST) / NST) & 1), a.wait_ns)) { fail(); break; }
        if (*abort_flag) break;
        const uint8_t* src = a.ws_f3 + (size_t)(bh * a.NC + c) * kF3Rec;
        mbar_arrive_expect_tx(&full[s], (uint32_t)kF3Rec);
        bulk_load(stage(s), src, (uint32_t)kF3Rec, &full[s]);
      }
      if (*abort_flag) {  // drain the loads still in flight
        for (int cc = (c > NST ? c - NST : 0); cc < c; ++cc)
          mbar_wait(&full[cc % NST], (uint32_t)((cc / NST) & 1), a.wait_ns);
      }
    }
  } else if (warp < 2) {
    // ------------------------------------------------------------ state chain
    const int r = tid;  // S row; columns c0 .. c0 + 31
    float sreg[32];
#pragma unroll
    for (int n = 0; n < 32; ++n) sreg[n] = 0.f;
    if (a.S_in) {
      const float* src = a.S_in + ((size_t)bh * 64 + r) * 64 + c0;
#pragma unroll
      for (int n = 0; n < 32; n += 4) {
        const float4 v4 = *reinterpret_cast<const float4*>(src + n);
        sreg[n] = v4.x; sreg[n + 1] = v4.y; sreg[n + 2] = v4.z; sreg[n + 3] = v4.w;
      }
    }
    auto store_s = [&](int buf) {  // row r, columns 0..31 of the tile
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pk[e] = pack_bf16(sreg[8 * j + 2 * e], sreg[8 * j + 2 * e + 1]);
        *reinterpret_cast<uint4*>(sm + L::SB + buf * 8192 + sw128(r, 8 * j)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    };
    store_s(0);
    fence_proxy_async();
    named_bar(1, 64);
    for (int c = 0; c < NC; ++c) {
      const int s = c % NST, p = c % NB;
      bool ok = mbar_wait(&full[s], (uint32_t)((c / NST) & 1), a.wait_ns);
      if (ok && tid == 0) {  // the TMEM buffer's previous chunk has been read by the outputs
        ok = c < NB || mbar_wait(&odone[p], (uint32_t)(((c - NB) / NB) & 1), a.wait_ns);
        if (ok) {
          tc_fence_after();
          const uint32_t sA = smem_u32(stage(s) + L::MQ), sS = smem_u32(sm + L::SB + p * 8192);
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16(tmem + 32 * p, kdesc<128>(sA, ks), mndesc(sS, ks), idesc_bf16(128, 32, false, true),
                      ks > 0 ? 1u : 0u);
          umma_commit(&mdone[p]);
        }
      }
      if (!ok) fail();
      // a product that was not issued leaves mdone incomplete: the bounded
      // wait runs out and the barrier below takes every chain thread out
      if (!mbar_wait(&mdone[p], (uint32_t)((c / NB) & 1), a.wait_ns)) fail();
      // the accumulator is read warp by warp (a warp that saw a failure
      // skips it); the barrier at the end of the chunk takes both warps out
      if (!__any_sync(0xffffffffu, *abort_flag != 0)) {
        tc_fence_after();
        uint32_t acc[32];
        tmem_ld32(tmem + lane_off + 32 * p, acc);
        tmem_wait_ld();
        tc_fence_before();
        const uint8_t* st = stage(s);
        const float gl = reinterpret_cast<const float*>(st + L::GO)[0];
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // S1 = Gamma_last S0 + b + (-M S0), row r, this CTA's columns
          const uint4 raw = *reinterpret_cast<const uint4*>(st + L::BO + sw128(r, c0 + 8 * j));
          const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 b2 = __bfloat1622float2(pb[e]);
            const int n = 8 * j + 2 * e;
            sreg[n] = fmaf(gl, sreg[n], b2.x + __uint_as_float(acc[n]));
            sreg[n + 1] = fmaf(gl, sreg[n + 1], b2.y + __uint_as_float(acc[n + 1]));
          }
        }
        mbar_arrive(&empty[s]);
        if (c + 1 < NC) store_s((c + 1) % NB);  // its previous reader (chunk c + 1 - NB) is done
        fence_proxy_async();
      }
      // the next chunk's S0 image is complete before thread 0 issues its product
      if (named_bar_any(1, 64, *abort_flag != 0)) break;
    }
    if (!*abort_flag && a.S_out) {
      float* dst = a.S_out + ((size_t)bh * 64 + r) * 64 + c0;
#pragma unroll
      for (int n = 0; n < 32; n += 4)
        *reinterpret_cast<float4*>(dst + n) = make_float4(sreg[n], sreg[n + 1], sreg[n + 2], sreg[n + 3]);
    }
  } else {
    // ------------------------------------------------------------ outputs (TMEM lanes 64..127)
    const int otid = tid - 64, t = otid;
    for (int c = 0; c < NC; ++c) {
      const int s = c % NST, p = c % NB;
      if (!mbar_wait(&mdone[p], (uint32_t)((c / NB) & 1), a.wait_ns) ||
          !mbar_wait(&full[s], (uint32_t)((c / NST) & 1), a.wait_ns))
        fail();
      if (named_bar_any(2, 64, *abort_flag != 0)) break;
      tc_fence_after();
      uint32_t acc[32];
      tmem_ld32(tmem + lane_off + 32 * p, acc);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&odone[p]);
      const uint8_t* st = stage(s);
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 raw = *reinterpret_cast<const uint4*>(st + L::OO + sw128(t, c0 + 8 * j));
        const __nv_bfloat162* po = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 o2 = __bfloat1622float2(po[e]);
          const int n = 8 * j + 2 * e;
          pk[4 * j + e] = pack_bf16(__uint_as_float(acc[n]) + o2.x, __uint_as_float(acc[n + 1]) + o2.y);
        }
      }
      mbar_arrive(&empty[s]);
      const int tg = c * kC + t;
      if (tg < a.T) {
        uint4* dst = reinterpret_cast<uint4*>(a.o + (((size_t)b * a.T + tg) * a.H + h) * 64 + c0);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      }
    }
    if (half == 0 && !*abort_flag) {  // carry: last key, the last W - 1 pairs, position
      if (a.kprev_out)
        a.kprev_out[(size_t)bh * 64 + otid] = a.k[(((size_t)b * a.T + (a.T - 1)) * a.H + h) * 64 + otid];
      const int Wr = W - 1;
      for (int idx = otid; idx < Wr * 64; idx += 64) {
        const int i = idx >> 6, col = idx & 63;
        const int64_t pp = pos + a.T - Wr + i;  // global pair index
        const int j = (int)(pp - pos);
        const int slot = (int)(((pp % Wr) + Wr) % Wr);
        const bool ok = pp >= a.shift;  // slots of pairs that do not exist hold zeros
        const __nv_bfloat16 z = __float2bfloat16_rn(0.f);
        if (a.winx_out)
          a.winx_out[((size_t)bh * Wr + slot) * 64 + col] = ok ? pair_x(a, b, h, j, col, pos) : z;
        if (a.winv_out)
          a.winv_out[((size_t)bh * Wr + slot) * 64 + col] = ok ? pair_v(a, b, h, j, col, pos) : z;
      }
      if (a.pos_out && otid == 0) a.pos_out[bh] = pos + a.T;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

}  // namespace

bool tc_f3_supported(const FwdArgs& a) {
  if (a.variant != FALCON_3 || a.dtype != FALCON_BF16 || a.chunk != 64 || a.T < 1) return false;
  return a.dk == 64 && a.dv == 64 && a.W >= 2 && a.W <= kWMax;
}

size_t tc_f3_ws_bytes(int B, int T, int H) {
  const size_t NC = (size_t)(T + kC - 1) / kC;
  return 256 + (size_t)B * H * NC * kF3Rec;
}

int launch_tc_f3(const FwdArgs& fa) {
  F3Args ta;
  ta.B = fa.B; ta.T = fa.T; ta.H = fa.H; ta.W = fa.W; ta.NC = (fa.T + kC - 1) / kC;
  ta.shift = fa.shift;
  ta.eps = fa.eps; ta.eps_gamma = fa.eps_gamma;
  ta.beta = fa.beta; ta.lam = fa.lam; ta.pos_in = fa.pos_in;
  ta.kprev_in = reinterpret_cast<const __nv_bfloat16*>(fa.kprev_in);
  ta.winx_in = reinterpret_cast<const __nv_bfloat16*>(fa.winx_in);
  ta.winv_in = reinterpret_cast<const __nv_bfloat16*>(fa.winv_in);
  ta.S_in = fa.S_in;
  ta.k = reinterpret_cast<const __nv_bfloat16*>(fa.k);
  ta.v = reinterpret_cast<const __nv_bfloat16*>(fa.v);
  ta.S_out = fa.S_out;
  ta.kprev_out = reinterpret_cast<__nv_bfloat16*>(fa.kprev_out);
  ta.winx_out = reinterpret_cast<__nv_bfloat16*>(fa.winx_out);
  ta.winv_out = reinterpret_cast<__nv_bfloat16*>(fa.winv_out);
  ta.pos_out = fa.pos_out;
  ta.status = reinterpret_cast<uint32_t*>(fa.ws);
  ta.ws_f3 = reinterpret_cast<uint8_t*>(fa.ws) + 256;
  ta.o = reinterpret_cast<__nv_bfloat16*>(fa.o);
  ta.wait_ns = wait_limit_ns();
  ta.stall = take_test_stall() ? 1 : 0;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, fa.q, fa.B, fa.T, fa.H, 64, 64) || !make_map(&mk, fa.k, fa.B, fa.T, fa.H, 64, kKP) ||
      !make_map(&mv, fa.v, fa.B, fa.T, fa.H, 64, kKP))
    return FALCON_ERR_CUDA;
  {  // per-chunk operators, persistent: one CTA per SM
    auto k = f3_chunk_kernel;
    const size_t smem = F3ChunkSmem::TOTAL;
    if (!set_smem_limit(reinterpret_cast<const void*>(k), smem)) return FALCON_ERR_CUDA;
    const long items = (long)ta.NC * fa.B * fa.H;
    dim3 grid((unsigned)std::min<long>(items, (long)sm_count()));
    record_event(fa, 0);
    if (launch_overlapped(fa, k, grid, dim3(256), smem, mq, mk, mv, ta) != FALCON_OK) return FALCON_ERR_CUDA;
    record_event(fa, 1);
  }
  {  // the chain and the outputs, two CTAs per (b, h) (32 value columns each)
    auto k = f3_chain_kernel;
    const size_t smem = F3ChainSmem::TOTAL;
    if (!set_smem_limit(reinterpret_cast<const void*>(k), smem)) return FALCON_ERR_CUDA;
    if (launch_overlapped(fa, k, dim3(2 * fa.B * fa.H), dim3(F3ChainSmem::kThreads), smem, ta) != FALCON_OK)
      return FALCON_ERR_CUDA;
    record_event(fa, 2);
  }
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace falcon
