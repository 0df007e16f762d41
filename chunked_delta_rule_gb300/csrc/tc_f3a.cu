// Tensor-core chunk forward for Falcon-3A (additive write averaged over a
// window of the last W pairs), bf16 inputs, fp32 state, chunk 64,
// d_k = d_v = 64, 2 <= W <= 16.
//
// The additive write needs no solve [JC Falcon家族六个变体各管一段;
// FW 三种等价形式]: with c_s = eta_s / n_s (eta_s from the window-average key
// energy e_s, n_s the existing pairs in the window of step s, zero when there
// are none), a chunk of steps t0..t0+63 touches the keys x_kappa, values
// v_kappa of the pairs j = t0 - W + 1 + kappa, kappa = 0 .. 62 + W, and
//   M'_{t,kappa} = sum_{s <= t, kappa in window(s)} exp(g_t - g_s) c_s
//                = gamma_t M'_{t-1,kappa} + c_t [t <= kappa <= t + W - 1]
//   O    = diag(Gamma) Q S0 + (Q X^T (.) M') V  = diag(Gamma) Q S0 + O0
//   S1   = Gamma_last S0 + (diag(m) X)^T V      = Gamma_last S0 + b,   m_kappa = M'_{63,kappa}
// (in-chunk cumulative log-decay g, Gamma = exp(g), clamped decay
// [JC 数学上的稳定阀门:正衰减钳制]).  The recurrence for M' only multiplies by
// gamma <= 1, so no decay ratio is ever formed.  The state enters only
// through the scalar decay Gamma_last and the product Q S0, so everything
// else is formed for all chunks at once:
//  (a) f3a_chunk_kernel, persistent over (b, h, chunk) on every SM (four
//      CTAs per SM): TMA of the 80 key rows, 80 value rows and 64 query rows;
//      window statistics, P^T = X Q^T (keys in TMEM lanes), M' by the
//      recurrence along t, P~^T and X~ = diag(m) X in place, then
//      [b ; O0] = [X~ | P~^T]^T V in one product (M = 128, K = 80); b, O0
//      (bf16, 128B-swizzled 64 x 64 tiles) and Gamma leave by bulk copies.
//  (b) f3a_chain_kernel, two CTAs per (b, h), each owning 32 value columns
//      (S's columns evolve independently): S1 = Gamma_last S0 + b on the
//      fp32 state in registers (no product on the chain), and off it
//      O = diag(Gamma) Q S0 + O0 with Q S0 one tcgen05 product per chunk
//      (N = 32), the outputs stored by 32-byte rows; a producer warp streams
//      Q, its half of b and O0 (stored by halves) and the gates ahead; two
//      output warpgroups take alternate chunks.  The chain's only coupling
//      across chunks is the scalar decay, so when one chain per (b, h)
//      would leave SMs idle the chunks split into G groups:
//      f3a_group_kernel sums each group's b with its decays (from a zero
//      state), and the chain CTAs of group g (lighter, two per SM) start
//      from S_in carried through the earlier groups' totals.
// Every wait is bounded; on timeout a kernel records an error in the
// workspace status word and leaves its loop (the chain kernel computes
// nothing when the first kernel recorded one).

#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_util.cuh"

namespace falcon {

using namespace tc;
using namespace tcu;

namespace {

constexpr int kKeys = 80;  // key / value rows per chunk (C + W - 1 <= 79, padded)

struct F3aArgs {
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
  uint8_t* ws_f3a;    // per chunk: b | Gamma | O0 (kF3aChunkWs bytes)
  __nv_bfloat16* o;   // [B, T, H, 64]
  uint64_t wait_ns;   // limit of every bounded wait
  int stall;          // failure-detection test hook: the per-chunk kernel's first CTA waits on
                      // a barrier that nothing completes, and so records a timeout
  // the chain in G groups of CPG chunks (G = 1: one group): group g of (b, h)
  // starts from the state the groups before it leave, gdec[g'] S + gtot[g']
  int G, CPG;
  float* gtot;        // [B H][G][64][64] fp32: a group's state from a zero start
  float* gdec;        // [B H][G]: the product of its chunks' Gamma_last
};

// per chunk in the workspace: b | Gamma (64 fp32) | O0, b and O0 bf16 by
// halves of 32 value columns ([2][64 rows][32], 4 KB each, pieces placed by
// half_off; only the chain's elementwise work reads them, so each chain CTA
// loads its own half)
constexpr size_t kF3aChunkWs = 8192 + 256 + 8192;
constexpr size_t kF3aGam = 8192, kF3aO0 = 8192 + 256;

// Byte offset of the 16-byte piece p (columns 8 p .. 8 p + 7) of row r in
// one half of such a tile: the piece index XOR (r >> 1) & 3 puts eight
// consecutive rows' pieces on different banks.
__device__ __forceinline__ int half_off(int r, int p) { return r * 64 + 16 * (p ^ ((r >> 1) & 3)); }

// a 64-value fp32 row as bf16 into a [2][64][32] half-major tile
__device__ __forceinline__ void store_row_halves(uint8_t* tile, int r, const float* v) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t pk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) pk[e] = pack_bf16(v[8 * j + 2 * e], v[8 * j + 2 * e + 1]);
    *reinterpret_cast<uint4*>(tile + (j >> 2) * 4096 + half_off(r, j & 3)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

struct F3aChunkSmem {
  // X (80 key rows, then X~) | P~^T (80 rows; then O0's staging) | V (80 rows) | Q | gates | b's staging
  static constexpr size_t XO = 0, PO = 10240, VO = 20480, QO = 30720, GO = 38912, BST = 40960;
  static constexpr size_t BAR = BST + 8192 + 256;
  static constexpr size_t MISC = BAR + 32;
  static constexpr size_t TOTAL = MISC + 64 + 1024;
  static constexpr uint32_t TX = 2 * 10240 + 8192;
  // gates (fp32 offsets in GO): key energy, key existence, c, gamma, Gamma, g, warp sums
  static constexpr int G_NRM = 0, G_EX = 80, G_C = 160, G_GMA = 224, G_GAM = 288, G_G = 352, G_WS = 416;
  static_assert(GO + (G_WS + 2) * 4 <= BST, "gates fit");
  // TMEM: P^T (keys in lanes) | [b ; O0]
  static constexpr uint32_t COL_PT = 0, COL_D = 64, NCOLS = 128;
};

template <int NST_, int NB_>
struct F3aChainSmemT {
  // stages in flight: each CTA streams ~25 KB per chunk, so the loads in
  // flight (NST stages) set its bandwidth at the memory latency
  static constexpr int NST = NST_;
  // stage: Q | this CTA's half of b | Gamma | its half of O0
  static constexpr size_t QO = 0, BO = 8192, GO = BO + 4096, OO = GO + 256, STAGE = 17408;
  static constexpr int NB = NB_;                   // S0 tiles and TMEM accumulators in flight
  static constexpr uint32_t NCOLS = NB * 32 <= 128 ? 128 : 256;
  static constexpr size_t SB = NST * STAGE;        // S0 of chunk c in SB + (c % NB) 8192 (MN-major B,
                                                   // this CTA's 32 columns in columns 0..31)
  static constexpr size_t BAR = SB + NB * 8192;
  static constexpr size_t MISC = BAR + 256;
  static constexpr size_t TOTAL = MISC + 16 + 1024;
  static constexpr uint32_t TX = 8192 + 4096 + 256 + 4096;
  static constexpr int kThreads = 384;  // outputs 0..3 and 8..11 (alternate chunks), chain 4..5,
                                        // producer 6, issuer 7
  static_assert(OO + 4096 <= STAGE && STAGE % 1024 == 0, "stage layout");
  static_assert(TOTAL <= 232448, "shared memory budget");
  static_assert((2 * NST + 3 * NB) * 8 <= 256, "barriers");
};
// one chain CTA per SM for (b, h) over all chunks; two per SM for groups of chunks
using F3aChainSmem = F3aChainSmemT<6, 6>;
using F3aChainSmemG = F3aChainSmemT<4, 4>;

// Key (x) and value of local pair j of (b, h): j >= 1 from the sequence,
// j = 0 the carried key with the first value, j < 0 the carried window ring.
__device__ __forceinline__ __nv_bfloat16 pair_x(const F3aArgs& a, int b, int h, int j, int col, int64_t pos) {
  if (j >= a.shift) return a.k[(((size_t)b * a.T + (j - a.shift)) * a.H + h) * 64 + col];
  if (j == 0) return a.kprev_in ? a.kprev_in[((size_t)b * a.H + h) * 64 + col] : __float2bfloat16_rn(0.f);
  if (!a.winx_in || pos + j < a.shift) return __float2bfloat16_rn(0.f);
  const int Wr = a.W - 1;
  return a.winx_in[(((size_t)b * a.H + h) * Wr + ring_slot(pos + j, Wr)) * 64 + col];
}
__device__ __forceinline__ __nv_bfloat16 pair_v(const F3aArgs& a, int b, int h, int j, int col, int64_t pos) {
  if (j >= 0) return a.v[(((size_t)b * a.T + j) * a.H + h) * 64 + col];
  if (!a.winv_in || pos + j < a.shift) return __float2bfloat16_rn(0.f);
  const int Wr = a.W - 1;
  return a.winv_in[(((size_t)b * a.H + h) * Wr + ring_slot(pos + j, Wr)) * 64 + col];
}


// ======================================================================
// (a) per-chunk operands b, O0 and Gamma, every (b, h, chunk) in parallel
// ======================================================================
__global__ void __launch_bounds__(128, 4)
    f3a_chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k80,
                     const __grid_constant__ CUtensorMap tm_v80, F3aArgs a) {
  using L = F3aChunkSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);  // [0] keys and values, [1] products, [2] queries
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
  float* gt = reinterpret_cast<float*>(sm + L::GO);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int W = a.W;
  const int n_items = a.NC * a.B * a.H;  // item = (b, h, chunk), chunk fastest
  // launched overlapping the stream's previous grid: wait for it before any
  // read; then (every CTA of this persistent grid being resident) let the
  // chain kernel launch and wait for this grid in hardware
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the call's status word starts clear (the grid is resident as a whole, so
  // no CTA of it records a timeout a full wait limit before this runs)
  if (blockIdx.x == 0 && tid == 0) atomicExch(a.status, 0u);
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_init(&bar[2], 1);
    mbar_init(&bar[3], 1);  // the test hook's (never completed)
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
  // keys and values of an item (their tiles are free once its second
  // product is done), and its queries (free once P^T is done): thread 0
  auto issue_xv = [&](int item) {
    const int c = item % a.NC, bh = item / a.NC, b = bh / a.H, h = bh % a.H;
    const int j0 = c * kC - W + 1;  // first pair of the chunk's keys
    mbar_arrive_expect_tx(&bar[0], 2 * 10240);
    tma_load_4d(sm + L::XO, &tm_k80, &bar[0], 0, h, j0 - a.shift, b);
    tma_load_4d(sm + L::VO, &tm_v80, &bar[0], 0, h, j0, b);
  };
  auto issue_q = [&](int item) {
    const int c = item % a.NC, bh = item / a.NC, b = bh / a.H, h = bh % a.H;
    mbar_arrive_expect_tx(&bar[2], 8192);
    tma_load_4d(sm + L::QO, &tm_q, &bar[2], 0, h, c * kC, b);
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
  int issued = 0, issued_q = 0, n_mma = 0;  // loads issued, product groups committed (thread 0)
  // failure-detection test hook: the first CTA waits, before it loads
  // anything, on a barrier that nothing completes; the bounded wait runs
  // out, the timeout is recorded and the CTA takes no item
  if (a.stall && blockIdx.x == 0 && tid == 0 && !mbar_wait(&bar[3], 0, a.wait_ns)) {
    *abort_flag = 1;
    atomicExch(a.status, kStatusTimeout);
  }
  __syncthreads();
  const int first_item = *abort_flag ? n_items : (int)blockIdx.x;
  if (tid == 0 && first_item < n_items) {
    issue_xv(first_item);
    issue_q(first_item);
    ++issued;
    ++issued_q;
  }
  float lam_n = 0.f, beta_n = 0.f;
  if (first_item < n_items) gate_in(first_item, lam_n, beta_n);
  int it = 0;
  for (int item = first_item; item < n_items; item += gridDim.x, ++it) {
    const int c = item % a.NC, bh = item / a.NC, b = bh / a.H, h = bh % a.H;
    const int t0 = c * kC, j0 = t0 - W + 1;
    const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
    const bool step_ok = tid < 64 && t0 + tid < a.T;
    const float lam_c = lam_n, beta = beta_n;
    gate_in(item + gridDim.x, lam_n, beta_n);  // the next item's gate inputs, in flight meanwhile
    const float ell = step_ok ? clamped_log_decay(lam_c, a.eps_gamma) : 0.f;
    if (!mbar_wait(&bar[0], (uint32_t)(it & 1), a.wait_ns)) {
      *abort_flag = 1;
      atomicExch(a.status, kStatusTimeout);
    }
    if (j0 < 1) {  // keys before the sequence: carried key and window ring
      for (int idx = tid; idx < W * 64; idx += 128) {
        const int kap = idx >> 6, col = idx & 63, j = j0 + kap;
        if (j < a.shift) {
          *reinterpret_cast<__nv_bfloat16*>(sm + L::XO + sw128(kap, col)) = pair_x(a, b, h, j, col, pos);
          if (j < 0)
            *reinterpret_cast<__nv_bfloat16*>(sm + L::VO + sw128(kap, col)) = pair_v(a, b, h, j, col, pos);
        }
      }
    }
    __syncthreads();
    if (tid < kKeys) {  // key energy and existence of pair j0 + kappa
      const int j = j0 + tid;
      float n = 0.f;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint4 raw = *reinterpret_cast<const uint4*>(sm + L::XO + sw128(tid, 8 * m));
        const __nv_bfloat162* px = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x2 = __bfloat1622float2(px[e]);
          n = fmaf(x2.x, x2.x, n);
          n = fmaf(x2.y, x2.y, n);
        }
      }
      gt[L::G_NRM + tid] = n;
      gt[L::G_EX + tid] = (pos + j >= a.shift && j < a.T) ? 1.f : 0.f;
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
      float n = 0.f, e = 0.f;
      for (int q = 0; q < W; ++q) {
        const float ex = gt[L::G_EX + tid + q];
        n += ex;
        e += ex * gt[L::G_NRM + tid + q];
      }
      const float cs = (step_ok && n > 0.f) ? beta / (a.eps + e / n) / n : 0.f;
      gt[L::G_C + tid] = cs;
      gt[L::G_GMA + tid] = __expf(ell);
      gt[L::G_GAM + tid] = __expf(g);
      gt[L::G_G + tid] = g;
    }
    if (tid == 0) bulk_wait_read0();  // the previous item's tiles have left P~^T's and b's staging
    fence_proxy_async();
    tc_fence_before();
    if (__syncthreads_or(*abort_flag)) break;
    tc_fence_after();
    if (tid == 0 && !mbar_wait(&bar[2], (uint32_t)(it & 1), a.wait_ns)) {
      *abort_flag = 1;
      atomicExch(a.status, kStatusTimeout);
    }
    if (tid == 0 && !*abort_flag) {  // P^T = X Q^T over 128 A rows (rows >= 80 are not read back)
      const uint32_t sX = smem_u32(sm + L::XO), sQ = smem_u32(sm + L::QO);
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tmem + L::COL_PT, kdesc<128>(sX, ks), kdesc<64>(sQ, ks), idesc_bf16(128, 64),
                  ks > 0 ? 1u : 0u);
      umma_commit(&bar[1]);
      ++n_mma;
    }
    if (!mbar_wait(&bar[1], 0u, a.wait_ns)) {  // each item commits bar[1] twice: parities 0, 1
      *abort_flag = 1;
      atomicExch(a.status, kStatusTimeout);
    }
    tc_fence_after();
    if (tid == 0 && item + (int)gridDim.x < n_items && !*abort_flag) {  // the query tile is read
      issue_q(item + gridDim.x);
      ++issued_q;
    }
    if (quad < 3) {  // keys kappa = 32 quad + lane < 80
      const int kap = 32 * quad + lane;
      const float* cs = gt + L::G_C;
      const float* gm = gt + L::G_GMA;
      const bool kex = kap < kKeys && gt[L::G_EX + kap] != 0.f;  // a pair that does not exist writes nothing
      float mcur = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {  // 32 columns t of P^T at a time, M' carried along t
        uint32_t pr[32];
        tmem_ld32(tmem + lane_off + L::COL_PT + 32 * hh, pr);
        tmem_wait_ld();
        float pv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int t = 32 * hh + i;
          const bool in_win = kex && t <= kap && kap <= t + W - 1;
          mcur = fmaf(gm[t], mcur, in_win ? cs[t] : 0.f);
          pv[i] = __uint_as_float(pr[i]) * mcur;
        }
        if (kap < kKeys) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) pk[e] = pack_bf16(pv[8 * j + 2 * e], pv[8 * j + 2 * e + 1]);
            *reinterpret_cast<uint4*>(sm + L::PO + sw128(kap, 32 * hh + 8 * j)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
      if (kap < kKeys) {
        // X~ row kappa = m_kappa x_kappa in place
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          uint4* ptr = reinterpret_cast<uint4*>(sm + L::XO + sw128(kap, 8 * m));
          const uint4 in = *ptr;
          const __nv_bfloat162* px = reinterpret_cast<const __nv_bfloat162*>(&in);
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x2 = __bfloat1622float2(px[e]);
            pk[e] = pack_bf16(x2.x * mcur, x2.y * mcur);
          }
          *ptr = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && !*abort_flag) {  // [b ; O0] = [X~ | P~^T]^T V, A MN-major over two 80-row atoms, K = 80
      const uint32_t sA = smem_u32(sm + L::XO), sV = smem_u32(sm + L::VO);
      for (int ks = 0; ks < kKeys / 16; ++ks)
        umma_bf16(tmem + L::COL_D, sdesc_mn128_wide(sA + ks * 2048, 10240), mndesc(sV, ks),
                  idesc_bf16(128, 64, true, true), ks > 0 ? 1u : 0u);
      umma_commit(&bar[1]);
      ++n_mma;
    }
    if (!*abort_flag && !mbar_wait(&bar[1], 1u, a.wait_ns)) {
      *abort_flag = 1;
      atomicExch(a.status, kStatusTimeout);
    }
    tc_fence_after();
    // the tiles are read: the next item's loads go out while this one leaves
    const int next = item + gridDim.x;
    if (tid == 0 && next < n_items && !*abort_flag) {
      issue_xv(next);
      ++issued;
    }
    {  // rows 0..63: b -> its staging; rows 64..127: O0 -> P~^T's region
      const int row = 32 * quad + lane;
      float dv[64];
      tmem_ld64(tmem + lane_off + L::COL_D, dv);
      tmem_wait_ld();
      store_row_halves(quad < 2 ? sm + L::BST : sm + L::PO, row & 63, dv);
      if (tid < 64) reinterpret_cast<float*>(sm + L::BST + 8192)[tid] = gt[L::G_GAM + tid];
    }
    fence_proxy_async();
    tc_fence_before();
    if (__syncthreads_or(*abort_flag)) break;
    if (tid == 0) {
      uint8_t* dst = a.ws_f3a + (size_t)(bh * a.NC + c) * kF3aChunkWs;
      bulk_store(dst, sm + L::BST, 8192 + 256);
      bulk_store(dst + 8192 + 256, sm + L::PO, 8192);
      bulk_commit();
    }
  }
  if (tid == 0) {
    bulk_wait0();
    if (issued > it) mbar_wait(&bar[0], (uint32_t)(it & 1), a.wait_ns);  // loads still in flight
    if (issued_q > it) mbar_wait(&bar[2], (uint32_t)(it & 1), a.wait_ns);
    // a product still in flight (abort between issue and wait) completes before TMEM is freed
    if (n_mma > 0) mbar_wait(&bar[1], (uint32_t)((n_mma - 1) & 1), a.wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::NCOLS);
  }
}

// ======================================================================
// (b) the chain: S1 = Gamma_last S0 + b, O = diag(Gamma) Q S0 + O0
// ======================================================================
template <int NST_, int NB_, int MINB>
__global__ void __launch_bounds__(384, MINB)
    f3a_chain_kernel(const __grid_constant__ CUtensorMap tm_q, F3aArgs a) {
  using L = F3aChainSmemT<NST_, NB_>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  constexpr int NST = L::NST;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* full = bars;              // [NST] stage loaded
  uint64_t* empty = bars + NST;       // [NST] chain (64) and outputs (128) done with the stage
  constexpr int NB = L::NB;
  uint64_t* sready = bars + 2 * NST;  // [NB] S0 of the chunk in SB buffer p written (64)
  uint64_t* mdone = sready + NB;      // [NB] Q S0 into TMEM buffer p done
  uint64_t* odone = mdone + NB;       // [NB] outputs read TMEM buffer p (128)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // CTA (g, b, h, half): group g of the chunks of (b, h), 32 value columns
  const int BH = a.B * a.H;
  const int bh = (blockIdx.x >> 1) % BH, g = (blockIdx.x >> 1) / BH, half = blockIdx.x & 1;
  const int b = bh / a.H, h = bh % a.H;
  const int c0 = 32 * half;  // this CTA's value columns c0 .. c0 + 31
  const bool last_group = g == a.G - 1;
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
      mbar_init(&empty[i], 64 + 128);
    }
    for (int p = 0; p < NB; ++p) {
      mbar_init(&sready[p], 64);
      mbar_init(&mdone[p], 1);
      mbar_init(&odone[p], 128);
    }
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
  // the per-chunk kernel has completed (and its writes are visible) past
  // this wait; a timeout it recorded leaves its tiles incomplete: then no
  // chunk is computed and no carry is written
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const bool upstream_failed = *reinterpret_cast<volatile uint32_t*>(a.status) != 0u;
  if (upstream_failed) *abort_flag = 1;
  // this group's chunks cbase .. cbase + NC - 1 (local index c below)
  const int cbase = g * a.CPG;
  const int NC = upstream_failed ? 0 : max(0, min(a.NC - cbase, a.CPG));
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;

  if (warp == 6) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      int c = 0;
      for (; c < NC; ++c) {
        const int s = c % NST;
        if (c >= NST && !mbar_wait(&empty[s], (uint32_t)(((c - NST) / NST) & 1), a.wait_ns)) { fail(); break; }
        if (*abort_flag) break;
        uint8_t* st = stage(s);
        const uint8_t* src = a.ws_f3a + (size_t)(bh * a.NC + cbase + c) * kF3aChunkWs;
        mbar_arrive_expect_tx(&full[s], L::TX);
        tma_load_4d(st + L::QO, &tm_q, &full[s], 0, h, (cbase + c) * kC, b);
        bulk_load(st + L::BO, src + half * 4096, 4096, &full[s]);
        bulk_load(st + L::GO, src + kF3aGam, 256, &full[s]);
        bulk_load(st + L::OO, src + kF3aO0 + half * 4096, 4096, &full[s]);
      }
      if (*abort_flag) {  // drain the loads still in flight
        for (int cc = (c > NST ? c - NST : 0); cc < c; ++cc)
          mbar_wait(&full[cc % NST], (uint32_t)((cc / NST) & 1), a.wait_ns);
      }
    }
  } else if (warp == 7) {
    // ------------------------------------------------------------ product issuer
    if (lane == 0) {
      int n = 0;
      for (int c = 0; c < NC; ++c) {
        const int s = c % NST, p = c % NB;
        bool ok = mbar_wait(&full[s], (uint32_t)((c / NST) & 1), a.wait_ns) &&
                  mbar_wait(&sready[p], (uint32_t)((c / NB) & 1), a.wait_ns) &&
                  (c < NB || mbar_wait(&odone[p], (uint32_t)(((c - NB) / NB) & 1), a.wait_ns));
        if (!ok || *abort_flag) { fail(); break; }
        tc_fence_after();
        const uint32_t sQ = smem_u32(stage(s) + L::QO), sS = smem_u32(sm + L::SB + p * 8192);
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem + 32 * p, kdesc<64>(sQ, ks), mndesc(sS, ks), idesc_bf16(64, 32, false, true),
                    ks > 0 ? 1u : 0u);
        umma_commit(&mdone[p]);
        ++n;
      }
      if (n > 0) mbar_wait(&mdone[(n - 1) % NB], (uint32_t)(((n - 1) / NB) & 1), a.wait_ns);  // TMEM quiet
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ state chain
    const int r = 32 * (warp - 4) + lane;  // S row; columns c0 .. c0 + 31
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
    for (int gg = 0; gg < g; ++gg) {  // through the groups before this one
      const float dg = a.gdec[(size_t)bh * a.G + gg];
      const float* tg = a.gtot + (((size_t)bh * a.G + gg) * 64 + r) * 64 + c0;
#pragma unroll
      for (int n = 0; n < 32; n += 4) {
        const float4 v4 = *reinterpret_cast<const float4*>(tg + n);
        sreg[n] = fmaf(dg, sreg[n], v4.x); sreg[n + 1] = fmaf(dg, sreg[n + 1], v4.y);
        sreg[n + 2] = fmaf(dg, sreg[n + 2], v4.z); sreg[n + 3] = fmaf(dg, sreg[n + 3], v4.w);
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
    if (NC > 0) {
      store_s(0);
      fence_proxy_async();
      mbar_arrive(&sready[0]);
    }
    for (int c = 0; c < NC; ++c) {
      const int s = c % NST;
      if (!mbar_wait(&full[s], (uint32_t)((c / NST) & 1), a.wait_ns)) fail();
      // each chain thread leaves on its own after a failure: nothing in this
      // loop waits on the other chain threads (every wait is bounded)
      if (*abort_flag) break;
      const uint8_t* st = stage(s);
      const float gl = reinterpret_cast<const float*>(st + L::GO)[63];
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // S1 = Gamma_last S0 + b, row r, this CTA's columns
        const uint4 raw = *reinterpret_cast<const uint4*>(st + L::BO + half_off(r, j));
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 b2 = __bfloat1622float2(pb[e]);
          sreg[8 * j + 2 * e] = fmaf(gl, sreg[8 * j + 2 * e], b2.x);
          sreg[8 * j + 2 * e + 1] = fmaf(gl, sreg[8 * j + 2 * e + 1], b2.y);
        }
      }
      mbar_arrive(&empty[s]);
      if (c + 1 < NC) {  // the next chunk's S0 into its buffer, once the product that read it last is done
        const int pn = (c + 1) % NB;
        if (c + 1 >= NB && !mbar_wait(&mdone[pn], (uint32_t)(((c + 1 - NB) / NB) & 1), a.wait_ns)) fail();
        store_s(pn);
        fence_proxy_async();
        mbar_arrive(&sready[pn]);
      }
    }
    if (!*abort_flag && a.S_out && last_group) {
      float* dst = a.S_out + ((size_t)bh * 64 + r) * 64 + c0;
#pragma unroll
      for (int n = 0; n < 32; n += 4)
        *reinterpret_cast<float4*>(dst + n) = make_float4(sreg[n], sreg[n + 1], sreg[n + 2], sreg[n + 3]);
    }
  } else {
    // ------------------------------------------------------------ outputs
    // M = 64 accumulator (N = 32): row t = 16 quad + lane % 16 in lanes 0..15
    // of the warp's quadrant; the half-warps read columns 0..15 and 16..31.
    // Group og (warps 0..3, then 8..11) takes the chunks c with c % 2 == og.
    const int og = warp >= 8 ? 1 : 0, quad = warp & 3, otid = tid - (og ? 256 : 0);
    const int obar = 2 + og;
    const int t = 16 * quad + (lane & 15), hf = lane >> 4;
    const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
    for (int c = og; c < NC; c += 2) {
      const int s = c % NST, p = c % NB;
      if (!mbar_wait(&mdone[p], (uint32_t)((c / NB) & 1), a.wait_ns)) fail();
      tc_fence_after();
      if (named_bar_any(obar, 128, *abort_flag != 0)) break;
      uint32_t acc[16];
      tmem_ld16x2_16(tmem + lane_off + 32 * p, acc);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&odone[p]);
      const uint8_t* st = stage(s);
      const float gq = reinterpret_cast<const float*>(st + L::GO)[t];
      const int col = c0 + 16 * hf;  // this thread's 16 value columns
      uint4 o0[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) o0[j] = *reinterpret_cast<const uint4*>(st + L::OO + half_off(t, 2 * hf + j));
      mbar_arrive(&empty[s]);
      uint32_t pk[8];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const __nv_bfloat162* po = reinterpret_cast<const __nv_bfloat162*>(&o0[j]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 b2 = __bfloat1622float2(po[e]);
          const int n = 8 * j + 2 * e;
          pk[4 * j + e] = pack_bf16(fmaf(gq, __uint_as_float(acc[n]), b2.x), fmaf(gq, __uint_as_float(acc[n + 1]), b2.y));
        }
      }
      const int tg = (cbase + c) * kC + t;
      if (tg < a.T) {
        uint4* dst = reinterpret_cast<uint4*>(a.o + (((size_t)b * a.T + tg) * a.H + h) * 64 + col);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
    if (half == 0 && og == 0 && last_group && !*abort_flag) {  // carry: last key, the last W - 1 pairs, position
      if (a.kprev_out && otid < 64)
        a.kprev_out[(size_t)bh * 64 + otid] = a.k[(((size_t)b * a.T + (a.T - 1)) * a.H + h) * 64 + otid];
      const int Wr = W - 1;
      for (int idx = otid; idx < Wr * 64; idx += 128) {
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
    tmem_dealloc(tmem, L::NCOLS);
  }
}

// Group totals of the chain (every group but the last; G >= 2): from a zero
// state, T = Gamma_last T + b over the group's chunks, and D = the product of
// their Gamma_last.  Eight parts of 64 threads take an eighth of the chunks
// each (thread r: row r, all 64 columns; the next chunk's row is loaded
// before the current one is added), then the parts combine in order,
// T = (..(T0 D1 + T1) D2 + ..) D7 + T7.
constexpr int kGParts = 8;
constexpr int kGLd = 68;  // padded row of the part totals (rows on different banks)
__global__ void __launch_bounds__(64 * kGParts) f3a_group_kernel(F3aArgs a) {
  extern __shared__ float gsm[];  // [kGParts][64][kGLd] part totals, then [kGParts] part decays
  const int tid = threadIdx.x, r = tid & 63, part = tid >> 6;
  const int g = blockIdx.x % (a.G - 1), bh = blockIdx.x / (a.G - 1);
  const int cs = g * a.CPG, qp = (a.CPG + kGParts - 1) / kGParts;
  const int p0 = cs + part * qp, p1 = min(cs + min(a.CPG, (part + 1) * qp), a.NC);
  float t[64];
#pragma unroll
  for (int n = 0; n < 64; ++n) t[n] = 0.f;
  float d = 1.f;
  const bool failed = *reinterpret_cast<volatile uint32_t*>(a.status) != 0u;
  auto rec = [&](int c) { return a.ws_f3a + (size_t)(bh * a.NC + c) * kF3aChunkWs; };
  uint4 nx[8];
  float gn = 1.f;
  auto fetch = [&](int c) {  // row r of b and Gamma_last of chunk c
#pragma unroll
    for (int j = 0; j < 8; ++j) nx[j] = *reinterpret_cast<const uint4*>(rec(c) + (j >> 2) * 4096 + half_off(r, j & 3));
    gn = reinterpret_cast<const float*>(rec(c) + kF3aGam)[63];
  };
  if (!failed && p0 < p1) fetch(p0);
  for (int c = p0; c < p1 && !failed; ++c) {
    uint4 cur[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) cur[j] = nx[j];
    const float gl = gn;
    if (c + 1 < p1) fetch(c + 1);
    d *= gl;
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // eight 16-byte pieces of row r (four of each half)
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&cur[j]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 b2 = __bfloat1622float2(pb[e]);
        t[8 * j + 2 * e] = fmaf(gl, t[8 * j + 2 * e], b2.x);
        t[8 * j + 2 * e + 1] = fmaf(gl, t[8 * j + 2 * e + 1], b2.y);
      }
    }
  }
  float* mine = gsm + ((size_t)part * 64 + r) * kGLd;
#pragma unroll
  for (int n = 0; n < 64; n += 4) *reinterpret_cast<float4*>(mine + n) = make_float4(t[n], t[n + 1], t[n + 2], t[n + 3]);
  if (r == 0) gsm[kGParts * 64 * kGLd + part] = d;
  __syncthreads();
  const float* dp = gsm + kGParts * 64 * kGLd;
  constexpr int kCols = 64 / kGParts;
  const int col0 = kCols * part;  // this thread combines row r, columns col0 .. col0 + kCols - 1
  float* dst = a.gtot + (((size_t)bh * a.G + g) * 64 + r) * 64 + col0;
#pragma unroll
  for (int n = 0; n < kCols; ++n) {
    float v = gsm[(size_t)r * kGLd + col0 + n];
#pragma unroll
    for (int q = 1; q < kGParts; ++q) v = fmaf(dp[q], v, gsm[((size_t)q * 64 + r) * kGLd + col0 + n]);
    dst[n] = v;
  }
  if (tid == 0) {
    float dd = 1.f;
#pragma unroll
    for (int q = 0; q < kGParts; ++q) dd *= dp[q];
    a.gdec[(size_t)bh * a.G + g] = dd;
  }
}

}  // namespace

bool tc_f3a_supported(const FwdArgs& a) {
  if (a.variant != FALCON_3A || a.dtype != FALCON_BF16 || a.chunk != 64 || a.T < 1) return false;
  return a.dk == 64 && a.dv == 64 && a.W >= 2 && a.W <= 16;
}

// the chain's group totals and decays: at most kMaxG groups
constexpr int kMaxG = 16;
static size_t f3a_records_bytes(int B, int T, int H) {
  return 256 + (size_t)B * H * ((size_t)(T + kC - 1) / kC) * kF3aChunkWs;
}

// Groups of the chain: one, unless the chain CTAs of all (b, h) leave SMs
// idle; then as many as two light CTAs per SM allow (at least 8 chunks each).
static int f3a_groups(int BH, int NC) {
  if (NC < 16) return 1;
  return std::max(1, std::min({(2 * sm_count()) / (2 * BH), NC / 8, kMaxG}));
}

int tc_f3a_launches(const FwdArgs& a) {
  return f3a_groups(a.B * a.H, (a.T + kC - 1) / kC) > 1 ? 3 : 2;
}

size_t tc_f3a_ws_bytes(int B, int T, int H) {
  return f3a_records_bytes(B, T, H) + (size_t)B * H * kMaxG * (64 * 64 + 1) * 4;
}

int launch_tc_f3a(const FwdArgs& fa) {
  F3aArgs ta;
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
  ta.ws_f3a = reinterpret_cast<uint8_t*>(fa.ws) + 256;
  ta.o = reinterpret_cast<__nv_bfloat16*>(fa.o);
  ta.wait_ns = wait_limit_ns();
  ta.stall = take_test_stall() ? 1 : 0;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, fa.q, fa.B, fa.T, fa.H, 64, 64) || !make_map(&mk, fa.k, fa.B, fa.T, fa.H, 64, kKeys) ||
      !make_map(&mv, fa.v, fa.B, fa.T, fa.H, 64, kKeys))
    return FALCON_ERR_CUDA;
  {  // per-chunk operands, persistent: four CTAs per SM (TMEM and shared memory both allow four)
    auto k = f3a_chunk_kernel;
    const size_t smem = F3aChunkSmem::TOTAL;
    if (!set_smem_limit(reinterpret_cast<const void*>(k), smem)) return FALCON_ERR_CUDA;
    const long items = (long)ta.NC * fa.B * fa.H;
    dim3 grid((unsigned)std::min<long>(items, 4L * sm_count()));
    record_event(fa, 0);
    if (launch_overlapped(fa, k, grid, dim3(128), smem, mq, mk, mv, ta) != FALCON_OK) return FALCON_ERR_CUDA;
    record_event(fa, 1);
  }
  // The chain and the outputs, two CTAs per (b, h) (32 value columns each).
  // Long sequences with few heads leave SMs idle on one chain per (b, h):
  // then the chunks split into G groups whose CTAs (lighter, two per SM) run
  // side by side, each starting from the state that a pass over the earlier
  // groups' totals gives it.
  const int BH = fa.B * fa.H;
  const int G = f3a_groups(BH, ta.NC);
  ta.G = G;
  ta.CPG = (ta.NC + G - 1) / G;
  uint8_t* gbase = reinterpret_cast<uint8_t*>(fa.ws) + f3a_records_bytes(fa.B, fa.T, fa.H);
  ta.gtot = reinterpret_cast<float*>(gbase);
  ta.gdec = reinterpret_cast<float*>(gbase + (size_t)BH * kMaxG * 64 * 64 * 4);
  if (G > 1) {
    auto k = f3a_group_kernel;
    const size_t smem = (kGParts * 64 * kGLd + kGParts) * 4;
    if (!set_smem_limit(reinterpret_cast<const void*>(k), smem)) return FALCON_ERR_CUDA;
    k<<<dim3(BH * (G - 1)), dim3(64 * kGParts), smem, fa.stream>>>(ta);
    if (cudaGetLastError() != cudaSuccess) return FALCON_ERR_CUDA;
    record_event(fa, 2);
    auto kc = f3a_chain_kernel<F3aChainSmemG::NST, F3aChainSmemG::NB, 2>;
    const size_t smc = F3aChainSmemG::TOTAL;
    if (!set_smem_limit(reinterpret_cast<const void*>(kc), smc)) return FALCON_ERR_CUDA;
    if (launch_overlapped(fa, kc, dim3(2 * BH * G), dim3(F3aChainSmemG::kThreads), smc, mq, ta) != FALCON_OK)
      return FALCON_ERR_CUDA;
  } else {
    auto k = f3a_chain_kernel<F3aChainSmem::NST, F3aChainSmem::NB, 1>;
    const size_t smem = F3aChainSmem::TOTAL;
    if (!set_smem_limit(reinterpret_cast<const void*>(k), smem)) return FALCON_ERR_CUDA;
    if (launch_overlapped(fa, k, dim3(2 * BH), dim3(F3aChainSmem::kThreads), smem, mq, ta) != FALCON_OK)
      return FALCON_ERR_CUDA;
  }
  record_event(fa, G > 1 ? 3 : 2);
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace falcon
