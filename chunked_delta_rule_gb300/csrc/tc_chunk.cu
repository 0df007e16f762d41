// Tensor-core chunk forward for sm_103a (Falcon-1 / Falcon-1A, bf16 inputs,
// fp32 state, chunk 64, d_k = d_v in {64, 128}).
//
// Chunked form [FW 三种等价形式, 图4C; JC 三种视角看同一个更新]: per chunk
// of C = 64 steps with state S0 at its start, in-chunk cumulative log-decay
// g_r (clamped decay [JC 数学上的稳定阀门:正衰减钳制]) and Gamma_r = exp(g_r),
//   A_ri = eta_r exp(g_r - g_i) x_r.x_i (i < r),     T = (I + A)^{-1}
//   [W | U] = T [diag(eta Gamma) X | diag(eta) V]            (WY representation)
//   Delta   = U - W S0                  (Falcon-1A: Delta = diag(eta) V)
//   O       = diag(Gamma) Q S0 + (Q X^T (.) [exp(g_r - g_i)]_{i<=r}) Delta
//   S1      = Gamma_last S0 + (diag(exp(g_last - g)) X)^T Delta
//
// Two kernels per call:
//  (a) per-chunk kernel, fully parallel: TMA loads the shifted keys and the
//      values, one tcgen05 MMA forms the Gram matrix in TMEM,
//      the gates (clamped log-decay, its in-chunk prefix sum, NLMS step) are
//      formed from lambda, beta and the key norms, and T = (I + A)^{-1}
//      is found by blocked forward substitution: 16x16 diagonal blocks in
//      registers, off-diagonal blocks merged with warp-level tf32 MMAs in
//      shared memory (tc_wyu_kernel, one chunk per CTA, persistent).  A
//      second MMA forms [U ; W] = [T diag(eta) ; T diag(eta Gamma)] [V | X]
//      and both leave as bf16 images of 128B-swizzled tiles, with the gate
//      rows Gamma, exp(g_last - g), g and exp(g - g_block).
//  (b) sequential kernel, one CTA per (b, h) (per value slice for d = 128),
//      the fp32 state in registers: TMA and bulk copies bring the chunk's
//      operands while earlier chunks compute; every contraction is a
//      tcgen05 MMA with the accumulator in TMEM; the output tile leaves by
//      TMA store.  d = 64 runs in transition form (tc_fwd_chain_kernel:
//      three front warpgroups form each chunk's state-independent operands
//      [-M ; Q'] and [b ; P~ U] = [X~^T ; P~] [W | U], so the state chain is
//      one product per chunk); d = 128 (tc_fwd_kernel) has one warp that
//      issues every load and product for eight epilogue warps.
//  The input prologue (phi = L2 normalisation of q and k, gates from logits)
//  runs inside the d = 64 kernels when asked for.
// The second kernel is launched to overlap the first one's tail (programmatic
// dependent launch) and waits for it in hardware before reading its images.
// Every mbarrier wait is bounded; on timeout a kernel records an error in the
// workspace status word and leaves its chunk loop.

#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_util.cuh"

namespace falcon {

using namespace tc;
using namespace tcu;

namespace {

constexpr int kGateF = 256;      // fp32 gate slot per chunk in the workspace
constexpr int kLD = 68;          // fp32 row stride of the solve buffers (bank spread)
constexpr int kYL = 24;          // row stride of the 16x16 scratch blocks

struct TcArgs {
  int B, T, H, NC, NV;
  int shift;          // pair t uses key t - shift (1 prefix alignment, 0 same-step)
  float eps, eps_gamma;
  const float* beta;
  const float* lam;
  const int64_t* pos_in;
  const __nv_bfloat16* kprev_in;
  const float* S_in;
  const __nv_bfloat16* k;
  float* S_out;
  __nv_bfloat16* kprev_out;
  int64_t* pos_out;
  uint8_t* ws_T;      // [B*H*NC][2 d_k 128]: bf16 128B-swizzled images, W slabs | U slabs
  float* ws_g;        // [B*H*NC][kGateF]: Gamma, exp(g_last - g), g, exp(g - g_block)
  uint32_t* status;   // workspace status word
  int pro;            // prologue flags applied inside the d = 64 kernels (falcon_prologue_t)
  uint64_t wait_ns;   // limit of every bounded wait
  int stall;          // failure-detection test hook: the per-chunk kernel's first CTA waits on
                      // a barrier that nothing completes (the wait runs out, a timeout is recorded)
  // packed sequences (d = 64 only): sequence b's length is cu[b+1] - cu[b];
  // the per-chunk kernel takes the items of item_map[0 .. *item_count), the
  // sequential kernel stops after the sequence's last chunk (NULL: dense)
  const int32_t* cu;
  const int32_t* item_map;
  const int32_t* item_count;
  int packed;         // with cu: q, k, v, o are the packed [total, H, d] rows themselves, sequence b
                      // at rows cu[b] .. cu[b+1] - 1 (else a padded [B, T] batch)
  __nv_bfloat16* o;   // the output rows (packed: stored row by row, up to each sequence's end)
};

// ======================================================================
// (a) per-chunk gates and WY products, one chunk per CTA (persistent):
// besides the gates it leaves W = T diag(eta Gamma) X and U = T diag(eta) V
// (Falcon-1) or U = diag(eta) V (Falcon-1A) in the workspace as bf16 images
// of 128B-swizzled 64 x 64 tiles (d_k / 64 slabs each), so that the
// sequential kernel needs no per-chunk products of its own beyond P.
// ======================================================================
template <int DK>
struct WyuSmem {
  static constexpr size_t VX = 0;                  // V slabs | X slabs: [V | X] as one MN-major B of 2 DK / 64 atoms
  static constexpr size_t TI = 2 * DK * 128;       // [T diag(eta) ; T diag(eta Gamma)], 128 K-major rows;
                                                   // the solve's 16x16 scratch blocks before that; the
                                                   // W | U images (2 DK 128 bytes) after the product
  static constexpr size_t AT = TI + 16384;         // A, then T in place: [64][kLD] fp32
  static constexpr size_t E = AT + 64 * kLD * 4;   // g, eta, column factors, Gamma, beta (64 each)
  static constexpr size_t WS = E + 5 * 64 * 4;     // warp sums
  static constexpr size_t BAR = WS + 16;           // 3 mbarriers (the third only for the stall hook)
  static constexpr size_t MISC = BAR + 32;         // tmem addr, abort flag
  static constexpr size_t TOTAL = MISC + 16 + 1024;
};

template <bool SOLVE, int DK, bool MAP = false>  // MAP: the items of packed sequences' chunk map
__global__ void __launch_bounds__(128, DK == 64 ? 4 : 2) tc_wyu_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                                    const __grid_constant__ CUtensorMap tm_v,
                                                                    TcArgs a) {
  using L = WyuSmem<DK>;
  constexpr int kSl = DK / 64;                  // 64-column slabs of keys and values
  constexpr uint32_t kImg = 2 * DK * 128;       // W | U images of one chunk
  static_assert(kImg <= 16384 + 64 * kLD * 4, "the images are staged over the T image and A / T");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* Vs = sm + L::VX;
  uint8_t* Xs = sm + L::VX + DK * 128;
  uint8_t* TI = sm + L::TI;
  float* T = reinterpret_cast<float*>(sm + L::AT);  // A, overwritten by T block by block
  float* gs = reinterpret_cast<float*>(sm + L::E);
  float* es = gs + 64;
  float* cfs = gs + 128;
  float* gms = gs + 192;
  float* bs = gs + 256;
  float* wsum = reinterpret_cast<float*>(sm + L::WS);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // launched overlapping the stream's previous grid: wait for it before any
  // read; then (every CTA of this persistent grid being resident) let the
  // sequential kernel launch and wait for this grid in hardware
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // work item = (b, h, chunk) as (b H + h) NC + chunk, chunk fastest: all of
  // them, or for packed sequences the listed ones (those holding tokens)
  const int n_items = MAP ? *a.item_count : a.NC * a.B * a.H;
  auto real_item = [&](int item) { return MAP ? a.item_map[item] : item; };
  // the call's status word starts clear (the grid is resident as a whole,
  // so no CTA of it records a timeout a full wait limit before this runs)
  if (blockIdx.x == 0 && tid == 0) atomicExch(a.status, 0u);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_init(&bar[2], 1);
    fence_mbar_init();
  }
  if (SOLVE && warp == 0) {
    tmem_alloc(tmem_slot, 2 * DK);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = SOLVE ? *tmem_slot : 0u;
  // failure-detection test hook: the first CTA waits, before it loads
  // anything, on a barrier that nothing completes; the bounded wait runs
  // out, the timeout is recorded and the CTA takes no item
  if (a.stall && blockIdx.x == 0 && tid == 0 && !mbar_wait(&bar[2], 0, a.wait_ns)) {
    *abort_flag = 1;
    atomicExch(a.status, kStatusTimeout);
  }
  __syncthreads();
  const int first_item = *abort_flag ? n_items : (int)blockIdx.x;
  // the tiles of an item are fetched while the previous item finishes (TMA
  // into the tile buffers once the products that read them are done); its
  // gate inputs two items ahead, into registers (raw loads: their values are
  // first used two items later, so the loads stay in flight meanwhile)
  int issued = 0;  // tile loads issued (thread 0); item `it` waits for the it-th
  auto fetch_tiles = [&](int item) {
    const int ri = real_item(item);
    const int chunk = ri % a.NC, bh = ri / a.NC, b = bh / a.H, h = bh % a.H, t0 = chunk * kC;
    if (tid == 0) {
      // packed rows: sequence b from row cu[b] of one [total, H, d] batch row
      const int r0 = (MAP && a.packed) ? a.cu[b] + t0 : t0, bb = (MAP && a.packed) ? 0 : b;
      ++issued;
      mbar_arrive_expect_tx(&bar[0], kImg);
      for (int k = 0; k < kSl; ++k) {
        tma_load_4d(Vs + k * 8192, &tm_v, &bar[0], 64 * k, h, r0, bb);
        tma_load_4d(Xs + k * 8192, &tm_k, &bar[0], 64 * k, h, r0 - a.shift, bb);
      }
    }
  };
  auto fetch_gates = [&](int item, float& lam_r, float& beta_r, int64_t& pos_r) {
    lam_r = 0.f;
    beta_r = 0.f;
    pos_r = 0;
    if (item >= n_items) return;
    const int ri = real_item(item);
    const int chunk = ri % a.NC, bh = ri / a.NC, b = bh / a.H, h = bh % a.H, t0 = chunk * kC;
    const int t = t0 + tid;
    // a step past the sequence's end neither writes nor decays (packed rows:
    // those are the next sequence's)
    const int len = MAP ? a.cu[b + 1] - a.cu[b] : a.T;
    const bool step_ok = tid < 64 && t < len;
    const size_t grow = (MAP && a.packed) ? (size_t)a.cu[b] + (step_ok ? t : 0) : (size_t)b * a.T + (step_ok ? t : 0);
    const size_t gi = grow * a.H + h;
    lam_r = a.lam[gi];
    beta_r = a.beta[gi];
    pos_r = a.pos_in ? a.pos_in[bh] : 0;
  };
  constexpr int kIss = 96;  // issues the products and the image stores (warp 3 computes no key norms)
  float lam_n = 0.f, beta_n = 0.f, lam_nn = 0.f, beta_nn = 0.f;
  int64_t pos_n = 0, pos_nn = 0;
  if (first_item < n_items) {
    fetch_tiles(first_item);
    fetch_gates(first_item, lam_n, beta_n, pos_n);
    fetch_gates(first_item + gridDim.x, lam_nn, beta_nn, pos_nn);
  }
  int it = 0;
  for (int item = first_item; item < n_items; item += gridDim.x, ++it) {
  const int ri = real_item(item);
  const int chunk = ri % a.NC, bh = ri / a.NC;
  const int next = item + gridDim.x;
  const int t_row = chunk * kC + tid;
  const int len_b = MAP ? a.cu[bh / a.H + 1] - a.cu[bh / a.H] : a.T;
  const bool step_ok = tid < 64 && t_row < len_b;
  // the clamped decay and the step size, from gate logits when the prologue asks
  const float ell = step_ok ? logf(gate_gamma(lam_n, a.eps_gamma, a.pro)) : 0.f;
  const float beta = (step_ok && pos_n + t_row >= a.shift) ? gate_beta(beta_n, a.pro) : 0.f;
  lam_n = lam_nn;
  beta_n = beta_nn;
  pos_n = pos_nn;
  fetch_gates(item + 2 * gridDim.x, lam_nn, beta_nn, pos_nn);
  {  // gates: row tid <-> step chunk * 64 + tid
    float g = ell;  // inclusive prefix sum over the chunk
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float n = __shfl_up_sync(0xffffffffu, g, o);
      if (lane >= o) g += n;
    }
    if (lane == 31) wsum[warp] = g;
    __syncthreads();
    if (warp == 1) g += wsum[0];
    if (tid < 64) {
      gs[tid] = g;
      bs[tid] = beta;
    }
  }
  if (!mbar_wait(&bar[0], (uint32_t)(it & 1), a.wait_ns)) {
    *abort_flag = 1;
    atomicExch(a.status, kStatusTimeout);
  }
  const bool carried = chunk == 0 && a.kprev_in && a.shift;  // x_0 = the carried key
  if (carried && tid < DK)
    *reinterpret_cast<__nv_bfloat16*>(Xs + (tid >> 6) * 8192 + sw128(0, tid & 63)) = a.kprev_in[(size_t)bh * DK + tid];
  if (MAP && a.packed && chunk == 0 && a.shift && !a.kprev_in && tid < DK)  // not the previous sequence's key
    *reinterpret_cast<__nv_bfloat16*>(Xs + (tid >> 6) * 8192 + sw128(0, tid & 63)) = __float2bfloat16_rn(0.f);
  if constexpr (DK == 64) {  // the prologue is fused into the d = 64 path only
    // phi(k) = k / max(|k|, 1e-12) per key row, in place (the carried key is
    // a feature already)
    if ((a.pro & FALCON_PROLOGUE_L2NORM_QK) && tid < 64 && !(carried && tid == 0)) {
      uint4 raw[DK / 8];
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < DK / 8; ++j) {
        raw[j] = *reinterpret_cast<const uint4*>(Xs + (j >> 3) * 8192 + sw128(tid, 8 * (j & 7)));
        const __nv_bfloat162* px = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(px[e]);
          ss = fmaf(x.x, x.x, ss);
          ss = fmaf(x.y, x.y, ss);
        }
      }
      const float sc = 1.f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
      for (int j = 0; j < DK / 8; ++j) {
        const __nv_bfloat162* px = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(px[e]);
          pk[e] = pack_bf16(x.x * sc, x.y * sc);
        }
        *reinterpret_cast<uint4*>(Xs + (j >> 3) * 8192 + sw128(tid, 8 * (j & 7))) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
  }
  fence_proxy_async();
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  const size_t ci = (size_t)bh * a.NC + chunk;
  uint8_t* Wo = a.ws_T + ci * kImg;  // W slabs, then the U slabs DK 128 bytes further
  float* go = a.ws_g + ci * kGateF;
  if (SOLVE && !aborted && tid == kIss) {  // Gram matrix X X^T (M = 64: row r in lane 32 (r / 16) + r % 16)
    tc_fence_after();
    mma_chain(tmem, Xs, 64, Xs, 64, DK, idesc_bf16(64, 64), false);
    umma_commit(&bar[1]);
  }
  // NLMS step from the key energy, and the decay factors of each row
  if (tid < 64) {
    float n4[4] = {0.f, 0.f, 0.f, 0.f};  // four short chains
#pragma unroll
    for (int j = 0; j < DK / 8; ++j) {
      const uint4 raw = *reinterpret_cast<const uint4*>(Xs + (j >> 3) * 8192 + sw128(tid, 8 * (j & 7)));
      const __nv_bfloat162* px = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(px[e]);
        n4[e] = fmaf(x.x, x.x, n4[e]);
        n4[e] = fmaf(x.y, x.y, n4[e]);
      }
    }
    const float n = (n4[0] + n4[1]) + (n4[2] + n4[3]);
    const float eta = bs[tid] != 0.f ? bs[tid] / (a.eps + n) : 0.f;
    const float g = gs[tid];
    es[tid] = eta;
    cfs[tid] = __expf(gs[tid | 15] - g);  // exp(g_end(J) - g_r), J the row's 16-block
    gms[tid] = __expf(g);
    if (!aborted) {  // gates of the sequential kernel
      go[tid] = gms[tid];
      go[64 + tid] = __expf(gs[63] - g);
      go[128 + tid] = g;
      go[192 + tid] = __expf(g - gs[tid & ~15]);  // decay from the 16-block start
    }
  }
  if (tid == kIss) bulk_wait_read0();  // the previous item's image store has read its staging
  __syncthreads();

  if (!SOLVE) {  // additive write: U = diag(eta) V
    if (!aborted) {
#pragma unroll
      for (int k = 0; k < 4 * kSl; ++k) {
        const int idx = tid + 128 * k;
        const uint4 in = *reinterpret_cast<const uint4*>(Vs + idx * 16);
        const __nv_bfloat162* pin = reinterpret_cast<const __nv_bfloat162*>(&in);
        const float fr = es[(idx & 511) >> 3];
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(pin[e]);
          pk[e] = pack_bf16(x.x * fr, x.y * fr);
        }
        *reinterpret_cast<uint4*>(Wo + DK * 128 + idx * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    __syncthreads();  // the tiles are read
    if (__syncthreads_or(*abort_flag)) break;
    if (next < n_items) fetch_tiles(next);
    continue;
  }

  if (!aborted && !mbar_wait(&bar[1], 0, a.wait_ns)) {
    *abort_flag = 1;
    atomicExch(a.status, kStatusTimeout);
  }
  tc_fence_after();
  const int rl = 16 * warp + (lane & 15);  // this lane's Gram row
  const int hf = lane >> 4;                // and its half of the columns
  float grow[32];
  {
    uint32_t r32[32];
    tmem_ld16x2_32(tmem + ((uint32_t)(warp * 32) << 16), r32);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) grow[i] = __uint_as_float(r32[i]);
  }
  tc_fence_before();
  {  // A_ri = eta_r exp(g_r - g_i) G_ri (i < r), the decay factored per 16-block
    const float eta = es[rl], g = gs[rl], cfr = cfs[rl];
    const bool ratio_ok = cfr > 1e-30f;  // inside the row's block exp(g_r - g_i) = cf_i / cf_r
    const float inv = ratio_ok ? __fdividef(eta, cfr) : 0.f;
    float* Arow = T + rl * kLD;
    const int I = rl >> 4;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int J = 2 * hf + jj;
      const float* gr = grow + 16 * jj;  // columns 16 J .. 16 J + 15
      float av[16];
      if (J < I) {
        const float rf = eta * __expf(g - gs[16 * J + 15]);
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 c4 = *reinterpret_cast<const float4*>(cfs + 16 * J + i);
          av[i] = rf * c4.x * gr[i];
          av[i + 1] = rf * c4.y * gr[i + 1];
          av[i + 2] = rf * c4.z * gr[i + 2];
          av[i + 3] = rf * c4.w * gr[i + 3];
        }
      } else if (J == I) {
        if (ratio_ok) {
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 c4 = *reinterpret_cast<const float4*>(cfs + 16 * J + i);
            const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              av[i + e] = (16 * J + i + e < rl) ? inv * cc[e] * gr[i + e] : 0.f;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            av[i] = (16 * J + i < rl) ? eta * __expf(g - gs[16 * J + i]) * gr[i] : 0.f;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) av[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4*>(Arow + 16 * J + i) = make_float4(av[i], av[i + 1], av[i + 2], av[i + 3]);
    }
  }
  __syncthreads();

  // ---- T = (I + A)^{-1} in place; the 16x16 scratch blocks live in the
  // (not yet written) T image region
  float* Ysc = reinterpret_cast<float*>(TI);             // [2 warps][16 * kYL]
  float* Yc = reinterpret_cast<float*>(TI + 4096);       // [I-2][J] blocks, 4 x 16 * kYL
  const int w2 = warp & 1;
  if (warp < 2) {  // 16x16 diagonal blocks, one column per lane, forward substitution
    const int I = 2 * w2 + (lane >> 4), l = lane & 15;
    float tv[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float s = (r == l) ? 1.f : 0.f;
#pragma unroll
      for (int i = 0; i < r; ++i) s -= T[(16 * I + r) * kLD + 16 * I + i] * tv[i];
      tv[r] = s;
    }
    __syncwarp();  // every lane of the block has read its A rows
#pragma unroll
    for (int r = 0; r < 16; ++r) T[(16 * I + r) * kLD + 16 * I + l] = tv[r];
  }
  __syncthreads();
  if (warp < 2) {  // T_10 = -T_11 A_10 T_00 and T_32 = -T_33 A_32 T_22 (A_IJ replaced by T_IJ)
    const int I = w2 == 0 ? 1 : 3, J = I - 1;
    float acc[2][4] = {};
    warp_mm16(acc, T + 16 * I * kLD + 16 * J, kLD, T + 16 * J * kLD + 16 * J, kLD, lane);
    float* ys = Ysc + warp * 16 * kYL;
    warp_store16(ys, kYL, acc, 1.f, lane);
    __syncwarp();
    float acc2[2][4] = {};
    warp_mm16(acc2, T + 16 * I * kLD + 16 * I, kLD, ys, kYL, lane);
    warp_store16(T + 16 * I * kLD + 16 * J, kLD, acc2, -1.f, lane);
  }
  __syncthreads();
  {  // Y = A[32:64, 0:32] T[0:32, 0:32]: block (I, J) = (2 + warp / 2, warp % 2)
    const int I = 2 + (warp >> 1), J = warp & 1;
    float acc[2][4] = {};
    if (J == 0) {
      warp_mm16(acc, T + 16 * I * kLD, kLD, T, kLD, lane);
      warp_mm16(acc, T + 16 * I * kLD + 16, kLD, T + 16 * kLD, kLD, lane);
    } else {
      warp_mm16(acc, T + 16 * I * kLD + 16, kLD, T + 16 * kLD + 16, kLD, lane);
    }
    warp_store16(Yc + (2 * (I - 2) + J) * 16 * kYL, kYL, acc, 1.f, lane);
  }
  __syncthreads();
  {  // T[I][J] = -sum_{K=2..I} T[I][K] Y[K-2][J], block (I, J) = (2 + warp / 2, warp % 2)
    const int I = 2 + (warp >> 1), J = warp & 1;
    float acc[2][4] = {};
    for (int K = 2; K <= I; ++K)
      warp_mm16(acc, T + 16 * I * kLD + 16 * K, kLD, Yc + (2 * (K - 2) + J) * 16 * kYL, kYL, lane);
    warp_store16(T + 16 * I * kLD + 16 * J, kLD, acc, -1.f, lane);
  }
  __syncthreads();
  // ---- [T diag(eta) ; T diag(eta Gamma)] as one 128-row K-major bf16 operand
  {
    const int j = tid & 7;  // this thread's 8 columns are the same in every pass
    float eu[8], ew[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      eu[e] = es[8 * j + e];
      ew[e] = eu[e] * gms[8 * j + e];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int R = (tid >> 3) + 16 * k;
      const float4 lo4 = *reinterpret_cast<const float4*>(T + R * kLD + 8 * j);
      const float4 hi4 = *reinterpret_cast<const float4*>(T + R * kLD + 8 * j + 4);
      const float v[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
      uint32_t pw[4], pu[4];  // T's strict upper triangle holds exact zeros (A's did)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pu[e] = pack_bf16(v[2 * e] * eu[2 * e], v[2 * e + 1] * eu[2 * e + 1]);
        pw[e] = pack_bf16(v[2 * e] * ew[2 * e], v[2 * e + 1] * ew[2 * e + 1]);
      }
      const int off = R * 128 + 16 * (j ^ (R & 7));
      *reinterpret_cast<uint4*>(TI + off) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
      *reinterpret_cast<uint4*>(TI + 8192 + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  if (!aborted && tid == kIss) {  // [U . ; . W] = [T diag(eta) ; T diag(eta Gamma)] [V | X]
    tc_fence_after();
    const uint32_t sT = smem_u32(TI), sV = smem_u32(Vs);
    for (int ks = 0; ks < 4; ++ks)
      umma_bf16(tmem, sdesc_k128(sT + ks * 32), sdesc_mn128_wide(sV + ks * 2048, 8192),
                idesc_bf16(128, 2 * DK, false, true), ks > 0 ? 1u : 0u);
    umma_commit(&bar[1]);
  }
  if (!aborted && !mbar_wait(&bar[1], 1, a.wait_ns)) {
    *abort_flag = 1;
    atomicExch(a.status, kStatusTimeout);
  }
  tc_fence_after();
  if (next < n_items && !*abort_flag) fetch_tiles(next);  // the tiles are read
  {  // rows 0..63: U (columns 0..DK-1); rows 64..127: W (columns DK..2 DK-1),
     // staged from the T image buffer on (the product that read it and T is
     // done) in the workspace layout, then stored by one bulk copy
    const int r = (32 * warp + lane) & 63;
#pragma unroll 1
    for (int sl = 0; sl < kSl; ++sl) {
      float rv[64];
      tmem_ld64(tmem + ((uint32_t)(warp * 32) << 16) + (warp < 2 ? 0 : DK) + 64 * sl, rv);
      tmem_wait_ld();
      uint8_t* dst = TI + (warp < 2 ? DK * 128 : 0) + sl * 8192;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pk[e] = pack_bf16(rv[8 * j + 2 * e], rv[8 * j + 2 * e + 1]);
        *reinterpret_cast<uint4*>(dst + sw128(r, 8 * j)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
  }
  fence_proxy_async();
  tc_fence_before();
  if (__syncthreads_or(*abort_flag)) break;
  if (tid == kIss) {
    bulk_store(Wo, TI, kImg);
    bulk_commit();
  }
  }  // items
  if (tid == kIss) bulk_wait0();  // the last images are written
  if (tid == 0 && issued > it) mbar_wait(&bar[0], (uint32_t)(it & 1), a.wait_ns);  // a load still in flight
  tc_fence_before();
  __syncthreads();
  if (SOLVE && warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * DK);
  }
}

// ======================================================================
// (b) sequential state propagation and chunk outputs
// ======================================================================
template <int DK, int NV, bool SOLVE>
struct FwdSmem {
  static constexpr int kKS = DK / 64;                 // 64-column slabs of the d_k contractions
  static constexpr size_t XSZ = DK * 128, QSZ = DK * 128, VSZ = NV * 128;
  static constexpr size_t WSZ = SOLVE ? DK * 128 : 0, GSZ = 1024;  // W rows (K-major [64][DK]); 4 gate rows
  static constexpr size_t STAGE = XSZ + QSZ + VSZ + WSZ + GSZ;     // X | Q | U slice | W | gates
  static constexpr size_t ST0 = 0;
  static constexpr size_t PM = 2 * STAGE;              // decay-masked Q X^T, K-major rows
  static constexpr size_t SB = PM + 8192;              // S rows, MN-major [DK][NV]
  static constexpr size_t DL = SB + DK * 128;          // Delta rows (MN-major B)
  static constexpr size_t DD = DL + (SOLVE ? VSZ : 0); // diag(exp(g_last - g)) Delta rows
  static constexpr size_t OST = DD + VSZ;              // output staging [64][NV]
  static constexpr size_t SMALL = OST + NV * 128;      // gamma, dec, g, eta (4 x 64 fp32)
  static constexpr size_t BAR = SMALL + 4 * 64 * 4;    // full[2], mma
  static constexpr size_t MISC = BAR + 32;
  static constexpr size_t TOTAL = MISC + 16 + 1024;
  // TMEM columns: P and later P~ Delta share one block; X~^T Delta (DK rows as
  // DK / 64 blocks of 64), W S0 and Q S0 one block each
  static constexpr uint32_t COL_P = 0, COL_W = 64, COL_D1 = COL_W + DK, COL_OA = COL_D1 + NV,
                            COL_P2 = COL_OA + NV, NCOL = COL_P2 + 64;
  // P (then P~ Delta) of chunk c in buffer c % 2: the next chunk's P is
  // issued while this chunk's epilogues run
  __host__ __device__ static constexpr uint32_t col_p(int c) { return (c & 1) ? COL_P2 : COL_P; }
  static_assert(NCOL <= 512, "TMEM budget");
  static_assert(NV == 64, "value slice of 64 channels");
};

template <int DK, int NV, bool SOLVE>
__global__ void __launch_bounds__(288, 1)
    tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_o, TcArgs a) {
  using L = FwdSmem<DK, NV, SOLVE>;
  constexpr uint32_t kImg = 2 * DK * 128;  // W | U images of a chunk in the workspace
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* Pm = sm + L::PM;
  uint8_t* SB = sm + L::SB;
  uint8_t* DD = sm + L::DD;
  uint8_t* Ost = sm + L::OST;
  float* Gam = reinterpret_cast<float*>(sm + L::SMALL);
  float* dec = Gam + 64;
  float* gl = dec + 64;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* mbar = full + 2;   // D1 (then the second product group) done
  uint64_t* mbar_p = full + 3; // P done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x, split = blockIdx.y;
  const int b = bh / a.H, h = bh % a.H;
  const int c0 = split * NV;  // first value channel of this CTA
  auto stage = [&](int s) { return sm + L::ST0 + s * L::STAGE; };
  auto Xst = [&](int s) { return stage(s); };
  auto Qst = [&](int s) { return stage(s) + L::XSZ; };
  auto Ust = [&](int s) { return stage(s) + L::XSZ + L::QSZ; };
  auto Wst = [&](int s) { return stage(s) + L::XSZ + L::QSZ + L::VSZ; };
  auto Gst = [&](int s) {
    return reinterpret_cast<float*>(stage(s) + L::XSZ + L::QSZ + L::VSZ + L::WSZ);
  };

  auto issue_stage = [&](int c, int s) {
    const uint32_t bytes = (uint32_t)(L::XSZ + L::QSZ + L::VSZ + L::WSZ + L::GSZ);
    mbar_arrive_expect_tx(&full[s], bytes);
    for (int k = 0; k < L::kKS; ++k) {
      tma_load_4d(Xst(s) + k * 8192, &tm_k, &full[s], 64 * k, h, c * kC - a.shift, b);
      tma_load_4d(Qst(s) + k * 8192, &tm_q, &full[s], 64 * k, h, c * kC, b);
    }
    const size_t ci = (size_t)bh * a.NC + c;
    const uint8_t* img = a.ws_T + ci * kImg;  // W slabs | U slabs
    bulk_load(Ust(s), img + DK * 128 + (c0 / 64) * 8192, (uint32_t)L::VSZ, &full[s]);
    if (SOLVE) bulk_load(Wst(s), img, (uint32_t)L::WSZ, &full[s]);
    bulk_load(Gst(s), a.ws_g + ci * kGateF, (uint32_t)L::GSZ, &full[s]);
  };

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(mbar, 1);
    mbar_init(mbar_p, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the per-chunk kernel has completed (and its writes are visible) past
  // this wait; a timeout it recorded leaves its images incomplete: then no
  // chunk is computed and no carry is written
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const bool upstream_failed = *reinterpret_cast<volatile uint32_t*>(a.status) != 0u;
  if (upstream_failed) *abort_flag = 1;
  const int NC = upstream_failed ? 0 : a.NC;
  // warp 8, lane 0 (tid 256) issues every load and product; warps 0..7 do
  // the epilogues and hold the state
  const bool issuer = tid == 256;
  int issued[2] = {0, 0};  // loads issued per stage (the issuer's bookkeeping)
  if (issuer && NC > 0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the per-chunk kernel's images and gates
    asm volatile("fence.proxy.async.global;" ::: "memory");
    issue_stage(0, 0);
    issued[0] = 1;
  }

  // Thread roles on the M = 64 accumulators (P, W S0, Q S0, P~ Delta): row
  // r = 16 * quadrant + lane % 16 lives in lanes 0..15 of each TMEM quadrant;
  // the half-warps read its columns 0..31 and 32..63 (hf = lane / 16), so
  // every thread owns half a row.  Warps 0..3 form P~ and write the outputs,
  // warps 4..7 form Delta.
  static_assert(DK == 128 && NV == 64, "d_k = 128, 64-channel value slices");
  const int quad = warp & 3;
  const int hf = lane >> 4;
  const int r64 = 16 * quad + (lane & 15);
  const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
  const bool lo = warp < 4, hi = warp >= 4 && warp < 8;
  // The state update D2 is an M = 128 product (S row r in TMEM lane r):
  // warps w and w + 4 share quadrant w % 4, rows 32 (w % 4) + lane, columns
  // 0..31 and 32..63 of them; sreg holds those 32 values of S.
  const int s_row = 32 * quad + lane;
  const int s_c0 = (warp >= 4) ? 32 : 0;
  // 32 fp32 values as bf16 into columns col0 .. col0 + 31 of a swizzled row
  auto store_32 = [&](uint8_t* tile, int row, int col0, const float* v) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pk[e] = pack_bf16(v[8 * j + 2 * e], v[8 * j + 2 * e + 1]);
      *reinterpret_cast<uint4*>(tile + sw128(row, col0 + 8 * j)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  };
  auto store_half = [&](uint8_t* tile, int row, const float* v) { store_32(tile, row, 32 * hf, v); };
  auto ld_half = [&](uint32_t col, float* v) {  // this thread's row, its 32 columns from col
    uint32_t r32[32];
    tmem_ld16x2_32(tmem + lane_off + col, r32);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r32[i]);
  };

  float sreg[32];
#pragma unroll
  for (int n = 0; n < 32; ++n) sreg[n] = 0.f;
  if (a.S_in && warp < 8) {
    const size_t dv = (size_t)gridDim.y * NV;
    const float* src = a.S_in + ((size_t)bh * DK + s_row) * dv + c0 + s_c0;
#pragma unroll
    for (int n = 0; n < 32; ++n) sreg[n] = src[n];
  }
  if (warp < 8) store_32(SB, s_row, s_c0, sreg);
  fence_proxy_async();
  __syncthreads();

  const uint32_t sP = smem_u32(Pm), sS = smem_u32(SB), sDD = smem_u32(DD);
  uint32_t mph = 0, pph = 0;
  int n_pc = 0, n_mc = 0;  // the issuer's commits on mbar_p and mbar
  for (int c = 0; c < NC; ++c) {
    const int s = c & 1;
    const int t0 = c * kC;
    if (issuer && c + 1 < NC) {
      issue_stage(c + 1, s ^ 1);
      ++issued[s ^ 1];
    }
    if (!mbar_wait(&full[s], (c >> 1) & 1, a.wait_ns)) {
      *abort_flag = 1;
      atomicExch(a.status, kStatusTimeout);
    }
    if (c == 0 && a.kprev_in && a.shift) {  // x_0 = carried key
      for (int i = tid; i < DK; i += 288)
        *reinterpret_cast<__nv_bfloat16*>(Xst(0) + (i >> 6) * 8192 + sw128(0, i & 63)) =
            a.kprev_in[(size_t)bh * DK + i];
    }
    if (tid < 64) {  // Gamma, exp(g_last - g), g of the chunk's rows
      const float* G = Gst(s);
      Gam[tid] = G[tid];
      dec[tid] = G[64 + tid];
      gl[tid] = G[128 + tid];
    }
    if (__syncthreads_or(*abort_flag)) break;
    const float gam_last = Gam[63];
    // Delta rows: U - W S0 (Falcon-1, formed below) or U itself (Falcon-1A)
    const uint32_t sDL = SOLVE ? smem_u32(sm + L::DL) : smem_u32(Ust(s));

    if (!SOLVE) {  // diag(exp(g_last - g)) U (16-byte chunks)
      for (int idx = tid; idx < 512; idx += 288) {
        const int R = idx >> 3;
        const uint4 in = *reinterpret_cast<const uint4*>(Ust(s) + idx * 16);
        const __nv_bfloat162* pin = reinterpret_cast<const __nv_bfloat162*>(&in);
        const float fr = dec[R];
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(pin[e]);
          pk[e] = pack_bf16(x.x * fr, x.y * fr);
        }
        *reinterpret_cast<uint4*>(DD + idx * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    fence_proxy_async();  // the carried key and the scaled rows, for the products
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- P = Q X^T (committed alone: the P~ warps start on it), D1 = W S0,
    // then Oa = Q S0 (read only after the second group, whose commit covers it)
    if (issuer) {
      const uint32_t sQ = smem_u32(Qst(s)), sX = smem_u32(Xst(s));
      if (c == 0) {  // later chunks' P was issued during the chunk before
        mma_chain_mn(tmem + L::col_p(c), kdesc<64>, sQ, kdesc<64>, sX, DK, idesc_bf16(64, 64), false);
        umma_commit(mbar_p);
        ++n_pc;
      }
      if (SOLVE)
        mma_chain_mn(tmem + L::COL_D1, kdesc<64>, smem_u32(Wst(s)), mndesc, sS, DK,
                     idesc_bf16(64, NV, false, true), false);
      umma_commit(mbar);
      ++n_mc;
      mma_chain_mn(tmem + L::COL_OA, kdesc<64>, sQ, mndesc, sS, DK, idesc_bf16(64, NV, false, true),
                   false);
    }
    if ((lo && !mbar_wait(mbar_p, pph, a.wait_ns)) || (hi && SOLVE && !mbar_wait(mbar, mph, a.wait_ns))) {
      *abort_flag = 1;
      atomicExch(a.status, kStatusTimeout);
    }
    pph ^= 1;
    mph ^= 1;
    tc_fence_after();
    if (lo) {  // P~ = decay-masked P, columns 32 hf .. 32 hf + 31 of row r64
      float pv[32];
      ld_half(L::col_p(c), pv);
      const float gr = gl[r64];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = 32 * hf + i;
        pv[i] = (t <= r64) ? __expf(gr - gl[t]) * pv[i] : 0.f;
      }
      store_half(Pm, r64, pv);
    } else if (hi && SOLVE) {  // Delta = U - W S0, and diag(exp(g_last - g)) Delta
      float dv1[32];
      ld_half(L::COL_D1, dv1);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 raw = *reinterpret_cast<const uint4*>(Ust(s) + sw128(r64, 32 * hf + 8 * j));
        const __nv_bfloat162* pu = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 u2 = __bfloat1622float2(pu[e]);
          dv1[8 * j + 2 * e] = u2.x - dv1[8 * j + 2 * e];
          dv1[8 * j + 2 * e + 1] = u2.y - dv1[8 * j + 2 * e + 1];
        }
      }
      store_half(sm + L::DL, r64, dv1);
      const float dr = dec[r64];
#pragma unroll
      for (int n = 0; n < 32; ++n) dv1[n] *= dr;
      store_half(DD, r64, dv1);
    }
    fence_proxy_async();
    tc_fence_before();
    if (tid == 0) bulk_wait_read0();  // the previous output tile has left the staging buffer
    const bool ab2 = __syncthreads_or(*abort_flag);
    tc_fence_after();
    if (ab2) break;

    // ---- D2 = X^T diag(exp(g_last - g)) Delta, Ob = P~ Delta
    if (issuer) {
      const uint32_t sX = smem_u32(Xst(s));
      for (int ks = 0; ks < 4; ++ks)  // X^T over both 64-row atoms of d_k: one M = 128 product
        umma_bf16(tmem + L::COL_W, sdesc_mn128_wide(sX + ks * 2048, 8192), mndesc(sDD, ks),
                  idesc_bf16(128, NV, true, true), ks > 0 ? 1u : 0u);
      mma_chain_mn(tmem + L::col_p(c), kdesc<64>, sP, mndesc, sDL, 64, idesc_bf16(64, NV, false, true),
                   false);
      umma_commit(mbar);
      ++n_mc;
      if (c + 1 < NC) {  // the next chunk's P = Q X^T: its stage is loaded, its buffer free
        if (!mbar_wait(&full[s ^ 1], (uint32_t)(((c + 1) >> 1) & 1), a.wait_ns)) {
          *abort_flag = 1;
          atomicExch(a.status, kStatusTimeout);
        } else {
          tc_fence_after();
          mma_chain_mn(tmem + L::col_p(c + 1), kdesc<64>, smem_u32(Qst(s ^ 1)), kdesc<64>,
                       smem_u32(Xst(s ^ 1)), DK, idesc_bf16(64, 64), false);
          umma_commit(mbar_p);
          ++n_pc;
        }
      }
    }
    if (warp < 8 && !mbar_wait(mbar, mph, a.wait_ns)) {
      *abort_flag = 1;
      atomicExch(a.status, kStatusTimeout);
    }
    mph ^= 1;
    tc_fence_after();
    if (warp < 8) {  // S1 = Gamma_last S0 + D2
      float d2[32];
      {
        uint32_t r32[32];
        tmem_ld32(tmem + lane_off + L::COL_W + s_c0, r32);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) d2[i] = __uint_as_float(r32[i]);
      }
#pragma unroll
      for (int n = 0; n < 32; ++n) sreg[n] = gam_last * sreg[n] + d2[n];
      store_32(SB, s_row, s_c0, sreg);
    }
    if (lo) {  // O = diag(Gamma) Oa + Ob, this thread's 32 columns
      float oa[32], ob[32];
      ld_half(L::COL_OA, oa);
      ld_half(L::col_p(c), ob);
      const float gr = Gam[r64];
#pragma unroll
      for (int n = 0; n < 32; ++n) oa[n] = gr * oa[n] + ob[n];
      store_half(Ost, r64, oa);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      tma_store_4d(&tm_o, Ost, c0, h, t0, b);
      bulk_commit();
    }
  }
  if (tid == 0) bulk_wait0();
  // ---- carry out
  if (!*abort_flag) {
    if (a.S_out && warp < 8) {
      const size_t dv = (size_t)gridDim.y * NV;
      float* dst = a.S_out + ((size_t)bh * DK + s_row) * dv + c0 + s_c0;
#pragma unroll
      for (int n = 0; n < 32; ++n) dst[n] = sreg[n];
    }
    if (split == 0) {
      if (a.kprev_out)
        for (int i = tid; i < DK; i += 288)
          a.kprev_out[(size_t)bh * DK + i] = a.k[(((size_t)b * a.T + (a.T - 1)) * a.H + h) * DK + i];
      if (a.pos_out && tid == 0) a.pos_out[bh] = (a.pos_in ? a.pos_in[bh] : 0) + a.T;
    }
  } else if (issuer) {
    // drain the loads still in flight before the shared memory goes away
    for (int s = 0; s < 2; ++s)
      if (issued[s] > 0) mbar_wait(&full[s], (uint32_t)((issued[s] - 1) & 1), a.wait_ns);
  }
  if (issuer) {  // no product may still write TMEM when it is freed (the abort path)
    if (n_pc > 0) mbar_wait(mbar_p, (uint32_t)((n_pc - 1) & 1), a.wait_ns);
    if (n_mc > 0) mbar_wait(mbar, (uint32_t)((n_mc - 1) & 1), a.wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------------
// (b'') sequential kernel in transition form, d_k = d_v = 64.  With the
// chunk's state-independent operands formed ahead of the chain,
//   S1 = Gamma_last S0 + X~^T U - (X~^T W) S0 = Gamma_last S0 + b - M S0
//   O  = (diag(Gamma) Q - P~ W) S0 + P~ U     = Q' S0 + P~ U
// so the state chain carries ONE product per chunk, [-M ; Q'] S0 (M = 128,
// N = 64, K = 64), accumulated onto [b ; P~ U], which a front product
// [X~^T ; P~] [W | U] (M = 128, N = 128) left in TMEM: rows 0..63 of the
// result are the next state less Gamma_last S0, rows 64..127 the chunk's
// outputs.  Roles:
//   warps 4..15   NF = 3 fronts of four warps, chunk c on front c % NF:
//                 P^T = X Q^T -> P~^T (decay-masked) and X~ = diag(exp(g_last - g)) X,
//                 then [X~^T ; P~] [W | U] into TMEM buffer c % 2; its rows
//                 0..63 give -M, rows 64..127 (with the stage's Q) give Q',
//                 both as bf16 rows of one 128-row K-major operand
//   warps 0, 1    state chain: the product, then S1 = Gamma_last S0 + acc
//   warps 2, 3    outputs: O = acc rows 64..127, TMA store
// The fronts run up to two chunks ahead of the chain (two TMEM buffers and
// operand tiles); the chain's round trip per chunk is one product and one
// TMEM -> register -> shared-memory pass.  A front's own latency per chunk
// (two products, each with its epilogue) is several times the chain's, so
// three of them take turns.  Loads: the first NST chunks are issued at the
// start, and the front that finishes chunk c refills its stage with chunk
// c + NST (no producer warp: 16 warps keep 128 registers a thread).
// ----------------------------------------------------------------------
template <bool SOLVE, bool L2N>
struct ChainSmem {
  static constexpr int NST = 4;
  static constexpr size_t XO = 0, PO = 8192, WO = 16384, QO = 24576, UO = 32768, GO = 40960;
  static constexpr size_t STAGE = GO + (L2N ? 2048 : 1024);  // gates: Gamma, exp(g_last - g), g,
                                                             // exp(g - g_block), then phi's row scales
  static constexpr size_t AM = NST * STAGE;          // 2 x [-M ; Q']: 128 K-major bf16 rows
  static constexpr size_t SB = AM + 2 * 16384;       // S rows (MN-major B)
  static constexpr size_t OST = SB + 8192;           // two output staging tiles
  static constexpr size_t GL = OST + 2 * 8192;       // Gamma_last of each TMEM buffer's chunk
  static constexpr size_t BAR = GL + 16;
  static constexpr size_t MISC = BAR + 256;          // tmem address, abort flag, loads issued per stage
  static constexpr size_t TOTAL = MISC + 64 + 1024;
  static constexpr uint32_t TX = 2 * 8192 + (SOLVE ? 8192 : 0) + 8192 + 1024;
  static_assert(TOTAL <= 232448, "shared memory budget");
  static_assert(STAGE % 1024 == 0 && AM % 1024 == 0, "1 KB aligned tiles");
  static constexpr int NF = 3;                    // fronts
  static constexpr int kThreads = 32 * (4 + 4 * NF);  // chain, outputs, fronts
  // TMEM: P^T of front f (M = 64 layout) at 64 f; buffer p of the front product
  // at 64 NF + 128 p (columns 0..63: [M ; P~ W], 64..127: [b ; P~ U], the
  // chain's accumulator)
  static constexpr uint32_t NCOLS = 512;
  __host__ __device__ static constexpr uint32_t col_pt(int f) { return 64 * f; }
  static_assert(64 * NF + 256 <= NCOLS, "TMEM budget");
  __host__ __device__ static constexpr uint32_t col_f(int p) { return 64 * NF + 128 * p; }
  static constexpr int G_GAM = 0, G_DEC = 64, G_GL = 128, G_CF = 192;
  static constexpr int G_SQ = 256, G_SX = 320;
};

template <bool SOLVE, bool L2N, bool PK = false>  // PK: packed sequences' rows read and written in place
__global__ void __launch_bounds__(ChainSmem<SOLVE, L2N>::kThreads, 1)
    tc_fwd_chain_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_o, TcArgs a) {
  using L = ChainSmem<SOLVE, L2N>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  constexpr int NST = L::NST;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* full = bars;              // [NST] stage loaded
  constexpr int NF = L::NF;
  uint64_t* fmma = bars + NST;        // [NF] P^T of front f done
  uint64_t* f2mma = fmma + NF;        // [NF] front product of front f done
  uint64_t* fdone = f2mma + NF;       // [2] operand tile and TMEM buffer p ready for the chain
  uint64_t* cmma = fdone + 2;         // [2] chain product of buffer p done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
  volatile int* issued = reinterpret_cast<volatile int*>(sm + L::MISC + 8);  // [NST] loads issued per stage
  // chunks whose accumulators the chain / the output warps have read (monotonic
  // counts: a front that runs ahead waits on them rather than on an mbarrier
  // phase, whose parity could alias across two pending phases)
  volatile int* chain_read = reinterpret_cast<volatile int*>(sm + L::MISC + 24);
  volatile int* out_read = reinterpret_cast<volatile int*>(sm + L::MISC + 28);
  float* glast = reinterpret_cast<float*>(sm + L::GL);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int b = bh / a.H, h = bh % a.H;
  auto stage = [&](int s) { return sm + s * L::STAGE; };
  auto fail = [&]() {
    *abort_flag = 1;
    atomicExch(a.status, kStatusTimeout);
  };

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      issued[i] = 0;
    }
    *chain_read = 0;
    *out_read = 0;
    for (int f = 0; f < NF; ++f) {
      mbar_init(&fmma[f], 1);
      mbar_init(&f2mma[f], 1);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(&fdone[p], 128);
      mbar_init(&cmma[p], 1);
    }
    fence_mbar_init();
  }
  if (!SOLVE) {  // additive write: the W tiles stay zero, so M = 0 and Q' = diag(Gamma) Q
    for (int i = tid; i < NST * 512; i += L::kThreads)
      *reinterpret_cast<uint4*>(stage(i >> 9) + L::WO + (i & 511) * 16) = make_uint4(0, 0, 0, 0);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, L::NCOLS);
    tmem_relinquish();
    tc_fence_before();
  }
  fence_proxy_async();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int quad = warp & 3;
  const uint32_t lane_off = (uint32_t)(32 * quad) << 16;
  // the per-chunk kernel has completed (and its writes are visible) past
  // this wait; a timeout it recorded leaves its images incomplete: then no
  // chunk is computed and no carry is written
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const bool upstream_failed = *reinterpret_cast<volatile uint32_t*>(a.status) != 0u;
  if (upstream_failed) *abort_flag = 1;
  // a packed sequence ends with its last chunk that holds tokens
  const int NCb = a.cu ? min(a.NC, (a.cu[b + 1] - a.cu[b] + kC - 1) / kC) : a.NC;
  const int NC = upstream_failed ? 0 : NCb;
  // chunk c into stage c % NST (one thread; the stage's previous chunk is done)
  auto load_chunk = [&](int c) {
    const int s = c % NST;
    uint8_t* st = stage(s);
    const size_t ci = (size_t)bh * a.NC + c;
    mbar_arrive_expect_tx(&full[s], L::TX);
    const int r0 = PK ? a.cu[b] + c * kC : c * kC, bb = PK ? 0 : b;  // packed: one batch row
    tma_load_4d(st + L::XO, &tm_k, &full[s], 0, h, r0 - a.shift, bb);
    tma_load_4d(st + L::QO, &tm_q, &full[s], 0, h, r0, bb);
    if (SOLVE) bulk_load(st + L::WO, a.ws_T + ci * 16384, 8192, &full[s]);
    bulk_load(st + L::UO, a.ws_T + ci * 16384 + 8192, 8192, &full[s]);
    bulk_load(st + L::GO, a.ws_g + ci * kGateF, 1024, &full[s]);
    __threadfence_block();
    issued[s] = issued[s] + 1;  // one issuing thread per stage and chunk at a time
  };
  // bounded spin until a shared counter reaches a value (false on a timeout
  // or once another role gave up)
  auto spin_until = [&](volatile int* x, int target) {
    if (*x >= target) return true;
    const uint64_t t0 = globaltimer();
    while (*x < target)
      if (*abort_flag || globaltimer() - t0 > a.wait_ns) return false;
    return true;
  };
  if (tid == 0) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    for (int c = 0; c < NST && c < NC; ++c) load_chunk(c);
  }

  if (warp >= 4) {
    // ------------------------------------------------------------ fronts
    const int fr = (warp - 4) >> 2;          // this front; it takes the chunks c with c % NF == fr
    const int ftid = tid - 128 - 128 * fr;
    const int fbar = fr == 0 ? 1 : 4 + fr;   // its named barrier (3 and 4 are the chain's and the outputs')
    const int r = 16 * quad + (lane & 15);  // P^T row (key index) of this lane
    const int half = lane >> 4;             // P^T columns 32 half .. 32 half + 31
    uint32_t fph = 0, f2ph = 0;
    int n_f2 = 0;  // front products issued (ftid 0's bookkeeping)
    for (int c = fr; c < NC; c += NF) {
      const int s = c % NST, p = c & 1;
      // a front can reach chunk c before the stage's previous chunk c - NST
      // was even loaded: first see the load of chunk c issued, so that the
      // wait below is on the latest phase of the stage's barrier
      if (!spin_until(&issued[s], c / NST + 1) || !mbar_wait(&full[s], (uint32_t)((c / NST) & 1), a.wait_ns)) fail();
      uint8_t* st = stage(s);
      const float* gt = reinterpret_cast<const float*>(st + L::GO);
      const bool carried = c == 0 && a.kprev_in && a.shift;  // x_0 = the carried key
      if (carried && ftid < 64)
        *reinterpret_cast<__nv_bfloat16*>(st + L::XO + sw128(0, ftid)) = a.kprev_in[(size_t)bh * 64 + ftid];
      if (PK && c == 0 && a.shift && !a.kprev_in && ftid < 64)  // not the previous sequence's key
        *reinterpret_cast<__nv_bfloat16*>(st + L::XO + sw128(0, ftid)) = __float2bfloat16_rn(0.f);
      if constexpr (L2N) {  // row scales of the prologue's phi, 1 / max(|row|, 1e-12), of the query
                            // row and the key row r (the carried key is a feature already); the raw
                            // rows enter the products and the scales their epilogues
        float* gw = reinterpret_cast<float*>(st + L::GO);
        float pq = 0.f, px = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 rq = *reinterpret_cast<const uint4*>(st + L::QO + sw128(r, 32 * half + 8 * j));
          const uint4 rx = *reinterpret_cast<const uint4*>(st + L::XO + sw128(r, 32 * half + 8 * j));
          const __nv_bfloat162* hq = reinterpret_cast<const __nv_bfloat162*>(&rq);
          const __nv_bfloat162* hx = reinterpret_cast<const __nv_bfloat162*>(&rx);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 q2 = __bfloat1622float2(hq[e]), x2 = __bfloat1622float2(hx[e]);
            pq = fmaf(q2.x, q2.x, fmaf(q2.y, q2.y, pq));
            px = fmaf(x2.x, x2.x, fmaf(x2.y, x2.y, px));
          }
        }
        pq += __shfl_xor_sync(0xffffffffu, pq, 16);
        px += __shfl_xor_sync(0xffffffffu, px, 16);
        if (half == 0) {
          gw[L::G_SQ + r] = 1.f / fmaxf(sqrtf(pq), 1e-12f);
          gw[L::G_SX + r] = (carried && r == 0) ? 1.f : 1.f / fmaxf(sqrtf(px), 1e-12f);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      if (named_bar_any(fbar, 128, *abort_flag != 0)) break;
      tc_fence_after();
      if (ftid == 0) {  // P^T = X Q^T
        const uint32_t sX = smem_u32(st + L::XO), sQ = smem_u32(st + L::QO);
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem + L::col_pt(fr), kdesc<64>(sX, ks), kdesc<64>(sQ, ks), idesc_bf16(64, 64),
                    ks > 0 ? 1u : 0u);
        umma_commit(&fmma[fr]);
      }
      // the factors of this thread's 32 columns, gathered while the product runs
      const float* gl = gt + L::G_GL;
      const float* cf = gt + L::G_CF;
      const float gi = gl[r], cfr = cf[r];
      const int I = r >> 4;
      const bool ratio_ok = cfr > 1e-30f;
      float cfv[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 c4 = *reinterpret_cast<const float4*>(cf + 32 * half + i);
        cfv[i] = c4.x; cfv[i + 1] = c4.y; cfv[i + 2] = c4.z; cfv[i + 3] = c4.w;
      }
      float f[2];
#pragma unroll
      for (int J2 = 0; J2 < 2; ++J2) {
        const int J = 2 * half + J2;
        f[J2] = J > I ? __expf(gl[16 * J] - gi) : (J == I && ratio_ok ? __fdividef(1.f, cfr) : 0.f);
      }
      if (!mbar_wait(&fmma[fr], fph, a.wait_ns)) fail();
      fph ^= 1;
      tc_fence_after();
      {  // P~^T[r][t] = P[t][r] exp(g_t - g_r) for t >= r.  With cf_t = exp(g_t - g_{16 J(t)}):
         // exp(g_t - g_r) = cf_t exp(g_{16 J} - g_r) across blocks and cf_t / cf_r inside one
        uint32_t pr[32];
        tmem_ld16x2_32(tmem + lane_off + L::col_pt(fr), pr);
        tmem_wait_ld();
        float pv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int t = 32 * half + i;
          const float v = __uint_as_float(pr[i]) * cfv[i] * f[i >> 4];
          pv[i] = (t >= r) ? v : 0.f;
        }
        if (!ratio_ok) {  // exact decays in the row's own block
#pragma unroll
          for (int J2 = 0; J2 < 2; ++J2) {
            if (2 * half + J2 == I) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int t = 16 * I + i;
                pv[16 * J2 + i] = (t >= r) ? __expf(gl[t] - gi) * __uint_as_float(pr[16 * J2 + i]) : 0.f;
              }
            }
          }
        }
        if constexpr (L2N) {  // phi(x_r) . phi(q_t) from the raw rows
          const float sxr = gt[L::G_SX + r];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 s4 = *reinterpret_cast<const float4*>(gt + L::G_SQ + 32 * half + i);
            pv[i] *= sxr * s4.x; pv[i + 1] *= sxr * s4.y; pv[i + 2] *= sxr * s4.z; pv[i + 3] *= sxr * s4.w;
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) pk[e] = pack_bf16(pv[8 * j + 2 * e], pv[8 * j + 2 * e + 1]);
          *reinterpret_cast<uint4*>(st + L::PO + sw128(r, 32 * half + 8 * j)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      {  // X~ rows in place of X (the product that read X is complete)
        uint4 in[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) in[k] = *reinterpret_cast<const uint4*>(st + L::XO + (ftid + 128 * k) * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int idx = ftid + 128 * k;
          const float fr = L2N ? gt[L::G_DEC + (idx >> 3)] * gt[L::G_SX + (idx >> 3)]  // decay x phi's scale
                               : gt[L::G_DEC + (idx >> 3)];
          const __nv_bfloat162* pin = reinterpret_cast<const __nv_bfloat162*>(&in[k]);
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(pin[e]);
            pk[e] = pack_bf16(x.x * fr, x.y * fr);
          }
          *reinterpret_cast<uint4*>(st + L::XO + idx * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      named_bar(fbar, 128);
      tc_fence_after();
      if (ftid == 0) {  // [X~^T ; P~] [W | U] into TMEM buffer p, once the chunk two back left it
        if (c >= 2 && !(spin_until(chain_read, c - 1) && spin_until(out_read, c - 1))) {
          fail();
        } else {
          tc_fence_after();
          const uint32_t sA = smem_u32(st + L::XO), sB = smem_u32(st + L::WO);
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16(tmem + L::col_f(p), sdesc_mn128_wide(sA + ks * 2048, 8192),
                      sdesc_mn128_wide(sB + ks * 2048, 16384), idesc_bf16(128, 128, true, true),
                      ks > 0 ? 1u : 0u);
          umma_commit(&f2mma[fr]);
          ++n_f2;
        }
      }
      if (!mbar_wait(&f2mma[fr], f2ph, a.wait_ns)) fail();
      f2ph ^= 1;
      tc_fence_after();
      if (named_bar_any(fbar, 128, *abort_flag != 0)) break;
      {  // rows 0..63: -M -> tile rows 0..63; rows 64..127: Q' = diag(Gamma) Q - P~ W -> rows 64..127
        const int row = 32 * quad + lane;   // TMEM lane of this thread
        float mv[64];
        tmem_ld64(tmem + lane_off + L::col_f(p), mv);
        tmem_wait_ld();
        uint8_t* AMp = sm + L::AM + p * 16384;
        if (quad < 2) {
#pragma unroll
          for (int n = 0; n < 64; ++n) mv[n] = -mv[n];
        } else {
          const int t = row - 64;
          const float gq = L2N ? gt[L::G_GAM + t] * gt[L::G_SQ + t] : gt[L::G_GAM + t];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 raw = *reinterpret_cast<const uint4*>(st + L::QO + sw128(t, 8 * j));
            const __nv_bfloat162* pq2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 q2 = __bfloat1622float2(pq2[e]);
              mv[8 * j + 2 * e] = fmaf(gq, q2.x, -mv[8 * j + 2 * e]);
              mv[8 * j + 2 * e + 1] = fmaf(gq, q2.y, -mv[8 * j + 2 * e + 1]);
            }
          }
        }
        store_row64(AMp, row, mv);
        if (ftid == 0) glast[p] = gt[L::G_GAM + 63];
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&fdone[p]);
      named_bar(fbar, 128);  // nothing of the stage is read after this: refill it
      if (ftid == 0 && c + NST < NC && !*abort_flag) load_chunk(c + NST);
    }
    const bool ab = __any_sync(0xffffffffu, *abort_flag != 0);  // one answer per warp
    if (a.kprev_out && !ab && fr == 0 && ftid < 32) {  // the last key, as a feature (warp 4)
      const __nv_bfloat16* kl = a.k + (((size_t)b * a.T + (a.T - 1)) * a.H + h) * 64;
      const float k0 = __bfloat162float(kl[ftid]), k1 = __bfloat162float(kl[ftid + 32]);
      float sc = 1.f;
      if (L2N) {
        float ss = fmaf(k0, k0, k1 * k1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        sc = 1.f / fmaxf(sqrtf(ss), 1e-12f);
      }
      a.kprev_out[(size_t)bh * 64 + ftid] = __float2bfloat16_rn(k0 * sc);
      a.kprev_out[(size_t)bh * 64 + ftid + 32] = __float2bfloat16_rn(k1 * sc);
    }
    if (a.pos_out && !*abort_flag && fr == 0 && ftid == 0) a.pos_out[bh] = (a.pos_in ? a.pos_in[bh] : 0) + a.T;
    if (ftid == 0 && n_f2 > 0) mbar_wait(&f2mma[fr], (uint32_t)((n_f2 - 1) & 1), a.wait_ns);  // TMEM quiet
  } else if (warp < 2) {
    // ------------------------------------------------------------ state chain
    uint8_t* SB = sm + L::SB;
    const uint32_t sS = smem_u32(SB);
    const int r = 32 * warp + lane;  // S row = TMEM lane
    float sreg[64];
#pragma unroll
    for (int n = 0; n < 64; ++n) sreg[n] = 0.f;
    if (a.S_in) {
      const float* src = a.S_in + ((size_t)bh * 64 + r) * 64;
#pragma unroll
      for (int n = 0; n < 64; n += 4) {
        const float4 v = *reinterpret_cast<const float4*>(src + n);
        sreg[n] = v.x; sreg[n + 1] = v.y; sreg[n + 2] = v.z; sreg[n + 3] = v.w;
      }
    }
    store_row64(SB, r, sreg);
    fence_proxy_async();
    named_bar(3, 64);
    int n_c = 0;  // chain products issued (thread 0's bookkeeping)
    for (int c = 0; c < NC; ++c) {
      const int p = c & 1;
      if (!mbar_wait(&fdone[p], (uint32_t)((c >> 1) & 1), a.wait_ns)) fail();
      tc_fence_after();
      if (named_bar_any(3, 64, *abort_flag != 0)) break;
      const float gl_ = glast[p];
      if (tid == 0) {  // [b ; P~ U] += [-M ; Q'] S0
        const uint32_t sA = smem_u32(sm + L::AM + p * 16384);
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem + L::col_f(p) + 64, kdesc<128>(sA, ks), mndesc(sS, ks), idesc_bf16(128, 64, false, true),
                    1u);
        umma_commit(&cmma[p]);
        ++n_c;
      }
      if (!mbar_wait(&cmma[p], (uint32_t)((c >> 1) & 1), a.wait_ns)) fail();
      tc_fence_after();
      {  // S1 = Gamma_last S0 + acc, 32 columns at a time
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t d2[32];
          tmem_ld32(tmem + lane_off + L::col_f(p) + 64 + 32 * hh, d2);
          tmem_wait_ld();
#pragma unroll
          for (int n = 0; n < 32; ++n) sreg[32 * hh + n] = fmaf(gl_, sreg[32 * hh + n], __uint_as_float(d2[n]));
        }
        tc_fence_before();
        store_row64(SB, r, sreg);
      }
      fence_proxy_async();
      named_bar(3, 64);
      if (tid == 0) *chain_read = c + 1;  // both chain warps read this chunk's accumulator
    }
    if (!*abort_flag && a.S_out) {
      float* dst = a.S_out + ((size_t)bh * 64 + r) * 64;
#pragma unroll
      for (int n = 0; n < 64; n += 4)
        *reinterpret_cast<float4*>(dst + n) = make_float4(sreg[n], sreg[n + 1], sreg[n + 2], sreg[n + 3]);
    }
    if (tid == 0 && n_c > 0) {  // TMEM quiet before it is freed
      const int cl = n_c - 1;
      mbar_wait(&cmma[cl & 1], (uint32_t)((cl >> 1) & 1), a.wait_ns);
    }
  } else {
    // ------------------------------------------------------------ outputs
    const int t = 32 * (warp - 2) + lane;  // output row = TMEM lane 64 + t
    for (int c = 0; c < NC; ++c) {
      const int p = c & 1;
      if (!mbar_wait(&cmma[p], (uint32_t)((c >> 1) & 1), a.wait_ns)) fail();
      tc_fence_after();
      if (named_bar_any(4, 64, *abort_flag != 0)) break;
      uint8_t* Ost = sm + L::OST + p * 8192;
      if (tid == 64) bulk_wait_read1();  // the tile stored from this buffer two chunks ago is out
      named_bar(4, 64);
      {
        uint32_t ov[2][32];
        tmem_ld32(tmem + lane_off + L::col_f(p) + 64, ov[0]);
        tmem_ld32(tmem + lane_off + L::col_f(p) + 96, ov[1]);
        tmem_wait_ld();
        tc_fence_before();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int n = 8 * j + 2 * e;
            pk[e] = pack_bf16(__uint_as_float(ov[n >> 5][n & 31]), __uint_as_float(ov[(n + 1) >> 5][(n + 1) & 31]));
          }
          if (PK) {  // the row itself, if it belongs to the sequence
            if (c * kC + t < a.cu[b + 1] - a.cu[b])
              *reinterpret_cast<uint4*>(a.o + (((size_t)a.cu[b] + c * kC + t) * a.H + h) * 64 + 8 * j) =
                  make_uint4(pk[0], pk[1], pk[2], pk[3]);
          } else {
            *reinterpret_cast<uint4*>(Ost + sw128(t, 8 * j)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
      fence_proxy_async();
      named_bar(4, 64);
      if (tid == 64) {
        *out_read = c + 1;  // both output warps read this chunk's accumulator
        if (!PK) {
          tma_store_4d(&tm_o, Ost, 0, h, c * kC, b);
          bulk_commit();
        }
      }
    }
    if (tid == 64) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) {  // loads still in flight complete before the shared memory goes away
    for (int s = 0; s < NST; ++s)
      if (issued[s] > 0) mbar_wait(&full[s], (uint32_t)((issued[s] - 1) & 1), a.wait_ns);
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::NCOLS);
  }
}

// ---------------------------------------------------------------- host side
struct WsLayout {
  size_t status, T, g, total;
};
// Per chunk: the bf16 W | U images (2 d_k 128 bytes) and kGateF gate floats.
WsLayout ws_layout(int B, int T, int H, int chunk, int dk) {
  const size_t NC = (size_t)(T + chunk - 1) / chunk;
  WsLayout w;
  w.status = 0;
  w.T = 256;
  w.g = w.T + (size_t)B * H * NC * (2 * (size_t)dk * 128);
  w.total = align_up(w.g + (size_t)B * H * NC * kGateF * 4, 256);
  return w;
}

template <int DK, int NV, bool SOLVE>
int launch_t(const FwdArgs& fa, const TcArgs& ta) {
  const int BH = fa.B * fa.H;
  CUtensorMap mq, mk, mv, mo;
  // packed sequences read in place: the rows of all sequences as one batch row
  const int mB = ta.packed ? 1 : fa.B, mT = ta.packed ? (int)fa.packed_total : fa.T;
  if (!make_map(&mq, fa.q, mB, mT, fa.H, DK, 64) || !make_map(&mk, fa.k, mB, mT, fa.H, DK, 64) ||
      !make_map(&mv, fa.v, mB, mT, fa.H, fa.dv, 64) || !make_map(&mo, fa.o, mB, mT, fa.H, fa.dv, 64))
    return FALCON_ERR_CUDA;
  if constexpr (DK == 64) {
    {  // per-chunk gates, W and U
      auto k = ta.item_map ? tc_wyu_kernel<SOLVE, 64, true> : tc_wyu_kernel<SOLVE, 64, false>;
      const size_t smem = WyuSmem<64>::TOTAL;
      if (!set_smem_limit(reinterpret_cast<const void*>(k), smem))
        return FALCON_ERR_CUDA;
      // persistent: four CTAs per SM (shared memory and TMEM both allow four)
      const long items = (long)ta.NC * BH;
      dim3 grid((unsigned)std::min<long>(items, 4L * sm_count()));
      record_event(fa, 0);
      if (launch_overlapped(fa, k, grid, dim3(128), smem, mk, mv, ta) != FALCON_OK) return FALCON_ERR_CUDA;
      record_event(fa, 1);
    }
    {  // transition form: producer warp, front warpgroup, chain and output warps
      const bool l2n = (ta.pro & FALCON_PROLOGUE_L2NORM_QK) != 0;
      auto k = ta.packed ? (l2n ? tc_fwd_chain_kernel<SOLVE, true, true> : tc_fwd_chain_kernel<SOLVE, false, true>)
                         : (l2n ? tc_fwd_chain_kernel<SOLVE, true, false> : tc_fwd_chain_kernel<SOLVE, false, false>);
      const size_t smem = l2n ? ChainSmem<SOLVE, true>::TOTAL : ChainSmem<SOLVE, false>::TOTAL;
      if (!set_smem_limit(reinterpret_cast<const void*>(k), smem))
        return FALCON_ERR_CUDA;
      // overlaps the per-chunk kernel's tail with its launch and set-up
      if (launch_overlapped(fa, k, dim3(BH), dim3(ChainSmem<SOLVE, false>::kThreads), smem, mq, mk, mo, ta) !=
          FALCON_OK)
        return FALCON_ERR_CUDA;
      record_event(fa, 2);
    }
  } else {
    {  // per-chunk gates, W and U (d = 128: two CTAs per SM)
      auto k = tc_wyu_kernel<SOLVE, DK>;
      const size_t smem = WyuSmem<DK>::TOTAL;
      if (!set_smem_limit(reinterpret_cast<const void*>(k), smem))
        return FALCON_ERR_CUDA;
      const long items = (long)ta.NC * BH;
      dim3 grid((unsigned)std::min<long>(items, 2L * sm_count()));
      record_event(fa, 0);
      if (launch_overlapped(fa, k, grid, dim3(128), smem, mk, mv, ta) != FALCON_OK) return FALCON_ERR_CUDA;
      record_event(fa, 1);
    }
    {
      auto k = tc_fwd_kernel<DK, NV, SOLVE>;
      const size_t smem = FwdSmem<DK, NV, SOLVE>::TOTAL;
      if (!set_smem_limit(reinterpret_cast<const void*>(k), smem))
        return FALCON_ERR_CUDA;
      dim3 grid(BH, fa.dv / NV);
      if (launch_overlapped(fa, k, grid, dim3(288), smem, mq, mk, mo, ta) != FALCON_OK) return FALCON_ERR_CUDA;
      record_event(fa, 2);
    }
  }
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace

bool tc_chunk_supported(const FwdArgs& a) {
  if (tc_f2_supported(a) || tc_f3a_supported(a) || tc_f3_supported(a)) return true;
  if (a.variant != FALCON_1 && a.variant != FALCON_1A) return false;
  if (a.dtype != FALCON_BF16 || a.chunk != 64 || a.T < 1) return false;
  if (a.dk != a.dv || (a.dk != 64 && a.dk != 128)) return false;
  return true;
}

int tc_chunk_launches(const FwdArgs& a) {
  if (tc_f3a_supported(a)) return tc_f3a_launches(a);
  return tc_f2_supported(a) ? 1 : 2;
}

size_t tc_chunk_ws_bytes(int B, int T, int H, int dk, int, int chunk, int variant) {
  if (variant == FALCON_2 || variant == FALCON_2A) return 256;  // status word only
  if (variant == FALCON_3A) return tc_f3a_ws_bytes(B, T, H);
  if (variant == FALCON_3) return tc_f3_ws_bytes(B, T, H);
  return ws_layout(B, T, H, chunk, dk).total;
}

int launch_tc_chunk(const FwdArgs& fa) {
  if (tc_f2_supported(fa)) return launch_tc_f2(fa);
  if (tc_f3a_supported(fa)) return launch_tc_f3a(fa);
  if (tc_f3_supported(fa)) return launch_tc_f3(fa);
  const WsLayout w = ws_layout(fa.B, fa.T, fa.H, 64, fa.dk);
  uint8_t* ws = reinterpret_cast<uint8_t*>(fa.ws);
  TcArgs ta;
  ta.B = fa.B; ta.T = fa.T; ta.H = fa.H; ta.NC = (fa.T + kC - 1) / kC;
  ta.shift = fa.shift;
  ta.eps = fa.eps; ta.eps_gamma = fa.eps_gamma;
  ta.beta = fa.beta; ta.lam = fa.lam; ta.pos_in = fa.pos_in;
  ta.kprev_in = reinterpret_cast<const __nv_bfloat16*>(fa.kprev_in);
  ta.S_in = fa.S_in;
  ta.k = reinterpret_cast<const __nv_bfloat16*>(fa.k);
  ta.S_out = fa.S_out;
  ta.kprev_out = reinterpret_cast<__nv_bfloat16*>(fa.kprev_out);
  ta.pos_out = fa.pos_out;
  ta.ws_T = ws + w.T;
  ta.ws_g = reinterpret_cast<float*>(ws + w.g);
  ta.status = reinterpret_cast<uint32_t*>(ws + w.status);
  ta.NV = 64;
  ta.pro = fa.dk == 64 ? fa.prologue : 0;  // fused into the d = 64 kernels (else applied before)
  ta.wait_ns = wait_limit_ns();
  ta.stall = take_test_stall() ? 1 : 0;
  ta.cu = fa.dk == 64 ? fa.cu : nullptr;
  ta.item_map = ta.cu ? fa.item_map : nullptr;
  ta.item_count = ta.cu ? fa.item_count : nullptr;
  ta.packed = ta.cu && fa.packed_total > 0 ? 1 : 0;
  ta.o = reinterpret_cast<__nv_bfloat16*>(fa.o);
  const bool solve = fa.variant == FALCON_1;
  if (fa.dk == 64) return solve ? launch_t<64, 64, true>(fa, ta) : launch_t<64, 64, false>(fa, ta);
  return solve ? launch_t<128, 64, true>(fa, ta) : launch_t<128, 64, false>(fa, ta);
}

// The items of packed sequences, (b H + h) NC + chunk for every chunk that
// holds tokens, in that order, then their count at map[B H NC] and the
// sequences' item offsets at map[B H NC + 1 + b]: one block scans the chunk
// counts 1024 sequences at a time, then every thread fills items, finding
// an item's sequence by bisection over the offsets.
__global__ void __launch_bounds__(1024) varlen_item_map_kernel(const int32_t* cu, int B, int H, int NC,
                                                              int32_t* map) {
  __shared__ int32_t scan[1024];
  __shared__ int32_t base;
  int32_t* off = map + (size_t)B * H * NC + 1;  // [B + 1]
  const int tid = threadIdx.x;
  if (tid == 0) base = 0;
  __syncthreads();
  for (int b0 = 0; b0 < B; b0 += 1024) {
    const int b = b0 + tid;
    const int n = b < B ? min(NC, max(0, (cu[b + 1] - cu[b] + kC - 1) / kC)) * H : 0;
    scan[tid] = n;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {  // inclusive prefix sum
      const int v = tid >= o ? scan[tid - o] : 0;
      __syncthreads();
      scan[tid] += v;
      __syncthreads();
    }
    if (b < B) off[b] = base + scan[tid] - n;
    __syncthreads();
    if (tid == 1023) base += scan[1023];
    __syncthreads();
  }
  const int total = base;
  if (tid == 0) {
    off[B] = total;
    map[(size_t)B * H * NC] = total;
  }
  __syncthreads();
  for (int i = tid; i < total; i += 1024) {
    int lo = 0, hi = B - 1;  // the last b with off[b] <= i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (off[mid] <= i) lo = mid;
      else hi = mid - 1;
    }
    const int r = i - off[lo], nc = (off[lo + 1] - off[lo]) / H;
    map[i] = (lo * H + r / nc) * NC + r % nc;
  }
}

bool tc_chunk_takes_map(const FwdArgs& a) {
  return !tc_f2_supported(a) && !tc_f3a_supported(a) && !tc_f3_supported(a) && a.dk == 64;
}

int launch_varlen_item_map(const int32_t* cu, int B, int H, int NC, int32_t* map, cudaStream_t s) {
  varlen_item_map_kernel<<<1, 1024, 0, s>>>(cu, B, H, NC, map);
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace falcon
