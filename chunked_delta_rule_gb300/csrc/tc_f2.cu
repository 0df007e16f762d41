// Tensor-core chunk forward for Falcon-2 / Falcon-2A (NLMS step per value
// channel), bf16 inputs, fp32 state, chunk 64, d_k = d_v in {64, 128}.
//
// Per chunk with state S0, in-chunk cumulative log-decay g (clamped decay
// [JC 数学上的稳定阀门:正衰减钳制]) and Gamma_r = exp(g_r)
// [FW 三种等价形式; JC Falcon家族六个变体各管一段]:
//   eta_rj  = beta_rj / (eps + |x_r|^2)         (zero for a pair that does not exist)
//   L_ri    = exp(g_r - g_i) x_r . x_i   (i < r), shared by every channel
//   Delta_rj = eta_rj (v_rj - Gamma_r (X S0)_rj - sum_{i<r} L_ri Delta_ij)
//              (Falcon-2A: Delta = eta (.) V)
//   O       = diag(Gamma) Q S0 + (Q X^T (.) [exp(g_t - g_r)]_{r<=t}) Delta
//   S1      = Gamma_last S0 + X~^T Delta,   X~ = diag(exp(g_last - g)) X
// The per-channel systems are one batched forward substitution with the
// shared L: each channel is solved by one thread.
//
// One CTA per (b, h, slice of 64 value channels).  Channel-major products
// put a channel in a TMEM lane, so the solving thread reads its own row:
//   warps 4..7  front (runs a chunk ahead): gates, [X ; Q] X^T -> L^T (fp32)
//               and the decay-masked P~ (bf16), then Q~ = diag(Gamma) Q in place
//   warps 0..3  back: the fp32 state S^T stays in TMEM (a channel per lane,
//               both 64-lane halves hold it); [S0^T ; S0^T] [X ; Q~]^T gives
//               (X S0)^T and (Q~ S0)^T; warps 0, 1 solve for Delta, warps 2, 3
//               form X~ and write the output tile; [Delta^T ; Delta^T] P~^T and
//               [Delta^T ; Delta^T] X~ accumulate the output and the state;
//               thread 0 also refills a stage by TMA (X | Q per 64-column
//               slab, the V and beta slices) as soon as its chunk is done.
// Every wait is bounded; on timeout the kernel records an error in the
// workspace status word and leaves its chunk loop.

#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_util.cuh"

namespace falcon {

using namespace tc;
using namespace tcu;

namespace {

struct F2Args {
  int B, T, H, dv, NC;
  int shift;  // pair t uses key t - shift (1 prefix alignment, 0 same-step)
  float eps, eps_gamma;
  const float* lam;
  const int64_t* pos_in;
  const __nv_bfloat16* kprev_in;
  const float* S_in;
  const __nv_bfloat16* k;
  float* S_out;
  __nv_bfloat16* kprev_out;
  int64_t* pos_out;
  uint32_t* status;
};

template <int DK>
struct F2Smem {
  static constexpr int kSl = DK / 64;               // 64-column slabs of d_k
  // stage: [X ; Q] per slab (X rows 0..63, Q rows 64..127; X~ and Q~ in place)
  static constexpr size_t XQ = 0;
  static constexpr size_t VS = XQ + kSl * 16384;    // V slice, bf16 swizzled rows
  static constexpr size_t BS = VS + 8192;           // beta slice, fp32 [64][64]
  static constexpr size_t LT = BS + 16384;          // L: diagonal 16x16 blocks fp32 [4][col][row] at +0,
                                                    // all of L as bf16 K-major rows at +8192
  static constexpr size_t PT = LT + 16384;          // P~, bf16 K-major rows t
  static constexpr size_t GT = PT + 8192;           // gates
  static constexpr size_t STAGE = GT + 2048;
  static constexpr int NST = 2;
  static constexpr size_t SA = NST * STAGE;         // [S0^T ; S0^T], K-major, 128 rows
  static constexpr size_t DA = SA + kSl * 16384;    // [Delta^T ; Delta^T], K-major, 128 rows
  static constexpr size_t OST = DA + 16384;         // output staging tile
  static constexpr size_t BAR = OST + 8192;
  static constexpr size_t MISC = BAR + 128;
  static constexpr size_t TOTAL = MISC + 16 + 1024;
  static constexpr uint32_t TX = kSl * 16384 + 8192 + 16384;
  static_assert(STAGE % 1024 == 0, "1 KB aligned stages");
  static_assert(TOTAL <= 232448, "shared memory budget");
  // gates (fp32 offsets in GT)
  static constexpr int G_INV = 0, G_GAM = 64, G_DEC = 128, G_G = 192, G_CFE = 256, G_WS = 320;
  // TMEM: S^T | [(X S0)^T | O^T] x 2 | [G ; P] (front) | E: sum_{i in earlier blocks} L_ri Delta_i
  static constexpr uint32_t COL_S = 0, COL_YO = DK, COL_F = DK + 256, COL_E = DK + 320, NCOLS = 512;
  static_assert(COL_E + 64 <= NCOLS, "TMEM budget");
};

template <int DK, bool SOLVE>
__global__ void __launch_bounds__(256, 1)
    tc_f2_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_beta,
                 const __grid_constant__ CUtensorMap tm_o, F2Args a) {
  using L = F2Smem<DK>;
  constexpr int kSl = L::kSl, NST = L::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* full = bars;             // [NST]
  uint64_t* fdone = bars + NST;      // [NST]
  uint64_t* fmma = bars + 2 * NST;
  uint64_t* bmma = fmma + 1;         // [2]
  uint64_t* tmma = bmma + 2;         // trailing update of the solve done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x, slice = blockIdx.y;
  const int b = bh / a.H, h = bh % a.H;
  const int c0 = 64 * slice;  // first value channel of this CTA
  const int NC = a.NC;
  auto stage = [&](int s) { return sm + s * L::STAGE; };
  auto fail = [&]() {
    *abort_flag = 1;
    atomicExch(a.status, kStatusTimeout);
  };

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&fdone[i], 128);
    }
    mbar_init(fmma, 1);
    mbar_init(&bmma[0], 1);
    mbar_init(&bmma[1], 1);
    mbar_init(tmma, 1);
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

  // TMA of chunk c into stage c % NST (issued by thread 0)
  auto load_chunk = [&](int c) {
    const int s = c % NST;
    uint8_t* st = stage(s);
    mbar_arrive_expect_tx(&full[s], L::TX);
#pragma unroll
    for (int s2 = 0; s2 < kSl; ++s2) {
      tma_load_4d(st + L::XQ + s2 * 16384, &tm_k, &full[s], 64 * s2, h, c * kC - a.shift, b);
      tma_load_4d(st + L::XQ + s2 * 16384 + 8192, &tm_q, &full[s], 64 * s2, h, c * kC, b);
    }
    tma_load_4d(st + L::VS, &tm_v, &full[s], c0, h, c * kC, b);
    tma_load_4d(st + L::BS, &tm_beta, &full[s], c0, h, c * kC, b);
  };
  if (tid == 0)
    for (int c = 0; c < NST && c < NC; ++c) load_chunk(c);

  if (warp >= 4) {
    // ------------------------------------------------------------ front
    const int ftid = tid - 128;
    const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
    const int row = 32 * quad + lane;  // 0..63: Gram row r; 64..127: P row t = row - 64
    uint32_t fph = 0;
    float lam_next = (ftid < 64 && ftid < a.T) ? a.lam[((size_t)b * a.T + ftid) * a.H + h] : 0.f;
    for (int c = 0; c < NC; ++c) {
      const int s = c % NST;
      const float lam_cur = lam_next;
      {
        const int tn = (c + 1) * kC + ftid;
        lam_next = (ftid < 64 && c + 1 < NC && tn < a.T) ? a.lam[((size_t)b * a.T + tn) * a.H + h] : 0.f;
      }
      if (!mbar_wait(&full[s], (uint32_t)((c / NST) & 1))) fail();
      uint8_t* st = stage(s);
      float* gt = reinterpret_cast<float*>(st + L::GT);
      if (c == 0 && a.kprev_in && a.shift && ftid < DK)  // x_0 = carried key
        *reinterpret_cast<__nv_bfloat16*>(st + L::XQ + (ftid >> 6) * 16384 + sw128(0, ftid & 63)) =
            a.kprev_in[(size_t)bh * DK + ftid];
      // gates: inclusive prefix sum of the clamped log-decay over the chunk
      float g = 0.f;
      if (ftid < 64) {
        const int t = c * kC + ftid;
        g = t < a.T ? clamped_log_decay(lam_cur, a.eps_gamma) : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float n = __shfl_up_sync(0xffffffffu, g, o);
          if (lane >= o) g += n;
        }
        if (lane == 31) gt[L::G_WS + (warp - 4)] = g;
      }
      named_bar(1, 128);
      if (ftid < 64) {
        if (warp == 5) g += gt[L::G_WS];
        gt[L::G_G + ftid] = g;
        gt[L::G_GAM + ftid] = __expf(g);
      }
      named_bar(1, 128);
      if (ftid < 64) {
        gt[L::G_DEC + ftid] = __expf(gt[L::G_G + 63] - g);
        gt[L::G_CFE + ftid] = __expf(gt[L::G_G + (ftid | 15)] - g);  // exp(g_end(block) - g)
      }
      fence_proxy_async();
      tc_fence_before();
      if (named_bar_any(1, 128, *abort_flag != 0)) break;
      tc_fence_after();
      if (ftid == 0) {  // [G ; P] = [X ; Q] X^T
        const uint32_t sXQ = smem_u32(st + L::XQ);
        for (int ks = 0; ks < DK / 16; ++ks)
          umma_bf16(tmem + L::COL_F, kdesc<128>(sXQ, ks), kdesc<128>(sXQ, ks), idesc_bf16(128, 64),
                    ks > 0 ? 1u : 0u);
        umma_commit(fmma);
      }
      if (!mbar_wait(fmma, fph)) fail();
      fph ^= 1;
      tc_fence_after();
      {
        float v[64];
        tmem_ld64(tmem + lane_off + L::COL_F, v);
        tmem_wait_ld();
        const float* gg = gt + L::G_G;
        const float* cfe = gt + L::G_CFE;
        // exp(g_x - g_i), i <= x: exp(g_x - g_end(J)) cfe_i for i in an earlier block J,
        // cfe_i / cfe_x inside the row's own block (exact exponentials if that ratio underflows)
        const int x = row & 63, I = x >> 4;
        const float gx = gg[x], cfx = cfe[x];
        const bool ratio_ok = cfx > 1e-30f;
        const float inv = ratio_ok ? __fdividef(1.f, cfx) : 0.f;
        float w[64];
        const float4* cf4 = reinterpret_cast<const float4*>(cfe);
#pragma unroll
        for (int J = 0; J < 4; ++J) {
          // row factor of block J: exp(g_x - g_end(J)) before the row's block, 1 / cf_x in it, 0 after
          const float f = J < I ? __expf(gx - gg[16 * J + 15]) : (J == I ? inv : 0.f);
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4) {
            const float4 c4 = cf4[4 * J + i4];
            const int i = 16 * J + 4 * i4;
            w[i] = f * c4.x * v[i];
            w[i + 1] = f * c4.y * v[i + 1];
            w[i + 2] = f * c4.z * v[i + 2];
            w[i + 3] = f * c4.w * v[i + 3];
          }
        }
        if (!ratio_ok) {  // exact exponentials inside the row's own block
#pragma unroll
          for (int J = 0; J < 4; ++J) {
            if (J == I) {
#pragma unroll
              for (int i = 0; i < 16; ++i) w[16 * J + i] = __expf(gx - gg[16 * J + i]) * v[16 * J + i];
            }
          }
        }
        if (quad < 2) {  // Gram row r = x: 1 / (eps + |x_r|^2) and column r of L^T
          float n = 0.f;
#pragma unroll
          for (int j = 0; j < 64; ++j) n = (j == x) ? v[j] : n;
          const int t = c * kC + x;
          const bool exists = t < a.T && pos + t >= a.shift;
          gt[L::G_INV + x] = exists ? 1.f / (a.eps + n) : 0.f;
          if (SOLVE) {  // row x of L: its diagonal block in fp32, the whole row in bf16
#pragma unroll
            for (int i = 0; i < 64; ++i) w[i] = (i < x) ? w[i] : 0.f;
            // diagonal block transposed: [block][column i][row], so a column is contiguous
            float* ld = reinterpret_cast<float*>(st + L::LT) + I * 256 + (x & 15);
#pragma unroll
            for (int J = 0; J < 4; ++J) {
              if (J == I) {
#pragma unroll
                for (int i = 0; i < 16; ++i) ld[16 * i] = w[16 * J + i];
              }
            }
            store_row64(st + L::LT + 8192, x, w);
          }
        } else {  // P row t = x: P~[t][r] = exp(g_t - g_r) q_t . x_r for r <= t
#pragma unroll
          for (int i = 0; i < 64; ++i) w[i] = (i <= x) ? w[i] : 0.f;
          store_row64(st + L::PT, x, w);
        }
      }
      // Q~ = diag(Gamma) Q in place (the product that read Q is complete)
#pragma unroll
      for (int k = 0; k < 4 * kSl; ++k) {
        const int idx = ftid + 128 * k;
        const int sl = idx >> 9, rem = idx & 511, t = rem >> 3;
        uint4* ptr = reinterpret_cast<uint4*>(st + L::XQ + sl * 16384 + 8192 + rem * 16);
        const uint4 in = *ptr;
        const __nv_bfloat162* pin = reinterpret_cast<const __nv_bfloat162*>(&in);
        const float fr = gt[L::G_GAM + t];
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 q2 = __bfloat1622float2(pin[e]);
          pk[e] = pack_bf16(q2.x * fr, q2.y * fr);
        }
        *ptr = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&fdone[s]);
    }
    if (slice == 0 && a.kprev_out && !*abort_flag && ftid < DK)
      a.kprev_out[(size_t)bh * DK + ftid] = a.k[(((size_t)b * a.T + (a.T - 1)) * a.H + h) * DK + ftid];
    if (slice == 0 && a.pos_out && !*abort_flag && ftid == 0)
      a.pos_out[bh] = (a.pos_in ? a.pos_in[bh] : 0) + a.T;
  } else {
    // ------------------------------------------------------------ back
    const int L_ = tid;             // TMEM lane of this thread (0..127)
    const int j = L_ & 63;          // value channel (in the slice) of this lane
    const bool solver = warp < 2;
    uint8_t* SA = sm + L::SA;
    uint8_t* DA = sm + L::DA;
    uint8_t* OST = sm + L::OST;
    // initial state S^T into TMEM (both halves)
#pragma unroll
    for (int pc = 0; pc < DK / 32; ++pc) {
      uint32_t r[32];
#pragma unroll
      for (int n = 0; n < 32; ++n)
        r[n] = __float_as_uint(a.S_in ? a.S_in[((size_t)bh * DK + 32 * pc + n) * a.dv + c0 + j] : 0.f);
      tmem_st32(tmem + lane_off + L::COL_S + 32 * pc, r);
    }
    tmem_wait_st();
    tc_fence_before();
    named_bar(2, 128);
    tc_fence_after();
    uint32_t bph = 0, tph = 0;
    int c = 0;
    for (; c < NC; ++c) {
      const int s = c % NST, p = c & 1;
      if (!mbar_wait(&fdone[s], (uint32_t)((c / NST) & 1))) fail();
      tc_fence_after();
      uint8_t* st = stage(s);
      const float* gt = reinterpret_cast<const float*>(st + L::GT);
      const uint32_t col_yo = L::COL_YO + 128 * p;
      {  // S0^T row -> bf16 operand row; Gamma_last S0 back into TMEM
        const float gC = gt[L::G_GAM + 63];
#pragma unroll
        for (int pc = 0; pc < DK / 32; ++pc) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + L::COL_S + 32 * pc, r);
          tmem_wait_ld();
          uint8_t* slab = SA + (pc >> 1) * 16384;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              pk[e] = pack_bf16(__uint_as_float(r[8 * m + 2 * e]), __uint_as_float(r[8 * m + 2 * e + 1]));
            *reinterpret_cast<uint4*>(slab + sw128(L_, 32 * (pc & 1) + 8 * m)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
#pragma unroll
          for (int n = 0; n < 32; ++n) r[n] = __float_as_uint(gC * __uint_as_float(r[n]));
          tmem_st32(tmem + lane_off + L::COL_S + 32 * pc, r);
        }
        tmem_wait_st();
      }
      fence_proxy_async();
      tc_fence_before();
      if (named_bar_any(2, 128, *abort_flag != 0)) break;
      tc_fence_after();
      if (tid == 0) {  // [(X S0)^T | (Q~ S0)^T] = [S0^T ; S0^T] [X ; Q~]^T
        const uint32_t sSA = smem_u32(SA), sXQ = smem_u32(st + L::XQ);
        for (int ks = 0; ks < DK / 16; ++ks)
          umma_bf16(tmem + col_yo, kdesc<128>(sSA, ks), kdesc<128>(sXQ, ks), idesc_bf16(128, 128),
                    ks > 0 ? 1u : 0u);
        umma_commit(&bmma[0]);
      }
      if (!mbar_wait(&bmma[0], bph)) fail();
      tc_fence_after();
      if (solver) {
        const float* bsl = reinterpret_cast<const float*>(st + L::BS);
        const float* inv = gt + L::G_INV;
        float acc[64];
        if (SOLVE) {
          uint32_t y[32];
          const float* gam = gt + L::G_GAM;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            tmem_ld32(tmem + lane_off + col_yo + 32 * hf, y);
            tmem_wait_ld();
#pragma unroll
            for (int n = 0; n < 32; ++n) {
              const int r = 32 * hf + n;
              const float vr = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(st + L::VS + sw128(r, j)));
              acc[r] = vr - gam[r] * __uint_as_float(y[n]);
            }
          }
          // forward substitution for this channel in 16-row blocks: inside a block
          // in registers with the fp32 diagonal block of L; the contributions of
          // finished blocks to all later rows accumulate in TMEM (E) by one MMA
          // [Delta^T ; Delta^T]_(block) L_(:, block)^T per block
          const float* ldiag = reinterpret_cast<const float*>(st + L::LT);
          const uint32_t sDA = smem_u32(DA), sLb = smem_u32(st + L::LT + 8192);
#pragma unroll
          for (int I = 0; I < 4; ++I) {
            if (I > 0) {  // E holds sum over the finished blocks
              if (!mbar_wait(tmma, tph)) fail();
              tph ^= 1;
              tc_fence_after();
              uint32_t e[16];
              tmem_ld16(tmem + lane_off + L::COL_E + 16 * I, e);
              tmem_wait_ld();
#pragma unroll
              for (int r = 0; r < 16; ++r) acc[16 * I + r] -= __uint_as_float(e[r]);
            }
#pragma unroll
            float eb[16];  // eta of the block's rows for this channel
#pragma unroll
            for (int r = 0; r < 16; ++r) eb[r] = bsl[(16 * I + r) * 64 + j] * inv[16 * I + r];
#pragma unroll
            for (int i = 0; i < 16; ++i) {  // right-looking: Delta_i, then its share of the later rows
              const float d = eb[i] * acc[16 * I + i];
              acc[16 * I + i] = d;
              const float* col = ldiag + I * 256 + 16 * i;  // L[16 I + r][16 I + i], r = 0..15
#pragma unroll
              for (int r4 = (i + 1) >> 2; r4 < 4; ++r4) {
                const float4 l4 = *reinterpret_cast<const float4*>(col + 4 * r4);
                const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  if (4 * r4 + e > i) acc[16 * I + 4 * r4 + e] = fmaf(-lv[e], d, acc[16 * I + 4 * r4 + e]);
              }
            }
            {  // this block of Delta^T (bf16) in both halves of the operand
              uint32_t pk[8];
#pragma unroll
              for (int e2 = 0; e2 < 8; ++e2) pk[e2] = pack_bf16(acc[16 * I + 2 * e2], acc[16 * I + 2 * e2 + 1]);
#pragma unroll
              for (int hlf = 0; hlf < 2; ++hlf) {
                const uint4 u = make_uint4(pk[4 * hlf], pk[4 * hlf + 1], pk[4 * hlf + 2], pk[4 * hlf + 3]);
                *reinterpret_cast<uint4*>(DA + sw128(L_, 16 * I + 8 * hlf)) = u;
                *reinterpret_cast<uint4*>(DA + sw128(L_ + 64, 16 * I + 8 * hlf)) = u;
              }
            }
            if (I < 3) {
              fence_proxy_async();
              tc_fence_before();
              named_bar(4, 64);
              tc_fence_after();
              if (tid == 0) {
                umma_bf16(tmem + L::COL_E, kdesc<128>(sDA, I), kdesc<64>(sLb, I), idesc_bf16(128, 64),
                          I > 0 ? 1u : 0u);
                umma_commit(tmma);
              }
            }
          }
        } else {  // additive write: Delta = eta (.) V
#pragma unroll
          for (int r = 0; r < 64; ++r) {
            const float vr = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(st + L::VS + sw128(r, j)));
            acc[r] = bsl[r * 64 + j] * inv[r] * vr;
          }
        }
        if (!SOLVE) {
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) pk[e] = pack_bf16(acc[8 * m + 2 * e], acc[8 * m + 2 * e + 1]);
            const uint4 u = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(DA + sw128(L_, 8 * m)) = u;
            *reinterpret_cast<uint4*>(DA + sw128(L_ + 64, 8 * m)) = u;
          }
        }
      } else {  // X~ rows in place of X (the product that read X is complete)
        const float* dec = gt + L::G_DEC;
#pragma unroll
        for (int k = 0; k < 8 * kSl; ++k) {
          const int idx = (L_ - 64) + 64 * k;
          const int sl = idx >> 9, rem = idx & 511, r = rem >> 3;
          uint4* ptr = reinterpret_cast<uint4*>(st + L::XQ + sl * 16384 + rem * 16);
          const uint4 in = *ptr;
          const __nv_bfloat162* pin = reinterpret_cast<const __nv_bfloat162*>(&in);
          const float fr = dec[r];
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x2 = __bfloat1622float2(pin[e]);
            pk[e] = pack_bf16(x2.x * fr, x2.y * fr);
          }
          *ptr = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      named_bar(2, 128);
      tc_fence_after();
      if (tid == 0) {
        const uint32_t sDA = smem_u32(DA), sPT = smem_u32(st + L::PT), sXQ = smem_u32(st + L::XQ);
        // O^T += [Delta^T ; Delta^T] P~^T
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem + col_yo + 64, kdesc<128>(sDA, ks), kdesc<64>(sPT, ks), idesc_bf16(128, 64), 1u);
        // S^T += [Delta^T ; Delta^T] X~  (X~ MN-major over the d_k slabs)
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem + L::COL_S, kdesc<128>(sDA, ks), sdesc_mn128_wide(sXQ + ks * 2048, 16384),
                    idesc_bf16(128, DK, false, true), 1u);
        umma_commit(&bmma[1]);
      }
      if (!mbar_wait(&bmma[1], bph)) fail();
      bph ^= 1;
      tc_fence_after();
      if (tid == 0 && c + NST < NC) load_chunk(c + NST);  // nothing reads this stage any more
      if (!solver) {  // output tile: O[t][j] from the channel-major accumulator
        uint32_t o[2][32];
        tmem_ld32(tmem + lane_off + col_yo + 64, o[0]);
        tmem_ld32(tmem + lane_off + col_yo + 96, o[1]);
        tmem_wait_ld();
        if (tid == 64) bulk_wait_read0();  // the previous tile has left the staging buffer
        named_bar(3, 64);
        const bool even = (j & 1) == 0;
#pragma unroll
        for (int tp = 0; tp < 32; ++tp) {
          const float a0 = __uint_as_float(o[tp >> 4][(2 * tp) & 31]);
          const float a1 = __uint_as_float(o[tp >> 4][(2 * tp + 1) & 31]);
          const float recv = __shfl_xor_sync(0xffffffffu, even ? a1 : a0, 1);
          if (even)
            *reinterpret_cast<uint32_t*>(OST + sw128(2 * tp, j)) = pack_bf16(a0, recv);
          else
            *reinterpret_cast<uint32_t*>(OST + sw128(2 * tp + 1, j - 1)) = pack_bf16(recv, a1);
        }
        fence_proxy_async();
        named_bar(3, 64);
        if (tid == 64) {
          tma_store_4d(&tm_o, OST, c0, h, c * kC, b);
          bulk_commit();
        }
      }
    }
    if (tid == 64) bulk_wait0();
    if (tid == 0 && *abort_flag) {  // drain the loads still in flight
      for (int cc = c; cc < NC && cc < c + NST; ++cc) mbar_wait(&full[cc % NST], (uint32_t)((cc / NST) & 1));
    }
    if (solver && !*abort_flag && a.S_out) {
#pragma unroll
      for (int pc = 0; pc < DK / 32; ++pc) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + L::COL_S + 32 * pc, r);
        tmem_wait_ld();
#pragma unroll
        for (int n = 0; n < 32; ++n)
          a.S_out[((size_t)bh * DK + 32 * pc + n) * a.dv + c0 + j] = __uint_as_float(r[n]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::NCOLS);
  }
}

template <int DK, bool SOLVE>
int launch_f2_t(const FwdArgs& fa, const F2Args& ta) {
  CUtensorMap mk, mq, mv, mb, mo;
  if (!make_map(&mk, fa.k, fa.B, fa.T, fa.H, DK, 64) || !make_map(&mq, fa.q, fa.B, fa.T, fa.H, DK, 64) ||
      !make_map(&mv, fa.v, fa.B, fa.T, fa.H, fa.dv, 64) || !make_map(&mo, fa.o, fa.B, fa.T, fa.H, fa.dv, 64) ||
      !make_map_f32(&mb, fa.beta, fa.B, fa.T, fa.H, fa.dv, 64, 64))
    return FALCON_ERR_CUDA;
  auto k = tc_f2_kernel<DK, SOLVE>;
  const size_t smem = F2Smem<DK>::TOTAL;
  if (!set_smem_limit(reinterpret_cast<const void*>(k), smem)) return FALCON_ERR_CUDA;
  dim3 grid(fa.B * fa.H, fa.dv / 64);
  // the call's status word starts clear; a bounded wait that runs out sets it
  if (cudaMemsetAsync(ta.status, 0, sizeof(uint32_t), fa.stream) != cudaSuccess) return FALCON_ERR_CUDA;
  record_event(fa, 0);
  k<<<grid, 256, smem, fa.stream>>>(mk, mq, mv, mb, mo, ta);
  record_event(fa, 1);
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace

bool tc_f2_supported(const FwdArgs& a) {
  if (a.variant != FALCON_2 && a.variant != FALCON_2A) return false;
  if (a.dtype != FALCON_BF16 || a.chunk != 64 || a.T < 1) return false;
  return a.dk == a.dv && (a.dk == 64 || a.dk == 128);
}

int launch_tc_f2(const FwdArgs& fa) {
  F2Args ta;
  ta.B = fa.B; ta.T = fa.T; ta.H = fa.H; ta.dv = fa.dv; ta.NC = (fa.T + kC - 1) / kC;
  ta.shift = fa.shift;
  ta.eps = fa.eps; ta.eps_gamma = fa.eps_gamma;
  ta.lam = fa.lam; ta.pos_in = fa.pos_in;
  ta.kprev_in = reinterpret_cast<const __nv_bfloat16*>(fa.kprev_in);
  ta.S_in = fa.S_in;
  ta.k = reinterpret_cast<const __nv_bfloat16*>(fa.k);
  ta.S_out = fa.S_out;
  ta.kprev_out = reinterpret_cast<__nv_bfloat16*>(fa.kprev_out);
  ta.pos_out = fa.pos_out;
  ta.status = reinterpret_cast<uint32_t*>(fa.ws);
  const bool solve = fa.variant == FALCON_2;
  if (fa.dk == 64) return solve ? launch_f2_t<64, true>(fa, ta) : launch_f2_t<64, false>(fa, ta);
  return solve ? launch_f2_t<128, true>(fa, ta) : launch_f2_t<128, false>(fa, ta);
}

}  // namespace falcon
