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
//   O    = diag(Gamma) Q S0 + (Q X^T (.) M') V
//   S1   = Gamma_last S0 + (diag(m) X)^T V,     m_kappa = M'_{63,kappa}
// (in-chunk cumulative log-decay g, Gamma = exp(g), clamped decay
// [JC 数学上的稳定阀门:正衰减钳制]).  The recurrence for M' only multiplies by
// gamma <= 1, so no decay ratio is ever formed.
//
// One CTA per (b, h), warp-specialised like the Falcon-1 sequential kernel:
//   warp 8      producer: TMA of the 80 key rows, 80 value rows and 64 query rows
//   warps 4..7  front, even chunks, and warps 9..12 front, odd chunks (each up
//               to NST chunks ahead of the back): window statistics, P^T = X Q^T
//               (keys in TMEM lanes; one TMEM block per front), M' by the
//               recurrence along t, P~^T and X~ = diag(m) X in place
//   warps 0..3  back: [0 ; Oa] = [0 ; Q] S0 and [D2 ; Ob] = [X~ | P~^T]^T V in one
//               go, S1 = Gamma_last S0 + D2, O = diag(Gamma) Oa + Ob
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
};

struct F3aSmem {
  static constexpr int NST = 4;
  // X (80 key rows, then X~) | P~^T (80 rows) | zero rows | Q | V (80 rows) | gates
  static constexpr size_t XO = 0, PO = 10240, ZO = 20480, QO = 28672, VO = 36864, GO = 47104;
  static constexpr size_t STAGE = 49152;
  static constexpr size_t SB = NST * STAGE;         // S rows (MN-major B)
  static constexpr size_t OST = SB + 8192;          // two output staging tiles
  static constexpr size_t BAR = OST + 2 * 8192;
  static constexpr size_t MISC = BAR + 128;
  static constexpr size_t TOTAL = MISC + 16 + 1024;
  static constexpr uint32_t TX = 2 * 10240 + 8192;
  static_assert(TOTAL <= 232448, "shared memory budget");
  // gates (fp32 offsets in GO): key energy, key existence, c, gamma, Gamma, g, warp sums
  static constexpr int G_NRM = 0, G_EX = 80, G_C = 160, G_GMA = 224, G_GAM = 288, G_G = 352, G_WS = 416;
  static_assert(GO + (G_WS + 2) * 4 <= STAGE, "gates fit the stage");
  // TMEM: P^T of the even-chunk front (keys in lanes) | [0 ; Oa] | [D2 ; Ob] |
  // P^T of the odd-chunk front
  static constexpr uint32_t COL_PT = 0, COL_B1 = 64, COL_B2 = 128, COL_PT1 = 192, NCOLS = 256;
  static constexpr int kThreads = 416;  // 13 warps
};

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

__global__ void __launch_bounds__(F3aSmem::kThreads, 1)
    tc_f3a_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k80,
                  const __grid_constant__ CUtensorMap tm_v80, const __grid_constant__ CUtensorMap tm_o,
                  F3aArgs a) {
  using L = F3aSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  constexpr int NST = L::NST;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* full = bars;              // [NST]
  uint64_t* empty = bars + NST;       // [NST]
  uint64_t* fdone = bars + 2 * NST;   // [NST]
  uint64_t* fmma = bars + 3 * NST;    // [2]: P^T of front 0 / 1 done
  uint64_t* bmma = fmma + 2;          // both back products done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.x;
  const int b = bh / a.H, h = bh % a.H;
  const int NC = a.NC, W = a.W;
  auto stage = [&](int s) { return sm + s * L::STAGE; };
  auto fail = [&]() {
    *abort_flag = 1;
    atomicExch(a.status, kStatusTimeout);
  };

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&fdone[i], 128);
    }
    mbar_init(&fmma[0], 1);
    mbar_init(&fmma[1], 1);
    mbar_init(bmma, 1);
    fence_mbar_init();
  }
  for (int i = tid; i < NST * 512; i += L::kThreads)  // the zero rows of [0 ; Q]
    *reinterpret_cast<uint4*>(stage(i >> 9) + L::ZO + (i & 511) * 16) = make_uint4(0, 0, 0, 0);
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
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int c = 0;
      for (; c < NC; ++c) {
        const int s = c % NST;
        if (c >= NST && !mbar_wait(&empty[s], (uint32_t)(((c - NST) / NST) & 1))) { fail(); break; }
        if (*abort_flag) break;
        uint8_t* st = stage(s);
        const int j0 = c * kC - W + 1;  // first pair of the chunk's keys
        mbar_arrive_expect_tx(&full[s], L::TX);
        tma_load_4d(st + L::XO, &tm_k80, &full[s], 0, h, j0 - a.shift, b);
        tma_load_4d(st + L::VO, &tm_v80, &full[s], 0, h, j0, b);
        tma_load_4d(st + L::QO, &tm_q, &full[s], 0, h, c * kC, b);
      }
      if (*abort_flag) {  // drain the loads still in flight
        for (int cc = (c > NST ? c - NST : 0); cc < c; ++cc)
          mbar_wait(&full[cc % NST], (uint32_t)((cc / NST) & 1));
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ front
    // fg = 0: warps 4..7, chunks 0, 2, 4, ...; fg = 1: warps 9..12, chunks 1, 3, ...
    const int fg = warp >= 9 ? 1 : 0;
    const int ftid = tid - (fg ? 288 : 128);
    const int fbar = fg ? 5 : 1;  // named barrier of this front
    const uint32_t col_pt = fg ? L::COL_PT1 : L::COL_PT;
    uint64_t* fm = &fmma[fg];
    uint32_t fph = 0;
    // gate inputs of step c * 64 + ftid, loaded one chunk ahead
    auto gate_in = [&](int c, float& lam, float& beta) {
      const int tg = c * kC + ftid;
      const bool ok = ftid < 64 && c < NC && tg < a.T;
      const size_t gi = ((size_t)b * a.T + (ok ? tg : 0)) * a.H + h;
      lam = ok ? a.lam[gi] : 0.f;
      beta = ok ? a.beta[gi] : 0.f;
    };
    float lam_n, beta_n;
    gate_in(fg, lam_n, beta_n);
    for (int c = fg; c < NC; c += 2) {
      const int s = c % NST;
      const int t0 = c * kC, j0 = t0 - W + 1;
      const bool step_ok = ftid < 64 && t0 + ftid < a.T;
      const float lam_c = lam_n, beta = beta_n;
      gate_in(c + 2, lam_n, beta_n);
      const float ell = step_ok ? clamped_log_decay(lam_c, a.eps_gamma) : 0.f;
      if (!mbar_wait(&full[s], (uint32_t)((c / NST) & 1))) fail();
      uint8_t* st = stage(s);
      float* gt = reinterpret_cast<float*>(st + L::GO);
      if (j0 < 1) {  // keys before the sequence: carried key and window ring
        for (int idx = ftid; idx < W * 64; idx += 128) {
          const int kap = idx >> 6, col = idx & 63, j = j0 + kap;
          if (j < a.shift) {
            *reinterpret_cast<__nv_bfloat16*>(st + L::XO + sw128(kap, col)) = pair_x(a, b, h, j, col, pos);
            if (j < 0)
              *reinterpret_cast<__nv_bfloat16*>(st + L::VO + sw128(kap, col)) = pair_v(a, b, h, j, col, pos);
          }
        }
      }
      named_bar(fbar, 128);
      if (ftid < kKeys) {  // key energy and existence of pair j0 + kappa
        const int j = j0 + ftid;
        float n = 0.f;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint4 raw = *reinterpret_cast<const uint4*>(st + L::XO + sw128(ftid, 8 * m));
          const __nv_bfloat162* px = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x2 = __bfloat1622float2(px[e]);
            n = fmaf(x2.x, x2.x, n);
            n = fmaf(x2.y, x2.y, n);
          }
        }
        gt[L::G_NRM + ftid] = n;
        gt[L::G_EX + ftid] = (pos + j >= a.shift && j < a.T) ? 1.f : 0.f;
      }
      float g = ell;  // inclusive prefix sum of the log-decay over the chunk
      if (ftid < 64) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float n = __shfl_up_sync(0xffffffffu, g, o);
          if (lane >= o) g += n;
        }
        if (lane == 31) gt[L::G_WS + (ftid >> 5)] = g;
      }
      named_bar(fbar, 128);
      if (ftid < 64) {  // step t = ftid: window statistics and decays
        if ((ftid >> 5) == 1) g += gt[L::G_WS];
        float n = 0.f, e = 0.f;
        for (int q = 0; q < W; ++q) {
          const float ex = gt[L::G_EX + ftid + q];
          n += ex;
          e += ex * gt[L::G_NRM + ftid + q];
        }
        const float cs = (step_ok && n > 0.f) ? beta / (a.eps + e / n) / n : 0.f;
        gt[L::G_C + ftid] = cs;
        gt[L::G_GMA + ftid] = __expf(ell);
        gt[L::G_GAM + ftid] = __expf(g);
        gt[L::G_G + ftid] = g;
      }
      fence_proxy_async();
      tc_fence_before();
      if (named_bar_any(fbar, 128, *abort_flag != 0)) break;
      tc_fence_after();
      if (ftid == 0) {  // P^T = X Q^T over 128 A rows (rows >= 80 are not read back)
        const uint32_t sX = smem_u32(st + L::XO), sQ = smem_u32(st + L::QO);
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem + col_pt, kdesc<128>(sX, ks), kdesc<64>(sQ, ks), idesc_bf16(128, 64),
                    ks > 0 ? 1u : 0u);
        umma_commit(fm);
      }
      if (!mbar_wait(fm, fph)) fail();
      fph ^= 1;
      tc_fence_after();
      if (quad < 3) {  // keys kappa = 32 quad + lane < 80
        const int kap = 32 * quad + lane;
        float pv[64];
        tmem_ld64(tmem + lane_off + col_pt, pv);
        tmem_wait_ld();
        if (kap < kKeys) {
          const float* cs = gt + L::G_C;
          const float* gm = gt + L::G_GMA;
          const bool kex = gt[L::G_EX + kap] != 0.f;  // a pair that does not exist writes nothing
          float mcur = 0.f;
#pragma unroll
          for (int t = 0; t < 64; ++t) {
            const bool in_win = kex && t <= kap && kap <= t + W - 1;
            mcur = fmaf(gm[t], mcur, in_win ? cs[t] : 0.f);
            pv[t] *= mcur;
          }
          store_row64(st + L::PO, kap, pv);
          // X~ row kappa = m_kappa x_kappa in place
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            uint4* ptr = reinterpret_cast<uint4*>(st + L::XO + sw128(kap, 8 * m));
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
      mbar_arrive(&fdone[s]);
    }
    if (!*abort_flag && fg == 0) {  // carry: last key, the last W - 1 pairs, position
      if (a.kprev_out && ftid < 64)
        a.kprev_out[(size_t)bh * 64 + ftid] = a.k[(((size_t)b * a.T + (a.T - 1)) * a.H + h) * 64 + ftid];
      const int Wr = W - 1;
      for (int idx = ftid; idx < Wr * 64; idx += 128) {
        const int i = idx >> 6, col = idx & 63;
        const int64_t p = pos + a.T - Wr + i;  // global pair index
        const int j = (int)(p - pos);
        const int slot = (int)(((p % Wr) + Wr) % Wr);
        const bool ok = p >= a.shift;  // slots of pairs that do not exist hold zeros
        const __nv_bfloat16 z = __float2bfloat16_rn(0.f);
        if (a.winx_out)
          a.winx_out[((size_t)bh * Wr + slot) * 64 + col] = ok ? pair_x(a, b, h, j, col, pos) : z;
        if (a.winv_out)
          a.winv_out[((size_t)bh * Wr + slot) * 64 + col] = ok ? pair_v(a, b, h, j, col, pos) : z;
      }
      if (a.pos_out && ftid == 0) a.pos_out[bh] = pos + a.T;
    }
  } else {
    // ------------------------------------------------------------ back
    // warps 0, 1: S rows 32 w + lane (lanes 0..63 of the stacked products);
    // warps 2, 3: output rows 32 (w - 2) + lane (lanes 64..127)
    uint8_t* SB = sm + L::SB;
    const uint32_t sS = smem_u32(SB);
    const bool srow = warp < 2;
    const int r = 32 * (warp & 1) + lane;
    float sreg[64];
#pragma unroll
    for (int n = 0; n < 64; ++n) sreg[n] = 0.f;
    if (srow && a.S_in) {
      const float* src = a.S_in + ((size_t)bh * 64 + r) * 64;
#pragma unroll
      for (int n = 0; n < 64; n += 4) {
        const float4 v4 = *reinterpret_cast<const float4*>(src + n);
        sreg[n] = v4.x; sreg[n + 1] = v4.y; sreg[n + 2] = v4.z; sreg[n + 3] = v4.w;
      }
    }
    if (srow) store_row64(SB, r, sreg);
    fence_proxy_async();
    named_bar(2, 128);
    uint32_t bph = 0;
    for (int c = 0; c < NC; ++c) {
      const int s = c % NST;
      if (!mbar_wait(&fdone[s], (uint32_t)((c / NST) & 1))) fail();
      tc_fence_after();
      uint8_t* st = stage(s);
      if (named_bar_any(2, 128, *abort_flag != 0)) break;
      const float* gt = reinterpret_cast<const float*>(st + L::GO);
      const float gfac = srow ? gt[L::G_GAM + 63] : gt[L::G_GAM + r];
      if (tid == 0) {
        // [0 ; Oa] = [0 ; Q] S0
        const uint32_t sA1 = smem_u32(st + L::ZO);
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem + L::COL_B1, kdesc<128>(sA1, ks), mndesc(sS, ks), idesc_bf16(128, 64, false, true),
                    ks > 0 ? 1u : 0u);
        // [D2 ; Ob] = [X~ | P~^T]^T V, A MN-major over two 80-row atoms, K = 80 keys
        const uint32_t sA2 = smem_u32(st + L::XO), sV = smem_u32(st + L::VO);
        for (int ks = 0; ks < kKeys / 16; ++ks)
          umma_bf16(tmem + L::COL_B2, sdesc_mn128_wide(sA2 + ks * 2048, 10240), mndesc(sV, ks),
                    idesc_bf16(128, 64, true, true), ks > 0 ? 1u : 0u);
        umma_commit(bmma);
      }
      uint8_t* Ost = sm + L::OST + (c & 1) * 8192;
      if (!mbar_wait(bmma, bph)) fail();
      bph ^= 1;
      tc_fence_after();
      if (tid == 0) mbar_arrive(&empty[s]);  // nothing reads this stage any more
      if (srow) {  // S1 = Gamma_last S0 + D2
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t d2[32];
          tmem_ld32(tmem + lane_off + L::COL_B2 + 32 * hf, d2);
          tmem_wait_ld();
#pragma unroll
          for (int n = 0; n < 32; ++n) sreg[32 * hf + n] = gfac * sreg[32 * hf + n] + __uint_as_float(d2[n]);
        }
        store_row64(SB, r, sreg);
      } else {  // O = diag(Gamma) Oa + Ob
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t oa[32], ob[32];
          tmem_ld32(tmem + lane_off + L::COL_B1 + 32 * hf, oa);
          tmem_ld32(tmem + lane_off + L::COL_B2 + 32 * hf, ob);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int n = 8 * j + 2 * e;
              pk[e] = pack_bf16(gfac * __uint_as_float(oa[n]) + __uint_as_float(ob[n]),
                                gfac * __uint_as_float(oa[n + 1]) + __uint_as_float(ob[n + 1]));
            }
            *reinterpret_cast<uint4*>(Ost + sw128(r, 32 * hf + 8 * j)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      named_bar(2, 128);
      tc_fence_after();
      if (tid == 0) {
        tma_store_4d(&tm_o, Ost, 0, h, c * kC, b);
        bulk_commit();
        bulk_wait_read1();  // the tile stored one chunk ago has left its buffer
      }
    }
    if (tid == 0) bulk_wait0();
    if (!*abort_flag && srow && a.S_out) {
      float* dst = a.S_out + ((size_t)bh * 64 + r) * 64;
#pragma unroll
      for (int n = 0; n < 64; n += 4)
        *reinterpret_cast<float4*>(dst + n) = make_float4(sreg[n], sreg[n + 1], sreg[n + 2], sreg[n + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::NCOLS);
  }
}

}  // namespace

bool tc_f3a_supported(const FwdArgs& a) {
  if (a.variant != FALCON_3A || a.dtype != FALCON_BF16 || a.chunk != 64 || a.T < 1) return false;
  return a.dk == 64 && a.dv == 64 && a.W >= 2 && a.W <= 16;
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
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, fa.q, fa.B, fa.T, fa.H, 64, 64) || !make_map(&mk, fa.k, fa.B, fa.T, fa.H, 64, kKeys) ||
      !make_map(&mv, fa.v, fa.B, fa.T, fa.H, 64, kKeys) || !make_map(&mo, fa.o, fa.B, fa.T, fa.H, 64, 64))
    return FALCON_ERR_CUDA;
  auto k = tc_f3a_kernel;
  const size_t smem = F3aSmem::TOTAL;
  if (!set_smem_limit(reinterpret_cast<const void*>(k), smem)) return FALCON_ERR_CUDA;
  // the call's status word starts clear; a bounded wait that runs out sets it
  if (cudaMemsetAsync(ta.status, 0, sizeof(uint32_t), fa.stream) != cudaSuccess) return FALCON_ERR_CUDA;
  record_event(fa, 0);
  k<<<fa.B * fa.H, F3aSmem::kThreads, smem, fa.stream>>>(mq, mk, mv, mo, ta);
  record_event(fa, 1);
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace falcon
