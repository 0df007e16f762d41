// Backward of the Falcon forward step by step for a window of pairs:
// Falcon-3 and 3A at any window W the shared memory holds, and every
// one-pair variant (W = 1) at d = 128; d_k = d_v = D in {32, 64, 128}, bf16 or
// fp32 inputs, fp32 arithmetic.
//
// The pages give the forward only [FW Falcon 家族; JC Falcon家族六个变体各管一段];
// the gradient is the chain rule through the step written per t, with the
// window's pairs p = t - a (a = 0 .. W-1), m_a = 1 when the pair exists,
//   n = sum m_a, e = sum m_a |x_a|^2 / max(n, 1), eta = beta / (eps + e)
//   (zero when n = 0; a dv-vector for Falcon-2/2A), c_a = m_a eta / max(n, 1),
//   Z = gamma S_{t-1},  r_a = v_a - Z^T x_a (additive: v_a),  delta_a = c_a (.) r_a,
//   S_t = Z + sum_a x_a delta_a^T,  o_t = S_t^T q_t.
// Going back in time with dS (the gradient of S_t):
//   dS += q do^T;  dq = S_t do;
//   dd_a = dS^T x_a;  dc_a = r_a (.) dd_a;  regression: dr_a = c_a (.) dd_a,
//   dv_a += dr_a, dx_a += dS delta_a - gamma S_{t-1} dr_a; additive:
//   dv_a += c_a (.) dd_a, dx_a += dS delta_a;
//   deta = sum_a m_a dc_a / max(n, 1) (summed over channels for a scalar
//   eta), dbeta = deta / (eps + e), de = -<deta, eta> / (eps + e),
//   dx_a += 2 de m_a x_a / max(n, 1);
//   dZ = dS - sum_a x_a dr_a^T (additive: dS), dgamma = <dZ, S_{t-1}>,
//   dlambda = -dgamma where the clamp passes it, dS_{t-1} = gamma dZ.
//
// Every column j of S runs its own recurrence (r_a, delta_a, dd_a and dr_a
// at column j read only column j), so the work splits by columns: a CTA of
// four warps takes 16 columns of one (b, h), a warp four of them, a lane one
// column and every eighth row.  Sums over rows are shuffles across the eight
// lanes of a column; the forward needs nothing else, and each warp keeps its
// own ring of the window's pairs, so the forward steps run without a block
// barrier.  What the backward sums over columns -- dx_a (a d_k vector per
// pair and step), dq, dgamma and the eta gradient -- is linear, so each CTA
// sums its 16 columns (shuffles within the warp, then the four warps through
// shared memory) and writes the per-step partial sums; a second kernel adds
// the column groups, gathers each pair's key gradient over the W steps that
// read the pair, and applies the key-norm term and the gates' gradients.
// dv, the state gradient and the per-channel beta gradient stay per column.
//
// A forward pass keeps the state at every 64-step block start in the
// workspace; then, block by block from the end, the block's states are
// recomputed into the workspace and its steps reversed.

#include "common.cuh"

namespace falcon {

namespace {

constexpr int kBW = 64;   // steps per recomputed block
constexpr int kCPC = 16;  // state columns a CTA takes
constexpr int kNT = 128;  // four warps, four columns each
constexpr int kNW = kNT / 32;

template <int D>
struct WinCfg {
  static constexpr int EPT = D / 8;     // rows a lane holds (every eighth)
  static constexpr int VPL = D / 32;    // elements of a D-vector per lane
  static constexpr int NCG = D / kCPC;  // column groups of a head
};

// Per-step partial sums of a column group: dx_a for the W window positions
// [W][D], dq [D], the eta-gradient sum and dgamma.
__host__ __device__ inline int win_part_floats(int D, int W) { return (W * D + D + 2 + 3) & ~3; }

// Shared-memory layout in floats.  Each warp has its own forward and
// backward ring of W + 2 pairs (the step's window, the pair written a step
// ahead, one spare): keys [W+2][D], its four columns' values [W+2][4],
// |x|^2 and existence [W+2]; the backward ring also gathers the four
// columns' value gradients [W+2][4].  Then the per-warp partial sums of a
// backward step.
struct WinLayout {
  int ring;                                // floats of one warp's rings
  int fx, fv, fe, fm, bx, bv, be, bm, gv;  // offsets inside a warp's rings
  int part;                                // [kNW][win_part_floats]
  int total;
};

__host__ __device__ inline WinLayout win_layout(int D, int W) {
  WinLayout L;
  const int R = W + 2;
  int o = 0;
  auto take = [&](int n) { const int at = o; o += (n + 3) & ~3; return at; };
  L.fx = take(R * D); L.fv = take(R * 4); L.fe = take(R); L.fm = take(R);
  L.bx = take(R * D); L.bv = take(R * 4); L.be = take(R); L.bm = take(R); L.gv = take(R * 4);
  L.ring = o;
  o = kNW * L.ring;
  L.part = take(kNW * win_part_floats(D, W));
  L.total = o;
  return L;
}

struct WinArgs {
  int B, T, H, W;
  float eps, eps_gamma;
  int shift;
  const void* q;
  const void* k;
  const void* v;
  const void* dO;
  const float* beta;
  const float* lam;
  const float* S_in;
  const void* kprev_in;
  const void* winx_in;
  const void* winv_in;
  const int64_t* pos_in;
  const float* dS_final;
  void* dq;
  void* dk;
  void* dv;
  float* dbeta;
  float* dlam;
  float* dS_in;
  void* dk_prev;
  void* dwin_x;
  void* dwin_v;
  float* st;    // per (b, h, column group): block-start states [NB][kNT][EPT], block states [kBW + 1][kNT][EPT]
  float* part;  // per (b, h, t, column group): win_part_floats partial sums
  float* scal;  // per (b, h, t): 1 / (eps + e), eta (1 per channel), 1 / max(n, 1), has a pair
};

template <typename Tin>
__device__ __forceinline__ float ldw(const void* p, size_t i) {
  return to_f32(reinterpret_cast<const Tin*>(p)[i]);
}
template <typename Tin>
__device__ __forceinline__ void stw(void* p, size_t i, float x) {
  reinterpret_cast<Tin*>(p)[i] = from_f32<Tin>(x);
}

__device__ __forceinline__ float warp_total(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// sum over the eight lanes of a column (lane bits 0..2)
__device__ __forceinline__ float col_total(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  return v;
}
// Sum of v[m] over the four columns of the warp (lane bits 3, 4), scattered:
// lane (jj, g) ends with the totals of elements jj N/4 .. jj N/4 + N/4 - 1 in
// v[0 .. N/4 - 1].  Each level hands the half of the values that the partner
// keeps and adds the half it receives.
template <int N>
__device__ __forceinline__ void quad_reduce_scatter(float (&v)[N], int lane) {
  static_assert(N >= 4 && (N & 3) == 0, "four lanes share the rows");
#pragma unroll
  for (int n = N, off = 16; n > N / 4; n >>= 1, off >>= 1) {
    const int half = n >> 1;
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
}

template <typename Tin, int D, bool ADD, bool PERCH>
__global__ void __launch_bounds__(kNT) falcon_bwd_win_kernel(WinArgs a) {
  using C = WinCfg<D>;
  constexpr int EPT = C::EPT, VPL = C::VPL, NCG = C::NCG;
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  const int W = a.W, R = W + 2;
  const WinLayout L = win_layout(D, W);
  const int KP = win_part_floats(D, W);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int jj = lane >> 3, g = lane & 7;  // the lane's column of the warp's four, its row group
  const int bh = blockIdx.x / NCG, cg = blockIdx.x % NCG;
  const int j = kCPC * cg + 4 * warp + jj;  // state column
  const int b = bh / a.H, h = bh % a.H;
  const int T = a.T, NB = (T + kBW - 1) / kBW;
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  float* ring = sm + warp * L.ring;
  float *fxr = ring + L.fx, *fvr = ring + L.fv, *fer = ring + L.fe, *fmr = ring + L.fm;
  float *bxr = ring + L.bx, *bvr = ring + L.bv, *ber = ring + L.be, *bmr = ring + L.bm, *gvr = ring + L.gv;
  float* pall = sm + L.part;          // [kNW][KP]
  float* pw = pall + warp * KP;       // this warp's partial sums
  float* stw_base = a.st + (size_t)blockIdx.x * (NB + kBW + 1) * kNT * EPT;
  auto st_at = [&](int k, int m) { return stw_base + ((size_t)k * EPT + m) * kNT + tid; };  // k: block or NB + step
  auto row = [&](int m) { return g + 8 * m; };
  auto gidx = [&](int t) { return ((size_t)b * T + t) * a.H + h; };
  auto slot = [&](int p) { const int s = p % R; return s < 0 ? s + R : s; };
  // slot of the carried window ring (W > 1) that holds pair p < 0 of this call
  auto ring_slot = [&](int p) {
    const int s = (int)((pos + p) % (W - 1));
    return s < 0 ? s + W - 1 : s;
  };

  // ---- pairs: the warp fetches pair p (key, its four columns' values) into
  // registers, then puts it into one of its rings; a pair that does not exist
  // (or lies outside the call) reads as zeros
  auto fetch_pair = [&](int p, float (&X)[VPL], float& V, bool& ex) {
    ex = pos + p >= a.shift && p < T && p >= -(W - 1);
    size_t kr = 0, vr = 0;
    int src = 0;  // 0: none, 1: this call's k and v, 2: the carried key, 3: the carried ring
    if (ex) {
      if (p >= 0) {
        const int kt = p - a.shift;
        src = kt >= 0 ? 1 : (a.kprev_in ? 2 : 4);
        kr = kt >= 0 ? gidx(kt) * D : (size_t)bh * D;
        vr = gidx(p) * D;
      } else if (a.winx_in) {  // pos + p >= shift >= 0 here
        src = 3;
        kr = vr = ((size_t)bh * (W - 1) + ring_slot(p)) * D;
      }
    }
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      const int i = lane + 32 * u;
      X[u] = src == 1 ? ldw<Tin>(a.k, kr + i) : src == 2 ? ldw<Tin>(a.kprev_in, kr + i)
                                              : src == 3 ? ldw<Tin>(a.winx_in, kr + i) : 0.f;
    }
    const int c = kCPC * cg + 4 * warp + (lane & 3);
    V = 0.f;
    if (lane < 4 && (src == 1 || src == 2 || src == 4)) V = ldw<Tin>(a.v, vr + c);
    else if (lane < 4 && src == 3) V = ldw<Tin>(a.winv_in, vr + c);
  };
  auto put_pair = [&](int p, const float (&X)[VPL], float V, bool ex, float* xr, float* vr, float* er,
                      float* mr) {
    const int s = slot(p);
    float en = 0.f;
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      xr[s * D + lane + 32 * u] = X[u];
      en = fmaf(X[u], X[u], en);
    }
    if (lane < 4) vr[s * 4 + lane] = V;
    en = warp_total(en);
    if (lane == 0) {
      er[s] = en;
      mr[s] = ex ? 1.f : 0.f;
    }
  };
  float fx[VPL], bx[VPL], fv = 0.f, bv = 0.f;  // the next pair of the forward / backward ring
  bool fex = false, bex = false;

  // ---- the step's gates (fetched a step ahead) and its scalars from a ring
  // holding the pairs t-W+1 .. t
  struct Gate {
    float lam, beta;  // lambda_t and beta_t (this lane's channel for Falcon-2/2A)
  };
  auto load_gate = [&](int t) {
    Gate gt;
    gt.lam = a.lam[gidx(t)];
    gt.beta = PERCH ? a.beta[gidx(t) * D + j] : a.beta[gidx(t)];
    return gt;
  };
  struct Scal {
    float inv_n, den;
    bool has;
  };
  auto scalars = [&](int t, const float* er, const float* mr) {
    float n = 0.f, es = 0.f;
    int s = slot(t);
#pragma unroll 4
    for (int q = 0; q < W; ++q) {
      n += mr[s];
      es = fmaf(mr[s], er[s], es);
      s = s == 0 ? R - 1 : s - 1;
    }
    Scal c;
    c.has = n > 0.f;
    c.inv_n = 1.f / fmaxf(n, 1.f);
    c.den = c.has ? a.eps + es * c.inv_n : 1.f;
    return c;
  };
  auto gamma_of = [&](float lam) { return fminf(fmaxf(1.f - lam, a.eps_gamma), 1.f); };

  // ---- one forward step of the lane's column on S (S_{t-1} in, S_t out),
  // the forward ring holding the pairs t-W+1 .. t.  The warp first puts pair
  // t + 1 (read by no step before t + 1) and fetches pair t + 2.
  auto fwd_one = [&](int t, int t_end, float (&S)[EPT], Gate& gn) {
    const Gate gt = gn;
    if (t + 1 < t_end) gn = load_gate(t + 1);
    put_pair(t + 1, fx, fv, fex, fxr, fvr, fer, fmr);
    fetch_pair(t + 2, fx, fv, fex);
    const Scal c = scalars(t, fer, fmr);
    const float gam = gamma_of(gt.lam);
    const float ce = c.has ? c.inv_n * gt.beta / c.den : 0.f;  // c_a / m_a at this column
    float acc[EPT];
#pragma unroll
    for (int m = 0; m < EPT; ++m) acc[m] = 0.f;
    const int s0 = slot(t);
#pragma unroll 4
    for (int q = 0; q < W; ++q) {
      const int s = s0 - q < 0 ? s0 - q + R : s0 - q;
      const float* xs = fxr + s * D;
      float x[EPT];
#pragma unroll
      for (int m = 0; m < EPT; ++m) x[m] = xs[row(m)];
      float dlt;
      if (ADD) {
        dlt = fmr[s] * ce * fvr[s * 4 + jj];
      } else {
        float u = 0.f;
#pragma unroll
        for (int m = 0; m < EPT; ++m) u = fmaf(x[m], S[m], u);
        u = col_total(u);
        dlt = fmr[s] * ce * (fvr[s * 4 + jj] - gam * u);
      }
#pragma unroll
      for (int m = 0; m < EPT; ++m) acc[m] = fmaf(x[m], dlt, acc[m]);
    }
#pragma unroll
    for (int m = 0; m < EPT; ++m) S[m] = fmaf(gam, S[m], acc[m]);
    __syncwarp();  // the put is seen by step t + 1
  };
  // the forward ring for a run of steps from t0: pairs t0-W+1 .. t0 in place,
  // pair t0 + 1 fetched; returns the gates of step t0
  auto fwd_ring_start = [&](int t0) {
    __syncwarp();
    for (int p = t0 - W + 1; p <= t0; ++p) {
      fetch_pair(p, fx, fv, fex);
      put_pair(p, fx, fv, fex, fxr, fvr, fer, fmr);
    }
    fetch_pair(t0 + 1, fx, fv, fex);
    __syncwarp();
    return load_gate(t0);
  };

  // ---- pass 1: forward, the state at every block start; the final state
  float Snext[EPT];  // S_t of the backward step t (the state after it)
#pragma unroll
  for (int m = 0; m < EPT; ++m) Snext[m] = a.S_in ? a.S_in[((size_t)bh * D + row(m)) * D + j] : 0.f;
  if (T > 0) {
    Gate gn = fwd_ring_start(0);
    for (int t = 0; t < T; ++t) {
      if (t % kBW == 0) {
#pragma unroll
        for (int m = 0; m < EPT; ++m) *st_at(t / kBW, m) = Snext[m];
      }
      fwd_one(t, T, Snext, gn);
    }
  }

  // ---- pass 2: backward, block by block from the end
  float dS[EPT];
#pragma unroll
  for (int m = 0; m < EPT; ++m) dS[m] = a.dS_final ? a.dS_final[((size_t)bh * D + row(m)) * D + j] : 0.f;
  if (cg == 0) {
    if (a.shift == 1 && T >= 1) {  // the last key is the key of no pair of this call
      for (int i = tid; i < D; i += kNT) stw<Tin>(a.dk, gidx(T - 1) * D + i, 0.f);
    }
    if (a.dk_prev && (a.shift == 0 || T == 0)) {  // the carried key is read by no pair
      for (int i = tid; i < D; i += kNT) stw<Tin>(a.dk_prev, (size_t)bh * D + i, 0.f);
    }
  }
  for (int i = lane; i < R * 4; i += 32) gvr[i] = 0.f;
  float qn[EPT], dn = 0.f;  // q (the lane's rows) and do (its column) of the next step
#pragma unroll
  for (int m = 0; m < EPT; ++m) qn[m] = 0.f;
  Gate gb{0.f, 0.f};  // the gates of the next step
  if (T > 0) {
    __syncwarp();
    for (int p = T - W; p < T; ++p) {  // the window of step T - 1
      fetch_pair(p, bx, bv, bex);
      put_pair(p, bx, bv, bex, bxr, bvr, ber, bmr);
    }
    fetch_pair(T - 1 - W, bx, bv, bex);  // enters at the start of step T - 1
    __syncwarp();
#pragma unroll
    for (int m = 0; m < EPT; ++m) qn[m] = ldw<Tin>(a.q, gidx(T - 1) * D + row(m));
    dn = ldw<Tin>(a.dO, gidx(T - 1) * D + j);
    gb = load_gate(T - 1);
  }
  const size_t prow = (size_t)bh * T;  // partial-sum and scalar rows of this (b, h)
  for (int blk = NB - 1; blk >= 0; --blk) {
    const int t0 = blk * kBW, t1 = min(T, t0 + kBW);
    {  // recompute and record the block's states: NB + (t - t0) holds S_{t-1}
      float S[EPT];
#pragma unroll
      for (int m = 0; m < EPT; ++m) S[m] = *st_at(blk, m);
      Gate gn = fwd_ring_start(t0);
      for (int t = t0; t < t1; ++t) {
#pragma unroll
        for (int m = 0; m < EPT; ++m) *st_at(NB + (t - t0), m) = S[m];
        if (t + 1 < t1) fwd_one(t, t1, S, gn);  // the block's last state is not needed
      }
    }
    float Spn[EPT];
    for (int t = t1 - 1; t >= t0; --t) {
      const int tl = t - t0;
      const Gate gt = gb;
      if (t >= 1) gb = load_gate(t - 1);
      float Sp[EPT], qc[EPT];
      const float dc = dn;
#pragma unroll
      for (int m = 0; m < EPT; ++m) {
        Sp[m] = t < t1 - 1 ? Spn[m] : *st_at(NB + tl, m);
        qc[m] = qn[m];
      }
      if (tl >= 1) {
#pragma unroll
        for (int m = 0; m < EPT; ++m) Spn[m] = *st_at(NB + tl - 1, m);
      }
      if (t >= 1) {
#pragma unroll
        for (int m = 0; m < EPT; ++m) qn[m] = ldw<Tin>(a.q, gidx(t - 1) * D + row(m));
        dn = ldw<Tin>(a.dO, gidx(t - 1) * D + j);
        // pair t - W enters the ring (its slot held pair t + 2, written out two steps ago)
        put_pair(t - W, bx, bv, bex, bxr, bvr, ber, bmr);
        fetch_pair(t - W - 1, bx, bv, bex);
      }
      const Scal c = scalars(t, ber, bmr);
      const float gam = gamma_of(gt.lam);
      const float eta_j = c.has ? gt.beta / c.den : 0.f;
#pragma unroll
      for (int m = 0; m < EPT; ++m) dS[m] = fmaf(qc[m], dc, dS[m]);  // dS += q do^T
      float dz[EPT];  // sum_a x_a dr_a at the lane's rows
#pragma unroll
      for (int m = 0; m < EPT; ++m) dz[m] = 0.f;
      float deta = 0.f;  // sum_a m_a r_a dd_a / max(n, 1) at this column
      const int s0 = slot(t);
#pragma unroll (EPT <= 8 ? 4 : 2)
      for (int q = 0; q < W; ++q) {
        const int s = s0 - q < 0 ? s0 - q + R : s0 - q;
        const float* xs = bxr + s * D;
        float x[EPT];
#pragma unroll
        for (int m = 0; m < EPT; ++m) x[m] = xs[row(m)];
        float u = 0.f, dd = 0.f;
#pragma unroll
        for (int m = 0; m < EPT; ++m) {
          if (!ADD) u = fmaf(x[m], Sp[m], u);
          dd = fmaf(x[m], dS[m], dd);
        }
        if (!ADD) u = col_total(u);
        dd = col_total(dd);
        const float cm = bmr[s] * c.inv_n, cc = cm * eta_j;
        const float r = ADD ? bvr[s * 4 + jj] : bvr[s * 4 + jj] - gam * u;
        const float dlt = cc * r, dr = ADD ? 0.f : cc * dd;
        if (g == 0) gvr[s * 4 + jj] += cc * dd;
        deta = fmaf(cm, r * dd, deta);
        // dx_a over the warp's columns: dS delta_a - gamma S_{t-1} dr_a
        float vals[EPT];
#pragma unroll
        for (int m = 0; m < EPT; ++m) {
          vals[m] = ADD ? dS[m] * dlt : fmaf(dS[m], dlt, -gam * Sp[m] * dr);
          if (!ADD) dz[m] = fmaf(x[m], dr, dz[m]);
        }
        quad_reduce_scatter<EPT>(vals, lane);
#pragma unroll
        for (int i = 0; i < EPT / 4; ++i) pw[q * D + row(jj * (EPT / 4) + i)] = vals[i];
      }
      {  // dq = S_t do over the warp's columns
        float vals[EPT];
#pragma unroll
        for (int m = 0; m < EPT; ++m) vals[m] = Snext[m] * dc;
        quad_reduce_scatter<EPT>(vals, lane);
#pragma unroll
        for (int i = 0; i < EPT / 4; ++i) pw[W * D + row(jj * (EPT / 4) + i)] = vals[i];
      }
      // dZ = dS - sum_a x_a dr_a^T, dgamma = <dZ, S_{t-1}>, dS_{t-1} = gamma dZ
      float gsum = 0.f;
#pragma unroll
      for (int m = 0; m < EPT; ++m) {
        const float z = dS[m] - dz[m];
        gsum = fmaf(z, Sp[m], gsum);
        dS[m] = gam * z;
        Snext[m] = Sp[m];
      }
      gsum = warp_total(gsum);
      const float ew = warp_total(g == 0 ? (PERCH ? deta * eta_j : deta) : 0.f);
      if (lane == 0) {
        pw[W * D + D] = ew;
        pw[W * D + D + 1] = gsum;
      }
      if (PERCH && g == 0) a.dbeta[gidx(t) * D + j] = c.has ? deta / c.den : 0.f;
      __syncthreads();
      {  // the CTA's 16 columns: the four warps' partial sums
        float* dst = a.part + ((prow + t) * NCG + cg) * KP;
        for (int i = tid; i < W * D + D + 2; i += kNT)
          dst[i] = (pall[i] + pall[KP + i]) + (pall[2 * KP + i] + pall[3 * KP + i]);
        if (cg == 0 && tid == 0) {
          float* sc = a.scal + (prow + t) * 4;
          sc[0] = 1.f / c.den;
          sc[1] = PERCH ? 1.f : eta_j;
          sc[2] = c.inv_n;
          sc[3] = c.has ? 1.f : 0.f;
        }
      }
      __syncthreads();
      if (g == 0) {  // pair t is complete: its value gradient leaves, the slot clears
        const int s = slot(t);
        stw<Tin>(a.dv, gidx(t) * D + j, gvr[s * 4 + jj]);
        gvr[s * 4 + jj] = 0.f;
      }
    }
  }
  __syncwarp();
  // the carried window ring's values (pairs -W+1 .. -1; zero when T = 0)
  if (W > 1 && a.dwin_v && g == 0) {
    for (int p = -(W - 1); p < 0; ++p)
      stw<Tin>(a.dwin_v, ((size_t)bh * (W - 1) + ring_slot(p)) * D + j, T > 0 ? gvr[slot(p) * 4 + jj] : 0.f);
  }
  if (a.dS_in) {
#pragma unroll
    for (int m = 0; m < EPT; ++m) a.dS_in[((size_t)bh * D + row(m)) * D + j] = dS[m];
  }
}

// Sums over the column groups, per pair and per step: row r of a (b, h) is
// pair p = r - (W - 1); its key gradient gathers dx_a of the steps
// t = p + a (a < W) that read it, plus the key-norm term 2 de_t m_p x_p / n_t;
// for p >= 0 the row also writes dq_t, and (one thread) dbeta_t and dlambda_t.
template <typename Tin, int D, bool PERCH>
__global__ void __launch_bounds__(256) falcon_bwd_win_reduce_kernel(WinArgs a) {
  constexpr int NCG = WinCfg<D>::NCG, RPB = 256 / D;
  const int W = a.W, T = a.T, KP = win_part_floats(D, W);
  const int i = threadIdx.x % D;
  const int r = blockIdx.x * RPB + threadIdx.x / D;
  const int bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
  if (r >= T + W - 1) return;
  const int p = r - (W - 1);
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  auto gidx = [&](int t) { return ((size_t)b * T + t) * a.H + h; };
  const size_t prow = (size_t)bh * T;
  auto part_at = [&](int t, int c, int k) { return a.part[((prow + t) * NCG + c) * KP + k]; };
  // the pair's key (zero when the pair does not exist)
  const bool ex = pos + p >= a.shift;
  float x = 0.f;
  if (ex) {
    if (p >= 0) {
      const int kt = p - a.shift;
      if (kt >= 0) x = ldw<Tin>(a.k, gidx(kt) * D + i);
      else if (a.kprev_in) x = ldw<Tin>(a.kprev_in, (size_t)bh * D + i);
    } else if (a.winx_in) {
      const int s = (int)((pos + p) % (W - 1));
      x = ldw<Tin>(a.winx_in, ((size_t)bh * (W - 1) + s) * D + i);
    }
  }
  float gk = 0.f;
  for (int q = 0; q < W; ++q) {
    const int t = p + q;
    if (t < 0 || t >= T) continue;
    float et = 0.f;
#pragma unroll
    for (int c = 0; c < NCG; ++c) {
      gk += part_at(t, c, q * D + i);
      et += part_at(t, c, W * D + D);
    }
    const float* sc = a.scal + (prow + t) * 4;
    if (ex && sc[3] != 0.f) {
      const float de = -et * sc[1] * sc[0];  // -<deta, eta> / (eps + e)
      gk = fmaf(2.f * de * sc[2], x, gk);
    }
  }
  if (p >= 0) {
    if (a.shift == 0) stw<Tin>(a.dk, gidx(p) * D + i, gk);
    else if (p >= 1) stw<Tin>(a.dk, gidx(p - 1) * D + i, gk);
    else if (a.dk_prev) stw<Tin>(a.dk_prev, (size_t)bh * D + i, gk);
    const int t = p;
    float dq = 0.f;
#pragma unroll
    for (int c = 0; c < NCG; ++c) dq += part_at(t, c, W * D + i);
    stw<Tin>(a.dq, gidx(t) * D + i, dq);
    if (i == 0) {
      float et = 0.f, dg = 0.f;
#pragma unroll
      for (int c = 0; c < NCG; ++c) {
        et += part_at(t, c, W * D + D);
        dg += part_at(t, c, W * D + D + 1);
      }
      const float* sc = a.scal + (prow + t) * 4;
      if (!PERCH) a.dbeta[gidx(t)] = sc[3] != 0.f ? et * sc[0] : 0.f;
      const float om = 1.f - a.lam[gidx(t)];
      a.dlam[gidx(t)] = (om >= a.eps_gamma && om <= 1.f) ? -dg : 0.f;
    }
  } else if (a.dwin_x) {
    const int s = (int)((pos + p) % (W - 1) + (W - 1)) % (W - 1);
    stw<Tin>(a.dwin_x, ((size_t)bh * (W - 1) + s) * D + i, gk);
  }
}

template <int D>
size_t win_smem_bytes(int W) {
  return (size_t)win_layout(D, W).total * sizeof(float);
}

size_t win_smem_for(int d, int W) {
  return d == 32 ? win_smem_bytes<32>(W) : d == 64 ? win_smem_bytes<64>(W) : win_smem_bytes<128>(W);
}

struct WinWs {
  size_t st, part, scal, total;  // float offsets
};
WinWs win_ws(int B, int T, int H, int d, int W) {
  const size_t NB = (size_t)(T + kBW - 1) / kBW, BH = (size_t)B * H;
  WinWs w;
  w.st = 0;
  w.part = BH * (NB + kBW + 1) * d * d;
  w.scal = w.part + BH * T * (d / kCPC) * win_part_floats(d, W);
  w.total = w.scal + BH * T * 4;
  return w;
}

template <typename Tin, int D>
int launch_win_d(const WinArgs& a, bool add, bool perch, cudaStream_t stream) {
  const size_t smem = win_smem_bytes<D>(a.W);
  auto go = [&](auto kern) {
    if (!set_smem_limit(reinterpret_cast<const void*>(kern), smem)) return FALCON_ERR_CUDA;
    kern<<<a.B * a.H * WinCfg<D>::NCG, kNT, smem, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
  };
  int st;
  if (add) st = perch ? go(falcon_bwd_win_kernel<Tin, D, true, true>) : go(falcon_bwd_win_kernel<Tin, D, true, false>);
  else st = perch ? go(falcon_bwd_win_kernel<Tin, D, false, true>) : go(falcon_bwd_win_kernel<Tin, D, false, false>);
  if (st != FALCON_OK) return st;
  const int rows = a.T + a.W - 1;
  if (rows <= 0) return FALCON_OK;
  dim3 grid((unsigned)((rows + 256 / D - 1) / (256 / D)), (unsigned)(a.B * a.H));
  if (perch) falcon_bwd_win_reduce_kernel<Tin, D, true><<<grid, 256, 0, stream>>>(a);
  else falcon_bwd_win_reduce_kernel<Tin, D, false><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace

bool backward_window_supported(int variant, int dk, int dv, int window) {
  if (dk != dv || (dk != 32 && dk != 64 && dk != 128)) return false;
  const int W = effective_window(variant, window);
  if (W < 1 || W > 64) return false;
  return win_smem_for(dk, W) <= 232448;
}

size_t backward_window_ws_bytes(int B, int T, int H, int d, int window) {
  return win_ws(B, T, H, d, window).total * sizeof(float);
}

int launch_backward_window(const FwdArgs& f, const void* dO, const float* dS_final, void* dq, void* dk, void* dv,
                           float* dbeta, float* dlam, float* dS_in, void* dk_prev, void* dwin_x, void* dwin_v) {
  WinArgs a;
  a.B = f.B; a.T = f.T; a.H = f.H; a.W = f.W;
  a.eps = f.eps; a.eps_gamma = f.eps_gamma; a.shift = f.shift;
  a.q = f.q; a.k = f.k; a.v = f.v; a.dO = dO; a.beta = f.beta; a.lam = f.lam;
  a.S_in = f.S_in; a.kprev_in = f.kprev_in; a.pos_in = f.pos_in; a.dS_final = dS_final;
  a.winx_in = f.W > 1 ? f.winx_in : nullptr;
  a.winv_in = f.W > 1 ? f.winv_in : nullptr;
  a.dq = dq; a.dk = dk; a.dv = dv; a.dbeta = dbeta; a.dlam = dlam; a.dS_in = dS_in; a.dk_prev = dk_prev;
  a.dwin_x = f.W > 1 ? dwin_x : nullptr;
  a.dwin_v = f.W > 1 ? dwin_v : nullptr;
  if ((a.dwin_x == nullptr) != (a.dwin_v == nullptr)) return FALCON_ERR_INVALID_ARG;
  const WinWs w = win_ws(f.B, f.T, f.H, f.dk, f.W);
  float* ws = reinterpret_cast<float*>(f.ws);
  a.st = ws + w.st;
  a.part = ws + w.part;
  a.scal = ws + w.scal;
  const bool add = variant_additive(f.variant), perch = variant_per_channel(f.variant);
  const bool bf = f.dtype == FALCON_BF16;
  switch (f.dk) {
    case 32: return bf ? launch_win_d<__nv_bfloat16, 32>(a, add, perch, f.stream) : launch_win_d<float, 32>(a, add, perch, f.stream);
    case 64: return bf ? launch_win_d<__nv_bfloat16, 64>(a, add, perch, f.stream) : launch_win_d<float, 64>(a, add, perch, f.stream);
    default: return bf ? launch_win_d<__nv_bfloat16, 128>(a, add, perch, f.stream) : launch_win_d<float, 128>(a, add, perch, f.stream);
  }
}

}  // namespace falcon
