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
//   dS += q do^T;  dq = gamma S_{t-1} do + sum_a x_a (delta_a . do);
//   dd_a = dS^T x_a;  dc_a = r_a (.) dd_a;  regression: dr_a = c_a (.) dd_a,
//   dv_a += dr_a, dx_a += dS delta_a - gamma S_{t-1} dr_a; additive:
//   dv_a += c_a (.) dd_a, dx_a += dS delta_a;
//   deta = sum_a m_a dc_a / max(n, 1) (summed over channels for a scalar
//   eta), dbeta = deta / (eps + e), de = -<deta, eta> / (eps + e),
//   dx_a += 2 de m_a x_a / max(n, 1);
//   dZ = dS - sum_a x_a dr_a^T (additive: dS), dgamma = <dZ, S_{t-1}>,
//   dlambda = -dgamma where the clamp passes it, dS_{t-1} = gamma dZ.
// A pair is read by the W steps p .. p + W - 1, so its key and value
// gradients gather in a ring of W accumulators while the steps run
// backwards, and leave for dk / dv (or the carried key and window ring) at
// step p, the last to read it.
//
// One CTA per (b, h).  A forward pass keeps the state at every 64-step block
// start in the workspace; then, block by block from the end, the block's
// states are recomputed into the workspace and its steps reversed.  Thread
// (j, g) owns the state column j and the rows g + RS m.  Sums over rows (the
// S^T x_a and dS^T x_a of a group of eight pairs) go through a table of
// partial sums per row group; sums over columns (dS delta_a - gamma S dr_a
// and S do) are a reduce-scatter across the warp's 32 columns by shuffles,
// then across the warps of a row group through shared memory.

#include "common.cuh"

namespace falcon {

namespace {

constexpr int kBW = 64;  // steps per recomputed block
constexpr int kGP = 8;   // pairs per reduction group

template <int D>
struct WinCfg {
  static constexpr int NT = D == 32 ? 64 : (D == 64 ? 256 : 512);
  static constexpr int RS = NT / D;   // row groups
  static constexpr int EPT = D / RS;  // state elements per thread
  static constexpr int NCB = D / 32;  // 32-column blocks of a row group
  static constexpr int NW = NT / 32;
  static constexpr int VPL = D / 32;  // elements of a D-vector per lane (one warp)
};

// Shared-memory layout in floats (W chosen at run time).  The rings hold
// W + 2 pairs: the window of the step, the pair a step ahead (written while
// the step runs) and the slot a slower warp may still read from the step before.
struct WinLayout {
  int xf, vf, ef, mf;          // forward ring: keys, values [W+2][D]; |x|^2, exists [W+2]
  int xb, vb, eb, mb, gx, gv;  // backward ring and its key / value gradients [W+2][D]
  int dl, dr;                  // delta_a, dr_a of the step's pairs [W][D] (by window position a)
  int qs, ds, y0;              // q_t, do_t [2][D] (by step parity), S_{t-1} do_t [D]
  int part;                    // row-sum partials [RS][2 kGP][D]
  int cpart;                   // column-sum partials [NCB][kGP + 1][D]
  int dots;                    // delta_a . do [W]
  int red;                     // block reductions [4 NW]
  int total;
};

__host__ __device__ inline WinLayout win_layout(int D, int W, int RS, int NCB, int NW) {
  WinLayout L;
  int o = 0;
  const int R = W + 2;
  auto take = [&](int n) { const int at = o; o += (n + 3) & ~3; return at; };
  L.xf = take(R * D); L.vf = take(R * D); L.ef = take(R); L.mf = take(R);
  L.xb = take(R * D); L.vb = take(R * D); L.eb = take(R); L.mb = take(R);
  L.gx = take(R * D); L.gv = take(R * D);
  L.dl = take(W * D); L.dr = take(W * D);
  L.qs = take(2 * D); L.ds = take(2 * D); L.y0 = take(D);
  L.part = take(RS * 2 * kGP * D);
  L.cpart = take(NCB * (kGP + 1) * D);
  L.dots = take(W);
  L.red = take(4 * NW);
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
  float* ws;  // per (b, h): block-start states [NB][D*D], then the block's states [kBW][D*D]
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

// Sum of v[m] over the warp's 32 lanes for each of 16 m, scattered: lanes
// 2m and 2m + 1 end with the total of element m.  Each level hands the half
// of the values that the partner keeps and adds the half it receives.
template <int N>
__device__ __forceinline__ float lane_reduce_scatter(float (&v)[N], int lane) {
  static_assert(N == 16, "16 values a lane");
#pragma unroll
  for (int n = N, off = 16; n > 1; n >>= 1, off >>= 1) {
    const int half = n >> 1;
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

template <typename Tin, int D, bool ADD, bool PERCH>
__global__ void __launch_bounds__(WinCfg<D>::NT, 1) falcon_bwd_win_kernel(WinArgs a) {
  using C = WinCfg<D>;
  constexpr int NT = C::NT, RS = C::RS, EPT = C::EPT, NW = C::NW, VPL = C::VPL;
  constexpr bool PRE_SP = EPT <= 16;  // registers allow the next step's saved state to load early
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  const int W = a.W, R = W + 2;
  const WinLayout L = win_layout(D, W, RS, C::NCB, NW);
  float *xf = sm + L.xf, *vf = sm + L.vf, *ef = sm + L.ef, *mf = sm + L.mf;
  float *xb = sm + L.xb, *vb = sm + L.vb, *eb = sm + L.eb, *mb = sm + L.mb;
  float *gx = sm + L.gx, *gv = sm + L.gv, *dl = sm + L.dl, *drs = sm + L.dr;
  float *qs = sm + L.qs, *ds = sm + L.ds, *y0 = sm + L.y0;
  float *part = sm + L.part, *cpart = sm + L.cpart, *dots = sm + L.dots, *red = sm + L.red;

  const int tid = threadIdx.x, j = tid % D, rg = tid / D, lane = tid & 31, warp = tid >> 5;
  const int cb = j >> 5;
  const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
  const int T = a.T, NB = (T + kBW - 1) / kBW;
  const int64_t pos = a.pos_in ? a.pos_in[bh] : 0;
  float* ckpt = a.ws + (size_t)bh * (NB + kBW) * D * D;
  float* sts = ckpt + (size_t)NB * D * D;
  auto row = [&](int m) { return rg + RS * m; };
  auto gidx = [&](int t) { return ((size_t)b * T + t) * a.H + h; };
  auto slot = [&](int p) { const int s = p % R; return s < 0 ? s + R : s; };
  // slot of the carried window ring (W > 1) that holds pair p < 0 of this call
  auto ring_slot = [&](int p) {
    const int s = (int)((pos + p) % (W - 1));
    return s < 0 ? s + W - 1 : s;
  };

  // ---- pairs: warp 0 fetches pair p into registers, then puts it into a
  // ring; a pair that does not exist (or lies outside the call) reads as zeros
  auto fetch_pair = [&](int p, float (&X)[VPL], float (&V)[VPL], bool& ex) {
    ex = pos + p >= a.shift && p < T && p >= -(W - 1);
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      const int i = lane + 32 * u;
      float x = 0.f, v = 0.f;
      if (ex) {
        if (p >= 0) {
          const int kt = p - a.shift;
          if (kt >= 0) x = ldw<Tin>(a.k, gidx(kt) * D + i);
          else if (a.kprev_in) x = ldw<Tin>(a.kprev_in, (size_t)bh * D + i);
          v = ldw<Tin>(a.v, gidx(p) * D + i);
        } else if (a.winx_in) {  // pos + p >= shift >= 0 here
          const size_t r = (size_t)bh * (W - 1) + ring_slot(p);
          x = ldw<Tin>(a.winx_in, r * D + i);
          v = ldw<Tin>(a.winv_in, r * D + i);
        }
      }
      X[u] = x;
      V[u] = v;
    }
  };
  auto put_pair = [&](int p, const float (&X)[VPL], const float (&V)[VPL], bool ex, float* xr, float* vr,
                      float* er, float* mr) {
    const int s = slot(p);
    float en = 0.f;
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      xr[s * D + lane + 32 * u] = X[u];
      vr[s * D + lane + 32 * u] = V[u];
      en = fmaf(X[u], X[u], en);
    }
    en = warp_total(en);
    if (lane == 0) {
      er[s] = en;
      mr[s] = ex ? 1.f : 0.f;
    }
  };
  float fx[VPL], fv[VPL], bx[VPL], bv[VPL];  // warp 0: the next pair of the forward / backward ring
  bool fex = false, bex = false;

  // ---- the step's gates (fetched a step ahead) and its scalars from a ring
  // holding the pairs t-W+1 .. t
  struct Gate {
    float lam, beta;  // lambda_t and beta_t (this thread's channel for Falcon-2/2A)
  };
  auto load_gate = [&](int t) {
    Gate g;
    g.lam = a.lam[gidx(t)];
    g.beta = PERCH ? a.beta[gidx(t) * D + j] : a.beta[gidx(t)];
    return g;
  };
  struct Scal {
    float inv_n, den;
    bool has;
  };
  auto scalars = [&](int t, const float* er, const float* mr) {
    float n = 0.f, es = 0.f;
    for (int q = 0; q < W; ++q) {
      const int s = slot(t - q);
      n += mr[s];
      es = fmaf(mr[s], er[s], es);
    }
    Scal c;
    c.has = n > 0.f;
    c.inv_n = 1.f / fmaxf(n, 1.f);
    c.den = c.has ? a.eps + es * c.inv_n : 1.f;
    return c;
  };
  auto gamma_of = [&](float lam) { return fminf(fmaxf(1.f - lam, a.eps_gamma), 1.f); };

  // ---- one forward step on the register state S (S_{t-1} in, S_t out) with
  // the forward ring holding the pairs t-W+1 .. t.  Warp 0 first puts pair
  // t + 1 into the ring (its slot is read by no step in flight) and fetches
  // pair t + 2; the step's barriers make the put visible to step t + 1.
  auto fwd_one = [&](int t, int t_end, float (&S)[EPT], Gate& gn) {
    const Gate g = gn;
    if (t + 1 < t_end) gn = load_gate(t + 1);
    if (warp == 0) {
      put_pair(t + 1, fx, fv, fex, xf, vf, ef, mf);
      fetch_pair(t + 2, fx, fv, fex);
    }
    const Scal c = scalars(t, ef, mf);
    const float gam = gamma_of(g.lam);
    const float ce = c.has ? c.inv_n * g.beta / c.den : 0.f;  // c_a / m_a for this column
    if (!ADD) {
      for (int g0 = 0; g0 < W; g0 += kGP) {
        const int ng = min(kGP, W - g0);
        for (int q = 0; q < ng; ++q) {  // S^T x_a over this thread's rows
          const float* xs = xf + slot(t - g0 - q) * D;
          float su = 0.f;
#pragma unroll
          for (int m = 0; m < EPT; ++m) su = fmaf(xs[row(m)], S[m], su);
          part[(rg * 2 * kGP + q) * D + j] = su;
        }
        __syncthreads();
        for (int q = rg; q < ng; q += RS) {  // pair q's sums for column j, one row group each
          float u = 0.f;
#pragma unroll
          for (int gg = 0; gg < RS; ++gg) u += part[(gg * 2 * kGP + q) * D + j];
          const int s = slot(t - g0 - q);
          dl[(g0 + q) * D + j] = mf[s] * ce * (vf[s * D + j] - gam * u);
        }
        __syncthreads();
      }
#pragma unroll
      for (int m = 0; m < EPT; ++m) S[m] *= gam;
      for (int q = 0; q < W; ++q) {
        const float* xs = xf + slot(t - q) * D;
        const float dj = dl[q * D + j];
#pragma unroll
        for (int m = 0; m < EPT; ++m) S[m] = fmaf(xs[row(m)], dj, S[m]);
      }
    } else {  // additive: delta_a = c_a v_a needs no sum over rows
#pragma unroll
      for (int m = 0; m < EPT; ++m) S[m] *= gam;
      for (int q = 0; q < W; ++q) {
        const int s = slot(t - q);
        const float* xs = xf + s * D;
        const float dj = mf[s] * ce * vf[s * D + j];
#pragma unroll
        for (int m = 0; m < EPT; ++m) S[m] = fmaf(xs[row(m)], dj, S[m]);
      }
      __syncthreads();
    }
  };
  // forward ring for a run of steps from t0: pairs t0-W+1 .. t0 in place,
  // pair t0 + 1 fetched; returns the gates of step t0
  auto fwd_ring_start = [&](int t0) {
    __syncthreads();
    if (warp == 0) {
      for (int p = t0 - W + 1; p <= t0; ++p) {
        fetch_pair(p, fx, fv, fex);
        put_pair(p, fx, fv, fex, xf, vf, ef, mf);
      }
      fetch_pair(t0 + 1, fx, fv, fex);
    }
    const Gate g = load_gate(t0);
    __syncthreads();
    return g;
  };

  // ---- pass 1: forward, the state at every block start
  if (T > 0) {
    float S[EPT];
#pragma unroll
    for (int m = 0; m < EPT; ++m) S[m] = a.S_in ? a.S_in[(size_t)bh * D * D + row(m) * D + j] : 0.f;
    Gate gn = fwd_ring_start(0);
    for (int t = 0; t < T; ++t) {
      if (t % kBW == 0) {
#pragma unroll
        for (int m = 0; m < EPT; ++m) ckpt[(size_t)(t / kBW) * D * D + row(m) * D + j] = S[m];
      }
      fwd_one(t, T, S, gn);
    }
  }

  // ---- pass 2: backward, block by block from the end
  float dS[EPT];
#pragma unroll
  for (int m = 0; m < EPT; ++m) dS[m] = a.dS_final ? a.dS_final[(size_t)bh * D * D + row(m) * D + j] : 0.f;
  if (a.shift == 1 && T >= 1) {  // the last key is the key of no pair of this call
    for (int i = tid; i < D; i += NT) stw<Tin>(a.dk, gidx(T - 1) * D + i, 0.f);
  }
  if (a.dk_prev && (a.shift == 0 || T == 0)) {  // the carried key is read by no pair
    for (int i = tid; i < D; i += NT) stw<Tin>(a.dk_prev, (size_t)bh * D + i, 0.f);
  }
  __syncthreads();
  for (int i = tid; i < R * D; i += NT) {
    gx[i] = 0.f;
    gv[i] = 0.f;
  }
  float qn = 0.f, dn = 0.f;  // q and do of the step after next (threads tid < D)
  Gate gb{0.f, 0.f};         // the gates of the next step
  if (T > 0) {
    if (warp == 0) {  // the window of step T - 1, and the pair that enters at its start
      for (int p = T - W; p < T; ++p) {
        fetch_pair(p, bx, bv, bex);
        put_pair(p, bx, bv, bex, xb, vb, eb, mb);
      }
      fetch_pair(T - 1 - W, bx, bv, bex);
    }
    if (tid < D) {
      qs[((T - 1) & 1) * D + tid] = ldw<Tin>(a.q, gidx(T - 1) * D + tid);
      ds[((T - 1) & 1) * D + tid] = ldw<Tin>(a.dO, gidx(T - 1) * D + tid);
      if (T >= 2) {
        qn = ldw<Tin>(a.q, gidx(T - 2) * D + tid);
        dn = ldw<Tin>(a.dO, gidx(T - 2) * D + tid);
      }
    }
    gb = load_gate(T - 1);
  }
  for (int blk = NB - 1; blk >= 0; --blk) {
    const int t0 = blk * kBW, t1 = min(T, t0 + kBW);
    {  // recompute and record the block's states: sts[t - t0] = S_{t-1}
      float S[EPT];
#pragma unroll
      for (int m = 0; m < EPT; ++m) S[m] = ckpt[(size_t)blk * D * D + row(m) * D + j];
      Gate gn = fwd_ring_start(t0);
      for (int t = t0; t < t1; ++t) {
#pragma unroll
        for (int m = 0; m < EPT; ++m) sts[(size_t)(t - t0) * D * D + row(m) * D + j] = S[m];
        if (t + 1 < t1) fwd_one(t, t1, S, gn);  // the block's last state is not needed
      }
      __syncthreads();
    }
    float Spn[PRE_SP ? EPT : 1];
    for (int t = t1 - 1; t >= t0; --t) {
      const int tl = t - t0;
      const Gate g = gb;
      if (t >= 1) gb = load_gate(t - 1);
      float Sp[EPT];
      if (PRE_SP && t < t1 - 1) {
#pragma unroll
        for (int m = 0; m < EPT; ++m) Sp[m] = Spn[PRE_SP ? m : 0];
      } else {
#pragma unroll
        for (int m = 0; m < EPT; ++m) Sp[m] = sts[(size_t)tl * D * D + row(m) * D + j];
      }
      if (PRE_SP && tl >= 1) {
#pragma unroll
        for (int m = 0; m < EPT; ++m) Spn[PRE_SP ? m : 0] = sts[(size_t)(tl - 1) * D * D + row(m) * D + j];
      }
      // pair t - W enters the ring (its slot held pair t + 2, written out two
      // steps ago); q and do of step t - 1 go to the other parity's buffer
      if (warp == 0 && t >= 1) {
        put_pair(t - W, bx, bv, bex, xb, vb, eb, mb);
        fetch_pair(t - W - 1, bx, bv, bex);
      }
      if (tid < D && t >= 1) {
        qs[((t - 1) & 1) * D + tid] = qn;
        ds[((t - 1) & 1) * D + tid] = dn;
        if (t >= 2) {
          qn = ldw<Tin>(a.q, gidx(t - 2) * D + tid);
          dn = ldw<Tin>(a.dO, gidx(t - 2) * D + tid);
        }
      }
      const float* qc = qs + (t & 1) * D;
      const float* dc = ds + (t & 1) * D;
      const Scal c = scalars(t, eb, mb);
      const float gam = gamma_of(g.lam);
      const float eta_j = c.has ? g.beta / c.den : 0.f;
      // dS += q do^T
      const float doj = dc[j];
#pragma unroll
      for (int m = 0; m < EPT; ++m) dS[m] = fmaf(qc[row(m)], doj, dS[m]);
      float deta = 0.f;  // sum over this thread's pairs of m_a r_a dd_a / max(n, 1) (column j)
      for (int g0 = 0; g0 < W; g0 += kGP) {
        const int ng = min(kGP, W - g0);
        // S_{t-1}^T x_a and dS^T x_a over this thread's rows
        for (int q = 0; q < ng; ++q) {
          const float* xs = xb + slot(t - g0 - q) * D;
          float su = 0.f, sd = 0.f;
#pragma unroll
          for (int m = 0; m < EPT; ++m) {
            const float xv = xs[row(m)];
            if (!ADD) su = fmaf(xv, Sp[m], su);
            sd = fmaf(xv, dS[m], sd);
          }
          if (!ADD) part[(rg * 2 * kGP + 2 * q) * D + j] = su;
          part[(rg * 2 * kGP + 2 * q + 1) * D + j] = sd;
        }
        __syncthreads();
        for (int q = rg; q < ng; q += RS) {  // pair q's sums for column j, one row group each
          float u = 0.f, dd = 0.f;
#pragma unroll
          for (int gg = 0; gg < RS; ++gg) {
            if (!ADD) u += part[(gg * 2 * kGP + 2 * q) * D + j];
            dd += part[(gg * 2 * kGP + 2 * q + 1) * D + j];
          }
          const int s = slot(t - g0 - q);
          const float cm = mb[s] * c.inv_n, cc = cm * eta_j;
          const float r = ADD ? vb[s * D + j] : vb[s * D + j] - gam * u;
          dl[(g0 + q) * D + j] = cc * r;
          drs[(g0 + q) * D + j] = ADD ? 0.f : cc * dd;
          gv[s * D + j] += cc * dd;
          deta = fmaf(cm, r * dd, deta);
        }
        __syncthreads();
        // column sums: dS delta_a - gamma S_{t-1} dr_a, and (first group) S_{t-1} do,
        // 16 rows at a time; lane l (l even) ends with row g + RS (16 hh + l / 2)
#pragma unroll 2
        for (int q = 0; q < ng; ++q) {
          const float dj = dl[(g0 + q) * D + j], rj = drs[(g0 + q) * D + j];
#pragma unroll
          for (int hh = 0; hh < EPT / 16; ++hh) {
            float vals[16];
#pragma unroll
            for (int mm = 0; mm < 16; ++mm) {
              const int m = 16 * hh + mm;
              vals[mm] = ADD ? dS[m] * dj : fmaf(dS[m], dj, -gam * Sp[m] * rj);
            }
            const float tot = lane_reduce_scatter<16>(vals, lane);
            if ((lane & 1) == 0) cpart[(cb * (kGP + 1) + q) * D + rg + RS * (16 * hh + (lane >> 1))] = tot;
          }
        }
        if (g0 == 0) {
#pragma unroll
          for (int hh = 0; hh < EPT / 16; ++hh) {
            float vals[16];
#pragma unroll
            for (int mm = 0; mm < 16; ++mm) vals[mm] = Sp[16 * hh + mm] * doj;
            const float tot = lane_reduce_scatter<16>(vals, lane);
            if ((lane & 1) == 0) cpart[(cb * (kGP + 1) + kGP) * D + rg + RS * (16 * hh + (lane >> 1))] = tot;
          }
        }
        __syncthreads();
        for (int idx = tid; idx < (ng + 1) * D; idx += NT) {
          const int q = idx / D, i = idx % D;
          if (q == ng && g0 != 0) continue;
          const int qq = q == ng ? kGP : q;
          float tot = 0.f;
#pragma unroll
          for (int bb = 0; bb < C::NCB; ++bb) tot += cpart[(bb * (kGP + 1) + qq) * D + i];
          if (q == ng) y0[i] = tot;
          else gx[slot(t - g0 - q) * D + i] += tot;
        }
        // the next group writes cpart only after its first barrier
      }
      // delta_a . do, and the step's sum for the gradient of eta
      for (int q = warp; q < W; q += NW) {
        float sdot = 0.f;
        for (int i = lane; i < D; i += 32) sdot = fmaf(dl[q * D + i], dc[i], sdot);
        sdot = warp_total(sdot);
        if (lane == 0) dots[q] = sdot;
      }
      {
        float rv = PERCH ? deta * eta_j : deta;
        rv = warp_total(rv);
        if (lane == 0) red[warp] = rv;
      }
      __syncthreads();
      float etot = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) etot += red[w];
      // de = -<deta, eta> / (eps + e)
      const float de = c.has ? -(PERCH ? etot : etot * eta_j) / c.den : 0.f;
      if (PERCH) {  // a one-pair variant: row group 0 holds the column's deta
        if (rg == 0) a.dbeta[gidx(t) * D + j] = c.has ? deta / c.den : 0.f;
      } else if (tid == 0) {
        a.dbeta[gidx(t)] = c.has ? etot / c.den : 0.f;
      }
      for (int i = tid; i < D; i += NT) {  // dq, and the key-norm term of dx_a
        float dqv = gam * y0[i];
        for (int q = 0; q < W; ++q) {
          const int s = slot(t - q);
          const float xv = xb[s * D + i];
          dqv = fmaf(xv, dots[q], dqv);
          gx[s * D + i] = fmaf(2.f * de * mb[s] * c.inv_n, xv, gx[s * D + i]);
        }
        stw<Tin>(a.dq, gidx(t) * D + i, dqv);
      }
      // dZ = dS - sum_a x_a dr_a^T, dgamma = <dZ, S_{t-1}>, dS_{t-1} = gamma dZ
      if (!ADD) {
        for (int q = 0; q < W; ++q) {
          const float* xs = xb + slot(t - q) * D;
          const float rj = drs[q * D + j];
#pragma unroll
          for (int m = 0; m < EPT; ++m) dS[m] = fmaf(-xs[row(m)], rj, dS[m]);
        }
      }
      float gsum = 0.f;
#pragma unroll
      for (int m = 0; m < EPT; ++m) {
        gsum = fmaf(dS[m], Sp[m], gsum);
        dS[m] *= gam;
      }
      gsum = warp_total(gsum);
      if (lane == 0) red[NW + warp] = gsum;
      __syncthreads();
      if (tid == 0) {
        float dg = 0.f;
        for (int w = 0; w < NW; ++w) dg += red[NW + w];
        const float om = 1.f - g.lam;
        a.dlam[gidx(t)] = (om >= a.eps_gamma && om <= 1.f) ? -dg : 0.f;
      }
      // pair t is complete (no later step reads it): its gradients leave and
      // its accumulators clear for the pair that takes the slot
      for (int i = tid; i < D; i += NT) {
        const int s = slot(t);
        const float gk = gx[s * D + i], gvv = gv[s * D + i];
        if (a.shift == 0) stw<Tin>(a.dk, gidx(t) * D + i, gk);
        else if (t >= 1) stw<Tin>(a.dk, gidx(t - 1) * D + i, gk);
        else if (a.dk_prev) stw<Tin>(a.dk_prev, (size_t)bh * D + i, gk);
        stw<Tin>(a.dv, gidx(t) * D + i, gvv);
        gx[s * D + i] = 0.f;
        gv[s * D + i] = 0.f;
      }
    }
  }
  __syncthreads();
  // the carried window ring's pairs -W+1 .. -1 (complete after step 0; zero when T = 0)
  if (W > 1 && a.dwin_x) {
    for (int idx = tid; idx < (W - 1) * D; idx += NT) {
      const int p = -(W - 1) + idx / D, i = idx % D;
      const size_t r = ((size_t)bh * (W - 1) + ring_slot(p)) * D + i;
      stw<Tin>(a.dwin_x, r, T > 0 ? gx[slot(p) * D + i] : 0.f);
      stw<Tin>(a.dwin_v, r, T > 0 ? gv[slot(p) * D + i] : 0.f);
    }
  }
  if (a.dS_in) {
#pragma unroll
    for (int m = 0; m < EPT; ++m) a.dS_in[(size_t)bh * D * D + row(m) * D + j] = dS[m];
  }
}

template <int D>
size_t win_smem_bytes(int W) {
  using C = WinCfg<D>;
  return (size_t)win_layout(D, W, C::RS, C::NCB, C::NW).total * sizeof(float);
}

size_t win_smem_for(int d, int W) {
  return d == 32 ? win_smem_bytes<32>(W) : d == 64 ? win_smem_bytes<64>(W) : win_smem_bytes<128>(W);
}

template <typename Tin, int D>
int launch_win_d(const WinArgs& a, bool add, bool perch, cudaStream_t stream) {
  const size_t smem = win_smem_bytes<D>(a.W);
  auto go = [&](auto kern) {
    if (!set_smem_limit(reinterpret_cast<const void*>(kern), smem)) return FALCON_ERR_CUDA;
    kern<<<a.B * a.H, WinCfg<D>::NT, smem, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
  };
  if (add) return perch ? go(falcon_bwd_win_kernel<Tin, D, true, true>) : go(falcon_bwd_win_kernel<Tin, D, true, false>);
  return perch ? go(falcon_bwd_win_kernel<Tin, D, false, true>) : go(falcon_bwd_win_kernel<Tin, D, false, false>);
}

}  // namespace

bool backward_window_supported(int variant, int dk, int dv, int window) {
  if (dk != dv || (dk != 32 && dk != 64 && dk != 128)) return false;
  const int W = effective_window(variant, window);
  if (W < 1 || W > 64) return false;
  return win_smem_for(dk, W) <= 232448;
}

size_t backward_window_ws_bytes(int B, int T, int H, int d) {
  const size_t NB = (size_t)(T + kBW - 1) / kBW;
  return (size_t)B * H * (NB + kBW) * d * d * sizeof(float);
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
  a.ws = reinterpret_cast<float*>(f.ws);
  const bool add = variant_additive(f.variant), perch = variant_per_channel(f.variant);
  const bool bf = f.dtype == FALCON_BF16;
  switch (f.dk) {
    case 32: return bf ? launch_win_d<__nv_bfloat16, 32>(a, add, perch, f.stream) : launch_win_d<float, 32>(a, add, perch, f.stream);
    case 64: return bf ? launch_win_d<__nv_bfloat16, 64>(a, add, perch, f.stream) : launch_win_d<float, 64>(a, add, perch, f.stream);
    default: return bf ? launch_win_d<__nv_bfloat16, 128>(a, add, perch, f.stream) : launch_win_d<float, 128>(a, add, perch, f.stream);
  }
}

}  // namespace falcon
