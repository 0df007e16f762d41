// C ABI of libfalcon.so: argument checks on the host, workspace sizing and
// dispatch to the kernels.  Nothing here allocates device memory.

#include <atomic>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "tc_ptx.cuh"

using namespace falcon;

namespace falcon {

// Failure-detection test hook state (falcon_test_hooks): process-wide.
static std::atomic<uint64_t> g_wait_limit_ns{0};
static std::atomic<int> g_stall{0};

uint64_t wait_limit_ns() {
  const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v ? v : tc::kWaitLimitNs;
}

bool take_test_stall() { return g_stall.exchange(0, std::memory_order_relaxed) != 0; }

}  // namespace falcon

namespace {

bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

int check_params(const falcon_params_t* p, bool need_T_pos) {
  if (!p) return FALCON_ERR_INVALID_ARG;
  if (p->B < 1 || p->H < 1 || p->T < 0 || (need_T_pos && p->T < 1)) return FALCON_ERR_INVALID_ARG;
  if (p->variant < FALCON_1 || p->variant > FALCON_3A) return FALCON_ERR_INVALID_ARG;
  if (p->dtype != FALCON_BF16 && p->dtype != FALCON_F32) return FALCON_ERR_INVALID_ARG;
  if (p->impl < FALCON_IMPL_AUTO || p->impl > FALCON_IMPL_SCAN) return FALCON_ERR_INVALID_ARG;
  if (p->pairing != FALCON_PAIR_PREFIX && p->pairing != FALCON_PAIR_SAME_STEP) return FALCON_ERR_INVALID_ARG;
  if (!(p->eps > 0.f) || !(p->eps_gamma > 0.f) || !(p->eps_gamma <= 1.f)) return FALCON_ERR_INVALID_ARG;
  if (!dim_ok(p->dk) || !dim_ok(p->dv)) return FALCON_ERR_UNSUPPORTED;
  if (p->chunk != 16 && p->chunk != 32 && p->chunk != 64) return FALCON_ERR_UNSUPPORTED;
  if (variant_windowed(p->variant) && (p->window < 1 || p->window > 64)) return FALCON_ERR_UNSUPPORTED;
  if (p->prologue & ~(FALCON_PROLOGUE_L2NORM_QK | FALCON_PROLOGUE_GATE_LOGITS)) return FALCON_ERR_INVALID_ARG;
  return FALCON_OK;
}

size_t elem_size(int dtype) { return dtype == FALCON_BF16 ? 2 : 4; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  auto pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + nb && pb < pa + na;
}

FwdArgs make_args(const falcon_params_t* p, const void* q, const void* k, const void* v,
                  const float* beta, const float* lambda, void* o, void* stream) {
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.B = p->B; a.T = p->T; a.H = p->H; a.dk = p->dk; a.dv = p->dv; a.chunk = p->chunk;
  a.W = effective_window(p->variant, p->window);
  a.eps = p->eps; a.eps_gamma = p->eps_gamma; a.variant = p->variant; a.dtype = p->dtype;
  a.shift = p->pairing == FALCON_PAIR_PREFIX ? 1 : 0;
  a.q = q; a.k = k; a.v = v; a.beta = beta; a.lam = lambda; a.o = o;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return a;
}

bool aligned16(const FwdArgs& a) {
  const void* ps[7] = {a.q, a.k, a.v, a.o, a.kprev_in, a.winx_in, a.winv_in};
  for (const void* x : ps)
    if (reinterpret_cast<uintptr_t>(x) & 15) return false;
  return true;
}

// Kernel family for the chunk forward: the forced one, or for AUTO the
// tensor-core path, then the window recurrence (Falcon-3), then the portable
// chunk kernel.  -1: the forced family does not cover the params.
int pick_impl(const falcon_params_t* p, const FwdArgs& a) {
  const bool tc_ok = tc_chunk_supported(a), scan_ok = window_scan_supported(a);
  switch (p->impl) {
    case FALCON_IMPL_GENERIC: return FALCON_IMPL_GENERIC;
    case FALCON_IMPL_TC: return tc_ok ? FALCON_IMPL_TC : -1;
    case FALCON_IMPL_SCAN: return scan_ok ? FALCON_IMPL_SCAN : -1;
    default: return tc_ok ? FALCON_IMPL_TC : scan_ok ? FALCON_IMPL_SCAN : FALCON_IMPL_GENERIC;
  }
}

}  // namespace

extern "C" {

const char* falcon_strerror(int code) {
  switch (code) {
    case FALCON_OK: return "ok";
    case FALCON_ERR_INVALID_ARG: return "invalid argument";
    case FALCON_ERR_UNSUPPORTED: return "unsupported shape or combination";
    case FALCON_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case FALCON_ERR_CUDA: return "CUDA error";
    case FALCON_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown error";
  }
}

const char* falcon_version(void) { return "falcon-gb300 0.1 sm_103a"; }

void falcon_test_hooks(uint64_t wait_limit_ns, int32_t stall) {
  g_wait_limit_ns.store(wait_limit_ns, std::memory_order_relaxed);
  g_stall.store(stall ? 1 : 0, std::memory_order_relaxed);
}

int falcon_workspace_status(const void* workspace, void* stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const void* word = workspace;
  if (!word) {
    void* scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st != FALCON_OK) return st;
    word = scratch;
  }
  if (reinterpret_cast<uintptr_t>(word) & 255) return FALCON_ERR_WORKSPACE;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FALCON_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return FALCON_ERR_CUDA;
  if (v == 0) return FALCON_OK;
  const uint32_t zero = 0;
  if (cudaMemcpy(const_cast<void*>(word), &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return FALCON_ERR_CUDA;
  return FALCON_ERR_TIMEOUT;
}

// workspace of the kernel family alone (no prologue buffers), 256-byte multiple
static size_t kernel_ws_bytes(const falcon_params_t* p) {
  FwdArgs a = make_args(p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
  const int impl = pick_impl(p, a);
  if (impl == FALCON_IMPL_TC) return align_up(tc_chunk_ws_bytes(p->B, p->T, p->H, p->dk, p->dv, p->chunk, p->variant), 256);
  if (impl == FALCON_IMPL_SCAN) return window_scan_ws_bytes(p->B, p->T, p->H, a.W);
  return 0;
}

static size_t prologue_bytes(const falcon_params_t* p, bool with_o) {
  return prologue_ws_bytes(p->B, p->T, p->H, p->dk, p->dv, p->dtype, variant_per_channel(p->variant), with_o);
}

static bool ws_ok(const void* ws, size_t have, size_t need) {
  return need == 0 || (ws && have >= need && (reinterpret_cast<uintptr_t>(ws) & 255) == 0);
}

static ProArgs pro_args(const falcon_params_t* p, const int32_t* cu, const void* q, const void* k,
                        const void* v, const float* beta, const float* lambda) {
  ProArgs a;
  std::memset(&a, 0, sizeof(a));
  a.B = p->B; a.T = p->T; a.H = p->H; a.dk = p->dk; a.dv = p->dv; a.dtype = p->dtype;
  a.flags = p->prologue; a.perch = variant_per_channel(p->variant) ? 1 : 0;
  a.cu = cu; a.q = q; a.k = k; a.v = v; a.beta = beta; a.lam = lambda;
  return a;
}

size_t falcon_workspace_size(const falcon_params_t* p) {
  if (check_params(p, false) != FALCON_OK) return 0;
  if (pick_impl(p, make_args(p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr)) < 0) return 0;
  return kernel_ws_bytes(p) + (p->prologue ? prologue_bytes(p, false) : 0);
}

// packed sequences' chunk map (B H NC items, their count and B + 1 sequence offsets, int32)
static size_t varlen_map_bytes(const falcon_params_t* p) {
  return align_up(((size_t)p->B * p->H * ((p->T + 63) / 64) + 1 + p->B + 1) * 4, 256);
}

size_t falcon_varlen_workspace_size(const falcon_params_t* p) {
  if (check_params(p, false) != FALCON_OK) return 0;
  if (pick_impl(p, make_args(p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr)) < 0) return 0;
  return kernel_ws_bytes(p) + prologue_bytes(p, true) + varlen_map_bytes(p);
}

// The prologue runs inside the kernels on the pipelined d = 64 tensor-core
// path (Falcon-1 / 1A): the per-chunk kernel normalises its key rows and
// forms the gates from logits, the sequential kernel scales its products by
// the rows' inverse norms.  Every other path, and rows off a 16-byte
// boundary (which the tensor maps cannot take; pass null pointers to ask
// about the plan alone), take it from a gather pass.
static bool prologue_fused(const falcon_params_t* p, const void* q = nullptr, const void* k = nullptr,
                           const void* v = nullptr) {
  if (!p->prologue || p->dk != 64 || (p->variant != FALCON_1 && p->variant != FALCON_1A)) return false;
  for (const void* x : {q, k, v})
    if (reinterpret_cast<uintptr_t>(x) & 15) return false;
  return pick_impl(p, make_args(p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr)) ==
         FALCON_IMPL_TC;
}

// The packed-sequence chunk map that the Falcon-1 / 1A d = 64 tensor-core
// kernels take in place of the padded batch's every chunk.
struct VarlenMap {
  const int32_t* cu;
  const int32_t* item_map;  // B H NC entries, then the count
  int NC;
  int64_t packed_total;     // > 0: the call's tensors are the packed rows themselves
};

// The kernel family a chunk forward with these args runs: pick_impl, then
// the portable kernel for rows off a 16-byte boundary; -1 if none.
static int resolve_impl(const falcon_params_t* p, const FwdArgs& a) {
  int impl = pick_impl(p, a);
  if (impl < 0) return impl;
  // the window recurrence's 16-byte async copies and the tensor-core
  // kernels' TMA maps and 16-byte stores need rows on 16-byte boundaries
  if ((impl == FALCON_IMPL_SCAN || impl == FALCON_IMPL_TC) && !aligned16(a)) {
    if (p->impl == impl) return -2;
    impl = FALCON_IMPL_GENERIC;
  }
  return impl;
}

static int chunk_fwd_impl(const falcon_params_t* p, const void* q, const void* k, const void* v,
                          const float* beta, const float* lambda, const falcon_carry_t* carry_in,
                          void* o, falcon_carry_t* carry_out, void* workspace,
                          size_t workspace_bytes, void* stream, void* const* events, int n_events,
                          const VarlenMap* vm = nullptr) {
  int st = check_params(p, false);
  if (st != FALCON_OK) return st;
  if (p->T > 0 && (!q || !k || !v || !beta || !lambda || !o)) return FALCON_ERR_INVALID_ARG;
  if (p->prologue && !prologue_fused(p, q, k, v)) {  // phi / gate logits: one pass into the workspace, then the features path
    if (pick_impl(p, make_args(p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr)) < 0)
      return FALCON_ERR_UNSUPPORTED;
    const size_t kws = kernel_ws_bytes(p);
    if (!ws_ok(workspace, workspace_bytes, kws + prologue_bytes(p, false))) return FALCON_ERR_WORKSPACE;
    ProArgs pa = pro_args(p, nullptr, q, k, v, beta, lambda);
    prologue_carve(pa, reinterpret_cast<uint8_t*>(workspace) + kws, false, nullptr);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaEvent_t* ev = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(events));
    if (ev && n_events > 0) cudaEventRecord(ev[0], s);
    st = launch_prologue(pa, s);
    if (st != FALCON_OK) return st;
    falcon_params_t p0 = *p;
    p0.prologue = 0;
    return chunk_fwd_impl(&p0, pa.qo, pa.ko, pa.vo, pa.bo, pa.lo, carry_in, o, carry_out,
                          kws ? workspace : nullptr, kws, stream, events ? events + 1 : nullptr,
                          events ? n_events - 1 : 0);
  }
  FwdArgs a = make_args(p, q, k, v, beta, lambda, o, stream);
  a.prologue = p->prologue;  // nonzero here only on the fused path
  const size_t es = elem_size(p->dtype);
  const size_t BH = (size_t)p->B * p->H;
  const int Wr = a.W - 1;
  if (carry_in) {
    a.S_in = carry_in->S; a.kprev_in = carry_in->k_prev; a.pos_in = carry_in->pos;
    if (Wr > 0) { a.winx_in = carry_in->win_x; a.winv_in = carry_in->win_v; }
  }
  if (carry_out) {
    a.S_out = carry_out->S; a.kprev_out = carry_out->k_prev; a.pos_out = carry_out->pos;
    if (Wr > 0) { a.winx_out = carry_out->win_x; a.winv_out = carry_out->win_v; }
  }
  if (carry_in && carry_out) {
    const size_t nS = BH * p->dk * p->dv * 4, nK = BH * p->dk * es, nP = BH * 8;
    const size_t nWX = BH * (size_t)(Wr > 0 ? Wr : 0) * p->dk * es;
    const size_t nWV = BH * (size_t)(Wr > 0 ? Wr : 0) * p->dv * es;
    const void* ins[5] = {a.S_in, a.kprev_in, a.pos_in, a.winx_in, a.winv_in};
    const size_t nin[5] = {nS, nK, nP, nWX, nWV};
    const void* outs[5] = {a.S_out, a.kprev_out, a.pos_out, a.winx_out, a.winv_out};
    for (int i = 0; i < 5; ++i)
      for (int j = 0; j < 5; ++j)
        if (overlaps(ins[i], nin[i], outs[j], nin[j])) return FALCON_ERR_INVALID_ARG;
  }
  a.ws = workspace; a.ws_bytes = workspace_bytes;
  a.events = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(events));
  a.n_events = n_events;
  const int impl = resolve_impl(p, a);
  if (impl == -2) return FALCON_ERR_INVALID_ARG;
  if (impl < 0) return FALCON_ERR_UNSUPPORTED;
  if (vm && impl == FALCON_IMPL_TC && tc_chunk_takes_map(a)) {
    a.cu = vm->cu;
    a.item_map = vm->item_map;
    a.item_count = vm->item_map + (size_t)p->B * p->H * vm->NC;
    a.packed_total = vm->packed_total;
  } else if (vm && vm->packed_total > 0) {
    return FALCON_ERR_UNSUPPORTED;  // packed rows are read in place by that path only
  }
  if (impl == FALCON_IMPL_SCAN) {
    const size_t need = window_scan_ws_bytes(p->B, p->T, p->H, a.W);
    if (need > 0 && (!workspace || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255) != 0))
      return FALCON_ERR_WORKSPACE;
    return launch_window_scan(a);
  }
  if (impl == FALCON_IMPL_TC) {
    const size_t need = tc_chunk_ws_bytes(p->B, p->T, p->H, p->dk, p->dv, p->chunk, p->variant);
    if (need > 0 && (!workspace || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255) != 0))
      return FALCON_ERR_WORKSPACE;
    return launch_tc_chunk(a);
  }
  return launch_generic_chunk(a);
}

int falcon_chunk_fwd(const falcon_params_t* p, const void* q, const void* k, const void* v,
                     const float* beta, const float* lambda, const falcon_carry_t* carry_in,
                     void* o, falcon_carry_t* carry_out, void* workspace, size_t workspace_bytes,
                     void* stream) {
  return chunk_fwd_impl(p, q, k, v, beta, lambda, carry_in, o, carry_out, workspace,
                        workspace_bytes, stream, nullptr, 0);
}

int falcon_chunk_fwd_timed(const falcon_params_t* p, const void* q, const void* k, const void* v,
                           const float* beta, const float* lambda, const falcon_carry_t* carry_in,
                           void* o, falcon_carry_t* carry_out, void* workspace,
                           size_t workspace_bytes, void* stream, void* const* events,
                           int32_t n_events) {
  int32_t launches = 0;
  const int st = falcon_chunk_fwd_plan(p, nullptr, &launches);
  if (st != FALCON_OK) return st;
  if (!events || n_events != launches + 1) return FALCON_ERR_INVALID_ARG;
  for (int i = 0; i < n_events; ++i)
    if (!events[i]) return FALCON_ERR_INVALID_ARG;
  return chunk_fwd_impl(p, q, k, v, beta, lambda, carry_in, o, carry_out, workspace,
                        workspace_bytes, stream, events, n_events);
}

int falcon_chunk_fwd_plan(const falcon_params_t* p, int32_t* impl_out, int32_t* launches_out) {
  int st = check_params(p, false);
  if (st != FALCON_OK) return st;
  FwdArgs a = make_args(p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
  const int impl = pick_impl(p, a);
  if (impl < 0) return FALCON_ERR_UNSUPPORTED;
  if (impl_out) *impl_out = impl;
  if (launches_out)
    *launches_out = (impl == FALCON_IMPL_TC ? tc_chunk_launches(a) : impl == FALCON_IMPL_SCAN ? 2 : 1) +
                    (p->prologue && !prologue_fused(p) ? 1 : 0);
  return FALCON_OK;
}

int falcon_chunk_fwd_varlen(const falcon_params_t* p, const int32_t* cu_seqlens, int64_t total_tokens,
                            const void* q, const void* k, const void* v, const float* beta,
                            const float* lambda, const falcon_carry_t* carry_in, void* o,
                            falcon_carry_t* carry_out, void* workspace, size_t workspace_bytes,
                            void* stream) {
  int st = check_params(p, false);
  if (st != FALCON_OK) return st;
  if (!cu_seqlens || total_tokens < 0 || total_tokens > (int64_t)p->B * p->T) return FALCON_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!q || !k || !v || !beta || !lambda || !o)) return FALCON_ERR_INVALID_ARG;
  if (pick_impl(p, make_args(p, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr)) < 0)
    return FALCON_ERR_UNSUPPORTED;
  const size_t kws = kernel_ws_bytes(p), pws = prologue_bytes(p, true);
  if (!ws_ok(workspace, workspace_bytes, kws + pws + varlen_map_bytes(p))) return FALCON_ERR_WORKSPACE;
  ProArgs pa = pro_args(p, cu_seqlens, q, k, v, beta, lambda);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  falcon_carry_t co_state;  // the chunk pass gives the state; the rest depends on each length
  std::memset(&co_state, 0, sizeof(co_state));
  if (carry_out) co_state.S = carry_out->S;
  const int W = effective_window(p->variant, p->window), shift = p->pairing == FALCON_PAIR_PREFIX ? 1 : 0;
  // the Falcon-1 / 1A d = 64 tensor-core kernels take only the chunks that
  // hold tokens (a map built here), and read the packed rows in place (the
  // prologue inside them); every other path reads a padded batch gathered
  // into the workspace
  VarlenMap vm;
  vm.cu = cu_seqlens;
  vm.item_map = reinterpret_cast<const int32_t*>(reinterpret_cast<uint8_t*>(workspace) + kws + pws);
  vm.NC = (p->T + 63) / 64;
  vm.packed_total = 0;
  auto with_carry = [&](FwdArgs x) {
    if (carry_in) {
      x.S_in = carry_in->S; x.kprev_in = carry_in->k_prev; x.pos_in = carry_in->pos;
      if (x.W > 1) { x.winx_in = carry_in->win_x; x.winv_in = carry_in->win_v; }
    }
    return x;
  };
  const FwdArgs au = with_carry(make_args(p, q, k, v, beta, lambda, o, stream));
  const bool in_place = total_tokens > 0 && W == 1 && resolve_impl(p, au) == FALCON_IMPL_TC &&
                        tc_chunk_takes_map(au) && (!p->prologue || prologue_fused(p, q, k, v));
  if (in_place) {
    vm.packed_total = total_tokens;
    st = launch_varlen_item_map(cu_seqlens, p->B, p->H, vm.NC, const_cast<int32_t*>(vm.item_map), s);
    if (st != FALCON_OK) return st;
    st = chunk_fwd_impl(p, q, k, v, beta, lambda, carry_in, o, &co_state, kws ? workspace : nullptr, kws,
                        stream, nullptr, 0, &vm);
    if (st != FALCON_OK) return st;
    return launch_varlen_finish(pa, nullptr, o, W, shift, carry_in, carry_out, s);
  }
  void* o_pad = nullptr;
  prologue_carve(pa, reinterpret_cast<uint8_t*>(workspace) + kws, true, &o_pad);
  falcon_params_t p0 = *p;
  p0.prologue = 0;
  const FwdArgs ad = with_carry(make_args(&p0, pa.qo, pa.ko, pa.vo, pa.bo, pa.lo, o_pad, stream));
  const bool mapped = resolve_impl(&p0, ad) == FALCON_IMPL_TC && tc_chunk_takes_map(ad);
  pa.skip_tail = mapped ? 1 : 0;
  st = launch_prologue(pa, s);
  if (st != FALCON_OK) return st;
  if (mapped) {
    st = launch_varlen_item_map(cu_seqlens, p->B, p->H, vm.NC, const_cast<int32_t*>(vm.item_map), s);
    if (st != FALCON_OK) return st;
  }
  st = chunk_fwd_impl(&p0, pa.qo, pa.ko, pa.vo, pa.bo, pa.lo, carry_in, o_pad, &co_state,
                      kws ? workspace : nullptr, kws, stream, nullptr, 0, mapped ? &vm : nullptr);
  if (st != FALCON_OK) return st;
  return launch_varlen_finish(pa, o_pad, o, W, shift, carry_in, carry_out, s);
}

int falcon_recurrent_step(const falcon_params_t* p, const void* q, const void* k, const void* v,
                          const float* beta, const float* lambda, falcon_carry_t* carry, void* o,
                          void* stream) {
  int st = check_params(p, true);
  if (st != FALCON_OK) return st;
  if (p->T != 1) return FALCON_ERR_INVALID_ARG;
  if (!q || !k || !v || !beta || !lambda || !o || !carry || !carry->S || !carry->k_prev || !carry->pos)
    return FALCON_ERR_INVALID_ARG;
  FwdArgs a = make_args(p, q, k, v, beta, lambda, o, stream);
  a.prologue = p->prologue;
  if (a.W > 1 && (!carry->win_x || !carry->win_v)) return FALCON_ERR_INVALID_ARG;
  a.S_in = a.S_out = carry->S;
  a.kprev_in = a.kprev_out = carry->k_prev;
  a.pos_in = a.pos_out = carry->pos;
  if (a.W > 1) { a.winx_in = a.winx_out = carry->win_x; a.winv_in = a.winv_out = carry->win_v; }
  return launch_recurrent_step(a);
}

size_t falcon_masked_parallel_workspace_size(const falcon_params_t* p) {
  if (check_params(p, true) != FALCON_OK) return 0;
  const int W = effective_window(p->variant, p->window);
  return masked_parallel_ws_bytes(p->B, p->T, p->H, p->dk, p->dv, W);
}

int falcon_masked_parallel_ref_gpu(const falcon_params_t* p, const void* q, const void* k,
                                   const void* v, const float* beta, const float* lambda, void* o,
                                   float* S_final, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  int st = check_params(p, true);
  if (st != FALCON_OK) return st;
  if (!q || !k || !v || !beta || !lambda || !o || !S_final) return FALCON_ERR_INVALID_ARG;
  if (p->prologue) return FALCON_ERR_UNSUPPORTED;  // takes features and gates
  const int W = effective_window(p->variant, p->window);
  if (p->T > 1024 || (size_t)p->T * W > 2048) return FALCON_ERR_UNSUPPORTED;
  const size_t need = masked_parallel_ws_bytes(p->B, p->T, p->H, p->dk, p->dv, W);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return FALCON_ERR_WORKSPACE;
  FwdArgs a = make_args(p, q, k, v, beta, lambda, o, stream);
  a.S_out = S_final;
  a.ws = workspace; a.ws_bytes = workspace_bytes;
  return launch_masked_parallel(a);
}

size_t falcon_backward_workspace_size(const falcon_params_t* p) {
  if (check_params(p, false) != FALCON_OK || !backward_supported(p->variant, p->dk, p->dv, p->window) ||
      p->prologue)
    return 0;
  return backward_ws_bytes(p->variant, p->B, p->T, p->H, p->dk, p->window);
}

int falcon_backward_carry(const falcon_params_t* p, const void* q, const void* k, const void* v,
                          const float* beta, const float* lambda, const falcon_carry_t* carry_in,
                          const void* dO, const float* dS_final, void* dq, void* dk, void* dv, float* dbeta,
                          float* dlambda, const falcon_carry_t* dcarry, void* workspace, size_t workspace_bytes,
                          void* stream) {
  int st = check_params(p, false);
  if (st != FALCON_OK) return st;
  if (!backward_supported(p->variant, p->dk, p->dv, p->window) || p->prologue) return FALCON_ERR_UNSUPPORTED;
  if (p->T > 0 && (!q || !k || !v || !beta || !lambda || !dO || !dq || !dk || !dv || !dbeta || !dlambda))
    return FALCON_ERR_INVALID_ARG;
  const size_t need = backward_ws_bytes(p->variant, p->B, p->T, p->H, p->dk, p->window);
  if (need > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0))
    return FALCON_ERR_WORKSPACE;
  FwdArgs a = make_args(p, q, k, v, beta, lambda, nullptr, stream);
  const int Wr = a.W - 1;
  if (carry_in) {
    a.S_in = carry_in->S; a.kprev_in = carry_in->k_prev; a.pos_in = carry_in->pos;
    if (Wr > 0) { a.winx_in = carry_in->win_x; a.winv_in = carry_in->win_v; }
    if ((a.winx_in == nullptr) != (a.winv_in == nullptr)) return FALCON_ERR_INVALID_ARG;
  }
  float* dS_in = dcarry ? dcarry->S : nullptr;
  void* dk_prev = dcarry ? dcarry->k_prev : nullptr;
  void* dwin_x = dcarry && Wr > 0 ? dcarry->win_x : nullptr;
  void* dwin_v = dcarry && Wr > 0 ? dcarry->win_v : nullptr;
  if ((dwin_x == nullptr) != (dwin_v == nullptr)) return FALCON_ERR_INVALID_ARG;
  // the gradients must not overlap the inputs or one another
  const size_t es = elem_size(p->dtype), BH = (size_t)p->B * p->H, BTH = BH * p->T;
  const size_t nbeta = BTH * (variant_per_channel(p->variant) ? p->dv : 1) * 4;
  const size_t nring_x = BH * (Wr > 0 ? Wr : 0) * p->dk * es, nring_v = BH * (Wr > 0 ? Wr : 0) * p->dv * es;
  const void* ins[11] = {q, k, v, beta, lambda, dO, dS_final, a.S_in, a.kprev_in, a.winx_in, a.winv_in};
  const size_t nin[11] = {BTH * p->dk * es, BTH * p->dk * es, BTH * p->dv * es, nbeta, BTH * 4,
                          BTH * p->dv * es, BH * p->dk * p->dv * 4, BH * p->dk * p->dv * 4, BH * p->dk * es,
                          nring_x, nring_v};
  const void* outs[9] = {dq, dk, dv, dbeta, dlambda, dS_in, dk_prev, dwin_x, dwin_v};
  const size_t nout[9] = {BTH * p->dk * es, BTH * p->dk * es, BTH * p->dv * es, nbeta, BTH * 4,
                          BH * p->dk * p->dv * 4, BH * p->dk * es, nring_x, nring_v};
  for (int i = 0; i < 9; ++i) {
    for (int j = 0; j < 11; ++j)
      if (overlaps(outs[i], nout[i], ins[j], nin[j])) return FALCON_ERR_INVALID_ARG;
    for (int j = i + 1; j < 9; ++j)
      if (overlaps(outs[i], nout[i], outs[j], nout[j])) return FALCON_ERR_INVALID_ARG;
  }
  a.ws = workspace; a.ws_bytes = workspace_bytes;
  return launch_backward(a, dO, dS_final, dq, dk, dv, dbeta, dlambda, dS_in, dk_prev, dwin_x, dwin_v);
}

int falcon_backward(const falcon_params_t* p, const void* q, const void* k, const void* v,
                    const float* beta, const float* lambda, const falcon_carry_t* carry_in,
                    const void* dO, const float* dS_final, void* dq, void* dk, void* dv,
                    float* dbeta, float* dlambda, float* dS_in, void* dk_prev, void* workspace,
                    size_t workspace_bytes, void* stream) {
  falcon_carry_t dc;
  dc.S = dS_in; dc.k_prev = dk_prev; dc.win_x = nullptr; dc.win_v = nullptr; dc.pos = nullptr;
  return falcon_backward_carry(p, q, k, v, beta, lambda, carry_in, dO, dS_final, dq, dk, dv, dbeta, dlambda, &dc,
                               workspace, workspace_bytes, stream);
}

}  // extern "C"
