// Shared device/host helpers of the Falcon GB300 library (internal).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <utility>

#include "falcon.h"

namespace falcon {

// ---------------------------------------------------------------- dtypes
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__host__ __device__ inline bool variant_additive(int v) {
  return v == FALCON_1A || v == FALCON_2A || v == FALCON_3A;
}
__host__ __device__ inline bool variant_per_channel(int v) { return v == FALCON_2 || v == FALCON_2A; }
__host__ __device__ inline bool variant_windowed(int v) { return v == FALCON_3 || v == FALCON_3A; }
__host__ __device__ inline int effective_window(int v, int w) { return variant_windowed(v) ? w : 1; }

// Decay with the positive-decay floor: gamma = clamp(1 - lambda, eps_gamma, 1);
// its log is then >= log(eps_gamma) > -inf.
__device__ __forceinline__ float clamped_log_decay(float lam, float eps_gamma) {
  float g = fminf(fmaxf(1.0f - lam, eps_gamma), 1.0f);
  return logf(g);
}

// Ring slot of the pair with global index p (p >= 1) in a ring of Wr slots.
__host__ __device__ inline int ring_slot(int64_t p, int Wr) { return (int)(p % (int64_t)Wr); }

// Everything one chunk-forward call needs, resolved on the host.
struct FwdArgs {
  int B, T, H, dk, dv, chunk, W;  // W: effective window (1 outside Falcon-3/3A)
  float eps, eps_gamma;
  int variant, dtype;
  int shift;                // pair t uses key t - shift: 1 prefix alignment, 0 same-step
  const void* q;
  const void* k;
  const void* v;
  const float* beta;
  const float* lam;
  const float* S_in;        // may be NULL (zero state)
  const void* kprev_in;     // may be NULL (zero key)
  const void* winx_in;      // may be NULL
  const void* winv_in;      // may be NULL
  const int64_t* pos_in;    // may be NULL (pos = 0)
  void* o;
  float* S_out;             // may be NULL
  void* kprev_out;          // may be NULL
  void* winx_out;           // may be NULL
  void* winv_out;           // may be NULL
  int64_t* pos_out;         // may be NULL
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
  cudaEvent_t* events;      // optional: recorded before the first and after every kernel
  int n_events;
  int prologue;             // falcon_prologue_t flags applied inside the kernel (recurrent step)
  // packed sequences (varlen): sequence b's tokens are rows 0 .. len_b - 1
  // of batch row b of a padded batch, or (packed_total > 0) rows cu[b] ..
  // cu[b+1] - 1 of the packed tensors; the Falcon-1 / 1A d = 64 tensor-core
  // kernels skip the chunks past its last (NULL: dense)
  const int32_t* cu;
  const int32_t* item_map;  // the (b, h, chunk) items that hold tokens, as (b H + h) NC + chunk
  const int32_t* item_count;
  int64_t packed_total;     // > 0: q, k, v, beta, lambda, o are the packed rows themselves (that many)
};

// Gates with the optional logit prologue: gamma = clamp(1 - lambda) or
// clamp(sigmoid(-a)); beta or sigmoid(b).
__device__ __forceinline__ float gate_gamma(float lam, float eps_gamma, int prologue) {
  const float g = (prologue & FALCON_PROLOGUE_GATE_LOGITS) ? 1.f / (1.f + __expf(lam)) : 1.0f - lam;
  return fminf(fmaxf(g, eps_gamma), 1.0f);
}
__device__ __forceinline__ float gate_beta(float b, int prologue) {
  return (prologue & FALCON_PROLOGUE_GATE_LOGITS) ? 1.f / (1.f + __expf(-b)) : b;
}

// Inputs of the prologue / varlen gather and its dense outputs.
struct ProArgs {
  int B, T, H, dk, dv, dtype, flags, perch;
  const int32_t* cu;        // NULL: dense rows (b, t) at b * T + t; else packed sequences
  const void* q;
  const void* k;
  const void* v;
  const float* beta;
  const float* lam;
  void* qo;
  void* ko;
  void* vo;
  float* bo;
  float* lo;
  int skip_tail;            // packed sequences: rows of the chunks past a sequence's last are not written
};
size_t prologue_ws_bytes(int B, int T, int H, int dk, int dv, int dtype, bool perch, bool with_o);
void prologue_carve(ProArgs& a, void* base, bool with_o, void** o_pad);
int launch_prologue(const ProArgs& a, cudaStream_t s);
int launch_varlen_finish(const ProArgs& a, const void* o_pad, void* o, int W, int shift,
                         const falcon_carry_t* ci, falcon_carry_t* co, cudaStream_t s);
// Whether launch_tc_chunk runs the Falcon-1 / 1A d = 64 kernels for these
// args (the path that takes a packed-sequence chunk map), and the kernel that
// builds that map (B H NC + B + 2 int32) from cu_seqlens.
bool tc_chunk_takes_map(const FwdArgs& a);
int launch_varlen_item_map(const int32_t* cu, int B, int H, int NC, int32_t* map, cudaStream_t s);

// Record the caller's event i on the stream (no-op without events).
inline void record_event(const FwdArgs& a, int i) {
  if (a.events && i < a.n_events) cudaEventRecord(a.events[i], a.stream);
}

// Launchers (each returns a FALCON_* code; host-side checks only).
int launch_generic_chunk(const FwdArgs& a);
size_t generic_chunk_smem_bytes(int dk, int dvs, int c, int W);
int launch_recurrent_step(const FwdArgs& a);
int launch_masked_parallel(const FwdArgs& a);
size_t masked_parallel_ws_bytes(int B, int T, int H, int dk, int dv, int W);
int launch_tc_chunk(const FwdArgs& a);
bool tc_chunk_supported(const FwdArgs& a);
int tc_chunk_launches(const FwdArgs& a);
size_t tc_chunk_ws_bytes(int B, int T, int H, int dk, int dv, int chunk, int variant);
bool tc_f2_supported(const FwdArgs& a);
int launch_tc_f2(const FwdArgs& a);
bool tc_f3a_supported(const FwdArgs& a);
int launch_tc_f3a(const FwdArgs& a);
size_t tc_f3a_ws_bytes(int B, int T, int H);
int tc_f3a_launches(const FwdArgs& a);  // 2, or 3 when the chain runs in groups
bool tc_f3_supported(const FwdArgs& a);
int launch_tc_f3(const FwdArgs& a);
size_t tc_f3_ws_bytes(int B, int T, int H);
bool window_scan_supported(const FwdArgs& a);
size_t window_scan_ws_bytes(int B, int T, int H, int W);
int launch_window_scan(const FwdArgs& a);
size_t backward_ws_bytes(int variant, int B, int T, int H, int d, int window);
bool backward_chunk_supported(int variant, int dk, int dv, int T);
size_t backward_chunk_ws_bytes(int B, int T, int H);
int launch_backward_chunk(const FwdArgs& f, const void* dO, const float* dS_final, void* dq, void* dk,
                          void* dv, float* dbeta, float* dlam, float* dS_in, void* dk_prev);
bool backward_supported(int variant, int dk, int dv, int window);
int launch_backward(const FwdArgs& f, const void* dO, const float* dS_final, void* dq, void* dk,
                    void* dv, float* dbeta, float* dlam, float* dS_in, void* dk_prev, void* dwin_x,
                    void* dwin_v);
bool backward_window_supported(int variant, int dk, int dv, int window);
size_t backward_window_ws_bytes(int B, int T, int H, int d, int window);
int launch_backward_window(const FwdArgs& f, const void* dO, const float* dS_final, void* dq, void* dk,
                           void* dv, float* dbeta, float* dlam, float* dS_in, void* dk_prev, void* dwin_x,
                           void* dwin_v);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Limit of the bounded device-side waits of the next launch (2 s unless the
// failure-detection test hook set another), and whether that hook asked the
// next Falcon-1 / 1A, 3 or 3A tensor-core call to stall one wait (consumed here).
uint64_t wait_limit_ns();
bool take_test_stall();
// Device address of the allocation-free entry point's scratch array on the
// current device (its first 4 bytes are that entry point's status word).
int noalloc_scratch(void** out);

// Raise a kernel's dynamic shared-memory limit, once per kernel and device
// (the attribute call costs host time on every launch otherwise).
inline bool set_smem_limit(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(kernel, dev);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess)
    return false;
  done[key] = bytes;
  return true;
}

}  // namespace falcon
