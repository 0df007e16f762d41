// Chunk forward for callers that cannot allocate device memory.
//
// Some hosts hand a kernel library nothing but input/output pointers and a
// stream: plugin interfaces of inference runtimes that expose no allocator,
// or services that fix their memory budget at start-up and forbid any
// allocation while serving.  Such callers cannot provide the scratch buffer
// falcon_chunk_fwd asks for.  This entry point runs the same tensor-core
// kernels with their scratch in a fixed array that lives in the library's
// own device image instead.

#include "common.cuh"

namespace {

// 32 MiB: enough for every call whose falcon_workspace_size is at most that,
// i.e. B * H * ceil(T / 64) <= 1927 chunks at d = 64 (16 KB of bf16 images +
// 1 KB of gates per chunk) and <= 992 chunks at d = 128 (32 KB + 1 KB), after
// a 256-byte status word.  Every device that loads the library holds this
// array until exit.
constexpr size_t kScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

}  // namespace

namespace falcon {

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from the
// runtime; it is looked up on every call (cheap once the library's device
// code is loaded on the device) so that it stays right if the module is
// loaded again, e.g. after a cudaDeviceReset.
int noalloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FALCON_ERR_CUDA;
  *out = p;
  return FALCON_OK;
}

}  // namespace falcon

extern "C" int falcon_chunk_fwd_noalloc(const falcon_params_t* p, const void* q, const void* k,
                                        const void* v, const float* beta, const float* lambda,
                                        const falcon_carry_t* carry_in, void* o,
                                        falcon_carry_t* carry_out, void* stream) {
  // covered: the Falcon-1 / Falcon-1A tensor-core path (the kernels that keep
  // per-chunk images in the scratch)
  if (p && ((p->variant != FALCON_1 && p->variant != FALCON_1A) || p->prologue)) return FALCON_ERR_UNSUPPORTED;
  int32_t impl = 0;
  int st = falcon_chunk_fwd_plan(p, &impl, nullptr);
  if (st != FALCON_OK) return st;
  if (impl != FALCON_IMPL_TC) return FALCON_ERR_UNSUPPORTED;
  if (falcon_workspace_size(p) > kScratchBytes) return FALCON_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = falcon::noalloc_scratch(&scratch);
  if (st != FALCON_OK) return st;
  // the status word is the one part of the scratch that must start at zero
  if (cudaMemsetAsync(scratch, 0, 256, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FALCON_ERR_CUDA;
  return falcon_chunk_fwd(p, q, k, v, beta, lambda, carry_in, o, carry_out, scratch, kScratchBytes,
                          stream);
}
