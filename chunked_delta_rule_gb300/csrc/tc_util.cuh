// Device and host helpers shared by the tensor-core kernels (internal):
// shared-memory alignment, bf16 packing, named barriers, UMMA chains and
// descriptors over 128B-swizzled tiles, TMEM row loads and stores, and the
// TMA tensor maps of the [B, T, H, D] activations.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace falcon {
namespace tcu {

using namespace tc;

constexpr int kC = 64;                    // chunk length of the tensor-core paths
constexpr uint32_t kStatusTimeout = 1;    // workspace status: a bounded wait gave up

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barrier that also returns whether any participating thread passed
// `pred`: every thread takes the same branch after it.
__device__ __forceinline__ bool named_bar_any(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Issue a chain of K/16 MMAs: D = A (M rows, K) * B (N rows, K)^T, both K-major
// 128B-swizzled; K beyond 64 continues in the next 64-column slab.
__device__ __forceinline__ void mma_chain(uint32_t d_tmem, const uint8_t* A, int a_rows,
                                          const uint8_t* Bm, int b_rows, int K, uint32_t idesc,
                                          bool accumulate) {
  const uint32_t a0 = smem_u32(A), b0 = smem_u32(Bm);
  for (int ks = 0; ks < K / 16; ++ks) {
    const uint32_t off = (ks & 3) * 32;
    const uint32_t slab = ks >> 2;
    const uint64_t ad = sdesc_k128(a0 + slab * a_rows * 128 + off);
    const uint64_t bd = sdesc_k128(b0 + slab * b_rows * 128 + off);
    umma_bf16(d_tmem, ad, bd, idesc, (ks > 0 || accumulate) ? 1u : 0u);
  }
}

// Load 64 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
  tmem_ld32(taddr + 32, r);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[32 + i] = __uint_as_float(r[i]);
}

// MN-major operand chain: D = A^T-or-B with 64 elements along M/N, K rows of
// 128 B in the swizzled layout; K steps of 16 rows = 2048 B.
__device__ __forceinline__ void mma_chain_mn(uint32_t d_tmem, uint64_t (*adesc)(uint32_t, int),
                                             uint32_t a0, uint64_t (*bdesc)(uint32_t, int),
                                             uint32_t b0, int K, uint32_t idesc, bool accumulate) {
  for (int ks = 0; ks < K / 16; ++ks)
    umma_bf16(d_tmem, adesc(a0, ks), bdesc(b0, ks), idesc, (ks > 0 || accumulate) ? 1u : 0u);
}
// descriptor of K step ks for a K-major operand (64-col slabs of `rows` rows)
template <int ROWS>
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int ks) {
  return sdesc_k128(base + (ks >> 2) * ROWS * 128 + (ks & 3) * 32);
}
// descriptor of K step ks for an MN-major operand (16 K rows per step)
__device__ __forceinline__ uint64_t mndesc(uint32_t base, int ks) {
  return sdesc_mn128(base + ks * 2048);
}

// Row r (K-major or MN-major rows of 64 bf16 are the same swizzled image):
// write 64 fp32 values as bf16 with 16-byte stores.
__device__ __forceinline__ void store_row64(uint8_t* tile, int r, const float* v) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t pk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) pk[e] = pack_bf16(v[8 * j + 2 * e], v[8 * j + 2 * e + 1]);
    *reinterpret_cast<uint4*>(tile + sw128(r, 8 * j)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// 32 lanes x 16 consecutive fp32 columns from TMEM (the thread's lane).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns from registers to TMEM (the
// thread's lane of the warp's quadrant).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- host side
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

inline EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// [B, T, H, D] bf16 tensor, box of 64 columns x `rows` time steps.
inline bool make_map(CUtensorMap* m, const void* base, int B, int T, int H, int D, int rows) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)T * H * D * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B, T, H, D] fp32 tensor without swizzle, box of `cols` columns x `rows`
// time steps (D * 4 bytes must be a multiple of 16).
inline bool make_map_f32(CUtensorMap* m, const void* base, int B, int T, int H, int D, int cols, int rows) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4, (cuuint64_t)T * H * D * 4};
  cuuint32_t box[4] = {(cuuint32_t)cols, 1, (cuuint32_t)rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Streaming multiprocessors of the current device (looked up once per device).
inline int sm_count() {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

// Launch overlapping the stream's previous grid (programmatic stream
// serialization): the kernel waits for it in hardware (griddepcontrol.wait)
// before it reads what that grid wrote.  Plain launch when the caller times
// each kernel with events.
template <typename Kern, typename... Args>
inline int launch_overlapped(const FwdArgs& fa, Kern k, dim3 grid, dim3 block, size_t smem, Args... args) {
  if (fa.events) {
    k<<<grid, block, smem, fa.stream>>>(args...);
    return cudaGetLastError() == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = fa.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...) == cudaSuccess ? FALCON_OK : FALCON_ERR_CUDA;
}

}  // namespace tcu
}  // namespace falcon
