// Tensor-core chunk forward (placeholder until the tcgen05 kernels land).
#include "common.cuh"

namespace falcon {

bool tc_chunk_supported(const FwdArgs&) { return false; }
int tc_chunk_launches(const FwdArgs&) { return 0; }
size_t tc_chunk_ws_bytes(int, int, int, int, int, int, int) { return 0; }
int launch_tc_chunk(const FwdArgs&) { return FALCON_ERR_UNSUPPORTED; }

}  // namespace falcon
