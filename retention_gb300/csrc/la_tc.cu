// la_tc.cu -- placeholder until the tensor-core kernel lands.
#include "la_common.cuh"
namespace la {
bool chunk_tc_supports(const ChunkArgs &) { return false; }
int launch_chunk_tc(const ChunkArgs &, cudaStream_t, int *) { return LA_ERR_UNSUPPORTED; }
}  // namespace la
