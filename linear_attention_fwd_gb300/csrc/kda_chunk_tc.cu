// KDA chunkwise forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {

bool chunk_tc_supported(int, int, kda_dtype_t) { return false; }

cudaError_t launch_chunk_tc(const ChunkArgs &, int, int, kda_dtype_t, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace kda
