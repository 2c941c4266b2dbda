// chunk_tc.cu -- tensor-core (TMA + tcgen05/TMEM) kernel for phase 2 of OSDN.
#include "common.cuh"

namespace osdn {
// Set by any kernel of this library whose bounded device-side wait gave up.
__device__ unsigned int g_timeout_flag = 0;
}  // namespace osdn

cudaError_t osdn_launch_chunk_tc(const OsdnChunkArgs&, cudaStream_t) { return cudaErrorNotSupported; }

cudaError_t osdn_read_and_clear_timeout(unsigned int* flag, cudaStream_t s) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(flag, osdn::g_timeout_flag, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    if (*flag) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(osdn::g_timeout_flag, &zero, sizeof(unsigned int));
    }
    return e;
}
