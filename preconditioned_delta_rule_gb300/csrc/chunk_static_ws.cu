// chunk_static_ws.cu -- osdn_chunk_fwd_static_ws: the chunk forward with no allocation at all.
//
// osdn_chunk_fwd's fast tensor-core path needs 32.5 KiB of scratch per chunk of each head, which the
// caller normally passes in.  Some callers cannot allocate device memory when they call: an
// engine that reserves all GPU memory in one plan at start-up and must not allocate afterwards,
// or code that cannot accept an allocator call (its latency, its implicit synchronisation, or its
// possible failure) in the middle of a step.  For them this entry point uses a fixed scratch
// array that lives in the library's own device memory instead.
#include "common.cuh"

namespace {

// Capacity: 1008 chunks of one head (33280 bytes each), e.g. 15 heads x 4096 tokens.
constexpr size_t kStaticWsBytes = static_cast<size_t>(32) << 20;

// File-scope device scratch.  Every GPU that loads this library holds these 32 MiB until the
// process exits.  In host code `g_chunk_ws` only names the symbol: its device address on the
// current device comes from cudaGetSymbolAddress, looked up on every call (it allocates nothing,
// and a fresh lookup stays valid if the device's context was torn down and made again).
static __device__ __align__(256) unsigned char g_chunk_ws[kStaticWsBytes];

}  // namespace

extern "C" {

osdn_status osdn_chunk_fwd_static_ws(const void* q, const void* k, const void* k_tilde, const void* v,
                                     osdn_dtype dtype, const float* beta, const float* alpha, int alpha_per_key,
                                     const float* S0, void* o,
                                     float* S_out, int B, int T, int H, int K, int V, int chunk,
                                     float scale, void* stream) {
    // the same argument checks as osdn_chunk_fwd, before the capacity test
    OsdnChunkArgs a{};
    bool empty = false;
    const osdn_status st = osdn_chunk_validate(q, k, k_tilde, v, dtype, beta, alpha, alpha_per_key, S0, o, S_out, B,
                                               T, H, K, V, chunk, scale, &a, &empty);
    if (st != OSDN_OK || empty) return st;
    // scratch only where the tensor-core path runs (a channel gate or fp32 inputs take the
    // CUDA-core kernel, which needs none)
    const size_t need = osdn_chunk_scratch_bytes(a);
    if (need > kStaticWsBytes) return OSDN_ERR_CAPACITY;
    void* ws = nullptr;
    if (need > 0) {
        // Everything the two kernels read from the scratch is written earlier in the same call,
        // so nothing needs clearing between calls.
        if (cudaGetSymbolAddress(&ws, g_chunk_ws) != cudaSuccess) return OSDN_ERR_CUDA;
    }
    return osdn_chunk_fwd(q, k, k_tilde, v, dtype, beta, alpha, alpha_per_key, S0, o, S_out, B, T, H, K, V, chunk,
                          scale, ws, need, stream);
}

}  // extern "C"
