// varlen.cu -- packed variable-length sequences (cu_seqlens) for the layer forward.
//
// "OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention": the
// recurrence of Algorithm 1 / Eqs. (2), (4), (7) runs per sequence; packed prefill concatenates
// N sequences along the token axis, sequence n owning rows cu[n] .. cu[n+1]-1, each starting from
// its own d0[n], S0[n] and ending in its own d_out[n], S_out[n].
//
// The sequences are scattered into an [N, Tp, H, .] batch (Tp = max_len rounded up to the chunk)
// and the batched layer forward runs on it.  A padding token carries k = q = v = 0, beta = 0,
// retention 1 and state gate 1, which leaves both states exactly unchanged: its phase-1 step is
// g s with s = k . k = 0, and in phase 2 its row of A and of T' = T diag(beta) is zero, so its rows
// of U, W and X are zero and it adds nothing to S.  Padding only follows a sequence's last token,
// so no real token reads a padded one (every intra-chunk product is causal).  The outputs o and k~
// of the real tokens are gathered back; a sequence of length 0 returns its d0 (ones) and S0
// (zeros) as given.
//
// Every cu_seqlens entry is checked on the device (0 <= cu[n] <= cu[n+1] <= total, length <= Tp);
// a sequence that fails is treated as empty (nothing is read or written for it) and a flag is
// raised that osdn_check reports as OSDN_ERR_SHAPE.
#include <stdint.h>

#include "common.cuh"

namespace osdn {

__device__ unsigned int g_varlen_bad = 0;

namespace {

constexpr int kMaxTensors = 6;
constexpr int kThreads = 256;

struct PackTensor {
    const unsigned char* packed;  // [total, row_bytes]
    unsigned char* padded;        // [N * Tp, row_bytes]
    long long row_bytes;          // a multiple of 4
    uint32_t fill;                // padding word (0, or the bits of 1.0f)
};
struct PackArgs {
    PackTensor t[kMaxTensors];
    int nt;
    const int* cu;
    int N, Tp;
    long long total;
};

// Length of sequence n, or -1 (and the flag raised) when its cu entries are not a valid range.
__device__ __forceinline__ int seq_len(const int* cu, int n, long long total, int Tp, int& start) {
    const int s = cu[n], e = cu[n + 1];
    if (s < 0 || e < s || static_cast<long long>(e) > total || e - s > Tp) {
        atomicExch(&g_varlen_bad, 1u);
        return -1;
    }
    start = s;
    return e - s;
}

template <typename W>
__device__ __forceinline__ void copy_words(const unsigned char* src, unsigned char* dst, long long bytes, int lane) {
    const W* s = reinterpret_cast<const W*>(src);
    W* d = reinterpret_cast<W*>(dst);
    const int n = static_cast<int>(bytes / static_cast<long long>(sizeof(W)));
    for (int w = lane; w < n; w += 32) d[w] = s[w];
}
template <typename W>
__device__ __forceinline__ void fill_words(unsigned char* dst, long long bytes, uint32_t fill, int lane) {
    W v;
    uint32_t* p = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int i = 0; i < static_cast<int>(sizeof(W) / 4); ++i) p[i] = fill;
    W* d = reinterpret_cast<W*>(dst);
    const int n = static_cast<int>(bytes / static_cast<long long>(sizeof(W)));
    for (int w = lane; w < n; w += 32) d[w] = v;
}

// One warp per padded row p = (n, t), grid-stride over the rows: every tensor's row is copied from
// packed row cu[n] + t when t is within sequence n, else filled with its padding word.
__global__ void __launch_bounds__(kThreads) pack_kernel(PackArgs a) {
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(a.N) * a.Tp;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    for (long long p = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); p < rows; p += warps) {
        const int n = static_cast<int>(p / a.Tp), t = static_cast<int>(p - static_cast<long long>(n) * a.Tp);
        int start = 0;
        const int len = seq_len(a.cu, n, a.total, a.Tp, start);
        for (int i = 0; i < a.nt; ++i) {
            const PackTensor& x = a.t[i];
            unsigned char* dst = x.padded + p * x.row_bytes;
            const bool v16 = (x.row_bytes & 15) == 0;
            if (t < len) {
                const unsigned char* src = x.packed + (static_cast<long long>(start) + t) * x.row_bytes;
                if (v16) copy_words<uint4>(src, dst, x.row_bytes, lane);
                else copy_words<uint32_t>(src, dst, x.row_bytes, lane);
            } else {
                if (v16) fill_words<uint4>(dst, x.row_bytes, x.fill, lane);
                else fill_words<uint32_t>(dst, x.row_bytes, x.fill, lane);
            }
        }
    }
}

struct UnpackArgs {
    PackTensor t[2];  // o and k~: padded -> packed, real rows only
    int nt;
    const int* cu;
    int N, Tp;
    long long total;
    const float* d0;  // [N, H*K] or null (ones)
    float* d_out;     // [N, H*K]
    int HK;
};

// The real rows of o and k~ back to the packed layout (one warp per padded row); for a sequence
// of length 0, d_out = d0.
__global__ void __launch_bounds__(kThreads) unpack_kernel(UnpackArgs a) {
    const int lane = threadIdx.x & 31;
    const long long rows = static_cast<long long>(a.N) * a.Tp;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    for (long long p = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); p < rows; p += warps) {
        const int n = static_cast<int>(p / a.Tp), t = static_cast<int>(p - static_cast<long long>(n) * a.Tp);
        int start = 0;
        const int len = seq_len(a.cu, n, a.total, a.Tp, start);
        if (t == 0 && len == 0) {
            for (int e = lane; e < a.HK; e += 32)
                a.d_out[static_cast<long long>(n) * a.HK + e] = a.d0 ? a.d0[static_cast<long long>(n) * a.HK + e] : 1.f;
        }
        if (t >= len) continue;
        for (int i = 0; i < a.nt; ++i) {
            const PackTensor& x = a.t[i];
            const unsigned char* src = x.padded + p * x.row_bytes;
            unsigned char* dst = const_cast<unsigned char*>(x.packed) + (static_cast<long long>(start) + t) * x.row_bytes;
            if ((x.row_bytes & 15) == 0) copy_words<uint4>(src, dst, x.row_bytes, lane);
            else copy_words<uint32_t>(src, dst, x.row_bytes, lane);
        }
    }
}

int grid_for(long long rows) {  // one warp per row, grid-stride
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long cap = static_cast<long long>(sms) * 8;
    const long long need = (rows + kThreads / 32 - 1) / (kThreads / 32);
    return static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
}

}  // namespace
}  // namespace osdn

size_t osdn_varlen_pad_bytes(const OsdnVarlenShape& v) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t rows = static_cast<size_t>(v.N) * v.Tp;
    const size_t e = v.elt;
    size_t b = 0;
    b += 3 * up(rows * v.H * v.K * e);          // q, k, k~
    b += 2 * up(rows * v.H * v.V * e);          // v, o
    b += up(rows * v.H * 4);                    // beta
    if (v.r_mode == 1) b += up(rows * v.H * 4);
    if (v.r_mode == 2) b += up(rows * v.H * v.K * 4);
    if (v.gated) b += up(rows * v.H * (v.gated == 2 ? v.K : 1) * 4);  // alpha
    return b;
}

cudaError_t osdn_launch_varlen_pack(const OsdnVarlenIo& io, const OsdnVarlenShape& v, cudaStream_t s) {
    using namespace osdn;
    PackArgs a{};
    const long long e = v.elt;
    const uint32_t one = 0x3f800000u;
    int i = 0;
    a.t[i++] = {static_cast<const unsigned char*>(io.q), static_cast<unsigned char*>(io.pq), v.H * v.K * e, 0u};
    a.t[i++] = {static_cast<const unsigned char*>(io.k), static_cast<unsigned char*>(io.pk), v.H * v.K * e, 0u};
    a.t[i++] = {static_cast<const unsigned char*>(io.v), static_cast<unsigned char*>(io.pv), v.H * v.V * e, 0u};
    a.t[i++] = {reinterpret_cast<const unsigned char*>(io.beta), reinterpret_cast<unsigned char*>(io.pbeta), v.H * 4LL, 0u};
    if (io.r) a.t[i++] = {reinterpret_cast<const unsigned char*>(io.r), reinterpret_cast<unsigned char*>(io.pr),
                          v.H * (v.r_mode == 2 ? v.K : 1) * 4LL, one};
    if (io.alpha) a.t[i++] = {reinterpret_cast<const unsigned char*>(io.alpha), reinterpret_cast<unsigned char*>(io.palpha),
                              v.H * (v.gated == 2 ? v.K : 1) * 4LL, one};
    a.nt = i;
    a.cu = io.cu;
    a.N = v.N;
    a.Tp = v.Tp;
    a.total = v.total;
    const long long rows = static_cast<long long>(v.N) * v.Tp;
    pack_kernel<<<grid_for(rows), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t osdn_launch_varlen_unpack(const OsdnVarlenIo& io, const OsdnVarlenShape& v, cudaStream_t s) {
    using namespace osdn;
    UnpackArgs a{};
    const long long e = v.elt;
    a.t[0] = {static_cast<const unsigned char*>(io.o), static_cast<unsigned char*>(io.po), v.H * v.V * e, 0u};
    a.t[1] = {static_cast<const unsigned char*>(io.k_tilde), static_cast<unsigned char*>(io.pkt), v.H * v.K * e, 0u};
    a.nt = 2;
    a.cu = io.cu;
    a.N = v.N;
    a.Tp = v.Tp;
    a.total = v.total;
    a.d0 = io.d0;
    a.d_out = io.d_out;
    a.HK = v.H * v.K;
    const long long rows = static_cast<long long>(v.N) * v.Tp;
    unpack_kernel<<<grid_for(rows), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t osdn_varlen_read_and_clear_flag(unsigned int* flag) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flag, osdn::g_varlen_bad, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    if (*flag) e = cudaMemcpyToSymbol(osdn::g_varlen_bad, &zero, sizeof(unsigned int));
    return e;
}
