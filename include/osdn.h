/*
 * osdn.h -- C ABI of the GB300 (sm_103a) OSDN forward path.
 *
 * OSDN ("OSDN: Improving Delta Rule with Provable Online Preconditioning in Linear Attention",
 * arXiv:2605.13473) is the delta rule with a diagonal, online-learned right preconditioner d on
 * the write side.  The forward path has three calls, and a fourth that chains the first two:
 *
 *   osdn_precond_scan  phase 1 (Section 4.2, Algorithm 1, Eq. (4); APF retention Eq. (7)):
 *                      per (batch, head), for t = 0..T-1:
 *                        k~_t   = d_t . k_t                                  (emitted first)
 *                        s_t    = k_t . k_t,  n_t = max(sum s_t, eps)
 *                        b      = beta_t if beta_aware else 1
 *                        d_{t+1}= clip(r_t d_t + eta b (1 - b <d_t, s_t>) / n_t * s_t, d_min, d_max)
 *   osdn_chunk_fwd     phase 2 (Section 4.1 Eq. (2), Section 4.3 Eqs. (5)-(6), Appendix A.2
 *                      Eqs. (8)-(11)): per (batch, head), with the original key on the read side
 *                      and the write key k~ on the write side,
 *                        u_t = v_t - S_{t-1} k_t,   S_t = S_{t-1} + beta_t u_t k~_t^T,
 *                        o_t = scale * S_t q_t      (readout after the write)
 *                      computed chunkwise (WY/UT form) with an fp32 state.
 *   osdn_decode_step   one token of both phases in place on (S, d): the recurrent form used at
 *                      generation time (the pages' single-token kernel, Appendix L).
 *   osdn_layer_fwd     osdn_precond_scan then osdn_chunk_fwd on its write keys (the pages'
 *                      chunk_osdn, Listing 1), with the two phases overlapped on the GPU.
 *   osdn_layer_fwd_host the same from HOST buffers, the copies overlapped with the compute.
 *
 * Conventions shared by every call
 *   - Every buffer is caller-owned DEVICE memory (cudaMalloc or equivalent; osdn_layer_fwd_host's
 *     inputs and outputs are the one exception, host memory); the library never allocates device
 *     memory, frees, or keeps pointers after the call returns.
 *   - Layouts are dense row-major: q, k, k~ [B,T,H,K]; v, o [B,T,H,V]; beta, r [B,T,H];
 *     S [B,H,V,K] (value-major: S[b,h,i,j] multiplies key coordinate j); d [B,H,K].
 *     Decode drops T: q, k [B,H,K]; v, o [B,H,V]; beta, r [B,H].
 *   - dtypes: q, k, k~, v, o are OSDN_F32, OSDN_BF16 or OSDN_F16 (one dtype per call, except the
 *     scan's k~ output dtype which is chosen separately); beta, r, d, S are always fp32.
 *   - All pointers must be 16-byte aligned.  K and V must each be 64 or 128.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is enqueued
 *     asynchronously; argument errors are detected on the host and returned before any launch.
 *   - Errors: OSDN_OK on success; OSDN_ERR_ARG (null pointer where one is required, negative or
 *     non-finite scalar, d_min > d_max), OSDN_ERR_SHAPE (sizes out of range, T not a multiple of
 *     the chunk), OSDN_ERR_DTYPE, OSDN_ERR_ALIGN, OSDN_ERR_UNSUPPORTED (valid but not built, e.g.
 *     K = 96), OSDN_ERR_CUDA (a launch failed; osdn_last_cuda_error() names the CUDA error),
 *     OSDN_ERR_TIMEOUT (a device-side bounded wait gave up; reported by osdn_check()),
 *     OSDN_ERR_CAPACITY (the request needs more scratch than osdn_chunk_fwd_static_ws has),
 *     OSDN_ERR_RANGE (reported by osdn_check(): a 16-bit tensor-core chunk call produced an inf or
 *     NaN in o or the final S, i.e. an input, the state or an intermediate left fp16's range).
 *   - Numeric range of the 16-bit tensor-core chunk path (K = V = 128, bf16/f16 inputs): its
 *     operands are fp16 (bf16 inputs convert exactly in fp16's normal range), so every input
 *     element, every entry of the state S and of the chunk intermediates T', W, U, X and L must
 *     stay below 65504 in magnitude.  Elements below fp16's normal range (6.1e-5) keep an absolute
 *     precision of 6e-8.  A call that left the range returns invalid results and osdn_check()
 *     reports OSDN_ERR_RANGE; rerun it with fp32 inputs (the fp32 CUDA-core path), or scale v and
 *     S0 by a power of two and o and S back (the rule is linear in (v, S0)).
 *   - Sizes are `int`; B*T*H*max(K,V) must stay below 2^31 elements per tensor.
 */
#ifndef OSDN_H
#define OSDN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    OSDN_OK = 0,
    OSDN_ERR_ARG = 1,
    OSDN_ERR_SHAPE = 2,
    OSDN_ERR_DTYPE = 3,
    OSDN_ERR_ALIGN = 4,
    OSDN_ERR_UNSUPPORTED = 5,
    OSDN_ERR_CUDA = 6,
    OSDN_ERR_TIMEOUT = 7,
    OSDN_ERR_CAPACITY = 8,
    OSDN_ERR_RANGE = 9
} osdn_status;

typedef enum { OSDN_F32 = 0, OSDN_BF16 = 1, OSDN_F16 = 2 } osdn_dtype;

/*
 * Phase 1: preconditioner scan (Algorithm 1 / Eq. (4); Eq. (7) when r != NULL).
 *   k        [B,T,H,K] keys, dtype k_dtype (read)
 *   beta     [B,T,H] fp32 write gates in (0,1) (read)
 *   r        fp32 APF retention; NULL means r = 1 (Eq. (4)).  r_per_key = 0: [B,T,H], one
 *            r_{t,h} broadcast over K (Eq. (7)); r_per_key = 1: [B,T,H,K], the vector retention
 *            diag(r_t) of Appendix A.5 (Prop. A.3), one gate per key coordinate.  Other values of
 *            r_per_key return OSDN_ERR_ARG.  With 16-bit keys and K = 128 both layouts run the
 *            blocked scan (vector gates: every 64-token block by Jacobi sweeps on the clipped
 *            recurrence, the gates staged with the keys); fp32 keys or K = 64 take the
 *            token-by-token kernel.
 *   d0       [B,H,K] fp32 initial preconditioner; NULL means d = 1.  Used as given (not clamped).
 *   k_tilde  [B,T,H,K] write keys k~_t = d_t . k_t, dtype kt_dtype (written)
 *   d_out    [B,H,K] fp32 final d_{T} (written; may alias d0)
 *   eta >= 0; d_min <= d_max (use -INFINITY/+INFINITY to switch the box off); eps > 0 floors
 *   the SQUARED key norm; beta_aware = 1 feeds beta_t into the step (Listing 1 default),
 *   0 uses 1 there (the memory write keeps beta either way).
 *   workspace, workspace_bytes
 *            optional caller-owned device scratch (16-byte aligned).  When it holds at least
 *            osdn_precond_scan_workspace_bytes(...) bytes, the blocked scan (bf16/f16 keys,
 *            K = 128) only fixes the step sizes and block-start states and a second, fully
 *            parallel kernel writes k_tilde from them; with NULL or a smaller workspace the scan
 *            kernel writes k_tilde itself (slower).  Results are bit-identical either way.  The
 *            workspace is overwritten; its contents on return are unspecified.
 *   T may be 0 (then d_out = d0 or 1).
 */
osdn_status osdn_precond_scan(const void* k, osdn_dtype k_dtype, const float* beta,
                              const float* r, int r_per_key, const float* d0, void* k_tilde,
                              osdn_dtype kt_dtype, float* d_out, int B, int T, int H, int K,
                              float eta, float d_min, float d_max, float eps, int beta_aware,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Workspace size in bytes that lets osdn_precond_scan write k_tilde from its parallel kernel (0
 * when that path does not apply: then no workspace is ever used).  For bf16/f16 keys with K = 128
 * it is 4 * B * H * (T + 256 * ceil(T / 64)) bytes: one fp32 step size per token and the fp32
 * (hi, lo) state at the start of each 64-token block. */
size_t osdn_precond_scan_workspace_bytes(int B, int T, int H, int K, osdn_dtype k_dtype);

/*
 * Phase 2: chunkwise preconditioned delta rule (Eqs. (2), (5), (8)-(11)).
 *   q, k, k_tilde [B,T,H,K], v [B,T,H,V], all of dtype `dtype` (read)
 *   beta     [B,T,H] fp32 (read)
 *   alpha    [B,T,H] fp32 state gate of the gated variant (OSGDN, Appendix B.1, Eqs. (13)-(15)),
 *            or NULL for none.  With it every token first scales the state, Sbar = alpha_t S_{t-1},
 *            then e_t = v_t - Sbar k_t, S_t = Sbar + beta_t e_t k~_t^T (post-gate residual).
 *            Gates are read as given (the pages' gates lie in (0, 1]).
 *   alpha_per_key
 *            1: alpha is [B,T,H,K], one state gate per key channel (OSKDA, Appendix B.2: KDA's
 *            K x V state Diag(alpha_t) S_{t-1}; the state here is its V x K transpose, so column i
 *            is scaled by alpha_{t,i}).  With a workspace of osdn_chunk_fwd_gated_workspace_bytes(
 *            ..., 2) bytes, bf16/f16 inputs with K = V = 128 run on the tensor cores (the chunk
 *            form of Listing 3: with Gamma the channels' cumulative gates inside a chunk, the Gram
 *            and scores of K . Gamma and Q . Gamma against K~ / Gamma as split-bf16 products,
 *            fp32 UT inverse, fp16 operands in the state pass).  That path needs every channel's
 *            decay over a chunk (a product of 64 gates) above 1e-30.  Otherwise, or with a smaller
 *            workspace, the fp32 CUDA-core kernel runs.  0: one per head (OSGDN).  Ignored without
 *            alpha; other values OSDN_ERR_ARG.
 *   S0       [B,H,V,K] fp32 initial state; NULL means zeros
 *   o        [B,T,H,V] outputs o_t = scale * S_t q_t, dtype `dtype` (written)
 *   S_out    [B,H,V,K] fp32 final state (written; may alias S0)
 *   chunk    chunk length C; 64 is the only value built.  T must be a multiple of C (T = 0 is
 *            allowed and copies S0 to S_out).
 *   scale    multiplies q (1.0 gives o_t = S_t q_t as in the equations; Listing 1 uses K^-1/2).
 *   workspace, workspace_bytes
 *            optional caller-owned device scratch (16-byte aligned).  When it holds at least
 *            B * H * (T / 64) * 33280 bytes, the tensor-core path splits into a parallel kernel
 *            over all chunks (everything that does not depend on S: the UT transform T' and W,
 *            kept as fp16 in the workspace) and a serial kernel over chunks; with NULL or a
 *            smaller workspace one fused kernel does both (slower, no scratch).  With few heads
 *            (B*H*(V/64) CTAs leave most SMs idle) and at least 32 chunks, a workspace of
 *            osdn_chunk_fwd_workspace_bytes(...) bytes (more than the above) also lets the serial
 *            pass run in segments side by side: each later segment starts from a zero state
 *            beside a pass that carries the product of the chunk transitions (I - K~^T W)
 *            (Appendix A.2, Eq. (10)); the segment start states are chained afterwards and the
 *            later segments' outputs corrected.  The paths agree to the fp16 operand rounding
 *            (o may differ by one unit of its last place).  The workspace is overwritten; its
 *            contents on return are unspecified.
 * bf16/f16 inputs with K = V = 128 run on the tensor-core kernels (TMA + tcgen05, fp16
 * operands, fp32 accumulation, fp32 state); other shapes and fp32 inputs run an fp32
 * CUDA-core kernel (which needs no workspace).
 */
osdn_status osdn_chunk_fwd(const void* q, const void* k, const void* k_tilde, const void* v,
                           osdn_dtype dtype, const float* beta, const float* alpha, int alpha_per_key,
                           const float* S0, void* o,
                           float* S_out, int B, int T, int H, int K, int V, int chunk,
                           float scale, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace size in bytes that lets osdn_chunk_fwd use its fastest tensor-core path for these
 * arguments (0 when that path does not apply: then no workspace is ever used).  For K = V = 128
 * and chunk 64 it is B * H * (T / 64) * 33280 bytes (for each chunk of each head 32 KiB of fp16
 * images and the chunk's decay factors of the gated variant), plus, where the serial pass runs
 * in segments (few heads, long sequences; depends on the device's SM count), the segment scratch:
 * the transition pass's fp16 outputs (B*T*H*K*2 bytes) and three fp32 states per head and
 * segment. */
size_t osdn_chunk_fwd_workspace_bytes(int B, int T, int H, int K, int V, int chunk,
                                      osdn_dtype dtype);

/* The same for a gated call: gated = 0 (no gate, as above), 1 (one state gate per head) or 2 (one
 * per key channel, alpha_per_key = 1).  With gated = 2 and K = V = 128 it is B * H * (T / 64) *
 * 66048 bytes: besides T', -W and L, each chunk of each head keeps Q . Gamma and K~ . Gamma_C /
 * Gamma (fp16) and Gamma_C (Gamma: the channels' cumulative gates within the chunk), which lets
 * osdn_chunk_fwd run that call on the tensor cores (a smaller workspace runs the fp32 CUDA-core
 * kernel).  0 for invalid arguments. */
size_t osdn_chunk_fwd_gated_workspace_bytes(int B, int T, int H, int K, int V, int chunk,
                                            osdn_dtype dtype, int gated);

/*
 * One OSDN layer forward: phase 1 then phase 2, the pages' chunk_osdn (Listing 1: returns o, the
 * final state S and the final preconditioner d) as one call.  Arguments as osdn_precond_scan and
 * osdn_chunk_fwd; q, k, v and the write keys share `dtype`.
 *   k_tilde  [B,T,H,K] write keys, dtype `dtype` (written; the phase-2 input)
 *   o, S_out as osdn_chunk_fwd; d_out as osdn_precond_scan (both written)
 *   r, r_per_key as osdn_precond_scan (vector retention always takes the two separate calls)
 *   alpha, alpha_per_key as osdn_chunk_fwd (the OSGDN / OSKDA state gate; phase 1 does not use it)
 *   workspace, workspace_bytes
 *            optional caller-owned device scratch (16-byte aligned).  With at least
 *            osdn_layer_fwd_workspace_bytes(...) bytes, bf16/f16 inputs with K = V = 128 and
 *            fewer than one (batch, head) per SM run phase 1 and the S-independent part of
 *            phase 2 in one cooperative launch (each chunk's prep starts as soon as phase 1 has
 *            passed it, on the SMs phase 1 leaves free), then the serial phase-2 kernel.  Other
 *            cases run osdn_precond_scan then osdn_chunk_fwd, giving each its part of the
 *            workspace when it fits.  Results equal the two calls' in every case.
 *   T must be a multiple of `chunk` (64).
 */
osdn_status osdn_layer_fwd(const void* q, const void* k, const void* v, osdn_dtype dtype, const float* beta,
                           const float* r, int r_per_key, const float* alpha, int alpha_per_key, const float* d0,
                           const float* S0, void* k_tilde, void* o,
                           float* S_out, float* d_out, int B, int T, int H, int K, int V, int chunk,
                           float eta, float d_min, float d_max, float eps, float scale, int beta_aware,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Workspace size in bytes for osdn_layer_fwd's fastest path with these arguments (0 when no
 * workspace is ever used). */
size_t osdn_layer_fwd_workspace_bytes(int B, int T, int H, int K, int V, int chunk, osdn_dtype dtype);

/* The same for a gated call (gated = 0, 1 or 2 as for osdn_chunk_fwd_gated_workspace_bytes). */
size_t osdn_layer_fwd_gated_workspace_bytes(int B, int T, int H, int K, int V, int chunk, osdn_dtype dtype,
                                            int gated);

/*
 * The layer forward over packed variable-length sequences (cu_seqlens).  N sequences are
 * concatenated along the token axis: sequence n owns rows cu_seqlens[n] .. cu_seqlens[n+1]-1 of
 * q, k, v [total, H, K|V] (dtype `dtype`), beta, alpha [total, H] fp32, r [total, H] (or
 * [total, H, K] with r_per_key = 1); it starts from d0[n] [H, K] and S0[n] [H, V, K] (NULL: ones,
 * zeros) and ends in d_out[n], S_out[n] ([N, H, K] and [N, H, V, K], fp32, written).  k_tilde
 * [total, H, K] and o [total, H, V] are written.  Each sequence gets exactly the result it would
 * get alone (Algorithm 1 and Eqs. (2), (4), (7), and Appendix B.1 with alpha, per sequence).
 *   cu_seqlens  device int32 [N + 1], non-decreasing from 0 to total (read on the device; a
 *               sequence whose range is not within [0, total] or is longer than max_len is
 *               skipped and the next osdn_check reports OSDN_ERR_SHAPE)
 *   total       packed tokens (rows of q); max_len >= every sequence length (host value)
 *   workspace, workspace_bytes
 *               required: at least osdn_layer_fwd_varlen_workspace_bytes(...) bytes, 16-byte
 *               aligned (OSDN_ERR_ARG when missing or smaller).  It holds the sequences scattered
 *               into an [N, Tp, H, .] batch, Tp = max_len rounded up to the chunk, with padding
 *               tokens that leave d and S unchanged (k = q = v = 0, beta = 0, retention and state
 *               gate 1), and the batched layer's own workspace; the outputs are gathered back.
 * Other arguments as osdn_layer_fwd.  A sequence of length 0 returns d0 and S0 unchanged.
 */
osdn_status osdn_layer_fwd_varlen(const void* q, const void* k, const void* v, osdn_dtype dtype, const float* beta,
                                  const float* r, int r_per_key, const float* alpha, int alpha_per_key,
                                  const int* cu_seqlens, int N,
                                  long long total, int max_len, const float* d0, const float* S0, void* k_tilde,
                                  void* o, float* S_out, float* d_out, int H, int K, int V, int chunk, float eta,
                                  float d_min, float d_max, float eps, float scale, int beta_aware, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Workspace size for osdn_layer_fwd_varlen: r_mode 0 (no retention), 1 (one per head) or 2 (one
 * per key coordinate); gated 0 (no alpha), 1 (one per head) or 2 (one per key channel).  0 for
 * invalid arguments. */
size_t osdn_layer_fwd_varlen_workspace_bytes(int N, int max_len, int H, int K, int V, int chunk, osdn_dtype dtype,
                                             int r_mode, int gated);

/*
 * The layer forward on HOST buffers (the pages' chunk_osdn, Listing 1, as one call from host
 * memory), with the copies overlapped with the compute.  Algorithm 1 and Eqs. (2), (4), (7) are
 * recurrences over the token axis that carry only (d, S), so the call splits the sequence into
 * `segments` consecutive pieces of T / segments tokens and runs osdn_layer_fwd on piece i from
 * piece i-1's final (d, S), kept on the device.  Piece i+1's inputs are copied in on `h2d_stream`
 * while piece i computes on `stream`, and piece i's o is copied out on `d2h_stream` meanwhile.
 *   q, k, v, beta, r, alpha, d0, S0
 *            HOST arrays, layouts and meaning as osdn_layer_fwd (NULL d0 / S0: ones / zeros; NULL
 *            r / alpha: none).  They must stay unchanged until the call's work on `stream` is
 *            complete.  Page-locked memory lets the copies overlap the compute; pageable memory
 *            gives the same results without the overlap.
 *   o, S_out, d_out
 *            HOST arrays [B,T,H,V] (dtype), [B,H,V,K] and [B,H,K] fp32 (written; valid once
 *            `stream` has completed the call's work).  The write keys are not returned.
 *   segments number of pieces; T / segments must be a whole number of chunks (OSDN_ERR_SHAPE
 *            otherwise; segments <= 0: OSDN_ERR_ARG).  1 runs copy-in, compute, copy-out in turn.
 *            Each piece boundary rounds the carried d to fp32 once (within the call d is carried
 *            as an fp32 pair), so results can differ from one osdn_layer_fwd call in the last bits.
 *   workspace, workspace_bytes
 *            required caller-owned DEVICE scratch, 256-byte aligned (OSDN_ERR_ALIGN otherwise), of
 *            at least osdn_layer_fwd_host_workspace_bytes(...) bytes (OSDN_ERR_ARG otherwise):
 *            two (d, S) state buffers, two staging slots of one piece's inputs and outputs, and
 *            the per-piece layer workspace.
 *   stream, h2d_stream, d2h_stream
 *            the compute stream and two copy streams (NULL copy streams mean `stream`: correct,
 *            without overlap).  Work queued on `stream` before the call comes first; everything the
 *            call queues is complete once `stream` reaches the point after the call.
 * T = 0 waits for `stream`, then writes d_out = d0 (or ones) and S_out = S0 (or zeros) on the
 * host.  Errors: the argument checks of osdn_layer_fwd, then OSDN_ERR_CUDA if a copy or an event
 * call fails.
 */
osdn_status osdn_layer_fwd_host(const void* q, const void* k, const void* v, osdn_dtype dtype, const float* beta,
                                const float* r, int r_per_key, const float* alpha, int alpha_per_key,
                                const float* d0, const float* S0, void* o, float* S_out, float* d_out, int B,
                                int T, int H, int K, int V, int chunk, float eta, float d_min, float d_max,
                                float eps, float scale, int beta_aware, int segments, void* workspace,
                                size_t workspace_bytes, void* stream, void* h2d_stream, void* d2h_stream);

/* Device workspace size for osdn_layer_fwd_host: r_mode 0 / 1 / 2 and gated 0 / 1 / 2 as for
 * osdn_layer_fwd_varlen_workspace_bytes.  0 for invalid arguments (including T = 0). */
size_t osdn_layer_fwd_host_workspace_bytes(int B, int T, int H, int K, int V, int chunk, osdn_dtype dtype,
                                           int r_mode, int gated, int segments);

/*
 * The layer backward: gradients of a loss through osdn_layer_fwd's outputs o, S_out and d_out
 * with respect to q, k, v, beta, r, d0 and S0 (the pages' training path; the reverse sweep of the
 * projected d recurrence passes no gradient through a clipped coordinate: the clip's derivative
 * is 1 on [d_min, d_max] and 0 outside).  Inputs as osdn_layer_fwd (alpha must be NULL: the gated
 * variant's backward is not built, OSDN_ERR_UNSUPPORTED); upstream gradients fp32:
 *   dout [B,T,H,V] (required), dS [B,H,V,K] and dd [B,H,K] (NULL: zero).
 * Outputs fp32 (written): dq, dk [B,T,H,K], dv [B,T,H,V], dbeta [B,T,H], dr (the layout of r;
 * required when r is given), dd0 [B,H,K] and dS0 [B,H,V,K] (NULL: not written).
 *   workspace  required, at least osdn_layer_bwd_workspace_bytes(...) bytes (fp32 write keys,
 *              their gradient, the state at every 64-token chunk start and d at every block
 *              start).
 * The sweeps are token-recurrent fp32 on the CUDA cores (S checkpointed per chunk and rebuilt
 * backward within it): exact to fp32 rounding, not fast.
 */
osdn_status osdn_layer_bwd(const void* q, const void* k, const void* v, osdn_dtype dtype, const float* beta,
                           const float* r, int r_per_key, const float* alpha, const float* d0, const float* S0,
                           const float* dout, const float* dS, const float* dd, float* dq, float* dk, float* dv,
                           float* dbeta, float* dr, float* dd0, float* dS0, int B, int T, int H, int K, int V,
                           float eta, float d_min, float d_max, float eps, float scale, int beta_aware,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Workspace size for osdn_layer_bwd (0 for unsupported head sizes or empty problems). */
size_t osdn_layer_bwd_workspace_bytes(int B, int T, int H, int K, int V);

/*
 * osdn_chunk_fwd for callers that cannot allocate device memory when they call -- for example an
 * engine that reserves all GPU memory in one plan at start-up and allocates nothing afterwards,
 * or code that cannot accept an allocator call (its latency, its implicit synchronisation, its
 * possible failure) in the middle of a step.  No counterpart in the paper: this is a property of
 * this library's interface, not of the method.
 *   Same arguments as osdn_chunk_fwd without the workspace, and the results osdn_chunk_fwd gives
 *   with a workspace of B * H * (T / 64) * 33280 bytes (its two-kernel tensor-core path, without
 *   the segment split): that scratch comes from a fixed 32 MiB array in the library's own device
 *   memory (file-scope; every GPU that loads the library holds it until the process exits).
 *   Capacity: B * H * (T / 64) * 33280 <= 32 MiB, i.e. B * H * (T / 64) <= 1008 chunks;
 *   larger requests return OSDN_ERR_CAPACITY before any launch.  Calls that need no scratch (fp32
 *   inputs, other head sizes) run the CUDA-core kernel as osdn_chunk_fwd does.
 *   Neither the library nor this call allocates (no cudaMalloc/cudaFree or allocating routine).
 *   Every call looks up the array's device address on the current device
 *   (cudaGetSymbolAddress, which allocates nothing); the first call on a device also loads the
 *   library's device code there, so make that first call before any stream capture.  The
 *   argument checks are osdn_chunk_fwd's and come before the capacity test; only calls that take
 *   the two-kernel tensor-core path need scratch, so a per-channel gate (alpha_per_key = 1: here the
 *   CUDA-core kernel, as osdn_chunk_fwd without a workspace) or fp32 inputs are never refused for
 *   capacity.
 *   All calls share the one array and nothing in it needs to start at zero (each call writes all
 *   the scratch it reads), but calls whose work overlaps on the GPU -- on different streams, or
 *   from different threads -- race on it: serialise them.
 */
osdn_status osdn_chunk_fwd_static_ws(const void* q, const void* k, const void* k_tilde,
                                     const void* v, osdn_dtype dtype, const float* beta,
                                     const float* alpha, int alpha_per_key, const float* S0, void* o, float* S_out, int B, int T, int H,
                                     int K, int V, int chunk, float scale, void* stream);

/*
 * One decode token for every (batch, head), in place (recurrent form of both phases):
 *   k~ = d . k (old d); d <- clip(r d + eta b (1 - b <d, k.k>) / max(|k|^2, eps) k.k);
 *   S <- alpha S (the OSGDN state gate, Appendix B.1; alpha NULL: none);
 *   u = v - S k;  S <- S + beta u k~^T;  o = scale * S q.
 *   q, k [B,H,K], v [B,H,V] of dtype `dtype`; beta [B,H] fp32; r fp32 or NULL: [B,H] with
 *   r_per_key = 0, or [B,H,K] (one gate per key coordinate, diag(r_t)) with r_per_key = 1;
 *   alpha [B,H] fp32 or NULL ([B,H,K] with alpha_per_key = 1: one gate per key channel, OSKDA);
 *   S [B,H,V,K] fp32 and d [B,H,K] fp32 are read and overwritten; o [B,H,V] dtype `dtype`.
 */
osdn_status osdn_decode_step(const void* q, const void* k, const void* v, osdn_dtype dtype,
                             const float* beta, const float* r, int r_per_key, const float* alpha,
                             int alpha_per_key, float* S, float* d, void* o,
                             int B, int H, int K, int V, float eta, float d_min, float d_max,
                             float eps, float scale, int beta_aware, void* stream);

/* Waits for `stream`, then reports OSDN_ERR_TIMEOUT if any kernel of this library gave up a
 * bounded device-side wait since the last check, OSDN_ERR_SHAPE if a varlen call met an invalid
 * cu_seqlens range, OSDN_ERR_RANGE if a 16-bit tensor-core chunk call produced a non-finite
 * output (all three flags are cleared), OSDN_ERR_CUDA if the stream holds a CUDA error, else
 * OSDN_OK. */
osdn_status osdn_check(void* stream);

/*
 * Failure-detection hook (not a method parameter; the paper has no counterpart).  Sets how many
 * times the fused layer call's chunk-prep workers poll for a value that its phase-1 CTAs publish
 * before they give up (0 restores the default, about 2-4 s of polling).  A small limit makes those
 * bounded waits run out while phase 1 is still working: the kernels then drain what they issued
 * and exit normally, the call's results are invalid, and osdn_check reports OSDN_ERR_TIMEOUT.
 * Process-wide; meant for tests, never needed in normal use.
 */
void osdn_set_poll_limit(unsigned int polls);

/* Human-readable name of a status code (static storage, never NULL). */
const char* osdn_status_string(int status);

/* Name of the CUDA error behind the calling thread's most recent OSDN_ERR_CUDA return
 * ("cudaSuccess" if there was none); static storage, never NULL. */
const char* osdn_last_cuda_error(void);

/* ABI version: major * 10000 + minor * 100 + patch. */
int osdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OSDN_H */
