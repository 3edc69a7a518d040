/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * The library computes exact softmax attention FlashAttention-style: Q and
 * K/V are tiled, an online softmax keeps a running row max and normaliser,
 * and the N x N score matrix never reaches device memory.  Sources for the
 * operations:
 *   - attention itself: S = Q K^T, P = softmax(S), O = P V
 *     (Flash Attention, ostralyan.com, "The Memory Wall Problem");
 *   - the tiled, single-pass computation with running statistics
 *     (FlashAttention: exact attention made fast by counting memory traffic,
 *     "The method"; Flash Attention, "Online Softmax Algorithm" and
 *     "Block-Wise Attention Computation");
 *   - one log-sum-exp per row kept by the forward, and the backward that
 *     recomputes P block by block from Q, K, V and that statistic
 *     (FlashAttention and IO-aware exact attention, "Core ideas").
 *
 * Conventions shared by every entry point
 *   - Tensors q, k, v, o, dO, dq, dk, dv are DEVICE pointers to contiguous
 *     bf16 arrays of shape [B][H][N][d] (d innermost).  lse is a device
 *     pointer to fp32 [B][H][N].  Every pointer must be 16-byte aligned.
 *     (The host-memory entry points fa_fwd_host and fa_fwd_bwd_host take
 *     HOST pointers instead, with no alignment rule, and a device staging
 *     area; see their section.)
 *   - d must be 64 or 128.  N >= 1 is any length up to 2^30 (the last tile
 *     is masked).  B, H >= 1.  B == 0, H == 0 or N == 0 is an empty problem:
 *     FA_OK, no work.  B * H * ceil(N / 128) must be at most 2^27 - 1 (grid
 *     limits); larger problems return FA_ERR_INVALID_ARG.
 *   - scale multiplies Q K^T before the softmax; it must be finite and > 0
 *     (usually 1/sqrt(d)).
 *   - causal = 1: key j is visible to query i iff j <= i (N_q = N_k = N;
 *     fa_fwd_ex / fa_bwd_ex below state the rule for N_q != N_k).
 *     causal = 0: every key is visible.
 *   - lse[i] = ln( sum over visible j of exp(scale * q_i . k_j) ).
 *   - The caller owns every buffer, including the backward workspace.  The
 *     library allocates no device memory per call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and run on the current device, which must be sm_103
 *     (GB300).  Argument errors are reported before anything is launched.
 *     A kernel whose internal pipeline wait exceeds the wait bound gives up
 *     cleanly and records FA_ERR_TIMEOUT in a per-device error word that
 *     fa_last_device_error() reads.
 *   - Thread safety: calls on distinct streams may come from distinct host
 *     threads.
 *   - CUDA graphs: fa_fwd, fa_fwd_gqa, fa_fwd_ex, fa_fwd_sparse, fa_bwd,
 *     fa_bwd_gqa, fa_bwd_ex, fa_bwd_sparse and the host-memory entry points
 *     may be captured on a stream and replayed; a replay computes on what the
 *     buffers hold then.  Make one eager call on the device first (it looks
 *     up the device and the driver's tensor-map encoder once).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st*` */

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, scale or flag */
  FA_ERR_UNSUPPORTED = 2, /* d not in {64,128}, or device is not sm_103 */
  FA_ERR_LAUNCH = 3,      /* a CUDA runtime call or kernel launch failed */
  FA_ERR_TIMEOUT = 4,     /* a kernel gave up on a pipeline wait */
  FA_ERR_NO_DEVICE = 5,   /* no CUDA device is current */
  FA_ERR_DEVICE = 6       /* the stream reported an asynchronous CUDA error */
} fa_status;

/*
 * Forward: o = softmax(scale * q k^T [causal]) v, and lse.
 * Outputs o ([B][H][N][d] bf16) and lse ([B][H][N] fp32) are overwritten.
 * Source: Flash Attention, "Core Flash Attention Algorithm" (tiled forward
 * with running max and sum); FlashAttention and IO-aware exact attention,
 * "Core ideas" (one log-sum-exp per row; only O and the row statistic are
 * written).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, struct CUstream_st* stream);

/*
 * Grouped key/value heads (GQA; MQA when H_kv = 1).  Same as fa_fwd, except
 * that k and v have H_kv heads: bf16 [B][H_kv][N][d], H_kv >= 1 dividing H.
 * Query head h attends with key/value head h / (H / H_kv) (consecutive query
 * heads share one K, V).  fa_fwd is this with H_kv = H.  H_kv outside
 * 1 ... H or not dividing H => FA_ERR_INVALID_ARG.  Source: Flash Attention,
 * "Evolution: Flash Attention 2 & 3" (multi-query and grouped-query support;
 * the grouping itself is the library's reading).
 */
fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int H_kv, int N, int d, float scale, int causal,
                     struct CUstream_st* stream);

/*
 * General forward: grouped key/value heads and query and key lengths that
 * differ.  q, o: bf16 [B][H][N_q][d]; k, v: bf16 [B][H_kv][N_k][d]; lse: fp32
 * [B][H][N_q].  H_kv as in fa_fwd_gqa.  Query row i attends to keys 0 ...
 * N_k - 1 (causal = 0), or to keys j <= i + (N_k - N_q) (causal = 1: the last
 * query row is aligned with the last key, as for a block of new queries
 * appended after N_k - N_q earlier positions; needs N_k >= N_q).
 *   - N_q == 0 (or B == 0 or H == 0) is an empty problem: FA_OK, no work.
 *   - N_k == 0 with N_q >= 1, or causal with N_k < N_q, or N_q or N_k
 *     above 2^30 => FA_ERR_INVALID_ARG.  B * H * ceil(N_q / 128) must be
 *     at most 2^27 - 1.
 * fa_fwd_gqa is this with N_q = N_k = N.  Source: Flash Attention,
 * "Evolution: Flash Attention 2 & 3" (variable sequence lengths; the causal
 * alignment for N_q != N_k is the library's reading).
 */
fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H, int H_kv, int N_q, int N_k, int d, float scale, int causal,
                    struct CUstream_st* stream);

/*
 * Bytes of device workspace fa_bwd needs: fp32 row statistics, two per row
 * (-lse log2 e and -D with D = rowsum(dO * o)) with each head padded to whole
 * 128-row tiles, i.e. B*H*ceil(N/128)*256 floats, followed by an fp32 dQ
 * accumulator of shape [B][H][N][d]; each region rounded up to 256 bytes.
 * 0 for an empty problem or invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward: given dO = dL/do, writes dq, dk, dv (bf16 [B][H][N][d],
 * overwritten).  o and lse must be the outputs of fa_fwd with the same
 * q, k, v, B, H, N, d, scale and causal.  P is recomputed block by block
 * from q, k and lse; no N x N matrix is stored (FlashAttention: exact
 * attention made fast by counting memory traffic, "The method";
 * FlashAttention and IO-aware exact attention, "Backward by recomputation").
 * The gradient formulas are the chain rule through the softmax:
 *   D_i = sum_c dO_ic o_ic,  dS_ij = P_ij (dO_i . v_j - D_i),
 *   dq = scale dS k,  dk = scale dS^T q,  dv = P^T dO.
 * workspace: device pointer, 256-byte aligned, at least
 * fa_bwd_workspace_size(B, H, N, d) bytes; its contents on entry are
 * ignored and on exit are unspecified.  Smaller => FA_ERR_INVALID_ARG.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, void* workspace, size_t workspace_bytes,
                 struct CUstream_st* stream);

/*
 * Backward for grouped key/value heads: the counterpart of fa_fwd_gqa.  k, v,
 * dk, dv are bf16 [B][H_kv][N][d]; dk and dv of a key/value head are the sums
 * of the gradients through it of its H / H_kv query heads (chain rule through
 * the shared K, V).  The workspace is fa_bwd_workspace_size(B, H, N, d)
 * (query heads).  fa_bwd is this with H_kv = H.
 */
fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dO, void* dq, void* dk, void* dv, int B, int H,
                     int H_kv, int N, int d, float scale, int causal, void* workspace,
                     size_t workspace_bytes, struct CUstream_st* stream);

/*
 * General backward: the counterpart of fa_fwd_ex.  q, o, dO, dq: bf16
 * [B][H][N_q][d]; k, v, dk, dv: bf16 [B][H_kv][N_k][d]; lse: fp32 [B][H][N_q]
 * from fa_fwd_ex with the same arguments.  The workspace depends on the
 * query side only: fa_bwd_workspace_size(B, H, N_q, d) bytes.
 *   - N_q == 0 with B, H, N_k >= 1: dk and dv are set to zero (sums over no
 *     query rows) with two cudaMemsetAsync on `stream`; nothing else is read.
 *   - Other sizes and errors as for fa_fwd_ex.
 * fa_bwd_gqa is this with N_q = N_k = N.
 */
fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, int B, int H, int H_kv, int N_q,
                    int N_k, int d, float scale, int causal, void* workspace,
                    size_t workspace_bytes, struct CUstream_st* stream);

/*
 * Block-sparse attention: fa_fwd_ex and fa_bwd_ex restricted by a block
 * mask.  block_mask is a DEVICE pointer to ceil(N_q/128) x ceil(N_k/128)
 * bytes, row-major (row = 128-row block of queries, column = 128-key block),
 * shared by every batch and head; a nonzero byte keeps the block, zero drops
 * it: key j is visible to query i only if byte [i/128][j/128] is nonzero,
 * and, when causal, j <= i + N_k - N_q.  Dropped blocks are neither loaded
 * nor computed.  A query row that sees no key gets o = 0 and lse = -inf and
 * contributes nothing to dq, dk or dv; a key that no row sees gets dk = dv = 0.
 * block_mask == NULL is the dense computation of fa_fwd_ex / fa_bwd_ex.
 * Both sides of the mask are limited to 4096 blocks (N_q, N_k <= 524288);
 * larger => FA_ERR_INVALID_ARG.  fa_bwd_sparse needs the o and lse of
 * fa_fwd_sparse with the same mask, and the workspace of fa_bwd_ex.  Source:
 * FlashAttention: exact attention made fast by counting memory traffic, "The
 * method" (the block-sparse extension, Sec 3.3); Flash Attention, "Sparse
 * Flash Attention" (predefined block-sparse patterns).  The mask's form and
 * the empty-row convention are the library's reading.
 */
fa_status fa_fwd_sparse(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int H_kv, int N_q, int N_k, int d, float scale, int causal,
                        const unsigned char* block_mask, struct CUstream_st* stream);
fa_status fa_bwd_sparse(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                        int H, int H_kv, int N_q, int N_k, int d, float scale, int causal,
                        const unsigned char* block_mask, void* workspace,
                        size_t workspace_bytes, struct CUstream_st* stream);

/*
 * Forward with a chosen key tile: fa_fwd_ex computed with K and V streamed in
 * tiles of key_tile keys (64 or 128; fa_fwd_ex uses 128).  Same arguments,
 * outputs and errors as fa_fwd_ex, plus key_tile: any other value returns
 * FA_ERR_UNSUPPORTED before anything is launched.  The results of the two
 * tile sizes agree to rounding (the online softmax sums the keys in another
 * grouping); fa_bwd_ex accepts the o and lse of either.  This is the block-
 * size axis of the IO analysis: FlashAttention: exact attention made fast by
 * counting memory traffic, "The decisive evidence" (Fig. 2, runtime against
 * block size); the pages' block-size rule itself (Flash Attention, "Memory &
 * Performance Analysis") is not used.
 */
fa_status fa_fwd_tiled(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int H_kv, int N_q, int N_k, int d, float scale, int causal,
                       int key_tile, struct CUstream_st* stream);

/*
 * Backward with no workspace argument and no allocation.  The paper has no
 * counterpart; this entry point exists for callers that cannot allocate
 * device memory: plugins inside a host framework that owns all device memory
 * and gives them none, and latency-critical loops that must not call
 * cudaMalloc (it may synchronise the device and takes unbounded time).
 *
 * Same arguments, semantics and outputs as fa_bwd minus the workspace: the
 * scratch (the row statistics and the fp32 dQ accumulator) lives in a 64 MiB
 * array that the library holds on every device that loads it, until the
 * process exits.
 *   - Capacity: fa_bwd_workspace_size(B, H, N, d) must be <= 64 MiB
 *     (67108864 bytes): up to about 129,000 rows (B*H*N) at d=128 and
 *     254,000 at d=64 (N a multiple of 128); larger problems return
 *     FA_ERR_INVALID_ARG before anything is launched.
 *   - The first call on a device looks up the array's device address (a
 *     one-time runtime query, with that device current); make that first
 *     call before any stream capture.
 *   - Every call on a device shares the one array.  Each call rewrites the
 *     statistics and re-zeroes the accumulator before use, so earlier
 *     contents never leak into a result, but calls that overlap on the GPU
 *     (on different streams without ordering between them) race on the array
 *     and give wrong gradients.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, float scale, int causal,
                         struct CUstream_st* stream);

/*
 * Host-memory entry points: the forward (fa_fwd_host), or the forward and
 * the backward (fa_fwd_bwd_host), for inputs and outputs that live in HOST
 * memory.  The computation is that of fa_fwd_sparse and fa_bwd_sparse with
 * the same shapes and arguments (same kernels; with block_mask == NULL, that
 * of fa_fwd_ex and fa_bwd_ex), so the sources are theirs; the copies around
 * it are the library's own.
 *   - block_mask: NULL, or a DEVICE pointer to the block mask of
 *     fa_fwd_sparse (same layout and limits), shared by every head and so by
 *     every group.
 *   - q, k, v, dO are HOST pointers to the inputs and o, lse, dq, dk, dv HOST
 *     pointers to the outputs, with the shapes of fa_fwd_ex / fa_bwd_ex
 *     (bf16 [B][H][N_q][d] for q, o, dO, dq; bf16 [B][H_kv][N_k][d] for k, v,
 *     dk, dv; fp32 [B][H][N_q] for lse).  No alignment is required.
 *   - dev: a DEVICE staging area owned by the caller, 256-byte aligned, of at
 *     least fa_fwd_host_device_bytes(...) or fa_fwd_bwd_host_device_bytes(...)
 *     bytes (the latter with the same `chunks`).  It holds the device copy of
 *     every tensor and the backward workspace; its contents on entry are
 *     ignored and on exit unspecified.  The *_device_bytes functions return
 *     0 for an empty problem or invalid sizes.
 *   - The key/value heads are cut into `chunks` groups of consecutive heads
 *     (0 = the library's choice, 8; at most 64, at most B * H_kv); a group
 *     takes its H / H_kv query heads along.  For each group the inputs are
 *     copied to the device on one internal stream, its kernels run on
 *     `stream`, and its outputs are copied back on a second internal stream,
 *     so the copies of one group overlap the kernels and copies of the
 *     others.  The internal streams and events are created once per device
 *     and kept until the process exits.
 *   - Asynchronous like every other call: nothing in `dev` is overwritten
 *     before the work already on `stream` has finished, and `stream` passes
 *     this call only once the last output has reached host memory, so
 *     cudaStreamSynchronize(stream) makes the outputs readable.  The host
 *     inputs must stay valid and unchanged until then.
 *   - Host buffers should be page-locked (cudaHostAlloc, cudaHostRegister):
 *     with pageable memory the copies are correct but do not overlap.
 *   - Results: o, lse, dk and dv equal those of the device entry points on
 *     the same inputs bit for bit; dq equals them up to the order of its fp32
 *     additions (which already varies between calls of fa_bwd_ex).
 *   - Errors: argument errors (the rules of fa_fwd_ex, a null host pointer
 *     for a non-empty tensor, a misaligned or short staging area) return
 *     FA_ERR_INVALID_ARG before anything is enqueued.  A CUDA error part way
 *     returns FA_ERR_LAUNCH or the failing kernel call's status; the outputs
 *     are then unspecified.  Calls on one device are enqueued one at a time
 *     (a per-device lock).
 */
size_t fa_fwd_host_device_bytes(int B, int H, int H_kv, int N_q, int N_k, int d);
size_t fa_fwd_bwd_host_device_bytes(int B, int H, int H_kv, int N_q, int N_k, int d,
                                    int chunks);
fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int H_kv, int N_q, int N_k, int d, float scale, int causal,
                      const unsigned char* block_mask, void* dev, size_t dev_bytes, int chunks,
                      struct CUstream_st* stream);
fa_status fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO, void* o,
                          float* lse, void* dq, void* dk, void* dv, int B, int H, int H_kv,
                          int N_q, int N_k, int d, float scale, int causal,
                          const unsigned char* block_mask, void* dev, size_t dev_bytes,
                          int chunks, struct CUstream_st* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns FA_OK, FA_ERR_TIMEOUT (a kernel gave up on a wait), or
 * FA_ERR_DEVICE when the synchronisation itself reported a CUDA error.
 */
fa_status fa_last_device_error(struct CUstream_st* stream);

/*
 * Raw error word of the last recorded device error on the current device
 * (code | site << 8 | block << 32), without clearing it; 0 if none.
 * Synchronises `stream` first.  For diagnostics.
 */
unsigned long long fa_device_error_word(struct CUstream_st* stream);

/*
 * Bound, in nanoseconds, on every internal pipeline wait of kernels launched
 * after this call (process-wide).  0 restores the default of 2 seconds.
 */
void fa_set_wait_timeout_ns(unsigned long long ns);

/* Static description of a status code. */
const char* fa_strerror(int status);

/* Library version string. */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
