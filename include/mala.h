/*
 * mala.h -- C ABI of libmala.so: MassAlloc Attention (MALA) on GB300 (sm_103a).
 *
 * MALA is causal softmax attention that forms every legal Q K^T score tile and
 * then runs the post-score work of a tile (softmax update, V load, P V; in the
 * backward pass P, dP, dS, dQ, dK, dV) only when some valid query row of the
 * tile gives one of its keys a normalised contribution of at least tau / L_q,
 * where L_q is the number of keys visible to that row.
 *
 * Source of every definition below: "MassAlloc Attention: Let Attention
 * Allocate Its Own Compute" -- §2.1 (scores, L_q, threshold tau/L_q), §2.2
 * Eq. (1)-(3) (forward test against the running online-softmax state),
 * Eq. (4) (backward test against the saved log-normaliser), Algorithm 1
 * (forward), Algorithm 2 (backward), App. A.1 (fused forward, backward and
 * split-KV decoding); the split merge is the (m, l, u) identity of "Why exact
 * attention does not need a quadratic matrix", Method/Mechanism.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers, owned by the caller.  The
 *    library never allocates or frees device memory; scratch space comes in
 *    through the `workspace` argument of the calls that need it.
 *  - Layouts are dense, row-major, head dimension fastest:
 *      prefill  q, o, dout, dq          [batch, seqlen_q, heads_q,  head_dim]
 *               k, v, dk, dv            [batch, seqlen_k, heads_kv, head_dim]
 *               lse                     [batch, heads_q, seqlen_q]   (float)
 *      decode   q, o                    [batch, heads_q, head_dim]
 *               k_cache, v_cache        [batch, cache_len, heads_kv, head_dim]
 *               lse                     [batch, heads_q]              (float)
 *    Query head h reads key/value head h / (heads_q / heads_kv).
 *  - Pointers must be 16-byte aligned.
 *  - Scores are s = softmax_scale * (q . k) computed in fp32; lse is the
 *    natural-log log-sum-exp over the retained keys (m + log l of Algorithm 1).
 *    Gradients are with respect to the unscaled q, k and v.
 *  - tau >= 0.  tau == 0 runs no test at all and gives dense attention
 *    through the same kernels (§2.3: tau -> 0 recovers full attention).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Argument errors are reported synchronously, before any
 *    launch, and leave all outputs untouched.  A failed launch returns
 *    MALA_ERR_CUDA.  Kernels that wait on on-chip barriers bound every wait;
 *    an expired wait is recorded in a device status word that
 *    mala_device_status() reads.
 *  - Optional instrumentation outputs may be NULL:
 *      retained_counts  int32, number of retained tiles per unit of work
 *      tile_mask        uint8, 1 = tile retained, 0 = tile skipped; the call
 *                       writes the entry of every legal tile and leaves the
 *                       others unchanged (zero the buffer first).
 */
#ifndef MALA_H_
#define MALA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MALA_OK = 0,
  MALA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad shape, tau < 0 or NaN */
  MALA_ERR_UNSUPPORTED = 2,  /* well-formed but not built: head_dim, tile size, dtype, or more than
                                2^31 - 1 CTAs (batch x heads_q x tiles along the longer sequence) */
  MALA_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than the *_workspace_size() */
  MALA_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
  MALA_ERR_TIMEOUT = 5       /* a bounded device-side wait expired (device status) */
} mala_status;

typedef enum {
  MALA_BF16 = 0,
  MALA_FP32 = 1
} mala_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* mala_status_string(mala_status status);

/*
 * MALA forward pass (Algorithm 1; test of Eq. (3)).
 *
 * For every query block of block_q rows, legal key blocks are visited from the
 * diagonal toward earlier keys; each tile's scores are formed, and the tile is
 * skipped iff  rowmax(S) - m - log(l) < log(tau / L_q)  for every valid row
 * with a legal key in the tile (a row with l = 0 retains).  Skipped tiles load
 * no V and leave (m, l, O) unchanged.  Writes o = O / l and lse = m + log l.
 *
 *  q [batch, seqlen_q, heads_q, head_dim]      in_dtype
 *  k, v [batch, seqlen_k, heads_kv, head_dim]  in_dtype
 *  o [batch, seqlen_q, heads_q, head_dim]      out_dtype
 *  lse [batch, heads_q, seqlen_q]              float
 *  causal: 1 = key k visible to query q iff k <= q (requires seqlen_q ==
 *          seqlen_k), L_q = q + 1;  0 = all keys visible, L_q = seqlen_k.
 *  block_q == block_k, in {64, 128}.  head_dim in {64, 128}.
 *  retained_counts: [batch, heads_q, ceil(seqlen_q / block_q)]
 *  tile_mask:       [batch, heads_q, ceil(seqlen_q / block_q), ceil(seqlen_k / block_k)]
 *  Needs no workspace.
 */
mala_status mala_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv,
                     int head_dim, mala_dtype in_dtype, mala_dtype out_dtype, int causal,
                     int block_q, int block_k, float tau, float softmax_scale,
                     int32_t* retained_counts, uint8_t* tile_mask, void* stream);

/*
 * Forward with given tile decisions (the matched-work study of the paper,
 * §3 "Normalized-Mass Allocation at Matched Work" and App. C.2).
 *
 * Softmax attention renormalised over the tiles tile_keep marks: no Eq. (3)
 * test is made; every legal tile with tile_keep != 0 is kept, every other
 * tile skipped, in the order mala_fwd visits them.  A row none of whose kept
 * tiles holds a legal key gets o = 0 and lse = -inf.  Runs on the CUDA cores
 * (an evaluation path, not the tensor-core kernel).
 *
 *  tile_keep [batch, heads_q, ceil(seqlen_q / block_q), ceil(seqlen_k / block_k)]
 *            uint8, device, required.
 *  Other arguments as for mala_fwd (tau is not taken).
 */
mala_status mala_fwd_forced(const void* q, const void* k, const void* v, void* o, float* lse,
                            int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv,
                            int head_dim, mala_dtype in_dtype, mala_dtype out_dtype, int causal,
                            int block_q, int block_k, float softmax_scale, const uint8_t* tile_keep,
                            int32_t* retained_counts, uint8_t* tile_mask, void* stream);

/*
 * Reference mass of every (query block, key tile) region (App. C.2: the
 * screening-disabled reference gives "the probability mass of every candidate
 * region"):
 *   region_mass[b, h, i, j] = sum over the valid rows q of query block i and
 *   the legal keys k of tile j of exp(scale * q . k - lse[b, h, q]).
 * With lse from a dense (tau = 0) forward each block's masses add up to its
 * number of valid rows.  Illegal tiles get 0.  CUDA cores.
 *
 *  q [batch, seqlen_q, heads_q, head_dim], k [batch, seqlen_k, heads_kv, head_dim]  in_dtype
 *  lse [batch, heads_q, seqlen_q] float (natural log), input
 *  region_mass [batch, heads_q, ceil(seqlen_q / block_q), ceil(seqlen_k / block_k)] float, output
 *  Shape rules as for mala_fwd.
 */
mala_status mala_region_mass(const void* q, const void* k, const float* lse, float* region_mass,
                             int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv,
                             int head_dim, mala_dtype in_dtype, int causal, int block_q, int block_k,
                             float softmax_scale, void* stream);

/* Bytes of device workspace mala_bwd needs for these sizes. */
size_t mala_bwd_workspace_size(int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv,
                               int head_dim, mala_dtype in_dtype, mala_dtype grad_dtype);

/*
 * MALA backward pass (Algorithm 2; test of Eq. (4)).
 *
 * Key-major: for each key block, the query blocks with a legal entry are
 * visited in ascending order; the recomputed tile S_ji is skipped iff
 * S_ji - lse_i < log(tau / L_i) for every valid causal entry.  Retained tiles
 * run P = exp(S - lse), dP = V dO^T, dS = P * (dP - rowsum(O * dO)),
 * dV += P dO, dK += dS Q, dQ += dS^T K.  Skipped tiles load no dO.
 *
 *  q, o, dout [batch, seqlen_q, heads_q, head_dim]   in_dtype
 *  k, v       [batch, seqlen_k, heads_kv, head_dim]  in_dtype
 *  lse        [batch, heads_q, seqlen_q] float, as written by mala_fwd
 *  dq         [batch, seqlen_q, heads_q, head_dim]   grad_dtype
 *  dk, dv     [batch, seqlen_k, heads_kv, head_dim]  grad_dtype
 *  workspace: >= mala_bwd_workspace_size(...) bytes, 256-byte aligned; its
 *             contents on entry do not matter.
 *  retained_counts: [batch, heads_q, ceil(seqlen_k / block_k)]
 *  tile_mask:       [batch, heads_q, ceil(seqlen_q / block_q), ceil(seqlen_k / block_k)]
 *  Other arguments as for mala_fwd.
 *
 * Range: with bf16 inputs and head_dim 128 (the tensor-core kernel) the
 * post-score products take fp16 operands, which hold every bf16 value of
 * magnitude up to 65504 (exactly from 2^-17 up).  A finite q, k, v or dout
 * element beyond 65504 sets bit 4 of the device status word
 * (mala_device_status returns MALA_ERR_INVALID_ARG) and the gradients of that
 * call are not valid.  fp32 inputs and the other shapes have no such limit.
 */
mala_status mala_bwd(const void* q, const void* k, const void* v, const void* o,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv,
                     int batch, int seqlen_q, int seqlen_k, int heads_q, int heads_kv,
                     int head_dim, mala_dtype in_dtype, mala_dtype grad_dtype, int causal,
                     int block_q, int block_k, float tau, float softmax_scale,
                     void* workspace, size_t workspace_bytes,
                     int32_t* retained_counts, uint8_t* tile_mask, void* stream);

/*
 * Variable-length prefill: mala_fwd / mala_bwd over a batch of sequences of
 * different lengths packed along one token axis (§2.1 counts L_q per query
 * row; each sequence is its own causal context).
 *
 * Sequence b holds the token rows cu_seqlens[b] .. cu_seqlens[b + 1] - 1 and
 * attends only within itself; each gives exactly what mala_fwd / mala_bwd
 * give on that sequence alone (batch 1, seqlen_q = seqlen_k = its length).
 *
 *  q, o, dout, dq   [total_tokens, heads_q,  head_dim]
 *  k, v, dk, dv     [total_tokens, heads_kv, head_dim]
 *  lse              [heads_q, total_tokens]  (float)
 *  cu_seqlens       [batch + 1] int32, device memory, 4-byte aligned, with
 *                   0 <= cu_seqlens[b] <= cu_seqlens[b + 1] <= total_tokens
 *                   and no sequence longer than max_seqlen (1 <= max_seqlen <= total_tokens)
 *  retained_counts  mala_fwd_varlen: [batch, heads_q, ceil(max_seqlen / block_q)];
 *                   mala_bwd_varlen: [batch, heads_q, ceil(max_seqlen / block_k)]
 *  tile_mask        [batch, heads_q, T, T], T = ceil(max_seqlen / block): a
 *                   sequence's entries past its own tiles are not written
 *  workspace        mala_bwd_varlen: >= mala_bwd_varlen_workspace_size(...) bytes
 * Everything else (dtypes, causal flag, tiles, tau, scale) as mala_fwd / mala_bwd.
 * The bounds are read on the device: a sequence that breaks them sets bit 2
 * of the device status word (mala_device_status) and is not computed (its
 * outputs are not written); the other sequences are unaffected.  A null or
 * misaligned cu_seqlens, or max_seqlen outside [1, total_tokens], returns
 * MALA_ERR_INVALID_ARG.
 */
mala_status mala_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int32_t* cu_seqlens, int batch, int total_tokens, int max_seqlen,
                            int heads_q, int heads_kv, int head_dim, mala_dtype in_dtype,
                            mala_dtype out_dtype, int causal, int block_q, int block_k, float tau,
                            float softmax_scale, int32_t* retained_counts, uint8_t* tile_mask,
                            void* stream);

/* Bytes of device workspace mala_bwd_varlen needs for these sizes. */
size_t mala_bwd_varlen_workspace_size(int total_tokens, int heads_q, int heads_kv, int head_dim,
                                      mala_dtype in_dtype, mala_dtype grad_dtype);

mala_status mala_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                            const void* dout, const float* lse, void* dq, void* dk, void* dv,
                            const int32_t* cu_seqlens, int batch, int total_tokens, int max_seqlen,
                            int heads_q, int heads_kv, int head_dim, mala_dtype in_dtype,
                            mala_dtype grad_dtype, int causal, int block_q, int block_k, float tau,
                            float softmax_scale, void* workspace, size_t workspace_bytes,
                            int32_t* retained_counts, uint8_t* tile_mask, void* stream);

/* Bytes of device workspace mala_decode needs for these sizes. */
size_t mala_decode_workspace_size(int batch, int heads_q, int head_dim, int num_splits);

/*
 * MALA split-KV decode (App. A.1 "Fused decoding execution"; §2.4).
 *
 * One new query per sequence against a cache of cache_len tokens that already
 * holds the current token, so L = cache_len for every row.  The
 * T = ceil(cache_len / block_k) key tiles are cut into num_splits contiguous
 * ranges of ceil(T / num_splits) tiles.  Each split starts from its own empty
 * (m, l), visits its tiles newest to oldest, scores every tile, and skips a
 * tile iff rowmax - m - log l < log(tau / cache_len) for all query heads of
 * the KV-head group (the group is the query block; l = 0 retains).  Retained
 * tiles load V and run softmax and P V.  The splits' (m, l, u) summaries are
 * merged exactly: m = max m_s, l = sum e^(m_s - m) l_s, u = sum e^(m_s - m) u_s,
 * o = u / l, lse = m + log l.
 *
 *  q [batch, heads_q, head_dim]                     in_dtype
 *  k_cache, v_cache [batch, cache_len, heads_kv, head_dim]  in_dtype
 *  o [batch, heads_q, head_dim]                     out_dtype
 *  lse [batch, heads_q]                             float
 *  heads_q / heads_kv in {1, 2, 4, 8}; head_dim in {64, 128}; block_k in {64, 128};
 *  1 <= num_splits <= 256.
 *  workspace: >= mala_decode_workspace_size(...) bytes, 256-byte aligned.
 *  retained_counts: [batch, heads_kv, num_splits]
 *  tile_mask:       [batch, heads_kv, ceil(cache_len / block_k)]
 */
mala_status mala_decode(const void* q, const void* k_cache, const void* v_cache, void* o,
                        float* lse, int batch, int cache_len, int heads_q, int heads_kv,
                        int head_dim, mala_dtype in_dtype, mala_dtype out_dtype, int block_k,
                        int num_splits, float tau, float softmax_scale,
                        void* workspace, size_t workspace_bytes,
                        int32_t* retained_counts, uint8_t* tile_mask, void* stream);

/*
 * MALA split-KV decode with per-head decisions (§2.2 states the skip rule per
 * query block; here each query head is its own one-row block).
 *
 * Same arguments, layouts, workspace and errors as mala_decode, and the same
 * split partition, order and merge.  The difference is who decides: each query
 * head tests every tile against its own (m, l) and log(tau / cache_len), and
 * a head that skips a tile leaves its (m, l, u) unchanged.  A tile's K is
 * always read; its V is read when any head of the KV group keeps it, since
 * the heads share it.  tau = 0 gives the same dense result as mala_decode.
 *
 *  retained_counts: [batch, heads_q, num_splits]   tiles each query head kept per split
 *  tile_mask:       [batch, heads_q, ceil(cache_len / block_k)]
 */
mala_status mala_decode_per_head(const void* q, const void* k_cache, const void* v_cache, void* o,
                                 float* lse, int batch, int cache_len, int heads_q, int heads_kv,
                                 int head_dim, mala_dtype in_dtype, mala_dtype out_dtype, int block_k,
                                 int num_splits, float tau, float softmax_scale,
                                 void* workspace, size_t workspace_bytes,
                                 int32_t* retained_counts, uint8_t* tile_mask, void* stream);

/*
 * Variable-length MALA split-KV decode: mala_decode over a batch whose
 * sequences hold different numbers of cached tokens (App. A.1; §2.1 counts
 * L per query, and a decoding query's L is its own cache length, current
 * token included).
 *
 * Sequence b attends to the first cache_lens[b] rows of its cache and tests
 * tiles against log(tau / cache_lens[b]).  Its ceil(cache_lens[b] / block_k)
 * tiles are cut into num_splits ranges exactly as mala_decode cuts a cache of
 * that length, so each sequence gives what mala_decode gives on its cache
 * truncated to cache_lens[b].
 *
 *  cache_lens [batch]                               int32, device memory, 4-byte aligned
 *  k_cache, v_cache [batch, max_cache_len, heads_kv, head_dim]  (rows past a
 *      sequence's length are never read into results)
 *  tile_mask [batch, heads_kv, ceil(max_cache_len / block_k)]: entries of a
 *      sequence's tiles past ceil(cache_lens[b] / block_k) are not written.
 *  Everything else as mala_decode, with max_cache_len in place of cache_len.
 *
 * The lengths are read on the device.  A length outside [1, max_cache_len]
 * sets bit 2 of the device status word (mala_device_status) and that
 * sequence's o and lse come out NaN; the other sequences are unaffected.
 * A null or misaligned cache_lens returns MALA_ERR_INVALID_ARG.
 */
mala_status mala_decode_varlen(const void* q, const void* k_cache, const void* v_cache, void* o,
                               float* lse, const int32_t* cache_lens, int batch, int max_cache_len,
                               int heads_q, int heads_kv, int head_dim, mala_dtype in_dtype,
                               mala_dtype out_dtype, int block_k, int num_splits, float tau,
                               float softmax_scale, void* workspace, size_t workspace_bytes,
                               int32_t* retained_counts, uint8_t* tile_mask, void* stream);

/*
 * mala_decode without a workspace argument, for callers that cannot allocate
 * device memory: for example a serving process whose device memory is all
 * handed out by a fixed pool at start-up and that may not call cudaMalloc
 * afterwards, or a host framework that calls this library from a plugin with
 * no allocator and no way to pass scratch space through its own interface.
 * The paper has no counterpart; it is the same split-KV decode and merge as
 * mala_decode (same arguments, same kernels, same results), except that the
 * per-split (m, l, u) records live in a fixed array inside the library.
 *
 *  - The array holds mala_decode_noalloc_max_floats() floats (1 Mi floats,
 *    4 MiB) on every device that loads the library, until the process exits.
 *    A call needs num_splits * batch * heads_q * (head_dim + 4) floats; larger
 *    shapes return MALA_ERR_WORKSPACE before anything is launched.
 *  - The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *    library routine.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents (every split rewrites its whole record before the merge reads
 *    it, so nothing needs clearing).  Calls that may overlap on the GPU -- on
 *    different streams without ordering between them -- race on the array and
 *    must not be issued; calls on one stream are ordered and safe.
 */
mala_status mala_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o,
                                float* lse, int batch, int cache_len, int heads_q, int heads_kv,
                                int head_dim, mala_dtype in_dtype, mala_dtype out_dtype, int block_k,
                                int num_splits, float tau, float softmax_scale,
                                int32_t* retained_counts, uint8_t* tile_mask, void* stream);

/* Capacity, in floats, of the array mala_decode_noalloc uses (see above). */
size_t mala_decode_noalloc_max_floats(void);

/*
 * Synchronise `stream`, then read and clear the device status word that the
 * kernels set.  Bits: 1 = a bounded on-chip wait expired (the kernel gave up
 * and its outputs are not valid); 2 = mala_decode_varlen read a sequence
 * length outside [1, max_cache_len], or mala_fwd_varlen / mala_bwd_varlen
 * read sequence bounds that break their contract; 4 = a bf16 input of the
 * tensor-core backward lies beyond fp16's range (see mala_bwd); 8 = only in
 * the bounds-checked build (libmala_debug.so, compiled with -DMALA_DEBUG): a
 * TMA box origin or global index of the tensor-core or decode kernels fell
 * outside the extents checked on the host; the access was skipped.
 * *device_code receives the raw word
 * (0 = no event).  Returns MALA_OK (word 0), MALA_ERR_TIMEOUT (bit 1 set),
 * MALA_ERR_INVALID_ARG (any other bit), or MALA_ERR_CUDA if synchronisation
 * failed.
 */
mala_status mala_device_status(void* stream, int* device_code);

/*
 * Test hook for failure detection (no counterpart in the paper).  The next
 * mala_fwd / mala_fwd_varlen call that runs on the tensor-core kernel has one
 * CTA leave its first K tile unloaded: that CTA's bounded waits expire (after
 * about 2 s), it gives up without writing its outputs, and bit 1 of the device
 * status word is set (mala_device_status returns MALA_ERR_TIMEOUT).  Nothing
 * faults or hangs, and later calls run normally.  One-shot, process-wide.
 */
void mala_test_drop_next_load(void);

/* Number of kernels this library has launched in this process (host counter). */
uint64_t mala_launch_count(void);

/* The cudaError_t behind this thread's most recent MALA_ERR_CUDA (0 if none),
 * and its description (static string). */
int mala_last_cuda_error(void);
const char* mala_cuda_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* MALA_H_ */
