/*
 * sparse_mla.h -- C ABI of the GB300 (sm_103a) sparse MLA attention forward (DSA top-k) and
 * its backward.
 *
 * The operation (FlashMLA PR #196, "Problem" and "Fix"; FlashMLA PR #216, "Summary";
 * FlashMLA PR #198, "Summary" item 2):
 *   For every query row t and head h, only the slots j of the row's index list that satisfy
 *       j < L_t   and   0 <= indices[t][j] < s_kv
 *   take part, where L_t = clamp(topk_length[t], 0, topk) when topk_length is given and
 *   L_t = topk otherwise.  With K = kv[:, :d_qk] and V = kv[:, :d_v] (the same latent row),
 *       logit_j   = sm_scale * <q[t,h,:], K[idx_j]>
 *       m         = max_j logit_j                         -> max_logits[t,h]
 *       lse[t,h]  = m + ln sum_j exp(logit_j - m)         (natural log, sink excluded)
 *       O[t,h,:]  = sum_j exp(logit_j - m) V[idx_j] / (sum_j exp(logit_j - m)
 *                                                      + [attn_sink] exp(attn_sink[h] - m))
 *   A row without any counted slot yields O = 0, lse = +inf, max_logits = -inf, with or
 *   without a sink.  Slots beyond L_t are never read, so their index values are unconstrained
 *   (e.g. INT_MAX padding is fine).  A duplicated index counts once per slot.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers to contiguous row-major buffers.  The caller
 *     owns every buffer; the library allocates nothing and keeps no pointer after the call.
 *   - bf16 tensors are passed as `void*` holding IEEE bfloat16 values.
 *   - The work is enqueued on `stream` and is asynchronous: a return value of SMLA_OK only
 *     means the launch was accepted.  No launch happens when an error code is returned.
 *   - s_q == 0 is a no-op that returns SMLA_OK (pointers are then not inspected).
 *   - Supported shapes: h_q a positive multiple of 64 (<= 1024), d_qk in {512, 576},
 *     d_v == 512, topk >= 1, sm_scale finite and > 0, s_q * h_q <= INT32_MAX.
 *   - Alignment: q and kv (or kv_pool) 16-byte aligned; every other pointer 4-byte aligned.
 *   - Requires an sm_103a device (GB300).
 */
#ifndef SPARSE_MLA_GB300_H_
#define SPARSE_MLA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SMLA_ABI_VERSION 4

typedef struct CUstream_st* smla_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  SMLA_OK = 0,
  SMLA_ERR_NULL_PTR = 1,       /* a required pointer is NULL */
  SMLA_ERR_BAD_SHAPE = 2,      /* a size or scalar argument is outside the supported set */
  SMLA_ERR_MISALIGNED = 3,     /* a pointer violates the alignment rule above */
  SMLA_ERR_LAUNCH = 4,         /* the CUDA launch (or a CUDA query) failed */
  SMLA_ERR_DEVICE_TIMEOUT = 5, /* a device-side wait gave up (see sparse_mla_device_status) */
  SMLA_ERR_TENSOR_MAP = 6,     /* the TMA descriptor for an operand could not be encoded */
  SMLA_ERR_WORKSPACE = 7       /* split-KV workspace missing or smaller than required */
} smla_status;

/*
 * Sparse MLA forward over one shared latent KV (FlashMLA PR #196, "Problem": the sparse
 * prefill forward; one latent KV stream, h_kv = 1).
 *   q            [s_q, h_q, d_qk]  bf16
 *   kv           [s_kv, 1, d_qk]   bf16; V is kv[:, :, :d_v]
 *   indices      [s_q, 1, topk]    int32; any value, -1 / <0 / >= s_kv mean "no key"
 *   topk_length  [s_q]             int32 or NULL (FlashMLA PR #216, "Summary")
 *   attn_sink    [h_q]             fp32 or NULL (logit units of sm_scale * q.k)
 *   out          [s_q, h_q, d_v]   bf16   (written)
 *   lse          [s_q, h_q]        fp32   (written)
 *   max_logits   [s_q, h_q]        fp32   (written)
 * When topk_length is NULL, each row's work is bounded by its last valid slot, found by a
 * scan in the kernel prologue (FlashMLA PR #196, "Fix"); results are identical to passing
 * that length explicitly.  A row's counted slots are packed into dense 64-slot blocks, so
 * invalid entries anywhere in the row cost no compute; the result does not depend on where
 * they sit.
 */
smla_status sparse_mla_fwd(const void* q, const void* kv, const int32_t* indices,
                           const int32_t* topk_length, const float* attn_sink, float sm_scale,
                           int d_v, void* out, float* lse, float* max_logits, int64_t s_q,
                           int64_t s_kv, int h_q, int d_qk, int topk, smla_stream_t stream);

/*
 * Same forward over a paged KV cache (FlashMLA PR #216, "Dynamic top-k": decode with
 * per-request top-k token positions in a cache of 64-token pages).
 *   kv_pool      [pool_rows, 1, d_qk] bf16; pool_rows = number of pages * page_block
 *   block_table  [s_q / s_q_per_req, max_blocks] int32: page id of each page_block-token
 *                block of every request; a negative entry marks an unmapped page
 *   seqlens_k    [s_q / s_q_per_req] int32 KV length of each request, or NULL to use
 *                s_kv_per_req for all requests
 *   indices      [s_q, 1, topk] int32 token positions within the row's request
 * Query row t belongs to request t / s_q_per_req (s_q must be a multiple of s_q_per_req).
 * Position p of request b is read from pool row block_table[b][p / page_block] * page_block
 * + p % page_block, and counts iff 0 <= p < seqlens_k[b], p / page_block < max_blocks, the
 * table entry is >= 0 and the row is < pool_rows; any other position is an invalid slot and is
 * never used as an address (FlashMLA PR #216, "Summary").
 * All other arguments and outputs are as in sparse_mla_fwd.
 */
smla_status sparse_mla_fwd_paged(const void* q, const void* kv_pool, int64_t pool_rows,
                                 const int32_t* block_table, int max_blocks, int page_block,
                                 const int32_t* seqlens_k, int64_t s_kv_per_req, int s_q_per_req,
                                 const int32_t* indices, const int32_t* topk_length,
                                 const float* attn_sink, float sm_scale, int d_v, void* out,
                                 float* lse, float* max_logits, int64_t s_q, int h_q, int d_qk,
                                 int topk, smla_stream_t stream);

/*
 * Split-KV variants, for calls with fewer (row, 64-head group) items than SMs (small-batch
 * decode).  Each row's slot list [0, L_t) is cut into n_split contiguous ranges of
 * ceil(ceil(L_t / n_split) / 64) * 64 slots; every (row, head group, range) is one work unit
 * whose partial result (unnormalised O, exponent offset, sum, max) goes to `workspace`, and a
 * second kernel on the same stream merges a row's ranges with log-sum-exp weights (the sink
 * joins the denominator there) and writes out / lse / max_logits.  Same semantics and
 * outputs as sparse_mla_fwd / sparse_mla_fwd_paged up to summation order; with n_split == 1
 * they are the same call (no workspace needed).
 *   n_split          1 .. 64
 *   workspace        device buffer of at least sparse_mla_splitkv_workspace_size(s_q, h_q,
 *                    n_split) bytes, 256-byte aligned, owned by the caller; its contents
 *                    need no initialisation and are meaningless after the call.  Two calls
 *                    in flight at once must not share a workspace.
 * Errors as in the base calls, plus SMLA_ERR_BAD_SHAPE for n_split outside 1..64 and
 * SMLA_ERR_WORKSPACE when the workspace is NULL or too small (n_split > 1).
 */
size_t sparse_mla_splitkv_workspace_size(int64_t s_q, int h_q, int n_split);

smla_status sparse_mla_fwd_splitkv(const void* q, const void* kv, const int32_t* indices,
                                   const int32_t* topk_length, const float* attn_sink, float sm_scale,
                                   int d_v, void* out, float* lse, float* max_logits, int64_t s_q,
                                   int64_t s_kv, int h_q, int d_qk, int topk, int n_split,
                                   void* workspace, size_t workspace_bytes, smla_stream_t stream);

smla_status sparse_mla_fwd_paged_splitkv(const void* q, const void* kv_pool, int64_t pool_rows,
                                         const int32_t* block_table, int max_blocks, int page_block,
                                         const int32_t* seqlens_k, int64_t s_kv_per_req,
                                         int s_q_per_req, const int32_t* indices,
                                         const int32_t* topk_length, const float* attn_sink,
                                         float sm_scale, int d_v, void* out, float* lse,
                                         float* max_logits, int64_t s_q, int h_q, int d_qk, int topk,
                                         int n_split, void* workspace, size_t workspace_bytes,
                                         smla_stream_t stream);

/*
 * Allocation-free form of sparse_mla_fwd_paged_splitkv: the split-KV partial results go to a
 * scratch array that lives in the library itself (a 32 MiB __device__ array per device)
 * instead of a caller workspace, so the call needs no buffer besides its inputs and outputs.
 *   - Problems whose partial results do not fit, i.e. sparse_mla_splitkv_workspace_size(s_q,
 *     h_q, n_split) > 32 MiB (33554432 bytes), are rejected with SMLA_ERR_WORKSPACE before
 *     anything runs.
 *   - Nothing in the scratch has to start at zero (every work unit writes its whole partial
 *     result before the merge reads it), so the call clears nothing.
 *   - Races: all calls on one device share the one scratch array.  Two calls whose kernels
 *     may overlap (different streams, or different host threads without ordering) corrupt
 *     each other's partial results; callers must order them (same stream, or an event or
 *     synchronisation between them).  Calls on different devices are independent.
 * With n_split == 1 the scratch is not used.  Other arguments, outputs and errors are as in
 * sparse_mla_fwd_paged_splitkv.
 */
smla_status sparse_mla_fwd_paged_splitkv_static(
    const void* q, const void* kv_pool, int64_t pool_rows, const int32_t* block_table, int max_blocks,
    int page_block, const int32_t* seqlens_k, int64_t s_kv_per_req, int s_q_per_req,
    const int32_t* indices, const int32_t* topk_length, const float* attn_sink, float sm_scale, int d_v,
    void* out, float* lse, float* max_logits, int64_t s_q, int h_q, int d_qk, int topk, int n_split,
    smla_stream_t stream);

/*
 * End-to-end form of sparse_mla_fwd for inputs and outputs that live in HOST memory: the
 * host -> device copies of the inputs, the forward and the device -> host copies of the
 * outputs, pipelined over row chunks so that the copies of one chunk overlap the compute of
 * another.  Rows are independent, so the results are bit-identical to one sparse_mla_fwd call.
 *   *_host       host buffers with the layouts of sparse_mla_fwd (inputs read, outputs
 *                written); page-locked (pinned) memory is needed for the copies to overlap
 *   *_dev        caller-owned device buffers of the full sizes, with the alignment rules of
 *                sparse_mla_fwd; the inputs are copied into them and the outputs computed in
 *                them.  topk_length_dev / attn_sink_dev are NULL exactly when their host
 *                counterparts are (kv_host / kv_dev may be NULL only when s_kv == 0)
 *   n_chunks     1 .. 64: the rows are cut into n_chunks ranges of ceil(s_q / n_chunks) rows
 *   stream       the compute stream; when it has finished, every output copy has finished
 *   copy_in      stream of the host -> device copies (kv and attn_sink first, then each chunk)
 *   copy_out     stream of the device -> host copies
 * The copies start after the work already queued on `stream`, so the call is ordered on
 * `stream` as a whole.  The three streams are ordered with CUDA events from a pool that the
 * first call on a device creates and keeps until exit (no memory is allocated); calls from
 * several host threads take turns while they enqueue.  The call only enqueues work:
 * synchronise `stream` before reading the host outputs.  Every argument is checked before
 * anything is enqueued; SMLA_ERR_LAUNCH (a failed copy, event or launch) can come after
 * earlier chunks were enqueued.
 */
smla_status sparse_mla_fwd_host(const void* q_host, const void* kv_host, const int32_t* indices_host,
                                const int32_t* topk_length_host, const float* attn_sink_host, float sm_scale,
                                int d_v, void* out_host, float* lse_host, float* max_logits_host, int64_t s_q,
                                int64_t s_kv, int h_q, int d_qk, int topk, void* q_dev, void* kv_dev,
                                int32_t* indices_dev, int32_t* topk_length_dev, float* attn_sink_dev, void* out_dev,
                                float* lse_dev, float* max_logits_dev, int n_chunks, smla_stream_t stream,
                                smla_stream_t copy_in, smla_stream_t copy_out);

/*
 * Reads (and, when reset != 0, clears) the device-side status word that kernels set when one
 * of their bounded waits gave up: SMLA_OK or SMLA_ERR_DEVICE_TIMEOUT.  Synchronises with the
 * device (a blocking copy of one int); SMLA_ERR_LAUNCH if that copy fails.
 */
smla_status sparse_mla_device_status(int reset);

/*
 * Diagnostic of the failure-detection path: launches a one-thread kernel that runs the same
 * bounded mbarrier wait the forward kernels use, on a barrier nothing ever completes.  After
 * limit_ns (1 .. 2e9 ns) of device time the wait gives up, the kernel sets the status word to
 * SMLA_ERR_DEVICE_TIMEOUT and returns; the context stays usable.  Read the result with
 * sparse_mla_device_status after synchronising.  SMLA_ERR_BAD_SHAPE for a limit out of range.
 */
smla_status sparse_mla_selftest_wait_timeout(uint64_t limit_ns, smla_stream_t stream);

/*
 * Sparse MLA backward over one shared latent KV (FlashMLA PR #198, "Summary" item 1: the
 * sparse MLA backward, dK / dV scattered into the shared latent rows).  It returns the
 * gradients of  L = sum_{t,h,d} dout[t,h,d] * O[t,h,d]  for the forward above:
 *   p_j      = exp(sm_scale <q[t,h,:], K[idx_j]> - lse_full[t,h]),
 *              lse_full = ln(exp(lse[t,h]) + [attn_sink] exp(attn_sink[h]))
 *   D[t,h]   = <dout[t,h,:], out[t,h,:]>,   dS_j = p_j (<dout[t,h,:], V[idx_j]> - D[t,h])
 *   dq[t,h,:]            = sm_scale sum_j dS_j K[idx_j]
 *   dkv[idx_j, :d_qk]   += sm_scale dS_j q[t,h,:]     (summed over every row, head and slot)
 *   dkv[idx_j, :d_v]    += p_j dout[t,h,:]
 *   dsink[h]            += -exp(attn_sink[h] - lse_full[t,h]) D[t,h]
 * over the same counted slots as the forward (j < L_t and 0 <= idx < s_kv; duplicated indices
 * count once per slot).  A row without a counted slot contributes nothing (its dq is 0).
 *   q, kv, indices, topk_length, attn_sink, sm_scale, d_v: as for sparse_mla_fwd
 *   out          [s_q, h_q, d_v]   bf16   the forward's output (16-byte aligned)
 *   dout         [s_q, h_q, d_v]   bf16   gradient of the loss w.r.t. out (16-byte aligned)
 *   lse          [s_q, h_q]        fp32   the forward's lse (natural log, sink excluded)
 *   dq           [s_q, h_q, d_qk]  fp32   (written)
 *   dkv          [s_kv, d_qk]      fp32   (written: zeroed on the stream, then accumulated
 *                                          with fp32 atomics, so the summation order and the
 *                                          last bits vary from run to run); may be NULL only
 *                                          when s_kv == 0
 *   dsink        [h_q]             fp32 or NULL (written when attn_sink is given: zeroed,
 *                                          then accumulated; zeroed otherwise)
 * Every row's work is bounded by L_t (topk_length, or topk); slots in [0, L_t) that do not
 * count are masked.  Uses no workspace and allocates nothing.  With s_q == 0, dkv and dsink
 * are zeroed and nothing else happens.  Every error except SMLA_ERR_LAUNCH is returned before
 * anything is enqueued; SMLA_ERR_LAUNCH may come after the zeroing of dkv and dsink was
 * queued, which then leaves them zeroed.
 */
smla_status sparse_mla_bwd(const void* q, const void* kv, const void* out, const void* dout,
                           const int32_t* indices, const int32_t* topk_length, const float* attn_sink,
                           const float* lse, float sm_scale, int d_v, float* dq, float* dkv, float* dsink,
                           int64_t s_q, int64_t s_kv, int h_q, int d_qk, int topk, smla_stream_t stream);

/* Static, human-readable description of a status code.  Never NULL. */
const char* sparse_mla_status_string(smla_status status);

/* SMLA_ABI_VERSION of the loaded library. */
int sparse_mla_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MLA_GB300_H_ */
