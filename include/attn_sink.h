/*
 * attn_sink.h -- C ABI of a GB300 (sm_103a) library for attention with an
 * attention sink.
 *
 * Two forms of the sink are implemented:
 *
 *  1. A learnable per-head sink logit (flash-attention PR "feat: Implement Sink
 *     Attention", Description; sglang PR "openai oss attention sink support
 *     with trtllm-gen backend", Summary of Changes).  For query head h the
 *     value sink[h] is one extra logit that enters the softmax denominator and
 *     carries no value vector:
 *         m_i   = max(sink[h], max_j s_ij)
 *         Z_i   = exp(sink[h] - m_i) + sum_j exp(s_ij - m_i)
 *         O_i   = sum_j exp(s_ij - m_i) v_j / Z_i
 *         LSE_i = m_i + ln Z_i
 *     with s_ij = scale * q_i . k_j over the keys j that row i sees.  sink is
 *     in the units of the scaled logits.  sink == NULL means "no sink"
 *     (sink = -inf, i.e. plain softmax attention).
 *
 *  2. First-window + last-window KV selection over a paged KV cache (sglang PR
 *     "To implement attention-sink", Motivation and the review's suggested
 *     code: keep the first 1024 and the last 7168 tokens of every sequence).
 *     A query at absolute position p sees the keys
 *         [0, min(F, p+1))  U  [max(p+1-W, min(F, p+1)), p+1)
 *     where F = win_first and W = win_last.  win_last <= 0 turns selection
 *     off (plain causal).  The window is applied per sequence, token-exactly;
 *     partial pages are masked per token.  Selection needs causal attention.
 *
 * Conventions shared by every entry point:
 *  - Tensors are device pointers owned by the caller; the library keeps no
 *    pointer after it returns.  Layouts are dense row-major as documented.
 *  - bf16 tensors hold raw IEEE bfloat16 bits (attn_bf16).
 *  - Work is queued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and is asynchronous: a zero return means "validated and
 *    launched", not "finished".
 *  - Query row t of a request with Lq queries and Lk keys sits at absolute
 *    position Lk - Lq + t (bottom-right alignment: a cached prefix precedes
 *    the new chunk).  A row that sees no key has O = 0 and LSE = sink (or
 *    -inf without a sink); its gradients are 0.
 *  - scale <= 0 selects 1/sqrt(head_dim).
 *  - Scratch memory (split-KV partials, the fp32 dQ accumulator) is taken
 *    from a library-owned stream-ordered pool on `stream` and returned on
 *    the same stream; no call synchronises the host.
 *  - Return values: ATTN_SINK_OK, or a negative status.  The text of the
 *    last failure of the calling thread is available from
 *    attn_sink_last_error().
 *  - Out-of-range page ids and sequence lengths longer than the page table
 *    are caught on the device: the offending load is skipped and a sticky
 *    device status is set, which attn_sink_device_status() reports.
 *  - One call takes at most 65535 requests (batch) in the forward, paged
 *    forward, decode and append entry points, and at most 65535 * 128 query
 *    rows per request in the forward ones (each is one grid dimension of the
 *    launch); larger calls return ATTN_SINK_ERR_UNSUPPORTED.
 */
#ifndef ATTN_SINK_H
#define ATTN_SINK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t attn_bf16;

enum {
    ATTN_SINK_OK = 0,
    ATTN_SINK_ERR_INVALID = -1,      /* NULL pointer, negative size, bad flag combination */
    ATTN_SINK_ERR_UNSUPPORTED = -2,  /* head_dim, group size, page_size or a size limit   */
    ATTN_SINK_ERR_CUDA = -3,         /* a CUDA call failed (allocation, launch)            */
    ATTN_SINK_ERR_DEVICE = -4        /* a device-side check failed (see device_status)     */
};

/* Device-side status bits reported by attn_sink_device_status(). */
enum {
    ATTN_SINK_DEV_PAGE_OOB = 1,      /* a page-table entry was outside [0, num_pages)       */
    ATTN_SINK_DEV_SEQLEN_OOB = 2,    /* a sequence length exceeded max_pages * page_size    */
    ATTN_SINK_DEV_TIMEOUT = 4,       /* a pipeline wait ran out of time; the kernel gave up */
    ATTN_SINK_DEV_LAYOUT = 8         /* the dynamic shared-memory base was not 1024-byte
                                        aligned; the forward kernel did nothing            */
};

/*
 * Forward attention with a sink over varlen requests (prefill, chunked
 * extend, training forward).  Pages: flash-attention PR "feat: Implement Sink
 * Attention" (Key Changes: forward functions and their variable-length
 * counterparts take the sink); sglang PR "openai oss attention sink support with trtllm-gen backend" (Highlights: the extend path
 * passes sink=).
 *
 *   q            (total_q, hq, head_dim) bf16, total_q = cu_seqlens_q[batch]
 *   k, v         (total_k, hkv, head_dim) bf16; request b owns key rows
 *                [cu_seqlens_k[b], cu_seqlens_k[b+1]) (cached prefix then chunk)
 *   sink         (hq,) fp32 or NULL
 *   cu_seqlens_q, cu_seqlens_k   (batch+1,) int32 device, non-decreasing, [0]=0
 *   total_q, total_k             host row counts of q and k/v (the tensors'
 *                first extents); cu_seqlens_*[batch] must not exceed them --
 *                rows past them are never read or written and set
 *                ATTN_SINK_DEV_SEQLEN_OOB
 *   max_seqlen_q, max_seqlen_k   host upper bounds of the per-request lengths
 *                (size the grid; no device-to-host read)
 *   win_first, win_last          window selection (needs causal = 1)
 *   out          (total_q, hq, head_dim) bf16
 *   lse          (hq, total_q) fp32, natural log, includes the sink; may be NULL
 * Supported: head_dim 64 or 128; hq % hkv == 0.  A request's results depend on its
 * own rows only: the value rows that its last key tile covers past its last
 * key (another request's, or beyond cu_seqlens_k[batch]) are replaced by zeros
 * in shared memory, so they may hold anything, NaN included.
 * Input range: the online softmax exponentiates each tile against a running
 * reference that may lag the true row maximum by up to a factor 2^64, so the
 * un-normalised weights reach 2^64 and the fp32 accumulator of P V stays
 * finite while max|v| * Lk < 1.8e19 (|v| < 1.7e13 at a million keys); an
 * exact softmax would stay finite for any finite value.
 */
int attn_sink_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v,
                  const float* sink, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                  int batch, int total_q, int total_k, int hq, int hkv, int head_dim,
                  int max_seqlen_q, int max_seqlen_k,
                  int win_first, int win_last, int causal, float scale,
                  attn_bf16* out, float* lse, void* stream);

/*
 * attn_sink_fwd with explicit row strides, for packed layouts (the varlen
 * forward functions of flash-attention PR "feat: Implement Sink Attention",
 * Key Changes, come in packed-QKV and packed-KV forms).  q_row_stride,
 * k_row_stride, v_row_stride are the distances in elements between
 * consecutive token rows of q, k and v (0: contiguous, heads * head_dim).
 * Within a row the heads stay contiguous, head_dim elements apart.  A packed
 * (total, hq + 2*hkv, head_dim) QKV buffer is q = base, k = base + hq*head_dim,
 * v = base + (hq+hkv)*head_dim, all with row stride (hq + 2*hkv)*head_dim.
 * Strides must be 0 or >= heads*head_dim and multiples of 8; out stays
 * contiguous.  Everything else as in attn_sink_fwd.
 */
int attn_sink_fwd_strided(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v,
                          long long q_row_stride, long long k_row_stride, long long v_row_stride,
                          const float* sink, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                          int batch, int total_q, int total_k, int hq, int hkv, int head_dim,
                          int max_seqlen_q, int max_seqlen_k,
                          int win_first, int win_last, int causal, float scale,
                          attn_bf16* out, float* lse, void* stream);

/*
 * Paged single-token decode with a sink and optional first/last-window
 * selection.  Pages: sglang PR "openai oss attention sink support with trtllm-gen backend" (Highlights: the decode path passes
 * sink=); sglang PR "To implement attention-sink" (page table rows built from the first and last
 * windows, per sequence); flash-attention PR "feat: Implement Sink Attention" (a user reports the sink
 * giving wrong decode results through the KV-cache API -- here the sink is
 * folded exactly once, after the split-KV partials are merged).
 *
 *   q            (batch, hq, head_dim) bf16, one new token per request
 *   k_cache, v_cache  (num_pages, page_size, hkv, head_dim) bf16
 *   page_table   (batch, max_pages) int32 physical page ids; logical token t
 *                of request b lives in page page_table[b][t / page_size],
 *                row t % page_size.  Entries past a request's last page are
 *                never read.
 *   seqlens      (batch,) int32: cache length including the new token
 *   sink         (hq,) fp32 or NULL
 *   out          (batch, hq, head_dim) bf16
 *   lse          (batch, hq) fp32 or NULL
 * Supported: head_dim 64 or 128; hq % hkv == 0; page_size >= 1.
 */
int attn_sink_decode_paged(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                           const int32_t* page_table, int max_pages, const int32_t* seqlens,
                           int batch, int hq, int hkv, int head_dim, int page_size, int num_pages,
                           const float* sink, int win_first, int win_last, float scale,
                           attn_bf16* out, float* lse, void* stream);

/*
 * Allocation-free paged decode.  The paper has no counterpart: this entry
 * point exists for callers that cannot allocate device memory at call time
 * (an engine that reserved the whole GPU up front, a latency-critical path
 * that must not take the allocator's locks or its implicit synchronisation,
 * a host that only hands the library existing buffers).
 *
 * Same arguments, semantics and results as attn_sink_decode_paged (up to
 * rounding when it has to use longer splits), but its split-KV scratch lives
 * in one static 32 MiB device array inside the library instead of coming
 * from a memory pool.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *  - The array is shared by every call on a device and keeps the previous
 *    call's contents; every scratch entry a call reads is written earlier in
 *    the same call, so nothing needs clearing.  Calls whose work overlaps on
 *    the GPU (e.g. on two streams without ordering between them) race on the
 *    array: order them on one stream or with events.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture.
 *  - A GPU holds the 32 MiB from the moment the library's module is loaded
 *    on it until the process exits.
 *  - Requests whose partials cannot fit in 32 MiB even with one split per
 *    (request, head) -- batch * hq * (head_dim * 4 + 8) bytes -- are
 *    rejected with ATTN_SINK_ERR_UNSUPPORTED and a message naming the size.
 */
int attn_sink_decode_paged_noalloc(const attn_bf16* q, const attn_bf16* k_cache,
                                   const attn_bf16* v_cache, const int32_t* page_table,
                                   int max_pages, const int32_t* seqlens, int batch, int hq,
                                   int hkv, int head_dim, int page_size, int num_pages,
                                   const float* sink, int win_first, int win_last, float scale,
                                   attn_bf16* out, float* lse, void* stream);

/*
 * Writes new tokens' K/V rows into a paged cache (the cache update that
 * precedes attention in KV-cache decode: flash-attention PR "feat: Implement
 * Sink Attention", Description; a request's tokens are reached through its
 * page-table row: sglang PR "To implement attention-sink", suggested code).
 *
 *   k_new, v_new   (rows, hkv, head_dim) bf16; request b's new rows are
 *                  [cu_new[b], cu_new[b+1]), or row b alone when cu_new is NULL
 *   cu_new         (batch+1,) int32 device or NULL (then max_new must be 1)
 *   seqlens        (batch,) int32 device: cache length INCLUDING the new rows,
 *                  so request b's n_b new rows become its logical tokens
 *                  seqlens[b] - n_b .. seqlens[b] - 1
 *   page_table     (batch, max_pages) int32 device, as in attn_sink_decode_paged
 *   max_new        host upper bound of n_b (sizes the grid); a request with more
 *                  new rows than max_new has its extra rows left unwritten and
 *                  sets ATTN_SINK_DEV_SEQLEN_OOB
 *   k_cache, v_cache   (num_pages, page_size, hkv, head_dim) bf16, written in place
 * A row whose slot would fall outside the cache (page id outside
 * [0, num_pages), or more new rows than cached tokens) is skipped and sets
 * ATTN_SINK_DEV_PAGE_OOB / ATTN_SINK_DEV_SEQLEN_OOB.  Rows of different
 * requests must not share a slot (the write order between them is undefined).
 * Supported: head_dim 64 or 128.
 */
int attn_sink_kv_append(const attn_bf16* k_new, const attn_bf16* v_new, const int32_t* cu_new,
                        const int32_t* seqlens, const int32_t* page_table, int max_pages, int batch,
                        int hkv, int head_dim, int page_size, int num_pages, int max_new,
                        attn_bf16* k_cache, attn_bf16* v_cache, void* stream);

/*
 * Paged decode with the new token's K/V appended in the same call: writes
 * k_new[b], v_new[b] ((batch, hkv, head_dim) bf16) at logical token
 * seqlens[b] - 1 of each request, then runs attn_sink_decode_paged on the
 * updated caches (KV-cache decode with a sink: flash-attention PR "feat:
 * Implement Sink Attention", Description).  Every other argument as in
 * attn_sink_decode_paged; k_cache / v_cache are written.  The call makes no
 * host synchronisation and depends only on its arguments, so it can be
 * captured in a CUDA graph (its scratch comes from a stream-ordered pool).
 */
int attn_sink_decode_paged_append(const attn_bf16* q, const attn_bf16* k_new, const attn_bf16* v_new,
                                  attn_bf16* k_cache, attn_bf16* v_cache, const int32_t* page_table,
                                  int max_pages, const int32_t* seqlens, int batch, int hq, int hkv,
                                  int head_dim, int page_size, int num_pages, const float* sink,
                                  int win_first, int win_last, float scale, attn_bf16* out,
                                  float* lse, void* stream);

/*
 * attn_sink_fwd on HOST-resident tensors: the library copies each request's
 * q / k / v rows to the device, runs the forward for that request and copies
 * its out / lse rows back, pipelined on library-owned streams so that the copies
 * of neighbouring requests overlap the kernel (same arithmetic and results as
 * attn_sink_fwd).  All tensor arguments, cu_seqlens_q and cu_seqlens_k
 * included, are host pointers; the layouts are those of attn_sink_fwd and the
 * row counts come from cu_seqlens_*[batch].  Host buffers should be
 * page-locked (cudaHostAlloc / cudaHostRegister) for the copies to overlap;
 * pageable buffers still give correct results, without overlap.  Returns once
 * the work is queued; `stream` waits for all of it (synchronise `stream`
 * before reading out / lse).  Device scratch for the whole batch comes from the
 * library's stream-ordered pool.  Supported: head_dim 64 or 128; hq % hkv == 0.
 */
int attn_sink_fwd_host(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v,
                       const float* sink, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                       int batch, int hq, int hkv, int head_dim, int win_first, int win_last,
                       int causal, float scale, attn_bf16* out, float* lse, void* stream);

/*
 * Varlen extend / prefill whose keys and values live in a paged cache (the
 * serving extend path: sglang PR "openai oss attention sink support with
 * trtllm-gen backend", Highlights: the extend path passes sink=; the prefix is
 * reached through the page table: sglang PR "To implement attention-sink",
 * suggested code).  Request b's query rows [cu_seqlens_q[b], cu_seqlens_q[b+1])
 * are the LAST Lq_b of its seqlens_k[b] cached tokens (bottom-right causal
 * alignment, as in attn_sink_fwd).
 *
 *   q            (total_q, hq, 64) bf16
 *   k_new, v_new (total_q, hkv, 64) bf16, the chunk's own K/V, or both NULL.
 *                When given they are first appended into the cache at the
 *                chunk's positions (attn_sink_kv_append with cu_new =
 *                cu_seqlens_q); when NULL the cache must already hold them.
 *   k_cache, v_cache  (num_pages, page_size, hkv, 64) bf16
 *   page_table   (batch, max_pages) int32 device
 *   seqlens_k    (batch,) int32 device, prefix + chunk
 *   max_seqlen_q, max_seqlen_k   host upper bounds (grid sizing, append grid)
 *   sink, win_first, win_last, causal, scale, out, lse: as in attn_sink_fwd
 * Supported: head_dim 64 or 128; hq % hkv == 0; page_size a power of two >= 8
 * (a 128-key tile is then one TMA copy per page segment).  Cache slots that a
 * request does not own (the rest of its last page, any other page) never
 * reach its results and may hold anything, NaN included.
 */
int attn_sink_fwd_paged(const attn_bf16* q, const attn_bf16* k_new, const attn_bf16* v_new,
                        attn_bf16* k_cache, attn_bf16* v_cache, const int32_t* page_table,
                        int max_pages, const int32_t* cu_seqlens_q, const int32_t* seqlens_k,
                        int batch, int total_q, int hq, int hkv, int head_dim, int page_size,
                        int num_pages, int max_seqlen_q, int max_seqlen_k, const float* sink,
                        int win_first, int win_last, int causal, float scale, attn_bf16* out,
                        float* lse, void* stream);

/*
 * Backward of attn_sink_fwd: gradients of sum(dout * out) with respect to q,
 * k, v and the sink.  Page: flash-attention PR "feat: Implement Sink Attention" (Key Changes: the
 * backward pass computes and returns the gradient of the learnable sink).
 * dsink[h] = -sum_i exp(sink[h] - LSE_i) * rowsum(dout_i * out_i).
 *
 *   q, k, v, sink, cu_seqlens_*, sizes, windows, causal, scale: as in attn_sink_fwd
 *   out, lse     the forward's outputs (lse is required here)
 *   dout         (total_q, hq, head_dim) bf16
 *   dq           (total_q, hq, head_dim) bf16
 *   dk, dv       (total_k, hkv, head_dim) bf16 (summed over the query heads
 *                of each KV head)
 *   dsink        (hq,) fp32; must be non-NULL iff sink is non-NULL; written
 *                (not accumulated)
 * Supported: head_dim 64 or 128 (one pass each: 128-row query steps at 64,
 * 64-row steps at 128); hq % hkv == 0.  A request's gradients depend on
 * its own rows only: the rows that its last query or key tile covers past its
 * own (another request's, or past total_q / total_k) are replaced by zeros in
 * shared memory, so they may hold anything, NaN included.
 */
int attn_sink_bwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, const float* sink,
                  const attn_bf16* out, const float* lse, const attn_bf16* dout,
                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                  int batch, int total_q, int total_k, int hq, int hkv, int head_dim,
                  int max_seqlen_q, int max_seqlen_k,
                  int win_first, int win_last, int causal, float scale,
                  attn_bf16* dq, attn_bf16* dk, attn_bf16* dv, float* dsink, void* stream);

/*
 * attn_sink_bwd with explicit row strides for q, k, v (inputs) and dq, dk, dv
 * (outputs), for packed QKV / KV layouts (as in attn_sink_fwd_strided; a packed
 * dQKV output uses the same offsets and stride as the packed QKV input).  out,
 * lse and dout stay contiguous.  With any of the dk / dv strides non-zero, dk/dv
 * rows past cu_seqlens_k[batch] are left untouched (instead of zeroed).
 */
int attn_sink_bwd_strided(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v,
                          long long q_row_stride, long long k_row_stride, long long v_row_stride,
                          const float* sink, const attn_bf16* out, const float* lse,
                          const attn_bf16* dout, const int32_t* cu_seqlens_q,
                          const int32_t* cu_seqlens_k, int batch, int total_q, int total_k, int hq,
                          int hkv, int head_dim, int max_seqlen_q, int max_seqlen_k,
                          int win_first, int win_last, int causal, float scale,
                          attn_bf16* dq, attn_bf16* dk, attn_bf16* dv,
                          long long dq_row_stride, long long dk_row_stride, long long dv_row_stride,
                          float* dsink, void* stream);

/*
 * The visible token ranges of each decode request, as the decode kernels
 * compute them on the device (sglang PR "To implement attention-sink", suggested code: first window
 * [:F] and last window [L-W:L], per sequence).
 *   seqlens  (batch,) int32 device
 *   ranges   (batch, 4) int32 device: a0, b0, a1, b1 with visible =
 *            [a0,b0) U [a1,b1), disjoint and increasing.
 */
int attn_sink_visible_ranges(const int32_t* seqlens, int batch, int win_first, int win_last,
                             int32_t* ranges, void* stream);

/*
 * The physical KV slot of every visible token, in the order the decode
 * kernels read them: slot = page_table[b][t / page_size] * page_size
 * + t % page_size for the visible logical tokens t of request b.
 *   slots    (batch, max_visible) int32 device; row b holds the request's
 *            visible slots followed by -1 padding (and -1 where a page id
 *            is outside [0, num_pages), which also sets
 *            ATTN_SINK_DEV_PAGE_OOB).  max_visible must be at least the
 *            largest visible count.
 */
int attn_sink_visible_slots(const int32_t* seqlens, const int32_t* page_table, int max_pages,
                            int batch, int page_size, int num_pages, int win_first, int win_last,
                            int32_t* slots, int max_visible, void* stream);

/*
 * Reads and clears the sticky device status (a bitwise OR of the
 * ATTN_SINK_DEV_* bits set by kernels since the last call) for the current
 * device.  Synchronises `stream`.  Returns the bits, or ATTN_SINK_ERR_CUDA.
 */
int attn_sink_device_status(void* stream);

/*
 * Self-test of the bounded wait behind every pipeline barrier of the kernels
 * (no counterpart on the pages: it is how a stalled pipeline is detected).
 * Launches one single-thread kernel on `stream` that waits on an mbarrier of
 * its own.  complete != 0: the barrier's phase is completed first and the wait
 * returns at once (no status).  complete == 0: nothing arrives, the wait gives
 * up after its time limit (1 s), sets ATTN_SINK_DEV_TIMEOUT and the kernel
 * returns; the context stays usable.  Asynchronous; returns ATTN_SINK_OK or
 * ATTN_SINK_ERR_CUDA (launch failure).
 */
int attn_sink_selftest_wait(int complete, void* stream);

/* Text of the calling thread's last failure ("" if none).  Never NULL. */
const char* attn_sink_last_error(void);

/* Library version string. */
const char* attn_sink_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_SINK_H */
