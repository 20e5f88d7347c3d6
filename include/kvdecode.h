/*
 * kvdecode.h -- C ABI of the GB300 (sm_103a) KV-cached decoder-step library.
 *
 * The library implements the data-parallel hot path of KV-cached autoregressive
 * decoding: appending the new tokens' K/V to a per-layer cache, single-query
 * attention over that cache and over cross-attention K/V computed once per audio
 * window, the k-token causal verify pass of speculative decoding, the greedy
 * accept-to-first-mismatch step, and the beam-search cache reorder.
 *
 * Sources (web pages; cited by title and section):
 *   [W] readoss.com, "Whisper のデコーダー内部：Beam Search、Logit フィルター、KV キャッシュ"
 *   [S] agentlenshq.com, "추측 디코딩으로 Whisper 추론 속도 2배 향상"
 *   [N] agentlenshq.com, "nanoVLM における KV キャッシュ実装"
 *   [A] aitime.ge, Whisper speculative-decoding article ("The quick brown sock/fox" example)
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Memory: every tensor pointer is DEVICE memory owned by the caller. The library
 *    never allocates, frees or synchronises. Calls are asynchronous on `stream`
 *    (a cudaStream_t; NULL is the legacy default stream) and contain no host
 *    synchronisation, so they can be captured in a CUDA graph.
 *  - Host errors: a non-KVD_OK status is returned synchronously and nothing is
 *    launched (null pointers, unsupported shapes, misalignment, a workspace that is
 *    too small). KVD_ERR_CUDA reports a launch failure (cudaGetLastError).
 *  - Device errors: conditions only visible on the device (a length past the
 *    capacity, a parent outside its window, a draft id outside the vocabulary, a
 *    NaN logit) are written to `*dev_err` with an atomic compare-and-swap from 0, so
 *    the first code wins; the offending unit of work is skipped, nothing traps and
 *    nothing spins. `dev_err` (device int32) may be NULL to ignore them. The caller
 *    reads and clears it when it chooses.
 *  - Layout: a per-layer cache is K, V : [batch, n_kv_heads, capacity, head_dim],
 *    head_dim contiguous ([N] "KV キャッシュが推論を最適化する方法": the per-layer key
 *    and value tensors are kept as (batch, heads, seq_len_cached, head_dim)). Other
 *    strides are given in elements. head_dim must be 64. Pointers and the strides
 *    times the element size must be multiples of 16 bytes.
 *  - Types: KVD_F16 or KVD_BF16 for q, the cache and the outputs; arithmetic is fp32
 *    and outputs are rounded to nearest even. greedy_accept reads fp32 logits.
 *  - Workspace: the attention and accept calls split work across thread blocks and
 *    merge partial results through `workspace` (device memory, at least
 *    kvd_workspace_size() bytes, 256-byte aligned). Its first KVD_WS_COUNTER_BYTES
 *    hold arrival counters that MUST be zero before the first call that uses the
 *    buffer; every call returns them to zero when it completes. One workspace may be
 *    shared by calls on one stream; calls that may run concurrently need separate
 *    workspaces.
 *  - Flags: KVD_FLAG_PDL launches the kernel with programmatic stream serialization
 *    (programmatic dependent launch): it may start while the previous kernel on the
 *    stream is still running, waits for that kernel to finish before reading any
 *    input or writing any output, and lets the next kernel start once its own first
 *    copies are issued. KVD_FLAG_EARLY_KV (attention only; implies KVD_FLAG_PDL) also
 *    reads `lens` and starts copying cached K/V BEFORE that wait. Use it only when no
 *    kernel that can still be running writes those cache positions or `lens`: cross
 *    K/V written once per audio window qualify, and so does a self cache whose new
 *    tokens come through the fused append (they are never read from the cache in the
 *    call that appends them). q, the new tokens, outputs and the workspace are always
 *    accessed after the wait.
 *  - Threading: no global mutable state except a per-device attribute cache; calls
 *    from several host threads are safe.
 */
#ifndef KVDECODE_H
#define KVDECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kvd_stream_t; /* identical to cudaStream_t */

typedef enum kvd_status {
    KVD_OK = 0,
    KVD_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad alignment, aliasing */
    KVD_ERR_UNSUPPORTED = 2,  /* head_dim != 64, qlen > 16, beam > 8, ... */
    KVD_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than kvd_workspace_size() */
    KVD_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    /* device-side codes, written to *dev_err */
    KVD_ERR_LEN_OVERFLOW = 16, /* a length < 0 or > capacity (or lens + q > capacity) */
    KVD_ERR_BAD_INDEX = 17,    /* a beam parent outside its window's block */
    KVD_ERR_BAD_TOKEN = 18,    /* a draft id outside [0, vocab) */
    KVD_ERR_NAN = 19,          /* a NaN among the logits */
    KVD_ERR_TIMEOUT = 20       /* a bounded wait for a shared-memory copy gave up; the
                                  workspace counters may be left non-zero: re-zero them */
} kvd_status;

typedef enum kvd_dtype { KVD_F16 = 0, KVD_BF16 = 1 } kvd_dtype;

typedef enum kvd_op {
    KVD_OP_DECODE_ATTN = 0,
    KVD_OP_VERIFY_ATTN = 1,
    KVD_OP_GREEDY_ACCEPT = 2,
    KVD_OP_SAMPLE_ACCEPT = 3
} kvd_op;

enum {
    KVD_FLAG_PDL = 1u << 0,
    KVD_FLAG_EARLY_KV = 1u << 1,
    /* Test only. kvd_prefill_attn: the attention kernel's producer does not issue the
     * copy of the first K tile, so that copy's wait and the rows' waits run out after
     * about one second each; the call must then report KVD_ERR_TIMEOUT through dev_err,
     * leave the outputs unwritten, release its tensor memory and leave the stream
     * usable. kvd_decode_attn / kvd_verify_attn / kvd_decode_attn_noalloc: in the last
     * split of every (row, KV head) unit the first stage of K/V tiles expects more
     * bytes than its copies bring (a split whose range starts past the row's length
     * has no stage), so that stage never completes and the split's tile waits run out
     * after about one second; it drains and gives up without sending its partial
     * (in a cluster merge the first CTA's bounded wait for it then runs out); the call
     * must report KVD_ERR_TIMEOUT, leave those units' outputs unwritten, and leave the
     * stream usable (a workspace merge also leaves that unit's arrival counter
     * non-zero: re-zero the workspace). The timeout paths are exercised without any
     * fault. */
    KVD_FLAG_TEST_STALL = 1u << 8
};

#define KVD_WS_COUNTER_BYTES 65536
#define KVD_HEAD_DIM 64
#define KVD_MAX_QLEN 16
#define KVD_MAX_BEAM 8
#define KVD_MAX_VOCAB 524288
#define KVD_MAX_LAYERS_PER_CALL 64

/* The new tokens' K/V for a fused append inside an attention call. */
typedef struct kvd_new_tokens {
    const void *k_new;  /* device [kv_batch, n_kv_heads, qlen, 64], contiguous */
    const void *v_new;  /* same shape                                         */
    int32_t *lens_out;  /* device [kv_batch] or NULL: receives lens + qlen     */
    float rope_base;    /* 0: no rotation. > 0: rotary encoding (kvd_rope's    */
                        /* definition, this base) of the call's queries and    */
                        /* new keys at the new tokens' absolute positions      */
                        /* lens[b] + j, inside the attention launch; the       */
                        /* cache receives the rotated keys, q is not written   */
} kvd_new_tokens;

/* One layer's cache: K and V share the shape and strides. */
typedef struct kvd_cache {
    void *k;
    void *v;
    int64_t stride_b;   /* elements between consecutive batch rows            */
    int64_t stride_h;   /* elements between consecutive KV heads               */
    int64_t stride_t;   /* elements between consecutive positions (>= 64)      */
    int32_t batch;      /* rows of the cache (kv batch)                        */
    int32_t n_kv_heads;
    int32_t head_dim;   /* must be 64                                          */
    int32_t capacity;   /* positions allocated per (row, head)                 */
} kvd_cache;

/*
 * kvd_kv_append -- write the new tokens' K/V into the cache.
 *
 * [N] "KV キャッシュが推論を最適化する方法", steps 2-3 (only the newest token's K/V are
 * computed and added to the cache); [W] "Inference 抽象と KV キャッシュ" (the
 * self-attention projections of the new token are concatenated along the sequence
 * axis). Here the cache is preallocated, so the append is an O(q) write, not a
 * reallocation.
 *
 *   K[b, h, lens_in[b] + j, :] = k_new[b, h, j, :]  (same for V), j < q, b < batch
 *   lens_out[b] = lens_in[b] + q                     (if lens_out != NULL)
 *
 * k_new, v_new : device [batch, n_kv_heads, q, 64], contiguous
 * lens_in      : device int32 [batch], read only
 * lens_out     : device int32 [batch] or NULL; must not alias lens_in. Every layer of
 *                a step may pass the same lens_out: it writes the same values.
 * Device error : lens_in[b] < 0 or lens_in[b] + q > capacity -> KVD_ERR_LEN_OVERFLOW,
 *                row b is not written and lens_out[b] = lens_in[b].
 */
kvd_status kvd_kv_append(kvd_dtype dtype, const kvd_cache *cache, int32_t batch, int32_t q,
                         const void *k_new, const void *v_new, const int32_t *lens_in,
                         int32_t *lens_out, uint32_t flags, int32_t *dev_err,
                         kvd_stream_t stream);

/*
 * kvd_kv_append_rope -- the append, with the keys rotary-encoded as they are written.
 *
 * [N] "nanoVLM における KV キャッシュ実装": the language model passes start_pos so that
 * the rotary encoding of the new tokens matches their absolute positions. As
 * kvd_kv_append, except that key row j of batch row b is written rotated at position
 * lens_in[b] + j (kvd_rope's definition, base rope_base > 0; the same bits as kvd_rope
 * followed by kvd_kv_append). V rows are written as they are.
 */
kvd_status kvd_kv_append_rope(kvd_dtype dtype, const kvd_cache *cache, int32_t batch, int32_t q,
                              const void *k_new, const void *v_new, const int32_t *lens_in,
                              int32_t *lens_out, float rope_base, uint32_t flags,
                              int32_t *dev_err, kvd_stream_t stream);

/*
 * kvd_decode_attn -- one query token per row attends over the cache.
 *
 * [N] "KV キャッシュが推論を最適化する方法", step 4 (the current token's query meets the
 * cached K/V); [W] "Inference 抽象と KV キャッシュ" (attention sees the full
 * concatenated sequence, the token just appended included; cross-attention K/V are
 * computed from the encoder output once and reused); [N] "nanoVLM における技術的実装"
 * item 1 (grouped attention: n_q_heads / n_kv_heads query heads share a KV head).
 *
 *   out[r, hq, 0, :] = sum_{t < len} softmax_t(scale * q[r,hq] . K[b,h,t]) V[b,h,t]
 *   b = r / rows_per_kv, h = hq / (n_q_heads / kv->n_kv_heads),
 *   len = lens ? lens[b] : fixed_len
 *
 * q, out       : device [batch, n_q_heads, 1, 64], contiguous
 * kv           : cache with kv->batch >= batch / rows_per_kv
 * lens         : device int32 [batch / rows_per_kv] (e.g. lens_out of kv_append) or
 *                NULL to use fixed_len (cross-attention: 1500 encoder frames)
 * append       : NULL, or the new token's K/V ([kv_batch, n_kv_heads, 1, 64]) to append
 *                in the same launch: they are written at position lens[b] and attention
 *                runs over lens[b] + 1 positions (lens = the length BEFORE the append,
 *                required); lens_out, if given, receives lens + 1. This equals
 *                kvd_kv_append followed by kvd_decode_attn, without the extra launch.
 * rows_per_kv  : rows r .. r+rows_per_kv-1 share cache row r / rows_per_kv (beam rows
 *                of one audio window share its cross K/V); batch % rows_per_kv == 0
 * len == 0 gives a zero output. Long caches are split across thread blocks and the
 * partial results merged with their log-sum-exp weights (flash-decoding). One query
 * vector per KV head runs on CUDA cores; two or more (grouped-query heads, beam rows
 * sharing a window) form a small GEMM and run on the tensor cores.
 * Device error : len < 0 or len (+1 when appending) > capacity -> KVD_ERR_LEN_OVERFLOW,
 *                output and cache left as is.
 */
kvd_status kvd_decode_attn(kvd_dtype dtype, int32_t batch, int32_t n_q_heads, const void *q,
                           const kvd_cache *kv, const int32_t *lens, int32_t fixed_len,
                           const kvd_new_tokens *append, int32_t rows_per_kv, float scale,
                           void *out, void *workspace, size_t workspace_bytes, uint32_t flags,
                           int32_t *dev_err, kvd_stream_t stream);

/*
 * kvd_decode_attn_noalloc -- kvd_decode_attn for callers that cannot allocate.
 *
 * The pages have no counterpart: this is a library convenience. Some callers cannot
 * hand the library a workspace: a plugin or custom-op interface that passes an op
 * only its input and output pointers, a server that reserves its whole memory budget
 * at start-up and may not allocate in the decode loop, or a host that must not take
 * the allocator's locks or device-wide synchronisation at that point. For them this
 * entry point takes the same arguments as kvd_decode_attn minus the workspace, and
 * does the same computation with the same kernel, merging split partial results in a
 * fixed scratch buffer of KVD_NOALLOC_SCRATCH_BYTES compiled into the library (every
 * GPU that loads the library holds it until the process exits). It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 *  - Set-up: the first call on each device looks up the scratch address there
 *    (cudaGetSymbolAddress, with that device current), after the host checks below
 *    have passed. Make that first call before any stream capture. The address is kept
 *    for the life of the process: do not call this entry point again after a
 *    cudaDeviceReset (or anything else that destroys the device's primary context)
 *    in the same process.
 *  - Host checks come first, exactly as for kvd_decode_attn: an invalid argument, or a
 *    shape whose split merge needs more than the buffer holds (KVD_ERR_WORKSPACE; use
 *    kvd_decode_attn with a workspace), returns with nothing enqueued on `stream`.
 *  - Only a plan that merges splits through the buffer (a handful of (row, KV head)
 *    units over a long range) uses its arrival counters. For such a plan the call first
 *    clears those counters on `stream` (a memset of the library's own buffer, a few
 *    bytes per unit), then launches the kernel. That memset sits between the previous
 *    kernel on the stream and this one, so for those shapes KVD_FLAG_PDL and
 *    KVD_FLAG_EARLY_KV give no overlap with the previous kernel. Other shapes launch
 *    the kernel alone, and the flags behave as in kvd_decode_attn.
 *  - All calls on a device share the one buffer: calls that can overlap on the GPU
 *    (different streams, or graphs replayed concurrently) race and give wrong results.
 *    Serialise them on one stream.
 */
#define KVD_NOALLOC_SCRATCH_BYTES (512u * 1024u)
kvd_status kvd_decode_attn_noalloc(kvd_dtype dtype, int32_t batch, int32_t n_q_heads,
                                   const void *q, const kvd_cache *kv, const int32_t *lens,
                                   int32_t fixed_len, const kvd_new_tokens *append,
                                   int32_t rows_per_kv, float scale, void *out, uint32_t flags,
                                   int32_t *dev_err, kvd_stream_t stream);

/*
 * kvd_noalloc_test_fill_counters -- test support for kvd_decode_attn_noalloc.
 *
 * No counterpart on the pages. Fills the arrival counters of the built-in scratch
 * buffer (its first KVD_WS_COUNTER_BYTES) with `byte_value` on `stream`, as a call that
 * stopped early after a timed-out wait could leave them, so that a test can check that
 * the next kvd_decode_attn_noalloc call still starts its merge from zero. Not for use
 * while a kvd_decode_attn_noalloc call may be running on another stream.
 */
kvd_status kvd_noalloc_test_fill_counters(uint8_t byte_value, kvd_stream_t stream);

/*
 * kvd_verify_attn -- a block of qlen query tokens per row in one pass.
 *
 * [S] "추측 디코딩이란?" and [A]: the main model checks all candidate tokens in a single
 * forward pass. The block's K/V are already appended (kvd_kv_append with q = qlen),
 * so query i sits at absolute position len - qlen + i:
 *
 *   causal:     out[r,hq,i,:] = sum_{t <= len - qlen + i} softmax(...) V_t
 *   non-causal: out[r,hq,i,:] = sum_{t < len} softmax(...) V_t   (cross-attention)
 *
 * q, out : device [batch, n_q_heads, qlen, 64], contiguous; 1 <= qlen <= 16.
 * append  : NULL, or the block's K/V ([kv_batch, n_kv_heads, qlen, 64]) appended in the
 *           same launch at positions lens[b] .. lens[b]+qlen-1 (lens = the length
 *           before the append); attention then runs as if kvd_kv_append had run first.
 * The Q.K^T and P.V products run on the tensor cores. Other arguments and errors as
 * kvd_decode_attn; a causal row with len < qlen sees only its visible positions and a
 * query with no visible position gets a zero output.
 */
kvd_status kvd_verify_attn(kvd_dtype dtype, int32_t batch, int32_t n_q_heads, int32_t qlen,
                           const void *q, const kvd_cache *kv, const int32_t *lens,
                           int32_t fixed_len, const kvd_new_tokens *append,
                           int32_t rows_per_kv, int32_t causal, float scale, void *out,
                           void *workspace, size_t workspace_bytes, uint32_t flags,
                           int32_t *dev_err, kvd_stream_t stream);

/*
 * kvd_prefill_attn -- prefill: the first forward pass over a prompt.
 *
 * [N] "KV キャッシュが推論を最適化する方法" (prefill fills the cache with the whole
 * prompt, decoding then adds one token per step); [W] "Inference 抽象と KV キャッシュ"
 * (the first pass covers the initial tokens). Two launches on `stream`: the prompt's
 * K/V rows j < plens[b] are written at positions lens_in[b] + j and
 * lens_out[b] = lens_in[b] + plens[b]; then, per head,
 *
 *   out[b,hq,j,:] = sum_{t <= lens_in[b] + j} softmax_t(scale * q[b,hq,j] . K[b,h,t]) V[b,h,t]
 *
 * for j < plens[b] (h = hq / (n_q_heads / n_kv_heads)); rows j >= plens[b] of `out` are
 * written as zeros. lens_in > 0 continues a cached prefix (chunked prefill).
 *
 * q, out        : device [batch, n_q_heads, max_len, 64], contiguous, 16-byte aligned
 * k_new, v_new  : device [batch, n_kv_heads, max_len, 64], contiguous, 16-byte aligned
 * kv            : the layer's cache (any strides kvd_cache allows)
 * lens_in       : device int32 [batch] or NULL (every row starts empty)
 * plens         : device int32 [batch], prompt lengths in [0, max_len]
 * lens_out      : device int32 [batch] or NULL; must not alias lens_in
 * rope_base    : 0, or > 0 to rotary-encode the prompt (kvd_rope's definition): query
 *                row j and key row j at position lens_in[b] + j; the cache receives the
 *                rotated keys, q is not written (the same bits as kvd_rope first)
 * Q.K^T and P.V run on the tensor cores, fp32 accumulation, output rounded to nearest.
 * Device errors: lens_in + plens outside [0, capacity] or plens outside [0, max_len] ->
 * KVD_ERR_LEN_OVERFLOW; that row's cache is untouched, lens_out keeps lens_in and its
 * output rows are zeros. No workspace; the buffers are caller-owned.
 */
kvd_status kvd_prefill_attn(kvd_dtype dtype, int32_t batch, int32_t n_q_heads, int32_t max_len,
                            const void *q, const kvd_cache *kv, const void *k_new,
                            const void *v_new, const int32_t *lens_in, const int32_t *plens,
                            int32_t *lens_out, float scale, float rope_base, void *out,
                            uint32_t flags, int32_t *dev_err, kvd_stream_t stream);

/*
 * kvd_rope -- rotary position encoding at absolute positions (in place).
 *
 * [N] "nanoVLM における KV キャッシュ実装" (start_pos keeps the rotary encoding of new
 * tokens at their absolute positions). The pages give no formula; this is the usual
 * rotate-half form: for i < 32, theta_i = base^(-i/32) and a = pos * theta_i,
 *   y[i] = x[i] cos a - x[i+32] sin a,   y[i+32] = x[i+32] cos a + x[i] sin a,
 * with token j of row b at pos0[b] + j. Run it on a step's queries and new keys (before
 * kvd_kv_append, the fused append, or kvd_prefill_attn).
 *
 * q : device [batch, n_q_heads, n, 64] or NULL;  k : device [batch, n_k_heads, n, 64]
 *     or NULL; contiguous, 16-byte aligned, rotated in place (one launch for both).
 * pos0 : device int32 [batch] or NULL (0). base > 0 (10000 for the usual encoding).
 * fp32 arithmetic (sin/cos with full argument reduction), rounded to the storage type.
 * No device errors; dev_err is accepted for symmetry.
 */
kvd_status kvd_rope(kvd_dtype dtype, int32_t batch, int32_t n, void *q, int32_t n_q_heads,
                    void *k, int32_t n_k_heads, const int32_t *pos0, float base, uint32_t flags,
                    int32_t *dev_err, kvd_stream_t stream);

/*
 * kvd_greedy_accept -- greedy verification of k draft tokens.
 *
 * [W] "Inference 抽象と KV キャッシュ" (GreedyDecoder: argmax at temperature 0);
 * [S] "추측 디코딩이란?" and [A] (accept candidates up to the first mismatch, replace
 * the mismatch by the main model's token, drop the rest); [S] "배치 크기 고려사항"
 * (in a batch all rows must match to advance together: n_min).
 *
 *   a_i    = argmax_v logits[b, i, v], i = 0..k (lowest index on ties; a NaN ranks
 *            above every number and the first NaN wins; -inf is an ordinary value)
 *   n_b    = min { i < k : draft[b, i] != a_i }, or k if all match
 *   next_b = a_{n_b}           (the correction, or the bonus token when n_b == k)
 *   emitted tokens: draft[b, 0..n_b-1] followed by next_b; the caller rolls its
 *   caches back to L_before + n_b + 1 positions (a length change only).
 *
 * logits     : device fp32 [batch, k+1, vocab], contiguous; 1 <= k <= 16
 * draft      : device int32 [batch, k]
 * n_accepted, next_token : device int32 [batch]
 * n_min      : device int32 [1] or NULL -- min_b n_b
 * argmax     : device int32 [batch, k+1] or NULL -- every a_i
 * Device errors: a draft id outside [0, vocab) -> KVD_ERR_BAD_TOKEN (it never
 * matches); a NaN logit -> KVD_ERR_NAN (outputs still follow the rule above).
 */
kvd_status kvd_greedy_accept(const float *logits, int32_t batch, int32_t k, int32_t vocab,
                             const int32_t *draft, int32_t *n_accepted, int32_t *next_token,
                             int32_t *n_min, int32_t *argmax, void *workspace,
                             size_t workspace_bytes, uint32_t flags, int32_t *dev_err,
                             kvd_stream_t stream);

/*
 * kvd_sample_accept -- temperature sampling and stochastic speculative
 * acceptance.
 *
 * [W] "Inference 抽象と KV キャッシュ" (GreedyDecoder above temperature 0 samples from
 * Categorical(logits / T)); [S] "추측 디코딩이란?" (Leviathan et al.'s speculative
 * decoding, whose sampling form is the rejection rule below). With
 * p_i = softmax(target[b, i] / T), q_i = softmax(draft[b, i] / T), x_i = drafts[b, i]:
 *
 *   for i < k: accept x_i iff r[b, i] * q_i(x_i) < p_i(x_i); stop at the first rejection
 *   n_accepted[b] = n (the first rejected i, or k)
 *   next_token[b] = a draw with u[b] from max(0, p_n - q_n) normalised (p_n if that is
 *                   all 0) when n < k, else from p_k
 *   a draw from weights w with u in [0, 1): the smallest id whose running sum (id order)
 *   exceeds u * sum(w); the last id with w > 0 if rounding leaves none
 *
 * The emitted tokens are drafts[b, 0..n-1] followed by next_token[b]; their joint
 * distribution is the main model's. k = 0: plain temperature sampling of target row 0.
 *
 * target : device fp32 [batch, k+1, vocab]; draft: device fp32 [batch, k, vocab]
 * drafts : device int32 [batch, k]; r: device fp32 [batch, k]; u: device fp32 [batch]
 *          (the caller's uniforms in [0, 1); the library draws no random numbers)
 * temperature > 0; 0 <= k <= 7 (KVD_ERR_UNSUPPORTED above).
 * n_accepted, next_token : device int32 [batch]
 * workspace : kvd_workspace_size(KVD_OP_SAMPLE_ACCEPT, batch, .., qlen = k, .., vocab)
 *             bytes, 256-byte aligned (the rows' per-segment softmax sums)
 * fp32 arithmetic; a draw whose u * sum(w) lies within fp32 rounding of a boundary may
 * land on either neighbour. Two launches: the rows' softmax sums over the whole GPU,
 * then one thread-block cluster per batch row for the decision and the draw.
 * Device errors: a drafted id outside [0, vocab) -> KVD_ERR_BAD_TOKEN (rejected); a NaN
 * logit -> KVD_ERR_NAN (counted as -inf).
 */
kvd_status kvd_sample_accept(const float *target, const float *draft, const int32_t *drafts,
                             int32_t batch, int32_t k, int32_t vocab, float temperature,
                             const float *r, const float *u, int32_t *n_accepted,
                             int32_t *next_token, void *workspace, size_t workspace_bytes,
                             uint32_t flags, int32_t *dev_err, kvd_stream_t stream);

/*
 * kvd_beam_reorder_kv -- reorder the self-attention caches of all layers.
 *
 * [W] "Inference 抽象と KV キャッシュ" (BeamSearchDecoder.update, rearrange_kv_cache):
 * after beams are re-ranked the key/value tensors are put in the new beam order, so
 * that no beam continues another beam's cache.
 *
 *   for every layer l < n_layers, K and V, row r < rows, head h, position t < len_r:
 *     C'[l][r, h, t, :] = C[l][parent[r], h, t, :]
 *   len_r = lens ? lens[r] : fixed_len. Rows are grouped in windows of `beam`; a
 *   parent must lie in its row's window [w*beam, (w+1)*beam).
 *
 * In place and allocation-free: each thread block reads, for one window and one
 * tile of positions, every source row it needs before writing any row, so repeated
 * parents (a beam with several children) and cycles are handled without scratch.
 * Rows whose parent is themselves are not touched. Cross-attention K/V are not part
 * of the reorder (they are shared per window).
 *
 * layers   : host array of n_layers caches (n_layers <= 64), each with batch >= rows
 * parent   : device int32 [rows]; beam in 1..8; rows % beam == 0
 * lens     : device int32 [rows] or NULL to use fixed_len
 * Device errors: parent outside its window -> KVD_ERR_BAD_INDEX (row left as is);
 * len_r < 0 or > capacity -> KVD_ERR_LEN_OVERFLOW (row left as is).
 */
kvd_status kvd_beam_reorder_kv(kvd_dtype dtype, const kvd_cache *layers, int32_t n_layers,
                               int32_t rows, int32_t beam, const int32_t *parent,
                               const int32_t *lens, int32_t fixed_len, uint32_t flags,
                               int32_t *dev_err, kvd_stream_t stream);

/*
 * kvd_beam_select -- logit filters and one beam-search selection step.
 *
 * [W] "LogitFilter チェーン" (SuppressBlank: blank ids and EOT -> -inf at the first
 * sampling position only; SuppressTokens: listed ids -> -inf at every position) and
 * [W] "Inference 抽象と KV キャッシュ" (BeamSearchDecoder.update). For every window w
 * of `beam` rows r = w*beam + j:
 *   x_r      = logits[r] with the masks applied (a NaN counts as -inf)
 *   lp_r(t)  = x_r[t] - log sum_u exp(x_r[u])          (all -inf if x_r is all -inf)
 *   step 1   : the beam+1 ids of largest x_r (ties: lower id) -> row_token, row_logprob
 *   step 2   : continuation (j, t) scores cum[r] + lp_r(t) (a NaN cum counts as -inf)
 *   step 3   : from the highest score down (ties: lower j, then better rank in the row)
 *              EOT continuations are finished, the others kept until `beam` are kept
 *   outputs  : kept continuation s at w*beam + s -> parent (absolute row, the input of
 *              kvd_beam_reorder_kv), token, new_cum; n_finished[w]; finished f at
 *              w*beam + f -> fin_parent, fin_score (slots past n_finished: -1, -inf)
 * fp32 arithmetic; every id and parent is decided by exact comparisons of fp32 values.
 * Greedy decoding with the filters: beam = 1, parent = NULL, token = row_token[r][0].
 *
 * logits      : device fp32 [windows*beam, vocab], contiguous; beam+1 <= vocab <=
 *               KVD_MAX_VOCAB; windows <= 2^24
 * cum         : device fp32 [windows*beam] or NULL (zeros)
 * suppress    : device int32 [n_suppress] (duplicates allowed); blank: device int32
 *               [n_blank], read only when first_step != 0; eot in [0, vocab) (host int)
 * row_token, row_logprob : device [windows*beam, beam+1] or NULL
 * parent, token, new_cum, fin_parent, fin_score : device [windows*beam];
 * n_finished  : device int32 [windows] -- all NULL (no walk) or all non-NULL
 * beam in 1..8 (KVD_ERR_UNSUPPORTED otherwise). No workspace: one thread-block cluster
 * per window merges through distributed shared memory.
 * Device errors: a suppress/blank id outside [0, vocab) -> KVD_ERR_BAD_TOKEN (skipped);
 * a NaN logit or cum -> KVD_ERR_NAN (outputs still follow the rules above); a bounded
 * wait for a copy that gave up -> KVD_ERR_TIMEOUT (outputs undefined).
 */
kvd_status kvd_beam_select(const float *logits, int32_t windows, int32_t beam, int32_t vocab,
                           const float *cum, const int32_t *suppress, int32_t n_suppress,
                           const int32_t *blank, int32_t n_blank, int32_t eot,
                           int32_t first_step, int32_t *row_token, float *row_logprob,
                           int32_t *parent, int32_t *token, float *new_cum,
                           int32_t *n_finished, int32_t *fin_parent, float *fin_score,
                           uint32_t flags, int32_t *dev_err, kvd_stream_t stream);

/*
 * kvd_workspace_size -- bytes of workspace a call needs (always includes the
 * KVD_WS_COUNTER_BYTES counter region). Arguments not used by `op` are ignored:
 *   KVD_OP_DECODE_ATTN : batch, n_q_heads, n_kv_heads, rows_per_kv, max_len
 *   KVD_OP_VERIFY_ATTN : the same plus qlen
 *   KVD_OP_GREEDY_ACCEPT: batch, qlen = k, vocab
 *   KVD_OP_SAMPLE_ACCEPT: batch, qlen = k, vocab
 * max_len is an upper bound of the attended length (the capacity, or fixed_len).
 * Returns 0 for invalid arguments.
 */
size_t kvd_workspace_size(kvd_op op, int32_t batch, int32_t n_q_heads, int32_t n_kv_heads,
                          int32_t rows_per_kv, int32_t qlen, int32_t max_len, int32_t vocab);

/* Human-readable name of a status code (static storage). */
const char *kvd_status_string(kvd_status status);

/* Library version as 10000*major + 100*minor + patch. */
int32_t kvd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVDECODE_H */
