/*
 * sink_attn.h -- C ABI of libsinkattn, grouped-query attention with per-head
 * attention sinks (the gpt-oss attention layer) on NVIDIA GB300 (sm_103a).
 *
 * The operation.  For a query row at position p of sequence b and query head
 * h, with G = num_qo_heads / num_kv_heads and kv head g = floor(h / G):
 *
 *   J     = { j : 0 <= j <= p, j < L_b, and (window == 0 or j > p - window) }
 *   s_j   = sm_scale * <q[h], k[b, g, j]>
 *   sigma = sinks[h]  (-inf when sinks == NULL)
 *   out   = sum_{j in J} exp(s_j - M) v[b, g, j] / (exp(sigma - M) + sum_{j in J} exp(s_j - M))
 *   lse   = M + log(exp(sigma - M) + sum_{j in J} exp(s_j - M)),   M = max(sigma, max_J s_j)
 *
 * i.e. a softmax over the scores plus one extra per-head logit, the sink,
 * which takes part in the denominator and has no value vector.  A row with no
 * visible key gets out = 0 and lse = sigma.  lse is a natural logarithm and
 * includes the sink.
 *
 * Sources: "GPT-OSS on day 0" (Perplexity), section "Attention: GQA with
 * attention sinks" (one pretrained sink parameter per attention head that
 * joins the softmax) and section "GPT-OSS kernels / Sink Attention" (the sink
 * is an extra bias term beside the Q.K products; the online softmax seeds its
 * running max with the sink, and a sequence split counts the sink in one chunk
 * only).  NVIDIA gpt-oss launch article, introduction: layers alternate full
 * causal context and a 128-token sliding window (window = 128 here means the
 * keys j in (p - 128, p]).  vLLM "GPT-OSS optimisations on NVIDIA Blackwell",
 * section "FlashInfer integration": an FP8 KV cache.
 *
 * Conventions shared by every call.
 *  - Memory: every pointer argument is caller-owned.  Device pointers must stay
 *    valid until the work queued on `stream` has finished.  The library
 *    allocates no device memory per call; scratch for split-KV lives in a
 *    caller-given workspace.
 *  - Asynchrony: every call only queues kernels on `stream` and returns; none
 *    synchronises the host.  Results are ready when the stream's work is done.
 *  - Launch chaining: every kernel of the library is launched with
 *    programmatic stream serialization and waits for the grid before it
 *    (griddepcontrol.wait) before touching memory, so its inputs may come from
 *    any earlier work on the stream.  It also lets the next grid on the stream
 *    be scheduled before it finishes (griddepcontrol.launch_dependents): a
 *    caller's kernel launched after it WITH the programmatic-serialization
 *    attribute must wait for its grid dependency (griddepcontrol.wait /
 *    cudaGridDependencySynchronize) before reading this call's results.
 *    Kernels launched without that attribute, copies and events see plain
 *    stream order.
 *  - Errors: argument errors are detected on the host before any launch and
 *    return SA_ERR_INVALID_ARG (malformed) or SA_ERR_UNSUPPORTED (well formed
 *    but outside what the kernels handle); nothing is launched then.  A failed
 *    launch returns SA_ERR_CUDA.  sa_last_error() gives a one-line message for
 *    the calling thread's most recent failure.  Conditions that only the
 *    device can see (a sequence longer than max_kv_len, a page index outside
 *    the pool, a pipeline wait that ran out its time limit) are recorded in a
 *    device status word that sa_device_status() reads; the kernels never trap.
 *  - Layouts: all tensors are dense with the innermost dimension contiguous
 *    unless a stride argument says otherwise.  head_dim must be 64.
 *  - Threads: the calls are re-entrant; concurrent calls on different streams
 *    are independent.
 */
#ifndef SINK_ATTN_H
#define SINK_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SA_VERSION 10000 /* 1.0.0 */

typedef enum {
    SA_OK = 0,
    SA_ERR_INVALID_ARG = 1, /* malformed argument; nothing launched */
    SA_ERR_UNSUPPORTED = 2, /* valid but not handled (head_dim != 64, ...); nothing launched */
    SA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than sa_decode_workspace_size() */
    SA_ERR_CUDA = 4,        /* a CUDA call or launch failed; see sa_last_error() */
    SA_ERR_TIMEOUT = 5      /* (sa_device_status only) a device wait ran out its limit */
} sa_status_t;

typedef enum {
    SA_KV_BF16 = 0,     /* bfloat16 K and V */
    SA_KV_FP8_E4M3 = 1  /* OCP FP8 E4M3 codes; real value = code * k_scale (resp. v_scale) */
} sa_kv_dtype_t;

/*
 * A paged KV cache.  Token t of sequence b, kv head g, lives in page
 *   page = page_table[b * page_table_stride + t / page_size]   (page_table != NULL)
 *   page = b                                                   (page_table == NULL)
 * at element offset  page * stride_page + g * stride_head + (t % page_size) * stride_token
 * of `k` (resp. `v`); the head_dim elements of one token are contiguous.
 * HND pages ([num_pages, num_kv_heads, page_size, head_dim]) and NHD pages
 * ([num_pages, page_size, num_kv_heads, head_dim]) are both expressible.
 * Requirements: k and v 16-byte aligned; every stride times the element size
 * a multiple of 16 bytes; page_size a multiple of 16; head_dim == 64.
 * The page table is int32 in device memory, one row of page_table_stride
 * entries per sequence, and must hold ceil(max_kv_len / page_size) entries per
 * row.  A page index outside [0, num_pages) is not read: the kernels load
 * zeros for it and set SA_DEVICE_BAD_PAGE in the device status word.
 */
typedef struct {
    const void *k;
    const void *v;
    int32_t dtype;            /* sa_kv_dtype_t */
    int32_t num_pages;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t page_size;
    int32_t page_table_stride;
    int64_t stride_page;      /* elements */
    int64_t stride_head;      /* elements */
    int64_t stride_token;     /* elements */
    const int32_t *page_table;
    float k_scale;            /* FP8 only: real = code * k_scale; ignored for bf16 */
    float v_scale;            /* FP8 only */
} sa_kv_desc_t;

/* Bits of the device status word (sa_device_status). */
#define SA_DEVICE_SEQLEN_RANGE 0x1u /* a seqlen was < 0 or > max_kv_len: clamped */
#define SA_DEVICE_BAD_PAGE 0x2u     /* a page index outside [0, num_pages): read as zeros */
#define SA_DEVICE_TIMEOUT 0x4u      /* a pipeline wait ran out its limit: output undefined */
#define SA_DEVICE_BAD_QLEN 0x8u     /* prefill: a query length was < 0 or > L_kv or > max_q_len;
                                       multi-token decode: 0 < seqlens[b] < q_len */
#define SA_DEVICE_BAD_TOKEN 0x10u   /* rope_append: a token's sequence id or position was out of
                                       range (that token's rows were skipped) */

/*
 * sa_decode -- one query token per sequence against its paged KV cache.
 * Source: "GPT-OSS on day 0", sections "Sink Attention" (the online softmax
 * seeded with the sink; parallel over heads and KV length) and the NVIDIA
 * launch article's introduction (window).
 *
 *   q          device bf16 [batch, num_qo_heads, 64]; row b is sequence b's query,
 *              at position seqlens[b] - 1 (its own key is already in the cache)
 *   kv         KV cache descriptor (host struct, read during the call only)
 *   seqlens    device int32 [batch]: keys held by each sequence (0 allowed)
 *   batch      >= 0 (0: no-op)
 *   num_qo_heads  multiple of kv->num_kv_heads, at most 8 query heads per kv head
 *   max_kv_len host upper bound on seqlens[]; sizes the work split.  A larger
 *              seqlen is clamped on the device and flagged.
 *   sinks      device fp32 [num_qo_heads] (natural-log units, not scaled by
 *              sm_scale), or NULL for no sink
 *   window     0 = full causal; w > 0 = the w most recent keys
 *   sm_scale   softmax scale applied to q.k (finite)
 *   out        device bf16 [batch, num_qo_heads, 64] (round to nearest even)
 *   lse        device fp32 [batch, num_qo_heads] or NULL
 *   workspace  device scratch of at least sa_decode_workspace_size(...) bytes,
 *              16-byte aligned; may be NULL when that size is 0
 *   num_splits 0 = choose automatically (sa_decode_num_splits); 1 = no split;
 *              S > 1 = cut every sequence's visible keys into S chunks whose
 *              partial states are merged (sink once) by a second kernel
 *   stream     CUDA stream (0 = legacy default stream)
 * Returns SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_WORKSPACE or SA_ERR_CUDA.
 */
sa_status_t sa_decode(const void *q, const sa_kv_desc_t *kv, const int32_t *seqlens,
                      int32_t batch, int32_t num_qo_heads, int32_t max_kv_len,
                      const float *sinks, int32_t window, float sm_scale,
                      void *out, float *lse, void *workspace, size_t workspace_bytes,
                      int32_t num_splits, cudaStream_t stream);

/*
 * Number of KV chunks sa_decode uses for num_splits = 0 on the current device.
 * Depends only on the arguments and the device's SM count (no device sync).
 */
int32_t sa_decode_num_splits(int32_t batch, int32_t num_kv_heads, int32_t max_kv_len,
                             int32_t window);

/*
 * Workspace bytes sa_decode needs.  num_splits = 0 gives the size for the
 * automatic choice (num_kv_heads is needed for it); 1 gives 0.
 * Layout when S > 1: fp32 o_part [S, batch, num_qo_heads, head_dim] followed
 * (at a 256-byte aligned offset) by fp32 lse_part [S, batch, num_qo_heads].
 */
size_t sa_decode_workspace_size(int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t max_kv_len, int32_t window,
                                int32_t num_splits);

/*
 * sa_decode_multi -- q_len (1..SA_MAX_DECODE_TOKENS) new query tokens per
 * sequence against its paged KV cache, for example the draft tokens a
 * speculative or multi-token-prediction decoder asks the model to verify
 * ("GPT-OSS on day 0": the engine's speculative and MTP decoders).  Each block
 * reads a kv head's keys once for every token and query head of the group.
 *   q          device bf16 [batch * q_len, num_qo_heads, 64]; row b * q_len + k
 *              is token k of sequence b, at position seqlens[b] - q_len + k
 *              (all q_len tokens' keys are already in the cache), so token k
 *              sees keys <= its position (and, with a window, the w most recent)
 *   out, lse   device bf16 [batch * q_len, num_qo_heads, 64] / fp32
 *              [batch * q_len, num_qo_heads] or NULL, rows as q
 *   workspace  at least sa_decode_multi_workspace_size(...) bytes when split
 *   num_splits 0 = sa_decode_multi_num_splits(...); otherwise as sa_decode
 *   other arguments as sa_decode; q_len = 1 is sa_decode.
 * q_len >= 2 on a bf16 cache runs on the tensor cores (tcgen05): the group's
 * q_len x G query rows against 64-key tiles, two key streams per block.
 * A sequence with 0 < seqlens[b] < q_len sets SA_DEVICE_BAD_QLEN; its tokens
 * at negative positions see no key (out = 0, lse = sink).  seqlens[b] = 0
 * marks an empty slot: every token of it gives out = 0, lse = sink, unflagged.
 * Returns SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED (q_len outside
 * [1, SA_MAX_DECODE_TOKENS]), SA_ERR_WORKSPACE or SA_ERR_CUDA.
 */
#define SA_MAX_DECODE_TOKENS 8
sa_status_t sa_decode_multi(const void *q, int32_t q_len, const sa_kv_desc_t *kv,
                            const int32_t *seqlens, int32_t batch, int32_t num_qo_heads,
                            int32_t max_kv_len, const float *sinks, int32_t window,
                            float sm_scale, void *out, float *lse, void *workspace,
                            size_t workspace_bytes, int32_t num_splits, cudaStream_t stream);

/*
 * Number of KV chunks sa_decode_multi uses for num_splits = 0 on the current
 * device, for a cache of type kv_dtype (an sa_kv_dtype_t).  q_len >= 2 on a
 * bf16 cache runs the tensor-core multi-token kernel (two blocks per SM, so
 * fewer chunks fill the GPU); otherwise this is sa_decode_num_splits.  Depends
 * only on the arguments and the device (no device sync).
 */
int32_t sa_decode_multi_num_splits(int32_t batch, int32_t q_len, int32_t num_kv_heads,
                                   int32_t max_kv_len, int32_t window, int32_t kv_dtype);

/*
 * Workspace bytes sa_decode_multi needs.  num_splits = 0 gives a size that
 * covers the automatic choice for either cache type (the larger of the two
 * sa_decode_multi_num_splits counts).  Layout when S > 1: fp32 o_part
 * [S, batch * q_len, num_qo_heads, head_dim] followed (at a 256-byte aligned
 * offset) by fp32 lse_part [S, batch * q_len, num_qo_heads].
 */
size_t sa_decode_multi_workspace_size(int32_t batch, int32_t q_len, int32_t num_qo_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t max_kv_len,
                                      int32_t window, int32_t num_splits);

/*
 * sa_decode_partial -- the first half of a split decode, exposed for callers
 * that merge partial states themselves (for example states gathered from
 * several devices that each hold part of a sequence's keys).
 * Chunking: for sequence b the visible keys are [lo, L_b) with
 * lo = max(0, L_b - window) (window > 0) or 0; with a = lo rounded down to a
 * multiple of 16 and T = ceil(tiles / num_splits) 16-key tiles per chunk
 * (tiles = ceil(max_kv_len / 16), or ceil((min(window, max_kv_len) + 15) / 16)
 * when window > 0), chunk s covers keys [a + 16*T*s, a + 16*T*(s+1)) within
 * [lo, L_b).  Chunk s writes the SINK-FREE state
 *   o_part[s, b, h, :] = sum_j exp(s_j - m) v_j / sum_j exp(s_j - m)   (fp32)
 *   lse_part[s, b, h]  = m + log(sum_j exp(s_j - m))                   (fp32)
 * with o = 0 and lse = -inf for an empty chunk.  sa_merge_states(... sinks ...)
 * of these partials equals sa_decode.  Arguments as sa_decode; o_part is
 * device fp32 [num_splits, batch, num_qo_heads, 64], lse_part device fp32
 * [num_splits, batch, num_qo_heads].  num_splits >= 1.
 */
sa_status_t sa_decode_partial(const void *q, const sa_kv_desc_t *kv, const int32_t *seqlens,
                              int32_t batch, int32_t num_qo_heads, int32_t max_kv_len,
                              int32_t window, float sm_scale, int32_t num_splits,
                              float *o_part, float *lse_part, cudaStream_t stream);

/*
 * sa_merge_states -- merge S partial attention states with the sink counted once.
 * Source: "GPT-OSS on day 0", section "Sink Attention": when attention is
 * split into chunks along the sequence, the sink may enter only once.
 *   M   = max(sigma_h, max_s lse_part[s, n, h])
 *   Z   = exp(sigma_h - M) + sum_s exp(lse_part[s, n, h] - M)
 *   out = sum_s exp(lse_part[s, n, h] - M) o_part[s, n, h, :] / Z   (bf16, RNE)
 *   lse_out = M + log(Z)
 * A partial with lse = -inf carries no weight; if every partial is -inf and
 * there is no sink, out = 0 and lse_out = -inf.
 *   o_part   device fp32 [num_splits, n, num_heads, head_dim]
 *   lse_part device fp32 [num_splits, n, num_heads]
 *   sinks    device fp32 [num_heads] or NULL
 *   out      device bf16 [n, num_heads, head_dim];  lse_out device fp32 [n, num_heads] or NULL
 * head_dim must be a multiple of 4 and at most 256; num_splits >= 1.
 */
sa_status_t sa_merge_states(const float *o_part, const float *lse_part, int32_t num_splits,
                            int32_t n, int32_t num_heads, int32_t head_dim,
                            const float *sinks, void *out, float *lse_out, cudaStream_t stream);

/*
 * sa_prefill -- causal (or sliding-window) attention of a ragged batch of
 * query blocks against the KV cache, on tcgen05 tensor cores.
 * Source: "GPT-OSS on day 0", section "Sink Attention" (prefill and decode
 * templates both carry the sink); NVIDIA launch article, introduction.
 *   q            device bf16 [total_q, num_qo_heads, 64], rows of sequence b at
 *                cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
 *   cu_seqlens_q device int32 [batch + 1], cu[0] = 0, non-decreasing
 *   total_q      rows of q and out (= cu_seqlens_q[batch]); the kernels read and
 *                write no row at or past it
 *   kv           KV cache descriptor, bf16 or FP8-E4M3; holds each sequence's
 *                keys, the queries' own keys included.  With an FP8 cache the
 *                products run in f16: q is rounded to f16 (|q| < 65504 assumed)
 *                and the codes are widened exactly
 *   seqlens_kv   device int32 [batch]: keys of sequence b (L_kv,b >= L_q,b)
 *   max_q_len, max_kv_len  host upper bounds on the query / key lengths
 *   sinks, window as sa_decode; sm_scale > 0 (SA_ERR_UNSUPPORTED otherwise)
 *   out          device bf16 [total_q, num_qo_heads, 64]
 *   lse          device fp32 [total_q, num_qo_heads] or NULL
 * Query i of sequence b sits at position L_kv,b - L_q,b + i (bottom-right aligned).
 * Returns SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED or SA_ERR_CUDA.
 */
sa_status_t sa_prefill(const void *q, const int32_t *cu_seqlens_q, int32_t total_q, const sa_kv_desc_t *kv,
                       const int32_t *seqlens_kv, int32_t batch, int32_t num_qo_heads,
                       int32_t max_q_len, int32_t max_kv_len, const float *sinks,
                       int32_t window, float sm_scale, void *out, float *lse,
                       cudaStream_t stream);

/*
 * sa_prefill_q8 -- sa_prefill with the query given as E4M3 codes on an
 * FP8-E4M3 cache (vLLM "GPT-OSS optimisations on NVIDIA Blackwell": part of
 * the attention runs in FP8).  S = Q K^T runs on the FP8 tensor cores
 * (kind::f8f6f4) straight from the cache's codes; P V as in sa_prefill.
 *   q        device uint8 [total_q, num_qo_heads, 64]: E4M3 codes, value =
 *            code * q_scale (sa_rope_append can write them)
 *   q_scale  finite, nonzero
 * Other arguments, layouts and results as sa_prefill.  SA_ERR_UNSUPPORTED
 * for a bf16 cache.
 */
sa_status_t sa_prefill_q8(const void *q, float q_scale, const int32_t *cu_seqlens_q, int32_t total_q,
                          const sa_kv_desc_t *kv, const int32_t *seqlens_kv, int32_t batch,
                          int32_t num_qo_heads, int32_t max_q_len, int32_t max_kv_len,
                          const float *sinks, int32_t window, float sm_scale, void *out, float *lse,
                          cudaStream_t stream);

/*
 * sa_rope_yarn_table -- fill a HOST buffer with the rotary table that
 * sa_rope_append reads: for each position p in [0, max_position), 64 floats,
 * cos(p * f_i) * mscale for i = 0..31 then sin(p * f_i) * mscale.
 * Frequencies follow YaRN ("GPT-OSS on day 0": YaRN position encoding as in
 * DeepSeek-V3), evaluated in double precision:
 *   f_i = theta^(-i/32) blended with f_i / factor by a ramp over the
 *   dimension index between floor(c(beta_fast)) and ceil(c(beta_slow)), where
 *   c(n) = 64 ln(original_max_position / (2 pi n)) / (2 ln theta) is the
 *   dimension that turns n times over the original context; dimensions below
 *   the ramp keep f_i, those above it use f_i / factor.
 *   mscale = 0.1 ln(factor) + 1 (1 when factor <= 1): q and k are both scaled,
 *   so q.k grows by mscale^2.
 * factor <= 1 gives plain rotary embeddings.  head_dim must be 64.
 * Returns SA_OK or SA_ERR_INVALID_ARG (NULL table, max_position < 1, theta <= 1,
 * original_max_position < 1, beta_fast <= 0, beta_slow <= 0, non-finite values)
 * or SA_ERR_UNSUPPORTED (head_dim != 64).  Copy the buffer to the device.
 */
sa_status_t sa_rope_yarn_table(float *table, int32_t max_position, int32_t head_dim, double theta,
                               double factor, int32_t original_max_position, double beta_fast,
                               double beta_slow);

/*
 * sa_rope_append -- the step in front of attention for T new tokens (vLLM
 * "GPT-OSS optimisations on NVIDIA Blackwell": RoPE, query and KV-cache
 * write as one operator).  One pass over the inputs:
 *   q_out[t, h] = rotate(q[t, h], positions[t])
 *   cache K at (seq_ids[t], positions[t], g) = rotate(k[t, g], positions[t])
 *   cache V at (seq_ids[t], positions[t], g) = v[t, g]
 * where rotate mixes dims i and i + 32 with the table row of the position:
 * (x_i c_i - x_{i+32} s_i, x_{i+32} c_i + x_i s_i).  The cache slot of
 * sequence b at position p is page kv->page_table[b, p / page_size] (page b
 * without a table), token slot p % page_size, in the descriptor's strides.
 * An FP8 cache stores e4m3(value / scale) (k_scale, v_scale; round to nearest
 * even, saturated to +-448); a bf16 cache the value rounded to nearest even.
 *   q            device bf16 [num_tokens, num_qo_heads, 64]
 *   k, v         device bf16 [num_tokens, kv->num_kv_heads, 64]
 *   seq_ids      device int32 [num_tokens], each in [0, batch)
 *   positions    device int32 [num_tokens], each in [0, max_position)
 *   table        device fp32 [max_position, 64] from sa_rope_yarn_table
 *   kv           the cache to write (kv->k and kv->v are written)
 *   batch        rows of kv->page_table (sequences), or pages when it is NULL
 *   q_out        device [num_tokens, num_qo_heads, 64]: bf16 (q_out_scale = 0;
 *                may alias q) or, for q_out_scale > 0, E4M3 codes of
 *                rotate(q) / q_out_scale (round to nearest even, saturated),
 *                the query input of sa_prefill_q8
 * A token whose sequence id or position is out of range, or whose table entry
 * lies past the table row, is skipped and sets SA_DEVICE_BAD_TOKEN; one whose
 * page is outside [0, num_pages) is skipped and sets SA_DEVICE_BAD_PAGE.
 * Returns SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED or SA_ERR_CUDA.
 */
sa_status_t sa_rope_append(const void *q, const void *k, const void *v, int32_t num_tokens,
                           int32_t num_qo_heads, const int32_t *seq_ids, const int32_t *positions,
                           const float *table, int32_t max_position, const sa_kv_desc_t *kv,
                           int32_t batch, void *q_out, float q_out_scale, cudaStream_t stream);

/*
 * sa_decode_static_workspace -- sa_decode for callers that cannot allocate
 * device memory.  The pages have no counterpart; this is an interface
 * convenience of the library.
 *
 * A split decode needs scratch for its per-chunk partial states, which
 * sa_decode takes from the caller.  Some callers cannot provide it: a plugin
 * inside a host program that owns all device memory and hands it only its
 * input and output tensors, or a caller on a latency-critical path that must
 * not call cudaMalloc (it may synchronise the device).  This entry point keeps
 * the scratch in a fixed array of SA_STATIC_WORKSPACE_BYTES in device memory
 * that the library declares itself; every GPU that loads the library holds that
 * array until the process exits.  It calls no allocator.
 *
 * Arguments, results and errors are those of sa_decode without the workspace
 * pair.  A split that needs more than SA_STATIC_WORKSPACE_BYTES of scratch
 * (see sa_decode_workspace_size) is refused with SA_ERR_WORKSPACE before any
 * launch; ask for fewer chunks or use sa_decode.  The first call on each
 * device looks up the array's device address (cudaGetSymbolAddress); make that
 * first call before any stream capture on that device.
 *
 * All calls share the one array and it keeps whatever the last call left in
 * it.  Nothing in it needs to start at zero (each call writes every entry it
 * later reads), but two calls whose work overlaps on the GPU -- on different
 * streams, or from different threads -- race on it: order them.
 */
#define SA_STATIC_WORKSPACE_BYTES (16u << 20) /* 16 MiB */
sa_status_t sa_decode_static_workspace(const void *q, const sa_kv_desc_t *kv, const int32_t *seqlens,
                                       int32_t batch, int32_t num_qo_heads, int32_t max_kv_len,
                                       const float *sinks, int32_t window, float sm_scale, void *out,
                                       float *lse, int32_t num_splits, cudaStream_t stream);

/*
 * sa_selftest_wait_timeout -- exercise the failure path of the pipeline waits
 * on the device: two blocks wait on a shared-memory barrier that nothing
 * completes, through the same bounded wait as every kernel of the library
 * (about 1 s), then set SA_DEVICE_TIMEOUT and return.  The context stays
 * usable.  For failure-detection tests; queues work on `stream` and returns.
 * Returns SA_OK or SA_ERR_CUDA.
 */
sa_status_t sa_selftest_wait_timeout(cudaStream_t stream);

/*
 * sa_device_status -- synchronise `stream`, then read and clear the device
 * status word (SA_DEVICE_* bits) of the current device.  The only call that
 * blocks the host.  Returns SA_OK or SA_ERR_CUDA.
 */
sa_status_t sa_device_status(cudaStream_t stream, uint32_t *flags_out);

const char *sa_status_string(sa_status_t status);
const char *sa_last_error(void);  /* thread-local; "" when none */
int sa_version(void);             /* SA_VERSION */

#ifdef __cplusplus
}
#endif

#endif /* SINK_ATTN_H */
