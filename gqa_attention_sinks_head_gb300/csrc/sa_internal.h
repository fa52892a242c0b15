// sa_internal.h -- host-side structures shared by the C ABI (api.cu) and the
// kernel launchers (decode.cu, merge.cu, prefill.cu).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/sink_attn.h"

namespace sa {

constexpr int kHeadDim = 64;   // the kernels handle head_dim 64 only
constexpr int kTile = 16;      // decode: keys per tile (one mma M dimension)
constexpr int kMaxGroup = 8;   // decode: query heads per kv head (mma N = 8)

// Decode launch description (one call of sa_decode / sa_decode_partial).
struct DecodeParams {
    const void *q;             // bf16 [B * q_len, Hq, 64]
    const int32_t *seqlens;    // [B]
    const int32_t *page_table; // [B, table_stride] or nullptr
    const float *sinks;        // [Hq] or nullptr (final mode only)
    void *out;                 // final: bf16 [B * q_len, Hq, 64]
    float *lse;                // final: [B * q_len, Hq] or nullptr
    float *o_part;             // partial: [S, B * q_len, Hq, 64]
    float *lse_part;           // partial: [S, B * q_len, Hq]
    uint32_t *status;          // device status word
    int32_t batch, num_qo_heads, num_kv_heads, group;
    int32_t q_len;             // query tokens per sequence (1..8), at positions L - q_len .. L - 1
    int32_t page_size, table_stride, num_pages, max_kv_len;
    int32_t window, num_splits, tiles_per_split;
    int32_t partial;           // 1: write sink-free partial states; 0: final output
    int32_t dim_token, dim_head, dim_page;  // tensor-map dimension (1..3) of each coordinate
    float score_scale;         // multiplies q.k to give base-2 logits
    float out_scale;           // multiplies the normalised value sum (FP8: v_scale)
};

struct MergeParams {
    const float *o_part;
    const float *lse_part;
    const float *sinks;
    void *out;
    float *lse_out;
    int32_t num_splits, n, num_heads, head_dim;
};

// Prefill launch description.
struct PrefillParams {
    const int32_t *cu_seqlens_q;  // [B+1]
    const int32_t *seqlens_kv;    // [B]
    const int32_t *page_table;    // [B, table_stride] or nullptr
    const float *sinks;           // [Hq] or nullptr
    void *out;                    // bf16 [total_q, Hq, 64]
    float *lse;                   // [total_q, Hq] or nullptr
    uint32_t *status;
    int32_t batch, num_qo_heads, num_kv_heads, group, heads_per_cta;
    int32_t page_size, table_stride, num_pages, max_q_len, max_kv_len;
    int32_t window, num_q_tiles;
    int32_t box_rows;                       // keys per K / V tensor-map box: 16, or 64 when a 64-key tile lies in one page
    int32_t dim_token, dim_head, dim_page;  // tensor-map dimension (1..3) of each KV coordinate
    float score_scale;                      // sm_scale * log2(e) (* k_scale for an FP8 cache)
    float out_scale;                        // 1 (v_scale for an FP8 cache)
};

// Rotary embedding + cache append launch description.
struct RopeParams {
    const void *q, *k, *v;        // bf16 [T, Hq, 64], [T, Hkv, 64], [T, Hkv, 64]
    const int32_t *seq_ids;       // [T]
    const int32_t *positions;     // [T]
    const float *table;           // [max_position, 64]: cos (scaled) in 0..31, sin (scaled) in 32..63
    void *q_out;                  // bf16 [T, Hq, 64]
    void *k_cache, *v_cache;      // written
    const int32_t *page_table;    // [batch, table_stride] or nullptr (page = sequence)
    uint32_t *status;
    int64_t stride_page, stride_head, stride_token;  // elements
    int32_t num_tokens, num_qo_heads, num_kv_heads, batch, max_position;
    int32_t page_size, table_stride, num_pages;
    int32_t fp8;                  // cache holds E4M3 codes
    float k_inv_scale, v_inv_scale;  // FP8: 1 / k_scale, 1 / v_scale
    int32_t q_fp8;                // q_out holds E4M3 codes of q / q_scale
    float q_inv_scale;
};

// Record `fmt` as the calling thread's sa_last_error() message and return st.
sa_status_t set_last_error(sa_status_t st, const char *fmt, ...);

// Launch `kernel` on `stream` with programmatic stream serialization: its
// blocks may be scheduled while the kernel before it on the stream drains
// (the kernel itself waits for that grid before any global memory access).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Runs `set` (a per-kernel cudaFuncSetAttribute) once per device: `flags`
// is a static array owned by the caller, indexed by device.  The flag is
// atomic, so concurrent first calls from several host threads are well
// defined: each may run `set`, which the runtime allows from any thread and
// which is idempotent, and every later call sees the flag and skips it.
constexpr int kMaxDevices = 64;
template <typename F>
cudaError_t once_per_device(std::atomic<int> (&flags)[kMaxDevices], F &&set)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const bool tracked = dev >= 0 && dev < kMaxDevices;
    if (tracked && flags[dev].load(std::memory_order_acquire) != 0)
        return cudaSuccess;
    e = set();
    if (e == cudaSuccess && tracked)
        flags[dev].store(1, std::memory_order_release);
    return e;
}

// Launchers (return the launch error, if any).
cudaError_t launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                          bool fp8, cudaStream_t stream);
cudaError_t decode_occupancy(bool fp8, int *blocks_per_sm);
// bf16 cache, q_len 2..8: tq maps q as [B * q_len, Hq, 64] with a box of
// (64, group, q_len); tk / tv take 16-key boxes
cudaError_t launch_decode_mt(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const DecodeParams &p, cudaStream_t stream);
cudaError_t decode_mt_occupancy(int *blocks_per_sm);
cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream);
cudaError_t launch_rope_append(const RopeParams &p, cudaStream_t stream);
cudaError_t launch_wait_timeout_selftest(uint32_t *status, cudaStream_t stream);
cudaError_t launch_prefill(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const PrefillParams &p, bool fp8, bool q8, cudaStream_t stream);

}  // namespace sa
