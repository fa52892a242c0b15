// rope.cu -- the step in front of attention for a batch of new tokens: rotary
// position embedding (YaRN-scaled frequencies) of q and k, and the write of
// k and v into the paged cache, in one pass over the inputs.
//
// "GPT-OSS on day 0" (Perplexity), model overview: YaRN position encoding as
// in DeepSeek-V3; vLLM "GPT-OSS optimisations on NVIDIA Blackwell", list of
// fusions: RoPE, the query and the KV-cache write as one operator.
//
// Memory-bound: every head row (one token's q, k or v of one head: 64 bf16)
// is read once and written once.  Four threads share a row: thread s handles
// dims 8s..8s+7 of the first half and the same dims of the second half, the
// pairs the rotation mixes, with 16-byte loads and stores; each thread takes
// three rows and loads all of them before it stores any.  cos and sin come
// from a table the host fills in double precision (sa_rope_yarn_table), so no
// large-angle argument reduction runs in fp32 on the device.
#include <cuda_bf16.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace {

constexpr int kRowsPerBlock = 64;  // rows one pass of the block covers (4 threads per row)
constexpr int kRowsPerThread = 3;
constexpr int kThreads = 4 * kRowsPerBlock;

__device__ __forceinline__ void unpack8(const uint4 &w, float (&f)[8])
{
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 pack8_bf16(const float (&f)[8])
{
    return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
}

// Eight fp32 values -> eight E4M3 codes (round to nearest even, saturated to
// +-448), lowest element in the lowest byte.
__device__ __forceinline__ uint2 pack8_e4m3(const float (&f)[8], float inv_scale)
{
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        unsigned short d;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
            : "=h"(d)
            : "f"(f[2 * i + 1] * inv_scale), "f"(f[2 * i] * inv_scale));
        h[i] = d;
    }
    return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

// One head row: rotate (unless it is v) and store.  x1/x2 hold dims 8s..8s+7
// of the two halves.
template <bool kCacheFp8, bool kQFp8>
__device__ __forceinline__ void finish_row(const RopeParams &p, int t, int j, int pos, int b, int sub, float (&x1)[8],
                                           float (&x2)[8])
{
    const bool is_q = j < p.num_qo_heads;
    const bool is_v = j >= p.num_qo_heads + p.num_kv_heads;
    const int g = is_q ? 0 : (is_v ? j - p.num_qo_heads - p.num_kv_heads : j - p.num_qo_heads);
    if (!is_v) {
        const float4 *tab = reinterpret_cast<const float4 *>(p.table + static_cast<int64_t>(pos) * kHeadDim);
        const float4 c0 = __ldg(tab + 2 * sub), c1 = __ldg(tab + 2 * sub + 1);
        const float4 s0 = __ldg(tab + 8 + 2 * sub), s1 = __ldg(tab + 8 + 2 * sub + 1);
        const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float a = x1[i], bb = x2[i];
            x1[i] = a * c[i] - bb * s[i];
            x2[i] = bb * c[i] + a * s[i];
        }
    }
    if (is_q) {
        const int64_t qoff = (static_cast<int64_t>(t) * p.num_qo_heads + j) * kHeadDim;
        if (kQFp8) {
            uint8_t *dst = reinterpret_cast<uint8_t *>(p.q_out) + qoff;
            *reinterpret_cast<uint2 *>(dst + 8 * sub) = pack8_e4m3(x1, p.q_inv_scale);
            *reinterpret_cast<uint2 *>(dst + kHeadDim / 2 + 8 * sub) = pack8_e4m3(x2, p.q_inv_scale);
        } else {
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.q_out) + qoff;
            *reinterpret_cast<uint4 *>(dst + 8 * sub) = pack8_bf16(x1);
            *reinterpret_cast<uint4 *>(dst + kHeadDim / 2 + 8 * sub) = pack8_bf16(x2);
        }
        return;
    }
    // cache slot of (sequence b, position pos, kv head g)
    if (p.page_table ? pos / p.page_size >= p.table_stride : pos >= p.page_size) {
        if (sub == 0)
            atomicOr(p.status, SA_DEVICE_BAD_TOKEN);
        return;
    }
    const int page = p.page_table ? __ldg(p.page_table + static_cast<int64_t>(b) * p.table_stride + pos / p.page_size)
                                  : b;
    if (page < 0 || page >= p.num_pages) {
        if (sub == 0)
            atomicOr(p.status, SA_DEVICE_BAD_PAGE);
        return;
    }
    const int64_t off = static_cast<int64_t>(page) * p.stride_page + static_cast<int64_t>(g) * p.stride_head +
                        static_cast<int64_t>(pos % p.page_size) * p.stride_token;
    if (kCacheFp8) {
        uint8_t *dst = reinterpret_cast<uint8_t *>(is_v ? p.v_cache : p.k_cache) + off;
        const float inv = is_v ? p.v_inv_scale : p.k_inv_scale;
        *reinterpret_cast<uint2 *>(dst + 8 * sub) = pack8_e4m3(x1, inv);
        *reinterpret_cast<uint2 *>(dst + kHeadDim / 2 + 8 * sub) = pack8_e4m3(x2, inv);
    } else {
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(is_v ? p.v_cache : p.k_cache) + off;
        *reinterpret_cast<uint4 *>(dst + 8 * sub) = pack8_bf16(x1);
        *reinterpret_cast<uint4 *>(dst + kHeadDim / 2 + 8 * sub) = pack8_bf16(x2);
    }
}

// Each thread takes kRowsPerThread rows, kRowsPerBlock apart, and issues all
// their loads before the first store: more bytes in flight per thread.  Four
// blocks per SM (64 registers, a few words spilled to L1) measured faster than
// three without spills: more rows in flight per SM.
template <bool kCacheFp8, bool kQFp8>
__global__ void __launch_bounds__(kThreads, 4) rope_append_kernel(const RopeParams p)
{
    // launched as a programmatic dependent: the grid before it has finished
    // (and its writes are visible) before any global access below
    griddep_wait();
    griddep_launch_dependents();
    const int sub = threadIdx.x & 3;
    const uint32_t heads = p.num_qo_heads + 2 * p.num_kv_heads;
    const uint32_t nrows = static_cast<uint32_t>(p.num_tokens) * heads;  // < 2^31 (checked on the host)
    const uint32_t row0 = blockIdx.x * (kRowsPerBlock * kRowsPerThread) + (threadIdx.x >> 2);
    uint4 w1[kRowsPerThread], w2[kRowsPerThread];
    int tt[kRowsPerThread], jj[kRowsPerThread], pp[kRowsPerThread], bb[kRowsPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
        const uint32_t row = row0 + r * kRowsPerBlock;
        tt[r] = -1;
        if (row >= nrows)
            continue;
        const int t = static_cast<int>(row / heads);
        const int j = static_cast<int>(row - static_cast<uint32_t>(t) * heads);
        const bool is_q = j < p.num_qo_heads;
        const bool is_v = j >= p.num_qo_heads + p.num_kv_heads;
        const int g = is_q ? 0 : (is_v ? j - p.num_qo_heads - p.num_kv_heads : j - p.num_qo_heads);
        const __nv_bfloat16 *src =
            is_q ? reinterpret_cast<const __nv_bfloat16 *>(p.q) +
                       (static_cast<int64_t>(t) * p.num_qo_heads + j) * kHeadDim
                 : reinterpret_cast<const __nv_bfloat16 *>(is_v ? p.v : p.k) +
                       (static_cast<int64_t>(t) * p.num_kv_heads + g) * kHeadDim;
        w1[r] = __ldg(reinterpret_cast<const uint4 *>(src + 8 * sub));
        w2[r] = __ldg(reinterpret_cast<const uint4 *>(src + kHeadDim / 2 + 8 * sub));
        tt[r] = t;
        jj[r] = j;
        pp[r] = __ldg(p.positions + t);
        bb[r] = __ldg(p.seq_ids + t);
    }
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
        if (tt[r] < 0)
            continue;
        if (pp[r] < 0 || pp[r] >= p.max_position || bb[r] < 0 || bb[r] >= p.batch) {
            if (sub == 0 && jj[r] == 0)
                atomicOr(p.status, SA_DEVICE_BAD_TOKEN);
            continue;
        }
        float x1[8], x2[8];
        unpack8(w1[r], x1);
        unpack8(w2[r], x2);
        finish_row<kCacheFp8, kQFp8>(p, tt[r], jj[r], pp[r], bb[r], sub, x1, x2);
    }
}

}  // namespace

cudaError_t launch_rope_append(const RopeParams &p, cudaStream_t stream)
{
    const int64_t rows = static_cast<int64_t>(p.num_tokens) * (p.num_qo_heads + 2 * p.num_kv_heads);
    const int64_t per_block = static_cast<int64_t>(kRowsPerBlock) * kRowsPerThread;
    const int64_t blocks = (rows + per_block - 1) / per_block;
    if (blocks == 0)
        return cudaSuccess;
    const unsigned nb = static_cast<unsigned>(blocks);
    auto kernel = p.fp8 ? (p.q_fp8 ? rope_append_kernel<true, true> : rope_append_kernel<true, false>)
                        : (p.q_fp8 ? rope_append_kernel<false, true> : rope_append_kernel<false, false>);
    return launch_pdl(kernel, dim3(nb), dim3(kThreads), 0, stream, p);
}

}  // namespace sa
