// merge.cu -- merge of split attention states with the sink counted once.
//
// "GPT-OSS on day 0" (Perplexity), section "Sink Attention": when the
// softmax is split into chunks along the sequence, the sink may enter only
// once.  Each chunk s leaves a sink-free state (o_s, lse_s); for one (row n,
// head h):
//   M = max(sigma_h, max_s lse_s),  Z = exp(sigma_h - M) + sum_s exp(lse_s - M)
//   out = sum_s exp(lse_s - M) o_s / Z,  lse = M + log Z.
// One warp per (n, h): the lanes first take the max of the S log-sum-exps,
// then each lane accumulates a float4 slice of the head dimension over the
// chunks (reads are float4-coalesced across the warp).
#include <cuda_bf16.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace {

constexpr int kMergeWarps = 8;

__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t NH = static_cast<int64_t>(p.n) * p.num_heads;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
    if (row >= NH)
        return;
    const int h = static_cast<int>(row % p.num_heads);
    const float sigma = p.sinks ? __ldg(p.sinks + h) : -INFINITY;

    float M = sigma;
    for (int s = lane; s < p.num_splits; s += 32)
        M = fmaxf(M, __ldg(p.lse_part + s * NH + row));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

    const int D = p.head_dim;
    __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(p.out) + row * D;
    if (M == -INFINITY) {  // no key anywhere and no sink
        for (int d = 4 * lane; d < D; d += 128) {
            out[d] = out[d + 1] = out[d + 2] = out[d + 3] = __float2bfloat16(0.f);
        }
        if (lane == 0 && p.lse_out)
            p.lse_out[row] = -INFINITY;
        return;
    }
    float Z = sigma == -INFINITY ? 0.f : expf(sigma - M);
    // up to 256 dims: two float4 per lane
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
    const int d0 = 4 * lane, d1 = 4 * lane + 128;
    for (int s = 0; s < p.num_splits; ++s) {
        const float ls = __ldg(p.lse_part + s * NH + row);
        if (ls == -INFINITY)
            continue;
        const float w = expf(ls - M);
        Z += w;
        const float *o = p.o_part + (s * NH + row) * D;
        if (d0 < D) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(o + d0));
            acc0.x += w * v.x, acc0.y += w * v.y, acc0.z += w * v.z, acc0.w += w * v.w;
        }
        if (d1 < D) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(o + d1));
            acc1.x += w * v.x, acc1.y += w * v.y, acc1.z += w * v.z, acc1.w += w * v.w;
        }
    }
    const float inv = 1.f / Z;
    if (d0 < D) {
        uint2 pk = make_uint2(pack_bf16(acc0.x * inv, acc0.y * inv), pack_bf16(acc0.z * inv, acc0.w * inv));
        *reinterpret_cast<uint2 *>(out + d0) = pk;
    }
    if (d1 < D) {
        uint2 pk = make_uint2(pack_bf16(acc1.x * inv, acc1.y * inv), pack_bf16(acc1.z * inv, acc1.w * inv));
        *reinterpret_cast<uint2 *>(out + d1) = pk;
    }
    if (lane == 0 && p.lse_out)
        p.lse_out[row] = M + logf(Z);
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream)
{
    const int64_t rows = static_cast<int64_t>(p.n) * p.num_heads;
    const int64_t blocks = (rows + kMergeWarps - 1) / kMergeWarps;
    merge_kernel<<<static_cast<unsigned>(blocks), kMergeWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace sa
