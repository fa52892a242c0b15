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
// chunks (reads are float4-coalesced across the warp).  For head_dim 64 and
// up to 16 chunks the two half-warps take alternate chunks, and every load
// (the log-sum-exps and all value slices) is issued before any is used: one
// memory round trip instead of two.
#include <cuda_bf16.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace {

constexpr int kMergeWarps = 8;

__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeParams p)
{
    // Launched as a programmatic dependent of the split decode: wait here until
    // that grid has finished and its partial states are visible (returns at
    // once when there is no such dependency).
    griddep_wait();
    griddep_launch_dependents();  // the next call's grid may be scheduled as this one drains
    const int lane = threadIdx.x & 31;
    const int64_t NH = static_cast<int64_t>(p.n) * p.num_heads;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
    if (row >= NH)
        return;
    const int h = static_cast<int>(row % p.num_heads);
    const float sigma = p.sinks ? __ldg(p.sinks + h) : -INFINITY;
    const int S = p.num_splits;
    const int D = p.head_dim;
    __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(p.out) + row * D;

    if (D == 64 && S <= 16) {
        const int half = lane >> 4, d = 4 * (lane & 15);  // chunks half, half + 2, ..; dims d .. d + 3
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int s = half + 2 * k;
            v[k] = s < S ? __ldg(reinterpret_cast<const float4 *>(p.o_part + (s * NH + row) * 64 + d))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float ls = lane < S ? __ldg(p.lse_part + lane * NH + row) : -INFINITY;
        float M = fmaxf(sigma, ls);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        if (M == -INFINITY) {  // no key anywhere and no sink
            if (lane < 16)
                *reinterpret_cast<uint2 *>(out + d) = make_uint2(0u, 0u);
            if (lane == 0 && p.lse_out)
                p.lse_out[row] = -INFINITY;
            return;
        }
        const float w_lane = ls == -INFINITY ? 0.f : expf(ls - M);  // lane s: chunk s's weight
        float Z = w_lane;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            Z += __shfl_xor_sync(0xffffffffu, Z, off);
        Z += sigma == -INFINITY ? 0.f : expf(sigma - M);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float w = __shfl_sync(0xffffffffu, w_lane, (half + 2 * k) & 31);  // 0 past S
            acc.x += w * v[k].x, acc.y += w * v[k].y, acc.z += w * v[k].z, acc.w += w * v[k].w;
        }
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, 16);  // the two halves' chunks
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, 16);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, 16);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, 16);
        const float inv = 1.f / Z;
        if (lane < 16)
            *reinterpret_cast<uint2 *>(out + d) =
                make_uint2(pack_bf16(acc.x * inv, acc.y * inv), pack_bf16(acc.z * inv, acc.w * inv));
        if (lane == 0 && p.lse_out)
            p.lse_out[row] = M + logf(Z);
        return;
    }

    // lane s holds lse of chunk s (chunks past 32 fold in below)
    float ls = lane < S ? __ldg(p.lse_part + lane * NH + row) : -INFINITY;
    float M = fmaxf(sigma, ls);
    for (int s = lane + 32; s < S; s += 32)
        M = fmaxf(M, __ldg(p.lse_part + s * NH + row));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

    if (M == -INFINITY) {  // no key anywhere and no sink
        for (int d = 4 * lane; d < D; d += 128)
            *reinterpret_cast<uint2 *>(out + d) = make_uint2(0u, 0u);
        if (lane == 0 && p.lse_out)
            p.lse_out[row] = -INFINITY;
        return;
    }
    // weights: lane s holds exp(lse_s - M) for the first 32 chunks
    const float w_lane = ls == -INFINITY ? 0.f : expf(ls - M);
    float Z = w_lane;
    for (int s = lane + 32; s < S; s += 32) {
        const float l2 = __ldg(p.lse_part + s * NH + row);
        Z += l2 == -INFINITY ? 0.f : expf(l2 - M);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        Z += __shfl_xor_sync(0xffffffffu, Z, off);
    Z += sigma == -INFINITY ? 0.f : expf(sigma - M);

    // every lane accumulates a float4 slice (two slices when D > 128); the
    // loads of all chunks are independent, so they are issued together
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
    const int d0 = 4 * lane, d1 = 4 * lane + 128;
#pragma unroll 4
    for (int s = 0; s < S; ++s) {
        float w = __shfl_sync(0xffffffffu, w_lane, s & 31);
        if (s >= 32) {
            const float l2 = __ldg(p.lse_part + s * NH + row);
            w = l2 == -INFINITY ? 0.f : expf(l2 - M);
        }
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
    if (d0 < D)
        *reinterpret_cast<uint2 *>(out + d0) =
            make_uint2(pack_bf16(acc0.x * inv, acc0.y * inv), pack_bf16(acc0.z * inv, acc0.w * inv));
    if (d1 < D)
        *reinterpret_cast<uint2 *>(out + d1) =
            make_uint2(pack_bf16(acc1.x * inv, acc1.y * inv), pack_bf16(acc1.z * inv, acc1.w * inv));
    if (lane == 0 && p.lse_out)
        p.lse_out[row] = M + logf(Z);
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream)
{
    const int64_t rows = static_cast<int64_t>(p.n) * p.num_heads;
    const int64_t blocks = (rows + kMergeWarps - 1) / kMergeWarps;
    // Programmatic dependent launch: the merge grid may be scheduled while the
    // kernel before it on the stream drains; griddepcontrol.wait above orders
    // the reads.
    return launch_pdl(merge_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kMergeWarps * 32), 0, stream, p);
}

}  // namespace sa
