// tmem_softmax.cuh -- one 64-key tile of the per-row online softmax, with S in
// tensor memory: the masking of edge tiles and the max / exp2 / sum / P pass.
// Shared by the tcgen05 kernels (prefill.cu, decode_mt.cu), where one thread
// owns one query row (TMEM lane) of a 128-row accumulator.
#pragma once

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace tsm {

constexpr int kCols = 64;                  // keys per tile: the S columns of a row
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest tolerated p

// Edge tiles (straddling the causal diagonal, the window's lower edge or the
// sequence end): overwrite the hidden keys' scores in TMEM with -inf, by
// select, so that NaN scores past the sequence vanish too.  The row sees the
// tile's columns lo .. hi (none when hi < lo).  A 32-column chunk that every
// row of the warp sees whole is skipped.  Interior tiles skip this and the
// softmax body carries no mask arithmetic.
__device__ __forceinline__ void mask_tile(uint32_t s_addr, int lo, int hi)
{
    // column e is visible iff (unsigned)(e - lo) <= span
    const uint32_t span = hi >= lo ? static_cast<uint32_t>(hi - lo) : 0u;
    const int lo_eff = hi >= lo ? lo : (1 << 20);
#pragma unroll 1
    for (int c = 0; c < kCols / 32; ++c) {
        if (__all_sync(0xffffffffu, lo <= 32 * c && hi >= 32 * c + 31))
            continue;
        uint32_t v[32];
        tmem_ld32(s_addr + 32 * c, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
            v[i] = static_cast<uint32_t>(32 * c + i - lo_eff) <= span ? v[i] : 0xff800000u;
        tmem_st32(s_addr + 32 * c, v);
    }
    tmem_st_wait();
}

// One 64-key tile of the online softmax for the query row this thread owns.
// Pass 1 reads S (TMEM) 16 columns at a time for the row max; pass 2 reads it
// again, forms p = 2^(s*scale - m) (fma.f32x2, ex2; ex2 of -inf is exactly 0),
// adds p into two paired sums (add.f32x2), packs p to bf16 and stores it as P
// over the leading columns of S.  When m moved, O is rescaled.
template <bool FP8>
__device__ __forceinline__ void softmax_tile(uint32_t s_addr, uint32_t o_addr, float scale, bool o_live, float &m,
                                             float &l)
{
    constexpr int kChunk = 16;  // columns per TMEM read: few live registers at two blocks per SM
    uint32_t sr[kChunk];
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int c = 0; c < kCols / kChunk; ++c) {
        tmem_ld16(s_addr + kChunk * c, sr);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kChunk; i += 8)
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                mx[q4] = max3f(mx[q4], __uint_as_float(sr[i + 2 * q4]), __uint_as_float(sr[i + 2 * q4 + 1]));
    }
    const float mt = max3f(mx[0], mx[1], fmaxf(mx[2], mx[3])) * scale;  // scale > 0
    const bool upd = mt > m + kRescaleThreshold;
    const bool any_upd = __any_sync(0xffffffffu, upd);
    float alpha = 1.f;
    if (upd) {
        alpha = ex2(m - mt);  // m = -inf gives 0
        l *= alpha;
        m = mt;
    }
    const float negmu = m == -INFINITY ? 0.f : -m;
    const uint64_t scale2 = f2_pack(scale, scale);
    const uint64_t negmu2 = f2_pack(negmu, negmu);
    uint64_t ls2[2] = {0ull, 0ull};
#pragma unroll
    for (int c = 0; c < kCols / kChunk; ++c) {
        tmem_ld16(s_addr + kChunk * c, sr);
        tmem_ld_wait();
        uint32_t pk[kChunk / 2];
#pragma unroll
        for (int i = 0; i < kChunk; i += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), scale2, negmu2), x0, x1);
            const float p0 = ex2(x0);
            const float p1 = ex2(x1);
            ls2[(i >> 1) & 1] = f2_add(ls2[(i >> 1) & 1], f2_pack(p0, p1));
            pk[i >> 1] = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
        }
        tmem_st8(s_addr + (kChunk / 2) * c, pk);  // P columns [8c, 8c+8): S columns already read
    }
    float a0, a1, b0, b1;
    f2_unpack(ls2[0], a0, a1);
    f2_unpack(ls2[1], b0, b1);
    l += (a0 + a1) + (b0 + b1);
    if (any_upd && o_live) {
        // O holds earlier tiles at the old max: rescale it.  PV of this tile
        // waits for the P handshake, and PV of the previous tile completed
        // before this S was reported.
#pragma unroll
        for (int c = 0; c < kHeadDim / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(o_addr + 32 * c, ov);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
                ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(o_addr + 32 * c, ov);
        }
    }
}


// softmax_tile with the row's 64 scores held in registers: one TMEM read of S
// (two 32-column loads, one wait), the edge mask applied by select (column e
// is visible iff lo <= e <= hi; `edge` false skips it), the max, the p pass
// and one 32-column store of P.  Two TMEM round trips per tile instead of
// eight, for kernels whose softmax sits on the critical chain and can spare
// the registers.
template <bool FP8>
__device__ __forceinline__ void softmax_tile_r(uint32_t s_addr, uint32_t o_addr, float scale, bool o_live, bool edge,
                                               int lo, int hi, float &m, float &l)
{
    uint32_t sa[32], sb[32];
    tmem_ld32(s_addr, sa);
    tmem_ld32(s_addr + 32, sb);
    tmem_ld_wait();
    if (edge) {
        const uint32_t span = hi >= lo ? static_cast<uint32_t>(hi - lo) : 0u;
        const int lo_eff = hi >= lo ? lo : (1 << 20);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            sa[i] = static_cast<uint32_t>(i - lo_eff) <= span ? sa[i] : 0xff800000u;
            sb[i] = static_cast<uint32_t>(32 + i - lo_eff) <= span ? sb[i] : 0xff800000u;
        }
    }
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        mx[0] = max3f(mx[0], __uint_as_float(sa[i]), __uint_as_float(sa[i + 1]));
        mx[1] = max3f(mx[1], __uint_as_float(sa[i + 2]), __uint_as_float(sa[i + 3]));
        mx[2] = max3f(mx[2], __uint_as_float(sb[i]), __uint_as_float(sb[i + 1]));
        mx[3] = max3f(mx[3], __uint_as_float(sb[i + 2]), __uint_as_float(sb[i + 3]));
    }
    const float mt = max3f(mx[0], mx[1], fmaxf(mx[2], mx[3])) * scale;  // scale > 0
    const bool upd = mt > m + kRescaleThreshold;
    const bool any_upd = __any_sync(0xffffffffu, upd);
    float alpha = 1.f;
    if (upd) {
        alpha = ex2(m - mt);  // m = -inf gives 0
        l *= alpha;
        m = mt;
    }
    const float negmu = m == -INFINITY ? 0.f : -m;
    const uint64_t scale2 = f2_pack(scale, scale);
    const uint64_t negmu2 = f2_pack(negmu, negmu);
    uint64_t ls2[2] = {0ull, 0ull};
    uint32_t pk[32];
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
        const uint32_t *src = i < 32 ? sa + i : sb + (i - 32);
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(src[0]), __uint_as_float(src[1])), scale2, negmu2), x0, x1);
        const float p0 = ex2(x0);
        const float p1 = ex2(x1);
        ls2[(i >> 1) & 1] = f2_add(ls2[(i >> 1) & 1], f2_pack(p0, p1));
        pk[i >> 1] = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
    }
    tmem_st32(s_addr, pk);  // P over S columns 0 .. 31 (all of S is in registers)
    float a0, a1, b0, b1;
    f2_unpack(ls2[0], a0, a1);
    f2_unpack(ls2[1], b0, b1);
    l += (a0 + a1) + (b0 + b1);
    if (any_upd && o_live) {
        // O holds earlier tiles at the old max: rescale it (PV of the
        // previous tile completed before this S was reported)
#pragma unroll
        for (int c = 0; c < kHeadDim / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(o_addr + 32 * c, ov);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
                ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(o_addr + 32 * c, ov);
        }
    }
}

}  // namespace tsm
}  // namespace sa
