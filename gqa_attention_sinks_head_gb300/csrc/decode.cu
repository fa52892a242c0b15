// decode.cu -- paged-KV sink-attention decode for sm_103a.
//
// One thread block per (KV chunk, kv head g, sequence b).  The G <= 8 query
// heads of kv head g share every K/V byte the block reads: the scores of a
// 16-key tile are one tensor-core product S^T = K . Q^T (keys on the mma M
// dimension, the group's heads on N = 8), and the value update is a second
// product O^T += V^T . P^T, so no head re-reads the cache and the fp32 math
// never runs on the FMA pipe at a rate the HBM stream cannot hide.
//
// Pipeline: warp 4 is the producer.  It walks the page table (32 entries
// prefetched ahead in registers) and issues one TMA tile copy per 16-key page
// slice of K and of V (2 KB each in bf16, 1 KB in FP8) into a ring of
// stages, completing on an mbarrier with transaction bytes.  Warps 0-3 are consumers:
// stage i holds four tiles, one per consumer warp.  The tiles land in shared
// memory with the TMA 128-byte (bf16) / 64-byte (FP8) swizzle so that the
// ldmatrix reads below are free of bank conflicts.
//
// Per tile and consumer warp: ldmatrix K -> 4 (bf16) mma for S^T; online
// softmax in base 2 (max via 3 warp shuffles per head pair); P packed to
// 16-bit and transposed in registers with movmatrix into the B operand of the
// value product; ldmatrix.trans V -> 4 mma for O^T.  The softmax follows
// "GPT-OSS on day 0" (Perplexity), section "Sink Attention": a running max m
// and a scale sum d per head, with m started at the head's sink and d at 1
// -- in warp 0 of the unsplit call only, so that the sink is counted once;
// every other warp (and every chunk of a split call) starts from m = -inf,
// d = 0.  At the end the block merges its four warp states through shared
// memory and writes either the final output (bf16 + natural-log lse) or a
// sink-free partial state for sa_merge_states.
//
// FP8-E4M3 caches (vLLM "GPT-OSS optimisations on NVIDIA Blackwell", FP8 KV
// cache) are widened in registers to f16 (cvt e4m3x2 -> f16x2, exact for
// every code), the products run as f16 mma, and k_scale (resp. v_scale) is
// folded into the score scale (resp. the output scale).  Q is rounded to f16
// for that path.
//
// Multi-token decode (q_len 2..8 new tokens per sequence, as a speculative or
// multi-token-prediction verifier sends them; "GPT-OSS on day 0", the engine's
// speculative and MTP decoders): token k of sequence b sits at position
// L_b - q_len + k.  Each consumer warp owns one token (q_len <= 4) or two
// (TPW = 2, q_len 5..8: two softmax chains interleaved on the same K/V
// fragments); the warps that own the same tokens split the tiles of a stage,
// and a warp's tiles of a stage run as one block of 32 or 64 keys.  The block
// still reads each K/V byte of the kv head once for all tokens and heads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>
#include <type_traits>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
// Pipeline depth.  3 stages x 4 resident blocks per SM keep as many bytes in
// flight as 4 x 3 (192 KB of bf16 K/V per SM), with more blocks to hide the
// per-block prologue and fewer waves for short (window) calls.  FP8 tiles are
// half the size, so the FP8 kernel runs twice the stages for the same bytes.
constexpr int kDefaultStages = 3;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest tolerated p

template <bool FP8>
struct DecodeCfg {
    static constexpr int kRowBytes = kHeadDim * (FP8 ? 1 : 2);  // 64 or 128
    static constexpr int kTileBytes = kTile * kRowBytes;        // 1 KB or 2 KB
};

constexpr int kMaxTPW = 2;  // query tokens per consumer warp (q_len <= 8)
constexpr int kMaxOrderedBatch = 128;  // batches up to this size run longest sequence first
// Row stride (floats) of the block-merge scratch [slot][head][dim]: 4 floats of
// padding put the 8 heads of a warp's float4 reads and of the fragment writes
// in different banks.
constexpr int kRedStride = kHeadDim + 4;

template <bool FP8, int kStages>
struct DecodeSmem {
    // K and V tiles of each stage, one per consumer warp (1 KB aligned).
    uint8_t k[kStages][kConsumerWarps][DecodeCfg<FP8>::kTileBytes];
    uint8_t v[kStages][kConsumerWarps][DecodeCfg<FP8>::kTileBytes];
    float red_m[kConsumerWarps][kMaxTPW][kMaxGroup];
    float red_l[kConsumerWarps][kMaxTPW][kMaxGroup];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int32_t seq;                     // the sequence this block serves
    int32_t lens[kMaxOrderedBatch];  // scratch: the batch's lengths, for the ordering
};

// Byte offset of 16-byte chunk `chunk` of row `row` in a swizzled tile.
template <bool FP8>
__device__ __forceinline__ uint32_t swz(int row, int chunk)
{
    if constexpr (FP8)  // 64-byte rows, 64B swizzle: chunk ^= (row / 2) % 4
        return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
    else  // 128-byte rows, 128B swizzle: chunk ^= row % 8
        return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// kJoint: a warp that owns several tiles of a stage (2..8 query tokens) runs
// them as one block; the one-token kernel is built without that path.  With
// two tokens per warp (TPW 2) that takes more registers: two blocks per SM.
template <bool FP8, int kStages, int TPW, bool kJoint>
__global__ void __launch_bounds__(kThreads, TPW == 1 ? 4 : (kJoint ? 2 : 3)) decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                          const __grid_constant__ CUtensorMap tmv,
                                                                          const DecodeParams p)
{
    using Cfg = DecodeCfg<FP8>;
    extern __shared__ uint8_t smem_raw[];
    // the per-warp O^T partials of the final merge reuse the K tiles
    static_assert(sizeof(float) * kConsumerWarps * TPW * kMaxGroup * kRedStride <=
                      sizeof(uint8_t) * kStages * kConsumerWarps * Cfg::kTileBytes,
                  "merge scratch must fit in the K tiles");
    DecodeSmem<FP8, kStages> &sm =
        *reinterpret_cast<DecodeSmem<FP8, kStages> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    // launched as a programmatic dependent: the grid before it has finished
    // (and its writes are visible) before any global access below
    griddep_wait();
    griddep_launch_dependents();  // the next grid (a merge, the next call) may be scheduled
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int g = blockIdx.y;
    // Longest sequences first: block z serves the sequence of rank z in
    // decreasing length (ties by index), so that the blocks of a ragged batch
    // start longest first and no long one starts last (list scheduling,
    // longest job first).  Only unsplit calls: split chunks are of equal
    // length already, and a windowed call gives every sequence the same keys.
    const bool ordered = p.batch <= kMaxOrderedBatch && p.window == 0 && p.num_splits == 1;
    if (ordered) {
        for (int i = threadIdx.x; i < p.batch; i += kThreads)
            sm.lens[i] = __ldg(p.seqlens + i);
        __syncthreads();
        for (int i = threadIdx.x; i < p.batch; i += kThreads) {
            const int li = sm.lens[i];
            int rank = 0;
            for (int k = 0; k < p.batch; ++k) {
                const int lk = sm.lens[k];
                rank += (lk > li || (lk == li && k < i)) ? 1 : 0;
            }
            if (rank == static_cast<int>(blockIdx.z))
                sm.seq = i;
        }
        __syncthreads();
    }
    const int b = ordered ? sm.seq : static_cast<int>(blockIdx.z);

    // ---- the block's key range: the union over its query tokens -----------
    const int qlen = p.q_len;
    int L = __ldg(p.seqlens + b);
    if (L < 0 || L > p.max_kv_len) {
        if (threadIdx.x == 0)
            atomicOr(p.status, SA_DEVICE_SEQLEN_RANGE);
        L = min(max(L, 0), p.max_kv_len);
    }
    if (L > 0 && L < qlen && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
        atomicOr(p.status, SA_DEVICE_BAD_QLEN);  // tokens at negative positions see no key (L = 0: empty slot)
    // token k sits at L - qlen + k and sees keys (pos - window, pos]
    const int lo = p.window > 0 ? max(0, L - qlen + 1 - p.window) : 0;  // first key of token 0
    const int t_begin = (lo & ~(kTile - 1)) + kTile * p.tiles_per_split * split;  // tile-aligned
    const int t_first = max(t_begin, lo);
    const int t_end = min(L, t_begin + kTile * p.tiles_per_split);
    const int ntiles = t_end > t_first ? (t_end - t_begin + kTile - 1) / kTile : 0;
    const int nstages = (ntiles + kConsumerWarps - 1) / kConsumerWarps;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // Token slots of this consumer warp.  The qlen tokens form G = ceil(qlen /
    // TPW) groups, group g holding tokens g, g + G, ..; warp w takes group
    // w % G, and the `rep` warps that share a group take the stage's tiles j
    // with j % rep == w / G.  Two tokens per warp (TPW 2) interleave two
    // independent softmax chains on the same K/V fragments.
    const int ngroups = max((qlen + TPW - 1) / TPW, 1);
    const int tok0_w = warp % ngroups;
    const int rep = (kConsumerWarps - 1 - tok0_w) / ngroups + 1;
    const int rep_idx = warp / ngroups;
    const int ntok = (TPW == 2 && tok0_w + ngroups < qlen) ? 2 : 1;

    // consumer state (per token slot), kept past the role split for the block-level merge
    float m[TPW][2], l[TPW][2], o[TPW][4][4];
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt) {
        m[tt][0] = m[tt][1] = -INFINITY;
        l[tt][0] = l[tt][1] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                o[tt][i][j] = 0.f;
    }
    const int r = lane >> 2;  // mma row group: key r / r+8 of a tile; head r in the B operand
    const int c = lane & 3;   // mma column pair: heads 2c, 2c+1 of the accumulators

    if (warp == kConsumerWarps) {
        // =================== producer: page-table walk + TMA ================
        if (lane == 0) {
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
        }
        const int32_t *trow = p.page_table ? p.page_table + static_cast<int64_t>(b) * p.table_stride : nullptr;
        auto page_of = [&](int tile) -> int {
            if (tile >= ntiles)
                return 0;
            if (!trow)
                return b;
            return __ldg(trow + (t_begin + tile * kTile) / p.page_size);
        };
        int pg_cur = page_of(lane);        // lane j: page of tile 32k + j
        int pg_next = page_of(32 + lane);  // the next 32, one batch ahead
        const uint64_t pol = l2_policy_evict_first();
        for (int st = 0; st < nstages; ++st) {
            const int buf = st % kStages;
            const int tile0 = st * kConsumerWarps;
            if (tile0 > 0 && (tile0 & 31) == 0) {
                pg_cur = pg_next;
                pg_next = page_of(tile0 + 32 + lane);
            }
            const int page = __shfl_sync(0xffffffffu, pg_cur, (tile0 & 31) + (lane & (kConsumerWarps - 1)));
            if (st >= kStages && !mbar_wait(&sm.empty[buf], ((st / kStages) - 1) & 1, p.status))
                break;
            const int nt = min(kConsumerWarps, ntiles - tile0);
            if (lane == 0)
                mbar_arrive_expect_tx(&sm.full[buf], static_cast<uint32_t>(nt * 2 * Cfg::kTileBytes));
            __syncwarp();
            if (lane < nt) {
                if (page < 0 || page >= p.num_pages)
                    atomicOr(p.status, SA_DEVICE_BAD_PAGE);  // the TMA box falls outside: zeros
                const int slot = (t_begin + (tile0 + lane) * kTile) % p.page_size;
                // coordinates in the tensor map's dimension order (dim 0 = head_dim)
                const int c1 = p.dim_token == 1 ? slot : (p.dim_head == 1 ? g : page);
                const int c2 = p.dim_token == 2 ? slot : (p.dim_head == 2 ? g : page);
                const int c3 = p.dim_token == 3 ? slot : (p.dim_head == 3 ? g : page);
                tma_load_4d_hint(sm.k[buf][lane], &tmk, &sm.full[buf], 0, c1, c2, c3, pol);
                tma_load_4d_hint(sm.v[buf][lane], &tmv, &sm.full[buf], 0, c1, c2, c3, pol);
            }
        }
    } else {
        // =================== consumers ======================================
        const int h0 = g * p.group;

        // Q^T as the B operand (K dimension = head_dim, N = the group's heads),
        // and each token slot's visible key range within this chunk.
        uint32_t qf[TPW][4][2];
        int tf[TPW], te[TPW];
#pragma unroll
        for (int tt = 0; tt < TPW; ++tt) {
            const int tok = tok0_w + ngroups * tt;
            const int hi_k = L - qlen + tok + 1;  // one past the token's own position
            const int lo_k = p.window > 0 ? max(0, hi_k - p.window) : 0;
            tf[tt] = max(t_first, lo_k);
            te[tt] = min(t_end, hi_k);
            const __nv_bfloat16 *qrow =
                reinterpret_cast<const __nv_bfloat16 *>(p.q) +
                ((static_cast<int64_t>(b) * qlen + min(tok, qlen - 1)) * p.num_qo_heads + h0 + r) * kHeadDim;
            const bool ok = r < p.group && tt < ntok;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                if constexpr (FP8) {
                    // k-step ks pairs (4c, 4c+1) and (4c+2, 4c+3) of the 16-dim block,
                    // the order in which the E4M3 K bytes arrive (see below).
                    uint2 w = ok ? *reinterpret_cast<const uint2 *>(qrow + 16 * ks + 4 * c) : make_uint2(0, 0);
                    __nv_bfloat162 x01 = *reinterpret_cast<__nv_bfloat162 *>(&w.x);
                    __nv_bfloat162 x23 = *reinterpret_cast<__nv_bfloat162 *>(&w.y);
                    qf[tt][ks][0] = pack_f16(__bfloat162float(x01.x), __bfloat162float(x01.y));
                    qf[tt][ks][1] = pack_f16(__bfloat162float(x23.x), __bfloat162float(x23.y));
                } else {
                    qf[tt][ks][0] = ok ? *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 2 * c) : 0u;
                    qf[tt][ks][1] = ok ? *reinterpret_cast<const uint32_t *>(qrow + 16 * ks + 2 * c + 8) : 0u;
                }
            }
        }

        // Running state for heads 2c, 2c+1 (m in base 2; l a per-lane partial
        // sum).  The sink seeds one warp per token (the first that holds it).
        if (!p.partial && rep_idx == 0 && p.sinks) {
#pragma unroll
            for (int tt = 0; tt < TPW; ++tt) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int n = 2 * c + j;
                    if (n < p.group && tt < ntok) {
                        m[tt][j] = __ldg(p.sinks + h0 + n) * kLog2e;  // m starts at the sink ...
                        l[tt][j] = (r == 0) ? 1.f : 0.f;              // ... and d at 1 (counted once)
                    }
                }
            }
        }
        const int lr = lane & 7;
        const int mi = lane >> 3;
        // Tiles j0, j0 + jstep, .. (NT of them) of stage buffer buf, taken as one
        // block of NT x 16 keys: NT independent score products, one max / rescale
        // decision and one softmax pass, then NT value products.  NT > 1 gives a
        // warp that owns several tiles of a stage (multi-token decode) NT
        // independent dependency chains instead of NT chains in a row.
        auto run_tiles = [&](auto ntc, int buf, int st, int j0, int jstep) {
            constexpr int NT = decltype(ntc)::value;
            int tok0[NT];
            uint32_t kt[NT], vt[NT];
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                const int j = j0 + i * jstep;
                tok0[i] = t_begin + (st * kConsumerWarps + j) * kTile;
                kt[i] = smem_u32(sm.k[buf][j]);
                vt[i] = smem_u32(sm.v[buf][j]);
            }
#pragma unroll
            for (int tt = 0; tt < TPW; ++tt) {
                const int t_first = tf[tt], t_end = te[tt];
                bool vis = false, edge = false;
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    vis |= tok0[i] + kTile > t_first && tok0[i] < t_end;
                    edge |= tok0[i] < t_first || tok0[i] + kTile > t_end;
                }
                if (tt >= ntok || !vis)
                    continue;  // no key of these tiles is visible to the token
                float (&mm)[2] = m[tt];
                float (&ll)[2] = l[tt];
                float (&oo)[4][4] = o[tt];

                // ---- S^T = K . Q^T  (16 keys x 8 heads per tile, fp32) ----------
                float s[NT][4];
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
                    if constexpr (FP8) {
#pragma unroll
                        for (int j2 = 0; j2 < 2; ++j2) {
                            uint32_t R0, R1, R2, R3;
                            ldsm_x4(kt[i] + swz<true>((mi & 1) * 8 + lr, 2 * j2 + (mi >> 1)), R0, R1, R2, R3);
                            uint32_t k0l, k0h, k1l, k1h;
                            e4m3x4_to_f16x2x2(R0, k0l, k0h);
                            e4m3x4_to_f16x2x2(R1, k1l, k1h);
                            mma_f16(s[i], k0l, k1l, k0h, k1h, qf[tt][2 * j2][0], qf[tt][2 * j2][1]);
                            e4m3x4_to_f16x2x2(R2, k0l, k0h);
                            e4m3x4_to_f16x2x2(R3, k1l, k1h);
                            mma_f16(s[i], k0l, k1l, k0h, k1h, qf[tt][2 * j2 + 1][0], qf[tt][2 * j2 + 1][1]);
                        }
                    } else {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            uint32_t a0, a1, a2, a3;
                            ldsm_x4(kt[i] + swz<false>((mi & 1) * 8 + lr, 2 * ks + (mi >> 1)), a0, a1, a2, a3);
                            mma_bf16(s[i], a0, a1, a2, a3, qf[tt][ks][0], qf[tt][ks][1]);
                        }
                    }
                }

                // ---- online softmax (base 2) -----------------------------------
                // s[i][0]: key r, head 2c   s[i][1]: key r, head 2c+1
                // s[i][2]: key r+8, head 2c s[i][3]: key r+8, head 2c+1
#pragma unroll
                for (int i = 0; i < NT; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        s[i][e] *= p.score_scale;
                uint32_t vm01[NT], vm23[NT];
#pragma unroll
                for (int i = 0; i < NT; ++i)
                    vm01[i] = vm23[i] = 0xffffffffu;
                if (edge) {
#pragma unroll
                    for (int i = 0; i < NT; ++i) {
                        const bool v0 = tok0[i] + r >= t_first && tok0[i] + r < t_end;
                        const bool v8 = tok0[i] + r + 8 >= t_first && tok0[i] + r + 8 < t_end;
                        s[i][0] = v0 ? s[i][0] : -INFINITY;
                        s[i][1] = v0 ? s[i][1] : -INFINITY;
                        s[i][2] = v8 ? s[i][2] : -INFINITY;
                        s[i][3] = v8 ? s[i][3] : -INFINITY;
                        // value rows outside the range are zeroed (a NaN there must not leak via 0 * NaN)
                        const int k0 = tok0[i] + 2 * c, k8 = tok0[i] + 2 * c + 8;
                        vm01[i] = ((k0 >= t_first && k0 < t_end) ? 0x0000ffffu : 0u) |
                                  ((k0 + 1 >= t_first && k0 + 1 < t_end) ? 0xffff0000u : 0u);
                        vm23[i] = ((k8 >= t_first && k8 < t_end) ? 0x0000ffffu : 0u) |
                                  ((k8 + 1 >= t_first && k8 + 1 < t_end) ? 0xffff0000u : 0u);
                    }
                }
                // The running max moves only when some score of the block exceeds it
                // by more than kRescaleThreshold (log2 units): p stays below 2^8,
                // the result is unchanged (numerator and denominator share m), and
                // most blocks skip the cross-lane max and the O rescale.
                float tm0[NT], tm1[NT];  // per-tile maxima, reduced as a tree
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    tm0[i] = fmaxf(s[i][0], s[i][2]);
                    tm1[i] = fmaxf(s[i][1], s[i][3]);
                }
#pragma unroll
                for (int w = 1; w < NT; w *= 2)
#pragma unroll
                    for (int i = 0; i + w < NT; i += 2 * w) {
                        tm0[i] = fmaxf(tm0[i], tm0[i + w]);
                        tm1[i] = fmaxf(tm1[i], tm1[i + w]);
                    }
                float mx0 = tm0[0], mx1 = tm1[0];
                // (-inf - -inf is NaN: a lane with nothing visible never asks)
                const bool grow = mx0 - mm[0] > kRescaleThreshold || mx1 - mm[1] > kRescaleThreshold;
                if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    const float mn0 = fmaxf(mm[0], mx0);
                    const float mn1 = fmaxf(mm[1], mx1);
                    // alpha = 0 from m = -inf (l and O are still 0); 1 while nothing is visible
                    const float al0 = mn0 == -INFINITY ? 1.f : ex2(mm[0] - mn0);
                    const float al1 = mn1 == -INFINITY ? 1.f : ex2(mm[1] - mn1);
                    ll[0] *= al0;
                    ll[1] *= al1;
                    mm[0] = mn0;
                    mm[1] = mn1;
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt) {
                        oo[mt][0] *= al0;
                        oo[mt][1] *= al1;
                        oo[mt][2] *= al0;
                        oo[mt][3] *= al1;
                    }
                }
                const float mu0 = mm[0] == -INFINITY ? 0.f : mm[0];  // keep exp2 finite
                const float mu1 = mm[1] == -INFINITY ? 0.f : mm[1];
                // P (key-major C layout) -> P^T as the B operand (K = keys, N = heads)
                uint32_t pb[NT][2];
                float ps0[NT], ps1[NT];  // per-tile sums of p, reduced as a tree
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    const float p0 = ex2(s[i][0] - mu0);
                    const float p1 = ex2(s[i][1] - mu1);
                    const float p2 = ex2(s[i][2] - mu0);
                    const float p3 = ex2(s[i][3] - mu1);
                    ps0[i] = p0 + p2;
                    ps1[i] = p1 + p3;
                    if constexpr (FP8) {
                        pb[i][0] = movmatrix_t(pack_f16(p0, p1));
                        pb[i][1] = movmatrix_t(pack_f16(p2, p3));
                    } else {
                        pb[i][0] = movmatrix_t(pack_bf16(p0, p1));
                        pb[i][1] = movmatrix_t(pack_bf16(p2, p3));
                    }
                }
#pragma unroll
                for (int w = 1; w < NT; w *= 2)
#pragma unroll
                    for (int i = 0; i + w < NT; i += 2 * w) {
                        ps0[i] += ps0[i + w];
                        ps1[i] += ps1[i + w];
                    }
                ll[0] += ps0[0];
                ll[1] += ps1[0];

                // ---- O^T += V^T . P^T -------------------------------------------
                // Value rows outside a tile's visible range are zeroed (vm01, vm23)
                // on edge blocks only; interior blocks skip the masks.
                auto pv = [&](auto masked) {
                    constexpr bool kMasked = decltype(masked)::value;
#pragma unroll
                    for (int i = 0; i < NT; ++i) {
                        auto mk = [&](uint32_t x, uint32_t vm) { return kMasked ? (x & vm) : x; };
                        if constexpr (FP8) {
#pragma unroll
                            for (int j2 = 0; j2 < 2; ++j2) {
                                uint32_t R0, R1, R2, R3;
                                ldsm_x4_t(vt[i] + swz<true>((mi & 1) * 8 + lr, 2 * j2 + (mi >> 1)), R0, R1, R2, R3);
                                // rows of m-tile 2*j2 (+1): row r <-> dim 16ch + 2r, row r+8 <-> 16ch + 2r + 1;
                                // byte pairs (0, 2) and (1, 3) of each word, gathered by one permute
                                uint32_t v0l, v0h, v1l, v1h, v2l, v2h, v3l, v3h;
                                e4m3x4_to_f16x2x2(prmt(R0, 0x3120u), v0l, v0h);
                                e4m3x4_to_f16x2x2(prmt(R1, 0x3120u), v1l, v1h);
                                e4m3x4_to_f16x2x2(prmt(R2, 0x3120u), v2l, v2h);
                                e4m3x4_to_f16x2x2(prmt(R3, 0x3120u), v3l, v3h);
                                mma_f16(oo[2 * j2], mk(v0l, vm01[i]), mk(v0h, vm01[i]), mk(v1l, vm23[i]),
                                        mk(v1h, vm23[i]), pb[i][0], pb[i][1]);
                                mma_f16(oo[2 * j2 + 1], mk(v2l, vm01[i]), mk(v2h, vm01[i]), mk(v3l, vm23[i]),
                                        mk(v3h, vm23[i]), pb[i][0], pb[i][1]);
                            }
                        } else {
#pragma unroll
                            for (int mt = 0; mt < 4; ++mt) {
                                uint32_t a0, a1, a2, a3;
                                ldsm_x4_t(vt[i] + swz<false>((mi >> 1) * 8 + lr, 2 * mt + (mi & 1)), a0, a1, a2, a3);
                                mma_bf16(oo[mt], mk(a0, vm01[i]), mk(a1, vm01[i]), mk(a2, vm23[i]), mk(a3, vm23[i]),
                                         pb[i][0], pb[i][1]);
                            }
                        }
                    }
                };
                if (edge)
                    pv(std::true_type{});
                else
                    pv(std::false_type{});
            }
        };
        for (int st = 0; st < nstages; ++st) {
            const int buf = st % kStages;
            if (!mbar_wait(&sm.full[buf], (st / kStages) & 1, p.status))
                break;
            const int nt = min(kConsumerWarps, ntiles - st * kConsumerWarps);  // tiles of this stage
            int j = rep_idx;
            if constexpr (kJoint) {
                // the warp's tiles of the stage: four at once, else in pairs
                if (rep == 1 && nt == kConsumerWarps) {
                    run_tiles(std::integral_constant<int, 4>{}, buf, st, 0, 1);
                    j = nt;
                }
                for (; j + rep < nt; j += 2 * rep)
                    run_tiles(std::integral_constant<int, 2>{}, buf, st, j, rep);
            }
            for (; j < nt; j += rep)
                run_tiles(std::integral_constant<int, 1>{}, buf, st, j, rep);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.empty[buf]);
        }
#pragma unroll
        for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                l[tt][j] += __shfl_xor_sync(0xffffffffu, l[tt][j], 4);
                l[tt][j] += __shfl_xor_sync(0xffffffffu, l[tt][j], 8);
                l[tt][j] += __shfl_xor_sync(0xffffffffu, l[tt][j], 16);
            }
    }
    __syncthreads();  // every warp is done with the tiles: their K area holds the merge scratch
    float *red_o = reinterpret_cast<float *>(&sm.k[0][0][0]);  // [warp][slot][head][kRedStride]
    if (warp < kConsumerWarps) {
#pragma unroll
        for (int tt = 0; tt < TPW; ++tt) {
            if (r == 0) {
                sm.red_m[warp][tt][2 * c] = m[tt][0];
                sm.red_m[warp][tt][2 * c + 1] = m[tt][1];
                sm.red_l[warp][tt][2 * c] = l[tt][0];
                sm.red_l[warp][tt][2 * c + 1] = l[tt][1];
            }
            float *w0 = red_o + ((warp * TPW + tt) * kMaxGroup + 2 * c) * kRedStride;  // head 2c
            float *w1 = w0 + kRedStride;                                                // head 2c + 1
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const int dlo = FP8 ? 16 * mt + 2 * r : 16 * mt + r;
                const int dhi = FP8 ? dlo + 1 : dlo + 8;
                w0[dlo] = o[tt][mt][0];
                w1[dlo] = o[tt][mt][1];
                w0[dhi] = o[tt][mt][2];
                w1[dhi] = o[tt][mt][3];
            }
        }
    }
    __syncthreads();

    // ---- merge the warp states of each token; thread t: head t/16, dims 4*(t%16).. ----
    if (threadIdx.x < 128) {
        const int n = threadIdx.x >> 4;
        const int d0 = (threadIdx.x & 15) * 4;
        for (int k = 0; k < qlen && n < p.group; ++k) {
            // slots holding token k: slot k / G of the warps w with w % G == k % G
            const int w0 = k % ngroups;
            const int wstep = ngroups;
            const int tt = k / ngroups;
            float M = -INFINITY;
            for (int w = w0; w < kConsumerWarps; w += wstep)
                M = fmaxf(M, sm.red_m[w][tt][n]);
            float Ls = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
            if (M != -INFINITY) {
                for (int w = w0; w < kConsumerWarps; w += wstep) {
                    const float sc = ex2(sm.red_m[w][tt][n] - M);
                    Ls += sc * sm.red_l[w][tt][n];
                    const float4 src =
                        *reinterpret_cast<const float4 *>(red_o + ((w * TPW + tt) * kMaxGroup + n) * kRedStride + d0);
                    acc[0] += sc * src.x;
                    acc[1] += sc * src.y;
                    acc[2] += sc * src.z;
                    acc[3] += sc * src.w;
                }
            }
            const float inv = Ls > 0.f ? p.out_scale / Ls : 0.f;
            const float lse = Ls > 0.f ? (M + lg2(Ls)) * kLn2 : -INFINITY;
            const int h = g * p.group + n;
            const int64_t qrow = static_cast<int64_t>(b) * qlen + k;  // row of token k
            if (p.partial) {
                const int64_t row = (static_cast<int64_t>(split) * p.batch * qlen + qrow) * p.num_qo_heads + h;
                *reinterpret_cast<float4 *>(p.o_part + row * kHeadDim + d0) =
                    make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
                if (d0 == 0)
                    p.lse_part[row] = lse;
            } else {
                const int64_t row = qrow * p.num_qo_heads + h;
                uint2 pk;
                pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
                pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
                *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + row * kHeadDim + d0) = pk;
                if (d0 == 0 && p.lse)
                    p.lse[row] = lse;
            }
        }
    }
}

template <bool FP8, int kStages>
size_t decode_smem_bytes()
{
    return sizeof(DecodeSmem<FP8, kStages>) + 1024;  // + slack for the 1 KB alignment
}

template <bool FP8, int kStages, int TPW, bool kJoint>
cudaError_t prepare_decode()
{
    // one cudaFuncSetAttribute per device and variant
    static std::atomic<int> done[kMaxDevices];
    return once_per_device(done, [] {
        return cudaFuncSetAttribute(decode_kernel<FP8, kStages, TPW, kJoint>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(decode_smem_bytes<FP8, kStages>()));
    });
}

template <bool FP8, int kStages>
cudaError_t occupancy_of(int *blocks_per_sm)
{
    cudaError_t e = prepare_decode<FP8, kStages, 1, false>();
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_kernel<FP8, kStages, 1, false>,
                                                         kThreads, decode_smem_bytes<FP8, kStages>());
}

template <bool FP8, int kStages, int TPW, bool kJoint>
cudaError_t launch_of(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, cudaStream_t stream)
{
    cudaError_t e = prepare_decode<FP8, kStages, TPW, kJoint>();
    if (e != cudaSuccess)
        return e;
    const dim3 grid(p.num_splits, p.num_kv_heads, p.batch);
    return launch_pdl(decode_kernel<FP8, kStages, TPW, kJoint>, grid, dim3(kThreads), decode_smem_bytes<FP8, kStages>(),
                      stream, tk, tv, p);
}

}  // namespace

cudaError_t decode_occupancy(bool fp8, int *blocks_per_sm)
{
    return fp8 ? occupancy_of<true, 2 * kDefaultStages>(blocks_per_sm)
               : occupancy_of<false, kDefaultStages>(blocks_per_sm);
}

cudaError_t launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, bool fp8,
                          cudaStream_t stream)
{
    // two tokens per consumer warp past four tokens (measured: for q_len 2..4
    // the fourth block per SM that one token per warp allows is worth more than
    // the second chain); from 2 tokens on, a warp takes its tiles of a stage
    // together (q_len 5..8: 2 blocks per SM, 10-12 % over one tile at a time
    // at 3 blocks per SM)
    constexpr int S = kDefaultStages;
    if (p.q_len > 4)
        return fp8 ? launch_of<true, 2 * S, 2, true>(tk, tv, p, stream) : launch_of<false, S, 2, true>(tk, tv, p, stream);
    if (p.q_len > 1)
        return fp8 ? launch_of<true, 2 * S, 1, true>(tk, tv, p, stream) : launch_of<false, S, 1, true>(tk, tv, p, stream);
    return fp8 ? launch_of<true, 2 * S, 1, false>(tk, tv, p, stream) : launch_of<false, S, 1, false>(tk, tv, p, stream);
}

}  // namespace sa
