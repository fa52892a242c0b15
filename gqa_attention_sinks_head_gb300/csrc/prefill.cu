// prefill.cu -- causal / sliding-window sink-attention prefill on tcgen05.
//
// One thread block per (128-query tile, pair of query heads of one kv group,
// sequence), two blocks per SM.  The two heads share every K/V tile: the block
// streams 64-key tiles of K and V through a 4-stage shared-memory ring filled
// by TMA (16-key boxes, so a paged cache needs no special case; one 64-key box
// per operand when no tile straddles a page), and both heads' products run on
// the 5th-generation tensor cores with their accumulators in tensor memory
// (256 columns per block):
//
//   TMEM columns   0..63   S_0 = Q_0 K^T (fp32), its first 32 columns reused for P_0 (bf16 pairs)
//                 64..127  O_0 (fp32)
//                128..191  S_1 / P_1       192..255  O_1
//
// Warp roles (320 threads):
//   warp 0      producer: Q tiles once, then K and V tiles (page-table walk, TMA;
//               for an FP8 cache the E4M3 codes, into a staging area)
//   warp 1      MMA issuer: S_t = Q_t K^T (SS form), O_t += P_t V (P from TMEM, TS form);
//               also zeroes the rows of the last V tile that lie past the sequence
//   warps 2-5   softmax of head 0, warps 6-9 softmax of head 1: one thread per query
//               row; warp w reads TMEM lanes 32*(w%4) .. +31, so each group of four
//               warps covers all 128 rows.  For an FP8 cache they also widen the
//               staged codes to f16, two tiles ahead.  At the end each warp stages
//               its 32 output rows in its head's Q tile and stores whole rows.
//
// Two blocks per SM give four independent softmax streams per SM, and one
// block's prologue, tail and epilogue overlap the other block's work.  Per key
// tile the MMA warp issues, for each head t: PV_t(j) once P_t(j) is in TMEM,
// then at once QK_t(j+1).  The tensor pipe runs a thread's MMAs in order, so
// the commit that reports S_t(j+1) also proves that PV_t(j) read P_t(j) and
// finished writing O_t; the softmax may then rescale O_t.
//
// Softmax ("GPT-OSS on day 0" (Perplexity), section "Sink Attention"): each
// row keeps a running max m (base 2) and sum l, started at the head's sink
// (m = sink * log2 e, l = 1) so the sink enters the denominator once and has
// no value vector.  m only moves when a tile's max exceeds it by more than 8
// (a factor 256): the probabilities then stay below 2^8, the result is the
// same because numerator and denominator share m, and the O rescale (a TMEM
// round trip) becomes rare.  Causal and window masks (NVIDIA gpt-oss launch
// article, introduction: full context alternating with a 128-token window)
// are applied only on tiles that straddle a boundary.
//
// FP8-E4M3 caches (vLLM "GPT-OSS optimisations on NVIDIA Blackwell", FP8 KV
// cache): TMA brings each key tile's E4M3 codes into a 3-slot staging area.
// The softmax warps, right after handing over P of tile j, widen tile j + 2
// (cvt e4m3x2 -> f16x2, exact for every code) into the 3-stage ring of f16
// tiles (128-byte swizzle) the MMAs read, zeroing rows past the sequence end;
// each of the 4 x NH warps takes an equal share, so the widening is spread
// over all four SM sub-partitions instead of loading the producer's.  The softmax warps convert their Q tile from
// bf16 to f16 in place once, P is stored as f16, the products run as
// kind::f16 with f16 operands, and k_scale (resp. v_scale) is folded into the
// score scale (resp. the output scale).
//
// E4M3 queries on an FP8 cache (Q8; the same vLLM passage: part of the
// attention in FP8): Q arrives as E4M3 codes and S = Q K^T runs as
// kind::f8f6f4 straight from the TMA-staged key codes (64-byte swizzle, two
// 32-byte K steps), so only V is widened; the MMA warp releases a staging slot
// once the QK products that read it have completed.
#include <cuda_bf16.h>

#include <type_traits>

#include "sa_internal.h"
#include "sa_ptx.cuh"
#include "tmem_softmax.cuh"

namespace sa {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 64;   // keys per tile
constexpr int kThreads = 320;
constexpr int kFirstSoftmaxWarp = 2;
constexpr uint32_t kQTileBytes = BM * kHeadDim * 2;   // 16 KB
constexpr uint32_t kKVTileBytes = BN * kHeadDim * 2;  // 8 KB
constexpr uint32_t kBoxBytes = 16 * kHeadDim * 2;     // one 16-key box
constexpr uint32_t kKV8TileBytes = BN * kHeadDim;     // 4 KB of E4M3 codes
constexpr uint32_t kBox8Bytes = 16 * kHeadDim;        // one 16-key box of codes
constexpr uint32_t kTmemCols = 256;
__host__ __device__ constexpr uint32_t col_s(int t) { return 128u * t; }        // S_t / P_t
__host__ __device__ constexpr uint32_t col_o(int t) { return 128u * t + 64u; }  // O_t
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;
// Q, K both K-major; V is MN-major (dims contiguous).  f16 operands for an FP8 cache.
template <bool FP8>
constexpr uint32_t kIdescQK = idesc_f32acc(BM, BN, 0, FP8);
constexpr uint32_t kIdescQK8 = idesc_e4m3_f32acc(BM, BN);  // E4M3 Q and K
template <bool FP8>
constexpr uint32_t kIdescPV = idesc_f32acc(BM, kHeadDim, 1, FP8);

using tsm::mask_tile;
using tsm::softmax_tile;
static_assert(BN == tsm::kCols, "the softmax helpers take 64-key tiles");

template <bool FP8>
struct PrefillSmem {
    static constexpr int kStages = FP8 ? 3 : 4;  // 16-bit K/V ring (FP8: widened two tiles ahead)
    static constexpr int kStaged = FP8 ? 3 : 1;  // FP8: slots of E4M3 codes in flight
    uint8_t q[2][kQTileBytes];
    uint8_t k[kStages][kKVTileBytes];
    uint8_t v[kStages][kKVTileBytes];
    uint8_t k8[kStaged][FP8 ? kKV8TileBytes : 16];  // E4M3 staging (64-byte swizzle)
    uint8_t v8[kStaged][FP8 ? kKV8TileBytes : 16];
    uint64_t q_full;
    uint64_t q_conv;  // FP8: Q converted to f16
    uint64_t st_full[kStaged];
    uint64_t k8_empty[kStaged];  // Q8: the QK products that read a staging slot have completed
    uint64_t st_empty[kStaged];  // FP8: the softmax warps have widened the slot's codes
    uint64_t k_full[kStages];
    uint64_t v_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full[2];
    uint64_t p_full[2][kStages];  // per head and ring stage: P of the stage's tile is in TMEM
    uint64_t o_done[2];
    uint32_t tmem_base;
};
static_assert(sizeof(PrefillSmem<false>) + 1024 <= 113 * 1024, "two blocks must fit one SM's shared memory");
static_assert(sizeof(PrefillSmem<true>) + 1024 <= 113 * 1024, "two blocks must fit one SM's shared memory");

// bf16 pair -> f16 pair (round to nearest; |x| < 65504 assumed).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x)
{
    return pack_f16(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

// One key tile of E4M3 codes (64 rows of 64 bytes as TMA wrote them with the
// 64-byte swizzle: 16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3)) ->
// f16 values in the 128-byte-swizzled layout of a 16-bit tile (chunk c of row
// r at chunk c ^ (r & 7)).  Rows at or past `valid` become zeros.  Thread
// `tid` of `nthr` takes the 16-byte chunks tid, tid + nthr, ..
__device__ __forceinline__ void widen_tile(const uint8_t *src, uint8_t *dst, int valid, int tid, int nthr)
{
#pragma unroll 1
    for (int i = tid; i < BN * 4; i += nthr) {
        const int r = i >> 2, c = i & 3;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (r < valid)
            w = *reinterpret_cast<const uint4 *>(src + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
        uint4 lo, hi;
        e4m3x4_to_f16x2x2(w.x, lo.x, lo.y);
        e4m3x4_to_f16x2x2(w.y, lo.z, lo.w);
        e4m3x4_to_f16x2x2(w.z, hi.x, hi.y);
        e4m3x4_to_f16x2x2(w.w, hi.z, hi.w);
        *reinterpret_cast<uint4 *>(dst + r * 128 + (((2 * c) ^ (r & 7)) << 4)) = lo;
        *reinterpret_cast<uint4 *>(dst + r * 128 + (((2 * c + 1) ^ (r & 7)) << 4)) = hi;
    }
}

// One thread's 16-byte chunk of a key tile, placed once: its row, the chunk's
// offset among the E4M3 codes (64-byte swizzle) and the offsets of its two
// f16 halves in the widened tile (128-byte swizzle).  With NH = 2 the 256
// softmax threads cover a tile's 256 chunks, one each.
struct WidenPlan {
    int r;
    uint32_t src, lo, hi;
};
__device__ __forceinline__ WidenPlan widen_plan(int i)
{
    const int r = i >> 2, c = i & 3;
    return WidenPlan{r, static_cast<uint32_t>(r * 64 + ((c ^ ((r >> 1) & 3)) << 4)),
                     static_cast<uint32_t>(r * 128 + (((2 * c) ^ (r & 7)) << 4)),
                     static_cast<uint32_t>(r * 128 + (((2 * c + 1) ^ (r & 7)) << 4))};
}
__device__ __forceinline__ void widen_chunk(const uint8_t *src, uint8_t *dst, const WidenPlan &w, int valid)
{
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (w.r < valid)
        x = *reinterpret_cast<const uint4 *>(src + w.src);
    uint4 lo, hi;
    e4m3x4_to_f16x2x2(x.x, lo.x, lo.y);
    e4m3x4_to_f16x2x2(x.y, lo.z, lo.w);
    e4m3x4_to_f16x2x2(x.z, hi.x, hi.y);
    e4m3x4_to_f16x2x2(x.w, hi.z, hi.w);
    *reinterpret_cast<uint4 *>(dst + w.lo) = lo;
    *reinterpret_cast<uint4 *>(dst + w.hi) = hi;
}

__device__ __forceinline__ void kv_coords(const PrefillParams &p, int slot, int g, int page, int &c1, int &c2,
                                          int &c3)
{
    c1 = p.dim_token == 1 ? slot : (p.dim_head == 1 ? g : page);
    c2 = p.dim_token == 2 ? slot : (p.dim_head == 2 ? g : page);
    c3 = p.dim_token == 3 ? slot : (p.dim_head == 3 ? g : page);
}

// NH: query heads per block, 2 (a pair of one kv group) or 1 (odd groups).
// A compile-time count lets the MMA warp's per-head loop unroll, with every
// head's TMEM columns and barriers fixed, which shortens the P -> next S
// round trip that bounds the kernel.
template <bool FP8, bool Q8, int NH>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const PrefillParams p)
{
    static_assert(FP8 || !Q8, "E4M3 queries need an FP8 cache");
    constexpr int kStages = PrefillSmem<FP8>::kStages;
    constexpr uint32_t kQBytes = Q8 ? kQTileBytes / 2 : kQTileBytes;  // bytes TMA brings per Q tile
    extern __shared__ uint8_t smem_raw[];
    PrefillSmem<FP8> &sm =
        *reinterpret_cast<PrefillSmem<FP8> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // launched as a programmatic dependent: the grid before it has finished
    // (and its writes are visible) before any global access below
    griddep_wait();
    griddep_launch_dependents();  // the next call's grid may be scheduled as this one drains
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int h0 = blockIdx.x * NH;
    const int g = h0 / p.group;
    const int qt = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);  // heavy tiles first
    const int b = blockIdx.z;

    // ---- sequence geometry (uniform over the block) ----------------------
    const int q_beg = __ldg(p.cu_seqlens_q + b);
    int Lq = __ldg(p.cu_seqlens_q + b + 1) - q_beg;
    int Lkv = __ldg(p.seqlens_kv + b);
    if (Lkv < 0 || Lkv > p.max_kv_len) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            atomicOr(p.status, SA_DEVICE_SEQLEN_RANGE);
        Lkv = min(max(Lkv, 0), p.max_kv_len);
    }
    if (Lq < 0 || Lq > Lkv || Lq > p.max_q_len) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            atomicOr(p.status, SA_DEVICE_BAD_QLEN);
        Lq = min(max(Lq, 0), min(Lkv, p.max_q_len));
    }
    const int q0 = qt * BM;
    if (q0 >= Lq)
        return;
    const int rows = min(BM, Lq - q0);
    const int off = Lkv - Lq;  // query i sits at position off + i
    const int p_first = off + q0;
    const int p_last = off + q0 + rows - 1;
    const int k_lo = p.window > 0 ? max(0, p_first - p.window + 1) : 0;
    const int j_first = k_lo / BN;
    const int ntiles = p_last / BN - j_first + 1;

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        mbar_init(&sm.q_conv, 4 * NH);
        for (int i = 0; i < PrefillSmem<FP8>::kStaged; ++i) {
            mbar_init(&sm.st_full[i], 1);
            mbar_init(&sm.k8_empty[i], 1);
            mbar_init(&sm.st_empty[i], 4 * NH);
        }
        for (int i = 0; i < kStages; ++i) {
            // FP8: every softmax warp arrives after widening its share
            mbar_init(&sm.k_full[i], FP8 ? 4 * NH : 1);
            mbar_init(&sm.v_full[i], FP8 ? 4 * NH : 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&sm.s_full[t], 1);
            for (int i = 0; i < kStages; ++i)
                mbar_init(&sm.p_full[t][i], 4);
            mbar_init(&sm.o_done[t], 1);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // ============================ producer ============================
        if (lane == 0) {
            tma_prefetch_desc(&tmq);
            tma_prefetch_desc(&tmk);
            tma_prefetch_desc(&tmv);
            mbar_arrive_expect_tx(&sm.q_full, static_cast<uint32_t>(NH) * kQBytes);
            for (int t = 0; t < NH; ++t)
                tma_load_3d(sm.q[t], &tmq, &sm.q_full, 0, h0 + t, q_beg + q0);
        }
        const int32_t *trow = p.page_table ? p.page_table + static_cast<int64_t>(b) * p.table_stride : nullptr;
        auto boxes = [&](int it) { return min(BN / 16, (Lkv - (j_first + it) * BN + 15) / 16); };
        auto page_of = [&](int it) -> int {
            if (it >= ntiles || lane >= boxes(it))
                return 0;
            const int key = (j_first + it) * BN + 16 * lane;
            return trow ? __ldg(trow + key / p.page_size) : b;
        };
        if constexpr (FP8) {
            // codes of tile j -> staging slot j % kStaged; a slot is reused once
            // the softmax warps have widened (and proxy-fenced) the tile it held
            // and, Q8, the QK products that read its key codes have completed
            constexpr int kStaged = PrefillSmem<FP8>::kStaged;
            for (int j = 0; j < ntiles; ++j) {
                const int sb = j % kStaged;
                if (j >= kStaged) {
                    const uint32_t ph = ((j / kStaged) - 1) & 1;
                    if (!mbar_wait(&sm.st_empty[sb], ph, p.status) ||
                        (Q8 && !mbar_wait(&sm.k8_empty[sb], ph, p.status)))
                        break;
                }
                const int nbox = boxes(j);
                const int page = page_of(j);
                const int key = (j_first + j) * BN + 16 * lane;
                int c1 = 0, c2 = 0, c3 = 0;
                if (lane < nbox) {
                    if (page < 0 || page >= p.num_pages)
                        atomicOr(p.status, SA_DEVICE_BAD_PAGE);  // outside the map: the box reads zeros
                    kv_coords(p, key % p.page_size, g, page, c1, c2, c3);
                }
                if (lane == 0)
                    mbar_arrive_expect_tx(&sm.st_full[sb], 2u * static_cast<uint32_t>(nbox) * kBox8Bytes);
                __syncwarp();
                if (lane < nbox) {
                    tma_load_4d(sm.k8[sb] + lane * kBox8Bytes, &tmk, &sm.st_full[sb], 0, c1, c2, c3);
                    tma_load_4d(sm.v8[sb] + lane * kBox8Bytes, &tmv, &sm.st_full[sb], 0, c1, c2, c3);
                }
            }
        } else {
            // One box per lane, so that the copies' issue latencies overlap:
            // lanes 0-3 the tile's K boxes, lanes 4-7 its V boxes (a 64-key box
            // when no tile straddles a page: lanes 0 and 4).  A stage is refilled
            // once the products that read its previous tile u have completed:
            // Q K^T of tile u + 1 for the last head is issued behind every head's
            // P V of tile u, and the softmax of that head's S of tile u + 1 has
            // read it, so the last head's P barrier of tile u + 1 says so (no
            // commit of its own).  The P barriers are per ring stage: the next
            // phase of the one waited here needs a tile not yet loaded, so the
            // parity wait cannot mistake a phase two ahead for the awaited one.
            const int is_v = (lane >> 2) & 1, bi = lane & 3;
            const uint32_t box_bytes = static_cast<uint32_t>(p.box_rows) * kHeadDim * 2;
            auto nbox_of = [&](int it) { return p.box_rows == 64 ? 1 : boxes(it); };
            auto page_for = [&](int it) -> int {  // the page of this lane's box of tile it
                if (it >= ntiles || lane >= 8 || bi >= nbox_of(it))
                    return 0;
                const int key = (j_first + it) * BN + 16 * bi;
                return trow ? __ldg(trow + key / p.page_size) : b;
            };
            int next_page = page_for(0);
            for (int it = 0; it < ntiles; ++it) {
                const int stage = it % kStages;
                const int nbox = nbox_of(it);
                const int page = next_page;
                next_page = page_for(it + 1);  // one tile ahead: the table read overlaps the wait
                const int u1 = it - kStages + 1;  // the tile after the stage's previous one
                if (u1 > 0 && !mbar_wait(&sm.p_full[NH - 1][u1 % kStages], (u1 / kStages) & 1, p.status))
                    break;
                const int key = (j_first + it) * BN + 16 * bi;
                const bool mine = lane < 8 && bi < nbox;
                int c1 = 0, c2 = 0, c3 = 0;
                if (mine) {
                    if (page < 0 || page >= p.num_pages)
                        atomicOr(p.status, SA_DEVICE_BAD_PAGE);  // outside the map: the box reads zeros
                    kv_coords(p, key % p.page_size, g, page, c1, c2, c3);
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&sm.k_full[stage], static_cast<uint32_t>(nbox) * box_bytes);
                    mbar_arrive_expect_tx(&sm.v_full[stage], static_cast<uint32_t>(nbox) * box_bytes);
                }
                __syncwarp();
                if (mine)
                    tma_load_4d((is_v ? sm.v[stage] : sm.k[stage]) + bi * kBoxBytes, is_v ? &tmv : &tmk,
                                is_v ? &sm.v_full[stage] : &sm.k_full[stage], 0, c1, c2, c3);
            }
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ==========================
        // Descriptor bases; a K step adds to the start-address field (bytes >> 4):
        // 32 bytes (16 dims) for Q/K, 2048 bytes (16 keys) for V.
        // Q8: E4M3 Q and key codes, 64-byte rows with the 64-byte swizzle (8-row groups of 512 bytes)
        const uint64_t dq0 = Q8 ? smem_desc(smem_u32(sm.q[0]), 16, 512, 4u) : smem_desc_sw128(smem_u32(sm.q[0]), 16, 1024);
        const uint64_t dk0 = Q8 ? smem_desc(smem_u32(sm.k8[0]), 16, 512, 4u) : smem_desc_sw128(smem_u32(sm.k[0]), 16, 1024);
        const uint64_t dv0 = smem_desc_sw128(smem_u32(sm.v[0]), 16, 1024);
        // stage: ring stage of K (16-bit) or staging slot of the key codes (Q8)
        auto issue_qk = [&](int t, int stage) {
            const uint64_t dq = dq0 + static_cast<uint64_t>(t) * (kQTileBytes >> 4);  // q[1] follows q[0]
            if constexpr (Q8) {
                const uint64_t dk = dk0 + static_cast<uint64_t>(stage) * (kKV8TileBytes >> 4);
#pragma unroll
                for (int ks = 0; ks < kHeadDim / 32; ++ks)  // K = 32 one-byte elements per product
                    umma_ss_f8(tmem + col_s(t), dq + 2 * ks, dk + 2 * ks, kIdescQK8, ks > 0 ? 1u : 0u);
            } else {
                const uint64_t dk = dk0 + static_cast<uint64_t>(stage) * (kKVTileBytes >> 4);
#pragma unroll
                for (int ks = 0; ks < kHeadDim / 16; ++ks)
                    umma_ss(tmem + col_s(t), dq + 2 * ks, dk + 2 * ks, kIdescQK<FP8>, ks > 0 ? 1u : 0u);
            }
        };
        constexpr int kStaged = PrefillSmem<FP8>::kStaged;
        // K of tile j is ready: the 16-bit ring stage, or (Q8) the TMA of its staging slot
        auto wait_k = [&](int j) -> bool {
            if (Q8)
                return mbar_wait(&sm.st_full[j % kStaged], (j / kStaged) & 1, p.status);
            return mbar_wait(&sm.k_full[j % kStages], (j / kStages) & 1, p.status);
        };
        auto k_slot = [&](int j) { return Q8 ? j % kStaged : j % kStages; };
        auto issue_pv = [&](int t, int stage, bool accumulate) {
            const uint64_t dv = dv0 + static_cast<uint64_t>(stage) * (kKVTileBytes >> 4);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)  // K = 16 keys: 8 TMEM columns of P, 2 KB of V
                umma_ts(tmem + col_o(t), tmem + col_s(t) + 8 * kk, dv + 128 * kk, kIdescPV<FP8>,
                        (accumulate || kk > 0) ? 1u : 0u);
        };
        bool ok = mbar_wait((FP8 && !Q8) ? &sm.q_conv : &sm.q_full, 0, p.status) && wait_k(0);
        if (ok) {
            tc_fence_after();
            if (lane == 0) {
                for (int t = 0; t < NH; ++t) {
                    issue_qk(t, 0);
                    umma_commit(&sm.s_full[t]);
                }
                if (Q8)
                    umma_commit(&sm.k8_empty[0]);
            }
            __syncwarp();
        }
        // One key tile; LAST (compile time) marks the block's last tile, the
        // only one with no next Q K^T and the only one that can reach past the
        // sequence end, so the steady-state tiles carry neither test.
        auto tile = [&](auto LAST_, int it) -> bool {
            constexpr bool LAST = decltype(LAST_)::value;
            const int stage = it % kStages;
            // V of this tile, P of head 0 and K of the next tile (Q8: its staged
            // codes), checked together first; the bounded waits below only when
            // one is missing
            bool ready = false;
            {
                const int kn = LAST ? it : it + 1;
                uint64_t *kb = Q8 ? &sm.st_full[kn % kStaged] : &sm.k_full[kn % kStages];
                const uint32_t kp = Q8 ? (kn / kStaged) & 1 : (kn / kStages) & 1;
                ready = mbar_try_wait3(&sm.v_full[stage], (it / kStages) & 1, &sm.p_full[0][stage], (it / kStages) & 1,
                                       kb, kp);
            }
            if (!ready && !mbar_wait(&sm.v_full[stage], (it / kStages) & 1, p.status))
                return false;
            if constexpr (!FP8 && LAST) {  // (the FP8 widening zeroes these rows itself)
                const int key0 = (j_first + it) * BN;
                if (key0 + BN > Lkv) {
                    // value rows past the sequence may hold anything (NaN included):
                    // zero them so that p = 0 contributes exactly 0
                    const int first_bad = max(Lkv - key0, 0);
                    uint4 *vz = reinterpret_cast<uint4 *>(sm.v[stage]);
                    for (int i = first_bad * 8 + lane; i < BN * 8; i += 32)
                        vz[i] = make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();
                    __syncwarp();
                }
            }
#pragma unroll
            for (int t = 0; t < NH; ++t) {
                if (!(ready && t == 0) && !mbar_wait(&sm.p_full[t][stage], (it / kStages) & 1, p.status))
                    return false;
                tc_fence_after();
                if (lane == 0) {
                    issue_pv(t, stage, it > 0);
                    if constexpr (LAST)
                        umma_commit(&sm.o_done[t]);  // this head's O is final
                }
                if constexpr (!LAST) {
                    // (after head 0 the next K is known to be there)
                    const bool k_known = ready || t > 0;
                    if (!k_known && !wait_k(it + 1))
                        return false;
                    tc_fence_after();
                    if (lane == 0) {
                        issue_qk(t, k_slot(it + 1));
                        umma_commit(&sm.s_full[t]);
                    }
                }
                __syncwarp();
            }
            if (lane == 0) {
                if (FP8)  // (bf16: the producer watches the last head's P barriers instead)
                    umma_commit(&sm.kv_empty[stage]);
                if (Q8 && !LAST)
                    umma_commit(&sm.k8_empty[(it + 1) % kStaged]);  // every head's QK(it + 1) is issued
            }
            __syncwarp();
            return true;
        };
        for (int it = 0; ok && it + 1 < ntiles; ++it)
            ok = tile(std::false_type{}, it);
        if (ok && ntiles > 0)
            ok = tile(std::true_type{}, ntiles - 1);
        if ((!ok || ntiles == 0) && lane == 0)  // (gave up: release the epilogues, which then see the status)
            for (int t = 0; t < NH; ++t)
                umma_commit(&sm.o_done[t]);
        __syncwarp();
    } else if (((warp - kFirstSoftmaxWarp) >> 2) < NH) {
        // ============================ softmax =============================
        const int t = (warp - kFirstSoftmaxWarp) >> 2;
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + col_s(t);
        const uint32_t o_addr = tmem + lane_base + col_o(t);
        const int qi = q0 + row;
        const int pos = off + qi;
        const int h = h0 + t;
        float m = -INFINITY, l = 0.f;
        if (p.sinks) {
            m = __ldg(p.sinks + h) * kLog2e;  // the running max starts at the sink ...
            l = 1.f;                          // ... and the sum at 1
        }
        bool ok = true;
        if constexpr (FP8 && !Q8) {
            // this thread's Q row, bf16 -> f16 in place (the swizzle only
            // permutes 16-byte chunks within the row); lanes start at
            // different chunks so that no two of 8 lanes share banks
            ok = mbar_wait(&sm.q_full, 0, p.status);
            if (ok) {
                uint4 *qrow = reinterpret_cast<uint4 *>(sm.q[t] + row * 128);
#pragma unroll
                for (int c0 = 0; c0 < 8; ++c0) {
                    const int c = (c0 + lane) & 7;
                    uint4 w = qrow[c];
                    w.x = bf16x2_to_f16x2(w.x);
                    w.y = bf16x2_to_f16x2(w.y);
                    w.z = bf16x2_to_f16x2(w.z);
                    w.w = bf16x2_to_f16x2(w.w);
                    qrow[c] = w;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&sm.q_conv);
            }
        }
        // (the E4M3-query kernel keeps its scores in registers and has none to spare)
        const WidenPlan wplan = (FP8 && !Q8 && NH == 2) ? widen_plan(static_cast<int>(threadIdx.x) - 32 * kFirstSoftmaxWarp)
                                                        : WidenPlan{0, 0u, 0u, 0u};
        // FP8: widen the staged codes of tile j (K unless Q8, and V) into ring
        // stage j % kStages, this thread's share of the block's softmax threads
        auto widen = [&](int j) -> bool {
            constexpr int kStaged = PrefillSmem<FP8>::kStaged;
            const int sb = j % kStaged, stage = j % kStages;
            if (!mbar_wait(&sm.st_full[sb], (j / kStaged) & 1, p.status))
                return false;
            // the stage's previous tile (j - kStages): its products have completed
            if (j >= kStages && !mbar_wait(&sm.kv_empty[stage], ((j / kStages) - 1) & 1, p.status))
                return false;
            const int valid = min(BN, Lkv - (j_first + j) * BN);
            if constexpr (NH == 2 && !Q8) {
                // one chunk of K and one of V per thread, at the offsets placed once
                widen_chunk(sm.k8[sb], sm.k[stage], wplan, valid);
                widen_chunk(sm.v8[sb], sm.v[stage], wplan, valid);
            } else {
                const int wtid = static_cast<int>(threadIdx.x) - 32 * kFirstSoftmaxWarp;
                if (!Q8)  // (Q8: the QK products read the key codes where TMA put them)
                    widen_tile(sm.k8[sb], sm.k[stage], valid, wtid, 128 * NH);
                widen_tile(sm.v8[sb], sm.v[stage], valid, wtid, 128 * NH);
            }
            fence_proxy_async_smem();  // generic writes -> tensor-core reads; staging reads -> next TMA
            __syncwarp();
            if (lane == 0) {
                if (!Q8)
                    mbar_arrive(&sm.k_full[stage]);
                mbar_arrive(&sm.v_full[stage]);
                mbar_arrive(&sm.st_empty[sb]);
            }
            return true;
        };
        if constexpr (FP8)
            for (int j = 0; ok && j < min(ntiles, kStages - 1); ++j)
                ok = widen(j);
        // The row's visible keys, and the tiles it_lo .. it_hi - 1 that every
        // row of the block sees whole (the rest straddle the causal diagonal,
        // the window's lower edge or the sequence end), worked out once so that
        // the tile loop keeps two bounds live instead of the block's geometry.
        const int row_lo = p.window > 0 ? max(pos - p.window + 1, 0) : 0;
        const int row_hi = min(pos, Lkv - 1);
        // below: every row sees the keys from p_last - window + 1 on (window > 0)
        const int it_lo = p.window > 0 ? max(0, (p_last - p.window + BN) / BN - j_first) : 0;
        // above: every row sees the keys below min(p_first + 1, Lkv)
        const int it_hi = max(it_lo, min(p_first + 1, Lkv) / BN - j_first);
        for (int it = 0; ok && it < ntiles; ++it) {
            if (!mbar_wait(&sm.s_full[t], it & 1, p.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int key0 = (j_first + it) * BN;
            const bool edge = it < it_lo || it >= it_hi;  // this row sees keys row_lo .. row_hi of the tile
            if constexpr (Q8) {
                // the row's 64 scores in registers, the mask by select (measured
                // faster for E4M3 queries only: the other modes spill more)
                tsm::softmax_tile_r<true>(s_addr, o_addr, p.score_scale, it > 0, edge, row_lo - key0, row_hi - key0,
                                          m, l);
            } else {
                if (edge)
                    mask_tile(s_addr, row_lo - key0, row_hi - key0);
                softmax_tile<FP8>(s_addr, o_addr, p.score_scale, it > 0, m, l);  // (P in f16 for both FP8 modes)
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.p_full[t][it % kStages]);
            if constexpr (FP8)  // the tile two ahead, while the tensor pipe runs PV and the next QK
                if (it + kStages - 1 < ntiles)
                    ok = widen(it + kStages - 1);
        }
        // ---- epilogue: O / l, lse = (m + log2 l) ln 2 ----
        if (ok && mbar_wait(&sm.o_done[t], 0, p.status)) {
            tc_fence_after();
            const float inv = l > 0.f ? (FP8 ? p.out_scale : 1.f) / l : 0.f;
            const int64_t orow = static_cast<int64_t>(q_beg + qi) * p.num_qo_heads + h;
            // The warp's 32 rows of O, in bf16, go through this head's Q tile
            // (every product that read it has completed) so that the global
            // stores are whole 128-byte rows: chunk c of row r sits at chunk
            // c ^ (r & 7), which keeps both the row-wise writes and the
            // chunk-wise reads free of bank conflicts.
            uint8_t *stage_o = sm.q[t] + quarter * 32 * 128;
#pragma unroll
            for (int c = 0; c < kHeadDim / 32; ++c) {  // 32 columns of O at a time
                uint32_t ov[32];
                tmem_ld32(o_addr + 32 * c, ov);
                tmem_ld_wait();
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                    uint4 w;
                    w.x = pack_bf16(__uint_as_float(ov[8 * v4 + 0]) * inv, __uint_as_float(ov[8 * v4 + 1]) * inv);
                    w.y = pack_bf16(__uint_as_float(ov[8 * v4 + 2]) * inv, __uint_as_float(ov[8 * v4 + 3]) * inv);
                    w.z = pack_bf16(__uint_as_float(ov[8 * v4 + 4]) * inv, __uint_as_float(ov[8 * v4 + 5]) * inv);
                    w.w = pack_bf16(__uint_as_float(ov[8 * v4 + 6]) * inv, __uint_as_float(ov[8 * v4 + 7]) * inv);
                    *reinterpret_cast<uint4 *>(stage_o + lane * 128 + (((4 * c + v4) ^ (lane & 7)) << 4)) = w;
                }
            }
            __syncwarp();
            // eight lanes per row, four rows per store
            const int ch = lane & 7;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = 4 * i + (lane >> 3);
                const int qr = q0 + quarter * 32 + r;
                const uint4 w = *reinterpret_cast<const uint4 *>(stage_o + r * 128 + ((ch ^ (r & 7)) << 4));
                if (qr < Lq)
                    reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                              (static_cast<int64_t>(q_beg + qr) * p.num_qo_heads + h) * kHeadDim)[ch] = w;
            }
            if (qi < Lq && p.lse)
                p.lse[orow] = l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
        }
    }

    // ---- teardown: every TMEM access is done before the columns are freed ----
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool FP8>
size_t prefill_smem_bytes()
{
    return sizeof(PrefillSmem<FP8>) + 1024;  // + slack for the 1 KB alignment
}

template <bool FP8, bool Q8, int NH>
cudaError_t launch_of(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p,
                      cudaStream_t stream)
{
    static std::atomic<int> done[kMaxDevices];  // one cudaFuncSetAttribute per device and variant
    const cudaError_t e = once_per_device(done, [] {
        return cudaFuncSetAttribute(prefill_kernel<FP8, Q8, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(prefill_smem_bytes<FP8>()));
    });
    if (e != cudaSuccess)
        return e;
    const dim3 grid(p.num_qo_heads / p.heads_per_cta, p.num_q_tiles, p.batch);
    return launch_pdl(prefill_kernel<FP8, Q8, NH>, grid, dim3(kThreads), prefill_smem_bytes<FP8>(), stream, tq, tk, tv, p);
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const PrefillParams &p, bool fp8, bool q8, cudaStream_t stream)
{
    const bool pair = p.heads_per_cta == 2;
    if (q8)
        return pair ? launch_of<true, true, 2>(tq, tk, tv, p, stream) : launch_of<true, true, 1>(tq, tk, tv, p, stream);
    if (fp8)
        return pair ? launch_of<true, false, 2>(tq, tk, tv, p, stream)
                    : launch_of<true, false, 1>(tq, tk, tv, p, stream);
    return pair ? launch_of<false, false, 2>(tq, tk, tv, p, stream) : launch_of<false, false, 1>(tq, tk, tv, p, stream);
}

}  // namespace sa
