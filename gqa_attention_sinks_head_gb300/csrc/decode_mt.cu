// decode_mt.cu -- multi-token decode (2..8 query tokens per sequence) on tcgen05.
//
// A speculative or multi-token-prediction decoder ("GPT-OSS on day 0"
// (Perplexity), the engine's speculative and MTP decoders) sends q_len new
// tokens per sequence; token k of sequence b sits at position L_b - q_len + k
// and sees the keys up to its own position (and, with a window, the last
// `window` of them).
//
// One thread block per (KV chunk, kv head g, sequence b), as in the one-token
// decode, two blocks per SM.  The q_len tokens x G query heads of the group
// (R = q_len G <= 64 rows; row r: token r / G, head r % G) are the rows of a
// 128-row tensor-core tile, so each K/V byte the block reads serves all of
// them: S = Q K^T and O += P V run as tcgen05.mma with the accumulators in
// tensor memory, as in the prefill kernel.  The tile holds Q twice, at rows
// 0 and 64 (the rest zeros): the padding costs tensor-pipe time but no memory
// traffic, and the kernel is bound by the HBM stream of the cache.
//
// The chunk's keys are walked in 64-key tiles, alternately by two streams
// (even and odd tiles), each with its own S and O in TMEM and its own softmax
// state, so that one stream's softmax overlaps the other's products.  Stream
// s reads its rows from the copy of Q at tile row 64 s, so its softmax warps
// (TMEM lanes 64 s ..) run on other SM sub-partitions than the other stream's:
//
//   TMEM columns   0..63  S_0 / P_0    64..127  O_0
//                128..191 S_1 / P_1   192..255  O_1
//
// The MMA warp issues, per tile j of stream s = j % 2: P V(j) once P(j) is in
// TMEM, then at once Q K^T(j + 2) into the same S columns.  The tensor pipe
// runs one thread's MMAs in order, so the commit that reports S(j + 2) also
// proves that P V(j) read P(j) and finished writing O_s, and the softmax may
// rescale O_s.  That one commit per round, on the barrier of the ring stage
// both products read, also frees the stage for the producers.  At the end the two streams' states merge (common max,
// rescaled sums and outputs) into the block's result: the final bf16 output
// and lse, or a sink-free partial state for sa_merge_states; stream 1 hands
// its scaled O rows to stream 0 through shared memory.
//
// Warp roles (320 threads):
//   warps 0, 1, 6, 7  softmax, one thread per row: warp w reads TMEM lanes
//              32 (w % 4) .. + 31; stream 0 uses warps 0 .. nq-1 (lanes 0 ..),
//              stream 1 warps 6 .. 5+nq (lanes 64 ..), nq = ceil(R / 32) <= 2
//   warps 2-5  producers: K and V tiles through a 5-stage ring, two 16-key
//              boxes per warp and step (a 16-key box never straddles a page),
//              page-table entries read 32 boxes ahead.  Step i of the ring
//              carries K of tile i and V of tile i - 2: the pair that one round
//              of the MMA warp (P V(j), Q K^T(j + 2)) uses
//   warp 8     the two copies of Q, once (one TMA box of G heads x q_len tokens each)
//   warp 9     MMA issuer; also zeroes the rows of the last V tile that lie
//              past the chunk (the cache may hold anything, NaN included,
//              past the sequence end, and 0 * NaN is NaN)
//
// Softmax: the per-row online softmax of the prefill kernel (running max m
// in base 2, moved only when a tile's max exceeds it by more than 8; sum l),
// seeded at the head's sink ("GPT-OSS on day 0", section "Sink Attention":
// m = sink log2 e, l = 1) in stream 0 of an unsplit call only, so that the
// sink enters the denominator once.
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>

#include "sa_internal.h"
#include "sa_ptx.cuh"
#include "tmem_softmax.cuh"

namespace sa {
namespace {

constexpr int kRows = 128;                              // tensor-core tile rows (M)
constexpr int kKeys = tsm::kCols;                       // keys per tile (N of Q K^T)
constexpr int kStages = 5;                              // K/V ring depth
constexpr int kThreads = 320;
constexpr int kFirstProducerWarp = 2;  // warps 2-5 (free: the softmax warps are 0, 1, 6, 7)
constexpr int kProducerWarps = 4;
constexpr int kQWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kQBytes = kRows * kHeadDim * 2;      // 16 KB
constexpr uint32_t kTileBytes = kKeys * kHeadDim * 2;   // 8 KB
constexpr uint32_t kBoxBytes = 16 * kHeadDim * 2;       // one 16-key box
constexpr uint32_t kTmemCols = 256;
constexpr int kMaxOrderedBatch = 128;  // batches up to this size run longest sequence first
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;
// Q, K K-major; V MN-major (dims contiguous); bf16 operands, fp32 accumulators
constexpr uint32_t kIdescQK = idesc_f32acc(kRows, kKeys, 0);
constexpr uint32_t kIdescPV = idesc_f32acc(kRows, kHeadDim, 1);
__host__ __device__ constexpr uint32_t col_s(int s) { return 128u * s; }        // S_s / P_s
__host__ __device__ constexpr uint32_t col_o(int s) { return 128u * s + 64u; }  // O_s

struct MtSmem {
    uint8_t q[kQBytes];  // 1 KB aligned, like every tile below
    uint8_t k[kStages][kTileBytes];
    uint8_t v[kStages][kTileBytes];
    float xm[2][kRows / 2], xl[2][kRows / 2];  // each stream's row states, for the merge
    uint64_t q_full;
    uint64_t full[kStages];   // the step's K and V tiles have landed
    uint64_t done[kStages];   // the step's products have completed: its stage is free, and S of its tile is in TMEM
    uint64_t p_full[2];          // per stream: P of its current tile is in TMEM
    uint64_t o_done;             // every product has completed
    uint32_t tmem_base;
    int32_t seq;                       // the sequence this block serves
    int32_t lens[kMaxOrderedBatch];    // scratch: the batch's lengths, for the ordering
};
constexpr size_t kSmemBytes = sizeof(MtSmem) + 1024;  // + slack for the 1 KB alignment
static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two blocks must fit one SM's shared memory");

__device__ __forceinline__ void kv_coords(const DecodeParams &p, int slot, int g, int page, int &c1, int &c2,
                                          int &c3)
{
    c1 = p.dim_token == 1 ? slot : (p.dim_head == 1 ? g : page);
    c2 = p.dim_token == 2 ? slot : (p.dim_head == 2 ? g : page);
    c3 = p.dim_token == 3 ? slot : (p.dim_head == 3 ? g : page);
}

__global__ void __launch_bounds__(kThreads, 2)
    decode_mt_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    MtSmem &sm = *reinterpret_cast<MtSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // launched as a programmatic dependent: the grid before it has finished
    // (and its writes are visible) before any global access below
    griddep_wait();
    griddep_launch_dependents();  // the next grid (a merge, the next call) may be scheduled
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int g = blockIdx.y;
    // Longest sequences first: block z serves the sequence of rank z in
    // decreasing length (ties by index).  The blocks of a ragged batch then
    // start in that order, so no long one starts last and runs alone at the
    // end (list scheduling, longest job first).  Only unsplit calls: split
    // chunks are of equal length already, and a windowed call gives every
    // sequence the same keys.
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
    const int qlen = p.q_len;
    const int G = p.group;
    const int R = qlen * G;            // live rows of the tile
    const int nq = (R + 31) >> 5;      // softmax warps per stream (1 or 2)
    const int h0 = g * G;

    // ---- the block's key range: the union over its query tokens (as in the
    // one-token kernel: chunks of tiles_per_split 16-key tiles from the first
    // key of token 0, rounded down to 16) --------------------------------------
    int L = __ldg(p.seqlens + b);
    if (L < 0 || L > p.max_kv_len) {
        if (threadIdx.x == 0)
            atomicOr(p.status, SA_DEVICE_SEQLEN_RANGE);
        L = min(max(L, 0), p.max_kv_len);
    }
    if (L > 0 && L < qlen && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
        atomicOr(p.status, SA_DEVICE_BAD_QLEN);  // tokens at negative positions see no key (L = 0: empty slot)
    const int lo = p.window > 0 ? max(0, L - qlen + 1 - p.window) : 0;
    const int t_begin = (lo & ~(kTile - 1)) + kTile * p.tiles_per_split * split;
    const int t_first = max(t_begin, lo);
    const int t_end = min(L, t_begin + kTile * p.tiles_per_split);
    const int ntiles = t_end > t_first ? (t_end - t_begin + kKeys - 1) / kKeys : 0;
    const int nsteps = ntiles > 0 ? ntiles + 2 : 0;  // producer steps (below)

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.full[i], kProducerWarps);
            mbar_init(&sm.done[i], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sm.p_full[s], nq);
        }
        mbar_init(&sm.o_done, 1);
        fence_barrier_init();
    }
    // rows R .. 63 and 64 + R .. 127 of the Q tile are zeros (the two TMA
    // boxes fill rows 0 .. R-1 and 64 .. 63+R)
    for (int i = threadIdx.x; i < kRows * (kHeadDim / 8); i += kThreads)
        if ((i >> 3) % (kRows / 2) >= R)
            reinterpret_cast<uint4 *>(sm.q)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // generic writes -> tensor-core reads
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    const int quarter = warp & 3;
    const int s = warp >> 2;         // softmax warps: stream
    const int qd = quarter - 2 * s;  // softmax warps: quadrant within the stream's copy of Q
    const bool softmax_warp = warp < 8 && qd >= 0 && qd < nq;
    const int row = qd * 32 + lane;  // softmax warps: this thread's row
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float m = -INFINITY, l = 0.f;    // softmax warps: the row's running state

    if (warp == kQWarp) {
        // ============================ Q ===================================
        if (lane == 0) {
            tma_prefetch_desc(&tmq);
            if (ntiles > 0) {
                mbar_arrive_expect_tx(&sm.q_full, 2u * static_cast<uint32_t>(R) * kHeadDim * 2);
                tma_load_3d(sm.q, &tmq, &sm.q_full, 0, h0, b * qlen);
                tma_load_3d(sm.q + kQBytes / 2, &tmq, &sm.q_full, 0, h0, b * qlen);
            }
        }
    } else if (warp >= kFirstProducerWarp && warp < kFirstProducerWarp + kProducerWarps) {
        // ============================ producers ===========================
        // Producer warp pw issues two 16-key boxes of each step (lanes 0, 1):
        // boxes 2 (pw & 1) .. + 1 of the step's K tile (pw < 2) or V tile.
        // Four warps issue side by side: one warp's copies go out one after
        // another, and eight per step from one warp fall behind the HBM stream.
        const int pw = warp - kFirstProducerWarp;
        const int is_v = pw >> 1, bi = 2 * (pw & 1) + lane;
        if (lane == 0)
            tma_prefetch_desc(is_v ? &tmv : &tmk);
        const int32_t *trow = p.page_table ? p.page_table + static_cast<int64_t>(b) * p.table_stride : nullptr;
        auto nbox_of = [&](int j) { return min(kKeys / 16, (t_end - (t_begin + j * kKeys) + 15) / 16); };
        // Page-table entries: lane i holds the page of 16-key box 32 k + i of
        // the chunk while the tiles of boxes 32 k .. 32 k + 31 are issued, and
        // the next 32 are already on their way (a table read from HBM takes
        // longer than a tile's turn)
        auto box_page = [&](int u) -> int {
            const int key = t_begin + 16 * u;
            if (key >= t_end)
                return 0;
            return trow ? __ldg(trow + key / p.page_size) : b;
        };
        // this warp's tile of step i: K of tile i, or V of tile i - 2
        const int lag = is_v ? 2 : 0;
        int pg_cur = box_page(lane), pg_next = box_page(32 + lane);
        const uint64_t pol = l2_policy_evict_first();  // each cache byte is read once
        uint8_t *const base = is_v ? &sm.v[0][0] : &sm.k[0][0];
        const CUtensorMap *map = is_v ? &tmv : &tmk;
        int issued = 0;
        for (int i = 0; i < nsteps; ++i) {
            // step i: K of tile i and V of tile i - 2, the pair one MMA round uses
            const int stage = i % kStages;
            const int t = i - lag;
            const int nb = t >= 0 && t < ntiles ? max(0, min(2, nbox_of(t) - 2 * (pw & 1))) : 0;
            const int u = (kKeys / 16) * max(t, 0);  // the tile's first box
            if (t > 0 && (u & 31) == 0) {
                pg_cur = pg_next;
                pg_next = box_page(u + 32 + lane);
            }
            const int page = __shfl_sync(0xffffffffu, pg_cur, (u & 31) + (bi & 3));
            // the stage's previous step i - kStages: its products have completed
            if (i >= kStages && !mbar_wait(&sm.done[stage], ((i / kStages) - 1) & 1, p.status))
                break;
            const bool mine = lane < nb;
            int c1 = 0, c2 = 0, c3 = 0;
            if (mine) {
                if (page < 0 || page >= p.num_pages)
                    atomicOr(p.status, SA_DEVICE_BAD_PAGE);  // the TMA box falls outside: zeros
                kv_coords(p, (t_begin + t * kKeys + 16 * bi) % p.page_size, g, page, c1, c2, c3);
            }
            if (lane == 0)
                mbar_arrive_expect_tx(&sm.full[stage], static_cast<uint32_t>(nb) * kBoxBytes);
            __syncwarp();
            if (mine)
                tma_load_4d_hint(base + stage * kTileBytes + bi * kBoxBytes, map, &sm.full[stage], 0, c1, c2, c3,
                                 pol);
            issued = i + 1;
        }
        // every copy this block started has landed before it may exit (the
        // consumers wait for them too, unless they stopped on an error)
        for (int i = max(0, issued - kStages); i < issued; ++i)
            if (!mbar_wait(&sm.full[i % kStages], (i / kStages) & 1, p.status))
                break;
    } else if (warp == kMmaWarp) {
        // ============================ MMA issuer ==========================
        // Descriptor bases; a K step adds to the start-address field (bytes >> 4):
        // 32 bytes (16 dims) for Q/K, 2048 bytes (16 keys) for V.
        const uint64_t dq = smem_desc_sw128(smem_u32(sm.q), 16, 1024);
        const uint64_t dk0 = smem_desc_sw128(smem_u32(sm.k[0]), 16, 1024);
        const uint64_t dv0 = smem_desc_sw128(smem_u32(sm.v[0]), 16, 1024);
        auto issue_qk = [&](int s, int stage) {
            const uint64_t dk = dk0 + static_cast<uint64_t>(stage) * (kTileBytes >> 4);
#pragma unroll
            for (int ks = 0; ks < kHeadDim / 16; ++ks)
                umma_ss(tmem + col_s(s), dq + 2 * ks, dk + 2 * ks, kIdescQK, ks > 0 ? 1u : 0u);
        };
        auto issue_pv = [&](int s, int stage, bool accumulate) {
            const uint64_t dv = dv0 + static_cast<uint64_t>(stage) * (kTileBytes >> 4);
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk)  // K = 16 keys: 8 TMEM columns of P, 2 KB of V
                umma_ts(tmem + col_o(s), tmem + col_s(s) + 8 * kk, dv + 128 * kk, kIdescPV,
                        (accumulate || kk > 0) ? 1u : 0u);
        };
        bool ok = ntiles == 0 || mbar_wait(&sm.q_full, 0, p.status);
        // steps 0 and 1: the first tile of each stream (K only)
        for (int i = 0; ok && i < min(2, nsteps); ++i) {
            ok = mbar_wait(&sm.full[i], 0, p.status);
            if (!ok)
                break;
            tc_fence_after();
            if (lane == 0) {
                if (i < ntiles)
                    issue_qk(i, i);
                umma_commit(&sm.done[i]);
            }
            __syncwarp();
        }
        // round j: P V(j) and Q K^T(j + 2), both from step j + 2.  QK (compile
        // time): there is a tile j + 2; TAIL: the round's tile may reach past the
        // chunk (only the last one can).  The steady rounds carry neither test.
        // ring stage and phase of step j + 2, advanced round by round (no
        // division by the ring depth on the issue path)
        int stage = 2 % kStages, sphase = 0;
        auto round = [&](auto QK_, auto TAIL_, int j) -> bool {
            constexpr bool QK = decltype(QK_)::value, TAIL = decltype(TAIL_)::value;
            const int s = j & 1;
            const uint32_t ph = static_cast<uint32_t>(sphase);
            // P(j) and step i, checked together first; the bounded waits only
            // when one is missing
            const bool ready = mbar_try_wait2(&sm.p_full[s], (j >> 1) & 1, &sm.full[stage], ph);
            if (!ready && (!mbar_wait(&sm.p_full[s], (j >> 1) & 1, p.status) ||
                           !mbar_wait(&sm.full[stage], ph, p.status)))
                return false;
            if constexpr (TAIL) {
                const int key0 = t_begin + j * kKeys;
                if (key0 + kKeys > t_end) {
                    // value rows past the chunk: zeros, so that p = 0 contributes exactly 0
                    uint4 *vz = reinterpret_cast<uint4 *>(sm.v[stage]);
                    for (int e = (t_end - key0) * (kHeadDim / 8) + lane; e < kKeys * (kHeadDim / 8); e += 32)
                        vz[e] = make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();
                    __syncwarp();
                }
            }
            tc_fence_after();
            if (lane == 0) {
                issue_pv(s, stage, j >= 2);
                if constexpr (QK)
                    issue_qk(s, stage);
                umma_commit(&sm.done[stage]);  // frees step i and reports S(i)
            }
            __syncwarp();
            if (++stage == kStages) {
                stage = 0;
                sphase ^= 1;
            }
            return true;
        };
        for (int j = 0; ok && j + 2 < ntiles; ++j)
            ok = round(std::true_type{}, std::false_type{}, j);
        for (int j = max(0, ntiles - 2); ok && j < ntiles; ++j)
            ok = round(std::false_type{}, std::true_type{}, j);
        if (lane == 0)
            umma_commit(&sm.o_done);
        __syncwarp();
    } else if (softmax_warp) {
        // ============================ softmax =============================
        const uint32_t s_addr = tmem + lane_base + col_s(s);
        const uint32_t o_addr = tmem + lane_base + col_o(s);
        const bool live = row < R;
        const int tok = live ? row / G : 0;
        const int n = live ? row % G : 0;
        // keys [vlo, vhi) of the chunk are visible to the row's token; rows
        // past R see all (their results are not written)
        const int hi_k = L - qlen + tok + 1;  // one past the token's own position
        const int lo_k = p.window > 0 ? max(0, hi_k - p.window) : 0;
        const int vlo = live ? max(t_first, lo_k) : t_begin;
        const int vhi = live ? min(t_end, hi_k) : t_begin + ntiles * kKeys;
        if (s == 0 && !p.partial && p.sinks && live) {
            m = __ldg(p.sinks + h0 + n) * kLog2e;  // the running max starts at the sink ...
            l = 1.f;                               // ... and the sum at 1
        }
        for (int j = s; j < ntiles; j += 2) {
            // S(j): the products of step j (ring barriers complete in step
            // order, so the phase of step j - kStages is complete by now)
            if (!mbar_wait(&sm.done[j % kStages], (j / kStages) & 1, p.status))
                break;
            tc_fence_after();
            const int key0 = t_begin + j * kKeys;
            const bool edge = __any_sync(0xffffffffu, vlo > key0 || vhi < key0 + kKeys);
            tsm::softmax_tile_r<false>(s_addr, o_addr, p.score_scale, j >= 2, edge, vlo - key0, vhi - 1 - key0, m, l);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.p_full[s]);
        }
        sm.xm[s][row] = m;
        sm.xl[s][row] = l;
    }
    __syncthreads();  // both streams' row states are in shared memory

    // ---- epilogue: merge the two streams' states of each row, normalise ----
    // Stream 1 leaves its scaled O rows in shared memory (the K ring, free once
    // every product has completed); stream 0 adds its own and writes the row.
    constexpr int kXoStride = kHeadDim + 4;  // floats; the pad spreads the rows' banks
    float *xo = reinterpret_cast<float *>(&sm.k[0][0]);
    static_assert(sizeof(float) * (kRows / 2) * kXoStride <= sizeof(MtSmem::k), "O hand-off fits the K ring");
    const bool have0 = ntiles > 0, have1 = ntiles > 1;  // streams that wrote their O
    float a_s = 0.f, lse = -INFINITY;
    bool ok = true;
    if (softmax_warp) {
        const float m0 = sm.xm[0][row], l0 = sm.xl[0][row];
        const float m1 = sm.xm[1][row], l1 = sm.xl[1][row];
        const float M = fmaxf(m0, m1);
        const float f0 = m0 == -INFINITY ? 0.f : ex2(m0 - M);
        const float f1 = m1 == -INFINITY ? 0.f : ex2(m1 - M);
        const float Ls = l0 * f0 + l1 * f1;
        const float inv = Ls > 0.f ? p.out_scale / Ls : 0.f;
        lse = Ls > 0.f ? (M + lg2(Ls)) * kLn2 : -INFINITY;
        a_s = (s == 0 ? f0 : f1) * inv;
        if (have0) {
            ok = mbar_wait(&sm.o_done, 0, p.status);
            tc_fence_after();
        }
        if (s == 1 && have1) {
#pragma unroll
            for (int c = 0; c < kHeadDim / 16; ++c) {
                uint32_t o1[16];
                tmem_ld16(tmem + lane_base + col_o(1) + 16 * c, o1);
                tmem_ld_wait();
                float4 *dst = reinterpret_cast<float4 *>(xo + row * kXoStride + 16 * c);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_float4(__uint_as_float(o1[4 * i]) * a_s, __uint_as_float(o1[4 * i + 1]) * a_s,
                                         __uint_as_float(o1[4 * i + 2]) * a_s, __uint_as_float(o1[4 * i + 3]) * a_s);
            }
        }
    }
    __syncthreads();  // stream 1's O rows are in shared memory

    if (softmax_warp && s == 0) {
        const bool live = row < R && ok;
        const int tok = row / G, n = row % G;
        const int64_t qrow = static_cast<int64_t>(b) * qlen + tok;
        const int h = h0 + n;
#pragma unroll
        for (int c = 0; c < kHeadDim / 16; ++c) {  // 16 dims at a time
            uint32_t o0[16];
            if (have0) {
                tmem_ld16(tmem + lane_base + col_o(0) + 16 * c, o0);
                tmem_ld_wait();
            }
            float v[16];
            const float4 *x1 = reinterpret_cast<const float4 *>(xo + row * kXoStride + 16 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 w = have1 ? x1[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                v[4 * i + 0] = (have0 ? __uint_as_float(o0[4 * i + 0]) * a_s : 0.f) + w.x;
                v[4 * i + 1] = (have0 ? __uint_as_float(o0[4 * i + 1]) * a_s : 0.f) + w.y;
                v[4 * i + 2] = (have0 ? __uint_as_float(o0[4 * i + 2]) * a_s : 0.f) + w.z;
                v[4 * i + 3] = (have0 ? __uint_as_float(o0[4 * i + 3]) * a_s : 0.f) + w.w;
            }
            if (live) {
                if (p.partial) {
                    const int64_t prow = (static_cast<int64_t>(split) * p.batch * qlen + qrow) * p.num_qo_heads + h;
                    float4 *dst = reinterpret_cast<float4 *>(p.o_part + prow * kHeadDim + 16 * c);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                } else {
                    const int64_t orow = qrow * p.num_qo_heads + h;
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + orow * kHeadDim +
                                                           16 * c);
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        dst[i] = make_uint4(pack_bf16(v[8 * i], v[8 * i + 1]), pack_bf16(v[8 * i + 2], v[8 * i + 3]),
                                            pack_bf16(v[8 * i + 4], v[8 * i + 5]),
                                            pack_bf16(v[8 * i + 6], v[8 * i + 7]));
                }
            }
        }
        if (live) {
            if (p.partial)
                p.lse_part[(static_cast<int64_t>(split) * p.batch * qlen + qrow) * p.num_qo_heads + h] = lse;
            else if (p.lse)
                p.lse[qrow * p.num_qo_heads + h] = lse;
        }
    }

    // ---- teardown: every TMEM access is done before the columns are freed ----
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

namespace {

cudaError_t prepare_decode_mt()
{
    static std::atomic<int> done[kMaxDevices];  // one cudaFuncSetAttribute per device
    return once_per_device(done, [] {
        return cudaFuncSetAttribute(decode_mt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmemBytes));
    });
}

}  // namespace

// Blocks per SM: the launch bounds reserve registers for two, so shared
// memory decides (two blocks resident, as measured on GB300;
// cudaOccupancyMaxActiveBlocksPerMultiprocessor reports one for this kernel).
cudaError_t decode_mt_occupancy(int *blocks_per_sm)
{
    int dev = 0, smem_sm = 0, reserved = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess)
        return e;
    *blocks_per_sm = std::min(2, smem_sm / static_cast<int>(kSmemBytes + reserved));
    return cudaSuccess;
}

cudaError_t launch_decode_mt(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const DecodeParams &p, cudaStream_t stream)
{
    const cudaError_t e = prepare_decode_mt();
    if (e != cudaSuccess)
        return e;
    const dim3 grid(p.num_splits, p.num_kv_heads, p.batch);
    return launch_pdl(decode_mt_kernel, grid, dim3(kThreads), kSmemBytes, stream, tq, tk, tv, p);
}

}  // namespace sa
