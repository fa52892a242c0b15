// api.cu -- the C ABI of libsinkattn (see include/sink_attn.h).
//
// Host-side argument validation (before any launch), the split-KV heuristic,
// TMA tensor-map encoding (cuTensorMapEncodeTiled through the runtime's
// driver entry point, so the library links no libcuda), and the device status
// word.  Every call only queues work on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/sink_attn.h"
#include "sa_internal.h"

namespace {

thread_local char g_err[512] = {0};

sa_status_t fail(sa_status_t st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

sa_status_t cuda_fail(cudaError_t e, const char *what)
{
    return fail(SA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- status word
__device__ uint32_t g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t *g_status_ptr[kMaxDevices] = {nullptr};
int g_sm_count[kMaxDevices] = {0};
int g_bps[3][kMaxDevices] = {{0}};  // blocks per SM: decode bf16, decode fp8, multi-token tcgen05

cudaError_t status_ptr(uint32_t **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess)
            return e;
        g_status_ptr[dev] = static_cast<uint32_t *>(p);
    }
    *out = g_status_ptr[dev];
    return cudaSuccess;
}

// SM count and the occupancy of a decode kernel (kind: 0 the one-token bf16
// kernel, 1 its FP8 build, 2 the multi-token tcgen05 kernel) on the current
// device (cached).
bool device_shape(int kind, int *sms, int *bps)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            return false;
        }
        g_sm_count[dev] = n;
    }
    if (!g_bps[kind][dev]) {
        int b = 0;
        const cudaError_t e = kind == 2 ? sa::decode_mt_occupancy(&b) : sa::decode_occupancy(kind == 1, &b);
        if (e != cudaSuccess || b <= 0) {
            cudaGetLastError();
            b = 1;
        }
        g_bps[kind][dev] = b;
    }
    *sms = g_sm_count[dev];
    *bps = g_bps[kind][dev];
    return true;
}

// ---------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
    });
    return fn;
}

// A 4-d map over one KV tensor: dim 0 = head_dim, dims 1..3 = token/head/page
// ordered by increasing stride.  Box: all of head_dim x `rows` tokens.
// dim_*: which map dimension carries each coordinate.
sa_status_t encode_kv_map(CUtensorMap *map, const void *base, bool fp8, const sa_kv_desc_t *kv, int rows,
                          int *dim_token, int *dim_head, int *dim_page)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return fail(SA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int64_t esz = fp8 ? 1 : 2;
    struct Ax {
        int64_t stride;
        int64_t extent;
        int kind;  // 0 token, 1 head, 2 page
    } ax[3] = {{kv->stride_token, kv->page_size, 0}, {kv->stride_head, kv->num_kv_heads, 1},
               {kv->stride_page, kv->num_pages, 2}};
    std::stable_sort(ax, ax + 3, [](const Ax &a, const Ax &b) { return a.stride < b.stride; });
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(kv->head_dim), 0, 0, 0};
    cuuint64_t strides[3];
    cuuint32_t box[4] = {static_cast<cuuint32_t>(kv->head_dim), 1, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    for (int i = 0; i < 3; ++i) {
        dims[i + 1] = static_cast<cuuint64_t>(ax[i].extent);
        strides[i] = static_cast<cuuint64_t>(ax[i].stride * esz);
        if (ax[i].kind == 0) {
            box[i + 1] = static_cast<cuuint32_t>(rows);
            *dim_token = i + 1;
        } else if (ax[i].kind == 1) {
            *dim_head = i + 1;
        } else {
            *dim_page = i + 1;
        }
    }
    CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                    const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    fp8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(SA_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled rejected the KV layout (CUresult %d)", (int)r);
    return SA_OK;
}

// ---------------------------------------------------------------- validation
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sa_status_t check_kv(const sa_kv_desc_t *kv, int32_t batch, int32_t num_qo_heads, int32_t max_kv_len)
{
    if (!kv)
        return fail(SA_ERR_INVALID_ARG, "kv descriptor is NULL");
    if (!kv->k || !kv->v)
        return fail(SA_ERR_INVALID_ARG, "kv->k / kv->v is NULL");
    if (kv->dtype != SA_KV_BF16 && kv->dtype != SA_KV_FP8_E4M3)
        return fail(SA_ERR_INVALID_ARG, "kv->dtype %d is not a sa_kv_dtype_t", (int)kv->dtype);
    if (kv->num_kv_heads <= 0 || kv->num_pages <= 0 || kv->page_size <= 0 || kv->head_dim <= 0)
        return fail(SA_ERR_INVALID_ARG, "kv sizes must be positive (heads %d, pages %d, page_size %d, dim %d)",
                    kv->num_kv_heads, kv->num_pages, kv->page_size, kv->head_dim);
    if (num_qo_heads <= 0 || num_qo_heads % kv->num_kv_heads != 0)
        return fail(SA_ERR_INVALID_ARG, "num_qo_heads %d is not a positive multiple of num_kv_heads %d",
                    num_qo_heads, kv->num_kv_heads);
    if (kv->head_dim != sa::kHeadDim)
        return fail(SA_ERR_UNSUPPORTED, "head_dim %d: only 64 is supported", kv->head_dim);
    if (num_qo_heads / kv->num_kv_heads > sa::kMaxGroup)
        return fail(SA_ERR_UNSUPPORTED, "%d query heads per kv head: at most %d are supported",
                    num_qo_heads / kv->num_kv_heads, sa::kMaxGroup);
    if (kv->page_size % 16 != 0)
        return fail(SA_ERR_UNSUPPORTED, "page_size %d is not a multiple of 16", kv->page_size);
    if (kv->num_kv_heads > 65535)
        return fail(SA_ERR_UNSUPPORTED, "more than 65535 kv heads");
    if (!aligned16(kv->k) || !aligned16(kv->v))
        return fail(SA_ERR_UNSUPPORTED, "kv->k / kv->v must be 16-byte aligned");
    const int64_t esz = kv->dtype == SA_KV_FP8_E4M3 ? 1 : 2;
    const int64_t st[3] = {kv->stride_page, kv->stride_head, kv->stride_token};
    for (int i = 0; i < 3; ++i) {
        if (st[i] <= 0)
            return fail(SA_ERR_INVALID_ARG, "kv strides must be positive");
        if ((st[i] * esz) % 16 != 0 || st[i] * esz >= (int64_t(1) << 40))
            return fail(SA_ERR_UNSUPPORTED, "kv stride %lld elements is not a multiple of 16 bytes below 2^40",
                        (long long)st[i]);
    }
    if (kv->dtype == SA_KV_FP8_E4M3 &&
        (!std::isfinite(kv->k_scale) || !std::isfinite(kv->v_scale) || kv->k_scale == 0.f))
        return fail(SA_ERR_INVALID_ARG, "FP8 scales must be finite (k_scale nonzero)");
    const int64_t need = (static_cast<int64_t>(max_kv_len) + kv->page_size - 1) / kv->page_size;
    if (kv->page_table) {
        if (kv->page_table_stride < need)
            return fail(SA_ERR_INVALID_ARG, "page_table_stride %d < ceil(max_kv_len / page_size) = %lld",
                        kv->page_table_stride, (long long)need);
    } else {
        if (kv->num_pages < batch || kv->page_size < max_kv_len)
            return fail(SA_ERR_INVALID_ARG,
                        "without a page table sequence b uses page b: need num_pages >= batch and "
                        "page_size >= max_kv_len");
    }
    return SA_OK;
}

int32_t eff_tiles(int32_t max_kv_len, int32_t window, int32_t q_len = 1)
{
    if (max_kv_len <= 0)
        return 0;
    if (window > 0)  // the q_len tokens' windows span window + q_len - 1 keys, not tile-aligned
        return (std::min(window + q_len - 1, max_kv_len) + 15 + sa::kTile - 1) / sa::kTile;
    return (max_kv_len + sa::kTile - 1) / sa::kTile;
}

constexpr int kMaxSplits = 256;

// Pick the chunk count that minimises (waves of blocks) x (tiles per block
// + a fixed per-block cost), over the SM count times resident blocks per SM.
// overhead_tiles: a block's fixed cost in 16-key tiles (8 for the one-token
// kernel; the tcgen05 multi-token block, with its TMEM allocation, Q load,
// pipeline fill and two-stream merge, costs about 64).
int32_t choose_splits(int32_t batch, int32_t hkv, int32_t max_kv_len, int32_t window, int sms, int bps,
                      double overhead_tiles = 8.0)
{
    const int32_t tiles = eff_tiles(max_kv_len, window);
    if (tiles <= 1 || batch <= 0)
        return 1;
    const double kOverheadTiles = overhead_tiles;
    // A chunk of fewer than 32 tiles (512 keys) costs more in its fixed block
    // setup and in the merge (one more partial per row) than it saves: measured
    // on GB300 for B = 1..4, L = 256..8192 with the calls replayed from a graph.
    constexpr int32_t kMinTilesPerChunk = 32;
    const int64_t units = static_cast<int64_t>(batch) * hkv;
    const int64_t slots = static_cast<int64_t>(std::max(1, sms)) * std::max(1, bps);
    int32_t best = 1;
    double best_cost = 1e300;
    const int32_t smax = std::max<int32_t>(
        1, std::min<int32_t>(std::min<int32_t>(kMaxSplits, tiles / kMinTilesPerChunk), 65535));
    for (int32_t s = 1; s <= smax; ++s) {
        const int64_t per = (tiles + s - 1) / s;
        const int64_t waves = (units * s + slots - 1) / slots;
        const double cost = static_cast<double>(waves) * (static_cast<double>(per) + kOverheadTiles);
        if (cost < best_cost * 0.98) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t partial_bytes(int32_t S, int32_t batch, int32_t hq, int32_t dim)
{
    const size_t rows = static_cast<size_t>(S) * batch * hq;
    return align256(rows * dim * sizeof(float)) + align256(rows * sizeof(float));
}

sa_status_t check_decode_common(const void *q, const sa_kv_desc_t *kv, const int32_t *seqlens, int32_t batch,
                                int32_t num_qo_heads, int32_t max_kv_len, int32_t window, float sm_scale)
{
    if (batch < 0 || max_kv_len < 0 || window < 0)
        return fail(SA_ERR_INVALID_ARG, "batch, max_kv_len and window must be >= 0");
    if (batch > 65535)
        return fail(SA_ERR_UNSUPPORTED, "batch %d > 65535", batch);
    if (!std::isfinite(sm_scale))
        return fail(SA_ERR_INVALID_ARG, "sm_scale must be finite");
    sa_status_t st = check_kv(kv, batch, num_qo_heads, max_kv_len);
    if (st != SA_OK)
        return st;
    if (batch > 0 && (!q || !seqlens))
        return fail(SA_ERR_INVALID_ARG, "q / seqlens is NULL");
    if (q && !aligned16(q))
        return fail(SA_ERR_UNSUPPORTED, "q must be 16-byte aligned");
    return SA_OK;
}

sa_status_t launch_decode_kernel(const void *q, int32_t q_len, const sa_kv_desc_t *kv, const int32_t *seqlens,
                                 int32_t batch, int32_t num_qo_heads, int32_t max_kv_len, const float *sinks,
                                 int32_t window, float sm_scale, void *out, float *lse, float *o_part,
                                 float *lse_part, int32_t S, bool partial, cudaStream_t stream)
{
    const bool fp8 = kv->dtype == SA_KV_FP8_E4M3;
    sa::DecodeParams p;
    std::memset(&p, 0, sizeof p);
    CUtensorMap tk, tv;
    int dt = 0, dh = 0, dp = 0;
    sa_status_t st = encode_kv_map(&tk, kv->k, fp8, kv, sa::kTile, &dt, &dh, &dp);
    if (st != SA_OK)
        return st;
    st = encode_kv_map(&tv, kv->v, fp8, kv, sa::kTile, &dt, &dh, &dp);
    if (st != SA_OK)
        return st;
    uint32_t *status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess)
        return cuda_fail(e, "device status word");
    const float kLog2e = 1.44269504088896340736f;
    p.q = q;
    p.seqlens = seqlens;
    p.page_table = kv->page_table;
    p.sinks = sinks;
    p.out = out;
    p.lse = lse;
    p.o_part = o_part;
    p.lse_part = lse_part;
    p.status = status;
    p.batch = batch;
    p.num_qo_heads = num_qo_heads;
    p.num_kv_heads = kv->num_kv_heads;
    p.group = num_qo_heads / kv->num_kv_heads;
    p.q_len = q_len;
    p.page_size = kv->page_size;
    p.table_stride = kv->page_table_stride;
    p.num_pages = kv->num_pages;
    p.max_kv_len = max_kv_len;
    p.window = window;
    p.num_splits = S;
    p.tiles_per_split = std::max<int32_t>(1, (eff_tiles(max_kv_len, window, q_len) + S - 1) / S);
    p.partial = partial ? 1 : 0;
    p.dim_token = dt;
    p.dim_head = dh;
    p.dim_page = dp;
    p.score_scale = sm_scale * kLog2e * (fp8 ? kv->k_scale : 1.f);  // FP8: codes widen to their values
    p.out_scale = fp8 ? kv->v_scale : 1.f;
    if (q_len > 1 && !fp8 && q_len * p.group <= 64) {
        // several tokens on a bf16 cache: the tcgen05 kernel, whose Q tile is
        // one TMA box of the group's heads x the sequence's q_len tokens
        EncodeTiledFn fn = encode_fn();
        if (!fn)
            return fail(SA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        CUtensorMap tq;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(sa::kHeadDim), static_cast<cuuint64_t>(num_qo_heads),
                                    static_cast<cuuint64_t>(batch) * static_cast<cuuint64_t>(q_len)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(sa::kHeadDim) * 2,
                                       static_cast<cuuint64_t>(num_qo_heads) * sa::kHeadDim * 2};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(sa::kHeadDim), static_cast<cuuint32_t>(p.group),
                                   static_cast<cuuint32_t>(q_len)};
        const cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = fn(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(SA_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled rejected q (CUresult %d)", (int)r);
        e = sa::launch_decode_mt(tq, tk, tv, p, stream);
        if (e != cudaSuccess)
            return cuda_fail(e, "multi-token decode launch");
        return SA_OK;
    }
    e = sa::launch_decode(tk, tv, p, fp8, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode launch");
    return SA_OK;
}

}  // namespace

sa_status_t sa::set_last_error(sa_status_t st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

extern "C" {

const char *sa_status_string(sa_status_t s)
{
    switch (s) {
    case SA_OK: return "SA_OK";
    case SA_ERR_INVALID_ARG: return "SA_ERR_INVALID_ARG";
    case SA_ERR_UNSUPPORTED: return "SA_ERR_UNSUPPORTED";
    case SA_ERR_WORKSPACE: return "SA_ERR_WORKSPACE";
    case SA_ERR_CUDA: return "SA_ERR_CUDA";
    case SA_ERR_TIMEOUT: return "SA_ERR_TIMEOUT";
    }
    return "unknown sa_status_t";
}

const char *sa_last_error(void) { return g_err; }

int sa_version(void) { return SA_VERSION; }

int32_t sa_decode_num_splits(int32_t batch, int32_t num_kv_heads, int32_t max_kv_len, int32_t window)
{
    int sms = 0, bps = 0;
    if (!device_shape(0, &sms, &bps)) {
        sms = 152;  // no device visible: size for a GB300
        bps = 4;
    }
    return choose_splits(batch, std::max(1, num_kv_heads), max_kv_len, window, sms, bps);
}

int32_t sa_decode_multi_num_splits(int32_t batch, int32_t q_len, int32_t num_kv_heads, int32_t max_kv_len,
                                   int32_t window, int32_t kv_dtype)
{
    if (q_len <= 1 || kv_dtype != SA_KV_BF16)  // the one-token kernel's blocks
        return sa_decode_num_splits(batch, num_kv_heads, max_kv_len, window);
    int sms = 0, bps = 0;
    if (!device_shape(2, &sms, &bps)) {
        sms = 152;
        bps = 2;
    }
    // measured on GB300 (B = 64, L ~ U[1024, 8192], q_len 4): 1 chunk 111 us,
    // 2 chunks 125 us, 4 chunks 146 us
    return choose_splits(batch, std::max(1, num_kv_heads), max_kv_len, window, sms, bps, 64.0);
}

size_t sa_decode_workspace_size(int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t max_kv_len, int32_t window, int32_t num_splits)
{
    if (batch <= 0 || num_qo_heads <= 0 || head_dim <= 0 || num_splits < 0)
        return 0;
    const int32_t S = num_splits == 0 ? sa_decode_num_splits(batch, num_kv_heads, max_kv_len, window) : num_splits;
    return S <= 1 ? 0 : partial_bytes(S, batch, num_qo_heads, head_dim);
}

}  // extern "C"

namespace {

// sa_decode and sa_decode_multi: rows = batch * q_len query rows.
sa_status_t decode_impl(const void *q, int32_t q_len, const sa_kv_desc_t *kv, const int32_t *seqlens,
                        int32_t batch, int32_t num_qo_heads, int32_t max_kv_len, const float *sinks,
                        int32_t window, float sm_scale, void *out, float *lse, void *workspace,
                        size_t workspace_bytes, int32_t num_splits, cudaStream_t stream)
{
    g_err[0] = 0;
    sa_status_t st = check_decode_common(q, kv, seqlens, batch, num_qo_heads, max_kv_len, window, sm_scale);
    if (st != SA_OK)
        return st;
    if (q_len < 1 || q_len > SA_MAX_DECODE_TOKENS)
        return fail(SA_ERR_UNSUPPORTED, "q_len %d outside [1, %d]", q_len, SA_MAX_DECODE_TOKENS);
    if (num_splits < 0 || num_splits > kMaxSplits)
        return fail(SA_ERR_INVALID_ARG, "num_splits %d outside [0, %d]", num_splits, kMaxSplits);
    if (batch > 0 && !out)
        return fail(SA_ERR_INVALID_ARG, "out is NULL");
    if (out && !aligned16(out))
        return fail(SA_ERR_UNSUPPORTED, "out must be 16-byte aligned");
    if (static_cast<int64_t>(batch) * q_len > 65535 * 8)
        return fail(SA_ERR_UNSUPPORTED, "batch * q_len too large");
    if (batch == 0)
        return SA_OK;
    const int32_t rows = batch * q_len;
    const int32_t S = num_splits != 0 ? num_splits
                      : sa_decode_multi_num_splits(batch, q_len, kv->num_kv_heads, max_kv_len, window, kv->dtype);
    if (S <= 1)
        return launch_decode_kernel(q, q_len, kv, seqlens, batch, num_qo_heads, max_kv_len, sinks, window,
                                    sm_scale, out, lse, nullptr, nullptr, 1, false, stream);
    const size_t need = partial_bytes(S, rows, num_qo_heads, kv->head_dim);
    if (!workspace || workspace_bytes < need)
        return fail(SA_ERR_WORKSPACE, "split decode (%d chunks) needs %zu workspace bytes, got %zu", S, need,
                    workspace ? workspace_bytes : size_t(0));
    if (!aligned16(workspace))
        return fail(SA_ERR_UNSUPPORTED, "workspace must be 16-byte aligned");
    float *o_part = static_cast<float *>(workspace);
    float *lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                align256(static_cast<size_t>(S) * rows * num_qo_heads *
                                                         kv->head_dim * sizeof(float)));
    st = launch_decode_kernel(q, q_len, kv, seqlens, batch, num_qo_heads, max_kv_len, nullptr, window, sm_scale,
                              nullptr, nullptr, o_part, lse_part, S, true, stream);
    if (st != SA_OK)
        return st;
    return sa_merge_states(o_part, lse_part, S, rows, num_qo_heads, kv->head_dim, sinks, out, lse, stream);
}

}  // namespace

extern "C" {

sa_status_t sa_decode(const void *q, const sa_kv_desc_t *kv, const int32_t *seqlens, int32_t batch,
                      int32_t num_qo_heads, int32_t max_kv_len, const float *sinks, int32_t window,
                      float sm_scale, void *out, float *lse, void *workspace, size_t workspace_bytes,
                      int32_t num_splits, cudaStream_t stream)
{
    return decode_impl(q, 1, kv, seqlens, batch, num_qo_heads, max_kv_len, sinks, window, sm_scale, out, lse,
                       workspace, workspace_bytes, num_splits, stream);
}

size_t sa_decode_multi_workspace_size(int32_t batch, int32_t q_len, int32_t num_qo_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t max_kv_len, int32_t window, int32_t num_splits)
{
    if (batch <= 0 || q_len <= 0 || num_qo_heads <= 0 || head_dim <= 0 || num_splits < 0)
        return 0;
    // (num_splits = 0: enough for the automatic choice on either cache type)
    const int32_t S =
        num_splits != 0
            ? num_splits
            : std::max(sa_decode_multi_num_splits(batch, q_len, num_kv_heads, max_kv_len, window, SA_KV_BF16),
                       sa_decode_multi_num_splits(batch, q_len, num_kv_heads, max_kv_len, window, SA_KV_FP8_E4M3));
    return S <= 1 ? 0 : partial_bytes(S, batch * q_len, num_qo_heads, head_dim);
}

sa_status_t sa_decode_multi(const void *q, int32_t q_len, const sa_kv_desc_t *kv, const int32_t *seqlens,
                            int32_t batch, int32_t num_qo_heads, int32_t max_kv_len, const float *sinks,
                            int32_t window, float sm_scale, void *out, float *lse, void *workspace,
                            size_t workspace_bytes, int32_t num_splits, cudaStream_t stream)
{
    return decode_impl(q, q_len, kv, seqlens, batch, num_qo_heads, max_kv_len, sinks, window, sm_scale, out, lse,
                       workspace, workspace_bytes, num_splits, stream);
}

sa_status_t sa_decode_partial(const void *q, const sa_kv_desc_t *kv, const int32_t *seqlens, int32_t batch,
                              int32_t num_qo_heads, int32_t max_kv_len, int32_t window, float sm_scale,
                              int32_t num_splits, float *o_part, float *lse_part, cudaStream_t stream)
{
    g_err[0] = 0;
    sa_status_t st = check_decode_common(q, kv, seqlens, batch, num_qo_heads, max_kv_len, window, sm_scale);
    if (st != SA_OK)
        return st;
    if (num_splits < 1 || num_splits > 65535)
        return fail(SA_ERR_INVALID_ARG, "num_splits %d outside [1, 65535]", num_splits);
    if (batch > 0 && (!o_part || !lse_part))
        return fail(SA_ERR_INVALID_ARG, "o_part / lse_part is NULL");
    if (o_part && !aligned16(o_part))
        return fail(SA_ERR_UNSUPPORTED, "o_part must be 16-byte aligned");
    if (batch == 0)
        return SA_OK;
    return launch_decode_kernel(q, 1, kv, seqlens, batch, num_qo_heads, max_kv_len, nullptr, window, sm_scale,
                                nullptr, nullptr, o_part, lse_part, num_splits, true, stream);
}

sa_status_t sa_merge_states(const float *o_part, const float *lse_part, int32_t num_splits, int32_t n,
                            int32_t num_heads, int32_t head_dim, const float *sinks, void *out, float *lse_out,
                            cudaStream_t stream)
{
    if (num_splits < 1 || n < 0 || num_heads <= 0)
        return fail(SA_ERR_INVALID_ARG, "num_splits >= 1, n >= 0 and num_heads > 0 required");
    if (head_dim <= 0 || head_dim % 4 != 0 || head_dim > 256)
        return fail(SA_ERR_UNSUPPORTED, "head_dim %d: a multiple of 4 up to 256 is supported", head_dim);
    if (n == 0)
        return SA_OK;
    if (!o_part || !lse_part || !out)
        return fail(SA_ERR_INVALID_ARG, "o_part / lse_part / out is NULL");
    if (!aligned16(o_part) || (reinterpret_cast<uintptr_t>(out) & 7u) != 0)
        return fail(SA_ERR_UNSUPPORTED, "o_part must be 16-byte and out 8-byte aligned");
    if (static_cast<int64_t>(n) * num_heads * num_splits * head_dim >= (int64_t(1) << 40))
        return fail(SA_ERR_UNSUPPORTED, "merge too large");
    sa::MergeParams p;
    p.o_part = o_part;
    p.lse_part = lse_part;
    p.sinks = sinks;
    p.out = out;
    p.lse_out = lse_out;
    p.num_splits = num_splits;
    p.n = n;
    p.num_heads = num_heads;
    p.head_dim = head_dim;
    cudaError_t e = sa::launch_merge(p, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "merge launch");
    return SA_OK;
}

}  // extern "C"

namespace {

// sa_prefill (bf16 q) and sa_prefill_q8 (E4M3 q codes, value = code * q_scale)
sa_status_t prefill_impl(const void *q, bool q8, float q_scale, const int32_t *cu_seqlens_q, int32_t total_q,
                         const sa_kv_desc_t *kv, const int32_t *seqlens_kv, int32_t batch, int32_t num_qo_heads,
                         int32_t max_q_len, int32_t max_kv_len, const float *sinks, int32_t window,
                         float sm_scale, void *out, float *lse, cudaStream_t stream)
{
    g_err[0] = 0;
    if (batch < 0 || total_q < 0 || max_q_len < 0 || max_kv_len < 0 || window < 0)
        return fail(SA_ERR_INVALID_ARG, "batch, total_q, max_q_len, max_kv_len and window must be >= 0");
    if (!std::isfinite(sm_scale))
        return fail(SA_ERR_INVALID_ARG, "sm_scale must be finite");
    if (!(sm_scale > 0.f))
        return fail(SA_ERR_UNSUPPORTED, "sa_prefill needs sm_scale > 0");
    if (batch > 65535)
        return fail(SA_ERR_UNSUPPORTED, "batch %d > 65535", batch);
    sa_status_t st = check_kv(kv, batch, num_qo_heads, max_kv_len);
    if (st != SA_OK)
        return st;
    if (batch == 0 || total_q == 0 || max_q_len == 0)
        return SA_OK;
    if (!q || !cu_seqlens_q || !seqlens_kv || !out)
        return fail(SA_ERR_INVALID_ARG, "q / cu_seqlens_q / seqlens_kv / out is NULL");
    if (!aligned16(q) || !aligned16(out))
        return fail(SA_ERR_UNSUPPORTED, "q and out must be 16-byte aligned");
    const int group = num_qo_heads / kv->num_kv_heads;
    sa::PrefillParams p;
    std::memset(&p, 0, sizeof p);
    CUtensorMap tq, tk, tv;
    int dt = 0, dh = 0, dp = 0;
    const bool fp8 = kv->dtype == SA_KV_FP8_E4M3;
    if (q8 && !fp8)
        return fail(SA_ERR_UNSUPPORTED, "E4M3 queries need an FP8-E4M3 cache");
    if (q8 && (!std::isfinite(q_scale) || q_scale == 0.f))
        return fail(SA_ERR_INVALID_ARG, "q_scale must be finite and nonzero");
    // bf16: one box per 64-key tile when no tile straddles a page (contiguous
    // sequences, or pages holding a multiple of 64 keys); else 16-key boxes
    const int box_rows =
        (!fp8 && ((!kv->page_table && kv->page_size >= 64) || kv->page_size % 64 == 0)) ? 64 : 16;
    st = encode_kv_map(&tk, kv->k, fp8, kv, box_rows, &dt, &dh, &dp);
    if (st != SA_OK)
        return st;
    st = encode_kv_map(&tv, kv->v, fp8, kv, box_rows, &dt, &dh, &dp);
    if (st != SA_OK)
        return st;
    {
        EncodeTiledFn fn = encode_fn();
        if (!fn)
            return fail(SA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(sa::kHeadDim), static_cast<cuuint64_t>(num_qo_heads),
                                    static_cast<cuuint64_t>(total_q)};
        const cuuint64_t esz = q8 ? 1 : 2;
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(sa::kHeadDim) * esz,
                                       static_cast<cuuint64_t>(num_qo_heads) * sa::kHeadDim * esz};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(sa::kHeadDim), 1, 128};
        const cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = fn(&tq, q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void *>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        q8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(SA_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled rejected q (CUresult %d)", (int)r);
    }
    uint32_t *status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess)
        return cuda_fail(e, "device status word");
    const float kLog2e = 1.44269504088896340736f;
    p.cu_seqlens_q = cu_seqlens_q;
    p.seqlens_kv = seqlens_kv;
    p.page_table = kv->page_table;
    p.sinks = sinks;
    p.out = out;
    p.lse = lse;
    p.status = status;
    p.batch = batch;
    p.num_qo_heads = num_qo_heads;
    p.num_kv_heads = kv->num_kv_heads;
    p.group = group;
    p.heads_per_cta = (group % 2 == 0) ? 2 : 1;  // the two heads of a block share one kv head
    p.page_size = kv->page_size;
    p.table_stride = kv->page_table_stride;
    p.num_pages = kv->num_pages;
    p.max_q_len = max_q_len;
    p.max_kv_len = max_kv_len;
    p.window = window;
    p.num_q_tiles = (max_q_len + 127) / 128;
    p.box_rows = box_rows;
    p.dim_token = dt;
    p.dim_head = dh;
    p.dim_page = dp;
    // FP8: the kernel widens each code to its E4M3 value in f16 (Q8: products of the codes)
    p.score_scale = sm_scale * kLog2e * (fp8 ? kv->k_scale : 1.f) * (q8 ? q_scale : 1.f);
    p.out_scale = fp8 ? kv->v_scale : 1.f;
    if (p.num_q_tiles > 65535)
        return fail(SA_ERR_UNSUPPORTED, "max_q_len too large");
    e = sa::launch_prefill(tq, tk, tv, p, fp8, q8, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "prefill launch");
    return SA_OK;
}

}  // namespace

extern "C" {

sa_status_t sa_prefill(const void *q, const int32_t *cu_seqlens_q, int32_t total_q, const sa_kv_desc_t *kv,
                       const int32_t *seqlens_kv, int32_t batch, int32_t num_qo_heads, int32_t max_q_len,
                       int32_t max_kv_len, const float *sinks, int32_t window, float sm_scale, void *out,
                       float *lse, cudaStream_t stream)
{
    return prefill_impl(q, false, 1.f, cu_seqlens_q, total_q, kv, seqlens_kv, batch, num_qo_heads, max_q_len,
                        max_kv_len, sinks, window, sm_scale, out, lse, stream);
}

sa_status_t sa_prefill_q8(const void *q, float q_scale, const int32_t *cu_seqlens_q, int32_t total_q,
                          const sa_kv_desc_t *kv, const int32_t *seqlens_kv, int32_t batch, int32_t num_qo_heads,
                          int32_t max_q_len, int32_t max_kv_len, const float *sinks, int32_t window,
                          float sm_scale, void *out, float *lse, cudaStream_t stream)
{
    return prefill_impl(q, true, q_scale, cu_seqlens_q, total_q, kv, seqlens_kv, batch, num_qo_heads, max_q_len,
                        max_kv_len, sinks, window, sm_scale, out, lse, stream);
}

sa_status_t sa_rope_yarn_table(float *table, int32_t max_position, int32_t head_dim, double theta,
                               double factor, int32_t original_max_position, double beta_fast, double beta_slow)
{
    g_err[0] = 0;
    if (!table || max_position < 1)
        return fail(SA_ERR_INVALID_ARG, "table is NULL or max_position < 1");
    if (head_dim != sa::kHeadDim)
        return fail(SA_ERR_UNSUPPORTED, "head_dim %d: only 64 is supported", head_dim);
    if (!std::isfinite(theta) || !(theta > 1.0) || !std::isfinite(factor) || original_max_position < 1 ||
        !(beta_fast > 0.0) || !(beta_slow > 0.0) || !std::isfinite(beta_fast) || !std::isfinite(beta_slow))
        return fail(SA_ERR_INVALID_ARG, "theta > 1, finite factor, original_max_position >= 1 and "
                                        "beta_fast, beta_slow > 0 required");
    constexpr int half = sa::kHeadDim / 2;
    const double kPi = 3.14159265358979323846;
    double freq[half];
    double mscale = 1.0;
    // the dimension index that turns n times over the original context
    auto turns_dim = [&](double n) {
        return sa::kHeadDim * std::log(original_max_position / (2.0 * kPi * n)) / (2.0 * std::log(theta));
    };
    double lo = 0.0, hi = 0.0;
    if (factor > 1.0) {
        lo = std::max(std::floor(turns_dim(beta_fast)), 0.0);
        hi = std::min(std::ceil(turns_dim(beta_slow)), double(sa::kHeadDim - 1));
        if (hi == lo)
            hi = lo + 0.001;
        mscale = 0.1 * std::log(factor) + 1.0;
    }
    for (int i = 0; i < half; ++i) {
        const double f = std::pow(theta, -2.0 * i / sa::kHeadDim);
        if (factor > 1.0) {
            const double ramp = std::min(std::max((i - lo) / (hi - lo), 0.0), 1.0);
            freq[i] = f * (1.0 - ramp) + (f / factor) * ramp;
        } else {
            freq[i] = f;
        }
    }
    for (int64_t p = 0; p < max_position; ++p) {
        float *row = table + p * sa::kHeadDim;
        for (int i = 0; i < half; ++i) {
            const double a = static_cast<double>(p) * freq[i];
            row[i] = static_cast<float>(std::cos(a) * mscale);
            row[half + i] = static_cast<float>(std::sin(a) * mscale);
        }
    }
    return SA_OK;
}

sa_status_t sa_rope_append(const void *q, const void *k, const void *v, int32_t num_tokens, int32_t num_qo_heads,
                           const int32_t *seq_ids, const int32_t *positions, const float *table,
                           int32_t max_position, const sa_kv_desc_t *kv, int32_t batch, void *q_out,
                           float q_out_scale, cudaStream_t stream)
{
    g_err[0] = 0;
    if (num_tokens < 0 || batch < 0 || max_position < 1)
        return fail(SA_ERR_INVALID_ARG, "num_tokens and batch must be >= 0, max_position >= 1");
    sa_status_t st = check_kv(kv, batch, num_qo_heads, 0);
    if (st != SA_OK)
        return st;
    if (!std::isfinite(q_out_scale) || q_out_scale < 0.f)
        return fail(SA_ERR_INVALID_ARG, "q_out_scale must be 0 (bf16 q_out) or finite and > 0 (E4M3 q_out)");
    if (num_tokens == 0)
        return SA_OK;
    if (!q || !k || !v || !seq_ids || !positions || !table || !q_out)
        return fail(SA_ERR_INVALID_ARG, "q / k / v / seq_ids / positions / table / q_out is NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_out) || !aligned16(table))
        return fail(SA_ERR_UNSUPPORTED, "q, k, v, q_out and table must be 16-byte aligned");
    if (static_cast<int64_t>(num_tokens) * (num_qo_heads + 2 * kv->num_kv_heads) >= (int64_t(1) << 31))
        return fail(SA_ERR_UNSUPPORTED, "num_tokens * (num_qo_heads + 2 * num_kv_heads) must be below 2^31");
    uint32_t *status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess)
        return cuda_fail(e, "device status word");
    const bool fp8 = kv->dtype == SA_KV_FP8_E4M3;
    sa::RopeParams p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.k = k;
    p.v = v;
    p.seq_ids = seq_ids;
    p.positions = positions;
    p.table = table;
    p.q_out = q_out;
    p.k_cache = const_cast<void *>(kv->k);
    p.v_cache = const_cast<void *>(kv->v);
    p.page_table = kv->page_table;
    p.status = status;
    p.stride_page = kv->stride_page;
    p.stride_head = kv->stride_head;
    p.stride_token = kv->stride_token;
    p.num_tokens = num_tokens;
    p.num_qo_heads = num_qo_heads;
    p.num_kv_heads = kv->num_kv_heads;
    p.batch = batch;
    p.max_position = max_position;
    p.page_size = kv->page_size;
    p.table_stride = kv->page_table_stride;
    p.num_pages = kv->num_pages;
    p.fp8 = fp8 ? 1 : 0;
    p.k_inv_scale = fp8 ? 1.f / kv->k_scale : 1.f;
    p.v_inv_scale = fp8 ? 1.f / kv->v_scale : 1.f;
    p.q_fp8 = q_out_scale > 0.f ? 1 : 0;
    p.q_inv_scale = q_out_scale > 0.f ? 1.f / q_out_scale : 1.f;
    e = sa::launch_rope_append(p, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "rope_append launch");
    return SA_OK;
}

sa_status_t sa_selftest_wait_timeout(cudaStream_t stream)
{
    g_err[0] = 0;
    uint32_t *status = nullptr;
    cudaError_t e = status_ptr(&status);
    if (e != cudaSuccess)
        return cuda_fail(e, "device status word");
    e = sa::launch_wait_timeout_selftest(status, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "self-test launch");
    return SA_OK;
}

sa_status_t sa_device_status(cudaStream_t stream, uint32_t *flags_out)
{
    uint32_t *dptr = nullptr;
    cudaError_t e = status_ptr(&dptr);
    if (e != cudaSuccess)
        return cuda_fail(e, "device status word");
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "stream synchronize");
    uint32_t v = 0;
    e = cudaMemcpy(&v, dptr, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "status read");
    const uint32_t zero = 0;
    e = cudaMemcpy(dptr, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess)
        return cuda_fail(e, "status clear");
    if (flags_out)
        *flags_out = v;
    return SA_OK;
}

}  // extern "C"
