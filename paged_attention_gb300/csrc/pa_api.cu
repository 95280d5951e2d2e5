// pa_api.cu -- the C ABI: argument validation, workspace layout, TMA
// descriptor encoding and launches.  Declarations and the contract of every
// entry point are in include/pa.h.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "pa_internal.cuh"

namespace pa {

struct DecodeParams;  // pa_decode.cu
cudaError_t launch_assign(const WsLayout& L, const int32_t* ctx, const int32_t* ql,
                          const uint8_t* mask, void* ws, cudaStream_t stream);
cudaError_t launch_combine(const WsLayout& L, const void* ws, const void* partial, void* out,
                           float* lse, int grid, cudaStream_t stream);
int decode_smem_bytes(const pa_problem& p);
int decode_threads(const pa_problem& p);
const void* decode_kernel_ptr(const pa_problem& p);
cudaError_t launch_decode_from_api(const pa_problem& p, const WsLayout& L,
                                   const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv,
                                   const int32_t* block_table,
                                   const int32_t* ctx, const int32_t* ql, const float* ks,
                                   const float* vs, void* ws, void* partial, void* out, float* lse,
                                   cudaStream_t stream, bool take_hook = true,
                                   int static_splits = 0, int cluster_size = 1);
bool decode_has_mail(const pa_problem& p);
int decode_cluster_grid(const pa_problem& p, int C);
int prefill_smem_bytes(int D, bool fp8);
const void* prefill_kernel_ptr(int D, bool fp8);
cudaError_t launch_prefill_from_api(const pa_problem& p, const WsLayout& L, const void* q,
                                    const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const int32_t* block_table,
                                    const int32_t* ctx, const int32_t* ql, const float* qs,
                                    const float* ks, const float* vs, void* ws, void* partial,
                                    void* out, float* lse, cudaStream_t stream);

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sm_count[kMaxDevices] = {0};

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return -1;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// rows (query token x head) of one decode unit, rounded up to 16-row tiles
int decode_row_tiles(const pa_problem& p) {
    const int rows = (p.num_q_heads / p.num_kv_heads) * p.max_q_len;
    if (rows <= 16) return 1;
    if (rows <= 32) return 2;
    if (rows <= 64) return 4;
    return -1;
}

pa_status check_problem(const pa_problem* pp, int mode) {
    if (!pp) return PA_ERR_INVALID_ARG;
    const pa_problem& p = *pp;
    if (mode != PA_MODE_DECODE && mode != PA_MODE_PREFILL) return PA_ERR_INVALID_ARG;
    if (p.num_seqs < 1 || p.num_q_heads < 1 || p.num_kv_heads < 1 ||
        p.num_q_heads % p.num_kv_heads != 0 || p.num_pages < 1 || p.max_pages_per_seq < 1 ||
        p.total_q_tokens < 0 || p.max_q_len < 0 || p.max_context_len < p.max_q_len ||
        p.mask_q_tiles < 0 || p.mask_kv_tiles < 0 || p.num_ctas < 0 || p.balance_rows < 0 ||
        !std::isfinite(p.sm_scale) || p.sm_scale < 0.f || p.window < 0)
        return PA_ERR_INVALID_ARG;

    if (p.layout != PA_NHD && p.layout != PA_HND) return PA_ERR_INVALID_ARG;
    if (p.kv_dtype != PA_BF16 && p.kv_dtype != PA_FP8_E4M3) return PA_ERR_INVALID_ARG;
    if (p.q_dtype != PA_BF16 && p.q_dtype != PA_FP8_E4M3) return PA_ERR_INVALID_ARG;
    if (p.q_scale_mode != PA_SCALE_PER_TENSOR && p.q_scale_mode != PA_SCALE_PER_ROW)
        return PA_ERR_INVALID_ARG;
    if ((p.mask_q_tiles > 0) != (p.mask_kv_tiles > 0)) return PA_ERR_INVALID_ARG;
    if (p.head_dim != 64 && p.head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (p.page_size != 16 && p.page_size != 32 && p.page_size != 64 && p.page_size != 128 &&
        p.page_size != 256)
        return PA_ERR_UNSUPPORTED;
    if ((int64_t)p.max_pages_per_seq * p.page_size < p.max_context_len) return PA_ERR_INVALID_ARG;
    const int G = p.num_q_heads / p.num_kv_heads;
    if (mode == PA_MODE_DECODE) {
        if (p.mask_q_tiles > 0) return PA_ERR_INVALID_ARG;   // masks are a prefill feature
        const int RT = decode_row_tiles(p);
        if (RT < 0 || (p.head_dim == 128 && RT > 2)) return PA_ERR_UNSUPPORTED;
        if (p.kv_dtype == PA_FP8_E4M3 && p.head_dim != 128) return PA_ERR_UNSUPPORTED;
        if (p.q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    } else {
        if (G > 128 || 128 % G != 0) return PA_ERR_UNSUPPORTED;
        // the E4M3 prefill takes E4M3 Q, K and V together, head_dim 128
        if (p.kv_dtype != p.q_dtype) return PA_ERR_UNSUPPORTED;
        if (p.kv_dtype == PA_FP8_E4M3 && p.head_dim != 128) return PA_ERR_UNSUPPORTED;
    }
    return PA_OK;
}

int resolve_ctas(const pa_problem& p, int mode) {
    if (p.num_ctas > 0) return p.num_ctas;
    const int sms = sm_count();
    if (sms <= 0) return -1;
    int per_sm = 1;
    const void* k = nullptr;
    int smem = 0, threads = 0;
    if (mode == PA_MODE_DECODE) {
        k = decode_kernel_ptr(p);
        smem = decode_smem_bytes(p);
        threads = decode_threads(p);
    } else {
        k = prefill_kernel_ptr(p.head_dim, p.kv_dtype == PA_FP8_E4M3);
        smem = prefill_smem_bytes(p.head_dim, p.kv_dtype == PA_FP8_E4M3);
        threads = 384;
    }
    if (k && smem > 0) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return -1;
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, threads, smem) == cudaSuccess &&
            occ > 0)
            per_sm = occ;
        else
            return -1;
    }
    return sms * per_sm;
}

int rows_cap_for(const pa_problem& p, int mode) {
    if (mode == PA_MODE_PREFILL) return kPrefillRows;
    return 16 * decode_row_tiles(p);
}

bool encode_kv_map(const pa_problem& p, const void* base, CUtensorMap* map) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int e = p.kv_dtype == PA_BF16 ? 2 : 1;
    const cuuint64_t D = p.head_dim, ps = p.page_size, H = p.num_kv_heads, NP = p.num_pages;
    // logical order (d, slot, head, page); NHD vs HND differ only in strides
    cuuint64_t dims[4] = {D, ps, H, NP};
    cuuint64_t strides[3];
    if (p.layout == PA_NHD) {
        strides[0] = H * D * e;
        strides[1] = D * e;
        strides[2] = ps * H * D * e;
    } else {
        strides[0] = D * e;
        strides[1] = ps * D * e;
        strides[2] = H * ps * D * e;
    }
    const int rows = p.page_size < 64 ? p.page_size : 64;
    cuuint32_t box[4] = {(cuuint32_t)(128 / e < (int)D ? 128 / e : (int)D), (cuuint32_t)rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, p.kv_dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                    4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// bf16 K/V with head_dim 128, as (d % 64, slot % 8, column block, slot / 8,
// page) with the head folded into the column-block coordinate (NHD: chunk =
// 2 head + d / 64) or into the page coordinate (HND: page * H + head).  A box
// of up to 64 of a page's rows lands as 8-token groups, each the two
// 128-byte-swizzled [8 x 128 B] column blocks: one copy per page (or per 64
// tokens of a larger page), for the decode and the prefill kernels alike.
bool encode_kv_map_grouped(const pa_problem& p, const void* base, CUtensorMap* map) {
    auto fn = encode_fn();
    if (!fn || p.kv_dtype != PA_BF16 || p.head_dim != 128) return false;
    const cuuint64_t D = p.head_dim, ps = p.page_size, H = p.num_kv_heads, NP = p.num_pages;
    cuuint64_t dims[5], strides[4];
    if (p.layout == PA_NHD) {
        const cuuint64_t tok = H * D * 2;
        dims[0] = 64; dims[1] = 8; dims[2] = 2 * H; dims[3] = ps / 8; dims[4] = NP;
        strides[0] = tok; strides[1] = 128; strides[2] = 8 * tok; strides[3] = ps * tok;
    } else {
        dims[0] = 64; dims[1] = 8; dims[2] = 2; dims[3] = ps / 8; dims[4] = NP * H;
        strides[0] = D * 2; strides[1] = 128; strides[2] = 8 * D * 2; strides[3] = ps * D * 2;
    }
    const cuuint32_t rows = p.page_size < 64 ? p.page_size : 64;
    cuuint32_t box[5] = {64, 8, 2, rows / 8, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The K and V maps of a call: by 8-token group for bf16 with head_dim 128,
// else (d, slot, head, page) boxes of up to 64 slots.
bool encode_kv_maps(const pa_problem& p, const void* k, const void* v, CUtensorMap* tk,
                    CUtensorMap* tv) {
    if (p.kv_dtype == PA_BF16 && p.head_dim == 128)
        return encode_kv_map_grouped(p, k, tk) && encode_kv_map_grouped(p, v, tv);
    return encode_kv_map(p, k, tk) && encode_kv_map(p, v, tv);
}

// Q viewed as (d, head, token): box = 128 bytes of d (64 bf16 or 128 E4M3
// elements) x G heads x box_tokens tokens
bool encode_q_map(const pa_problem& p, const void* base, int box_tokens, CUtensorMap* map) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int G = p.num_q_heads / p.num_kv_heads;
    const cuuint64_t e = p.q_dtype == PA_FP8_E4M3 ? 1 : 2;
    const cuuint64_t D = p.head_dim, Hq = p.num_q_heads;
    const cuuint64_t T = p.total_q_tokens > 0 ? p.total_q_tokens : 1;
    cuuint64_t dims[3] = {D, Hq, T};
    cuuint64_t strides[2] = {D * e, Hq * D * e};
    cuuint32_t box[3] = {(cuuint32_t)(128 / e), (cuuint32_t)G, (cuuint32_t)box_tokens};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, e == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    3, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

pa_status make_layout(const pa_problem* p, int mode, WsLayout& L) {
    pa_status st = check_problem(p, mode);
    if (st != PA_OK) return st;
    const int N = resolve_ctas(*p, mode);
    if (N <= 0) return PA_ERR_CUDA;
    if (!layout_for(*p, mode, N, rows_cap_for(*p, mode), L)) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

// Prefill mode.  A batch without a block mask is split in two: the sequences
// with 1 <= G * q_len <= kMixedDecodeRows (decode steps of a mixed batch) get
// a decode-mode task map that the decode kernel runs (64-token tiles, one
// unit per (sequence, KV head), balanced over its own persistent CTAs); the
// others get the prefill map.  A decode unit fills a few of the 128 rows of a
// tensor-core tile, so the prefill kernel would stream its K/V at a fraction
// of the decode kernel's rate.  Both maps live in one workspace: the prefill
// map first (its header, at offset 0, also takes the decode kernel's device
// faults), the decode map from the next 256-byte boundary; the partials
// likewise.
struct PrefillLayout {
    WsLayout L;          // the prefill map
    WsLayout Ld;         // the decode map (split only)
    pa_problem pd;       // the problem as the decode kernel sees it
    bool split;
    int64_t part_off;    // Ld's partials inside the partial workspace
    int64_t total_bytes, partial_bytes;
};

pa_status make_prefill_layout(const pa_problem* p, PrefillLayout& M) {
    pa_status st = make_layout(p, PA_MODE_PREFILL, M.L);
    if (st != PA_OK) return st;
    M.split = false;
    M.part_off = 0;
    M.total_bytes = M.L.total_bytes;
    M.partial_bytes = M.L.partial_bytes;
    const int G = p->num_q_heads / p->num_kv_heads;
    // (the decode kernel takes a bf16 Q: an E4M3 batch stays on one map)
    if (p->mask_q_tiles > 0 || G > kMixedDecodeRows || p->q_dtype != PA_BF16) return PA_OK;
    const int small_q = kMixedDecodeRows / G;
    M.pd = *p;
    if (M.pd.max_q_len > small_q) M.pd.max_q_len = small_q;
    if (check_problem(&M.pd, PA_MODE_DECODE) != PA_OK) return PA_OK;
    const int Nd = resolve_ctas(M.pd, PA_MODE_DECODE);
    if (Nd <= 0) return PA_ERR_CUDA;
    WsLayout& Ld = M.Ld;
    if (!layout_for(M.pd, PA_MODE_DECODE, Nd, rows_cap_for(M.pd, PA_MODE_DECODE), Ld))
        return PA_ERR_INVALID_ARG;
    const int64_t base = align256(M.L.total_bytes);
    for (int64_t* o : {&Ld.off_header, &Ld.off_cta_ptr, &Ld.off_tasks, &Ld.off_task_cta,
                       &Ld.off_units, &Ld.off_ntiles, &Ld.off_prefix, &Ld.off_nsplit,
                       &Ld.off_slot0, &Ld.off_done, &Ld.off_fix, &Ld.off_active, &Ld.off_cu_q,
                       &Ld.off_seq_unit0})
        *o += base;
    Ld.off_err_header = M.L.off_header;
    Ld.max_q_len = p->max_q_len;   // both Assigns check the caller's lengths
    Ld.cls = 1;
    Ld.small_q = small_q;
    M.L.cls = 2;
    M.L.small_q = small_q;
    M.split = true;
    M.total_bytes = base + Ld.total_bytes;
    M.part_off = align256(M.L.partial_bytes);
    M.partial_bytes = M.part_off + Ld.partial_bytes;
    return PA_OK;
}

// Static split-K workspace: a 256-byte header (its error word is where
// pa_last_device_error reads it), the completion counters of the in-kernel
// finalizer (kDoneWords per unit), then, for S > 1, the partials of the U * S
// static tasks.  The header and counters are cleared at every call.
constexpr int kMaxStaticSplits = 64;

// The library's split count: the smallest power of two giving at least eight
// tasks per CTA, at most 4 (measured on the bf16 decode batch, 512 units on
// 152 SMs: S = 1, 2, 4, 8 took 0.332, 0.310, 0.284, 0.473 ms; finer splits
// pay for more partial states than they gain in balance).
int static_splits_for(const pa_problem& p, int num_splits, int N) {
    if (num_splits > 0) return num_splits;
    const int64_t U = (int64_t)p.num_seqs * p.num_kv_heads;
    const int64_t want = (8 * (int64_t)N + U - 1) / U;
    int S = 1;
    while (S < want && S < 4) S *= 2;
    return S;
}

// Clusters: with S in {2, 4, 8} and a kernel variant that has room for the
// DSM mailbox, the S splits of a unit run on the S CTAs of one cluster and
// merge on chip (cluster = S); else the splits merge through the partial
// workspace (cluster = 1).  The grid is then a multiple of S: the largest
// co-resident one, or problem->num_ctas when that is a multiple of S.
// `query_grid` false: decide without touching the device (size queries).
pa_status make_static_layout(const pa_problem* p, int num_splits, WsLayout& L, int& S,
                             int& cluster, bool query_grid) {
    pa_status st = make_layout(p, PA_MODE_DECODE, L);
    if (st != PA_OK) return st;
    if (num_splits < 0 || num_splits > kMaxStaticSplits) return PA_ERR_INVALID_ARG;
    S = static_splits_for(*p, num_splits, L.N);
    cluster = 1;
    if ((S == 2 || S == 4 || S == 8) && decode_has_mail(*p)) {
        if (p->num_ctas > 0) {
            if (p->num_ctas % S == 0) cluster = S;
        } else if (query_grid) {
            const int g = decode_cluster_grid(*p, S);
            if (g >= S) {
                cluster = S;
                L.N = g;
            }
        } else {
            cluster = S;
        }
    }
    const int64_t U = (int64_t)p->num_seqs * p->num_kv_heads;
    L.off_header = 0;
    L.off_err_header = 0;
    L.off_done = kHeaderWords * 4;
    L.total_bytes = align256(L.off_done + U * kDoneWords * 4);
    L.partial_slots = S > 1 ? U * S : 0;   // (kept in cluster mode too: one size per S)
    L.partial_bytes = L.partial_slots * (int64_t)L.rows_cap * (L.D + 1) * 4;
    return PA_OK;
}

// Combine walks (unit, 4-row chunk) items: up to 8 CTAs of 128 threads per
// SM, never more than the items of the largest possible fix list
int combine_grid(const WsLayout& L) {
    int64_t grid = 8 * (int64_t)sm_count();
    const int64_t items = (int64_t)L.unit_cap * ((L.rows_cap + 3) / 4);
    if (grid > items) grid = items;
    return grid < 1 ? 1 : (int)grid;
}

std::atomic<int64_t*> g_trace{nullptr};
std::atomic<int64_t> g_trace_cap{0};
std::atomic<int32_t> g_test_skip{-1};
std::atomic<uint64_t> g_test_limit{0};

}  // namespace

void take_task_trace(int64_t** trace, int64_t* capacity) {
    *trace = g_trace.load();
    *capacity = *trace != nullptr ? g_trace_cap.load() : 0;
}

void take_test_hook(int32_t* skip_entry, uint64_t* wait_limit_ns) {
    const int32_t s = g_test_skip.exchange(-1);
    const uint64_t l = g_test_limit.exchange(0);
    *skip_entry = s;
    *wait_limit_ns = (s >= 0 && l > 0) ? l : kWaitLimitNs;
}

bool layout_for(const pa_problem& p, int mode, int N, int rows_cap, WsLayout& L) {
    std::memset(&L, 0, sizeof(L));
    const int G = p.num_q_heads / p.num_kv_heads;
    L.mode = mode;
    L.B = p.num_seqs;
    L.Hq = p.num_q_heads;
    L.Hkv = p.num_kv_heads;
    L.G = G;
    L.D = p.head_dim;
    L.N = N;
    L.kv_tile = mode == PA_MODE_DECODE ? kDecodeTile : kPrefillTile;
    if (mode == PA_MODE_DECODE)
        L.qtok = p.max_q_len > 0 ? p.max_q_len : 1;
    else
        L.qtok = (p.mask_q_tiles > 0 && G == 1) ? kPrefillHalfRows : kPrefillRows / G;
    int64_t ucap;
    if (mode == PA_MODE_DECODE)
        ucap = (int64_t)p.num_seqs * p.num_kv_heads;
    else
        ucap = (int64_t)p.num_kv_heads * (ceil_div(p.total_q_tokens, L.qtok) + p.num_seqs);
    if (ucap < 1) ucap = 1;
    if (ucap > (1 << 30)) return false;
    L.unit_cap = (int32_t)ucap;
    L.task_cap = L.unit_cap + N;
    L.max_kv_tiles = ceil_div(p.max_context_len > 0 ? p.max_context_len : 1, L.kv_tile);
    L.has_mask = p.mask_q_tiles > 0 ? 1 : 0;
    L.rows_cap = rows_cap;
    L.balance_rows = p.balance_rows > 0 ? p.balance_rows : kDefaultBalanceRows;
    L.unit_cost = p.unit_cost > 0 ? p.unit_cost
                  : p.unit_cost < 0 ? 0
                  : (mode == PA_MODE_DECODE ? PA_DEFAULT_UNIT_COST_DECODE
                                            : PA_DEFAULT_UNIT_COST_PREFILL);
    L.total_q = p.total_q_tokens;
    L.max_q_len = p.max_q_len;
    L.max_ctx = p.max_context_len;
    L.mask_q_tiles = p.mask_q_tiles;
    L.mask_kv_tiles = p.mask_kv_tiles;
    L.window = p.window;
    int64_t off = 0;
    auto take = [&](int64_t bytes) {
        int64_t o = off;
        off = align256(off + bytes);
        return o;
    };
    L.off_header = take(kHeaderWords * 4);
    L.off_cta_ptr = take((int64_t)(N + 1) * 4);
    L.off_tasks = take((int64_t)L.task_cap * 16);
    L.off_task_cta = take((int64_t)L.task_cap * 4);
    L.off_units = take((int64_t)L.unit_cap * 16);
    L.off_ntiles = take((int64_t)L.unit_cap * 4);
    L.off_prefix = take((int64_t)L.unit_cap * 8);
    L.off_nsplit = take((int64_t)L.unit_cap * 4);
    L.off_slot0 = take((int64_t)L.unit_cap * 4);
    L.off_done = take((int64_t)L.unit_cap * kDoneWords * 4);
    L.off_fix = take((int64_t)L.unit_cap * 4);
    L.off_active = take(L.has_mask ? (int64_t)L.unit_cap * L.max_kv_tiles * 4 : 4);
    L.off_cu_q = take((int64_t)(p.num_seqs + 1) * 4);
    L.off_seq_unit0 = take((int64_t)(p.num_seqs + 1) * 4);
    L.off_err_header = L.off_header;
    L.total_bytes = off;
    L.partial_slots = L.task_cap;
    L.partial_bytes = L.partial_slots * (int64_t)L.rows_cap * (L.D + 1) * 4;
    return true;
}

// ------------------------------------------- fixed scratch of pa_decode_noalloc
// One array per device for the whole process: the task map at offset 0, the
// split-K partials after it.  Being part of the module image, it exists on
// every device that loads the library.  In host code the name below is only a
// host-side stand-in that the CUDA runtime links to the device copy; the
// device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device, looked up on the first
// call for that device and cached.
pa_status noalloc_scratch(char** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return PA_ERR_CUDA;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = static_cast<char*>(g_noalloc_ptr[dev]);
    return PA_OK;
}

}  // namespace

namespace {
pa_status prefill_body(const pa_problem* problem, const void* q, const float* q_scale,
                       const void* k_cache, const void* v_cache, const int32_t* block_table,
                       const int32_t* context_lens, const int32_t* q_lens, const float* k_scale,
                       const float* v_scale, const uint8_t* block_mask, const void* assign_ws,
                       size_t assign_ws_bytes, void* partial_ws, size_t partial_ws_bytes,
                       void* out, float* lse, void* stream) {
    PrefillLayout M;
    pa_status st = make_prefill_layout(problem, M);
    if (st != PA_OK) return st;
    // the kernels read the active-tile lists pa_assign built from the mask;
    // the mask itself must be given exactly when the problem declares one
    if ((problem->mask_q_tiles > 0) != (block_mask != nullptr)) return PA_ERR_INVALID_ARG;
    const WsLayout& L = M.L;
    const pa_problem& p = *problem;
    if (p.total_q_tokens == 0) return PA_OK;   // no query row: nothing to compute
    if (!q || !k_cache || !v_cache || !block_table || !context_lens || !q_lens || !assign_ws ||
        !out || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(out, 16) || !aligned(block_table, 4) || !aligned(assign_ws, 256))
        return PA_ERR_INVALID_ARG;
    if (p.q_dtype == PA_FP8_E4M3 &&
        (!q_scale || !k_scale || !v_scale || !aligned(q_scale, 4) || !aligned(k_scale, 4) ||
         !aligned(v_scale, 4)))
        return PA_ERR_INVALID_ARG;
    if (assign_ws_bytes < (size_t)M.total_bytes) return PA_ERR_WORKSPACE;
    if (partial_ws_bytes < (size_t)M.partial_bytes || !partial_ws || !aligned(partial_ws, 16))
        return PA_ERR_WORKSPACE;
    CUtensorMap tq, tk, tv;
    if (!encode_q_map(p, q, kPrefillHalfRows / (p.num_q_heads / p.num_kv_heads), &tq) ||
        !encode_kv_maps(p, k_cache, v_cache, &tk, &tv))
        return PA_ERR_INVALID_ARG;
    const cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    if (M.split) {
        // the decode-shaped sequences first, on the decode kernel (same K/V
        // maps)
        CUtensorMap tqd;
        if (!encode_q_map(M.pd, q, M.pd.max_q_len > 0 ? M.pd.max_q_len : 1, &tqd))
            return PA_ERR_INVALID_ARG;
        // (the wait-timeout test hook is left for the prefill kernel)
        e = launch_decode_from_api(M.pd, M.Ld, tqd, tk, tv,
                                   block_table, context_lens, q_lens, k_scale, v_scale,
                                   const_cast<void*>(assign_ws),
                                   static_cast<char*>(partial_ws) + M.part_off, out, lse, s,
                                   false);
    }
    if (e == cudaSuccess)
        e = launch_prefill_from_api(p, L, q, tq, tk, tv, block_table, context_lens, q_lens,
                                    q_scale, k_scale, v_scale, const_cast<void*>(assign_ws),
                                    partial_ws, out, lse, s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
}  // namespace

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_DEVICE_CHECK: return "PA_ERR_DEVICE_CHECK";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
        default: return "PA_ERR_UNKNOWN";
    }
}

const char* pa_version(void) { return "paged_attention_gb300 0.1 (sm_103a)"; }

pa_status pa_num_ctas(const pa_problem* problem, int mode, int32_t* num_ctas) {
    if (!num_ctas) return PA_ERR_INVALID_ARG;
    pa_status st = check_problem(problem, mode);
    if (st != PA_OK) return st;
    const int n = resolve_ctas(*problem, mode);
    if (n <= 0) return PA_ERR_CUDA;
    *num_ctas = n;
    return PA_OK;
}

size_t pa_assign_workspace_size(const pa_problem* problem, int mode) {
    if (mode == PA_MODE_PREFILL) {
        PrefillLayout M;
        return make_prefill_layout(problem, M) == PA_OK ? (size_t)M.total_bytes : 0;
    }
    WsLayout L;
    if (make_layout(problem, mode, L) != PA_OK) return 0;
    return (size_t)L.total_bytes;
}

size_t pa_partial_workspace_size(const pa_problem* problem, int mode) {
    if (mode == PA_MODE_PREFILL) {
        PrefillLayout M;
        return make_prefill_layout(problem, M) == PA_OK ? (size_t)M.partial_bytes : 0;
    }
    WsLayout L;
    if (make_layout(problem, mode, L) != PA_OK) return 0;
    return (size_t)L.partial_bytes;
}

pa_status pa_assign(const pa_problem* problem, int mode, const int32_t* context_lens,
                    const int32_t* q_lens, const uint8_t* block_mask, void* assign_ws,
                    size_t assign_ws_bytes, void* stream) {
    PrefillLayout M;
    pa_status st = mode == PA_MODE_PREFILL ? make_prefill_layout(problem, M)
                                           : make_layout(problem, mode, M.L);
    if (st != PA_OK) return st;
    if (mode != PA_MODE_PREFILL) {
        M.split = false;
        M.total_bytes = M.L.total_bytes;
    }
    const WsLayout& L = M.L;
    if (!context_lens || !q_lens || !assign_ws || !aligned(assign_ws, 256) ||
        !aligned(context_lens, 4) || !aligned(q_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (L.has_mask && !block_mask) return PA_ERR_INVALID_ARG;
    if (assign_ws_bytes < (size_t)M.total_bytes) return PA_ERR_WORKSPACE;
    cudaError_t e = launch_assign(L, context_lens, q_lens, L.has_mask ? block_mask : nullptr,
                                  assign_ws, (cudaStream_t)stream);
    if (e == cudaSuccess && M.split)
        e = launch_assign(M.Ld, context_lens, q_lens, nullptr, assign_ws, (cudaStream_t)stream);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode_splitk(const pa_problem* problem, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* block_table,
                           const int32_t* context_lens, const int32_t* q_lens,
                           const float* k_scale, const float* v_scale, const void* assign_ws,
                           size_t assign_ws_bytes, void* partial_ws, size_t partial_ws_bytes,
                           void* out, float* lse, void* stream) {
    WsLayout L;
    pa_status st = make_layout(problem, PA_MODE_DECODE, L);
    if (st != PA_OK) return st;
    const pa_problem& p = *problem;
    if (p.total_q_tokens == 0) return PA_OK;   // no query row: nothing to compute
    if (!q || !k_cache || !v_cache || !block_table || !context_lens || !q_lens || !assign_ws ||
        !out || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(out, 16) || !aligned(block_table, 4) || !aligned(assign_ws, 256))
        return PA_ERR_INVALID_ARG;
    if (p.kv_dtype == PA_FP8_E4M3 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
    if (assign_ws_bytes < (size_t)L.total_bytes) return PA_ERR_WORKSPACE;
    if (partial_ws_bytes < (size_t)L.partial_bytes || (!partial_ws && L.partial_bytes > 0) ||
        !aligned(partial_ws, 16))
        return PA_ERR_WORKSPACE;
    CUtensorMap tq, tk, tv;
    if (!encode_q_map(p, q, p.max_q_len > 0 ? p.max_q_len : 1, &tq)) return PA_ERR_INVALID_ARG;
    if (!encode_kv_maps(p, k_cache, v_cache, &tk, &tv)) return PA_ERR_INVALID_ARG;
    cudaError_t e = launch_decode_from_api(p, L, tq, tk, tv,
                                           block_table,
                                           context_lens, q_lens, k_scale, v_scale,
                                           const_cast<void*>(assign_ws), partial_ws, out, lse,
                                           (cudaStream_t)stream);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_combine(const pa_problem* problem, int mode, const void* assign_ws,
                     size_t assign_ws_bytes, const void* partial_ws, size_t partial_ws_bytes,
                     void* out, float* lse, void* stream) {
    PrefillLayout M;
    pa_status st = mode == PA_MODE_PREFILL ? make_prefill_layout(problem, M)
                                           : make_layout(problem, mode, M.L);
    if (st != PA_OK) return st;
    if (mode != PA_MODE_PREFILL) {
        M.split = false;
        M.total_bytes = M.L.total_bytes;
        M.partial_bytes = M.L.partial_bytes;
    }
    if (problem->total_q_tokens == 0) return PA_OK;   // no query row: nothing to combine
    if (!assign_ws || !out || !aligned(out, 16) || !aligned(assign_ws, 256))
        return PA_ERR_INVALID_ARG;
    if (assign_ws_bytes < (size_t)M.total_bytes) return PA_ERR_WORKSPACE;
    if (partial_ws_bytes < (size_t)M.partial_bytes || !partial_ws || !aligned(partial_ws, 16))
        return PA_ERR_WORKSPACE;
    // The bf16 decode kernel finalizes its split units itself (the last task
    // of a unit to finish merges its partials), and a decode-mode unit always
    // has a visible key: nothing is left for a bf16 decode-mode map, nor for
    // the decode part of a prefill-mode workspace (always bf16).  E4M3 decode
    // maps and the prefill kernel's map need this pass.
    if (mode == PA_MODE_DECODE && problem->kv_dtype == PA_BF16) return PA_OK;
    const cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_combine(M.L, assign_ws, partial_ws, out, lse, combine_grid(M.L), s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode_noalloc(const pa_problem* problem, const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_table,
                            const int32_t* context_lens, const int32_t* q_lens,
                            const float* k_scale, const float* v_scale, void* out, float* lse,
                            int32_t* device_error, void* stream) {
    WsLayout L;
    pa_status st = make_layout(problem, PA_MODE_DECODE, L);
    if (st != PA_OK) return st;
    const pa_problem& p = *problem;
    if (p.total_q_tokens == 0) {   // no query row: nothing to compute, no error
        if (device_error != nullptr && (!aligned(device_error, 4) ||
                                        cudaMemsetAsync(device_error, 0, 4,
                                                        (cudaStream_t)stream) != cudaSuccess))
            return aligned(device_error, 4) ? PA_ERR_CUDA : PA_ERR_INVALID_ARG;
        return PA_OK;
    }
    if (!q || !k_cache || !v_cache || !block_table || !context_lens || !q_lens || !out ||
        !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(context_lens, 4) || !aligned(q_lens, 4) ||
        !aligned(device_error, 4))
        return PA_ERR_INVALID_ARG;
    if (p.kv_dtype == PA_FP8_E4M3 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
    // task map first, partials from the next 256-byte boundary; both must fit
    const int64_t part_off = align256(L.total_bytes);
    if (part_off + L.partial_bytes > (int64_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    CUtensorMap tq, tk, tv;
    if (!encode_q_map(p, q, p.max_q_len > 0 ? p.max_q_len : 1, &tq)) return PA_ERR_INVALID_ARG;
    if (!encode_kv_maps(p, k_cache, v_cache, &tk, &tv)) return PA_ERR_INVALID_ARG;
    char* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != PA_OK) return st;
    void* ws = scratch;
    void* partial = scratch + part_off;
    const cudaStream_t s = (cudaStream_t)stream;
    // Assign resets the error word and the completion counters and rewrites
    // every word read below
    cudaError_t e = launch_assign(L, context_lens, q_lens, nullptr, ws, s);
    if (e == cudaSuccess)
        e = launch_decode_from_api(p, L, tq, tk, tv, block_table,
                                   context_lens, q_lens, k_scale, v_scale, ws, partial, out, lse,
                                   s);
    // (the bf16 decode kernel finalizes split units itself; E4M3 needs Combine)
    if (e == cudaSuccess && p.kv_dtype == PA_FP8_E4M3)
        e = launch_combine(L, ws, partial, out, lse, combine_grid(L), s);
    if (e == cudaSuccess && device_error)
        e = cudaMemcpyAsync(device_error, scratch + L.off_header + H_ERROR * 4, 4,
                            cudaMemcpyDeviceToDevice, s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_static_workspace_size(const pa_problem* problem, int32_t num_splits) {
    WsLayout L;
    int S = 0, cluster = 1;
    if (make_static_layout(problem, num_splits, L, S, cluster, false) != PA_OK) return 0;
    return (size_t)(L.total_bytes + L.partial_bytes);
}

pa_status pa_static_num_splits(const pa_problem* problem, int32_t num_splits, int32_t* out) {
    if (!out) return PA_ERR_INVALID_ARG;
    WsLayout L;
    int S = 0, cluster = 1;
    pa_status st = make_static_layout(problem, num_splits, L, S, cluster, false);
    if (st != PA_OK) return st;
    *out = S;
    return PA_OK;
}

pa_status pa_decode_static(const pa_problem* problem, int32_t num_splits, const void* q,
                           const void* k_cache, const void* v_cache, const int32_t* block_table,
                           const int32_t* context_lens, const int32_t* q_lens,
                           const float* k_scale, const float* v_scale, void* ws, size_t ws_bytes,
                           void* out, float* lse, void* stream) {
    WsLayout L;
    int S = 0, cluster = 1;
    pa_status st = make_static_layout(problem, num_splits, L, S, cluster, true);
    if (st != PA_OK) return st;
    const pa_problem& p = *problem;
    if (!ws || !aligned(ws, 256)) return PA_ERR_INVALID_ARG;
    if (ws_bytes < (size_t)(L.total_bytes + L.partial_bytes)) return PA_ERR_WORKSPACE;
    const cudaStream_t s = (cudaStream_t)stream;
    // the error word and the completion counters start at zero
    if (cudaMemsetAsync(ws, 0, (size_t)L.total_bytes, s) != cudaSuccess) return PA_ERR_CUDA;
    if (p.total_q_tokens == 0) return PA_OK;   // no query row: nothing to compute
    if (!q || !k_cache || !v_cache || !block_table || !context_lens || !q_lens || !out ||
        !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(context_lens, 4) || !aligned(q_lens, 4))
        return PA_ERR_INVALID_ARG;
    if (p.kv_dtype == PA_FP8_E4M3 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
    CUtensorMap tq, tk, tv;
    if (!encode_q_map(p, q, p.max_q_len > 0 ? p.max_q_len : 1, &tq)) return PA_ERR_INVALID_ARG;
    if (!encode_kv_maps(p, k_cache, v_cache, &tk, &tv)) return PA_ERR_INVALID_ARG;
    cudaError_t e = launch_decode_from_api(p, L, tq, tk, tv, block_table, context_lens,
                                           q_lens, k_scale, v_scale, ws,
                                           static_cast<char*>(ws) + L.total_bytes, out, lse, s,
                                           true, S, cluster);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_prefill(const pa_problem* problem, const void* q, const void* k_cache,
                     const void* v_cache, const int32_t* block_table,
                     const int32_t* context_lens, const int32_t* q_lens, const float* k_scale,
                     const float* v_scale, const uint8_t* block_mask, const void* assign_ws,
                     size_t assign_ws_bytes, void* partial_ws, size_t partial_ws_bytes,
                     void* out, float* lse, void* stream) {
    // an E4M3 Q comes with its scales: pa_prefill_fp8
    if (problem && problem->q_dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    return prefill_body(problem, q, nullptr, k_cache, v_cache, block_table, context_lens, q_lens,
                        k_scale, v_scale, block_mask, assign_ws, assign_ws_bytes, partial_ws,
                        partial_ws_bytes, out, lse, stream);
}

pa_status pa_prefill_fp8(const pa_problem* problem, const void* q, const float* q_scale,
                         const void* k_cache, const void* v_cache, const int32_t* block_table,
                         const int32_t* context_lens, const int32_t* q_lens,
                         const float* k_scale, const float* v_scale,
                         const uint8_t* block_mask, const void* assign_ws,
                         size_t assign_ws_bytes, void* partial_ws, size_t partial_ws_bytes,
                         void* out, float* lse, void* stream) {
    if (!problem) return PA_ERR_INVALID_ARG;
    if (problem->q_dtype != PA_FP8_E4M3 || problem->kv_dtype != PA_FP8_E4M3)
        return PA_ERR_UNSUPPORTED;
    return prefill_body(problem, q, q_scale, k_cache, v_cache, block_table, context_lens, q_lens,
                        k_scale, v_scale, block_mask, assign_ws, assign_ws_bytes, partial_ws,
                        partial_ws_bytes, out, lse, stream);
}

pa_status pa_set_task_trace(int64_t* trace, int64_t capacity) {
    if (capacity < 0 || (trace == nullptr) != (capacity == 0) || !aligned(trace, 8))
        return PA_ERR_INVALID_ARG;
    g_trace_cap.store(capacity);
    g_trace.store(trace);
    return PA_OK;
}

pa_status pa_test_inject_wait_timeout(int32_t skip_entry, int64_t wait_limit_ns) {
    if (skip_entry < 0) {
        g_test_skip.store(-1);
        g_test_limit.store(0);
        return PA_OK;
    }
    if (wait_limit_ns < 1000000 || wait_limit_ns > 1000000000) return PA_ERR_INVALID_ARG;
    g_test_limit.store((uint64_t)wait_limit_ns);
    g_test_skip.store(skip_entry);
    return PA_OK;
}

pa_status pa_read_task_map(const pa_problem* problem, int mode, const void* assign_ws,
                           size_t assign_ws_bytes, int32_t* counts, int32_t* cta_ptr,
                           int32_t* tasks, int32_t* units, int32_t* unit_ntiles,
                           int32_t* unit_nsplit, int32_t* unit_slot0, int32_t* active,
                           void* stream) {
    if (mode != PA_MODE_DECODE && mode != PA_MODE_PREFILL && mode != PA_MAP_DECODE_PART)
        return PA_ERR_INVALID_ARG;
    PrefillLayout M;
    pa_status st = mode == PA_MODE_DECODE ? make_layout(problem, mode, M.L)
                                          : make_prefill_layout(problem, M);
    if (st != PA_OK) return st;
    if (mode == PA_MODE_DECODE) M.total_bytes = M.L.total_bytes;
    if (!assign_ws || !counts) return PA_ERR_INVALID_ARG;
    if (assign_ws_bytes < (size_t)M.total_bytes) return PA_ERR_WORKSPACE;
    if (mode == PA_MAP_DECODE_PART && !M.split) {   // a masked batch has no decode part
        for (int i = 0; i < 4; ++i) counts[i] = 0;
        return PA_OK;
    }
    const WsLayout& L = mode == PA_MAP_DECODE_PART ? M.Ld : M.L;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t hdr[kHeaderWords];
    const char* ws = reinterpret_cast<const char*>(assign_ws);
    if (cudaMemcpyAsync(hdr, ws + L.off_header, sizeof hdr, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return PA_ERR_CUDA;
    const int U = hdr[H_UNITS], T = hdr[H_TASKS];
    counts[0] = U;
    counts[1] = T;
    counts[2] = hdr[H_SLOTS];
    counts[3] = hdr[H_CTAS];
    struct Copy {
        void* dst;
        int64_t off;
        int64_t bytes;
    } copies[] = {
        {cta_ptr, L.off_cta_ptr, (int64_t)(L.N + 1) * 4},
        {tasks, L.off_tasks, (int64_t)T * 16},
        {units, L.off_units, (int64_t)U * 16},
        {unit_ntiles, L.off_ntiles, (int64_t)U * 4},
        {unit_nsplit, L.off_nsplit, (int64_t)U * 4},
        {unit_slot0, L.off_slot0, (int64_t)U * 4},
        {active, L.off_active, L.has_mask ? (int64_t)U * L.max_kv_tiles * 4 : 0},
    };
    for (const Copy& c : copies) {
        if (!c.dst || c.bytes <= 0) continue;
        if (cudaMemcpyAsync(c.dst, ws + c.off, (size_t)c.bytes, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess)
            return PA_ERR_CUDA;
    }
    return cudaStreamSynchronize(s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_last_device_error(const void* assign_ws, int32_t* code, void* stream) {
    if (!assign_ws || !code) return PA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t v = 0;
    const char* ws = reinterpret_cast<const char*>(assign_ws);  // header is at offset 0
    if (cudaMemcpyAsync(&v, ws + H_ERROR * 4, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return PA_ERR_CUDA;
    *code = v;
    if (v == PA_DEV_OK) return PA_OK;
    if (v == PA_DEV_WAIT_TIMEOUT) return PA_ERR_TIMEOUT;
    return PA_ERR_DEVICE_CHECK;
}

}  // extern "C"
