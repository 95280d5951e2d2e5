// pa_assign.cu -- the Assign pass: units, tile lists, load-balanced task map.
//
// "基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 (Assign: cut every KV
// sequence into tiles and build a task map that balances the work per CTA),
// 三.3 (均分调度: every CTA carries a similar amount of KV work; a GPU-resident
// task map drives the persistent compute CTAs), 二.1 (the block mask is
// compacted into an ascending active-KV-tile list with a warp ballot,
// popcount and prefix rank).
//
// Prefill mode: three launches on the caller's stream:
//   1. assign_seq_kernel   (1 CTA)      validate lengths; cu_q and the first
//                                       unit of every sequence (block scans)
//   2. assign_units_kernel (warp/unit)  unit -> (b, hk, q0, nq), tile count,
//                                       active-tile list (ballot + popc)
//   3. assign_map_kernel   (1 CTA)      cost prefix, CTA ownership in closed
//                                       form, tasks, split slots, cta_ptr
// Decode mode: one launch (assign_decode_kernel, 1 CTA) does all three --
// its units are (b, hk) in order, so nothing needs a search.
// Closed form used in 3: with C the total cost and N CTAs, CTA c owns
// [a_c, a_{c+1}), a_c = floor(c*C/N); the owner of cost x (0 <= x < C) is
// floor(((x+1)*N - 1) / C).
#include <mutex>

#include "pa_internal.cuh"

namespace pa {

namespace {

constexpr int kScanThreads = 1024;

// Block-wide exclusive scan of one int64 per thread; *total gets the sum.
__device__ int64_t block_exscan(int64_t v, int64_t* total, int64_t* sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t w = lane < nwarps ? sm[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sm[lane] = w;  // inclusive per warp
    }
    __syncthreads();
    int64_t excl = (x - v) + (warp > 0 ? sm[warp - 1] : 0);
    *total = sm[nwarps - 1];
    __syncthreads();
    return excl;
}

// The same for three values at once (one set of barriers); sm: 3 * 32 int64.
__device__ void block_exscan3(const int64_t (&v)[3], int64_t (&excl)[3], int64_t (&total)[3],
                              int64_t* sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int64_t x[3] = {v[0], v[1], v[2]};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            int64_t y = __shfl_up_sync(0xffffffffu, x[i], o);
            if (lane >= o) x[i] += y;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int i = 0; i < 3; ++i) sm[i * 32 + warp] = x[i];
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            int64_t w = lane < nwarps ? sm[i * 32 + lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int64_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            sm[i * 32 + lane] = w;  // inclusive per warp
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        excl[i] = (x[i] - v[i]) + (warp > 0 ? sm[i * 32 + warp - 1] : 0);
        total[i] = sm[i * 32 + nwarps - 1];
    }
    __syncthreads();
}

__device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// query tokens of a sequence that this map covers (see WsLayout::cls)
__device__ __forceinline__ int class_ql(const WsLayout& L, int q) {
    if (L.cls == 1) return q <= L.small_q ? q : 0;
    if (L.cls == 2) return q > L.small_q ? q : 0;
    return q;
}

__device__ __forceinline__ int units_of_seq(const WsLayout& L, int ql) {
    if (L.mode == PA_MODE_DECODE) return L.Hkv;
    return L.Hkv * (int)ceil_div64(ql, L.qtok);
}

__global__ void __launch_bounds__(kScanThreads)
assign_seq_kernel(WsLayout L, const int32_t* __restrict__ ctx, const int32_t* __restrict__ ql,
                  void* ws) {
    __shared__ int64_t sm[32];
    int32_t* header = ws_ptr<int32_t>(ws, L.off_header);
    int32_t* cu_q = ws_ptr<int32_t>(ws, L.off_cu_q);
    int32_t* seq_u0 = ws_ptr<int32_t>(ws, L.off_seq_unit0);
    const int tid = threadIdx.x;
    const int chunk = (L.B + kScanThreads - 1) / kScanThreads;
    const int b0 = min(L.B, tid * chunk), b1 = min(L.B, b0 + chunk);
    int64_t sq = 0, su = 0;
    int bad = 0;
    for (int b = b0; b < b1; ++b) {
        int q = ql[b], c = ctx[b];
        if (q < 0 || c < q || c > L.max_ctx || q > L.max_q_len) bad = 1;
        q = max(0, min(q, L.max_q_len));
        sq += q;
        su += units_of_seq(L, class_ql(L, q));
    }
    int64_t tq, tu;
    int64_t eq = block_exscan(sq, &tq, sm);
    int64_t eu = block_exscan(su, &tu, sm);
    for (int b = b0; b < b1; ++b) {
        int q = max(0, min(ql[b], L.max_q_len));
        cu_q[b] = (int32_t)eq;
        seq_u0[b] = (int32_t)eu;
        eq += q;
        eu += units_of_seq(L, class_ql(L, q));
    }
    bad = __syncthreads_or(bad);
    if (tid == 0) {
        cu_q[L.B] = (int32_t)tq;
        seq_u0[L.B] = (int32_t)tu;
        bad = bad || tq != L.total_q || tu > L.unit_cap;
        for (int i = 0; i < kHeaderWords; ++i) header[i] = 0;
        header[H_UNITS] = bad ? 0 : (int32_t)tu;
        header[H_ERROR] = bad ? PA_DEV_BAD_LENGTHS : PA_DEV_OK;
        header[H_CTAS] = L.N;
        header[H_MODE] = L.mode;
    }
}

__global__ void assign_units_kernel(WsLayout L, const int32_t* __restrict__ ctx,
                                    const int32_t* __restrict__ ql,
                                    const uint8_t* __restrict__ mask, void* ws) {
    const int32_t* header = ws_ptr<int32_t>(ws, L.off_header);
    const int32_t* seq_u0 = ws_ptr<int32_t>(ws, L.off_seq_unit0);
    int4* units = ws_ptr<int4>(ws, L.off_units);
    int32_t* ntiles = ws_ptr<int32_t>(ws, L.off_ntiles);
    int32_t* active = ws_ptr<int32_t>(ws, L.off_active);
    const int lane = threadIdx.x & 31;
    const int u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int U = header[H_UNITS];
    if (u >= U) return;
    // sequence owning unit u: the last b with seq_u0[b] <= u
    int lo = 0, hi = L.B;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (seq_u0[mid] <= u) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int q_b = class_ql(L, max(0, min(ql[b], L.max_q_len))), c_b = ctx[b];
    const int nqt = L.mode == PA_MODE_DECODE ? 1 : (int)ceil_div64(q_b, L.qtok);
    const int local = u - seq_u0[b];
    const int hk = local / nqt, qt = local % nqt;
    int q0, nq;
    int64_t keys;
    if (L.mode == PA_MODE_DECODE) {
        q0 = 0;
        nq = q_b;
        keys = nq > 0 ? c_b : 0;
    } else {
        q0 = qt * L.qtok;
        nq = min(L.qtok, q_b - q0);
        keys = (int64_t)c_b - q_b + q0 + nq;
    }
    const int nreach = (int)ceil_div64(keys, L.kv_tile);
    // with a sliding window the unit's tiles start at the first one its first
    // query (position ctx - q_len + q0) can see
    const int first = nq > 0 ? window_first_tile(L.window, c_b - q_b + q0, L.kv_tile) : 0;
    int n = nreach - first;
    if (L.has_mask) {
        // active-KV-tile compaction: ballot the kept predicates of 32 tiles,
        // popcount them, write each kept tile at its prefix rank
        const int mq = q0 / kMaskTile;
        const uint8_t* mrow = mask + ((int64_t)b * L.mask_q_tiles + mq) * L.mask_kv_tiles;
        int32_t* out = active + (int64_t)u * L.max_kv_tiles;
        int base = 0;
        for (int k0 = first; k0 < nreach; k0 += 32) {
            const int kt = k0 + lane;
            const bool keep = kt < nreach && kt < L.mask_kv_tiles && mq < L.mask_q_tiles &&
                              mrow[kt] != 0;
            const uint32_t bal = __ballot_sync(0xffffffffu, keep);
            if (keep) out[base + __popc(bal & ((1u << lane) - 1u))] = kt;
            base += __popc(bal);
        }
        n = base;
    }
    if (lane == 0) {
        units[u] = make_int4(b, hk, q0, nq);
        ntiles[u] = n;
    }
}

__device__ __forceinline__ int64_t unit_weight(const WsLayout& L, int nq) {
    int64_t w = ceil_div64((int64_t)L.G * nq, L.balance_rows);
    return w < 1 ? 1 : w;
}

// Visit the CTAs owning tiles of a unit (cost prefix P, n tiles of weight w):
// f(cta, t_lo, t_hi) for every CTA with at least one of them.
template <typename F>
__device__ __forceinline__ void for_each_owner(int64_t P, int n, int64_t w, int64_t C, int N,
                                               F f) {
    if (n <= 0) return;
    const int64_t x0 = P, x1 = P + (int64_t)(n - 1) * w;
    const int c0 = (int)(((x0 + 1) * N - 1) / C);
    const int c1 = (int)(((x1 + 1) * N - 1) / C);
    for (int c = c0; c <= c1; ++c) {
        const int64_t a = (int64_t)c * C / N, a1 = (int64_t)(c + 1) * C / N;
        const int64_t tlo = a <= P ? 0 : ceil_div64(a - P, w);
        int64_t thi = ceil_div64(a1 - P, w);
        if (thi > n) thi = n;
        if (thi > tlo) f(c, (int)tlo, (int)thi);
    }
}

// Units whose tile count, weight and split count the map pass keeps in
// shared memory (3 x 4 bytes each); larger maps read them from the workspace.
constexpr int kMapCacheUnits = 12288;
constexpr int kMapCacheBytes = kMapCacheUnits * 12;

// Cost prefix, ownership, tasks, split slots, combine fix list and cta_ptr,
// for the U units already written (one CTA; sm: 3 * 32 int64 of shared
// memory; cache: kMapCacheBytes of shared memory or nullptr).  Each thread
// owns a contiguous run of units; with the cache, the units' tile counts and
// weights are staged once with coalesced loads, and a unit's prefix is
// rebuilt from the thread's running sum instead of being read back.
__device__ void assign_map_body(const WsLayout& L, void* ws, int64_t* sm, int32_t* cache) {
    int32_t* header = ws_ptr<int32_t>(ws, L.off_header);
    const int4* units = ws_ptr<int4>(ws, L.off_units);
    const int32_t* ntiles = ws_ptr<int32_t>(ws, L.off_ntiles);
    int64_t* prefix = ws_ptr<int64_t>(ws, L.off_prefix);
    int32_t* nsplit = ws_ptr<int32_t>(ws, L.off_nsplit);
    int32_t* slot0 = ws_ptr<int32_t>(ws, L.off_slot0);
    int4* tasks = ws_ptr<int4>(ws, L.off_tasks);
    int32_t* task_cta = ws_ptr<int32_t>(ws, L.off_task_cta);
    int32_t* cta_ptr = ws_ptr<int32_t>(ws, L.off_cta_ptr);
    int32_t* fix = ws_ptr<int32_t>(ws, L.off_fix);
    int32_t* done = ws_ptr<int32_t>(ws, L.off_done);
    const int U = header[H_UNITS];
    const int N = L.N;
    const int tid = threadIdx.x;
    const int chunk = (U + kScanThreads - 1) / kScanThreads;
    const int u0 = min(U, tid * chunk), u1 = min(U, u0 + chunk);

    const bool cached = cache != nullptr && U <= kMapCacheUnits;
    int32_t* c_n = cache;                                   // [U] tiles
    int32_t* c_w = cache + (cached ? U : 0);                // [U] weight
    int32_t* c_s = cache + (cached ? 2 * U : 0);            // [U] tasks (splits)
    if (cached) {
        for (int u = tid; u < U; u += blockDim.x) {
            c_n[u] = ntiles[u];
            c_w[u] = (int32_t)unit_weight(L, units[u].w);
        }
        __syncthreads();
    }
    auto n_of = [&](int u) -> int { return cached ? c_n[u] : ntiles[u]; };
    auto w_of = [&](int u) -> int64_t { return cached ? (int64_t)c_w[u] : unit_weight(L, units[u].w); };
    auto nq_of = [&](int u) -> int { return units[u].w; };

    // cost prefix
    int64_t cost = 0;
    // a unit with tiles also costs L.unit_cost, ahead of its first tile
    const int64_t h = L.unit_cost;
    for (int u = u0; u < u1; ++u) {
        const int n = n_of(u);
        cost += (n > 0 ? h : 0) + (int64_t)n * w_of(u);
    }
    int64_t C;
    const int64_t run0 = block_exscan(cost, &C, sm);

    // tasks per unit, split slots, units the combine pass must finish
    int64_t cnt[3] = {0, 0, 0};   // tasks, split slots, fix-list entries
    {
        int64_t run = run0;
        for (int u = u0; u < u1; ++u) {
            const int n = n_of(u);
            const int64_t w = w_of(u);
            prefix[u] = run;
            const int64_t hu = n > 0 ? h : 0;
            int S = 0;
            for_each_owner(run + hu, n, w, C, N, [&](int, int, int) { ++S; });
            run += hu + (int64_t)n * w;
            nsplit[u] = S;
            // completion counters of the in-kernel finalizer of split units
#pragma unroll
            for (int i = 0; i < kDoneWords; ++i) done[(int64_t)u * kDoneWords + i] = 0;
            if (cached) c_s[u] = S;
            cnt[0] += S;
            cnt[1] += S > 1 ? S : 0;
            cnt[2] += (S != 1 && nq_of(u) > 0) ? 1 : 0;
        }
    }
    int64_t base[3], tot[3];
    block_exscan3(cnt, base, tot, sm);
    const int64_t T = tot[0], Sl = tot[1], F = tot[2];
    {
        int64_t run = run0, t_run = base[0], s_run = base[1], f_run = base[2];
        for (int u = u0; u < u1; ++u) {
            const int n = n_of(u);
            const int64_t w = w_of(u);
            const int S = cached ? c_s[u] : nsplit[u];
            const int s0 = S > 1 ? (int)s_run : -1;
            slot0[u] = s0;
            int k = 0;
            const int64_t hu = n > 0 ? h : 0;
            for_each_owner(run + hu, n, w, C, N, [&](int c, int tlo, int thi) {
                tasks[t_run + k] = make_int4(u, tlo, thi, S > 1 ? s0 + k : -1);
                task_cta[t_run + k] = c;
                ++k;
            });
            run += hu + (int64_t)n * w;
            t_run += S;
            s_run += S > 1 ? S : 0;
            if (S != 1 && nq_of(u) > 0) fix[f_run++] = u;
        }
    }
    __syncthreads();
    // cta_ptr[c] = number of tasks owned by CTAs < c.  task_cta is sorted, so
    // task k starts every CTA in (task_cta[k-1], task_cta[k]]; CTAs after the
    // last task's start at T.
    for (int k = tid; k < (int)T; k += blockDim.x) {
        const int c = task_cta[k];
        const int prev = k > 0 ? task_cta[k - 1] : -1;
        for (int cc = prev + 1; cc <= c; ++cc) cta_ptr[cc] = k;
    }
    {
        const int last = T > 0 ? task_cta[T - 1] : -1;
        for (int c = last + 1 + tid; c <= N; c += blockDim.x) cta_ptr[c] = (int)T;
    }
    if (tid == 0) {
        header[H_TASKS] = (int32_t)T;
        header[H_SLOTS] = (int32_t)Sl;
        header[H_FIX] = (int32_t)F;
    }
}

__global__ void __launch_bounds__(kScanThreads) assign_map_kernel(WsLayout L, void* ws) {
    __shared__ int64_t sm[3 * 32];
    extern __shared__ int32_t map_cache[];   // kMapCacheBytes
    grid_launch_dependents();   // the compute kernel may become resident meanwhile
    assign_map_body(L, ws, sm, map_cache);
}

// Decode mode in one launch: units are (b, hk) in order, Hkv per sequence,
// so the three passes need no search and fit one CTA.
__global__ void __launch_bounds__(kScanThreads)
assign_decode_kernel(WsLayout L, const int32_t* __restrict__ ctx, const int32_t* __restrict__ ql,
                     void* ws) {
    __shared__ int64_t sm[3 * 32];
    grid_launch_dependents();   // the compute kernel may become resident meanwhile
    int32_t* header = ws_ptr<int32_t>(ws, L.off_header);
    int32_t* cu_q = ws_ptr<int32_t>(ws, L.off_cu_q);
    int32_t* seq_u0 = ws_ptr<int32_t>(ws, L.off_seq_unit0);
    int4* units = ws_ptr<int4>(ws, L.off_units);
    int32_t* ntiles = ws_ptr<int32_t>(ws, L.off_ntiles);
    const int tid = threadIdx.x;
    // lengths: validate, cu_q
    const int chunk = (L.B + kScanThreads - 1) / kScanThreads;
    const int b0 = min(L.B, tid * chunk), b1 = min(L.B, b0 + chunk);
    int64_t sq = 0;
    int bad = 0;
    for (int b = b0; b < b1; ++b) {
        int q = ql[b], c = ctx[b];
        if (q < 0 || c < q || c > L.max_ctx || q > L.max_q_len) bad = 1;
        sq += max(0, min(q, L.max_q_len));
    }
    int64_t tq;
    int64_t eq = block_exscan(sq, &tq, sm);
    for (int b = b0; b < b1; ++b) {
        cu_q[b] = (int32_t)eq;
        seq_u0[b] = b * L.Hkv;
        eq += max(0, min(ql[b], L.max_q_len));
    }
    const int64_t tu = (int64_t)L.B * L.Hkv;
    bad = __syncthreads_or(bad) || tq != L.total_q || tu > L.unit_cap;
    if (tid == 0) {
        cu_q[L.B] = (int32_t)tq;
        seq_u0[L.B] = (int32_t)tu;
        for (int i = 0; i < kHeaderWords; ++i) header[i] = 0;
        header[H_UNITS] = bad ? 0 : (int32_t)tu;
        header[H_ERROR] = bad ? PA_DEV_BAD_LENGTHS : PA_DEV_OK;
        header[H_CTAS] = L.N;
        header[H_MODE] = L.mode;
    }
    // units (b, hk): all q_len[b] queries over all ctx[b] keys
    const int U = bad ? 0 : (int)tu;
    for (int u = tid; u < U; u += blockDim.x) {
        const int b = u / L.Hkv, hk = u - b * L.Hkv;
        const int nq = class_ql(L, ql[b]);
        const int64_t keys = nq > 0 ? ctx[b] : 0;
        units[u] = make_int4(b, hk, 0, nq);
        // with a sliding window the unit's tiles start at the first one its
        // first query (position ctx - nq) can see
        const int first = nq > 0 ? window_first_tile(L.window, ctx[b] - nq, L.kv_tile) : 0;
        ntiles[u] = (int)ceil_div64(keys, L.kv_tile) - first;
    }
    __syncthreads();   // header, units and tiles visible to the whole CTA
    assign_map_body(L, ws, sm, nullptr);
}

}  // namespace

cudaError_t launch_assign(const WsLayout& L, const int32_t* ctx, const int32_t* ql,
                          const uint8_t* mask, void* ws, cudaStream_t stream) {
    if (L.mode == PA_MODE_DECODE) {
        assign_decode_kernel<<<1, kScanThreads, 0, stream>>>(L, ctx, ql, ws);
        return cudaGetLastError();
    }
    assign_seq_kernel<<<1, kScanThreads, 0, stream>>>(L, ctx, ql, ws);
    const int warps = 8;
    const int grid = (L.unit_cap + warps - 1) / warps;
    assign_units_kernel<<<grid > 0 ? grid : 1, warps * 32, 0, stream>>>(L, ctx, ql, mask, ws);
    // the shared-memory opt-in, once per device (host threads may race here)
    static std::mutex attr_mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(attr_mu);
        if (dev < 0 || dev >= 64 || !attr_set[dev]) {
            e = cudaFuncSetAttribute(assign_map_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kMapCacheBytes);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) attr_set[dev] = true;
        }
    }
    assign_map_kernel<<<1, kScanThreads, kMapCacheBytes, stream>>>(L, ws);
    return cudaGetLastError();
}

}  // namespace pa
