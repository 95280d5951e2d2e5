// pa_prefill.cu -- persistent causal / block-sparse prefill on tcgen05 + TMEM.
//
// "基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 Prefill (tile
// scheduling by batch, head and query tile; pipelined TMA loads of Q/K/V into
// multi-stage shared memory; QK, causal mask, fp32 online softmax, PV;
// epilogue normalisation), 二.1 (only the KV tiles of the active-tile list
// are loaded and multiplied), 二.2 (warp specialisation: a producer resolves
// page ids and issues K then V by TMA while the consumers compute; two
// consumer groups each own one half of the query tile; K and V buffers are
// released separately, K right after QK).  "vLLM Triton Attention Backend
// Deep Dive": Q blocks pack the G q heads of one KV head into one MMA tile;
// the persistent grid is fixed at the SM count.
//
// In a batch without a block mask the sequences of at most 16 rows (G x
// q_len: the decode steps of a mixed batch) never reach this kernel: they
// run on the decode kernel over a task map of their own (pa_api.cu).
//
// GB300 design (one CTA per SM, 384 threads = 3 warpgroups).  A unit is up
// to 256 query rows (G heads x 256/G tokens), computed as two 128-row halves
// that share every K/V tile.  Registers: of the 168 per thread the block is
// launched with, setmaxnreg leaves warpgroup 0 with 88 and gives the two
// softmax warpgroups 200 each: 128*88 + 256*200 <= 384*168.
//   warp 0      TMA producer: the unit's Q halves once per task, then for
//               every active 128-token KV tile its K, one copy per page,
//               into its own entry of a ring (128-byte swizzle, rows stored
//               by 8-token group); warp 3 fills the V entries the same way.
//   warps 1-2   warp 1 allocates the 512 TMEM columns; lane 0 of warp 1+h
//               issues every MMA of half h:
//               S_h = Q_h K^T (M=128, N=128, K=D, both operands K-major in
//               shared memory) into TMEM, and O_h += P_h V (M=128, N=D,
//               K=128) with P_h read from TMEM (written over S_h by the
//               softmax) and V read MN-major from shared memory, so V is
//               never transposed.  Per tile j each issuer runs
//                 PV_h(j), QK_h(j+1)
//               so the tensor cores work on one half while the other half's
//               softmax runs; MMAs of one thread execute in issue order,
//               which keeps QK_h(j+1) from overwriting P_h(j) before PV_h(j)
//               has read it.  Warp 1 also zeroes V rows past the context.
//   warp 3      fills the V entries of the ring (see warp 0); with E4M3 K/V
//               it converts V tiles to f16 instead, and warp 0 fills every
//               entry.
//   warps 4-7   softmax for half 0, warps 8-11 for half 1: thread = query row
//               = TMEM lane.  Reads its S row (tcgen05.ld), applies the
//               causal / context / window mask on the tiles that need it
//               (a warp-uniform test per tile), keeps the running max lazily (O is
//               rescaled in TMEM only when the max grows by more than 2^8),
//               writes P (bf16) back into TMEM, and at the end of the task
//               normalises O and writes the output row (or split partial)
//               and its LSE.
// TMEM columns: half h uses [256h, 256h+128) for S (and P over its first 64
// columns) and [256h+128, 256h+128+D) for O.
#include "pa_internal.cuh"

namespace pa {

struct PrefillParams {
    WsLayout L;
    const int32_t* block_table;
    const int32_t* ctx;
    const int32_t* ql;
    void* ws;
    float* part_o;
    float* part_lse;
    __nv_bfloat16* out;
    float* lse;
    int32_t page_size;
    int32_t num_pages;
    int32_t max_pages_per_seq;
    int32_t rows_per_box;    // min(page_size, 64)
    int32_t boxes_per_tile;  // 128 / rows_per_box
    // coordinates of a grouped K/V box (bf16, D = 128): chunk = kv_chunk_mul *
    // head; last coordinate = page * kv_page_mul + head * kv_head_add
    int32_t kv_chunk_mul;
    int32_t kv_page_mul;
    int32_t kv_head_add;
    int32_t test_skip_it;    // test hook: CTA 0 leaves this K/V ring entry unfilled (-1 none)
    int32_t store_v8;        // bit 0: out, bit 1: the partials are 32-byte aligned
    // E4M3 Q/K/V: Q scale (one, or one per (token, q head)), one K and one V scale
    const float* q_scale;
    const float* k_scale;
    const float* v_scale;
    int32_t q_scale_per_row;
    int64_t* trace;          // task trace (pa_set_task_trace), or nullptr
    int64_t trace_cap;
    float sm_scale;
    uint64_t wait_limit_ns;
};

template <int D, bool FP8 = false>
struct PrefillCfg {
    static constexpr int kElem = FP8 ? 1 : 2;        // bytes per Q/K/V element
    static constexpr int kHalves = D * kElem / 128;  // 128-byte column blocks of a row
    static constexpr int kRegion = 128 * 128;        // 128 rows x 128 bytes
    static constexpr int kQTileBytes = kHalves * kRegion;
    static constexpr int kQBytes = 2 * kQTileBytes;  // two 128-row halves
    static constexpr int kKVBytes = kHalves * kRegion;
    // K/V tiles are stored by 8-token group: group g holds its kHalves
    // column blocks of 8 rows x 128 bytes (1 KB each) at g * kGroupStride.
    // One tensor copy of a page then fills whole groups of both column
    // blocks, and the 8-row groups of each column block still sit at one
    // uniform stride, as the MMA descriptors need.  With one column block
    // (E4M3, or bf16 with D = 64) this is the plain row-major tile.
    static constexpr int kGroupStride = kHalves * 1024;
    // ring entries (each a K or a V tile)
    static constexpr int kEntries = FP8 ? 6 : (D == 128 ? 5 : 8);
    // producer warps (warp 0, and warp 3 for bf16); for E4M3 warp 3 instead
    // turns each V tile into f16, double-buffered, for an f16 PV
    static constexpr int kProducers = FP8 ? 1 : 2;
    static constexpr int kVhBytes = 2 * kRegion;     // f16 V tile: two 64-dim column blocks
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + kQBytes;
    static constexpr int kOffVh = kOffKV + kEntries * kKVBytes;
    static constexpr int kOffBar = kOffVh + (FP8 ? 2 * kVhBytes : 0);
    static constexpr int kNumBars = 2 + 2 * kEntries + 9 + (FP8 ? 4 : 0);
    // after the TMEM slot and the abort flag: the last phase armed with a copy,
    // per ring entry, and that of the Q buffer
    static constexpr int kOffArmed = kOffBar + kNumBars * 8 + 16;
    static constexpr int kSmemBytes = kOffArmed + (4 * (kEntries + 1) + 15) / 16 * 16 + 1024;
    static constexpr int kThreads = 384;
    static constexpr int kRegsLaunch = 168;          // 65536 / 384, rounded down to 8
    static constexpr int kRegsProducer = 88;
    static constexpr int kRegsSoftmax = 200;
    static_assert(128 * kRegsProducer + 256 * kRegsSoftmax <= kThreads * kRegsLaunch,
                  "register split exceeds the launch allocation");
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kSmemBytes <= 232448, "shared memory");
};

__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// WINDOW: the instantiation that takes a sliding window; the other one
// carries no window arithmetic in its softmax.  FP8: E4M3 Q, K and V
// ("基于Triton-TLE…", 二: FP8 prefill) -- QK^T on kind::f8f6f4 (K = 32 per
// instruction) straight from the E4M3 Q and K tiles (both K-major); the
// softmax scales S by q_scale * k_scale and writes its f16 exponentials into
// tensor memory as they are; warp 3 (not a producer here) turns every E4M3
// V tile into an f16 tile (exact), double-buffered, and PV runs as a
// kind::f16 MMA (f16 P, f16 V, MN-major).  v_scale is applied to O in the
// epilogue.
template <int D, bool WINDOW, bool FP8>
__global__ void __launch_bounds__(384, 1)
prefill_kernel(const __grid_constant__ PrefillParams P, const __grid_constant__ CUtensorMap tmq,
               const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    using Cfg = PrefillCfg<D, FP8>;
    static_assert(!FP8 || D == 128, "E4M3 prefill: head_dim 128");
    constexpr int E = Cfg::kEntries;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
    uint64_t* q_full = bars + 0;
    uint64_t* q_empty = bars + 1;
    uint64_t* kv_full = bars + 2;             // [E]
    uint64_t* kv_empty = kv_full + E;         // [E]
    uint64_t* s_full = kv_empty + E;          // [2]
    uint64_t* p_full = s_full + 2;            // [2]
    uint64_t* o_done = p_full + 2;            // [2]
    uint64_t* o_free = o_done + 2;            // [2]
    uint64_t* mma_done = o_free + 2;
    uint64_t* vh_full = mma_done + 1;         // [2] E4M3: f16 V buffer written
    uint64_t* vh_empty = vh_full + 2;         // [2] E4M3: f16 V buffer read by both PVs
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* armed = reinterpret_cast<int*>(smem + Cfg::kOffArmed);   // [E] entries, then Q
    const WsLayout& L = P.L;
    int32_t* header = ws_ptr<int32_t>(P.ws, L.off_header);
    int32_t* err_hdr = ws_ptr<int32_t>(P.ws, L.off_err_header);   // device faults
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t lim = P.wait_limit_ns;

    grid_dependency_wait();   // Assign's task map is complete
    if (header[H_CTAS] != (int)gridDim.x) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(err_hdr, PA_DEV_BAD_LENGTHS);
        return;
    }
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 2);                 // one commit from each MMA warp
        for (int e = 0; e < E; ++e) {
            mbar_init(&kv_full[e], 1);      // armed by the warp that fills it
            mbar_init(&kv_empty[e], 2);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&s_full[h], 1);
            mbar_init(&p_full[h], 128);
            mbar_init(&o_done[h], 1);
            mbar_init(&o_free[h], 128);
        }
        mbar_init(mma_done, 2);
        if constexpr (FP8) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(&vh_full[b], 1);
                mbar_init(&vh_empty[b], 2);      // one commit from each MMA warp
            }
        }
        *abort_flag = 0;
        for (int i = 0; i < E + 1; ++i) armed[i] = -1;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (mbar_try_wait(bar, parity)) return;   // the usual case, checked first
        if (*abort_flag) return;
        if (!mbar_wait_or_abort(bar, parity, lim, abort_flag)) {
            *abort_flag = 1;
            set_device_error(err_hdr, PA_DEV_WAIT_TIMEOUT);
        }
    };

    const int32_t* cta_ptr = ws_ptr<int32_t>(P.ws, L.off_cta_ptr);
    const int4* tasks = ws_ptr<int4>(P.ws, L.off_tasks);
    const int4* units = ws_ptr<int4>(P.ws, L.off_units);
    const int32_t* cu_q = ws_ptr<int32_t>(P.ws, L.off_cu_q);
    const int32_t* active = ws_ptr<int32_t>(P.ws, L.off_active);
    const int k_begin = cta_ptr[blockIdx.x], k_end = cta_ptr[blockIdx.x + 1];
    const int G = L.G, Hq = L.Hq;
    const int half_tokens = kPrefillHalfRows / G;   // query tokens per 128-row half

    // KV tile at position t of unit u's list: the active list with a block
    // mask; else the tiles from the first one the unit's first query can see
    // (position p0 = ctx - q_len + q0; 0 without a sliding window) onwards
    auto tile_of = [&](int u, int t, int p0) -> int {
        return L.has_mask ? active[(int64_t)u * L.max_kv_tiles + t]
                          : t + (WINDOW ? window_first_tile(L.window, p0, kPrefillTile) : 0);
    };

    if (warp < 4) {
      regs_dec<Cfg::kRegsProducer>();
      if (warp == 0 || (warp == 3 && !FP8)) {
        // --------------------------------------------------------- producers
        // A tensor copy holds its issuing thread for hundreds of cycles, so
        // with two producer warps (bf16) warp 0 fills the K entries and warp 3
        // the V entries, each issuing one page per lane: the two copy chains
        // run side by side.  With one (E4M3) warp 0 fills both.  Warp 0 also
        // loads Q.
        const int pw = warp == 0 ? 0 : 1;
        constexpr int kP = Cfg::kProducers;
        if (lane == 0) {
            prefetch_tmap(&tmq);
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
        }
        const int ps = P.page_size, rpb = P.rows_per_box, nbox = P.boxes_per_tile;
        const uint32_t box_bytes = (uint32_t)rpb * 128u * Cfg::kHalves;
        int e_it = 0, task_it = 0;
        TaskRec mine;
        for (int k = k_begin; k < k_end; ++k, ++task_it) {
            if (((k - k_begin) & 31) == 0)
                mine = load_task_rec(tasks, units, P.ctx, P.ql, cu_q, k + lane, k_end);
            const TaskRec rec = shfl_task_rec(mine, (k - k_begin) & 31);
            const int u = rec.tk.x, b = rec.un.x, hk = rec.un.y, q0 = rec.un.z;
            const int H = G * rec.un.w > kPrefillHalfRows ? 2 : 1;
            const int ctx_b = rec.ctx;
            const int npg = (ctx_b + ps - 1) / ps;
            const int32_t* bt_row = P.block_table + (int64_t)b * P.max_pages_per_seq;
            if (pw == 0) wait(q_empty, (uint32_t)(task_it & 1) ^ 1u);
            if (pw == 0) {
                // lane 0 arms the Q buffer, then lane h * kHalves + c copies half
                // h's column block c (one tensor copy per lane)
                const bool go = __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
                if (lane == 0 && go) {
                    armed[E] = task_it;
                    mbar_arrive_expect_tx(q_full, (uint32_t)H * Cfg::kQTileBytes);
                }
                __syncwarp();
                if (go && lane < H * Cfg::kHalves) {
                    const int h = lane / Cfg::kHalves, c = lane % Cfg::kHalves;
                    tma_load_3d(smem + Cfg::kOffQ + h * Cfg::kQTileBytes + c * Cfg::kRegion, &tmq,
                                q_full, (128 / Cfg::kElem) * c, hk * G,
                                rec.cuq + q0 + h * half_tokens);
                }
            }
            __syncwarp();
            // block-table window: 32 page ids read lane-parallel; the next
            // window's ids are requested one window ahead
            int win_lo = -(1 << 30), win_val = -1;
            int nxt_lo = -(1 << 30), nxt_val = -1;
            const int p0 = ctx_b - rec.ql + q0;
            for (int t = rec.tk.y; t < rec.tk.z; ++t) {
                const int kt = tile_of(u, t, p0);
                uint32_t bytes = 0;
                int pg[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    pg[j] = -1;
                    if (j >= nbox) continue;
                    const int tok0 = kt * kPrefillTile + j * rpb;
                    if (tok0 >= ctx_b) continue;
                    const int lp = tok0 / ps;
                    if (lp - win_lo < 0 || lp - win_lo >= 32) {
                        win_val = (lp == nxt_lo) ? nxt_val
                                                 : ((lp + lane < npg) ? __ldg(bt_row + lp + lane) : -1);
                        win_lo = lp;
                        nxt_lo = lp + 32;
                        nxt_val = (nxt_lo + lane < npg) ? __ldg(bt_row + nxt_lo + lane) : -1;
                    }
                    int page = __shfl_sync(0xffffffffu, win_val, lp - win_lo);
                    if (page < 0 || page >= P.num_pages) {
                        if (lane == 0) set_device_error(err_hdr, PA_DEV_BAD_PAGE);
                        page = -1;
                    }
                    pg[j] = page;
                    if (page >= 0) bytes += box_bytes;
                }
                // K first (QK needs it first), then V, each into its own ring entry
#pragma unroll
                for (int kv = 0; kv < 2; ++kv, ++e_it) {
                    if (kP == 2 && kv != pw) continue;   // the other warp's entry
                    const int e = e_it % E;
                    wait(&kv_empty[e], (uint32_t)((e_it / E) & 1) ^ 1u);
                    // lane 0 arms the entry; then lane j issues box j: both column
                    // blocks of its tokens in one copy, laid out by 8-token group.
                    // test hook: CTA 0 leaves one entry unfilled, so that the MMA
                    // warps' bounded wait runs out (the abort path, without a fault)
                    const bool skip = P.test_skip_it == e_it && blockIdx.x == 0;
                    const bool go = __shfl_sync(0xffffffffu, *abort_flag, 0) == 0 && !skip;
                    if (lane == 0 && go) {
                        armed[e] = e_it / E;
                        mbar_arrive_expect_tx(&kv_full[e], bytes);
                    }
                    __syncwarp();
                    if (go && lane < 8) {
                        const int j = lane;
                        int page = -1;
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj)
                            if (jj == j) page = pg[jj];
                        if (page >= 0) {
                            const int slot0 = (kt * kPrefillTile + j * rpb) % ps;
                            uint8_t* dst = smem + Cfg::kOffKV + e * Cfg::kKVBytes +
                                           (j * rpb / 8) * Cfg::kGroupStride;
                            if constexpr (Cfg::kHalves == 2)
                                tma_load_5d(dst, kv ? &tmv : &tmk, &kv_full[e], 0, 0,
                                            hk * P.kv_chunk_mul, slot0 / 8,
                                            page * P.kv_page_mul + hk * P.kv_head_add);
                            else
                                tma_load_4d(dst, kv ? &tmv : &tmk, &kv_full[e], 0, slot0, hk,
                                            page);
                        }
                    }
                    __syncwarp();
                }
            }
        }
    } else if (FP8 && warp == 3) {
        // --------------------------------------------- V converter (E4M3)
        // Each V tile, as it lands in the ring, becomes an f16 tile in one of
        // two buffers laid out as a bf16 V tile would be (two 64-dim column
        // blocks, 128-byte swizzle), so that PV runs as an f16 MMA with P in
        // f16 -- the softmax then writes its f16 exponentials as they are.
        // Rows of keys past the context are written as zeros (E4M3 NaN codes
        // in stale slots would otherwise poison 0 * V).  The ring entry goes
        // back to the producer as soon as its bytes are in registers.
        int e_it = 0, vt = 0;
        TaskRec mine;
        for (int k = k_begin; k < k_end; ++k) {
            if (((k - k_begin) & 31) == 0)
                mine = load_task_rec(tasks, units, P.ctx, P.ql, cu_q, k + lane, k_end);
            const TaskRec rec = shfl_task_rec(mine, (k - k_begin) & 31);
            const int u = rec.tk.x;
            const int n = rec.tk.z - rec.tk.y;
            const int ctx_b = rec.ctx;
            for (int j = 0; j < n; ++j, ++vt) {
                const int eV = e_it + 2 * j + 1;
                const int kt = tile_of(u, rec.tk.y + j, ctx_b - rec.ql + rec.un.z);
                const int first_bad = ctx_b - kt * kPrefillTile;   // rows >= this are zeros
                wait(&kv_full[eV % E], (uint32_t)((eV / E) & 1));
                wait(&vh_empty[vt & 1], (uint32_t)((vt >> 1) & 1) ^ 1u);
                const uint8_t* src = smem + Cfg::kOffKV + (eV % E) * Cfg::kKVBytes;
                uint8_t* dst = smem + Cfg::kOffVh + (vt & 1) * Cfg::kVhBytes;
#pragma unroll 1
                for (int rr = 0; rr < kPrefillTile / 32; ++rr) {
                    const int r = rr * 32 + lane;
                    const bool ok = r < first_bad;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        // source chunks 4 half .. 4 half + 3 = head dims [64 half, +64)
                        uint4 w[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            w[c] = *reinterpret_cast<const uint4*>(src + swz128(r, 4 * half + c));
                        uint8_t* blk = dst + half * Cfg::kRegion;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint32_t x[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
                            uint32_t h[8];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                h[2 * q] = ok ? e4m3x2_to_f16x2((uint16_t)(x[q] & 0xffffu)) : 0u;
                                h[2 * q + 1] = ok ? e4m3x2_to_f16x2((uint16_t)(x[q] >> 16)) : 0u;
                            }
                            *reinterpret_cast<uint4*>(blk + swz128(r, 2 * c)) =
                                make_uint4(h[0], h[1], h[2], h[3]);
                            *reinterpret_cast<uint4*>(blk + swz128(r, 2 * c + 1)) =
                                make_uint4(h[4], h[5], h[6], h[7]);
                        }
                    }
                }
                __syncwarp();
                // the E4M3 entry is free (both of its releases), the f16 tile ready
                if (lane == 0) {
                    mbar_arrive(&kv_empty[eV % E]);
                    mbar_arrive(&kv_empty[eV % E]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&vh_full[vt & 1]);
            }
            e_it += 2 * n;
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------ MMA issuers
        // warp 1 issues every MMA of half 0, warp 2 those of half 1: each
        // issue blocks until the tensor pipe nearly drains it, so with one
        // issuer per half one warp does its waits while the other issues.
        // A token passed through two named barriers keeps the segments in
        // the order half 0, half 1, half 0, ...: without it both halves'
        // MMAs interleave on the pipe, finish together, and the two softmax
        // groups then run at the same time while the tensor pipe idles.
        // Both warps release each ring entry and the Q buffer (two commits
        // per barrier phase).
        constexpr uint32_t idesc_qk = FP8 ? idesc_e4m3_f32(128, 128, false, false)
                                          : idesc_bf16_f32(128, 128, false, false);
        // E4M3: PV is an f16 MMA over the converter's f16 V tile and an f16 P
        constexpr uint32_t idesc_pv = FP8 ? idesc_f16_f32(128, D, false, true)
                                          : idesc_bf16_f32(128, D, false, true);
        // Descriptor bases: the start-address field is the low bits of a
        // descriptor, so a byte offset within the buffer is added as offset >> 4.
        const uint64_t dQ = smem_desc_sw128(smem_u32(smem + Cfg::kOffQ), 16, 1024);
        // K (K-major) and V (MN-major) tiles: 8-row groups kGroupStride apart,
        // the second column block 1 KB after the first
        const uint64_t dK = smem_desc_sw128(smem_u32(smem + Cfg::kOffKV), 16, Cfg::kGroupStride);
        const uint64_t dV = smem_desc_sw128(smem_u32(smem + Cfg::kOffKV), 1024, Cfg::kGroupStride);
        const uint64_t dVh = smem_desc_sw128(smem_u32(smem + Cfg::kOffVh), Cfg::kRegion, 1024);
        int e_it = 0, task_it = 0, vt = 0;
        int p_cnt = 0, of_cnt = 0;   // phases of this warp's half
        TaskRec mine;

        auto issue_qk = [&](int h, int e) {   // S_h = Q_h K^T from ring entry e
            const uint64_t a0 = dQ + (uint64_t)((h * Cfg::kQTileBytes) >> 4);
            const uint64_t b0 = dK + (uint64_t)((e * Cfg::kKVBytes) >> 4);
            const uint32_t d = tmem + h * 256;
            // each instruction takes 32 bytes of every row's K dimension
#pragma unroll
            for (int kk = 0; kk < D * Cfg::kElem / 32; ++kk) {
                // column block kk / 4: kRegion further on in Q, 1 KB in K
                const uint64_t qoff = (uint64_t)((((kk >> 2) * Cfg::kRegion) + (kk & 3) * 32) >> 4);
                const uint64_t koff = (uint64_t)((((kk >> 2) * 1024) + (kk & 3) * 32) >> 4);
                if constexpr (FP8)
                    tc_mma_ss_f8(d, a0 + qoff, b0 + koff, idesc_qk, kk > 0 ? 1u : 0u);
                else
                    tc_mma_ss(d, a0 + qoff, b0 + koff, idesc_qk, kk > 0 ? 1u : 0u);
            }
            tc_commit(&s_full[h]);
        };
        auto issue_pv = [&](int h, int e, bool first) {   // O_h += P_h V from ring entry e
            // (E4M3: e is the f16 V buffer)
            const uint64_t b0 = FP8 ? dVh + (uint64_t)((e * Cfg::kVhBytes) >> 4)
                                    : dV + (uint64_t)((e * Cfg::kKVBytes) >> 4);
            const uint32_t d = tmem + h * 256 + 128, a = tmem + h * 256;
#pragma unroll
            // 16 keys per instruction: two 8-row groups of V (the f16 copy of an
            // E4M3 V tile is plain row-major: two 1 KB groups per column block)
            constexpr int kStep = FP8 ? 2 * 1024 : 2 * Cfg::kGroupStride;
            for (int kk = 0; kk < kPrefillTile / 16; ++kk)
                tc_mma_ts(d, a + kk * 8, b0 + (uint64_t)((kk * kStep) >> 4), idesc_pv,
                          (!first || kk > 0) ? 1u : 0u);
            tc_commit(&o_done[h]);
        };

        const int h = warp - 1;                // the half this warp issues for
        // segment token: half 1 waits for half 0's segment (barrier 2); half 0
        // waits for half 1's previous segment (barrier 3), except the first
        bool first_segment = true;
        auto token_wait = [&]() {
            if (h == 1)
                named_bar_sync(2, 64);
            else if (!first_segment)
                named_bar_sync(3, 64);
            first_segment = false;
        };
        auto token_pass = [&]() { named_bar_arrive(h == 0 ? 2 : 3, 64); };
        for (int k = k_begin; k < k_end; ++k, ++task_it) {
            if (((k - k_begin) & 31) == 0)
                mine = load_task_rec(tasks, units, P.ctx, P.ql, cu_q, k + lane, k_end);
            const TaskRec rec = shfl_task_rec(mine, (k - k_begin) & 31);
            const int u = rec.tk.x;
            const bool mine_half = h == 0 || G * rec.un.w > kPrefillHalfRows;
            const int n = rec.tk.z - rec.tk.y;
            const int ctx_b = rec.ctx;
            wait(q_full, (uint32_t)(task_it & 1));
            // prologue: QK of tile 0
            {
                const int eK = e_it;
                wait(&kv_full[eK % E], (uint32_t)((eK / E) & 1));
                token_wait();
                if (lane == 0) {
                    tc_fence_after();
                    if (mine_half) issue_qk(h, eK % E);
                    tc_commit(&kv_empty[eK % E]);
                    if (n == 1) tc_commit(q_empty);
                }
                __syncwarp();
                token_pass();
            }
            for (int j = 0; j < n; ++j, ++vt) {
                const int eV = e_it + 2 * j + 1, eKn = e_it + 2 * j + 2;
                if constexpr (FP8)
                    wait(&vh_full[vt & 1], (uint32_t)((vt >> 1) & 1));   // f16 V ready
                else
                    wait(&kv_full[eV % E], (uint32_t)((eV / E) & 1));
                if constexpr (!FP8) {
                    // zero V rows of keys past the context (P is 0 there, 0 * NaN is
                    // not): warp 1 writes, both MMA warps meet before their PV
                    const int kt = tile_of(u, rec.tk.y + j, ctx_b - rec.ql + rec.un.z);
                    const int first_bad = ctx_b - kt * kPrefillTile;
                    if (first_bad < kPrefillTile) {
                        if (h == 0) {
                            uint8_t* sVp = smem + Cfg::kOffKV + (eV % E) * Cfg::kKVBytes;
                            const int r0 = first_bad < 0 ? 0 : first_bad;
                            for (int idx = lane; idx < (kPrefillTile - r0) * Cfg::kHalves * 8;
                                 idx += 32) {
                                const int r = r0 + idx / (Cfg::kHalves * 8);
                                const int rem = idx % (Cfg::kHalves * 8);
                                *reinterpret_cast<uint4*>(sVp + (r >> 3) * Cfg::kGroupStride +
                                                          (rem >> 3) * 1024 +
                                                          swz128(r & 7, rem & 7)) =
                                    make_uint4(0u, 0u, 0u, 0u);
                            }
                            fence_proxy_async_smem();
                        }
                        named_bar_sync(1, 64);
                    }
                }
                if (j + 1 < n) wait(&kv_full[eKn % E], (uint32_t)((eKn / E) & 1));
                if (mine_half) {
                    wait(&p_full[h], (uint32_t)(p_cnt & 1));
                    ++p_cnt;
                    if (j == 0) {
                        wait(&o_free[h], (uint32_t)(of_cnt & 1) ^ 1u);
                        ++of_cnt;
                    }
                }
                token_wait();
                if (lane == 0) {
                    if (mine_half) {
                        tc_fence_after();
                        issue_pv(h, FP8 ? (vt & 1) : eV % E, j == 0);
                        if (j + 1 < n) issue_qk(h, eKn % E);
                    }
                    // (E4M3: the converter released the V entry; PV read the f16 copy)
                    tc_commit(FP8 ? &vh_empty[vt & 1] : &kv_empty[eV % E]);
                    if (j + 1 < n) tc_commit(&kv_empty[eKn % E]);
                    if (j + 1 == n - 1) tc_commit(q_empty);
                }
                __syncwarp();
                token_pass();
            }
            e_it += 2 * n;
        }
        // consume half 1's last token so every barrier arrival is matched
        if (h == 0 && !first_segment) named_bar_sync(3, 64);
        if (lane == 0) {
            tc_commit(mma_done);
            mbar_wait(mma_done, 0, lim);
        }
        __syncwarp();
      }
    } else {
        regs_inc<Cfg::kRegsSoftmax>();
        // --------------------------------------------------- softmax (2 halves)
        const int h = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int row = wq * 32 + lane;              // row inside the half = TMEM lane
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + h * 256, tO = tS + 128;
        const float scale_log2 = P.sm_scale * kLog2e;
        int s_cnt = 0, o_cnt = 0;
        TaskRec mine;
        for (int k = k_begin; k < k_end; ++k) {
            if (((k - k_begin) & 31) == 0)
                mine = load_task_rec(tasks, units, P.ctx, P.ql, cu_q, k + lane, k_end);
            const TaskRec rec = shfl_task_rec(mine, (k - k_begin) & 31);
            if (threadIdx.x == 128) trace_task_start(P.trace, P.trace_cap, k);   // half 0, row 0
            const int u = rec.tk.x, hk = rec.un.y, q0 = rec.un.z;
            const int R = G * rec.un.w;
            if (h == 1 && R <= kPrefillHalfRows) continue;   // half 1 idle for this unit
            const int r = h * kPrefillHalfRows + row;        // row inside the unit
            const bool row_ok = r < R;
            // the row's logit scale (E4M3: times its Q scale and the K scale)
            float sl2 = scale_log2;
            if constexpr (FP8) {
                const int64_t qi = P.q_scale_per_row
                                       ? (int64_t)(rec.cuq + q0 + r / G) * Hq + hk * G + r % G
                                       : 0;
                sl2 = scale_log2 * (row_ok ? __ldg(P.q_scale + qi) : 1.f) * __ldg(P.k_scale);
            }
            const int ctx_b = rec.ctx;
            const int p_row = ctx_b - rec.ql + q0 + r / G;   // last key this row sees
            const int key_last = p_row < ctx_b - 1 ? p_row : ctx_b - 1;
            // first key this row sees: p - window + 1 with a sliding window
            // ("HiLS-Attention", 二.1 local branch)
            const int key_first = WINDOW ? p_row - L.window + 1 : -(1 << 30);
            const int p0 = ctx_b - rec.ql + q0;
            const int n = rec.tk.z - rec.tk.y;
            // a warp whose 32 rows are all padding (units of a few rows: short
            // sequences of a masked batch, or the last q tile of a sequence)
            // keeps the barrier protocol but skips the math: MMA rows are
            // independent and padding rows are never written
            const bool warp_live = __any_sync(0xffffffffu, row_ok);
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                const int kt = tile_of(u, rec.tk.y + j, p0);
                wait(&s_full[h], (uint32_t)(s_cnt & 1));
                ++s_cnt;
                tc_fence_after();
                if (!warp_live) {
                    if (j > 0) ++o_cnt;   // PV of the previous tile: nothing to wait for
                    tc_fence_before();
                    mbar_arrive(&p_full[h]);
                    continue;
                }
                const int limc = row_ok ? key_last - kt * kPrefillTile : -1;   // valid: c <= limc
                const int lowc = key_first - kt * kPrefillTile;                // and c >= lowc
                // every key of the tile visible to every row of the warp: no mask
                // work in either pass (a warp-uniform test, once a tile)
                const bool tile_full = __all_sync(
                    0xffffffffu, limc >= kPrefillTile - 1 && (!WINDOW || lowc <= 0));
                // pass 1: row max of the raw scores (sm_scale >= 0 keeps the order),
                // 32 columns at a time; the two softmax warps on each SM
                // sub-partition hide each other's TMEM latency
                // (four scalar chains, no array: nothing of the loop in local memory)
                float mxa = -INFINITY, mxb = -INFINITY, mxc = -INFINITY, mxd = -INFINITY;
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {
                    float s[32];
                    tmem_ld32(tS + c4 * 32, s);
                    tmem_wait_ld();
                    reg_fence32(s);
                    if (!tile_full) {
                        const int lim = limc - c4 * 32, low = lowc - c4 * 32;
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (!(c <= lim && (!WINDOW || c >= low))) s[c] = -INFINITY;
                    }
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {   // three-input max: 2 scores a step
                        mxa = fmax3(mxa, s[c], s[c + 1]);
                        mxb = fmax3(mxb, s[c + 2], s[c + 3]);
                        mxc = fmax3(mxc, s[c + 4], s[c + 5]);
                        mxd = fmax3(mxd, s[c + 6], s[c + 7]);
                    }
                }
                const float mx = fmaxf(fmaxf(mxa, mxb), fmaxf(mxc, mxd)) * sl2;
                // lazy max: move m (and rescale O, l) only when it grows by > 2^8
                float alpha = 1.f;
                bool resc = false;
                if (mx > m + 8.f) {
                    if (m != -INFINITY) {
                        alpha = ex2(m - mx);
                        resc = true;
                    }
                    m = mx;
                }
                const float mu = m == -INFINITY ? 0.f : m;
                // pass 2: P = exp2(s * scale - m) in bf16, two exponentials per MUFU
                // operation (x <= 8 since m trails the row max by at most 8, and f16
                // holds such x to 2^-9 relative, below P's own bf16 rounding); keys
                // [32c, 32c+32) go to S columns [16c, 16c+16), which every later
                // chunk has already read
                float2 suma = make_float2(0.f, 0.f), sumb = make_float2(0.f, 0.f);
                const float2 sl2x2 = make_float2(sl2, sl2), nmu2 = make_float2(-mu, -mu);
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {
                    float s[32];
                    tmem_ld32(tS + c4 * 32, s);
                    tmem_wait_ld();
                    reg_fence32(s);
                    // keys outside [lowc, limc] (a diagonal, context-end or window
                    // tile) become -inf, whose exponential is 0: every chunk then
                    // takes the same path
                    if (!tile_full) {
                        const int lim = limc - c4 * 32, low = lowc - c4 * 32;
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (!(c <= lim && (!WINDOW || c >= low))) s[c] = -INFINITY;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        // packed f32x2: the scaled scores and the row sums
                        const float2 a = __ffma2_rn(make_float2(s[c], s[c + 1]), sl2x2, nmu2);
                        const uint32_t e2 = ex2_h2(a.x, a.y);
                        float2& acc = ((c >> 1) & 1) ? sumb : suma;
                        if constexpr (FP8) {
                            // f16 P as computed; the pair straight into the f32 sums
                            add_f16x2_to_f32(acc, e2);
                            pk[c >> 1] = e2;
                        } else {
                            const float2 pf =
                                __half22float2(*reinterpret_cast<const __half2*>(&e2));
                            acc = __fadd2_rn(acc, pf);
                            pk[c >> 1] = pack_bf16x2(pf.x, pf.y);
                        }
                    }
                    tmem_st16(tS + c4 * 16, pk);
                }
                // O is rescaled only after the previous tile's PV has written it;
                // without a rescale nothing here touches O (PV of this tile is
                // issued after the arrival below, behind the previous one)
                if (__any_sync(0xffffffffu, resc)) {
                    if (j > 0) wait(&o_done[h], (uint32_t)(o_cnt & 1));
                    tc_fence_after();
                    const float f = resc ? alpha : 1.f;
#pragma unroll 1
                    for (int c4 = 0; c4 < D / 32; ++c4) {
                        float o[32];
                        tmem_ld32(tO + c4 * 32, o);
                        tmem_wait_ld();
                        reg_fence32(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= f;
                        tmem_st32(tO + c4 * 32, o);
                    }
                }
                if (j > 0) ++o_cnt;   // that PV's phase, waited for or not
                l = l * alpha + ((suma.x + suma.y) + (sumb.x + sumb.y));
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&p_full[h]);
            }
            // ---- epilogue: O / l -> output row (or split partial), LSE
            if (n > 0) {
                wait(&o_done[h], (uint32_t)(o_cnt & 1));
                ++o_cnt;
            }
            tc_fence_after();
            float inv = l > 0.f ? 1.f / l : 0.f;
            if constexpr (FP8) inv *= __ldg(P.v_scale);   // one V scale for the cache
            const float lse_nat = l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
            const int token = rec.cuq + q0 + r / G, head = hk * G + r % G;
#pragma unroll 1
            for (int c4 = 0; c4 < (warp_live ? D / 32 : 0); ++c4) {
                float o[32];
                tmem_ld32(tO + c4 * 32, o);
                tmem_wait_ld();
                reg_fence32(o);
                // 32-byte stores where the buffer allows (the rows' scattered
                // stores are the epilogue's cost: half as many instructions)
                if (row_ok) {
                    if (rec.tk.w < 0) {
                        __nv_bfloat16* dst = P.out + ((int64_t)token * Hq + head) * D + c4 * 32;
                        if (P.store_v8 & 1) {
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                uint32_t w[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    w[e] = pack_bf16x2(o[16 * q + 2 * e] * inv, o[16 * q + 2 * e + 1] * inv);
                                st_global_v8(dst + 16 * q, w);
                            }
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                reinterpret_cast<uint4*>(dst)[q] = make_uint4(
                                    pack_bf16x2(o[8 * q] * inv, o[8 * q + 1] * inv),
                                    pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                                    pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                                    pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
                        }
                    } else {
                        float* dst = P.part_o + ((int64_t)rec.tk.w * L.rows_cap + r) * D + c4 * 32;
                        if (P.store_v8 & 2) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t w[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(o[8 * q + e] * inv);
                                st_global_v8(dst + 8 * q, w);
                            }
                        } else {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                reinterpret_cast<float4*>(dst)[q] =
                                    make_float4(o[4 * q] * inv, o[4 * q + 1] * inv,
                                                o[4 * q + 2] * inv, o[4 * q + 3] * inv);
                        }
                    }
                }
            }
            if (row_ok) {
                if (rec.tk.w < 0) {
                    if (P.lse != nullptr) P.lse[(int64_t)token * Hq + head] = lse_nat;
                } else {
                    P.part_lse[(int64_t)rec.tk.w * L.rows_cap + r] = lse_nat;
                }
            }
            tc_fence_before();
            mbar_arrive(&o_free[h]);
            if (threadIdx.x == 128) trace_task_end(P.trace, P.trace_cap, k);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // After an abort, wait (bounded) for every copy the producers armed before
    // the CTA exits.  Nothing arms a barrier after the abort, and each armed
    // phase is one warp's arrival with its copies' bytes, so waiting for the
    // last armed phase of every entry waits for every copy in flight.  The MMA
    // warps already waited for all their MMAs (the mma_done commit).
    if (*abort_flag && threadIdx.x == 0) {
        for (int e = 0; e < E; ++e)
            if (armed[e] >= 0) mbar_wait(&kv_full[e], (uint32_t)(armed[e] & 1), kDrainLimitNs);
        if (armed[E] >= 0) mbar_wait(q_full, (uint32_t)(armed[E] & 1), kDrainLimitNs);
    }
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
}

int prefill_smem_bytes(int D, bool fp8) {
    if (fp8) return D == 128 ? PrefillCfg<128, true>::kSmemBytes : -1;
    if (D == 128) return PrefillCfg<128>::kSmemBytes;
    if (D == 64) return PrefillCfg<64>::kSmemBytes;
    return -1;
}

int prefill_threads() { return 384; }

const void* prefill_kernel_ptr(int D, bool fp8) {
    if (fp8) return D == 128 ? (const void*)prefill_kernel<128, false, true> : nullptr;
    if (D == 128) return (const void*)prefill_kernel<128, false, false>;
    if (D == 64) return (const void*)prefill_kernel<64, false, false>;
    return nullptr;
}

namespace {
template <int D, bool WINDOW, bool FP8>
cudaError_t launch_prefill_variant(const PrefillParams& P, const CUtensorMap& tq,
                                   const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                                   cudaStream_t stream) {
    using Cfg = PrefillCfg<D, FP8>;
    const void* kern = (const void*)prefill_kernel<D, WINDOW, FP8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_dependent(prefill_kernel<D, WINDOW, FP8>, dim3(grid), dim3(Cfg::kThreads),
                            Cfg::kSmemBytes, stream, P, tq, tk, tv);
}
}  // namespace

cudaError_t launch_prefill_from_api(const pa_problem& p, const WsLayout& L, const void* q,
                                    const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const int32_t* block_table,
                                    const int32_t* ctx, const int32_t* ql, const float* qs,
                                    const float* ks, const float* vs, void* ws, void* partial,
                                    void* out, float* lse, cudaStream_t stream) {
    (void)q;
    PrefillParams P;
    P.L = L;
    P.block_table = block_table;
    P.ctx = ctx;
    P.ql = ql;
    P.ws = ws;
    P.part_o = reinterpret_cast<float*>(partial);
    P.part_lse = P.part_o + L.partial_slots * L.rows_cap * L.D;
    P.out = reinterpret_cast<__nv_bfloat16*>(out);
    P.lse = lse;
    P.page_size = p.page_size;
    P.num_pages = p.num_pages;
    P.max_pages_per_seq = p.max_pages_per_seq;
    P.rows_per_box = p.page_size < 64 ? p.page_size : 64;
    P.boxes_per_tile = kPrefillTile / P.rows_per_box;
    P.kv_chunk_mul = p.layout == PA_NHD ? 2 : 0;
    P.kv_page_mul = p.layout == PA_NHD ? 1 : p.num_kv_heads;
    P.kv_head_add = p.layout == PA_NHD ? 0 : 1;
    // a row's 32-element chunk starts 64 (bf16) or 128 (fp32) bytes apart
    // from the buffer's start, so 32-byte stores need only a 32-byte base
    P.store_v8 = ((reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0) |
                 ((reinterpret_cast<uintptr_t>(partial) & 31u) == 0 ? 2 : 0);
    P.q_scale = qs;
    P.k_scale = ks;
    P.v_scale = vs;
    P.q_scale_per_row = p.q_scale_mode == PA_SCALE_PER_ROW ? 1 : 0;
    P.sm_scale = p.sm_scale;
    take_test_hook(&P.test_skip_it, &P.wait_limit_ns);
    take_task_trace(&P.trace, &P.trace_cap);
    const bool win = p.window > 0;
    const bool fp8 = p.q_dtype == PA_FP8_E4M3;
    cudaError_t e = cudaErrorInvalidValue;
    if (fp8 && p.head_dim == 128)
        e = win ? launch_prefill_variant<128, true, true>(P, tq, tk, tv, L.N, stream)
                : launch_prefill_variant<128, false, true>(P, tq, tk, tv, L.N, stream);
    else if (!fp8 && p.head_dim == 128)
        e = win ? launch_prefill_variant<128, true, false>(P, tq, tk, tv, L.N, stream)
                : launch_prefill_variant<128, false, false>(P, tq, tk, tv, L.N, stream);
    else if (!fp8 && p.head_dim == 64)
        e = win ? launch_prefill_variant<64, true, false>(P, tq, tk, tv, L.N, stream)
                : launch_prefill_variant<64, false, false>(P, tq, tk, tv, L.N, stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pa
