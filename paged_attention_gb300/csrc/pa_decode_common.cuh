// pa_decode_common.cuh -- parameters and the TMA producer warp shared by the
// split-K decode kernels (bf16 K/V in pa_decode.cu, E4M3 K/V in
// pa_decode_fp8.cu).
//
// "基于Triton-TLE优化Tencent HPC-Ops Attention", 二.2 (the producer resolves
// page ids ahead of the buffer wait; K/V land in a multi-stage shared-memory
// ring guarded by full / empty barriers) and 三.2 (paged K/V through one tile
// descriptor whose strides absorb NHD vs HND).
#pragma once

#include "pa_internal.cuh"

namespace pa {

struct DecodeParams {
    WsLayout L;
    const int32_t* block_table;
    const int32_t* ctx;
    const int32_t* ql;
    const float* k_scale;
    const float* v_scale;
    void* ws;
    float* part_o;
    float* part_lse;
    __nv_bfloat16* out;
    float* lse;
    int32_t page_size;
    int32_t num_pages;
    int32_t max_pages_per_seq;
    int32_t rows_per_box;     // min(page_size, 64)
    int32_t boxes_per_tile;   // 64 / rows_per_box
    int32_t q_box_tokens;     // tokens per Q TMA box (max q_len)
    // bf16 K/V with head_dim 128 come in boxes of a page's rows by 8-token
    // group (see pa_api's grouped K/V map): chunk coordinate kv_chunk_mul *
    // head, last coordinate page * kv_page_mul + head * kv_head_add
    int32_t kv_chunk_mul;
    int32_t kv_page_mul;
    int32_t kv_head_add;
    int32_t test_skip_it;     // test hook: CTA 0 leaves this KV tile's stage unfilled (-1 none)
    int32_t static_splits;    // 0: tasks from the Assign map; S > 0: static split-K, S splits
    int32_t cluster_size;     // static split-K on clusters of S CTAs (DSM merge); else 1
    int64_t* trace;           // task trace (pa_set_task_trace), or nullptr
    int64_t trace_cap;
    float sm_scale;
    uint64_t wait_limit_ns;
};

// Static split-K ("基于Triton-TLE…", 一 Static Split-K: a fixed split count,
// the mapping resolved from the program id, no task map built or read).  Of
// the U * S static tasks (U = B * Hkv units), CTA c runs c, c + N, c + 2N, ...
// (N CTAs); task i is split s = i % S of unit u = i / S and covers the unit's
// KV tiles [s*n/S, (s+1)*n/S) (n tiles; fewer than S leaves empty splits).
template <bool kMayBeStatic>
__device__ __forceinline__ void cta_task_range(const DecodeParams& P, int& k_begin, int& k_end) {
    if (kMayBeStatic && P.static_splits > 0) {
        const int64_t T = (int64_t)P.L.B * P.L.Hkv * P.static_splits;
        const int64_t c = blockIdx.x, N = gridDim.x;
        k_begin = 0;
        k_end = c < T ? (int)((T - c + N - 1) / N) : 0;
    } else {
        const int32_t* cta_ptr = ws_ptr<int32_t>(P.ws, P.L.off_cta_ptr);
        k_begin = cta_ptr[blockIdx.x];
        k_end = cta_ptr[blockIdx.x + 1];
    }
}

// Record of static task k (k < k_end) of this CTA, for lane `lane`; all 32
// lanes call it together (the query offset cu_q of the task's sequence -- the
// sum of the q_lens before it -- is a warp-wide prefix over q_lens).  Lengths
// are checked as Assign checks them; a sequence that fails gets empty tasks
// and PA_DEV_BAD_LENGTHS.
__device__ __forceinline__ TaskRec static_task_rec(const DecodeParams& P, int k, int k_end,
                                                   int lane, int32_t* err_hdr) {
    const WsLayout& L = P.L;
    const int S = P.static_splits;
    const bool valid = k < k_end;
    const int64_t i = (int64_t)blockIdx.x + (int64_t)k * gridDim.x;
    const int u = valid ? (int)(i / S) : 0, s = valid ? (int)(i % S) : 0;
    const int b = u / L.Hkv, hk = u - b * L.Hkv;
    const int q = valid ? P.ql[b] : 0, c = valid ? P.ctx[b] : 0;
    int cuq = 0, run = 0;
    const int bmax = __reduce_max_sync(0xffffffffu, valid ? b : 0);
    for (int c0 = 0; c0 <= bmax; c0 += 32) {
        const int qq = c0 + lane < L.B ? P.ql[c0 + lane] : 0;
        const int v = max(0, min(qq, L.max_q_len));
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        const int ex = __shfl_sync(0xffffffffu, inc - v, (b - c0) & 31);
        if (b >= c0 && b < c0 + 32) cuq = run + ex;
        run += __shfl_sync(0xffffffffu, inc, 31);
    }
    TaskRec r;
    r.tk = make_int4(u, 0, 0, -1);
    r.un = make_int4(b, hk, 0, 0);
    r.ctx = c;
    r.ql = q;
    r.cuq = cuq;
    const bool bad = q < 0 || c < q || c > L.max_ctx || q > L.max_q_len || cuq + q > L.total_q;
    if (valid && bad) set_device_error(err_hdr, PA_DEV_BAD_LENGTHS);
    if (!valid || bad || q == 0) return r;
    const int n = (c + kDecodeTile - 1) / kDecodeTile - window_first_tile(L.window, c - q, kDecodeTile);
    r.tk = make_int4(u, (int)((int64_t)s * n / S), (int)((int64_t)(s + 1) * n / S),
                     S > 1 ? u * S + s : -1);
    r.un.w = q;
    return r;
}

// Record of task k of this CTA's list, for lane `lane` (all 32 lanes call it):
// from the Assign map, or the static split-K mapping.  Only the kernel
// instantiations built with kMayBeStatic carry the static-path code.
template <bool kMayBeStatic>
__device__ __forceinline__ TaskRec fetch_task_rec(const DecodeParams& P, int k, int k_end,
                                                  int lane, int32_t* err_hdr) {
    if (kMayBeStatic && P.static_splits > 0) return static_task_rec(P, k, k_end, lane, err_hdr);
    const WsLayout& L = P.L;
    return load_task_rec(ws_ptr<int4>(P.ws, L.off_tasks), ws_ptr<int4>(P.ws, L.off_units), P.ctx,
                         P.ql, ws_ptr<int32_t>(P.ws, L.off_cu_q), k, k_end);
}

// Split count and first partial slot of split unit u.
template <bool kMayBeStatic>
__device__ __forceinline__ int2 unit_splits(const DecodeParams& P, int u) {
    if (kMayBeStatic && P.static_splits > 0) return make_int2(P.static_splits, u * P.static_splits);
    return make_int2(ws_ptr<int32_t>(P.ws, P.L.off_nsplit)[u],
                     ws_ptr<int32_t>(P.ws, P.L.off_slot0)[u]);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile written by TMA
// with the 128-byte swizzle (128-byte rows, 1024-byte aligned tile).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// The producer warps of a decode kernel (kProducerWarps of them; this is
// warp `pw`).  Warp 0 loads, per task, the unit's Q rows (G heads x q_len
// tokens) into one of two Q slots.  KV tile it belongs to warp
// it % kProducerWarps, which takes the page ids (32 at a time, one coalesced
// warp load, the next 32 requested one window ahead), for E4M3 also the
// pages' K/V scales, and issues the TMA boxes of K and V into ring stage
// it % kStages.  One thread issuing every copy of a CTA is slow (each
// tensor copy holds its thread for hundreds of cycles), so the tiles are
// dealt out over several warps; kStages % kProducerWarps == 0 keeps every
// stage with one warp.
//
// Cfg supplies the shared-memory geometry: kStages, kProducerWarps, kFP8,
// kHalves (128-byte column blocks per K/V row), kHalfBytes, kKBytes (V follows
// K in a stage), kStageBytes, kElem, kQHalves, kQHalfBytes, kQSlotBytes,
// kOffQ, and kTilesPerStage: 1, or 2 for a stage that holds the task's KV
// tiles t and t+1 as one 128-row K block followed by one 128-row V block
// (tile t+1 is left unloaded past the task's end; the scales of a stage are
// then 8 per K/V, tile-major).  `wait` is the kernel's bounded mbarrier wait (it turns into a no-op
// once the CTA has aborted, so the loop structure is kept).  After an abort
// the producers arm no barrier and issue no copy; `armed` (shared, kStages + 2
// ints, -1 at start) records per ring stage and per Q slot the last phase
// armed with a copy, so that decode_drain can wait for every copy still in
// flight before the CTA exits.
template <class Cfg, class Wait>
__device__ __forceinline__ void decode_produce(const DecodeParams& P, const CUtensorMap* tmq,
                                               const CUtensorMap* tmk, const CUtensorMap* tmv,
                                               uint8_t* smem, uint64_t* full, uint64_t* empty,
                                               uint64_t* q_full, uint64_t* q_empty,
                                               float* scales, volatile int* abort_flag,
                                               int* armed, int32_t* err_hdr, int k_begin,
                                               int k_end, int pw, int lane, Wait& wait) {
    static_assert(Cfg::kStages % Cfg::kProducerWarps == 0,
                  "every ring stage must stay with one producer warp");
    const WsLayout& L = P.L;
    const int G = L.G;
    if (lane == 0) {
        prefetch_tmap(tmq);
        prefetch_tmap(tmk);
        prefetch_tmap(tmv);
    }
    constexpr int TPS = Cfg::kTilesPerStage;
    static_assert(TPS == 1 || (TPS == 2 && Cfg::kHalves == 1), "two tiles a stage: E4M3 only");
    constexpr int kSubBytes = kDecodeTile * 128;   // one tile's K (or V) in a two-tile stage
    const int ps = P.page_size, rpb = P.rows_per_box, nbox = P.boxes_per_tile;
    const uint32_t box_bytes = (uint32_t)rpb * 128u * Cfg::kHalves;
    const uint32_t q_bytes = (uint32_t)Cfg::kQHalves * G * P.q_box_tokens * 128u;
    int it = 0, task_it = 0;
    TaskRec mine;
    for (int k = k_begin; k < k_end; ++k, ++task_it) {
        if (((k - k_begin) & 31) == 0)
            mine = fetch_task_rec<Cfg::kStatic>(P, k + lane, k_end, lane, err_hdr);
        const TaskRec rec = shfl_task_rec(mine, (k - k_begin) & 31);
        const int4 tk = rec.tk;
        const int4 un = rec.un;
        const int b = un.x, hk = un.y;
        const int ctx_b = rec.ctx;
        const int npg = (ctx_b + ps - 1) / ps;
        const int32_t* bt_row = P.block_table + (int64_t)b * P.max_pages_per_seq;
        // Q rows of the unit into slot task_it & 1
        const int qs = task_it & 1;
        if (pw == 0) wait(&q_empty[qs], (uint32_t)((task_it >> 1) & 1) ^ 1u);
        if (pw == 0) {
            // lane 0 arms the slot, then lane h copies column block h (a tensor
            // copy holds its issuing thread for hundreds of cycles)
            const bool go = __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
            if (lane == 0 && go) {
                armed[Cfg::kStages + qs] = task_it >> 1;
                mbar_arrive_expect_tx(&q_full[qs], q_bytes);
            }
            __syncwarp();
            if (go && lane < Cfg::kQHalves)
                tma_load_3d(smem + Cfg::kOffQ + qs * Cfg::kQSlotBytes + lane * Cfg::kQHalfBytes,
                            tmq, &q_full[qs], 64 * lane, hk * G, rec.cuq + un.z);
        }
        __syncwarp();
        // block-table window: 32 page ids (and, for FP8, their K/V scales)
        // read lane-parallel; the ids of the next window are requested one
        // window ahead so that a refresh does not wait on a global load
        int win_lo = -(1 << 30), win_val = -1;
        int nxt_lo = -(1 << 30), nxt_val = -1;
        float win_ks = 0.f, win_vs = 0.f;
        // sliding window: task positions count from the unit's first visible tile
        const int first = window_first_tile(L.window, ctx_b - rec.ql + un.z, kDecodeTile);
        for (int t = tk.y; t < tk.z; t += TPS, ++it) {
            if (Cfg::kProducerWarps > 1 && it % Cfg::kProducerWarps != pw) continue;
            const int s = it % Cfg::kStages;
            wait(&empty[s], (uint32_t)((it / Cfg::kStages) & 1) ^ 1u);
            const int kt = t + first;
            if constexpr (TPS == 2) {
                // Two tiles a stage (E4M3, one 128-byte column block): every
                // step is lane-parallel -- lane = (kv, tile m, box j) finds its
                // own page, scale and bytes, so the warp spends a few dozen
                // instructions a stage however many boxes the pages need.
                const int kv = lane >> 3, m = (lane >> 2) & 1, j = lane & 3;
                const int tok0 = (kt + m) * kDecodeTile + j * rpb;
                const bool want = lane < 16 && j < nbox && t + m < tk.z && tok0 < ctx_b;
                const int lp = want ? tok0 / ps : 0;
                const int lp_lo = __reduce_min_sync(0xffffffffu, want ? lp : (1 << 30));
                const int lp_hi = __reduce_max_sync(0xffffffffu, want ? lp : -(1 << 30));
                if (lp_lo <= lp_hi && (lp_lo < win_lo || lp_hi - win_lo >= 32)) {
                    win_val = (lp_lo == nxt_lo) ? nxt_val
                                                : ((lp_lo + lane < npg) ? __ldg(bt_row + lp_lo + lane) : -1);
                    win_lo = lp_lo;
                    nxt_lo = lp_lo + 32;
                    nxt_val = (nxt_lo + lane < npg) ? __ldg(bt_row + nxt_lo + lane) : -1;
                    const bool okp = win_val >= 0 && win_val < P.num_pages;
                    const int64_t si = (int64_t)(okp ? win_val : 0) * L.Hkv + hk;
                    win_ks = okp ? __ldg(P.k_scale + si) : 0.f;
                    win_vs = okp ? __ldg(P.v_scale + si) : 0.f;
                }
                const int src = want ? lp - win_lo : 0;
                int page = __shfl_sync(0xffffffffu, win_val, src);
                const float ks = __shfl_sync(0xffffffffu, win_ks, src);
                const float vs = __shfl_sync(0xffffffffu, win_vs, src);
                if (want && (page < 0 || page >= P.num_pages)) {
                    set_device_error(err_hdr, PA_DEV_BAD_PAGE);
                    page = -1;
                }
                const bool load = want && page >= 0;
                const uint32_t bytes =
                    (uint32_t)__popc(__ballot_sync(0xffffffffu, load)) * box_bytes;
                uint8_t* dst = smem + s * Cfg::kStageBytes + kv * Cfg::kKBytes + m * kSubBytes +
                               j * rpb * 128;
                const bool skip = P.test_skip_it == it && blockIdx.x == 0;
                const bool go = __shfl_sync(0xffffffffu, *abort_flag, 0) == 0 && !skip;
                if (go && lane < 16)
                    scales[(s * 2 + kv) * 8 + m * 4 + j] = load ? (kv ? vs : ks) : 0.f;
                __syncwarp();
                if (lane == 0 && go) {
                    armed[s] = it / Cfg::kStages;
                    mbar_arrive_expect_tx(&full[s], bytes);
                }
                __syncwarp();
                if (go && load)
                    tma_load_4d(dst, kv ? tmv : tmk, &full[s], 0,
                                ((kt + m) * kDecodeTile + j * rpb) % ps, hk, page);
                __syncwarp();
                continue;
            }
            int pg[4 * TPS];
            float ksc[4 * TPS], vsc[4 * TPS];
            uint32_t bytes = 0;
#pragma unroll
            for (int jm = 0; jm < 4 * TPS; ++jm) {
                // box j of the stage's tile m
                const int m = jm / 4, j = jm % 4;
                pg[jm] = -1;
                ksc[jm] = vsc[jm] = 0.f;
                if (j >= nbox || t + m >= tk.z) continue;
                const int tok0 = (kt + m) * kDecodeTile + j * rpb;
                if (tok0 >= ctx_b) continue;
                const int lp = tok0 / ps;
                if (lp - win_lo < 0 || lp - win_lo >= 32) {
                    win_val = (lp == nxt_lo) ? nxt_val
                                             : ((lp + lane < npg) ? __ldg(bt_row + lp + lane) : -1);
                    win_lo = lp;
                    nxt_lo = lp + 32;
                    nxt_val = (nxt_lo + lane < npg) ? __ldg(bt_row + nxt_lo + lane) : -1;
                    if (Cfg::kFP8) {
                        const bool okp = win_val >= 0 && win_val < P.num_pages;
                        const int64_t si = (int64_t)(okp ? win_val : 0) * L.Hkv + hk;
                        win_ks = okp ? __ldg(P.k_scale + si) : 0.f;
                        win_vs = okp ? __ldg(P.v_scale + si) : 0.f;
                    }
                }
                int page = __shfl_sync(0xffffffffu, win_val, lp - win_lo);
                if (Cfg::kFP8) {
                    ksc[jm] = __shfl_sync(0xffffffffu, win_ks, lp - win_lo);
                    vsc[jm] = __shfl_sync(0xffffffffu, win_vs, lp - win_lo);
                }
                if (page < 0 || page >= P.num_pages) {
                    if (lane == 0) set_device_error(err_hdr, PA_DEV_BAD_PAGE);
                    page = -1;
                }
                pg[jm] = page;
                if (page >= 0) bytes += 2u * box_bytes;
            }
            uint8_t* stK = smem + s * Cfg::kStageBytes;
            uint8_t* stV = stK + Cfg::kKBytes;
            // test hook: CTA 0 leaves one stage unfilled, so that its consumers'
            // bounded wait runs out (the abort path, exercised without a fault)
            const bool skip = P.test_skip_it == it && blockIdx.x == 0;
            const bool go = __shfl_sync(0xffffffffu, *abort_flag, 0) == 0 && !skip;
            if (lane == 0 && go) {
                if (Cfg::kFP8) {
#pragma unroll
                    for (int jm = 0; jm < 4 * TPS; ++jm) {
                        scales[(s * 2 + 0) * 4 * TPS + jm] = pg[jm] >= 0 ? ksc[jm] : 0.f;
                        scales[(s * 2 + 1) * 4 * TPS + jm] = pg[jm] >= 0 ? vsc[jm] : 0.f;
                    }
                }
                armed[s] = it / Cfg::kStages;
                mbar_arrive_expect_tx(&full[s], bytes);
            }
            __syncwarp();
            // one box per lane: a tensor copy holds its issuing thread for
            // hundreds of cycles, the SM takes a new one every ~90
            if (go) {
                if constexpr (Cfg::kHalves == 2) {
                    // two column blocks: lane = (kv, box j), one copy per page
                    // (or per 64 tokens of a larger page) holding both blocks,
                    // laid out by 8-token group
                    if (lane < 2 * nbox) {
                        const int kv = lane / nbox, j = lane - kv * nbox;
                        int page = -1;
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            if (jj == j) page = pg[jj];
                        if (page >= 0) {
                            const int slot0 = (kt * kDecodeTile + j * rpb) % ps;
                            tma_load_5d((kv ? stV : stK) + (j * rpb / 8) * Cfg::kGroupStride,
                                        kv ? tmv : tmk, &full[s], 0, 0, hk * P.kv_chunk_mul,
                                        slot0 / 8, page * P.kv_page_mul + hk * P.kv_head_add);
                        }
                    }
                } else if (lane < 8 * TPS * Cfg::kHalves) {
                    // one column block: lane = (kv, tile m, box j)
                    const int kv = lane / (4 * TPS * Cfg::kHalves);
                    const int jm = (lane / Cfg::kHalves) % (4 * TPS), h = lane % Cfg::kHalves;
                    const int m = jm / 4, j = jm % 4;
                    int page = -1;
#pragma unroll
                    for (int jj = 0; jj < 4 * TPS; ++jj)
                        if (jj == jm) page = pg[jj];
                    if (page >= 0) {
                        const int slot0 = ((kt + m) * kDecodeTile + j * rpb) % ps;
                        tma_load_4d((kv ? stV : stK) + m * kSubBytes + h * Cfg::kHalfBytes +
                                        j * rpb * 128,
                                    kv ? tmv : tmk, &full[s], h * (128 / Cfg::kElem), slot0, hk,
                                    page);
                    }
                }
            }
            __syncwarp();
        }
    }
}

// In-kernel finalizer of split units ("基于Triton-TLE…", 三.3: the partial
// states of one output are merged by whoever completes it, in place of a
// separate Combine pass).  Called by every thread of a named-barrier group
// (bar_id, nthreads) right after the group wrote its rows of a split task's
// normalised partial: each writer fences, one leader thread counts the task
// done on done_word, and the group learns (through *flag, shared) whether it
// was the unit's last task to finish -- S tasks in all -- and so must merge.
// Nobody waits for another CTA.
__device__ __forceinline__ bool split_task_done(int32_t* done_word, int S, int bar_id,
                                                int nthreads, bool leader, volatile int* flag) {
    __threadfence();
    named_bar_sync(bar_id, nthreads);
    if (leader) *flag = atomicAdd(done_word, 1) == S - 1 ? 1 : 0;
    named_bar_sync(bar_id, nthreads);
    const bool last = *flag != 0;
    if (last) __threadfence();
    return last;
}

// Writes one output row from the merged sums of its parts: out = acc / den,
// lse = M + ln den (den = 0: no visible key, out = 0 and lse = -inf).
template <int DPL>
__device__ __forceinline__ void write_merged_row(const DecodeParams& P, int64_t out_row,
                                                 const float (&acc)[DPL], float den, float M,
                                                 int lane) {
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat16* dst = P.out + out_row * P.L.D + lane * DPL;
    if constexpr (DPL == 4) {
        uint2 v;
        v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(dst) = v;
    } else {
#pragma unroll
        for (int e = 0; e < DPL; e += 2)
            *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
    }
    if (P.lse != nullptr && lane == 0)
        P.lse[out_row] = den > 0.f ? M + lg2(den) * kLn2 : -INFINITY;
}

// Cluster-DSM merge of static split-K ("基于Triton-TLE…", 三.3: the CTAs of a
// hardware cluster publish their partial softmax states into distributed
// shared memory, merge them on chip, and shard the merge by head).  With
// static split-K on clusters of C = S CTAs, the C CTAs of a cluster run the
// C splits of one unit in the same round: task i = c + j*N is split i % S of
// unit i / S, and for c = kS .. kS+S-1 the unit is the same (N % S == 0) and
// the split is the CTA's rank.  Each CTA writes its split's normalised rows
// O_r and lse_r into its own mailbox (rows of D + kMailPad floats, lse at D).
// Per round:
//   - every consumer thread fences at cluster scope; after the group barrier
//     one leader arrives on mail_full of every CTA of the cluster (release);
//   - all wait for their own mail_full (acquire): C arrivals = every mailbox
//     of the cluster written;
//   - the CTA of rank q merges the rows r = q (mod C) from all C mailboxes
//     through DSM and writes out / lse (no global partial, no Combine);
//   - after the group barrier the leader arrives on every CTA's mail_empty;
//     a CTA waits for its own mail_empty (all peers read its mailbox) before
//     it writes its mailbox again in the next round.
// All CTAs of a cluster run the same number of rounds (the unit of a round
// is common to the cluster), and a cluster-wide barrier at the kernel's end
// keeps every mailbox alive until its readers are done.
constexpr int kMailPad = 4;   // 16-byte aligned rows

template <int D>
__device__ __forceinline__ void cluster_merge_rows(const DecodeParams& P, const float* box, int R,
                                                   int rank, int C, int w, int nw,
                                                   int64_t row0_out, int G, int Hq, int hk,
                                                   int lane) {
    constexpr int DPL = D / 32;
    constexpr int kStride = D + kMailPad;
    const uint32_t base = smem_u32(box);
    for (int r = rank + C * w; r < R; r += C * nw) {
        const uint32_t row = base + (uint32_t)(r * kStride) * 4u;
        float M = -INFINITY;
        for (int q = 0; q < C; ++q) M = fmaxf(M, ld_dsm_f32(mapa_shared(row + D * 4, q)));
        float den = 0.f;
        float acc[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
        if (M != -INFINITY) {
            for (int q = 0; q < C; ++q) {
                const float lq = ld_dsm_f32(mapa_shared(row + D * 4, q));
                if (lq == -INFINITY) continue;
                const float wq = ex2((lq - M) * kLog2e);
                den += wq;
                const uint32_t src = mapa_shared(row + (uint32_t)(lane * DPL) * 4u, q);
                if constexpr (DPL == 4) {
                    const float4 v = ld_dsm_f32x4(src);
                    acc[0] += wq * v.x;
                    acc[1] += wq * v.y;
                    acc[2] += wq * v.z;
                    acc[3] += wq * v.w;
                } else {
                    const float2 v = ld_dsm_f32x2(src);
                    acc[0] += wq * v.x;
                    acc[1] += wq * v.y;
                }
            }
        }
        write_merged_row<DPL>(P, (row0_out + r / G) * Hq + hk * G + r % G, acc, den, M, lane);
    }
}

// Row r of a split unit, finalized: m = max_k lse_k, w_k = e^(lse_k - m),
// out = sum_k w_k O_k / sum_k w_k, lse = m + ln sum_k w_k over its S partials
// (slots s0 .. s0+S-1).  One warp per row, DPL head_dim elements per lane.
// The partials were written by other CTAs: read through L2 (ld.cg).
template <int DPL>
__device__ __forceinline__ void finalize_split_row(const DecodeParams& P, int s0, int S, int r,
                                                int64_t out_row, int lane) {
    const WsLayout& L = P.L;
    float M = -INFINITY;
    for (int k = 0; k < S; ++k)
        M = fmaxf(M, __ldcg(P.part_lse + (int64_t)(s0 + k) * L.rows_cap + r));
    float den = 0.f;
    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
    if (M != -INFINITY) {
        for (int k = 0; k < S; ++k) {
            const int64_t prow = (int64_t)(s0 + k) * L.rows_cap + r;
            const float lk = __ldcg(P.part_lse + prow);
            if (lk == -INFINITY) continue;
            const float w = ex2((lk - M) * kLog2e);
            den += w;
            const float* src = P.part_o + prow * L.D + lane * DPL;
            if constexpr (DPL == 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
                acc[0] += w * v.x;
                acc[1] += w * v.y;
                acc[2] += w * v.z;
                acc[3] += w * v.w;
            } else {
#pragma unroll
                for (int e = 0; e < DPL; ++e) acc[e] += w * __ldcg(src + e);
            }
        }
    }
    write_merged_row<DPL>(P, out_row, acc, den, M, lane);
}

// After an abort: wait (bounded) until every copy this producer warp armed
// has landed -- for each of its ring stages (and, warp 0, the Q slots) the
// phase last armed with a copy -- so that no tensor copy is still writing
// shared memory when the CTA exits.  Nothing arms a barrier after the abort,
// so each such phase completes exactly when its bytes arrive.
template <class Cfg>
__device__ __forceinline__ void decode_drain(uint64_t* full, uint64_t* q_full, const int* armed,
                                             const volatile int* abort_flag, int pw, int lane) {
    if (!*abort_flag || lane != 0) return;
    for (int s = pw; s < Cfg::kStages; s += Cfg::kProducerWarps)
        if (armed[s] >= 0) mbar_wait(&full[s], (uint32_t)(armed[s] & 1), kDrainLimitNs);
    if (pw == 0)
        for (int qs = 0; qs < 2; ++qs)
            if (armed[Cfg::kStages + qs] >= 0)
                mbar_wait(&q_full[qs], (uint32_t)(armed[Cfg::kStages + qs] & 1), kDrainLimitNs);
}

}  // namespace pa
