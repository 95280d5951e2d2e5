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
    int32_t kv_one_box;       // 1: one 5-D TMA box fills both column blocks of a tile
    int32_t test_skip_it;     // test hook: CTA 0 leaves this KV tile's stage unfilled (-1 none)
    float sm_scale;
    uint64_t wait_limit_ns;
};

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
// kOffQ.  `wait` is the kernel's bounded mbarrier wait (it turns into a no-op
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
    const int4* tasks = ws_ptr<int4>(P.ws, L.off_tasks);
    const int4* units = ws_ptr<int4>(P.ws, L.off_units);
    const int32_t* cu_q = ws_ptr<int32_t>(P.ws, L.off_cu_q);
    if (lane == 0) {
        prefetch_tmap(tmq);
        prefetch_tmap(tmk);
        prefetch_tmap(tmv);
    }
    const int ps = P.page_size, rpb = P.rows_per_box, nbox = P.boxes_per_tile;
    const uint32_t box_bytes = (uint32_t)rpb * 128u * Cfg::kHalves;
    const uint32_t q_bytes = (uint32_t)Cfg::kQHalves * G * P.q_box_tokens * 128u;
    int it = 0, task_it = 0;
    TaskRec mine;
    for (int k = k_begin; k < k_end; ++k, ++task_it) {
        if (((k - k_begin) & 31) == 0)
            mine = load_task_rec(tasks, units, P.ctx, P.ql, cu_q, k + lane, k_end);
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
        for (int t = tk.y; t < tk.z; ++t, ++it) {
            if (Cfg::kProducerWarps > 1 && it % Cfg::kProducerWarps != pw) continue;
            const int s = it % Cfg::kStages;
            wait(&empty[s], (uint32_t)((it / Cfg::kStages) & 1) ^ 1u);
            const int kt = t + first;
            int pg[4];
            float ksc[4], vsc[4];
            uint32_t bytes = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                pg[j] = -1;
                ksc[j] = vsc[j] = 0.f;
                if (j >= nbox) continue;
                const int tok0 = kt * kDecodeTile + j * rpb;
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
                    ksc[j] = __shfl_sync(0xffffffffu, win_ks, lp - win_lo);
                    vsc[j] = __shfl_sync(0xffffffffu, win_vs, lp - win_lo);
                }
                if (page < 0 || page >= P.num_pages) {
                    if (lane == 0) set_device_error(err_hdr, PA_DEV_BAD_PAGE);
                    page = -1;
                }
                pg[j] = page;
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
                    for (int j = 0; j < 4; ++j) {
                        scales[(s * 2 + 0) * 4 + j] = pg[j] >= 0 ? ksc[j] : 0.f;
                        scales[(s * 2 + 1) * 4 + j] = pg[j] >= 0 ? vsc[j] : 0.f;
                    }
                }
                armed[s] = it / Cfg::kStages;
                mbar_arrive_expect_tx(&full[s], bytes);
            }
            __syncwarp();
            // one box per lane: a tensor copy holds its issuing thread for
            // hundreds of cycles, the SM takes a new one every ~90
            if (go) {
                if (Cfg::kHalves == 2 && P.kv_one_box) {
                    // pages of >= 64 tokens: one box = both column blocks (lane 0 K, lane 1 V)
                    const int slot0 = (kt * kDecodeTile) % ps;
                    if (lane < 2 && pg[0] >= 0)
                        tma_load_5d(lane ? stV : stK, lane ? tmv : tmk, &full[s], 0, slot0, 0, hk,
                                    pg[0]);
                } else if (lane < 8 * Cfg::kHalves) {
                    // lane = (kv, page j, column block h)
                    const int kv = lane / (4 * Cfg::kHalves);
                    const int j = (lane / Cfg::kHalves) % 4, h = lane % Cfg::kHalves;
                    int page = -1;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        if (jj == j) page = pg[jj];
                    if (page >= 0) {
                        const int slot0 = (kt * kDecodeTile + j * rpb) % ps;
                        tma_load_4d((kv ? stV : stK) + h * Cfg::kHalfBytes + j * rpb * 128,
                                    kv ? tmv : tmk, &full[s], h * (128 / Cfg::kElem), slot0, hk,
                                    page);
                    }
                }
            }
            __syncwarp();
        }
    }
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
