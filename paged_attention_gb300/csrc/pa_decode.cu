// pa_decode.cu -- persistent split-K decode compute (memory-bound path).
//
// "基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 (Split-K Compute:
// persistent CTAs follow the task map, compute QK, softmax and PV per KV
// chunk and emit a local output and its LSE), 三.1 (small-M geometry: all
// G*q_len query rows of one KV head share each K/V tile, so the tile is read
// once for the whole GQA group and every MTP token), 三.2 (paged K/V reached
// through one 4-D tile descriptor whose strides absorb NHD vs HND), 二.2
// (producer warp resolves page ids ahead of the buffer wait, K/V land in a
// multi-stage shared-memory ring guarded by full/empty barriers).
//
// GB300 design.  One CTA per SM (persistent grid = Assign's CTA count):
//   warp 0            TMA producer.  Per task it loads the unit's Q rows
//                     (G heads x q_len tokens) into one of two Q slots; per
//                     64-token KV tile it reads the page ids (32 at a time,
//                     one coalesced warp load) and issues one TMA box per
//                     page and 128-byte column block of K and of V into a
//                     multi-stage ring (128-byte swizzle).
//   warps 1..         consumers, NG groups x RT row tiles x 4 token slices.
//                     Group g takes the CTA's tiles with index % NG == g, so
//                     NG tiles are in flight at once.  Warp (g, rt, ts) owns
//                     rows [16rt, 16rt+16) of the unit and tokens
//                     [16ts, 16ts+16) of its tiles; S = Q K^T and O += P V run
//                     on mma.sync (bf16 in, fp32 accumulate, P stays in
//                     registers), with a lazily moved running max (O is
//                     rescaled only when the max grows by more than 2^8).  At
//                     the end of a task the NG x 4 slices of each row tile
//                     merge their (m, l, O) through shared memory.
// The work is HBM-bound (<= 48 flop per KV byte even at 64 rows of FP8), so
// mma.sync is far from its limit; what matters is enough K/V bytes in flight
// per SM (the ring) and enough independent warps to hide the MMA / shuffle
// latency chains (the groups).
// FP8 (E4M3) K/V: each consumer converts its share of the tile to bf16 in a
// double-buffered per-slice buffer (exact), k_scale folds into the softmax
// scale, v_scale into P.
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
    float sm_scale;
    uint64_t wait_limit_ns;
};

template <int D, int RT, bool FP8, int NG, int STAGES>
struct DecodeCfg {
    static constexpr int kGroupWarps = 4 * RT;
    static constexpr int kConsumerWarps = kGroupWarps * NG;
    static constexpr int kWarps = 1 + kConsumerWarps;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int kElem = FP8 ? 1 : 2;
    static constexpr int kHalves = D * kElem / 128;          // 128-B column blocks of a K/V row
    static constexpr int kHalfBytes = kDecodeTile * 128;      // one column block of a tile
    static constexpr int kKBytes = kHalves * kHalfBytes;
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kQRows = 16 * RT;
    static constexpr int kQHalves = D / 64;                   // Q is bf16
    static constexpr int kQHalfBytes = kQRows * 128;
    static constexpr int kQSlotBytes = kQHalves * kQHalfBytes;
    static constexpr int kCvtHalves = D * 2 / 128;           // bf16 column blocks
    static constexpr int kCvtHalfBytes = 16 * 128;
    static constexpr int kCvtKBytes = kCvtHalves * kCvtHalfBytes;
    static constexpr int kCvtBuf = 2 * kCvtKBytes;           // K + V of one slice
    static constexpr int kCvtTotal = FP8 ? 4 * 2 * kCvtBuf : 0;
    static constexpr int kMergeFloats = 16 * D + 32;
    static constexpr int kMergeBytes = kConsumerWarps * kMergeFloats * 4;
    static constexpr int kScaleBytes = FP8 ? STAGES * 2 * 4 * 4 : 0;
    static constexpr int kOffQ = STAGES * kStageBytes;
    static constexpr int kOffCvt = kOffQ + 2 * kQSlotBytes;
    static constexpr int kOffMerge = kOffCvt + kCvtTotal;
    static constexpr int kOffScale = kOffMerge + kMergeBytes;
    static constexpr int kOffBar = (kOffScale + kScaleBytes + 15) / 16 * 16;
    static constexpr int kNumBars = 2 * STAGES + 4;
    static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(!FP8 || D == 128, "FP8 decode is built for head_dim 128");
    static_assert(!FP8 || NG == 1, "FP8 decode uses one tile group");
    static_assert(kQHalfBytes % 1024 == 0, "Q slot alignment");
    // Group g consumes the tiles with index % NG == g.  Every ring stage must
    // always be consumed by the same group: a group that reused a stage after
    // the other group could wait on a full barrier two phases ahead, where the
    // parity test cannot tell the phases apart.
    static_assert(STAGES % NG == 0, "stages must be a multiple of the tile groups");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int D, int RT, bool FP8, int NG, int STAGES>
__global__ void __launch_bounds__(32 * (1 + 4 * RT * NG), 1)
decode_kernel(const __grid_constant__ DecodeParams P, const __grid_constant__ CUtensorMap tmq,
              const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    using Cfg = DecodeCfg<D, RT, FP8, NG, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
    uint64_t* empty = full + STAGES;
    uint64_t* q_full = empty + STAGES;       // 2 slots
    uint64_t* q_empty = q_full + 2;          // 2 slots
    volatile int* abort_flag = reinterpret_cast<volatile int*>(q_empty + 2);
    float* scales = reinterpret_cast<float*>(smem + Cfg::kOffScale);   // [stage][k|v][box]
    const WsLayout& L = P.L;
    int32_t* header = ws_ptr<int32_t>(P.ws, L.off_header);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t lim = P.wait_limit_ns;

    if (header[H_CTAS] != (int)gridDim.x) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(header, PA_DEV_BAD_LENGTHS);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], Cfg::kGroupWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], Cfg::kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (*abort_flag) return;
        if (!mbar_wait(bar, parity, lim)) {
            *abort_flag = 1;
            set_device_error(header, PA_DEV_WAIT_TIMEOUT);
        }
    };

    const int32_t* cta_ptr = ws_ptr<int32_t>(P.ws, L.off_cta_ptr);
    const int4* tasks = ws_ptr<int4>(P.ws, L.off_tasks);
    const int4* units = ws_ptr<int4>(P.ws, L.off_units);
    const int32_t* cu_q = ws_ptr<int32_t>(P.ws, L.off_cu_q);
    const int k_begin = cta_ptr[blockIdx.x], k_end = cta_ptr[blockIdx.x + 1];
    const int G = L.G, Hq = L.Hq;

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tmap(&tmq);
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
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
            wait(&q_empty[qs], (uint32_t)((task_it >> 1) & 1) ^ 1u);
            if (lane == 0) {
                if (*abort_flag) {
                    mbar_arrive(&q_full[qs]);
                } else {
                    mbar_arrive_expect_tx(&q_full[qs], q_bytes);
                    uint8_t* qdst = smem + Cfg::kOffQ + qs * Cfg::kQSlotBytes;
#pragma unroll
                    for (int h = 0; h < Cfg::kQHalves; ++h)
                        tma_load_3d(qdst + h * Cfg::kQHalfBytes, &tmq, &q_full[qs], 64 * h, hk * G,
                                    rec.cuq + un.z);
                }
            }
            __syncwarp();
            int win_lo = -(1 << 30), win_val = -1;
            for (int t = tk.y; t < tk.z; ++t, ++it) {
                const int s = it % STAGES;
                wait(&empty[s], (uint32_t)((it / STAGES) & 1) ^ 1u);
                const int kt = t;
                int pg[4];
                uint32_t bytes = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    pg[j] = -1;
                    if (j >= nbox) continue;
                    const int tok0 = kt * kDecodeTile + j * rpb;
                    if (tok0 >= ctx_b) continue;
                    const int lp = tok0 / ps;
                    if (lp - win_lo < 0 || lp - win_lo >= 32) {
                        win_lo = lp;
                        win_val = (lp + lane < npg) ? __ldg(bt_row + lp + lane) : -1;
                    }
                    int page = __shfl_sync(0xffffffffu, win_val, lp - win_lo);
                    if (page < 0 || page >= P.num_pages) {
                        if (lane == 0) set_device_error(header, PA_DEV_BAD_PAGE);
                        page = -1;
                    }
                    pg[j] = page;
                    if (page >= 0) bytes += 2u * box_bytes;
                }
                if (lane == 0) {
                    uint8_t* stK = smem + s * Cfg::kStageBytes;
                    uint8_t* stV = stK + Cfg::kKBytes;
                    if (FP8) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int64_t si = (int64_t)(pg[j] < 0 ? 0 : pg[j]) * L.Hkv + hk;
                            scales[(s * 2 + 0) * 4 + j] = pg[j] >= 0 ? P.k_scale[si] : 0.f;
                            scales[(s * 2 + 1) * 4 + j] = pg[j] >= 0 ? P.v_scale[si] : 0.f;
                        }
                    }
                    if (*abort_flag) {
                        mbar_arrive(&full[s]);
                    } else {
                        mbar_arrive_expect_tx(&full[s], bytes);
                        if (Cfg::kHalves == 2 && P.kv_one_box) {
                            // pages of >= 64 tokens: one box = both column blocks
                            const int slot0 = (kt * kDecodeTile) % ps;
                            if (pg[0] >= 0) {
                                tma_load_5d(stK, &tmk, &full[s], 0, slot0, 0, hk, pg[0]);
                                tma_load_5d(stV, &tmv, &full[s], 0, slot0, 0, hk, pg[0]);
                            }
                        } else
#pragma unroll
                        for (int kv = 0; kv < 2; ++kv) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                if (pg[j] < 0) continue;
                                const int slot0 = (kt * kDecodeTile + j * rpb) % ps;
#pragma unroll
                                for (int h = 0; h < Cfg::kHalves; ++h)
                                    tma_load_4d((kv ? stV : stK) + h * Cfg::kHalfBytes + j * rpb * 128,
                                                kv ? &tmv : &tmk, &full[s], h * (128 / Cfg::kElem),
                                                slot0, hk, pg[j]);
                            }
                        }
                    }
                }
                __syncwarp();
            }
        }
    } else {
        // ------------------------------------------------------- consumers
        const int cw = warp - 1;
        const int grp = cw / Cfg::kGroupWarps;
        const int rt = (cw % Cfg::kGroupWarps) >> 2, ts = cw & 3;
        const int g = lane >> 2, q4 = lane & 3;
        const float scale_log2 = P.sm_scale * kLog2e;
        float* merge = reinterpret_cast<float*>(smem + Cfg::kOffMerge);
        int it = 0, task_it = 0;
        TaskRec mine;
        for (int k = k_begin; k < k_end; ++k, ++task_it) {
            if (((k - k_begin) & 31) == 0)
                mine = load_task_rec(tasks, units, P.ctx, P.ql, cu_q, k + lane, k_end);
            const TaskRec rec = shfl_task_rec(mine, (k - k_begin) & 31);
            const int4 tk = rec.tk;
            const int4 un = rec.un;
            const int hk = un.y, q0 = un.z, nq = un.w;
            const int R = G * nq;
            const int ctx_b = rec.ctx, ql_b = rec.ql;
            const int tok_base = rec.cuq + q0;
            const int pbase = ctx_b - ql_b + q0;
            const int r_lo = 16 * rt + g, r_hi = r_lo + 8;
            const bool v_lo = r_lo < R, v_hi = r_hi < R;
            const int p_lo = pbase + r_lo / G, p_hi = pbase + r_hi / G;

            // Q fragments (A operand, rows x D) from the TMA-filled slot
            uint32_t qf[D / 16][4];
            {
                const int qs = task_it & 1;
                wait(&q_full[qs], (uint32_t)((task_it >> 1) & 1));
                const uint32_t qbase = smem_u32(smem + Cfg::kOffQ + qs * Cfg::kQSlotBytes);
                const int mi = lane >> 3;
                const int row = 16 * rt + 8 * (mi & 1) + (lane & 7);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int ch = 2 * kk + (mi >> 1);
                    ldsm_x4(qbase + (ch >> 3) * Cfg::kQHalfBytes + swz(row, ch & 7), qf[kk][0],
                            qf[kk][1], qf[kk][2], qf[kk][3]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_empty[qs]);
            }
            float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
            float o[D / 8][4];
#pragma unroll
            for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

            for (int t = tk.y; t < tk.z; ++t, ++it) {
                if (NG > 1 && (it % NG) != grp) continue;
                const int s = it % STAGES;
                wait(&full[s], (uint32_t)((it / STAGES) & 1));
                const int kt = t;
                const int tok_s0 = kt * kDecodeTile + 16 * ts;
                uint8_t* stK = smem + s * Cfg::kStageBytes;
                uint8_t* stV = stK + Cfg::kKBytes;
                uint32_t kbase, vbase;
                int rowbase, halfstride;
                float kscale = 1.f, vscale = 1.f;
                if constexpr (FP8) {
                    const int box = (16 * ts) / P.rows_per_box;
                    kscale = scales[(s * 2 + 0) * 4 + box];
                    vscale = scales[(s * 2 + 1) * 4 + box];
                    uint8_t* buf = smem + Cfg::kOffCvt + (ts * 2 + (it & 1)) * Cfg::kCvtBuf;
                    uint8_t* Kc = buf;
                    uint8_t* Vc = buf + Cfg::kCvtKBytes;
                    constexpr int kRowsPer = 16 / RT;
                    const int r0 = rt * kRowsPer;
                    // E4M3 row = 128 bytes = 8 chunks of 16 values
                    for (int idx = lane; idx < kRowsPer * 8; idx += 32) {
                        const int tr = r0 + idx / 8, c = idx % 8;
                        const int srow = 16 * ts + tr;
                        const bool live = tok_s0 + tr < ctx_b;
                        const int cb = 2 * (c & 3), hb = c >> 2;
#pragma unroll
                        for (int kv = 0; kv < 2; ++kv) {
                            const uint8_t* src = (kv ? stV : stK) + swz(srow, c);
                            uint8_t* dst = (kv ? Vc : Kc) + hb * Cfg::kCvtHalfBytes;
                            uint4 raw = *reinterpret_cast<const uint4*>(src);
                            uint32_t w[8];
                            const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                w[2 * i] = live ? e4m3x2_to_bf16x2((uint16_t)(in[i] & 0xffffu)) : 0u;
                                w[2 * i + 1] = live ? e4m3x2_to_bf16x2((uint16_t)(in[i] >> 16)) : 0u;
                            }
                            *reinterpret_cast<uint4*>(dst + swz(tr, cb)) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                            *reinterpret_cast<uint4*>(dst + swz(tr, cb + 1)) =
                                make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                    named_bar_sync(1 + ts, 32 * RT);
                    kbase = smem_u32(Kc);
                    vbase = smem_u32(Vc);
                    rowbase = 0;
                    halfstride = Cfg::kCvtHalfBytes;
                } else {
                    if (tok_s0 + 15 >= ctx_b) {
                        // tokens past the context: zero their V rows (P is 0 there,
                        // but 0 * NaN would poison O)
                        for (int idx = lane; idx < 16 * Cfg::kHalves * 8; idx += 32) {
                            const int tr = idx / (Cfg::kHalves * 8);
                            const int rem = idx % (Cfg::kHalves * 8);
                            if (tok_s0 + tr >= ctx_b)
                                *reinterpret_cast<uint4*>(stV + (rem >> 3) * Cfg::kHalfBytes +
                                                          swz(16 * ts + tr, rem & 7)) =
                                    make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    kbase = smem_u32(stK);
                    vbase = smem_u32(stV);
                    rowbase = 16 * ts;
                    halfstride = Cfg::kHalfBytes;
                }

                // S = Q K^T : 16 rows x 16 tokens, even / odd k-steps in two chains
                float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                float sb[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                {
                    const int mi = lane >> 3;
                    const int trow = rowbase + 8 * (mi >> 1) + (lane & 7);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int dch = 2 * kk + (mi & 1);
                        const uint32_t addr = kbase + (dch >> 3) * halfstride + swz(trow, dch & 7);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(addr, b0, b1, b2, b3);
                        if (kk & 1) {
                            mma_bf16_16816(sb[0], qf[kk], b0, b1);
                            mma_bf16_16816(sb[1], qf[kk], b2, b3);
                        } else {
                            mma_bf16_16816(sa[0], qf[kk], b0, b1);
                            mma_bf16_16816(sa[1], qf[kk], b2, b3);
                        }
                    }
                }
                // mask + online softmax (log2 domain, lazily moved max)
                const float cs = scale_log2 * kscale;
                float sv[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = tok_s0 + 8 * j + 2 * q4 + e;
                        const bool okl = v_lo && tok < ctx_b && tok <= p_lo;
                        const bool okh = v_hi && tok < ctx_b && tok <= p_hi;
                        sv[j][e] = okl ? (sa[j][e] + sb[j][e]) * cs : -INFINITY;
                        sv[j][2 + e] = okh ? (sa[j][2 + e] + sb[j][2 + e]) * cs : -INFINITY;
                    }
                }
                float mx_lo = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
                float mx_hi = fmaxf(fmaxf(sv[0][2], sv[0][3]), fmaxf(sv[1][2], sv[1][3]));
                mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
                mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
                mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
                mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
                float al_lo = 1.f, al_hi = 1.f;
                bool resc = false;
                if (mx_lo > m_lo + 8.f) {
                    if (m_lo != -INFINITY) {
                        al_lo = ex2(m_lo - mx_lo);
                        resc = true;
                    }
                    m_lo = mx_lo;
                }
                if (mx_hi > m_hi + 8.f) {
                    if (m_hi != -INFINITY) {
                        al_hi = ex2(m_hi - mx_hi);
                        resc = true;
                    }
                    m_hi = mx_hi;
                }
                const float mu_lo = m_lo == -INFINITY ? 0.f : m_lo;
                const float mu_hi = m_hi == -INFINITY ? 0.f : m_hi;
                float p[2][4];
                float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    p[j][0] = ex2(sv[j][0] - mu_lo);
                    p[j][1] = ex2(sv[j][1] - mu_lo);
                    p[j][2] = ex2(sv[j][2] - mu_hi);
                    p[j][3] = ex2(sv[j][3] - mu_hi);
                    sum_lo += p[j][0] + p[j][1];
                    sum_hi += p[j][2] + p[j][3];
                }
                l_lo = l_lo * al_lo + sum_lo;
                l_hi = l_hi * al_hi + sum_hi;
                if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
                    for (int j = 0; j < D / 8; ++j) {
                        o[j][0] *= al_lo;
                        o[j][1] *= al_lo;
                        o[j][2] *= al_hi;
                        o[j][3] *= al_hi;
                    }
                }
                uint32_t pa[4];
                pa[0] = pack_bf16x2(p[0][0] * vscale, p[0][1] * vscale);
                pa[1] = pack_bf16x2(p[0][2] * vscale, p[0][3] * vscale);
                pa[2] = pack_bf16x2(p[1][0] * vscale, p[1][1] * vscale);
                pa[3] = pack_bf16x2(p[1][2] * vscale, p[1][3] * vscale);
                // O += P V : V^T fragments via ldmatrix.trans
                {
                    const int mi = lane >> 3;
                    const int trow = rowbase + 8 * (mi & 1) + (lane & 7);
#pragma unroll
                    for (int jd = 0; jd < D / 8; jd += 2) {
                        const int dch = jd + (mi >> 1);
                        const uint32_t addr = vbase + (dch >> 3) * halfstride + swz(trow, dch & 7);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(addr, b0, b1, b2, b3);
                        mma_bf16_16816(o[jd], pa, b0, b1);
                        mma_bf16_16816(o[jd + 1], pa, b2, b3);
                    }
                }
                if constexpr (!FP8) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                }
            }

            // ---- merge the NG x 4 slices of this row tile
            l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
            l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
            l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
            l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
            // slice index inside the row tile: (group, token slice)
            const int slice = grp * 4 + ts;
            float* mb = merge + (rt * NG * 4 + slice) * Cfg::kMergeFloats;
            if (q4 == 0) {
                mb[g] = m_lo;
                mb[g + 8] = m_hi;
                mb[16 + g] = l_lo;
                mb[16 + g + 8] = l_hi;
            }
#pragma unroll
            for (int j = 0; j < D / 8; ++j) {
                const int d = 8 * j + 2 * q4;
                *reinterpret_cast<float2*>(mb + 32 + g * D + d) = make_float2(o[j][0], o[j][1]);
                *reinterpret_cast<float2*>(mb + 32 + (g + 8) * D + d) =
                    make_float2(o[j][2], o[j][3]);
            }
            named_bar_sync(5 + rt, 128 * NG);
            {
                constexpr int DPL = D / 32;            // elements of D per lane
                constexpr int kSlices = 4 * NG;
                constexpr int kRowsPerWarp = 16 / kSlices;
                const float* m0 = merge + (rt * kSlices) * Cfg::kMergeFloats;
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i) {
                    const int rr = slice * kRowsPerWarp + i;
                    const int r = 16 * rt + rr;
                    float M = -INFINITY;
#pragma unroll
                    for (int kk = 0; kk < kSlices; ++kk) M = fmaxf(M, m0[kk * Cfg::kMergeFloats + rr]);
                    float Lsum = 0.f;
                    float acc[DPL];
#pragma unroll
                    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
#pragma unroll
                    for (int kk = 0; kk < kSlices; ++kk) {
                        const float* mk = m0 + kk * Cfg::kMergeFloats;
                        const float w = mk[rr] == -INFINITY ? 0.f : ex2(mk[rr] - M);
                        Lsum += w * mk[16 + rr];
#pragma unroll
                        for (int e = 0; e < DPL; ++e) acc[e] += w * mk[32 + rr * D + lane * DPL + e];
                    }
                    if (r < R) {
                        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
                        const float lse_nat = Lsum > 0.f ? (M + lg2(Lsum)) * kLn2 : -INFINITY;
                        const int token = tok_base + r / G, head = hk * G + r % G;
                        if (tk.w < 0) {
                            __nv_bfloat16* dst =
                                P.out + ((int64_t)token * Hq + head) * D + lane * DPL;
                            if constexpr (DPL == 4) {
                                uint2 v;
                                v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
                                v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
                                *reinterpret_cast<uint2*>(dst) = v;
                            } else {
                                *reinterpret_cast<uint32_t*>(dst) =
                                    pack_bf16x2(acc[0] * inv, acc[1] * inv);
                            }
                            if (P.lse != nullptr && lane == 0)
                                P.lse[(int64_t)token * Hq + head] = lse_nat;
                        } else {
                            const int64_t prow = (int64_t)tk.w * L.rows_cap + r;
                            float* dst = P.part_o + prow * D + lane * DPL;
#pragma unroll
                            for (int e = 0; e < DPL; ++e) dst[e] = acc[e] * inv;
                            if (lane == 0) P.part_lse[prow] = lse_nat;
                        }
                    }
                }
            }
            named_bar_sync(5 + rt, 128 * NG);
        }
    }
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // the consumers stopped waiting: give copies already issued time to land
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 200000ull) {
        }
    }
}

template <int D, int RT, bool FP8, int NG, int STAGES>
static cudaError_t launch_variant(const DecodeParams& P, const CUtensorMap& tq,
                                  const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t stream) {
    using Cfg = DecodeCfg<D, RT, FP8, NG, STAGES>;
    auto kern = decode_kernel<D, RT, FP8, NG, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<P.L.N, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(P, tq, tk, tv);
    return cudaGetLastError();
}

// (head_dim, row tiles, fp8, tile groups, stages) built
#ifndef PA_DECODE_NG_128_1
#define PA_DECODE_NG_128_1 2
#endif
#ifndef PA_DECODE_ST_128_1
#define PA_DECODE_ST_128_1 4
#endif
#define PA_DECODE_VARIANTS(X)                                             \
    X(128, 1, false, PA_DECODE_NG_128_1, PA_DECODE_ST_128_1)              \
    X(128, 2, false, 1, 4)    \
    X(64, 1, false, 2, 8)     \
    X(64, 2, false, 1, 8)     \
    X(64, 4, false, 1, 6)     \
    X(128, 1, true, 1, 6)     \
    X(128, 2, true, 1, 5)

int decode_smem_bytes(int D, int RT, bool fp8) {
#define X(d, rt, f8, ng, st) \
    if (D == d && RT == rt && fp8 == f8) return DecodeCfg<d, rt, f8, ng, st>::kSmemBytes;
    PA_DECODE_VARIANTS(X)
#undef X
    return -1;
}

int decode_threads(int D, int RT, bool fp8) {
#define X(d, rt, f8, ng, st) \
    if (D == d && RT == rt && fp8 == f8) return DecodeCfg<d, rt, f8, ng, st>::kThreads;
    PA_DECODE_VARIANTS(X)
#undef X
    return -1;
}

const void* decode_kernel_ptr(int D, int RT, bool fp8) {
#define X(d, rt, f8, ng, st) \
    if (D == d && RT == rt && fp8 == f8) return (const void*)decode_kernel<d, rt, f8, ng, st>;
    PA_DECODE_VARIANTS(X)
#undef X
    return nullptr;
}

static cudaError_t launch_decode(const DecodeParams& P, int D, int RT, bool fp8,
                                 const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, cudaStream_t stream) {
#define X(d, rt, f8, ng, st)             \
    if (D == d && RT == rt && fp8 == f8) \
        return launch_variant<d, rt, f8, ng, st>(P, tq, tk, tv, stream);
    PA_DECODE_VARIANTS(X)
#undef X
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_from_api(const pa_problem& p, const WsLayout& L, int RT,
                                   const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, bool kv_one_box,
                                   const int32_t* block_table,
                                   const int32_t* ctx, const int32_t* ql, const float* ks,
                                   const float* vs, void* ws, void* partial, void* out, float* lse,
                                   cudaStream_t stream) {
    DecodeParams P;
    P.L = L;
    P.block_table = block_table;
    P.ctx = ctx;
    P.ql = ql;
    P.k_scale = ks;
    P.v_scale = vs;
    P.ws = ws;
    P.part_o = reinterpret_cast<float*>(partial);
    P.part_lse = P.part_o + L.partial_slots * L.rows_cap * L.D;
    P.out = reinterpret_cast<__nv_bfloat16*>(out);
    P.lse = lse;
    P.page_size = p.page_size;
    P.num_pages = p.num_pages;
    P.max_pages_per_seq = p.max_pages_per_seq;
    P.rows_per_box = p.page_size < kDecodeTile ? p.page_size : kDecodeTile;
    P.boxes_per_tile = kDecodeTile / P.rows_per_box;
    P.q_box_tokens = p.max_q_len > 0 ? p.max_q_len : 1;
    P.kv_one_box = kv_one_box ? 1 : 0;
    P.sm_scale = p.sm_scale;
    P.wait_limit_ns = 1000000000ull;
    return launch_decode(P, p.head_dim, RT, p.kv_dtype == PA_FP8_E4M3, tq, tk, tv, stream);
}

}  // namespace pa
