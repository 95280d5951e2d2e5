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
//   warps 0..P-1      TMA producers (pa_decode_common.cuh), tile it on warp
//                     it % P: per task the unit's Q rows (G heads x q_len
//                     tokens) into one of two Q slots; per 64-token KV tile
//                     the page ids (32 at a time, one coalesced warp load) and
//                     one TMA box per page of K and of V (a 64-token tile of a
//                     larger page is one box) into a multi-stage ring
//                     (128-byte swizzle); with two column blocks (bf16,
//                     D = 128) a box carries both, stored by 8-token group.
//   warps P..         consumers, NG groups x RT row tiles x 4 token slices.
//                     Group g takes the CTA's tiles with index % NG == g, so
//                     NG tiles are in flight at once.  Warp (g, rt, ts) owns
//                     rows [16rt, 16rt+16) of the unit and tokens
//                     [16ts, 16ts+16) of its tiles; S = Q K^T and O += P V run
//                     on mma.sync (bf16 in, fp32 accumulate, P stays in
//                     registers), with a lazily moved running max (O is
//                     rescaled only when the max grows by more than 2^8).  At
//                     the end of a task the NG x 4 slices of each row tile
//                     merge their (m, l, O) through shared memory.
// The work is HBM-bound (<= 2 * 32 flop per KV byte at 32 rows), so mma.sync
// is far from its limit; what matters is enough K/V bytes in flight per SM
// (the ring), enough producer threads issuing copies, and enough independent
// warps to hide the MMA / shuffle latency chains (the groups).  E4M3 K/V
// caches run in pa_decode_fp8.cu.
#include "pa_decode_common.cuh"

namespace pa {


template <int D, int RT, int NG, int STAGES, bool STATIC = false>
struct DecodeCfg {
    static constexpr bool kStatic = STATIC;   // static split-K task source (no Assign map)
    static constexpr int kStages = STAGES;
    static constexpr int kTilesPerStage = 1;                  // one 64-token KV tile a stage
    static constexpr int kProducerWarps = STAGES % 4 == 0 ? 4 : 2;
    static constexpr bool kFP8 = false;
    static constexpr int kGroupWarps = 4 * RT;
    static constexpr int kConsumerWarps = kGroupWarps * NG;
    static constexpr int kWarps = kProducerWarps + kConsumerWarps;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int kElem = 2;
    static constexpr int kHalves = D * kElem / 128;          // 128-B column blocks of a K/V row
    static constexpr int kHalfBytes = kDecodeTile * 128;      // one column block of a tile
    static constexpr int kKBytes = kHalves * kHalfBytes;
    // K/V tiles by 8-token group: group g holds its kHalves column blocks of
    // 8 rows x 128 bytes at g * kGroupStride (one block: plain row-major)
    static constexpr int kGroupStride = kHalves * 1024;
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kQRows = 16 * RT;
    static constexpr int kQHalves = D / 64;                   // Q is bf16
    static constexpr int kQHalfBytes = kQRows * 128;
    static constexpr int kQSlotBytes = kQHalves * kQHalfBytes;
    static constexpr int kMergeFloats = 16 * D + 32;
    static constexpr int kMergeBytes = kConsumerWarps * kMergeFloats * 4;
    static constexpr int kOffQ = STAGES * kStageBytes;
    static constexpr int kOffMerge = kOffQ + 2 * kQSlotBytes;
    static constexpr int kOffBar = (kOffMerge + kMergeBytes + 15) / 16 * 16;
    static constexpr int kNumBars = 2 * STAGES + 4;
    static constexpr int kOffArmed = kOffBar + kNumBars * 8 + 16;   // after the abort flag
    static constexpr int kOffFlag = kOffArmed + (4 * (STAGES + 2) + 15) / 16 * 16;  // [RT]
    // static split-K on a cluster: the DSM mailbox of one task's rows and its
    // two mbarriers (only where it fits, and for one row tile)
    static constexpr int kOffMail = kOffFlag + 16;
    static constexpr int kMailWanted = kQRows * (D + kMailPad) * 4;
    static constexpr bool kHasMail =
        STATIC && RT == 1 && kOffMail + kMailWanted + 16 + 1024 <= 232448;
    static constexpr int kOffMailBar = kOffMail + (kHasMail ? kMailWanted : 0);
    static constexpr int kSmemBytes = kOffMailBar + 16 + 1024;
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(kQHalfBytes % 1024 == 0, "Q slot alignment");
    // Group g consumes the tiles with index % NG == g.  Every ring stage must
    // always be consumed by the same group: a group that reused a stage after
    // the other group could wait on a full barrier two phases ahead, where the
    // parity test cannot tell the phases apart.
    static_assert(STAGES % NG == 0, "stages must be a multiple of the tile groups");
    static_assert(kSmemBytes <= 232448, "shared memory");
};


template <int D, int RT, int NG, int STAGES, bool STATIC>
__global__ void __launch_bounds__(DecodeCfg<D, RT, NG, STAGES>::kThreads, 1)
decode_kernel(const __grid_constant__ DecodeParams P, const __grid_constant__ CUtensorMap tmq,
              const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    using Cfg = DecodeCfg<D, RT, NG, STAGES, STATIC>;
    // byte offset in a K/V tile of row `row`, 16-byte chunk c of its 8 * kHalves
    auto kv_off = [](int row, int c) -> uint32_t {
        return (uint32_t)((row >> 3) * Cfg::kGroupStride + (c >> 3) * 1024) + swz(row & 7, c & 7);
    };
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
    uint64_t* empty = full + STAGES;
    uint64_t* q_full = empty + STAGES;       // 2 slots
    uint64_t* q_empty = q_full + 2;          // 2 slots
    volatile int* abort_flag = reinterpret_cast<volatile int*>(q_empty + 2);
    int* armed = reinterpret_cast<int*>(smem + Cfg::kOffArmed);   // last phase armed per stage
    volatile int* fin_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffFlag);
    float* mbox = reinterpret_cast<float*>(smem + Cfg::kOffMail);
    uint64_t* mail_full = reinterpret_cast<uint64_t*>(smem + Cfg::kOffMailBar);
    uint64_t* mail_empty = mail_full + 1;
    // static split-K on clusters of S CTAs: split states merged through DSM
    const bool use_cluster = Cfg::kHasMail && P.cluster_size > 1;
    const int C = use_cluster ? P.cluster_size : 1;
    const WsLayout& L = P.L;
    int32_t* header = ws_ptr<int32_t>(P.ws, L.off_header);
    int32_t* err_hdr = ws_ptr<int32_t>(P.ws, L.off_err_header);   // device faults
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t lim = P.wait_limit_ns;

    grid_dependency_wait();   // Assign's task map is complete
    if (!STATIC && header[H_CTAS] != (int)gridDim.x) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(err_hdr, PA_DEV_BAD_LENGTHS);
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
        for (int s = 0; s < STAGES + 2; ++s) armed[s] = -1;
        if (use_cluster) {
            mbar_init(mail_full, C);    // one arrival from each CTA of the cluster
            mbar_init(mail_empty, C);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (use_cluster) cluster_sync_all();   // every peer's barriers initialised

    auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (mbar_try_wait(bar, parity)) return;   // the usual case, checked first
        if (*abort_flag) return;
        if (!mbar_wait_or_abort(bar, parity, lim, abort_flag)) {
            *abort_flag = 1;
            set_device_error(err_hdr, PA_DEV_WAIT_TIMEOUT);
        }
    };
    auto wait_cluster = [&](uint64_t* bar, uint32_t parity) {
        if (*abort_flag) return;
        if (!mbar_wait_cluster(bar, parity, lim, abort_flag)) {
            *abort_flag = 1;
            set_device_error(err_hdr, PA_DEV_WAIT_TIMEOUT);
        }
    };

    int32_t* done = ws_ptr<int32_t>(P.ws, L.off_done);
    int k_begin, k_end;
    cta_task_range<STATIC>(P, k_begin, k_end);
    const int G = L.G, Hq = L.Hq;

    if (warp < Cfg::kProducerWarps) {
        decode_produce<Cfg>(P, &tmq, &tmk, &tmv, smem, full, empty, q_full, q_empty, nullptr,
                            abort_flag, armed, err_hdr, k_begin, k_end, warp, lane, wait);
    } else {
        // ------------------------------------------------------- consumers
        const int cw = warp - Cfg::kProducerWarps;
        const int grp = cw / Cfg::kGroupWarps;
        const int rt = (cw % Cfg::kGroupWarps) >> 2, ts = cw & 3;
        const int g = lane >> 2, q4 = lane & 3;
        const float scale_log2 = P.sm_scale * kLog2e;
        float* merge = reinterpret_cast<float*>(smem + Cfg::kOffMerge);
        int it = 0, task_it = 0, mround = 0;
        const uint32_t rank = use_cluster ? cluster_ctarank() : 0u;
        TaskRec mine;
        const bool tracer = threadIdx.x == Cfg::kProducerWarps * 32;   // task trace
        for (int k = k_begin; k < k_end; ++k, ++task_it) {
            if (((k - k_begin) & 31) == 0)
                mine = fetch_task_rec<STATIC>(P, k + lane, k_end, lane, err_hdr);
            const TaskRec rec = shfl_task_rec(mine, (k - k_begin) & 31);
            if (tracer) trace_task_start(P.trace, P.trace_cap, k);
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
            // sliding window: keys > p - window (no bound without a window), and
            // task positions count from the unit's first visible tile
            const int w_lo = L.window > 0 ? p_lo - L.window : -1;
            const int w_hi = L.window > 0 ? p_hi - L.window : -1;
            const int first = window_first_tile(L.window, pbase, kDecodeTile);

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
                const int kt = t + first;
                const int tok_s0 = kt * kDecodeTile + 16 * ts;
                uint8_t* stK = smem + s * Cfg::kStageBytes;
                uint8_t* stV = stK + Cfg::kKBytes;
                if (tok_s0 + 15 >= ctx_b) {
                    // tokens past the context: zero their V rows (P is 0 there,
                    // but 0 * NaN would poison O)
                    for (int idx = lane; idx < 16 * Cfg::kHalves * 8; idx += 32) {
                        const int tr = idx / (Cfg::kHalves * 8);
                        const int rem = idx % (Cfg::kHalves * 8);
                        if (tok_s0 + tr >= ctx_b)
                            *reinterpret_cast<uint4*>(stV + kv_off(16 * ts + tr, rem)) =
                                make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                const uint32_t kbase = smem_u32(stK), vbase = smem_u32(stV);
                const int rowbase = 16 * ts;

                // S = Q K^T : 16 rows x 16 tokens, even / odd k-steps in two chains
                float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                float sb[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                {
                    const int mi = lane >> 3;
                    const int trow = rowbase + 8 * (mi >> 1) + (lane & 7);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int dch = 2 * kk + (mi & 1);
                        const uint32_t addr = kbase + kv_off(trow, dch);
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
                const float cs = scale_log2;
                float sv[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = tok_s0 + 8 * j + 2 * q4 + e;
                        const bool okl = v_lo && tok < ctx_b && tok <= p_lo && tok > w_lo;
                        const bool okh = v_hi && tok < ctx_b && tok <= p_hi && tok > w_hi;
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
                pa[0] = pack_bf16x2(p[0][0], p[0][1]);
                pa[1] = pack_bf16x2(p[0][2], p[0][3]);
                pa[2] = pack_bf16x2(p[1][0], p[1][1]);
                pa[3] = pack_bf16x2(p[1][2], p[1][3]);
                // O += P V : V^T fragments via ldmatrix.trans
                {
                    const int mi = lane >> 3;
                    const int trow = rowbase + 8 * (mi & 1) + (lane & 7);
#pragma unroll
                    for (int jd = 0; jd < D / 8; jd += 2) {
                        const int dch = jd + (mi >> 1);
                        const uint32_t addr = vbase + kv_off(trow, dch);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(addr, b0, b1, b2, b3);
                        mma_bf16_16816(o[jd], pa, b0, b1);
                        mma_bf16_16816(o[jd + 1], pa, b2, b3);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
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
            // the mailbox is rewritten below: every peer has read this CTA's
            // previous round
            if (use_cluster && tk.w >= 0 && mround > 0)
                wait_cluster(mail_empty, (uint32_t)((mround - 1) & 1));
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
                        } else if (use_cluster) {
                            float* dst = mbox + r * (D + kMailPad);
#pragma unroll
                            for (int e = 0; e < DPL; ++e) dst[lane * DPL + e] = acc[e] * inv;
                            if (lane == 0) dst[D] = lse_nat;
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
            if (use_cluster && tk.w >= 0) {
                // the cluster's S CTAs hold the S splits of this unit: merge
                // them through DSM, rows sharded by rank (one row tile here)
                fence_acq_rel_cluster();
                named_bar_sync(5 + rt, 128 * NG);
                if (slice == 0 && lane == 0)
                    for (int q = 0; q < C; ++q)
                        mbar_arrive_cluster(mapa_shared(smem_u32(mail_full), (uint32_t)q));
                wait_cluster(mail_full, (uint32_t)(mround & 1));
                cluster_merge_rows<D>(P, mbox, R, (int)rank, C, slice, 4 * NG, tok_base, G, Hq,
                                      hk, lane);
                named_bar_sync(5 + rt, 128 * NG);
                if (slice == 0 && lane == 0)
                    for (int q = 0; q < C; ++q)
                        mbar_arrive_cluster(mapa_shared(smem_u32(mail_empty), (uint32_t)q));
                ++mround;
            } else if (tk.w >= 0) {
                // a split unit: the last of its tasks to finish merges the
                // partials of this row tile into the output (no Combine pass)
                const int u = tk.x;
                const int2 sp = unit_splits<STATIC>(P, u);   // (S, first slot)
                if (split_task_done(done + (int64_t)u * kDoneWords + rt, sp.x, 5 + rt, 128 * NG,
                                    slice == 0 && lane == 0, fin_flag + rt)) {
                    constexpr int kRowsPerWarp = 16 / (4 * NG);
#pragma unroll
                    for (int i = 0; i < kRowsPerWarp; ++i) {
                        const int r = 16 * rt + slice * kRowsPerWarp + i;
                        if (r < R)
                            finalize_split_row<D / 32>(
                                P, sp.y, sp.x, r,
                                (int64_t)(tok_base + r / G) * Hq + hk * G + r % G, lane);
                    }
                }
            }
            named_bar_sync(5 + rt, 128 * NG);
            if (tracer) trace_task_end(P.trace, P.trace_cap, k);
        }
    }
    grid_launch_dependents();
    // every warp is done: after an abort the producers wait for their copies
    // still in flight
    __syncthreads();
    if (warp < Cfg::kProducerWarps) decode_drain<Cfg>(full, q_full, armed, abort_flag, warp, lane);
    // no CTA leaves while a peer may still read its mailbox or arrive on it
    if (use_cluster) cluster_sync_all();
}

template <int D, int RT, int NG, int STAGES>
static cudaError_t launch_variant(const DecodeParams& P, const CUtensorMap& tq,
                                  const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t stream) {
    using Cfg = DecodeCfg<D, RT, NG, STAGES>;
    using CfgS = DecodeCfg<D, RT, NG, STAGES, true>;
    const bool st = P.static_splits > 0;
    auto kern = st ? decode_kernel<D, RT, NG, STAGES, true> : decode_kernel<D, RT, NG, STAGES, false>;
    const int smem = st ? CfgS::kSmemBytes : Cfg::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (st && P.cluster_size > 1)
        e = launch_in_clusters(kern, dim3(P.L.N), dim3(Cfg::kThreads), smem, stream,
                               P.cluster_size, P, tq, tk, tv);
    else
        e = launch_dependent(kern, dim3(P.L.N), dim3(Cfg::kThreads), smem, stream, P, tq, tk, tv);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Static split-K on clusters of C CTAs: 0 if the variant has no DSM mailbox,
// else the largest grid of co-resident clusters (C * clusters).
template <int D, int RT, int NG, int STAGES>
static int cluster_grid_variant(int C) {
    using CfgS = DecodeCfg<D, RT, NG, STAGES, true>;
    if (!CfgS::kHasMail) return 0;
    auto kern = decode_kernel<D, RT, NG, STAGES, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             CfgS::kSmemBytes) != cudaSuccess)
        return 0;
    return max_cluster_grid((const void*)kern, CfgS::kThreads, CfgS::kSmemBytes, C);
}

// (head_dim, row tiles, tile groups, stages) built
#ifndef PA_DECODE_NG_128_1
#define PA_DECODE_NG_128_1 2
#endif
#ifndef PA_DECODE_ST_128_1
#define PA_DECODE_ST_128_1 4
#endif
#define PA_DECODE_VARIANTS(X)                                             \
    X(128, 1, PA_DECODE_NG_128_1, PA_DECODE_ST_128_1)              \
    X(128, 2, 1, 4)    \
    X(64, 1, 2, 8)     \
    X(64, 2, 1, 8)     \
    X(64, 4, 1, 6)

// E4M3 K/V: the kernels of pa_decode_fp8.cu
int decode_fp8_row_tiles(int rows);
int decode_fp8_smem_bytes(int nt);
int decode_fp8_threads(int nt);
const void* decode_fp8_kernel_ptr(int nt);
cudaError_t launch_decode_fp8(const DecodeParams& P, int nt, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream);

namespace {

// query rows of one decode unit (G heads x the longest q_len)
int unit_rows(const pa_problem& p) {
    return (p.num_q_heads / p.num_kv_heads) * (p.max_q_len > 0 ? p.max_q_len : 1);
}
// 16-row tiles of the bf16 kernel
int bf16_row_tiles(int rows) { return rows <= 16 ? 1 : rows <= 32 ? 2 : 4; }
bool is_fp8(const pa_problem& p) { return p.kv_dtype == PA_FP8_E4M3; }

}  // namespace

int decode_smem_bytes(const pa_problem& p) {
    if (is_fp8(p))
        return p.head_dim == 128 ? decode_fp8_smem_bytes(decode_fp8_row_tiles(unit_rows(p))) : -1;
    const int D = p.head_dim, RT = bf16_row_tiles(unit_rows(p));
#define X(d, rt, ng, st) \
    if (D == d && RT == rt) return DecodeCfg<d, rt, ng, st>::kSmemBytes;
    PA_DECODE_VARIANTS(X)
#undef X
    return -1;
}

int decode_threads(const pa_problem& p) {
    if (is_fp8(p))
        return p.head_dim == 128 ? decode_fp8_threads(decode_fp8_row_tiles(unit_rows(p))) : -1;
    const int D = p.head_dim, RT = bf16_row_tiles(unit_rows(p));
#define X(d, rt, ng, st) \
    if (D == d && RT == rt) return DecodeCfg<d, rt, ng, st>::kThreads;
    PA_DECODE_VARIANTS(X)
#undef X
    return -1;
}

const void* decode_kernel_ptr(const pa_problem& p) {
    if (is_fp8(p))
        return p.head_dim == 128 ? decode_fp8_kernel_ptr(decode_fp8_row_tiles(unit_rows(p)))
                                 : nullptr;
    const int D = p.head_dim, RT = bf16_row_tiles(unit_rows(p));
#define X(d, rt, ng, st) \
    if (D == d && RT == rt) return (const void*)decode_kernel<d, rt, ng, st, false>;
    PA_DECODE_VARIANTS(X)
#undef X
    return nullptr;
}

static cudaError_t launch_decode(const DecodeParams& P, int D, int RT, const CUtensorMap& tq,
                                 const CUtensorMap& tk, const CUtensorMap& tv,
                                 cudaStream_t stream) {
#define X(d, rt, ng, st) \
    if (D == d && RT == rt) return launch_variant<d, rt, ng, st>(P, tq, tk, tv, stream);
    PA_DECODE_VARIANTS(X)
#undef X
    return cudaErrorInvalidValue;
}

int decode_fp8_cluster_grid(int nt, int C);
bool decode_fp8_has_mail(int nt);

// Static split-K on clusters of C CTAs for this problem: whether the kernel
// variant carries the DSM mailbox, and the persistent grid (0 if not).
bool decode_has_mail(const pa_problem& p) {
    if (is_fp8(p)) return p.head_dim == 128 && decode_fp8_has_mail(decode_fp8_row_tiles(unit_rows(p)));
    const int D = p.head_dim, RT = bf16_row_tiles(unit_rows(p));
#define X(d, rt, ng, st) \
    if (D == d && RT == rt) return DecodeCfg<d, rt, ng, st, true>::kHasMail;
    PA_DECODE_VARIANTS(X)
#undef X
    return false;
}

int decode_cluster_grid(const pa_problem& p, int C) {
    if (is_fp8(p))
        return p.head_dim == 128 ? decode_fp8_cluster_grid(decode_fp8_row_tiles(unit_rows(p)), C)
                                 : 0;
    const int D = p.head_dim, RT = bf16_row_tiles(unit_rows(p));
#define X(d, rt, ng, st) \
    if (D == d && RT == rt) return cluster_grid_variant<d, rt, ng, st>(C);
    PA_DECODE_VARIANTS(X)
#undef X
    return 0;
}

cudaError_t launch_decode_from_api(const pa_problem& p, const WsLayout& L,
                                   const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv,
                                   const int32_t* block_table,
                                   const int32_t* ctx, const int32_t* ql, const float* ks,
                                   const float* vs, void* ws, void* partial, void* out, float* lse,
                                   cudaStream_t stream, bool take_hook, int static_splits,
                                   int cluster_size) {
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
    P.kv_chunk_mul = p.layout == PA_NHD ? 2 : 0;
    P.kv_page_mul = p.layout == PA_NHD ? 1 : p.num_kv_heads;
    P.kv_head_add = p.layout == PA_NHD ? 0 : 1;
    P.sm_scale = p.sm_scale;
    P.static_splits = static_splits;
    P.cluster_size = cluster_size;
    P.test_skip_it = -1;
    P.wait_limit_ns = kWaitLimitNs;
    if (take_hook) take_test_hook(&P.test_skip_it, &P.wait_limit_ns);
    // the task trace follows the Assign map's task numbering: not on the
    // static path, nor on the decode part of a mixed batch
    P.trace = nullptr;
    P.trace_cap = 0;
    if (take_hook && static_splits == 0) take_task_trace(&P.trace, &P.trace_cap);
    if (is_fp8(p)) {
        if (p.head_dim != 128) return cudaErrorInvalidValue;
        return launch_decode_fp8(P, decode_fp8_row_tiles(unit_rows(p)), tq, tk, tv, stream);
    }
    return launch_decode(P, p.head_dim, bf16_row_tiles(unit_rows(p)), tq, tk, tv, stream);
}

}  // namespace pa
