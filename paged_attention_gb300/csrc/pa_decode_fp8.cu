// pa_decode_fp8.cu -- split-K decode compute for E4M3 K/V caches on legacy
// mma.sync, the kernel of the static split-K path (pa_decode_static).  The
// Assign-map decode runs on the tcgen05 kernel of pa_decode_fp8_tc.cu.
//
// "基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 (Split-K Compute:
// persistent CTAs follow the task map and emit a final or partial output with
// its LSE), 三.1 (small-M geometry: the G*q_len query rows of one KV head
// share every K/V tile), 三.2 (paged K/V through one tile descriptor for NHD
// and HND); FP8 KV with fp32 scales per (page, KV head).
//
// GB300 design.  One CTA per SM, persistent over Assign's task map:
//   warps 0..3   the shared TMA producer (pa_decode_common.cuh), tile
//                it on warp it % 4: the unit's Q rows into one of two Q slots,
//                64-token K and V tiles of E4M3 bytes into a kStages ring,
//                each page's scales beside them.
//   warps 4..11  consumers: 2 tile groups (one warpgroup each) x 4 token
//                slices.  Group g takes the tiles with index % 2 == g; warp
//                (g, ts) owns tokens [16ts, 16ts+16) of its tiles and all
//                R = G*q_len <= 8*NT rows.
// Launched with 168 registers a thread (three warps per SM sub-partition);
// setmaxnreg moves them to 72 for the producer warpgroup and 216 for the
// consumers, who hold the O^T accumulators (32*NT floats) in registers.
// The decode is HBM-bound: at ~70 % of HBM an SM must retire a 16 KB tile
// every ~1100 cycles, so the consumers may not spend a shared-memory round
// trip and a barrier per tile on turning E4M3 into something the MMA takes.
// Instead the bytes go from the ring straight into mma.sync fragments:
//   - Scores are computed transposed, S^T = K Q^T (m16n8k16, M = 16 tokens,
//     N = 8 rows per n-tile, K = head_dim).  The K operand is then the
//     row-major E4M3 tile, and a thread's A-fragment pairs are consecutive
//     bytes of one token's row once head_dim is visited in a permuted order:
//     thread quad q reads bytes [32q, 32q+32) of a row, k-block kk uses the 4
//     bytes at 32q + 4kk.  Each 16-bit pair converts with one exact
//     cvt.rn.f16x2.e4m3x2.  Q is converted once per task to f16 in shared
//     memory and read in the same order.
//   - P^T leaves the score accumulators in the C-fragment layout; one
//     movmatrix transpose per 8x8 block makes it the B operand of
//     O^T = V^T P^T.  The V^T A-fragments pair two tokens' bytes at one
//     head_dim position (one prmt for two fragment registers), again
//     converted exactly by cvt.rn.f16x2.e4m3x2.  P is f16 and carries v_scale
//     times a power of two that brings the warp's first v_scale of the task to
//     [1, 2); the merge divides it out.  (P <= 2^8 after the lazy max, so
//     pages whose v_scale is within 2^7 of that first one stay inside the f16
//     range; the conversion saturates beyond.)  V bytes of tokens past the
//     context are zeroed: the E4M3 NaN codes would otherwise turn 0 * V into
//     NaN.
//   - A warp releases its ring stage as soon as its slice's 128 bytes of K
//     and V are in registers; no converted copy is written and no barrier is
//     taken per tile.
// Per task the 4*NG partial (m, l, O) states of the unit merge through
// shared memory (two rounds, fixed order: deterministic).
#include "pa_decode_common.cuh"

namespace pa {

// GENERAL: the instantiation that also takes the static split-K task source
// and the sliding window (the only one built); with GENERAL = false the loops
// carry neither.
template <int NT, int STAGES, bool GENERAL = false>
struct DecodeFp8Cfg {
    static constexpr bool kStatic = GENERAL;   // may take the static split-K task source
    static constexpr int D = 128;
    // geometry the shared producer reads
    static constexpr int kStages = STAGES;
    static constexpr int kTilesPerStage = 1;                  // one 64-token KV tile a stage
    static constexpr int kProducerWarps = 4;                 // the whole first warpgroup
    static constexpr bool kFP8 = true;
    static constexpr int kElem = 1;
    static constexpr int kHalves = 1;                         // a K/V row is 128 bytes
    static constexpr int kHalfBytes = kDecodeTile * 128;      // 64 rows x 128 B
    static constexpr int kKBytes = kHalfBytes;
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kRows = 8 * NT;                      // unit rows covered
    static constexpr int kQHalves = 2;                        // Q is bf16: two column blocks
    static constexpr int kQHalfBytes = kRows * 128;
    static constexpr int kQSlotBytes = kQHalves * kQHalfBytes;
    // consumers
    static constexpr int NG = 2;                              // tile groups
    static constexpr int kConsumerWarps = 4 * NG;
    static constexpr int kConsumerThreads = 32 * kConsumerWarps;
    static constexpr int kThreads = 128 + kConsumerThreads;   // producer warpgroup + consumers
    static constexpr int kRegsLaunch = 168;
    static constexpr int kRegsProducer = 72;
    static constexpr int kRegsConsumer = 216;
    static_assert(128 * kRegsProducer + kConsumerThreads * kRegsConsumer <=
                      kThreads * kRegsLaunch,
                  "setmaxnreg split exceeds the registers the block is launched with");
    static constexpr int kQhBytes = kRows * D * 2;            // f16 Q
    static constexpr int kMergeStride = D + 4;                // floats per merge row
    static constexpr int kMergeBufs = 4;
    static constexpr int kMergeBytes = kMergeBufs * kRows * kMergeStride * 4;
    static constexpr int kMLBytes = kConsumerWarps * kRows * 2 * 4;
    static constexpr int kScaleBytes = STAGES * 2 * 4 * 4;
    static constexpr int kOffQ = STAGES * kStageBytes;
    static constexpr int kOffQh = kOffQ + 2 * kQSlotBytes;
    static constexpr int kOffMerge = kOffQh + kQhBytes;
    static constexpr int kOffML = kOffMerge + kMergeBytes;
    static constexpr int kOffScale = kOffML + kMLBytes;
    static constexpr int kOffBar = (kOffScale + kScaleBytes + 15) / 16 * 16;
    static constexpr int kNumBars = 2 * STAGES + 4;
    static constexpr int kOffArmed = kOffBar + kNumBars * 8 + 16;   // after the abort flag
    static constexpr int kOffFlag = kOffArmed + (4 * (STAGES + 2) + 15) / 16 * 16;
    // static split-K on a cluster: the DSM mailbox of one task's rows and its
    // two mbarriers (only where it fits)
    static constexpr int kOffMail = kOffFlag + 16;
    static constexpr int kMailWanted = kRows * (D + kMailPad) * 4;
    static constexpr bool kHasMail = GENERAL && kOffMail + kMailWanted + 16 + 1024 <= 232448;
    static constexpr int kOffMailBar = kOffMail + (kHasMail ? kMailWanted : 0);
    static constexpr int kSmemBytes = kOffMailBar + 16 + 1024;
    static_assert(NT >= 1 && NT <= 4, "rows per unit");
    // every ring stage is always consumed by the same group (a group that
    // reused a stage after the other could wait two phases ahead)
    static_assert(STAGES % NG == 0, "stages must be a multiple of the tile groups");
    static_assert(kQHalfBytes % 1024 == 0, "Q slot alignment for the 128-byte swizzle");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// 16-byte chunk c (head_dim [8c, 8c+8)) of f16 Q row r: chunks 8..15 are
// XOR-ed with 2 and odd rows with 1, so that the eight lanes of each
// 128-bit load phase (two rows, four thread quads) hit eight distinct bank
// groups.
__device__ __forceinline__ int qh_chunk(int c, int r) { return c ^ ((c >> 3) << 1) ^ (r & 1); }

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
    return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <int NT, int STAGES, bool GENERAL>
__global__ void __launch_bounds__(384, 1)
decode_fp8_kernel(const __grid_constant__ DecodeParams P, const __grid_constant__ CUtensorMap tmq,
                  const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    using Cfg = DecodeFp8Cfg<NT, STAGES, GENERAL>;
    static_assert(Cfg::kThreads == 384, "launch bounds");
    constexpr int NG = Cfg::NG;
    constexpr int D = Cfg::D;
    constexpr int kRows = Cfg::kRows;
    constexpr int kCW = Cfg::kConsumerWarps;
    constexpr int kCT = Cfg::kConsumerThreads;
    constexpr int kBarConsumers = 1;           // named barrier of the consumer warps
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
    const bool use_cluster = Cfg::kHasMail && P.static_splits > 0 && P.cluster_size > 1;
    const int C = use_cluster ? P.cluster_size : 1;
    float* scales = reinterpret_cast<float*>(smem + Cfg::kOffScale);   // [stage][k|v][box]
    const WsLayout& L = P.L;
    int32_t* header = ws_ptr<int32_t>(P.ws, L.off_header);
    int32_t* err_hdr = ws_ptr<int32_t>(P.ws, L.off_err_header);   // device faults
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t lim = P.wait_limit_ns;

    grid_dependency_wait();   // Assign's task map is complete
    if ((!GENERAL || P.static_splits == 0) && header[H_CTAS] != (int)gridDim.x) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(err_hdr, PA_DEV_BAD_LENGTHS);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);          // the 4 slice warps of the stage's group
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], kCW);
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

    int k_begin, k_end;
    cta_task_range<GENERAL>(P, k_begin, k_end);

    if (warp < 4) {
        regs_dec<Cfg::kRegsProducer>();
        decode_produce<Cfg>(P, &tmq, &tmk, &tmv, smem, full, empty, q_full, q_empty, scales,
                            abort_flag, armed, err_hdr, k_begin, k_end, warp, lane, wait);
    } else {
        regs_inc<Cfg::kRegsConsumer>();
        // ------------------------------------------------------- consumers
        const int cw = warp - 4;
        const int grp = cw >> 2, ts = cw & 3;
        const int g = lane >> 2, q4 = lane & 3;
        const int G = L.G, Hq = L.Hq;
        const float scale_log2 = P.sm_scale * kLog2e;
        uint8_t* qh = smem + Cfg::kOffQh;
        float* mbuf = reinterpret_cast<float*>(smem + Cfg::kOffMerge);
        float* ml = reinterpret_cast<float*>(smem + Cfg::kOffML);
        // scale box of this warp's token slice (a slice never spans two pages)
        const int box = (16 * ts) / P.rows_per_box;
        // byte offsets of this thread's four 16-byte Q chunks in n-tile 0
        // (n-tile nt adds nt * 8 rows; 8 is even, so the swizzle is unchanged)
        uint32_t qoff[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qoff[i] = g * (D * 2) + (qh_chunk(4 * q4 + i, g) << 4);
        // byte offsets inside a stage of this thread's K pieces (token rows g
        // and g+8 of the slice, bytes [32q4, 32q4+32)) and V pieces (token rows
        // 2q4, 2q4+1, 2q4+8, 2q4+9, bytes [16g, 16g+16))
        const int kr0 = 16 * ts + g, vr0 = 16 * ts + 2 * q4;
        const uint32_t koff[4] = {swz(kr0, 2 * q4), swz(kr0, 2 * q4 + 1), swz(kr0 + 8, 2 * q4),
                                  swz(kr0 + 8, 2 * q4 + 1)};
        const uint32_t voff[4] = {swz(vr0, g), swz(vr0 + 1, g), swz(vr0 + 8, g),
                                  swz(vr0 + 9, g)};
        int it = 0, task_it = 0, mround = 0;
        const uint32_t rank = use_cluster ? cluster_ctarank() : 0u;
        TaskRec mine;
        for (int k = k_begin; k < k_end; ++k, ++task_it) {
            if (((k - k_begin) & 31) == 0)
                mine = fetch_task_rec<GENERAL>(P, k + lane, k_end, lane, err_hdr);
            const TaskRec rec = shfl_task_rec(mine, (k - k_begin) & 31);
            const int4 tk = rec.tk;
            const int4 un = rec.un;
            const int hk = un.y, q0 = un.z, nq = un.w;
            const int R = G * nq;
            const int ctx_b = rec.ctx, ql_b = rec.ql;
            const int tok_base = rec.cuq + q0;
            const int pbase = ctx_b - ql_b + q0;
            // this thread's rows are 8nt + 2q4 + e; the last key each may see,
            // its own position p (p <= ctx - 1 in decode; -1 for padding
            // rows).  With a sliding window ("HiLS-Attention", 二.1 local
            // branch) the row sees the keys p - window < j <= p: tok is visible
            // iff tok <= lastk and tok + win > lastk (win is huge without one).
            int lastk[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = 8 * nt + 2 * q4 + e;
                    const int pr = pbase + r / G;
                    lastk[nt][e] = r < R ? (pr < ctx_b - 1 ? pr : ctx_b - 1) : -1;
                }
            const int win = GENERAL && L.window > 0 ? L.window : (1 << 30);
            // task positions count from the unit's first visible tile; every
            // row of the unit sees a key when it is >= first_open
            const int first = GENERAL ? window_first_tile(L.window, pbase, kDecodeTile) : 0;
            const int first_open = GENERAL && L.window > 0 ? pbase + nq - L.window : 0;

            // ---- Q of the unit: bf16 slot -> f16 rows in head_dim order, then
            // release the slot.  Every consumer warp has left the previous
            // task's merge when it passes this barrier.
            {
                const int qs = task_it & 1;
                wait(&q_full[qs], (uint32_t)((task_it >> 1) & 1));
                const uint8_t* qslot = smem + Cfg::kOffQ + qs * Cfg::kQSlotBytes;
                for (int idx = threadIdx.x - 128; idx < kRows * 16; idx += kCT) {
                    const int r = idx >> 4, c = idx & 15;
                    const uint4 v = lds128(qslot + (c >> 3) * Cfg::kQHalfBytes + swz(r, c & 7));
                    const uint4 h = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y),
                                               bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
                    *reinterpret_cast<uint4*>(qh + r * (D * 2) + (qh_chunk(c, r) << 4)) = h;
                }
                named_bar_sync(kBarConsumers, kCT);
                if (lane == 0) mbar_arrive(&q_empty[qs]);
            }

            float m[NT][2], l[NT][2];
            float o[8][NT][4];
            float vpow = 0.f;   // set at this warp's first tile of the task
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                m[nt][0] = m[nt][1] = -INFINITY;
                l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
                for (int mb = 0; mb < 8; ++mb)
                    o[mb][nt][0] = o[mb][nt][1] = o[mb][nt][2] = o[mb][nt][3] = 0.f;
            }

            for (int t = tk.y; t < tk.z; ++t, ++it) {
                if (NG > 1 && (it % NG) != grp) continue;
                const int s = it % STAGES;
                wait(&full[s], (uint32_t)((it / STAGES) & 1));
                const uint8_t* stK = smem + s * Cfg::kStageBytes;
                const uint8_t* stV = stK + Cfg::kKBytes;
                const float ksc = scales[(s * 2 + 0) * 4 + box];
                const float vsc = scales[(s * 2 + 1) * 4 + box];
                // this slice's K and V bytes; then the stage goes back to the
                // producer
                uint4 kw[2][2], vw[4];
                kw[0][0] = lds128(stK + koff[0]);
                kw[0][1] = lds128(stK + koff[1]);
                kw[1][0] = lds128(stK + koff[2]);
                kw[1][1] = lds128(stK + koff[3]);
                // V bytes: before the score product (their latency hides under
                // it) unless the 32-row tile needs those registers
                constexpr bool kEarlyV = NT <= 3;
                auto load_v = [&]() {
                    vw[0] = lds128(stV + voff[0]);
                    vw[1] = lds128(stV + voff[1]);
                    vw[2] = lds128(stV + voff[2]);
                    vw[3] = lds128(stV + voff[3]);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);   // the stage's bytes are in registers
                    // tokens past the context (slots after the last one of the
                    // sequence, or pages not loaded): P is 0 there, but E4M3 NaN
                    // codes would still poison the product
                    const int tok_v = (t + first) * kDecodeTile + 16 * ts;
                    if (tok_v + 15 >= ctx_b) {
                        const int dt[4] = {2 * q4, 2 * q4 + 1, 2 * q4 + 8, 2 * q4 + 9};
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            if (tok_v + dt[x] >= ctx_b) vw[x] = make_uint4(0u, 0u, 0u, 0u);
                    }
                };
                if (kEarlyV) load_v();

                // ---- S^T = K Q^T over head_dim in the permuted order; with
                // registers to spare, even and odd k-blocks accumulate in
                // separate chains
                constexpr int kChains = NT <= 3 ? 2 : 1;
                float sacc[2][NT][4];
#pragma unroll
                for (int h = 0; h < kChains; ++h)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        sacc[h][nt][0] = sacc[h][nt][1] = sacc[h][nt][2] = sacc[h][nt][3] = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {            // 16-byte chunk of each Q row
                    uint4 qv[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        qv[nt] = lds128(qh + nt * 8 * (D * 2) + qoff[i]);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {        // k-block kk = 2i + h
                        const int kk = 2 * i + h;
                        const uint32_t w0 = word_of(kw[0][kk >> 2], kk & 3);
                        const uint32_t w1 = word_of(kw[1][kk >> 2], kk & 3);
                        uint32_t a[4];
                        a[0] = e4m3x2_to_f16x2((uint16_t)(w0 & 0xffffu));
                        a[1] = e4m3x2_to_f16x2((uint16_t)(w1 & 0xffffu));
                        a[2] = e4m3x2_to_f16x2((uint16_t)(w0 >> 16));
                        a[3] = e4m3x2_to_f16x2((uint16_t)(w1 >> 16));
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_f16_16816(sacc[h % kChains][nt], a, word_of(qv[nt], 2 * h),
                                          word_of(qv[nt], 2 * h + 1));
                    }
                }

                if (!kEarlyV) load_v();

                // ---- mask + online softmax (log2 domain, lazily moved max)
                const int tok0 = (t + first) * kDecodeTile + 16 * ts;   // the slice's first token
                const int tok = tok0 + g;                                // token of sacc[.][0..1]
                const float cs = scale_log2 * ksc;
                float sv[NT][4];
                bool need = false;
                // every row sees every token of the slice: no mask to apply
                const bool open = GENERAL ? R == kRows && tok0 + 15 <= pbase && tok0 >= first_open
                                          : R == kRows && tok0 + 15 <= pbase;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float s0 = kChains == 2 ? sacc[0][nt][e] + sacc[1][nt][e]
                                                      : sacc[0][nt][e];
                        const float s2 = kChains == 2 ? sacc[0][nt][2 + e] + sacc[1][nt][2 + e]
                                                      : sacc[0][nt][2 + e];
                        bool vis0, vis8;
                        if constexpr (GENERAL) {
                            vis0 = tok <= lastk[nt][e] && tok + win > lastk[nt][e];
                            vis8 = tok + 8 <= lastk[nt][e] && tok + 8 + win > lastk[nt][e];
                        } else {
                            vis0 = tok <= lastk[nt][e];
                            vis8 = tok + 8 <= lastk[nt][e];
                        }
                        sv[nt][e] = open || vis0 ? s0 * cs : -INFINITY;
                        sv[nt][2 + e] = open || vis8 ? s2 * cs : -INFINITY;
                        need |= fmaxf(sv[nt][e], sv[nt][2 + e]) > m[nt][e] + 8.f;
                    }
                if (__any_sync(0xffffffffu, need)) {
                    // row max over the 8 lanes holding the row's tokens
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            float mx = fmaxf(sv[nt][e], sv[nt][2 + e]);
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                            if (mx > m[nt][e] + 8.f) {
                                const float al = ex2(m[nt][e] - mx);   // 0 while m = -inf
                                m[nt][e] = mx;
                                l[nt][e] *= al;
#pragma unroll
                                for (int mb = 0; mb < 8; ++mb) {
                                    o[mb][nt][e] *= al;
                                    o[mb][nt][2 + e] *= al;
                                }
                            }
                        }
                }
                // P = 2^(s - m); the PV operand (f16) carries v_scale times the
                // power of two that brought this warp's first v_scale of the
                // task to [1, 2) -- P then stays far inside the f16 range for
                // scales within 2^7 of that one, and saturates beyond
                if (vpow == 0.f) {
                    const uint32_t ex = (__float_as_uint(vsc) >> 23) & 0xffu;
                    vpow = ex == 0u || ex == 255u ? 1.f
                                                  : __uint_as_float((254u - (ex < 253u ? ex : 253u)) << 23);
                }
                const float vsw = vsc * vpow;
                uint32_t pb[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float mu0 = m[nt][0] == -INFINITY ? 0.f : m[nt][0];
                    const float mu1 = m[nt][1] == -INFINITY ? 0.f : m[nt][1];
                    const float p0 = ex2(sv[nt][0] - mu0), p1 = ex2(sv[nt][1] - mu1);
                    const float p2 = ex2(sv[nt][2] - mu0), p3 = ex2(sv[nt][3] - mu1);
                    l[nt][0] += p0 + p2;
                    l[nt][1] += p1 + p3;
                    // [token][row] 8x8 blocks -> [row][token]: the B fragments
                    pb[nt][0] = movmatrix_trans(pack_f16x2_sat(p0 * vsw, p1 * vsw));
                    pb[nt][1] = movmatrix_trans(pack_f16x2_sat(p2 * vsw, p3 * vsw));
                }

                // ---- O^T += V^T P^T; A-fragment rows are head_dim in the order
                // thread g <-> [16g, 16g+16), block mb <-> pair (16g+2mb, +1)
#pragma unroll
                for (int mb = 0; mb < 8; ++mb) {
                    const int wi = mb >> 1;
                    const uint32_t v0 = word_of(vw[0], wi), v1 = word_of(vw[1], wi);
                    const uint32_t v2 = word_of(vw[2], wi), v3 = word_of(vw[3], wi);
                    // {t0.d, t1.d, t0.d+1, t1.d+1} -> the (d, d+1) fragment pair
                    const uint32_t x01 = (mb & 1) ? interleave_bytes<2>(v0, v1)
                                                  : interleave_bytes<0>(v0, v1);
                    const uint32_t x23 = (mb & 1) ? interleave_bytes<2>(v2, v3)
                                                  : interleave_bytes<0>(v2, v3);
                    uint32_t a[4];
                    a[0] = e4m3x2_to_f16x2((uint16_t)(x01 & 0xffffu));
                    a[1] = e4m3x2_to_f16x2((uint16_t)(x01 >> 16));
                    a[2] = e4m3x2_to_f16x2((uint16_t)(x23 & 0xffffu));
                    a[3] = e4m3x2_to_f16x2((uint16_t)(x23 >> 16));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_f16_16816(o[mb][nt], a, pb[nt][0], pb[nt][1]);
                }
            }

            // ---- merge the 4*NG partial (m, l, O) states of this unit
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float v = l[nt][e];
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    l[nt][e] = v;
                    if (g == 0) {
                        const int r = 8 * nt + 2 * q4 + e;
                        ml[(cw * kRows + r) * 2] = m[nt][e];
                        ml[(cw * kRows + r) * 2 + 1] = v;
                    }
                }
            named_bar_sync(kBarConsumers, kCT);
            // weight 2^(m_w - M) of this warp's state, M = the rows' max over warps
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = 8 * nt + 2 * q4 + e;
                    float M = -INFINITY;
#pragma unroll
                    for (int w = 0; w < kCW; ++w) M = fmaxf(M, ml[(w * kRows + r) * 2]);
                    const float wgt = m[nt][e] == -INFINITY ? 0.f : ex2(m[nt][e] - M) / vpow;
#pragma unroll
                    for (int mb = 0; mb < 8; ++mb) {
                        o[mb][nt][e] *= wgt;
                        o[mb][nt][2 + e] *= wgt;
                    }
                }
            // buffer ts holds the sum over the tile groups of slice ts, as
            // [row][head_dim] fp32
            float* sbuf = mbuf + ts * (kRows * Cfg::kMergeStride);
            auto put = [&](bool add) {
#pragma unroll
                for (int mb = 0; mb < 8; ++mb)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int r = 8 * nt + 2 * q4 + e;
                            float2* dst = reinterpret_cast<float2*>(
                                sbuf + r * Cfg::kMergeStride + 16 * g + 2 * mb);
                            float2 v = make_float2(o[mb][nt][e], o[mb][nt][2 + e]);
                            if (add) {
                                const float2 old = *dst;
                                v.x += old.x;
                                v.y += old.y;
                            }
                            *dst = v;
                        }
            };
            if (NG == 2) {
                if (grp == 1) put(false);
                named_bar_sync(kBarConsumers, kCT);
                if (grp == 0) put(true);
            } else {
                put(false);
            }
            // the mailbox is rewritten below: every peer has read this CTA's
            // previous round
            if (use_cluster && tk.w >= 0 && mround > 0)
                wait_cluster(mail_empty, (uint32_t)((mround - 1) & 1));
            named_bar_sync(kBarConsumers, kCT);
            // one warp per row, 4 head_dim values per lane
            for (int r = cw; r < R; r += kCW) {
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kCW; ++w) M = fmaxf(M, ml[(w * kRows + r) * 2]);
                float Lsum = 0.f;
#pragma unroll
                for (int w = 0; w < kCW; ++w) {
                    const float mw = ml[(w * kRows + r) * 2];
                    if (mw != -INFINITY) Lsum += ex2(mw - M) * ml[(w * kRows + r) * 2 + 1];
                }
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int b = 0; b < Cfg::kMergeBufs; ++b) {
                    const float4 v = *reinterpret_cast<const float4*>(
                        mbuf + (b * kRows + r) * Cfg::kMergeStride + 4 * lane);
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
                const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
                const float lse_nat = Lsum > 0.f ? (M + lg2(Lsum)) * kLn2 : -INFINITY;
                const int token = tok_base + r / G, head = hk * G + r % G;
                if (tk.w < 0) {
                    uint2 v;
                    v.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                    v.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                    *reinterpret_cast<uint2*>(P.out + ((int64_t)token * Hq + head) * D + 4 * lane) = v;
                    if (P.lse != nullptr && lane == 0) P.lse[(int64_t)token * Hq + head] = lse_nat;
                } else if (use_cluster) {
                    float* dst = mbox + r * (D + kMailPad);
                    *reinterpret_cast<float4*>(dst + 4 * lane) =
                        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                    if (lane == 0) dst[D] = lse_nat;
                } else {
                    const int64_t prow = (int64_t)tk.w * L.rows_cap + r;
                    *reinterpret_cast<float4*>(P.part_o + prow * D + 4 * lane) =
                        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                    if (lane == 0) P.part_lse[prow] = lse_nat;
                }
            }
            if (use_cluster && tk.w >= 0) {
                // the cluster's S CTAs hold the S splits of this unit: merge
                // them through DSM, rows sharded by rank
                fence_acq_rel_cluster();
                named_bar_sync(kBarConsumers, kCT);
                if (threadIdx.x == 128)
                    for (int q = 0; q < C; ++q)
                        mbar_arrive_cluster(mapa_shared(smem_u32(mail_full), (uint32_t)q));
                wait_cluster(mail_full, (uint32_t)(mround & 1));
                cluster_merge_rows<D>(P, mbox, R, (int)rank, C, cw, kCW, tok_base, G, Hq, hk,
                                      lane);
                named_bar_sync(kBarConsumers, kCT);
                if (threadIdx.x == 128)
                    for (int q = 0; q < C; ++q)
                        mbar_arrive_cluster(mapa_shared(smem_u32(mail_empty), (uint32_t)q));
                ++mround;
            }
            if constexpr (GENERAL) {
                // static split-K: the last of a unit's tasks to finish merges
                // its partials (there is no Combine pass on that path).  With
                // an Assign map the partials are left to pa_combine: in this
                // kernel's loop the finalizer costs more than that launch.
                if (tk.w >= 0 && P.static_splits > 0 && !use_cluster) {
                    const int u = tk.x;
                    const int2 sp = unit_splits<GENERAL>(P, u);   // (S, first slot)
                    if (split_task_done(ws_ptr<int32_t>(P.ws, L.off_done) + (int64_t)u * kDoneWords,
                                        sp.x, kBarConsumers, kCT, threadIdx.x == 128, fin_flag))
                        for (int r = cw; r < R; r += kCW)
                            finalize_split_row<4>(
                                P, sp.y, sp.x, r,
                                (int64_t)(tok_base + r / G) * Hq + hk * G + r % G, lane);
                }
            }
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

// (8-row tiles, ring stages) built
#define PA_DECODE_FP8_VARIANTS(X) \
    X(1, 8)                       \
    X(2, 8)                       \
    X(3, 8)                       \
    X(4, 8)

int decode_fp8_row_tiles(int rows) { return (rows + 7) / 8; }

// The Assign-map E4M3 decode runs on the tensor-core kernel
// (pa_decode_fp8_tc.cu); these describe it for the persistent-grid query.
int decode_fp8_tc_smem_bytes(int rows);
int decode_fp8_tc_threads(int rows);
const void* decode_fp8_tc_kernel_ptr(int rows);
int decode_fp8_smem_bytes(int nt) { return decode_fp8_tc_smem_bytes(8 * nt); }
int decode_fp8_threads(int nt) { return decode_fp8_tc_threads(8 * nt); }
const void* decode_fp8_kernel_ptr(int nt) { return decode_fp8_tc_kernel_ptr(8 * nt); }

// static split-K (this file's kernel, the instantiation with the static
// task source)
template <int NT, int STAGES>
static cudaError_t launch_fp8_variant(const DecodeParams& P, const CUtensorMap& tq,
                                      const CUtensorMap& tk, const CUtensorMap& tv,
                                      cudaStream_t stream) {
    using Cfg = DecodeFp8Cfg<NT, STAGES, true>;
    auto kern = decode_fp8_kernel<NT, STAGES, true>;
    const int smem = Cfg::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (P.static_splits > 0 && P.cluster_size > 1)
        e = launch_in_clusters(kern, dim3(P.L.N), dim3(Cfg::kThreads), smem, stream,
                               P.cluster_size, P, tq, tk, tv);
    else
        e = launch_dependent(kern, dim3(P.L.N), dim3(Cfg::kThreads), smem, stream, P, tq, tk, tv);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int NT, int STAGES>
static int fp8_cluster_grid_variant(int C) {
    using CfgG = DecodeFp8Cfg<NT, STAGES, true>;
    if (!CfgG::kHasMail) return 0;
    auto kern = decode_fp8_kernel<NT, STAGES, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             CfgG::kSmemBytes) != cudaSuccess)
        return 0;
    return max_cluster_grid((const void*)kern, CfgG::kThreads, CfgG::kSmemBytes, C);
}

bool decode_fp8_has_mail(int nt) {
#define X(n, st) \
    if (nt == n) return DecodeFp8Cfg<n, st, true>::kHasMail;
    PA_DECODE_FP8_VARIANTS(X)
#undef X
    return false;
}

int decode_fp8_cluster_grid(int nt, int C) {
#define X(n, st) \
    if (nt == n) return fp8_cluster_grid_variant<n, st>(C);
    PA_DECODE_FP8_VARIANTS(X)
#undef X
    return 0;
}

cudaError_t launch_decode_fp8_tc(const DecodeParams& P, int rows, const CUtensorMap& tq,
                                 const CUtensorMap& tk, const CUtensorMap& tv,
                                 cudaStream_t stream);

cudaError_t launch_decode_fp8(const DecodeParams& P, int nt, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    // the Assign map (with or without a window) runs on the tensor-core kernel
    // (pa_decode_fp8_tc.cu); static split-K on this file's kernel
    if (P.static_splits == 0) return launch_decode_fp8_tc(P, 8 * nt, tq, tk, tv, stream);
#define X(n, st) \
    if (nt == n) return launch_fp8_variant<n, st>(P, tq, tk, tv, stream);
    PA_DECODE_FP8_VARIANTS(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace pa
