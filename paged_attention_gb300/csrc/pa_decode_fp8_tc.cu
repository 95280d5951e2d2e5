// pa_decode_fp8_tc.cu -- split-K decode compute for E4M3 K/V caches on the
// tcgen05 tensor cores (kind::f8f6f4), the E4M3 bytes read by the MMA
// straight from the TMA ring.
//
// "基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 (Split-K Compute:
// persistent CTAs follow the task map and emit a final or partial output with
// its LSE), 三.1 (small-M geometry: the G*q_len query rows of one KV head
// share every K/V tile), 三.2 (paged K/V through one tile descriptor for NHD
// and HND); FP8 KV with fp32 scales per (page, KV head).
//
// The decode is HBM-bound: at 70 % of HBM an SM has ~2,200 cycles for the
// 32 KB of K and V of 128 tokens.  Converting those bytes in registers for a
// legacy MMA costs more than that budget, so here the tensor core reads them
// as they landed, and the scores are computed transposed -- the key tokens
// are the MMA's M = 128 rows and the few query rows its N:
//   S^T = K Q^T   M = 128 tokens (two 64-token KV tiles of one ring stage),
//                 N = 3 * NR (NR = query rows rounded up to 16), K = 128:
//                 K is the E4M3 tile, K-major; Q enters as three E4M3 terms
//                 t1 + t2 + t3 of q * 2^e (a power of two per row that puts
//                 its largest element in (224, 448]), which carry q to about
//                 2^-12 relative -- finer than the bf16 q itself.
//   O^T += V^T P^T  M = 128 head dims, N = NR query rows, K = 128 tokens:
//                 V^T is the same V tile read MN-major (no transpose is
//                 written); P^T comes as two E4M3 terms (P and its rounding
//                 residual, about 2^-8 relative), two MMAs per 32 tokens.
// Accumulators live in tensor memory: two S^T buffers (128 columns apart)
// and O^T (NR columns).
//
// Warps (352 threads, one CTA per SM):
//   0-7  softmax, two warpgroups: thread t of a warpgroup = TMEM lane t =
//        token t of the stage's 128; warpgroup w owns the query rows
//        [w NR/2, (w+1) NR/2).  Per stage a thread reads its token's S^T
//        columns (the three Q terms summed), turns them into
//        y = s * sm_scale * log2(e) * 2^-e * k_scale + log2(v_scale) per
//        row, and writes P' = 2^(y - m) as two E4M3 bytes into the P^T
//        operand in shared memory (so v_scale rides in P', and each token's
//        1/v_scale goes into the row sums l).  m is a per-row running
//        maximum shared by the warpgroup's 128 threads: a stage only changes
//        it when some y exceeds m + 8 (one barrier-or per stage decides);
//        then the tile's row maxima are reduced across the threads and O^T
//        and l are rescaled.  The softmax warps also turn Q into its three
//        E4M3 terms at the start of a task and write O / LSE (or the split
//        partial) at its end.
//   8    QK issuer (lane 0) and TMEM owner: S^T of stage g into buffer g % 2.
//   9    PV issuer (lane 0): O^T += V^T P^T of stage g once its P is written;
//        its commits release the ring stage and the P^T buffer.
//   10   TMA producer (pa_decode_common.cuh, two 64-token tiles a stage).
// Registers are handed out per four warps, so eleven warps cost twelve.
#include "pa_decode_common.cuh"

namespace pa {

template <int NR>
struct DecodeTcCfg {
    static_assert(NR == 16 || NR == 32, "query rows of a unit: 16 or 32");
    static constexpr bool kStatic = false;   // the Assign map only
    static constexpr int D = 128;
    // geometry the shared producer reads
    // the deepest ring that fits beside the other buffers: every stage not
    // held by QK, softmax or PV is a copy in flight
    static constexpr int kStages = NR == 16 ? 6 : 4;
    static constexpr int kTilesPerStage = 2;
    static constexpr int kProducerWarps = 2;
    static constexpr bool kFP8 = true;
    static constexpr int kElem = 1;
    static constexpr int kHalves = 1;
    static constexpr int kHalfBytes = kDecodeTile * 128;
    static constexpr int kKBytes = 2 * kDecodeTile * 128;    // 128 token rows of K
    static constexpr int kStageBytes = 2 * kKBytes;          // K rows, then V rows
    static constexpr int kRows = NR;
    static constexpr int kQHalves = 2;                        // bf16 Q: two column blocks
    static constexpr int kQHalfBytes = NR * 128;
    static constexpr int kQSlotBytes = kQHalves * kQHalfBytes;
    // operands written by the softmax warps
    static constexpr int kTerms = 3;                          // E4M3 terms of Q
    static constexpr int kNQK = kTerms * NR;
    static constexpr int kQtBytes = kNQK * 128;
    static constexpr int kPTermBytes = NR * 128;              // one P^T term, NR x 128 tokens
    // P^T layout: 32 rows MN-major (each token's 32 row bytes contiguous,
    // 32-byte swizzle; one 16-byte store per warpgroup), 16 rows K-major (each
    // row's 128 token bytes, 128-byte swizzle; byte stores)
    static constexpr bool kPMN = NR == 32;
    static constexpr int kOffQ = kStages * kStageBytes;
    static constexpr int kOffQt = kOffQ + 2 * kQSlotBytes;
    static constexpr int kOffP = kOffQt + kQtBytes;           // [buffer][term]
    static constexpr int kOffEpi = kOffP + 2 * 2 * kPTermBytes;   // f32 O rows, NR x D
    static constexpr int kOffRed = kOffEpi + NR * D * 4;          // [warpgroup][warp][32]
    static constexpr int kOffRowM = kOffRed + 2 * 4 * 32 * 4;     // running max per row, [2 tasks]
    static constexpr int kOffRowC = kOffRowM + 2 * 32 * 4;    // sm_scale log2(e) 2^-e per row
    static constexpr int kOffScale = kOffRowC + 32 * 4;       // [stage][k|v][8 boxes]
    static constexpr int kOffBar = kOffScale + kStages * 2 * 8 * 4;
    static constexpr int kNumBars = 2 * kStages + 4 + 8 + 4;
    static constexpr int kOffArmed = kOffBar + kNumBars * 8 + 16;   // after TMEM slot, abort flag
    static constexpr int kSmemBytes = kOffArmed + (4 * (kStages + 2) + 15) / 16 * 16 + 1024;
    static constexpr int kThreads = 384;   // 8 softmax, QK, PV, 2 producer warps
    static constexpr uint32_t kTmemCols = 256;
    static constexpr uint32_t kColS = 128;          // S^T buffer b at column b * kColS
    static constexpr uint32_t kColO = 224;
    static_assert(kNQK <= 128 && kColO + NR <= kTmemCols, "tensor-memory columns");
    static_assert(kOffQ % 1024 == 0 && kOffQt % 1024 == 0 && kOffP % 1024 == 0 &&
                      kQHalfBytes % 1024 == 0 && kPTermBytes % 1024 == 0,
                  "128-byte-swizzled operands start on 1024-byte boundaries");
    static_assert(kStages % kProducerWarps == 0, "every stage stays with one producer warp");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// Reduce NR per-thread values across the 32 lanes of a warp, each row on its
// own: the exchange halves the rows a lane keeps at every step, so after it
// lane l holds row l % NR reduced over the warp (31 shuffles for 32 rows).
template <int NR, class Op>
__device__ __forceinline__ float warp_reduce_rows(float (&v)[NR], int lane, Op op) {
#pragma unroll
    for (int half = NR / 2; half >= 1; half >>= 1) {
        const bool up = (lane & half) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float keep = up ? v[i + half] : v[i];
            const float send = up ? v[i] : v[i + half];
            v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, half));
        }
    }
    float r = v[0];
#pragma unroll
    for (int off = NR; off < 32; off <<= 1) r = op(r, __shfl_xor_sync(0xffffffffu, r, off));
    return r;
}

// tcgen05.ld / st of N consecutive 32-bit columns (N = 8 or 16) of this
// warp's 32 lanes.
template <int N>
__device__ __forceinline__ void tmem_ld_rows(uint32_t taddr, float* v) {
    if constexpr (N == 16) {
        tmem_ld16(taddr, v);
    } else {
        static_assert(N == 8, "8 or 16 columns");
        uint32_t* r = reinterpret_cast<uint32_t*>(v);
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                       "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr)
                     : "memory");
    }
}
template <int N>
__device__ __forceinline__ void reg_fence_rows(float* v) {
    if constexpr (N == 16) {
        reg_fence16(v);
    } else {
        asm volatile("" : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                          "+f"(v[6]), "+f"(v[7]));
    }
}
template <int N>
__device__ __forceinline__ void tmem_st_rows(uint32_t taddr, const float* v) {
    const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
    if constexpr (N == 16) {
        tmem_st16(taddr, r);
    } else {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                     ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]),
                       "r"(r[5]), "r"(r[6]), "r"(r[7])
                     : "memory");
    }
}

// Initial running maximum: finite, so 2^(y - m) of a masked score (y = -inf)
// is 0, and below every finite score minus 8.
constexpr float kNoMax = -1e30f;

// Two E4M3 bytes (low byte first) -> two f32, exact.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t two) {
    const uint32_t h = e4m3x2_to_f16x2(two);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Byte offset of byte `col` of row `row` in a 128-byte-swizzled operand tile.
__device__ __forceinline__ uint32_t swz_byte(int row, int col) {
    return (uint32_t)(row * 128 + (((col >> 4) ^ (row & 7)) << 4) + (col & 15));
}

template <int NR>
__global__ void __launch_bounds__(384, 1)
decode_fp8_tc_kernel(const __grid_constant__ DecodeParams P, const __grid_constant__ CUtensorMap tmq,
                     const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
    using Cfg = DecodeTcCfg<NR>;
    constexpr int S = Cfg::kStages;
    constexpr int D = Cfg::D;
    constexpr int kBarAll = 3;                   // named barrier of all 8 softmax warps
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
    uint64_t* empty = full + S;
    uint64_t* q_full = empty + S;      // [2]
    uint64_t* q_empty = q_full + 2;    // [2]
    uint64_t* s_full = q_empty + 2;    // [2]
    uint64_t* s_free = s_full + 2;     // [2]
    uint64_t* p_full = s_free + 2;     // [2]
    uint64_t* p_empty = p_full + 2;    // [2]
    uint64_t* o_full = p_empty + 2;
    uint64_t* o_free = o_full + 1;
    uint64_t* qt_full = o_free + 1;
    uint64_t* mma_done = qt_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + Cfg::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* armed = reinterpret_cast<int*>(smem + Cfg::kOffArmed);
    float* scales = reinterpret_cast<float*>(smem + Cfg::kOffScale);
    float* red = reinterpret_cast<float*>(smem + Cfg::kOffRed);      // [4 warps][32 rows]
    float* row_m = reinterpret_cast<float*>(smem + Cfg::kOffRowM);
    float* row_c = reinterpret_cast<float*>(smem + Cfg::kOffRowC);
    const WsLayout& L = P.L;
    int32_t* header = ws_ptr<int32_t>(P.ws, L.off_header);
    int32_t* err_hdr = ws_ptr<int32_t>(P.ws, L.off_err_header);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t lim = P.wait_limit_ns;

    grid_dependency_wait();   // Assign's task map is complete
    if (header[H_CTAS] != (int)gridDim.x) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(err_hdr, PA_DEV_BAD_LENGTHS);
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);              // the PV commit of the stage
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 8);             // one arrival per softmax warp
            mbar_init(&p_full[i], 8);
            mbar_init(&p_empty[i], 1);
        }
        mbar_init(o_full, 1);
        mbar_init(o_free, 8);                     // one per softmax warp
        mbar_init(qt_full, 1);
        mbar_init(mma_done, 2);                   // the QK and the PV warp
        *abort_flag = 0;
        for (int s = 0; s < S + 2; ++s) armed[s] = -1;
        fence_mbar_init();
    }
    if (warp == 8) {
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

    int k_begin, k_end;
    cta_task_range<false>(P, k_begin, k_end);
    const int G = L.G, Hq = L.Hq;

    if (warp >= 10) {
        // --------------------------------------------------------- producers
        decode_produce<Cfg>(P, &tmq, &tmk, &tmv, smem, full, empty, q_full, q_empty, scales,
                            abort_flag, armed, err_hdr, k_begin, k_end, warp - 10, lane, wait);
    } else if (warp == 8 || warp == 9) {
        // ----------------------------------------------------- MMA issuers
        // warp 8 issues the QKs, warp 9 the PVs: each commit tracks the MMAs
        // of its own thread, and a PV never waits behind the next stage's QK
        // (whose copies may still be in flight), so a stage goes back to the
        // producer as soon as its softmax is done.
        constexpr uint32_t idesc_qk = idesc_e4m3_f32(128, Cfg::kNQK, false, false);
        constexpr uint32_t idesc_pv = idesc_e4m3_f32(128, NR, true, Cfg::kPMN);
        // K-major operands (K as A, Q terms and P^T as B): 128-byte rows, 8-row
        // groups 1024 bytes apart.  V^T as A is MN-major: 128 head dims along
        // M in one 128-byte row per token, 8-token groups 1024 bytes apart.
        const uint64_t dKV = smem_desc_sw128(smem_u32(smem), 16, 1024);
        const uint64_t dQt = smem_desc_sw128(smem_u32(smem + Cfg::kOffQt), 16, 1024);
        // P^T: K-major with the 128-byte swizzle, or MN-major with the 32-byte
        // one (32 row bytes per token, 8-token groups 256 bytes apart)
        const uint64_t dP = Cfg::kPMN ? smem_desc_sw32(smem_u32(smem + Cfg::kOffP), 16, 256)
                                      : smem_desc_sw128(smem_u32(smem + Cfg::kOffP), 16, 1024);
        constexpr int kPStep = Cfg::kPMN ? 32 * 32 : 32;   // bytes per 32 tokens of P^T
        const bool qk_warp = warp == 8;
        int g = 0, task_it = 0, o_tasks = 0;
        TaskRec mine;
        for (int k = k_begin; k < k_end; ++k, ++task_it) {
            if (((k - k_begin) & 31) == 0)
                mine = fetch_task_rec<false>(P, k + lane, k_end, lane, err_hdr);
            const TaskRec rec = shfl_task_rec(mine, (k - k_begin) & 31);
            const int n2 = (rec.tk.z - rec.tk.y + 1) / 2;
            if (qk_warp) {
                wait(qt_full, (uint32_t)(task_it & 1));        // this task's Q terms
                for (int i = 0; i < n2; ++i, ++g) {
                    const int s = g % S, b = g & 1;
                    wait(&full[s], (uint32_t)((g / S) & 1));
                    wait(&s_free[b], (uint32_t)((g >> 1) & 1) ^ 1u);
                    if (lane == 0) {
                        tc_fence_after();
                        const uint64_t a0 = dKV + (uint64_t)((s * Cfg::kStageBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma_ss_f8(tmem + b * Cfg::kColS, a0 + (uint64_t)((kk * 32) >> 4),
                                         dQt + (uint64_t)((kk * 32) >> 4), idesc_qk,
                                         kk > 0 ? 1u : 0u);
                        tc_commit(&s_full[b]);
                    }
                    __syncwarp();
                }
            } else {
                for (int i = 0; i < n2; ++i, ++g) {
                    const int s = g % S, b = g & 1;
                    wait(&p_full[b], (uint32_t)((g >> 1) & 1));
                    if (i == 0) {
                        wait(o_free, (uint32_t)(o_tasks & 1) ^ 1u);   // last epilogue read O^T
                        ++o_tasks;
                    }
                    if (lane == 0) {
                        tc_fence_after();
                        const uint64_t a0 =
                            dKV + (uint64_t)((s * Cfg::kStageBytes + Cfg::kKBytes) >> 4);
#pragma unroll
                        for (int term = 0; term < 2; ++term)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc_mma_ss_f8(
                                    tmem + Cfg::kColO, a0 + (uint64_t)((kk * 32 * 128) >> 4),
                                    dP + (uint64_t)(((b * 2 + term) * Cfg::kPTermBytes + kk * kPStep) >> 4),
                                    idesc_pv, (i == 0 && term == 0 && kk == 0) ? 0u : 1u);
                        // the stage's K was read by its QK, whose scores the
                        // softmax consumed before P was written
                        tc_commit(&empty[s]);
                        tc_commit(&p_empty[b]);
                        if (i == n2 - 1) tc_commit(o_full);
                    }
                    __syncwarp();
                }
            }
        }
        if (lane == 0) {
            tc_commit(mma_done);
            mbar_wait(mma_done, 0, lim);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- softmax
        // warpgroup wg owns query rows [wg * HR, wg * HR + HR) of the unit;
        // thread t of a warpgroup = TMEM lane t = token t of the stage
        constexpr int HR = NR / 2;
        const int wg = warp >> 2, wq = warp & 3;
        const int t = threadIdx.x & 127;
        const int rb = wg * HR;
        const int bar_wg = 1 + wg;                 // named barrier of this warpgroup
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float scale_log2 = P.sm_scale * kLog2e;
        float* redw = red + wg * 128;              // [4 warps][32] of this warpgroup
        const int rpb_log = __ffs(P.rows_per_box) - 1;   // rows per box: a power of two
        uint8_t* qt = smem + Cfg::kOffQt;
        // Q rows of task number `ti` (R of them) -> three E4M3 terms (rows
        // R..NR-1 are zeros); thread u = threadIdx.x of the 256 takes row u / 8,
        // head dims [16 (u % 8), +16).  Also sets the rows' scale factor c and
        // clears their running maximum (task parity ti & 1).
        auto convert_q = [&](int ti, int R) {
            {
                const int qs = ti & 1;
                wait(&q_full[qs], (uint32_t)((ti >> 1) & 1));
                const int u = threadIdx.x;
                const int r = u >> 3, qd = u & 7;
                if (r < NR) {
                    const uint8_t* src = smem + Cfg::kOffQ + qs * Cfg::kQSlotBytes +
                                         (qd >> 2) * Cfg::kQHalfBytes;
                    float v[16];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint4 w = *reinterpret_cast<const uint4*>(
                            src + swz(r, (qd & 3) * 2 + c));
                        const uint32_t ws4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            v[8 * c + 2 * e] = __uint_as_float(ws4[e] << 16);
                            v[8 * c + 2 * e + 1] = __uint_as_float(ws4[e] & 0xffff0000u);
                        }
                    }
                    float amax = 0.f;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        if (r >= R) v[e] = 0.f;
                        amax = fmaxf(amax, fabsf(v[e]));
                    }
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
                    // 2^e with amax * 2^e in (224, 448]: exact scaling
                    int ex = 0;
                    if (amax > 0.f) {
                        frexpf(448.f / amax, &ex);
                        ex -= 1;
                        if (ldexpf(amax, ex) > 448.f) ex -= 1;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = ldexpf(v[e], ex);
                    // t1 = e4m3(x), t2 = e4m3(x - t1), t3 = e4m3(x - t1 - t2)
#pragma unroll 1
                    for (int term = 0; term < 3; ++term) {
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 16; e += 4) {
                            const uint16_t a = f32x2_to_e4m3x2(v[e], v[e + 1]);
                            const uint16_t b2 = f32x2_to_e4m3x2(v[e + 2], v[e + 3]);
                            pk[e / 4] = (uint32_t)a | ((uint32_t)b2 << 16);
                            const float2 fa = e4m3x2_to_f32x2(a);
                            const float2 fb = e4m3x2_to_f32x2(b2);
                            v[e] -= fa.x;
                            v[e + 1] -= fa.y;
                            v[e + 2] -= fb.x;
                            v[e + 3] -= fb.y;
                        }
                        *reinterpret_cast<uint4*>(qt + swz(term * NR + r, qd)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                    if (qd == 0) {
                        row_c[r] = ldexpf(scale_log2, -ex);
                        row_m[(ti & 1) * 32 + r] = kNoMax;
                    }
                }
                fence_proxy_async_smem();
                named_bar_sync(kBarAll, 256);
                if (threadIdx.x == 0) {
                    mbar_arrive(qt_full);
                    mbar_arrive(&q_empty[qs]);
                }
            }
        };
        int g = 0, task_it = 0, o_tasks = 0;
        TaskRec mine;
        bool fetched = false;   // `mine` already holds the batch of the next task
        for (int k = k_begin; k < k_end; ++k, ++task_it) {
            if (((k - k_begin) & 31) == 0 && !fetched)
                mine = fetch_task_rec<false>(P, k + lane, k_end, lane, err_hdr);
            fetched = false;
            const TaskRec rec = shfl_task_rec(mine, (k - k_begin) & 31);
            if (threadIdx.x == 0) trace_task_start(P.trace, P.trace_cap, k);
            const int4 tk = rec.tk;
            const int hk = rec.un.y, nq = rec.un.w;
            const int R = G * nq;
            float* rm = row_m + (task_it & 1) * 32;   // this task's running maxima
            if (k == k_begin) convert_q(task_it, R);   // later tasks: converted early
            const int ctx_b = rec.ctx;
            const int tok_base = rec.cuq + rec.un.z;
            const int pbase = ctx_b - rec.ql + rec.un.z;
            const int n = tk.z - tk.y, n2 = (n + 1) / 2;
            const int first = window_first_tile(L.window, pbase, kDecodeTile);

            // m starts at -1e30 (not -inf): 2^(y - m) stays 0 for y = -inf, and
            // any finite y exceeds m + 8, so the first stage sets the maxima
            float c[HR], m[HR], m8[HR], l[HR];
#pragma unroll
            for (int r = 0; r < HR; ++r) {
                c[r] = row_c[rb + r];
                m[r] = kNoMax;
                m8[r] = kNoMax;
                l[r] = 0.f;
            }

            for (int i = 0; i < n2; ++i, ++g) {
                const int s = g % S, b = g & 1;
                const int kt0 = tk.y + 2 * i + first;          // first KV tile of the stage
                const int tok = kt0 * kDecodeTile + t;
                const bool valid = (t < kDecodeTile || tk.y + 2 * i + 1 < tk.z) && tok < ctx_b;
                // row r = G * (query token) + head sees this key iff its
                // position p = pbase + r / G has tok <= p and, with a sliding
                // window ("HiLS-Attention", 二.1 local branch), tok > p - window:
                // the rows [r_lo, r_hi), here relative to this warpgroup's first
                const int d0 = tok - pbase;
                int r_lo = (d0 > 0 ? d0 * G : 0) - rb, r_hi = R - rb;
                if (L.window > 0) {
                    const int64_t h = (int64_t)(d0 + L.window) * G;
                    r_hi = (h < R ? (int)(h > 0 ? h : 0) : R) - rb;
                }
                if (!valid) r_lo = r_hi;
                // ---- pass 1: y for every row.  The stage's own barrier is
                // waited too (it completed before its QK was issued): it orders
                // the producer's scale stores before these reads.
                wait(&s_full[b], (uint32_t)((g >> 1) & 1));
                wait(&full[s], (uint32_t)((g / S) & 1));
                tc_fence_after();
                const int box = (t >> 6) * 4 + ((t & 63) >> rpb_log);
                const float ks = scales[(s * 2 + 0) * 8 + box];
                const float vs = scales[(s * 2 + 1) * 8 + box];
                const float lvs = valid ? lg2(vs) : 0.f;
                const float ivs = valid ? 1.f / vs : 0.f;
                float y[HR];
                bool need = false;
                {
                    float a1[HR], a2[HR], a3[HR];
                    const uint32_t tS = tmem + lane_off + b * Cfg::kColS + rb;
                    tmem_ld_rows<HR>(tS, a1);
                    tmem_ld_rows<HR>(tS + NR, a2);
                    tmem_ld_rows<HR>(tS + 2 * NR, a3);
                    tmem_wait_ld();
                    reg_fence_rows<HR>(a1);
                    reg_fence_rows<HR>(a2);
                    reg_fence_rows<HR>(a3);
                    // y = (t1 + t2 + t3) * c * k_scale + log2(v_scale), two rows
                    // per packed f32x2 operation
                    const float2 ks2 = make_float2(ks, ks), lv2 = make_float2(lvs, lvs);
#pragma unroll
                    for (int r = 0; r < HR; r += 2) {
                        const float2 sum = __fadd2_rn(
                            __fadd2_rn(make_float2(a1[r], a1[r + 1]), make_float2(a2[r], a2[r + 1])),
                            make_float2(a3[r], a3[r + 1]));
                        const float2 yy = __ffma2_rn(
                            sum, __fmul2_rn(make_float2(c[r], c[r + 1]), ks2), lv2);
                        y[r] = yy.x;
                        y[r + 1] = yy.y;
                    }
                    // rows that do not see this key (the last stages of a sequence,
                    // a sliding window, tokens past the context)
                    if (r_lo > 0 || r_hi < HR) {
#pragma unroll
                        for (int r = 0; r < HR; ++r)
                            if (r < r_lo || r >= r_hi) y[r] = -INFINITY;
                    }
#pragma unroll
                    for (int r = 0; r < HR; ++r) need |= y[r] > m8[r];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[b]);
                // ---- the running max moves only when a score outgrows it by 2^8
                if (named_bar_or(bar_wg, 128, need)) {
                    float mx[HR];
#pragma unroll
                    for (int r = 0; r < HR; ++r) mx[r] = y[r];
                    const float wm = warp_reduce_rows<HR>(
                        mx, lane, [](float x, float z) { return fmaxf(x, z); });
                    if (lane < HR) redw[wq * 32 + lane] = wm;
                    named_bar_sync(bar_wg, 128);
                    if (t < HR) {
                        const float tm = fmaxf(fmaxf(redw[t], redw[32 + t]),
                                               fmaxf(redw[64 + t], redw[96 + t]));
                        rm[rb + t] = fmaxf(rm[rb + t], tm);
                    }
                    named_bar_sync(bar_wg, 128);
                    bool resc = false;
                    float alpha[HR];
#pragma unroll
                    for (int r = 0; r < HR; ++r) {
                        const float mn = rm[rb + r];
                        alpha[r] = m[r] == mn ? 1.f : ex2(m[r] - mn);
                        resc |= alpha[r] != 1.f;
                        l[r] *= alpha[r];
                        m[r] = mn;
                        m8[r] = mn + 8.f;
                    }
                    if (resc && i > 0) {
                        // O^T row t (head dim t), this warpgroup's columns, times
                        // alpha, once the previous stage's PV has landed
                        wait(&p_empty[(g - 1) & 1], (uint32_t)(((g - 1) >> 1) & 1));
                        tc_fence_after();
                        float o[HR];
                        const uint32_t tO = tmem + lane_off + Cfg::kColO + rb;
                        tmem_ld_rows<HR>(tO, o);
                        tmem_wait_ld();
                        reg_fence_rows<HR>(o);
#pragma unroll
                        for (int r = 0; r < HR; ++r) o[r] *= alpha[r];
                        tmem_st_rows<HR>(tO, o);
                        tmem_wait_st();
                    }
                }
                // ---- pass 2: P' = 2^(y - m) in f32 (l += P' / v_scale), then as
                // two E4M3 terms, P_hi = e4m3(P') and P_lo = e4m3(P' - P_hi)
                // (the difference taken in f16), into P^T buffer b
                wait(&p_empty[b], (uint32_t)((g >> 1) & 1) ^ 1u);
                uint8_t* p0 = smem + Cfg::kOffP + b * 2 * Cfg::kPTermBytes;
                uint8_t* p1 = p0 + Cfg::kPTermBytes;
                uint32_t hw[HR / 4], lw[HR / 4];
                const float2 iv2 = make_float2(ivs, ivs);
#pragma unroll
                for (int r = 0; r < HR; r += 2) {
                    const float2 pf = make_float2(ex2(y[r] - m[r]), ex2(y[r + 1] - m[r + 1]));
                    const uint32_t e2 = pack_f16x2_sat(pf.x, pf.y);
                    const float2 lsum = __ffma2_rn(pf, iv2, make_float2(l[r], l[r + 1]));
                    l[r] = lsum.x;
                    l[r + 1] = lsum.y;
                    const uint16_t hi = f16x2_to_e4m3x2(e2);
                    const uint16_t lo = f16x2_to_e4m3x2(hsub2_u32(e2, e4m3x2_to_f16x2(hi)));
                    if ((r & 2) == 0) {
                        hw[r / 4] = hi;
                        lw[r / 4] = lo;
                    } else {
                        hw[r / 4] |= (uint32_t)hi << 16;
                        lw[r / 4] |= (uint32_t)lo << 16;
                    }
                }
                if constexpr (Cfg::kPMN) {
                    // MN-major P^T: token t's 32 row bytes, this warpgroup's 16 of
                    // them as one 16-byte chunk (32-byte swizzle: chunk ^ bit 2 of t)
                    const uint32_t off = (uint32_t)(t * 32 + ((wg ^ ((t >> 2) & 1)) << 4));
                    *reinterpret_cast<uint4*>(p0 + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4*>(p1 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                } else {
                    // K-major P^T: row r's 128 token bytes
#pragma unroll
                    for (int r = 0; r < HR; ++r) {
                        if (rb + r >= R) break;
                        p0[swz_byte(rb + r, t)] = (uint8_t)(hw[r / 4] >> (8 * (r & 3)));
                        p1[swz_byte(rb + r, t)] = (uint8_t)(lw[r / 4] >> (8 * (r & 3)));
                    }
                }
                // V rows of tokens past the context or of the stage's unloaded
                // tile: P' is 0 there, but stale bytes may hold E4M3 NaN codes
                if (!valid && wg == 0) {
                    uint4* vrow = reinterpret_cast<uint4*>(smem + s * Cfg::kStageBytes +
                                                           Cfg::kKBytes + t * 128);
#pragma unroll
                    for (int q = 0; q < 8; ++q) vrow[q] = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[b]);
            }

            // ---- the next task's Q terms now: its first QK overlaps this epilogue
            if (k + 1 < k_end) {
                if (((k + 1 - k_begin) & 31) == 0) {
                    mine = fetch_task_rec<false>(P, k + 1 + lane, k_end, lane, err_hdr);
                    fetched = true;
                }
                const TaskRec nrec = shfl_task_rec(mine, (k + 1 - k_begin) & 31);
                convert_q(task_it + 1, G * nrec.un.w);
            }

            // ---- epilogue: l summed over the 128 tokens (warp sums), raw O^T of
            // this warpgroup's rows into the f32 staging rows, one barrier, then
            // thread t finishes row rb + t / 8, head dims [16 (t % 8), +16):
            // O / l (bf16, or the f32 split partial) and the LSE
            {
                const float wl = warp_reduce_rows<HR>(l, lane,
                                                      [](float x, float z) { return x + z; });
                if (lane < HR) redw[wq * 32 + lane] = wl;
                float* epi = reinterpret_cast<float*>(smem + Cfg::kOffEpi);   // [NR][D]
                float o[HR];
                if (n2 > 0) {
                    wait(o_full, (uint32_t)(o_tasks & 1));
                    ++o_tasks;
                    tc_fence_after();
                    tmem_ld_rows<HR>(tmem + lane_off + Cfg::kColO + rb, o);
                    tmem_wait_ld();
                    reg_fence_rows<HR>(o);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(o_free);     // O^T may be overwritten
                } else {
#pragma unroll
                    for (int r = 0; r < HR; ++r) o[r] = 0.f;
                }
#pragma unroll
                for (int r = 0; r < HR; ++r) epi[(rb + r) * D + t] = o[r];
                named_bar_sync(bar_wg, 128);
                const int rr = t >> 3, r = rb + rr, c16 = (t & 7) * 16;
                if (rr < HR && r < R) {
                    const float ls = (redw[rr] + redw[32 + rr]) + (redw[64 + rr] + redw[96 + rr]);
                    const float inv = ls > 0.f ? 1.f / ls : 0.f;
                    const int rt = r / G;
                    const int token = tok_base + rt, head = hk * G + (r - rt * G);
                    if ((t & 7) == 0) {
                        const float lse_nat = ls > 0.f ? (rm[r] + lg2(ls)) * kLn2 : -INFINITY;
                        if (tk.w < 0) {
                            if (P.lse != nullptr) P.lse[(int64_t)token * Hq + head] = lse_nat;
                        } else {
                            P.part_lse[(int64_t)tk.w * L.rows_cap + r] = lse_nat;
                        }
                    }
                    const float4* src = reinterpret_cast<const float4*>(epi + r * D + c16);
                    float4 v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        v[q] = src[q];
                        v[q].x *= inv;
                        v[q].y *= inv;
                        v[q].z *= inv;
                        v[q].w *= inv;
                    }
                    if (tk.w < 0) {
                        uint4* dst = reinterpret_cast<uint4*>(
                            P.out + ((int64_t)token * Hq + head) * D + c16);
                        dst[0] = make_uint4(pack_bf16x2(v[0].x, v[0].y), pack_bf16x2(v[0].z, v[0].w),
                                            pack_bf16x2(v[1].x, v[1].y), pack_bf16x2(v[1].z, v[1].w));
                        dst[1] = make_uint4(pack_bf16x2(v[2].x, v[2].y), pack_bf16x2(v[2].z, v[2].w),
                                            pack_bf16x2(v[3].x, v[3].y), pack_bf16x2(v[3].z, v[3].w));
                    } else {
                        float4* dst = reinterpret_cast<float4*>(
                            P.part_o + ((int64_t)tk.w * L.rows_cap + r) * D + c16);
#pragma unroll
                        for (int q = 0; q < 4; ++q) dst[q] = v[q];
                    }
                }
            }
            if (threadIdx.x == 0) trace_task_end(P.trace, P.trace_cap, k);
        }
    }

    grid_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp >= 10) decode_drain<Cfg>(full, q_full, armed, abort_flag, warp - 10, lane);
    __syncthreads();
    if (warp == 8) tmem_dealloc(tmem, Cfg::kTmemCols);
}

namespace {
template <int NR>
cudaError_t launch_tc_variant(const DecodeParams& P, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t stream) {
    using Cfg = DecodeTcCfg<NR>;
    auto kern = decode_fp8_tc_kernel<NR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = launch_dependent(kern, dim3(P.L.N), dim3(Cfg::kThreads), Cfg::kSmemBytes, stream, P, tq,
                         tk, tv);
    return e != cudaSuccess ? e : cudaGetLastError();
}
}  // namespace

// The tensor-core E4M3 decode for units of `rows` query rows (at most 32):
// its shared memory, threads and entry point, and its launch.
int decode_fp8_tc_smem_bytes(int rows) {
    return rows <= 16 ? DecodeTcCfg<16>::kSmemBytes
                      : rows <= 32 ? DecodeTcCfg<32>::kSmemBytes : -1;
}
int decode_fp8_tc_threads(int rows) { return rows <= 32 ? 384 : -1; }
const void* decode_fp8_tc_kernel_ptr(int rows) {
    return rows <= 16 ? (const void*)decode_fp8_tc_kernel<16>
                      : rows <= 32 ? (const void*)decode_fp8_tc_kernel<32> : nullptr;
}
cudaError_t launch_decode_fp8_tc(const DecodeParams& P, int rows, const CUtensorMap& tq,
                                 const CUtensorMap& tk, const CUtensorMap& tv,
                                 cudaStream_t stream) {
    if (rows <= 16) return launch_tc_variant<16>(P, tq, tk, tv, stream);
    if (rows <= 32) return launch_tc_variant<32>(P, tq, tk, tv, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
