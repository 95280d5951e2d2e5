// pa_prefill.cu -- persistent causal / block-sparse prefill on tcgen05 + TMEM.
//
// "基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 Prefill (tile
// scheduling by batch, head and query tile; pipelined TMA loads of Q/K/V into
// multi-stage shared memory; QK, causal mask, fp32 online softmax, PV;
// epilogue normalisation), 二.1 (only the KV tiles of the active-tile list
// are loaded and multiplied), 二.2 (warp specialisation: a producer resolves
// page ids and issues K then V by TMA while compute runs; K/V buffers are
// released as soon as the MMAs that read them complete).  "vLLM Triton
// Attention Backend Deep Dive": Q blocks pack the G q heads of one KV head
// into one MMA tile; the persistent grid is fixed at the SM count.
//
// GB300 design (one CTA per SM, 192 threads):
//   warp 0      TMA producer: Q tile (128 rows = 128/G tokens x G heads,
//               128-byte swizzled) once per task, then K and V of every
//               active 128-token tile page by page into a 2-stage ring.
//   warp 1      allocates 512 TMEM columns; lane 0 issues every tcgen05.mma:
//               S[buf] = Q K^T (M=128, N=128, K=D, both operands K-major in
//               shared memory) into one of two TMEM S buffers, then
//               O += P V (M=128, N=D, K=128; P K-major, V MN-major: no
//               transpose of V is ever made).  Completion is signalled with
//               tcgen05.commit on mbarriers.  The warp also zeroes V rows past
//               the context before they are multiplied.
//   warps 2-5   softmax warpgroup: thread = query row = TMEM lane.  Reads its
//               S row (tcgen05.ld), applies the causal / context mask, keeps
//               the running max lazily (O is rescaled in TMEM only when the
//               max grows by more than 2^8), writes P (bf16) into shared
//               memory for the PV MMA, and finally normalises O and writes
//               the output row (or the split partial) and its LSE.
// While the softmax works on tile j, the tensor cores already compute
// S_{j+1} into the other TMEM buffer.
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
    float sm_scale;
    uint64_t wait_limit_ns;
};

template <int D>
struct PrefillCfg {
    static constexpr int kHalves = D / 64;           // 128-byte column blocks of a row
    static constexpr int kRegion = 128 * 128;        // 128 rows x 128 bytes
    static constexpr int kQBytes = kHalves * kRegion;
    static constexpr int kPBytes = 2 * kRegion;      // 128 keys = 2 column blocks
    static constexpr int kKVBytes = kHalves * kRegion;
    static constexpr int kStages = 2;
    static constexpr int kStageBytes = 2 * kKVBytes;
    static constexpr int kOffQ = 0;
    static constexpr int kOffP = kOffQ + kQBytes;
    static constexpr int kOffStage = kOffP + kPBytes;
    static constexpr int kOffBar = kOffStage + kStages * kStageBytes;
    static constexpr int kSlack = 16384;             // guard space after the data
    static constexpr int kSmemBytes = kOffBar + 256 + kSlack + 1024;
    static constexpr int kThreads = 192;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr int kOCol = 256;                // S buffers at columns 0 and 128
};

enum PrefillBar {
    B_Q_FULL = 0,
    B_Q_EMPTY = 1,
    B_KV_FULL = 2,   // 2 stages
    B_KV_EMPTY = 4,  // 2 stages
    B_S_FULL = 6,    // 2 buffers
    B_S_FREE = 8,    // 2 buffers
    B_P_FULL = 10,
    B_O_DONE = 11,
    B_O_FREE = 12,
    B_MMA_DONE = 13,
    B_COUNT = 14
};

__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* header, uint64_t limit) {
    if (*abort_flag) return;
    if (!mbar_wait(bar, parity, limit)) {
        *abort_flag = 1;
        set_device_error(header, PA_DEV_WAIT_TIMEOUT);
    }
}

template <int D>
__global__ void __launch_bounds__(192, 1)
prefill_kernel(const __grid_constant__ PrefillParams P, const __grid_constant__ CUtensorMap tmq,
               const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    using Cfg = PrefillCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffBar + 128);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffBar + 132);
    const WsLayout& L = P.L;
    int32_t* header = ws_ptr<int32_t>(P.ws, L.off_header);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t lim = P.wait_limit_ns;

    if (header[H_CTAS] != (int)gridDim.x) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(header, PA_DEV_BAD_LENGTHS);
        return;
    }
    if (threadIdx.x == 0) {
        mbar_init(&bar[B_Q_FULL], 1);
        mbar_init(&bar[B_Q_EMPTY], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar[B_KV_FULL + s], 1);
            mbar_init(&bar[B_KV_EMPTY + s], 1);
            mbar_init(&bar[B_S_FULL + s], 1);
            mbar_init(&bar[B_S_FREE + s], 128);
        }
        mbar_init(&bar[B_P_FULL], 128);
        mbar_init(&bar[B_O_DONE], 1);
        mbar_init(&bar[B_O_FREE], 128);
        mbar_init(&bar[B_MMA_DONE], 1);
        *abort_flag = 0;
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

    const int32_t* cta_ptr = ws_ptr<int32_t>(P.ws, L.off_cta_ptr);
    const int4* tasks = ws_ptr<int4>(P.ws, L.off_tasks);
    const int4* units = ws_ptr<int4>(P.ws, L.off_units);
    const int32_t* cu_q = ws_ptr<int32_t>(P.ws, L.off_cu_q);
    const int32_t* active = ws_ptr<int32_t>(P.ws, L.off_active);
    const int k_begin = cta_ptr[blockIdx.x], k_end = cta_ptr[blockIdx.x + 1];
    const int G = L.G, Hq = L.Hq;

    auto tile_of = [&](int u, int t) -> int {
        return L.has_mask ? active[(int64_t)u * L.max_kv_tiles + t] : t;
    };

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tmap(&tmq);
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
        }
        const int ps = P.page_size, rpb = P.rows_per_box, nbox = P.boxes_per_tile;
        const uint32_t box_bytes = (uint32_t)rpb * 128u * Cfg::kHalves;
        int kv_it = 0, task_it = 0;
        for (int k = k_begin; k < k_end; ++k, ++task_it) {
            const int4 tk = tasks[k];
            const int4 un = units[tk.x];
            const int b = un.x, hk = un.y, q0 = un.z;
            const int ctx_b = P.ctx[b];
            const int npg = (ctx_b + ps - 1) / ps;
            const int32_t* bt_row = P.block_table + (int64_t)b * P.max_pages_per_seq;
            wait_or_abort(&bar[B_Q_EMPTY], (uint32_t)(task_it & 1) ^ 1u, abort_flag, header, lim);
            if (lane == 0) {
                if (*abort_flag) {
                    mbar_arrive(&bar[B_Q_FULL]);
                } else {
                    mbar_arrive_expect_tx(&bar[B_Q_FULL], Cfg::kQBytes);
#pragma unroll
                    for (int h = 0; h < Cfg::kHalves; ++h)
                        tma_load_3d(smem + Cfg::kOffQ + h * Cfg::kRegion, &tmq, &bar[B_Q_FULL],
                                    64 * h, hk * G, cu_q[b] + q0);
                }
            }
            __syncwarp();
            int win_lo = -(1 << 30), win_val = -1;
            for (int t = tk.y; t < tk.z; ++t, ++kv_it) {
                const int st = kv_it & 1;
                wait_or_abort(&bar[B_KV_EMPTY + st], (uint32_t)((kv_it >> 1) & 1) ^ 1u, abort_flag,
                              header, lim);
                const int kt = tile_of(tk.x, t);
                uint8_t* sK = smem + Cfg::kOffStage + st * Cfg::kStageBytes;
                uint8_t* sV = sK + Cfg::kKVBytes;
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
                    if (*abort_flag) {
                        mbar_arrive(&bar[B_KV_FULL + st]);
                    } else {
                        mbar_arrive_expect_tx(&bar[B_KV_FULL + st], bytes);
                        // all K boxes first (QK needs them first), then V
#pragma unroll
                        for (int kv = 0; kv < 2; ++kv) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                if (pg[j] < 0) continue;
                                const int slot0 = (kt * kPrefillTile + j * rpb) % ps;
#pragma unroll
                                for (int h = 0; h < Cfg::kHalves; ++h)
                                    tma_load_4d((kv ? sV : sK) + h * Cfg::kRegion + j * rpb * 128,
                                                kv ? &tmv : &tmk, &bar[B_KV_FULL + st], 64 * h,
                                                slot0, hk, pg[j]);
                            }
                        }
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
        const uint32_t sQ = smem_u32(smem + Cfg::kOffQ);
        const uint32_t sP = smem_u32(smem + Cfg::kOffP);
        int kv_it = 0, s_it = 0, p_it = 0, task_it = 0;

        auto issue_pv = [&](int st, bool first) {
            wait_or_abort(&bar[B_P_FULL], (uint32_t)(p_it & 1), abort_flag, header, lim);
            ++p_it;
            if (first)
                wait_or_abort(&bar[B_O_FREE], (uint32_t)(task_it & 1) ^ 1u, abort_flag, header, lim);
            if (lane == 0) {
                tc_fence_after();
                const uint32_t sV =
                    smem_u32(smem + Cfg::kOffStage + st * Cfg::kStageBytes + Cfg::kKVBytes);
#pragma unroll
                for (int kk = 0; kk < kPrefillTile / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(
                        sP + (kk >> 2) * Cfg::kRegion + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(sV + kk * 16 * 128, Cfg::kRegion, 1024);
                    tc_mma_ss(tmem + Cfg::kOCol, a, bd, idesc_pv, (!first || kk > 0) ? 1u : 0u);
                }
                tc_commit(&bar[B_O_DONE]);
                tc_commit(&bar[B_KV_EMPTY + st]);
            }
            __syncwarp();
        };

        for (int k = k_begin; k < k_end; ++k, ++task_it) {
            const int4 tk = tasks[k];
            const int4 un = units[tk.x];
            const int ctx_b = P.ctx[un.x];
            const int n = tk.z - tk.y;
            wait_or_abort(&bar[B_Q_FULL], (uint32_t)(task_it & 1), abort_flag, header, lim);
            int prev_st = 0;
            for (int j = 0; j < n; ++j, ++kv_it, ++s_it) {
                const int st = kv_it & 1;
                const int kt = tile_of(tk.x, tk.y + j);
                wait_or_abort(&bar[B_KV_FULL + st], (uint32_t)((kv_it >> 1) & 1), abort_flag, header,
                              lim);
                uint8_t* sK = smem + Cfg::kOffStage + st * Cfg::kStageBytes;
                const int first_bad = ctx_b - kt * kPrefillTile;   // first key row past the context
                if (first_bad < kPrefillTile) {
                    uint8_t* sV = sK + Cfg::kKVBytes;
                    const int r0 = first_bad < 0 ? 0 : first_bad;
                    for (int idx = lane; idx < (kPrefillTile - r0) * Cfg::kHalves * 8; idx += 32) {
                        const int r = r0 + idx / (Cfg::kHalves * 8);
                        const int rem = idx % (Cfg::kHalves * 8);
                        *reinterpret_cast<uint4*>(sV + (rem >> 3) * Cfg::kRegion + swz128(r, rem & 7)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                const int sb = s_it & 1;
                wait_or_abort(&bar[B_S_FREE + sb], (uint32_t)((s_it >> 1) & 1) ^ 1u, abort_flag,
                              header, lim);
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t sKa = smem_u32(sK);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = (kk >> 2) * Cfg::kRegion + (kk & 3) * 32;
                        tc_mma_ss(tmem + sb * 128, smem_desc_sw128(sQ + koff, 16, 1024),
                                  smem_desc_sw128(sKa + koff, 16, 1024), idesc_qk,
                                  kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&bar[B_S_FULL + sb]);
                    if (j == n - 1) tc_commit(&bar[B_Q_EMPTY]);
                }
                __syncwarp();
                if (j > 0) issue_pv(prev_st, j - 1 == 0);
                prev_st = st;
            }
            if (n > 0) issue_pv(prev_st, n == 1);
        }
        if (lane == 0) {
            tc_commit(&bar[B_MMA_DONE]);
            mbar_wait(&bar[B_MMA_DONE], 0, lim);
        }
        __syncwarp();
    } else {
        // -------------------------------------------------- softmax warpgroup
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float scale_log2 = P.sm_scale * kLog2e;
        uint8_t* sPb = smem + Cfg::kOffP;
        int s_it = 0, o_it = 0, task_it = 0;
        for (int k = k_begin; k < k_end; ++k, ++task_it) {
            const int4 tk = tasks[k];
            const int4 un = units[tk.x];
            const int b = un.x, hk = un.y, q0 = un.z, nq = un.w;
            const int R = G * nq;
            const int ctx_b = P.ctx[b], ql_b = P.ql[b];
            const bool row_ok = row < R;
            const int p_row = ctx_b - ql_b + q0 + row / G;           // last key this row sees
            const int key_last = p_row < ctx_b - 1 ? p_row : ctx_b - 1;
            float m = -INFINITY, l = 0.f;
            const int n = tk.z - tk.y;
            for (int j = 0; j < n; ++j, ++s_it) {
                const int kt = tile_of(tk.x, tk.y + j);
                const int sb = s_it & 1;
                wait_or_abort(&bar[B_S_FULL + sb], (uint32_t)((s_it >> 1) & 1), abort_flag, header,
                              lim);
                tc_fence_after();
                float s[128];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(tmem + lane_off + sb * 128 + c4 * 32, s + c4 * 32);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bar[B_S_FREE + sb]);
                const int limc = row_ok ? key_last - kt * kPrefillTile : -1;   // valid: c <= limc
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    s[c] = c <= limc ? s[c] * scale_log2 : -INFINITY;
                    mx = fmaxf(mx, s[c]);
                }
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
                if (j > 0) {
                    wait_or_abort(&bar[B_O_DONE], (uint32_t)(o_it & 1), abort_flag, header, lim);
                    ++o_it;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, resc)) {
                    const float f = resc ? alpha : 1.f;
#pragma unroll
                    for (int c4 = 0; c4 < D / 32; ++c4) {
                        float o[32];
                        tmem_ld32(tmem + lane_off + Cfg::kOCol + c4 * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= f;
                        tmem_st32(tmem + lane_off + Cfg::kOCol + c4 * 32, o);
                    }
                    tmem_wait_st();
                }
                float sum = 0.f;
#pragma unroll
                for (int ch = 0; ch < 16; ++ch) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p0 = ex2(s[ch * 8 + 2 * e] - mu);
                        const float p1 = ex2(s[ch * 8 + 2 * e + 1] - mu);
                        sum += p0 + p1;
                        w[e] = pack_bf16x2(p0, p1);
                    }
                    *reinterpret_cast<uint4*>(sPb + (ch >> 3) * Cfg::kRegion + swz128(row, ch & 7)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
                l = l * alpha + sum;
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bar[B_P_FULL]);
            }
            // ---- epilogue: O / l -> output row (or split partial), LSE
            if (n > 0) {
                wait_or_abort(&bar[B_O_DONE], (uint32_t)(o_it & 1), abort_flag, header, lim);
                ++o_it;
            }
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const float lse_nat = l > 0.f ? (m + lg2(l)) * kLn2 : -INFINITY;
            const int token = cu_q[b] + q0 + row / G, head = hk * G + row % G;
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
                float o[32];
                tmem_ld32(tmem + lane_off + Cfg::kOCol + c4 * 32, o);
                tmem_wait_ld();
                if (row_ok) {
                    if (tk.w < 0) {
                        uint4* dst = reinterpret_cast<uint4*>(
                            P.out + ((int64_t)token * Hq + head) * D + c4 * 32);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            dst[q] = make_uint4(pack_bf16x2(o[8 * q] * inv, o[8 * q + 1] * inv),
                                                pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                                                pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                                                pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
                    } else {
                        float4* dst = reinterpret_cast<float4*>(
                            P.part_o + ((int64_t)tk.w * L.rows_cap + row) * D + c4 * 32);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[q] = make_float4(o[4 * q] * inv, o[4 * q + 1] * inv,
                                                 o[4 * q + 2] * inv, o[4 * q + 3] * inv);
                    }
                }
            }
            if (row_ok) {
                if (tk.w < 0) {
                    if (P.lse != nullptr) P.lse[(int64_t)token * Hq + head] = lse_nat;
                } else {
                    P.part_lse[(int64_t)tk.w * L.rows_cap + row] = lse_nat;
                }
            }
            tc_fence_before();
            mbar_arrive(&bar[B_O_FREE]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
}

int prefill_smem_bytes(int D, bool fp8) {
    if (fp8) return -1;
    if (D == 128) return PrefillCfg<128>::kSmemBytes;
    if (D == 64) return PrefillCfg<64>::kSmemBytes;
    return -1;
}

const void* prefill_kernel_ptr(int D, bool fp8) {
    if (fp8) return nullptr;
    if (D == 128) return (const void*)prefill_kernel<128>;
    if (D == 64) return (const void*)prefill_kernel<64>;
    return nullptr;
}

cudaError_t launch_prefill_from_api(const pa_problem& p, const WsLayout& L, const void* q,
                                    const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const int32_t* block_table,
                                    const int32_t* ctx, const int32_t* ql, const float* ks,
                                    const float* vs, void* ws, void* partial, void* out,
                                    float* lse, cudaStream_t stream) {
    (void)q;
    (void)ks;
    (void)vs;
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
    P.sm_scale = p.sm_scale;
    P.wait_limit_ns = 1000000000ull;
    const void* kern = prefill_kernel_ptr(p.head_dim, false);
    const int smem = prefill_smem_bytes(p.head_dim, false);
    if (!kern || smem <= 0) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (p.head_dim == 128)
        prefill_kernel<128><<<L.N, 192, smem, stream>>>(P, tq, tk, tv);
    else
        prefill_kernel<64><<<L.N, 192, smem, stream>>>(P, tq, tk, tv);
    return cudaGetLastError();
}

}  // namespace pa
