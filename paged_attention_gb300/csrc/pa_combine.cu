// pa_combine.cu -- the Combine pass of split-K attention.
//
// "基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 (Combine: re-weight each
// chunk's local output by its LSE into a result equal to full attention) and
// 三.3 (the softmax-aware merge: m = max of the parts, weights exp(m_k - m)).
// Partials hold normalised O_k and LSE_k (natural log), so
//   O = sum_k e^(lse_k - m) O_k / sum_k e^(lse_k - m),  lse = m + ln sum_k e^(lse_k - m).
// Also writes O = 0, lse = -inf for units that received no task (no visible key).
//
// Grid-stride over (unit, chunk of ROWS rows) items of the units Assign listed
// as needing a combine, so that a 256-row prefill unit spreads over many CTAs;
// each thread owns 4 consecutive elements of D of one row (coalesced fp32
// reads).  The partials are merged online, four at a time, with every load of
// a group issued before any use (no LSE-then-O dependent round trip).
#include "pa_internal.cuh"

namespace pa {

namespace {

constexpr int kCombineThreads = 128;

template <int D>
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(WsLayout L, const void* __restrict__ ws, const float* __restrict__ part_o,
               const float* __restrict__ part_lse, __nv_bfloat16* __restrict__ out,
               float* __restrict__ lse) {
    constexpr int TPR = D / 4;                    // threads per row
    constexpr int ROWS = kCombineThreads / TPR;   // rows per item
    const int32_t* header = ws_ptr<int32_t>(ws, L.off_header);
    const int4* units = ws_ptr<int4>(ws, L.off_units);
    const int32_t* nsplit = ws_ptr<int32_t>(ws, L.off_nsplit);
    const int32_t* slot0 = ws_ptr<int32_t>(ws, L.off_slot0);
    const int32_t* fix = ws_ptr<int32_t>(ws, L.off_fix);
    const int32_t* cu_q = ws_ptr<int32_t>(ws, L.off_cu_q);
    grid_dependency_wait();   // the compute pass's partials are complete
    const int nfix = header[H_FIX];
    const int chunks = (L.rows_cap + ROWS - 1) / ROWS;   // items per unit
    const int sub = threadIdx.x / TPR, d = (threadIdx.x % TPR) * 4;
    for (int64_t i = blockIdx.x; i < (int64_t)nfix * chunks; i += gridDim.x) {
        const int f = (int)(i / chunks), c = (int)(i % chunks);
        const int u = fix[f];
        const int4 un = units[u];
        const int R = L.G * un.w;
        const int r = c * ROWS + sub;
        if (r >= R) continue;
        const int S = nsplit[u], s0 = slot0[u];
        const int token = cu_q[un.x] + un.z + r / L.G, head = un.y * L.G + r % L.G;
        float m = -INFINITY, den = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k0 = 0; k0 < S; k0 += 4) {
            float lk[4];
            float4 ok[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                lk[j] = -INFINITY;
                ok[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (k0 + j < S) {
                    const int64_t row = (int64_t)(s0 + k0 + j) * L.rows_cap + r;
                    lk[j] = part_lse[row];
                    ok[j] = *reinterpret_cast<const float4*>(part_o + row * D + d);
                }
            }
            const float mn = fmaxf(m, fmaxf(fmaxf(lk[0], lk[1]), fmaxf(lk[2], lk[3])));
            if (mn == -INFINITY) continue;
            const float sc = m == -INFINITY ? 0.f : ex2((m - mn) * kLog2e);
            den *= sc;
            acc.x *= sc;
            acc.y *= sc;
            acc.z *= sc;
            acc.w *= sc;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (lk[j] == -INFINITY) continue;
                const float w = ex2((lk[j] - mn) * kLog2e);
                den += w;
                acc.x += w * ok[j].x;
                acc.y += w * ok[j].y;
                acc.z += w * ok[j].z;
                acc.w += w * ok[j].w;
            }
            m = mn;
        }
        if (m != -INFINITY) {
            const float inv = 1.f / den;
            acc.x *= inv;
            acc.y *= inv;
            acc.z *= inv;
            acc.w *= inv;
        }
        uint2 packed;
        packed.x = pack_bf16x2(acc.x, acc.y);
        packed.y = pack_bf16x2(acc.z, acc.w);
        *reinterpret_cast<uint2*>(out + ((int64_t)token * L.Hq + head) * D + d) = packed;
        if (lse != nullptr && d == 0)
            lse[(int64_t)token * L.Hq + head] = m == -INFINITY ? -INFINITY : m + lg2(den) * kLn2;
    }
}

}  // namespace

cudaError_t launch_combine(const WsLayout& L, const void* ws, const void* partial, void* out,
                           float* lse, int grid, cudaStream_t stream) {
    const float* po = reinterpret_cast<const float*>(partial);
    const float* pl = po + L.partial_slots * L.rows_cap * L.D;
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
    cudaError_t e;
    if (L.D == 128)
        e = launch_dependent(combine_kernel<128>, dim3(grid), dim3(kCombineThreads), 0, stream, L,
                             ws, po, pl, o, lse);
    else if (L.D == 64)
        e = launch_dependent(combine_kernel<64>, dim3(grid), dim3(kCombineThreads), 0, stream, L,
                             ws, po, pl, o, lse);
    else
        return cudaErrorInvalidValue;
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pa
