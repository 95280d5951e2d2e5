// pa_combine.cu -- the Combine pass of split-K attention.
//
// "基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 (Combine: re-weight each
// chunk's local output by its LSE into a result equal to full attention) and
// 三.3 (the softmax-aware merge: m = max of the parts, weights exp(m_k - m)).
// Partials hold normalised O_k and LSE_k (natural log), so
//   O = sum_k e^(lse_k - m) O_k / sum_k e^(lse_k - m),  lse = m + ln sum_k e^(lse_k - m).
// Also writes O = 0, lse = -inf for units that received no task (no visible key).
//
// Persistent grid over the units Assign listed as needing a combine; each
// thread owns 4 consecutive elements of D of one row (coalesced fp32 reads).
#include "pa_internal.cuh"

namespace pa {

namespace {

template <int D>
__global__ void __launch_bounds__(128) combine_kernel(WsLayout L, const void* __restrict__ ws,
                                                      const float* __restrict__ part_o,
                                                      const float* __restrict__ part_lse,
                                                      __nv_bfloat16* __restrict__ out,
                                                      float* __restrict__ lse) {
    constexpr int TPR = D / 4;            // threads per row
    constexpr int ROWS = 128 / TPR;       // rows in flight per CTA
    const int32_t* header = ws_ptr<int32_t>(ws, L.off_header);
    const int4* units = ws_ptr<int4>(ws, L.off_units);
    const int32_t* nsplit = ws_ptr<int32_t>(ws, L.off_nsplit);
    const int32_t* slot0 = ws_ptr<int32_t>(ws, L.off_slot0);
    const int32_t* fix = ws_ptr<int32_t>(ws, L.off_fix);
    const int32_t* cu_q = ws_ptr<int32_t>(ws, L.off_cu_q);
    grid_dependency_wait();   // the compute pass's partials are complete
    const int nfix = header[H_FIX];
    const int sub = threadIdx.x / TPR, d = (threadIdx.x % TPR) * 4;
    for (int f = blockIdx.x; f < nfix; f += gridDim.x) {
        const int u = fix[f];
        const int4 un = units[u];
        const int S = nsplit[u], s0 = slot0[u];
        const int R = L.G * un.w;
        const int tok0 = cu_q[un.x] + un.z;
        for (int r = sub; r < R; r += ROWS) {
            const int token = tok0 + r / L.G, head = un.y * L.G + r % L.G;
            float m = -INFINITY;
            for (int k = 0; k < S; ++k)
                m = fmaxf(m, part_lse[(int64_t)(s0 + k) * L.rows_cap + r]);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            float den = 0.f;
            if (m != -INFINITY) {
                for (int k = 0; k < S; ++k) {
                    const int64_t row = (int64_t)(s0 + k) * L.rows_cap + r;
                    const float lk = part_lse[row];
                    if (lk == -INFINITY) continue;
                    const float w = ex2((lk - m) * kLog2e);
                    const float4 o = *reinterpret_cast<const float4*>(part_o + row * D + d);
                    den += w;
                    acc.x += w * o.x;
                    acc.y += w * o.y;
                    acc.z += w * o.z;
                    acc.w += w * o.w;
                }
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
                lse[(int64_t)token * L.Hq + head] =
                    m == -INFINITY ? -INFINITY : m + lg2(den) * kLn2;
        }
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
        e = launch_dependent(combine_kernel<128>, dim3(grid), dim3(128), 0, stream, L, ws, po, pl,
                             o, lse);
    else if (L.D == 64)
        e = launch_dependent(combine_kernel<64>, dim3(grid), dim3(128), 0, stream, L, ws, po, pl,
                             o, lse);
    else
        return cudaErrorInvalidValue;
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pa
