// pa_internal.cuh -- shared definitions of the CUDA library (not part of the ABI).
//
// Workspace layout of the Assign pass, launch-parameter structs and thin
// inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// ldmatrix, mma.sync, tcgen05 and fast exp2/log2.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "pa.h"

namespace pa {

// ------------------------------------------------------------ constants

constexpr int kDecodeTile = 64;      // KV tokens per decode tile
constexpr int kPrefillTile = 128;    // KV tokens per prefill tile (= mask tile)
constexpr int kPrefillHalfRows = 128;  // rows of one tcgen05 M=128 tile
constexpr int kPrefillRows = 256;    // rows (query token x head) per prefill unit (2 halves)
constexpr int kMaskTile = 128;       // block-mask tile edge
constexpr int kDefaultBalanceRows = 128;
// A prefill-mode batch without a block mask sends every sequence with
// 1 <= G * q_len <= kMixedDecodeRows (decode steps, short speculative runs)
// to the decode kernel, through a second, decode-mode task map.
constexpr int kMixedDecodeRows = 16;
constexpr int kHeaderWords = 64;
// Completion counters per unit in the Assign workspace: one per 16-row tile
// of a decode unit (the bf16 decode kernel finalizes split units per row
// tile).
constexpr int kDoneWords = 4;

// header word indices inside the Assign workspace
enum HeaderWord {
    H_UNITS = 0,
    H_TASKS = 1,
    H_SLOTS = 2,
    H_CTAS = 3,
    H_ERROR = 4,
    H_FIX = 5,
    H_MODE = 6,
};

// First KV tile (of `tile` tokens) any row of a unit can see under a sliding
// window: its first query sits at position p0 and sees keys > p0 - window.
__host__ __device__ inline int window_first_tile(int window, int p0, int tile) {
    if (window <= 0) return 0;
    const int lo = p0 - window + 1;
    return lo > 0 ? lo / tile : 0;
}

// Byte offsets of every array inside the Assign workspace.  Computed on the
// host from the problem (layout_for) and passed to every kernel by value.
struct WsLayout {
    int32_t mode;
    int32_t B, Hq, Hkv, G, D;
    int32_t N;            // persistent CTAs
    int32_t kv_tile;      // 64 decode / 128 prefill
    int32_t qtok;         // query tokens per unit (prefill: 256/G, or 128 for G=1 with a
                          // mask; decode: all)
    int32_t unit_cap;
    int32_t task_cap;
    int32_t max_kv_tiles; // row stride of the active-tile lists
    int32_t has_mask;
    int32_t rows_cap;     // partial rows per slot
    int32_t balance_rows;
    int32_t unit_cost;        // Assign's fixed cost of a unit with tiles (tile-weight units)
    int32_t total_q;
    int32_t max_q_len, max_ctx;
    int32_t mask_q_tiles, mask_kv_tiles;
    // which sequences this map covers: 0 all; 1 those with 1 <= q_len <=
    // small_q (the decode map of a mixed batch); 2 those with q_len > small_q
    // (its prefill map).  The other sequences get no units, or (decode mode)
    // units without query rows.
    int32_t cls, small_q;
    int32_t window;   // sliding window (0 = none): the query at p sees keys p - window < j <= p
    int64_t off_err_header;   // header whose error word device faults go to
    int64_t off_header, off_cta_ptr, off_tasks, off_task_cta, off_units, off_ntiles,
        off_prefix, off_nsplit, off_slot0, off_done, off_fix, off_active, off_cu_q,
        off_seq_unit0;   // off_done: completion counters, kDoneWords per unit
    int64_t total_bytes;
    int64_t partial_slots;
    int64_t partial_bytes;
};

// fills `L` for (problem, mode, N); returns false on invalid dims
bool layout_for(const pa_problem& p, int mode, int N, int rows_cap, WsLayout& L);

// Bounded-wait limit of a normal launch.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// The wait-timeout test hook (pa_test_inject_wait_timeout): returns the ring
// entry CTA 0's producer should leave unfilled (-1: none) and the wait limit
// for the next compute launch, and disarms the hook.
void take_test_hook(int32_t* skip_entry, uint64_t* wait_limit_ns);
// The task trace set by pa_set_task_trace (nullptr, 0 when none).
void take_task_trace(int64_t** trace, int64_t* capacity);

template <typename T>
__host__ __device__ inline T* ws_ptr(void* ws, int64_t off) {
    return reinterpret_cast<T*>(reinterpret_cast<char*>(ws) + off);
}
template <typename T>
__host__ __device__ inline const T* ws_ptr(const void* ws, int64_t off) {
    return reinterpret_cast<const T*>(reinterpret_cast<const char*>(ws) + off);
}

// ------------------------------------------------------- device helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void set_device_error(int32_t* header, int code) {
    atomicOr(header + H_ERROR, code);
}

// Programmatic dependent launch.  A kernel launched with
// launch_dependent() may start while the previous kernel on the stream is
// still running; grid_dependency_wait() blocks until that kernel has finished
// and its memory is visible (a no-op for an ordinary launch).
// grid_launch_dependents() lets the next such kernel start early.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kernel` so that it may overlap the tail of the kernel before it on
// `stream` (it must call grid_dependency_wait() before reading that kernel's
// output).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launch `kernel` in thread-block clusters of `cluster` CTAs along x (the
// grid must be a multiple of it).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_in_clusters(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t stream, int cluster, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Largest grid of clusters of `cluster` CTAs that are co-resident on the
// current device for this kernel (0 if none).
inline int max_cluster_grid(const void* kernel, int threads, int smem, int cluster) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cluster);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return 0;
    return n * cluster;
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// mbarrier ----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: spins until the phase with `parity` completes or `limit_ns`
// elapses.  Returns false on timeout (the caller records the error and
// carries on without the data, so no wait can hang the GPU).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && globaltimer() - t0 > limit_ns) return false;
    }
}
// The same, but it also gives up as soon as the CTA's abort flag is raised
// (another warp's wait ran out): the CTA then winds down without waiting for
// data that will not come.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity,
                                                   uint64_t limit_ns, const volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && (*abort || globaltimer() - t0 > limit_ns)) return false;
    }
}

// Limit of each wait while a CTA that gave up drains its own copies in
// flight (a tensor copy lands within microseconds; this only bounds the
// wait should one never land).
constexpr uint64_t kDrainLimitNs = 100000000ull;

// Thread-block clusters and distributed shared memory ------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster (a CTA-wide barrier across the cluster).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of `addr` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void fence_acq_rel_cluster() {
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
}
// Arrive, with release at cluster scope, on an mbarrier of (possibly) another CTA.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     cluster_addr)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait with acquire at cluster scope (the phase was completed by
// arrivals of other CTAs of the cluster); gives up on the CTA's abort flag.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns, const volatile int* abort) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 255u) == 0 && (*abort || globaltimer() - t0 > limit_ns)) return false;
    }
}
__device__ __forceinline__ float ld_dsm_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_dsm_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ float2 ld_dsm_f32x2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                 : "=f"(v.x), "=f"(v.y)
                 : "r"(addr)
                 : "memory");
    return v;
}

// TMA ----------------------------------------------------------------------
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3), "r"(c4)
        : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Named barriers (ids 1..15; id 0 is __syncthreads) -------------------------
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// Named barrier that also returns whether `pred` held in any of its threads.
__device__ __forceinline__ bool named_bar_or(int id, int threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %3, 0;\n\t"
        "bar.red.or.pred q, %1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(threads), "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void named_bar_arrive(int id, int threads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ldmatrix / mma.sync -------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One 32-byte global store of eight 32-bit words (sm_100 and later); the
// address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Hardware base-2 exponential / logarithm (MUFU), flushing denormals.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Two base-2 exponentials in one MUFU operation: f16 inputs and results.
__device__ __forceinline__ uint32_t ex2_h2(float lo, float hi) {
    uint32_t x, y;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(x) : "f"(hi), "f"(lo));
    asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// acc.x += low f16 of h2, acc.y += high f16 (mixed-precision add, exact
// conversion, one instruction each)
__device__ __forceinline__ void add_f16x2_to_f32(float2& acc, uint32_t h2) {
    asm("{\n\t.reg .f16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.f16 %0, lo, %0;\n\t"
        "add.rn.f32.f16 %1, hi, %1;\n\t}"
        : "+f"(acc.x), "+f"(acc.y)
        : "r"(h2));
}
// max(a, b, c) in one instruction (three-input max.f32 of sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// D = A(16x16 f16, row) * B(16x8 f16, col) + D, fp32 accumulate
__device__ __forceinline__ void mma_f16_16816(float* d, const uint32_t* a, uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit values spread over the warp in the
// mma fragment layout (lane l holds row l/4, columns 2(l%4), 2(l%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Two E4M3 bytes (low byte first) -> packed f16x2, exact (hardware).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
    return h2;
}

// Packed bf16x2 -> f16x2, rounded to nearest; values beyond the f16 range
// saturate to +-65504.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
    uint32_t d;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// f32 pair -> packed f16x2, rounded to nearest; beyond the f16 range the
// values saturate to +-65504 instead of becoming infinite.
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Bytes J and J+1 of two words, interleaved: {a.J, b.J, a.J+1, b.J+1} from
// the lowest byte up (two 16-bit pairs, each holding one byte of a and one of b).
template <int J>
__device__ __forceinline__ uint32_t interleave_bytes(uint32_t a, uint32_t b) {
    constexpr uint32_t sel = (uint32_t)(5 + J) << 12 | (uint32_t)(J + 1) << 8 |
                             (uint32_t)(4 + J) << 4 | (uint32_t)J;
    return prmt(a, b, sel);
}

}  // namespace pa

// ------------------------------------------------------------- tcgen05 / TMEM
namespace pa {

// Shared-memory matrix descriptor for tcgen05.mma (128-byte swizzle).
//   bits [0,14) start >> 4, [16,30) leading byte offset >> 4,
//   [32,46) stride byte offset >> 4, [46,48) version = 1,
//   [61,64) layout = 2 (128-byte swizzle).
// K-major operand: rows of 128 B (64 bf16 along K), 8-row atoms 1024 B apart
// (SBO = 1024); LBO unused.  MN-major operand: 128 B along M/N per K row,
// 8 K rows per atom (SBO = 1024 between K groups), LBO = byte distance between
// 64-element M/N blocks.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// The same with the 32-byte swizzle (layout type 6): 32-byte rows, 8-row
// atoms of 256 bytes.  An MN-major operand 32 bytes wide along M/N takes
// SBO = 256 between its 8-row K groups.
__device__ __forceinline__ uint64_t smem_desc_sw32(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (6ull << 61);
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, dense.
//   [4,6) D fmt = 1 (f32), [7,10) A fmt = 1 (bf16), [10,13) B fmt = 1 (bf16),
//   bit 15 A MN-major, bit 16 B MN-major, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Per-warpgroup register budget (all 4 warps of a warpgroup execute it).
template <int N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(smem_slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]  (A: 128 lanes = rows, 2 bf16 per 32-bit column)
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Instruction descriptor, kind::f16: f16 A and B (format 0), fp32 D, dense.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Instruction descriptor, kind::f8f6f4: E4M3 A and B (format 0), fp32 D;
// otherwise laid out as for kind::f16.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D[tmem] (+)= A[smem] * B[smem], 8-bit operands (K = 32 per instruction)
__device__ __forceinline__ void tc_mma_ss_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], 8-bit operands (A: 128 lanes = rows, 4 per 32-bit column)
__device__ __forceinline__ void tc_mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Two f16 values (packed) -> two E4M3 bytes, round to nearest, saturating to +-448.
__device__ __forceinline__ uint16_t f16x2_to_e4m3x2(uint32_t h2) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(d) : "r"(h2));
    return d;
}
// Task trace (diagnostics, pa_set_task_trace): task k of the map is recorded
// as trace[3k] = the time its CTA starts it, trace[3k + 1] = the time it is
// done (%globaltimer, ns), trace[3k + 2] = the CTA.  One thread per CTA calls
// these; nothing is written without a trace buffer.
__device__ __forceinline__ void trace_task_start(int64_t* trace, int64_t cap, int k) {
    if (trace != nullptr && k < cap) {
        trace[3 * (int64_t)k] = (int64_t)globaltimer();
        trace[3 * (int64_t)k + 2] = (int64_t)blockIdx.x;
    }
}
__device__ __forceinline__ void trace_task_end(int64_t* trace, int64_t cap, int k) {
    if (trace != nullptr && k < cap) trace[3 * (int64_t)k + 1] = (int64_t)globaltimer();
}

// Two f32 values -> two E4M3 bytes (lo in the low byte), round to nearest,
// saturating to +-448.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// arrive (once) on an mbarrier when all previously issued MMAs of this thread complete
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// After tcgen05.wait::ld: tie 32 loaded registers to this point.  The load's
// destination registers are written asynchronously; without this the compiler
// may read them before the wait (it sees them defined by the load asm).
__device__ __forceinline__ void reg_fence32(float* v) {
    asm volatile(""
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                   "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                   "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]),
                   "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]),
                   "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]),
                   "+f"(v[30]), "+f"(v[31]));
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit: thread t of the warp gets lane (base + t),
// columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// 32 lanes x 16 columns of 32-bit (see tmem_ld32).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void reg_fence16(float* v) {
    asm volatile(""
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                   "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                   "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
    const uint32_t* r = reinterpret_cast<const uint32_t*>(v);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

}  // namespace pa

// ------------------------------------------------------------ task records
namespace pa {

// One task of the map with its unit and the sequence lengths it needs.
struct TaskRec {
    int4 tk;   // {unit, t0, t1, slot}
    int4 un;   // {b, hk, q0, nq}
    int ctx, ql, cuq;
};

// Lane `lane` of a warp loads task k (if k < k_end): the three dependent
// loads run in parallel across the warp's lanes, once per 32 tasks.
__device__ __forceinline__ TaskRec load_task_rec(const int4* tasks, const int4* units,
                                                 const int32_t* ctx, const int32_t* ql,
                                                 const int32_t* cu_q, int k, int k_end) {
    TaskRec r;
    r.tk = make_int4(0, 0, 0, -1);
    r.un = make_int4(0, 0, 0, 0);
    r.ctx = r.ql = r.cuq = 0;
    if (k < k_end) {
        r.tk = tasks[k];
        r.un = units[r.tk.x];
        r.ctx = ctx[r.un.x];
        r.ql = ql[r.un.x];
        r.cuq = cu_q[r.un.x];
    }
    return r;
}

__device__ __forceinline__ TaskRec shfl_task_rec(const TaskRec& r, int src) {
    TaskRec o;
    o.tk.x = __shfl_sync(0xffffffffu, r.tk.x, src);
    o.tk.y = __shfl_sync(0xffffffffu, r.tk.y, src);
    o.tk.z = __shfl_sync(0xffffffffu, r.tk.z, src);
    o.tk.w = __shfl_sync(0xffffffffu, r.tk.w, src);
    o.un.x = __shfl_sync(0xffffffffu, r.un.x, src);
    o.un.y = __shfl_sync(0xffffffffu, r.un.y, src);
    o.un.z = __shfl_sync(0xffffffffu, r.un.z, src);
    o.un.w = __shfl_sync(0xffffffffu, r.un.w, src);
    o.ctx = __shfl_sync(0xffffffffu, r.ctx, src);
    o.ql = __shfl_sync(0xffffffffu, r.ql, src);
    o.cuq = __shfl_sync(0xffffffffu, r.cuq, src);
    return o;
}

}  // namespace pa
