/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged-KV-cache attention forward.
 *
 * The operation ("基于Triton-TLE优化Tencent HPC-Ops Attention", 一.2 "Prefill
 * 与 Decode"): for every new query token of every sequence, softmax attention
 * over that sequence's cached keys and values, which live in fixed-size
 * physical pages reached through a per-sequence block table.  Decode runs as
 * three passes -- Assign (tile the KV, build a load-balanced task map),
 * Split-K compute (persistent CTAs write final or partial O and LSE),
 * Combine (LSE-rescale the partials into the exact softmax).  Prefill runs
 * causal or block-sparse attention over the same paged cache, and also takes
 * the mixed chunked-prefill + decode batch (xdnf.cn "Chunked Prefill" hybrid
 * batch article).  The arguments follow the pages' statement of the problem:
 * Q [tokens, Hq, D]; K/V caches [pages, page_size, Hkv, D] (NHD) or
 * [pages, Hkv, page_size, D] (HND) ("基于Triton-TLE…", 三.2: both layouts read
 * through one projected tile descriptor); block_table, context_lens, q_lens,
 * sm_scale; FP8 (E4M3) K/V with fp32 scales per (page, KV head); a 0/1 block
 * mask over 128x128 (query, key) tiles.
 *
 * Semantics (identical to the fp64 oracle the tests compare against):
 *   query i of sequence b sits at absolute position p = context_lens[b] -
 *   q_lens[b] + i and attends to keys j <= p (keys j < context_lens[b]); with
 *   a block mask also only keys whose tile (i/128, j/128) is kept.  q head h
 *   reads KV head h / (Hq/Hkv).  out = softmax(sm_scale * q.K^T) V in bf16;
 *   lse = natural log of sum_j exp(sm_scale * q.k_j) in fp32.  A row with no
 *   visible key gets out = 0 and lse = -inf.
 *
 * Conventions
 *   - Every pointer argument except those marked "host" is a DEVICE pointer.
 *     The caller owns every buffer; the library allocates no device memory
 *     and keeps no per-call state.  (It caches, per device, the SM count and
 *     per-kernel attributes.  The one exception is pa_decode_noalloc, whose
 *     fixed scratch array belongs to the library.)
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  All calls
 *     are asynchronous on that stream except pa_read_task_map and
 *     pa_last_device_error, which synchronise it.
 *   - Host-side validation never throws: bad arguments return
 *     PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED / PA_ERR_WORKSPACE and launch
 *     nothing.  Launch failures return PA_ERR_CUDA.
 *   - Faults the device detects (a block-table entry outside [0, num_pages),
 *     q_lens > context_lens, lengths above the declared maxima, a wait that
 *     ran out of time) never trap: the kernel records a code in the Assign
 *     workspace, skips the offending access and finishes; the outputs of that
 *     call are then unspecified.  Read the code with pa_last_device_error.
 *   - Tensors are dense and row-major with the shapes given; every base
 *     pointer must be 16-byte aligned.  The prefill epilogue stores 32 bytes
 *     at a time into out and the partial workspace when they are 32-byte
 *     aligned (16 otherwise; same results, a little slower).
 *   - With total_q_tokens == 0 there is no query row: pa_decode_splitk,
 *     pa_decode_noalloc, pa_prefill and pa_combine return PA_OK without
 *     launching anything, and their buffers may be NULL (pa_assign still
 *     writes an empty task map).
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null pointer, bad dimension, misaligned buffer       */
    PA_ERR_UNSUPPORTED = 2,  /* valid but not built (head_dim, page_size, GQA ratio) */
    PA_ERR_WORKSPACE = 3,    /* a workspace smaller than the *_workspace_size query, or a
                                problem too large for the scratch of pa_decode_noalloc */
    PA_ERR_CUDA = 4,         /* a CUDA runtime call failed                           */
    PA_ERR_DEVICE_CHECK = 5, /* the device recorded a fault (pa_last_device_error)   */
    PA_ERR_TIMEOUT = 6       /* a bounded device wait ran out                        */
} pa_status;

/* KV cache layouts ("基于Triton-TLE…", 三.2). */
enum { PA_NHD = 0, PA_HND = 1 };
/* Element types of the KV cache (and of Q, see q_dtype).  FP8 is OCP E4M3FN.
 * Decode: E4M3 K/V with fp32 scales per (page, KV head), K and V separately,
 * and a bf16 Q.  Prefill (pa_prefill_fp8): E4M3 Q, K and V with one fp32
 * scale for K, one for V, and Q scales per q_scale_mode. */
enum { PA_BF16 = 0, PA_FP8_E4M3 = 1 };
/* E4M3 Q scales ("基于Triton-TLE…", 三: the two quantisation types of the FP8
 * prefill): one fp32 for the whole Q (quant type 0), or one per (token, q
 * head), laid out [total_q_tokens, Hq] (quant type 1).  K and V are per
 * tensor in both. */
enum { PA_SCALE_PER_TENSOR = 0, PA_SCALE_PER_ROW = 1 };
/* Assign modes.
 *   PA_MODE_DECODE:  one unit per (sequence, KV head) holding all q_lens[b]
 *                    queries (G*max_q_len rows: at most 32 for head_dim 128,
 *                    64 for head_dim 64; larger groups use the prefill
 *                    mode); 64-token KV tiles.
 *   PA_MODE_PREFILL: one unit per (sequence, KV head, q tile of 256/G tokens;
 *                    128 tokens when G = 1 with a block mask) = up to 256
 *                    rows, computed as two 128-row tensor-core tiles that
 *                    share every K/V tile; 128-token KV tiles; block mask
 *                    allowed.  Used by pa_prefill for prefill and mixed
 *                    batches. */
enum { PA_MODE_DECODE = 0, PA_MODE_PREFILL = 1 };
/* pa_read_task_map only: the decode-mode map that pa_assign(PA_MODE_PREFILL)
 * builds for the decode-shaped sequences of a batch (see pa_prefill). */
enum { PA_MAP_DECODE_PART = 2 };

/* Device error codes written by the kernels (read with pa_last_device_error). */
enum {
    PA_DEV_OK = 0,
    PA_DEV_BAD_LENGTHS = 1,    /* q_lens > context_lens, negative, above the maxima, or
                                  sum(q_lens) != total_q_tokens: the task map is empty */
    PA_DEV_BAD_PAGE = 2,       /* a block-table entry used was outside [0, num_pages)  */
    PA_DEV_WAIT_TIMEOUT = 4    /* a pipeline wait ran out of time                      */
};

/* Problem description, passed by host pointer and copied by every call. */
typedef struct pa_problem {
    int32_t num_seqs;          /* B                                                  */
    int32_t num_q_heads;       /* Hq                                                 */
    int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0, G = Hq/Hkv                      */
    int32_t head_dim;          /* D: 64 or 128                                       */
    int32_t page_size;         /* tokens per page: 16, 32, 64, 128 or 256             */
    int32_t num_pages;         /* pages in the cache pool (bound for block_table)     */
    int32_t max_pages_per_seq; /* row stride of block_table                          */
    int32_t total_q_tokens;    /* sum of q_lens = rows of q / out                    */
    int32_t max_q_len;         /* >= every q_lens[b]                                 */
    int32_t max_context_len;   /* >= every context_lens[b]                           */
    int32_t layout;            /* PA_NHD or PA_HND                                   */
    int32_t kv_dtype;          /* PA_BF16 or PA_FP8_E4M3                             */
    int32_t mask_q_tiles;      /* block mask dims per sequence; 0 = no mask          */
    int32_t mask_kv_tiles;
    int32_t num_ctas;          /* persistent CTAs; 0 = the library's choice          */
    int32_t balance_rows;      /* Assign weight divisor; 0 = 128                     */
    float sm_scale;            /* softmax scale applied to q.k; finite and >= 0      */
    int32_t window;            /* sliding window ("HiLS-Attention", 二.1 local
                                  branch): 0 = none, else the query at position p
                                  sees only the keys p - window < j <= p.  Both
                                  modes, bf16 and E4M3 K/V.  Negative: invalid. */
    int32_t q_dtype;           /* PA_BF16 (0), or PA_FP8_E4M3: the E4M3 prefill of
                                  pa_prefill_fp8, which needs kv_dtype PA_FP8_E4M3
                                  and head_dim 128; decode takes bf16 Q only     */
    int32_t q_scale_mode;      /* E4M3 Q: PA_SCALE_PER_TENSOR or PA_SCALE_PER_ROW    */
    int32_t unit_cost;         /* Assign's fixed cost of a unit with tiles, in the
                                  units of a tile's weight (the work a CTA spends
                                  on a unit besides its tiles); 0 = the library's
                                  choice (PA_DEFAULT_UNIT_COST_*), < 0 = none   */
} pa_problem;

/* The library's fixed cost per unit when pa_problem.unit_cost is 0, by Assign
 * mode (the decode part of a mixed batch takes the decode value).  Measured
 * on GB300: with none, the CTAs that draw many short units finish up to 30 %
 * after the mean (per-task timings from pa_set_task_trace); these values
 * bring the slowest within ~5 % on the decode and prefill batches. */
#define PA_DEFAULT_UNIT_COST_DECODE 6
#define PA_DEFAULT_UNIT_COST_PREFILL 4

/* Human-readable name of a pa_status or PA_DEV_* code set. */
PA_API const char* pa_status_string(int status);

/* Library version string. */
PA_API const char* pa_version(void);

/* Persistent CTA count that pa_assign and the compute pass of `mode` use for
 * this problem on the current device (problem->num_ctas if non-zero).  In
 * prefill mode this is the prefill kernel's; the decode part of a mixed batch
 * uses pa_num_ctas(PA_MODE_DECODE) of the problem with max_q_len capped at
 * 16 / G.  *num_ctas: host out. */
PA_API pa_status pa_num_ctas(const pa_problem* problem, int mode, int32_t* num_ctas);

/* Bytes of the Assign workspace for (problem, mode).  Its content (task map,
 * unit table, active-tile lists, error word; in prefill mode without a block
 * mask also the decode part's map) is private to the library. */
PA_API size_t pa_assign_workspace_size(const pa_problem* problem, int mode);

/* Bytes of the split-K partial workspace (fp32 O and LSE per split slot; in
 * prefill mode without a block mask also the decode part's slots). */
PA_API size_t pa_partial_workspace_size(const pa_problem* problem, int mode);

/*
 * Assign ("基于Triton-TLE…", 一.2: tile each sequence's KV and build a
 * load-balanced task map; 二.1: keep only the KV tiles the block mask keeps,
 * compacted into an ascending active-tile list).
 *   context_lens, q_lens: int32 [B]
 *   block_mask: uint8 [B][mask_q_tiles][mask_kv_tiles] or NULL (prefill mode only)
 *   assign_ws: >= pa_assign_workspace_size bytes, 256-byte aligned; written.
 * Clears the device error word.  Units are (b, hk) in decode mode and
 * (b, hk, q tile) in prefill mode; tile t of unit u weighs
 * w_u = max(1, ceil(G*rows/balance_rows)); CTA c owns the cost interval
 * [floor(c*C/N), floor((c+1)*C/N)) of the total cost C; a task is a maximal
 * run of one unit's tiles inside one CTA; split units get partial slots.
 * Prefill mode without a block mask builds two such maps: a decode-mode map
 * (units (b, hk), 64-token tiles, the decode kernel's CTA count) over the
 * sequences with 1 <= G*q_lens[b] <= 16, and the prefill-mode map over the
 * others; each map treats the other part's sequences as having no query.
 */
PA_API pa_status pa_assign(const pa_problem* problem, int mode, const int32_t* context_lens,
                    const int32_t* q_lens, const uint8_t* block_mask, void* assign_ws,
                    size_t assign_ws_bytes, void* stream);

/*
 * Split-K decode compute ("基于Triton-TLE…", 一.2 Split-K Compute; 三.1 small-M
 * query geometry: the G*q_len rows of one KV head share every K/V tile read).
 * Persistent CTAs walk the task map of pa_assign(PA_MODE_DECODE): per 64-token
 * KV tile a page lookup, a TMA load of K and V into a multi-stage shared-memory
 * ring, S = sm_scale * Q K^T, online softmax (fp32), O += P V.  An unsplit
 * unit writes out / lse directly.  A split unit's tasks write normalised
 * partial O and LSE to partial_ws.  With bf16 K/V each then counts itself
 * done on a completion counter in assign_ws, and the last one to finish
 * merges the unit's partials into out / lse ("基于Triton-TLE…", 三.3), so the
 * call leaves nothing for pa_combine and no task ever waits for another CTA.
 * With E4M3 K/V the partials are left to pa_combine (in that kernel the
 * finalizer costs more than the launch it saves).
 *   q: bf16 [total_q_tokens][Hq][D]
 *   k_cache, v_cache: bf16 or E4M3 bytes, NHD or HND (see above)
 *   block_table: int32 [B][max_pages_per_seq]; only entries of pages holding a
 *     token < context_lens[b] are read
 *   k_scale, v_scale: fp32 [num_pages][Hkv] (FP8 only; else may be NULL)
 *   assign_ws: from pa_assign(..., PA_MODE_DECODE, ...) on the same stream
 *   partial_ws: >= pa_partial_workspace_size(problem, PA_MODE_DECODE) bytes
 *   out: bf16 [total_q_tokens][Hq][D];  lse: fp32 [total_q_tokens][Hq] or NULL
 */
PA_API pa_status pa_decode_splitk(const pa_problem* problem, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* block_table,
                           const int32_t* context_lens, const int32_t* q_lens,
                           const float* k_scale, const float* v_scale, const void* assign_ws,
                           size_t assign_ws_bytes, void* partial_ws, size_t partial_ws_bytes,
                           void* out, float* lse, void* stream);

/*
 * Combine ("基于Triton-TLE…", 一.2 Combine; 三.3 merge of partial softmax
 * states with m = max, w_k = exp(m_k - m)).  For every unit split into S > 1
 * tasks: m = max_k lse_k, O = sum_k e^(lse_k - m) O_k / sum_k e^(lse_k - m),
 * lse = m + ln sum_k e^(lse_k - m).  Units with no visible key get O = 0,
 * lse = -inf.  Units written directly by the compute pass are not touched.
 * The bf16 decode kernel finalizes its own split units, and a decode-mode
 * unit always sees at least one key, so for a bf16 decode-mode workspace (and
 * for the decode part of a prefill-mode one) nothing is left: the call
 * validates its arguments and returns PA_OK without launching.  It finishes
 * E4M3 decode-mode maps and, in prefill mode, the prefill map.
 *   mode: the mode assign_ws was built with.
 */
PA_API pa_status pa_combine(const pa_problem* problem, int mode, const void* assign_ws,
                     size_t assign_ws_bytes, const void* partial_ws, size_t partial_ws_bytes,
                     void* out, float* lse, void* stream);

/*
 * Static split-K decode ("基于Triton-TLE…", 一.2, the Static Split-K
 * paragraph: a fixed split count, no Assign, a shorter launch chain; 三.3:
 * the regular split mapping is resolved from the program id, no task map is
 * built or read).  Every unit (sequence, KV head) is cut into the same number
 * S of splits: of the U * S tasks (U = B * Hkv), persistent CTA c of N runs
 * tasks c, c + N, c + 2N, ...; task i is split s = i % S of unit u = i / S
 * and covers the unit's 64-token KV tiles [s*n/S, (s+1)*n/S) of its n (a unit
 * of fewer than S tiles has empty splits, which carry no weight).  The compute
 * is that of pa_decode_splitk (same kernels, same semantics, sliding window
 * included); split units are finalized in the kernel by the last of their
 * tasks to finish, so this is one memset and one kernel launch per call.  It
 * does not rebalance ragged batches: the dynamic path (pa_assign +
 * pa_decode_splitk) does.
 *   num_splits: S in 1 .. 64, or 0 for the library's choice (the smallest
 *     power of two giving each CTA eight tasks or more, at most 4); see
 *     pa_static_num_splits.  With S = 2, 4 or 8 and a grid that is a multiple
 *     of S (the library's grid, or problem->num_ctas), and where the kernel
 *     variant has room for it (bf16 units of <= 16 rows, E4M3 units of <= 24),
 *     the S splits of a unit run on the S CTAs of one thread-block cluster and
 *     merge on chip through distributed shared memory (三.3): each CTA
 *     publishes its split's rows in a shared-memory mailbox, and the CTA of
 *     rank q merges the rows r = q (mod S) from all mailboxes and writes them;
 *     no partials go through global memory.  Otherwise the splits merge
 *     through ws and completion counters.
 *   ws: >= pa_static_workspace_size(problem, num_splits) bytes, 256-byte
 *     aligned; its first 256 bytes hold the device error word that
 *     pa_last_device_error reads.  The call clears the error word and the
 *     completion counters itself (a memset on `stream`); the rest needs no
 *     initialisation.
 *   Other arguments as pa_decode_splitk.  Lengths are checked on the device
 *   as pa_assign checks them (PA_DEV_BAD_LENGTHS; such a sequence's rows are
 *   not written).
 */
PA_API size_t pa_static_workspace_size(const pa_problem* problem, int32_t num_splits);
/* The split count S that pa_decode_static uses for (problem, num_splits) on
 * the current device; *splits: host out. */
PA_API pa_status pa_static_num_splits(const pa_problem* problem, int32_t num_splits,
                                      int32_t* splits);
PA_API pa_status pa_decode_static(const pa_problem* problem, int32_t num_splits, const void* q,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, const int32_t* context_lens,
                                  const int32_t* q_lens, const float* k_scale,
                                  const float* v_scale, void* ws, size_t ws_bytes, void* out,
                                  float* lse, void* stream);

/* Size of the fixed device scratch array behind pa_decode_noalloc: 32 MiB. */
#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * Whole decode (Assign, Split-K compute and, for E4M3 K/V, Combine: the
 * same passes and results as pa_assign + pa_decode_splitk + pa_combine in
 * PA_MODE_DECODE)
 * with every workspace taken from a fixed scratch array inside the library
 * instead of caller buffers.  The call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.  The pages describe no such entry
 * point; it is an addition of this library.
 *
 * Who it is for: callers that cannot hand the library device memory at call
 * time -- a serving engine that gave all free HBM to its KV-cache page pool up
 * front, or a plain C host with no device allocator of its own.  An
 * allocation inside the call would also cost latency and can synchronise the
 * device.
 *
 * The scratch is one file-scope device array of PA_NOALLOC_SCRATCH_BYTES
 * bytes.  Every GPU that loads the library holds it, whether or not this
 * entry point is called, until the process exits.
 *
 * Limit: the problem must fit, i.e. pa_assign_workspace_size (rounded up to
 * 256) + pa_partial_workspace_size, both for PA_MODE_DECODE, must be at most
 * PA_NOALLOC_SCRATCH_BYTES; otherwise the call returns PA_ERR_WORKSPACE and
 * launches nothing (use the caller-workspace entry points for such problems).
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it.  Make that
 * first call on every device before any stream capture starts.  The cached
 * address belongs to the device's current context: after cudaDeviceReset on a
 * device this entry point must not be called there again in the same process.
 *
 * Sharing: all calls on one device use the same array.  Two calls that may
 * run at the same time on one device (different streams without ordering,
 * several host threads) race and corrupt each other's results; order them on
 * one stream or synchronise between them.  Nothing needs clearing between
 * calls: Assign rewrites every scratch word the later passes read, and its
 * first kernel resets the device error word.
 *
 *   Arguments as pa_decode_splitk (out and lse receive the final result).
 *   device_error: int32, DEVICE pointer or NULL.  When given, the device
 *     error word of this call (PA_DEV_* bits) is copied there, on `stream`,
 *     after the last pass.
 */
PA_API pa_status pa_decode_noalloc(const pa_problem* problem, const void* q, const void* k_cache,
                                   const void* v_cache, const int32_t* block_table,
                                   const int32_t* context_lens, const int32_t* q_lens,
                                   const float* k_scale, const float* v_scale, void* out,
                                   float* lse, int32_t* device_error, void* stream);

/*
 * Prefill / mixed-batch compute ("基于Triton-TLE…", 一.2 Prefill: tile
 * scheduling by (batch, head, q tile), pipelined QK / causal mask / fp32 online
 * softmax / PV, epilogue; 二.1 active-tile list; 二.2 page-aware TMA pipeline;
 * "vLLM Triton Attention Backend Deep Dive": Q blocks pack the G heads of one
 * KV head, persistent fixed grid).  Walks the task map of
 * pa_assign(PA_MODE_PREFILL) with 256-row GQA-packed q tiles and 128-token KV
 * tiles on the tcgen05 tensor cores (accumulators in tensor memory).
 * Arguments as pa_decode_splitk, plus block_mask: the mask given to pa_assign,
 * non-NULL exactly when problem->mask_q_tiles > 0 (else PA_ERR_INVALID_ARG);
 * the kernels follow the active-tile lists pa_assign built from it.  In a batch without a block mask, the sequences with
 * 1 <= G*q_lens[b] <= 16 (the decode steps of a mixed chunked-prefill + decode
 * batch) run first, on the decode kernel of pa_decode_splitk over their own
 * task map: such a unit would fill a few of the 128 rows of a tensor-core
 * tile.  With a block mask every sequence takes the prefill path.
 */
PA_API pa_status pa_prefill(const pa_problem* problem, const void* q, const void* k_cache,
                     const void* v_cache, const int32_t* block_table,
                     const int32_t* context_lens, const int32_t* q_lens, const float* k_scale,
                     const float* v_scale, const uint8_t* block_mask, const void* assign_ws,
                     size_t assign_ws_bytes, void* partial_ws, size_t partial_ws_bytes,
                     void* out, float* lse, void* stream);

/*
 * FP8 prefill ("基于Triton-TLE…", 二: FP8 prefill over NHD/HND, two
 * quantisation types, dense or block-sparse; 二.2: the warp-specialised
 * pipeline also carries the quantisation scales).  problem->q_dtype and
 * kv_dtype must both be PA_FP8_E4M3 and head_dim 128 (else
 * PA_ERR_UNSUPPORTED); pa_assign, pa_assign_workspace_size and
 * pa_partial_workspace_size take the same problem in PA_MODE_PREFILL.  Every
 * sequence runs on the tensor-core kernel (no decode part): QK^T and PV are
 * E4M3 tcgen05 MMAs with fp32 accumulation; the probabilities enter PV as
 * two E4M3 terms (P and the rounding residual), about the precision of a
 * bf16 P.  The scores are sm_scale * q_scale * k_scale * (q8 . k8) and
 * out = v_scale * softmax(scores) V8 (bf16), lse as in pa_prefill.
 *   q:        uint8 E4M3 [total_q_tokens, Hq, 128].
 *   q_scale:  fp32, [1] (PA_SCALE_PER_TENSOR) or [total_q_tokens, Hq]
 *             (PA_SCALE_PER_ROW); positive and finite.
 *   k_scale, v_scale: fp32 [1] each, positive and finite.
 *   Other arguments as pa_prefill (caches are uint8 E4M3).  A partial
 *   workspace of the pa_partial_workspace_size this problem reports.
 */
PA_API pa_status pa_prefill_fp8(const pa_problem* problem, const void* q, const float* q_scale,
                                const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* context_lens,
                                const int32_t* q_lens, const float* k_scale, const float* v_scale,
                                const uint8_t* block_mask, const void* assign_ws,
                                size_t assign_ws_bytes, void* partial_ws,
                                size_t partial_ws_bytes, void* out, float* lse, void* stream);

/*
 * Test hook: copy the task map out of assign_ws (synchronises `stream`).
 * counts (host, int32[4]) = {units, tasks, slots, ctas}.  Each other host
 * array may be NULL; sizes: cta_ptr [ctas+1], tasks [tasks][4] = {unit, t0,
 * t1, slot} (t = positions in the unit's tile list), units [units][4] =
 * {b, hk, q0, nq}, unit_ntiles [units], unit_nsplit [units], unit_slot0
 * [units], active [units][max_kv_tiles] (only with a block mask; tile lists),
 * where max_kv_tiles = ceil(max_context_len / kv_tile), kv_tile 64 (decode) or
 * 128 (prefill).  mode PA_MAP_DECODE_PART reads the decode part of a
 * pa_assign(PA_MODE_PREFILL) workspace (kv_tile 64; all counts 0 when the
 * batch has a block mask or G > 16).
 */
PA_API pa_status pa_read_task_map(const pa_problem* problem, int mode, const void* assign_ws,
                           size_t assign_ws_bytes, int32_t* counts, int32_t* cta_ptr,
                           int32_t* tasks, int32_t* units, int32_t* unit_ntiles,
                           int32_t* unit_nsplit, int32_t* unit_slot0, int32_t* active,
                           void* stream);

/*
 * Test hook (the pages describe no such call; it exists to exercise the
 * failure path of the bounded waits without a GPU fault).  The next compute
 * launch in this process (the decode kernel of pa_decode_splitk or
 * pa_decode_noalloc, or the tensor-core kernel of pa_prefill -- not the
 * decode kernel pa_prefill runs first for a mixed batch's decode-shaped
 * sequences) runs with every pipeline wait limited to
 * wait_limit_ns, and in its CTA 0 the producer leaves K/V ring entry number
 * skip_entry (counted from 0 in issue order) unfilled.  The consumer waiting
 * for that entry runs out of time: the launch records PA_DEV_WAIT_TIMEOUT,
 * every CTA stops waiting, waits for the tensor copies it issued, frees its
 * tensor memory and finishes; the outputs of that call are unspecified.  The
 * hook disarms itself after that one launch.  skip_entry < 0 disarms it.
 * wait_limit_ns: 1e6 .. 1e9 (else PA_ERR_INVALID_ARG).
 */
PA_API pa_status pa_test_inject_wait_timeout(int32_t skip_entry, int64_t wait_limit_ns);

/*
 * Task trace (diagnostics: how evenly the persistent CTAs share a launch's
 * work; the pages describe no such call).  While a buffer is set, every
 * compute launch that walks an Assign task map -- the decode kernel of
 * pa_decode_splitk and pa_decode_noalloc, the tensor-core kernel of
 * pa_prefill / pa_prefill_fp8; not the static path and not the decode part of
 * a mixed batch -- records, for task k of its map (k < capacity):
 *   trace[3k]     the %globaltimer (ns) when its CTA starts the task,
 *   trace[3k + 1] the %globaltimer when the CTA is done with it,
 *   trace[3k + 2] the CTA index.
 * One thread per CTA writes; the rest of the kernel is unchanged.  Tasks
 * number as in pa_read_task_map.  Entries of tasks that did not run keep their
 * previous contents, so clear the buffer before the launch to be traced.
 *   trace: int64 [capacity][3], DEVICE pointer, 8-byte aligned, or NULL to stop
 *          tracing (then capacity must be 0).  The caller keeps it alive while set.
 * The setting is process-wide and stays until changed.
 */
PA_API pa_status pa_set_task_trace(int64_t* trace, int64_t capacity);

/* Read (and keep) the device error word of assign_ws into *code (host);
 * synchronises `stream`.  Returns PA_OK when *code == PA_DEV_OK, else
 * PA_ERR_DEVICE_CHECK (or PA_ERR_TIMEOUT when only the timeout bit is set). */
PA_API pa_status pa_last_device_error(const void* assign_ws, int32_t* code, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
