/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for paged-KV-cache attention
 * forward, the split-K Assign task map and the split-K Combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load or call this file.  It shares no
 * code, header, table or helper with the CUDA library, and the CUDA library
 * never calls it.
 *
 * Sources (pages are cited by title and section):
 *  [HPC]   "基于Triton-TLE优化Tencent HPC-Ops Attention" (flagos.csdn.net):
 *          sec. 一.2 "Prefill 与 Decode" -- paged KV through a block table,
 *          block mask, Assign / Split-K / Combine; sec. 二.1 active-tile list;
 *          sec. 三.3 the softmax-aware merge of (m, l, O) partial states.
 *  [HYB]   "Chunked Prefill" hybrid batch article (xdnf.cn news 311566),
 *          "混合批次计算图与内存访问不对称性": decode rows see the whole cache,
 *          a chunk is causal over its own tokens and unmasked over history.
 *  [VLLM]  "vLLM Triton Attention Backend Deep Dive", "Q Blocks": all q heads
 *          of one KV head are processed together (GQA grouping).
 *  [OCP8]  OCP 8-bit floating point specification, E4M3 ("fn") encoding:
 *          bias 7, no infinities, S.1111.111 is NaN, max normal 448.
 *
 * Readings taken where the pages are silent:
 *  - context_lens[b] is the total KV length including the q_lens[b] new
 *    tokens; query i of sequence b sits at absolute position
 *    p = ctx[b] - ql[b] + i and sees keys j <= p (bottom-right causal).
 *  - q head h reads KV head h / (Hq / Hkv) (contiguous groups).
 *  - LSE is the natural log of sum_j exp(sm_scale * q.k_j).
 *  - a row with no visible key has O = 0 and LSE = -inf.
 *  - the block mask is [B][mask_q_tiles][mask_kv_tiles], shared by all heads;
 *    row index = local query index / mask_tile, column = key / mask_tile.
 *  - FP8 K/V are E4M3FN bytes times an fp32 scale per (page, KV head).
 *  - Assign follows the procedure written out above oracle_assign().
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Problem description.  Mirrored field by field in oracle/__init__.py. */
typedef struct {
    int32_t num_seqs;          /* B                                          */
    int32_t num_q_heads;       /* Hq                                         */
    int32_t num_kv_heads;      /* Hkv, divides Hq                            */
    int32_t head_dim;          /* D                                          */
    int32_t page_size;         /* tokens per physical page                   */
    int32_t num_pages;         /* pages in the pool                          */
    int32_t max_pages_per_seq; /* row stride of block_table                  */
    int32_t layout;            /* 0 = NHD [page][slot][head][d]; 1 = HND [page][head][slot][d] */
    int32_t kv_dtype;          /* 0 = bf16 bit patterns; 1 = E4M3FN bytes    */
    int32_t mask_q_tiles;      /* 0 = no block mask                          */
    int32_t mask_kv_tiles;
    int32_t mask_tile;         /* tokens per mask tile edge (128)            */
    double sm_scale;
    int32_t window;            /* 0: none; else sliding window: query p sees keys
                                  p - window < j <= p ("HiLS-Attention", 二.1
                                  local branch; the bounds are our reading) */
    int32_t q_dtype;           /* 0 = bf16 bit patterns; 1 = E4M3FN bytes times q_scale */
    int32_t q_scale_mode;      /* E4M3 Q: 0 = one scale; 1 = one per (token, q head) */
    int32_t kv_scale_mode;     /* E4M3 K/V: 0 = one scale per (page, KV head);
                                  1 = one scale for the whole cache             */
} oracle_problem;

/* ---------------------------------------------------------------- decoding */

/* bf16 is the upper half of an IEEE binary32; exact in binary64. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* [OCP8] E4M3FN: sign, 4 exponent bits (bias 7), 3 mantissa bits.
 * exponent 0 is subnormal: 2^-6 * m/8; S.1111.111 is NaN; no infinities. */
double oracle_e4m3_to_double(uint8_t byte)
{
    int sign = (byte >> 7) & 1;
    int e = (byte >> 3) & 0xF;
    int m = byte & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* ------------------------------------------------------------- attention */

/* Where the key (or value) vector of sequence b at logical position j for KV
 * head hk starts, read through the block table ([HPC] 一.2: "根据 Block Table
 * 定位物理 K/V Page"): returns the element offset of d = 0 and stores the
 * (page, head) index for the FP8 scale.  Sets *bad and returns -1 when the
 * page index is outside the pool. */
static int64_t kv_offset(const oracle_problem* P, const int32_t* block_table, int b, int j, int hk,
                         int64_t* scale_idx, int* bad)
{
    int32_t page = block_table[(int64_t)b * P->max_pages_per_seq + j / P->page_size];
    int slot = j % P->page_size;
    if (page < 0 || page >= P->num_pages) {
        *bad = 1;
        return -1;
    }
    *scale_idx = (int64_t)page * P->num_kv_heads + hk;
    if (P->layout == 0)
        return (((int64_t)page * P->page_size + slot) * P->num_kv_heads + hk) * P->head_dim;
    return (((int64_t)page * P->num_kv_heads + hk) * P->page_size + slot) * P->head_dim;
}

/* Element d of a cached vector starting at offset off: bf16 decoded, or E4M3
 * decoded times the (page, head) scale. */
static double kv_value(const oracle_problem* P, const void* cache, const float* scale, int64_t off,
                       int64_t scale_idx, int d)
{
    if (P->kv_dtype == 0)
        return oracle_bf16_to_double(((const uint16_t*)cache)[off + d]);
    return oracle_e4m3_to_double(((const uint8_t*)cache)[off + d]) *
           (double)scale[P->kv_scale_mode == 1 ? 0 : scale_idx];
}

/* Element d of query row (token, h): bf16 decoded, or the E4M3 byte decoded
 * times its scale (one for the tensor, or one per (token, q head): the two
 * FP8 quantisation types of "基于Triton-TLE…", 二 / 三). */
static double q_value(const oracle_problem* P, const void* q, const float* q_scale,
                      int64_t token, int h, int d)
{
    const int64_t i = (token * P->num_q_heads + h) * (int64_t)P->head_dim + d;
    if (P->q_dtype == 0)
        return oracle_bf16_to_double(((const uint16_t*)q)[i]);
    return oracle_e4m3_to_double(((const uint8_t*)q)[i]) *
           (double)q_scale[P->q_scale_mode == 1 ? token * P->num_q_heads + h : 0];
}

/* Visibility of key j to local query i of sequence b: inside the context,
 * not after the query's own position (causal), inside the sliding window when
 * one is set, inside [key_lo, key_hi) and, when a block mask is given, inside a
 * kept tile. */
static int visible(const oracle_problem* P, const uint8_t* mask, int b, int i, int64_t p, int j,
                   int64_t key_lo, int64_t key_hi)
{
    if (j > p || j < key_lo || j >= key_hi)
        return 0;
    if (P->window > 0 && (int64_t)j <= p - P->window)
        return 0;
    if (mask && P->mask_q_tiles > 0) {
        int qt = i / P->mask_tile, kt = j / P->mask_tile;
        if (qt >= P->mask_q_tiles || kt >= P->mask_kv_tiles)
            return 0;
        return mask[((int64_t)b * P->mask_q_tiles + qt) * P->mask_kv_tiles + kt] != 0;
    }
    return 1;
}

/*
 * Attention forward for a list of (token, q head) rows.
 *
 * For each requested row r = token * Hq + h, with b the sequence owning the
 * token, i its index among the sequence's new tokens, p = ctx[b]-ql[b]+i and
 * hk = h / (Hq/Hkv):
 *     s_j   = sm_scale * sum_d Q[token][h][d] * K_j[d]     for visible j
 *     m     = max_j s_j
 *     L     = sum_j exp(s_j - m)
 *     O[d]  = sum_j exp(s_j - m) * V_j[d] / L
 *     LSE   = m + ln L
 * (the plain softmax attention that [HPC] 一.2 says Combine reproduces exactly;
 * the visibility rule of [HYB]).  key_lo/key_hi restrict the keys (used to
 * build split-K partials); pass 0 and INT64_MAX for the full range.
 *
 * q: bf16 bits, or E4M3 bytes (q_dtype 1), [total_tokens][Hq][D]; q_scale:
 * fp32 [1] or [total_tokens][Hq] (E4M3 Q only).  rows == NULL means all rows
 * in order.
 * out: [n_rows][D], lse: [n_rows].  Returns 0, or -1 on bad arguments,
 * -2 if a block-table entry used is outside the pool, -3 if ql > ctx.
 */
int oracle_attention(const oracle_problem* P, const void* q, const float* q_scale,
                     const void* k_cache,
                     const void* v_cache, const float* k_scale, const float* v_scale,
                     const int32_t* block_table, const int32_t* context_lens,
                     const int32_t* q_lens, const uint8_t* block_mask, const int64_t* rows,
                     int64_t n_rows, int64_t key_lo, int64_t key_hi, double* out, double* lse,
                     int num_threads)
{
    const int B = P->num_seqs, Hq = P->num_q_heads, Hkv = P->num_kv_heads, D = P->head_dim;
    int64_t* cu;
    int64_t total = 0;
    int max_ctx = 0, status = 0, b;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || P->page_size <= 0)
        return -1;
    if (P->kv_dtype == 1 && (!k_scale || !v_scale))
        return -1;
    if (P->q_dtype == 1 && !q_scale)
        return -1;
    cu = (int64_t*)malloc(sizeof(int64_t) * (size_t)(B + 1));
    if (!cu)
        return -1;
    cu[0] = 0;
    for (b = 0; b < B; ++b) {
        if (q_lens[b] < 0 || context_lens[b] < 0 || q_lens[b] > context_lens[b]) {
            free(cu);
            return -3;
        }
        cu[b + 1] = cu[b] + q_lens[b];
        if (context_lens[b] > max_ctx)
            max_ctx = context_lens[b];
    }
    total = cu[B];
    if (!rows && n_rows != total * Hq) {
        free(cu);
        return -1;
    }
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif

#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
        unsigned char* vis = (unsigned char*)malloc((size_t)(max_ctx > 0 ? max_ctx : 1));
        int64_t r;
#pragma omp for schedule(dynamic, 4)
        for (r = 0; r < n_rows; ++r) {
            int64_t row = rows ? rows[r] : r;
            int64_t token = row / Hq;
            int h = (int)(row % Hq);
            int hk = h / (Hq / Hkv);
            int lo = 0, hi = B, sb, i, j, d, any = 0, bad = 0;
            int64_t p;
            double m = -INFINITY, L = 0.0;
            double* o = out + r * D;
            if (token < 0 || token >= total) {
#pragma omp atomic write
                status = -1;
                continue;
            }
            /* sequence owning this token: the last sb with cu[sb] <= token */
            while (hi - lo > 1) {
                int mid = (lo + hi) / 2;
                if (cu[mid] <= token)
                    lo = mid;
                else
                    hi = mid;
            }
            sb = lo;
            i = (int)(token - cu[sb]);
            p = (int64_t)context_lens[sb] - q_lens[sb] + i;
            for (j = 0; j < context_lens[sb]; ++j) {
                vis[j] = (unsigned char)visible(P, block_mask, sb, i, p, j, key_lo, key_hi);
                if (!vis[j])
                    continue;
                double acc = 0.0;
                int64_t si = 0, off = kv_offset(P, block_table, sb, j, hk, &si, &bad);
                if (off < 0) {
                    vis[j] = 0;
                    continue;
                }
                for (d = 0; d < D; ++d)
                    acc += q_value(P, q, q_scale, token, h, d) *
                           kv_value(P, k_cache, k_scale, off, si, d);
                s[j] = P->sm_scale * acc;
                if (!any || s[j] > m)
                    m = s[j];
                any = 1;
            }
            for (d = 0; d < D; ++d)
                o[d] = 0.0;
            if (!any) {
                lse[r] = -INFINITY;
            } else {
                for (j = 0; j < context_lens[sb]; ++j)
                    if (vis[j])
                        L += exp(s[j] - m);
                for (j = 0; j < context_lens[sb]; ++j) {
                    if (!vis[j])
                        continue;
                    double w = exp(s[j] - m) / L;
                    int64_t si = 0, off = kv_offset(P, block_table, sb, j, hk, &si, &bad);
                    if (off < 0)
                        continue;
                    for (d = 0; d < D; ++d)
                        o[d] += w * kv_value(P, v_cache, v_scale, off, si, d);
                }
                lse[r] = m + log(L);
            }
            if (bad) {
#pragma omp atomic write
                status = -2;
            }
        }
        free(s);
        free(vis);
    }
    free(cu);
    return status;
}

/* --------------------------------------------------------------- combine */

/*
 * Merge S split-K partial results of one output row ([HPC] 一.2 "Combine":
 * re-weight each chunk's local output by its LSE; 三.3 the merge with
 * m = max, w_k = exp(m_k - m)).  Partials hold the normalised local output
 * O_k and LSE_k of their key subset:
 *     m   = max_k LSE_k
 *     O   = sum_k exp(LSE_k - m) O_k / sum_k exp(LSE_k - m)
 *     LSE = m + ln sum_k exp(LSE_k - m)
 * Splits with LSE_k = -inf (no visible key) carry no weight; if all are
 * -inf the row is O = 0, LSE = -inf.
 */
void oracle_combine(int S, int D, const double* o_parts, const double* lse_parts, double* o,
                    double* lse)
{
    double m = -INFINITY, den = 0.0;
    int k, d;
    for (k = 0; k < S; ++k)
        if (lse_parts[k] > m)
            m = lse_parts[k];
    for (d = 0; d < D; ++d)
        o[d] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    for (k = 0; k < S; ++k) {
        if (lse_parts[k] == -INFINITY)
            continue;
        double w = exp(lse_parts[k] - m);
        den += w;
        for (d = 0; d < D; ++d)
            o[d] += w * o_parts[(int64_t)k * D + d];
    }
    for (d = 0; d < D; ++d)
        o[d] /= den;
    *lse = m + log(den);
}

/* ---------------------------------------------------------------- assign */

/*
 * Assign: split every unit's KV into tiles and hand the tiles to num_ctas
 * CTAs so that each CTA gets an equal share of the work ([HPC] 一.2 "Assign:
 * 将各 KV 序列切成 Tile,并按 CTA 工作量生成负载均衡的 Task Map"; 三.3 "均分
 * 调度": every CTA carries a similar amount of KV work).  The pages give the
 * goal, not the procedure; this is the procedure, written tile by tile:
 *
 *  1. Units.  mode 0 (decode): u = b*Hkv + hk, all ql[b] queries of the
 *     sequence, rows R_u = G*ql[b], key length L_u = ctx[b].
 *     mode 1 (prefill / mixed): q tiles of qtok = 256/G tokens ([VLLM] "Q
 *     Blocks": G heads x qtok tokens = 256 rows, two 128-row MMA tiles that
 *     share every K/V tile); with a block mask and G = 1, qtok = 128 so a
 *     unit never spans two mask rows; units ordered by b, hk, qt;
 *     q0 = qt*qtok, nq = min(qtok, ql-q0), R_u = G*nq,
 *     L_u = ctx - ql + q0 + nq (keys up to the tile's last query).
 *     A sequence with ql = 0 has no units in mode 1 and empty units in mode 0.
 *  2. Tiles of kv_tile keys.  Without a mask the unit's tile list is
 *     0 .. ceil(L_u/kv_tile)-1.  With a mask (mode 1 only, kv_tile equal to
 *     the mask tile) it is the ascending list of kt with kt*kv_tile < L_u and
 *     mask[b][q0/mask_tile][kt] != 0 ([HPC] 二.1 active-KV-tile list).
 *     n_u = length of the list.
 *  3. Weight w_u = max(1, ceil(R_u / balance_rows)).  A unit with tiles also
 *     carries a fixed cost h_u = unit_cost (0 for a unit without tiles): the
 *     work a CTA spends on a unit besides its tiles (its queries in, its
 *     rows out), in the units of a tile's weight.
 *  4. Cost prefix P_u = sum_{u'<u} (h_u' + n_u' w_u'), total C.  CTA c owns
 *     the cost interval [a_c, a_{c+1}) with a_c = floor(c*C/N).  List
 *     position t of unit u sits at cost P_u + h_u + t*w_u and belongs to the
 *     CTA whose interval contains it.
 *  5. A task is a maximal run of one unit's positions owned by one CTA.
 *     Tasks are ordered by CTA, then cost; cta_ptr[c] is the first task of
 *     CTA c.  The k-th task of a unit has split index k; S_u = task count.
 *  6. slot = -1 if S_u == 1, else slot0_u + k where
 *     slot0_u = sum_{u'<u, S_u'>1} S_u'.  unit_slot0 = -1 when S_u <= 1.
 *  7. Units with n_u = 0 get no task (S_u = 0).
 *
 * Outputs (caller allocates):
 *   units[unit_cap][4]         = {b, hk, q0, nq}
 *   unit_ntiles[unit_cap]      = n_u
 *   active[unit_cap][max_kv_tiles] = the unit's tile list (first n_u used)
 *   cta_ptr[N+1]; tasks[task_cap][4] = {u, t0, t1, slot} (t = list positions)
 *   unit_nsplit[unit_cap] = S_u; unit_slot0[unit_cap]
 *   counts[3] = {U, n_tasks, n_slots}
 * Returns 0, -1 on bad arguments, -4 if a capacity is too small.
 */
int oracle_assign(int mode, int B, int Hq, int Hkv, int N, int kv_tile, int balance_rows,
                  const int32_t* ctx, const int32_t* ql, const uint8_t* mask, int mask_q_tiles,
                  int mask_kv_tiles, int mask_tile, int32_t* units, int32_t* unit_ntiles,
                  int32_t* active, int max_kv_tiles, int32_t* cta_ptr, int32_t* tasks,
                  int64_t task_cap, int32_t* unit_nsplit, int32_t* unit_slot0, int32_t* counts,
                  int64_t unit_cap, int window, int unit_cost)
{
    int G, qtok, b, hk, c;
    int64_t U = 0, u, C, n_tasks = 0, slots = 0;
    int64_t* prefix;
    int64_t* bound;
    int64_t* weight;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || N <= 0 || kv_tile <= 0 || balance_rows <= 0 ||
        unit_cost < 0)
        return -1;
    G = Hq / Hkv;
    if (mode == 1 && (G > 128 || 128 % G))
        return -1;
    if (mask && (mode != 1 || kv_tile != mask_tile))
        return -1;
    qtok = (mask && G == 1) ? 128 : 256 / G;

    /* 1-3: units, tile lists, weights */
    for (b = 0; b < B; ++b) {
        int nqt = (mode == 0) ? 1 : (ql[b] + qtok - 1) / qtok;
        for (hk = 0; hk < Hkv; ++hk) {
            int qt;
            for (qt = 0; qt < nqt; ++qt) {
                int q0, nq, t, n = 0;
                int64_t L;
                if (U >= unit_cap)
                    return -4;
                if (mode == 0) {
                    q0 = 0;
                    nq = ql[b];
                    L = nq > 0 ? ctx[b] : 0;
                } else {
                    q0 = qt * qtok;
                    nq = ql[b] - q0 < qtok ? ql[b] - q0 : qtok;
                    L = (int64_t)ctx[b] - ql[b] + q0 + nq;
                }
                units[U * 4 + 0] = b;
                units[U * 4 + 1] = hk;
                units[U * 4 + 2] = q0;
                units[U * 4 + 3] = nq;
                /* sliding window: the unit's first query (position ctx - ql + q0)
                 * sees no key before p0 - window + 1; tiles wholly before it are
                 * not the unit's */
                t = 0;
                if (window > 0) {
                    int64_t lo = (int64_t)ctx[b] - ql[b] + q0 - window + 1;
                    if (lo > 0)
                        t = (int)(lo / kv_tile);
                }
                for (; (int64_t)t * kv_tile < L; ++t) {
                    int keep = 1;
                    if (mask) {
                        int mq = q0 / mask_tile;
                        keep = (mq < mask_q_tiles && t < mask_kv_tiles) &&
                               mask[((int64_t)b * mask_q_tiles + mq) * mask_kv_tiles + t] != 0;
                    }
                    if (!keep)
                        continue;
                    if (n >= max_kv_tiles)
                        return -4;
                    active[U * max_kv_tiles + n] = t;
                    ++n;
                }
                unit_ntiles[U] = n;
                ++U;
            }
        }
    }

    /* 4: cost prefix and CTA boundaries */
    prefix = (int64_t*)malloc(sizeof(int64_t) * (size_t)(U + 1));
    weight = (int64_t*)malloc(sizeof(int64_t) * (size_t)(U + 1));
    bound = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N + 1));
    if (!prefix || !bound || !weight) {
        free(prefix);
        free(weight);
        free(bound);
        return -1;
    }
    prefix[0] = 0;
    for (u = 0; u < U; ++u) {
        int64_t R = (int64_t)G * units[u * 4 + 3];
        weight[u] = (R + balance_rows - 1) / balance_rows;
        if (weight[u] < 1)
            weight[u] = 1;
        prefix[u + 1] = prefix[u] + (unit_ntiles[u] > 0 ? unit_cost : 0) + unit_ntiles[u] * weight[u];
    }
    C = prefix[U];
    for (c = 0; c <= N; ++c)
        bound[c] = (int64_t)c * C / N;

    /* 5-7: walk every tile in cost order and cut tasks */
    for (c = 0; c <= N; ++c)
        cta_ptr[c] = 0;
    for (u = 0; u < U; ++u) {
        int64_t w = weight[u];
        int t, cur_cta = -1;
        unit_nsplit[u] = 0;
        for (t = 0; t < unit_ntiles[u]; ++t) {
            int64_t x = prefix[u] + unit_cost + t * w;
            int owner = 0;
            /* owner = the last CTA whose interval starts at or before x */
            while (owner + 1 < N && bound[owner + 1] <= x)
                ++owner;
            if (owner != cur_cta) {
                if (n_tasks >= task_cap) {
                    free(prefix);
                    free(weight);
                    free(bound);
                    return -4;
                }
                tasks[n_tasks * 4 + 0] = (int32_t)u;
                tasks[n_tasks * 4 + 1] = t;
                tasks[n_tasks * 4 + 2] = t + 1;
                tasks[n_tasks * 4 + 3] = unit_nsplit[u]; /* split index k for now */
                ++n_tasks;
                ++unit_nsplit[u];
                cta_ptr[owner + 1] += 1;
                cur_cta = owner;
            } else {
                tasks[(n_tasks - 1) * 4 + 2] = t + 1;
            }
        }
    }
    for (c = 0; c < N; ++c)
        cta_ptr[c + 1] += cta_ptr[c];
    for (u = 0; u < U; ++u) {
        if (unit_nsplit[u] > 1) {
            unit_slot0[u] = (int32_t)slots;
            slots += unit_nsplit[u];
        } else {
            unit_slot0[u] = -1;
        }
    }
    for (u = 0; u < n_tasks; ++u) {
        int32_t uu = tasks[u * 4 + 0];
        tasks[u * 4 + 3] = unit_nsplit[uu] > 1 ? unit_slot0[uu] + tasks[u * 4 + 3] : -1;
    }
    counts[0] = (int32_t)U;
    counts[1] = (int32_t)n_tasks;
    counts[2] = (int32_t)slots;
    free(prefix);
    free(weight);
    free(bound);
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
