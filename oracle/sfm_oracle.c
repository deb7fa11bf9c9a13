/*
 * sfm_oracle.c -- plain, slow CPU reference for sparse shared-KV MLA attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path may call, link or
 * load this file; only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code with the CUDA
 * library: its own struct, its own element decoders, its own set logic.
 *
 * What it computes (all arithmetic in fp64 from the stored bf16/fp16/int8
 * inputs), following the pages' definitions:
 *
 *   O = softmax(Q . K~^T . softmax_scale) . V~,  K~ = V~          (1)
 *   LSE = log sum exp(S - max S) + max S,  S = Q K~^T . scale       (2)
 *
 *   (1),(2): "sparse_flash_mla" doc (zh), 功能说明 / 计算公式; same formula
 *   in the English doc ("Function") and the SparseAttnSharedkv README.
 *
 * The attended rows K~ of one query row are two disjoint sources:
 *   - ori_kv: a window [p - win_left, p + win_right] intersected with
 *     [0, kv_len) (ori_mask_mode 4), the causal prefix [0, p] (mode 3) or all
 *     of [0, kv_len) (mode 0); ori_win_left/right = -1 means unbounded
 *     ("sparse_flash_mla" doc, 参数说明: ori_mask_mode, ori_win_left,
 *     ori_win_right).  When ori_topk > 0 the ori source is instead the valid
 *     entries of ori_sparse_indices inside that same set (token-wise sparse
 *     selection of the kv_quant_sparse_flash_attention guide, 属性参数:
 *     sparse_block_size = 1, sparse_mode 0/3); with sparse_block_size > 1
 *     (block-wise selection, same 属性参数 row: the tokens of a block share
 *     the decision) entry e selects tokens e*sbs .. e*sbs + sbs - 1, each kept
 *     only inside that set.
 *   - cmp_kv: slot j is visible iff (j+1)*cmp_ratio <= p_cmp + 1 under
 *     cmp_mask_mode 3 (right-down causal), always under mode 0.  HCA attends
 *     every visible slot; CSA attends the valid entries of cmp_sparse_indices
 *     (-1 = invalid, valid first) ("sparse_flash_mla" doc, 功能说明: SWA / CSA
 *     / HCA; 参数说明: cmp_sparse_indices, cmp_residual_kv).
 * Query row i of batch b sits at p = kv_len - q_len + i (right-down
 * alignment; "sparse_flash_mla" doc, CP切分示例: the q start the kernel
 * derives is the prefix length minus the query length).
 * The cmp side uses the pre-compression length cmp_len*cmp_ratio + residual
 * (参数说明: the residual recovers the cmp-side mask length), so p_cmp = that length -
 * q_len + i; under the documented contract it equals p.
 *
 * Readings taken where the pages are silent (each listed in the design notes):
 *   sinks: per-head fp32 logit added to the denominator only,
 *          Z' = Z + exp(sink - m); the LSE excludes it.
 *   empty attended set (or query row beyond seqused_q): O = 0, LSE = -inf.
 *   CSA entries that are negative, >= cmp_len or not visible are skipped;
 *   duplicates count once per occurrence.
 *   packed rows: k[d] = int8[d] * scale[d / 128] for d < 512, then the rope
 *   values; V = k[0:512] (kv_quant_sparse_flash_attention guide, 计算公式 and
 *   the "A2/A3 C8 NoPE" table: 512 int8 + 64 rope + 4 fp32 scales = 656 B).
 *   FP8 packed rows (the guide's "Ascend 950 INT8/FP8 C8 NoPE" section, same
 *   528 / 656-byte layout): the 512 NoPE bytes are FLOAT8_E4M3FN values,
 *   k[d] = e4m3(byte d) * scale[d / 128].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* The oracle's own view of one problem.  Layout codes: 0 = BSND, 1 = TND,
 * 2 = paged.  Element codes: 0 = bf16, 1 = fp16.  All pointers are host. */
typedef struct oracle_problem {
    int32_t q_n, d_qk, d_v, rope_dim;
    int32_t batch, q_s, q_t;
    int32_t ori_s, cmp_s;            /* BSND capacity per batch entry */
    int32_t layout_q, layout_kv;
    int32_t dtype, kv_packed;
    int32_t ori_bs, cmp_bs, ori_bt_stride, cmp_bt_stride;
    int64_t ori_row_stride, cmp_row_stride;   /* bytes between rows */
    int64_t ori_rows, cmp_rows;               /* rows held by each buffer */
    int32_t ori_topk, cmp_topk, cmp_ratio, ori_sbs;
    int32_t ori_mask_mode, cmp_mask_mode, win_left, win_right;
    int32_t has_ori, has_cmp, has_sinks;
    double softmax_scale;
    const uint16_t *q;
    const uint8_t *ori_kv, *cmp_kv;
    const int32_t *ori_idx, *cmp_idx, *ori_bt, *cmp_bt;
    const int32_t *cu_q, *cu_ori, *cu_cmp, *used_q, *used_ori, *used_cmp, *residual;
    const float *sinks;
} oracle_problem;

enum { OR_OK = 0, OR_ERR_ARG = 1, OR_ERR_RANGE = 2, OR_ERR_CAP = 3 };

/* ---------------- element decoders (exact) ---------------- */
static double dec_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static double dec_fp16(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(m + 1024), e - 25);
    return s ? -v : v;
}

static double dec_half(const oracle_problem *P, uint16_t h)
{
    return P->dtype == 0 ? dec_bf16(h) : dec_fp16(h);
}

/* FLOAT8_E4M3FN (the OCP 8-bit floating point format the kv_quant guide names
 * for its A5 rows): sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent 0 is subnormal (m/8 * 2^-6); exponent 15 with mantissa 7 is NaN
 * and there is no infinity, so the largest finite value is 1.75 * 2^8 = 448. */
static double dec_e4m3(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(m + 8), e - 10);
    return s ? -v : v;
}

/* ---------------- per-token lengths and position ---------------- */
typedef struct {
    int b, i, q_len, kv_len, cmp_len, residual, p, p_cmp, in_range;
} tok_info;

static int token_info(const oracle_problem *P, int t, tok_info *o)
{
    int b, i, qcap;
    if (P->layout_q == 0) {
        if (P->q_s <= 0) return OR_ERR_ARG;
        b = t / P->q_s;
        i = t % P->q_s;
        qcap = P->q_s;
        if (b >= P->batch) return OR_ERR_RANGE;
    } else {
        if (!P->cu_q) return OR_ERR_ARG;
        b = -1;
        for (int k = 0; k < P->batch; ++k)
            if (P->cu_q[k] <= t && t < P->cu_q[k + 1]) { b = k; break; }
        if (b < 0) return OR_ERR_RANGE;
        i = t - P->cu_q[b];
        qcap = P->cu_q[b + 1] - P->cu_q[b];
    }
    o->b = b;
    o->i = i;
    o->q_len = P->used_q ? P->used_q[b] : qcap;
    if (P->used_ori) o->kv_len = P->used_ori[b];
    else if (P->layout_kv == 1) o->kv_len = P->cu_ori[b + 1] - P->cu_ori[b];
    else if (P->layout_kv == 0) o->kv_len = P->ori_s;
    else return OR_ERR_ARG;                     /* paged needs seqused_ori_kv */
    if (!P->has_ori) o->kv_len = 0;
    if (P->has_cmp) {
        if (P->used_cmp) o->cmp_len = P->used_cmp[b];
        else if (P->layout_kv == 1) o->cmp_len = P->cu_cmp[b + 1] - P->cu_cmp[b];
        else if (P->layout_kv == 0) o->cmp_len = P->cmp_s;
        else return OR_ERR_ARG;
    } else {
        o->cmp_len = 0;
    }
    o->residual = P->residual ? P->residual[b] : 0;
    o->p = o->kv_len - o->q_len + i;
    o->p_cmp = o->cmp_len * P->cmp_ratio + o->residual - o->q_len + i;
    o->in_range = i < o->q_len;
    return OR_OK;
}

/* ---------------- the attended set ---------------- */
/* ori window bounds [lo, hi] (inclusive) for mask mode 0 / 3 / 4 */
static void ori_bounds(const oracle_problem *P, const tok_info *ti, int64_t *lo, int64_t *hi)
{
    int64_t p = ti->p, n = ti->kv_len;
    *lo = 0;
    *hi = n - 1;
    if (P->ori_mask_mode == 3) {
        if (p < *hi) *hi = p;
    } else if (P->ori_mask_mode == 4) {
        if (P->win_left >= 0 && p - P->win_left > *lo) *lo = p - P->win_left;
        if (P->win_right >= 0 && p + P->win_right < *hi) *hi = p + P->win_right;
    }
}

static int cmp_visible(const oracle_problem *P, const tok_info *ti, int64_t j)
{
    if (P->cmp_mask_mode != 3) return 1;
    return (j + 1) * (int64_t)P->cmp_ratio <= (int64_t)ti->p_cmp + 1;
}

/* Enumerate the attended rows of token t: src 0 = ori, 1 = cmp, pos = logical
 * position (ori token position or cmp slot).  Returns the count; writes at
 * most cap entries.  Order: ori rows, then cmp rows, each in input order. */
static int64_t attended(const oracle_problem *P, int t, const tok_info *ti, int32_t *src, int32_t *pos,
                        int64_t cap)
{
    int64_t n = 0;
    if (!ti->in_range) return 0;
    if (P->has_ori && ti->kv_len > 0) {
        int64_t lo, hi;
        ori_bounds(P, ti, &lo, &hi);
        if (P->ori_topk > 0) {
            /* entry k selects the sbs tokens [e * sbs, (e + 1) * sbs); each
             * token is then kept only inside the ori mask set */
            const int32_t *row = P->ori_idx + (int64_t)t * P->ori_topk;
            const int64_t sbs = P->ori_sbs > 1 ? P->ori_sbs : 1;
            for (int k = 0; k < P->ori_topk; ++k) {
                if (row[k] < 0) continue;
                for (int64_t j = 0; j < sbs; ++j) {
                    const int64_t e = (int64_t)row[k] * sbs + j;
                    if (e >= ti->kv_len || e < lo || e > hi) continue;
                    if (n < cap) { src[n] = 0; pos[n] = (int32_t)e; }
                    ++n;
                }
            }
        } else {
            for (int64_t e = lo; e <= hi; ++e) {
                if (n < cap) { src[n] = 0; pos[n] = (int32_t)e; }
                ++n;
            }
        }
    }
    if (P->has_cmp && ti->cmp_len > 0) {
        if (P->cmp_topk > 0) {
            const int32_t *row = P->cmp_idx + (int64_t)t * P->cmp_topk;
            for (int k = 0; k < P->cmp_topk; ++k) {
                int64_t e = row[k];
                if (e < 0 || e >= ti->cmp_len || !cmp_visible(P, ti, e)) continue;
                if (n < cap) { src[n] = 1; pos[n] = (int32_t)e; }
                ++n;
            }
        } else {
            for (int64_t j = 0; j < ti->cmp_len; ++j) {
                if (!cmp_visible(P, ti, j)) continue;
                if (n < cap) { src[n] = 1; pos[n] = (int32_t)j; }
                ++n;
            }
        }
    }
    return n;
}

/* ---------------- row addressing and decoding ---------------- */
static const uint8_t *row_ptr(const oracle_problem *P, const tok_info *ti, int src, int64_t pos)
{
    const uint8_t *base = src ? P->cmp_kv : P->ori_kv;
    int64_t stride = src ? P->cmp_row_stride : P->ori_row_stride;
    int64_t nrows = src ? P->cmp_rows : P->ori_rows;
    int64_t row;
    if (P->layout_kv == 0) {
        row = (int64_t)ti->b * (src ? P->cmp_s : P->ori_s) + pos;
    } else if (P->layout_kv == 1) {
        row = (int64_t)(src ? P->cu_cmp[ti->b] : P->cu_ori[ti->b]) + pos;
    } else {
        int bs = src ? P->cmp_bs : P->ori_bs;
        const int32_t *bt = src ? P->cmp_bt : P->ori_bt;
        int bts = src ? P->cmp_bt_stride : P->ori_bt_stride;
        int64_t blk = bt[(int64_t)ti->b * bts + pos / bs];
        row = blk * bs + pos % bs;
    }
    if (row < 0 || row >= nrows) return NULL;
    return base + row * stride;
}

/* decode one attended row into k[0..d_qk) (fp64, exact) */
static void decode_row(const oracle_problem *P, const uint8_t *r, double *k)
{
    if (!P->kv_packed) {
        for (int d = 0; d < P->d_qk; ++d) {
            uint16_t h;
            memcpy(&h, r + 2 * d, 2);
            k[d] = dec_half(P, h);
        }
        return;
    }
    float scale[4];
    memcpy(scale, r + 512 + 2 * P->rope_dim, 16);
    if (P->kv_packed == 2)
        for (int d = 0; d < 512; ++d) k[d] = dec_e4m3(r[d]) * (double)scale[d / 128];
    else
        for (int d = 0; d < 512; ++d) k[d] = (double)(int8_t)r[d] * (double)scale[d / 128];
    for (int j = 0; j < P->rope_dim; ++j) {
        uint16_t h;
        memcpy(&h, r + 512 + 2 * j, 2);
        k[512 + j] = dec_half(P, h);
    }
}

/* ---------------- exported API ---------------- */
/* the E4M3 decoder on its own, for the tests that pin it */
double oracle_dec_e4m3(int32_t code) { return dec_e4m3((uint8_t)code); }

int oracle_token_info(const oracle_problem *P, int32_t t, int32_t *out9)
{
    tok_info ti;
    int rc = token_info(P, t, &ti);
    if (rc) return rc;
    out9[0] = ti.b; out9[1] = ti.i; out9[2] = ti.q_len; out9[3] = ti.kv_len; out9[4] = ti.cmp_len;
    out9[5] = ti.residual; out9[6] = ti.p; out9[7] = ti.p_cmp; out9[8] = ti.in_range;
    return OR_OK;
}

/* Attended set of token t; returns the count (>= 0) or -error. */
int64_t oracle_attended(const oracle_problem *P, int32_t t, int32_t *src, int32_t *pos, int64_t cap)
{
    tok_info ti;
    int rc = token_info(P, t, &ti);
    if (rc) return -rc;
    return attended(P, t, &ti, src, pos, cap);
}

/* Forward for the listed tokens.  O: n x q_n x d_v, lse: n x q_n (fp64). */
int oracle_forward(const oracle_problem *P, const int32_t *tokens, int32_t n, double *O, double *lse,
                   int32_t nthreads)
{
    int err = OR_OK;
    if (P->d_v != 512 || (P->kv_packed && P->d_qk != 512 + P->rope_dim) || (!P->kv_packed && P->d_qk != 512))
        return OR_ERR_ARG;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int64_t tasks = (int64_t)n * P->q_n;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t task = 0; task < tasks; ++task) {
        int ti_idx = (int)(task / P->q_n), h = (int)(task % P->q_n);
        int t = tokens[ti_idx];
        double *o = O + task * P->d_v;
        tok_info ti;
        for (int d = 0; d < P->d_v; ++d) o[d] = 0.0;
        lse[task] = -INFINITY;
        if (token_info(P, t, &ti)) {
#pragma omp atomic write
            err = OR_ERR_ARG;
            continue;
        }
        int64_t cnt = attended(P, t, &ti, NULL, NULL, 0);
        if (cnt == 0) continue;
        int32_t *src = (int32_t *)malloc(sizeof(int32_t) * cnt);
        int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * cnt);
        double *s = (double *)malloc(sizeof(double) * cnt);
        double *qv = (double *)malloc(sizeof(double) * P->d_qk);
        double *k = (double *)malloc(sizeof(double) * P->d_qk);
        attended(P, t, &ti, src, pos, cnt);
        const uint16_t *qh = P->q + ((int64_t)t * P->q_n + h) * P->d_qk;
        for (int d = 0; d < P->d_qk; ++d) qv[d] = dec_half(P, qh[d]);
        /* S = Q . K~^T . softmax_scale */
        double m = -INFINITY;
        int bad = 0;
        for (int64_t a = 0; a < cnt; ++a) {
            const uint8_t *r = row_ptr(P, &ti, src[a], pos[a]);
            if (!r) { bad = 1; break; }
            decode_row(P, r, k);
            double acc = 0.0;
            for (int d = 0; d < P->d_qk; ++d) acc += qv[d] * k[d];
            s[a] = acc * P->softmax_scale;
            if (s[a] > m) m = s[a];
        }
        if (bad) {
#pragma omp atomic write
            err = OR_ERR_RANGE;
        } else {
            /* softmax: Z = sum exp(s - m); O = sum exp(s - m) v / (Z + sink term) */
            double Z = 0.0;
            for (int64_t a = 0; a < cnt; ++a) Z += exp(s[a] - m);
            double denom = Z;
            if (P->has_sinks) denom += exp((double)P->sinks[h] - m);
            for (int64_t a = 0; a < cnt; ++a) {
                const uint8_t *r = row_ptr(P, &ti, src[a], pos[a]);
                decode_row(P, r, k);
                double w = exp(s[a] - m) / denom;
                for (int d = 0; d < P->d_v; ++d) o[d] += w * k[d];
            }
            lse[task] = m + log(Z);
        }
        free(src); free(pos); free(s); free(qv); free(k);
    }
    return err;
}

int oracle_abi_version(void) { return 1; }
