// sfm_internal.cuh -- shared device/host definitions of the sfm library.
//
// Everything the planner, the attention kernel and the combine kernel agree
// on lives here: the kernel parameter block, the metadata layout and the
// per-query-row lengths, window and attended-position counts.  The attended
// set follows the
// "sparse_flash_mla" doc (zh), 参数说明 (ori_mask_mode, ori_win_left/right,
// cmp_mask_mode, cmp_sparse_indices, cmp_residual_kv) and the right-down
// alignment p = kv_len - q_len + i of its CP切分示例.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sfm.h"

namespace sfm {

// ----------------------------------------------------------------------------
// metadata layout (int32 words)
//   [0, HDR)                  header (H_* below)
//   ws[G + 1]                 worker split ranges: worker c owns splits [ws[c], ws[c+1])
//   sp[T + 1]                 split prefix per query row: row t owns splits [sp[t], sp[t+1])
//   cp[T + 1]                 cost prefix per query row (attended rows + per-split overhead)
//   rec[T][8]                 per query row: b, kv_len, cmp_len, p_cmp, lo, hi, n_ori, n_cmp
//   own[Wcap]                 owning query row of every split
//   srec[Wcap][16]            per split (64-byte aligned): t, first split of t, splits of t,
//                             split size of t, then t's rec[8]; one 64-byte load gives a
//                             kernel everything it needs about a split
//   wrec[G][32]               per worker: first and end unit, 2 spare words, then the
//                             srec of its first unit's split (one load to start work)
// ----------------------------------------------------------------------------
constexpr int32_t kMetaMagic = 0x53464d31;   // "SFM1"
constexpr int kHdr = 16;
constexpr int kRecWords = 8;
enum MetaHeader {
    H_MAGIC = 0, H_FPRINT = 1, H_TOKENS = 2, H_WORKERS = 3, H_SPLIT = 4, H_PATH = 5,
    H_TOTAL_SPLITS = 6, H_FLAGS = 7, H_LENFLAGS = 8, H_WCAP = 9
};
// modelled cost of one split beyond its rows, in rows: a split pays the
// latency of its metadata / Q / first-tile loads and of its epilogue
// whatever its length, so splits are balanced first by count, then by rows
constexpr int kSplitOverheadRows = 128;

// A row with n attended positions gets ceil(n / S) splits of equal size
// (rounded up to 32 rows; never more than S when S is a multiple of 32, so
// the last split is never empty).  Depends on the row's own n and the params
// only, which keeps results batch invariant.
// Division by a divisor fixed for the launch (a block size), by
// multiplication: with l = ceil(log2 d) and M = ceil(2^(32 + l) / d),
// floor(n M / 2^(32 + l)) = floor(n / d) for every 0 <= n < 2^32 (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994).
// M < 2^33 is kept as lo + hi 2^32 with hi 0 or 1.
struct FastDiv {
    uint32_t lo, hi, l, d;
};

inline FastDiv make_fastdiv(uint32_t d)
{
    FastDiv f{0, 0, 0, d};
    if (d == 0) return f;
    while ((1ull << f.l) < d) ++f.l;
    const uint64_t m = ((1ull << (32 + f.l)) + d - 1) / d;
    f.lo = (uint32_t)m;
    f.hi = (uint32_t)(m >> 32);
    return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f)
{
    const uint64_t t = (uint64_t)__umulhi(n, f.lo) + (f.hi ? n : 0u);
    return (uint32_t)(t >> f.l);
}

// a / b for a >= 0, b > 0: a 32-bit division when both fit (64-bit integer
// division is a long dependent instruction sequence on the GPU)
__host__ __device__ inline int64_t div_nonneg(int64_t a, int64_t b)
{
    if ((((uint64_t)a | (uint64_t)b) >> 32) == 0) return (int64_t)((uint32_t)a / (uint32_t)b);
    return a / b;
}

// number of splits of a row with n attended positions
__host__ __device__ inline int64_t num_splits(int64_t n, int S)
{
    return n > 0 ? div_nonneg(n + S - 1, S) : 0;
}

__host__ __device__ inline int split_size(int64_t n, int S)
{
    if (n <= 0) return S;
    const int64_t ns = num_splits(n, S);
    const int64_t sz = div_nonneg(n + ns - 1, ns);
    return (int)((sz + 31) & ~(int64_t)31);
}

// floor(a / b) for 32-bit a, b >= 1: a float estimate (32-bit conversions
// are cheap, 64-bit ones and integer division are not) corrected exactly; the
// estimate is within one of the quotient whenever a < 2^24, and an estimate
// that needs more than two corrections falls back to the division
__device__ __forceinline__ uint32_t udiv_est(uint32_t a, uint32_t b)
{
    uint32_t q = __float2uint_rz(__fdividef(__uint2float_rz(a), __uint2float_rz(b)));
    if ((uint64_t)q * b > a) --q;
    else if (((uint64_t)q + 1) * b <= a) ++q;
    if ((uint64_t)q * b > a || ((uint64_t)q + 1) * b <= a) q = a / b;
    return q;
}

// num_splits / split_size with the launch's precomputed division by split_rows
__device__ __forceinline__ int64_t num_splits_dev(int64_t n, const FastDiv &sd)
{
    if (n <= 0) return 0;
    const int64_t a = n + sd.d - 1;
    return a <= 0xffffffffll ? (int64_t)fdiv((uint32_t)a, sd) : a / sd.d;
}
__device__ __forceinline__ int split_size_dev(int64_t n, const FastDiv &sd)
{
    if (n <= 0) return (int)sd.d;
    const int64_t ns = num_splits_dev(n, sd);
    const int64_t a = n + ns - 1;
    const int64_t sz = ns == 1 ? n : a <= 0xffffffffll ? (int64_t)udiv_est((uint32_t)a, (uint32_t)ns) : a / ns;
    return (int)((sz + 31) & ~(int64_t)31);
}

__host__ __device__ inline int64_t meta_ws_off() { return kHdr; }
__host__ __device__ inline int64_t meta_split_off(int G) { return kHdr + (int64_t)G + 1; }
__host__ __device__ inline int64_t meta_cost_off(int G, int T) { return kHdr + (int64_t)G + 1 + (int64_t)T + 1; }
__host__ __device__ inline int64_t meta_rec_off(int G, int T) { return meta_cost_off(G, T) + (int64_t)T + 1; }
constexpr int kSrecWords = 16;
constexpr int kWrecWords = 16;
__host__ __device__ inline int64_t meta_srec_off(int G, int T, int64_t wcap)
{
    (void)wcap;
    return (meta_rec_off(G, T) + (int64_t)kRecWords * T + 15) & ~(int64_t)15;
}
__host__ __device__ inline int64_t meta_wrec_off(int G, int T, int64_t wcap)
{
    return meta_srec_off(G, T, wcap) + (int64_t)kSrecWords * wcap;
}
__host__ __device__ inline int64_t meta_words(int G, int T, int64_t wcap)
{
    int64_t n = meta_wrec_off(G, T, wcap) + (int64_t)kWrecWords * G;
    return n < 1024 ? 1024 : n;
}

// the attention path a plan was made for (recorded in the plan header)
enum PathId : int32_t { PATH_TC = 2 };

// ----------------------------------------------------------------------------
// kernel parameter block (passed by value)
// ----------------------------------------------------------------------------
struct KParams {
    int32_t q_n, d_qk, d_v, rope;
    int32_t batch, q_s, T;                 // T = query rows ("tokens")
    int32_t ori_s, cmp_s;                  // BSND per-batch capacity
    int32_t ori_max, cmp_max;              // paged: declared max lengths (length capacity)
    int32_t layout_q, layout_kv, dtype, packed;
    int32_t kv_fp8;                        // packed NoPE bytes are FLOAT8_E4M3FN (else int8)
    int32_t ori_bs, cmp_bs, ori_bt_stride, cmp_bt_stride;
    FastDiv ori_bs_div, cmp_bs_div;        // division by the block sizes
    FastDiv q_s_div, ratio_div, split_div; // by q_s, cmp_ratio and split_rows
    int64_t ori_row_stride, cmp_row_stride, ori_rows, cmp_rows;
    int32_t ori_topk, cmp_topk, cmp_ratio, ori_mask_mode, cmp_mask_mode, win_left, win_right;
    int32_t sbs_log2;                      // log2 of the tokens per ori_sparse_indices entry
    int32_t has_cmp, return_lse;
    float scale;                            // softmax_scale
    float scale_log2;                       // softmax_scale * log2(e)
    // plan
    int32_t G, split_rows, fingerprint, path;
    int32_t head_groups;                    // groups of 64 heads: a token
                                            // with n splits owns head_groups * n work units, group-major
    int64_t ws_capacity_splits;
    int32_t max_splits;                     // splits a row can have: row t's partials use workspace
                                            // slots t * max_splits .. t * max_splits + max_splits - 1
    int64_t wcap;                           // capacity of the split -> row map
    // tensors
    const void *q;
    const uint8_t *ori_kv, *cmp_kv;
    const int32_t *ori_idx, *cmp_idx, *ori_bt, *cmp_bt;
    const int32_t *cu_q, *cu_ori, *cu_cmp, *used_q, *used_ori, *used_cmp, *residual;
    const float *sinks;
    const int32_t *meta;
    int32_t *meta_w;
    void *out;
    float *lse;
    uint16_t *ws_o;   // [slot][512 / 8][q_n][8] normalised partial O, bf16, chunk-major
    float *ws_lse;    // [slot][q_n] partial LSE
    int32_t *status;
    int32_t *dbg_rows;   // attended-row dump (sfm_debug_attended): [T][dbg_cap] resolver entries, or NULL
    int64_t dbg_cap;
    int32_t *dbg_counts; // [T] attended positions per row (clamped to dbg_cap)
};

__device__ __forceinline__ void set_status(const KParams &kp, int bits)
{
    if (kp.status) atomicOr(kp.status, bits);
}

// ----------------------------------------------------------------------------
// per query row: lengths, position, window, attended-position counts
// ----------------------------------------------------------------------------
struct Tok {
    int32_t b, i, q_len, kv_len, cmp_len, p, p_cmp, valid;
    int32_t lo, hi;        // ori window, inclusive (hi < lo: empty)
    int32_t n_ori, n_cmp;  // attended positions of each source (topk entries or contiguous rows)
};

// L2 prefetch of the 128-byte line holding p (an ordinary per-thread
// instruction; no alignment rule)
__device__ __forceinline__ void prefetch_line_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Four FLOAT8_E4M3FN bytes of w (byte 0 first) -> fp32, exactly: the PTX
// conversion to fp16 pairs is exact (every E4M3 value, subnormals included,
// is an fp16 value) and fp16 -> fp32 is exact.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float (&f)[4])
{
    uint32_t lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}\n"
        : "=r"(lo), "=r"(hi) : "r"(w));
    const __half2 a = *reinterpret_cast<const __half2 *>(&lo), b = *reinterpret_cast<const __half2 *>(&hi);
    const float2 fa = __half22float2(a), fb = __half22float2(b);
    f[0] = fa.x;
    f[1] = fa.y;
    f[2] = fb.x;
    f[3] = fb.y;
}

__device__ __forceinline__ int32_t clamp_len(const KParams &kp, int64_t v, int64_t cap)
{
    if (v < 0 || v > cap) {
        set_status(kp, SFM_STATUS_BAD_LENGTH);
        v = v < 0 ? 0 : cap;
    }
    return (int32_t)v;
}

__device__ inline Tok token_info(const KParams &kp, int t)
{
    Tok k;
    int32_t qcap;
    if (kp.layout_q == SFM_LAYOUT_BSND) {
        k.b = (int)fdiv((uint32_t)t, kp.q_s_div);
        k.i = t - k.b * kp.q_s;
        qcap = kp.q_s;
    } else {
        int lo = 0, hi = kp.batch - 1;          // largest b with cu_q[b] <= t
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (__ldg(kp.cu_q + mid) <= t) lo = mid; else hi = mid - 1;
        }
        k.b = lo;
        k.i = t - __ldg(kp.cu_q + lo);
        qcap = __ldg(kp.cu_q + lo + 1) - __ldg(kp.cu_q + lo);
    }
    const int b = k.b;
    k.q_len = kp.used_q ? clamp_len(kp, __ldg(kp.used_q + b), qcap) : qcap;

    int64_t cap;
    int64_t kv;
    if (kp.layout_kv == SFM_LAYOUT_BSND) cap = kp.ori_s;
    else if (kp.layout_kv == SFM_LAYOUT_TND) cap = __ldg(kp.cu_ori + b + 1) - __ldg(kp.cu_ori + b);
    else cap = kp.ori_max;      // paged: the declared max length (the planner sees no block table)
    kv = kp.used_ori ? (int64_t)__ldg(kp.used_ori + b) : cap;
    k.kv_len = clamp_len(kp, kv, cap);

    k.cmp_len = 0;
    if (kp.has_cmp) {
        if (kp.layout_kv == SFM_LAYOUT_BSND) cap = kp.cmp_s;
        else if (kp.layout_kv == SFM_LAYOUT_TND) cap = __ldg(kp.cu_cmp + b + 1) - __ldg(kp.cu_cmp + b);
        else cap = kp.cmp_max;
        int64_t c = kp.used_cmp ? (int64_t)__ldg(kp.used_cmp + b) : cap;
        k.cmp_len = clamp_len(kp, c, cap);
    }
    const int64_t r = kp.residual ? (int64_t)__ldg(kp.residual + b) : 0;
    k.p = k.kv_len - k.q_len + k.i;
    const int64_t pc = (int64_t)k.cmp_len * kp.cmp_ratio + r - k.q_len + k.i;
    k.p_cmp = (int32_t)pc;
    k.valid = (t < kp.T) && (k.i < k.q_len);

    // ori window [lo, hi]
    int64_t lo = 0, hi = (int64_t)k.kv_len - 1, p = k.p;
    if (kp.ori_mask_mode == 3) {
        if (p < hi) hi = p;
    } else if (kp.ori_mask_mode == 4) {
        if (kp.win_left >= 0 && p - kp.win_left > lo) lo = p - kp.win_left;
        if (kp.win_right >= 0 && p + kp.win_right < hi) hi = p + kp.win_right;
    }
    if (hi < lo) { lo = 0; hi = -1; }
    k.lo = (int32_t)lo;
    k.hi = (int32_t)hi;

    k.n_ori = 0;
    k.n_cmp = 0;
    if (k.valid && k.kv_len > 0) k.n_ori = kp.ori_topk > 0 ? kp.ori_topk << kp.sbs_log2 : (int32_t)(hi - lo + 1);
    if (k.valid && kp.has_cmp && k.cmp_len > 0) {
        if (kp.cmp_topk > 0) {
            k.n_cmp = kp.cmp_topk;
        } else if (kp.cmp_mask_mode == 3) {
            // slots j with (j+1)*ratio <= pc+1
            int64_t v = (pc + 1) < 0 ? 0 : (pc + 1) <= 0xffffffffll ? (int64_t)fdiv((uint32_t)(pc + 1), kp.ratio_div)
                                                                    : (pc + 1) / kp.cmp_ratio;
            k.n_cmp = (int32_t)(v < k.cmp_len ? v : k.cmp_len);
        } else {
            k.n_cmp = k.cmp_len;
        }
    }
    return k;
}

// metadata sanity check shared by the kernels that consume a plan
__device__ __forceinline__ bool meta_ok(const KParams &kp)
{
    const int32_t *m = kp.meta;
    return m[H_MAGIC] == kMetaMagic && m[H_FPRINT] == kp.fingerprint && m[H_TOKENS] == kp.T &&
           m[H_WORKERS] == kp.G && m[H_SPLIT] == kp.split_rows && m[H_PATH] == kp.path && m[H_FLAGS] == 0;
}

// first split of query row t / the row owning split w (binary search)
__device__ __forceinline__ int split_owner(const int32_t *sp, int T, int w)
{
    int lo = 0, hi = T - 1;     // largest t with sp[t] <= w
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (sp[mid] <= w) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ----------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched with
// launch_dependent() may start while its predecessor in the stream is still
// running; it must call grid_dependency_wait() before it reads anything the
// predecessor writes.  grid_launch_dependents() lets the next kernel start.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ----------------------------------------------------------------------------
// host-side launchers (one per translation unit)
// ----------------------------------------------------------------------------
cudaError_t launch_plan(const KParams &kp, cudaStream_t st);
cudaError_t launch_attn_tc(const KParams &kp, cudaStream_t st);
cudaError_t launch_combine(const KParams &kp, cudaStream_t st);

}  // namespace sfm
