// sfm_host.cu -- the C-ABI entry points declared in include/sfm.h.
//
// Host-side validation follows the parameter tables of the "sparse_flash_mla"
// doc (zh), 约束说明 / 参数组约束: kv_n = 1, d = 512, q_n in 1..128, the
// SWA / CSA / HCA attribute combinations of 计算模式参数组, the layout pairs of
// the layout匹配关系表 and the paged block-size rule.  Tensor values are not
// read here (the pages leave their validity to the caller); the kernels
// bounds-check them instead.
#include <math.h>
#include <string.h>

#include "sfm_internal.cuh"

namespace sfm {
namespace {

inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

constexpr int64_t kMaxPoolRows = ((int64_t)1 << 31) - 2;

int64_t num_tokens(const sfm_params &p)
{
    return p.layout_q == SFM_LAYOUT_BSND ? (int64_t)p.batch_size * p.max_seqlen_q : (int64_t)p.total_q;
}

// tokens per ori_sparse_indices entry (0 means the token-wise default)
int sparse_block(const sfm_params &p) { return p.sparse_block_size == 0 ? 1 : p.sparse_block_size; }

bool is_packed(const sfm_params &p)
{
    return p.kv_format == SFM_KV_INT8_PACKED || p.kv_format == SFM_KV_FP8_PACKED;
}

int64_t row_bytes(const sfm_params &p)
{
    if (is_packed(p)) return 512 + 2 * (int64_t)p.rope_head_dim + 16;
    return 2 * (int64_t)p.head_dim;
}

int validate_params(const sfm_params *pp)
{
    if (!pp) return SFM_ERR_INVALID_ARG;
    const sfm_params &p = *pp;
    if (p.num_heads_q < 1 || p.num_heads_q > 128) return SFM_ERR_INVALID_ARG;
    if (p.num_heads_kv != 1) return SFM_ERR_UNSUPPORTED;
    if (p.head_dim != 512) return SFM_ERR_UNSUPPORTED;
    if (p.dtype != SFM_DTYPE_BF16 && p.dtype != SFM_DTYPE_FP16) return SFM_ERR_INVALID_ARG;
    if (p.kv_format == SFM_KV_PLAIN) {
        if (p.rope_head_dim != 0) return SFM_ERR_INVALID_ARG;
    } else if (is_packed(p)) {
        if (p.rope_head_dim != 0 && p.rope_head_dim != 64) return SFM_ERR_INVALID_ARG;
    } else {
        return SFM_ERR_INVALID_ARG;
    }
    if (p.layout_q != SFM_LAYOUT_BSND && p.layout_q != SFM_LAYOUT_TND) return SFM_ERR_LAYOUT;
    if (p.layout_kv != SFM_LAYOUT_BSND && p.layout_kv != SFM_LAYOUT_TND && p.layout_kv != SFM_LAYOUT_PAGED)
        return SFM_ERR_LAYOUT;
    if (p.layout_kv != SFM_LAYOUT_PAGED && p.layout_kv != p.layout_q) return SFM_ERR_LAYOUT;
    if (p.batch_size <= 0 || p.max_seqlen_q <= 0) return SFM_ERR_INVALID_ARG;
    if (p.layout_q == SFM_LAYOUT_TND && p.total_q <= 0) return SFM_ERR_INVALID_ARG;
    if (num_tokens(p) > (int64_t)INT32_MAX / 2) return SFM_ERR_INVALID_ARG;
    if (p.has_ori_kv != 1) return SFM_ERR_UNSUPPORTED;
    if (p.has_cmp_kv != 0 && p.has_cmp_kv != 1) return SFM_ERR_INVALID_ARG;
    if (p.ori_mask_mode != 0 && p.ori_mask_mode != 3 && p.ori_mask_mode != 4) return SFM_ERR_INVALID_ARG;
    if (p.cmp_mask_mode != 0 && p.cmp_mask_mode != 3) return SFM_ERR_INVALID_ARG;
    if (p.ori_win_left < -1 || p.ori_win_right < -1) return SFM_ERR_INVALID_ARG;
    if (p.ori_topk < 0 || p.cmp_topk < 0) return SFM_ERR_INVALID_ARG;
    {
        const int sbs = sparse_block(p);
        if (sbs < 1 || sbs > 128 || (sbs & (sbs - 1))) return SFM_ERR_INVALID_ARG;
        if (sbs > 1 && p.ori_topk == 0) return SFM_ERR_INVALID_ARG;
        if (sbs > 1 && p.layout_kv == SFM_LAYOUT_PAGED && p.ori_block_size % sbs) return SFM_ERR_LAYOUT;
        if ((int64_t)p.ori_topk * sbs > INT32_MAX) return SFM_ERR_INVALID_ARG;
    }
    if (p.max_seqlen_ori_kv <= 0) return SFM_ERR_INVALID_ARG;
    if (!p.has_cmp_kv) {
        if (p.cmp_topk != 0 || p.cmp_ratio != 1) return SFM_ERR_INVALID_ARG;    // SWA: cmp_topk 0, cmp_ratio 1
    } else {
        if (p.cmp_ratio <= 0) return SFM_ERR_INVALID_ARG;
        if (p.max_seqlen_cmp_kv < 0) return SFM_ERR_INVALID_ARG;
    }
    if (p.layout_kv == SFM_LAYOUT_PAGED) {
        if (p.ori_block_size < 16 || p.ori_block_size > 1024 || p.ori_block_size % 16) return SFM_ERR_LAYOUT;
        if (p.has_cmp_kv && (p.cmp_block_size < 16 || p.cmp_block_size > 1024 || p.cmp_block_size % 16))
            return SFM_ERR_LAYOUT;
    }
    if (p.return_lse != 0 && p.return_lse != 1) return SFM_ERR_INVALID_ARG;
    if (p.kernel_hint < 0 || p.kernel_hint > 2) return SFM_ERR_INVALID_ARG;
    if (p.kernel_hint == 1) return SFM_ERR_UNSUPPORTED;   // the CUDA-core kernel is retired
    if (p.split_policy != SFM_SPLIT_BATCH_INVARIANT && p.split_policy != SFM_SPLIT_OCCUPANCY)
        return SFM_ERR_INVALID_ARG;
    return SFM_OK;
}

// Required length tensors (both calls): 参数组约束 / Paged Attention参数组.
int validate_lengths(const sfm_params &p, const sfm_tensors *t)
{
    if (!t) return SFM_ERR_INVALID_ARG;
    if (p.layout_q == SFM_LAYOUT_TND && !t->cu_seqlens_q) return SFM_ERR_INVALID_ARG;
    if (p.layout_kv == SFM_LAYOUT_TND) {
        if (!t->cu_seqlens_ori_kv) return SFM_ERR_INVALID_ARG;
        if (p.has_cmp_kv && !t->cu_seqlens_cmp_kv) return SFM_ERR_INVALID_ARG;
    }
    if (p.layout_kv == SFM_LAYOUT_PAGED) {
        if (!t->seqused_ori_kv) return SFM_ERR_INVALID_ARG;
        if (p.has_cmp_kv && !t->seqused_cmp_kv) return SFM_ERR_INVALID_ARG;
    }
    if (p.has_cmp_kv && p.cmp_mask_mode == 3 && !t->cmp_residual_kv) return SFM_ERR_INVALID_ARG;
    return SFM_OK;
}

int num_sms(int *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SFM_ERR_CUDA;
    if (cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SFM_ERR_CUDA;
    return SFM_OK;
}

// Upper bound of attended positions of one query row.
int64_t max_positions(const sfm_params &p)
{
    int64_t ori;
    if (p.ori_topk > 0) {
        ori = (int64_t)p.ori_topk * sparse_block(p);
    } else {
        ori = p.max_seqlen_ori_kv;
        if (p.ori_mask_mode == 4 && p.ori_win_left >= 0 && p.ori_win_right >= 0) {
            const int64_t w = (int64_t)p.ori_win_left + p.ori_win_right + 1;
            if (w < ori) ori = w;
        }
    }
    int64_t cmp = 0;
    if (p.has_cmp_kv) cmp = p.cmp_topk > 0 ? p.cmp_topk : p.max_seqlen_cmp_kv;
    return ori + cmp;
}

struct Plan {
    int32_t path, G, split_rows;
    int64_t T, max_splits_per_token;
};

int head_groups(const sfm_params &p) { return (p.num_heads_q + 63) / 64; }

// Occupancy policy: when the batch-invariant plan leaves CTAs without a work
// unit, re-cut every row into k chunks, k chosen by a cost model of the step,
// in half-tiles.  A CTA runs ceil(units / G) units one after the other; a
// unit costs its 32-row tiles, at least three (shorter units hide behind the
// kernel's start-up), plus one tile of epilogue; splitting a row adds the
// combine launch (one tile) and half a tile per chunk of the row to merge.
// Fitted to decode steps timed on one GPU with 64 and 128 heads at 4 to 16
// rows.  The model is evaluated on the params' upper bound of a row's
// positions, so the plan still does not depend on the lengths.
void occupancy_split(const sfm_params &p, Plan *pl, int64_t mp)
{
    const int64_t hg = head_groups(p);
    const int64_t units_inv = pl->T * hg * pl->max_splits_per_token;
    if (pl->T <= 0 || mp <= 0 || units_inv >= pl->G) return;
    const int64_t tiles = (mp + 31) / 32;
    auto cost = [&](int64_t k) {
        const int64_t waves = (pl->T * hg * k + pl->G - 1) / pl->G;
        const int64_t per_unit = (tiles + k - 1) / k;
        return 2 * waves * ((per_unit > 3 ? per_unit : 3) + 1) + (k > 1 ? 2 + k : 0);
    };
    int64_t best_k = pl->max_splits_per_token, best = cost(best_k);
    const int64_t kmax = tiles < pl->G ? tiles : pl->G;     // more chunks than CTAs only adds waves
    for (int64_t k = best_k + 1; k <= kmax; ++k) {
        const int64_t c = cost(k);
        if (c < best) best = c, best_k = k;
    }
    if (best_k == pl->max_splits_per_token) return;
    const int64_t rows = 32 * ((tiles + best_k - 1) / best_k);
    pl->split_rows = (int32_t)rows;
    pl->max_splits_per_token = (mp + rows - 1) / rows;
}

// Split size: decode-shaped calls (few query rows per sequence) cut each
// row's attended positions into fixed chunks so the SMs share the work;
// prefill-shaped calls have enough rows and keep one split per row.  The
// choice depends on the params only, never on the lengths.
int make_plan(const sfm_params &p, Plan *pl)
{
    int sms = 0;
    int rc = num_sms(&sms);
    if (rc) return rc;
    // One attention kernel (tensor cores) covers every supported shape: plain
    // bf16 / fp16 rows and packed int8 / fp8 rows with or without the rope
    // part; more than 64 heads run as two work units (head groups) per split.
    pl->path = PATH_TC;
    // The kernel keeps one CTA per SM and leaves one SM to the planner kernel
    // that runs just before it (the attention kernel's set-up overlaps the
    // planner; a CTA placed on the planner's SM would start late).
    pl->G = sms > 1 ? sms - 1 : sms;
    pl->T = num_tokens(p);
    const bool decode_like = p.max_seqlen_q <= 16;
    // Tensor-core tiles are 32 rows.  The split size is a constant of the
    // path and head count (a row's splits never depend on the batch), chosen
    // so that the decode workloads' units about fill the SMs once: up to 64
    // heads, splits of 5 tiles (CSA decode: 32 rows x 4 splits = 128 units);
    // 128 heads, each split is two work units, splits of 64 tiles (HCA and
    // packed decode, 64 rows of at most 2048 positions: one split per row,
    // 128 units, no partials to merge).  Measured on one GPU against
    // 768-row splits: HCA decode step -13 %, packed decode -8 %.  Batches of
    // fewer rows leave SMs idle unless the params ask for the occupancy
    // policy, which re-cuts the rows so the units fill the SMs.
    const int split = p.num_heads_q > 64 ? 2048 : 160;
    pl->split_rows = decode_like ? split : (1 << 30);
    const int64_t mp = max_positions(p);
    pl->max_splits_per_token = decode_like ? (mp + pl->split_rows - 1) / pl->split_rows : 1;
    if (p.split_policy == SFM_SPLIT_OCCUPANCY) occupancy_split(p, pl, mp);
    return SFM_OK;
}

uint32_t fingerprint(const sfm_params &p, const Plan &pl)
{
    uint32_t h = 2166136261u;
    auto mix = [&](uint32_t v) {
        for (int i = 0; i < 4; ++i) {
            h ^= (v >> (8 * i)) & 0xffu;
            h *= 16777619u;
        }
    };
    const int32_t *f = reinterpret_cast<const int32_t *>(&p);
    for (size_t i = 0; i < sizeof(sfm_params) / sizeof(int32_t); ++i) mix((uint32_t)f[i]);
    mix((uint32_t)pl.path);
    mix((uint32_t)pl.G);
    mix((uint32_t)pl.split_rows);
    mix((uint32_t)pl.T);
    return h;
}

size_t ws_lse_offset(const sfm_params &p, int64_t cap)
{
    size_t o = (size_t)cap * p.num_heads_q * 512 * sizeof(uint16_t);
    return (o + 255) & ~(size_t)255;
}


size_t workspace_bytes_for(const sfm_params &p, const Plan &pl)
{
    if (pl.max_splits_per_token <= 1) return 0;
    const int64_t cap = pl.T * pl.max_splits_per_token;
    return ws_lse_offset(p, cap) + (size_t)cap * p.num_heads_q * sizeof(float);
}

void fill_common(KParams &kp, const sfm_params &p, const Plan &pl)
{
    memset(&kp, 0, sizeof(kp));
    kp.q_n = p.num_heads_q;
    kp.d_v = 512;
    kp.rope = is_packed(p) ? p.rope_head_dim : 0;
    kp.d_qk = 512 + kp.rope;
    kp.batch = p.batch_size;
    kp.q_s = p.max_seqlen_q;
    kp.T = (int32_t)pl.T;
    kp.ori_s = p.layout_kv == SFM_LAYOUT_BSND ? p.max_seqlen_ori_kv : 0;
    kp.cmp_s = p.layout_kv == SFM_LAYOUT_BSND ? p.max_seqlen_cmp_kv : 0;
    kp.ori_max = p.max_seqlen_ori_kv;
    kp.cmp_max = p.max_seqlen_cmp_kv;
    kp.layout_q = p.layout_q;
    kp.layout_kv = p.layout_kv;
    kp.dtype = p.dtype;
    kp.packed = is_packed(p);
    kp.kv_fp8 = p.kv_format == SFM_KV_FP8_PACKED;
    kp.ori_bs = p.ori_block_size;
    kp.cmp_bs = p.cmp_block_size;
    kp.q_s_div = make_fastdiv(kp.q_s > 0 ? (uint32_t)kp.q_s : 1u);
    kp.ratio_div = make_fastdiv(p.cmp_ratio > 0 ? (uint32_t)p.cmp_ratio : 1u);
    kp.split_div = make_fastdiv(pl.split_rows > 0 ? (uint32_t)pl.split_rows : 1u);
    kp.ori_bs_div = make_fastdiv(p.ori_block_size > 0 ? (uint32_t)p.ori_block_size : 1u);
    kp.cmp_bs_div = make_fastdiv(p.cmp_block_size > 0 ? (uint32_t)p.cmp_block_size : 1u);
    kp.ori_topk = p.ori_topk;
    {
        int l = 0;
        while ((1 << l) < sparse_block(p)) ++l;
        kp.sbs_log2 = l;
    }
    kp.cmp_topk = p.has_cmp_kv ? p.cmp_topk : 0;
    kp.cmp_ratio = p.cmp_ratio;
    kp.ori_mask_mode = p.ori_mask_mode;
    kp.cmp_mask_mode = p.cmp_mask_mode;
    kp.win_left = p.ori_win_left;
    kp.win_right = p.ori_win_right;
    kp.has_cmp = p.has_cmp_kv;
    kp.return_lse = p.return_lse;
    kp.G = pl.G;
    kp.split_rows = pl.split_rows;
    kp.path = pl.path;
    kp.fingerprint = (int32_t)fingerprint(p, pl);
    kp.head_groups = head_groups(p);
    kp.wcap = pl.T * pl.max_splits_per_token;
    kp.max_splits = (int32_t)(pl.max_splits_per_token < INT32_MAX ? pl.max_splits_per_token : INT32_MAX);
}

void fill_lengths(KParams &kp, const sfm_tensors &t)
{
    kp.cu_q = t.cu_seqlens_q;
    kp.cu_ori = t.cu_seqlens_ori_kv;
    kp.cu_cmp = t.cu_seqlens_cmp_kv;
    kp.used_q = t.seqused_q;
    kp.used_ori = t.seqused_ori_kv;
    kp.used_cmp = t.seqused_cmp_kv;
    kp.residual = t.cmp_residual_kv;
    kp.ori_bt_stride = t.ori_block_table_stride;
    kp.cmp_bt_stride = t.cmp_block_table_stride;
}

int validate_tensors(const sfm_params &p, const sfm_tensors *t)
{
    int rc = validate_lengths(p, t);
    if (rc) return rc;
    if (!t->q || !t->ori_kv) return SFM_ERR_INVALID_ARG;
    if (!aligned16(t->q) || !aligned16(t->ori_kv)) return SFM_ERR_LAYOUT;
    const int64_t rb = row_bytes(p);
    if (t->ori_row_stride < rb || t->ori_row_stride % 16 || t->ori_rows <= 0) return SFM_ERR_LAYOUT;
    // the kernel names a KV row with 31 bits (the top bit tells the pools apart)
    if (t->ori_rows > kMaxPoolRows || (p.has_cmp_kv && t->cmp_rows > kMaxPoolRows)) return SFM_ERR_UNSUPPORTED;
    if (p.has_cmp_kv) {
        if (!t->cmp_kv) return SFM_ERR_INVALID_ARG;
        if (!aligned16(t->cmp_kv)) return SFM_ERR_LAYOUT;
        if (t->cmp_row_stride < rb || t->cmp_row_stride % 16 || t->cmp_rows <= 0) return SFM_ERR_LAYOUT;
    } else if (t->cmp_kv || t->cmp_sparse_indices || t->cmp_block_table) {
        return SFM_ERR_INVALID_ARG;   // SWA takes no cmp tensors (计算模式参数组)
    }
    if (p.cmp_topk > 0 && !t->cmp_sparse_indices) return SFM_ERR_INVALID_ARG;
    if (p.has_cmp_kv && p.cmp_topk == 0 && t->cmp_sparse_indices) return SFM_ERR_INVALID_ARG;  // HCA
    if (p.ori_topk > 0 && !t->ori_sparse_indices) return SFM_ERR_INVALID_ARG;
    if (p.ori_topk == 0 && t->ori_sparse_indices) return SFM_ERR_INVALID_ARG;
    if (p.layout_kv == SFM_LAYOUT_PAGED) {
        if (!t->ori_block_table || t->ori_block_table_stride <= 0) return SFM_ERR_INVALID_ARG;
        if (p.has_cmp_kv && (!t->cmp_block_table || t->cmp_block_table_stride <= 0)) return SFM_ERR_INVALID_ARG;
    } else if (t->ori_block_table || t->cmp_block_table) {
        return SFM_ERR_INVALID_ARG;
    }
    return SFM_OK;
}

cudaEvent_t g_prof_begin = nullptr, g_prof_end = nullptr;

// sfm_forward() with an optional attended-row dump (sfm_debug_attended):
// validation, the kernel parameter block, the attention kernel and, when a
// row can have more than one split, the combine kernel.
int enqueue_forward(const sfm_params *params, const sfm_tensors *in, const int32_t *metadata, size_t metadata_n,
                    float softmax_scale, void *out, float *lse, void *workspace, size_t workspace_bytes,
                    int32_t *status, sfm_stream_t stream, int32_t *dbg_rows, int64_t dbg_cap, int32_t *dbg_counts)
{
    int rc = validate_params(params);
    if (rc) return rc;
    const sfm_params &p = *params;
    rc = validate_tensors(p, in);
    if (rc) return rc;
    if (!out || !metadata || !isfinite(softmax_scale)) return SFM_ERR_INVALID_ARG;
    if ((uintptr_t)metadata & 15u) return SFM_ERR_LAYOUT;
    if (!aligned16(out)) return SFM_ERR_LAYOUT;
    if (p.return_lse ? !lse : lse != nullptr) return SFM_ERR_INVALID_ARG;
    Plan pl;
    rc = make_plan(p, &pl);
    if (rc) return rc;
    if (metadata_n < (size_t)meta_words(pl.G, (int)pl.T, pl.T * pl.max_splits_per_token)) return SFM_ERR_WORKSPACE;
    const size_t need = workspace_bytes_for(p, pl);
    if (workspace_bytes < need || (need && !workspace) || ((uintptr_t)workspace & 255u)) return SFM_ERR_WORKSPACE;

    KParams kp;
    fill_common(kp, p, pl);
    fill_lengths(kp, *in);
    kp.scale = softmax_scale;
    kp.scale_log2 = softmax_scale * 1.4426950408889634f;
    kp.q = in->q;
    kp.ori_kv = static_cast<const uint8_t *>(in->ori_kv);
    kp.cmp_kv = static_cast<const uint8_t *>(in->cmp_kv);
    kp.ori_row_stride = in->ori_row_stride;
    kp.cmp_row_stride = in->cmp_row_stride;
    kp.ori_rows = in->ori_rows;
    kp.cmp_rows = in->cmp_rows;
    kp.ori_idx = in->ori_sparse_indices;
    kp.cmp_idx = in->cmp_sparse_indices;
    kp.ori_bt = in->ori_block_table;
    kp.cmp_bt = in->cmp_block_table;
    kp.sinks = in->sinks;
    kp.meta = metadata;
    kp.out = out;
    kp.lse = lse;
    kp.status = status;
    kp.dbg_rows = dbg_rows;
    kp.dbg_cap = dbg_cap;
    kp.dbg_counts = dbg_counts;
    if (need) {
        const int64_t cap = pl.T * pl.max_splits_per_token;
        kp.ws_capacity_splits = cap;
        kp.ws_o = static_cast<uint16_t *>(workspace);
        kp.ws_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + ws_lse_offset(p, cap));
    }
    cudaStream_t st = (cudaStream_t)stream;
    if (g_prof_begin && cudaEventRecord(g_prof_begin, st) != cudaSuccess) return SFM_ERR_CUDA;
    if (launch_attn_tc(kp, st) != cudaSuccess) return SFM_ERR_CUDA;
    if (g_prof_end && cudaEventRecord(g_prof_end, st) != cudaSuccess) return SFM_ERR_CUDA;
    // at most one split per row: the attention kernel finishes every row
    // itself (rows without a split included), so there is nothing to merge
    if (pl.max_splits_per_token > 1 && launch_combine(kp, st) != cudaSuccess) return SFM_ERR_CUDA;
    return SFM_OK;
}


}  // namespace
}  // namespace sfm

using namespace sfm;

extern "C" {

int sfm_abi_version(void) { return SFM_ABI_VERSION; }

int sfm_set_profile_events(void *begin, void *end)
{
    if ((begin == nullptr) != (end == nullptr)) return SFM_ERR_INVALID_ARG;
    g_prof_begin = (cudaEvent_t)begin;
    g_prof_end = (cudaEvent_t)end;
    return SFM_OK;
}

const char *sfm_error_string(int code)
{
    switch (code) {
    case SFM_OK: return "ok";
    case SFM_ERR_INVALID_ARG: return "invalid argument";
    case SFM_ERR_UNSUPPORTED: return "unsupported combination";
    case SFM_ERR_LAYOUT: return "layout, stride or alignment rule broken";
    case SFM_ERR_WORKSPACE: return "workspace or metadata buffer too small";
    case SFM_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown error";
    }
}

int sfm_metadata_size(const sfm_params *params, size_t *n_int32)
{
    int rc = validate_params(params);
    if (rc) return rc;
    if (!n_int32) return SFM_ERR_INVALID_ARG;
    Plan pl;
    rc = make_plan(*params, &pl);
    if (rc) return rc;
    *n_int32 = (size_t)meta_words(pl.G, (int)pl.T, pl.T * pl.max_splits_per_token);
    return SFM_OK;
}

int sfm_workspace_size(const sfm_params *params, size_t *bytes)
{
    int rc = validate_params(params);
    if (rc) return rc;
    if (!bytes) return SFM_ERR_INVALID_ARG;
    Plan pl;
    rc = make_plan(*params, &pl);
    if (rc) return rc;
    *bytes = workspace_bytes_for(*params, pl);
    return SFM_OK;
}

int sfm_metadata(const sfm_params *params, const sfm_tensors *lengths, int32_t *metadata, size_t metadata_n,
                 sfm_stream_t stream)
{
    int rc = validate_params(params);
    if (rc) return rc;
    rc = validate_lengths(*params, lengths);
    if (rc) return rc;
    if (!metadata) return SFM_ERR_INVALID_ARG;
    if ((uintptr_t)metadata & 15u) return SFM_ERR_LAYOUT;
    Plan pl;
    rc = make_plan(*params, &pl);
    if (rc) return rc;
    if (metadata_n < (size_t)meta_words(pl.G, (int)pl.T, pl.T * pl.max_splits_per_token)) return SFM_ERR_WORKSPACE;
    KParams kp;
    fill_common(kp, *params, pl);
    fill_lengths(kp, *lengths);
    kp.meta_w = metadata;
    kp.meta = metadata;
    return launch_plan(kp, (cudaStream_t)stream) == cudaSuccess ? SFM_OK : SFM_ERR_CUDA;
}

int sfm_forward(const sfm_params *params, const sfm_tensors *in, const int32_t *metadata, size_t metadata_n,
                float softmax_scale, void *out, float *lse, void *workspace, size_t workspace_bytes,
                int32_t *status, sfm_stream_t stream)
{
    return enqueue_forward(params, in, metadata, metadata_n, softmax_scale, out, lse, workspace, workspace_bytes,
                           status, stream, nullptr, 0, nullptr);
}

int sfm_debug_attended(const sfm_params *params, const sfm_tensors *in, const int32_t *metadata,
                       size_t metadata_n, float softmax_scale, void *out, float *lse, void *workspace,
                       size_t workspace_bytes, int32_t *rows, int64_t cap, int32_t *counts, int32_t *status,
                       sfm_stream_t stream)
{
    if (!rows || !counts || cap <= 0) return SFM_ERR_INVALID_ARG;
    return enqueue_forward(params, in, metadata, metadata_n, softmax_scale, out, lse, workspace, workspace_bytes,
                           status, stream, rows, cap, counts);
}

}  // extern "C"
