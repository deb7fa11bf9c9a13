/*
 * sfm.h -- C-ABI of the GB300 (sm_103a) sparse shared-KV MLA attention library.
 *
 * The library computes, for every query row and head,
 *
 *     O   = softmax(Q . K~^T . softmax_scale) . V~,      K~ = V~,  kv_n = 1, d = 512
 *     LSE = log sum exp(S - max S) + max S,              S  = Q K~^T . softmax_scale
 *
 * ("sparse_flash_mla" doc (zh), 功能说明 / 计算公式; the English doc's
 * "Function" section and the SparseAttnSharedkv README give the same formula),
 * where the attended rows K~ of one query row are the union of two sources:
 *
 *   ori_kv  a sliding window [p - ori_win_left, p + ori_win_right] cut to
 *           [0, kv_len) (ori_mask_mode 4), the causal prefix [0, p] (mode 3)
 *           or all rows (mode 0); -1 for a window side means unbounded.  With
 *           ori_topk > 0 the ori source is instead the valid entries of
 *           ori_sparse_indices inside that set (the token-wise sparse form of
 *           the kv_quant_sparse_flash_attention guide, 属性参数:
 *           sparse_block_size = 1, sparse_mode 0 / 3).
 *   cmp_kv  compressed rows; slot j is visible iff (j + 1) * cmp_ratio <=
 *           p_cmp + 1 (cmp_mask_mode 3) or always (mode 0).  HCA (cmp_topk = 0)
 *           attends every visible slot; CSA (cmp_topk > 0) the valid entries of
 *           cmp_sparse_indices (-1 = invalid, valid entries first).
 *
 * with p = kv_len - q_len + i for query row i (right-down alignment, CP切分示例)
 * and p_cmp = cmp_len * cmp_ratio + cmp_residual_kv - q_len + i (参数说明: the
 * residual recovers the cmp-side mask length; equal to p under the documented
 * contract).
 * Optional per-head fp32 sinks add exp(sink - m) to the softmax denominator
 * only; the LSE excludes them.  An empty attended set gives O = 0 and
 * LSE = -inf.
 *
 * Two-call contract ("sparse_flash_mla" doc, 功能说明 and 函数原型): first
 * sfm_metadata() builds the split-KV work plan on the device, then
 * sfm_forward() consumes it.  Both calls take the SAME sfm_params; the plan
 * carries a fingerprint of them and sfm_forward() refuses (status bit
 * SFM_STATUS_METADATA_MISMATCH, outputs zeroed) a plan made for other params.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers of the current CUDA device,
 *     except the sfm_params / sfm_tensors structs themselves, which live in
 *     host memory and are read during the call only.
 *   - The caller owns every buffer (inputs, outputs, metadata, workspace,
 *     status).  The library allocates nothing on the device and never
 *     synchronises: work is enqueued on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and completes in stream order.
 *   - Return value: SFM_OK or an sfm_error code for a host-side rejection
 *     (nothing is enqueued then).  Tensor VALUES are checked on the device
 *     (indices, block ids, lengths); a bad value never faults: the row is
 *     skipped and a bit is OR-ed into *status (if status != NULL).
 *   - Element types: q / out / plain KV rows are bf16 or fp16 (sfm_params.dtype).
 *     Packed KV rows are bytes (see SFM_KV_INT8_PACKED).  Indices, lengths and
 *     block tables are int32; sinks and LSE are fp32.
 */
#ifndef SFM_H
#define SFM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SFM_ABI_VERSION 4

/* A cudaStream_t, passed as an untyped pointer so this header needs no CUDA headers. */
typedef void *sfm_stream_t;

/* Layouts ("sparse_flash_mla" doc, 参数说明: layout_q / layout_kv and the
 * layout匹配关系表).  SFM_LAYOUT_PAGED is the pages' PA_BBND / PA_BSND / PA_ND:
 * (blocks, block_size, 1, row) addressed through a block table. */
enum sfm_layout { SFM_LAYOUT_BSND = 0, SFM_LAYOUT_TND = 1, SFM_LAYOUT_PAGED = 2 };

enum sfm_dtype { SFM_DTYPE_BF16 = 0, SFM_DTYPE_FP16 = 1 };

/* KV row formats.
 *   SFM_KV_PLAIN        512 bf16/fp16 values per row (1024 bytes).
 *   SFM_KV_INT8_PACKED  kv_quant_sparse_flash_attention guide, "A2/A3 C8 NoPE"
 *                       table: bytes [0,512) int8 NoPE, then rope_head_dim
 *                       (0 or 64) bf16/fp16 rope values, then 4 fp32 scales,
 *                       one per 128-dim tile: 656 bytes (rope 64) or 528 bytes
 *                       (rope 0).  K~[d] = int8[d] * scale[d / 128] for
 *                       d < 512, followed by the rope values; V~ = K~[0:512];
 *                       q has 512 + rope_head_dim dims, out has 512.
 *   SFM_KV_FP8_PACKED   the same guide, "Ascend 950 INT8/FP8 C8 NoPE" section:
 *                       the same 528 / 656-byte rows with the 512 NoPE bytes
 *                       FLOAT8_E4M3FN values (sign, 4 exponent bits biased by
 *                       7, 3 mantissa bits, no infinity, S.1111.111 = NaN):
 *                       K~[d] = e4m3(byte d) * scale[d / 128]. */
enum sfm_kv_format { SFM_KV_PLAIN = 0, SFM_KV_INT8_PACKED = 1, SFM_KV_FP8_PACKED = 2 };

/* How sfm_metadata sizes the split-KV chunks of a query row ("sparse_flash_mla"
 * doc, 确定性计算: deterministic results and batch invariance are the default).
 *   SFM_SPLIT_BATCH_INVARIANT  a row is cut into chunks whose size depends
 *       only on the head count and the query shape (max_seqlen_q): a row's O
 *       and LSE are bit for bit the same whatever other rows share the batch
 *       and however many there are.  Batches much smaller than one row per
 *       SM leave SMs idle (a 128-head row of 1152 positions is two work
 *       units, so 8 such rows keep 16 SMs busy).
 *   SFM_SPLIT_OCCUPANCY        where the batch-invariant plan has fewer work
 *       units than the kernel has CTAs, the chunk size is chosen from the
 *       number of query rows and the SM count as well, so the units fill the
 *       SMs; otherwise the plan is the batch-invariant one.  Results are
 *       deterministic for given params and lengths, but a row's rounding can
 *       change with the batch size. */
enum sfm_split_policy { SFM_SPLIT_BATCH_INVARIANT = 0, SFM_SPLIT_OCCUPANCY = 1 };

/* Host-side return codes. */
enum sfm_error {
    SFM_OK = 0,
    SFM_ERR_INVALID_ARG = 1,   /* a scalar out of range or a required pointer missing */
    SFM_ERR_UNSUPPORTED = 2,   /* a combination the library does not implement */
    SFM_ERR_LAYOUT = 3,        /* layout pair / stride / alignment rule broken */
    SFM_ERR_WORKSPACE = 4,     /* workspace or metadata buffer too small */
    SFM_ERR_CUDA = 5           /* a CUDA runtime call failed (launch, attribute query) */
};

/* Device status bits, OR-ed into *status by the kernels (never reset by the
 * library: the caller zeroes the word before a call it wants to inspect). */
#define SFM_STATUS_BAD_INDEX          0x01  /* an index entry >= its source length: skipped */
#define SFM_STATUS_BAD_BLOCK          0x02  /* a block id / row outside the cache: row skipped */
#define SFM_STATUS_BAD_LENGTH         0x04  /* a length above its tensor's capacity: clamped */
#define SFM_STATUS_METADATA_MISMATCH  0x08  /* metadata built for other params: outputs zeroed */
#define SFM_STATUS_WORKSPACE_OVERFLOW 0x10  /* plan needs more workspace than given: outputs zeroed */
#define SFM_STATUS_PLAN_OVERFLOW      0x20  /* plan larger than int32 counters allow: outputs zeroed */
#define SFM_STATUS_TIMEOUT            0x40  /* a kernel pipeline wait gave up (bounded spin): outputs undefined */

/* Scalar attributes shared by sfm_metadata() and sfm_forward().  Field names
 * follow the pages' parameter tables ("sparse_flash_mla" doc, 参数说明). */
typedef struct sfm_params {
    int32_t num_heads_q;       /* q_n, 1..128 */
    int32_t num_heads_kv;      /* kv_n, must be 1 */
    int32_t head_dim;          /* d of V~ and of the output, must be 512 */
    int32_t rope_head_dim;     /* packed rows only: 0 or 64 extra score dims; plain rows: 0 */
    int32_t batch_size;        /* b (> 0) */
    int32_t max_seqlen_q;      /* BSND: q_s, the q tensor's S dim; TND: max q length */
    int32_t total_q;           /* TND: q_t, rows of q; ignored for BSND */
    int32_t max_seqlen_ori_kv; /* BSND: S dim of ori_kv; TND / paged: max ori length */
    int32_t max_seqlen_cmp_kv; /* BSND: S dim of cmp_kv; TND / paged: max cmp length */
    int32_t ori_topk;          /* 0: window over ori_kv; > 0: ori_sparse_indices last dim */
    int32_t cmp_topk;          /* CSA: cmp_sparse_indices last dim (> 0); SWA / HCA: 0 */
    int32_t cmp_ratio;         /* SWA: 1; CSA / HCA: > 0 */
    int32_t ori_mask_mode;     /* 0 no mask, 3 right-down causal, 4 band (window) */
    int32_t cmp_mask_mode;     /* 0 no mask, 3 right-down causal */
    int32_t ori_win_left;      /* -1 (unbounded) or >= 0 past rows */
    int32_t ori_win_right;     /* -1 (unbounded) or >= 0 future rows */
    int32_t layout_q;          /* SFM_LAYOUT_BSND or SFM_LAYOUT_TND */
    int32_t layout_kv;         /* BSND, TND or PAGED; non-paged must equal layout_q */
    int32_t has_ori_kv;        /* must be 1 (every supported mode reads ori_kv) */
    int32_t has_cmp_kv;        /* 0: SWA; 1: CSA or HCA */
    int32_t dtype;             /* enum sfm_dtype of q, out and plain KV rows */
    int32_t kv_format;         /* enum sfm_kv_format */
    int32_t ori_block_size;    /* paged: rows per ori block, multiple of 16, <= 1024 */
    int32_t cmp_block_size;    /* paged with cmp_kv: rows per cmp block, multiple of 16, <= 1024 */
    int32_t return_lse;        /* 1: write LSE (fp32, token-major x q_n) */
    int32_t kernel_hint;       /* 0 or 2: the tensor-core kernel, which takes every supported
                                  shape (up to 128 heads, plain or packed rows; packed rows
                                  are computed with fp16 operands, bf16 q converted exactly,
                                  and rope-0 packed rows with a zero rope block, as if
                                  padded); 1 (the former CUDA-core kernel): SFM_ERR_UNSUPPORTED */
    int32_t sparse_block_size; /* ori_topk > 0 only: tokens per selected block; 0 or 1 =
                                  token-wise (each ori_sparse_indices entry is a token),
                                  2..128 (a power of two, dividing ori_block_size when
                                  paged) = block-wise: entry e selects tokens
                                  [e * sparse_block_size, (e + 1) * sparse_block_size),
                                  each still under the ori mask ([QSFA] / [SFA] 属性参数:
                                  sparse_block_size; the tokens of a block share the
                                  selection decision) */
    int32_t split_policy;      /* enum sfm_split_policy (0 = batch invariant) */
} sfm_params;

/* Device tensors of one call.  Shapes (row = one KV row of row_stride bytes):
 *   q                    BSND (b, q_s, q_n, dq) / TND (q_t, q_n, dq), dq = 512 + rope_head_dim
 *   ori_kv, cmp_kv       BSND (b, S, 1, row) / TND (t, 1, row) / PAGED (blocks, block_size, 1, row)
 *   ori_sparse_indices   (tokens, 1, ori_topk) int32, -1 = invalid (ori_topk > 0 only)
 *   cmp_sparse_indices   (tokens, 1, cmp_topk) int32, -1 = invalid (CSA only)
 *   *_block_table        (b, block_table_stride) int32 block ids (PAGED only)
 *   cu_seqlens_*         (b + 1) int32 prefix sums (TND)
 *   seqused_*            (b) int32 valid counts (seqused_ori_kv required for PAGED,
 *                        seqused_cmp_kv required for PAGED cmp_kv; each overrides the
 *                        length taken from the shape or cu_seqlens)
 *   cmp_residual_kv      (b) int32, 0 <= r < cmp_ratio (required when cmp_mask_mode = 3)
 *   sinks                (q_n) fp32 or NULL
 * Row strides are in bytes, >= the row size and a multiple of 16 (rows may be
 * padded between rows, 公共参数组); *_rows is the number of rows
 * the buffer holds (used to bounds-check every resolved row; at most
 * 2^31 - 2, SFM_ERR_UNSUPPORTED above).  Base pointers must be 16-byte
 * aligned. */
typedef struct sfm_tensors {
    const void *q;
    const void *ori_kv;
    int64_t ori_row_stride;
    int64_t ori_rows;
    const void *cmp_kv;
    int64_t cmp_row_stride;
    int64_t cmp_rows;
    const int32_t *ori_sparse_indices;
    const int32_t *cmp_sparse_indices;
    const int32_t *ori_block_table;
    int32_t ori_block_table_stride;
    const int32_t *cmp_block_table;
    int32_t cmp_block_table_stride;
    const int32_t *cu_seqlens_q;
    const int32_t *cu_seqlens_ori_kv;
    const int32_t *cu_seqlens_cmp_kv;
    const int32_t *seqused_q;
    const int32_t *seqused_ori_kv;
    const int32_t *seqused_cmp_kv;
    const int32_t *cmp_residual_kv;
    const float *sinks;
} sfm_tensors;

/* Number of int32 metadata elements sfm_metadata() writes for these params on
 * the current device (>= 1024, the pages' fixed size; larger when the number
 * of query rows or SMs needs more).  Host only, enqueues nothing. */
int sfm_metadata_size(const sfm_params *params, size_t *n_int32);

/* Device workspace bytes sfm_forward() needs for these params (split-KV
 * partial results; 0 when no query row is split).  Host only. */
int sfm_workspace_size(const sfm_params *params, size_t *bytes);

/* "sparse_flash_mla_metadata": enqueue the device-side planner.  It reads the
 * length tensors of `lengths` (cu_seqlens_*, seqused_*, cmp_residual_kv; other
 * fields are ignored and may be NULL), computes every query row's attended-row
 * count, cuts it into equal splits of at most a fixed size (by default a
 * function of that row's own count and the params only, so a row's result
 * does not depend on the rest of the batch: 确定性计算 / batch invariance;
 * see sfm_params.split_policy) and balances the splits over the SMs.
 * metadata: device int32[metadata_n], 16-byte aligned (SFM_ERR_LAYOUT
 * otherwise), metadata_n >= sfm_metadata_size().
 * Ordering: the planner is launched as a programmatic dependent of the kernel
 * before it in the stream and reads the length tensors before waiting for
 * that kernel to finish (it waits before writing `metadata`).  The kernels
 * of this library never write length tensors, copies and ordinary kernels
 * finish before it starts; a kernel of the caller's that triggers its
 * dependents early (griddepcontrol.launch_dependents) must not write the
 * length tensors after that trigger. */
int sfm_metadata(const sfm_params *params, const sfm_tensors *lengths, int32_t *metadata, size_t metadata_n,
                 sfm_stream_t stream);

/* "sparse_flash_mla": enqueue the attention for every query row.
 * out: device, q's token-major layout with 512 dims per head, dtype of q.
 * lse: device fp32 (tokens x q_n), required iff params->return_lse (NULL
 *      otherwise; replaces the pages' scalar placeholder).
 * workspace: device, >= sfm_workspace_size() bytes, 256-byte aligned.
 * status: device int32 or NULL (see SFM_STATUS_*).
 * Deterministic: the same inputs give bitwise the same outputs. */
int sfm_forward(const sfm_params *params, const sfm_tensors *inputs, const int32_t *metadata, size_t metadata_n,
                float softmax_scale, void *out, float *lse, void *workspace, size_t workspace_bytes,
                int32_t *status, sfm_stream_t stream);

/* Size of the fixed device workspace used by sfm_forward_noalloc(): 32 MiB. */
#define SFM_NOALLOC_WORKSPACE_BYTES ((size_t)32 << 20)

/* sfm_forward() for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists because some callers of
 * this library cannot call cudaMalloc when they run attention -- a graph
 * replayed with its memory frozen, a plug-in whose host framework owns every
 * allocation, a latency-critical path that must not allocate -- yet
 * sfm_forward() needs sfm_workspace_size() bytes of scratch for split-KV
 * partial results.
 *
 * Same arguments and behaviour as sfm_forward() minus the workspace: the
 * scratch comes from a fixed SFM_NOALLOC_WORKSPACE_BYTES device array that is
 * part of the library's module (every GPU that loads the module keeps it
 * until the process exits).  Nothing is allocated by this call: no cudaMalloc,
 * no cudaFree, no allocating library routine.  The caller still owns and
 * passes the inputs, the metadata, out, lse and status.
 *   - Returns SFM_ERR_WORKSPACE, enqueuing nothing, when these params need
 *     more than SFM_NOALLOC_WORKSPACE_BYTES of workspace.
 *   - Each call that needs scratch looks up the array's device address on
 *     the current device (cudaGetSymbolAddress, which allocates nothing); the
 *     first such call on a device loads the module, so make it before any
 *     stream capture.  The address is not cached, so calls made after a
 *     device reset use the array of the re-loaded module.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents: calls whose kernels may overlap on the GPU (unordered
 *     streams) race on it.  Every scratch word is written before it is read
 *     within a call, so nothing needs clearing between calls. */
int sfm_forward_noalloc(const sfm_params *params, const sfm_tensors *inputs, const int32_t *metadata,
                        size_t metadata_n, float softmax_scale, void *out, float *lse, int32_t *status,
                        sfm_stream_t stream);

/* Test hook: sfm_forward() (same arguments, same kernels, same outputs)
 * that also records every KV row the attention kernel's resolver hands to
 * its copy warps, so the attended sets of the kernel that computes O can be
 * compared exactly with a reference.  For query row t and attended position
 * k (ori positions first, then cmp, in index order; k < cap):
 *   rows[t * cap + k] = -1                       the entry is skipped (masked,
 *                                                 invalid or out of range),
 *                     = r (>= 0)                 row r of the ori_kv buffer,
 *                     = (int32_t)(r | 1u << 31)  row r of the cmp_kv buffer,
 * where r counts rows of row_stride bytes from the buffer's base (for PAGED
 * caches: block id * block_size + offset, after the block table).
 * counts[t] = attended positions of row t (clamped to cap); rows with no
 * position and entries at k >= counts[t] are left as the caller filled them
 * (fill counts with 0).  Positions at or beyond cap are not recorded and set
 * SFM_STATUS_BAD_LENGTH.  rows / counts: device int32, caller-owned. */
int sfm_debug_attended(const sfm_params *params, const sfm_tensors *inputs, const int32_t *metadata,
                       size_t metadata_n, float softmax_scale, void *out, float *lse, void *workspace,
                       size_t workspace_bytes, int32_t *rows, int64_t cap, int32_t *counts, int32_t *status,
                       sfm_stream_t stream);

/* Optional instrumentation for benchmarks: with both handles non-NULL (two
 * cudaEvent_t of the current device), every following sfm_forward() records
 * `begin` on its stream right before its main attention kernel and `end`
 * right after it, so the caller can time that kernel alone with
 * cudaEventElapsedTime.  (NULL, NULL) turns it off.  Process-wide setting,
 * not synchronised: set it from the thread that calls sfm_forward(). */
int sfm_set_profile_events(void *begin, void *end);

/* Static description of an sfm_error code. */
const char *sfm_error_string(int code);

/* SFM_ABI_VERSION of the loaded library. */
int sfm_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SFM_H */
