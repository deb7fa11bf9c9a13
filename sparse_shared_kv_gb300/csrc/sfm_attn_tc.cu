// sfm_attn_tc.cu -- tensor-core (tcgen05 / TMEM) split-KV attention for
// plain bf16 / fp16 KV rows.
//
// One persistent CTA per SM walks the work units the planner gave its worker.
// A unit is one split of one query row for one group of up to 64 heads; the
// units of a row are ordered group-major, so consecutive units of a worker
// usually share their Q rows and Q is only reloaded when the (row, group)
// changes.  Per 32-row KV tile of a unit:
//   resolver warp 9      resolves the attended rows (window / compressed /
//                        indices through the block tables) up to 16 tiles
//                        ahead, eight tiles per batch so that a batch costs
//                        two dependent memory round trips, into a ring of
//                        row numbers in shared memory;
//   producer warps 0-3   stream each tile's 32 rows (1 KB each, 8 rows per
//                        warp) with cp.async into the 128-byte-swizzled
//                        operand layout (four stages) and, when the (row,
//                        head group) changes, the unit's 64 Q rows (16 per
//                        warp).  Four copy warps keep more requests in
//                        flight per SM than two (about 38 vs 33 GB/s per SM
//                        with all SMs loading).  16-byte cp.async
//                        gathers sustain about 5 TB/s of random 1 KB rows on
//                        this part; TMA row gathers (tile::gather4) reach
//                        about 1.8 TB/s, one-row TMA boxes about 0.7 TB/s;
//   MMA warps 8, 10      S = Q.K~^T            (M=128, N=32 or 64, K=512 / 576) -> TMEM
//   (and 11 for packed)  as independent accumulation chains, one per
//                        issuing warp (two for plain rows, three for packed);
//   MMA in warp 6        O += P.V~             (M=128, N=256, K=2x32)  -> TMEM
//                        both products read the SAME staged tile (K-major
//                        for S, MN-major for P.V); four S buffers, two P
//                        buffers.  A chain of small dependent MMAs from one
//                        thread is bound by per-instruction latency, not by
//                        the math, so S is split in two chains on two warps
//                        and P.V has its own issuing warp;
//   softmax warps 4-7    warps 4-5: one thread per head row -- scale, mask,
//                        running max with lazy rescaling, exp2, row sum, P
//                        (bf16/fp16) into shared memory; warps 6-7 rescale the
//                        upper half of O.  The epilogue pulls O out of TMEM
//                        into registers (releasing TMEM for the next unit's
//                        first P.V) and writes the output (single split) or
//                        the split's bf16 partial O and fp32 LSE for the
//                        combine kernel.
//
// M=128 rows with at most 64 heads: the upper 64 rows of the Q operand alias
// the next column block (their scores are never read), and O uses a
// block-diagonal P so that TMEM rows 0-63 accumulate O[:, 0:256] and rows
// 64-127 accumulate O[:, 256:512] in 256 columns: A = [P;0] with V[:, :256]
// for the first two reduction steps, A = [0;P] with V[:, 256:] for the next.
//
// Softmax follows the pages' definition (S = Q.K~^T * softmax_scale, softmax
// over the attended rows, LSE = max S + log sum exp(S - max S)); scores are
// kept in the log2 domain (x = S * log2 e) and the running max is only moved
// when a row's max grows by more than 8 (a factor 256), which leaves O / l
// unchanged mathematically and keeps fp32 far from overflow.
//
// Every wait is bounded (2 s); a timeout raises the CTA's abort flag, every
// role leaves its loop at its next wait, in-flight copies and MMAs are
// drained, TMEM is freed and SFM_STATUS_TIMEOUT is reported.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "sfm_internal.cuh"
#include "sfm_tc.cuh"

namespace sfm {

namespace {

using namespace tc;

constexpr int NT = 32;                       // KV rows per tile
constexpr int kThreads = 384;               // 12 warps: three warpgroups
constexpr int kProducers = 4;               // KV copy warps
constexpr uint32_t KV_BLOCK = NT * 128;      // one 64-column block of one stage (32 rows)
constexpr uint32_t PK_ROW = 656;             // packed row: int8[512], rope bf16[64], fp32 scale[4]
constexpr uint32_t MISC_BYTES = 4608;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_O = 0;                 // O: columns [0, 256)
constexpr uint32_t TM_S = 256;               // S: chain c, stage s at [256 + 128 c + 32 s, +32)
constexpr float kRescaleThreshold = 8.0f;    // log2 units
constexpr int kRing = 16;                    // resolved tiles in flight
constexpr int kResolveBatch = 8;             // tiles per resolver batch
constexpr int kFirstBatch = 4;               // tiles of a worker's first resolver batch
constexpr int kPrefetchTiles = 4;            // tiles past the stages whose rows are prefetched to L2

// Shared-memory layout.  Plain rows: Q (8 column blocks of 64 values), P,
// four 32-row bf16 stages.  Packed rows: Q and K carry 9 column blocks (512
// NoPE values + 64 rope values), two fp16 stages, two raw stages of 32
// packed rows (the copy target the producers convert from) and each fp16
// stage's per-row scales (4 per row, one per 128-value tile).
// MODE 0: plain rows; 1: packed rows whose dequantised values are rounded
// once to fp16 (int8); 2: packed rows computed from their exact unscaled
// values with the scales applied in fp32 (E4M3).
template <int MODE>
struct Lay {
    static constexpr bool PK = MODE > 0;
    static constexpr int QB = PK ? 9 : 8;                        // 64-column blocks of a Q / K row
    static constexpr int kStages = PK ? 2 : 4;                   // bf16 KV stages == S buffers
    static constexpr uint32_t Q_OFF = 0;                         // QB blocks x 64 rows x 128 B
    static constexpr uint32_t P_OFF = QB * 8192;                 // 192 rows x 128 B: zero / P / zero
    static constexpr uint32_t KV_OFF = P_OFF + 24576;
    static constexpr uint32_t KV_COL = kStages * KV_BLOCK;       // stride between 64-column blocks
    static constexpr uint32_t RAW_OFF = KV_OFF + QB * KV_COL;
    static constexpr uint32_t RAW_STAGE = NT * PK_ROW;
    static constexpr uint32_t SCL_OFF = RAW_OFF + (PK ? 2 * RAW_STAGE : 0);   // [stage][tile][32 rows] fp32 scales
    static constexpr uint32_t SCL_BYTES = MODE == 2 ? kStages * 4 * NT * 4 : 0;
    static constexpr uint32_t MISC_OFF = (SCL_OFF + SCL_BYTES + 1023u) & ~1023u;
    static constexpr uint32_t EPI_OFF = MISC_OFF + MISC_BYTES;   // epilogue staging, 1 KB per softmax warp
    static constexpr uint32_t kSmemBytes = EPI_OFF + 4 * 1024 + 1024;   // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(P_OFF == Q_OFF + QB * 8192, "the last Q block's alias rows must be P's leading zero rows");
};

// barrier slots (8 bytes each) at MISC_OFF
enum Bar {
    B_KV_FULL = 0,     // [4] 128 copy-completion arrivals + the row-mask word
    B_KV_EMPTY = 4,    // [4] P.V of the tile done
    B_S_FULL = 8,      // [4] both halves of S of the tile in TMEM
    B_S_FREE = 12,     // [4] both head warps read S
    B_P_FULL = 16,     // [2] P written and O rescaled by all four softmax warps
    B_O_DONE = 18,     // [2] P.V of tiles with that parity done
    B_Q_FULL = 20,     // 128 copy-completion arrivals
    B_Q_EMPTY = 21,    // both S issuers done with Q
    B_ALPHA = 22,      // [4] per-tile rescale factors published
    B_STATS = 26,      // final (max, sum) of the unit published
    B_TEARDOWN = 27,
    B_ROW_FULL = 28,   // [16] resolved rows of a tile in the ring
    B_ROW_EMPTY = 44,  // [16] the four producer warps took them
    B_TEARDOWN_PV = 60,
    B_TEARDOWN_S2 = 61,
    B_TEARDOWN_S3 = 62,
    B_SV_DONE = 63,    // [2] packed rows: every S product of the tile on that stage has read it
    kNumBars = 65
};
// offsets inside the misc area
constexpr uint32_t TMEM_SLOT_REL = 576;
constexpr uint32_t ABORT_REL = 580;
constexpr uint32_t VALID_REL = 592;      // [4] row-valid words
constexpr uint32_t ALPHA_REL = 1024;     // [4][64] floats
constexpr uint32_t STATS_REL = 2048;     // [64][2] floats
constexpr uint32_t RING_REL = 2560;      // [16][32] int32 row entries
static_assert(kNumBars * 8 <= TMEM_SLOT_REL && VALID_REL + 16 <= 1024, "barrier area");
static_assert(RING_REL + kRing * NT * 4 <= MISC_BYTES, "misc area");

struct Unit {
    int t, w, h0, nh, nsplit, pos0, pos1, ntiles, key;
    Tok k;
};

// Unit u of the plan from its split's 64-byte record (query row, first split
// and split count of the row, the row's split size and lengths / window /
// position counts): the split, head group and row range of the unit.
__device__ __forceinline__ Unit unit_decode(const KParams &kp, int4 r0, int4 r1, int4 r2, int u)
{
    Unit s;
    const int HG = kp.head_groups;
    s.t = r0.x;
    const int s_beg = r0.y;
    s.nsplit = r0.z;
    const int size = r0.w;
    const int local = u - s_beg * HG;
    // head group of the unit: units of a row are group-major, at most two
    // groups (128 heads)
    const int hg = (HG > 1 && s.nsplit > 0 && local >= s.nsplit) ? 1 : 0;
    const int sidx = local - hg * s.nsplit;
    s.w = sidx;          // the row's workspace slot t * max_splits + sidx holds its partial
    s.h0 = hg * 64;
    s.nh = min(64, kp.q_n - s.h0);
    s.key = s.t * HG + hg;
    Tok &k = s.k;
    k.b = r1.x;
    k.kv_len = r1.y;
    k.cmp_len = r1.z;
    k.p_cmp = r1.w;
    k.lo = r2.x;
    k.hi = r2.y;
    k.n_ori = r2.z;
    k.n_cmp = r2.w;
    k.i = 0;
    k.q_len = 0;
    k.p = 0;
    k.valid = 1;
    const int n = k.n_ori + k.n_cmp;
    s.pos0 = sidx * size;
    s.pos1 = min(n, s.pos0 + size);
    const int rows = s.pos1 > s.pos0 ? s.pos1 - s.pos0 : 0;
    s.ntiles = rows > 0 ? (rows + NT - 1) / NT : 1;   // an empty split still runs one masked tile
    return s;
}

__device__ __forceinline__ Unit unit_info(const KParams &kp, const int32_t *srec, int u)
{
    const int4 *r = reinterpret_cast<const int4 *>(srec + (int64_t)(u / kp.head_groups) * kSrecWords);
    return unit_decode(kp, __ldg(r), __ldg(r + 1), __ldg(r + 2), u);
}

// byte b of w as a signed 8-bit integer, converted exactly to float: the
// sign-extended byte (prmt sign-replicate selector) added to the bit pattern
// of 1.5 * 2^23, whose unit in the last place is 1, minus 1.5 * 2^23
__device__ __forceinline__ float i8_to_f32(uint32_t w, int b)
{
    const uint32_t sel = (uint32_t)b | ((8u | b) << 4) | ((8u | b) << 8) | ((8u | b) << 12);
    uint32_t v;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(v) : "r"(w), "r"(sel));
    return __int_as_float(0x4B400000 + (int)v) - 12582912.0f;
}

// eight bf16 values -> eight fp16 values (round to nearest; exact for
// magnitudes in fp16's normal range)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v)
{
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = __uint_as_float(w[i] << 16), b = __uint_as_float(w[i] & 0xffff0000u);
        __half2 h = __floats2half2_rn(a, b);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16)
{
    if (bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Row entries of this lane's row in tiles i0 .. i0+K-1 of the unit: -1 for a
// skipped or masked position, else the pool row with bit 31 set for the
// compressed pool; out-of-range indices (BAD_INDEX) and rows outside the
// cache (BAD_BLOCK) are skipped and flagged in the status word.  Every load
// is unconditional, from the real address or from an always-valid one, so
// that the K index loads and then the K block-table loads each go out back to
// back: a batch costs two memory round trips whatever K is.
template <int K>
__device__ __forceinline__ void resolve_tiles(const KParams &kp, const Unit &s, int i0, int lane, int32_t (&ent)[K])
{
    const Tok &k = s.k;
    const int32_t *safe = kp.meta;      // any readable int32
    int e[K];
    bool in[K], cmp[K];
    // 1. positions -> logical rows (the index tensors for top-k sources)
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const int pos = s.pos0 + (i0 + j) * NT + lane;
        in[j] = pos < s.pos1;
        cmp[j] = pos >= k.n_ori;
        const int jj = pos - k.n_ori;
        const bool from_idx = in[j] && (cmp[j] ? kp.cmp_topk > 0 : kp.ori_topk > 0);
        const int32_t *ip = !from_idx ? safe
                            : cmp[j]  ? kp.cmp_idx + (int64_t)s.t * kp.cmp_topk + jj
                                      : kp.ori_idx + (int64_t)s.t * kp.ori_topk + (pos >> kp.sbs_log2);
        const int v = __ldg(ip);
        e[j] = from_idx ? v : (cmp[j] ? jj : k.lo + pos);
    }
    int err = 0;
#pragma unroll
    for (int j = 0; j < K; ++j) {
        bool ok = in[j];
        if (ok && !cmp[j] && kp.ori_topk > 0) {
            // block-wise entries: the block start, then this position's token in it
            const int pos = s.pos0 + (i0 + j) * NT + lane;
            const int64_t blk0 = (int64_t)e[j] << kp.sbs_log2;
            const int64_t tok = blk0 + (pos & ((1 << kp.sbs_log2) - 1));
            if (e[j] >= 0 && blk0 >= k.kv_len) err |= SFM_STATUS_BAD_INDEX;
            ok = e[j] >= 0 && tok < k.kv_len && tok >= k.lo && tok <= k.hi;
            e[j] = ok ? (int)tok : 0;
        } else if (ok && cmp[j] && kp.cmp_topk > 0) {
            if (e[j] >= k.cmp_len) err |= SFM_STATUS_BAD_INDEX;
            ok = e[j] >= 0 && e[j] < k.cmp_len &&
                 (kp.cmp_mask_mode != 3 || (int64_t)(e[j] + 1) * kp.cmp_ratio <= (int64_t)k.p_cmp + 1);
        }
        in[j] = ok;
    }
    // 2. logical rows -> pool rows
    int64_t row[K];
    if (kp.layout_kv == SFM_LAYOUT_PAGED) {
        int32_t blk[K], off[K];
        bool inb[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int bs = cmp[j] ? kp.cmp_bs : kp.ori_bs;
            const int bts = cmp[j] ? kp.cmp_bt_stride : kp.ori_bt_stride;
            const int ee = in[j] ? e[j] : 0;
            const int bi = (int)fdiv((uint32_t)ee, cmp[j] ? kp.cmp_bs_div : kp.ori_bs_div);
            off[j] = ee - bi * bs;
            inb[j] = in[j] && bi < bts;
            const int32_t *bp = inb[j] ? (cmp[j] ? kp.cmp_bt : kp.ori_bt) + (int64_t)k.b * bts + bi : safe;
            blk[j] = __ldg(bp);
        }
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int bs = cmp[j] ? kp.cmp_bs : kp.ori_bs;
            row[j] = (inb[j] && blk[j] >= 0) ? (int64_t)blk[j] * bs + off[j] : -1;
        }
    } else if (kp.layout_kv == SFM_LAYOUT_TND) {
        const int64_t base_o = __ldg(kp.cu_ori + k.b);
        const int64_t base_c = kp.has_cmp ? (int64_t)__ldg(kp.cu_cmp + k.b) : 0;
#pragma unroll
        for (int j = 0; j < K; ++j) row[j] = (cmp[j] ? base_c : base_o) + e[j];
    } else {
#pragma unroll
        for (int j = 0; j < K; ++j) row[j] = (int64_t)k.b * (cmp[j] ? kp.cmp_s : kp.ori_s) + e[j];
    }
#pragma unroll
    for (int j = 0; j < K; ++j) {
        int32_t v = -1;
        if (in[j]) {
            const int64_t nrows = cmp[j] ? kp.cmp_rows : kp.ori_rows;
            if (row[j] < 0 || row[j] >= nrows) err |= SFM_STATUS_BAD_BLOCK;
            else v = static_cast<int32_t>(static_cast<uint32_t>(row[j]) | (cmp[j] ? 0x80000000u : 0u));
        }
        ent[j] = v;
    }
    if (err) set_status(kp, err);
}

// Rows without a split, when a plan has at most one split per row and no
// combine kernel follows the attention kernel: O = 0 and LSE = -inf for every
// row with no split (every row when the plan was made for other params), and
// the plan's status, as the combine kernel writes them otherwise.  Rows are
// spread over the CTAs of the grid.  Kept out of line so the attention
// kernel's own code and registers do not change with it.
__device__ __noinline__ void finish_rows_without_split(const int32_t *meta, bool ok, int G, int T, int qn, void *out,
                                                       float *lse, int32_t *status)
{
    const int tid = threadIdx.x;
    const int32_t *spt = meta + meta_split_off(G);
    if (blockIdx.x == 0 && tid == 0 && status) {
        if (!ok) atomicOr(status, SFM_STATUS_METADATA_MISMATCH | meta[H_FLAGS]);
        else if (meta[H_LENFLAGS]) atomicOr(status, meta[H_LENFLAGS]);
    }
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        if (ok && spt[t + 1] > spt[t]) continue;          // uniform over the CTA
        uint4 *o4 = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + (int64_t)t * qn * 512);
        for (int i = tid; i < qn * 64; i += kThreads) o4[i] = make_uint4(0, 0, 0, 0);
        if (lse)
            for (int h = tid; h < qn; h += kThreads) lse[(int64_t)t * qn + h] = -INFINITY;
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) sfm_attn_tc_kernel(const KParams kp)
{
    using L = Lay<MODE>;
    constexpr bool PK = MODE > 0;          // packed rows
    constexpr bool EX = MODE == 2;         // packed rows with exact scores
    constexpr int QB = L::QB, kStages = L::kStages;
    // Independent accumulation chains of S (TMEM: chain c, buffer b at
    // TM_S + 32 (c * kSBufs + b)).  Plain rows: two chains (dimensions 0-255
    // and 256-511), one buffer per stage, issued by warps 8 and 10.  Packed
    // rows rounded to fp16: three chains of 192 dimensions (warps 8, 10, 11).
    // Packed rows with exact scores: one chain per 128-value scale tile and
    // one for the rope part, so that the products are exact products of the
    // unscaled values and the softmax applies each row's fp32 tile scales;
    // five chains leave room for one buffer only, issued by warps 8 (tiles 0,
    // 1), 10 (tiles 2, 3) and 11 (rope).  The tensor pipe takes products from
    // several issuing warps at once, while one warp issues one about every
    // 100-130 ns whatever its size.
    constexpr int kChains = EX ? 5 : PK ? 3 : 2;
    constexpr int kIssuers = PK ? 3 : 2;
    constexpr int kSBufs = EX ? 1 : kStages;
    static_assert(kChains * kSBufs * NT <= 256, "S buffers fit next to O in TMEM");
    constexpr uint32_t Q_OFF = L::Q_OFF, P_OFF = L::P_OFF, KV_COL = L::KV_COL, MISC_OFF = L::MISC_OFF;
    constexpr uint32_t EPI_OFF = L::EPI_OFF, TMEM_SLOT_OFF = MISC_OFF + TMEM_SLOT_REL, ABORT_OFF = MISC_OFF + ABORT_REL;
    constexpr uint32_t VALID_OFF = MISC_OFF + VALID_REL, ALPHA_OFF = MISC_OFF + ALPHA_REL;
    constexpr uint32_t STATS_OFF = MISC_OFF + STATS_REL, RING_OFF = MISC_OFF + RING_REL;
    // Column block a of stage st sits at KV_OFF + a * KV_COL + st * KV_BLOCK, so
    // stages 2j and 2j+1 form one contiguous 64-row operand per column block.
    auto kv_at = [](uint32_t st, uint32_t a) -> uint32_t { return L::KV_OFF + a * KV_COL + st * KV_BLOCK; };
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(base);
    const uint32_t bar0 = sb + MISC_OFF;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + ABORT_OFF);
    uint32_t *valid_s = reinterpret_cast<uint32_t *>(base + VALID_OFF);
    float *scl = reinterpret_cast<float *>(base + L::SCL_OFF);     // packed rows: [stage][tile][row] scales
    float *alpha_s = reinterpret_cast<float *>(base + ALPHA_OFF);
    float *stats_s = reinterpret_cast<float *>(base + STATS_OFF);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool bf16 = kp.dtype == SFM_DTYPE_BF16;   // input / output dtype
    // Operand dtype of the products.  Packed rows compute in fp16: int8 x
    // scale rounded to fp16 (11-bit significand) keeps S within the LSE
    // tolerance where bf16 (8-bit) does not; bf16 Q is converted exactly
    // (magnitudes up to 65504).
    const bool mma_bf16 = PK ? false : bf16;
    grid_launch_dependents();    // the next kernel (the combine, or the next planner) may launch; it waits for this grid

    // ---------------- set-up ----------------
    for (uint32_t i = tid; i < 24576u / 16u; i += kThreads)
        reinterpret_cast<uint4 *>(base + P_OFF)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(B_KV_FULL + s), PK ? kProducers + 1 : 32 * kProducers + 1);
            mbar_init(bar(B_KV_EMPTY + s), 1);
            mbar_init(bar(B_S_FULL + s), kIssuers);
            mbar_init(bar(B_S_FREE + s), 2);
        }
        for (int a = 0; a < 4; ++a) mbar_init(bar(B_ALPHA + a), 2);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_P_FULL + b), 4);
            mbar_init(bar(B_O_DONE + b), 1);
        }
        for (int r = 0; r < kRing; ++r) {
            mbar_init(bar(B_ROW_FULL + r), 1);
            mbar_init(bar(B_ROW_EMPTY + r), kProducers);
        }
        mbar_init(bar(B_Q_FULL), (PK && kp.dtype == SFM_DTYPE_BF16) ? kProducers : 32 * kProducers);
        mbar_init(bar(B_Q_EMPTY), kIssuers);
        mbar_init(bar(B_STATS), 2);
        mbar_init(bar(B_TEARDOWN), 1);
        mbar_init(bar(B_TEARDOWN_PV), 1);
        mbar_init(bar(B_TEARDOWN_S2), 1);
        mbar_init(bar(B_TEARDOWN_S3), 1);
        for (int s = 0; s < 2; ++s) mbar_init(bar(B_SV_DONE + s), kIssuers);
        *abort_flag = 0;
        fence_barrier_init();
    }
    fence_proxy_async_smem();
    if (warp == 8) {
        tmem_alloc(sb + TMEM_SLOT_OFF, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(base + TMEM_SLOT_OFF);

    // While the planner still runs: pull this CTA's share of the index
    // tensors, block tables and Q into L2 (they do not depend on the plan),
    // so the first dependent loads after the plan hit L2.  Issued by a lane
    // of an S-issuing warp, which has nothing to do until the first tile
    // lands (issuing these from the resolver delayed its first loads).
    if (tid == 10 * 32 + 1) {
        const int G = gridDim.x, c = blockIdx.x;
        constexpr int64_t kCap = 256 * 1024;
        prefetch_share(kp.cmp_idx, (int64_t)kp.T * kp.cmp_topk * 4, c, G, kCap);
        prefetch_share(kp.ori_idx, (int64_t)kp.T * kp.ori_topk * 4, c, G, kCap);
        if (kp.layout_kv == SFM_LAYOUT_PAGED) {
            prefetch_share(kp.ori_bt, (int64_t)kp.batch * kp.ori_bt_stride * 4, c, G, kCap);
            if (kp.has_cmp) prefetch_share(kp.cmp_bt, (int64_t)kp.batch * kp.cmp_bt_stride * 4, c, G, kCap);
        }
        prefetch_share(kp.q, (int64_t)kp.T * kp.q_n * kp.d_qk * 2, c, G, kCap);
    }

    // everything above overlapped the planner; the plan is read from here on
    grid_dependency_wait();
    // one round trip: the header check and this worker's record (its unit
    // range and its first unit's split record) are independent loads
    const int32_t *sp = kp.meta + meta_srec_off(kp.G, kp.T, kp.wcap);   // split records
    const int4 *wr = reinterpret_cast<const int4 *>(kp.meta + meta_wrec_off(kp.G, kp.T, kp.wcap) +
                                                    (int64_t)blockIdx.x * kWrecWords);
    const int4 w0 = __ldg(wr), w1 = __ldg(wr + 1), w2 = __ldg(wr + 2), w3 = __ldg(wr + 3);
    const bool ok = meta_ok(kp);
    const int u_beg = ok ? w0.x : 0;
    const int u_end = ok ? w0.y : 0;
    const Unit first = unit_decode(kp, w1, w2, w3, u_beg);

    int32_t *ring = reinterpret_cast<int32_t *>(base + RING_OFF);


    if (warp == 9) {
        // ======================= row resolver =======================
        // Lane L resolves row L of every tile, kResolveBatch tiles at a time,
        // and publishes each tile's 32 entries in ring slot (tile % kRing).
        int g = 0;
        bool stop = false;
        const bool pf_all = !PK && kp.split_rows < (1 << 30);     // plain rows, decode-shaped plan
        Unit cur = first;
        for (int u = u_beg; u < u_end && !stop; ++u) {
            const Unit nxt = u + 1 < u_end ? unit_info(kp, sp, u + 1) : cur;   // prefetched
            const Unit &s = cur;
            // publish tiles i0 .. i0 + K - 1 of the unit, then pull into L2
            // the rows of the tiles that wait for a stage to drain before
            // their copies start, so that those copies hit L2: for plain
            // rows of decode-shaped plans every tile from kStages on,
            // otherwise the worker's tiles kStages .. kStages +
            // kPrefetchTiles - 1 (prefill rows share most of their rows, and
            // more prefetching only added traffic there); one bulk prefetch
            // per plain row, line prefetches for packed rows
            auto publish = [&](int i0, int K, const int32_t *ent) {
                if (kp.dbg_rows) {
                    // attended-row dump: the entries exactly as the copy warps
                    // will consume them, at the row's attended position
                    for (int j = 0; j < K; ++j) {
                        const int pos = s.pos0 + (i0 + j) * NT + lane;
                        if (pos < s.pos1) {
                            if (pos < kp.dbg_cap) kp.dbg_rows[(int64_t)s.t * kp.dbg_cap + pos] = ent[j];
                            else set_status(kp, SFM_STATUS_BAD_LENGTH);
                        }
                    }
                    if (i0 == 0 && s.w == 0 && s.h0 == 0 && lane == 0)
                        kp.dbg_counts[s.t] = (int32_t)min((int64_t)(s.k.n_ori + s.k.n_cmp), kp.dbg_cap);
                }
                for (int j = 0; j < K; ++j) {
                    const int i = i0 + j;
                    if (i >= s.ntiles) break;
                    const int gi = g + i, slot = gi % kRing, use = gi / kRing;
                    if (use >= 1 && !warp_wait(bar(B_ROW_EMPTY + slot), (use - 1) & 1, abort_flag)) {
                        stop = true;
                        return;
                    }
                    ring[slot * NT + lane] = ent[j];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_ROW_FULL + slot));
                }
                for (int j = 0; j < K; ++j) {
                    const int gi = g + i0 + j;
                    if (i0 + j < s.ntiles && gi >= kStages && (pf_all || gi < kStages + kPrefetchTiles) && ent[j] != -1) {
                        const int64_t r = ent[j] & 0x7fffffff;
                        const uint8_t *row = ent[j] < 0 ? kp.cmp_kv + r * kp.cmp_row_stride : kp.ori_kv + r * kp.ori_row_stride;
                        if constexpr (!PK) {
                            prefetch_l2(row, QB * 128u);         // one bulk prefetch per 1 KB row
                        } else {
                            // the row's own lines only: 656 bytes, or 528 without
                            // the rope part (line prefetches: one bulk prefetch
                            // per packed row was slower for E4M3 rows)
                            if (kp.rope > 0) {
#pragma unroll
                                for (uint32_t o = 0; o < PK_ROW; o += 128) prefetch_line_l2(row + o);
                                prefetch_line_l2(row + PK_ROW - 1);
                            } else {
#pragma unroll
                                for (uint32_t o = 0; o < PK_ROW - 128; o += 128) prefetch_line_l2(row + o);
                                prefetch_line_l2(row + PK_ROW - 129);
                            }
                        }
                    }
                }
            };
            int i0 = 0;
            if (g == 0 && s.ntiles > 0) {
                // the worker's first tiles: a short batch (fewer instructions
                // before the first publish)
                int32_t ent[kFirstBatch];
                resolve_tiles<kFirstBatch>(kp, s, 0, lane, ent);
                publish(0, kFirstBatch, ent);
                i0 = kFirstBatch;
            }
            for (; i0 < s.ntiles && !stop; i0 += kResolveBatch) {
                int32_t ent[kResolveBatch];
                resolve_tiles<kResolveBatch>(kp, s, i0, lane, ent);
                publish(i0, kResolveBatch, ent);
            }
            g += s.ntiles;
            cur = nxt;
        }
    } else if (warp < kProducers) {
        // ======================= producers =======================
        // The four warps share every tile: warp pw copies rows 8pw..8pw+7,
        // one 1 KB row per step (row address broadcast from the ring entry's
        // lane; lane L copies 16-byte chunks L and L + 32: 512 contiguous
        // bytes per warp instruction).  Copies arrive on the stage barrier by
        // themselves when they land.  Each warp also copies 16 of the unit's
        // 64 Q rows when the (row, head group) changes.
        const int pw = warp;
        constexpr int kRowsPerWarp = NT / kProducers;
        const uint8_t *zero_src = static_cast<const uint8_t *>(kp.q);
        int g = 0, nq = 0, prev_key = -1;
        bool stop = false;
        // the unit's Q rows (16 heads per warp); rows past the group's heads are zero
        auto copy_q = [&](const Unit &s) -> bool {
            if (nq > 0 && !warp_wait(bar(B_Q_EMPTY), (nq - 1) & 1, abort_flag)) return false;
            const int QROW = (int)kp.d_qk * 2;             // bytes of one Q head row in the input
            const int QC = QROW / 16;                      // its 16-byte chunks (the rest of the QB blocks: zero)
            const uint8_t *qrow = static_cast<const uint8_t *>(kp.q) + ((int64_t)s.t * kp.q_n + s.h0) * QROW;
#pragma unroll 4
            for (int rr = 0; rr < 64 / kProducers; ++rr) {
                const int hh = pw * (64 / kProducers) + rr;
                const bool live = hh < s.nh;
#pragma unroll
                for (int part = 0; part < (QB * 8 + 31) / 32; ++part) {
                    const int C = lane + part * 32;
                    if (C < QB * 8) {
                        const uint32_t dst = sb + Q_OFF + (C >> 3) * 8192u + sw128(hh, C & 7);
                        const bool in_row = live && C < QC;
                        cp_async16(dst, in_row ? qrow + (int64_t)hh * QROW + C * 16 : zero_src, in_row ? 16u : 0u);
                    }
                }
            }
            if (PK && bf16) {
                // bf16 Q -> fp16 in place once this warp's rows have landed
                cp_async_commit();
                cp_async_wait<0>();
                __syncwarp();
                for (int rr = 0; rr < 64 / kProducers; ++rr) {
                    const int hh = pw * (64 / kProducers) + rr;
#pragma unroll
                    for (int part = 0; part < (QB * 8 + 31) / 32; ++part) {
                        const int C = lane + part * 32;
                        if (C < QB * 8) {
                            uint4 *q4 = reinterpret_cast<uint4 *>(base + Q_OFF + (C >> 3) * 8192u + sw128(hh, C & 7));
                            *q4 = bf16x8_to_f16x8(*q4);
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_Q_FULL));
            } else {
                cp_async_arrive_noinc(bar(B_Q_FULL));
            }
            ++nq;
            prev_key = s.key;
            return true;
        };
        // packed rows: dequantize this warp's 8 rows of tile p from its raw
        // stage into fp16 stage p % kStages (int8 or E4M3 x the row's
        // per-128 fp32 scale, rounded once; the 64 rope values converted to
        // fp16)
        int pend = -1;
        uint32_t pend_vm = 0;
        const bool fp8 = PK && kp.kv_fp8;
        // rope-0 packed rows (528 bytes) keep the 576-dim computation: their
        // rope operand block is zero in K and in Q, so the products are those
        // of the same row padded with a zero rope part
        const bool has_rope = kp.rope > 0;
        const uint32_t row_bytes = has_rope ? PK_ROW : PK_ROW - 128, scale_off = row_bytes - 16;
        auto convert = [&](int p, uint32_t vmask, bool last) -> bool {
            if (last) cp_async_wait<0>(); else cp_async_wait<1>();
            __syncwarp();
            const int st = p & (kStages - 1), use = p / kStages;
            if (use >= 1 && !warp_wait(bar(B_KV_EMPTY + st), (use - 1) & 1, abort_flag)) return false;
            const uint8_t *rawp = base + L::RAW_OFF + (p & 1) * L::RAW_STAGE;
#pragma unroll 2
            for (int k = 0; k < kRowsPerWarp; ++k) {
                const int rr = pw * kRowsPerWarp + k;
                const uint8_t *row = rawp + rr * PK_ROW;
                const uint4 v = *reinterpret_cast<const uint4 *>(row + 16 * lane);   // dims 16 lane .. +15
                const float sc = *reinterpret_cast<const float *>(row + scale_off + 4 * (lane >> 3));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t o[8];
                // MODE 1: value x scale in fp32, rounded once to fp16.
                // MODE 2: the unscaled values (every int8 and every E4M3
                // value is an fp16 value, so the conversion is exact); the
                // scale is applied in fp32 to the products (S) and, after S
                // has read the stage, to the values in place (for P.V)
                const float vs = EX ? 1.f : sc;
                if (fp8) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float f[4];
                        e4m3x4_to_f32(w[q], f);
                        o[2 * q] = pack2(f[0] * vs, f[1] * vs, false);
                        o[2 * q + 1] = pack2(f[2] * vs, f[3] * vs, false);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        o[2 * q] = pack2(i8_to_f32(w[q], 0) * vs, i8_to_f32(w[q], 1) * vs, false);
                        o[2 * q + 1] = pack2(i8_to_f32(w[q], 2) * vs, i8_to_f32(w[q], 3) * vs, false);
                    }
                }
                if (EX && (lane & 7) == 0) scl[(st * 4 + (lane >> 3)) * NT + rr] = sc;
                const uint32_t dst = sb + kv_at(st, lane >> 2);
                *reinterpret_cast<uint4 *>(base + (dst - sb) + sw128(rr, (lane & 3) * 2)) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4 *>(base + (dst - sb) + sw128(rr, (lane & 3) * 2 + 1)) =
                    make_uint4(o[4], o[5], o[6], o[7]);
                if (lane < 8) {                          // rope: input dtype -> fp16; rope-0 rows: zeros
                    uint4 r4 = make_uint4(0, 0, 0, 0);
                    if (has_rope) {
                        r4 = *reinterpret_cast<const uint4 *>(row + 512 + 16 * lane);
                        if (bf16) r4 = bf16x8_to_f16x8(r4);
                    }
                    *reinterpret_cast<uint4 *>(base + kv_at(st, 8) + sw128(rr, lane)) = r4;
                }
            }
            fence_proxy_async_smem();      // generic-proxy writes -> tensor-core reads
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_KV_FULL + st));
            if (pw == 0 && lane == 0) {
                valid_s[st] = vmask;                     // the tile's row-valid bits
                mbar_arrive(bar(B_KV_FULL + st));        // release: the word is visible with the phase
            }
            return true;
        };
        Unit cur = first;
        for (int u = u_beg; u < u_end && !stop; ++u) {
            const Unit nxt = u + 1 < u_end ? unit_info(kp, sp, u + 1) : cur;   // prefetched
            const Unit &s = cur;
            const bool reload = s.key != prev_key;
            // the worker's first Q goes out at once, while the resolver still
            // waits for its first rows; later ones after the unit's first tile
            const bool q_first = reload && nq == 0;
            if (q_first && !copy_q(s)) { stop = true; break; }
            for (int i = 0; i < s.ntiles; ++i) {
                const int gi = g + i, slot = gi % kRing, st = gi & (kStages - 1), use = gi / kStages;
                if (!warp_wait(bar(B_ROW_FULL + slot), (gi / kRing) & 1, abort_flag)) { stop = true; break; }
                const int32_t e = ring[slot * NT + lane];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_ROW_EMPTY + slot));
                const uint8_t *row = nullptr;
                if (e != -1) {
                    const int64_t r = e & 0x7fffffff;
                    row = e < 0 ? kp.cmp_kv + r * kp.cmp_row_stride : kp.ori_kv + r * kp.ori_row_stride;
                }
                const uint32_t vm = __ballot_sync(0xffffffffu, row != nullptr);
                const unsigned long long my_row = reinterpret_cast<unsigned long long>(row);
                if constexpr (!PK) {
                    if (use >= 1 && !warp_wait(bar(B_KV_EMPTY + st), (use - 1) & 1, abort_flag)) { stop = true; break; }
                    const uint32_t stage = sb + kv_at(st, 0);
#pragma unroll
                    for (int k = 0; k < kRowsPerWarp; ++k) {
                        const int rr = pw * kRowsPerWarp + k;
                        const uint8_t *src = reinterpret_cast<const uint8_t *>(__shfl_sync(0xffffffffu, my_row, rr));
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const int C = lane + half * 32;
                            const uint32_t dst = stage + (C >> 3) * KV_COL + sw128(rr, C & 7);
                            cp_async16(dst, src ? src + C * 16 : zero_src, src ? 16u : 0u);
                        }
                    }
                    cp_async_arrive_noinc(bar(B_KV_FULL + st));
                    if (pw == 0 && lane == 0) {
                        valid_s[st] = vm;                        // the tile's row-valid bits
                        mbar_arrive(bar(B_KV_FULL + st));        // release: the word is visible with the phase
                    }
                } else {
                    // packed rows: 656 bytes each (41 x 16) into raw stage gi % 2,
                    // then convert the tile copied one step earlier
                    const uint32_t raw = sb + L::RAW_OFF + (gi & 1) * L::RAW_STAGE;
#pragma unroll
                    for (int k = 0; k < kRowsPerWarp; ++k) {
                        const int rr = pw * kRowsPerWarp + k;
                        const uint8_t *src = reinterpret_cast<const uint8_t *>(__shfl_sync(0xffffffffu, my_row, rr));
                        const uint32_t dst = raw + rr * PK_ROW;
                        cp_async16(dst + lane * 16, src ? src + lane * 16 : zero_src, src ? 16u : 0u);
                        if (lane < (int)(row_bytes / 16) - 32)
                            cp_async16(dst + (32 + lane) * 16, src ? src + (32 + lane) * 16 : zero_src, src ? 16u : 0u);
                    }
                    cp_async_commit();
                    if (pend >= 0 && !convert(pend, pend_vm, false)) { stop = true; break; }
                    pend = gi;
                    pend_vm = vm;
                }
                // a reloaded Q after the unit's first tile: that tile's rows
                // are usually resolved by then, and Q waits for the S issuers
                if (i == 0 && reload && !q_first && !copy_q(s)) { stop = true; break; }
            }
            g += s.ntiles;
            cur = nxt;
        }
        if constexpr (PK) {
            if (!stop && pend >= 0) convert(pend, pend_vm, true);
        }
        cp_async_wait<0>();
    } else if (warp == 8 || warp == 10 || (kIssuers > 2 && warp == 11)) {
        // ======================= S issuers =======================
        // S(i) needs tile i staged and its S buffer free.  Its reduction
        // steps run as independent accumulation chains: plain rows one per
        // issuing warp, warps 8 and 10 (dimensions 0..255 and 256..511), into
        // TMEM column ranges chain c, stage st at TM_S + 32 (c kStages + st);
        // packed rows five chains (the four 128-value scale tiles and the rope
        // part) into one buffer, TM_S + 32 c, warp 8 issuing tiles 0 and 1,
        // warp 10 tiles 2 and 3 (interleaved), warp 11 the rope part.  The
        // softmax adds the chains (packed rows: with each row's tile scales).
        // For plain rows an even tile and the next tile of the same unit are
        // computed together as one N=64 product, which halves the number of
        // S instructions (the tensor pipe's instruction rate, not its math,
        // bounds these small products).  P.V is issued by warp 6.
        if (lane == 0) {
            const int c = warp == 8 ? 0 : warp == 10 ? 1 : 2;     // this warp's chain
            const uint32_t id_s = idesc_f16(128, NT, mma_bf16, false, false);
            const uint32_t id_s2 = idesc_f16(128, 2 * NT, mma_bf16, false, false);
            int g = 0, nq = 0, prev_key = -1;
            bool stop = false;
            Unit cur = first;
            for (int u = u_beg; u < u_end && !stop; ++u) {
                const Unit nxt = u + 1 < u_end ? unit_info(kp, sp, u + 1) : cur;
                const Unit &s = cur;
                const bool next_reloads = u + 1 < u_end && nxt.key != s.key;
                if (s.key != prev_key) {
                    if (!mbar_wait(bar(B_Q_FULL), nq & 1, abort_flag)) break;
                    ++nq;
                    prev_key = s.key;
                }
                for (int i = 0; i < s.ntiles;) {
                    const int gi = g + i, st = gi & (kStages - 1), use = gi / kStages;
                    // an even tile and the next one of the same unit share one
                    // 64-row S (stages 2j, 2j+1 are one operand)
                    // (packed rows have two stages only: a pair would hold both
                    // and stop the conversion of the next tile from overlapping)
                    const int nt = (!PK && (gi & 1) == 0 && i + 1 < s.ntiles) ? 2 : 1;
                    bool good = true;
                    for (int j = 0; j < nt && good; ++j) {
                        good = mbar_wait(bar(B_KV_FULL + st + j), use & 1, abort_flag);
                        if (!EX) good = good && (use == 0 || mbar_wait(bar(B_S_FREE + st + j), (use - 1) & 1, abort_flag));
                        else good = good && (gi == 0 || mbar_wait(bar(B_S_FREE), (gi - 1) & 1, abort_flag));
                    }
                    if (!good) {
                        stop = true;
                        break;
                    }
                    fence_proxy_async_smem();    // cp.async (generic proxy) writes -> tensor-core reads
                    tc_fence_after();
                    const uint32_t id = nt == 2 ? id_s2 : id_s;
                    if constexpr (!EX) {
                        // this warp's chain c covers reduction steps [kSteps c, kSteps (c + 1)).
                        // Each descriptor is built here, which paces the products at ~50 ns
                        // instead of ~30.  Issued back to back from precomputed descriptors
                        // they made every workload slower (CSA prefill +24 %, HCA decode
                        // +3 %, FP8 rows +6 % in A/B runs on one GPU), and still did as M=64
                        // products (half of Q's shared-memory reads) or with the S issuers
                        // yielding to a pending P.V.
                        constexpr int kSteps = QB * 4 / kChains;
#pragma unroll 3
                        for (int k = 0; k < kSteps; ++k) {
                            const uint32_t d = tmem + TM_S + c * (kStages * NT) + st * NT;
                            const uint32_t kk = c * kSteps + k, blk = kk >> 2, sub = (kk & 3) * 32u;
                            umma_f16(d, sdesc_sw128(sb + Q_OFF + blk * 8192u + sub, 16, 1024),
                                     sdesc_sw128(sb + kv_at(st, blk) + sub, 16, 1024), id, k > 0);
                        }
                        for (int j = 0; j < nt; ++j) umma_commit(bar(B_S_FULL + st + j));
                    } else {
                        // chains 2c and 2c + 1 (tiles: 8 reduction steps over
                        // column blocks 2 t, 2 t + 1), or the rope chain 4
                        // (4 steps over block 8), interleaved step by step
                        const int c0 = c < 2 ? 2 * c : 4, nch = c < 2 ? 2 : 1, nsteps = c < 2 ? 8 : 4;
#pragma unroll 2
                        for (int k = 0; k < nsteps; ++k) {
                            for (int j = 0; j < nch; ++j) {
                                const int cc = c0 + j;
                                const uint32_t kk = cc < 4 ? 8 * cc + k : 32 + k, blk = kk >> 2, sub = (kk & 3) * 32u;
                                umma_f16(tmem + TM_S + cc * NT, sdesc_sw128(sb + Q_OFF + blk * 8192u + sub, 16, 1024),
                                         sdesc_sw128(sb + kv_at(st, blk) + sub, 16, 1024), id, k > 0);
                            }
                        }
                        umma_commit(bar(B_S_FULL));
                        umma_commit(bar(B_SV_DONE + st));        // the stage may now be rescaled for P.V
                    }
                    i += nt;
                    if (i == s.ntiles && next_reloads) umma_commit(bar(B_Q_EMPTY));
                }
                g += s.ntiles;
                cur = nxt;
            }
            // drain: every MMA this thread issued has completed before TMEM is freed
            const uint32_t tb = bar(c == 0 ? B_TEARDOWN : c == 1 ? B_TEARDOWN_S2 : B_TEARDOWN_S3);
            umma_commit(tb);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(tb, 0) && globaltimer_ns() - t0 < kTimeoutNs) {
            }
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ======================= softmax / epilogue =======================
        // Warps 4-5 own the score rows (heads) and O[:, 0:256]; warps 6-7 own
        // O[:, 256:512] of the same heads.  Warps 4-5 publish each tile's
        // rescale factor and the unit's final (max, sum) through one-way
        // mbarriers; only warps 6-7 wait on them.
        const int r = tid - 128;             // TMEM lane == score row
        const bool head_row = r < 64;
        const int h = r & 63;
        const int wl = warp - 4;
        const uint32_t lane_base = static_cast<uint32_t>(wl * 32) << 16;
        const float sl2 = kp.scale_log2;
        const uint32_t id_pv = idesc_f16(128, 256, mma_bf16, false, true);
        const uint64_t p_desc = sdesc_sw128(sb + P_OFF, 16, 1024);                 // P.V's A base (warp 6)
        const uint64_t v_desc = sdesc_sw128(sb + kv_at(0, 0), KV_COL, 1024);       // P.V's B base, MN-major
        uint8_t *stage = base + EPI_OFF + static_cast<uint32_t>(wl) * 1024u;
        int g = 0, ks = 0;
        bool stop = false;
        Unit cur = first;
        for (int u = u_beg; u < u_end && !stop; ++u) {
            const Unit nxt = u + 1 < u_end ? unit_info(kp, sp, u + 1) : cur;
            const Unit &s = cur;
            const bool live_head = head_row && h < s.nh;
            float m = -INFINITY, l = 0.f;
            for (int i = 0; i < s.ntiles; ++i) {
                const int gi = g + i, st = gi & (kStages - 1), use = gi / kStages, pb = gi & 1;
                float alpha = 1.f;
                uint32_t pw[NT / 2];
                if (head_row) {
                    const int sbuf = EX ? 0 : st;
                    if (!warp_wait(bar(B_S_FULL + sbuf), EX ? (gi & 1) : (use & 1), abort_flag)) { stop = true; break; }
                    tc_fence_after();
                    // packed rows: the tile's scales were written with it (this
                    // wait orders them); plain rows wait after releasing S
                    if (EX && !warp_wait(bar(B_KV_FULL + st), use & 1, abort_flag)) { stop = true; break; }
                    uint32_t sv[NT];
                    if constexpr (!EX) {
                        uint32_t sa[NT / 2], sc[NT / 2];
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {        // the chains' partial sums of S, 16 columns at a time
                            tmem_ld16(tmem + lane_base + TM_S + st * NT + hf * 16, sa);
                            tmem_ld16(tmem + lane_base + TM_S + kStages * NT + st * NT + hf * 16, sc);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < NT / 2; ++j)
                                sv[hf * 16 + j] = __float_as_uint(__uint_as_float(sa[j]) + __uint_as_float(sc[j]));
#pragma unroll
                            for (int cc = 2; cc < kChains; ++cc) {       // the third chain (packed rows)
                                tmem_ld16(tmem + lane_base + TM_S + cc * kStages * NT + st * NT + hf * 16, sa);
                                tmem_wait_ld();
#pragma unroll
                                for (int j = 0; j < NT / 2; ++j)
                                    sv[hf * 16 + j] = __float_as_uint(__uint_as_float(sv[hf * 16 + j]) +
                                                                      __uint_as_float(sa[j]));
                            }
                        }
                    } else {
                        // S = sum over the four tiles of scale_t(row) x (q_t . k_t)
                        // (exact products of the unscaled values, scaled in fp32)
                        // plus the rope part, in a fixed order
                        // chains 0 and 4 first (the product and the rope part),
                        // then chains 1-3 folded in; the S buffer is released
                        // as soon as every chain is in registers
                        const float *sct = scl + st * 4 * NT;
                        uint32_t s0[NT], s1[NT];
                        tmem_ld16(tmem + lane_base + TM_S + 0 * NT, *reinterpret_cast<uint32_t(*)[16]>(&s0[0]));
                        tmem_ld16(tmem + lane_base + TM_S + 0 * NT + 16, *reinterpret_cast<uint32_t(*)[16]>(&s0[16]));
                        tmem_ld16(tmem + lane_base + TM_S + 4 * NT, *reinterpret_cast<uint32_t(*)[16]>(&s1[0]));
                        tmem_ld16(tmem + lane_base + TM_S + 4 * NT + 16, *reinterpret_cast<uint32_t(*)[16]>(&s1[16]));
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < NT; ++j)
                            sv[j] = __float_as_uint(fmaf(sct[j], __uint_as_float(s0[j]), __uint_as_float(s1[j])));
#pragma unroll
                        for (int cc = 1; cc < 4; ++cc) {
                            tmem_ld16(tmem + lane_base + TM_S + cc * NT, *reinterpret_cast<uint32_t(*)[16]>(&s0[0]));
                            tmem_ld16(tmem + lane_base + TM_S + cc * NT + 16, *reinterpret_cast<uint32_t(*)[16]>(&s0[16]));
                            tmem_wait_ld();
                            if (cc == 3) {
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0) mbar_arrive(bar(B_S_FREE + sbuf));
                            }
#pragma unroll
                            for (int j = 0; j < NT; ++j)
                                sv[j] = __float_as_uint(fmaf(sct[cc * NT + j], __uint_as_float(s0[j]), __uint_as_float(sv[j])));
                        }
                    }
                    if constexpr (!EX) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(B_S_FREE + sbuf));
                        // tile i landed before its S was computed; this wait
                        // only orders the row-mask word
                        if (!warp_wait(bar(B_KV_FULL + st), use & 1, abort_flag)) { stop = true; break; }
                    }
                    float x[NT];
                    if (live_head) {
                        const uint32_t vm = valid_s[st];
#pragma unroll
                        for (int j = 0; j < NT; ++j) x[j] = ((vm >> j) & 1u) ? __uint_as_float(sv[j]) : -INFINITY;
                        float mx[NT / 2];
#pragma unroll
                        for (int j = 0; j < NT / 2; ++j) mx[j] = fmaxf(x[2 * j], x[2 * j + 1]);
#pragma unroll
                        for (int w2 = NT / 4; w2 >= 1; w2 >>= 1)
#pragma unroll
                            for (int j = 0; j < w2; ++j) mx[j] = fmaxf(mx[j], mx[j + w2]);
                        const float tmax = mx[0] * sl2;   // softmax_scale > 0 keeps the arg-max
                        if (tmax > m + kRescaleThreshold) {
                            alpha = (m == -INFINITY) ? 0.f : fast_exp2(m - tmax);
                            m = tmax;
                        }
                    }
                    // the tile's rescale factor is final once its maximum is
                    // known: published before the exponentials, so warps 6-7
                    // (and the P.V issue behind them) need not wait for those
                    alpha_s[(gi & 3) * 64 + r] = alpha;      // four-slot ring, whatever the stage count
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_ALPHA + (gi & 3)));
                    if (live_head) {
                        float ps[NT / 2];
                        if (m == -INFINITY) {
#pragma unroll
                            for (int j = 0; j < NT / 2; ++j) {
                                ps[j] = 0.f;
                                pw[j] = 0u;
                            }
                        } else {
                            const float nm = -m;
#pragma unroll
                            for (int j = 0; j < NT / 2; ++j) {
                                const float p0 = fast_exp2(fmaf(x[2 * j], sl2, nm));
                                const float p1 = fast_exp2(fmaf(x[2 * j + 1], sl2, nm));
                                ps[j] = p0 + p1;
                                pw[j] = pack2(p0, p1, mma_bf16);
                            }
                        }
#pragma unroll
                        for (int w2 = NT / 4; w2 >= 1; w2 >>= 1)
#pragma unroll
                            for (int j = 0; j < w2; ++j) ps[j] += ps[j + w2];
                        l = l * alpha + ps[0];
                    }
                } else {
                    if constexpr (EX) {
                        // V of the tile: once every S product has read the
                        // stage, scale its unscaled NoPE values in place by
                        // their row's tile scale (rounded once to fp16) for P.V
                        if (!warp_wait(bar(B_KV_FULL + st), use & 1, abort_flag) ||
                            !warp_wait(bar(B_SV_DONE + st), use & 1, abort_flag)) {
                            stop = true;
                            break;
                        }
                        // thread t of warps 6-7 (t = 0..63) takes 16-byte
                        // position t % 8 of rows t / 8 + 8 j (j = 0..3) in all
                        // eight column blocks; a warp covers 512 contiguous bytes
                        const float *sct = scl + st * 4 * NT;
                        const int t64 = tid - 192, r0 = t64 >> 3;
                        uint8_t *p0 = base + kv_at(st, 0) + r0 * 128 + (t64 & 7) * 16;
#pragma unroll
                        for (int tile = 0; tile < 4; ++tile) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float sc = sct[tile * NT + r0 + 8 * j];
                                // the scale as fp16 when it is a normal fp16 value
                                // (V is then rounded twice, within the output
                                // tolerance); otherwise fp32 products
                                const bool h = fabsf(sc) >= 6.103515625e-05f && fabsf(sc) <= 65504.f;
                                const __half2 sh = __float2half2_rn(sc);
#pragma unroll
                                for (int b2 = 0; b2 < 2; ++b2) {
                                    uint4 *pc = reinterpret_cast<uint4 *>(p0 + (2 * tile + b2) * KV_COL + j * 1024);
                                    uint4 v = *pc;
                                    uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        if (h) {
                                            const __half2 r2 = __hmul2(*reinterpret_cast<const __half2 *>(&w4[e]), sh);
                                            w4[e] = *reinterpret_cast<const uint32_t *>(&r2);
                                        } else {
                                            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w4[e]));
                                            w4[e] = pack2(f.x * sc, f.y * sc, false);
                                        }
                                    }
                                    *pc = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                                }
                            }
                        }
                        fence_proxy_async_smem();        // generic-proxy writes -> the P.V product
                    }
                    if (!warp_wait(bar(B_ALPHA + (gi & 3)), (gi >> 2) & 1, abort_flag)) { stop = true; break; }
                    alpha = alpha_s[(gi & 3) * 64 + h];
                }
                // rescale this warp's half of O once P.V(i-1) has landed in it
                if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    const int gp = gi - 1;
                    if (!warp_wait(bar(B_O_DONE + (gp & 1)), (gp >> 1) & 1, abort_flag)) { stop = true; break; }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_base + TM_O + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                        tmem_st32(tmem + lane_base + TM_O + c * 32, o);
                    }
                    tmem_wait_st();
                }
                if (head_row) {
                    // P buffer pb was last read by P.V(i-2)
                    if (gi >= 2 && !warp_wait(bar(B_O_DONE + pb), ((gi - 2) >> 1) & 1, abort_flag)) {
                        stop = true;
                        break;
                    }
                    if (live_head) {
#pragma unroll
                        for (int c = 0; c < NT / 8; ++c)
                            *reinterpret_cast<uint4 *>(base + P_OFF + sw128(64 + r, pb * 4 + c)) =
                                make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_P_FULL + pb));
                if (warp == 6) {
                    // P.V(i) once all four warps have written P(i) / rescaled O
                    if (lane == 0) {
                        if (mbar_wait(bar(B_P_FULL + pb), (gi >> 1) & 1, abort_flag)) {
                            tc_fence_after();
                            // descriptors: bases plus compile-time offsets (the start-address
                            // field is address / 16 in the low 14 bits; operand addresses stay
                            // below 256 KB, so the add never carries out of it): P.V issues
                            // back to back instead of building each descriptor here
                            const uint64_t a_pb = p_desc + (pb * 64u >> 4);
                            const uint64_t b_st = v_desc + ((uint64_t)st * KV_BLOCK >> 4);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint32_t half = k >> 1, sub = k & 1;
                                const uint32_t a_off = ((half ? 0u : 8192u) + sub * 32u) >> 4;
                                const uint32_t b_off = (half * 4u * KV_COL + sub * 2048u) >> 4;
                                umma_f16(tmem + TM_O, a_pb + a_off, b_st + b_off, id_pv, (i > 0 || k > 0) ? 1u : 0u);
                            }
                            umma_commit(bar(B_KV_EMPTY + st));
                            umma_commit(bar(B_O_DONE + pb));
                        }
                    }
                    __syncwarp();
                    if (*abort_flag) { stop = true; break; }
                }
            }
            if (stop) break;
            // ---------------- epilogue ----------------
            const int gl = g + s.ntiles - 1;
            if (!warp_wait(bar(B_O_DONE + (gl & 1)), (gl >> 1) & 1, abort_flag)) break;
            tc_fence_after();
            float mm = m, ll = l;
            if (head_row) {
                stats_s[2 * r] = m;
                stats_s[2 * r + 1] = l;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_STATS));
            } else {
                if (!warp_wait(bar(B_STATS), ks & 1, abort_flag)) break;
                mm = stats_s[2 * h];
                ll = stats_s[2 * h + 1];
            }
            const bool final_split = s.nsplit == 1;
            const bool ws_ok = final_split || (kp.max_splits > 1 && s.w < kp.max_splits);
            const int64_t slot = (int64_t)s.t * kp.max_splits + s.w;
            if (!ws_ok && r == 0) set_status(kp, SFM_STATUS_WORKSPACE_OVERFLOW);
            float inv = 0.f;
            if (ll > 0.f) {
                float den = ll;
                if (final_split && kp.sinks) den += exp2f(__ldg(kp.sinks + s.h0 + h) * 1.4426950408889634f - mm);
                inv = 1.f / den;
            }
            // O out of TMEM (two 32-column chunks per wait), normalised and
            // packed to 16 bits.
            //  * a partial (bf16) goes to the workspace in chunk-major order
            //    ([split][dim / 8][head][8]): for each 8-dim chunk the 32
            //    lanes of a warp write 32 consecutive heads, 512 contiguous
            //    bytes per warp store, straight from registers;
            //  * a final split (output dtype) goes to the output rows through
            //    the warp's staging slice: each lane parks 32 bytes of its row
            //    (16-byte pieces rotated by lane), then lane L writes piece L%2
            //    of row 16k + L/2 (sixteen 32-byte row segments per store).
            const bool out_bf16 = final_split ? bf16 : true;
            const int dcol = head_row ? 0 : 256;
            const int hrow = (wl & 1) * 32 + lane;               // this lane's head within the group
            uint16_t *obase = final_split ? static_cast<uint16_t *>(kp.out) + ((int64_t)s.t * kp.q_n + s.h0) * 512
                                          : kp.ws_o + slot * kp.q_n * 512;
            const int srow = lane >> 1, spiece = lane & 1;
#pragma unroll 1
            for (int cc = 0; cc < 8; cc += 2) {
                uint32_t o[64];
                tmem_ld32(tmem + lane_base + TM_O + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
                tmem_ld32(tmem + lane_base + TM_O + cc * 32 + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
                tmem_wait_ld();
                // after the last chunk, TMEM is free for the next unit once
                // this warp's next P arrival (which follows this fence) completes
                if (cc == 6) tc_fence_before();
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    pk[j] = pack2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv, out_bf16);
                if (!final_split) {
                    if (ws_ok && hrow < s.nh) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {            // 8-dim chunk (dcol + 32 cc) / 8 + q
                            const int chunk = (dcol + cc * 32) / 8 + q;
                            *reinterpret_cast<uint4 *>(obase + ((int64_t)chunk * kp.q_n + s.h0 + hrow) * 8) =
                                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                        }
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < 4; ++r) {                // 16 columns per round
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            *reinterpret_cast<uint4 *>(stage + lane * 32 + ((q ^ (lane & 1)) << 4)) =
                                make_uint4(pk[r * 8 + 4 * q], pk[r * 8 + 4 * q + 1], pk[r * 8 + 4 * q + 2],
                                           pk[r * 8 + 4 * q + 3]);
                        __syncwarp();
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const int lr = k * 16 + srow, hh = (wl & 1) * 32 + lr;
                            const uint4 v =
                                *reinterpret_cast<const uint4 *>(stage + lr * 32 + ((spiece ^ (lr & 1)) << 4));
                            if (hh < s.nh)
                                *reinterpret_cast<uint4 *>(obase + (int64_t)hh * 512 + dcol + cc * 32 + r * 16 +
                                                           spiece * 8) = v;
                        }
                    }
                }
            }
            __syncwarp();
            if (head_row && h < s.nh && ws_ok) {
                const float lse = ll > 0.f ? (mm + log2f(ll)) * 0.6931471805599453f : -INFINITY;
                if (final_split) {
                    if (kp.lse) kp.lse[(int64_t)s.t * kp.q_n + s.h0 + h] = lse;
                } else {
                    kp.ws_lse[slot * kp.q_n + s.h0 + h] = lse;
                }
            }
            g += s.ntiles;
            ++ks;
            cur = nxt;
        }
    }

    if (warp == 6 && lane == 0) {
        // every P.V issued by this thread has completed before TMEM is freed
        umma_commit(bar(B_TEARDOWN_PV));
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar(B_TEARDOWN_PV), 0) && globaltimer_ns() - t0 < kTimeoutNs) {
        }
    }
    __syncwarp();

    if (kp.max_splits <= 1) {
        // at most one split per row: every row with attended positions was
        // finished by its unit and no combine kernel follows
        finish_rows_without_split(kp.meta, meta_ok(kp), kp.G, kp.T, kp.q_n, kp.out, kp.lse, kp.status);
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort_flag) set_status(kp, SFM_STATUS_TIMEOUT);
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int MODE>
cudaError_t launch_tc(const KParams &kp, cudaStream_t st)
{
    constexpr uint32_t smem = Lay<MODE>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(sfm_attn_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(sfm_attn_tc_kernel<MODE>, dim3(kp.G), dim3(kThreads), (size_t)smem, st, kp);
}

}  // namespace

cudaError_t launch_attn_tc(const KParams &kp, cudaStream_t st)
{
    // E4M3 rows: exact scores (see MODE 2); int8 rows: one fp16 rounding of
    // value x scale, which keeps the LSE far inside the tolerance
    if (!kp.packed) return launch_tc<0>(kp, st);
    return kp.kv_fp8 ? launch_tc<2>(kp, st) : launch_tc<1>(kp, st);
}

}  // namespace sfm
