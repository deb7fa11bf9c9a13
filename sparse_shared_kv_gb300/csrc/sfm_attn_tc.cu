// sfm_attn_tc.cu -- tensor-core (tcgen05 / TMEM) split-KV attention for
// plain bf16 / fp16 KV rows.
//
// One persistent CTA per SM walks the work units the planner gave its worker;
// a unit is one split for one group of up to 64 query heads (128 heads make
// two units per split, whose second pass over the split's rows hits L2).
// Per 64-row KV tile of a split:
//   producer warps 0-1   resolve the attended rows (window / compressed /
//                        indices through the block tables) and stream each
//                        1 KB row with cp.async into a 128-byte-swizzled
//                        shared-memory stage (two stages);
//   MMA warp 2           S = Q.K~^T            (M=128, N=64,  K=512)   -> TMEM
//                        O += P.V~             (M=128, N=256, K=2x64)  -> TMEM
//                        both reading the SAME staged tile (K-major for S,
//                        MN-major for P.V);
//   softmax warps 4-7    one thread per score row: scale, mask, running max
//                        with lazy rescaling, exp2, row sum, P (bf16/fp16)
//                        into shared memory; the epilogue normalises O and
//                        writes the output (single split) or the split's
//                        partial O and LSE for the combine kernel.
//
// M=128 rows with at most 64 heads: the upper 64 rows of the Q operand alias
// the next column block (their scores are never read), and O uses a
// block-diagonal P so that TMEM rows 0-63 accumulate O[:, 0:256] and rows
// 64-127 accumulate O[:, 256:512] in 256 columns: A = [P;0] with V[:, :256]
// for the first 64 reduction steps, A = [0;P] with V[:, 256:] for the next.
//
// Softmax follows the pages' definition (S = Q.K~^T * softmax_scale, softmax
// over the attended rows, LSE = max S + log sum exp(S - max S)); scores are
// kept in the log2 domain (x = S * log2 e) and the running max is only moved
// when a row's max grows by more than 8 (a factor 256), which leaves O / l
// unchanged mathematically and keeps fp32 far from overflow.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "sfm_internal.cuh"
#include "sfm_tc.cuh"

namespace sfm {

namespace {

using namespace tc;

constexpr int NT = 64;                       // KV rows per tile
constexpr int kThreads = 256;
constexpr uint32_t Q_OFF = 0;                // 8 blocks x 64 rows x 128 B
constexpr uint32_t P_OFF = 65536;            // 192 rows x 128 B: [0..63] zero, [64..127] P, [128..191] zero
constexpr uint32_t KV_OFF = 90112;           // 2 stages x 64 KB
constexpr uint32_t KV_STAGE = 65536;
constexpr uint32_t MISC_OFF = KV_OFF + 2 * KV_STAGE;   // 221184
constexpr uint32_t kSmemBytes = MISC_OFF + 1536 + 1024;   // misc block (1280 B used) + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_O = 0;                 // O: columns [0, 256)
constexpr uint32_t TM_S = 256;               // S buffers: [256, 320), [320, 384)
constexpr float kRescaleThreshold = 8.0f;    // log2 units

// barrier slots (8 bytes each) at MISC_OFF
enum Bar {
    B_KV_FULL = 0, B_KV_EMPTY = 2, B_S_FULL = 4, B_S_FREE = 6, B_P_FULL = 8, B_O_DONE = 9, B_Q_FULL = 10,
    B_Q_EMPTY = 11, B_O_FREE = 12, B_TEARDOWN = 13, B_ALPHA = 14, B_STATS = 16, kNumBars = 17
};
constexpr uint32_t TMEM_SLOT_OFF = MISC_OFF + 128;
constexpr uint32_t ABORT_OFF = MISC_OFF + 132;
constexpr uint32_t VALID_OFF = MISC_OFF + 144;   // [2 stages][2 words]
constexpr uint32_t ALPHA_OFF = MISC_OFF + 256;   // [2][64] floats
constexpr uint32_t STATS_OFF = MISC_OFF + 768;   // [64][2] floats

struct SplitInfo {
    int t, sidx, nsplit, pos0, pos1, ntiles;
    Tok k;
};

// The split's row and that row's lengths / window / position counts come
// from the plan (two dependent loads instead of a search and a length walk).
__device__ __forceinline__ SplitInfo split_info(const KParams &kp, const int32_t *sp, int w)
{
    SplitInfo s;
    s.t = kp.meta[meta_own_off(kp.G, kp.T) + w];
    const int32_t *rec = kp.meta + meta_rec_off(kp.G, kp.T) + (int64_t)kRecWords * s.t;
    const int s_beg = sp[s.t], s_end = sp[s.t + 1];
    s.nsplit = s_end - s_beg;
    s.sidx = w - s_beg;
    Tok &k = s.k;
    k.b = rec[0];
    k.kv_len = rec[1];
    k.cmp_len = rec[2];
    k.p_cmp = rec[3];
    k.lo = rec[4];
    k.hi = rec[5];
    k.n_ori = rec[6];
    k.n_cmp = rec[7];
    k.i = 0;
    k.q_len = 0;
    k.p = 0;
    k.valid = 1;
    const int n = k.n_ori + k.n_cmp;
    s.pos0 = s.sidx * kp.split_rows;
    s.pos1 = min(n, s.pos0 + kp.split_rows);
    const int rows = s.pos1 > s.pos0 ? s.pos1 - s.pos0 : 0;
    s.ntiles = rows > 0 ? (rows + NT - 1) / NT : 1;   // an empty split still runs one masked tile
    return s;
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

__global__ void __launch_bounds__(kThreads, 1) sfm_attn_tc_kernel(KParams kp)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(base);
    const uint32_t bar0 = sb + MISC_OFF;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + ABORT_OFF);
    uint32_t *valid_s = reinterpret_cast<uint32_t *>(base + VALID_OFF);
    float *alpha_s = reinterpret_cast<float *>(base + ALPHA_OFF);
    float *stats_s = reinterpret_cast<float *>(base + STATS_OFF);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool bf16 = kp.dtype == SFM_DTYPE_BF16;
    grid_launch_dependents();    // the combine kernel may launch; it waits for this grid

    // ---------------- set-up ----------------
    for (uint32_t i = tid; i < 24576u / 16u; i += kThreads)
        reinterpret_cast<uint4 *>(base + P_OFF)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        mbar_init(bar(B_KV_FULL + 0), 66);   // 64 copy-completion arrivals + 2 row-mask words
        mbar_init(bar(B_KV_FULL + 1), 66);
        mbar_init(bar(B_KV_EMPTY + 0), 1);
        mbar_init(bar(B_KV_EMPTY + 1), 1);
        mbar_init(bar(B_S_FULL + 0), 1);
        mbar_init(bar(B_S_FULL + 1), 1);
        mbar_init(bar(B_S_FREE + 0), 128);
        mbar_init(bar(B_S_FREE + 1), 128);
        mbar_init(bar(B_P_FULL), 128);
        mbar_init(bar(B_O_DONE), 1);
        mbar_init(bar(B_Q_FULL), 64);
        mbar_init(bar(B_Q_EMPTY), 1);
        mbar_init(bar(B_O_FREE), 128);
        mbar_init(bar(B_TEARDOWN), 1);
        mbar_init(bar(B_ALPHA + 0), 64);
        mbar_init(bar(B_ALPHA + 1), 64);
        mbar_init(bar(B_STATS), 64);
        *abort_flag = 0;
        fence_barrier_init();
    }
    fence_proxy_async_smem();
    if (warp == 2) {
        tmem_alloc(sb + TMEM_SLOT_OFF, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(base + TMEM_SLOT_OFF);

    // everything above overlapped the planner; the plan is read from here on
    grid_dependency_wait();
    const bool ok = meta_ok(kp);
    const int worker = blockIdx.x;
    const int32_t *sp = kp.meta + meta_split_off(kp.G);
    const int w_beg = ok ? kp.meta[meta_ws_off() + worker] : 0;
    const int w_end = ok ? kp.meta[meta_ws_off() + worker + 1] : 0;

    if (warp < 2) {
        // ======================= producer =======================
        // Thread pt owns tile row pt (and Q head row pt).  Copies arrive on the
        // stage barrier by themselves when they land (cp.async.mbarrier), so
        // the producer never waits for its own loads; it only waits for a
        // free stage.  Rows are resolved one tile ahead of the tile in flight.
        const int pt = tid;
        const uint8_t *zero_src = static_cast<const uint8_t *>(kp.q);
        int g = 0, ks = 0;
        bool stop = false;
        for (int u = w_beg; u < w_end && !stop; ++u) {
            const int w = u / kp.head_groups, h0 = (u - w * kp.head_groups) * 64;
            const int nh = min(64, kp.q_n - h0);
            const SplitInfo s = split_info(kp, sp, w);
            if (ks > 0 && !warp_wait(bar(B_Q_EMPTY), (ks - 1) & 1, abort_flag)) break;
            {
                // Q rows of this warp's 32 heads, one 1 KB row per step: lane L
                // copies 16-byte chunks L and L + 32 (512 contiguous bytes per
                // instruction)
                const uint8_t *qrow = static_cast<const uint8_t *>(kp.q) + ((int64_t)s.t * kp.q_n + h0) * 1024;
                for (int rr = 0; rr < 32; ++rr) {
                    const int hh = warp * 32 + rr;
                    const bool live = hh < nh;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int C = lane + half * 32;
                        const uint32_t dst = sb + Q_OFF + (C >> 3) * 8192u + sw128(hh, C & 7);
                        cp_async16(dst, live ? qrow + (int64_t)hh * 1024 + C * 16 : zero_src, live ? 16u : 0u);
                    }
                }
                cp_async_arrive_noinc(bar(B_Q_FULL));
            }
            auto resolve = [&](int i) -> const uint8_t * {
                const int pos = s.pos0 + i * NT + pt;
                if (pos >= s.pos1) return nullptr;
                int logical, src;
                return resolve_row(kp, s.k, s.t, pos, &logical, &src);
            };
            const uint8_t *rp[2];
            rp[0] = resolve(0);
            rp[1] = s.ntiles > 1 ? resolve(1) : nullptr;      // independent chains overlap
            for (int i = 0; i < s.ntiles; ++i, ++g) {
                const int st = g & 1, use = g >> 1;
                if (use >= 1 && !warp_wait(bar(B_KV_EMPTY + st), (use - 1) & 1, abort_flag)) {
                    stop = true;
                    break;
                }
                const uint8_t *row = rp[i & 1];
                __syncwarp();
                const uint32_t vm = __ballot_sync(0xffffffffu, row != nullptr);
                const uint32_t stage = sb + KV_OFF + st * KV_STAGE;
                // this warp's 32 tile rows, one row per step (pointer broadcast
                // from the lane that resolved it): 512 contiguous bytes per
                // warp instruction
                const unsigned long long my_row = reinterpret_cast<unsigned long long>(row);
                for (int rr = 0; rr < 32; ++rr) {
                    const uint8_t *src = reinterpret_cast<const uint8_t *>(__shfl_sync(0xffffffffu, my_row, rr));
                    const int tr = warp * 32 + rr;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int C = lane + half * 32;
                        const uint32_t dst = stage + (C >> 3) * 8192u + sw128(tr, C & 7);
                        cp_async16(dst, src ? src + C * 16 : zero_src, src ? 16u : 0u);
                    }
                }
                cp_async_arrive_noinc(bar(B_KV_FULL + st));
                if (lane == 0) {
                    valid_s[st * 2 + warp] = vm;          // this warp's 32 row-valid bits
                    mbar_arrive(bar(B_KV_FULL + st));     // release: the word is visible with the phase
                }
                // the next tile was resolved earlier; resolve the one after it now,
                // behind the copies in flight
                if (i >= 1 && i + 1 < s.ntiles) rp[(i + 1) & 1] = resolve(i + 1);
            }
            ++ks;
        }
        cp_async_wait<0>();
    } else if (warp == 2) {
        // ======================= MMA issuer =======================
        // One thread polls both inputs and issues whichever product is ready:
        // S(i) needs tile i staged and its S buffer free; P.V(i) needs P(i)
        // (and, for a split's first tile, the previous epilogue done with O).
        if (lane == 0) {
            const uint32_t id_s = idesc_f16(128, 64, bf16, false, false);
            const uint32_t id_pv = idesc_f16(128, 256, bf16, false, true);
            int g = 0, ks = 0;
            bool stop = false;
            for (int u = w_beg; u < w_end && !stop; ++u) {
                const int w = u / kp.head_groups;
                const SplitInfo s = split_info(kp, sp, w);
                if (!mbar_wait(bar(B_Q_FULL), ks & 1, abort_flag)) break;
                fence_proxy_async_smem();       // cp.async (generic proxy) writes -> tensor-core reads
                tc_fence_after();
                int ns = 0, npv = 0;             // next tile to issue S / P.V for
                uint64_t t_idle = 0;
                while (npv < s.ntiles) {
                    bool progressed = false;
                    if (ns < s.ntiles) {
                        const int gi = g + ns, st = gi & 1;
                        if (mbar_test(bar(B_KV_FULL + st), (gi >> 1) & 1) &&
                            (gi < 2 || mbar_test(bar(B_S_FREE + st), ((gi >> 1) - 1) & 1))) {
                            fence_proxy_async_smem();
                            tc_fence_after();
                            const uint32_t d = tmem + TM_S + st * 64;
                            const uint32_t kv = sb + KV_OFF + st * KV_STAGE;
#pragma unroll 8
                            for (int k = 0; k < 32; ++k) {
                                const uint32_t off = (k >> 2) * 8192u + (k & 3) * 32u;
                                umma_f16(d, sdesc_sw128(sb + Q_OFF + off, 16, 1024),
                                         sdesc_sw128(kv + off, 16, 1024), id_s, k > 0);
                            }
                            umma_commit(bar(B_S_FULL + st));
                            if (ns == s.ntiles - 1) umma_commit(bar(B_Q_EMPTY));
                            ++ns;
                            progressed = true;
                        }
                    }
                    if (npv < ns) {
                        const int gj = g + npv, st = gj & 1;
                        if (mbar_test(bar(B_P_FULL), gj & 1) &&
                            (npv > 0 || ks == 0 || mbar_test(bar(B_O_FREE), (ks - 1) & 1))) {
                            tc_fence_after();
                            const uint32_t kv = sb + KV_OFF + st * KV_STAGE;
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const int half = k >> 2, sub = k & 3;
                                const uint32_t a = sb + P_OFF + (half ? 0u : 8192u) + sub * 32u;
                                const uint32_t b = kv + half * 32768u + sub * 2048u;
                                umma_f16(tmem + TM_O, sdesc_sw128(a, 16, 1024), sdesc_sw128(b, 8192, 1024), id_pv,
                                         !(npv == 0 && k == 0));
                            }
                            umma_commit(bar(B_KV_EMPTY + st));
                            umma_commit(bar(B_O_DONE));
                            ++npv;
                            progressed = true;
                        }
                    }
                    if (progressed) {
                        t_idle = 0;
                    } else {
                        if (*abort_flag) { stop = true; break; }
                        const uint64_t now = globaltimer_ns();
                        if (t_idle == 0) t_idle = now;
                        else if (now - t_idle > kTimeoutNs) {
                            *abort_flag = 1;
                            stop = true;
                            break;
                        }
                    }
                }
                g += s.ntiles;
                ++ks;
            }
            // drain: every MMA issued so far has completed before TMEM is freed
            umma_commit(bar(B_TEARDOWN));
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar(B_TEARDOWN), 0) && globaltimer_ns() - t0 < kTimeoutNs) {
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ======================= softmax / epilogue =======================
        // Warps 4-5 own the score rows (heads) and O[:, 0:256]; warps 6-7 own
        // O[:, 256:512] of the same heads.  Warps 4-5 publish each tile's
        // rescale factor and the final (max, sum) through one-way mbarriers;
        // only warps 6-7 wait on them.
        const int r = tid - 128;             // TMEM lane == score row
        const bool head_row = r < 64;
        const int h = r & 63;
        const uint32_t lane_base = static_cast<uint32_t>((warp - 4) * 32) << 16;
        const float sl2 = kp.scale_log2;
        // epilogue staging: 2 KB per warp in P rows 64..127 (idle during the epilogue)
        uint8_t *stage = base + P_OFF + 8192u + static_cast<uint32_t>(warp - 4) * 2048u;
        int g = 0, ks = 0;
        for (int u = w_beg; u < w_end; ++u) {
            const int w = u / kp.head_groups, h0 = (u - w * kp.head_groups) * 64;
            const int nh = min(64, kp.q_n - h0);
            const SplitInfo s = split_info(kp, sp, w);
            float m = -INFINITY, l = 0.f;
            bool stop = false;
            for (int i = 0; i < s.ntiles; ++i) {
                const int gi = g + i, st = gi & 1;
                if (!warp_wait(bar(B_S_FULL + st), (gi >> 1) & 1, abort_flag)) { stop = true; break; }
                tc_fence_after();
                float alpha = 1.f;
                uint32_t pw[32];
                const bool live_head = head_row && h < nh;
                if (head_row) {
                    uint32_t sv[64];
                    tmem_ld32(tmem + lane_base + TM_S + st * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                    tmem_ld32(tmem + lane_base + TM_S + st * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(bar(B_S_FREE + st));
                    if (!warp_wait(bar(B_KV_FULL + st), (gi >> 1) & 1, abort_flag)) { stop = true; break; }
                    if (live_head) {
                        const uint32_t v0 = valid_s[st * 2 + 0], v1 = valid_s[st * 2 + 1];
                        float x[64];
#pragma unroll
                        for (int j = 0; j < 64; ++j) x[j] = __uint_as_float(sv[j]);
                        if ((v0 & v1) != 0xffffffffu) {
#pragma unroll
                            for (int j = 0; j < 64; ++j)
                                if (!(((j < 32 ? v0 >> j : v1 >> (j - 32)) & 1u))) x[j] = -INFINITY;
                        }
                        float mx[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) mx[j] = fmaxf(x[2 * j], x[2 * j + 1]);
#pragma unroll
                        for (int w2 = 16; w2 >= 1; w2 >>= 1)
#pragma unroll
                            for (int j = 0; j < w2; ++j) mx[j] = fmaxf(mx[j], mx[j + w2]);
                        const float tmax = mx[0] * sl2;   // softmax_scale > 0 keeps the arg-max
                        if (tmax > m + kRescaleThreshold) {
                            alpha = (m == -INFINITY) ? 0.f : fast_exp2(m - tmax);
                            m = tmax;
                        }
                        float ps[32];
                        if (m == -INFINITY) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                ps[j] = 0.f;
                                pw[j] = 0u;
                            }
                        } else {
                            const float nm = -m;
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const float p0 = fast_exp2(fmaf(x[2 * j], sl2, nm));
                                const float p1 = fast_exp2(fmaf(x[2 * j + 1], sl2, nm));
                                ps[j] = p0 + p1;
                                pw[j] = pack2(p0, p1, bf16);
                            }
                        }
#pragma unroll
                        for (int w2 = 16; w2 >= 1; w2 >>= 1)
#pragma unroll
                            for (int j = 0; j < w2; ++j) ps[j] += ps[j + w2];
                        l = l * alpha + ps[0];
                    }
                    alpha_s[(gi & 1) * 64 + r] = alpha;
                    mbar_arrive(bar(B_ALPHA + (gi & 1)));
                } else {
                    tc_fence_before();
                    mbar_arrive(bar(B_S_FREE + st));
                    if (!warp_wait(bar(B_ALPHA + (gi & 1)), (gi >> 1) & 1, abort_flag)) { stop = true; break; }
                    alpha = alpha_s[(gi & 1) * 64 + h];
                }
                if (gi >= 1 && !warp_wait(bar(B_O_DONE), (gi - 1) & 1, abort_flag)) { stop = true; break; }
                tc_fence_after();
                if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
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
                // the previous split's epilogue staged O through P rows 64..127:
                // all four warps must be done with it before a new P lands there
                if (i == 0 && ks > 0 && head_row && !warp_wait(bar(B_O_FREE), (ks - 1) & 1, abort_flag)) {
                    stop = true;
                    break;
                }
                if (live_head) {
                    uint8_t *prow = base + P_OFF;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(prow + sw128(64 + r, c)) =
                            make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(B_P_FULL));
            }
            if (stop) break;
            // ---------------- epilogue ----------------
            const int gl = g + s.ntiles - 1;
            if (!warp_wait(bar(B_O_DONE), gl & 1, abort_flag)) break;
            tc_fence_after();
            float mm = m, ll = l;
            if (head_row) {
                stats_s[2 * r] = m;
                stats_s[2 * r + 1] = l;
                mbar_arrive(bar(B_STATS));
            } else {
                if (!warp_wait(bar(B_STATS), ks & 1, abort_flag)) break;
                mm = stats_s[2 * h];
                ll = stats_s[2 * h + 1];
            }
            const bool final_split = s.nsplit == 1;
            const bool ws_ok = final_split || w < kp.ws_capacity_splits;
            if (!ws_ok && r == 0) set_status(kp, SFM_STATUS_WORKSPACE_OVERFLOW);
            float inv = 0.f;
            if (ll > 0.f) {
                float den = ll;
                if (final_split && kp.sinks) den += exp2f(__ldg(kp.sinks + h0 + h) * 1.4426950408889634f - mm);
                inv = 1.f / den;
            }
            // Coalesced stores: each thread parks its row chunk in its warp's
            // staging slice (64 B per row, 16-byte pieces rotated by row), then
            // lane L writes piece L%4 of row 8k + L/4: a warp store covers
            // eight whole 64-byte row segments.
            const int wl = warp - 4;
            const int srow = lane >> 2, spiece = lane & 3;
            auto rd_row = [&](int k) { return k * 8 + srow; };          // local row read back by this lane
            auto row_head = [&](int lr) { return (wl * 32 + lr) & 63; };
            auto row_dcol = [&](int lr) { return (wl * 32 + lr) < 64 ? 0 : 256; };
            if (final_split) {
                uint16_t *obase = static_cast<uint16_t *>(kp.out) + ((int64_t)s.t * kp.q_n + h0) * 512;
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {                    // 32 columns per chunk
                    uint32_t o[32];
                    __syncwarp();
                    tmem_ld32(tmem + lane_base + TM_O + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int j = q * 8;
                        *reinterpret_cast<uint4 *>(stage + lane * 64 + ((q ^ (lane & 3)) << 4)) = make_uint4(
                            pack2(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv, bf16),
                            pack2(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv, bf16),
                            pack2(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv, bf16),
                            pack2(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv, bf16));
                    }
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int lr = rd_row(k), hh = row_head(lr);
                        const uint4 v = *reinterpret_cast<const uint4 *>(stage + lr * 64 + ((spiece ^ (lr & 3)) << 4));
                        if (hh < nh)
                            *reinterpret_cast<uint4 *>(obase + (int64_t)hh * 512 + row_dcol(lr) + c * 32 + spiece * 8) = v;
                    }
                }
            } else if (ws_ok) {
                float *wbase = kp.ws_o + ((int64_t)w * kp.q_n + h0) * 512;
#pragma unroll 1
                for (int c = 0; c < 16; ++c) {                   // 16 columns per chunk
                    uint32_t o[16];
                    __syncwarp();
                    tmem_ld16(tmem + lane_base + TM_O + c * 16, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<float4 *>(stage + lane * 64 + ((q ^ (lane & 3)) << 4)) = make_float4(
                            __uint_as_float(o[4 * q]) * inv, __uint_as_float(o[4 * q + 1]) * inv,
                            __uint_as_float(o[4 * q + 2]) * inv, __uint_as_float(o[4 * q + 3]) * inv);
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int lr = rd_row(k), hh = row_head(lr);
                        const float4 v = *reinterpret_cast<const float4 *>(stage + lr * 64 + ((spiece ^ (lr & 3)) << 4));
                        if (hh < nh)
                            *reinterpret_cast<float4 *>(wbase + (int64_t)hh * 512 + row_dcol(lr) + c * 16 + spiece * 4) = v;
                    }
                }
            }
            __syncwarp();
            if (head_row && h < nh && ws_ok) {
                const float lse = ll > 0.f ? (mm + log2f(ll)) * 0.6931471805599453f : -INFINITY;
                const int64_t row = (int64_t)s.t * kp.q_n + h0 + h;
                if (final_split) {
                    if (kp.lse) kp.lse[row] = lse;
                } else {
                    kp.ws_lse[(int64_t)w * kp.q_n + h0 + h] = lse;
                }
            }
            tc_fence_before();
            mbar_arrive(bar(B_O_FREE));
            g += s.ntiles;
            ++ks;
        }
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort_flag) set_status(kp, SFM_STATUS_TIMEOUT);
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_attn_tc(const KParams &kp, cudaStream_t st)
{
    cudaError_t e = cudaFuncSetAttribute(sfm_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_dependent(sfm_attn_tc_kernel, dim3(kp.G), dim3(kThreads), kSmemBytes, st, kp);
}

}  // namespace sfm
