// sfm_attn_tc.cu -- tensor-core (tcgen05 / TMEM) split-KV attention for up
// to 64 query heads with plain bf16 / fp16 KV rows.
//
// One persistent CTA per SM walks the splits the planner gave its worker.
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
    B_Q_EMPTY = 11, B_O_FREE = 12, B_TEARDOWN = 13, B_SM_SYNC = 14, kNumBars = 15
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
    const bool ok = meta_ok(kp);
    const bool bf16 = kp.dtype == SFM_DTYPE_BF16;

    // ---------------- set-up ----------------
    for (uint32_t i = tid; i < 24576u / 16u; i += kThreads)
        reinterpret_cast<uint4 *>(base + P_OFF)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        mbar_init(bar(B_KV_FULL + 0), 64);
        mbar_init(bar(B_KV_FULL + 1), 64);
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
        mbar_init(bar(B_SM_SYNC), 128);
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

    const int worker = blockIdx.x;
    const int32_t *sp = kp.meta + meta_split_off(kp.G);
    const int w_beg = ok ? kp.meta[meta_ws_off() + worker] : 0;
    const int w_end = ok ? kp.meta[meta_ws_off() + worker + 1] : 0;

    if (warp < 2) {
        // ======================= producer =======================
        const int pt = tid;                 // tile row / Q head handled by this thread
        uint32_t pend_bar[3];
        int pend = 0;
        auto flush_one = [&]() {
            if (pend >= 3) cp_async_wait<2>();
            else if (pend == 2) cp_async_wait<1>();
            else cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(pend_bar[0]);
            pend_bar[0] = pend_bar[1];
            pend_bar[1] = pend_bar[2];
            --pend;
        };
        const uint8_t *zero_src = static_cast<const uint8_t *>(kp.q);
        int g = 0, ks = 0;
        bool stop = false;
        for (int w = w_beg; w < w_end && !stop; ++w) {
            const SplitInfo s = split_info(kp, sp, w);
            // Q of the query row (all 64 head rows; heads >= q_n are zero)
            while (pend) flush_one();
            if (ks > 0 && !warp_wait(bar(B_Q_EMPTY), (ks - 1) & 1, abort_flag)) break;
            __syncwarp();
            {
                const bool live = pt < kp.q_n;
                const uint8_t *src = live ? static_cast<const uint8_t *>(kp.q) +
                                                ((int64_t)s.t * kp.q_n + pt) * 1024
                                          : zero_src;
                for (int C = 0; C < 64; ++C) {
                    const uint32_t dst = sb + Q_OFF + (C >> 3) * 8192u + sw128(pt, C & 7);
                    cp_async16(dst, live ? src + C * 16 : zero_src, live ? 16u : 0u);
                }
                cp_async_commit();
                pend_bar[pend++] = bar(B_Q_FULL);
            }
            // rows of tile 0 resolve while Q streams in; tile i+1 resolves while
            // tile i streams in and while waiting for a free stage
            auto resolve = [&](int i) -> const uint8_t * {
                const int pos = s.pos0 + i * NT + pt;
                if (pos >= s.pos1) return nullptr;
                int logical, src;
                return resolve_row(kp, s.k, s.t, pos, &logical, &src);
            };
            const uint8_t *rp = resolve(0);
            const uint8_t *rp_next = s.ntiles > 1 ? resolve(1) : nullptr;   // independent chains overlap
            for (int i = 0; i < s.ntiles; ++i, ++g) {
                const int st = g & 1, use = g >> 1;
                if (use >= 1) {
                    // never block while holding copies whose arrival is deferred:
                    // the MMA warp may be waiting for exactly those rows
                    const bool ready = __all_sync(0xffffffffu, mbar_test(bar(B_KV_EMPTY + st), (use - 1) & 1));
                    if (!ready) {
                        while (pend) flush_one();
                        if (!warp_wait(bar(B_KV_EMPTY + st), (use - 1) & 1, abort_flag)) {
                            stop = true;
                            break;
                        }
                    }
                }
                __syncwarp();
                const uint32_t vm = __ballot_sync(0xffffffffu, rp != nullptr);
                if (lane == 0) valid_s[st * 2 + warp] = vm;
                const uint32_t stage = sb + KV_OFF + st * KV_STAGE;
                for (int C = 0; C < 64; ++C) {
                    const uint32_t dst = stage + (C >> 3) * 8192u + sw128(pt, C & 7);
                    cp_async16(dst, rp ? rp + C * 16 : zero_src, rp ? 16u : 0u);
                }
                cp_async_commit();
                pend_bar[pend++] = bar(B_KV_FULL + st);
                rp = rp_next;
                rp_next = i + 2 < s.ntiles ? resolve(i + 2) : nullptr;
                while (pend > 1) flush_one();
            }
            ++ks;
        }
        while (pend) flush_one();
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
            for (int w = w_beg; w < w_end && !stop; ++w) {
                const SplitInfo s = split_info(kp, sp, w);
                if (!mbar_wait(bar(B_Q_FULL), ks & 1, abort_flag)) break;
                tc_fence_after();
                int ns = 0, npv = 0;             // next tile to issue S / P.V for
                uint64_t t_idle = 0;
                while (npv < s.ntiles) {
                    bool progressed = false;
                    if (ns < s.ntiles) {
                        const int gi = g + ns, st = gi & 1;
                        if (mbar_test(bar(B_KV_FULL + st), (gi >> 1) & 1) &&
                            (gi < 2 || mbar_test(bar(B_S_FREE + st), ((gi >> 1) - 1) & 1))) {
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
        const int r = tid - 128;             // TMEM lane == score row
        const bool head_row = r < 64;
        const int h = r & 63;
        const uint32_t lane_base = static_cast<uint32_t>((warp - 4) * 32) << 16;
        const float sl2 = kp.scale_log2;
        int g = 0, ks = 0;
        uint32_t nsync = 0;                  // uses of the softmax-group barrier
        auto group_sync = [&]() -> bool {
            mbar_arrive(bar(B_SM_SYNC));
            return warp_wait(bar(B_SM_SYNC), (nsync++) & 1, abort_flag);
        };
        for (int w = w_beg; w < w_end; ++w) {
            const SplitInfo s = split_info(kp, sp, w);
            float m = -INFINITY, l = 0.f;
            bool stop = false;
            for (int i = 0; i < s.ntiles; ++i) {
                const int gi = g + i, st = gi & 1;
                if (!warp_wait(bar(B_S_FULL + st), (gi >> 1) & 1, abort_flag)) { stop = true; break; }
                tc_fence_after();
                uint32_t sv[64];
                if (warp < 6) {
                    tmem_ld32(tmem + lane_base + TM_S + st * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
                    tmem_ld32(tmem + lane_base + TM_S + st * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
                    tmem_wait_ld();
                }
                tc_fence_before();
                mbar_arrive(bar(B_S_FREE + st));
                if (!warp_wait(bar(B_KV_FULL + st), (gi >> 1) & 1, abort_flag)) { stop = true; break; }
                float alpha = 1.f;
                uint32_t pw[32];
                const bool live_head = head_row && h < kp.q_n;
                if (live_head) {
                    const uint32_t v0 = valid_s[st * 2 + 0], v1 = valid_s[st * 2 + 1];
                    float x[64];
                    float tmax = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const bool v = ((j < 32 ? v0 >> j : v1 >> (j - 32)) & 1u) != 0;
                        x[j] = v ? __uint_as_float(sv[j]) * sl2 : -INFINITY;
                        tmax = fmaxf(tmax, x[j]);
                    }
                    if (tmax > m + kRescaleThreshold) {
                        alpha = (m == -INFINITY) ? 0.f : exp2f(m - tmax);
                        m = tmax;
                    }
                    float sum = 0.f;
#pragma unroll
                    for (int j = 0; j < 64; j += 2) {
                        const float p0 = (m == -INFINITY) ? 0.f : exp2f(x[j] - m);
                        const float p1 = (m == -INFINITY) ? 0.f : exp2f(x[j + 1] - m);
                        sum += p0 + p1;
                        pw[j >> 1] = pack2(p0, p1, bf16);
                    }
                    l = l * alpha + sum;
                }
                if (head_row) alpha_s[(gi & 1) * 64 + r] = alpha;
                if (!group_sync()) { stop = true; break; }
                __syncwarp();
                const float my_alpha = head_row ? alpha : alpha_s[(gi & 1) * 64 + h];
                if (gi >= 1 && !warp_wait(bar(B_O_DONE), (gi - 1) & 1, abort_flag)) { stop = true; break; }
                tc_fence_after();
                if (i > 0 && __any_sync(0xffffffffu, my_alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_base + TM_O + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * my_alpha);
                        tmem_st32(tmem + lane_base + TM_O + c * 32, o);
                    }
                    tmem_wait_st();
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
            if (head_row) {
                stats_s[2 * r] = m;
                stats_s[2 * r + 1] = l;
            }
            if (!group_sync()) break;
            const float mm = stats_s[2 * h], ll = stats_s[2 * h + 1];
            const bool final_split = s.nsplit == 1;
            const bool store = h < kp.q_n && (final_split || w < kp.ws_capacity_splits);
            if (!final_split && w >= kp.ws_capacity_splits && r == 0) set_status(kp, SFM_STATUS_WORKSPACE_OVERFLOW);
            float inv = 0.f;
            if (ll > 0.f) {
                float den = ll;
                if (final_split && kp.sinks) den += exp2f(__ldg(kp.sinks + h) * 1.4426950408889634f - mm);
                inv = 1.f / den;
            }
            const int64_t row = (int64_t)s.t * kp.q_n + h;
            const int dcol = head_row ? 0 : 256;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t o[32];
                __syncwarp();
                tmem_ld32(tmem + lane_base + TM_O + c * 32, o);
                tmem_wait_ld();
                if (store && final_split) {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(kp.out) + row * 512 + dcol + c * 32);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int j = q4 * 8;
                        dst[q4] = make_uint4(pack2(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv, bf16),
                                             pack2(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv, bf16),
                                             pack2(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv, bf16),
                                             pack2(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv, bf16));
                    }
                } else if (store) {
                    float4 *dst = reinterpret_cast<float4 *>(kp.ws_o + ((int64_t)w * kp.q_n + h) * 512 + dcol + c * 32);
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4)
                        dst[q4] = make_float4(__uint_as_float(o[4 * q4]) * inv, __uint_as_float(o[4 * q4 + 1]) * inv,
                                              __uint_as_float(o[4 * q4 + 2]) * inv, __uint_as_float(o[4 * q4 + 3]) * inv);
                }
            }
            if (head_row && store) {
                const float lse = ll > 0.f ? (mm + log2f(ll)) * 0.6931471805599453f : -INFINITY;
                if (final_split) {
                    if (kp.lse) kp.lse[row] = lse;
                } else {
                    kp.ws_lse[(int64_t)w * kp.q_n + h] = lse;
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
    sfm_attn_tc_kernel<<<kp.G, kThreads, kSmemBytes, st>>>(kp);
    return cudaGetLastError();
}

}  // namespace sfm
