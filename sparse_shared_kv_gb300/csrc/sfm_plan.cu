// sfm_plan.cu -- device-side split-KV planner ("sparse_flash_mla_metadata").
//
// The pages' metadata call returns the AI Core / AI Vector Core task split
// computed from the same parameters as the main call ("sparse_flash_mla" doc,
// 功能说明 and the metadata row of 参数说明).  Here it is one CTA that reads the
// length tensors on the device (no host round trip) and writes:
//   * per query row t: its attended-position count n_t cut into
//     ceil(n_t / split_rows) equal splits -- a function of the row's own count and
//     the params only, so a row's arithmetic never depends on the rest of the
//     batch (the 确定性计算 section makes batch invariance the default);
//   * per query row: the lengths / window / position counts the attention
//     kernels need (so they skip the length walk), and the split -> row map;
//   * per worker (persistent CTA): a contiguous range of splits chosen so that
//     every worker gets about the same modelled cost (attended rows plus a
//     fixed per-split latency cost).
// Each row's lengths are read once (phase 1, one row per thread); the prefix
// sums (phase 2, contiguous runs per thread) recompute the counts from the
// per-row records, and the worker searches (phase 3) run on shared-memory
// copies of the prefixes when the rows fit.
#include "sfm_internal.cuh"

namespace sfm {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kSmemRows = 1024;          // rows whose records and prefixes stay in shared memory
constexpr int kMaxWorkers = 256;

// Exclusive prefix sums of two values per thread over the block: a shuffle
// scan inside each warp, then one warp scans the 32 warp totals.
__device__ __forceinline__ int64_t shfl_up64(int64_t v, int d)
{
    return __shfl_up_sync(0xffffffffu, v, d);
}

__device__ __forceinline__ void block_exclusive_scan2(int64_t &a, int64_t &b, int64_t *sa, int64_t *sb)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int64_t ia = a, ib = b;                 // inclusive within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t ua = shfl_up64(ia, d), ub = shfl_up64(ib, d);
        if (lane >= d) {
            ia += ua;
            ib += ub;
        }
    }
    if (lane == 31) {
        sa[warp] = ia;
        sb[warp] = ib;
    }
    __syncthreads();
    if (warp == 0) {
        int64_t wa = lane < kPlanThreads / 32 ? sa[lane] : 0, wb = lane < kPlanThreads / 32 ? sb[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t ua = shfl_up64(wa, d), ub = shfl_up64(wb, d);
            if (lane >= d) {
                wa += ua;
                wb += ub;
            }
        }
        if (lane < kPlanThreads / 32) {
            sa[lane] = wa;          // inclusive warp-total prefix
            sb[lane] = wb;
        }
    }
    __syncthreads();
    const int64_t base_a = warp > 0 ? sa[warp - 1] : 0, base_b = warp > 0 ? sb[warp - 1] : 0;
    a = base_a + ia - a;            // exclusive
    b = base_b + ib - b;
    __syncthreads();
}

// One CTA.  Rows up to kSmemRows keep their records and prefixes in shared
// memory, so after the length loads of phase 1 every phase reads shared
// memory only (no global write-then-read round trips).
__global__ void __launch_bounds__(kPlanThreads) sfm_plan_kernel(KParams kp)
{
    __shared__ int64_t s_a[32];
    __shared__ int64_t s_b[32];
    __shared__ int4 s_rec[kSmemRows][2];
    __shared__ int32_t s_sp[kSmemRows + 1];
    __shared__ int32_t s_cp[kSmemRows + 1];
    __shared__ int32_t s_ws[kMaxWorkers + 1];
    __shared__ int s_overflow;

    // the attention kernel may start its set-up now; it waits for this grid
    // to finish before it reads the plan.  This grid itself is launched as a
    // dependent of whatever ran before it on the stream (its launch latency
    // overlaps that kernel's tail) and waits for it before reading any input.
    grid_launch_dependents();
    grid_dependency_wait();

    int32_t *meta = kp.meta_w;
    const int T = kp.T, G = kp.G, S = kp.split_rows;
    int32_t *ws = meta + meta_ws_off();
    int32_t *sp = meta + meta_split_off(G);
    int32_t *cp = meta + meta_cost_off(G, T);
    int32_t *rec = meta + meta_rec_off(G, T);
    int32_t *own = meta + meta_own_off(G, T);
    int32_t *srec = meta + meta_srec_off(G, T, kp.wcap);
    int32_t *wrec = meta + meta_wrec_off(G, T, kp.wcap);
    const bool in_smem = T <= kSmemRows;
    const bool ws_smem = G <= kMaxWorkers;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_overflow = 0;
        meta[H_LENFLAGS] = 0;       // length problems found while planning are OR-ed here
    }
    __syncthreads();
    kp.status = meta + H_LENFLAGS;

    auto rec_of = [&](int t, int4 &r0, int4 &r1) {
        if (in_smem) {
            r0 = s_rec[t][0];
            r1 = s_rec[t][1];
        } else {
            const int32_t *r = rec + (int64_t)kRecWords * t;
            r0 = make_int4(r[0], r[1], r[2], r[3]);
            r1 = make_int4(r[4], r[5], r[6], r[7]);
        }
    };
    auto count = [&](int t) -> int64_t {
        int4 r0, r1;
        rec_of(t, r0, r1);
        return (int64_t)r1.z + r1.w;     // n_ori + n_cmp
    };

    // 1. every row once: lengths, window and position counts
    for (int t = tid; t < T; t += kPlanThreads) {
        const Tok k = token_info(kp, t);
        const int4 r0 = make_int4(k.b, k.kv_len, k.cmp_len, k.p_cmp), r1 = make_int4(k.lo, k.hi, k.n_ori, k.n_cmp);
        if (in_smem) {
            s_rec[t][0] = r0;
            s_rec[t][1] = r1;
        } else {
            int32_t *r = rec + (int64_t)kRecWords * t;
            r[0] = r0.x; r[1] = r0.y; r[2] = r0.z; r[3] = r0.w;
            r[4] = r1.x; r[5] = r1.y; r[6] = r1.z; r[7] = r1.w;
        }
    }
    __syncthreads();
    // 2. split / cost prefixes: each thread scans a contiguous run of rows and
    //    writes the split records of its rows
    const int per = (T + kPlanThreads - 1) / kPlanThreads;
    const int beg = min(T, tid * per), end = min(T, beg + per);
    int64_t sum_s = 0, sum_c = 0;
    for (int t = beg; t < end; ++t) {
        const int64_t n = count(t), ns = num_splits(n, S);
        sum_s += ns;
        sum_c += n + ns * kSplitOverheadRows;
    }
    int64_t ex_s = sum_s, ex_c = sum_c;
    block_exclusive_scan2(ex_s, ex_c, s_a, s_b);
    for (int t = beg; t < end; ++t) {
        const int64_t n = count(t), ns = num_splits(n, S);
        if (ex_s > INT32_MAX || ex_c > INT32_MAX || ex_s + ns > kp.wcap) s_overflow = 1;
        sp[t] = (int32_t)ex_s;
        cp[t] = (int32_t)ex_c;
        if (in_smem) {
            s_sp[t] = (int32_t)ex_s;
            s_cp[t] = (int32_t)ex_c;
        }
        if (ns > 0) {
            int4 r0, r1;
            rec_of(t, r0, r1);
            const int4 hd = make_int4(t, (int32_t)ex_s, (int32_t)ns, split_size(n, S));
            for (int64_t j = 0; j < ns && ex_s + j < kp.wcap; ++j) {
                own[ex_s + j] = t;
                int4 *d = reinterpret_cast<int4 *>(srec + (ex_s + j) * kSrecWords);
                d[0] = hd;
                d[1] = r0;
                d[2] = r1;
                d[3] = make_int4(0, 0, 0, 0);
            }
        }
        ex_s += ns;
        ex_c += n + ns * kSplitOverheadRows;
    }
    if ((beg < end && end == T) || (T == 0 && tid == 0)) {   // the run that ends the rows writes the totals
        if (ex_s > INT32_MAX || ex_c > INT32_MAX) s_overflow = 1;
        sp[T] = (int32_t)ex_s;
        cp[T] = (int32_t)ex_c;
        if (in_smem) {
            s_sp[T] = (int32_t)ex_s;
            s_cp[T] = (int32_t)ex_c;
        }
    }
    __syncthreads();

    // 3. worker ranges over work units: a unit is one split for one group of
    //    heads; row t owns units [sp[t] * HG, sp[t+1] * HG), group-major, so
    //    that consecutive units of a worker mostly share their Q rows.  Worker
    //    c starts at the first unit whose cumulative cost reaches c / G of the
    //    total.
    const int32_t *xsp = in_smem ? s_sp : sp;
    const int32_t *xcp = in_smem ? s_cp : cp;
    const int64_t HG = kp.head_groups;
    const int32_t W = xsp[T];
    const int64_t units = (int64_t)W * HG;
    if (units > INT32_MAX && tid == 0) s_overflow = 1;
    const int64_t total = (int64_t)xcp[T] * HG;
    for (int c = tid; c <= G; c += kPlanThreads) {
        int64_t u;
        if (c == 0) {
            u = 0;
        } else if (c == G) {
            u = units;
        } else {
            const int64_t target = div_nonneg(total * c, G);
            int lo = 0, hi = T;     // last row t whose cumulative cost <= target
            while (lo < hi) {
                int mid = (lo + hi + 1) >> 1;
                if ((int64_t)xcp[mid] * HG <= target) lo = mid; else hi = mid - 1;
            }
            if (lo >= T) {
                u = units;
            } else {
                const int64_t nu = (int64_t)(xsp[lo + 1] - xsp[lo]) * HG;
                const int64_t within = target - (int64_t)xcp[lo] * HG;
                const int64_t ucost = split_size(count(lo), S) + kSplitOverheadRows;
                int64_t k = div_nonneg(within + ucost - 1, ucost);
                if (k > nu) k = nu;
                u = (int64_t)xsp[lo] * HG + k;
            }
        }
        const int32_t v = (int32_t)(u < INT32_MAX ? u : INT32_MAX);
        ws[c] = v;
        if (ws_smem) s_ws[c] = v;
    }
    __syncthreads();
    // 4. per worker: its range and its first unit's split record in one place
    for (int c = tid; c < G; c += kPlanThreads) {
        const int32_t u0 = ws_smem ? s_ws[c] : ws[c], u1 = ws_smem ? s_ws[c + 1] : ws[c + 1];
        int4 *d = reinterpret_cast<int4 *>(wrec + (int64_t)c * kWrecWords);
        d[0] = make_int4(u0, u1, 0, 0);
        const int64_t w0 = div_nonneg(u0, HG);
        if (u0 < u1 && w0 < kp.wcap) {
            if (in_smem) {
                int lo = 0, hi = T - 1;          // the row owning split w0
                while (lo < hi) {
                    int mid = (lo + hi + 1) >> 1;
                    if (s_sp[mid] <= w0) lo = mid; else hi = mid - 1;
                }
                const int64_t n = count(lo), ns = s_sp[lo + 1] - s_sp[lo];
                int4 r0, r1;
                rec_of(lo, r0, r1);
                d[1] = make_int4(lo, s_sp[lo], (int32_t)ns, split_size(n, S));
                d[2] = r0;
                d[3] = r1;
                d[4] = make_int4(0, 0, 0, 0);
            } else {
                const int4 *src = reinterpret_cast<const int4 *>(srec + w0 * kSrecWords);
                d[1] = src[0];
                d[2] = src[1];
                d[3] = src[2];
                d[4] = src[3];
            }
        }
    }
    if (tid == 0) {
        meta[H_MAGIC] = kMetaMagic;
        meta[H_FPRINT] = kp.fingerprint;
        meta[H_TOKENS] = T;
        meta[H_WORKERS] = G;
        meta[H_SPLIT] = S;
        meta[H_PATH] = kp.path;
        meta[H_TOTAL_SPLITS] = W;
        meta[H_FLAGS] = s_overflow ? SFM_STATUS_PLAN_OVERFLOW : 0;
        meta[H_WCAP] = (int32_t)(kp.wcap < INT32_MAX ? kp.wcap : INT32_MAX);
        for (int j = 10; j < kHdr; ++j) meta[j] = 0;
    }
}

}  // namespace

cudaError_t launch_plan(const KParams &kp, cudaStream_t st)
{
    return launch_dependent(sfm_plan_kernel, dim3(1), dim3(kPlanThreads), (size_t)0, st, kp);
}

}  // namespace sfm
