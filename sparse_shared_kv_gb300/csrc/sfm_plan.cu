// sfm_plan.cu -- device-side split-KV planner ("sparse_flash_mla_metadata").
//
// The pages' metadata call returns the AI Core / AI Vector Core task split
// computed from the same parameters as the main call ("sparse_flash_mla" doc,
// 功能说明 and the metadata row of 参数说明).  Here it is one CTA that reads the
// length tensors on the device (no host round trip) and writes:
//   * per query row t: its attended-position count n_t cut into
//     ceil(n_t / split_rows) splits -- a function of the row's own count and
//     the params only, so a row's arithmetic never depends on the rest of the
//     batch (the 确定性计算 section makes batch invariance the default);
//   * per worker (persistent CTA or CTA pair): a contiguous range of splits
//     chosen so that every worker gets about the same modelled cost
//     (attended rows + a fixed per-split overhead).
#include "sfm_internal.cuh"

namespace sfm {

namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ void block_exclusive_scan2(int64_t &a, int64_t &b, int64_t *sa, int64_t *sb)
{
    const int tid = threadIdx.x;
    sa[tid] = a;
    sb[tid] = b;
    __syncthreads();
    for (int off = 1; off < kPlanThreads; off <<= 1) {
        int64_t va = 0, vb = 0;
        if (tid >= off) {
            va = sa[tid - off];
            vb = sb[tid - off];
        }
        __syncthreads();
        sa[tid] += va;
        sb[tid] += vb;
        __syncthreads();
    }
    const int64_t ia = sa[tid], ib = sb[tid];
    a = ia - a;    // exclusive
    b = ib - b;
    __syncthreads();
}

__global__ void __launch_bounds__(kPlanThreads) sfm_plan_kernel(KParams kp)
{
    __shared__ int64_t s_a[kPlanThreads];
    __shared__ int64_t s_b[kPlanThreads];
    __shared__ int s_overflow;

    int32_t *meta = kp.meta_w;
    const int T = kp.T, G = kp.G, S = kp.split_rows;
    int32_t *ws = meta + meta_ws_off();
    int32_t *sp = meta + meta_split_off(G);
    int32_t *cp = meta + meta_cost_off(G, T);
    int32_t *rec = meta + meta_rec_off(G, T);
    int32_t *own = meta + meta_own_off(G, T);
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_overflow = 0;
        meta[H_LENFLAGS] = 0;       // length problems found while planning are OR-ed here
    }
    __syncthreads();
    kp.status = meta + H_LENFLAGS;

    // 1. per-row split count and cost; each thread owns a contiguous run of rows
    const int per = (T + kPlanThreads - 1) / kPlanThreads;
    const int beg = min(T, tid * per), end = min(T, beg + per);
    int64_t sum_s = 0, sum_c = 0;
    for (int t = beg; t < end; ++t) {
        const Tok k = token_info(kp, t);
        const int64_t n = (int64_t)k.n_ori + k.n_cmp;
        const int64_t ns = n > 0 ? (n + S - 1) / S : 0;
        sum_s += ns;
        sum_c += n + ns * kSplitOverheadRows;
    }
    // 2. exclusive scan of the per-thread sums, then the per-row prefixes
    int64_t ex_s = sum_s, ex_c = sum_c;
    block_exclusive_scan2(ex_s, ex_c, s_a, s_b);
    for (int t = beg; t < end; ++t) {
        const Tok k = token_info(kp, t);
        const int64_t n = (int64_t)k.n_ori + k.n_cmp;
        const int64_t ns = n > 0 ? (n + S - 1) / S : 0;
        if (ex_s > INT32_MAX || ex_c > INT32_MAX || ex_s + ns > kp.wcap) s_overflow = 1;
        sp[t] = (int32_t)ex_s;
        cp[t] = (int32_t)ex_c;
        int32_t *r = rec + (int64_t)kRecWords * t;
        r[0] = k.b;
        r[1] = k.kv_len;
        r[2] = k.cmp_len;
        r[3] = k.p_cmp;
        r[4] = k.lo;
        r[5] = k.hi;
        r[6] = k.n_ori;
        r[7] = k.n_cmp;
        for (int64_t j = 0; j < ns && ex_s + j < kp.wcap; ++j) own[ex_s + j] = t;
        ex_s += ns;
        ex_c += n + ns * kSplitOverheadRows;
    }
    if (tid == kPlanThreads - 1) {
        if (ex_s > INT32_MAX || ex_c > INT32_MAX) s_overflow = 1;
        sp[T] = (int32_t)ex_s;
        cp[T] = (int32_t)ex_c;
    }
    __syncthreads();

    // 3. worker ranges: worker c starts at the first split whose cumulative
    //    cost reaches c / G of the total
    const int32_t W = sp[T];
    const int64_t total = cp[T];
    for (int c = tid; c <= G; c += kPlanThreads) {
        int32_t w;
        if (c == 0) {
            w = 0;
        } else if (c == G) {
            w = W;
        } else {
            const int64_t target = total * c / G;
            int lo = 0, hi = T;     // last row t with cp[t] <= target
            while (lo < hi) {
                int mid = (lo + hi + 1) >> 1;
                if (cp[mid] <= target) lo = mid; else hi = mid - 1;
            }
            if (lo >= T) {
                w = W;
            } else {
                const int64_t ns = sp[lo + 1] - sp[lo];
                const int64_t within = target - cp[lo];
                int64_t s = (within + S + kSplitOverheadRows - 1) / (S + kSplitOverheadRows);
                if (s > ns) s = ns;
                w = sp[lo] + (int32_t)s;
            }
        }
        ws[c] = w;
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
    sfm_plan_kernel<<<1, kPlanThreads, 0, st>>>(kp);
    return cudaGetLastError();
}

}  // namespace sfm
