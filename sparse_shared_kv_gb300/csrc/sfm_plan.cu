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
//   * per split: a 64-byte record with its row, the row's split count and
//     size, and the lengths / window / position counts the attention kernels
//     need (so they skip the length walk);
//   * per worker (persistent CTA): a contiguous range of work units chosen so
//     that every worker gets about the same modelled cost (attended rows plus
//     a fixed per-split latency cost), and its first unit's split record.
// Each row's lengths are read once (phase 1, one row per thread); the prefix
// sums (phase 2, contiguous runs per thread) recompute the counts from the
// per-row records; phase 3 writes the split and worker records in parallel
// (binary searches over shared-memory copies of the prefixes when the rows
// fit).  Every step after the length loads is a short chain per thread: the
// planner sits on the critical path of a decode step.
#include "sfm_internal.cuh"

namespace sfm {

namespace {

constexpr int kPlanThreads = 512;
constexpr int kSmemRows = 512;           // rows whose records stay in shared memory
constexpr int kMaxWorkers = 256;         // persistent workers (one per SM)
constexpr int kMaxSplits = 2048;         // splits whose row map fits in shared memory

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

// One CTA.  Rows up to kSmemRows keep their records in shared memory, so
// after the length loads of phase 1 no phase reads global memory.  No thread
// runs a serial chain longer than its rows' splits and worker boundaries: the
// planner sits on the critical path of a decode step.
__global__ void __launch_bounds__(kPlanThreads) sfm_plan_kernel(KParams kp)
{
    __shared__ int64_t s_a[32];
    __shared__ int64_t s_b[32];
    __shared__ int4 s_rec[kSmemRows][2];
    __shared__ int2 s_shape[kSmemRows];           // splits, split size
    __shared__ int32_t s_sp[kSmemRows];           // first split of each row
    __shared__ int32_t s_cp[kSmemRows];           // modelled cost before each row
    __shared__ int32_t s_ws[kMaxWorkers + 1];     // worker c's first unit
    __shared__ int32_t s_wrow[kMaxWorkers];       // the row of that unit
    __shared__ int32_t s_wbeg[kMaxWorkers];       // the row's first split
    __shared__ int32_t s_owner[kMaxSplits];       // split -> row (flat record writes)
    __shared__ int64_t s_tot[2];                  // splits, modelled cost
    __shared__ int s_overflow;
    __shared__ int s_lenflags;                    // length problems, while the rows stay in shared memory

    // the attention kernel may start its set-up now; it waits for this grid
    // to finish before it reads the plan.  This grid itself is launched as a
    // dependent of whatever ran before it on the stream (its launch latency
    // overlaps that kernel's tail).  It reads only the length tensors, which
    // no kernel of this library writes, and waits for its predecessor before
    // it writes the plan (a previous forward may still be reading an earlier
    // plan in the same buffer): while the rows fit in shared memory, the row
    // phase (the length loads) runs before that wait.
    grid_launch_dependents();

    int32_t *meta = kp.meta_w;
    const int T = kp.T, G = kp.G, S = kp.split_rows;
    int32_t *ws = meta + meta_ws_off();
    int32_t *sp = meta + meta_split_off(G);
    int32_t *cp = meta + meta_cost_off(G, T);
    int32_t *rec = meta + meta_rec_off(G, T);
    int32_t *srec = meta + meta_srec_off(G, T, kp.wcap);
    int32_t *wrec = meta + meta_wrec_off(G, T, kp.wcap);
    const bool in_smem = T <= kSmemRows;
    const int tid = threadIdx.x;
    if (!in_smem) grid_dependency_wait();
    if (tid == 0) {
        s_overflow = G > kMaxWorkers ? 1 : 0;
        s_tot[0] = s_tot[1] = 0;
        s_lenflags = 0;
        if (!in_smem) meta[H_LENFLAGS] = 0;       // length problems found while planning are OR-ed here
    }
    __syncthreads();
    kp.status = in_smem ? &s_lenflags : meta + H_LENFLAGS;

    auto rec_of = [&](int t, int4 &r0, int4 &r1) {
        if (in_smem) {
            r0 = s_rec[t][0];
            r1 = s_rec[t][1];
        } else {                         // 4-byte aligned only: scalar accesses
            const int32_t *r = rec + (int64_t)kRecWords * t;
            r0 = make_int4(r[0], r[1], r[2], r[3]);
            r1 = make_int4(r[4], r[5], r[6], r[7]);
        }
    };
    const int64_t HG = kp.head_groups;
    // a row's splits, their size and the modelled cost of each of its
    // head_groups * splits work units (rows plus a fixed per-unit latency cost)
    auto shape_of = [&](int64_t n) -> int2 {           // n = n_ori + n_cmp
        return make_int2((int)num_splits_dev(n, kp.split_div), split_size_dev(n, kp.split_div));
    };
    auto row_shape = [&](int t, int64_t &ns, int &size, int64_t &ucost) {
        int2 sh;
        if (in_smem) {
            sh = s_shape[t];
        } else {
            int4 r0, r1;
            rec_of(t, r0, r1);
            sh = shape_of((int64_t)r1.z + r1.w);
        }
        ns = sh.x;
        size = sh.y;
        ucost = size + kSplitOverheadRows;
    };

    // 1. every row once: lengths, window and position counts
    for (int t = tid; t < T; t += kPlanThreads) {
        const Tok k = token_info(kp, t);
        const int4 r0 = make_int4(k.b, k.kv_len, k.cmp_len, k.p_cmp), r1 = make_int4(k.lo, k.hi, k.n_ori, k.n_cmp);
        if (in_smem) {
            s_rec[t][0] = r0;
            s_rec[t][1] = r1;
            s_shape[t] = shape_of((int64_t)k.n_ori + k.n_cmp);
        } else {
            int32_t *r = rec + (int64_t)kRecWords * t;
            r[0] = r0.x; r[1] = r0.y; r[2] = r0.z; r[3] = r0.w;
            r[4] = r1.x; r[5] = r1.y; r[6] = r1.z; r[7] = r1.w;
        }
    }
    if (in_smem) grid_dependency_wait();
    __syncthreads();
    if (in_smem) {
        if (tid == 0) meta[H_LENFLAGS] = s_lenflags;
        kp.status = meta + H_LENFLAGS;
    }

    // 2. split and unit-cost prefixes over contiguous runs of rows per thread
    const int per = (T + kPlanThreads - 1) / kPlanThreads;
    const int beg = min(T, tid * per), end = min(T, beg + per);
    int64_t sum_s = 0, sum_c = 0;
    for (int t = beg; t < end; ++t) {
        int64_t ns, ucost;
        int size;
        row_shape(t, ns, size, ucost);
        sum_s += ns;
        sum_c += ns * HG * ucost;
    }
    int64_t ex_s = sum_s, ex_c = sum_c;
    block_exclusive_scan2(ex_s, ex_c, s_a, s_b);
    for (int t = beg; t < end; ++t) {     // per-row prefixes: the split table (global) and cost prefix
        int64_t ns, ucost;
        int size;
        row_shape(t, ns, size, ucost);
        if (ex_s > INT32_MAX || ex_c > INT32_MAX || ns > kp.max_splits) s_overflow = 1;
        sp[t] = (int32_t)ex_s;
        if (in_smem) {
            s_sp[t] = (int32_t)ex_s;
            s_cp[t] = (int32_t)ex_c;
        } else {
            cp[t] = (int32_t)ex_c;
        }
        ex_s += ns;
        ex_c += ns * HG * ucost;
    }
    if (beg < end && end == T) {          // the run that ends the rows holds the totals
        s_tot[0] = ex_s;
        s_tot[1] = ex_c;
    }
    __syncthreads();
    const int64_t W = s_tot[0], units = W * HG, total = s_tot[1];
    if (tid == 0 && (W > INT32_MAX || units > INT32_MAX || W > kp.wcap || total > INT32_MAX)) s_overflow = 1;
    auto sp_of = [&](int t) -> int64_t { return in_smem ? s_sp[t] : sp[t]; };
    auto cp_of = [&](int t) -> int64_t { return in_smem ? s_cp[t] : cp[t]; };

    // 3. two independent halves of the block, so that neither chain waits for
    //    the other:
    //    (a) threads [0, kHalf): each row's 64-byte split records;
    //    (b) threads [kHalf, 2 kHalf): the worker boundaries in each row.  A
    //        row's units are group-major (unit hg * ns + s is split s for head
    //        group hg), so consecutive units of a worker mostly share their Q
    //        rows.  Unit j of row t spans modelled cost [cp(t) + j ucost,
    //        cp(t) + (j + 1) ucost); worker c starts at the unit whose span
    //        holds target(c) = floor(c total / G), so every worker gets about
    //        the same cost.  The workers whose targets fall in the row and
    //        their units come from three divisions per row and a merge walk.
    constexpr int kHalf = kPlanThreads / 2;
    // split records go out in step 4 as one coalesced stream when the split
    // -> row map fits in shared memory; otherwise each row writes its own
    const bool flat = in_smem && W <= kMaxSplits;
    if (tid < kHalf) {
        for (int t = tid; t < T; t += kHalf) {
            int64_t ns, ucost;
            int size;
            row_shape(t, ns, size, ucost);
            const int64_t s0 = sp_of(t);
            if (flat) {
                for (int64_t j = 0; j < ns; ++j) s_owner[s0 + j] = t;
                continue;
            }
            int4 r0, r1;
            rec_of(t, r0, r1);
            const int4 hd = make_int4(t, (int32_t)s0, (int32_t)ns, size);
            for (int64_t j = 0; j < ns && s0 + j < kp.wcap; ++j) {
                int4 *d = reinterpret_cast<int4 *>(srec + (s0 + j) * kSrecWords);
                d[0] = hd;
                d[1] = r0;
                d[2] = r1;
            }
        }
        if (tid == 0) sp[T] = (int32_t)(W < INT32_MAX ? W : INT32_MAX);
    } else if (total > 0) {
        const bool small = (total + 1) * (G + 1) <= 0xffffffffll;     // boundary arithmetic fits 32 bits
        auto qdiv = [&](int64_t a, int64_t b) -> int64_t {
            return small ? (int64_t)udiv_est((uint32_t)a, (uint32_t)b) : a / b;
        };
        const int64_t tq = qdiv(total, G), tr = total - tq * G;      // target(c + 1) - target(c) = tq or tq + 1
        for (int t = tid - kHalf; t < T; t += kHalf) {
            int64_t ns, ucost;
            int size;
            row_shape(t, ns, size, ucost);
            const int64_t nu = ns * HG, c0 = cp_of(t), s0 = sp_of(t);
            if (nu == 0) continue;
            // workers c with c0 <= target(c) < c0 + nu ucost
            const int64_t c_first = qdiv(c0 * G + total - 1, total);
            int64_t c_end = qdiv((c0 + nu * ucost) * G + total - 1, total);
            if (c_end > G) c_end = G;
            if (c_first >= c_end) continue;
            const int64_t num = c_first * total;
            int64_t tgt = qdiv(num, G), rem = num - tgt * G;
            int64_t j = 0, ustart = c0;
            for (int64_t c = c_first; c < c_end; ++c) {
                while (j + 1 < nu && ustart + ucost <= tgt) {
                    ustart += ucost;
                    ++j;
                }
                if (c < kMaxWorkers) {
                    s_ws[c] = (int32_t)(s0 * HG + j);
                    s_wrow[c] = t;
                    s_wbeg[c] = (int32_t)s0;
                }
                tgt += tq;
                rem += tr;
                if (rem >= G) {
                    rem -= G;
                    ++tgt;
                }
            }
        }
    }
    if (tid == kHalf) {
        if (G <= kMaxWorkers) s_ws[G] = (int32_t)(units < INT32_MAX ? units : INT32_MAX);
        if (total == 0)                   // no work: every worker's range is empty
            for (int c = 0; c < G && c < kMaxWorkers; ++c) {
                s_ws[c] = 0;
                s_wrow[c] = 0;
                s_wbeg[c] = 0;
            }
    }
    __syncthreads();

    // 4. every thread writes consecutive 16-byte words of two flat streams,
    //    so that a warp's stores are contiguous:
    //    * the split records, words 0-2 of each 64-byte record (row, first
    //      split, split count and size; the row's two record words);
    //    * the worker records, words 0-3 (unit range; the first unit's row
    //      header and record words).
    auto row_word = [&](int t, int32_t first, int part) -> int4 {
        if (part == 0) {
            int64_t ns, ucost;
            int size;
            row_shape(t, ns, size, ucost);
            return make_int4(t, first, (int32_t)ns, size);
        }
        int4 r0, r1;
        rec_of(t, r0, r1);
        return part == 1 ? r0 : r1;
    };
    if (flat) {
        const int W3 = (int)W * 3;                 // W <= kMaxSplits: 32-bit arithmetic
        for (int i = tid; i < W3; i += kPlanThreads) {
            const int w = i / 3;
            const int part = i - w * 3, t = s_owner[w];
            reinterpret_cast<int4 *>(srec + (int64_t)w * kSrecWords)[part] = row_word(t, s_sp[t], part);
        }
    }
    const int GW = G < kMaxWorkers ? G : kMaxWorkers;
    for (int i = tid; i < GW * 4; i += kPlanThreads) {
        const int c = i >> 2, part = i & 3;
        const int32_t u0 = s_ws[c], u1 = s_ws[c + 1];
        int4 v;
        if (part == 0) v = make_int4(u0, u1, 0, 0);
        else if (u0 < u1) v = row_word(s_wrow[c], s_wbeg[c], part - 1);
        else continue;              // an empty range: the rest of the record is never read
        reinterpret_cast<int4 *>(wrec + (int64_t)c * kWrecWords)[part] = v;
    }
    for (int c = tid; c <= GW; c += kPlanThreads) ws[c] = s_ws[c];
    if (tid == 0) {
        meta[H_MAGIC] = kMetaMagic;
        meta[H_FPRINT] = kp.fingerprint;
        meta[H_TOKENS] = T;
        meta[H_WORKERS] = G;
        meta[H_SPLIT] = S;
        meta[H_PATH] = kp.path;
        meta[H_TOTAL_SPLITS] = (int32_t)(W < INT32_MAX ? W : INT32_MAX);
        meta[H_FLAGS] = s_overflow ? SFM_STATUS_PLAN_OVERFLOW : 0;
        meta[H_WCAP] = (int32_t)(kp.wcap < INT32_MAX ? kp.wcap : INT32_MAX);
        for (int j = 10; j < kHdr; ++j) meta[j] = 0;
    }
}

// The same plan for a decode batch of at most kSmallRows rows and fewer than
// kSmallThreads workers, in three short phases:
//   1. warps 0 and 1 take one row per lane (lengths, window, counts, split
//      shape) and scan the split counts and modelled costs of their 32 rows
//      with shuffles;
//   2. every thread finds, by binary search over the 64 row prefixes, the row
//      of each split record it writes (one flat stream) and the first unit of
//      worker c = thread index (the row whose cost span holds c total / G,
//      then the unit inside it by one division);
//   3. the worker records, as one flat stream.
// A plan of at most kStageSplits splits and kStageWorkers workers is built
// entirely in shared memory before the kernel's dependency wait (it reads
// only the length tensors) and only streamed out after it, so its
// computation overlaps the previous kernel; larger plans are built and
// written after the wait.  No thread runs a serial walk; the general kernel
// above serves larger batches.
constexpr int kSmallRows = 64;
constexpr int kSmallThreads = 512;
constexpr int kStageSplits = 384;        // plans this small are finished in shared memory
constexpr int kStageWorkers = 256;       // before the dependency wait, then streamed out

__global__ void __launch_bounds__(kSmallThreads) sfm_plan_small_kernel(KParams kp)
{
    __shared__ int4 s_r0[kSmallRows], s_r1[kSmallRows];   // the rows' record words
    __shared__ int2 s_shape[kSmallRows];                   // splits, split size
    __shared__ int64_t s_is[kSmallRows], s_ic[kSmallRows];  // inclusive split / cost prefix in the row's warp
    __shared__ int64_t s_wt[2][2];                         // warp totals: splits, cost
    __shared__ int32_t s_ws[kSmallThreads], s_wrow[kSmallThreads];
    __shared__ int s_flags[2];                             // length problems, per row warp
    __shared__ int s_over[2];                              // a row with too many splits, per row warp
    __shared__ int4 s_srec[kStageSplits * 3];              // staged split records (words 0..11)
    __shared__ int4 s_wrec[kStageWorkers * 4];             // staged worker records

    // reads only the length tensors before its dependency wait (everything
    // up to the stores works in shared memory); waits before it writes the plan
    grid_launch_dependents();

    int32_t *meta = kp.meta_w;
    const int T = kp.T, G = kp.G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t HG = kp.head_groups;
    int32_t *sp = meta + meta_split_off(G);
    int32_t *srec = meta + meta_srec_off(G, T, kp.wcap);
    int32_t *wrec = meta + meta_wrec_off(G, T, kp.wcap);

    // 1. rows
    if (warp < 2) {
        if (lane == 0) {
            s_flags[warp] = 0;
            s_over[warp] = 0;
        }
        __syncwarp();
        kp.status = &s_flags[warp];          // length problems of this warp's rows
        const int t = warp * 32 + lane;
        int64_t ns = 0, cost = 0;
        if (t < T) {
            const Tok k = token_info(kp, t);
            const int64_t n = (int64_t)k.n_ori + k.n_cmp;
            ns = num_splits_dev(n, kp.split_div);
            const int size = split_size_dev(n, kp.split_div);
            cost = ns * HG * (size + kSplitOverheadRows);
            s_r0[t] = make_int4(k.b, k.kv_len, k.cmp_len, k.p_cmp);
            s_r1[t] = make_int4(k.lo, k.hi, k.n_ori, k.n_cmp);
            s_shape[t] = make_int2((int)ns, size);
            if (ns > kp.max_splits) s_over[warp] = 1;
        }
        int64_t is = ns, ic = cost;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t us = shfl_up64(is, d), uc = shfl_up64(ic, d);
            if (lane >= d) {
                is += us;
                ic += uc;
            }
        }
        s_is[t] = is;
        s_ic[t] = ic;
        if (lane == 31) {
            s_wt[warp][0] = is;
            s_wt[warp][1] = ic;
        }
    }
    __syncthreads();

    // row prefixes over the whole batch (rows past T carry no splits and no cost)
    const int64_t W = s_wt[0][0] + s_wt[1][0];
    const int64_t total = s_wt[0][1] + s_wt[1][1];
    const int64_t units = W * HG;
    auto incl_s = [&](int t) -> int64_t { return s_is[t] + (t >= 32 ? s_wt[0][0] : 0); };
    auto incl_c = [&](int t) -> int64_t { return s_ic[t] + (t >= 32 ? s_wt[0][1] : 0); };
    // the first row whose inclusive prefix passes v (v below the batch total)
    auto find_row = [&](int64_t v, bool by_cost) -> int {
        int lo = 0, hi = T - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((by_cost ? incl_c(mid) : incl_s(mid)) > v) hi = mid; else lo = mid + 1;
        }
        return lo;
    };
    auto row_word = [&](int t, int part) -> int4 {
        if (part == 1) return s_r0[t];
        if (part == 2) return s_r1[t];
        const int2 sh = s_shape[t];
        return make_int4(t, (int32_t)(incl_s(t) - sh.x), sh.x, sh.y);
    };
    const int64_t WR = (W < kp.wcap ? W : kp.wcap) * 3;
    // a small plan is finished in shared memory before the dependency wait
    // (only its stores wait for the previous kernel); larger ones are
    // computed and written after it
    const bool staged = WR <= kStageSplits * 3 && G <= kStageWorkers;

    // 2. each worker's first unit (the row whose cost span holds c total / G,
    // then the unit inside it by one division), and the split records
    if (tid <= G) {
        int32_t u = 0, row = 0;
        if (tid == G) {
            u = (int32_t)(units < INT32_MAX ? units : INT32_MAX);
        } else if (total > 0) {
            const int64_t num = (int64_t)tid * total;
            const int64_t tgt = (total + 1) * (G + 1) <= 0xffffffffll ? (int64_t)udiv_est((uint32_t)num, (uint32_t)G)
                                                                     : num / G;
            row = find_row(tgt, true);
            const int2 sh = s_shape[row];
            const int64_t ucost = sh.y + kSplitOverheadRows, nu = (int64_t)sh.x * HG;
            const int64_t c0 = incl_c(row) - nu * ucost, off = tgt - c0;
            int64_t j = off <= 0xffffffffll ? (int64_t)udiv_est((uint32_t)off, (uint32_t)ucost) : off / ucost;
            if (j > nu - 1) j = nu - 1;
            u = (int32_t)((incl_s(row) - sh.x) * HG + j);
        }
        s_ws[tid] = u;
        s_wrow[tid] = row;
    }
    if (staged) {
        for (int i = tid; i < (int)WR; i += kSmallThreads) {
            const int w = i / 3, part = i - w * 3;
            s_srec[i] = row_word(find_row(w, false), part);
        }
        __syncthreads();
        // 3. worker records: the unit range, then the first unit's split record words
        for (int i = tid; i < G * 4; i += kSmallThreads) {
            const int c = i >> 2, part = i & 3;
            const int32_t u0 = s_ws[c], u1 = s_ws[c + 1];
            s_wrec[i] = part == 0 ? make_int4(u0, u1, 0, 0)
                                  : (u0 < u1 ? row_word(s_wrow[c], part - 1) : make_int4(0, 0, 0, 0));
        }
        __syncthreads();
    }

    grid_dependency_wait();                  // the plan may now be overwritten

    if (tid <= T) sp[tid] = tid < T ? (int32_t)(incl_s(tid) - s_shape[tid].x) : (int32_t)(W < INT32_MAX ? W : INT32_MAX);
    if (tid <= G) meta[meta_ws_off() + tid] = s_ws[tid];
    if (staged) {
        for (int i = tid; i < (int)WR; i += kSmallThreads)
            reinterpret_cast<int4 *>(srec + (int64_t)(i / 3) * kSrecWords)[i % 3] = s_srec[i];
        for (int i = tid; i < G * 4; i += kSmallThreads) {
            const int c = i >> 2, part = i & 3;
            if (part == 0 || s_ws[c] < s_ws[c + 1])          // an empty range: the rest is never read
                reinterpret_cast<int4 *>(wrec + (int64_t)c * kWrecWords)[part] = s_wrec[i];
        }
    } else {
        if (WR <= INT32_MAX) {                   // 32-bit index arithmetic
            for (int i = tid; i < (int)WR; i += kSmallThreads) {
                const int w = i / 3, part = i - w * 3;
                reinterpret_cast<int4 *>(srec + (int64_t)w * kSrecWords)[part] = row_word(find_row(w, false), part);
            }
        } else {
            for (int64_t i = tid; i < WR; i += kSmallThreads) {
                const int64_t w = i / 3;
                const int part = (int)(i - w * 3);
                reinterpret_cast<int4 *>(srec + w * kSrecWords)[part] = row_word(find_row(w, false), part);
            }
        }
        __syncthreads();
        // 3. worker records: the unit range, then the first unit's split record words
        for (int i = tid; i < G * 4; i += kSmallThreads) {
            const int c = i >> 2, part = i & 3;
            const int32_t u0 = s_ws[c], u1 = s_ws[c + 1];
            int4 v;
            if (part == 0) v = make_int4(u0, u1, 0, 0);
            else if (u0 < u1) v = row_word(s_wrow[c], part - 1);
            else continue;              // an empty range: the rest of the record is never read
            reinterpret_cast<int4 *>(wrec + (int64_t)c * kWrecWords)[part] = v;
        }
    }
    if (tid == 0) {
        const bool bad = W > INT32_MAX || units > INT32_MAX || W > kp.wcap || total > INT32_MAX;
        meta[H_MAGIC] = kMetaMagic;
        meta[H_FPRINT] = kp.fingerprint;
        meta[H_TOKENS] = T;
        meta[H_WORKERS] = G;
        meta[H_SPLIT] = kp.split_rows;
        meta[H_PATH] = kp.path;
        meta[H_TOTAL_SPLITS] = (int32_t)(W < INT32_MAX ? W : INT32_MAX);
        meta[H_FLAGS] = (s_over[0] | s_over[1] | bad) ? SFM_STATUS_PLAN_OVERFLOW : 0;
        meta[H_LENFLAGS] = s_flags[0] | s_flags[1];
        meta[H_WCAP] = (int32_t)(kp.wcap < INT32_MAX ? kp.wcap : INT32_MAX);
        for (int j = 10; j < kHdr; ++j) meta[j] = 0;
    }
}

}  // namespace

cudaError_t launch_plan(const KParams &kp, cudaStream_t st)
{
    if (kp.T <= kSmallRows && kp.G < kSmallThreads)
        return launch_dependent(sfm_plan_small_kernel, dim3(1), dim3(kSmallThreads), (size_t)0, st, kp);
    return launch_dependent(sfm_plan_kernel, dim3(1), dim3(kPlanThreads), (size_t)0, st, kp);
}

}  // namespace sfm
