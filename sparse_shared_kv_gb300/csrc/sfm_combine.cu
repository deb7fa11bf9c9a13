// sfm_combine.cu -- merge the split-KV partial results of each query row.
//
// For a row whose attended positions were cut into splits s = 0..n-1 with
// normalised partial outputs O_s (stored as bf16) and partial LSEs lse_s (fp32):
//   LSE = log sum_s exp(lse_s)                         (the row's log-sum-exp)
//   O   = sum_s exp(lse_s - LSE) O_s / (1 + exp(sink - LSE))
// The sink term is the per-head logit added once to the softmax denominator;
// it is applied here, after the merge, so the merge itself stays a plain
// associative log-sum-exp (the same merge the kv_quant_sparse_flash_attention
// guide uses the LSE for across decode context-parallel ranks).  Splits are
// merged in split order, so the result is deterministic.
//
// This kernel also writes the rows no split covers (empty attended set or a
// query row beyond seqused_q: O = 0, LSE = -inf) and, when the plan does not
// match the params, zeroes every output and flags the status word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "sfm_internal.cuh"

namespace sfm {

namespace {

constexpr int kThreads = 256;                 // 8 warps, one head each
constexpr int kHeadsPerBlock = kThreads / 32;

__device__ __forceinline__ uint32_t to_half2(float a, float b, int dtype)
{
    if (dtype == SFM_DTYPE_BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

constexpr int kUnrolled = 8;                  // splits whose loads are all issued up front

__device__ __forceinline__ void acc_bf16x8(float (&acc)[16], int base, float w, uint4 v)
{
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {      // bf16 pair -> two floats (exact)
        acc[base + 2 * e] = fmaf(w, __uint_as_float(wv[e] << 16), acc[base + 2 * e]);
        acc[base + 2 * e + 1] = fmaf(w, __uint_as_float(wv[e] & 0xffff0000u), acc[base + 2 * e + 1]);
    }
}

// grid (query rows, ceil(q_n / 8)); warp = head, lane = 16 consecutive dims.
// After the plan words, every load of a row with up to kUnrolled splits goes
// out at once (the split LSEs, one per lane, and both 16-byte pieces of every
// split's partial), so the merge costs three dependent round trips.
__global__ void __launch_bounds__(kThreads) sfm_combine_kernel(KParams kp)
{
    const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * kHeadsPerBlock + warp;
    grid_launch_dependents();    // the next launch on the stream may start its set-up
    grid_dependency_wait();      // partial results come from the attention launch before this one
    const int32_t *sp = kp.meta + meta_split_off(kp.G);
    const int32_t sp0 = sp[t], sp1 = sp[t + 1];      // independent of the header check
    const bool ok = meta_ok(kp);
    if (t == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        if (!ok) set_status(kp, SFM_STATUS_METADATA_MISMATCH | kp.meta[H_FLAGS]);
        else if (kp.meta[H_LENFLAGS]) set_status(kp, kp.meta[H_LENFLAGS]);
    }
    if (h >= kp.q_n) return;
    int ns = 0, s0 = 0;
    if (ok) {
        s0 = sp0;
        ns = sp1 - s0;
        if (ns == 1) return;      // finalised by the attention kernel
        if (ns > 1 && (int64_t)s0 + ns > kp.ws_capacity_splits) {
            if (lane == 0) set_status(kp, SFM_STATUS_WORKSPACE_OVERFLOW);
            ns = 0;
        }
    }
    const int64_t row = (int64_t)t * kp.q_n + h;
    // chunk-major partial: [split][dim / 8][head][8]; this lane's 16 dims are
    // chunks 2 lane and 2 lane + 1
    auto piece = [&](int sx, int q) -> const uint4 * {
        return reinterpret_cast<const uint4 *>(kp.ws_o + (int64_t)(s0 + sx) * kp.q_n * 512 +
                                               ((int64_t)(2 * lane + q) * kp.q_n + h) * 8);
    };
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    float L = -INFINITY;
    if (ns > 0 && ns <= kUnrolled) {
        const float my_lse = lane < ns ? kp.ws_lse[(int64_t)(s0 + lane) * kp.q_n + h] : -INFINITY;
        uint4 v[kUnrolled][2];
#pragma unroll
        for (int sx = 0; sx < kUnrolled; ++sx)
#pragma unroll
            for (int q = 0; q < 2; ++q) v[sx][q] = sx < ns ? *piece(sx, q) : make_uint4(0, 0, 0, 0);
        float m = my_lse;
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float z = (m != -INFINITY && lane < ns) ? expf(my_lse - m) : 0.f;
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        L = m == -INFINITY ? -INFINITY : m + logf(z);
        const float wl = (L != -INFINITY && lane < ns) ? expf(my_lse - L) : 0.f;
#pragma unroll
        for (int sx = 0; sx < kUnrolled; ++sx) {
            const float w = __shfl_sync(0xffffffffu, wl, sx);
            if (sx < ns) {
                acc_bf16x8(acc, 0, w, v[sx][0]);
                acc_bf16x8(acc, 8, w, v[sx][1]);
            }
        }
    } else if (ns > kUnrolled) {
        // LSE of the row over its splits: lane s holds split s (in chunks of 32)
        float m = -INFINITY;
        for (int c = 0; c < ns; c += 32)
            if (c + lane < ns) m = fmaxf(m, kp.ws_lse[(int64_t)(s0 + c + lane) * kp.q_n + h]);
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float z = 0.f;
        if (m != -INFINITY)
            for (int c = 0; c < ns; c += 32)
                if (c + lane < ns) z += expf(kp.ws_lse[(int64_t)(s0 + c + lane) * kp.q_n + h] - m);
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        L = m == -INFINITY ? -INFINITY : m + logf(z);
        if (L != -INFINITY) {
            for (int c = 0; c < ns; c += 32) {
                const int cn = min(32, ns - c);
                const float wl = lane < cn ? expf(kp.ws_lse[(int64_t)(s0 + c + lane) * kp.q_n + h] - L) : 0.f;
                for (int sx = 0; sx < cn; ++sx) {
                    const float w = __shfl_sync(0xffffffffu, wl, sx);
                    acc_bf16x8(acc, 0, w, *piece(c + sx, 0));
                    acc_bf16x8(acc, 8, w, *piece(c + sx, 1));
                }
            }
        }
    }
    if (L != -INFINITY && kp.sinks) {
        const float f = 1.f / (1.f + expf(__ldg(kp.sinks + h) - L));
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] *= f;
    }
    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(kp.out) + row * 512 + lane * 16);
    dst[0] = make_uint4(to_half2(acc[0], acc[1], kp.dtype), to_half2(acc[2], acc[3], kp.dtype),
                        to_half2(acc[4], acc[5], kp.dtype), to_half2(acc[6], acc[7], kp.dtype));
    dst[1] = make_uint4(to_half2(acc[8], acc[9], kp.dtype), to_half2(acc[10], acc[11], kp.dtype),
                        to_half2(acc[12], acc[13], kp.dtype), to_half2(acc[14], acc[15], kp.dtype));
    if (lane == 0 && kp.lse) kp.lse[row] = L;
}

__global__ void __launch_bounds__(256) sfm_debug_kernel(KParams kp)
{
    for (int t = blockIdx.x; t < kp.T; t += gridDim.x) {
        const Tok k = token_info(kp, t);
        const int n = k.n_ori + k.n_cmp;
        if (threadIdx.x == 0) kp.dbg_counts[t] = (int32_t)min((int64_t)n, kp.dbg_cap);
        if (n > kp.dbg_cap && threadIdx.x == 0) set_status(kp, SFM_STATUS_BAD_LENGTH);
        for (int pos = threadIdx.x; pos < n && pos < kp.dbg_cap; pos += blockDim.x) {
            int logical, src;
            const uint8_t *rp = resolve_row(kp, k, t, pos, &logical, &src);
            int32_t v = -1;
            if (rp) v = src ? (logical | 0x40000000) : logical;
            kp.dbg_rows[(int64_t)t * kp.dbg_cap + pos] = v;
        }
    }
}

}  // namespace

cudaError_t launch_combine(const KParams &kp, cudaStream_t st)
{
    if (kp.T == 0) return cudaSuccess;
    dim3 grid(kp.T, (kp.q_n + kHeadsPerBlock - 1) / kHeadsPerBlock);
    return launch_dependent(sfm_combine_kernel, grid, dim3(kThreads), (size_t)0, st, kp);
}

cudaError_t launch_debug(const KParams &kp, cudaStream_t st)
{
    const int grid = kp.T < 4096 ? (kp.T > 0 ? kp.T : 1) : 4096;
    sfm_debug_kernel<<<grid, 256, 0, st>>>(kp);
    return cudaGetLastError();
}

}  // namespace sfm
