// sfm_combine.cu -- merge the split-KV partial results of each query row.
//
// For a row whose attended positions were cut into splits s = 0..n-1 with
// normalised partial outputs O_s and partial LSEs lse_s:
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

constexpr int kThreads = 256;
constexpr int kMaxSplits = 64;    // per row, merged from shared memory in chunks of this size

__device__ __forceinline__ uint16_t to_half(float f, int dtype)
{
    if (dtype == SFM_DTYPE_BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(f));
    return __half_as_ushort(__float2half_rn(f));
}

__global__ void __launch_bounds__(kThreads) sfm_combine_kernel(KParams kp)
{
    __shared__ float s_w[kMaxSplits];
    __shared__ float s_red[2];
    const int t = blockIdx.x, tid = threadIdx.x;
    const bool ok = meta_ok(kp);
    if (!ok && t == 0 && tid == 0) set_status(kp, SFM_STATUS_METADATA_MISMATCH | kp.meta[H_FLAGS]);
    int ns = 0, s0 = 0;
    if (ok) {
        const int32_t *sp = kp.meta + meta_split_off(kp.G);
        s0 = sp[t];
        ns = sp[t + 1] - s0;
        if (ns == 1) return;      // finalised by the attention kernel
        if (ns > 1 && (int64_t)s0 + ns > kp.ws_capacity_splits) {
            if (tid == 0) set_status(kp, SFM_STATUS_WORKSPACE_OVERFLOW);
            ns = 0;
        }
    }
    for (int h = 0; h < kp.q_n; ++h) {
        const int64_t row = (int64_t)t * kp.q_n + h;
        uint16_t *o = reinterpret_cast<uint16_t *>(kp.out) + row * 512;
        if (ns == 0) {
            o[tid] = to_half(0.f, kp.dtype);
            o[tid + 256] = to_half(0.f, kp.dtype);
            if (tid == 0 && kp.lse) kp.lse[row] = -INFINITY;
            continue;
        }
        // LSE of the row: max then sum over the splits (thread 0, split order)
        __syncthreads();
        if (tid == 0) {
            float m = -INFINITY;
            for (int s = 0; s < ns; ++s) m = fmaxf(m, kp.ws_lse[(int64_t)(s0 + s) * kp.q_n + h]);
            float z = 0.f;
            if (m != -INFINITY)
                for (int s = 0; s < ns; ++s) z += expf(kp.ws_lse[(int64_t)(s0 + s) * kp.q_n + h] - m);
            s_red[0] = m;
            s_red[1] = z;
        }
        __syncthreads();
        const float m = s_red[0], z = s_red[1];
        const float L = m == -INFINITY ? -INFINITY : m + logf(z);
        float a0 = 0.f, a1 = 0.f;
        if (L != -INFINITY) {
            float sink_f = 1.f;
            if (kp.sinks) sink_f = 1.f / (1.f + expf(__ldg(kp.sinks + h) - L));
            for (int c0 = 0; c0 < ns; c0 += kMaxSplits) {
                const int cn = min(kMaxSplits, ns - c0);
                __syncthreads();
                if (tid < cn) s_w[tid] = expf(kp.ws_lse[(int64_t)(s0 + c0 + tid) * kp.q_n + h] - L);
                __syncthreads();
                for (int s = 0; s < cn; ++s) {
                    const float *os = kp.ws_o + ((int64_t)(s0 + c0 + s) * kp.q_n + h) * 512;
                    a0 = fmaf(s_w[s], os[tid], a0);
                    a1 = fmaf(s_w[s], os[tid + 256], a1);
                }
            }
            a0 *= sink_f;
            a1 *= sink_f;
        }
        o[tid] = to_half(a0, kp.dtype);
        o[tid + 256] = to_half(a1, kp.dtype);
        if (tid == 0 && kp.lse) kp.lse[row] = L;
    }
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
    sfm_combine_kernel<<<kp.T, kThreads, 0, st>>>(kp);
    return cudaGetLastError();
}

cudaError_t launch_debug(const KParams &kp, cudaStream_t st)
{
    const int grid = kp.T < 4096 ? (kp.T > 0 ? kp.T : 1) : 4096;
    sfm_debug_kernel<<<grid, 256, 0, st>>>(kp);
    return cudaGetLastError();
}

}  // namespace sfm
