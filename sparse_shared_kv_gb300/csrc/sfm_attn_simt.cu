// sfm_attn_simt.cu -- generic split-KV attention kernel (fp32 CUDA cores).
//
// Covers every configuration the boundary accepts: q_n 1..128, bf16 / fp16,
// BSND / TND / paged KV with padded rows, window / causal / unmasked ori,
// CSA / HCA compressed KV, token-wise ori indices and the INT8 / FP8 packed rows of
// the kv_quant_sparse_flash_attention guide (dequantised exactly to fp32 in
// shared memory: K~[d] = int8[d] * scale[d / 128]).
//
// One CTA = one worker of the plan x one group of HG heads.  For each split
// of its range it streams TR-row tiles of attended KV through shared memory
// and keeps an online softmax (running max m, sum l, unnormalised O) per head:
//   S = Q.K~^T * scale;  m' = max(m, max S);  O = O*e^(m-m') + e^(S-m') V~
// A row with a single split is finalised here (sinks, 1/denominator, LSE);
// otherwise the split's normalised O and its LSE go to the workspace for the
// combine kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "sfm_internal.cuh"

namespace sfm {

namespace {

constexpr int HG = 16;          // heads per CTA
constexpr int TR = 32;          // KV rows per tile
constexpr int kThreads = 256;   // 8 warps; warp w scores heads 2w, 2w+1
constexpr int kMaxDqk = 576;
constexpr int kStride = kMaxDqk + 1;   // padded fp32 row stride in shared memory

struct __align__(16) Smem {
    float q[HG][kStride];
    float k[TR][kStride];
    float p[HG][TR];
    float alpha[HG];
    const uint8_t *rowp[TR];
};

__device__ __forceinline__ float half_to_float(uint16_t h, int dtype)
{
    if (dtype == SFM_DTYPE_BF16) return __uint_as_float((uint32_t)h << 16);
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ uint16_t float_to_half(float f, int dtype)
{
    if (dtype == SFM_DTYPE_BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(f));
    return __half_as_ushort(__float2half_rn(f));
}

__device__ __forceinline__ float warp_max(float v)
{
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Load tile row r (16-byte chunks) into s.k[r][:] as fp32; zero for skipped rows.
__device__ __forceinline__ void load_tile(const KParams &kp, Smem &s, int nrows)
{
    const int tid = threadIdx.x;
    if (!kp.packed) {
        // 512 bf16/fp16 = 64 chunks of 8 values per row
        for (int c = tid; c < TR * 64; c += kThreads) {
            const int r = c >> 6, j = c & 63;
            const uint8_t *rp = s.rowp[r];
            float *dst = &s.k[r][j * 8];
            if (r < nrows && rp) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(rp) + j);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    dst[2 * e] = half_to_float((uint16_t)(w[e] & 0xffffu), kp.dtype);
                    dst[2 * e + 1] = half_to_float((uint16_t)(w[e] >> 16), kp.dtype);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) dst[e] = 0.f;
            }
        }
        return;
    }
    // packed: 32 int8 chunks (16 values each) + rope/8 chunks of 8 rope values
    const int rope_chunks = kp.rope / 8;
    const int per_row = 32 + rope_chunks;
    for (int c = tid; c < TR * per_row; c += kThreads) {
        const int r = c / per_row, j = c - r * per_row;
        const uint8_t *rp = s.rowp[r];
        if (j < 32) {
            float *dst = &s.k[r][j * 16];
            if (r < nrows && rp) {
                const float sc = __ldg(reinterpret_cast<const float *>(rp + 512 + 2 * kp.rope) + (j >> 3));
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(rp) + j);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                if (kp.kv_fp8) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float f[4];
                        e4m3x4_to_f32(w[q], f);
#pragma unroll
                        for (int e = 0; e < 4; ++e) dst[4 * q + e] = f[e] * sc;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int8_t x = (int8_t)((w[e >> 2] >> (8 * (e & 3))) & 0xffu);
                        dst[e] = (float)x * sc;
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) dst[e] = 0.f;
            }
        } else {
            const int jj = j - 32;
            float *dst = &s.k[r][512 + jj * 8];
            if (r < nrows && rp) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(rp + 512) + jj);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    dst[2 * e] = half_to_float((uint16_t)(w[e] & 0xffffu), kp.dtype);
                    dst[2 * e + 1] = half_to_float((uint16_t)(w[e] >> 16), kp.dtype);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) dst[e] = 0.f;
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads) sfm_attn_simt_kernel(KParams kp)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem &s = *reinterpret_cast<Smem *>(smem_raw);
    grid_launch_dependents();
    grid_dependency_wait();      // the plan comes from the preceding planner launch
    if (!meta_ok(kp)) return;   // the combine kernel zeroes the outputs and flags the status

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int worker = blockIdx.x;
    const int h0 = blockIdx.y * HG;
    const int nh = min(HG, kp.q_n - h0);
    const int G = kp.G, T = kp.T, SR = kp.split_rows;
    const int32_t *sp = kp.meta + meta_split_off(G);
    const int w_beg = kp.meta[meta_ws_off() + worker];
    const int w_end = kp.meta[meta_ws_off() + worker + 1];

    for (int w = w_beg; w < w_end; ++w) {
        const int t = split_owner(sp, T, w);
        const int nsplit = sp[t + 1] - sp[t];
        const int sidx = w - sp[t];
        const Tok k = token_info(kp, t);
        const int n = k.n_ori + k.n_cmp;
        const int size = split_size_dev(n, kp.split_div);
        const int pos0 = sidx * size;
        const int pos1 = min(n, pos0 + size);
        const bool final_split = nsplit == 1;
        const int64_t slot = (int64_t)t * kp.max_splits + sidx;     // the row's workspace slot for this split
        if (!final_split && (kp.max_splits <= 1 || sidx >= kp.max_splits)) {
            set_status(kp, SFM_STATUS_WORKSPACE_OVERFLOW);
            continue;
        }

        // Q of this row and head group -> fp32 shared memory
        __syncthreads();
        const uint16_t *qg = reinterpret_cast<const uint16_t *>(kp.q) + ((int64_t)t * kp.q_n + h0) * kp.d_qk;
        for (int e = tid; e < HG * kp.d_qk; e += kThreads) {
            const int h = e / kp.d_qk, d = e - h * kp.d_qk;
            s.q[h][d] = h < nh ? half_to_float(__ldg(qg + (int64_t)h * kp.d_qk + d), kp.dtype) : 0.f;
        }

        float acc[HG][2];
#pragma unroll
        for (int h = 0; h < HG; ++h) acc[h][0] = acc[h][1] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // heads 2*warp, 2*warp+1

        for (int base = pos0; base < pos1; base += TR) {
            const int nrows = min(TR, pos1 - base);
            __syncthreads();
            if (tid < TR) {
                const uint8_t *rp = nullptr;
                if (tid < nrows) {
                    int logical, src;
                    rp = resolve_row(kp, k, t, base + tid, &logical, &src);
                }
                s.rowp[tid] = rp;
            }
            __syncthreads();
            load_tile(kp, s, nrows);
            __syncthreads();

            // scores: lane = row, warp = 2 heads
            const int ha = 2 * warp, hb = 2 * warp + 1;
            float sa = 0.f, sb = 0.f;
            const float *kr = &s.k[lane][0];
            for (int d = 0; d < kp.d_qk; ++d) {
                const float kv = kr[d];
                sa = fmaf(s.q[ha][d], kv, sa);
                sb = fmaf(s.q[hb][d], kv, sb);
            }
            const bool live = lane < nrows && s.rowp[lane] != nullptr;
            sa = live ? sa * kp.scale : -INFINITY;
            sb = live ? sb * kp.scale : -INFINITY;
            const float ma = fmaxf(m0, warp_max(sa));
            const float mb = fmaxf(m1, warp_max(sb));
            const float pa = ma == -INFINITY ? 0.f : expf(sa - ma);
            const float pb = mb == -INFINITY ? 0.f : expf(sb - mb);
            const float aa = ma == -INFINITY ? 1.f : expf(m0 - ma);
            const float ab = mb == -INFINITY ? 1.f : expf(m1 - mb);
            l0 = l0 * aa + warp_sum(pa);
            l1 = l1 * ab + warp_sum(pb);
            m0 = ma;
            m1 = mb;
            s.p[ha][lane] = pa;
            s.p[hb][lane] = pb;
            if (lane == 0) {
                s.alpha[ha] = aa;
                s.alpha[hb] = ab;
            }
            __syncthreads();

            // O[h][d] for d = tid, tid + 256
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                const float al = s.alpha[h];
                float o0 = acc[h][0] * al, o1 = acc[h][1] * al;
                for (int r = 0; r < nrows; ++r) {
                    const float pr = s.p[h][r];
                    o0 = fmaf(pr, s.k[r][tid], o0);
                    o1 = fmaf(pr, s.k[r][tid + 256], o1);
                }
                acc[h][0] = o0;
                acc[h][1] = o1;
            }
        }

        // publish m, l of every head for the epilogue
        __syncthreads();
        if (lane == 0) {
            s.p[2 * warp][0] = m0;
            s.p[2 * warp][1] = l0;
            s.p[2 * warp + 1][0] = m1;
            s.p[2 * warp + 1][1] = l1;
        }
        __syncthreads();
        for (int h = 0; h < nh; ++h) {
            const int hh = h0 + h;
            const float m = s.p[h][0], l = s.p[h][1];
            const int64_t row = (int64_t)t * kp.q_n + hh;
            if (final_split) {
                float inv = 0.f;
                if (l > 0.f) {
                    float den = l;
                    if (kp.sinks) den += expf(__ldg(kp.sinks + hh) - m);
                    inv = 1.f / den;
                }
                uint16_t *o = reinterpret_cast<uint16_t *>(kp.out) + row * 512;
                o[tid] = float_to_half(acc[h][0] * inv, kp.dtype);
                o[tid + 256] = float_to_half(acc[h][1] * inv, kp.dtype);
                if (tid == 0 && kp.lse) kp.lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
            } else {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                // chunk-major partial: [split][dim / 8][head][8]
                uint16_t *o = kp.ws_o + slot * kp.q_n * 512;
                const int d0 = tid, d1 = tid + 256;
                o[((int64_t)(d0 >> 3) * kp.q_n + hh) * 8 + (d0 & 7)] = float_to_half(acc[h][0] * inv, SFM_DTYPE_BF16);
                o[((int64_t)(d1 >> 3) * kp.q_n + hh) * 8 + (d1 & 7)] = float_to_half(acc[h][1] * inv, SFM_DTYPE_BF16);
                if (tid == 0) kp.ws_lse[slot * kp.q_n + hh] = l > 0.f ? m + logf(l) : -INFINITY;
            }
        }
    }
}

}  // namespace

cudaError_t launch_attn_simt(const KParams &kp, cudaStream_t st)
{
    const size_t smem = sizeof(Smem);
    cudaError_t e = cudaFuncSetAttribute(sfm_attn_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(kp.G, (kp.q_n + HG - 1) / HG);
    return launch_dependent(sfm_attn_simt_kernel, grid, dim3(kThreads), smem, st, kp);
}

}  // namespace sfm
