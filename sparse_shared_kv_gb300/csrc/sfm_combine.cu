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
// match the params, zeroes every output and flags the status word.  It runs
// only when a row can have more than one split: for tensor-core plans of at
// most one split per row the attention kernel finishes every row itself.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "sfm_internal.cuh"

namespace sfm {

namespace {

constexpr int kThreads = 256;                 // 8 warps
constexpr int kChunksPerRow = 512 / 8;        // 16-byte pieces of a 512-dim row

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

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], float w, uint4 v)
{
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {      // bf16 pair -> two floats (exact)
        acc[2 * e] = fmaf(w, __uint_as_float(wv[e] << 16), acc[2 * e]);
        acc[2 * e + 1] = fmaf(w, __uint_as_float(wv[e] & 0xffff0000u), acc[2 * e + 1]);
    }
}

// Warps per 16-byte piece of the rows: one lane per head, ceil(q_n / 32)
// warps cover a piece of every head; a CTA covers 8 / that many pieces.
__host__ __device__ constexpr int warps_per_piece(int q_n) { return q_n <= 32 ? 1 : q_n <= 64 ? 2 : 4; }

// grid (query rows, 64 / pieces per CTA).  Thread = (head, piece): its loads
// (the split LSEs of its head, its piece of each split's partial) are
// coalesced across the warp's 32 heads, since partials are stored
// chunk-major ([slot][dim / 8][head][8]).  Row t's partials sit in workspace
// slots t * max_splits + s, so with up to kUnrolled possible splits every load
// -- plan words, sink, LSEs, pieces -- goes out at once and the merge costs
// one round trip (slots past the row's split count are loaded, never used).
// The merged pieces are transposed through shared memory so that each head's
// output bytes are written contiguously.
__global__ void __launch_bounds__(kThreads) sfm_combine_kernel(KParams kp)
{
    __shared__ uint4 s_out[128 * 8];            // [head][piece of this CTA]
    const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int HW = warps_per_piece(kp.q_n), PC = 8 / HW;
    const int wc = warp / HW;                   // piece within this CTA
    const int h = (warp - wc * HW) * 32 + lane;
    const int chunk = blockIdx.y * PC + wc;
    grid_launch_dependents();    // the next launch on the stream may start its set-up
    grid_dependency_wait();      // partial results come from the attention launch before this one
    const int32_t *sp = kp.meta + meta_split_off(kp.G);
    const int32_t sp0 = sp[t], sp1 = sp[t + 1];      // independent of the header check
    const bool ok = meta_ok(kp);
    const bool live = h < kp.q_n;
    const int hh = live ? h : 0;
    const int MS = kp.max_splits;
    const int64_t slot0 = (int64_t)t * MS;
    const float sink = kp.sinks ? __ldg(kp.sinks + hh) : 0.f;
    auto piece = [&](int sx) -> const uint4 * {
        return reinterpret_cast<const uint4 *>(kp.ws_o + (slot0 + sx) * kp.q_n * 512 + ((int64_t)chunk * kp.q_n + hh) * 8);
    };
    auto lse_of = [&](int sx) -> float { return kp.ws_lse[(slot0 + sx) * kp.q_n + hh]; };
    const bool early = MS > 1 && MS <= kUnrolled;
    float pl[kUnrolled];
    uint4 v[kUnrolled];
    if (early) {
#pragma unroll
        for (int sx = 0; sx < kUnrolled; ++sx) {
            pl[sx] = sx < MS ? lse_of(sx) : -INFINITY;
            v[sx] = sx < MS ? *piece(sx) : make_uint4(0, 0, 0, 0);
        }
    }
    if (t == 0 && blockIdx.y == 0 && threadIdx.x == 0) {     // after this thread's loads are out
        if (!ok) set_status(kp, SFM_STATUS_METADATA_MISMATCH | kp.meta[H_FLAGS]);
        else if (kp.meta[H_LENFLAGS]) set_status(kp, kp.meta[H_LENFLAGS]);
    }
    int ns = 0;
    if (ok) {
        ns = sp1 - sp0;
        if (ns == 1) return;      // finalised by the attention kernel (uniform over the CTA)
        if (ns > 1 && ns > MS) {
            if (threadIdx.x == 0) set_status(kp, SFM_STATUS_WORKSPACE_OVERFLOW);
            ns = 0;
        }
    }
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    float L = -INFINITY;
    if (ns > 0 && early) {
        float m = -INFINITY;
#pragma unroll
        for (int sx = 0; sx < kUnrolled; ++sx)
            if (sx < ns) m = fmaxf(m, pl[sx]);
        if (m != -INFINITY) {
            float z = 0.f;
#pragma unroll
            for (int sx = 0; sx < kUnrolled; ++sx)
                if (sx < ns) z += expf(pl[sx] - m);
            L = m + logf(z);
#pragma unroll
            for (int sx = 0; sx < kUnrolled; ++sx)
                if (sx < ns) acc_bf16x8(acc, expf(pl[sx] - L), v[sx]);
        }
    } else if (ns > 0) {
        float m = -INFINITY;
        for (int sx = 0; sx < ns; ++sx) m = fmaxf(m, lse_of(sx));
        if (m != -INFINITY) {
            float z = 0.f;
            for (int sx = 0; sx < ns; ++sx) z += expf(lse_of(sx) - m);
            L = m + logf(z);
            for (int sx = 0; sx < ns; ++sx) acc_bf16x8(acc, expf(lse_of(sx) - L), *piece(sx));
        }
    }
    if (L != -INFINITY && kp.sinks) {
        const float f = 1.f / (1.f + expf(sink - L));
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] *= f;
    }
    if (live) {
        s_out[h * PC + wc] = make_uint4(to_half2(acc[0], acc[1], kp.dtype), to_half2(acc[2], acc[3], kp.dtype),
                                        to_half2(acc[4], acc[5], kp.dtype), to_half2(acc[6], acc[7], kp.dtype));
        if (chunk == 0 && kp.lse) kp.lse[(int64_t)t * kp.q_n + h] = L;
    }
    __syncthreads();
    // PC consecutive pieces (16 PC bytes) of one head per group of PC threads
    uint4 *out = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(kp.out) + (int64_t)t * kp.q_n * 512);
    for (int i = threadIdx.x; i < kp.q_n * PC; i += kThreads) {
        const int oh = i / PC, op = i - oh * PC;
        out[(int64_t)oh * kChunksPerRow + blockIdx.y * PC + op] = s_out[oh * PC + op];
    }
}

}  // namespace

cudaError_t launch_combine(const KParams &kp, cudaStream_t st)
{
    if (kp.T == 0) return cudaSuccess;
    dim3 grid(kp.T, kChunksPerRow / (8 / warps_per_piece(kp.q_n)));
    return launch_dependent(sfm_combine_kernel, grid, dim3(kThreads), (size_t)0, st, kp);
}


}  // namespace sfm
