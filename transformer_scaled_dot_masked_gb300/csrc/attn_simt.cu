// CUDA-core attention kernel: fp32 arithmetic from fp32 or bf16 inputs.
//
// Computes softmax(scale * Q K^T + M) V ("Paper Deep Reading: Attention Is All
// You Need", §04, attention equation with the additive mask) one key block
// at a time with a running (online) softmax: per query row it keeps the
// running maximum and the running sum of exponentials, and rescales the
// partial output whenever the maximum grows.  This is exact algebra for the
// row softmax; only rounding differs from the two-pass definition.
//
// It serves the fp32 path (true fp32: no tensor cores, so no TF32 rounding)
// and is a plain baseline for the tensor-core kernel on bf16 inputs.
//
// Grid: (ceil(m / kRows), h, B); 128 threads = 4 warps; each warp owns
// kRowsPerWarp query rows, and lane l owns output columns l, l + 32, ... (up to
// the instantiation's maximum head width, 64 or 128).  Key/value blocks of 32
// rows are staged in shared memory as fp32.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "kernels.h"

namespace attn {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRows = kWarps * kRowsPerWarp;
constexpr int kKeys = 32;
constexpr int kDMaxAll = 128; // widest head this kernel takes

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float x, float *dst) { *dst = x; }
__device__ __forceinline__ void from_f32(float x, __nv_bfloat16 *dst) { *dst = __float2bfloat16_rn(x); }

// DMAX: maximum head width of the instantiation (64 or 128); d <= DMAX.
template <typename T, int DMAX>
__global__ void __launch_bounds__(kWarps * 32)
attn_simt_kernel(const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                 const int32_t *__restrict__ key_lengths, T *__restrict__ out, float *__restrict__ lse, int h,
                 int m, int n, int d, int mask_kind, int window, float scale_log2)
{
    constexpr int kStride = DMAX + 1; // padded row stride: lane-per-key reads hit distinct banks
    constexpr int kCols = DMAX / 32;  // output columns per lane
    __shared__ float sq[kRows][kStride];
    __shared__ float sk[kKeys][kStride];
    __shared__ float sv[kKeys][DMAX];

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int b = blockIdx.z;
    const int bh = b * h + blockIdx.y;
    const int q0 = blockIdx.x * kRows;
    const bool causal = (mask_kind & kMaskCausal) != 0;

    int kv_len = n;
    if ((mask_kind & kMaskKeyPadding) && key_lengths != nullptr) {
        kv_len = key_lengths[b];
        kv_len = kv_len < 0 ? 0 : (kv_len > n ? n : kv_len);
    }
    int kv_end = kv_len;
    if (causal) kv_end = min(kv_end, min(q0 + kRows, m)); // keys beyond the last row are never allowed
    int kv_begin = 0;
    if (window >= 0) { // keys within `window` of some row of this block
        kv_end = min(kv_end, min(q0 + kRows, m) + window);
        kv_begin = max(0, q0 - window) / kKeys * kKeys;
    }

    const T *Qh = Q + static_cast<size_t>(bh) * m * d;
    const T *Kh = K + static_cast<size_t>(bh) * n * d;
    const T *Vh = V + static_cast<size_t>(bh) * n * d;

    for (int t = threadIdx.x; t < kRows * DMAX; t += blockDim.x) {
        int r = t / DMAX, c = t % DMAX;
        sq[r][c] = (q0 + r < m && c < d) ? to_f32(Qh[static_cast<size_t>(q0 + r) * d + c]) : 0.f;
    }

    float run_max[kRowsPerWarp], run_sum[kRowsPerWarp], acc[kRowsPerWarp][kCols];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        run_max[rr] = -CUDART_INF_F;
        run_sum[rr] = 0.f;
#pragma unroll
        for (int cc = 0; cc < kCols; ++cc) acc[rr][cc] = 0.f;
    }

    for (int k0 = kv_begin; k0 < kv_end; k0 += kKeys) {
        __syncthreads();
        for (int t = threadIdx.x; t < kKeys * DMAX; t += blockDim.x) {
            int r = t / DMAX, c = t % DMAX;
            bool in = (k0 + r < n) && (c < d);
            sk[r][c] = in ? to_f32(Kh[static_cast<size_t>(k0 + r) * d + c]) : 0.f;
            sv[r][c] = in ? to_f32(Vh[static_cast<size_t>(k0 + r) * d + c]) : 0.f;
        }
        __syncthreads();

        const int j = k0 + lane; // this lane's key
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            const int r = warp * kRowsPerWarp + rr;
            const int i = q0 + r;
            float s = 0.f;
            for (int c = 0; c < d; ++c) s = fmaf(sq[r][c], sk[lane][c], s);
            const bool allowed = (j < kv_len) && !(causal && j > i) &&
                                 !(window >= 0 && (j < i - window || j > i + window));
            // scale folded with log2(e): exp(x) = exp2(x * log2 e)
            const float x = allowed ? s * scale_log2 : -CUDART_INF_F;
            float blk_max = x;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) blk_max = fmaxf(blk_max, __shfl_xor_sync(0xffffffffu, blk_max, off));
            const float new_max = fmaxf(run_max[rr], blk_max);
            if (new_max == -CUDART_INF_F) continue; // nothing allowed for this row yet
            const float p = allowed ? exp2f(x - new_max) : 0.f;
            const float alpha = exp2f(run_max[rr] - new_max); // 0 when run_max is -inf
            float blk_sum = p;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) blk_sum += __shfl_xor_sync(0xffffffffu, blk_sum, off);
            run_sum[rr] = run_sum[rr] * alpha + blk_sum;
            float a[kCols];
#pragma unroll
            for (int cc = 0; cc < kCols; ++cc) a[cc] = acc[rr][cc] * alpha;
#pragma unroll 8
            for (int jj = 0; jj < kKeys; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
                for (int cc = 0; cc < kCols; ++cc) a[cc] = fmaf(pj, sv[jj][lane + 32 * cc], a[cc]);
            }
#pragma unroll
            for (int cc = 0; cc < kCols; ++cc) acc[rr][cc] = a[cc];
            run_max[rr] = new_max;
        }
    }

    // lane rr of the warp writes row rr's log-sum-exp (weights are exp2(x - run_max) / run_sum)
    if (lse != nullptr && lane < kRowsPerWarp) {
        float mx = run_max[0], sm = run_sum[0];
#pragma unroll
        for (int rr = 1; rr < kRowsPerWarp; ++rr)
            if (lane == rr) mx = run_max[rr], sm = run_sum[rr];
        const int i = q0 + warp * kRowsPerWarp + lane;
        if (i < m) lse[static_cast<size_t>(bh) * m + i] = sm > 0.f ? (mx + __log2f(sm)) * 0.6931471805599453f : -CUDART_INF_F;
    }
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int i = q0 + warp * kRowsPerWarp + rr;
        if (i >= m) continue;
        const float inv = run_sum[rr] > 0.f ? 1.f / run_sum[rr] : 0.f; // no allowed key -> 0
        T *o = out + (static_cast<size_t>(bh) * m + i) * d;
#pragma unroll
        for (int cc = 0; cc < kCols; ++cc)
            if (lane + 32 * cc < d) from_f32(acc[rr][cc] * inv, o + lane + 32 * cc);
    }
}


template <int DMAX>
cudaError_t launch_simt_w(const Problem &p, cudaStream_t stream)
{
    const float scale_log2 = p.scale * 1.4426950408889634f;
    const int win = (p.mask_kind & kMaskWindow) ? p.window : -1;
    dim3 grid((p.m + kRows - 1) / kRows, p.h, p.B);
    if (p.bf16) {
        attn_simt_kernel<__nv_bfloat16, DMAX><<<grid, kWarps * 32, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(p.q), static_cast<const __nv_bfloat16 *>(p.k),
            static_cast<const __nv_bfloat16 *>(p.v), p.key_lengths, static_cast<__nv_bfloat16 *>(p.out), p.lse, p.h,
            p.m, p.n, p.d, p.mask_kind, win, scale_log2);
    } else {
        attn_simt_kernel<float, DMAX><<<grid, kWarps * 32, 0, stream>>>(
            static_cast<const float *>(p.q), static_cast<const float *>(p.k), static_cast<const float *>(p.v),
            p.key_lengths, static_cast<float *>(p.out), p.lse, p.h, p.m, p.n, p.d, p.mask_kind, win, scale_log2);
    }
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_simt(const Problem &p, cudaStream_t stream)
{
    if (p.d > kDMaxAll) return cudaErrorInvalidValue;
    return p.d <= 64 ? launch_simt_w<64>(p, stream) : launch_simt_w<128>(p, stream);
}

} // namespace attn
