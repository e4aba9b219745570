// CUDA-core backward of the attention: fp32 arithmetic from fp32 or bf16 tensors, any
// head width up to 128 (the tensor-core backward takes bf16 heads of width up to 64).
//
// The gradients of sum(dO * out) for out = softmax(scale * Q K^T + M) V ("Paper Deep
// Reading: Attention Is All You Need", §04 attention equation; the chain rule of it):
//
//     P_ij = exp(scale * Q_i . K_j - lse_i) for allowed (i, j), else 0
//     D_i = sum_c dO_ic O_ic,   dS_ij = P_ij (dO_i . V_j - D_i)
//     dQ_i = scale sum_j dS_ij K_j,   dK_j = scale sum_i dS_ij Q_i,   dV_j = sum_i P_ij dO_i
//
// with lse the forward's per-row log-sum-exp.  Two kernels: the rows pass (one CTA
// per 16 query rows of a head: D_i, then dQ over 32-key blocks staged in shared
// memory) and the keys pass (one CTA per 16 key rows: dK and dV over 32-query blocks,
// reading D from the rows pass).  Lane l of a warp owns columns l, l + 32, ... of its
// rows' gradients; P and dS are recomputed, never stored.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "kernels.h"

namespace attn {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRows = kWarps * kRowsPerWarp; // rows of Q (rows pass) or of K (keys pass) per CTA
constexpr int kBlock = 32;                   // keys (rows pass) or queries (keys pass) per staged block
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f32(float x, float *dst) { *dst = x; }
__device__ __forceinline__ void from_f32(float x, __nv_bfloat16 *dst) { *dst = __float2bfloat16_rn(x); }

__device__ __forceinline__ int key_length(const int32_t *key_lengths, int b, int n)
{
    if (key_lengths == nullptr) return n;
    const int len = key_lengths[b];
    return len < 0 ? 0 : (len > n ? n : len);
}

__device__ __forceinline__ bool allowed(int i, int j, int len, bool causal) { return j < len && !(causal && j > i); }

template <typename T, int DMAX>
__device__ __forceinline__ void stage_rows(float (*dst)[DMAX + 1], const T *src, int row0, int rows, int count, int d)
{
    for (int t = threadIdx.x; t < count * DMAX; t += blockDim.x) {
        const int r = t / DMAX, c = t % DMAX;
        dst[r][c] = (row0 + r < rows && c < d) ? to_f32(src[static_cast<size_t>(row0 + r) * d + c]) : 0.f;
    }
}

// Rows pass: D_i (to the workspace) and dQ for query rows q0 .. q0 + 15 of head bh.
template <typename T, int DMAX>
__global__ void __launch_bounds__(kWarps * 32)
attn_bwd_simt_rows_kernel(const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                          const T *__restrict__ O, const T *__restrict__ dO, const float *__restrict__ lse,
                          const int32_t *__restrict__ key_lengths, T *__restrict__ dQ, float *__restrict__ Dbuf,
                          int h, int m, int n, int d, int mask_kind, float scale)
{
    constexpr int kS = DMAX + 1; // padded stride: lane-per-row reads hit distinct banks
    constexpr int kCols = DMAX / 32;
    extern __shared__ float smem[]; // rows_smem_bytes<DMAX>()
    float(*sq)[kS] = reinterpret_cast<float(*)[kS]>(smem);
    float(*sdo)[kS] = sq + kRows;
    float(*sk)[kS] = sdo + kRows;
    float(*sv)[kS] = sk + kBlock;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int b = blockIdx.z, bh = b * h + blockIdx.y;
    const int q0 = blockIdx.x * kRows;
    const bool causal = (mask_kind & kMaskCausal) != 0;
    const int len = (mask_kind & kMaskKeyPadding) ? key_length(key_lengths, b, n) : n;
    const int kv_end = causal ? min(len, min(q0 + kRows, m)) : len;
    const size_t head_q = static_cast<size_t>(bh) * m * d, head_k = static_cast<size_t>(bh) * n * d;

    stage_rows<T, DMAX>(sq, Q + head_q, q0, m, kRows, d);
    stage_rows<T, DMAX>(sdo, dO + head_q, q0, m, kRows, d);
    __syncthreads();

    float Di[kRowsPerWarp], lse2[kRowsPerWarp], acc[kRowsPerWarp][kCols];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int r = warp * kRowsPerWarp + rr, i = q0 + r;
        float part = 0.f;
        if (i < m)
            for (int c = lane; c < d; c += 32) part = fmaf(sdo[r][c], to_f32(O[head_q + static_cast<size_t>(i) * d + c]), part);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        Di[rr] = part;
        if (i < m && lane == 0) Dbuf[static_cast<size_t>(bh) * m + i] = part;
        // -inf: no allowed key, the row contributes nothing
        lse2[rr] = i < m ? lse[static_cast<size_t>(bh) * m + i] * kLog2e : -CUDART_INF_F;
#pragma unroll
        for (int cc = 0; cc < kCols; ++cc) acc[rr][cc] = 0.f;
    }
    const float sl2 = scale * kLog2e;

    for (int k0 = 0; k0 < kv_end; k0 += kBlock) {
        __syncthreads();
        stage_rows<T, DMAX>(sk, K + head_k, k0, n, kBlock, d);
        stage_rows<T, DMAX>(sv, V + head_k, k0, n, kBlock, d);
        __syncthreads();
        const int j = k0 + lane; // this lane's key
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            const int r = warp * kRowsPerWarp + rr, i = q0 + r;
            if (lse2[rr] == -CUDART_INF_F) continue; // warp-uniform
            float s = 0.f, dp = 0.f;
            for (int c = 0; c < d; ++c) {
                s = fmaf(sq[r][c], sk[lane][c], s);
                dp = fmaf(sdo[r][c], sv[lane][c], dp);
            }
            const float p = allowed(i, j, len, causal) ? exp2f(s * sl2 - lse2[rr]) : 0.f;
            const float ds = p * (dp - Di[rr]);
#pragma unroll 8
            for (int jj = 0; jj < kBlock; ++jj) {
                const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
                for (int cc = 0; cc < kCols; ++cc) acc[rr][cc] = fmaf(dsj, sk[jj][lane + 32 * cc], acc[rr][cc]);
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int i = q0 + warp * kRowsPerWarp + rr;
        if (i >= m) continue;
        T *g = dQ + head_q + static_cast<size_t>(i) * d;
#pragma unroll
        for (int cc = 0; cc < kCols; ++cc)
            if (lane + 32 * cc < d) from_f32(scale * acc[rr][cc], g + lane + 32 * cc);
    }
}

// Keys pass: dK and dV for key rows k0 .. k0 + 15 of head bh (0 for keys no query sees).
template <typename T, int DMAX>
__global__ void __launch_bounds__(kWarps * 32)
attn_bwd_simt_keys_kernel(const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V,
                          const T *__restrict__ dO, const float *__restrict__ lse,
                          const int32_t *__restrict__ key_lengths, const float *__restrict__ Dbuf,
                          T *__restrict__ dK, T *__restrict__ dV, int h, int m, int n, int d, int mask_kind,
                          float scale)
{
    constexpr int kS = DMAX + 1;
    constexpr int kCols = DMAX / 32;
    extern __shared__ float smem[]; // keys_smem_bytes<DMAX>()
    float(*sk)[kS] = reinterpret_cast<float(*)[kS]>(smem);
    float(*sv)[kS] = sk + kRows;
    float(*sq)[kS] = sv + kRows;
    float(*sdo)[kS] = sq + kBlock;
    float *slse2 = &sdo[kBlock][0];
    float *sD = slse2 + kBlock;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int b = blockIdx.z, bh = b * h + blockIdx.y;
    const int key0 = blockIdx.x * kRows;
    const bool causal = (mask_kind & kMaskCausal) != 0;
    const int len = (mask_kind & kMaskKeyPadding) ? key_length(key_lengths, b, n) : n;
    const size_t head_q = static_cast<size_t>(bh) * m * d, head_k = static_cast<size_t>(bh) * n * d;

    stage_rows<T, DMAX>(sk, K + head_k, key0, n, kRows, d);
    stage_rows<T, DMAX>(sv, V + head_k, key0, n, kRows, d);

    float dk[kRowsPerWarp][kCols], dv[kRowsPerWarp][kCols];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
        for (int cc = 0; cc < kCols; ++cc) dk[rr][cc] = dv[rr][cc] = 0.f;
    const float sl2 = scale * kLog2e;
    // queries that may see a key of this block: with a causal mask, i >= key0
    const int i_begin = key0 < len ? (causal ? key0 / kBlock * kBlock : 0) : m;

    for (int i0 = i_begin; i0 < m; i0 += kBlock) {
        __syncthreads();
        stage_rows<T, DMAX>(sq, Q + head_q, i0, m, kBlock, d);
        stage_rows<T, DMAX>(sdo, dO + head_q, i0, m, kBlock, d);
        if (threadIdx.x < kBlock) {
            const int i = i0 + threadIdx.x;
            slse2[threadIdx.x] = i < m ? lse[static_cast<size_t>(bh) * m + i] * kLog2e : -CUDART_INF_F;
            sD[threadIdx.x] = i < m ? Dbuf[static_cast<size_t>(bh) * m + i] : 0.f;
        }
        __syncthreads();
        const int i = i0 + lane; // this lane's query
        const float l2 = slse2[lane], Dl = sD[lane];
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            const int r = warp * kRowsPerWarp + rr, j = key0 + r;
            float s = 0.f, dp = 0.f;
            for (int c = 0; c < d; ++c) {
                s = fmaf(sq[lane][c], sk[r][c], s);
                dp = fmaf(sdo[lane][c], sv[r][c], dp);
            }
            const bool ok = i < m && l2 != -CUDART_INF_F && allowed(i, j, len, causal);
            const float p = ok ? exp2f(s * sl2 - l2) : 0.f;
            const float ds = p * (dp - Dl);
#pragma unroll 8
            for (int ii = 0; ii < kBlock; ++ii) {
                const float pi = __shfl_sync(0xffffffffu, p, ii);
                const float dsi = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
                for (int cc = 0; cc < kCols; ++cc) {
                    dv[rr][cc] = fmaf(pi, sdo[ii][lane + 32 * cc], dv[rr][cc]);
                    dk[rr][cc] = fmaf(dsi, sq[ii][lane + 32 * cc], dk[rr][cc]);
                }
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int j = key0 + warp * kRowsPerWarp + rr;
        if (j >= n) continue;
        T *gk = dK + head_k + static_cast<size_t>(j) * d, *gv = dV + head_k + static_cast<size_t>(j) * d;
#pragma unroll
        for (int cc = 0; cc < kCols; ++cc)
            if (lane + 32 * cc < d) {
                from_f32(scale * dk[rr][cc], gk + lane + 32 * cc);
                from_f32(dv[rr][cc], gv + lane + 32 * cc);
            }
    }
}

template <int DMAX> constexpr size_t rows_smem_bytes() { return (2 * kRows + 2 * kBlock) * (DMAX + 1) * sizeof(float); }
template <int DMAX>
constexpr size_t keys_smem_bytes() { return ((2 * kRows + 2 * kBlock) * (DMAX + 1) + 2 * kBlock) * sizeof(float); }

template <typename T, int DMAX>
cudaError_t launch_bwd_simt_t(const BwdSimtProblem &p, cudaStream_t stream)
{
    cudaError_t e;
    // above the 48 KB default for DMAX = 128: raise the limit (idempotent, cheap)
    if ((e = cudaFuncSetAttribute(reinterpret_cast<const void *>(attn_bwd_simt_rows_kernel<T, DMAX>),
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(rows_smem_bytes<DMAX>()))) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(reinterpret_cast<const void *>(attn_bwd_simt_keys_kernel<T, DMAX>),
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(keys_smem_bytes<DMAX>()))) != cudaSuccess)
        return e;
    float *Dbuf = static_cast<float *>(p.workspace);
    const dim3 rows((p.m + kRows - 1) / kRows, p.h, p.B), keys((p.n + kRows - 1) / kRows, p.h, p.B);
    attn_bwd_simt_rows_kernel<T, DMAX><<<rows, kWarps * 32, rows_smem_bytes<DMAX>(), stream>>>(
        static_cast<const T *>(p.q), static_cast<const T *>(p.k), static_cast<const T *>(p.v),
        static_cast<const T *>(p.out), static_cast<const T *>(p.dout), p.lse, p.key_lengths, static_cast<T *>(p.dq),
        Dbuf, p.h, p.m, p.n, p.d, p.mask_kind, p.scale);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    attn_bwd_simt_keys_kernel<T, DMAX><<<keys, kWarps * 32, keys_smem_bytes<DMAX>(), stream>>>(
        static_cast<const T *>(p.q), static_cast<const T *>(p.k), static_cast<const T *>(p.v),
        static_cast<const T *>(p.dout), p.lse, p.key_lengths, Dbuf, static_cast<T *>(p.dk), static_cast<T *>(p.dv),
        p.h, p.m, p.n, p.d, p.mask_kind, p.scale);
    return cudaGetLastError();
}

} // namespace

size_t bwd_simt_workspace_bytes(int B, int h, int m) { return static_cast<size_t>(B) * h * m * sizeof(float); }

cudaError_t launch_bwd_simt(const BwdSimtProblem &p, cudaStream_t stream)
{
    if (p.d < 1 || p.d > 128) return cudaErrorInvalidValue;
    if (p.bf16)
        return p.d <= 64 ? launch_bwd_simt_t<__nv_bfloat16, 64>(p, stream)
                         : launch_bwd_simt_t<__nv_bfloat16, 128>(p, stream);
    return p.d <= 64 ? launch_bwd_simt_t<float, 64>(p, stream) : launch_bwd_simt_t<float, 128>(p, stream);
}

} // namespace attn
