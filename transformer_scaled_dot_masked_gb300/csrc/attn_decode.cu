// Incremental decoding: a few new query rows per (batch, head) against a cached
// K/V prefix, the decoder's per-step attention during generation ("Paper Deep
// Reading: Attention Is All You Need", §03 "Decoder layer": the decoder produces
// one position at a time and attends to the positions produced so far; the slide
// deck's "Training Details" / results slides use beam search).  Every new query
// sees the cached keys 0 .. len_b - 1 of its batch entry (the key-padding mask of
// the attention equation with len_b = the cache length), so the result is exactly
// attn_fwd with ATTN_MASK_KEY_PADDING.
//
// The work is memory-bound (each cached K and V row is read once per step and used
// by m <= 8 queries), so it runs on the CUDA cores and is split over the keys
// (split-KV): CTA (split, b*h) reads keys [split * chunk, (split + 1) * chunk) of
// one head.  Eight lanes share a key row (16 bytes each, so a warp load covers
// four whole rows), each eight-lane group keeps an online softmax over its rows,
// and the CTA merges its 32 groups.  With one split the CTA writes the output;
// otherwise it writes (max, sum, unnormalised O) and attn_decode_combine_kernel
// merges the splits.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <cstdint>

#include "kernels.h"

namespace attn {

namespace {

constexpr int kWarps = 8;
// D: head width (16, 32, 64 or 128).  Every lane holds 16 bytes (8 dims) of a key row,
// so a row spans D / 8 lanes and a warp reads 32 / (D / 8) rows per pass.
template <int D> __host__ __device__ constexpr int lanes_per_row() { return D / 8; }
template <int D> __host__ __device__ constexpr int rows_per_warp() { return 32 / (D / 8); }
template <int D> __host__ __device__ constexpr int rows_per_pass() { return kWarps * rows_per_warp<D>(); }
template <int D> __host__ __device__ constexpr int part_of() { return D + 2; } // floats of one partial: O, max, sum
// passes of rows each warp has in flight
template <int M>
__host__ __device__ constexpr int depth_of() { return M > 4 ? 3 : 4; }

// 16 bytes global -> shared without registers (zero-filled when !valid: no read).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Merge softmax state (m2, l2, a2) into (m, l, a): both are sums of exp2(x - m)
// weights over disjoint key sets.
template <int M>
__device__ __forceinline__ void merge(float (&m)[M], float (&l)[M], float (&a)[M][8], const float (&m2)[M],
                                      const float (&l2)[M], const float (&a2)[M][8])
{
#pragma unroll
    for (int q = 0; q < M; ++q) {
        const float mn = fmaxf(m[q], m2[q]);
        const float f1 = mn == -CUDART_INF_F ? 0.f : ex2f(m[q] - mn);
        const float f2 = mn == -CUDART_INF_F ? 0.f : ex2f(m2[q] - mn);
        l[q] = l[q] * f1 + l2[q] * f2;
#pragma unroll
        for (int e = 0; e < 8; ++e) a[q][e] = a[q][e] * f1 + a2[q][e] * f2;
        m[q] = mn;
    }
}

// M: query rows handled per (b, h) (the call's m rounded up to 1, 2, 4 or 8); D: head width.
template <int M, int D>
__global__ void __launch_bounds__(kWarps * 32, M == 1 ? 5 : 1)
attn_decode_kernel(const __nv_bfloat16 *__restrict__ Q, const __nv_bfloat16 *__restrict__ K,
                   const __nv_bfloat16 *__restrict__ V, const int32_t *__restrict__ lengths,
                   __nv_bfloat16 *__restrict__ out, float *__restrict__ lse, float *__restrict__ part, int h,
                   int m, int n, int chunk, int splits, float scale_log2)
{
    constexpr int kL = lanes_per_row<D>(), kRowsPerWarp = rows_per_warp<D>(), kRowsPerPass = rows_per_pass<D>();
    constexpr int kPart = part_of<D>();
    // each lane's 16-byte slices of its K and V rows, kDepth passes deep per warp; once
    // every copy has landed and been read, the same bytes hold the warps' partials
    constexpr int kDepth = depth_of<M>();
    constexpr int kRingBytes = kWarps * kDepth * 2 * 32 * 16;
    constexpr int kRedBytes = kWarps * M * kPart * 4;
    __shared__ __align__(16) unsigned char smem[kRingBytes > kRedBytes ? kRingBytes : kRedBytes];
    auto ring_at = [&](int w, int st) {
        return static_cast<uint32_t>(__cvta_generic_to_shared(smem)) + ((w * kDepth + st) * 2 * 32) * 16;
    };
    float(*red)[M][kPart] = reinterpret_cast<float(*)[M][kPart]>(smem);
    const int bh = blockIdx.x;
    const int split = blockIdx.y;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int r = lane / kL; // key row within the warp's kRowsPerWarp
    const int j = lane % kL; // 16-byte slice of the row: dims 8j .. 8j+7
    int len = n;
    if (lengths != nullptr) {
        len = __ldg(lengths + bh / h);
        len = len < 0 ? 0 : (len > n ? n : len);
    }
    const int k_begin = split * chunk;
    const int k_end = min(len, k_begin + chunk);

    // this lane's slice of every query row, pre-multiplied by scale * log2 e
    float q[M][8];
#pragma unroll
    for (int qi = 0; qi < M; ++qi) {
        if (qi < m) {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(Q + (static_cast<size_t>(bh) * m + qi) * D) + j);
            unpack8(u, q[qi]);
#pragma unroll
            for (int e = 0; e < 8; ++e) q[qi][e] *= scale_log2;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) q[qi][e] = 0.f;
        }
    }
    float mx[M], sm[M], acc[M][8];
#pragma unroll
    for (int qi = 0; qi < M; ++qi) {
        mx[qi] = -CUDART_INF_F;
        sm[qi] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[qi][e] = 0.f;
    }

    const uint4 *Kh = reinterpret_cast<const uint4 *>(K + static_cast<size_t>(bh) * n * D);
    const uint4 *Vh = reinterpret_cast<const uint4 *>(V + static_cast<size_t>(bh) * n * D);
    // Passes over the warp's rows are warp-uniform (the shuffles below need all 32
    // lanes); a row past the chunk is loaded as nothing and skipped after them.
    // Each lane copies its own 16-byte slices of the K and V rows of the next
    // kDepth - 1 passes into shared memory (cp.async, no registers held) and reads
    // back only what it copied, so its own wait_group is the only ordering needed.
    int row = k_begin + warp * kRowsPerWarp + r;
    const uint32_t my_ring = ring_at(warp, 0) + lane * 16;
    auto issue = [&](int prow, int st) {
        const bool v = prow < k_end;
        const size_t at = static_cast<size_t>(v ? prow : 0) * kL + j; // row 0 exists: n >= 1
        cp_async16(my_ring + st * (2 * 32 * 16), Kh + at, v);
        cp_async16(my_ring + st * (2 * 32 * 16) + 32 * 16, Vh + at, v);
        cp_async_commit();
    };
#pragma unroll
    for (int st = 0; st < kDepth - 1; ++st) issue(row + st * kRowsPerPass, st);
    int stage = 0;
    for (int base = k_begin + warp * kRowsPerWarp; base < k_end; base += kRowsPerPass, row += kRowsPerPass) {
        const bool valid = row < k_end;
        // the stage read in the previous pass is refilled (an empty group past the end)
        issue(row + (kDepth - 1) * kRowsPerPass, (stage + kDepth - 1) % kDepth);
        cp_async_wait<kDepth - 1>();
        const uint4 ku = ld_shared_u4(my_ring + stage * (2 * 32 * 16));
        const uint4 vu = ld_shared_u4(my_ring + stage * (2 * 32 * 16) + 32 * 16);
        stage = (stage + 1) % kDepth;
        float kf[8], vf[8];
        unpack8(ku, kf);
        unpack8(vu, vf);
#pragma unroll
        for (int qi = 0; qi < M; ++qi) {
            float x = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) x = fmaf(q[qi][e], kf[e], x);
            // the kL lanes of this row hold its kL partial dot products
#pragma unroll
            for (int off = 1; off < kL; off *= 2) x += __shfl_xor_sync(0xffffffffu, x, off);
            if (valid) {
                const float mn = fmaxf(mx[qi], x);
                const float alpha = ex2f(mx[qi] - mn); // 0 on the group's first row
                const float pw = ex2f(x - mn);
                sm[qi] = sm[qi] * alpha + pw;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[qi][e] = fmaf(pw, vf[e], acc[qi][e] * alpha);
                mx[qi] = mn;
            }
        }
    }
    cp_async_wait<0>(); // no copy may still target the ring when the CTA moves on
    // the warp's row groups (lanes j, j + kL, ...) into lanes 0 .. kL - 1
#pragma unroll
    for (int off = kL; off <= 16; off *= 2) {
        float m2[M], l2[M], a2[M][8];
#pragma unroll
        for (int qi = 0; qi < M; ++qi) {
            m2[qi] = __shfl_xor_sync(0xffffffffu, mx[qi], off);
            l2[qi] = __shfl_xor_sync(0xffffffffu, sm[qi], off);
#pragma unroll
            for (int e = 0; e < 8; ++e) a2[qi][e] = __shfl_xor_sync(0xffffffffu, acc[qi][e], off);
        }
        merge<M>(mx, sm, acc, m2, l2, a2);
    }
    __syncthreads(); // every warp is done with the ring: its bytes now hold the partials
    if (lane < kL) {
#pragma unroll
        for (int qi = 0; qi < M; ++qi) {
#pragma unroll
            for (int e = 0; e < 8; ++e) red[warp][qi][8 * j + e] = acc[qi][e];
            if (j == 0) {
                red[warp][qi][D] = mx[qi];
                red[warp][qi][D + 1] = sm[qi];
            }
        }
    }
    __syncthreads();
    // the CTA's warps: thread t < M * D merges dimension t % D of query t / D
    for (int t = threadIdx.x; t < M * D; t += blockDim.x) {
        const int qi = t / D, dim = t % D;
        if (qi >= m) continue;
        float mm = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, red[w][qi][D]);
        float ll = 0.f, aa = 0.f;
        if (mm != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = ex2f(red[w][qi][D] - mm);
                ll += red[w][qi][D + 1] * f;
                aa += red[w][qi][dim] * f;
            }
        }
        const size_t row = static_cast<size_t>(bh) * m + qi;
        if (splits == 1) {
            out[row * D + dim] = __float2bfloat16_rn(ll > 0.f ? aa / ll : 0.f); // no allowed key -> 0
            if (lse != nullptr && dim == 0)
                lse[row] = ll > 0.f ? (mm + __log2f(ll)) * 0.6931471805599453f : -CUDART_INF_F;
        } else {
            float *pp = part + (row * splits + split) * kPart;
            pp[dim] = aa;
            if (dim == 0) {
                pp[D] = mm;
                pp[D + 1] = ll;
            }
        }
    }
}

// One warp per (b, h, query row): merge the splits' (max, sum, O), divide, store.
template <int D>
__global__ void attn_decode_combine_kernel(const float *__restrict__ part, __nv_bfloat16 *__restrict__ out,
                                           float *__restrict__ lse, int rows, int splits)
{
    constexpr int kPart = part_of<D>();
    constexpr int kPer = (D + 31) / 32; // dimensions per lane
    const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= rows) return;
    const float *pr = part + static_cast<size_t>(row) * splits * kPart;
    float mm = -CUDART_INF_F;
    for (int s = lane; s < splits; s += 32) mm = fmaxf(mm, pr[s * kPart + D]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));
    float ll = 0.f, a[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) a[u] = 0.f;
    if (mm != -CUDART_INF_F) {
        for (int s = 0; s < splits; ++s) {
            const float *ps = pr + s * kPart;
            const float f = ex2f(ps[D] - mm); // 0 for a split with no key (max -inf)
            ll += ps[D + 1] * f;
#pragma unroll
            for (int u = 0; u < kPer; ++u)
                if (lane + 32 * u < D) a[u] += ps[lane + 32 * u] * f;
        }
    }
    const float inv = ll > 0.f ? 1.f / ll : 0.f;
#pragma unroll
    for (int u = 0; u < kPer; ++u)
        if (lane + 32 * u < D) out[static_cast<size_t>(row) * D + lane + 32 * u] = __float2bfloat16_rn(a[u] * inv);
    if (lse != nullptr && lane == 0) lse[row] = ll > 0.f ? (mm + __log2f(ll)) * 0.6931471805599453f : -CUDART_INF_F;
}

} // namespace

int decode_splits(int B, int h, int n, int sms)
{
    // Enough CTAs for about four waves, and no CTA reading more than 512 keys (so
    // heads with long caches do not finish alone), each reading at least 256 keys.
    const int max_splits = (n + 255) / 256;
    const long heads = static_cast<long>(B) * h;
    long want = (4L * sms + heads - 1) / heads;
    const long by_rows = (n + 511) / 512;
    if (want < by_rows) want = by_rows;
    if (want < 1) want = 1;
    if (want > max_splits) want = max_splits;
    if (want > 65535) want = 65535;
    return static_cast<int>(want);
}

size_t decode_workspace_bytes(int B, int h, int m, int n, int d, int sms)
{
    const int splits = decode_splits(B, h, n, sms);
    if (splits <= 1) return 0;
    return static_cast<size_t>(B) * h * m * splits * (d + 2) * sizeof(float);
}

namespace {

template <int D>
cudaError_t launch_decode_d(const Problem &p, void *workspace, int sms, cudaStream_t stream)
{
    const int splits = decode_splits(p.B, p.h, p.n, sms);
    constexpr int kRowsPerPass = rows_per_pass<D>();
    int chunk = (p.n + splits - 1) / splits;
    chunk = (chunk + kRowsPerPass - 1) / kRowsPerPass * kRowsPerPass;
    const float scale_log2 = p.scale * 1.4426950408889634f;
    const dim3 grid(p.B * p.h, splits);
    const auto *q = static_cast<const __nv_bfloat16 *>(p.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(p.k);
    const auto *v = static_cast<const __nv_bfloat16 *>(p.v);
    auto *o = static_cast<__nv_bfloat16 *>(p.out);
    float *part = static_cast<float *>(workspace);
    if (p.m <= 1)
        attn_decode_kernel<1, D><<<grid, kWarps * 32, 0, stream>>>(q, k, v, p.key_lengths, o, p.lse, part, p.h, p.m,
                                                                  p.n, chunk, splits, scale_log2);
    else if (p.m <= 2)
        attn_decode_kernel<2, D><<<grid, kWarps * 32, 0, stream>>>(q, k, v, p.key_lengths, o, p.lse, part, p.h, p.m,
                                                                  p.n, chunk, splits, scale_log2);
    else if (p.m <= 4)
        attn_decode_kernel<4, D><<<grid, kWarps * 32, 0, stream>>>(q, k, v, p.key_lengths, o, p.lse, part, p.h, p.m,
                                                                  p.n, chunk, splits, scale_log2);
    else
        attn_decode_kernel<8, D><<<grid, kWarps * 32, 0, stream>>>(q, k, v, p.key_lengths, o, p.lse, part, p.h, p.m,
                                                                  p.n, chunk, splits, scale_log2);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || splits == 1) return e;
    const int rows = p.B * p.h * p.m;
    attn_decode_combine_kernel<D><<<(rows + 7) / 8, 256, 0, stream>>>(part, o, p.lse, rows, splits);
    return cudaGetLastError();
}

} // namespace

bool decode_width_supported(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

cudaError_t launch_decode(const Problem &p, void *workspace, int sms, cudaStream_t stream)
{
    switch (p.d) {
    case 16: return launch_decode_d<16>(p, workspace, sms, stream);
    case 32: return launch_decode_d<32>(p, workspace, sms, stream);
    case 64: return launch_decode_d<64>(p, workspace, sms, stream);
    case 128: return launch_decode_d<128>(p, workspace, sms, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace attn
