// Projections of multi-head attention on tcgen05: the W^Q, W^K, W^V products
// that split the model width into heads, and the W^O product over the
// concatenated heads ("Paper Deep Reading: Attention Is All You Need", §04
// MultiHead equation: head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V),
// MultiHead = Concat(head_1, ..., head_h) W^O; no bias terms).
//
// One CTA computes a 128 x 128 tile of D = A B with fp32 accumulation in TMEM:
//   kProjIn   A = rows t0 .. t0+127 of x[b] ([B][L][K], K = d_model), B = columns
//             n0 .. n0+127 of W ([K][h*64]); the tile is heads n0/64 and n0/64 + 1,
//             stored straight into the head-split layout [B*h][L][64] (the
//             per-head W_i are column blocks of W).
//   kProjOut  A = the heads' outputs [B*h][L][64]: the 64-wide K step j reads head
//             j, so Concat needs no copy; B = columns n0 .. n0+127 of W^O
//             ([h*64][N]); the tile goes to out[b] ([B][L][N]).
// A tiles are K-major (64 bf16 = one 128-byte swizzle row per tile row), B tiles
// 64 x 64 MN-major, loaded by TMA through a 4-stage ring; each 64-wide K step is
// 4 x 2 MMAs of M128 N64 K16 into two 64-column accumulators.  The epilogue
// converts to bf16 through a swizzled shared-memory tile and TMA stores (rows
// past L are clipped).
//
// Warps: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2-5 epilogue.  Every
// mbarrier wait is bounded and reports through this file's status word.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

__device__ unsigned int g_proj_status_code;
__device__ unsigned int g_proj_status_info;

namespace {

constexpr int kTM = 128, kTN = 128, kTK = 64; // output tile and K step
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kATile = kTM * kTK * 2;    // 16 KiB
constexpr uint32_t kBHalf = kTK * 64 * 2;     // 8 KiB: 64 K rows x 64 N columns
constexpr uint32_t kTmemCols = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kIdesc = idesc_bf16_f32(kTM, 64, 0, 1); // A K-major, B MN-major, N = 64

struct alignas(1024) ProjSmem {
    uint8_t a[kStages][kATile];
    uint8_t b[kStages][2][kBHalf];
    uint8_t stage[2][kTM * 64 * 2]; // bf16 output halves, 128-byte swizzle
    uint64_t full[kStages], empty[kStages], acc_full, staged[2];
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, int *abort_flag, uint32_t site)
{
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t start = global_timer_ns();
    while (true) {
        for (int k = 0; k < 64; ++k)
            if (mbar_try_wait(a, parity)) return true;
        if (*reinterpret_cast<volatile int *>(abort_flag)) return false;
        if (global_timer_ns() - start > kWaitLimitNs) {
            *reinterpret_cast<volatile int *>(abort_flag) = 1;
            atomicOr(&g_proj_status_code, 1u);
            atomicCAS(&g_proj_status_info, 0u, site);
            return false;
        }
    }
}

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint32_t a = smem_addr(bar);
    const uint64_t start = global_timer_ns();
    while (!mbar_try_wait(a, parity))
        if (global_timer_ns() - start > kWaitLimitNs) return;
}

struct ProjParams {
    int mode, h, K;
};

__global__ void __launch_bounds__(kThreads, 1)
attn_proj_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w,
                 const __grid_constant__ CUtensorMap tm_out, const ProjParams p)
{
    extern __shared__ uint8_t smem_raw[];
    ProjSmem &sm = *reinterpret_cast<ProjSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                 ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32;
    const int n0 = blockIdx.x * kTN, t0 = blockIdx.y * kTM, b = blockIdx.z;
    const int ksteps = p.K / kTK;
    int *ab = &sm.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.acc_full, 1);
        mbar_init(&sm.staged[0], kTM);
        mbar_init(&sm.staged[1], kTM);
        sm.abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncwarp();
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        if (threadIdx.x == 0) {
            tma_prefetch_map(&tm_a);
            tma_prefetch_map(&tm_w);
            int issued = 0;
            for (int kk = 0; kk < ksteps; ++kk) {
                const int s = kk % kStages;
                if (!wait_bar(&sm.empty[s], ((kk / kStages) & 1) ^ 1, ab, 1)) break;
                mbar_arrive_expect_tx(&sm.full[s], kATile + 2 * kBHalf);
                if (p.mode == kProjIn)
                    tma_load_3d(sm.a[s], &tm_a, &sm.full[s], kk * kTK, t0, b);
                else
                    tma_load_3d(sm.a[s], &tm_a, &sm.full[s], 0, t0, b * p.h + kk);
                // W as a 2-D tensor (the third coordinate is 0)
                tma_load_3d(sm.b[s][0], &tm_w, &sm.full[s], n0, kk * kTK, 0);
                tma_load_3d(sm.b[s][1], &tm_w, &sm.full[s], n0 + 64, kk * kTK, 0);
                ++issued;
            }
            for (int kk = issued > kStages ? issued - kStages : 0; kk < issued; ++kk)
                drain_wait(&sm.full[kk % kStages], (kk / kStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (threadIdx.x == 32) {
            const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(0, 0, 1024) >> 32);
            const uint32_t a_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.a[0]), 16, 1024));
            const uint32_t b_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.b[0][0]), kBHalf, 1024));
            bool ok = true;
            for (int kk = 0; kk < ksteps && ok; ++kk) {
                const int s = kk % kStages;
                if (!(ok = wait_bar(&sm.full[s], (kk / kStages) & 1, ab, 2))) break;
                tc_fence_after();
                const uint32_t ad = a_lo + s * (kATile >> 4);
                const uint32_t acc = kk > 0 ? 1u : 0u;
#pragma unroll
                for (int nh = 0; nh < 2; ++nh) {
                    // A: 16 bf16 of K per step = 32 bytes; B: K rows 16kk.. = 2 KiB per step
                    const uint32_t bd = b_lo + (s * 2 + nh) * (kBHalf >> 4);
                    const uint32_t d = tmem + 64 * nh;
                    mma_ss_k<0, 0>(d, ad, bd, desc_hi, kIdesc, acc);
                    mma_ss_k<2, 128>(d, ad, bd, desc_hi, kIdesc, 1u);
                    mma_ss_k<4, 256>(d, ad, bd, desc_hi, kIdesc, 1u);
                    mma_ss_k<6, 384>(d, ad, bd, desc_hi, kIdesc, 1u);
                }
                mma_commit(&sm.empty[s]);
            }
            // the epilogue waits on this (also after an abort: every MMA issued is complete)
            mma_commit(&sm.acc_full);
        }
        __syncwarp();
    } else {
        // epilogue: thread t = output row t of the tile (TMEM lane t)
        const int t = (warp % 4) * 32 + threadIdx.x % 32;
        const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
        const bool ok = __all_sync(0xffffffffu, wait_bar(&sm.acc_full, 0, ab, 3));
        if (ok && !*reinterpret_cast<volatile int *>(ab)) {
            tc_fence_after();
#pragma unroll 1
            for (int nh = 0; nh < 2; ++nh) {
                uint32_t r[64];
                tmem_ld32(tmem + lane_base + 64 * nh, r);
                tmem_ld32(tmem + lane_base + 64 * nh + 32, r + 32);
                tmem_wait_ld();
                reg_fence32(r);
                reg_fence32(r + 32);
                const uint32_t row = smem_addr(sm.stage[nh]) + t * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 v;
                    v.x = pack_bf16x2(__uint_as_float(r[8 * c + 0]), __uint_as_float(r[8 * c + 1]));
                    v.y = pack_bf16x2(__uint_as_float(r[8 * c + 2]), __uint_as_float(r[8 * c + 3]));
                    v.z = pack_bf16x2(__uint_as_float(r[8 * c + 4]), __uint_as_float(r[8 * c + 5]));
                    v.w = pack_bf16x2(__uint_as_float(r[8 * c + 6]), __uint_as_float(r[8 * c + 7]));
                    st_shared_v4(row + ((c ^ (t & 7)) << 4), v);
                }
                fence_proxy_async_shared();
                mbar_arrive(&sm.staged[nh]);
            }
            if (t == 0) {
#pragma unroll 1
                for (int nh = 0; nh < 2; ++nh) {
                    if (!wait_bar(&sm.staged[nh], 0, ab, 4)) break;
                    if (p.mode == kProjIn)
                        tma_store_3d(&tm_out, sm.stage[nh], 0, t0, b * p.h + n0 / 64 + nh);
                    else
                        tma_store_3d(&tm_out, sm.stage[nh], n0 + 64 * nh, t0, b);
                }
                bulk_commit_group();
                bulk_wait_all();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

constexpr size_t kSmemBytes = sizeof(ProjSmem) + 1024;

} // namespace

cudaError_t launch_proj(const ProjProblem &pp, cudaStream_t stream)
{
    static bool configured[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!configured[dev]) {
            if ((e = cudaFuncSetAttribute(attn_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(kSmemBytes))) != cudaSuccess)
                return e;
            configured[dev] = true;
        }
    }
    if (pp.K % kTK != 0 || pp.N % kTN != 0) return cudaErrorInvalidValue;
    CUtensorMap ta, tw, to;
    const int BH = pp.B * pp.h;
    bool enc;
    if (pp.mode == kProjIn) {
        enc = encode_bf16_3d(&ta, pp.a, pp.K, pp.L, pp.B, kTM) && encode_bf16_3d(&to, pp.out, 64, pp.L, BH, kTM);
    } else {
        enc = encode_bf16_3d(&ta, pp.a, 64, pp.L, BH, kTM) && encode_bf16_3d(&to, pp.out, pp.N, pp.L, pp.B, kTM);
    }
    // W [K][N] as a 3-D tensor with one outer slice: 64 x 64 boxes
    enc = enc && encode_bf16_3d(&tw, pp.w, pp.N, pp.K, 1, kTK);
    if (!enc) return cudaErrorInvalidValue;
    ProjParams p;
    p.mode = pp.mode;
    p.h = pp.h;
    p.K = pp.K;
    const dim3 grid(pp.N / kTN, (pp.L + kTM - 1) / kTM, pp.B);
    attn_proj_kernel<<<grid, kThreads, kSmemBytes, stream>>>(ta, tw, to, p);
    return cudaGetLastError();
}

cudaError_t proj_status_read_and_clear(cudaStream_t stream, uint32_t *code, uint32_t *info)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned int c = 0, i = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&c, g_proj_status_code, sizeof c)) != cudaSuccess) return e;
    if ((e = cudaMemcpyFromSymbol(&i, g_proj_status_info, sizeof i)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_proj_status_code, &zero, sizeof zero)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_proj_status_info, &zero, sizeof zero)) != cudaSuccess) return e;
    *code = c;
    *info = i;
    return cudaSuccess;
}

} // namespace attn
