// Forward of the masked scaled dot-product attention for heads of width 128
// (bf16) on tcgen05 + TMA + TMEM: out = softmax(scale Q K^T + M) V, the attention
// equation of "Paper Deep Reading: Attention Is All You Need", §04, for the model
// variants whose heads are 128 wide (the variants table of the same page).
//
// One CTA per (batch, head, 128-row query tile), heaviest query tiles first.  Q and
// each 128-key tile of K and V are 128 x 128 bf16, loaded by TMA as two 64-column
// boxes (128-byte swizzle atoms) 16 KiB apart; K and V pass through a two-stage ring.
//   MMA:     S = Q K_j^T                (8 x M128 N128 K16: four K steps in each atom)
//   softmax: 4 warps, thread r = row r = TMEM lane r; masked scores, online softmax
//            (the row max of every key tile), P = exp2(S scale log2 e - max) as bf16
//            pairs in TMEM; O is rescaled in TMEM when a row's max grows
//   MMA:     O += P V_j                 (8 x M128 N128 K16, P from TMEM, V MN-major:
//            its two 64-column atoms are the two halves of N)
// The epilogue divides O by the row sum (0 for a row with no allowed key) and writes
// bf16 rows.  A restricted-attention window limits each CTA to the key tiles that
// meet its rows' windows and masks the rest of each row's range.
// TMEM (512 columns): S [0,128), P [128,192) bf16 pairs, O [256,384).
//
// Every mbarrier wait is bounded: one that runs out sets the CTA's abort flag and
// this file's status word, every role leaves its loop, waits (bounded) for its own
// copies and MMAs, and the CTA frees its TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

__device__ unsigned int g_wide_status_code;
__device__ unsigned int g_wide_status_info;

namespace {

constexpr int kBM = 128;                              // query rows per CTA
constexpr int kBN = 128;                              // keys per key tile
constexpr int kDW = 128;                              // head width
constexpr uint32_t kAtomBytes = 128 * 64 * 2;         // one 64-column atom of a 128-row tile
constexpr uint32_t kTileBytes = (kDW / 64) * kAtomBytes; // 32 KiB
constexpr int kStages = 2;
constexpr int kLoadWarp = 4, kMmaWarp = 5;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull; // 2 s
constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0, 0);  // Q (K-major) x K (K-major)
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kDW, 0, 1); // P (TMEM) x V (MN-major), N = 128

enum WideSite : uint32_t {
    kSiteLoadKvEmpty = 1, kSiteMmaQFull, kSiteMmaKvFull, kSiteMmaSFree, kSiteMmaPFull, kSiteSmSFull,
    kSiteSmPvDone
};

struct alignas(1024) WideSmem {
    uint8_t q[kTileBytes];
    uint8_t k[kStages][kTileBytes];
    uint8_t v[kStages][kTileBytes];
    uint64_t q_full, kv_full[kStages], kv_empty[kStages];
    uint64_t s_full, s_free, p_full, pv_done, drain;
    uint32_t tmem_base;
    int abort_flag;
};

struct WideParams {
    const int32_t *key_lengths; // nullptr unless key padding
    __nv_bfloat16 *out;
    float *lse;
    int BH, h, m, n, mask_kind, q_tiles;
    int window; // restricted attention: keys with |i - j| <= window stay; -1: none
    float scale_log2;
};

__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, int *abort_flag, uint32_t site)
{
    const uint64_t start = global_timer_ns();
    while (true) {
        for (int k = 0; k < 64; ++k)
            if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int *>(abort_flag)) return false;
        if (global_timer_ns() - start > kWaitLimitNs) {
            *reinterpret_cast<volatile int *>(abort_flag) = 1;
            atomicOr(&g_wide_status_code, 1u);
            atomicCAS(&g_wide_status_info, 0u, site);
            return false;
        }
    }
}

// Bounded wait for phase `parity` of `bar`.  false: gave up (or another role did).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, int *abort_flag, uint32_t site)
{
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    return wait_slow(a, parity, abort_flag, site);
}

// Wait, bounded and ignoring the abort flag, for work already in flight to complete.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint32_t a = smem_addr(bar);
    const uint64_t start = global_timer_ns();
    while (!mbar_try_wait(a, parity))
        if (global_timer_ns() - start > kWaitLimitNs) return;
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

__global__ void __launch_bounds__(kThreads, 1)
attn_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const WideParams p)
{
    extern __shared__ uint8_t smem_raw[];
    WideSmem &sm = *reinterpret_cast<WideSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                 ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // heaviest query tiles first: with a causal mask later query tiles see more keys
    const int qt = p.q_tiles - 1 - static_cast<int>(blockIdx.x) / p.BH;
    const int bh = static_cast<int>(blockIdx.x) % p.BH;
    const int q0 = qt * kBM;
    const bool causal = (p.mask_kind & kMaskCausal) != 0;
    int len = p.n;
    if (p.key_lengths != nullptr) {
        len = __ldg(p.key_lengths + bh / p.h);
        len = len < 0 ? 0 : (len > p.n ? p.n : len);
    }
    int kv_end = causal ? min(len, q0 + kBM) : len;
    int kv_lo = 0; // first key tile
    if (p.window >= 0) {
        // keys within `window` of some row q0 .. min(m, q0 + 128) - 1 of the tile
        kv_lo = max(0, q0 - p.window) / kBN;
        kv_end = min(kv_end, min(p.m, q0 + kBM) + p.window);
    }
    // key tiles [kv_lo, kv_lo + n_kv); fill f of the ring holds key tile kv_lo + f
    const int n_kv = kv_end > kv_lo * kBN ? (kv_end + kBN - 1) / kBN - kv_lo : 0;

    if (n_kv == 0) {
        // no allowed key for any row of this tile: output 0
        if (warp < 4) {
            const int i = q0 + warp * 32 + lane;
            if (i < p.m) {
                uint4 *orow = reinterpret_cast<uint4 *>(p.out + (static_cast<size_t>(bh) * p.m + i) * kDW);
                const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < kDW / 8; ++c) orow[c] = z;
                if (p.lse != nullptr) p.lse[static_cast<size_t>(bh) * p.m + i] = -CUDART_INF_F;
            }
        }
        return;
    }

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.kv_full[s], 1);
            mbar_init(&sm.kv_empty[s], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_free, kBM);
        mbar_init(&sm.p_full, kBM);
        mbar_init(&sm.pv_done, 1);
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncwarp();
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    int *ab = &sm.abort_flag;

    if (warp == kLoadWarp) {
        if (lane == 0) {
            tma_prefetch_map(&tm_q);
            tma_prefetch_map(&tm_k);
            tma_prefetch_map(&tm_v);
            mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
            tma_load_3d(sm.q, &tm_q, &sm.q_full, 0, q0, bh);
            tma_load_3d(sm.q + kAtomBytes, &tm_q, &sm.q_full, 64, q0, bh);
            int issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int st = j % kStages;
                if (!wait_bar(&sm.kv_empty[st], ((j / kStages) & 1) ^ 1, ab, kSiteLoadKvEmpty)) break;
                mbar_arrive_expect_tx(&sm.kv_full[st], 2 * kTileBytes);
                const int key0 = (kv_lo + j) * kBN;
                tma_load_3d(sm.k[st], &tm_k, &sm.kv_full[st], 0, key0, bh);
                tma_load_3d(sm.k[st] + kAtomBytes, &tm_k, &sm.kv_full[st], 64, key0, bh);
                tma_load_3d(sm.v[st], &tm_v, &sm.kv_full[st], 0, key0, bh);
                tma_load_3d(sm.v[st] + kAtomBytes, &tm_v, &sm.kv_full[st], 64, key0, bh);
                ++issued;
            }
            // copies still in flight must land before the CTA may exit
            drain_wait(&sm.q_full, 0);
            for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
                drain_wait(&sm.kv_full[j % kStages], (j / kStages) & 1);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(0, 0, 1024) >> 32);
            const uint32_t q_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.q), 16, 1024));
            const uint32_t k_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.k[0]), 16, 1024));
            // V as an MN-major B of N = 128: its two 64-column atoms kAtomBytes apart
            const uint32_t v_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.v[0]), kAtomBytes, 1024));
            constexpr uint32_t kStageUnits = kTileBytes >> 4;
            const uint32_t ts = tmem + kColS, tp = tmem + kColP, to = tmem + kColO;
            bool ok = wait_bar(&sm.q_full, 0, ab, kSiteMmaQFull);
            for (int j = 0; j <= n_kv && ok; ++j) {
                if (j < n_kv) {
                    // S(j) once K_j is in and the softmax has read S(j - 1)
                    const int st = j % kStages;
                    ok = wait_bar(&sm.kv_full[st], (j / kStages) & 1, ab, kSiteMmaKvFull);
                    if (ok && j > 0) ok = wait_bar(&sm.s_free, (j - 1) & 1, ab, kSiteMmaSFree);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kd = k_lo + st * kStageUnits;
                    // 16 columns (32 bytes, 2 units) per K step; the second atom 16 KiB
                    // (1024 units) on
                    mma_ss_k<0, 0>(ts, q_lo, kd, desc_hi, kIdescS, 0u);
                    mma_ss_k<2, 2>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<4, 4>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<6, 6>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<1024, 1024>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<1026, 1026>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<1028, 1028>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<1030, 1030>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_commit(&sm.s_full);
                }
                if (j >= 1) {
                    // O += P(j - 1) V(j - 1): keys 16kk.. are P columns 8kk.. (bf16 pairs)
                    // and V rows 16kk.. (2 KiB = 128 units per K step)
                    const int jp = j - 1, st = jp % kStages;
                    ok = wait_bar(&sm.p_full, jp & 1, ab, kSiteMmaPFull);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t vd = v_lo + st * kStageUnits;
                    const uint32_t acc0 = jp > 0 ? 1u : 0u;
                    mma_ts_k<0, 0>(to, tp, vd, desc_hi, kIdescPV, acc0);
                    mma_ts_k<8, 128>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<16, 256>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<24, 384>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<32, 512>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<40, 640>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<48, 768>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<56, 896>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_commit(&sm.pv_done);
                    mma_commit(&sm.kv_empty[st]);
                }
            }
            if (!ok) {
                // make sure no MMA is still writing TMEM when the CTA frees it
                mma_commit(&sm.drain);
                drain_wait(&sm.drain, 0);
            }
        }
        __syncwarp();
    } else {
        // softmax and epilogue: thread r = row r of the tile = TMEM lane r
        const int row = warp * 32 + lane;
        const int i = q0 + row;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t t_s = tmem + lane_base + kColS, t_p = tmem + lane_base + kColP;
        const uint32_t t_o = tmem + lane_base + kColO;
        const float sl2 = p.scale_log2;
        // keys allowed for row i: [lo, hi) (below the padded length, i + 1 causal, and
        // within `window` of i)
        int hi = causal ? min(len, i + 1) : len;
        int lo = 0;
        if (p.window >= 0) {
            hi = min(hi, i + p.window + 1);
            lo = i - p.window;
        }
        float m_run = -CUDART_INF_F, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv && ok; ++j) {
            ok = warp_all(wait_bar(&sm.s_full, j & 1, ab, kSiteSmSFull));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) tmem_ld32(t_s + 32 * c, sr + 32 * c);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) reg_fence32(sr + 32 * c);
            tc_fence_before();
            mbar_arrive(&sm.s_free);
            // scale first, then mask: a zero scale must not turn -inf into NaN
            const int key0 = (kv_lo + j) * kBN;
            const int cnt = hi - key0, cnt_lo = lo - key0;
            float x[kBN];
            float mt = -CUDART_INF_F;
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                x[c] = (c < cnt && c >= cnt_lo) ? __uint_as_float(sr[c]) * sl2 : -CUDART_INF_F;
                mt = fmaxf(mt, x[c]);
            }
            const float m_new = fmaxf(m_run, mt);
            // O and l hold nothing before the row's first allowed key: no rescale then
            const bool rescale = m_run != -CUDART_INF_F && m_new > m_run;
            const float alpha = rescale ? ex2(m_run - m_new) : 1.f;
            const float m_sub = m_new == -CUDART_INF_F ? 0.f : m_new;
            uint32_t pk[kBN / 2];
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int c2 = 0; c2 < kBN / 2; ++c2) {
                const float e0 = ex2(x[2 * c2] - m_sub), e1 = ex2(x[2 * c2 + 1] - m_sub);
                s0 += e0;
                s1 += e1;
                pk[c2] = pack_bf16x2(e0, e1);
            }
            if (j > 0) {
                // P and O are in use by the previous P V until it completes
                ok = warp_all(wait_bar(&sm.pv_done, (j - 1) & 1, ab, kSiteSmPvDone));
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                    for (int c = 0; c < kDW / 32; ++c) {
                        uint32_t orr[32];
                        tmem_ld32(t_o + 32 * c, orr);
                        tmem_wait_ld();
                        reg_fence32(orr);
#pragma unroll
                        for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                        tmem_st32(t_o + 32 * c, orr);
                    }
                }
            }
            tmem_st32(t_p, pk);
            tmem_st32(t_p + 32, pk + 32);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&sm.p_full);
            l_run = l_run * alpha + (s0 + s1);
            m_run = m_new;
        }
        if (ok) ok = warp_all(wait_bar(&sm.pv_done, (n_kv - 1) & 1, ab, kSiteSmPvDone));
        if (ok) {
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            if (p.lse != nullptr && i < p.m) // weights are exp2(x - m_run) / l: lse = (m_run + log2 l) ln 2
                p.lse[static_cast<size_t>(bh) * p.m + i] =
                    l_run > 0.f ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -CUDART_INF_F;
            uint4 *orow = reinterpret_cast<uint4 *>(p.out + (static_cast<size_t>(bh) * p.m + (i < p.m ? i : 0)) * kDW);
#pragma unroll 1
            for (int c = 0; c < kDW / 32; ++c) {
                uint32_t orr[32];
                tmem_ld32(t_o + 32 * c, orr);
                tmem_wait_ld();
                reg_fence32(orr);
                if (i < p.m) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(orr[8 * q + 0]) * inv, __uint_as_float(orr[8 * q + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(orr[8 * q + 2]) * inv, __uint_as_float(orr[8 * q + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(orr[8 * q + 4]) * inv, __uint_as_float(orr[8 * q + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(orr[8 * q + 6]) * inv, __uint_as_float(orr[8 * q + 7]) * inv);
                        orow[4 * c + q] = w;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

constexpr size_t kSmemBytes = sizeof(WideSmem) + 1024; // + alignment slack

} // namespace

cudaError_t launch_wide(const Problem &pb, cudaStream_t stream)
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
            if ((e = cudaFuncSetAttribute(attn_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(kSmemBytes))) != cudaSuccess)
                return e;
            configured[dev] = true;
        }
    }
    if (!pb.bf16 || pb.d != kDW) return cudaErrorInvalidValue;
    const int BH = pb.B * pb.h;
    CUtensorMap tq, tk, tv;
    if (!encode_bf16_3d(&tq, pb.q, kDW, pb.m, BH, kBM) || !encode_bf16_3d(&tk, pb.k, kDW, pb.n, BH, kBN) ||
        !encode_bf16_3d(&tv, pb.v, kDW, pb.n, BH, kBN))
        return cudaErrorInvalidValue;
    WideParams p;
    p.key_lengths = (pb.mask_kind & kMaskKeyPadding) ? pb.key_lengths : nullptr;
    p.out = static_cast<__nv_bfloat16 *>(pb.out);
    p.lse = pb.lse;
    p.BH = BH;
    p.h = pb.h;
    p.m = pb.m;
    p.n = pb.n;
    p.mask_kind = pb.mask_kind;
    p.q_tiles = (pb.m + kBM - 1) / kBM;
    p.window = (pb.mask_kind & kMaskWindow) ? pb.window : -1;
    p.scale_log2 = pb.scale * 1.4426950408889634f;
    const long long grid = static_cast<long long>(BH) * p.q_tiles;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    attn_wide_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

cudaError_t wide_status_read_and_clear(cudaStream_t stream, uint32_t *code, uint32_t *info)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned int c = 0, i = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&c, g_wide_status_code, sizeof c)) != cudaSuccess) return e;
    if ((e = cudaMemcpyFromSymbol(&i, g_wide_status_info, sizeof i)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_wide_status_code, &zero, sizeof zero)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_wide_status_info, &zero, sizeof zero)) != cudaSuccess) return e;
    *code = c;
    *info = i;
    return cudaSuccess;
}

} // namespace attn
