// Backward of the fused masked scaled dot-product attention for sm_103a:
// TMA + tcgen05 + TMEM.
//
// For each (batch, head), with S = scale * Q K^T + M, P = softmax(S) row-wise,
// O = P V and an upstream gradient dO (the chain rule of the attention equation,
// "Paper Deep Reading: Attention Is All You Need", §04 attention equation; the
// model is trained, slide deck "Training Details"):
//
//   dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic (= sum_j P_ij dP_ij),
//   dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// P is recomputed from Q, K and the forward's per-row log-sum-exp, never stored.
//
// Three launches:
//   attn_bwd_pre_kernel   D_i and (lse_i * log2 e, D_i) per query row, padded to
//                         whole 128-row tiles (padding rows: (+inf, 0) so their
//                         weights are 0); zeroes the fp32 dQ accumulator.
//   attn_bwd_kernel       one CTA per (key tile j of 128 keys, head): K_j, V_j stay
//                         in shared memory; dV_j and dK_j accumulate in TMEM over
//                         the query tiles i that can see key tile j (i >= j with a
//                         causal mask); each step adds its dQ_i part to the fp32
//                         accumulator with TMA reductions from shared memory.
//   attn_bwd_post_kernel  dQ = bf16(scale * accumulator).
//
// Per step (query tile i) of attn_bwd_kernel, keys as the MMA rows (four groups of
// four compute warps; thread t of each group owns key row t = TMEM lane t, group g
// takes the step's queries 32g .. 32g+31):
//   MMA:      S^T = K_j Q_i^T, dP^T = V_j dO_i^T     (4 + 4 x M128 N128 K16, K-major)
//   compute:  P^T = exp2(S^T scale log2 e - L_i), dS^T = P^T o (dP^T - D_i), masked;
//             P^T goes to TMEM as bf16 pairs, dS^T to shared memory as a K-major
//             [key][query] tile (two buffers, alternating by step)
//   MMA:      dV_j += P^T dO_i (A from TMEM), dK_j += dS^T Q_i (A K-major),
//             dQ_i  = dS K_j (dS^T read as an MN-major A); B operands MN-major
//   compute:  read dQ_i from TMEM (lane = query row), stage it in shared memory
//             and add it to the accumulator with one TMA reduction per group
// The steps overlap: S^T and dP^T are released as soon as every compute thread has
// read them, so step i+1's scores are computed while step i's weights are; step
// i's dQ is read out after step i+1's weights are written.
// The epilogue writes dV_j and scale * dK_j as bf16.
//
// TMEM (512 columns): S^T [0,128), dP^T [128,256), dV [256,320), dK [320,384),
// dQ [384,448), P^T [448,512).
//
// Every mbarrier wait is bounded; a wait that runs out sets the CTA's abort flag
// and this file's device status word, and every role leaves its loop.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

__device__ unsigned int g_bwd_status_code;
__device__ unsigned int g_bwd_status_info;

namespace {

constexpr int kBM = 128; // keys per CTA (TMEM lanes) and queries per step
constexpr int kD = 64;
constexpr int kStages = 2;
constexpr int kGroups = 4;                       // compute groups of four warps, 32 queries each per step
constexpr int kComputeThreads = kGroups * 128;
constexpr int kThreads = kComputeThreads + 64;   // + warp 16 TMA producer, warp 17 MMA issuer
constexpr int kLoadWarp = kGroups * 4;
constexpr int kMmaWarp = kLoadWarp + 1;
constexpr uint32_t kTileBytes = kBM * kD * 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 320, kColDQ = 384, kColPT = 448;
constexpr uint64_t kWaitLimitNs = 2000000000ull; // 2 s: far beyond any legitimate wait
constexpr uint32_t kIdescNN = idesc_bf16_f32(kBM, kBM, 0, 0); // both operands K-major, N = 128
constexpr uint32_t kIdescN64 = idesc_bf16_f32(kBM, kD, 0, 1); // B MN-major, N = 64
constexpr uint32_t kIdescDQ = idesc_bf16_f32(kBM, kD, 1, 1);  // A and B MN-major, N = 64

enum BwdSite : uint32_t {
    kSiteLoadQEmpty = 1, kSiteMmaKvFull, kSiteMmaQFull, kSiteMmaDqFull, kSiteMmaPReady, kSiteMmaDqFree,
    kSiteCmpQFull, kSiteCmpSdpFull, kSiteCmpDqFull, kSiteCmpSLoaded, kSiteCmpDqsFree, kSiteCmpDqsFull,
    kSiteMmaSLoaded
};

struct alignas(1024) BwdSmem {
    uint8_t k[kTileBytes];
    uint8_t v[kTileBytes];
    uint8_t q[kStages][kTileBytes];
    uint8_t dout[kStages][kTileBytes];
    // dS^T [key][query] bf16 of steps with even / odd index, 128-byte swizzle, two
    // blocks each: queries 0-63, queries 64-127
    uint8_t dst[2][2][kTileBytes];
    uint8_t dq_stage[2][kBM * 32 * 4]; // dQ columns 0-31 / 32-63: 128 rows x 32 fp32, 128-byte swizzle
    float2 ld[kStages][kBM];    // (lse * log2 e, D) of the step's query rows
    uint64_t kv_full, q_full[kStages], q_empty[kStages];
    uint64_t sdp_full, p_ready, dq_full, dq_free;
    uint64_t s_loaded; // every compute thread has read its S^T and dP^T columns out of TMEM
    uint64_t dqs_free[2], dqs_full[2]; // dq_stage[g] may be written / may be reduced into the accumulator
    uint64_t drain; // abort path only: completion of every MMA this CTA issued
    uint32_t tmem_base;
    int abort_flag;
};

struct BwdParams {
    const float2 *ld;        // [BH][m_pad] (lse * log2 e, D); padding rows (+inf, 0)
    float *dq_acc;           // [BH][m][64] fp32, zeroed by the pre kernel
    __nv_bfloat16 *dk, *dv;  // [BH][n][d]
    const int32_t *key_lengths;
    int BH, h, m, n, m_pad, mask_kind, q_tiles;
    int d;                   // head width in memory (a multiple of 8, <= 64); the tiles are 64 wide
    int group_heads;         // heads per group of the CTA order (their Q and dO share L2)
    int k_tiles;             // key tiles per head
    float scale_log2;        // scale * log2 e
    float scale;
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
            atomicOr(&g_bwd_status_code, 1u);
            atomicCAS(&g_bwd_status_info, 0u, site);
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

// Wait, bounded and ignoring the abort flag, for copies already in flight to land.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint32_t a = smem_addr(bar);
    const uint64_t start = global_timer_ns();
    while (!mbar_try_wait(a, parity))
        if (global_timer_ns() - start > kWaitLimitNs) return;
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// Keys of batch b allowed by padding (n without it).
__device__ __forceinline__ int key_len(const BwdParams &p, int bh)
{
    int len = p.n;
    if ((p.mask_kind & kMaskKeyPadding) && p.key_lengths != nullptr) {
        len = __ldg(p.key_lengths + bh / p.h);
        len = len < 0 ? 0 : (len > p.n ? p.n : len);
    }
    return len;
}

// ------------------------------------------------------------------ roles
__device__ __forceinline__ void load_role(BwdSmem &sm, const BwdParams &p, const CUtensorMap *tm_q,
                                          const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                                          const CUtensorMap *tm_do, int bh, int key0, int i_begin, int steps)
{
    int *ab = &sm.abort_flag;
    tma_prefetch_map(tm_q);
    tma_prefetch_map(tm_do);
    mbar_arrive_expect_tx(&sm.kv_full, 2 * kTileBytes);
    tma_load_3d(sm.k, tm_k, &sm.kv_full, 0, key0, bh);
    tma_load_3d(sm.v, tm_v, &sm.kv_full, 0, key0, bh);
    int issued = 0;
    for (int t = 0; t < steps; ++t) {
        const int s = t % kStages;
        if (!wait_bar(&sm.q_empty[s], ((t / kStages) & 1) ^ 1, ab, kSiteLoadQEmpty)) break;
        const int i0 = (i_begin + t) * kBM;
        mbar_arrive_expect_tx(&sm.q_full[s], 2 * kTileBytes + kBM * sizeof(float2));
        tma_load_3d(sm.q[s], tm_q, &sm.q_full[s], 0, i0, bh);
        tma_load_3d(sm.dout[s], tm_do, &sm.q_full[s], 0, i0, bh);
        bulk_load(sm.ld[s], p.ld + static_cast<size_t>(bh) * p.m_pad + i0, kBM * sizeof(float2), &sm.q_full[s]);
        ++issued;
    }
    // copies still in flight must land before the CTA may exit
    drain_wait(&sm.kv_full, 0);
    for (int t = issued > kStages ? issued - kStages : 0; t < issued; ++t)
        drain_wait(&sm.q_full[t % kStages], (t / kStages) & 1);
}

__device__ __forceinline__ void mma_role(BwdSmem &sm, uint32_t tmem, int steps)
{
    int *ab = &sm.abort_flag;
    const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(0, 0, 1024) >> 32);
    // K-major operands (rows x 64 bf16 = one 128-byte swizzle atom wide)
    const uint32_t k_km = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.k), 16, 1024));
    const uint32_t v_km = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.v), 16, 1024));
    const uint32_t q_km = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.q[0]), 16, 1024));
    const uint32_t do_km = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.dout[0]), 16, 1024));
    const uint32_t dst_km = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.dst[0][0]), 16, 1024));
    // the same tiles as MN-major operands (rows are the reduction dimension); dS^T
    // read as dS: its two 64-query blocks are the two M atoms, one tile apart
    const uint32_t k_mn = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.k), kTileBytes, 1024));
    const uint32_t q_mn = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.q[0]), kTileBytes, 1024));
    const uint32_t do_mn = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.dout[0]), kTileBytes, 1024));
    const uint32_t dst_mn = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.dst[0][0]), kTileBytes, 1024));
    constexpr uint32_t kStageUnits = kTileBytes >> 4; // descriptor units per stage
    const uint32_t ts = tmem + kColS, tdp = tmem + kColDP;
    const uint32_t tdv = tmem + kColDV, tdk = tmem + kColDK, tdq = tmem + kColDQ, tpt = tmem + kColPT;

    // S^T = K Q^T and dP^T = V dO^T of the step in stage s: 16 of the 64 columns
    // (32 bytes) per K step
    auto scores = [&](uint32_t su) {
        mma_ss_k<0, 0>(ts, k_km, q_km + su, desc_hi, kIdescNN, 0u);
        mma_ss_k<2, 2>(ts, k_km, q_km + su, desc_hi, kIdescNN, 1u);
        mma_ss_k<4, 4>(ts, k_km, q_km + su, desc_hi, kIdescNN, 1u);
        mma_ss_k<6, 6>(ts, k_km, q_km + su, desc_hi, kIdescNN, 1u);
        mma_ss_k<0, 0>(tdp, v_km, do_km + su, desc_hi, kIdescNN, 0u);
        mma_ss_k<2, 2>(tdp, v_km, do_km + su, desc_hi, kIdescNN, 1u);
        mma_ss_k<4, 4>(tdp, v_km, do_km + su, desc_hi, kIdescNN, 1u);
        mma_ss_k<6, 6>(tdp, v_km, do_km + su, desc_hi, kIdescNN, 1u);
        mma_commit(&sm.sdp_full);
    };

    bool ok = wait_bar(&sm.kv_full, 0, ab, kSiteMmaKvFull);
    if (ok) ok = wait_bar(&sm.q_full[0], 0, ab, kSiteMmaQFull);
    if (ok) {
        tc_fence_after();
        scores(0);
    }
    for (int t = 0; t < steps && ok; ++t) {
        const int s = t % kStages;
        const uint32_t su = static_cast<uint32_t>(s) * kStageUnits;
        if (t + 1 < steps) {
            // the next step's scores as soon as every compute thread has read this
            // step's out of TMEM: they run while this step's weights are computed
            const int s1 = (t + 1) % kStages;
            ok = wait_bar(&sm.s_loaded, t & 1, ab, kSiteMmaSLoaded);
            if (ok) ok = wait_bar(&sm.q_full[s1], ((t + 1) / kStages) & 1, ab, kSiteMmaQFull);
            if (!ok) break;
            tc_fence_after();
            scores(static_cast<uint32_t>(s1) * kStageUnits);
        }
        if (!(ok = wait_bar(&sm.p_ready, t & 1, ab, kSiteMmaPReady))) break;
        tc_fence_after();
        // dV += P^T dO (P^T in TMEM: queries 16kk.. are columns 8kk.., bf16 pairs),
        // dK += dS^T Q (dS^T K-major in shared memory: queries 0-63 in the first
        // block, 32 bytes per K step, 64-127 in the second, 16 KiB on); B operands
        // MN-major, rows 16kk.. at 2 KiB = 128 descriptor units per K step
        const uint32_t acc = t > 0 ? 1u : 0u;
        const uint32_t dob = do_mn + su, qb = q_mn + su;
        const uint32_t du = static_cast<uint32_t>(t & 1) * (2 * kStageUnits); // dS^T buffer
        const uint32_t dsk = dst_km + du, dsm = dst_mn + du;
        mma_ts_k<0, 0>(tdv, tpt, dob, desc_hi, kIdescN64, acc);
        mma_ts_k<8, 128>(tdv, tpt, dob, desc_hi, kIdescN64, 1u);
        mma_ts_k<16, 256>(tdv, tpt, dob, desc_hi, kIdescN64, 1u);
        mma_ts_k<24, 384>(tdv, tpt, dob, desc_hi, kIdescN64, 1u);
        mma_ts_k<32, 512>(tdv, tpt, dob, desc_hi, kIdescN64, 1u);
        mma_ts_k<40, 640>(tdv, tpt, dob, desc_hi, kIdescN64, 1u);
        mma_ts_k<48, 768>(tdv, tpt, dob, desc_hi, kIdescN64, 1u);
        mma_ts_k<56, 896>(tdv, tpt, dob, desc_hi, kIdescN64, 1u);
        mma_ss_k<0, 0>(tdk, dsk, qb, desc_hi, kIdescN64, acc);
        mma_ss_k<2, 128>(tdk, dsk, qb, desc_hi, kIdescN64, 1u);
        mma_ss_k<4, 256>(tdk, dsk, qb, desc_hi, kIdescN64, 1u);
        mma_ss_k<6, 384>(tdk, dsk, qb, desc_hi, kIdescN64, 1u);
        mma_ss_k<1024, 512>(tdk, dsk, qb, desc_hi, kIdescN64, 1u);
        mma_ss_k<1026, 640>(tdk, dsk, qb, desc_hi, kIdescN64, 1u);
        mma_ss_k<1028, 768>(tdk, dsk, qb, desc_hi, kIdescN64, 1u);
        mma_ss_k<1030, 896>(tdk, dsk, qb, desc_hi, kIdescN64, 1u);
        // Q_i and dO_i are read by nothing after dV and dK: the stage can be refilled
        mma_commit(&sm.q_empty[s]);
        if (t > 0) {
            // the compute warps have read the previous dQ out of TMEM
            if (!(ok = wait_bar(&sm.dq_free, (t - 1) & 1, ab, kSiteMmaDqFree))) break;
            tc_fence_after();
        }
        // dQ = dS K: dS^T read as an MN-major A (keys 16kk.. are rows 16kk.., 2 KiB
        // per K step), K_j rows 16kk.. as MN-major B
        mma_ss_k<0, 0>(tdq, dsm, k_mn, desc_hi, kIdescDQ, 0u);
        mma_ss_k<128, 128>(tdq, dsm, k_mn, desc_hi, kIdescDQ, 1u);
        mma_ss_k<256, 256>(tdq, dsm, k_mn, desc_hi, kIdescDQ, 1u);
        mma_ss_k<384, 384>(tdq, dsm, k_mn, desc_hi, kIdescDQ, 1u);
        mma_ss_k<512, 512>(tdq, dsm, k_mn, desc_hi, kIdescDQ, 1u);
        mma_ss_k<640, 640>(tdq, dsm, k_mn, desc_hi, kIdescDQ, 1u);
        mma_ss_k<768, 768>(tdq, dsm, k_mn, desc_hi, kIdescDQ, 1u);
        mma_ss_k<896, 896>(tdq, dsm, k_mn, desc_hi, kIdescDQ, 1u);
        mma_commit(&sm.dq_full); // every MMA of step t: P^T and dS^T consumed, dQ complete
    }
}

// Four groups of four compute warps.  Thread t of group g: key row t of the CTA's
// key tile for the score work on queries 32g .. 32g+31 of each step; query row t
// and dQ columns 16g .. 16g+15 for the dQ readout; in the epilogue, columns
// 32(g % 2) .. +31 of dV (g < 2) or dK (g >= 2) of key row t.
//
// Step t: read S^T, dP^T (releasing them for step t + 1's products), compute P^T
// and dS^T, wait for step t - 1's products to finish with the previous P^T and
// dS^T, write the new ones, then read out step t - 1's dQ (one step late, so that
// no thread waits for the products of the step it has just fed).
__device__ __forceinline__ void compute_role(BwdSmem &sm, const BwdParams &p, const CUtensorMap *tm_dq,
                                             uint32_t tmem, int bh, int key0, int len, int i_begin, int steps)
{
    const int warp = threadIdx.x / 32;
    const int g = warp / 4;              // query chunk of each step
    const int t = threadIdx.x % 128;     // TMEM lane
    const int half = g / 2;              // dQ staging block (columns 32 * half ..)
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + kColS + 32 * g, t_dp = tmem + lane_base + kColDP + 32 * g;
    const uint32_t t_pt = tmem + lane_base + kColPT + 16 * g;
    const uint32_t t_dq = tmem + lane_base + kColDQ + 16 * g;
    const bool causal = (p.mask_kind & kMaskCausal) != 0;
    const float sl2 = p.scale_log2;
    const int k = key0 + t;         // this thread's key
    const bool key_live = k < len;  // len <= n: keys past n (zero-filled rows) are never live
    // dS^T row t (this thread's key), queries 32g .. 32g+31: four 16-byte chunks
    // 4(g % 2) .. of the 128-byte row in block g / 2, swizzled with t % 8
    const uint32_t dst_row0 = smem_addr(sm.dst[0][g / 2]) + t * 128;
    const uint32_t dqs_row = smem_addr(sm.dq_stage[half]) + t * 128; // this thread's staging row
    const bool dq_issuer = t == 0 && g % 2 == 0;
    int *ab = &sm.abort_flag;
    bool ok = true;

    // dQ of step r into the accumulator: groups 2h and 2h+1 stage columns 32h ..
    // 32h+31 (row t at t * 128 bytes, 16-byte chunk c at c ^ (t % 8): conflict-free)
    // and one thread adds the block with a TMA reduction, which skips rows past m.
    // The block is rewritten only after the previous reduction has read it.
    auto dq_readout = [&](int r) -> bool {
        uint32_t qr[16];
        tmem_ld16(t_dq, qr);
        tmem_wait_ld();
        reg_fence16(qr);
        tc_fence_before();
        mbar_arrive(&sm.dq_free);
        if (dq_issuer) {
            bulk_wait_read_all();
            mbar_arrive(&sm.dqs_free[half]);
        }
        bool good = warp_all(wait_bar(&sm.dqs_free[half], r & 1, ab, kSiteCmpDqsFree));
        if (!good) return false;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c4 = 4 * (g % 2) + j;
            st_shared_v4(dqs_row + ((c4 ^ (t & 7)) << 4),
                         make_uint4(qr[4 * j], qr[4 * j + 1], qr[4 * j + 2], qr[4 * j + 3]));
        }
        fence_proxy_async_shared();
        mbar_arrive(&sm.dqs_full[half]);
        if (dq_issuer) {
            good = wait_bar(&sm.dqs_full[half], r & 1, ab, kSiteCmpDqsFull);
            if (good) {
                tma_reduce_add_3d(tm_dq, sm.dq_stage[half], 32 * half, (i_begin + r) * kBM, bh);
                bulk_commit_group();
            }
        }
        return warp_all(good);
    };

    for (int st = 0; st < steps && ok; ++st) {
        const int s = st % kStages;
        const int i0 = (i_begin + st) * kBM;
        ok = warp_all(wait_bar(&sm.q_full[s], (st / kStages) & 1, ab, kSiteCmpQFull));
        if (ok) ok = warp_all(wait_bar(&sm.sdp_full, st & 1, ab, kSiteCmpSdpFull));
        if (!ok) break;
        tc_fence_after();
        // Only the diagonal tile of a causal mask (i0 == key0: key t is allowed for
        // query row qq iff t <= qq) and padded key rows need masking; elsewhere the
        // whole warp takes the unmasked path.
        const bool diag = causal && i0 == key0;
        const bool plain = __all_sync(0xffffffffu, key_live) && !diag;
        const uint32_t ldv = smem_addr(sm.ld[s]) + 32 * g * 8; // float2 (L, D) per query row
        const uint32_t dst_row = dst_row0 + static_cast<uint32_t>(st & 1) * (2 * kTileBytes);
        uint32_t pp[16], pd[4];
        // (L, D) of rows qq, qq + 1 in one 16-byte load, issued two pairs ahead
        float4 ldq[3];
        ldq[0] = ld_shared_f4_ordered(ldv);
        ldq[1] = ld_shared_f4_ordered(ldv + 16);
        // the chunk is read and processed in two halves of 16 queries; every thread
        // has read both when it releases S^T and dP^T
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t sr[16], dr[16];
            tmem_ld16(t_s + 16 * hh, sr);
            tmem_ld16(t_dp + 16 * hh, dr);
            tmem_wait_ld();
            reg_fence16(sr);
            reg_fence16(dr);
            if (hh == 1) {
                tc_fence_before();
                mbar_arrive(&sm.s_loaded);
            }
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const int u = 8 * hh + v;
                const int qq = 32 * g + 2 * u;              // query rows qq, qq + 1 of the tile
                if (u + 2 < 16) ldq[(u + 2) % 3] = ld_shared_f4_ordered(ldv + (2 * u + 4) * 8);
                const float4 ld = ldq[u % 3];
                float e0 = ex2(fmaf(__uint_as_float(sr[2 * v]), sl2, -ld.x));
                float e1 = ex2(fmaf(__uint_as_float(sr[2 * v + 1]), sl2, -ld.z));
                if (!plain) {
                    e0 = (key_live && !(diag && t > qq)) ? e0 : 0.f;
                    e1 = (key_live && !(diag && t > qq + 1)) ? e1 : 0.f;
                }
                const float d0 = e0 * (__uint_as_float(dr[2 * v]) - ld.y);
                const float d1 = e1 * (__uint_as_float(dr[2 * v + 1]) - ld.w);
                pp[u] = pack_bf16x2(e0, e1);
                pd[u % 4] = pack_bf16x2(d0, d1);
                if (u % 4 == 3) {
                    // dS^T buffer st % 2 was last read by step st - 2's products,
                    // which completed before this thread wrote step st - 1's P^T
                    const int c4 = 4 * (g % 2) + u / 4;
                    st_shared_v4_ordered(dst_row + ((c4 ^ (t & 7)) << 4), make_uint4(pd[0], pd[1], pd[2], pd[3]));
                }
            }
        }
        if (st > 0) {
            // step st - 1's products have finished with P^T (and its dQ is ready)
            ok = warp_all(wait_bar(&sm.dq_full, (st - 1) & 1, ab, kSiteCmpDqFull));
            if (!ok) break;
            tc_fence_after();
        }
        tmem_st16(t_pt, pp);
        tmem_wait_st();
        tc_fence_before();
        fence_proxy_async_shared();
        mbar_arrive(&sm.p_ready);
        if (st > 0) ok = dq_readout(st - 1);
    }
    if (ok) {
        // the last step's dQ; its completion also covers every earlier product
        ok = warp_all(wait_bar(&sm.dq_full, (steps - 1) & 1, ab, kSiteCmpDqFull));
        if (ok) {
            tc_fence_after();
            ok = dq_readout(steps - 1);
        }
    }
    // the staging blocks must stay valid, and the sums land, before the CTA exits
    if (dq_issuer) bulk_wait_all();
    if (!ok) return;
    // 32 columns of dV (groups 0, 1) or scale * dK (groups 2, 3) of this thread's
    // key row: every MMA completed with the last dq_full
    tc_fence_after();
    uint32_t r[32];
    tmem_ld32(tmem + lane_base + (g < 2 ? kColDV : kColDK) + 32 * (g % 2), r);
    tmem_wait_ld();
    reg_fence32(r);
    if (k < p.n) {
        const float f = g < 2 ? 1.f : p.scale;
        uint4 *dst = reinterpret_cast<uint4 *>((g < 2 ? p.dv : p.dk) + (static_cast<size_t>(bh) * p.n + k) * p.d +
                                               32 * (g % 2));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (32 * (g % 2) + 8 * c >= p.d) break; // narrower heads: only the first d columns exist
            uint4 a;
            a.x = pack_bf16x2(__uint_as_float(r[8 * c + 0]) * f, __uint_as_float(r[8 * c + 1]) * f);
            a.y = pack_bf16x2(__uint_as_float(r[8 * c + 2]) * f, __uint_as_float(r[8 * c + 3]) * f);
            a.z = pack_bf16x2(__uint_as_float(r[8 * c + 4]) * f, __uint_as_float(r[8 * c + 5]) * f);
            a.w = pack_bf16x2(__uint_as_float(r[8 * c + 6]) * f, __uint_as_float(r[8 * c + 7]) * f);
            dst[c] = a;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dq, const BwdParams p)
{
    extern __shared__ uint8_t smem_raw[];
    BwdSmem &sm = *reinterpret_cast<BwdSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32;
    // Heads in groups whose Q and dO fit in L2 together, so the CTAs running at one time
    // share them; within a group, key tile j ascending first (with a causal mask the low
    // key tiles see the most queries).
    const int per_group = p.group_heads * p.k_tiles;
    const int grp = static_cast<int>(blockIdx.x) / per_group, r_in = static_cast<int>(blockIdx.x) - grp * per_group;
    const int heads = min(p.group_heads, p.BH - grp * p.group_heads); // the last group may be short
    const int j = r_in / heads;
    const int bh = grp * p.group_heads + r_in % heads;
    const int key0 = j * kBM;
    const int len = key_len(p, bh);
    const bool causal = (p.mask_kind & kMaskCausal) != 0;
    const int i_begin = causal ? j : 0; // causal: m == n, query tile i sees key tile j iff i >= j
    const int steps = key0 < len ? p.q_tiles - i_begin : 0;

    if (steps <= 0) {
        // no query sees any key of this tile: its gradients are 0
        const uint4 z = make_uint4(0, 0, 0, 0);
        const int row8 = p.d / 8; // 16-byte chunks per row
        for (int r = threadIdx.x; r < kBM * row8; r += blockDim.x) {
            const int kk = key0 + r / row8;
            if (kk >= p.n) continue;
            const size_t off = (static_cast<size_t>(bh) * p.n + kk) * row8 + r % row8;
            reinterpret_cast<uint4 *>(p.dv)[off] = z;
            reinterpret_cast<uint4 *>(p.dk)[off] = z;
        }
        return;
    }

    if (threadIdx.x == 0) {
        mbar_init(&sm.kv_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.q_full[s], 1);
            mbar_init(&sm.q_empty[s], 1);
        }
        mbar_init(&sm.sdp_full, 1);
        mbar_init(&sm.p_ready, kComputeThreads);
        mbar_init(&sm.dq_full, 1);
        mbar_init(&sm.dq_free, kComputeThreads);
        mbar_init(&sm.s_loaded, kComputeThreads);
        for (int g = 0; g < 2; ++g) {
            mbar_init(&sm.dqs_free[g], 1);
            mbar_init(&sm.dqs_full[g], 2 * kBM);
        }
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

    if (warp < kGroups * 4) {
        compute_role(sm, p, &tm_dq, tmem, bh, key0, len, i_begin, steps);
    } else if (warp == kLoadWarp) {
        if (threadIdx.x % 32 == 0) load_role(sm, p, &tm_q, &tm_k, &tm_v, &tm_do, bh, key0, i_begin, steps);
        __syncwarp();
    } else {
        if (threadIdx.x % 32 == 0) {
            mma_role(sm, tmem, steps);
            if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) {
                // make sure no MMA is still writing TMEM when the CTA frees it
                mma_commit(&sm.drain);
                drain_wait(&sm.drain, 0);
            }
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// D_i = sum_c dO_ic O_ic and (lse_i * log2 e, D_i) per query row (padding rows of
// the last tile: (+inf, 0)), and the row's 64 accumulator columns zeroed.  Eight
// threads per row, each with 16 bytes of O and dO and 32 bytes of the accumulator,
// so a warp's loads and stores cover whole consecutive rows; the eight partial dot
// products are summed with three shuffles.
__global__ void attn_bwd_pre_kernel(const __nv_bfloat16 *__restrict__ out, const __nv_bfloat16 *__restrict__ dout,
                                    const float *__restrict__ lse, float2 *__restrict__ ld,
                                    float *__restrict__ dq_acc, int BH, int m, int m_pad, int d)
{
    const size_t t = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t r = t / 8; // query row (BH * m_pad * 8 threads: a whole number of warps)
    const int part = static_cast<int>(t % 8);
    if (r >= static_cast<size_t>(BH) * m_pad) return; // whole warps only
    const int bh = static_cast<int>(r / m_pad), q = static_cast<int>(r % m_pad);
    const size_t row = static_cast<size_t>(bh) * m + q;
    float dsum = 0.f;
    if (q < m && 8 * part < d) {
        const uint4 a = reinterpret_cast<const uint4 *>(out + row * d)[part];
        const uint4 b = reinterpret_cast<const uint4 *>(dout + row * d)[part];
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            dsum = fmaf(__uint_as_float(av[u] << 16), __uint_as_float(bv[u] << 16), dsum);
            dsum = fmaf(__uint_as_float(av[u] & 0xffff0000u), __uint_as_float(bv[u] & 0xffff0000u), dsum);
        }
    }
    dsum += __shfl_xor_sync(0xffffffffu, dsum, 4);
    dsum += __shfl_xor_sync(0xffffffffu, dsum, 2);
    dsum += __shfl_xor_sync(0xffffffffu, dsum, 1);
    if (q >= m) {
        if (part == 0) ld[r] = make_float2(CUDART_INF_F, 0.f);
        return;
    }
    if (part == 0) ld[r] = make_float2(lse[row] * 1.4426950408889634f, dsum);
    float4 *acc = reinterpret_cast<float4 *>(dq_acc + row * kD);
    acc[part] = make_float4(0.f, 0.f, 0.f, 0.f);
    acc[part + 8] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ = bf16(scale * accumulator), eight elements per thread: chunk r is columns
// 8 (r % (d / 8)) .. of row r / (d / 8); the accumulator's rows are 64 wide.
__global__ void attn_bwd_post_kernel(const float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dq,
                                     size_t count8, float scale, int d)
{
    const size_t r = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (r >= count8) return;
    const size_t row = r / (d / 8), c8 = r % (d / 8);
    const float4 *src = reinterpret_cast<const float4 *>(dq_acc + row * kD + 8 * c8);
    const float4 a = src[0];
    const float4 b = src[1];
    uint4 o;
    o.x = pack_bf16x2(a.x * scale, a.y * scale);
    o.y = pack_bf16x2(a.z * scale, a.w * scale);
    o.z = pack_bf16x2(b.x * scale, b.y * scale);
    o.w = pack_bf16x2(b.z * scale, b.w * scale);
    reinterpret_cast<uint4 *>(dq)[r] = o;
}

constexpr size_t kSmemBytes = sizeof(BwdSmem) + 1024; // + alignment slack

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

} // namespace

size_t bwd_workspace_bytes(int B, int h, int m)
{
    const size_t BH = static_cast<size_t>(B) * h;
    const size_t m_pad = align_up(static_cast<size_t>(m), kBM);
    return align_up(BH * m * kD * sizeof(float), 256) + BH * m_pad * sizeof(float2);
}

cudaError_t launch_bwd(const BwdProblem &pb, cudaStream_t stream)
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
            if ((e = cudaFuncSetAttribute(attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(kSmemBytes))) != cudaSuccess)
                return e;
            configured[dev] = true;
        }
    }
    const int BH = pb.B * pb.h;
    const int m_pad = static_cast<int>(align_up(static_cast<size_t>(pb.m), kBM));
    float *dq_acc = static_cast<float *>(pb.workspace);
    float2 *ld = reinterpret_cast<float2 *>(static_cast<uint8_t *>(pb.workspace) +
                                            align_up(static_cast<size_t>(BH) * pb.m * kD * sizeof(float), 256));
    if (pb.d % 8 != 0 || pb.d < 8 || pb.d > kD) return cudaErrorInvalidValue;
    // rows of d elements in 64-wide, 128-row boxes: columns d .. 63 of a load read as zero
    CUtensorMap tq, tk, tv, tdo, tdq;
    if (!encode_bf16_3d(&tq, pb.q, pb.d, pb.m, BH, kBM) || !encode_bf16_3d(&tk, pb.k, pb.d, pb.n, BH, kBM) ||
        !encode_bf16_3d(&tv, pb.v, pb.d, pb.n, BH, kBM) || !encode_bf16_3d(&tdo, pb.dout, pb.d, pb.m, BH, kBM) ||
        !encode_rows_map_f32(&tdq, dq_acc, pb.m, BH))
        return cudaErrorInvalidValue;

    const size_t pre_threads = static_cast<size_t>(BH) * m_pad * 8;
    attn_bwd_pre_kernel<<<static_cast<unsigned>((pre_threads + 255) / 256), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(pb.out), static_cast<const __nv_bfloat16 *>(pb.dout), pb.lse, ld,
        dq_acc, BH, pb.m, m_pad, pb.d);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    BwdParams p;
    p.ld = ld;
    p.dq_acc = dq_acc;
    p.dk = static_cast<__nv_bfloat16 *>(pb.dk);
    p.dv = static_cast<__nv_bfloat16 *>(pb.dv);
    p.key_lengths = (pb.mask_kind & kMaskKeyPadding) ? pb.key_lengths : nullptr;
    p.BH = BH;
    p.h = pb.h;
    p.m = pb.m;
    p.n = pb.n;
    p.m_pad = m_pad;
    p.mask_kind = pb.mask_kind;
    p.q_tiles = m_pad / kBM;
    p.d = pb.d;
    p.scale_log2 = pb.scale * 1.4426950408889634f;
    p.scale = pb.scale;
    const int k_tiles = (pb.n + kBM - 1) / kBM;
    p.k_tiles = k_tiles;
    {
        // about 32 MB of Q and dO per group (a quarter of L2)
        const size_t qdo_head = 2ull * pb.m * kD * 2;
        const size_t g = (32ull << 20) / (qdo_head > 0 ? qdo_head : 1);
        p.group_heads = static_cast<int>(g < 1 ? 1 : (g > static_cast<size_t>(BH) ? BH : g));
    }
    attn_bwd_kernel<<<k_tiles * BH, kThreads, kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    const size_t count8 = static_cast<size_t>(BH) * pb.m * (pb.d / 8);
    attn_bwd_post_kernel<<<static_cast<unsigned>((count8 + 255) / 256), 256, 0, stream>>>(
        dq_acc, static_cast<__nv_bfloat16 *>(pb.dq), count8, pb.scale, pb.d);
    return cudaGetLastError();
}

cudaError_t bwd_status_read_and_clear(cudaStream_t stream, uint32_t *code, uint32_t *info)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned int c = 0, i = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&c, g_bwd_status_code, sizeof c)) != cudaSuccess) return e;
    if ((e = cudaMemcpyFromSymbol(&i, g_bwd_status_info, sizeof i)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_bwd_status_code, &zero, sizeof zero)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_bwd_status_info, &zero, sizeof zero)) != cudaSuccess) return e;
    *code = c;
    *info = i;
    return cudaSuccess;
}

} // namespace attn
