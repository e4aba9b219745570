// Forward of the masked scaled dot-product attention for heads of width 128
// (bf16) on tcgen05 + TMA + TMEM: out = softmax(scale Q K^T + M) V, the attention
// equation of "Paper Deep Reading: Attention Is All You Need", §04, for the model
// variants whose heads are 128 wide (the variants table of the same page).
//
// One CTA per (batch, head, pair of 128-row query tiles), heaviest pairs first;
// for heads of a single query and key tile, one CTA per pair of heads instead
// (attn_wide_kernel<true>).  The two tiles ("slots") share one stream of K and V
// tiles (head pairs: one K and V tile each) and take turns on the tensor cores:
// while one slot's softmax runs, the other slot's MMAs do.  Q and
// each 128-key tile of K and V are 128 x 128 bf16, loaded by TMA as two 64-column
// boxes (128-byte swizzle atoms) 16 KiB apart; K and V pass through two-stage rings
// of their own (a K tile is free a tile before its V tile is).
//   MMA:     S_s = Q_s K_t^T            (8 x M128 N128 K16: four K steps in each atom)
//   softmax: 4 warps per slot, thread r = row r = TMEM lane r; scores masked on
//            boundary tiles only; P = exp2(S scale log2 e - r) as bf16 pairs written
//            over the upper half of S, against a per-row reference r: the row max
//            of the row's first key tile, moved up only when a later tile's sum
//            exceeds 2^15 (by an exact power of two, or, when a weight
//            overflowed, to the max of the row's recomputed scores); O is rescaled
//            in TMEM only when r moves
//   MMA:     O_s += P_s V_t             (8 x M128 N128 K16, P from TMEM, V MN-major:
//            its two 64-column atoms are the two halves of N)
// Each slot has an MMA issuer; per key tile t the two issue, taking turns, O_0 +=
// P_0 V_(t-1), S_0 = Q_0 K_t^T, then O_1 += P_1 V_(t-1), S_1 = Q_1 K_t^T.  The tensor
// cores run a thread's MMAs in order, so S_s(t) overwrites P_s(t - 1) only after
// O_s += P_s V_(t-1) has read it, and the commit that signals S_s(t) also covers
// that P V: once the softmax sees S_s(t), O_s is free to rescale.  Each slot covers
// only the key tiles its rows can see (causal diagonal, padded length, window); the
// CTA loads their union.
// The epilogue divides O by the row sum (0 for a row with no allowed key) and stores
// the bf16 tile through the slot's Q buffer with TMA.
// TMEM (512 columns), per slot s at column 256 s: S [0,128) with P over [64,128)
// as bf16 pairs, O [128,256).
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
#include "softmax_tile.cuh"

namespace attn {

__device__ unsigned int g_wide_status_code;
__device__ unsigned int g_wide_status_info;

namespace {

constexpr int kBM = 128;                              // query rows per slot
constexpr int kBN = 128;                              // keys per key tile
constexpr int kDW = 128;                              // head width
constexpr int kSlots = 2;                             // query tiles (or heads) per CTA
constexpr uint32_t kAtomBytes = 128 * 64 * 2;         // one 64-column atom of a 128-row tile
constexpr uint32_t kTileBytes = (kDW / 64) * kAtomBytes; // 32 KiB
constexpr int kStages = 2;
constexpr int kLoadWarp = 4 * kSlots;
constexpr int kMmaWarp = kLoadWarp + 1; // MMA issuer of slot 0 (slot s: kMmaWarp + s); allocates TMEM
// three full warpgroups: two of softmax, one of control (loader, the two MMA
// issuers and an idle warp that completes it so that setmaxnreg can move
// registers to the softmax)
constexpr int kThreads = 384;
constexpr uint32_t kSoftmaxRegs = 200; // per thread, softmax warpgroups
constexpr uint32_t kControlRegs = 104; // per thread, control warpgroup
static_assert(2 * kSoftmaxRegs + kControlRegs <= 3 * 168, "register split exceeds the launch allocation");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSlotCols = 256, kColS = 0, kColP = 64, kColO = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull; // 2 s
constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0, 0);  // Q (K-major) x K (K-major)
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kDW, 0, 1); // P (TMEM) x V (MN-major), N = 128

enum WideSite : uint32_t {
    kSiteLoadKEmpty = 1, kSiteLoadVEmpty, kSiteMmaQFull, kSiteMmaKFull, kSiteMmaVFull, kSiteMmaPFull,
    kSiteSmSFull, kSiteSmODone, kSiteMmaTurn, kSiteSmStaged
};

struct alignas(1024) WideSmem {
    uint8_t q[kSlots][kTileBytes];
    uint8_t k[kStages][kTileBytes];
    uint8_t v[kStages][kTileBytes];
    uint64_t q_full[kSlots], k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
    uint64_t s_full[kSlots], p_full[kSlots], o_done[kSlots], drain[kSlots];
    uint64_t turn[kSlots]; // turn[s]: the other issuer has issued its group, slot s may go
    uint64_t staged[kSlots]; // slot s's output tile is in q[s], ready for the TMA store
    uint32_t tmem_base;
    int abort_flag;
};

static_assert(kBN == kTileKeys, "the shared softmax helpers take 128-key tiles");
static_assert(kSlots == 2, "the softmax role picks its slot's range with a two-way select");
static_assert(sizeof(WideSmem) + 1024 <= 227 * 1024, "shared memory per CTA");

struct WideParams {
    const __nv_bfloat16 *q, *k; // read only by the rare score recomputation
    const int32_t *key_lengths; // nullptr unless key padding
    __nv_bfloat16 *out;
    float *lse;
    int BH, h, m, n, mask_kind, q_pairs;
    int group_heads; // query-tile pairs: heads per group of the CTA order (their K and V share L2)
    int window;     // restricted attention: keys with |i - j| <= window stay; -1: none
    int head_pairs; // 1: m, n <= 128, and slot s of CTA c takes (batch, head) 2c + s (host side;
                    // the kernel is instantiated for each mode)
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

// mbarrier try_wait without a suspend-time hint (the hardware's own time limit).
__device__ __forceinline__ bool mbar_try_wait_nohint(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0;
}

// Bounded wait of the softmax warps for their scores: try_wait without the
// 20 us suspend hint, which resumes the warps sooner after the MMAs complete
// (a test_wait spin would take issue slots from the other slot's softmax).
__device__ __forceinline__ bool wait_scores(uint64_t *bar, uint32_t parity, int *abort_flag, uint32_t site)
{
    const uint32_t a = smem_addr(bar);
    const uint64_t start = global_timer_ns();
    while (true) {
        for (int k = 0; k < 64; ++k)
            if (mbar_try_wait_nohint(a, parity)) return true;
        if (*reinterpret_cast<volatile int *>(abort_flag)) return false;
        if (global_timer_ns() - start > kWaitLimitNs) {
            *reinterpret_cast<volatile int *>(abort_flag) = 1;
            atomicOr(&g_wide_status_code, 1u);
            atomicCAS(&g_wide_status_info, 0u, site);
            return false;
        }
    }
}

// Bounded wait that polls (test_wait) instead of suspending: a thread suspended in
// try_wait resumes a few hundred cycles after the phase completes, which the MMA
// issuers cannot afford (the tensor cores drain meanwhile).
__device__ __forceinline__ bool wait_poll(uint64_t *bar, uint32_t parity, int *abort_flag, uint32_t site)
{
    const uint32_t a = smem_addr(bar);
    if (mbar_test_wait(a, parity)) return true;
    const uint64_t start = global_timer_ns();
    while (true) {
        for (int k = 0; k < 256; ++k)
            if (mbar_test_wait(a, parity)) return true;
        if (*reinterpret_cast<volatile int *>(abort_flag)) return false;
        if (global_timer_ns() - start > kWaitLimitNs) {
            *reinterpret_cast<volatile int *>(abort_flag) = 1;
            atomicOr(&g_wide_status_code, 1u);
            atomicCAS(&g_wide_status_info, 0u, site);
            return false;
        }
    }
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// Key tiles [lo, hi) that rows q0s .. min(m, q0s + 128) - 1 can see; lo == hi when none.
__device__ __forceinline__ void slot_range(const WideParams &p, int q0s, int len, bool causal, int &lo, int &hi)
{
    lo = hi = 0;
    if (q0s >= p.m) return;
    int kv_end = causal ? min(len, q0s + kBM) : len;
    int first = 0;
    if (p.window >= 0) {
        first = max(0, q0s - p.window) / kBN;
        kv_end = min(kv_end, min(p.m, q0s + kBM) + p.window);
    }
    if (kv_end <= first * kBN) return;
    lo = first;
    hi = (kv_end + kBN - 1) / kBN;
}

// Scores of query row i of head bh against keys key0 .. key0+127, recomputed on
// the CUDA cores from Q and K in global memory (fp32 sums of exact bf16
// products), multiplied by scale * log2 e, and -inf where not allowed (column c
// is allowed iff cnt_lo <= c < cnt; allowed keys are below n).  Rows past m read
// as zero queries, as the TMA loads fill them.  Taken only when a tile's
// exponentials against the running reference overflowed, so it favours size
// over speed.
__device__ __forceinline__ void recompute_scores(const WideParams &p, int bh, int i, int key0, int cnt_lo, int cnt,
                                                  float (&x)[kBN])
{
    const bool row_in = i < p.m;
    const uint4 *qr = reinterpret_cast<const uint4 *>(p.q + (static_cast<size_t>(bh) * p.m + (row_in ? i : 0)) * kDW);
    float srow[kBN];
#pragma unroll 1
    for (int c = 0; c < kBN; ++c) {
        float v = -CUDART_INF_F;
        if (c < cnt && c >= cnt_lo) {
            const uint4 *kr = reinterpret_cast<const uint4 *>(p.k + (static_cast<size_t>(bh) * p.n + key0 + c) * kDW);
            float a = 0.f;
#pragma unroll 4
            for (int u = 0; u < kDW / 8; ++u) {
                const uint4 qa = row_in ? qr[u] : make_uint4(0, 0, 0, 0), ka = kr[u];
                const uint32_t qw[4] = {qa.x, qa.y, qa.z, qa.w}, kw[4] = {ka.x, ka.y, ka.z, ka.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a = fmaf(__uint_as_float(qw[e] << 16), __uint_as_float(kw[e] << 16), a);
                    a = fmaf(__uint_as_float(qw[e] & 0xffff0000u), __uint_as_float(kw[e] & 0xffff0000u), a);
                }
            }
            v = a * p.scale_log2;
        }
        srow[c] = v;
    }
#pragma unroll
    for (int c = 0; c < kBN; ++c) x[c] = srow[c];
}

__device__ __forceinline__ void zero_rows(const WideParams &p, int bh, int i)
{
    if (i >= p.m) return;
    uint4 *orow = reinterpret_cast<uint4 *>(p.out + (static_cast<size_t>(bh) * p.m + i) * kDW);
    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < kDW / 8; ++c) orow[c] = z;
    if (p.lse != nullptr) p.lse[static_cast<size_t>(bh) * p.m + i] = -CUDART_INF_F;
}

// kHeadPairs: the launch has one query tile and one key tile per head, and each
// CTA takes two heads (compiled separately so that the other launches carry none
// of it).
template <bool kHeadPairs>
__global__ void __launch_bounds__(kThreads, 1)
attn_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 const WideParams p)
{
    extern __shared__ uint8_t smem_raw[];
    WideSmem &sm = *reinterpret_cast<WideSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                 ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    constexpr bool hp = kHeadPairs;
    const bool causal = (p.mask_kind & kMaskCausal) != 0;
    // Slot s works on query rows q0s[s] .. q0s[s] + 127 of head bhs[s].  Query-tile
    // pairs: one head, two consecutive query tiles; heads in groups whose keys and values
    // fit in L2 together (the CTAs running at one time share them), heaviest pairs first
    // within a group (with a causal mask later query tiles see more keys).  Head pairs:
    // two heads, query tile 0; a slot past the last head has no rows.
    const int per_group = p.group_heads * p.q_pairs;
    const int grp = static_cast<int>(blockIdx.x) / per_group, r_in = static_cast<int>(blockIdx.x) - grp * per_group;
    const int g_heads = min(p.group_heads, p.BH - grp * p.group_heads); // the last group may be short
    int bhs[kSlots], q0s[kSlots], lens[kSlots], lo[kSlots], hi[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        if (hp) {
            bhs[s] = kSlots * static_cast<int>(blockIdx.x) + s;
            q0s[s] = 0;
        } else {
            bhs[s] = grp * p.group_heads + r_in % g_heads;
            q0s[s] = ((p.q_pairs - 1 - r_in / g_heads) * kSlots + s) * kBM;
        }
        int len = 0;
        if (bhs[s] < p.BH) {
            len = p.n;
            if (p.key_lengths != nullptr) {
                len = __ldg(p.key_lengths + bhs[s] / p.h);
                len = len < 0 ? 0 : (len > p.n ? p.n : len);
            }
            slot_range(p, q0s[s], len, causal, lo[s], hi[s]);
        } else {
            lo[s] = hi[s] = 0;
        }
        lens[s] = len;
    }
    // union of the slots' key tiles; fill f of the ring holds key tile t_lo + f
    int t_lo = 0x7fffffff, t_hi = 0;
#pragma unroll
    for (int s = 0; s < kSlots; ++s)
        if (hi[s] > lo[s]) {
            t_lo = min(t_lo, lo[s]);
            t_hi = max(t_hi, hi[s]);
        }

    if (t_hi == 0) {
        // no allowed key for any row of the CTA: output 0
        if (warp < kLoadWarp) {
            const int s = warp / 4;
            const int bh = s == 0 ? bhs[0] : bhs[1];
            if (bh < p.BH) zero_rows(p, bh, (s == 0 ? q0s[0] : q0s[1]) + (warp % 4) * 32 + lane);
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&sm.q_full[s], 1);
            mbar_init(&sm.s_full[s], 1);
            mbar_init(&sm.p_full[s], kBM);
            mbar_init(&sm.o_done[s], 1);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.k_full[s], 1);
            mbar_init(&sm.k_empty[s], kSlots); // one commit from each MMA issuer
            mbar_init(&sm.v_full[s], 1);
            mbar_init(&sm.v_empty[s], kSlots);
        }
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&sm.drain[s], 1);
            mbar_init(&sm.turn[s], 1);
            mbar_init(&sm.staged[s], kBM);
        }
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
    const int n_fill = t_hi - t_lo;

    // The two register regions never rejoin: each ends with its own CTA-wide
    // barrier (every thread arrives exactly once).
    if (warp < kLoadWarp) {
        regs_increase<kSoftmaxRegs>();
        // softmax and epilogue of slot s: thread r = row r of the tile = TMEM lane r
        const int s = warp / 4, quad = warp % 4;
        const int row = quad * 32 + lane;
        const int bh = s == 0 ? bhs[0] : bhs[1], len = s == 0 ? lens[0] : lens[1];
        const int q0_slot = s == 0 ? q0s[0] : q0s[1];
        const int i = q0_slot + row;
        const int my_lo = s == 0 ? lo[0] : lo[1];
        const int n_s = (s == 0 ? hi[0] : hi[1]) - my_lo;
        if (n_s == 0) {
            if (bh < p.BH) zero_rows(p, bh, i);
        } else {
            const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
            const uint32_t t_s = tmem + lane_base + s * kSlotCols + kColS;
            const uint32_t t_p = tmem + lane_base + s * kSlotCols + kColP;
            const uint32_t t_o = tmem + lane_base + s * kSlotCols + kColO;
            const float sl2 = p.scale_log2;
            // keys allowed for row i: [klo, khi) (below the padded length, i + 1 causal,
            // and within `window` of i)
            int khi = causal ? min(len, i + 1) : len;
            int klo = 0;
            if (p.window >= 0) {
                khi = min(khi, i + p.window + 1);
                klo = i - p.window;
            }
            float m_run = -CUDART_INF_F; // running reference, log2 units, as used for the exponentials
            float l_run = 0.f;           // running sum of the rounded weights relative to m_run
            bool ok = true;
            for (int jj = 0; jj < n_s && ok; ++jj) {
                ok = warp_all(wait_scores(&sm.s_full[s], jj & 1, ab, kSiteSmSFull));
                if (!ok) break;
                tc_fence_after();
                uint32_t sr[kBN];
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) tmem_ld32(t_s + 32 * c, sr + 32 * c);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) reg_fence32(sr + 32 * c);
                const int key0 = (my_lo + jj) * kBN;
                // column c of the tile is allowed for row i iff cnt_lo <= c < cnt; a tile
                // is a boundary tile when that fails for some column of some row
                const int cnt = khi - key0, cnt_lo = klo - key0;
                const bool boundary = (key0 + kBN > len) || (causal && key0 + kBN - 1 > q0_slot) ||
                                      (p.window >= 0 && (key0 < q0_slot + kBM - 1 - p.window ||
                                                         key0 + kBN - 1 > q0_slot + p.window));
                float x[kBN];
#pragma unroll
                for (int c = 0; c < kBN; ++c) x[c] = __uint_as_float(sr[c]);
                const bool prescaled = boundary; // x already multiplied by scale * log2 e
                if (boundary) {
                    // scale first, then mask: a zero scale must not turn -inf into NaN; one
                    // bit mask of allowed columns per 32 columns, one bit test per column
#pragma unroll
                    for (int ch = 0; ch < kBN / 32; ++ch) {
                        const int top = min(max(cnt - 32 * ch, 0), 32);
                        const int bot = min(max(cnt_lo - 32 * ch, 0), 32);
                        uint32_t msk = top >= 32 ? 0xffffffffu : (1u << top) - 1u;
                        msk &= bot >= 32 ? 0u : ~((1u << bot) - 1u);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            x[32 * ch + e] = (msk & (1u << e)) ? x[32 * ch + e] * sl2 : -CUDART_INF_F;
                    }
                }
                // Reference for the exponentials: the row max of the row's first tile with
                // an allowed key; later tiles keep it and check the tile's sum instead.
                float m_use = m_run, alpha = 1.f;
                bool grow = false;
                const bool first = m_run == -CUDART_INF_F;
                if (first) move_reference(x, prescaled, sl2, m_run, m_use, alpha, grow);
                uint32_t pk[kBN / 2];
                // the sum of the weights as rounded: the output is a weighted mean of
                // exactly the weights P V applies
                float tile_sum = weights_bf16_rounded(x, prescaled, sl2, m_use, pk);
                if (!first && !(tile_sum <= kFastSumLimit)) {
                    if (tile_sum < CUDART_INF_F) {
                        // finite but large: scale the weights by 2^-k (k an integer, so the
                        // bf16 values scale exactly) and move the reference up by k
                        const int k = ((__float_as_int(tile_sum) >> 23) & 0xff) - 127 - 7; // 8..120
                        const float f2k = __int_as_float((127 - k) << 23);                 // 2^-k
#pragma unroll
                        for (int c2 = 0; c2 < kBN / 2; ++c2) {
                            const float lo2 = __uint_as_float(pk[c2] << 16), hi2 = __uint_as_float(pk[c2] & 0xffff0000u);
                            pk[c2] = pack_bf16x2(lo2 * f2k, hi2 * f2k);
                        }
                        tile_sum *= f2k;
                        alpha = f2k;
                        m_use = m_run + static_cast<float>(k);
                        grow = true;
                    } else {
                        // some weight overflowed (the scores grew by 128 or more in log2
                        // units, or are not finite): recompute this row's scores from Q and
                        // K, already scaled and masked, and take their max
                        recompute_scores(p, bh, i, key0, cnt_lo, cnt, x);
                        move_reference(x, true, sl2, m_run, m_use, alpha, grow);
                        tile_sum = weights_bf16_rounded(x, true, sl2, m_use, pk);
                    }
                }
                if (jj > 0 && __any_sync(0xffffffffu, grow)) {
                    // the P V of the previous tile has completed (the commit that
                    // signalled this S covers it): move O to the new reference
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
                tmem_st32(t_p, pk);
                tmem_st32(t_p + 32, pk + 32);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sm.p_full[s]);
                l_run = l_run * alpha + tile_sum;
                m_run = m_use;
            }
            if (ok) ok = warp_all(wait_bar(&sm.o_done[s], 0, ab, kSiteSmODone));
            if (ok) {
                tc_fence_after();
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                // weights are exp2(x - m_run) / l: lse = (m_run + log2 l) ln 2 (l sums the
                // rounded weights: within 2^-8 relative of the sum before rounding)
                if (p.lse != nullptr && i < p.m)
                    p.lse[static_cast<size_t>(bh) * p.m + i] =
                        l_run > 0.f ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -CUDART_INF_F;
                // Output: each thread writes its row of O / l into the slot's Q tile, free
                // now that every MMA of the slot has completed, in the 128-byte-swizzled
                // layout of the Q boxes (16-byte chunk c of row r at chunk c ^ (r % 8) of
                // its 64-column atom); then one thread stores the tile with two TMA boxes,
                // which clip rows past m.
                const uint32_t stage = smem_addr(sm.q[s]) + row * 128;
#pragma unroll 1
                for (int c = 0; c < kDW / 32; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(t_o + 32 * c, orr);
                    tmem_wait_ld();
                    reg_fence32(orr);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(orr[8 * q + 0]) * inv, __uint_as_float(orr[8 * q + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(orr[8 * q + 2]) * inv, __uint_as_float(orr[8 * q + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(orr[8 * q + 4]) * inv, __uint_as_float(orr[8 * q + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(orr[8 * q + 6]) * inv, __uint_as_float(orr[8 * q + 7]) * inv);
                        const int chunk = (c & 1) * 4 + q; // 16-byte chunk within the 64-column atom
                        st_shared_v4(stage + (c >> 1) * kAtomBytes + ((chunk ^ (row & 7)) << 4), w);
                    }
                }
                fence_proxy_async_shared();
                mbar_arrive(&sm.staged[s]);
                if (row == 0) {
                    if (wait_bar(&sm.staged[s], 0, ab, kSiteSmStaged)) {
                        tma_store_3d(&tm_o, sm.q[s], 0, q0_slot, bh);
                        tma_store_3d(&tm_o, sm.q[s] + kAtomBytes, 64, q0_slot, bh);
                        bulk_commit_group();
                        // the tile must stay in shared memory until the stores have read it
                        bulk_wait_all();
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        return;
    }
    regs_decrease<kControlRegs>();
    if (warp == kLoadWarp) {
        if (lane == 0) {
            tma_prefetch_map(&tm_q);
            tma_prefetch_map(&tm_k);
            tma_prefetch_map(&tm_v);
            for (int s = 0; s < kSlots; ++s) {
                if (hi[s] == lo[s]) continue;
                mbar_arrive_expect_tx(&sm.q_full[s], kTileBytes);
                tma_load_3d(sm.q[s], &tm_q, &sm.q_full[s], 0, q0s[s], bhs[s]);
                tma_load_3d(sm.q[s] + kAtomBytes, &tm_q, &sm.q_full[s], 64, q0s[s], bhs[s]);
                if (hp) {
                    // head pairs: the slot's one key tile of K and V, in stage s of each ring
                    mbar_arrive_expect_tx(&sm.k_full[s], kTileBytes);
                    tma_load_3d(sm.k[s], &tm_k, &sm.k_full[s], 0, 0, bhs[s]);
                    tma_load_3d(sm.k[s] + kAtomBytes, &tm_k, &sm.k_full[s], 64, 0, bhs[s]);
                    mbar_arrive_expect_tx(&sm.v_full[s], kTileBytes);
                    tma_load_3d(sm.v[s], &tm_v, &sm.v_full[s], 0, 0, bhs[s]);
                    tma_load_3d(sm.v[s] + kAtomBytes, &tm_v, &sm.v_full[s], 64, 0, bhs[s]);
                }
            }
            // K and V in rings of their own: K_t is free once both slots' S(t) have
            // read it, V_t only after both P V(t), a tile later
            const int bh = bhs[0];
            int k_issued = 0, v_issued = 0;
            for (int f = 0; f < (hp ? 0 : n_fill); ++f) {
                const int st = f % kStages;
                const uint32_t par = ((f / kStages) & 1) ^ 1;
                const int key0 = (t_lo + f) * kBN;
                if (!wait_bar(&sm.k_empty[st], par, ab, kSiteLoadKEmpty)) break;
                mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
                tma_load_3d(sm.k[st], &tm_k, &sm.k_full[st], 0, key0, bh);
                tma_load_3d(sm.k[st] + kAtomBytes, &tm_k, &sm.k_full[st], 64, key0, bh);
                ++k_issued;
                if (!wait_bar(&sm.v_empty[st], par, ab, kSiteLoadVEmpty)) break;
                mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
                tma_load_3d(sm.v[st], &tm_v, &sm.v_full[st], 0, key0, bh);
                tma_load_3d(sm.v[st] + kAtomBytes, &tm_v, &sm.v_full[st], 64, key0, bh);
                ++v_issued;
            }
            // copies still in flight must land before the CTA may exit
            for (int s = 0; s < kSlots; ++s)
                if (hi[s] > lo[s]) {
                    drain_wait(&sm.q_full[s], 0);
                    if (hp) {
                        drain_wait(&sm.k_full[s], 0);
                        drain_wait(&sm.v_full[s], 0);
                    }
                }
            for (int f = k_issued > kStages ? k_issued - kStages : 0; f < k_issued; ++f)
                drain_wait(&sm.k_full[f % kStages], (f / kStages) & 1);
            for (int f = v_issued > kStages ? v_issued - kStages : 0; f < v_issued; ++f)
                drain_wait(&sm.v_full[f % kStages], (f / kStages) & 1);
        }
        __syncwarp();
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        // One issuer per slot; per key tile t each issues O_s += P_s V(t - 1), then
        // S_s = Q_s K_t^T.  The two take turns (slot 0, slot 1, slot 0, ...), passing
        // a token through turn[], so the tensor cores receive the groups in that order
        // and the slots stay half an iteration apart, while each issuer's waits
        // overlap the other's MMAs.  Every issuer commits once per fill of each ring,
        // whether its slot read the fill or not, after waiting for that fill to land.
        // Head pairs: one key tile per slot, in stage s, loaded once; each issuer waits
        // only for its own and frees nothing.
        if (lane == 0) {
            const int s = warp - kMmaWarp;
            const int my_lo = s == 0 ? lo[0] : lo[1];
            const int my_hi = s == 0 ? hi[0] : hi[1];
            const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(0, 0, 1024) >> 32);
            const uint32_t q_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.q[s]), 16, 1024));
            const uint32_t k_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.k[0]), 16, 1024));
            // V as an MN-major B of N = 128: its two 64-column atoms kAtomBytes apart
            const uint32_t v_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.v[0]), kAtomBytes, 1024));
            constexpr uint32_t kStageUnits = kTileBytes >> 4;
            const uint32_t ts = tmem + s * kSlotCols + kColS, tp = tmem + s * kSlotCols + kColP;
            const uint32_t to = tmem + s * kSlotCols + kColO;
            bool ok = true, q_in = false;
            for (int t = t_lo; t <= t_hi && ok; ++t) {
                // fill f of the rings holds key tile t; V(t - 1) is fill f - 1
                const int f = t - t_lo;
                const int st = hp ? s : f % kStages, pst = hp ? s : (f + kStages - 1) % kStages;
                const uint32_t k_par = hp ? 0u : (f / kStages) & 1, v_par = hp ? 0u : ((f - 1) / kStages) & 1;
                const bool do_pv = t - 1 >= my_lo && t - 1 < my_hi, do_s = t >= my_lo && t < my_hi;
                // this slot's own inputs first, while the other issuer may still be issuing
                if (t > t_lo && (!hp || do_pv)) ok = wait_poll(&sm.v_full[pst], v_par, ab, kSiteMmaVFull);
                if (ok && do_pv) ok = wait_poll(&sm.p_full[s], (t - 1 - my_lo) & 1, ab, kSiteMmaPFull);
                if (ok && t < t_hi && (!hp || do_s)) ok = wait_poll(&sm.k_full[st], k_par, ab, kSiteMmaKFull);
                if (ok && do_s && !q_in) ok = q_in = wait_bar(&sm.q_full[s], 0, ab, kSiteMmaQFull);
                // then the turn: slot 1 after slot 0 of the same tile, slot 0 after slot 1
                // of the previous one
                if (ok && (s == 1 || t > t_lo))
                    ok = wait_poll(&sm.turn[s], (s == 1 ? f : f - 1) & 1, ab, kSiteMmaTurn);
                if (!ok) break;
                tc_fence_after();
                if (do_pv) {
                    // O_s += P_s(t - 1) V(t - 1): keys 16kk.. are P columns 8kk..
                    // (bf16 pairs) and V rows 16kk.. (2 KiB = 128 units per K step)
                    const uint32_t vd = v_lo + pst * kStageUnits;
                    const uint32_t acc0 = t - 1 > my_lo ? 1u : 0u;
                    mma_ts_k<0, 0>(to, tp, vd, desc_hi, kIdescPV, acc0);
                    mma_ts_k<8, 128>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<16, 256>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<24, 384>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<32, 512>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<40, 640>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<48, 768>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    mma_ts_k<56, 896>(to, tp, vd, desc_hi, kIdescPV, 1u);
                    if (t == my_hi) mma_commit(&sm.o_done[s]);
                }
                // this issuer is done with V(t - 1): its share of freeing the stage
                if (t > t_lo && !hp) mma_commit(&sm.v_empty[pst]);
                if (do_s) {
                    // S_s(t) = Q_s K_t^T, after the P V above in the tensor pipe; 16
                    // columns (32 bytes, 2 units) per K step, the second atom 16 KiB
                    // (1024 units) on
                    const uint32_t kd = k_lo + st * kStageUnits;
                    mma_ss_k<0, 0>(ts, q_lo, kd, desc_hi, kIdescS, 0u);
                    mma_ss_k<2, 2>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<4, 4>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<6, 6>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<1024, 1024>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<1026, 1026>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<1028, 1028>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_ss_k<1030, 1030>(ts, q_lo, kd, desc_hi, kIdescS, 1u);
                    mma_commit(&sm.s_full[s]);
                }
                if (t < t_hi && !hp) mma_commit(&sm.k_empty[st]);
                mbar_arrive(&sm.turn[1 - s]); // the other slot's turn
            }
            if (!ok) {
                // make sure no MMA of this issuer is still writing TMEM when the CTA frees it
                mma_commit(&sm.drain[s]);
                drain_wait(&sm.drain[s], 0);
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
            if ((e = cudaFuncSetAttribute(attn_wide_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(kSmemBytes))) != cudaSuccess ||
                (e = cudaFuncSetAttribute(attn_wide_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(kSmemBytes))) != cudaSuccess)
                return e;
            configured[dev] = true;
        }
    }
    if (!pb.bf16 || pb.d != kDW) return cudaErrorInvalidValue;
    const int BH = pb.B * pb.h;
    CUtensorMap tq, tk, tv, to;
    if (!encode_bf16_3d(&tq, pb.q, kDW, pb.m, BH, kBM) || !encode_bf16_3d(&tk, pb.k, kDW, pb.n, BH, kBN) ||
        !encode_bf16_3d(&tv, pb.v, kDW, pb.n, BH, kBN) || !encode_bf16_3d(&to, pb.out, kDW, pb.m, BH, kBM))
        return cudaErrorInvalidValue;
    WideParams p;
    p.q = static_cast<const __nv_bfloat16 *>(pb.q);
    p.k = static_cast<const __nv_bfloat16 *>(pb.k);
    p.key_lengths = (pb.mask_kind & kMaskKeyPadding) ? pb.key_lengths : nullptr;
    p.out = static_cast<__nv_bfloat16 *>(pb.out);
    p.lse = pb.lse;
    p.BH = BH;
    p.h = pb.h;
    p.m = pb.m;
    p.n = pb.n;
    p.mask_kind = pb.mask_kind;
    p.q_pairs = (pb.m + kSlots * kBM - 1) / (kSlots * kBM);
    {
        // about 32 MB of keys and values per group (a quarter of L2)
        const size_t kv_head = 2ull * pb.n * kDW * 2;
        const size_t g = (32ull << 20) / (kv_head > 0 ? kv_head : 1);
        p.group_heads = static_cast<int>(g < 1 ? 1 : (g > static_cast<size_t>(BH) ? BH : g));
    }
    // one query tile and one key tile per head: two heads per CTA, so that the
    // second slot has rows (and the grid halves)
    p.head_pairs = (pb.m <= kBM && pb.n <= kBN && BH > 1) ? 1 : 0;
    p.window = (pb.mask_kind & kMaskWindow) ? pb.window : -1;
    p.scale_log2 = pb.scale * 1.4426950408889634f;
    const long long grid = p.head_pairs ? (BH + kSlots - 1) / kSlots : static_cast<long long>(BH) * p.q_pairs;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    if (p.head_pairs)
        attn_wide_kernel<true><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tq, tk, tv, to, p);
    else
        attn_wide_kernel<false><<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tq, tk, tv, to, p);
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
