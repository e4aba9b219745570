// Whole-head-resident masked attention for short sequences on sm_103a (TMA + tcgen05 + TMEM).
//
// softmax(scale * Q K^T + M) V for one 128-row query tile of one (batch, head) per
// CTA ("Paper Deep Reading: Attention Is All You Need", §04 attention equation with
// the mask M; the slide deck's "Three Applications of Attention": encoder
// self-attention with key padding, decoder self-attention with a causal mask,
// encoder-decoder attention).  A query tile with up to 256 keys fits in shared
// memory and TMEM at once, so each row's softmax is taken over the whole row: the
// exact row maximum first, then the exponentials, with no running rescale.  This
// path is bound by HBM bandwidth (every byte of Q, K, V and O is moved once; the
// query tiles of a head read its K and V from L2 after the first), so the kernel is
// built for many small CTAs in flight rather than for tensor-pipe throughput.
//
// One CTA of 160 threads per query tile: warps 0-3 own one query row per thread
// (TMEM lane t = row q0 + t), warp 4 issues the copies and the MMAs.
//   1. warp 4 issues the TMA loads, one copy per lane: Q (one 128-row box; rows past
//      m read as 0), then K, then V, in 64-row and 16-row boxes only up to the keys
//      some row may see (the padded length, or m under a causal mask, rounded up to
//      16), so padded keys cost almost no HBM traffic;
//   2. S = Q K^T into TMEM columns [0, kv_rows)      (4 x tcgen05.mma M128 N=kv_rows K16)
//   3. each row thread: pass 1 takes the row maximum over its allowed keys (32-column
//      TMEM loads that also return the chunk's maximum, taken as is for a chunk allowed
//      whole for the warp, over the allowed columns otherwise), pass 2
//      takes P = exp2(S * scale * log2 e - max), rounds it to bf16 pairs written over
//      the start of S, and sums the ROUNDED weights, so the output is a weighted mean
//      with exactly the weights the MMA applies (the log-sum-exp output uses the sum
//      before rounding, the exact statistic);
//   4. O = P V after S in TMEM                       (kv_rows / 16 x M128 N64 K16, P from TMEM),
//      issued 32 keys at a time as soon as every row has stored that chunk of P
//      (above 192 keys O lies over the last two chunks of S, whose weights each row
//      takes first and holds in registers: kernel variant kLong);
//   5. epilogue: O / sum in bf16; each warp stages its 32 rows in the (now free) Q
//      buffer with the 128-byte swizzle and stores them with one TMA copy, which clips
//      rows past m (and columns past d_k for narrow heads).
// Several CTAs share an SM (128 or 256 of its 512 TMEM columns each): while some
// compute, the loads of others are in flight.  A CTA issues its loads before it
// allocates TMEM, so a CTA waiting for columns already has its data coming.
//
// Launched as a programmatic dependent: the set-up above the dependency wait
// overlaps the previous kernel, and nothing touches global memory or TMEM before
// the wait.  Each CTA lets the next grid launch as soon as it starts; every kernel
// of this library allocates TMEM only after its own dependency wait, so a dependent
// never holds columns a CTA of this grid still waits for.
//
// Every mbarrier wait is bounded; a wait that runs out sets the abort flag and
// this file's status word, the CTA waits (bounded) for its own copies and MMAs,
// frees TMEM and exits without storing.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {

__device__ unsigned int g_resident_status_code;
__device__ unsigned int g_resident_status_info;

namespace {

constexpr int kRows = 128;     // query rows per head (TMEM lanes)
constexpr int kD = 64;         // tile width (narrower heads zero-padded by the loads)
constexpr int kKeyBox = 16;    // key rows of the small K/V load (the granule of the rows loaded)
constexpr int kKeyBoxBig = 64; // key rows of the large K/V load
constexpr uint32_t kQBytes = kRows * kD * 2;      // 16 KiB
constexpr uint32_t kRowBytes = kD * 2;            // one key row in shared memory
constexpr uint32_t kIdescPV = idesc_bf16_f32(kRows, kD, 0, 1); // P (TMEM) x V (MN-major)
constexpr uint64_t kDefaultWaitNs = 2000000000ull; // 2 s
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 0.2 s
// S takes up to 256 TMEM columns and O 64: above 192 keys O lies over the last two
// chunks of S, whose weights are taken first and held in registers (see pass 2)
static_assert(kResidentMaxKeys % 32 == 0 && kResidentMaxKeys <= 256, "S must fit 256 columns");
constexpr int kShortKeys = 192; // up to this many keys S and O never overlap

// where a wait gave up (the status word's info)
enum Site : uint32_t { kSiteQK = 1, kSiteS = 2, kSiteP = 3, kSiteV = 4, kSiteO = 5 };

struct Ctl {
    uint64_t qk_full, v_full, s_full, o_full, drain;
    uint64_t p_full[kResidentMaxKeys / 32]; // chunk c of P stored by every row
    uint32_t tmem_base;
    int abort_flag;
};

struct ResidentParams {
    const int32_t *key_lengths; // [B] or nullptr
    float *lse;                 // [B][h][m] natural log, or nullptr
    int h, m, n, mask_kind;
    int q_tiles;                // 128-row query tiles per head (one CTA each)
    int window;                 // restricted attention: keys with |i - j| <= window stay; -1: none
    int kv_cap;                 // key rows the K and V buffers hold: n rounded up to kKeyBox
    float scale_log2;
    uint64_t wait_ns;           // limit of every bounded wait
    int withhold_p_arrival;     // test hook: the first chunk's barrier waits for one arrival more
                                // than the row threads make, so the MMA issuer's wait runs out
};

__device__ __forceinline__ bool give_up(int *abort_flag, uint64_t start, uint64_t limit_ns, uint32_t site)
{
    if (*reinterpret_cast<volatile int *>(abort_flag)) return true;
    if (global_timer_ns() - start > limit_ns) {
        *reinterpret_cast<volatile int *>(abort_flag) = 1;
        atomicOr(&g_resident_status_code, 1u);
        atomicCAS(&g_resident_status_info, 0u, site);
        return true;
    }
    return false;
}

// Bounded wait that polls (test_wait): every wait of this kernel is on its critical
// path, and a warp suspended in try_wait resumes hundreds of cycles after the phase
// completes; the few warps of a CTA have nothing else to issue meanwhile.
__device__ __forceinline__ bool wait_poll(uint64_t *bar, uint32_t parity, int *abort_flag, uint64_t limit_ns,
                                          uint32_t site)
{
    const uint32_t a = smem_addr(bar);
    if (mbar_test_wait(a, parity)) return true;
    const uint64_t start = global_timer_ns();
    while (true) {
        for (int k = 0; k < 64; ++k)
            if (mbar_test_wait(a, parity)) return true;
        if (give_up(abort_flag, start, limit_ns, site)) return false;
    }
}

// Bounded wait that ignores the abort flag (to let in-flight work land on the way out).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint32_t a = smem_addr(bar);
    const uint64_t start = global_timer_ns();
    while (!mbar_try_wait(a, parity))
        if (global_timer_ns() - start > kDrainLimitNs) return;
}

// 32 consecutive TMEM columns of this warp's 32 lanes, as tmem_ld32, and their
// maximum, taken by the load itself (sm_103a): as fmaxf, a NaN column is passed
// over.  Both are valid after tmem_wait_ld.
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float &mx)
{
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, %32, [%33];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=f"(mx)
        : "r"(taddr));
}

// Row maximum of one 32-key chunk of raw scores.  kMask: only columns e of the chunk
// with lo_rel <= e < hi_rel count (a chunk that is allowed whole for every row of the
// warp skips the test); kLo: the lower bound applies (a window), else lo_rel <= 0.
template <bool kMask, bool kLo>
__device__ __forceinline__ float chunk_max(const uint32_t (&r)[32], int lo_rel, int hi_rel)
{
    if (!kMask) {
        float m0 = fmaxf(__uint_as_float(r[0]), __uint_as_float(r[1]));
        float m1 = fmaxf(__uint_as_float(r[2]), __uint_as_float(r[3]));
#pragma unroll
        for (int e = 4; e < 32; e += 4) {
            m0 = max3(m0, __uint_as_float(r[e]), __uint_as_float(r[e + 1]));
            m1 = max3(m1, __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
        }
        return fmaxf(m0, m1);
    }
    float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const float y = e < hi_rel && (!kLo || e >= lo_rel) ? __uint_as_float(r[e]) : -CUDART_INF_F;
        m4[e & 3] = fmaxf(m4[e & 3], y);
    }
    return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}

// acc0 += the bf16 in the low half of pk, acc1 += the one in the high half (exact
// bf16 values widened to fp32 inside the add).
__device__ __forceinline__ void add_bf16_pair(float &acc0, float &acc1, uint32_t pk)
{
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1) : "r"(pk));
}

// Weights exp2(S * scale * log2 e - mx) of one 32-key chunk as bf16 pairs (zero outside
// [lo_rel, hi_rel) when kMask; kLo as for chunk_max); adds the rounded weights to acc
// and, when kLse, the unrounded ones to accx.
template <bool kMask, bool kLse, bool kLo>
__device__ __forceinline__ void chunk_weights(const uint32_t (&r)[32], int lo_rel, int hi_rel, uint64_t mul2,
                                              uint64_t sub2, uint32_t (&pk)[16], float (&acc)[4], uint64_t &accx)
{
#pragma unroll
    for (int e2 = 0; e2 < 16; ++e2) {
        float a0, a1;
        unf2(fma2(f2(__uint_as_float(r[2 * e2]), __uint_as_float(r[2 * e2 + 1])), mul2, sub2), a0, a1);
        if (kMask) {
            a0 = 2 * e2 < hi_rel && (!kLo || 2 * e2 >= lo_rel) ? a0 : -CUDART_INF_F;
            a1 = 2 * e2 + 1 < hi_rel && (!kLo || 2 * e2 + 1 >= lo_rel) ? a1 : -CUDART_INF_F;
        }
        const float e0 = ex2(a0), e1 = ex2(a1);
        if (kLse) accx = add2(accx, f2(e0, e1));
        pk[e2] = pack_bf16x2(e0, e1);
        add_bf16_pair(acc[(2 * e2) & 3], acc[(2 * e2 + 1) & 3], pk[e2]);
    }
}

// 160 threads: warps 0-3 own one query row each per thread (TMEM lane = row); warp 4
// issues the copies, allocates TMEM and issues the MMAs.
constexpr int kRowThreads = kRows;
constexpr int kThreads = kRows + 32;
constexpr int kCtlWarp = 4;
constexpr int kMaxChunks = kResidentMaxKeys / 32;

// kLong: heads with more than 192 keys (S and O overlap in TMEM; two CTAs per SM at
// most by their 256 columns, so the row threads may hold two chunks of weights).
// kLse: the launch writes each row's log-sum-exp; kWin: the launch has a restricted-
// attention window (each compiled apart, so that the launches without them carry none
// of their arithmetic).
template <bool kLong, bool kLse, bool kWin>
__global__ void __launch_bounds__(kThreads, kLong ? 2 : 4)
attn_resident_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k64,
                     const __grid_constant__ CUtensorMap tm_k16, const __grid_constant__ CUtensorMap tm_v64,
                     const __grid_constant__ CUtensorMap tm_v16, const __grid_constant__ CUtensorMap tm_o32,
                     const ResidentParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *q_s = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t *k_s = q_s + kQBytes;
    uint8_t *v_s = k_s + p.kv_cap * kRowBytes;
    Ctl &c = *reinterpret_cast<Ctl *>(v_s + p.kv_cap * kRowBytes);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    // the query tiles of one head are neighbours in the grid (they read the same K, V)
    const int bh = blockIdx.x / p.q_tiles;
    const int q0 = (blockIdx.x % p.q_tiles) * kRows;
    const int rows = min(kRows, p.m - q0); // query rows of this tile
    int *ab = &c.abort_flag;

    if (tid == kCtlWarp * 32) {
        mbar_init(&c.qk_full, 1);
        mbar_init(&c.v_full, 1);
        mbar_init(&c.s_full, 1);
        for (int ch = 0; ch < kMaxChunks; ++ch)
            mbar_init(&c.p_full[ch], kRowThreads + (ch == 0 && p.withhold_p_arrival ? 1 : 0));
        mbar_init(&c.o_full, 1);
        mbar_init(&c.drain, 1);
        c.abort_flag = 0;
        fence_mbarrier_init();
    } else if (tid == kCtlWarp * 32 + 1) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_k64);
        tma_prefetch_map(&tm_k16);
        tma_prefetch_map(&tm_v64);
        tma_prefetch_map(&tm_v16);
        tma_prefetch_map(&tm_o32);
    }
    __syncthreads(); // barriers initialised
    // The next grid on the stream may launch now, once every CTA of this one has
    // started: its CTAs take free slots and wait for this grid to complete, so its
    // launch and set-up overlap this grid's work.  (It allocates no TMEM before this
    // grid completes, so no CTA here can be left waiting for columns it holds.)
    grid_launch_dependents();
    // Above: set-up only.  Below: reads and writes of global memory and TMEM, which
    // must follow the completion of the grid this one depends on (a no-op for an
    // ordinary launch).
    grid_dependency_wait();

    int len = p.n;
    if ((p.mask_kind & kMaskKeyPadding) && p.key_lengths != nullptr) {
        len = __ldg(p.key_lengths + bh / p.h);
        len = len < 0 ? 0 : (len > p.n ? p.n : len);
    }
    const bool causal = (p.mask_kind & kMaskCausal) != 0;
    int need = causal ? min(len, q0 + rows) : len; // keys some row of the tile may see
    if (kWin) need = min(need, q0 + rows + p.window);
    // key rows loaded and multiplied: whole 16-row boxes, at least one (an empty head
    // still runs the same steps on a box of real, finite keys and writes zeros)
    const int kv_rows = max(kKeyBox, (need + kKeyBox - 1) / kKeyBox * kKeyBox);
    const int nch = (kv_rows + 31) / 32; // 32-column chunks of scores
    // TMEM: S in [0, kv_rows); P (bf16 pairs) over [0, kv_rows / 2), chunk by chunk as
    // S is read; O after S, so that P V starts on the first chunks while later ones are
    // still being read.  Up to 64 keys: 128 columns (four CTAs compute per SM), else 256.
    // Above 192 keys O lies over S chunks 6 and 7: pass 2 takes their weights first.
    const uint32_t tmem_cols = kv_rows <= 64 ? 128u : 256u;
    const uint32_t col_o = kv_rows <= 64 ? 64u : 192u;
    const int held_lo = kLong && kv_rows > kShortKeys ? kShortKeys / 32 : nch; // first chunk under O
    const uint64_t lim = p.wait_ns;

    if (warp == kCtlWarp) {
        // Q and K first (the scores need them), then V, in large then small boxes; one
        // lane posts the bytes, then one lane issues each copy (a TMA issue costs tens of
        // cycles: a few large boxes load a head sooner)
        const int big = kv_rows / kKeyBoxBig, small = (kv_rows % kKeyBoxBig) / kKeyBox; // <= 3 each
        if (lane == 0) {
            mbar_arrive_expect_tx(&c.qk_full, kQBytes + kv_rows * kRowBytes);
            mbar_arrive_expect_tx(&c.v_full, kv_rows * kRowBytes);
        }
        __syncwarp();
        const int r0 = lane < big ? lane * kKeyBoxBig : big * kKeyBoxBig + (lane - big) * kKeyBox;
        if (lane < big) tma_load_3d(k_s + r0 * kRowBytes, &tm_k64, &c.qk_full, 0, r0, bh);
        else if (lane < big + small) tma_load_3d(k_s + r0 * kRowBytes, &tm_k16, &c.qk_full, 0, r0, bh);
        if (lane == 31) tma_load_3d(q_s, &tm_q, &c.qk_full, 0, q0, bh);
        __syncwarp();
        if (lane < big) tma_load_3d(v_s + r0 * kRowBytes, &tm_v64, &c.v_full, 0, r0, bh);
        else if (lane < big + small) tma_load_3d(v_s + r0 * kRowBytes, &tm_v16, &c.v_full, 0, r0, bh);
        __syncwarp();
        // may wait until other CTAs on this SM free their columns; the loads are in flight
        tmem_alloc(&c.tmem_base, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c.tmem_base;

    bool ok = true;
    if (warp == kCtlWarp) {
        if (lane == 0) {
            // ---- S = Q K^T
            ok = wait_poll(&c.qk_full, 0, ab, lim, kSiteQK);
            if (ok) {
                tc_fence_after();
                const uint32_t hi = static_cast<uint32_t>(smem_desc_sw128(0, 0, 1024) >> 32);
                const uint32_t q_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(q_s), 16, 1024));
                const uint32_t k_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(k_s), 16, 1024));
                const uint32_t idesc = idesc_bf16_f32(kRows, kv_rows, 0, 0);
                // 16 bf16 of the head dimension per step = 32 bytes along the swizzled rows
                mma_ss_k<0, 0>(tmem, q_lo, k_lo, hi, idesc, 0u);
                mma_ss_k<2, 2>(tmem, q_lo, k_lo, hi, idesc, 1u);
                mma_ss_k<4, 4>(tmem, q_lo, k_lo, hi, idesc, 1u);
                mma_ss_k<6, 6>(tmem, q_lo, k_lo, hi, idesc, 1u);
                mma_commit(&c.s_full);
            }
            // ---- O = P V: keys 16kk .. 16kk+15 per step: P columns 8kk .. (two bf16 per
            // column), V rows 16kk .. (2 KiB = 128 descriptor units)
            const int steps = kv_rows / 16;
            const uint32_t hi_w = static_cast<uint32_t>(smem_desc_sw128(0, 0, 1024) >> 32);
            const uint32_t v_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(v_s), kQBytes, 1024));
            ok = ok && wait_poll(&c.v_full, 0, ab, lim, kSiteV);
            for (int ch = 0; ch < nch && ok; ++ch) {
                ok = wait_poll(&c.p_full[ch], 0, ab, lim, kSiteP);
                if (!ok) break;
                tc_fence_after();
                for (int kk = 2 * ch; kk < min(2 * ch + 2, steps); ++kk)
                    mma_ts(tmem + col_o, tmem + 8 * kk, make_desc(v_lo + 128u * kk, hi_w), kIdescPV,
                           kk > 0 ? 1u : 0u);
            }
            if (ok) mma_commit(&c.o_full);
        }
        __syncwarp();
    } else {
        // ---- softmax of query row `row` (TMEM lane tid) over keys [lo, hi)
        const int row = q0 + tid;
        const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        int hi = causal ? min(len, row + 1) : len;
        int lo = 0;
        if (kWin) {
            hi = min(hi, row + p.window + 1);
            lo = row - p.window;
        }
        const float sl2 = p.scale_log2;
        const bool warp_live = warp * 32 < rows; // rows past m are never stored
        // the row threads' waits depend on the MMA issuer's, so they get twice its limit:
        // when something stalls, the first wait to run out is the one that names it
        ok = wait_poll(&c.s_full, 0, ab, 2 * lim, kSiteS);
        ok = __all_sync(0xffffffffu, ok);
        // chunks [c_lo, c_hi) hold an allowed key of some row of this warp; a chunk inside
        // [lo_max, hi_min) is allowed whole for every row of it (no mask arithmetic)
        const int c_hi = warp_live ? (__reduce_max_sync(0xffffffffu, hi) + 31) / 32 : 0;
        const int c_lo = kWin && warp_live ? max(0, __reduce_min_sync(0xffffffffu, lo)) / 32 : 0;
        const int hi_min = __reduce_min_sync(0xffffffffu, hi), lo_max = kWin ? __reduce_max_sync(0xffffffffu, lo) : 0;
        constexpr bool want_lse = kLse;
        float mraw = -CUDART_INF_F;
        float acc[4] = {0.f, 0.f, 0.f, 0.f}; // rounded weights: the output's divisor
        uint64_t accx = f2(0.f, 0.f);        // weights before rounding: the log-sum-exp
        if (ok) {
            tc_fence_after();
            // pass 1: row maximum of the raw scores over the allowed columns (scaled after:
            // scaling by a non-negative number keeps the order, and a zero scale must not
            // meet a masked -inf).  A chunk allowed whole for the warp takes the maximum
            // the load computes; a masked one takes it over its allowed columns.
            for (int ch = c_lo; ch < c_hi; ++ch) {
                uint32_t r[32];
                float cm;
                tmem_ld32_max(t_row + 32 * ch, r, cm);
                tmem_wait_ld();
                asm volatile("" : "+f"(cm)::"memory"); // cm is read after the wait
                if (!(32 * ch >= lo_max && 32 * ch + 32 <= hi_min)) {
                    reg_fence32(r);
                    cm = chunk_max<true, kWin>(r, lo - 32 * ch, hi - 32 * ch);
                }
                mraw = fmaxf(mraw, cm);
            }
        }
        const float mx = mraw == -CUDART_INF_F ? -CUDART_INF_F : mraw * sl2;
        const float msub = mx == -CUDART_INF_F ? 0.f : mx;
        const uint64_t mul2 = f2(sl2, sl2), sub2 = f2(-msub, -msub);
        // pass 2: bf16 pairs over the start of S (chunk ch to columns [16 ch, 16 ch + 16),
        // which only chunks this thread has already read occupied); each chunk is handed to
        // the MMA issuer as soon as every row has stored it
        auto weights_of = [&](int ch, uint32_t (&pk)[16]) {
            if (ch >= c_lo && ch < c_hi) {
                uint32_t r[32];
                tmem_ld32(t_row + 32 * ch, r);
                tmem_wait_ld();
                reg_fence32(r);
                const bool mk = !(32 * ch >= lo_max && 32 * ch + 32 <= hi_min);
                if (mk) chunk_weights<true, kLse, kWin>(r, lo - 32 * ch, hi - 32 * ch, mul2, sub2, pk, acc, accx);
                else chunk_weights<false, kLse, kWin>(r, lo - 32 * ch, hi - 32 * ch, mul2, sub2, pk, acc, accx);
            } else {
#pragma unroll
                for (int e2 = 0; e2 < 16; ++e2) pk[e2] = 0u;
            }
        };
        // Above 192 keys O lies over S chunks 6 and 7: their weights are taken first and
        // held in registers.  They are stored after the other chunks, into the columns of
        // S chunk 3, which this thread has read by then.  The first P V, which writes O,
        // follows chunk 0, which every row hands over only after reading chunks 6 and 7.
        uint32_t held[2][16];
        if (kLong && ok) {
#pragma unroll
            for (int hc = 0; hc < 2; ++hc)
                if (held_lo + hc < nch) weights_of(held_lo + hc, held[hc]);
        }
        for (int ch = 0; ch < nch; ++ch) {
            if (ok) {
                uint32_t pk[16];
                if (kLong && ch >= held_lo) {
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) pk[e2] = ch == held_lo ? held[0][e2] : held[1][e2];
                } else {
                    weights_of(ch, pk);
                }
                tmem_st16(t_row + 16 * ch, pk);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&c.p_full[ch]);
        }
        const float l = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        float s0, s1;
        unf2(accx, s0, s1);
        const float lx = s0 + s1;

        // ---- epilogue: O / l in bf16; each warp stages its 32 rows in its quarter of the
        // Q buffer (the S MMA, its last reader, is done) and stores them with one TMA copy
        ok = ok && wait_poll(&c.o_full, 0, ab, 2 * lim, kSiteO);
        ok = __all_sync(0xffffffffu, ok);
        uint32_t o[kD];
        if (ok) {
            tc_fence_after();
            tmem_ld32(t_row + col_o, o);
            tmem_ld32(t_row + col_o + 32, o + 32);
            tmem_wait_ld();
            reg_fence32(o);
            reg_fence32(o + 32);
        }
        tc_fence_before();
        if (ok && warp_live) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            if (want_lse && row < p.m) // the weights are exp2(y - mx): lse = (mx + log2 sum) ln 2
                p.lse[static_cast<size_t>(bh) * p.m + row] =
                    lx > 0.f ? (mx + __log2f(lx)) * 0.6931471805599453f : -CUDART_INF_F;
            // 128-byte swizzle: 16-byte chunk k of row r at chunk k ^ (r % 8) (conflict-free)
            const uint32_t stage_row = smem_addr(q_s) + tid * kRowBytes;
#pragma unroll
            for (int k8 = 0; k8 < kD / 8; ++k8) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(o[8 * k8 + 0]) * inv, __uint_as_float(o[8 * k8 + 1]) * inv);
                v.y = pack_bf16x2(__uint_as_float(o[8 * k8 + 2]) * inv, __uint_as_float(o[8 * k8 + 3]) * inv);
                v.z = pack_bf16x2(__uint_as_float(o[8 * k8 + 4]) * inv, __uint_as_float(o[8 * k8 + 5]) * inv);
                v.w = pack_bf16x2(__uint_as_float(o[8 * k8 + 6]) * inv, __uint_as_float(o[8 * k8 + 7]) * inv);
                st_shared_v4(stage_row + ((k8 ^ (tid & 7)) << 4), v);
            }
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
                // rows past m and columns past d are clipped by the copy
                tma_store_3d(&tm_o32, q_s + warp * 32 * kRowBytes, 0, q0 + warp * 32, bh);
                bulk_commit_group();
                bulk_wait_read_all(); // the staging rows must stay valid until the copy has read them
            }
        }
    }
    __syncthreads(); // every TMEM access of the CTA is done (or abandoned)
    if (warp == kCtlWarp) {
        if (*reinterpret_cast<volatile int *>(ab) != 0 && lane == 0) {
            // nothing asynchronous may still write shared memory or TMEM
            mma_commit(&c.drain);
            drain_wait(&c.drain, 0);
            drain_wait(&c.qk_full, 0);
            drain_wait(&c.v_full, 0);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

struct DeviceInfo {
    bool configured = false;
};

template <bool kLong, bool kLse, bool kWin>
const void *variant_fn()
{
    return reinterpret_cast<const void *>(attn_resident_kernel<kLong, kLse, kWin>);
}

size_t smem_bytes(int kv_cap) { return 1024 + kQBytes + 2u * kv_cap * (kD * 2) + sizeof(Ctl); }

} // namespace

bool resident_fits(int m, int n, int d) { return m >= 1 && n <= kResidentMaxKeys && d % 8 == 0 && d <= kD; }

cudaError_t launch_resident(const Problem &pb, cudaStream_t stream, const ResidentTestHook *hook)
{
    static DeviceInfo infos[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!pb.bf16 || !resident_fits(pb.m, pb.n, pb.d)) return cudaErrorInvalidValue;
    {
        std::lock_guard<std::mutex> lock(mu);
        DeviceInfo &di = infos[dev];
        if (!di.configured) {
            const struct {
                const void *fn;
                size_t bytes;
            } fns[8] = {{variant_fn<false, false, false>(), smem_bytes(kShortKeys)},
                        {variant_fn<false, false, true>(), smem_bytes(kShortKeys)},
                        {variant_fn<false, true, false>(), smem_bytes(kShortKeys)},
                        {variant_fn<false, true, true>(), smem_bytes(kShortKeys)},
                        {variant_fn<true, false, false>(), smem_bytes(kResidentMaxKeys)},
                        {variant_fn<true, false, true>(), smem_bytes(kResidentMaxKeys)},
                        {variant_fn<true, true, false>(), smem_bytes(kResidentMaxKeys)},
                        {variant_fn<true, true, true>(), smem_bytes(kResidentMaxKeys)}};
            for (const auto &f : fns)
                if ((e = cudaFuncSetAttribute(f.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(f.bytes))) != cudaSuccess)
                    return e;
            di.configured = true;
        }
    }
    const int BH = pb.B * pb.h;
    const int kv_cap = (pb.n + kKeyBox - 1) / kKeyBox * kKeyBox;
    // rows of d elements in 64-wide boxes: columns d .. 63 of a load read as zero and a
    // store writes only columns below d; rows past m (queries) or n (keys) read as zero
    CUtensorMap tq, tk64, tk16, tv64, tv16, to32;
    if (!encode_bf16_3d(&tq, pb.q, pb.d, pb.m, BH, kRows) || !encode_bf16_3d(&tk64, pb.k, pb.d, pb.n, BH, kKeyBoxBig) ||
        !encode_bf16_3d(&tk16, pb.k, pb.d, pb.n, BH, kKeyBox) ||
        !encode_bf16_3d(&tv64, pb.v, pb.d, pb.n, BH, kKeyBoxBig) || !encode_bf16_3d(&tv16, pb.v, pb.d, pb.n, BH, kKeyBox) ||
        !encode_bf16_3d(&to32, pb.out, pb.d, pb.m, BH, 32))
        return cudaErrorInvalidValue;
    ResidentParams p;
    p.key_lengths = (pb.mask_kind & kMaskKeyPadding) ? pb.key_lengths : nullptr;
    p.lse = pb.lse;
    p.h = pb.h;
    p.m = pb.m;
    p.q_tiles = (pb.m + kRows - 1) / kRows;
    p.n = pb.n;
    p.mask_kind = pb.mask_kind;
    p.window = (pb.mask_kind & kMaskWindow) ? pb.window : -1;
    p.kv_cap = kv_cap;
    p.scale_log2 = pb.scale * 1.4426950408889634f;
    p.wait_ns = hook != nullptr ? hook->wait_ns : kDefaultWaitNs;
    p.withhold_p_arrival = hook != nullptr ? hook->withhold_p_arrival : 0;
    cudaLaunchConfig_t cfg = {};
    const long long ctas = static_cast<long long>(BH) * p.q_tiles;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes(kv_cap);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pb.overlap_launch ? 1 : 0;
    const void *fn = kv_cap > kShortKeys ? (p.lse ? (p.window >= 0 ? variant_fn<true, true, true>() : variant_fn<true, true, false>())
                                                  : (p.window >= 0 ? variant_fn<true, false, true>() : variant_fn<true, false, false>()))
                                         : (p.lse ? (p.window >= 0 ? variant_fn<false, true, true>() : variant_fn<false, true, false>())
                                                  : (p.window >= 0 ? variant_fn<false, false, true>() : variant_fn<false, false, false>()));
    void *args[] = {&tq, &tk64, &tk16, &tv64, &tv16, &to32, &p};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t resident_status_read_and_clear(cudaStream_t stream, uint32_t *code, uint32_t *info)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned int c = 0, i = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&c, g_resident_status_code, sizeof c)) != cudaSuccess) return e;
    if ((e = cudaMemcpyFromSymbol(&i, g_resident_status_info, sizeof i)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_resident_status_code, &zero, sizeof zero)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_resident_status_info, &zero, sizeof zero)) != cudaSuccess) return e;
    *code = c;
    *info = i;
    return cudaSuccess;
}

} // namespace attn
