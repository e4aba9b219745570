// Fused masked scaled dot-product attention for sm_103a: TMA + tcgen05 + TMEM.
//
// What it computes is softmax(scale * Q K^T + M) V per (batch, head)
// ("Paper Deep Reading: Attention Is All You Need", §04 attention equation;
// M from §03 "Decoder layer" and §04), one 128-key tile at a time with an
// online softmax, so no score matrix larger than one tile ever exists.
//
// CTA organisation (persistent: one CTA per SM; CTA tiles dealt to CTAs in snake order)
//   warps 0-3  softmax group of slot 0 (thread t owns query row t of the slot)
//   warps 4-7  softmax group of slot 1
//   warp 8     TMA producer (one lane): Q tiles, then K/V tiles into a 4-stage ring
//   warp 9     MMA issuer of slot 0 (one lane) + TMEM allocation for the CTA
//   warp 10    MMA issuer of slot 1 (one lane), on another SM sub-partition
//   warp 11    idle: it completes the third warpgroup so that setmaxnreg can
//              move registers from it to the softmax warpgroups (200 each, vs 104)
// A CTA tile has two slots of 128 query rows each:
//   pair mode   two consecutive query tiles of one head; each K/V stage feeds both
//   split mode  query tile 0 of two different heads (m <= 128: the whole head's
//               queries, keys and values are resident at once)
//
// TMEM (512 columns, fp32 unless noted), per slot s at column 256*s:
//   S [0,128)   scores of the current key tile, Q K^T
//   P [128,192) exp2 weights as packed bf16 pairs: the A operand of the PV MMA
//   O [192,256) output accumulator
//
// Per key tile j of a slot:
//   MMA:     S = Q K_j^T                       (4 x tcgen05.mma M128 N128 K16, both K-major)
//   softmax: read S, mask (boundary tiles only), P = exp2(S * scale * log2 e - r)
//            against a per-row reference r, row sum, write P as bf16.  r is the
//            row max of the row's first key tile; later tiles keep r and check
//            the tile's row sum instead of taking a max (sum <= 2^15 bounds
//            every weight).  A larger sum moves r up by an integer k and scales
//            the weights by 2^-k exactly; an overflowed one recomputes the row's
//            scores and takes their max.  O and the running sum stay exact
//            multiples of the true ones and are rescaled only when r moves.
//   MMA:     O += P V_j                        (8 x tcgen05.mma M128 N64 K16, A from TMEM, V MN-major)
// Key tiles wholly beyond the causal diagonal or the padded length are never
// loaded or computed.  The epilogue divides O by the row sum (0 for a row with
// no allowed key) and writes the bf16 tile through shared memory with a TMA store.
//
// Every mbarrier wait is bounded (kWaitLimitNs).  A wait that runs out sets a
// shared abort flag and the device status word; all roles then leave their
// loops, wait (bounded) for their own asynchronous copies and MMAs, and the
// CTA frees its TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "softmax_tile.cuh"

namespace attn {

// Device status word: code (bit 0 = a bounded wait gave up) and info (which wait).
__device__ unsigned int g_flash_status_code;
__device__ unsigned int g_flash_status_info;

namespace {

constexpr int kBM = 128;   // query rows per slot
constexpr int kBN = 128;   // keys per key tile
constexpr int kD = 64;     // head width
constexpr int kSlots = 2;
constexpr int kStages = 4; // K/V ring depth
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;  // MMA issuer of slot 0; allocates and frees TMEM
constexpr int kMma1Warp = 10; // MMA issuer of slot 1
constexpr int kThreads = 384;           // three full warpgroups
constexpr uint32_t kSoftmaxRegs = 200;  // per thread, softmax warpgroups (setmaxnreg; spill-free)
constexpr uint32_t kControlRegs = 104;  // per thread, producer/MMA warpgroup
static_assert(2 * kSoftmaxRegs + kControlRegs <= 3 * 168, "register split exceeds the launch allocation");
constexpr uint32_t kTileBytes = kBM * kD * 2; // one 128 x 64 bf16 tile = 16 KiB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSlotCols = 256;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192;
constexpr int kTileRing = 4;              // CTA tile indices handed from the loader to the other roles
constexpr uint32_t kTileConsumers = 2 + 2 * 128; // two MMA issuers, two softmax warpgroups
constexpr uint64_t kWaitLimitNs = 2000000000ull; // 2 s
constexpr uint64_t kDrainLimitNs = 200000000ull; // 0.2 s

constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0, 0); // Q (K-major) x K^T (K-major)
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kD, 0, 1); // P (TMEM) x V (MN-major)

// Where a wait gave up (reported through the status word's info).
enum WaitSite : uint32_t {
    kSiteLoadQEmpty = 1, kSiteLoadKvEmpty, kSiteMmaQFull, kSiteMmaKvFull, kSiteMmaSFree,
    kSiteMmaPFull, kSiteMmaOFree, kSiteSmSFull, kSiteSmPvDone, kSiteSmPvLast, kSiteTileEmpty, kSiteTileFull,
    kSiteSmStageFree, kSiteSmStageFull
};

struct alignas(1024) SharedStorage {
    uint8_t q[kSlots][kTileBytes];
    uint8_t k[kStages][kTileBytes];
    uint8_t v[kStages][kTileBytes];
    uint8_t o_stage[kSlots][kTileBytes]; // output tile of each slot, SW128 layout, read by a TMA store
    uint64_t q_full[kSlots], q_empty[kSlots];
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[kSlots], s_free[kSlots], p_full[kSlots], pv_done[kSlots], o_free[kSlots];
    uint64_t drain[kSlots];
    uint64_t stage_free[kSlots], stage_full[kSlots]; // o_stage may be written / may be stored
    uint64_t tile_full[kTileRing], tile_empty[kTileRing];
    int tile_ring[kTileRing];
    uint32_t tmem_base;
    int abort_flag;
};

struct FlashParams {
    const __nv_bfloat16 *q, *k; // read only by the rare score recomputation
    const int32_t *key_lengths;
    __nv_bfloat16 *out;
    float *lse; // per-row log-sum-exp of the scaled scores (natural log), or nullptr
    int window; // restricted attention: keys with |i - j| <= window stay; -1: no window
    int BH, h, m, n, mask_kind;
    float scale_log2;
    int pair_mode;
    int num_tiles;
    int q_pairs;        // pair mode: query-tile pairs per head
    int group_heads;    // pair mode: heads per group of the tile order (their K and V share L2)
    int *tile_counter;  // [0] next tile to claim, [1] CTAs done; nullptr: static snake schedule
    int d;              // head width in memory (a multiple of 8, <= 64): narrower heads enter
                        // the 64-wide tiles zero-padded by the TMA loads and leave clipped by the store
};

struct Tile {
    int bh[kSlots];
    int q0[kSlots];
    int kv_len[kSlots]; // keys allowed by padding (n without padding)
    int kv_lo[kSlots];  // first key tile to process (0 without a window)
    int n_kv[kSlots];   // end of the key tiles to process (n_kv <= kv_lo: nothing allowed or slot unused)
    bool active[kSlots];
    bool shared_kv;
};

// The t-th CTA tile this CTA processes in round r: rounds walk the heaviest-first
// tile order, alternating direction (CTA c takes position c of even rounds and
// position G-1-c of odd rounds), which evens out the causal work per CTA (the
// heaviest and lightest tiles of consecutive rounds land on the same CTA).
__device__ __forceinline__ int tile_of(int r)
{
    const int k = (r & 1) ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
    return r * static_cast<int>(gridDim.x) + k;
}

// Sequence of CTA tiles one role of this CTA processes.  Static schedule: the
// snake order above.  Dynamic schedule (a zeroed counter in global memory): the
// loader claims the next tile of the heaviest-first order with an atomic add
// when it is about to load it, and hands the index to the MMA issuers and the
// softmax warpgroups through a small ring in shared memory, so CTAs on faster
// SMs simply take more tiles.  -1 ends the sequence.
struct TileFeed {
    uint32_t k = 0;

    __device__ __forceinline__ int produce(SharedStorage &sm, const FlashParams &p, bool &ok);
    __device__ __forceinline__ int consume(SharedStorage &sm, const FlashParams &p, bool &ok, bool warp_wide);
};

__device__ __forceinline__ Tile decode_tile(const FlashParams &p, int t)
{
    Tile T;
    if (p.pair_mode) {
        // Heads are taken in groups whose keys and values fit in L2 together; within a
        // group, heaviest pair first (with a causal mask later query tiles see more keys),
        // so the CTAs working at one time share a group's K and V through L2.
        const int per_group = p.group_heads * p.q_pairs;
        const int g = t / per_group, r = t - g * per_group;
        const int heads = min(p.group_heads, p.BH - g * p.group_heads); // the last group may be short
        const int pair = p.q_pairs - 1 - r / heads;
        const int bh = g * p.group_heads + r % heads;
        T.bh[0] = T.bh[1] = bh;
        T.q0[0] = pair * 2 * kBM;
        T.q0[1] = pair * 2 * kBM + kBM;
        T.shared_kv = true;
    } else {
        T.bh[0] = 2 * t;
        T.bh[1] = 2 * t + 1;
        T.q0[0] = T.q0[1] = 0;
        T.shared_kv = false;
    }
    const bool causal = (p.mask_kind & kMaskCausal) != 0;
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        T.active[s] = T.bh[s] < p.BH && T.q0[s] < p.m;
        T.kv_len[s] = 0;
        T.kv_lo[s] = 0;
        T.n_kv[s] = 0;
        if (!T.active[s]) continue;
        int len = p.n;
        if ((p.mask_kind & kMaskKeyPadding) && p.key_lengths != nullptr) {
            len = __ldg(p.key_lengths + T.bh[s] / p.h);
            len = len < 0 ? 0 : (len > p.n ? p.n : len);
        }
        int lim = causal ? min(len, T.q0[s] + kBM) : len;
        int lo = 0;
        if (p.window >= 0) {
            // keys within `window` of some row q0 .. min(m, q0 + 128) - 1 of the tile
            lo = max(0, T.q0[s] - p.window) / kBN;
            lim = min(lim, min(p.m, T.q0[s] + kBM) + p.window);
        }
        T.kv_len[s] = len;
        T.kv_lo[s] = lo;
        T.n_kv[s] = max(lo, (lim + kBN - 1) / kBN);
    }
    return T;
}

__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, int *abort_flag, uint32_t site)
{
    const uint64_t start = global_timer_ns();
    while (true) {
        for (int k = 0; k < 64; ++k)
            if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int *>(abort_flag)) return false;
        if (global_timer_ns() - start > kWaitLimitNs) {
            *reinterpret_cast<volatile int *>(abort_flag) = 1;
            atomicOr(&g_flash_status_code, 1u);
            atomicCAS(&g_flash_status_info, 0u, site);
            return false;
        }
    }
}

// Bounded wait for phase `parity` of `bar` to complete.  false: gave up (or another role did).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, int *abort_flag, uint32_t site)
{
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    return wait_slow(a, parity, abort_flag, site);
}

// Bounded wait that ignores the abort flag (used to drain in-flight work on the way out).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint32_t a = smem_addr(bar);
    const uint64_t start = global_timer_ns();
    while (!mbar_try_wait(a, parity))
        if (global_timer_ns() - start > kDrainLimitNs) return;
}

__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

// Loader side (one thread): claim the next tile and publish it to the ring.
__device__ __forceinline__ int TileFeed::produce(SharedStorage &sm, const FlashParams &p, bool &ok)
{
    if (p.tile_counter == nullptr) {
        const int t = tile_of(static_cast<int>(k++));
        return t < p.num_tiles ? t : -1;
    }
    int t = atomicAdd(p.tile_counter, 1);
    if (t >= p.num_tiles) t = -1;
    const uint32_t slot = k % kTileRing;
    ok = wait_bar(&sm.tile_empty[slot], ((k / kTileRing) & 1) ^ 1, &sm.abort_flag, kSiteTileEmpty);
    if (!ok) return -1;
    sm.tile_ring[slot] = t;
    mbar_arrive(&sm.tile_full[slot]); // release: the index is visible to whoever sees the phase
    ++k;
    return t;
}

// Consumer side: every thread of a consuming group reads the index and arrives.
__device__ __forceinline__ int TileFeed::consume(SharedStorage &sm, const FlashParams &p, bool &ok, bool warp_wide)
{
    if (p.tile_counter == nullptr) {
        const int t = tile_of(static_cast<int>(k++));
        return t < p.num_tiles ? t : -1;
    }
    const uint32_t slot = k % kTileRing;
    bool got = wait_bar(&sm.tile_full[slot], (k / kTileRing) & 1, &sm.abort_flag, kSiteTileFull);
    if (warp_wide) got = warp_all(got);
    ok = got;
    if (!ok) return -1;
    const int t = *reinterpret_cast<volatile int *>(&sm.tile_ring[slot]);
    mbar_arrive(&sm.tile_empty[slot]);
    ++k;
    return t;
}

// K/V stage rings.  Pair mode: one ring of kStages stages, one fill per key
// tile, read by both slots.  Split mode: each slot owns a ring of kStages / 2
// stages holding its own head's key tiles.  Every thread that waits on a
// stage's kv_full barrier thus sees each of that stage's phases in order, so a
// parity wait can never be satisfied by a phase two fills away.
struct StagePos {
    uint32_t st;    // stage index
    uint32_t phase; // parity of the fill
};

__device__ __forceinline__ StagePos ring_pos(bool pair_mode, int ring, uint32_t fill)
{
    if (pair_mode) return {fill % kStages, (fill / kStages) & 1u};
    constexpr uint32_t kHalf = kStages / 2;
    return {static_cast<uint32_t>(ring) * kHalf + fill % kHalf, (fill / kHalf) & 1u};
}

// Pair mode: the key tiles loaded for the CTA tile, [shared_lo, shared_hi): the
// union of the two slots' ranges (a slot with nothing to do adds nothing).
__device__ __forceinline__ int shared_lo(const Tile &T)
{
    const bool e0 = T.n_kv[0] <= T.kv_lo[0], e1 = T.n_kv[1] <= T.kv_lo[1];
    return e0 ? (e1 ? 0 : T.kv_lo[1]) : (e1 ? T.kv_lo[0] : min(T.kv_lo[0], T.kv_lo[1]));
}

__device__ __forceinline__ int shared_hi(const Tile &T)
{
    const bool e0 = T.n_kv[0] <= T.kv_lo[0], e1 = T.n_kv[1] <= T.kv_lo[1];
    return e0 ? (e1 ? 0 : T.n_kv[1]) : (e1 ? T.n_kv[0] : max(T.n_kv[0], T.n_kv[1]));
}

// Fills of slot s's ring that CTA tile T takes.
__device__ __forceinline__ uint32_t fills_of(const Tile &T, int s)
{
    // selects, not T.n_kv[s]: a runtime index would put the tile on the stack
    if (T.shared_kv) return static_cast<uint32_t>(shared_hi(T) - shared_lo(T));
    return static_cast<uint32_t>(s ? T.n_kv[1] - T.kv_lo[1] : T.n_kv[0] - T.kv_lo[0]);
}

// ------------------------------------------------------------------ roles
__device__ __forceinline__ void load_role(SharedStorage &sm, const FlashParams &p, const CUtensorMap *tm_q,
                                          const CUtensorMap *tm_k, const CUtensorMap *tm_v)
{
    tma_prefetch_map(tm_q);
    tma_prefetch_map(tm_k);
    tma_prefetch_map(tm_v);
    uint32_t q_cnt[kSlots] = {0, 0};
    uint32_t fill0 = 0, fill1 = 0; // fills of ring 0 and ring 1 (pair mode uses ring 0 only)
    bool ok = true;
    TileFeed feed;
    while (ok) {
        const int t = feed.produce(sm, p, ok);
        if (t < 0) break;
        const Tile T = decode_tile(p, t);
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
            if (T.n_kv[s] <= T.kv_lo[s]) continue;
            if (!(ok = wait_bar(&sm.q_empty[s], (q_cnt[s] & 1) ^ 1, &sm.abort_flag, kSiteLoadQEmpty))) break;
            mbar_arrive_expect_tx(&sm.q_full[s], kTileBytes);
            tma_load_3d(sm.q[s], tm_q, &sm.q_full[s], 0, T.q0[s], T.bh[s]);
            ++q_cnt[s];
        }
        // pair mode: each key tile of the union once (both slots read it); split mode:
        // each slot's own range into its own ring, the slots interleaved
        const int J0 = T.shared_kv ? shared_lo(T) : min(T.kv_lo[0], T.kv_lo[1]);
        const int J = T.shared_kv ? shared_hi(T) : max(T.n_kv[0], T.n_kv[1]);
        for (int j = J0; j < J && ok; ++j) {
#pragma unroll
            for (int s = 0; s < kSlots; ++s) {
                if (T.shared_kv ? s == 1 : (j < T.kv_lo[s] || j >= T.n_kv[s])) continue;
                const int ring = T.shared_kv ? 0 : s;
                const StagePos sp = ring_pos(p.pair_mode, ring, ring ? fill1 : fill0);
                if (!(ok = wait_bar(&sm.kv_empty[sp.st], sp.phase ^ 1, &sm.abort_flag, kSiteLoadKvEmpty))) break;
                mbar_arrive_expect_tx(&sm.kv_full[sp.st], 2 * kTileBytes);
                tma_load_3d(sm.k[sp.st], tm_k, &sm.kv_full[sp.st], 0, j * kBN, T.bh[s]);
                tma_load_3d(sm.v[sp.st], tm_v, &sm.kv_full[sp.st], 0, j * kBN, T.bh[s]);
                if (ring) ++fill1; else ++fill0;
            }
        }
    }
    // Tail: every stage and Q buffer must be released (its last copy landed and
    // the MMAs reading it completed) before the CTA may exit.
    for (int ring = 0; ring < (p.pair_mode ? 1 : kSlots); ++ring) {
        // the last fill of each stage that was used at all
        const uint32_t depth = p.pair_mode ? kStages : kStages / 2;
        const uint32_t fills = ring ? fill1 : fill0;
        for (uint32_t f = fills > depth ? fills - depth : 0; f < fills; ++f) {
            const StagePos sp = ring_pos(p.pair_mode, ring, f);
            if (ok) {
                wait_bar(&sm.kv_empty[sp.st], sp.phase, &sm.abort_flag, kSiteLoadKvEmpty);
            } else {
                drain_wait(&sm.kv_full[sp.st], sp.phase);
            }
        }
    }
    for (int s = 0; s < kSlots; ++s) {
        if (q_cnt[s] == 0) continue;
        if (ok) {
            wait_bar(&sm.q_empty[s], (q_cnt[s] - 1) & 1, &sm.abort_flag, kSiteLoadQEmpty);
        } else {
            drain_wait(&sm.q_full[s], (q_cnt[s] - 1) & 1);
        }
    }
}

// MMA issuer of one slot (one lane of its own warp): S_s(j) = Q_s K_j^T as soon
// as the softmax has read S_s(j-1), and O_s += P_s(j-1) V_(j-1) as soon as P is
// written.  Each slot has its own issuing thread so that neither slot's P V
// waits behind the other's in one thread's program order.  A K/V stage shared by
// both slots (pair mode) is released when both issuers have arrived on its
// kv_empty barrier (count 2): after their P V completes, or, for a slot that
// does not read that stage, once the stage is loaded (so the arrival can only
// count towards the stage's current fill).  Descriptors are computed once.
__device__ __forceinline__ void mma_role(SharedStorage &sm, const FlashParams &p, uint32_t tmem, int s)
{
    uint32_t q_cnt = 0, s_cnt = 0, p_cnt = 0, o_cnt = 0;
    uint32_t fill_base = 0; // fills of this slot's ring before the current CTA tile
    bool ok = true;
    int *ab = &sm.abort_flag;
    uint64_t *q_full = &sm.q_full[s], *q_empty = &sm.q_empty[s], *s_full = &sm.s_full[s];
    uint64_t *s_free = &sm.s_free[s], *p_full = &sm.p_full[s], *pv_done = &sm.pv_done[s], *o_free = &sm.o_free[s];
    const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(0, 0, 1024) >> 32);
    const uint32_t q_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.q[s]), 16, 1024));
    const uint32_t k_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.k[0]), 16, 1024));
    const uint32_t v_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.v[0]), kTileBytes, 1024));
    const uint32_t s_tmem = tmem + s * kSlotCols + kColS;
    const uint32_t p_tmem = tmem + s * kSlotCols + kColP;
    const uint32_t o_tmem = tmem + s * kSlotCols + kColO;
    TileFeed feed;
    while (ok) {
        const int t = feed.consume(sm, p, ok, false);
        if (t < 0) break;
        const Tile T = decode_tile(p, t);
        const int lo = s ? T.kv_lo[1] : T.kv_lo[0];
        const int n = max(0, (s ? T.n_kv[1] : T.n_kv[0]) - lo);
        // fill of this slot's first key tile; pair mode: stages of the union that
        // precede this slot's range are only acknowledged (below)
        const int J0 = T.shared_kv ? shared_lo(T) : lo;
        if (n > 0) {
            ok = wait_bar(q_full, q_cnt & 1, ab, kSiteMmaQFull);
            ++q_cnt;
        }
        if (ok && T.shared_kv) {
            for (int j = J0; j < lo && ok && n > 0; ++j) {
                const StagePos sp = ring_pos(p.pair_mode, s, fill_base + static_cast<uint32_t>(j - J0));
                ok = wait_bar(&sm.kv_full[sp.st], sp.phase, ab, kSiteMmaKvFull);
                if (ok) mbar_arrive(&sm.kv_empty[sp.st]);
            }
        }
        const uint32_t own_base = fill_base + static_cast<uint32_t>(n > 0 ? lo - J0 : 0);
        for (int j = 0; j <= n && ok; ++j) {
            if (j < n) {
                // S(j)
                const StagePos sp = ring_pos(p.pair_mode, s, own_base + j);
                ok = wait_bar(&sm.kv_full[sp.st], sp.phase, ab, kSiteMmaKvFull);
                if (ok) ok = wait_bar(s_free, (s_cnt & 1) ^ 1, ab, kSiteMmaSFree);
                if (!ok) break;
                tc_fence_after();
                const uint32_t kd = k_lo + sp.st * (kTileBytes >> 4);
                // 16 bf16 of K per step = 32 bytes (2 descriptor units) along the swizzled rows
                mma_ss_k<0, 0>(s_tmem, q_lo, kd, desc_hi, kIdescS, 0u);
                mma_ss_k<2, 2>(s_tmem, q_lo, kd, desc_hi, kIdescS, 1u);
                mma_ss_k<4, 4>(s_tmem, q_lo, kd, desc_hi, kIdescS, 1u);
                mma_ss_k<6, 6>(s_tmem, q_lo, kd, desc_hi, kIdescS, 1u);
                mma_commit(s_full);
                ++s_cnt;
                if (j == n - 1) mma_commit(q_empty);
            }
            if (j >= 1) {
                // P V(j - 1)
                const int jp = j - 1;
                ok = wait_bar(p_full, p_cnt & 1, ab, kSiteMmaPFull);
                if (!ok) break;
                ++p_cnt;
                tc_fence_after();
                if (jp == 0) {
                    // the first P V of a tile overwrites O: the previous epilogue must have read it
                    ok = wait_bar(o_free, (o_cnt & 1) ^ 1, ab, kSiteMmaOFree);
                    if (!ok) break;
                    ++o_cnt;
                    tc_fence_after();
                }
                const uint32_t st = ring_pos(p.pair_mode, s, own_base + jp).st;
                const uint32_t vd = v_lo + st * (kTileBytes >> 4);
                // keys 16kk..16kk+15 per step: P columns 8kk.. (two bf16 per column), V rows
                // 16kk.. (2 KiB = 128 descriptor units)
                const uint32_t acc0 = jp > 0 ? 1u : 0u;
                mma_ts_k<0, 0>(o_tmem, p_tmem, vd, desc_hi, kIdescPV, acc0);
                mma_ts_k<8, 128>(o_tmem, p_tmem, vd, desc_hi, kIdescPV, 1u);
                mma_ts_k<16, 256>(o_tmem, p_tmem, vd, desc_hi, kIdescPV, 1u);
                mma_ts_k<24, 384>(o_tmem, p_tmem, vd, desc_hi, kIdescPV, 1u);
                mma_ts_k<32, 512>(o_tmem, p_tmem, vd, desc_hi, kIdescPV, 1u);
                mma_ts_k<40, 640>(o_tmem, p_tmem, vd, desc_hi, kIdescPV, 1u);
                mma_ts_k<48, 768>(o_tmem, p_tmem, vd, desc_hi, kIdescPV, 1u);
                mma_ts_k<56, 896>(o_tmem, p_tmem, vd, desc_hi, kIdescPV, 1u);
                mma_commit(pv_done);
                mma_commit(&sm.kv_empty[st]);
            }
        }
        if (ok && T.shared_kv) {
            // stages of this CTA tile that only the other slot reads: arrive once each
            // is loaded (in fill order: after this slot's own range, or all of them
            // when this slot has nothing to do)
            const int J = shared_hi(T);
            for (int j = n > 0 ? lo + n : J0; j < J && ok; ++j) {
                const StagePos sp = ring_pos(p.pair_mode, s, fill_base + static_cast<uint32_t>(j - J0));
                ok = wait_bar(&sm.kv_full[sp.st], sp.phase, ab, kSiteMmaKvFull);
                if (ok) mbar_arrive(&sm.kv_empty[sp.st]);
            }
        }
        fill_base += fills_of(T, s);
    }
    if (!ok) {
        // make sure no MMA is still writing TMEM when the CTA frees it
        mma_commit(&sm.drain[s]);
        drain_wait(&sm.drain[s], 0);
    }
}

// Scores of query row i of head bh against keys key0 .. key0+127, recomputed on
// the CUDA cores from Q and K in global memory (fp32 sums of exact bf16
// products), multiplied by scale * log2 e, and -inf where not allowed (column c
// is allowed iff cnt_lo <= c < cnt; allowed keys are below n).  Rows past m read as zero
// queries, as the TMA loads fill them.  Taken only when a tile's exponentials
// against the running reference overflowed, so it favours size over speed.
template <bool kNarrow>
__device__ __forceinline__ void recompute_scores(const FlashParams &p, int bh, int i, int key0, int cnt_lo,
                                                 int cnt, float (&x)[kBN])
{
    const bool row_in = i < p.m;
    const int width = kNarrow ? p.d : kD; // elements per row in memory
    const __nv_bfloat16 *qr = p.q + (static_cast<size_t>(bh) * p.m + (row_in ? i : 0)) * width;
    float q[kD];
#pragma unroll
    for (int d = 0; d < kD; ++d) {
        if (kNarrow) {
            q[d] = 0.f;
            if (row_in && d < width) q[d] = __bfloat162float(qr[d]);
        } else {
            q[d] = row_in ? __bfloat162float(qr[d]) : 0.f;
        }
    }
    float srow[kBN];
#pragma unroll 1
    for (int c = 0; c < kBN; ++c) {
        float v = -CUDART_INF_F;
        if (c < cnt && c >= cnt_lo) {
            const __nv_bfloat16 *kr = p.k + (static_cast<size_t>(bh) * p.n + key0 + c) * width;
            float a = 0.f;
#pragma unroll
            for (int d = 0; d < kD; ++d)
                if (!kNarrow || d < width) a = fmaf(q[d], __bfloat162float(kr[d]), a);
            v = a * p.scale_log2;
        }
        srow[c] = v;
    }
#pragma unroll
    for (int c = 0; c < kBN; ++c) x[c] = srow[c];
}

// kWindow: the launch has a restricted-attention window (compiled separately so
// that launches without one run none of its bound arithmetic).
template <bool kWindow, bool kNarrow>
__device__ __forceinline__ void softmax_role(SharedStorage &sm, const FlashParams &p, const CUtensorMap *tm_o,
                                             uint32_t tmem, int slot)
{
    const int warp_in_group = (threadIdx.x / 32) % 4; // TMEM lane quadrant this warp may access
    const int row = warp_in_group * 32 + (threadIdx.x % 32);
    const uint32_t lane_base = static_cast<uint32_t>(warp_in_group * 32) << 16;
    const uint32_t t_s = tmem + lane_base + slot * kSlotCols + kColS;
    const uint32_t t_p = tmem + lane_base + slot * kSlotCols + kColP;
    const uint32_t t_o = tmem + lane_base + slot * kSlotCols + kColO;
    const bool causal = (p.mask_kind & kMaskCausal) != 0;
    const int win = kWindow ? p.window : -1;
    const float sl2 = p.scale_log2;
    int *ab = &sm.abort_flag;
    uint32_t s_cnt = 0, pv_cnt = 0, epi_cnt = 0;
    bool ok = true;
    if (row == 0) tma_prefetch_map(tm_o);
    const uint32_t stage_row = smem_addr(sm.o_stage[slot]) + row * (kD * 2);

    TileFeed feed;
    while (ok) {
        const int t = feed.consume(sm, p, ok, true);
        if (t < 0) break;
        const Tile T = decode_tile(p, t);
        // select this slot's fields without indexing the per-slot arrays at run time
        const bool active = slot ? T.active[1] : T.active[0];
        if (!active) continue;
        const int q0 = slot ? T.q0[1] : T.q0[0];
        const int bh = slot ? T.bh[1] : T.bh[0];
        const int kv_lo = slot ? T.kv_lo[1] : T.kv_lo[0];
        const int n_kv = slot ? T.n_kv[1] : T.n_kv[0];
        const int kv_len = slot ? T.kv_len[1] : T.kv_len[0];
        const int i = q0 + row;
        const int width = kNarrow ? p.d : kD; // elements per row in memory
        __nv_bfloat16 *orow = p.out + (static_cast<size_t>(bh) * p.m + i) * width;
        if (n_kv <= kv_lo) { // no allowed key for any row of this tile: output 0
            if (i < p.m) {
                uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < width / 8; ++c) reinterpret_cast<uint4 *>(orow)[c] = z;
                if (p.lse != nullptr) p.lse[static_cast<size_t>(bh) * p.m + i] = -CUDART_INF_F;
            }
            continue;
        }
        float m_run = -CUDART_INF_F; // running max, log2 units, as used for the exponentials
        float l_run = 0.f;           // running sum of the weights relative to m_run
        for (int j = kv_lo; j < n_kv; ++j) {
            ok = warp_all(wait_bar(&sm.s_full[slot], s_cnt & 1, ab, kSiteSmSFull));
            if (!ok) break;
            ++s_cnt;
            tc_fence_after();
            uint32_t sr[kBN];
#pragma unroll
            tmem_ld128(t_s, sr);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) reg_fence32(sr + c * 32);
            tc_fence_before();
            mbar_arrive(&sm.s_free[slot]); // S may be overwritten by the next Q K^T

            const int key0 = j * kBN;
            // keys allowed for row i are exactly those in one range [lo_i, hi_i): below
            // the padded length (and i + 1 for a causal mask), and within `win` of i
            // for a window; column c of the tile is allowed iff cnt_lo <= c < cnt
            int hi_i = causal ? min(kv_len, i + 1) : kv_len;
            int lo_i = 0;
            if (kWindow) {
                hi_i = min(hi_i, i + win + 1);
                lo_i = i - win;
            }
            const int cnt = hi_i - key0, cnt_lo = lo_i - key0;
            const bool boundary = (key0 + kBN > kv_len) || (causal && key0 + kBN - 1 > q0) ||
                                  (kWindow && (key0 < q0 + kBM - 1 - win || key0 + kBN - 1 > q0 + win));
            float x[kBN];
#pragma unroll
            for (int c = 0; c < kBN; ++c) x[c] = __uint_as_float(sr[c]);
            bool prescaled = boundary; // x already multiplied by scale * log2 e
            if (boundary) {
                // Scale first, then mask: a zero scale must not turn -inf into NaN.  The
                // allowed columns of a row are the range [cnt_lo, cnt) (cnt_lo <= 0
                // without a window).
                if (kWindow) {
                    // two bounds: one bit mask per 32 columns, then one bit test per column
#pragma unroll
                    for (int ch = 0; ch < kBN / 32; ++ch) {
                        const int hi = min(max(cnt - 32 * ch, 0), 32);
                        const int lo = min(max(cnt_lo - 32 * ch, 0), 32);
                        uint32_t m = hi >= 32 ? 0xffffffffu : (1u << hi) - 1u;
                        m &= lo >= 32 ? 0u : ~((1u << lo) - 1u);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            x[32 * ch + e] = (m & (1u << e)) ? x[32 * ch + e] * sl2 : -CUDART_INF_F;
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kBN; ++c) x[c] = c < cnt ? x[c] * sl2 : -CUDART_INF_F;
                }
            }

            // Reference for the exponentials.  The row max is taken only on the row's
            // first key tile; later tiles use the running reference and check the
            // result through the tile's row sum.
            float m_use = m_run, alpha = 1.f;
            bool grow = false;
            const bool first = m_run == -CUDART_INF_F;
            if (first) move_reference(x, prescaled, sl2, m_run, m_use, alpha, grow);
            uint32_t pk[kBN / 2];
            float tile_sum = weights_bf16(x, prescaled, sl2, m_use, pk);
            if (!first && !(tile_sum <= kFastSumLimit)) {
                float f = 1.f;
                if (tile_sum < CUDART_INF_F) {
                    // Finite but large: scale the weights by f = 2^-k (k an integer, so
                    // the bf16 values scale exactly) and move the reference up by k.
                    const int k = ((__float_as_int(tile_sum) >> 23) & 0xff) - 127 - 7; // 8..120
                    f = __int_as_float((127 - k) << 23);                               // 2^-k
                    alpha = f;
                    m_use = m_run + static_cast<float>(k);
                    grow = true;
                } else {
                    // Some weight overflowed (the scores grew by 128 or more in log2
                    // units, or are not finite).  The scores have left the registers:
                    // recompute this row's from Q and K, already scaled and masked,
                    // and take their max.
                    recompute_scores<kNarrow>(p, bh, i, key0, cnt_lo, cnt, x);
                    move_reference(x, true, sl2, m_run, m_use, alpha, grow);
                    weights_bf16(x, true, sl2, m_use, pk);
                }
                // Such a tile holds a key far above the row's reference, likely the
                // row's dominant one: its weights enter the row sum as rounded, the
                // values P V applies (the log-sum-exp then carries their rounding,
                // at most 2^-8 relative, on these rows alone).
                tile_sum = scale_and_sum(pk, f);
            }
            if (j > kv_lo) {
                // P and O are still in use by the previous P V until it completes;
                // waiting only now lets the exponentials above overlap with it
                ok = warp_all(wait_bar(&sm.pv_done[slot], pv_cnt & 1, ab, kSiteSmPvDone));
                if (!ok) break;
                ++pv_cnt;
                tc_fence_after();
            }
            if (j > kv_lo && __any_sync(0xffffffffu, grow)) {
                // move O to the new reference (rare: a large tile sum or a recomputation)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t orr[32];
                    tmem_ld32(t_o + 32 * h2, orr);
                    tmem_wait_ld();
                    reg_fence32(orr);
#pragma unroll
                    for (int c = 0; c < 32; ++c) orr[c] = __float_as_uint(__uint_as_float(orr[c]) * alpha);
                    tmem_st32(t_o + 32 * h2, orr);
                }
            }
            tmem_st32(t_p, pk);
            tmem_st32(t_p + 32, pk + 32);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&sm.p_full[slot]);
            l_run = l_run * alpha + tile_sum;
            m_run = m_use;
        }
        if (!ok) break;
        ok = warp_all(wait_bar(&sm.pv_done[slot], pv_cnt & 1, ab, kSiteSmPvLast));
        if (!ok) break;
        ++pv_cnt;
        tc_fence_after();
        uint32_t orr[kD];
        tmem_ld64(t_o, orr);
        tmem_wait_ld();
        reg_fence32(orr);
        reg_fence32(orr + 32);
        tc_fence_before();
        mbar_arrive(&sm.o_free[slot]);
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        if (p.lse != nullptr && i < p.m) // weights are exp2(x - m_run) / l: lse = (m_run + log2 l) ln 2
            p.lse[static_cast<size_t>(bh) * p.m + i] =
                l_run > 0.f ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -CUDART_INF_F;
        // Output: each thread writes its row of O / l into this slot's staging tile in
        // the 128-byte-swizzled layout (16-byte chunk c of row r at chunk c ^ (r % 8):
        // conflict-free), then one thread stores the tile with TMA, which clips rows
        // past m.  The staging tile is rewritten only after the previous store has
        // read it.
        if (row == 0) {
            bulk_wait_read_all();
            mbar_arrive(&sm.stage_free[slot]);
        }
        ok = warp_all(wait_bar(&sm.stage_free[slot], epi_cnt & 1, ab, kSiteSmStageFree));
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < kD / 8; ++c) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(orr[8 * c + 0]) * inv, __uint_as_float(orr[8 * c + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(orr[8 * c + 2]) * inv, __uint_as_float(orr[8 * c + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(orr[8 * c + 4]) * inv, __uint_as_float(orr[8 * c + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(orr[8 * c + 6]) * inv, __uint_as_float(orr[8 * c + 7]) * inv);
            st_shared_v4(stage_row + ((c ^ (row & 7)) << 4), v);
        }
        fence_proxy_async_shared();
        mbar_arrive(&sm.stage_full[slot]);
        if (row == 0) {
            ok = wait_bar(&sm.stage_full[slot], epi_cnt & 1, ab, kSiteSmStageFull);
            if (ok) {
                tma_store_3d(tm_o, sm.o_stage[slot], 0, q0, bh);
                bulk_commit_group();
            }
        }
        ok = warp_all(ok);
        ++epi_cnt;
    }
    // the staging tiles must stay valid, and the output written, until the stores complete
    if (row == 0) bulk_wait_all();
}

// kWindow: compiled separately for launches with a restricted-attention window;
// kNarrow: for heads narrower than 64 (row width read from the parameters).  Each
// kernel holds only the code it runs: its speed depends on instruction fetch (the
// short workloads are dominated by cold first tiles) and on code layout.
template <bool kWindow, bool kNarrow>
__global__ void __launch_bounds__(kThreads, 1)
attn_flash_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FlashParams p)
{
    extern __shared__ uint8_t smem_raw[];
    SharedStorage &sm = *reinterpret_cast<SharedStorage *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&sm.q_full[s], 1);
            mbar_init(&sm.q_empty[s], 1);
            mbar_init(&sm.s_full[s], 1);
            mbar_init(&sm.s_free[s], kBM);
            mbar_init(&sm.p_full[s], kBM);
            mbar_init(&sm.pv_done[s], 1);
            mbar_init(&sm.o_free[s], kBM);
            mbar_init(&sm.stage_free[s], 1);
            mbar_init(&sm.stage_full[s], kBM);
        }
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&sm.kv_full[st], 1);
            mbar_init(&sm.kv_empty[st], p.pair_mode ? 2 : 1); // pair mode: one arrival per slot issuer
        }
        for (int r = 0; r < kTileRing; ++r) {
            mbar_init(&sm.tile_full[r], 1);
            mbar_init(&sm.tile_empty[r], kTileConsumers);
        }
        mbar_init(&sm.drain[0], 1);
        mbar_init(&sm.drain[1], 1);
        sm.abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncwarp();
    // Set-up above overlaps the previous kernel's tail when launched as its programmatic
    // dependent.  Nothing below may read what that kernel writes before it completes,
    // and TMEM is allocated only after it has completed: a kernel that let this one
    // launch early may still have CTAs waiting for columns.
    grid_dependency_wait();
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    // The two register regions never rejoin: each branch ends with its own
    // CTA-wide barrier (every thread arrives exactly once) and returns.
    if (warp < 4 * kSlots) {
        regs_increase<kSoftmaxRegs>();
        softmax_role<kWindow, kNarrow>(sm, p, &tm_o, tmem, warp / 4);
        tc_fence_before();
        __syncthreads();
        return;
    }
    regs_decrease<kControlRegs>();
    if (warp == kLoadWarp) {
        if (threadIdx.x % 32 == 0) load_role(sm, p, &tm_q, &tm_k, &tm_v);
        __syncwarp();
    } else if (warp == kMmaWarp || warp == kMma1Warp) {
        if (threadIdx.x % 32 == 0) mma_role(sm, p, tmem, warp == kMmaWarp ? 0 : 1);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (p.tile_counter != nullptr && threadIdx.x == kLoadWarp * 32) {
        // every claim of this CTA precedes this point; the last CTA to get here
        // returns the counters to zero for the next call that uses the workspace
        __threadfence();
        if (atomicAdd(p.tile_counter + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            atomicExch(p.tile_counter, 0);
            atomicExch(p.tile_counter + 1, 0);
        }
    }
}

// ------------------------------------------------------------------ host side
struct DeviceInfo {
    int sms = 0;
    bool configured = false;
};

constexpr size_t kSmemBytes = sizeof(SharedStorage) + 1024; // + alignment slack

} // namespace

cudaError_t launch_flash(const Problem &pb, bool pair_mode, int *tile_counter, cudaStream_t stream)
{
    static DeviceInfo infos[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        DeviceInfo &di = infos[dev];
        if (!di.configured) {
            if ((e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
            const void *kernels[4] = {reinterpret_cast<const void *>(attn_flash_kernel<false, false>),
                                      reinterpret_cast<const void *>(attn_flash_kernel<true, false>),
                                      reinterpret_cast<const void *>(attn_flash_kernel<false, true>),
                                      reinterpret_cast<const void *>(attn_flash_kernel<true, true>)};
            for (const void *k : kernels)
                if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(kSmemBytes))) != cudaSuccess)
                    return e;
            di.configured = true;
        }
    }
    const int sms = infos[dev].sms;
    const int BH = pb.B * pb.h;
    if (pb.d % 8 != 0 || pb.d < 8 || pb.d > kD) return cudaErrorInvalidValue;
    // rows of d elements in 64-wide, 128-row boxes: columns d .. 63 of a load read as
    // zero, and a store writes only columns below d
    CUtensorMap tq, tk, tv, to;
    if (!encode_bf16_3d(&tq, pb.q, pb.d, pb.m, BH, kBM) || !encode_bf16_3d(&tk, pb.k, pb.d, pb.n, BH, kBN) ||
        !encode_bf16_3d(&tv, pb.v, pb.d, pb.n, BH, kBN) || !encode_bf16_3d(&to, pb.out, pb.d, pb.m, BH, kBM))
        return cudaErrorInvalidValue;
    FlashParams p;
    p.q = static_cast<const __nv_bfloat16 *>(pb.q);
    p.k = static_cast<const __nv_bfloat16 *>(pb.k);
    p.key_lengths = (pb.mask_kind & kMaskKeyPadding) ? pb.key_lengths : nullptr;
    p.out = static_cast<__nv_bfloat16 *>(pb.out);
    p.lse = pb.lse;
    p.window = (pb.mask_kind & kMaskWindow) ? pb.window : -1;
    p.d = pb.d;
    p.BH = BH;
    p.h = pb.h;
    p.m = pb.m;
    p.n = pb.n;
    p.mask_kind = pb.mask_kind;
    p.scale_log2 = pb.scale * 1.4426950408889634f;
    p.pair_mode = pair_mode ? 1 : 0;
    p.q_pairs = (pb.m + 2 * kBM - 1) / (2 * kBM);
    {
        // about 32 MB of keys and values per group: a quarter of L2, leaving room for the
        // query tiles and output tiles streaming through it
        const size_t kv_head = 2ull * pb.n * 64 * 2;
        const size_t g = (32ull << 20) / (kv_head > 0 ? kv_head : 1);
        p.group_heads = static_cast<int>(g < 1 ? 1 : (g > static_cast<size_t>(BH) ? BH : g));
    }
    p.num_tiles = pair_mode ? BH * p.q_pairs : (BH + 1) / 2;
    p.tile_counter = tile_counter;
    const int grid = p.num_tiles < sms ? p.num_tiles : sms;
    // compiled four times: with or without a window, full or narrower heads
    const bool narrow = pb.d != kD;
    auto kernel = p.window >= 0 ? (narrow ? attn_flash_kernel<true, true> : attn_flash_kernel<true, false>)
                                : (narrow ? attn_flash_kernel<false, true> : attn_flash_kernel<false, false>);
    if (!pb.overlap_launch) {
        kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, to, p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, p);
}

cudaError_t flash_status_read_and_clear(cudaStream_t stream, uint32_t *code, uint32_t *info)
{
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned int c = 0, i = 0, zero = 0;
    if ((e = cudaMemcpyFromSymbol(&c, g_flash_status_code, sizeof c)) != cudaSuccess) return e;
    if ((e = cudaMemcpyFromSymbol(&i, g_flash_status_info, sizeof i)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_flash_status_code, &zero, sizeof zero)) != cudaSuccess) return e;
    if ((e = cudaMemcpyToSymbol(g_flash_status_info, &zero, sizeof zero)) != cudaSuccess) return e;
    *code = c;
    *info = i;
    return cudaSuccess;
}

} // namespace attn
