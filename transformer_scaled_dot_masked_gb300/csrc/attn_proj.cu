// Projections of multi-head attention on tcgen05: the W^Q, W^K, W^V products
// that split the model width into heads, and the W^O product over the
// concatenated heads ("Paper Deep Reading: Attention Is All You Need", §04
// MultiHead equation: head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V),
// MultiHead = Concat(head_1, ..., head_h) W^O; no bias terms).
//
// Clusters of two CTAs (CTA pairs) walk 256 x 256 tiles of D = A B, persistent, one
// pair per co-resident cluster slot (a last tile of 128 columns when N is an odd
// multiple of 128).  Per 16 of K one tcgen05 MMA of M = 256 spans the pair: the first
// CTA issues it, each CTA holds 128 rows of the A tile and half of the B columns in
// its shared memory and its 128 rows of D (fp32) in its TMEM.  One launch may hold up
// to three products of the same shape (the W^Q, W^K and W^V products, whose row
// counts may differ): their tiles form one list, so the three share the pipeline
// fill and the last wave:
//   kProjIn   A = rows t0 .. t0+255 of x[b] ([B][L][K], K = d_model), B = columns
//             n0 .. n0+255 of W ([K][h*64]); each 64-column block of the tile is one
//             head, stored straight into the head-split layout [B*h][L][64] (the
//             per-head W_i are column blocks of W).
//   kProjOut  A = the heads' outputs [B*h][L][64]: the 64-wide K step j reads head
//             j, so Concat needs no copy; B = columns n0 .. n0+255 of W^O
//             ([h*64][N]); the tile goes to out[b] ([B][L][N]).
// A tiles are K-major (64 bf16 = one 128-byte swizzle row per tile row); B tiles
// are 64 x 64 MN-major blocks side by side (the descriptor's leading offset is the
// distance between them).  A 6-stage TMA ring of 32 KiB per CTA feeds 4 MMAs per
// 64-wide K step; each CTA's loads signal the first CTA's barrier, and each MMA
// group's commit reaches both CTAs.  Two 256-column TMEM accumulators alternate
// between tiles, so the epilogue of one tile (bf16 through per-warp swizzled
// staging slots, TMA stores, rows past L clipped) runs while the next tile
// accumulates.
//
// Warps: 0 TMA producer, 1 MMA issuer (first CTA) and TMEM owner, 2-5 epilogue.
// Every mbarrier wait is bounded and reports through this file's status word.
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

// A CTA pair (a cluster of two) computes 256 x 256 tiles of D with one M = 256 MMA
// per K step: each CTA holds 128 rows of the A tile and 128 of the 256 B columns in
// its shared memory, and its 128 rows of D in its TMEM.  A K step is 32 KiB of
// shared memory per CTA instead of 48 KiB for a 128 x 256 tile on one CTA, so a
// six-stage ring fits and hides twice the L2 latency.
constexpr int kTM = 128, kPairM = 256, kTN = 256, kTK = 64; // rows per CTA, per pair; columns; K step
constexpr int kStages = 6;
constexpr int kThreads = 192;
constexpr uint32_t kATile = kTM * kTK * 2;    // 16 KiB
constexpr uint32_t kBBlock = kTK * 64 * 2;    // 8 KiB: 64 K rows x 64 N columns
constexpr uint32_t kTmemCols = 512;           // two 256-column accumulators
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint16_t kBothCtas = 0x3;
constexpr uint32_t kEpilogueWarps = 4;

struct alignas(1024) ProjSmem {
    uint8_t a[kStages][kATile];
    uint8_t b[kStages][2][kBBlock]; // this CTA's half of the B columns: up to two 64-column blocks
    // output staging: per epilogue warp, two slots of its 32 rows x 64 columns (bf16,
    // 128-byte swizzle) used in turn
    uint8_t stage[kEpilogueWarps][2][32 * 64 * 2];
    uint64_t full[kStages];         // first CTA: both CTAs' bytes of a stage have landed
    uint64_t empty[kStages];        // each CTA: the pair's MMAs have read its stage
    uint64_t acc_full[2];           // each CTA: accumulator a holds a finished tile
    uint64_t acc_empty[2];          // first CTA: both CTAs' epilogues have read accumulator a
    uint64_t drain;
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
        if (global_timer_ns() - start > kWaitLimitNs / 10) return;
}

constexpr int kMaxProblems = 3; // the W^Q, W^K, W^V products of one layer in one launch

// Tensor maps of the launch's products: A, W and the output of product i.
struct ProjMaps {
    CUtensorMap a[kMaxProblems], w[kMaxProblems], out[kMaxProblems];
};

struct ProjParams {
    int mode, h, K, N, B, problems;
    int dk; // head width: a head is dk / 64 blocks of 64 columns
    int L[kMaxProblems];       // rows per batch entry of product i
    int m_tiles[kMaxProblems]; // 256-row pair tiles per batch entry of product i
    int tiles_of[kMaxProblems];
    int n_tiles, tiles;
};

struct TileId {
    int pi, b, t0, n0, ncols, L; // pi: product; t0: the pair tile's first row; ncols: 256, or 128 for a last half tile
};

// Tiles are numbered product by product; selects instead of indexing the
// parameter arrays with a run-time value.
__device__ __forceinline__ TileId tile_id(const ProjParams &p, int t)
{
    TileId id;
    id.pi = 0;
    if (p.problems > 1 && t >= p.tiles_of[0]) {
        t -= p.tiles_of[0];
        id.pi = 1;
        if (p.problems > 2 && t >= p.tiles_of[1]) {
            t -= p.tiles_of[1];
            id.pi = 2;
        }
    }
    const int mt = id.pi == 0 ? p.m_tiles[0] : (id.pi == 1 ? p.m_tiles[1] : p.m_tiles[2]);
    id.L = id.pi == 0 ? p.L[0] : (id.pi == 1 ? p.L[1] : p.L[2]);
    const int nt = t % p.n_tiles, mi = t / p.n_tiles;
    id.b = mi / mt;
    id.t0 = (mi % mt) * kPairM;
    id.n0 = nt * kTN;
    id.ncols = min(kTN, p.N - id.n0);
    return id;
}

__device__ __forceinline__ const CUtensorMap *pick(const CUtensorMap (&m)[kMaxProblems], int pi)
{
    return pi == 0 ? &m[0] : (pi == 1 ? &m[1] : &m[2]);
}

__global__ void __launch_bounds__(kThreads, 1)
attn_proj_kernel(const __grid_constant__ ProjMaps maps, const ProjParams p)
{
    extern __shared__ uint8_t smem_raw[];
    ProjSmem &sm = *reinterpret_cast<ProjSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                 ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32;
    const int ksteps = p.K / kTK;
    const uint32_t rank = cluster_ctarank(); // 0: the pair's first CTA, which issues the MMAs
    const int pair = blockIdx.x / 2, pairs = gridDim.x / 2;
    int *ab = &sm.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sm.acc_full[a], 1);
            mbar_init(&sm.acc_empty[a], 2 * kEpilogueWarps);
        }
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbarrier_init();
    }
    // Set-up above overlaps the previous kernel's tail when launched as its programmatic
    // dependent.  Nothing below may read what that kernel writes before it completes,
    // and TMEM is allocated only after it has completed: a kernel that let this one
    // launch early may still have CTAs waiting for columns.  Every CTA of this
    // (persistent) grid is resident, so the next grid may launch now: its CTAs take SMs
    // as this grid's leave and wait for it to complete.
    grid_launch_dependents();
    grid_dependency_wait();
    if (warp == 1) {
        tmem_alloc_pair(&sm.tmem_base, kTmemCols); // one warp of each CTA of the pair, together
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    // both CTAs' barriers are initialised before either signals the other's
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        if (threadIdx.x == 0) {
            for (int pi = 0; pi < p.problems; ++pi) {
                tma_prefetch_map(pick(maps.a, pi));
                tma_prefetch_map(pick(maps.w, pi));
            }
            uint32_t kc = 0, issued = 0;
            bool ok = true;
            for (int t = pair; t < p.tiles && ok; t += pairs) {
                const TileId id = tile_id(p, t);
                const int blocks = id.ncols / 128; // 64-column blocks of B in each CTA
                const int row0 = id.t0 + kTM * static_cast<int>(rank);
                const int col0 = id.n0 + (id.ncols / 2) * static_cast<int>(rank);
                const CUtensorMap *tm_a = pick(maps.a, id.pi), *tm_w = pick(maps.w, id.pi);
                for (int kk = 0; kk < ksteps; ++kk, ++kc) {
                    const uint32_t s = kc % kStages;
                    if (!(ok = wait_bar(&sm.empty[s], ((kc / kStages) & 1) ^ 1, ab, 1))) break;
                    // the first CTA's barrier counts both CTAs' bytes (rows past L arrive
                    // zero-filled and count too)
                    const uint32_t full_bar = map_shared_rank(smem_addr(&sm.full[s]), 0);
                    if (rank == 0) mbar_arrive_expect_tx(&sm.full[s], 2 * (kATile + blocks * kBBlock));
                    if (p.mode == kProjIn)
                        tma_load_3d_pair(sm.a[s], tm_a, full_bar, kk * kTK, row0, id.b);
                    else // K step kk: columns 64 (kk % (dk / 64)) .. of head kk / (dk / 64)
                        tma_load_3d_pair(sm.a[s], tm_a, full_bar, (kk % (p.dk / 64)) * 64, row0,
                                         id.b * p.h + kk / (p.dk / 64));
                    // W as a 3-D tensor with one outer slice
                    for (int q = 0; q < blocks; ++q)
                        tma_load_3d_pair(sm.b[s][q], tm_w, full_bar, col0 + 64 * q, kk * kTK, 0);
                    ++issued;
                }
            }
            // every stage this CTA loaded has been read by the pair's MMAs (each
            // completes one phase of this CTA's empty barrier) before the CTA leaves
            for (uint32_t c = issued > kStages ? issued - kStages : 0; c < issued; ++c)
                drain_wait(&sm.empty[c % kStages], (c / kStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (threadIdx.x == 32 && rank == 0) {
            const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(0, 0, 1024) >> 32);
            const uint32_t a_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.a[0]), 16, 1024));
            // B operands: 64-column blocks kBBlock apart (the leading offset)
            const uint32_t b_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.b[0][0]), kBBlock, 1024));
            uint32_t kc = 0;
            bool ok = true;
            int i = 0;
            for (int t = pair; t < p.tiles && ok; t += pairs, ++i) {
                const TileId id = tile_id(p, t);
                const int a = i & 1;
                // both epilogues have read this accumulator's previous tile
                if (!(ok = wait_bar(&sm.acc_empty[a], ((i >> 1) & 1) ^ 1, ab, 2))) break;
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(kPairM, id.ncols, 0, 1); // A K-major, B MN-major
                for (int kk = 0; kk < ksteps; ++kk, ++kc) {
                    const uint32_t s = kc % kStages;
                    if (!(ok = wait_bar(&sm.full[s], (kc / kStages) & 1, ab, 3))) break;
                    tc_fence_after();
                    const uint32_t ad = a_lo + s * (kATile >> 4);
                    const uint32_t bd = b_lo + s * 2 * (kBBlock >> 4);
                    const uint32_t d = tmem + 256 * a;
                    // A: 16 bf16 of K per step = 32 bytes; B: K rows 16kk.. = 2 KiB per step
                    mma_ss_k_pair<0, 0>(d, ad, bd, desc_hi, idesc, kk > 0 ? 1u : 0u);
                    mma_ss_k_pair<2, 128>(d, ad, bd, desc_hi, idesc, 1u);
                    mma_ss_k_pair<4, 256>(d, ad, bd, desc_hi, idesc, 1u);
                    mma_ss_k_pair<6, 384>(d, ad, bd, desc_hi, idesc, 1u);
                    mma_commit_pair(&sm.empty[s], kBothCtas);
                }
                if (ok) mma_commit_pair(&sm.acc_full[a], kBothCtas);
            }
            if (!ok) {
                // make sure no MMA is still writing TMEM when the pair frees it
                mma_commit_pair(&sm.drain, 0x1);
                drain_wait(&sm.drain, 0);
            }
        }
        __syncwarp();
    } else {
        // epilogue: warp w owns rows 32 (w % 4) .. +31 of this CTA's half of the tile
        // (its TMEM lane quadrant; thread = row).  Each 64-column block of its rows goes
        // through one of the warp's two staging slots in turn and out with one TMA
        // store issued by lane 0; a slot is rewritten once lane 0's store of the block
        // before last has read it.  No barrier spans more than one warp.
        const int quad = warp % 4, lane = threadIdx.x % 32;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        bool ok = true;
        int i = 0;
        uint32_t stored = 0; // blocks this warp has staged so far
        for (int t = pair; t < p.tiles && ok; t += pairs, ++i) {
            const TileId id = tile_id(p, t);
            const int a = i & 1;
            const int row0 = id.t0 + kTM * static_cast<int>(rank) + 32 * quad;
            ok = __all_sync(0xffffffffu, wait_bar(&sm.acc_full[a], (i >> 1) & 1, ab, 4));
            if (!ok) break;
            tc_fence_after();
            const CUtensorMap *tm_out = pick(maps.out, id.pi);
            const int blocks = id.ncols / 64;
            for (int q = 0; q < blocks; ++q, ++stored) {
                uint32_t v[64];
                tmem_ld64(tmem + lane_base + 256 * a + 64 * q, v);
                tmem_wait_ld();
                reg_fence32(v);
                reg_fence32(v + 32);
                if (q == blocks - 1) {
                    // the accumulator is free for the tile after next (one arrival per
                    // warp, on the first CTA's barrier)
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(map_shared_rank(smem_addr(&sm.acc_empty[a]), 0));
                }
                uint8_t *slot = sm.stage[quad][stored & 1];
                // each block's store is its own group: all but the latest have read their
                // source, the one that last used this slot included
                if (lane == 0) bulk_wait_read_1();
                __syncwarp();
                const uint32_t row = smem_addr(slot) + lane * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1]));
                    w.y = pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3]));
                    w.z = pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5]));
                    w.w = pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7]));
                    st_shared_v4(row + ((c ^ (lane & 7)) << 4), w);
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    // rows past L are clipped by the copy; a slot wholly past L is not stored
                    if (row0 < id.L) {
                        if (p.mode == kProjIn) // column c of the product: head c / dk, column c % dk of it
                            tma_store_3d(tm_out, slot, (id.n0 + 64 * q) % p.dk, row0,
                                         id.b * p.h + (id.n0 + 64 * q) / p.dk);
                        else
                            tma_store_3d(tm_out, slot, id.n0 + 64 * q, row0, id.b);
                    }
                    bulk_commit_group();
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    // neither CTA leaves, or frees the pair's columns, while the other may still read
    // its shared memory or signal its barriers
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

constexpr size_t kSmemBytes = sizeof(ProjSmem) + 1024;

} // namespace

cudaError_t launch_proj_multi(const ProjProblem *pps, int count, cudaStream_t stream)
{
    static int max_pairs[64] = {}; // co-resident CTA pairs per device, found once
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (max_pairs[dev] == 0) {
            if ((e = cudaFuncSetAttribute(attn_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(kSmemBytes))) != cudaSuccess)
                return e;
            int sms = 0;
            if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
            cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1));
            int clusters = 0;
            if ((e = cudaOccupancyMaxActiveClusters(&clusters, attn_proj_kernel, &cfg)) != cudaSuccess) return e;
            if (clusters < 1) return cudaErrorInvalidConfiguration;
            max_pairs[dev] = clusters;
        }
    }
    if (count < 1 || count > kMaxProblems) return cudaErrorInvalidValue;
    const ProjProblem &p0 = pps[0];
    if (p0.K % kTK != 0 || p0.N % 128 != 0) return cudaErrorInvalidValue;
    ProjMaps maps;
    ProjParams p;
    p.mode = p0.mode;
    p.h = p0.h;
    // dk: the head width, or for a plain product (h = 1) the whole output width
    if (p0.dk % 64 != 0 || p0.dk <= 0 || (p0.mode == kProjIn ? p0.N : p0.K) % p0.dk != 0) return cudaErrorInvalidValue;
    p.K = p0.K;
    p.N = p0.N;
    p.B = p0.B;
    p.dk = p0.dk;
    p.problems = count;
    p.n_tiles = (p0.N + kTN - 1) / kTN;
    p.tiles = 0;
    const int BH = p0.B * p0.h;
    for (int i = 0; i < kMaxProblems; ++i) {
        p.L[i] = 0;
        p.m_tiles[i] = 0;
        p.tiles_of[i] = 0;
    }
    for (int i = 0; i < count; ++i) {
        const ProjProblem &pp = pps[i];
        // one launch runs products of one shape: only the row count may differ
        if (pp.mode != p0.mode || pp.B != p0.B || pp.h != p0.h || pp.K != p0.K || pp.N != p0.N || pp.dk != p0.dk)
            return cudaErrorInvalidValue;
        bool enc;
        if (pp.mode == kProjIn) {
            enc = encode_bf16_3d(&maps.a[i], pp.a, pp.K, pp.L, pp.B, kTM) &&
                  encode_bf16_3d(&maps.out[i], pp.out, pp.dk, pp.L, BH, 32);
        } else {
            enc = encode_bf16_3d(&maps.a[i], pp.a, pp.dk, pp.L, BH, kTM) &&
                  encode_bf16_3d(&maps.out[i], pp.out, pp.N, pp.L, pp.B, 32);
        }
        // W [K][N] as a 3-D tensor with one outer slice: 64 x 64 boxes
        enc = enc && encode_bf16_3d(&maps.w[i], pp.w, pp.N, pp.K, 1, kTK);
        if (!enc) return cudaErrorInvalidValue;
        p.L[i] = pp.L;
        p.m_tiles[i] = (pp.L + kPairM - 1) / kPairM;
        p.tiles_of[i] = p.n_tiles * p.m_tiles[i] * pp.B;
        p.tiles += p.tiles_of[i];
    }
    for (int i = count; i < kMaxProblems; ++i) {
        maps.a[i] = maps.a[0];
        maps.w[i] = maps.w[0];
        maps.out[i] = maps.out[0];
    }
    if (p.tiles == 0) return cudaSuccess;
    // persistent: one CTA pair per co-resident cluster slot, at most one per tile
    const int pairs = p.tiles < max_pairs[dev] ? p.tiles : max_pairs[dev];
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.numAttrs = p0.overlap_launch ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, attn_proj_kernel, maps, p);
}

cudaError_t launch_proj(const ProjProblem &pp, cudaStream_t stream) { return launch_proj_multi(&pp, 1, stream); }

namespace {

// Between the concatenated layout [B][L][h][dk] and the head-split layout [B][h][L][dk],
// 16 bytes per thread (dk a multiple of 8): chunk c of head hh of row t of batch b.
__global__ void attn_heads_copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int L, int h,
                                       int dk8, size_t total, int split)
{
    const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const size_t c = idx % dk8;
    size_t rest = idx / dk8;
    const size_t hh = rest % h;
    rest /= h;
    const size_t t = rest % L, b = rest / L;
    const size_t heads = ((b * h + hh) * L + t) * dk8 + c; // idx is the concatenated position
    if (split) dst[heads] = src[idx];
    else dst[idx] = src[heads];
}

} // namespace

cudaError_t launch_heads_copy(const void *src, void *dst, int B, int L, int h, int dk, bool split,
                              cudaStream_t stream)
{
    if (dk % 8 != 0 || dk <= 0) return cudaErrorInvalidValue;
    const size_t total = static_cast<size_t>(B) * L * h * (dk / 8);
    if (total == 0) return cudaSuccess;
    const unsigned blocks = static_cast<unsigned>((total + 255) / 256);
    attn_heads_copy_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), L,
                                                        h, dk / 8, total, split ? 1 : 0);
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
