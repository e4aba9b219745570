// Projections of multi-head attention on tcgen05: the W^Q, W^K, W^V products
// that split the model width into heads, and the W^O product over the
// concatenated heads ("Paper Deep Reading: Attention Is All You Need", §04
// MultiHead equation: head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V),
// MultiHead = Concat(head_1, ..., head_h) W^O; no bias terms).
//
// A persistent CTA per SM walks 128 x 256 tiles of D = A B (fp32 accumulation in
// TMEM; a last tile of 128 columns when N is an odd multiple of 128).  One launch
// may hold up to three products of the same shape (the W^Q, W^K and W^V products,
// whose row counts may differ): their tiles form one list, so the three share the
// pipeline fill and the last wave:
//   kProjIn   A = rows t0 .. t0+127 of x[b] ([B][L][K], K = d_model), B = columns
//             n0 .. n0+255 of W ([K][h*64]); each 64-column block of the tile is one
//             head, stored straight into the head-split layout [B*h][L][64] (the
//             per-head W_i are column blocks of W).
//   kProjOut  A = the heads' outputs [B*h][L][64]: the 64-wide K step j reads head
//             j, so Concat needs no copy; B = columns n0 .. n0+255 of W^O
//             ([h*64][N]); the tile goes to out[b] ([B][L][N]).
// A tiles are K-major (64 bf16 = one 128-byte swizzle row per tile row); B tiles
// are 64 x 64 MN-major blocks, two side by side forming each N = 128 operand (the
// descriptor's leading offset is the distance between them).  A 4-stage TMA ring
// feeds 4 x 2 MMAs of M128 N128 K16 per 64-wide K step.  Two 256-column TMEM
// accumulators alternate between tiles, so the epilogue of one tile (bf16 through
// two swizzled shared-memory blocks used in turn, TMA stores, rows past L clipped)
// runs while the next tile accumulates.
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

constexpr int kTM = 128, kTN = 256, kTK = 64; // output tile and K step
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kATile = kTM * kTK * 2;    // 16 KiB
constexpr uint32_t kBBlock = kTK * 64 * 2;    // 8 KiB: 64 K rows x 64 N columns
constexpr uint32_t kTmemCols = 512;           // two 256-column accumulators
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kIdesc = idesc_bf16_f32(kTM, 128, 0, 1); // A K-major, B MN-major, N = 128

struct alignas(1024) ProjSmem {
    uint8_t a[kStages][kATile];
    uint8_t b[kStages][4][kBBlock];
    uint8_t stage[2][kTM * 64 * 2]; // bf16 output blocks of 64 columns, 128-byte swizzle, used in turn
    uint64_t full[kStages], empty[kStages];
    uint64_t acc_full[2], acc_empty[2]; // accumulator a holds a finished tile / may be overwritten
    uint64_t stage_free[2], staged[2];  // staging block j may be rewritten / holds a block to store
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
        if (global_timer_ns() - start > kWaitLimitNs) return;
}

constexpr int kMaxProblems = 3; // the W^Q, W^K, W^V products of one layer in one launch

// Tensor maps of the launch's products: A, W and the output of product i.
struct ProjMaps {
    CUtensorMap a[kMaxProblems], w[kMaxProblems], out[kMaxProblems];
};

struct ProjParams {
    int mode, h, K, N, B, problems;
    int dk; // head width: a head is dk / 64 blocks of 64 columns
    int m_tiles[kMaxProblems]; // 128-row tiles per batch entry of product i
    int tiles_of[kMaxProblems];
    int n_tiles, tiles;
};

struct TileId {
    int pi, b, t0, n0, ncols; // pi: product; ncols: 256, or 128 for a last half tile
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
    const int nt = t % p.n_tiles, mi = t / p.n_tiles;
    id.b = mi / mt;
    id.t0 = (mi % mt) * kTM;
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
    int *ab = &sm.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sm.acc_full[a], 1);
            mbar_init(&sm.acc_empty[a], kTM);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&sm.stage_free[j], 1);
            mbar_init(&sm.staged[j], kTM);
        }
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncwarp();
    // Set-up above overlaps the previous kernel's tail when launched as its programmatic
    // dependent.  Nothing below may read what that kernel writes before it completes,
    // and TMEM is allocated only after it has completed: a kernel that let this one
    // launch early may still have CTAs waiting for columns.
    grid_dependency_wait();
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
            for (int pi = 0; pi < p.problems; ++pi) {
                tma_prefetch_map(pick(maps.a, pi));
                tma_prefetch_map(pick(maps.w, pi));
            }
            uint32_t kc = 0, issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
                const TileId id = tile_id(p, t);
                const int blocks = id.ncols / 64;
                const CUtensorMap *tm_a = pick(maps.a, id.pi), *tm_w = pick(maps.w, id.pi);
                for (int kk = 0; kk < ksteps; ++kk, ++kc) {
                    const uint32_t s = kc % kStages;
                    if (!(ok = wait_bar(&sm.empty[s], ((kc / kStages) & 1) ^ 1, ab, 1))) break;
                    mbar_arrive_expect_tx(&sm.full[s], kATile + blocks * kBBlock);
                    if (p.mode == kProjIn)
                        tma_load_3d(sm.a[s], tm_a, &sm.full[s], kk * kTK, id.t0, id.b);
                    else // K step kk: columns 64 (kk % (dk / 64)) .. of head kk / (dk / 64)
                        tma_load_3d(sm.a[s], tm_a, &sm.full[s], (kk % (p.dk / 64)) * 64, id.t0,
                                    id.b * p.h + kk / (p.dk / 64));
                    // W as a 3-D tensor with one outer slice
                    for (int q = 0; q < blocks; ++q)
                        tma_load_3d(sm.b[s][q], tm_w, &sm.full[s], id.n0 + 64 * q, kk * kTK, 0);
                    ++issued;
                }
            }
            for (uint32_t c = issued > kStages ? issued - kStages : 0; c < issued; ++c)
                drain_wait(&sm.full[c % kStages], (c / kStages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (threadIdx.x == 32) {
            const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(0, 0, 1024) >> 32);
            const uint32_t a_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.a[0]), 16, 1024));
            // N = 128 operands: two 64-column blocks kBBlock apart (the leading offset)
            const uint32_t b_lo = static_cast<uint32_t>(smem_desc_sw128(smem_addr(sm.b[0][0]), kBBlock, 1024));
            uint32_t kc = 0;
            bool ok = true;
            int i = 0;
            for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x, ++i) {
                const TileId id = tile_id(p, t);
                const int a = i & 1;
                // the epilogue has read this accumulator's previous tile
                if (!(ok = wait_bar(&sm.acc_empty[a], ((i >> 1) & 1) ^ 1, ab, 2))) break;
                tc_fence_after();
                for (int kk = 0; kk < ksteps; ++kk, ++kc) {
                    const uint32_t s = kc % kStages;
                    if (!(ok = wait_bar(&sm.full[s], (kc / kStages) & 1, ab, 3))) break;
                    tc_fence_after();
                    const uint32_t ad = a_lo + s * (kATile >> 4);
                    const uint32_t acc = kk > 0 ? 1u : 0u;
                    for (int nq = 0; nq < id.ncols / 128; ++nq) {
                        // A: 16 bf16 of K per step = 32 bytes; B: K rows 16kk.. = 2 KiB per step
                        const uint32_t bd = b_lo + (s * 4 + 2 * nq) * (kBBlock >> 4);
                        const uint32_t d = tmem + 256 * a + 128 * nq;
                        mma_ss_k<0, 0>(d, ad, bd, desc_hi, kIdesc, acc);
                        mma_ss_k<2, 128>(d, ad, bd, desc_hi, kIdesc, 1u);
                        mma_ss_k<4, 256>(d, ad, bd, desc_hi, kIdesc, 1u);
                        mma_ss_k<6, 384>(d, ad, bd, desc_hi, kIdesc, 1u);
                    }
                    mma_commit(&sm.empty[s]);
                }
                if (ok) mma_commit(&sm.acc_full[a]);
            }
            if (!ok) {
                // make sure no MMA is still writing TMEM when the CTA frees it
                mma_commit(&sm.drain);
                drain_wait(&sm.drain, 0);
            }
        }
        __syncwarp();
    } else {
        // epilogue: thread r = output row r of the tile (TMEM lane r).  Each 64-column
        // block goes through one of two staging blocks in turn: block q is written
        // once the store of the block before last has read its staging block, and
        // stored by one thread; every use of staging block j completes one phase of
        // stage_free[j] and of staged[j], so both follow the use count.
        const int r = (warp % 4) * 32 + threadIdx.x % 32;
        const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
        bool ok = true;
        int i = 0;
        uint32_t uses[2] = {0, 0};
        for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x, ++i) {
            const TileId id = tile_id(p, t);
            const int a = i & 1;
            ok = __all_sync(0xffffffffu, wait_bar(&sm.acc_full[a], (i >> 1) & 1, ab, 4));
            if (!ok) break;
            tc_fence_after();
            const CUtensorMap *tm_out = pick(maps.out, id.pi);
            const int blocks = id.ncols / 64;
            for (int q = 0; q < blocks && ok; ++q) {
                const int j = q & 1;
                const uint32_t u = j ? uses[1] : uses[0];
                uint32_t v[64];
                tmem_ld32(tmem + lane_base + 256 * a + 64 * q, v);
                tmem_ld32(tmem + lane_base + 256 * a + 64 * q + 32, v + 32);
                tmem_wait_ld();
                reg_fence32(v);
                reg_fence32(v + 32);
                if (q == blocks - 1) {
                    // the accumulator is free for the tile after next
                    tc_fence_before();
                    mbar_arrive(&sm.acc_empty[a]);
                }
                if (r == 0) {
                    // each block's store is its own group: all but the last (the other
                    // staging block's) have read their source, this block's included
                    bulk_wait_read_1();
                    mbar_arrive(&sm.stage_free[j]);
                }
                ok = __all_sync(0xffffffffu, wait_bar(&sm.stage_free[j], u & 1, ab, 5));
                if (!ok) break;
                const uint32_t row = smem_addr(sm.stage[j]) + r * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1]));
                    w.y = pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3]));
                    w.z = pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5]));
                    w.w = pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7]));
                    st_shared_v4(row + ((c ^ (r & 7)) << 4), w);
                }
                fence_proxy_async_shared();
                mbar_arrive(&sm.staged[j]);
                if (r == 0) {
                    if ((ok = wait_bar(&sm.staged[j], u & 1, ab, 6))) {
                        if (p.mode == kProjIn) // column c of the product: head c / dk, column c % dk of it
                            tma_store_3d(tm_out, sm.stage[j], (id.n0 + 64 * q) % p.dk, id.t0,
                                         id.b * p.h + (id.n0 + 64 * q) / p.dk);
                        else
                            tma_store_3d(tm_out, sm.stage[j], id.n0 + 64 * q, id.t0, id.b);
                        bulk_commit_group();
                    }
                }
                ok = __all_sync(0xffffffffu, ok);
                if (j) ++uses[1]; else ++uses[0];
            }
        }
        if (r == 0) bulk_wait_all();
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

cudaError_t launch_proj_multi(const ProjProblem *pps, int count, cudaStream_t stream)
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
                  encode_bf16_3d(&maps.out[i], pp.out, pp.dk, pp.L, BH, kTM);
        } else {
            enc = encode_bf16_3d(&maps.a[i], pp.a, pp.dk, pp.L, BH, kTM) &&
                  encode_bf16_3d(&maps.out[i], pp.out, pp.N, pp.L, pp.B, kTM);
        }
        // W [K][N] as a 3-D tensor with one outer slice: 64 x 64 boxes
        enc = enc && encode_bf16_3d(&maps.w[i], pp.w, pp.N, pp.K, 1, kTK);
        if (!enc) return cudaErrorInvalidValue;
        p.m_tiles[i] = (pp.L + kTM - 1) / kTM;
        p.tiles_of[i] = p.n_tiles * p.m_tiles[i] * pp.B;
        p.tiles += p.tiles_of[i];
    }
    for (int i = count; i < kMaxProblems; ++i) {
        maps.a[i] = maps.a[0];
        maps.w[i] = maps.w[0];
        maps.out[i] = maps.out[0];
    }
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int grid = p.tiles < sms ? p.tiles : sms;
    if (!p0.overlap_launch) {
        attn_proj_kernel<<<grid, kThreads, kSmemBytes, stream>>>(maps, p);
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
