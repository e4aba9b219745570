// Internal launcher interface between the C-ABI layer (attn_api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

struct Problem {
    const void *q;
    const void *k;
    const void *v;
    const int32_t *key_lengths; // device [B]; nullptr unless key padding
    void *out;
    float *lse;                 // device [B][h][m] natural log of each row's softmax normaliser, or nullptr
    int B, h, m, n, d;
    int mask_kind;  // bit 0 key padding, bit 1 causal, bit 2 window
    int window = -1; // window half-width when bit 2 is set (keys with |i - j| <= window stay)
    float scale;    // >= 0
    bool bf16;      // element type of q, k, v, out (fp32 otherwise)
    bool overlap_launch = false; // tensor-core kernels: launched as a programmatic dependent of the
                                 // previous kernel on the stream (its prologue overlaps that kernel's tail)
};

enum : int { kMaskKeyPadding = 1, kMaskCausal = 2, kMaskWindow = 4 };

// CUDA-core kernel: fp32 arithmetic, d <= 64, any m, n.
cudaError_t launch_simt(const Problem &p, cudaStream_t stream);

// tcgen05/TMA kernel (bf16, d a multiple of 8 up to 64: narrower heads enter the
// 64-wide tiles zero-padded by the TMA loads and leave clipped by the TMA store).  pair_mode: each CTA tile holds two
// consecutive 128-row query tiles of one head sharing K/V; otherwise each
// CTA tile holds one 128-row query tile of each of two heads (m <= 128).
// tile_counter: two zeroed ints in global memory for the dynamic tile
// schedule (left zeroed on exit), or nullptr for the static schedule.
cudaError_t launch_flash(const Problem &p, bool pair_mode, int *tile_counter, cudaStream_t stream);

// Bytes of workspace the dynamic tile schedule needs.
constexpr size_t kWorkspaceBytes = 256;

// Incremental decoding (bf16, d in {16, 32, 64, 128}, m <= 8 queries per head, every
// query sees keys 0 .. len_b - 1): split-KV CUDA-core kernel plus a combine pass.
int decode_splits(int B, int h, int n, int sms);
bool decode_width_supported(int d);
size_t decode_workspace_bytes(int B, int h, int m, int n, int d, int sms);
cudaError_t launch_decode(const Problem &p, void *workspace, int sms, cudaStream_t stream);

// [BH][rows][64] bf16 viewed as a 3-D tensor (64, rows, BH) for TMA; box = 128
// rows x 64 columns of one (b, h), 128-byte swizzle, rows past `rows` read as 0.
bool encode_rows_map(CUtensorMap *map, const void *base, int rows, int BH);

// [outer][rows][inner] bf16 as a 3-D TMA tensor (inner a multiple of 8); box =
// box_rows rows x 64 elements of one outer index, 128-byte swizzle.
bool encode_bf16_3d(CUtensorMap *map, const void *base, int inner, int rows, int outer, int box_rows);

// [BH][rows][64] fp32 as a 3-D tensor for TMA reductions; box = 128 rows x 32
// columns (one 128-byte swizzle span), 128-byte swizzle.
bool encode_rows_map_f32(CUtensorMap *map, void *base, int rows, int BH);

// Backward: dQ, dK, dV (bf16, d a multiple of 8 up to 64) from Q, K, V, the forward's
// output and per-row log-sum-exp, and the output gradient.
struct BwdProblem {
    const void *q, *k, *v, *out, *dout; // bf16 [B][h][rows][d]
    const float *lse;                   // [B][h][m], natural log
    const int32_t *key_lengths;         // device [B]; nullptr unless key padding
    void *dq, *dk, *dv;                 // bf16, shaped like q, k, v
    void *workspace;                    // bwd_workspace_bytes(B, h, m), 256-byte aligned
    int B, h, m, n;
    int d = 64;                         // head width: a multiple of 8 up to 64 (narrower heads
                                        // enter the 64-wide tiles zero-padded)
    int mask_kind;
    float scale;
};

// CUDA-core backward (fp32 arithmetic; bf16 or fp32 tensors; any d up to 128): a rows
// pass (D and dQ) and a keys pass (dK and dV).  Workspace: D, B * h * m floats.
struct BwdSimtProblem {
    const void *q, *k, *v, *out, *dout; // [B][h][rows][d]
    const float *lse;                   // [B][h][m], natural log
    const int32_t *key_lengths;         // device [B]; nullptr unless key padding
    void *dq, *dk, *dv;
    void *workspace;                    // bwd_simt_workspace_bytes(B, h, m), 4-byte aligned
    int B, h, m, n, d;
    int mask_kind;
    float scale;
    bool bf16;
};
size_t bwd_simt_workspace_bytes(int B, int h, int m);
cudaError_t launch_bwd_simt(const BwdSimtProblem &p, cudaStream_t stream);

// Workspace of the backward: the fp32 dQ accumulator and the per-row table.
size_t bwd_workspace_bytes(int B, int h, int m);
cudaError_t launch_bwd(const BwdProblem &p, cudaStream_t stream);
cudaError_t bwd_status_read_and_clear(cudaStream_t stream, uint32_t *code, uint32_t *info);

// Projection GEMM of the multi-head wrapper (tcgen05).  kIn: out[b*h + j][t][:] =
// row t of x[b] (a [B][L][K] bf16 tensor) times columns dk j .. dk (j+1) - 1 of w
// ([K][N] bf16, N = h * dk).  kOut: out[b][t][:] = sum over heads j of row t of
// a[b*h + j] ([B*h][L][dk]) times rows dk j .. dk (j+1) - 1 of w ([h * dk][N]).
enum ProjMode : int { kProjIn = 0, kProjOut = 1 };
struct ProjProblem {
    ProjMode mode;
    const void *a;   // kIn: x [B][L][K]; kOut: heads [B*h][L][dk]
    const void *w;   // [K][N], K = d_model (kIn) or h * dk (kOut)
    void *out;       // kIn: [B*h][L][dk]; kOut: [B][L][N]
    int B, h, L, K, N;
    int dk = 64;     // head width (64 or 128): a head is dk / 64 blocks of 64 columns
    bool overlap_launch = false; // launched as a programmatic dependent of the previous kernel on the stream
};
cudaError_t launch_proj(const ProjProblem &p, cudaStream_t stream);
// Up to three products of one shape (mode, B, h, K, N; L may differ) in one launch.
cudaError_t launch_proj_multi(const ProjProblem *p, int count, cudaStream_t stream);
cudaError_t proj_status_read_and_clear(cudaStream_t stream, uint32_t *code, uint32_t *info);
// bf16 [B][L][h][dk] (concatenated heads) to [B][h][L][dk] (split) or back; dk a multiple of 8.
cudaError_t launch_heads_copy(const void *src, void *dst, int B, int L, int h, int dk, bool split,
                              cudaStream_t stream);

// Device status word of the flash kernel (bounded waits that gave up).
cudaError_t flash_status_read_and_clear(cudaStream_t stream, uint32_t *code, uint32_t *info);

// Whole-head-resident tcgen05/TMA kernel for short key sequences (bf16, d a multiple
// of 8 up to 64, n <= kResidentMaxKeys, any m): one 128-row query tile of one head per
// CTA with all of the head's keys, exact two-pass softmax per row.  Launched as a
// programmatic dependent of the previous kernel when p.overlap_launch is set
// (everything it reads or writes follows the dependency wait).
constexpr int kResidentMaxKeys = 256;
bool resident_fits(int m, int n, int d);
// Test hook of the bounded waits: a short wait limit, and the barrier on which the rows
// hand over their first chunk of weights waiting for one arrival more than they make,
// so that the MMA issuer's wait runs out.
struct ResidentTestHook {
    uint64_t wait_ns;
    int withhold_p_arrival;
};
cudaError_t launch_resident(const Problem &p, cudaStream_t stream, const ResidentTestHook *hook = nullptr);
cudaError_t resident_status_read_and_clear(cudaStream_t stream, uint32_t *code, uint32_t *info);

// tcgen05/TMA kernel for bf16 heads of width 128 (one 128-row query tile per CTA).
cudaError_t launch_wide(const Problem &p, cudaStream_t stream);
cudaError_t wide_status_read_and_clear(cudaStream_t stream, uint32_t *code, uint32_t *info);

} // namespace attn
