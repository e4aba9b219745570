// Internal launcher interface between the C-ABI layer (attn_api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace attn {

struct Problem {
    const void *q;
    const void *k;
    const void *v;
    const int32_t *key_lengths; // device [B]; nullptr unless key padding
    void *out;
    int B, h, m, n, d;
    int mask_kind;  // bit 0 key padding, bit 1 causal
    float scale;    // >= 0
    bool bf16;      // element type of q, k, v, out (fp32 otherwise)
};

enum : int { kMaskKeyPadding = 1, kMaskCausal = 2 };

// CUDA-core kernel: fp32 arithmetic, d <= 64, any m, n.
cudaError_t launch_simt(const Problem &p, cudaStream_t stream);

// tcgen05/TMA kernel (bf16, d == 64).  pair_mode: each CTA tile holds two
// consecutive 128-row query tiles of one head sharing K/V; otherwise each
// CTA tile holds one 128-row query tile of each of two heads (m <= 128).
// tile_counter: two zeroed ints in global memory for the dynamic tile
// schedule (left zeroed on exit), or nullptr for the static schedule.
cudaError_t launch_flash(const Problem &p, bool pair_mode, int *tile_counter, cudaStream_t stream);

// Bytes of workspace the dynamic tile schedule needs.
constexpr size_t kWorkspaceBytes = 256;

// Device status word of the flash kernel (bounded waits that gave up).
cudaError_t flash_status_read_and_clear(cudaStream_t stream, uint32_t *code, uint32_t *info);

} // namespace attn
