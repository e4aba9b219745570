// C-ABI layer: argument validation, kernel choice, launch on the caller's stream.
// The operation and its rules are documented in include/attn.h.
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>
#include <mutex>

#include "../../include/attn.h"
#include "kernels.h"

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void *a, uint64_t abytes, const void *b, uint64_t bbytes)
{
    if (a == nullptr || b == nullptr) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// Heads the tensor-core kernels take: bf16, d_k a multiple of 8 up to 64 (narrower
// heads run zero-padded to 64 inside the kernel).
bool tensor_core_head(const attn_dims &d) { return d.dtype == ATTN_BF16 && d.d_k % 8 == 0 && d.d_k <= 64; }

// Which kernel AUTO picks: tensor cores for tensor_core_head (one query tile per CTA
// with the head's keys and values resident, when a head has at most 256 keys; two
// heads per CTA tile when it has at most 128 queries; two query tiles of one head
// otherwise); CUDA cores for fp32 and for other bf16 head widths.
int auto_kernel(const attn_dims &d)
{
    if (tensor_core_head(d) && attn::resident_fits(d.m, d.n, d.d_k)) return ATTN_KERNEL_RESIDENT;
    if (tensor_core_head(d)) return d.m <= 128 ? ATTN_KERNEL_SHORT : ATTN_KERNEL_FLASH;
    if (d.dtype == ATTN_BF16 && d.d_k == 128) return ATTN_KERNEL_WIDE;
    return ATTN_KERNEL_SIMT;
}

bool scale_ok(float scale) { return scale == ATTN_SCALE_DEFAULT || (std::isfinite(scale) && scale >= 0.f); }

// The scale a kernel multiplies the scores by: the caller's, or 1/sqrt(d_k) for
// ATTN_SCALE_DEFAULT (the formula's scale).
float resolve_scale(float scale, int d_k)
{
    return scale == ATTN_SCALE_DEFAULT ? static_cast<float>(1.0 / std::sqrt(static_cast<double>(d_k))) : scale;
}

attn_status validate_dims(const attn_dims *dims, int mask_kind, float scale)
{
    if (dims == nullptr) return ATTN_ERR_NULL;
    if ((mask_kind & ~(ATTN_MASK_KEY_PADDING | ATTN_MASK_CAUSAL)) != 0) return ATTN_ERR_MASK;
    const attn_dims &d = *dims;
    if (d.dtype != ATTN_BF16 && d.dtype != ATTN_FP32) return ATTN_ERR_DTYPE;
    if (d.d_k < 1 || d.d_k > 128) return ATTN_ERR_DTYPE;
    if (d.B < 1 || d.h < 1 || d.m < 1 || d.n < 1) return ATTN_ERR_SHAPE;
    if (d.B > 65535 || d.h > 65535) return ATTN_ERR_SHAPE;                  // grid limits
    if ((mask_kind & ATTN_MASK_CAUSAL) && d.m != d.n) return ATTN_ERR_SHAPE; // queries and keys share positions
    if (!scale_ok(scale)) return ATTN_ERR_VALUE;
    return ATTN_OK;
}

attn_status validate(const void *Q, const void *K, const void *V, const int32_t *key_lengths, int mask_kind,
                     float scale, void *out, const attn_dims *dims)
{
    if (dims == nullptr || Q == nullptr || K == nullptr || V == nullptr || out == nullptr) return ATTN_ERR_NULL;
    if ((mask_kind & ATTN_MASK_KEY_PADDING) && key_lengths == nullptr) return ATTN_ERR_NULL;
    const attn_status st = validate_dims(dims, mask_kind, scale);
    if (st != ATTN_OK) return st;
    const attn_dims &d = *dims;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(out, 16)) return ATTN_ERR_ALIGN;
    if ((mask_kind & ATTN_MASK_KEY_PADDING) && !aligned(key_lengths, 4)) return ATTN_ERR_ALIGN;
    const uint64_t esz = d.dtype == ATTN_BF16 ? 2 : 4;
    const uint64_t qbytes = static_cast<uint64_t>(d.B) * d.h * d.m * d.d_k * esz;
    const uint64_t kbytes = static_cast<uint64_t>(d.B) * d.h * d.n * d.d_k * esz;
    if (overlaps(out, qbytes, Q, qbytes) || overlaps(out, qbytes, K, kbytes) || overlaps(out, qbytes, V, kbytes))
        return ATTN_ERR_ALIAS;
    if ((mask_kind & ATTN_MASK_KEY_PADDING) && overlaps(out, qbytes, key_lengths, 4ull * d.B))
        return ATTN_ERR_ALIAS;
    return ATTN_OK;
}

} // namespace

namespace {

attn_status run(const void *Q, const void *K, const void *V, const int32_t *key_lengths, int mask_kind, float scale,
                void *out, const attn_dims *dims, void *stream, int kernel, int *tile_counter, float *lse = nullptr,
                int window = -1, bool overlap_launch = false)
{
    // the window bit is accepted only from attn_fwd_window (window >= 0), which checks it
    const int checked = window >= 0 ? (mask_kind & ~ATTN_MASK_WINDOW) : mask_kind;
    const attn_status st = validate(Q, K, V, key_lengths, checked, scale, out, dims);
    if (st != ATTN_OK) return st;
    const attn_dims &d = *dims;
    if (kernel == ATTN_KERNEL_AUTO) kernel = auto_kernel(d);
    attn::Problem p;
    p.q = Q;
    p.k = K;
    p.v = V;
    p.key_lengths = (mask_kind & ATTN_MASK_KEY_PADDING) ? key_lengths : nullptr;
    p.out = out;
    p.lse = lse;
    p.B = d.B;
    p.h = d.h;
    p.m = d.m;
    p.n = d.n;
    p.d = d.d_k;
    p.mask_kind = mask_kind;
    p.window = window;
    p.scale = resolve_scale(scale, d.d_k);
    p.bf16 = d.dtype == ATTN_BF16;
    p.overlap_launch = overlap_launch;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (kernel) {
    case ATTN_KERNEL_SIMT:
        e = attn::launch_simt(p, s);
        break;
    case ATTN_KERNEL_FLASH:
        if (!tensor_core_head(d)) return ATTN_ERR_UNSUPPORTED;
        e = attn::launch_flash(p, /*pair_mode=*/true, tile_counter, s);
        break;
    case ATTN_KERNEL_WIDE:
        if (!p.bf16 || p.d != 128) return ATTN_ERR_UNSUPPORTED;
        e = attn::launch_wide(p, s);
        break;
    case ATTN_KERNEL_SHORT:
        if (!tensor_core_head(d) || p.m > 128) return ATTN_ERR_UNSUPPORTED;
        e = attn::launch_flash(p, /*pair_mode=*/false, tile_counter, s);
        break;
    case ATTN_KERNEL_RESIDENT:
        if (!tensor_core_head(d) || !attn::resident_fits(d.m, d.n, d.d_k)) return ATTN_ERR_UNSUPPORTED;
        p.overlap_launch = true; // every access of the kernel follows its dependency wait
        e = attn::launch_resident(p, s);
        break;
    default:
        return ATTN_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Scratch of attn_fwd_noalloc: a statically allocated device array (one per
// device that loads the library, held until the process exits).  Host code
// cannot use the symbol's name as a device address; its address is looked up
// once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

struct NoAllocDevice {
    std::mutex lock;
    void *ptr = nullptr; // set once a lookup has succeeded; kept for the life of the process
};
constexpr int kMaxDevices = 64;
NoAllocDevice g_noalloc_devices[kMaxDevices];

// Device address of g_noalloc_scratch on the current device.  The first successful
// lookup is kept; a failed one is not, so the next call tries again.
cudaError_t noalloc_scratch(void **ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    NoAllocDevice &d = g_noalloc_devices[dev];
    std::lock_guard<std::mutex> guard(d.lock);
    if (d.ptr == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        d.ptr = p;
    }
    *ptr = d.ptr;
    return cudaSuccess;
}

} // namespace

extern "C" {

attn_status attn_fwd_noalloc(const void *Q, const void *K, const void *V, const int32_t *key_lengths,
                             int mask_kind, float scale, void *out, const attn_dims *dims, void *stream)
{
    const attn_status st = validate(Q, K, V, key_lengths, mask_kind, scale, out, dims);
    if (st != ATTN_OK) return st;
    if (attn::kWorkspaceBytes > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_SCRATCH;
    void *scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return ATTN_ERR_CUDA;
    // The array keeps the previous call's contents.  Only the d_k <= 64 tensor-core
    // kernels read it (their tile counters); they leave it zeroed when they finish,
    // but not after an earlier call gave up a bounded wait, so it is cleared here.
    const int kernel = auto_kernel(*dims);
    if ((kernel == ATTN_KERNEL_FLASH || kernel == ATTN_KERNEL_SHORT) &&
        cudaMemsetAsync(scratch, 0, attn::kWorkspaceBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    return run(Q, K, V, key_lengths, mask_kind, scale, out, dims, stream, ATTN_KERNEL_AUTO,
               static_cast<int *>(scratch));
}


attn_status attn_fwd_kernel(const void *Q, const void *K, const void *V, const int32_t *key_lengths,
                            int mask_kind, float scale, void *out, const attn_dims *dims, void *stream,
                            int kernel)
{
    return run(Q, K, V, key_lengths, mask_kind, scale, out, dims, stream, kernel, nullptr);
}

size_t attn_workspace_size(void) { return attn::kWorkspaceBytes; }

attn_status attn_fwd_ws(const void *Q, const void *K, const void *V, const int32_t *key_lengths, int mask_kind,
                        float scale, void *out, const attn_dims *dims, void *stream, void *workspace,
                        size_t workspace_bytes)
{
    if (workspace == nullptr) return ATTN_ERR_NULL;
    if (workspace_bytes < attn::kWorkspaceBytes) return ATTN_ERR_SHAPE;
    if (!aligned(workspace, 16)) return ATTN_ERR_ALIGN;
    const attn_status st = validate(Q, K, V, key_lengths, mask_kind, scale, out, dims);
    if (st != ATTN_OK) return st;
    const attn_dims &d = *dims;
    const uint64_t esz = d.dtype == ATTN_BF16 ? 2 : 4;
    const uint64_t qbytes = static_cast<uint64_t>(d.B) * d.h * d.m * d.d_k * esz;
    const uint64_t kbytes = static_cast<uint64_t>(d.B) * d.h * d.n * d.d_k * esz;
    if (overlaps(workspace, workspace_bytes, out, qbytes) || overlaps(workspace, workspace_bytes, Q, qbytes) ||
        overlaps(workspace, workspace_bytes, K, kbytes) || overlaps(workspace, workspace_bytes, V, kbytes))
        return ATTN_ERR_ALIAS;
    if ((mask_kind & ATTN_MASK_KEY_PADDING) && overlaps(workspace, workspace_bytes, key_lengths, 4ull * d.B))
        return ATTN_ERR_ALIAS;
    return run(Q, K, V, key_lengths, mask_kind, scale, out, dims, stream, ATTN_KERNEL_AUTO,
               static_cast<int *>(workspace));
}

attn_status attn_fwd_window(const void *Q, const void *K, const void *V, const int32_t *key_lengths, int mask_kind,
                            int window, float scale, void *out, const attn_dims *dims, void *stream)
{
    if (!(mask_kind & ATTN_MASK_WINDOW))
        return run(Q, K, V, key_lengths, mask_kind, scale, out, dims, stream, ATTN_KERNEL_AUTO, nullptr);
    if (dims == nullptr) return ATTN_ERR_NULL;
    if ((mask_kind & ~(ATTN_MASK_KEY_PADDING | ATTN_MASK_CAUSAL | ATTN_MASK_WINDOW)) != 0) return ATTN_ERR_MASK;
    const attn_status st = validate(Q, K, V, key_lengths, mask_kind & ~ATTN_MASK_WINDOW, scale, out, dims);
    if (st != ATTN_OK) return st;
    if (dims->m != dims->n) return ATTN_ERR_SHAPE; // self-attention: queries and keys share positions
    if (window < 0) return ATTN_ERR_VALUE;
    return run(Q, K, V, key_lengths, mask_kind, scale, out, dims, stream, ATTN_KERNEL_AUTO, nullptr, nullptr,
               window);
}

attn_status attn_fwd(const void *Q, const void *K, const void *V, const int32_t *key_lengths, int mask_kind,
                     float scale, void *out, const attn_dims *dims, void *stream)
{
    return attn_fwd_kernel(Q, K, V, key_lengths, mask_kind, scale, out, dims, stream, ATTN_KERNEL_AUTO);
}

attn_status attn_fwd_lse(const void *Q, const void *K, const void *V, const int32_t *key_lengths, int mask_kind,
                         float scale, void *out, float *lse, const attn_dims *dims, void *stream)
{
    if (lse == nullptr) return ATTN_ERR_NULL;
    const attn_status st = validate(Q, K, V, key_lengths, mask_kind, scale, out, dims);
    if (st != ATTN_OK) return st;
    if (!aligned(lse, 4)) return ATTN_ERR_ALIGN;
    const attn_dims &d = *dims;
    const uint64_t esz = d.dtype == ATTN_BF16 ? 2 : 4;
    const uint64_t qbytes = static_cast<uint64_t>(d.B) * d.h * d.m * d.d_k * esz;
    const uint64_t kbytes = static_cast<uint64_t>(d.B) * d.h * d.n * d.d_k * esz;
    const uint64_t lbytes = static_cast<uint64_t>(d.B) * d.h * d.m * 4;
    if (overlaps(lse, lbytes, out, qbytes) || overlaps(lse, lbytes, Q, qbytes) || overlaps(lse, lbytes, K, kbytes) ||
        overlaps(lse, lbytes, V, kbytes))
        return ATTN_ERR_ALIAS;
    if ((mask_kind & ATTN_MASK_KEY_PADDING) && overlaps(lse, lbytes, key_lengths, 4ull * d.B))
        return ATTN_ERR_ALIAS;
    return run(Q, K, V, key_lengths, mask_kind, scale, out, dims, stream, ATTN_KERNEL_AUTO, nullptr, lse);
}

// Workspace of the backward for these dims: the tensor-core backward's (bf16 heads of a
// multiple of 8 up to 64) or the CUDA-core backward's (everything else up to 128 wide).
size_t bwd_need(const attn_dims &d)
{
    return tensor_core_head(d) ? attn::bwd_workspace_bytes(d.B, d.h, d.m) : attn::bwd_simt_workspace_bytes(d.B, d.h, d.m);
}

size_t attn_bwd_workspace_size(const attn_dims *dims)
{
    if (validate_dims(dims, 0, 1.0f) != ATTN_OK) return 0;
    return bwd_need(*dims);
}

attn_status attn_bwd(const void *Q, const void *K, const void *V, const void *out, const void *dout, const float *lse,
                     const int32_t *key_lengths, int mask_kind, float scale, void *dQ, void *dK, void *dV,
                     void *workspace, size_t workspace_bytes, const attn_dims *dims, void *stream)
{
    if (out == nullptr || dout == nullptr || lse == nullptr || dQ == nullptr || dK == nullptr || dV == nullptr ||
        workspace == nullptr)
        return ATTN_ERR_NULL;
    // Q, K, V, key_lengths, mask, scale and dims as for the forward; dQ stands in for out
    const attn_status st = validate(Q, K, V, key_lengths, mask_kind, scale, dQ, dims);
    if (st != ATTN_OK) return st;
    const attn_dims &d = *dims;
    if (!aligned(out, 16) || !aligned(dout, 16) || !aligned(dK, 16) || !aligned(dV, 16) || !aligned(lse, 4) ||
        !aligned(workspace, 256))
        return ATTN_ERR_ALIGN;
    const size_t need = bwd_need(d);
    if (workspace_bytes < need) return ATTN_ERR_SHAPE;
    const uint64_t esz = d.dtype == ATTN_BF16 ? 2 : 4;
    const uint64_t qbytes = static_cast<uint64_t>(d.B) * d.h * d.m * d.d_k * esz;
    const uint64_t kbytes = static_cast<uint64_t>(d.B) * d.h * d.n * d.d_k * esz;
    const uint64_t lbytes = static_cast<uint64_t>(d.B) * d.h * d.m * 4;
    struct Span {
        const void *p;
        uint64_t n;
    };
    const Span outs[4] = {{dQ, qbytes}, {dK, kbytes}, {dV, kbytes}, {workspace, need}};
    const Span ins[7] = {{Q, qbytes},   {K, kbytes},   {V, kbytes}, {out, qbytes},
                         {dout, qbytes}, {lse, lbytes},
                         {(mask_kind & ATTN_MASK_KEY_PADDING) ? key_lengths : nullptr, 4ull * d.B}};
    for (int a = 0; a < 4; ++a) {
        for (int b = a + 1; b < 4; ++b)
            if (overlaps(outs[a].p, outs[a].n, outs[b].p, outs[b].n)) return ATTN_ERR_ALIAS;
        for (int b = 0; b < 7; ++b)
            if (overlaps(outs[a].p, outs[a].n, ins[b].p, ins[b].n)) return ATTN_ERR_ALIAS;
    }
    if (!tensor_core_head(d)) {
        // fp32, and bf16 heads the tensor-core backward does not take: the CUDA cores
        attn::BwdSimtProblem p;
        p.q = Q;
        p.k = K;
        p.v = V;
        p.out = out;
        p.dout = dout;
        p.lse = lse;
        p.key_lengths = (mask_kind & ATTN_MASK_KEY_PADDING) ? key_lengths : nullptr;
        p.dq = dQ;
        p.dk = dK;
        p.dv = dV;
        p.workspace = workspace;
        p.B = d.B;
        p.h = d.h;
        p.m = d.m;
        p.n = d.n;
        p.d = d.d_k;
        p.mask_kind = mask_kind;
        p.scale = resolve_scale(scale, d.d_k);
        p.bf16 = d.dtype == ATTN_BF16;
        return attn::launch_bwd_simt(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    }
    attn::BwdProblem p;
    p.q = Q;
    p.k = K;
    p.v = V;
    p.out = out;
    p.dout = dout;
    p.lse = lse;
    p.key_lengths = (mask_kind & ATTN_MASK_KEY_PADDING) ? key_lengths : nullptr;
    p.dq = dQ;
    p.dk = dK;
    p.dv = dV;
    p.d = d.d_k;
    p.workspace = workspace;
    p.B = d.B;
    p.h = d.h;
    p.m = d.m;
    p.n = d.n;
    p.mask_kind = mask_kind;
    p.scale = resolve_scale(scale, d.d_k);
    return attn::launch_bwd(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

namespace {
// SM count of the current device (the decode kernel's split geometry); 0 on error.
int current_sms()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

attn_status validate_decode_dims(const attn_dims *dims)
{
    if (dims == nullptr) return ATTN_ERR_NULL;
    const attn_status st = validate_dims(dims, ATTN_MASK_KEY_PADDING, 1.0f);
    if (st != ATTN_OK) return st;
    if (dims->dtype != ATTN_BF16 || !attn::decode_width_supported(dims->d_k)) return ATTN_ERR_DTYPE;
    if (dims->m > 8) return ATTN_ERR_SHAPE;
    return ATTN_OK;
}
} // namespace

size_t attn_decode_workspace_size(const attn_dims *dims)
{
    if (validate_decode_dims(dims) != ATTN_OK) return 0;
    const int sms = current_sms();
    if (sms <= 0) return 0;
    return attn::decode_workspace_bytes(dims->B, dims->h, dims->m, dims->n, dims->d_k, sms);
}

attn_status attn_decode(const void *Q, const void *K, const void *V, const int32_t *cache_lengths, float scale,
                        void *out, float *lse, const attn_dims *dims, void *workspace, size_t workspace_bytes,
                        void *stream)
{
    attn_status st = validate_decode_dims(dims);
    if (st != ATTN_OK) return st;
    const int mask = cache_lengths != nullptr ? ATTN_MASK_KEY_PADDING : ATTN_MASK_NONE;
    st = validate(Q, K, V, cache_lengths, mask, scale, out, dims);
    if (st != ATTN_OK) return st;
    const attn_dims &d = *dims;
    const uint64_t qbytes = static_cast<uint64_t>(d.B) * d.h * d.m * d.d_k * 2;
    const uint64_t kbytes = static_cast<uint64_t>(d.B) * d.h * d.n * d.d_k * 2;
    const uint64_t lbytes = static_cast<uint64_t>(d.B) * d.h * d.m * 4;
    if (lse != nullptr) {
        if (!aligned(lse, 4)) return ATTN_ERR_ALIGN;
        if (overlaps(lse, lbytes, out, qbytes) || overlaps(lse, lbytes, Q, qbytes) ||
            overlaps(lse, lbytes, K, kbytes) || overlaps(lse, lbytes, V, kbytes) ||
            overlaps(lse, lbytes, cache_lengths, 4ull * d.B))
            return ATTN_ERR_ALIAS;
    }
    const int sms = current_sms();
    if (sms <= 0) return ATTN_ERR_CUDA;
    const size_t need = attn::decode_workspace_bytes(d.B, d.h, d.m, d.n, d.d_k, sms);
    if (need > 0) {
        if (workspace == nullptr) return ATTN_ERR_NULL;
        if (workspace_bytes < need) return ATTN_ERR_SHAPE;
        if (!aligned(workspace, 16)) return ATTN_ERR_ALIGN;
        if (overlaps(workspace, need, out, qbytes) || overlaps(workspace, need, Q, qbytes) ||
            overlaps(workspace, need, K, kbytes) || overlaps(workspace, need, V, kbytes) ||
            overlaps(workspace, need, cache_lengths, 4ull * d.B) || (lse && overlaps(workspace, need, lse, lbytes)))
            return ATTN_ERR_ALIAS;
    }
    attn::Problem p;
    p.q = Q;
    p.k = K;
    p.v = V;
    p.key_lengths = cache_lengths;
    p.out = out;
    p.lse = lse;
    p.B = d.B;
    p.h = d.h;
    p.m = d.m;
    p.n = d.n;
    p.d = d.d_k;
    p.mask_kind = mask;
    p.scale = resolve_scale(scale, d.d_k);
    p.bf16 = true;
    return attn::launch_decode(p, workspace, sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK
                                                                                                  : ATTN_ERR_CUDA;
}

namespace {
int mha_dk(const attn_mha_dims &d) { return d.d_k == 0 ? 64 : d.d_k; }

attn_status validate_mha_dims(const attn_mha_dims *d)
{
    if (d == nullptr) return ATTN_ERR_NULL;
    // 64 and 128 wide heads are whole 64-column blocks of the projections; narrower
    // ones (a multiple of 8 below 64) go through the concatenated layout
    if (d->d_k != 0 && d->d_k != 128 && !(d->d_k % 8 == 0 && d->d_k >= 8 && d->d_k <= 64)) return ATTN_ERR_DTYPE;
    if (d->B < 1 || d->h < 1 || d->m < 1 || d->n < 1 || d->d_model < 1) return ATTN_ERR_SHAPE;
    if (d->B > 65535 || d->h > 65535 || (static_cast<int64_t>(d->h) * mha_dk(*d)) % 128 != 0 ||
        d->d_model % 128 != 0)
        return ATTN_ERR_SHAPE;
    return ATTN_OK;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct MhaLayout {
    size_t q, k, v, o;    // byte offsets in the workspace: the head-split Q, K, V, O
    size_t qc, kc, vc;    // narrow heads: the concatenated projections (the heads' output reuses qc)
    size_t total;
};

// Heads whose width is a whole number of 64-column blocks go straight from the
// projections' epilogues into the head-split layout; narrower heads go through the
// concatenated layout [B][len][h * d_k] and a copy.
bool mha_direct(const attn_mha_dims &d) { return mha_dk(d) % 64 == 0; }

MhaLayout mha_layout(const attn_mha_dims &d)
{
    const size_t BH = static_cast<size_t>(d.B) * d.h;
    const size_t dk = static_cast<size_t>(mha_dk(d));
    MhaLayout L;
    L.q = 0;
    L.k = L.q + align256(BH * d.m * dk * 2);
    L.v = L.k + align256(BH * d.n * dk * 2);
    L.o = L.v + align256(BH * d.n * dk * 2);
    L.total = L.o + align256(BH * d.m * dk * 2);
    L.qc = L.kc = L.vc = 0;
    if (!mha_direct(d)) {
        L.qc = L.total;
        L.kc = L.qc + align256(BH * d.m * dk * 2);
        L.vc = L.kc + align256(BH * d.n * dk * 2);
        L.total = L.vc + align256(BH * d.n * dk * 2);
    }
    return L;
}
} // namespace

size_t attn_mha_workspace_size(const attn_mha_dims *dims)
{
    if (validate_mha_dims(dims) != ATTN_OK) return 0;
    return mha_layout(*dims).total;
}

attn_status attn_mha_fwd(const void *Xq, const void *Xkv, const void *Wq, const void *Wk, const void *Wv,
                         const void *Wo, const int32_t *key_lengths, int mask_kind, float scale, void *out,
                         const attn_mha_dims *dims, void *workspace, size_t workspace_bytes, void *stream)
{
    attn_status st = validate_mha_dims(dims);
    if (st != ATTN_OK) return st;
    if (!Xq || !Xkv || !Wq || !Wk || !Wv || !Wo || !out || !workspace) return ATTN_ERR_NULL;
    if ((mask_kind & ATTN_MASK_KEY_PADDING) && key_lengths == nullptr) return ATTN_ERR_NULL;
    if ((mask_kind & ~(ATTN_MASK_KEY_PADDING | ATTN_MASK_CAUSAL)) != 0) return ATTN_ERR_MASK;
    const attn_mha_dims &d = *dims;
    if ((mask_kind & ATTN_MASK_CAUSAL) && d.m != d.n) return ATTN_ERR_SHAPE;
    if (!scale_ok(scale)) return ATTN_ERR_VALUE;
    const void *ptrs[8] = {Xq, Xkv, Wq, Wk, Wv, Wo, out, workspace};
    for (const void *q : ptrs)
        if (!aligned(q, 16)) return ATTN_ERR_ALIGN;
    if (!aligned(workspace, 256)) return ATTN_ERR_ALIGN;
    if ((mask_kind & ATTN_MASK_KEY_PADDING) && !aligned(key_lengths, 4)) return ATTN_ERR_ALIGN;
    const MhaLayout L = mha_layout(d);
    if (workspace_bytes < L.total) return ATTN_ERR_SHAPE;
    const int dk = mha_dk(d);
    const uint64_t dm = d.d_model, hd = static_cast<uint64_t>(d.h) * dk;
    const uint64_t xq = static_cast<uint64_t>(d.B) * d.m * dm * 2, xkv = static_cast<uint64_t>(d.B) * d.n * dm * 2;
    const uint64_t wb = dm * hd * 2;
    struct Span {
        const void *p;
        uint64_t n;
    };
    const Span ins[7] = {{Xq, xq}, {Xkv, xkv}, {Wq, wb}, {Wk, wb}, {Wv, wb}, {Wo, wb},
                         {(mask_kind & ATTN_MASK_KEY_PADDING) ? key_lengths : nullptr, 4ull * d.B}};
    for (const Span &in : ins)
        if (overlaps(out, xq, in.p, in.n) || overlaps(workspace, L.total, in.p, in.n)) return ATTN_ERR_ALIAS;
    if (overlaps(out, xq, workspace, L.total)) return ATTN_ERR_ALIAS;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *Q = ws + L.q, *K = ws + L.k, *V = ws + L.v, *O = ws + L.o;
    if (!mha_direct(d)) {
        // Narrow heads: the projections as plain products into [B][len][h * d_k] (one
        // "head" as wide as the product), split into heads, attention, heads merged
        // back (into the Q product's space, free by then), the output projection.
        void *Qc = ws + L.qc, *Kc = ws + L.kc, *Vc = ws + L.vc;
        attn::ProjProblem in3[3];
        const struct {
            const void *x, *w;
            void *o;
            int L;
        } prods[3] = {{Xq, Wq, Qc, d.m}, {Xkv, Wk, Kc, d.n}, {Xkv, Wv, Vc, d.n}};
        for (int i = 0; i < 3; ++i) {
            in3[i].mode = attn::kProjIn;
            in3[i].a = prods[i].x;
            in3[i].w = prods[i].w;
            in3[i].out = prods[i].o;
            in3[i].B = d.B;
            in3[i].h = 1;
            in3[i].L = prods[i].L;
            in3[i].K = d.d_model;
            in3[i].N = d.h * dk;
            in3[i].dk = d.h * dk;
        }
        if (attn::launch_proj_multi(in3, 3, s) != cudaSuccess) return ATTN_ERR_CUDA;
        if (attn::launch_heads_copy(Qc, Q, d.B, d.m, d.h, dk, true, s) != cudaSuccess ||
            attn::launch_heads_copy(Kc, K, d.B, d.n, d.h, dk, true, s) != cudaSuccess ||
            attn::launch_heads_copy(Vc, V, d.B, d.n, d.h, dk, true, s) != cudaSuccess)
            return ATTN_ERR_CUDA;
        attn_dims ad{d.B, d.h, d.m, d.n, dk, ATTN_BF16};
        st = run(Q, K, V, key_lengths, mask_kind, scale, O, &ad, stream, ATTN_KERNEL_AUTO, nullptr);
        if (st != ATTN_OK) return st;
        if (attn::launch_heads_copy(O, Qc, d.B, d.m, d.h, dk, false, s) != cudaSuccess) return ATTN_ERR_CUDA;
        attn::ProjProblem po;
        po.mode = attn::kProjIn;
        po.a = Qc;
        po.w = Wo;
        po.out = out;
        po.B = d.B;
        po.h = 1;
        po.L = d.m;
        po.K = d.h * dk;
        po.N = d.d_model;
        po.dk = d.d_model;
        return attn::launch_proj(po, s) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    }
    attn::ProjProblem pp;
    pp.B = d.B;
    pp.h = d.h;
    pp.mode = attn::kProjIn;
    pp.K = d.d_model;
    pp.N = d.h * dk;
    pp.dk = dk;
    const struct {
        const void *x, *w;
        void *o;
        int L;
    } ins_proj[3] = {{Xq, Wq, Q, d.m}, {Xkv, Wk, K, d.n}, {Xkv, Wv, V, d.n}};
    attn::ProjProblem in3[3];
    for (int i = 0; i < 3; ++i) {
        in3[i] = pp;
        in3[i].a = ins_proj[i].x;
        in3[i].w = ins_proj[i].w;
        in3[i].out = ins_proj[i].o;
        in3[i].L = ins_proj[i].L;
        // a programmatic dependent of whatever ran before on the stream: only its
        // barrier set-up runs before that kernel completes
        in3[i].overlap_launch = true;
    }
    // the three input projections in one launch
    if (attn::launch_proj_multi(in3, 3, s) != cudaSuccess) return ATTN_ERR_CUDA;
    attn_dims ad{d.B, d.h, d.m, d.n, dk, ATTN_BF16};
    // the attention and the output projection each start as programmatic dependents of
    // the launch before them: their set-up overlaps its tail, and each waits for it to
    // complete before reading its output
    st = run(Q, K, V, key_lengths, mask_kind, scale, O, &ad, stream, ATTN_KERNEL_AUTO, nullptr, nullptr, -1, true);
    if (st != ATTN_OK) return st;
    pp.mode = attn::kProjOut;
    pp.a = O;
    pp.w = Wo;
    pp.out = out;
    pp.L = d.m;
    pp.K = d.h * dk;
    pp.N = d.d_model;
    pp.overlap_launch = true;
    return attn::launch_proj(pp, s) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

} // extern "C"

// ------------------------------------------------------------ host buffers
namespace {

constexpr int kHostChunksTarget = 8; // chunks per call (about: the cut follows (batch, head) slices)
constexpr int kHostComputeStreams = 2;
constexpr int kHostMaxChunks = 64;

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

struct HostPlan {
    size_t q_bytes, kv_bytes, len_off, ctr_off, total;
};

HostPlan host_plan(const attn_dims &d)
{
    const size_t esz = d.dtype == ATTN_BF16 ? 2 : 4;
    HostPlan p;
    p.q_bytes = static_cast<size_t>(d.B) * d.h * d.m * d.d_k * esz;
    p.kv_bytes = static_cast<size_t>(d.B) * d.h * d.n * d.d_k * esz;
    // [Q][K][V][out][lengths][one tile counter per compute stream]
    p.len_off = 2 * round256(p.q_bytes) + 2 * round256(p.kv_bytes);
    p.ctr_off = p.len_off + round256(4ull * d.B);
    p.total = p.ctr_off + kHostComputeStreams * attn::kWorkspaceBytes;
    return p;
}

// A chunk: batches [b0, b0 + nb) with all heads, or heads [h0, h0 + nh) of batch b0
// (nb == 1).  Either way its rows are contiguous in every tensor and its key
// lengths are lengths[b0 ...].
struct HostChunk {
    int b0, nb, h0, nh;
};

int host_chunks(const attn_dims &d, HostChunk *c)
{
    int k = 0;
    if (d.B >= kHostChunksTarget) {
        const int nb = (d.B + kHostChunksTarget - 1) / kHostChunksTarget;
        for (int b = 0; b < d.B; b += nb) c[k++] = {b, nb < d.B - b ? nb : d.B - b, 0, d.h};
    } else {
        int parts = (kHostChunksTarget + d.B - 1) / d.B;
        if (parts > d.h) parts = d.h;
        const int nh = (d.h + parts - 1) / parts;
        for (int b = 0; b < d.B; ++b)
            for (int h0 = 0; h0 < d.h; h0 += nh) c[k++] = {b, 1, h0, nh < d.h - h0 ? nh : d.h - h0};
    }
    return k;
}

// Streams and events of one device, made on first use and kept for the process.
struct HostDevice {
    std::mutex mu;
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr, comp[kHostComputeStreams] = {};
    cudaEvent_t start = nullptr, done = nullptr, ev_in[kHostMaxChunks] = {}, ev_comp[kHostMaxChunks] = {};
};
HostDevice g_host_devices[kMaxDevices];

cudaError_t host_device_setup(HostDevice &hd)
{
    if (hd.ready) return cudaSuccess;
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&hd.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&hd.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    for (auto &s : hd.comp)
        if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&hd.start, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&hd.done, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int i = 0; i < kHostMaxChunks; ++i) {
        if ((e = cudaEventCreateWithFlags(&hd.ev_in[i], cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&hd.ev_comp[i], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    hd.ready = true;
    return cudaSuccess;
}

} // namespace

extern "C" {

size_t attn_fwd_host_workspace_size(const attn_dims *dims)
{
    if (validate_dims(dims, 0, 1.f) != ATTN_OK) return 0;
    return host_plan(*dims).total;
}

attn_status attn_fwd_host(const void *Q, const void *K, const void *V, const int32_t *key_lengths, int mask_kind,
                          float scale, void *out, const attn_dims *dims, void *dev_workspace,
                          size_t dev_workspace_bytes, void *stream)
{
    if (dims == nullptr || Q == nullptr || K == nullptr || V == nullptr || out == nullptr) return ATTN_ERR_NULL;
    if ((mask_kind & ATTN_MASK_KEY_PADDING) && key_lengths == nullptr) return ATTN_ERR_NULL;
    attn_status st = validate_dims(dims, mask_kind, scale);
    if (st != ATTN_OK) return st;
    if (dev_workspace == nullptr) return ATTN_ERR_NULL;
    const attn_dims &d = *dims;
    const HostPlan plan = host_plan(d);
    if (dev_workspace_bytes < plan.total) return ATTN_ERR_SHAPE;
    if (!aligned(dev_workspace, 256)) return ATTN_ERR_ALIGN;
    if (overlaps(out, plan.q_bytes, Q, plan.q_bytes) || overlaps(out, plan.q_bytes, K, plan.kv_bytes) ||
        overlaps(out, plan.q_bytes, V, plan.kv_bytes))
        return ATTN_ERR_ALIAS;
    if ((mask_kind & ATTN_MASK_KEY_PADDING) && overlaps(out, plan.q_bytes, key_lengths, 4ull * d.B))
        return ATTN_ERR_ALIAS;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    HostDevice &hd = g_host_devices[dev];
    std::lock_guard<std::mutex> lock(hd.mu); // one call enqueues at a time: the events are reused
    if (host_device_setup(hd) != cudaSuccess) return ATTN_ERR_CUDA;

    const size_t esz = d.dtype == ATTN_BF16 ? 2 : 4;
    const size_t q_row = static_cast<size_t>(d.m) * d.d_k * esz; // bytes of one (batch, head) slice
    const size_t kv_row = static_cast<size_t>(d.n) * d.d_k * esz;
    HostChunk chunks[kHostMaxChunks];
    int nchunks = 1;
    chunks[0] = {0, d.B, 0, d.h};
    // chunks start at slice boundaries, which keep the 16-byte alignment the kernels need
    // only when a slice is a whole number of 16-byte units
    if (q_row % 16 == 0 && kv_row % 16 == 0) nchunks = host_chunks(d, chunks);
    uint8_t *ws = static_cast<uint8_t *>(dev_workspace);
    uint8_t *dq = ws, *dk = ws + round256(plan.q_bytes), *dv = dk + round256(plan.kv_bytes);
    uint8_t *dout = dv + round256(plan.kv_bytes);
    int32_t *dlen = reinterpret_cast<int32_t *>(ws + plan.len_off);
    uint8_t *ctr = ws + plan.ctr_off;
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    const uint8_t *hq = static_cast<const uint8_t *>(Q), *hk = static_cast<const uint8_t *>(K),
                  *hv = static_cast<const uint8_t *>(V);
    uint8_t *ho = static_cast<uint8_t *>(out);

    // everything already on the caller's stream comes first
    bool ok = cudaEventRecord(hd.start, user) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(hd.in, hd.start, 0) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(hd.out, hd.start, 0) == cudaSuccess;
    ok = ok && cudaMemsetAsync(ctr, 0, kHostComputeStreams * attn::kWorkspaceBytes, hd.in) == cudaSuccess;
    if (mask_kind & ATTN_MASK_KEY_PADDING)
        ok = ok && cudaMemcpyAsync(dlen, key_lengths, 4ull * d.B, cudaMemcpyHostToDevice, hd.in) == cudaSuccess;
    for (int c = 0; c < nchunks && ok; ++c) {
        const HostChunk &ch = chunks[c];
        const size_t bh0 = static_cast<size_t>(ch.b0) * d.h + ch.h0;
        const size_t units = static_cast<size_t>(ch.nb) * ch.nh;
        // inputs of chunk c, then its kernel as soon as they are in, then its output back
        ok = ok && cudaMemcpyAsync(dq + bh0 * q_row, hq + bh0 * q_row, units * q_row, cudaMemcpyHostToDevice,
                                   hd.in) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(dk + bh0 * kv_row, hk + bh0 * kv_row, units * kv_row, cudaMemcpyHostToDevice,
                                   hd.in) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(dv + bh0 * kv_row, hv + bh0 * kv_row, units * kv_row, cudaMemcpyHostToDevice,
                                   hd.in) == cudaSuccess;
        ok = ok && cudaEventRecord(hd.ev_in[c], hd.in) == cudaSuccess;
        cudaStream_t cs = hd.comp[c % kHostComputeStreams];
        ok = ok && cudaStreamWaitEvent(cs, hd.ev_in[c], 0) == cudaSuccess;
        if (!ok) break;
        attn_dims sub = d;
        sub.B = ch.nb;
        sub.h = ch.nh;
        st = attn_fwd_ws(dq + bh0 * q_row, dk + bh0 * kv_row, dv + bh0 * kv_row,
                         (mask_kind & ATTN_MASK_KEY_PADDING) ? dlen + ch.b0 : nullptr, mask_kind, scale,
                         dout + bh0 * q_row, &sub, cs, ctr + (c % kHostComputeStreams) * attn::kWorkspaceBytes,
                         attn::kWorkspaceBytes);
        if (st != ATTN_OK) break;
        ok = cudaEventRecord(hd.ev_comp[c], cs) == cudaSuccess;
        ok = ok && cudaStreamWaitEvent(hd.out, hd.ev_comp[c], 0) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(ho + bh0 * q_row, dout + bh0 * q_row, units * q_row, cudaMemcpyDeviceToHost,
                                   hd.out) == cudaSuccess;
    }
    // the caller's stream waits for the last copy back (which waited for every kernel)
    const bool joined = cudaEventRecord(hd.done, hd.out) == cudaSuccess &&
                        cudaStreamWaitEvent(user, hd.done, 0) == cudaSuccess;
    if (st != ATTN_OK) return st;
    return ok && joined ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_test_withheld_arrival(const void *Q, const void *K, const void *V, const int32_t *key_lengths,
                                       int mask_kind, float scale, void *out, const attn_dims *dims,
                                       uint64_t wait_ns, void *stream)
{
    const attn_status st = validate(Q, K, V, key_lengths, mask_kind, scale, out, dims);
    if (st != ATTN_OK) return st;
    const attn_dims &d = *dims;
    if (!tensor_core_head(d) || !attn::resident_fits(d.m, d.n, d.d_k)) return ATTN_ERR_UNSUPPORTED;
    if (wait_ns < 100000ull || wait_ns > 2000000000ull) return ATTN_ERR_VALUE;
    attn::Problem p;
    p.q = Q;
    p.k = K;
    p.v = V;
    p.key_lengths = (mask_kind & ATTN_MASK_KEY_PADDING) ? key_lengths : nullptr;
    p.out = out;
    p.lse = nullptr;
    p.B = d.B;
    p.h = d.h;
    p.m = d.m;
    p.n = d.n;
    p.d = d.d_k;
    p.mask_kind = mask_kind;
    p.scale = resolve_scale(scale, d.d_k);
    p.bf16 = true;
    attn::ResidentTestHook hook{wait_ns, 1};
    return attn::launch_resident(p, static_cast<cudaStream_t>(stream), &hook) == cudaSuccess ? ATTN_OK
                                                                                                 : ATTN_ERR_CUDA;
}

int attn_select_kernel(const attn_dims *dims, int mask_kind)
{
    if (validate_dims(dims, mask_kind, 1.0f) != ATTN_OK) return ATTN_KERNEL_AUTO;
    return auto_kernel(*dims);
}

attn_status attn_device_status(void *stream, int32_t *info)
{
    uint32_t code = 0, where = 0, bcode = 0, bwhere = 0;
    if (attn::flash_status_read_and_clear(static_cast<cudaStream_t>(stream), &code, &where) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (attn::bwd_status_read_and_clear(static_cast<cudaStream_t>(stream), &bcode, &bwhere) != cudaSuccess)
        return ATTN_ERR_CUDA;
    uint32_t pcode = 0, pwhere = 0;
    if (attn::proj_status_read_and_clear(static_cast<cudaStream_t>(stream), &pcode, &pwhere) != cudaSuccess)
        return ATTN_ERR_CUDA;
    uint32_t wcode = 0, wwhere = 0;
    if (attn::wide_status_read_and_clear(static_cast<cudaStream_t>(stream), &wcode, &wwhere) != cudaSuccess)
        return ATTN_ERR_CUDA;
    uint32_t rcode = 0, rwhere = 0;
    if (attn::resident_status_read_and_clear(static_cast<cudaStream_t>(stream), &rcode, &rwhere) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (code == 0 && rcode != 0) {
        code = rcode;
        where = 400 + rwhere; // resident-kernel wait sites are reported as 400 + site
    }
    if (code == 0 && wcode != 0) {
        code = wcode;
        where = 300 + wwhere; // wide-head wait sites are reported as 300 + site
    }
    if (code == 0 && bcode == 0 && pcode != 0) {
        code = pcode;
        where = 200 + pwhere; // projection wait sites are reported as 200 + site
    }
    if (code == 0 && bcode != 0) {
        code = bcode;
        where = 100 + bwhere; // backward wait sites are reported as 100 + site
    }
    if (info != nullptr) *info = static_cast<int32_t>(where);
    return code != 0 ? ATTN_ERR_DEVICE_TIMEOUT : ATTN_OK;
}

const char *attn_status_string(int status)
{
    switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "shape out of range (or causal mask with m != n)";
    case ATTN_ERR_DTYPE: return "unsupported dtype or head width";
    case ATTN_ERR_MASK: return "unknown mask bits";
    case ATTN_ERR_ALIGN: return "pointer not aligned (16 bytes for tensors, 4 for key_lengths)";
    case ATTN_ERR_UNSUPPORTED: return "the requested kernel cannot run this call";
    case ATTN_ERR_CUDA: return "CUDA runtime error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait; its output is incomplete";
    case ATTN_ERR_VALUE: return "scale must be finite and >= 0, or ATTN_SCALE_DEFAULT";
    case ATTN_ERR_ALIAS: return "out overlaps an input";
    case ATTN_ERR_SCRATCH: return "the call needs more scratch than attn_fwd_noalloc holds";
    default: return "unknown status";
    }
}

int32_t attn_version(void) { return (1 << 16) | 2; }

} // extern "C"
