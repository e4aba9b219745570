// Softmax arithmetic on one 128-key tile of a query row, shared by the tcgen05
// attention kernels: the reference the exponentials are taken against and the
// bf16 weights with their sum.  Part of the blockwise (online) form of the row
// softmax in the attention equation ("Paper Deep Reading: Attention Is All You
// Need", §04).
#pragma once

#include <cstdint>
#include <math_constants.h>

#include "ptx.cuh"

namespace attn {

constexpr int kTileKeys = 128; // keys per tile

// A key tile's exponentials are taken against the row's running reference max
// and kept when their sum is at most 2^15 (so is every weight).  A larger finite
// sum is brought back below 2^8 by an exact power of two; an infinite one (the
// row's scores grew by 128 or more in log2 units) recomputes that row's scores.
constexpr float kFastSumLimit = 32768.0f;

// Row max of one key tile (x holds scores, or scores * scale * log2 e when
// `prescaled`), in log2 units; moves the reference up to it if it is larger.
// alpha rescales what was accumulated against the old reference (0 when there
// was none).
__device__ __forceinline__ void move_reference(const float (&x)[kTileKeys], bool prescaled, float sl2, float m_run,
                                               float &m_use, float &alpha, bool &grow)
{
    // four independent chains of three-input max
    float mx[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) mx[k] = fmaxf(x[2 * k], x[2 * k + 1]);
#pragma unroll
    for (int c = 8; c < kTileKeys; c += 8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) mx[k] = max3(mx[k], x[c + 2 * k], x[c + 2 * k + 1]);
    }
    float row_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    if (!prescaled) row_max *= sl2;
    const float m_new = fmaxf(m_run, row_max);
    grow = m_new > m_run;
    m_use = grow ? m_new : m_run;
    alpha = grow ? ex2(m_run - m_new) : 1.f;
}

// Weights exp2(x * scale * log2 e - m_use) of one key tile as bf16 pairs (column
// 2c in the low half of pk[c]); returns their sum (before rounding).  The
// exponent argument and the sum use packed two-lane fp32 ops.
__device__ __forceinline__ float weights_bf16(const float (&x)[kTileKeys], bool prescaled, float sl2, float m_use,
                                              uint32_t (&pk)[kTileKeys / 2])
{
    const float m_sub = (m_use == -CUDART_INF_F) ? 0.f : m_use;
    const uint64_t mul2 = prescaled ? f2(1.f, 1.f) : f2(sl2, sl2);
    const uint64_t sub2 = f2(-m_sub, -m_sub);
    uint64_t acc2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
    for (int c2 = 0; c2 < kTileKeys / 2; ++c2) {
        const int c = 2 * c2;
        float a0, a1;
        unf2(fma2(f2(x[c], x[c + 1]), mul2, sub2), a0, a1);
        const float e0 = ex2(a0), e1 = ex2(a1);
        acc2[c2 & 1] = add2(acc2[c2 & 1], f2(e0, e1));
        pk[c2] = pack_bf16x2(e0, e1);
    }
    float s0, s1, s2, s3;
    unf2(acc2[0], s0, s1);
    unf2(acc2[1], s2, s3);
    return (s0 + s1) + (s2 + s3);
}

// acc0 += the bf16 in the low half of pk, acc1 += the one in the high half (exact
// bf16 values widened to fp32 inside the add).
__device__ __forceinline__ void add_bf16_pair(float &acc0, float &acc1, uint32_t pk)
{
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1) : "r"(pk));
}

// The same weights, returning the sum of the weights as rounded: the values the
// P V product applies, so that dividing by it makes the output a weighted mean of
// exactly those.
__device__ __forceinline__ float weights_bf16_rounded(const float (&x)[kTileKeys], bool prescaled, float sl2,
                                                      float m_use, uint32_t (&pk)[kTileKeys / 2])
{
    const float m_sub = (m_use == -CUDART_INF_F) ? 0.f : m_use;
    const uint64_t mul2 = prescaled ? f2(1.f, 1.f) : f2(sl2, sl2);
    const uint64_t sub2 = f2(-m_sub, -m_sub);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c2 = 0; c2 < kTileKeys / 2; ++c2) {
        const int c = 2 * c2;
        float a0, a1;
        unf2(fma2(f2(x[c], x[c + 1]), mul2, sub2), a0, a1);
        const float e0 = ex2(a0), e1 = ex2(a1);
        pk[c2] = pack_bf16x2(e0, e1);
        add_bf16_pair(acc[(2 * c2) & 3], acc[(2 * c2 + 1) & 3], pk[c2]);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Scales one key tile's packed bf16 weights by f (a power of two, so exactly) and
// returns the sum of the scaled weights as rounded.
__device__ __forceinline__ float scale_and_sum(uint32_t (&pk)[kTileKeys / 2], float f)
{
    uint64_t acc2 = f2(0.f, 0.f);
#pragma unroll
    for (int c2 = 0; c2 < kTileKeys / 2; ++c2) {
        const float lo = __uint_as_float(pk[c2] << 16) * f, hi = __uint_as_float(pk[c2] & 0xffff0000u) * f;
        pk[c2] = pack_bf16x2(lo, hi);
        acc2 = add2(acc2, f2(lo, hi));
    }
    float s0, s1;
    unf2(acc2, s0, s1);
    return s0 + s1;
}

} // namespace attn
