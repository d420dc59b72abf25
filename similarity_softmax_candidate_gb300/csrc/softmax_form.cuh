// The range-safe form of the readout's logits and softmax, shared by the
// streaming, direct and scalar kernels (kernels.cu) and the projected
// readout (project.cu).
//
// The logits are z_k = a * s_k with a = scale / temperature and s_k the
// similarity: the cosine, each norm clamped at 1e-8, or the dot (PR #69
// "cuda: add a fused candidate-scoring kernel for CLM and Kev", opening
// table). The softmax only sees z_k - max_j z_j. With v_k = sign(a) s_k / 2
// that difference is 2 |a| (v_k - max_j v_j), and
//   * |v_k| <= 1/2 for the cosine (s_k is divided by max(|q|, eps) and
//     |c . q| <= |c| |q|) and |v_k| <= FLT_MAX / 2 for the dot, so
//     v_k - max v is finite and <= 0;
//   * the product with 2 |a| (a finite: the host refuses a factor beyond
//     float32's range) can only overflow towards -inf, where exp is exactly 0.
// So no finite input gives NaN: nothing multiplies an overflowed factor by a
// similarity or subtracts two overflowed logits. What float32 cannot hold --
// a dot or squared norm beyond its range, or a non-finite input -- makes the
// row's value NaN, and the kernels skip a question with such a row, leaving
// its probabilities unwritten and setting a device status bit.
#pragma once

#include <math.h>

namespace cs {
namespace form {

constexpr float kNormEps = 1e-8f;    // the cosine's norm clamp
constexpr float kNormEps2 = 1e-16f;  // its square: max(|c|, eps) = sqrt(max(|c|^2, eps^2))

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fc00000); }

// Per-question scale w of the values: v_k = w * t_k for the dot, and
// w * t_k / max(|c_k|, eps) for the cosine, where qsq = |q|^2. When qsq is
// not finite, w is NaN, so that every row of the question is flagged.
__device__ __forceinline__ float value_scale(float factor, float qsq, bool cos) {
    const float h = copysignf(0.5f, factor);
    if (!cos) return h;
    return isfinite(qsq) ? h / fmaxf(sqrtf(qsq), kNormEps) : qnan();
}

// Value of a cosine row from its dot t and squared norm nsq; NaN when either
// left float32's range.
__device__ __forceinline__ float cos_value(float t, float nsq, float w) {
    const float v = t * rsqrtf(fmaxf(nsq, kNormEps2)) * w;
    return isfinite(nsq) && isfinite(v) ? v : qnan();
}

// Value of a cosine row whose norm nrm (not squared) was staged by a
// separate pass.
__device__ __forceinline__ float staged_cos_value(float t, float nrm, float w) {
    const float v = t / fmaxf(nrm, kNormEps) * w;
    return isfinite(nrm) && isfinite(v) ? v : qnan();
}

// Value of a dot row; NaN when the dot left float32's range.
__device__ __forceinline__ float dot_value(float t, float w) {
    const float v = t * w;
    return isfinite(v) ? v : qnan();
}

// exp(z_k - M) for x = v_k - max v (<= 0) and afac = |a|.
__device__ __forceinline__ float softmax_term(float afac, float x) { return __expf(2.f * (afac * x)); }

}  // namespace form
}  // namespace cs
