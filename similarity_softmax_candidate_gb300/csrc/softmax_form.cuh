// The range-safe form of the readout's logits and softmax, shared by the
// streaming, direct and scalar kernels (kernels.cu) and the projected
// readout (project.cu).
//
// The logits are z_k = a * s_k with a = scale / temperature and s_k the
// similarity: the cosine, each norm clamped at 1e-8, or the dot (PR #69
// "cuda: add a fused candidate-scoring kernel for CLM and Kev", opening
// table). The softmax only sees z_k - max_j z_j. The host splits a into a
// signed value scale w0 and a positive exponent scale (LogitForm), and a
// row's value is v_k = w s_k (w = w0 for the dot, w0 / max(|q|, eps) for the
// cosine), so that
//   z_k - max_j z_j = |a| (v_k - max_j v_j) / |w0| and
//   exp(z_k - max_j z_j) = 2^(kexp (v_k - max_j v_j)), kexp = |a| log2(e) / |w0|
// (change of base: e^x = 2^(x log2 e)). The parts are chosen so that
//   * v_k - max v is finite and <= 0, or -inf only where the exact exponent
//     is below -2^28 (exp is exactly 0 there too): for the cosine
//     |v_k| <= 1 (|c . q| <= |c| |q|); for the dot |w0| is 1, or 1/2 when
//     |a| < 2^-100, where the halving keeps the difference of two dots
//     finite;
//   * kexp (v_k - max v) cannot be NaN: kexp is finite (the host refuses
//     |a| > 2^126) and, with it, the product can only reach -inf.
// So no finite input gives NaN. What float32 cannot hold -- a dot or a
// squared norm beyond its range, or a non-finite input -- turns the row's
// value into NaN, which carries into the question's sum of exponentials;
// the kernels skip a question whose sum is NaN, leaving its probabilities
// unwritten, and set a device status bit.
#pragma once

#include <math.h>

namespace cs {
namespace form {

constexpr float kNormEps = 1e-8f;    // the cosine's norm clamp
constexpr float kNormEps2 = 1e-16f;  // its square: max(|c|, eps) = sqrt(max(|c|^2, eps^2))

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fc00000); }

// x itself when finite, NaN when x is infinite or NaN (x * 0 + x).
__device__ __forceinline__ float nan_unless_finite(float x) { return fmaf(x, 0.f, x); }

// v when g is finite, NaN otherwise (g * 0 + v), then NaN unless v is finite.
__device__ __forceinline__ float nan_unless_both_finite(float v, float g) {
    return nan_unless_finite(fmaf(g, 0.f, v));
}

// Per-question scale w of the values: w0 for the dot; w0 / max(|q|, eps)
// for the cosine, with qsq = |q|^2 (NaN when qsq is not finite, so that
// every row of the question is flagged).
__device__ __forceinline__ float value_scale(float w0, float qsq, bool cos) {
    if (!cos) return w0;
    return isfinite(qsq) ? w0 / fmaxf(sqrtf(qsq), kNormEps) : qnan();
}

// Value of a cosine row from its dot t and squared norm nsq; NaN when either
// left float32's range.
__device__ __forceinline__ float cos_value(float t, float nsq, float w) {
    const float n = fmaxf(nsq, kNormEps2);
    return nan_unless_both_finite(t * rsqrtf(n) * w, n);
}

// Value of a cosine row whose norm nrm (not squared) a separate pass staged.
__device__ __forceinline__ float staged_cos_value(float t, float nrm, float w) {
    const float n = fmaxf(nrm, kNormEps);
    return nan_unless_both_finite(t / n * w, n);
}

// Value of a dot row; NaN when the dot left float32's range.
__device__ __forceinline__ float dot_value(float t, float w) { return nan_unless_finite(t * w); }

// 2^y, the hardware's base-2 exponential (results below 2^-126 flush to 0).
__device__ __forceinline__ float exp2_approx(float y) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

// exp(z_k - M) for x = v_k - max v (<= 0).
__device__ __forceinline__ float softmax_term(float kexp, float x) { return exp2_approx(x * kexp); }

}  // namespace form
}  // namespace cs
