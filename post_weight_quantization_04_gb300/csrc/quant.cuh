// quant.cuh — the quantization grids shared by the GPTQ column loop and round-to-nearest.
//
// Symmetric grid (GPTQ's error-compensation loop page, `quantize_column`; GPTQ guide
// page, "Source code"): s = max(max|w|, 1e-12) / qmax, code = clip(round(w / s), -qmax,
// qmax), qmax = 2^(bits-1) - 1, dequantised code * s.
// Asymmetric grid (AutoGPTQ page, `quantize_weight`, `dequantize_weight` and the
// group-start parameters of `gptq_quantize_row`): s = (max - min) / maxq (1.0 if
// max == min), z = clamp(round(-min / s), 0, maxq), code = clamp(round(w / s + z), 0,
// maxq), maxq = 2^bits - 1, dequantised s * (code - z).
//
// Rounding is half-to-even. Scales are stored as fp32 and the grid is the stored scale.
// Every rounding decision equals the one taken in fp64 on the same fp32 inputs: the fast
// fp32 estimate is used only when it is at least 1e-3 away from a half-integer (its error
// is below 1e-4 for |w / s| < 1000, and beyond that the clamp decides); otherwise the
// quotient is recomputed in fp64 with IEEE division.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gptq {

struct Grid {
    float s;      // stored scale
    float inv_s;  // fp32 reciprocal, for the fast estimate only
    float z;      // zero point (integer valued; 0 for the symmetric grid)
};

__device__ __forceinline__ Grid sym_grid(float absmax, int qmax) {
    const double m = fmax((double)absmax, 1e-12);
    const float s = __double2float_rn(m / (double)qmax);
    return Grid{s, 1.0f / s, 0.0f};
}

__device__ __forceinline__ Grid asym_grid(float mn, float mx, int maxq) {
    const double sd = (mx > mn) ? ((double)mx - (double)mn) / (double)maxq : 1.0;
    const float s = __double2float_rn(sd);
    double z = rint(-(double)mn / (double)s);
    z = fmin(fmax(z, 0.0), (double)maxq);
    return Grid{s, 1.0f / s, (float)z};
}

// round(w / s (+ z)) with the quotient taken in fp64 (IEEE division); kept out of line so
// the rare near-half-point case does not weigh on the common path
__device__ __noinline__ float quotient_rint_f64(float w, float s, float z, int sym) {
    double td = (double)w / (double)s;
    if (!sym) td += (double)z;
    return (float)rint(td);
}

// Integer code of w on the grid, clamped to [lo, hi].
__device__ __forceinline__ int grid_code(float w, const Grid& g, bool sym, int lo, int hi) {
    const float t = sym ? w * g.inv_s : fmaf(w, g.inv_s, g.z);
    float r = rintf(t);
    if (fabsf(t - floorf(t) - 0.5f) < 1e-3f) r = quotient_rint_f64(w, g.s, g.z, sym ? 1 : 0);
    r = fminf(fmaxf(r, (float)lo), (float)hi);
    return (int)r;
}

// The same decision as grid_code, returned as an integer-valued float (no float<->int
// conversions on the caller's dependency chain). |t - rint(t)| > 0.499 is the same
// 1e-3-wide band around the half-points as grid_code's test.
__device__ __forceinline__ float grid_code_f(float w, const Grid& g, bool sym, float lo, float hi) {
    const float t = sym ? w * g.inv_s : fmaf(w, g.inv_s, g.z);
    float r = rintf(t);
    if (fabsf(t - r) > 0.499f) r = quotient_rint_f64(w, g.s, g.z, sym ? 1 : 0);
    return fminf(fmaxf(r, lo), hi);
}

__device__ __forceinline__ float grid_dequant_f(float code, const Grid& g, bool sym) {
    return sym ? code * g.s : g.s * (code - g.z);
}

__device__ __forceinline__ float grid_dequant(int code, const Grid& g, bool sym) {
    return sym ? (float)code * g.s : g.s * ((float)code - g.z);
}

}  // namespace gptq
