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
// Every rounding decision is the exact one for the fp32 inputs (the one fp64 takes: the
// quotient of two fp32 numbers is never within fp64 rounding of a half-point unless it
// is one). The fp32 estimate r = rint(w * (1/s) (+ z)) is off by at most one, and only
// next to a half-point; it is corrected by the signs of w - (r - z +- 1/2) s, each
// formed by one fma (exact product, a single rounding, so the sign is exact), with ties
// going to the even code. No branch, no fp64.
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

// zr: the range is widened to contain 0 first (the grid then has 0 as a point)
__device__ __forceinline__ Grid asym_grid(float mn, float mx, int maxq, bool zr) {
    if (zr) {
        mn = fminf(mn, 0.0f);
        mx = fmaxf(mx, 0.0f);
    }
    const double sd = (mx > mn) ? ((double)mx - (double)mn) / (double)maxq : 1.0;
    const float s = __double2float_rn(sd);
    double z = rint(-(double)mn / (double)s);
    z = fmin(fmax(z, 0.0), (double)maxq);
    return Grid{s, 1.0f / s, (float)z};
}

// round-half-even of w / s (+ z), exact, as an integer-valued float
__device__ __forceinline__ float grid_round(float w, const Grid& g, bool sym) {
    const float t = sym ? w * g.inv_s : fmaf(w, g.inv_s, g.z);
    const float r = rintf(t);
    const float m = sym ? r : r - g.z;              // the multiple of s that r stands for
    const float dh = fmaf(-(m + 0.5f), g.s, w);     // > 0: w / s lies above m + 1/2
    const float dl = fmaf(-(m - 0.5f), g.s, w);     // < 0: w / s lies below m - 1/2
    const float half = r * 0.5f;
    const bool odd = rintf(half) != half;
    const float up = (dh > 0.0f || (dh == 0.0f && odd)) ? 1.0f : 0.0f;
    const float dn = (dl < 0.0f || (dl == 0.0f && odd)) ? 1.0f : 0.0f;
    return r + up - dn;
}

// Integer code of w on the grid, clamped to [lo, hi].
__device__ __forceinline__ int grid_code(float w, const Grid& g, bool sym, int lo, int hi) {
    return (int)fminf(fmaxf(grid_round(w, g, sym), (float)lo), (float)hi);
}

// The same decision as grid_code, returned as an integer-valued float (no float<->int
// conversions on the caller's dependency chain).
__device__ __forceinline__ float grid_code_f(float w, const Grid& g, bool sym, float lo, float hi) {
    return fminf(fmaxf(grid_round(w, g, sym), lo), hi);
}

__device__ __forceinline__ float grid_dequant_f(float code, const Grid& g, bool sym) {
    return sym ? code * g.s : g.s * (code - g.z);
}

__device__ __forceinline__ float grid_dequant(int code, const Grid& g, bool sym) {
    return sym ? (float)code * g.s : g.s * ((float)code - g.z);
}

}  // namespace gptq
