// rotary.cuh -- rotation of one pair of the decoupled positional key in the append kernels.
//
// Pair (2i, 2i+1) of k^R = x W^KR turns by theta = pos * base^(-2i/d_rope) ("Embeddings II:
// MLA & Architectural Choices", decoupled RoPE): (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos).
// Positions reach 2^17, so theta (up to ~1.3e5 rad) needs the inverse frequency to ~1e-13 and
// the angle in double; sine, cosine and the products must hold the result well inside one bf16
// ulp of the exact rotation.  GB300's FP64 pipe is narrow, so this avoids double transcendental
// calls:
//   - base^(-j/m) (j = i, m = d_rope / 2) by two Newton steps in double on y^m base^j = 1 from
//     an fp32 seed: y <- y (1 - (y^m base^j - 1) / m) has error (m + 1)/2 e^2 after a step, so a
//     seed within ~2e-6 ends within a few double ulps;
//   - the angle as a fraction of a turn in double, reduced to [0, 1);
//   - sine and cosine in fp32 of that fraction (rounded to fp32, |error| <= 2^-25 of a turn),
//     corrected to first order in double by the rounding residual (second-order term < 2e-14);
//     what remains is the fp32 functions' own error, ~1e-7;
//   - the products in double, rounded to fp32 like every other column.
#pragma once

#include <cuda_runtime.h>
#include <math.h>

namespace lrkv {

// x^e for an integer e >= 0, by binary powering (a few roundings of double precision).
__device__ __forceinline__ double rope_ipow(double x, int e) {
    double r = 1.0;
    while (e > 0) {
        if (e & 1) r *= x;
        x *= x;
        e >>= 1;
    }
    return r;
}

// base^(-2i / d_rope) in double.
__device__ __forceinline__ double rope_inv_freq(int i, int d_rope, float base) {
    if (i == 0) return 1.0;
    const int m = d_rope / 2;
    const double P = rope_ipow((double)base, i);  // base^j, j = i
    if (!(P < 1e290)) return pow((double)base, -2.0 * i / d_rope);  // beyond the Newton form's range
    // 1/m exactly (m is a power of two for the supported widths; else one division)
    const double inv_m = (m & (m - 1)) == 0 ? __hiloint2double((1023 - (__ffs(m) - 1)) << 20, 0) : 1.0 / m;
    double y = (double)exp2f(-(float)i / (float)m * log2f(base));
    for (int s = 0; s < 2; ++s) {
        const double t = rope_ipow(y, m) * P;  // ~1
        y = fma(-y, (t - 1.0) * inv_m, y);
    }
    return y;
}

// Cosine and sine of the angle pos * inv_freq, inv_freq = rope_inv_freq(i, ...) of the pair.
__device__ __forceinline__ void rope_cos_sin(double inv_freq, int pos, double& cs, double& sn) {
    const double turns = (double)pos * inv_freq * 0.15915494309189533577;  // / 2 pi
    const double fr = turns - floor(turns);
    const float f = (float)fr;
    float sf, cf;
    sincospif(2.0f * f, &sf, &cf);
    const double dl = (fr - (double)f) * 6.283185307179586477;  // residual angle, rad
    sn = fma(dl, (double)cf, (double)sf);
    cs = fma(-dl, (double)sf, (double)cf);
}

// The fp32 pair (x0, x1) turned by the angle whose cosine and sine are cs, sn.
__device__ __forceinline__ void rope_apply(float& x0, float& x1, double cs, double sn) {
    const double y0 = (double)x0 * cs - (double)x1 * sn;
    const double y1 = (double)x0 * sn + (double)x1 * cs;
    x0 = (float)y0;
    x1 = (float)y1;
}

// Rotate the fp32 pair (x0, x1) by pos * inv_freq.
__device__ __forceinline__ void rope_rotate_f(float& x0, float& x1, double inv_freq, int pos) {
    double cs, sn;
    rope_cos_sin(inv_freq, pos, cs, sn);
    rope_apply(x0, x1, cs, sn);
}

// Rotate the fp32 pair (x0, x1) = columns (2i, 2i+1) of k^R at position pos.
__device__ __forceinline__ void rope_rotate(float& x0, float& x1, int i, int d_rope, int pos, float base) {
    rope_rotate_f(x0, x1, rope_inv_freq(i, d_rope, base), pos);
}

}  // namespace lrkv
