// exp2dd.cuh -- 2^x to about 1e-9 relative, as an unevaluated pair of
// floats, for the entries whose probability is large enough that the
// special-function unit's few-ulp error would move the sampled token.
//
// Method: the table-driven reduction of Tang ("Table-driven implementation
// of the exponential function in IEEE floating-point arithmetic", ACM TOMS
// 15(2), 1989), in base 2:  x = n + j/128 + f  with n, j integers,
// 0 <= j < 128 and |f| <= 1/256;  2^x = 2^n * 2^(j/128) * e^(f ln 2).
// 2^(j/128) comes from a 128-entry table of (hi, lo) float pairs filled by
// the host in double precision; e^t - 1 for |t| = |f ln 2| <= 0.0028 is its
// Taylor series t + t^2/2 + t^3/6 (the next term is below 2.3e-12).
#pragma once
#include <cstdint>

namespace specv {

// The (hi, lo) table of 2^(j/128), j = 0..127; one copy per device, written
// by the host when a handle is created on that device.  (The library is a
// single translation unit, so the definition lives here.)
__device__ float2 g_exp2_table[128];

constexpr float kLn2 = 0.693147180559945309f;

// 2^(xh + xl) for xh <= 0 (|xl| tiny compared with 1/256).  Returns (eh, el)
// with eh + el = 2^x to ~1e-9 relative; eh is a table entry times 2^n.
// Arguments below -125 are raised to -125 (the result is then < 2.4e-38,
// negligible next to the sums it enters).
__device__ __forceinline__ float2 exp2dd(float xh, float xl, const float2* tab) {
    xh = fmaxf(xh, -125.0f);
    const float kf = rintf(xh * 128.0f);
    const int K = static_cast<int>(kf);
    float f = fmaf(kf, -0.0078125f, xh);  // exact: xh and K/128 are close
    f = f + xl;
    const float t = f * kLn2;
    const float h = fmaf(t, 0.16666667f, 0.5f);
    const float P = fmaf(t * t, h, t);  // e^t - 1
    const int j = K & 127;
    const int n = K >> 7;  // floor(K / 128)
    const float2 T = tab[j];
    const float lo = fmaf(T.x, P, T.y);
    const float scale = __int_as_float((n + 127) << 23);
    return make_float2(T.x * scale, lo * scale);
}

}  // namespace specv
