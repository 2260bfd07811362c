// Double-float ("float-float") arithmetic for the rotation meshes whose
// transitions do not contract: a value is carried as an unevaluated sum
// hi + lo of two fp32 numbers (|lo| <= ulp(hi)/2), which holds about 48
// significant bits.  The building blocks are the classical error-free
// transformations (Dekker 1971; Knuth, TAOCP vol. 2, 4.2.2): the product
// a*b = p + e with e = fma(a, b, -p), and the sums TwoSum / FastTwoSum.
//
// cos_sin_ff gives cos(theta) and sin(theta) of an fp32 angle to about 1e-12
// absolute, each as a hi + lo pair:
//   1. theta = k pi/2 + r with |r| <= pi/4 (Cody & Waite 1980 reduction,
//      pi/2 split into three floats; r kept as hi + lo),
//   2. |r| = j/64 + r2 with |r2| <= 1/128, sin and cos of j/64 from a 52-entry
//      table (each as hi + lo, filled on the host in double precision),
//   3. sin r2 and 1 - cos r2 from their Taylor series (r2^5/120 and r2^4/24
//      are the last terms kept; the next ones are below 1e-15), combined
//      with the angle-addition formulas, and the quadrant k mod 4 applied.
#pragma once

#include <cmath>
#include <cuda_runtime.h>

namespace mgs {

struct SinCosTable {
    static constexpr int kEntries = 52;  // j = 0 .. 51 covers |r| <= pi/4 + rounding
    float4 e[kEntries];                  // (sin hi, sin lo, cos hi, cos lo) of j/64

    static SinCosTable build() {
        SinCosTable t;
        for (int j = 0; j < kEntries; ++j) {
            const double x = double(j) / 64.0, s = std::sin(x), c = std::cos(x);
            const float sh = float(s), ch = float(c);
            t.e[j] = make_float4(sh, float(s - double(sh)), ch, float(c - double(ch)));
        }
        return t;
    }
};

// a*b = p + e exactly
__host__ __device__ __forceinline__ void ff_two_prod(float a, float b, float &p, float &e) {
    p = a * b;
    e = fmaf(a, b, -p);
}
// a+b = s + e exactly, any magnitudes
__host__ __device__ __forceinline__ void ff_two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}
// a+b = s + e exactly when |a| >= |b| (or a == 0)
__host__ __device__ __forceinline__ void ff_fast_two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    e = b - (s - a);
}

// pi/2 = kPio2a + kPio2b + kPio2c + O(1e-23)
constexpr float kPio2a = 0x1.921fb6p+0f, kPio2b = -0x1.777a5cp-25f, kPio2c = -0x1.ee59dap-50f;
constexpr float kTwoOverPi = 0x1.45f306p-1f;

__host__ __device__ __forceinline__ void cos_sin_ff(float theta, const float4 *tab, float &ch, float &cl,
                                                   float &sh, float &sl) {
    // 1. r = theta - k pi/2.  theta - k*kPio2a is exact: both terms are
    // multiples of 2^-23 once |theta| >= 1 (for smaller theta, k = 0 or the
    // difference is a multiple of 2^-24 below 1), and the result is below 1.
    const float kf = rintf(theta * kTwoOverPi);
    const float r0 = fmaf(-kf, kPio2a, theta);
    float p, pe, rh, rl;
    ff_two_prod(kf, kPio2b, p, pe);
    ff_two_sum(r0, -p, rh, rl);
    rl = (rl - pe) - kf * kPio2c;
    ff_fast_two_sum(rh, rl, rh, rl);
    // 2. |r| = j/64 + r2 (j/64 exact; |r| - j/64 exact by Sterbenz's lemma)
    const float sg = rh < 0.f ? -1.f : 1.f;
    const float ar = fabsf(rh);
    int j = int(rintf(ar * 64.f));
    j = j < SinCosTable::kEntries - 1 ? j : SinCosTable::kEntries - 1;
    const float r2h = ar - float(j) * (1.f / 64.f);
    const float r2l = sg * rl;
    const float4 T = tab[j];  // S hi, S lo, C hi, C lo
    // 3. sin r2 = r2 - ds, cos r2 = 1 - dc, ds and dc small enough for fp32
    const float z = fmaf(2.f * r2h, r2l, r2h * r2h);              // r2^2
    const float dc = z * fmaf(-z, 1.f / 24.f, 0.5f);                // z/2 - z^2/24
    const float ds = r2h * z * fmaf(z, -1.f / 120.f, 1.f / 6.f);    // r2^3/6 - r2^5/120
    const float q = r2l - ds;                                       // sin r2 = r2h + q
    // sin|r| = S cos r2 + C sin r2 = (S + C r2h) + (C q - S dc + lo terms)
    float s1, s1e;
    ff_two_prod(T.z, r2h, p, pe);
    ff_fast_two_sum(T.x, p, s1, s1e);  // |S hi| >= 1/64 > |C r2h|, or S = 0
    const float slo = s1e + pe + T.y + fmaf(T.w, r2h, fmaf(T.z, q, -T.x * dc));
    float sin_h, sin_l;
    ff_fast_two_sum(s1, slo, sin_h, sin_l);
    // cos|r| = C cos r2 - S sin r2 = (C - S r2h) - (S q + C dc - lo terms)
    float c1, c1e;
    ff_two_prod(T.x, r2h, p, pe);
    ff_fast_two_sum(T.z, -p, c1, c1e);  // C hi >= cos(52/64) > |S r2h|
    const float clo = (c1e - pe + T.w) - fmaf(T.y, r2h, fmaf(T.x, q, T.z * dc));
    float cos_h, cos_l;
    ff_fast_two_sum(c1, clo, cos_h, cos_l);
    sin_h *= sg;
    sin_l *= sg;
    // quadrant: theta = r + k pi/2
    switch (int(kf) & 3) {
        case 0: sh = sin_h; sl = sin_l; ch = cos_h; cl = cos_l; break;
        case 1: sh = cos_h; sl = cos_l; ch = -sin_h; cl = -sin_l; break;
        case 2: sh = -sin_h; sl = -sin_l; ch = -cos_h; cl = -cos_l; break;
        default: sh = -cos_h; sl = -cos_l; ch = sin_h; cl = sin_l; break;
    }
}

// (x, y) <- (c x - s y, s x + c y) with every quantity a hi + lo pair.
__host__ __device__ __forceinline__ void ff_rot_fwd(float &xh, float &xl, float &yh, float &yl, float ch, float cl,
                                                    float sh, float sl) {
    float p1, e1, p2, e2, u, eu, v, ev;
    // c x - s y
    ff_two_prod(ch, xh, p1, e1);
    ff_two_prod(sh, yh, p2, e2);
    ff_two_sum(p1, -p2, u, eu);
    const float tu = (eu + (e1 - e2)) + (fmaf(ch, xl, cl * xh) - fmaf(sh, yl, sl * yh));
    // s x + c y
    ff_two_prod(sh, xh, p1, e1);
    ff_two_prod(ch, yh, p2, e2);
    ff_two_sum(p1, p2, v, ev);
    const float tv = (ev + (e1 + e2)) + (fmaf(sh, xl, sl * xh) + fmaf(ch, yl, cl * yh));
    ff_fast_two_sum(u, tu, xh, xl);
    ff_fast_two_sum(v, tv, yh, yl);
}

// (x, y) <- (c x + s y, -s x + c y), the transposed rotation.
__host__ __device__ __forceinline__ void ff_rot_bwd(float &xh, float &xl, float &yh, float &yl, float ch, float cl,
                                                    float sh, float sl) {
    ff_rot_fwd(xh, xl, yh, yl, ch, cl, -sh, -sl);
}

// x <- x + b (x a hi + lo pair, b an fp32 number)
__host__ __device__ __forceinline__ void ff_add(float &xh, float &xl, float b) {
    float s, e;
    ff_two_sum(xh, b, s, e);
    ff_fast_two_sum(s, e + xl, xh, xl);
}

}  // namespace mgs
