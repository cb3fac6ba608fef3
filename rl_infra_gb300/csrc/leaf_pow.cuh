// leaf_pow.cuh -- fl32(pow(x, alpha)) for a binary32 x > 0 and a binary64 alpha, without
// GB300's narrow binary64 pipe in the common case.
//
// The leaf of a priority is the binary64 power rounded to binary32.  On GB300 a binary64
// instruction occupies an SM's FP64 unit for ~19 cycles whatever the number of active lanes,
// and a binary64 pow is ~100 of them, so the power is evaluated here in double-float
// arithmetic on the FP32 pipe (pairs hi + lo of binary32 values, error-free transformations
// with fused multiply-add):
//   x = 2^e m, m in [1, 2);  k = the top 7 bits of m's fraction;  c_k ~ 1 / (1 + (k + 1/2)/128)
//   r = m c_k - 1 exactly (|r| <= 2^-8);  log2 x = e + log2(1/c_k) + log2(1 + r), the last by
//   the series r - r^2/2 + r^3/3 - r^4/4 + r^5/5 (truncation below 2^-50);
//   alpha = a0 + a1 + a2 exactly (three binary32 values); alpha e is split exactly into an
//   integer n and a fraction, so only |f| <= 1/2 + alpha needs double-float precision;
//   2^f = 2^(j/64) 2^g with |g| <= 1/128 and 2^g = exp(g ln 2) by its series to the 5th power.
// The value v carries a relative error well below 2^-44.  If every number within 2^-40 of v
// rounds to the same binary32 F, then x^alpha does, and so does any binary64 power within a
// few ulps of it: F is returned.  Otherwise (about one input in 2^15) and outside the normal
// range the binary64 pow decides.  The tables hold values computed in extended precision on
// the host.
#pragma once

#include <cmath>
#include <cstdint>
#include <cstring>

#if defined(__CUDACC__)
#define LP_HD __host__ __device__ __forceinline__
#else
#define LP_HD inline
#endif

namespace gbper {

struct LeafPowTables {
    float c[128];                 // c_k
    float lt_hi[128], lt_lo[128]; // log2(1 / c_k) as hi + lo
    float ex_hi[67], ex_lo[67];   // 2^(j/64), j = -33 .. 33, as hi + lo
    float log2e_hi, log2e_lo;     // 1 / ln 2
    float ln2_hi, ln2_lo;         // ln 2
};

struct LeafPowAlpha {
    double alpha;
    float a0, a1, a2;  // alpha = a0 + a1 + a2 exactly
    int kind;          // 0: general; 1: alpha == 0; 2: alpha == 1
};

// ---- bit access -------------------------------------------------------------------------------
LP_HD uint32_t lp_bits(float f)
{
#if defined(__CUDA_ARCH__)
    return __float_as_uint(f);
#else
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
#endif
}

LP_HD float lp_float(uint32_t u)
{
#if defined(__CUDA_ARCH__)
    return __uint_as_float(u);
#else
    float f;
    std::memcpy(&f, &u, 4);
    return f;
#endif
}

LP_HD float lp_fma(float a, float b, float c)
{
#if defined(__CUDA_ARCH__)
    return __fmaf_rn(a, b, c);
#else
    return std::fmaf(a, b, c);
#endif
}

LP_HD float lp_add(float a, float b)
{
#if defined(__CUDA_ARCH__)
    return __fadd_rn(a, b);
#else
    return a + b;
#endif
}

LP_HD float lp_sub(float a, float b)
{
#if defined(__CUDA_ARCH__)
    return __fsub_rn(a, b);
#else
    return a - b;
#endif
}

LP_HD float lp_mul(float a, float b)
{
#if defined(__CUDA_ARCH__)
    return __fmul_rn(a, b);
#else
    return a * b;
#endif
}

LP_HD float lp_rint(float a)
{
#if defined(__CUDA_ARCH__)
    return rintf(a);
#else
    return std::nearbyint(a);
#endif
}

// 2^k as a binary32, for -126 <= k <= 127
LP_HD float lp_pow2(int k) { return lp_float((uint32_t)(k + 127) << 23); }

// ---- double-float primitives (Dekker, Knuth) -------------------------------------------------
struct ff {
    float hi, lo;
};

LP_HD ff two_sum(float a, float b)
{
    const float s = lp_add(a, b);
    const float bb = lp_sub(s, a);
    const float e = lp_add(lp_sub(a, lp_sub(s, bb)), lp_sub(b, bb));
    return {s, e};
}

LP_HD ff fast_two_sum(float a, float b)  // |a| >= |b| or a == 0
{
    const float s = lp_add(a, b);
    return {s, lp_sub(b, lp_sub(s, a))};
}

LP_HD ff two_prod(float a, float b)
{
    const float p = lp_mul(a, b);
    return {p, lp_fma(a, b, -p)};
}

LP_HD ff ff_add(ff a, ff b)
{
    ff s = two_sum(a.hi, b.hi);
    const ff t = two_sum(a.lo, b.lo);
    s.lo = lp_add(s.lo, t.hi);
    s = fast_two_sum(s.hi, s.lo);
    s.lo = lp_add(s.lo, t.lo);
    return fast_two_sum(s.hi, s.lo);
}

LP_HD ff ff_add_f(ff a, float b)
{
    ff s = two_sum(a.hi, b);
    s.lo = lp_add(s.lo, a.lo);
    return fast_two_sum(s.hi, s.lo);
}

LP_HD ff ff_mul(ff a, ff b)
{
    ff p = two_prod(a.hi, b.hi);
    p.lo = lp_fma(a.hi, b.lo, p.lo);
    p.lo = lp_fma(a.lo, b.hi, p.lo);
    return fast_two_sum(p.hi, p.lo);
}

LP_HD ff ff_mul_f(ff a, float b)
{
    ff p = two_prod(a.hi, b);
    p.lo = lp_fma(a.lo, b, p.lo);
    return fast_two_sum(p.hi, p.lo);
}

// ---- the power ---------------------------------------------------------------------------------
// Returns true and the binary32 result in *out when the fast path decides; false when the
// caller must use the binary64 pow.  *v receives the double-float value (for tests).
LP_HD bool leaf_pow_fast(float x, const LeafPowAlpha &al, const LeafPowTables &tb, float *out,
                         ff *v = nullptr)
{
    const uint32_t xb = lp_bits(x);
    const int bexp = (int)((xb >> 23) & 0xFF);
    if (!(x > 0.0f) || bexp == 0 || bexp == 0xFF) return false;  // zero, subnormal, inf, nan
    if (al.kind == 1) {
        *out = 1.0f;
        return true;
    }
    if (al.kind == 2) {
        *out = x;
        return true;
    }
    const int e = bexp - 127;
    const float m = lp_float((xb & 0x007FFFFFu) | 0x3F800000u);  // [1, 2)
    const int k = (int)((xb >> 16) & 0x7F);
    // r = m c_k - 1, exactly, as a double-float
    const ff p = two_prod(m, tb.c[k]);
    const ff r = two_sum(lp_sub(p.hi, 1.0f), p.lo);
    // ln(1 + r) = r - r^2/2 + [r^3/3 - r^4/4 + r^5/5]
    const ff r2 = ff_mul(r, r);
    const float r3 = lp_mul(r2.hi, r.hi);
    const float tail = lp_mul(r3, lp_fma(r.hi, lp_fma(r.hi, 0.2f, -0.25f), 0.333333343f));
    // tail coefficients 1/3, -1/4, 1/5 in binary32: their rounding (<= 2^-24 relative of a term
    // below 2^-25) stays under 2^-49
    ff ln1p = ff_add(r, ff{-0.5f * r2.hi, -0.5f * r2.lo});
    ln1p = ff_add_f(ln1p, tail);
    // F = log2(1/c_k) + log2(1 + r), |F| <= 1
    const ff F = ff_add(ff{tb.lt_hi[k], tb.lt_lo[k]}, ff_mul(ln1p, ff{tb.log2e_hi, tb.log2e_lo}));
    // alpha e = sum of exact products a_i e, split into an integer and a fraction
    const float ef = (float)e;
    const ff q0 = two_prod(al.a0, ef), q1 = two_prod(al.a1, ef), q2 = two_prod(al.a2, ef);
    const float n1 = lp_rint(q0.hi);
    ff frac = two_sum(lp_sub(q0.hi, n1), q0.lo);
    frac = ff_add(frac, q1);
    frac = ff_add(frac, q2);
    // alpha F
    ff aF = ff_mul(ff{al.a0, al.a1}, F);
    aF = ff_add_f(aF, lp_mul(al.a2, F.hi));
    ff y = ff_add(frac, aF);  // |y| <= 1/2 + alpha + tiny
    const float n2 = lp_rint(y.hi);
    y = fast_two_sum(lp_sub(y.hi, n2), y.lo);
    const float nf = lp_add(n1, n2);
    if (!(nf > -140.0f && nf < 140.0f)) return false;
    const int n = (int)nf;
    // 2^y = 2^(j/64) exp(g ln 2), g = y - j/64
    const float jf = lp_rint(lp_mul(y.hi, 64.0f));
    const int j = (int)jf;
    if (j < -33 || j > 33) return false;
    const ff g = fast_two_sum(lp_sub(y.hi, lp_mul(jf, 0.015625f)), y.lo);
    const ff z = ff_mul(g, ff{tb.ln2_hi, tb.ln2_lo});
    // exp(z) = 1 + z + z^2/2 + [z^3/6 + z^4/24 + z^5/120]
    const ff z2 = ff_mul(z, z);
    const float z3 = lp_mul(z2.hi, z.hi);
    const float ztail = lp_mul(z3, lp_fma(z.hi, lp_fma(z.hi, 0.00833333377f, 0.0416666679f), 0.166666672f));
    ff ez = ff_add_f(ff{1.0f, 0.0f}, z.hi);
    ez = ff_add_f(ez, z.lo);
    ez = ff_add(ez, ff{0.5f * z2.hi, 0.5f * z2.lo});
    ez = ff_add_f(ez, ztail);
    ff val = ff_mul(ff{tb.ex_hi[j + 33], tb.ex_lo[j + 33]}, ez);
    // scale by 2^n; the result must stay a normal binary32 with room for the rounding test
    const int scale_exp = (int)((lp_bits(val.hi) >> 23) & 0xFF) - 127 + n;
    if (scale_exp < -120 || scale_exp > 126) return false;
    float s1, s2;
    if (n >= 0) {
        s1 = lp_pow2(n / 2);
        s2 = lp_pow2(n - n / 2);
    } else {
        s1 = lp_pow2(-((-n) / 2));
        s2 = lp_pow2(n + (-n) / 2);
    }
    val.hi = lp_mul(lp_mul(val.hi, s1), s2);
    val.lo = lp_mul(lp_mul(val.lo, s1), s2);
    if (v) *v = val;
    // rounding test: everything within 2^-40 of val must round to one binary32
    const float d = lp_mul(val.hi, 9.094947017729282e-13f);  // 2^-40
    const float lo = lp_add(val.hi, lp_sub(val.lo, d));
    const float hi = lp_add(val.hi, lp_add(val.lo, d));
    if (lo != hi) return false;
    *out = lp_add(val.hi, val.lo);
    return true;
}

// ---- host side: tables and alpha split ---------------------------------------------------------

inline void lp_split(long double v, float *hi, float *lo)
{
    *hi = (float)v;
    *lo = (float)(v - (long double)*hi);
}

inline LeafPowTables make_leaf_pow_tables()
{
    LeafPowTables t;
    for (int k = 0; k < 128; ++k) {
        const long double mk = 1.0L + ((long double)k + 0.5L) / 128.0L;
        t.c[k] = (float)(1.0L / mk);
        lp_split(-log2l((long double)t.c[k]), &t.lt_hi[k], &t.lt_lo[k]);
    }
    for (int j = -33; j <= 33; ++j) lp_split(exp2l((long double)j / 64.0L), &t.ex_hi[j + 33], &t.ex_lo[j + 33]);
    const long double ln2 = logl(2.0L);
    lp_split(1.0L / ln2, &t.log2e_hi, &t.log2e_lo);
    lp_split(ln2, &t.ln2_hi, &t.ln2_lo);
    return t;
}

inline LeafPowAlpha make_leaf_pow_alpha(double alpha)
{
    LeafPowAlpha a;
    a.alpha = alpha;
    a.a0 = (float)alpha;
    a.a1 = (float)(alpha - (double)a.a0);
    a.a2 = (float)(alpha - (double)a.a0 - (double)a.a1);
    a.kind = alpha == 0.0 ? 1 : (alpha == 1.0 ? 2 : 0);
    return a;
}

}  // namespace gbper
