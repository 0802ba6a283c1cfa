// quant_math.cuh -- the element path of the online E4M3 quantizers, shared by
// the standalone quantizers (quant.cu) and the GEMM's fused activation
// quantizer (gemm.cu): one FP32 scale per group, s = fl32(amax / 448), codes
// E4M3_RNE_satfinite(fl32(x / s)) with both divisions rounded to nearest.
// DeepSeek-V3 FP8 post (innerforce.co.kr), fine-grained quantization,
// Figure 7 (a); "Unified E4M3 format in DeepSeek-V3" (codingmall.com),
// Dynamic Scaling and Online Quantization.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fp8fg {
namespace {

FP8FG_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
FP8FG_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Division by the group scale.  The element code needs fl32(x / s) exactly
// (an IEEE round-to-nearest quotient).  For a normal scale it is computed
// with the reciprocal correction of Markstein ("Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 1990):
// with r = RN(1/s) (correctly rounded reciprocal, computed once per group)
// and q = RN(x r), which is within one ulp of x / s, the remainder
// x - s q is exact in one FMA and RN(q + (x - s q) r) is the correctly
// rounded quotient.  The remainder stays exact (no underflow) whenever
// |x / s| >= 2^-11 and s >= 2^-90; smaller quotients all encode to a signed
// zero in E4M3 (its smallest magnitude is 2^-9, the tie to zero at 2^-10),
// and the sign of the quotient is the sign of x (s > 0), which quant4 puts
// into the codes.  Scales below 2^-90 fall back to the full IEEE division.
// Bit-exactness against the oracle's IEEE division is tested.
struct GroupScale {
    float s, r;
    int mode;  // 0: s == 0 (codes keep only the sign), 1: reciprocal correction, 2: IEEE division
    FP8FG_DEV explicit GroupScale(float scale) : s(scale), r(0.0f) {
        if (s == 0.0f) {
            mode = 0;
        } else if (s >= 0x1p-90f) {
            mode = 1;
            r = __frcp_rn(s);
        } else {
            mode = 2;
        }
    }
};

// Four values -> four E4M3 codes (x0 in the lowest byte), for a group whose
// scale has mode kMode.  The quotients by the reciprocal correction are
// computed two lanes at a time (packed FP32; each lane rounds exactly as the
// scalar operations).  The sign of each code is taken from x's sign bit, ORed
// in at the end: a nonzero quotient already carries x's sign, and a quotient
// that rounds to zero must encode as a signed zero (0x80 for negative x),
// which is what the OR gives.  A zero scale leaves only the signs.  `signs`
// holds x_k's sign bit at bit 8k+7.  The mode is a template parameter: a
// caller branches once per group (with_mode) and the group's quads are then
// straight-line code the compiler interleaves -- with a branch inside every
// quad, each quad's dependent chain (multiply, two FMAs, conversion) ran
// after the previous one (measured: 0.6 us for the 32 codes of one thread).
template <int kMode>
FP8FG_DEV uint32_t quant4(float x0, float x1, float x2, float x3, uint32_t signs, const GroupScale& g) {
    if (kMode == 0) return signs;
    uint32_t lo, hi;
    if (kMode == 1) {
        // q = RN(x r); rem = x - s q (exact, one FMA); q' = RN(q + rem r)
        float q0 = x0, q1 = x1, q2 = x2, q3 = x3;
        mul2(q0, q1, g.r, g.r);
        mul2(q2, q3, g.r, g.r);
        float e0 = x0, e1 = x1, e2 = x2, e3 = x3;
        fma2(e0, e1, q0, q1, -g.s, -g.s);
        fma2(e2, e3, q2, q3, -g.s, -g.s);
        fma2(q0, q1, e0, e1, g.r, g.r);
        fma2(q2, q3, e2, e3, g.r, g.r);
        lo = cvt_e4m3x2(q0, q1);
        hi = cvt_e4m3x2(q2, q3);
    } else {
        lo = cvt_e4m3x2(__fdiv_rn(x0, g.s), __fdiv_rn(x1, g.s));
        hi = cvt_e4m3x2(__fdiv_rn(x2, g.s), __fdiv_rn(x3, g.s));
    }
    return (lo | (hi << 16)) | signs;
}

// Four FP32 values.
template <int kMode>
FP8FG_DEV uint32_t quant_quad(float a, float b, float c, float d, const GroupScale& g) {
    const uint32_t ab = __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x0073);
    const uint32_t cd = __byte_perm(__float_as_uint(c), __float_as_uint(d), 0x0073);
    return quant4<kMode>(a, b, c, d, __byte_perm(ab, cd, 0x5410) & 0x80808080u, g);
}

// Four BF16 values in two words (value 2i in the low half of word i, 2i+1 in
// the high half); the high byte of each BF16 value holds its sign bit.
template <int kMode>
FP8FG_DEV uint32_t quant_quad_bf16(uint32_t w0, uint32_t w1, const GroupScale& g) {
    return quant4<kMode>(bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1), __byte_perm(w0, w1, 0x7531) & 0x80808080u,
                         g);
}

template <int V>
struct ModeTag {
    static constexpr int value = V;
};

// Calls f(ModeTag<mode>{}) for the group's scale mode: the one branch of a
// group, outside the code that quantizes its elements.
template <class F>
FP8FG_DEV void with_mode(const GroupScale& g, F&& f) {
    if (g.mode == 1)
        f(ModeTag<1>{});
    else if (g.mode == 0)
        f(ModeTag<0>{});
    else
        f(ModeTag<2>{});
}

constexpr int kGroup = 128;

// Max |x| of the 128 BF16 values a lane quad holds (32 per lane), as in
// group_amax_bf16.
FP8FG_DEV float quad_amax_bf16(const uint4 (&v)[4]) {
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        m = __vmaxu2(m, __vmaxu2(__vmaxu2(v[k].x & 0x7FFF7FFFu, v[k].y & 0x7FFF7FFFu),
                                 __vmaxu2(v[k].z & 0x7FFF7FFFu, v[k].w & 0x7FFF7FFFu)));
    // xor < 4 stays inside the quad that owns the group
    m = __vmaxu2(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = __vmaxu2(m, __shfl_xor_sync(0xffffffffu, m, 1));
    const uint32_t hi = m >> 16, lo = m & 0xFFFFu;
    return __uint_as_float((hi > lo ? hi : lo) << 16);
}

}  // namespace
}  // namespace fp8fg
