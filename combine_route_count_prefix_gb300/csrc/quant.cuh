// quant.cuh -- the dynamic int8 quantisation code shared by the kernels that
// quantise rows (the FFN's per-row quantisations, the quantised dispatch).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

// Two floats -> one fp16x2 word (lo in the low half), round to nearest; exact
// for the integer codes in [-127, 127].
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Four integer-valued floats in [-128, 127] -> their two's-complement bytes in
// one word (a in the low byte).  Adding 1.5 * 2^23 is exact for them and leaves
// the integer in the low mantissa bits, so its low byte is the code's byte.
__device__ __forceinline__ uint32_t pack_i8x4(float a, float b, float c, float d) {
    const float kMagic = 12582912.0f;
    const uint32_t ua = __float_as_uint(__fadd_rn(a, kMagic));
    const uint32_t ub = __float_as_uint(__fadd_rn(b, kMagic));
    const uint32_t uc = __float_as_uint(__fadd_rn(c, kMagic));
    const uint32_t ud = __float_as_uint(__fadd_rn(d, kMagic));
    const uint32_t ab = __byte_perm(ua, ub, 0x0040);   // a.b0, b.b0 in bytes 0, 1
    const uint32_t cd = __byte_perm(uc, ud, 0x0040);
    return __byte_perm(ab, cd, 0x5410);
}

// Dynamic int8 quantisation codes of n values with scale s (s = amax / 127,
// amax the largest |v| of the row): for each value the round-half-even
// integer of the IEEE quotient v/s, clamped to [-127, 127]; all 0 when s == 0.
// rs = 1/s rounded to nearest.
// Fast path: x = v * rs differs from the exact quotient by at most 2^-23
// relatively, i.e. by less than 1.6e-5 for |v/s| <= 128, so rint(x) equals
// rint(v/s) unless x lies within that distance of a half-integer: the guard
// below keeps every x whose distance d = |x - rint(x)| to its integer is at
// most 0.5 - 3e-5.  For finite x, |x| <= 127 * (1 + 3 * 2^-24) < 127.5, so
// rint(x) needs no clamp.  The rare values beyond the guard (and non-finite
// x) take the IEEE division and the clamp, so every code is the same as
// clamp(rint(__fdiv_rn(v, s))).  The guard is tested for all n values before
// the one branch to the division, so the common case has no branch per value.
constexpr float kTieGuard = 0.5f - 3.0e-5f;

template <int n>
__device__ __forceinline__ void quant_codes(const float (&v)[n], float s, float rs, float (&q)[n]) {
    if (s == 0.0f) {
#pragma unroll
        for (int i = 0; i < n; ++i) q[i] = 0.0f;
        return;
    }
    bool slow = false;
#pragma unroll
    for (int i = 0; i < n; ++i) {
        const float x = __fmul_rn(v[i], rs);
        q[i] = rintf(x);
        slow = slow || !(fabsf(__fsub_rn(x, q[i])) <= kTieGuard);
    }
    if (slow) {
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float x = __fmul_rn(v[i], rs);
            if (!(fabsf(__fsub_rn(x, q[i])) <= kTieGuard))
                q[i] = fminf(fmaxf(rintf(__fdiv_rn(v[i], s)), -127.0f), 127.0f);
        }
    }
}

}  // namespace moe
