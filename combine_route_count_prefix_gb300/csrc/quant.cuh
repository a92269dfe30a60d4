// quant.cuh -- the dynamic int8 quantisation code shared by the kernels that
// quantise rows (the FFN's per-row quantisations, the quantised dispatch).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half a = __float2half_rn(lo), b = __float2half_rn(hi);
    return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
}

// Dynamic int8 quantisation code of v with scale s (s = amax / 127): the
// round-half-even integer of the IEEE quotient v/s, clamped to [-127, 127];
// 0 when s == 0.  rs = 1/s rounded to nearest.
// Fast path: x = v * rs differs from the exact quotient by at most 2^-23
// relatively, i.e. by less than 1.6e-5 for |v/s| <= 128, so rint(x) equals
// rint(v/s) unless x lies within that distance of a half-integer.  Those
// rare cases (and non-finite x) take the IEEE division, so the code is the
// same as rint(__fdiv_rn(v, s)) for every input.
__device__ __forceinline__ float quant_code(float v, float s, float rs) {
    if (s == 0.0f) return 0.0f;
    const float x = __fmul_rn(v, rs);
    float q = rintf(x);
    if (!(fabsf(fabsf(x - q) - 0.5f) >= 3.0e-5f)) q = rintf(__fdiv_rn(v, s));
    return fminf(fmaxf(q, -127.0f), 127.0f);
}

}  // namespace moe
