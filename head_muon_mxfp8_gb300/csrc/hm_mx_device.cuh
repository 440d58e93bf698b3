// Device helpers of G (MXFP8 quantization) shared by the requant kernels and
// the fused Newton-Schulz epilogue.  OCP Microscaling format (cited by the
// SS-HSDP paper as [28]): a 1x32 block shares the UE8M0 scale 2^e with
// e = clamp(floor(log2 amax) - 8, -127, 127); elements are E4M3.
#pragma once

#include <cstdint>

namespace hm {

// floor(log2 amax) read exactly from the fp32 bit pattern (subnormals
// included), minus the E4M3 emax 8, clamped to [-127, 127]; amax = 0 -> -127.
__device__ __forceinline__ int mx_scale_exponent(float amax) {
    const uint32_t bits = __float_as_uint(amax);
    const int ex = static_cast<int>(bits >> 23);
    int fl;
    if (ex == 0) {
        const uint32_t mant = bits & 0x7FFFFFu;
        if (mant == 0) return -127;
        fl = (31 - __clz(static_cast<int>(mant))) - 149;
    } else {
        fl = ex - 127;
    }
    const int e = fl - 8;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// 2^-e for e in [-127, 119] (always a normal fp32).
__device__ __forceinline__ float mx_inv_scale(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

}  // namespace hm
