// Per-group scale and cast arithmetic shared by the quantizer kernels.
//
// The amax of a group is taken on BF16 bit patterns: |x| is the pattern with
// the sign bit cleared, and for non-negative IEEE values the unsigned order of
// the patterns equals the numeric order, so an integer max is exact.  NaN
// patterns (exponent all ones, mantissa != 0) sort above infinity, which sorts
// above every finite value, so "amax pattern >= 0x7F80" detects a non-finite
// group.
//
// Scale exponents are read off the amax's exponent and mantissa fields; no
// logarithm is evaluated.  With amax = 1.m * 2^E (E = field - 127):
//  * UE8M0 round-up ("A Comprehensive FP8 Training Recipe ...", "What carries
//    the argument": scales rounded up to a power of two so the FP8 range is
//    never exceeded).  FMAX = 1.75 * 2^emax for both E4M3 (emax 8) and E5M2
//    (emax 15), so the smallest e with amax <= FMAX * 2^e is
//    E - emax, plus one when 1.m > 1.75, i.e. when the 7-bit mantissa field
//    exceeds 96.  Zero and subnormal amax give the clamp value -127.
//  * MX ("Characterization and Mitigation of Training Instabilities in
//    Microscaling Formats", "What carries the argument"): e = floor(log2 amax)
//    - emax = E - emax.
// Both are clamped to [-127, 127]; the scale byte is e + 127.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fp8hg {

enum { FMT_E4M3 = 0, FMT_E5M2 = 1 };

__device__ __forceinline__ uint32_t bf16_abs_max8(const uint4 &v) {
    const uint32_t m = 0x7FFF7FFFu;
    uint32_t a = __vmaxu2(__vmaxu2(v.x & m, v.y & m), __vmaxu2(v.z & m, v.w & m));
    return max(a & 0xFFFFu, a >> 16);
}

__device__ __forceinline__ int clamp_exp(int e) { return max(-127, min(127, e)); }

template <int FMT>
__device__ __forceinline__ int ue8m0_exponent(uint32_t amax_bits) {
    constexpr int emax = (FMT == FMT_E4M3) ? 8 : 15;
    const int ef = static_cast<int>(amax_bits >> 7);
    const int mf = static_cast<int>(amax_bits & 0x7F);
    if (ef == 0) return -127;
    return clamp_exp((ef - 127) - emax + (mf > 96 ? 1 : 0));
}

template <int FMT>
__device__ __forceinline__ int mx_exponent(uint32_t amax_bits) {
    constexpr int emax = (FMT == FMT_E4M3) ? 8 : 15;
    const int ef = static_cast<int>(amax_bits >> 7);
    if (ef == 0) return -127;
    return clamp_exp((ef - 127) - emax);
}

// The round-up rule on an FP32 amax pattern (sign cleared, finite): 1.m >
// 1.75 when the 23-bit mantissa field exceeds 0x600000; zero and subnormal
// amax give the clamp value -127 (any subnormal is below FMAX * 2^-127).
template <int FMT>
__device__ __forceinline__ int ue8m0_exponent_f32(uint32_t amax_bits) {
    constexpr int emax = (FMT == FMT_E4M3) ? 8 : 15;
    const int ef = static_cast<int>(amax_bits >> 23);
    const uint32_t mf = amax_bits & 0x7FFFFFu;
    if (ef == 0) return -127;
    return clamp_exp((ef - 127) - emax + (mf > 0x600000u ? 1 : 0));
}

// 2^n as a float for n in [-127, 127] (2^-127 is an FP32 subnormal).
__device__ __forceinline__ float pow2f(int n) {
    return (n >= -126) ? __uint_as_float(static_cast<uint32_t>(n + 127) << 23)
                       : __uint_as_float(1u << 22);
}

template <int FMT>
__device__ __forceinline__ uint32_t cvt2(float lo, float hi) {
    if constexpr (FMT == FMT_E4M3) return ptx::cvt_e4m3x2(lo, hi);
    else return ptx::cvt_e5m2x2(lo, hi);
}

// Largest finite magnitude of the format (for counting MX clamp events).
template <int FMT>
__device__ __forceinline__ float fp8_maxf() {
    return (FMT == FMT_E4M3) ? 448.0f : 57344.0f;
}

// Eight BF16 values (one 16-byte vector) -> eight FP8 codes (8 bytes).
// x * mul is exact: mul is a power of two and the product stays in FP32's
// normal range or underflows to values that round to zero in FP8 anyway.
// COUNT: add the number of scaled magnitudes beyond the format's maximum.
template <int FMT, bool COUNT>
__device__ __forceinline__ uint2 quant8(const uint4 &v, float mul, uint32_t &nsat) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16) * mul;
        const float hi = __uint_as_float(w[i] & 0xFFFF0000u) * mul;
        if constexpr (COUNT) {
            nsat += (fabsf(lo) > fp8_maxf<FMT>()) + (fabsf(hi) > fp8_maxf<FMT>());
        }
        p[i] = cvt2<FMT>(lo, hi);
    }
    return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

// Scale exponent for a group from its amax pattern; returns the scale byte and
// sets `mul` = 2^-e.  Non-finite groups give byte 0xFF (mul unused).
template <int FMT, bool MX>
__device__ __forceinline__ uint32_t group_scale(uint32_t amax_bits, float &mul) {
    if (amax_bits >= 0x7F80u) {
        mul = 0.0f;
        return 0xFFu;
    }
    const int e = MX ? mx_exponent<FMT>(amax_bits) : ue8m0_exponent<FMT>(amax_bits);
    mul = pow2f(-e);
    return static_cast<uint32_t>(e + 127);
}

constexpr uint32_t kNanCodes = 0x7F7F7F7Fu;

// How a group's scale is chosen and stored.
//  SCALE_UE8M0  power of two rounded up (one byte, e + 127)
//  SCALE_MX     power of two floor(log2 amax) - emax (one byte)
//  SCALE_F32    the FP32-scale variant: d = fl32(amax / FMAX) is stored and
//               x is multiplied by m = fl32(FMAX / amax) before the cast
//               (amax = 0: d = m = 1); both divisions correctly rounded.
enum { SCALE_UE8M0 = 0, SCALE_MX = 1, SCALE_F32 = 2 };

template <int FMT, int SM>
struct GroupScale {
    float mul;      // multiplier applied before the cast
    uint32_t byte;  // UE8M0 / MX scale byte (0xFF for a non-finite group)
    float d;        // FP32 scale (NaN for a non-finite group)
    bool nan;       // the group holds a NaN or an infinity
    __device__ __forceinline__ explicit GroupScale(uint32_t amax_bits) {
        nan = amax_bits >= 0x7F80u;
        if constexpr (SM == SCALE_F32) {
            const float fmax = fp8_maxf<FMT>();
            const float a = __uint_as_float(amax_bits << 16);  // BF16 -> FP32, exact
            byte = 0;
            if (nan) {
                d = __uint_as_float(0x7FC00000u);
                mul = 0.0f;
            } else if (a == 0.0f) {
                d = 1.0f;
                mul = 1.0f;
            } else {
                d = __fdiv_rn(a, fmax);
                mul = __fdiv_rn(fmax, a);
            }
        } else {
            byte = group_scale<FMT, SM == SCALE_MX>(amax_bits, mul);
            d = 0.0f;
        }
    }
    // The group's scale at element index idx of the caller's scale array
    // (bytes, or floats for SCALE_F32).
    __device__ __forceinline__ void store(uint8_t *s, int64_t idx) const {
        if constexpr (SM == SCALE_F32) reinterpret_cast<float *>(s)[idx] = d;
        else s[idx] = static_cast<uint8_t>(byte);
    }
};



}  // namespace fp8hg
