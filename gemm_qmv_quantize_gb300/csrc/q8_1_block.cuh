// q8_1_block.cuh -- Q8_1 quantization of one 32-value block by a quad of lanes
// (8 values per lane), shared by the standalone quantizer and the fused
// quantize + MMVQ prologue so that both produce the same bytes.
//
// Per block, every step one IEEE fp32 operation: d = max|x| / 127 (division),
// q = clamp(roundf(x / d), -127, 127) (ties away from zero), d8 = fp16_rn(d),
// s8 = fp16_rn(d * (float)sum q). The maximum and the integer sum are exact in
// any order, so the split over four lanes changes no result.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace qmv {

struct Q8Quad {
    uint32_t qlo, qhi;   // this lane's 8 quantized values, packed int8 (element order)
    float d;             // the block scale (fp32, before fp16 rounding)
    int sum;             // sum of the block's 32 values of q (every lane of the quad)
};

// Four int32 in [-127, 127] packed as int8 bytes, element order.
__device__ __forceinline__ uint32_t pack_s8x4(int a, int b, int c, int d)
{
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// v: the 8 consecutive values 8p..8p+7 of the block held by quad lane p = lane % 4.
// Every lane of the warp must call this together (it shuffles within quads).
//
// q = roundf(x / d) needs the correctly rounded quotient only where it decides the
// rounding. |x / d| <= 127 (1 + 2^-23), and x * fl(1/d) is within 2^-15 of fl(x / d)
// (two roundings of at most 2^-24 relative each), so when x * fl(1/d) lies farther
// than 2^-13 from a half-integer both round to the same integer, and there round to
// nearest (rint) and round half away (roundf) agree. Near a tie, or when 1/d
// overflows, the value is recomputed with the IEEE quotient and roundf. The clamp
// to [-127, 127] never binds: the largest quotient rounds to 127.
__device__ __forceinline__ Q8Quad q8_1_quantize_quad(const float (&v)[8])
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    Q8Quad r;
    r.d = amax / 127.0f;   // IEEE division (the library is built without fast-math)
    const float inv = 1.0f / r.d;
    const bool fast = isfinite(inv);
    const float rcp = r.d == 0.0f ? 0.0f : inv;   // d == 0: every q is 0
    int q[8];
    uint32_t slow = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float t = v[i] * rcp;
        const float n = rintf(t);
        q[i] = static_cast<int>(n);
        if (fabsf(t - n) > 0.5f - 0x1p-13f) slow |= 1u << i;
    }
    if (!fast && r.d != 0.0f) slow = 0xffu;
    if (slow) {   // rare: decide the rounding with the IEEE quotient
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (slow & (1u << i)) q[i] = static_cast<int>(fminf(fmaxf(roundf(v[i] / r.d), -127.0f), 127.0f));
    }
    r.qlo = pack_s8x4(q[0], q[1], q[2], q[3]);
    r.qhi = pack_s8x4(q[4], q[5], q[6], q[7]);
    int sum = __dp4a(static_cast<int>(r.qlo), 0x01010101, __dp4a(static_cast<int>(r.qhi), 0x01010101, 0));
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    r.sum = sum;
    return r;
}

__device__ __forceinline__ uint32_t q8_1_d8_bits(const Q8Quad &r) { return __half_as_ushort(__float2half_rn(r.d)); }

__device__ __forceinline__ uint32_t q8_1_s8_bits(const Q8Quad &r)
{
    return __half_as_ushort(__float2half_rn(r.d * static_cast<float>(r.sum)));
}

}  // namespace qmv
