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

// v: the 8 consecutive values 8p..8p+7 of the block held by quad lane p = lane % 4.
// Every lane of the warp must call this together (it shuffles within quads).
__device__ __forceinline__ Q8Quad q8_1_quantize_quad(const float (&v)[8])
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    Q8Quad r;
    r.d = amax / 127.0f;   // IEEE division (the library is built without fast-math)
    // q = roundf(v / d) needs the correctly rounded quotient only where it decides
    // the rounding: v * fl(1/d) is within 2^-15 of fl(v / d) (|v / d| <= 127, two
    // roundings of 2^-24 relative each), so away from a tie (fraction farther than
    // 2^-13 from 1/2) both round to the same integer; near a tie, divide exactly.
    const float rcp = 1.0f / r.d;
    const bool fast = isfinite(rcp);
    int sum = 0;
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int q = 0;
        if (r.d != 0.0f) {
            float t = v[i] * rcp;
            const float a = fabsf(t);
            if (!fast || fabsf((a - floorf(a)) - 0.5f) < 0x1p-13f) t = v[i] / r.d;
            t = roundf(t);
            t = fminf(fmaxf(t, -127.0f), 127.0f);
            q = static_cast<int>(t);
        }
        sum += q;
        packed[i >> 2] |= (static_cast<uint32_t>(q) & 0xffu) << (8 * (i & 3));
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    r.qlo = packed[0];
    r.qhi = packed[1];
    r.sum = sum;
    return r;
}

__device__ __forceinline__ uint32_t q8_1_d8_bits(const Q8Quad &r) { return __half_as_ushort(__float2half_rn(r.d)); }

__device__ __forceinline__ uint32_t q8_1_s8_bits(const Q8Quad &r)
{
    return __half_as_ushort(__float2half_rn(r.d * static_cast<float>(r.sum)));
}

}  // namespace qmv
