// quantize_q8_1.cu -- fp32 -> Q8_1 activation quantizer.
//
// MMVQ ("Machine Learning on NVIDIA CMP", sections "TL;DR" and "The DP2A patch")
// multiplies int8 weights nibbles against int8 activations; the activation row is
// quantized per call into 32-element blocks {fp16 d8, fp16 s8, int8 q[32]}:
//   d = max|x| / 127, q = clamp(round_half_away(x / d), -127, 127), s8 = d * sum q,
// every step one IEEE fp32 operation (division, roundf), fp16 by round to nearest even.
//
// One warp per block: lane i owns x_i (a coalesced 128-byte load), the block
// maximum and the integer sum are warp reductions, four lanes' bytes are gathered
// into one 32-bit store.
#include "qmv_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

constexpr int kWarpsPerCta = 8;

__global__ void __launch_bounds__(kWarpsPerCta * 32) quantize_q8_1_kernel(const float *__restrict__ x,
                                                                         uint8_t *__restrict__ xq,
                                                                         int64_t nblocks)
{
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t blk = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
    grid_dependency_wait();   // x may be written by the preceding kernel
    if (blk >= nblocks) return;

    const float v = x[blk * 32 + lane];
    float amax = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));

    const float d = amax / 127.0f;                 // IEEE division (no fast-math)
    int q = 0;
    if (d != 0.0f) {
        float r = roundf(v / d);                   // ties away from zero
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        q = static_cast<int>(r);
    }
    int sum = q;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);

    uint8_t *out = xq + blk * 36;
    // gather bytes of lanes 4i..4i+3 into lane 4i
    uint32_t packed = static_cast<uint32_t>(q) & 0xffu;
    packed |= __shfl_down_sync(0xffffffffu, packed, 1) << 8;
    packed |= __shfl_down_sync(0xffffffffu, packed, 2) << 16;
    if ((lane & 3) == 0) reinterpret_cast<uint32_t *>(out + 4)[lane >> 2] = packed;
    if (lane == 0) {
        const uint32_t d8 = __half_as_ushort(__float2half_rn(d));
        const uint32_t s8 = __half_as_ushort(__float2half_rn(d * static_cast<float>(sum)));
        reinterpret_cast<uint32_t *>(out)[0] = d8 | (s8 << 16);
    }
}

}  // namespace

cudaError_t launch_quantize_q8_1(const float *x, void *xq, int M, int64_t K, cudaStream_t s)
{
    const int64_t nblocks = static_cast<int64_t>(M) * (K / 32);
    const int64_t grid = (nblocks + kWarpsPerCta - 1) / kWarpsPerCta;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kWarpsPerCta * 32);
    cfg.stream = s;
    route_hit(kRouteQuantizeQ8_1);
    return cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel, x, static_cast<uint8_t *>(xq), nblocks);
}

}  // namespace qmv
