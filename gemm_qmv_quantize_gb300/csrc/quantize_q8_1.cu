// quantize_q8_1.cu -- fp32 -> Q8_1 activation quantizer.
//
// MMVQ ("Machine Learning on NVIDIA CMP", sections "TL;DR" and "The DP2A patch")
// multiplies the weights' nibbles against int8 activations; the activation row is
// quantized per call into 32-element blocks {fp16 d8, fp16 s8, int8 q[32]}:
// d = max|x| / 127, q = clamp(round_half_away(x / d), -127, 127), s8 = d * sum q
// (q8_1_block.cuh, shared with the fused quantize + MMVQ prologue).
//
// A quad of lanes per block: lane p of the quad loads x[8p .. 8p+7] with two
// 16-byte loads (32 contiguous bytes per lane, 1 KB per warp), the maximum and
// the sum are two shuffles each, and the lane stores its 8 bytes of q.
#include "q8_1_block.cuh"
#include "qmv_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerCta = kThreads / 4;

__global__ void __launch_bounds__(kThreads) quantize_q8_1_kernel(const float *__restrict__ x,
                                                                uint8_t *__restrict__ xq, int64_t nblocks,
                                                                int vec_loads)
{
    grid_launch_dependents();
    const int part = threadIdx.x & 3;
    const int64_t blk = static_cast<int64_t>(blockIdx.x) * kBlocksPerCta + (threadIdx.x >> 2);
    grid_dependency_wait();   // x may be written by the preceding kernel
    const bool live = blk < nblocks;
    float v[8];
    const float *src = x + (live ? blk : 0) * 32 + 8 * part;
    if (vec_loads) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(src));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(src) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __ldg(src + i);
    }
    const Q8Quad r = q8_1_quantize_quad(v);   // all lanes take part in the shuffles
    if (!live) return;
    uint32_t *out = reinterpret_cast<uint32_t *>(xq + blk * 36);
    out[1 + 2 * part] = r.qlo;
    out[2 + 2 * part] = r.qhi;
    if (part == 0) out[0] = q8_1_d8_bits(r) | (q8_1_s8_bits(r) << 16);
}

}  // namespace

cudaError_t launch_quantize_q8_1(const float *x, void *xq, int M, int64_t K, cudaStream_t s)
{
    const int64_t nblocks = static_cast<int64_t>(M) * (K / 32);
    const int64_t grid = (nblocks + kBlocksPerCta - 1) / kBlocksPerCta;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = set_launch_overlap_attr(attr);
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(quantize_q8_1_kernel), 0);
    if (e != cudaSuccess) return e;
    route_hit(kRouteQuantizeQ8_1);
    const int vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
    return cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel, x, static_cast<uint8_t *>(xq), nblocks, vec);
}

}  // namespace qmv
