// wq_mma.cu -- NVFP4 W4A16 and FP8 W8A16 skinny GEMM, M = 1..8 activation rows.
//
// QPN2 / QPN8 of "v100-skinny README", section "How QPN works": packed weights stay
// packed through HBM and are decoded only in registers, straight into the fp16
// operands of a tensor-core op, against fp16 activations. The page's Volta design
// (m8n8k4, load-time weight permutation, fp16 partials flushed to fp32 every 16)
// is not kept; what holds on sm_103a:
//  * Layout unchanged: codes are read as stored ([N][K/2] nibbles, [N][K/16]
//    E4M3 group scales, or [N][K] E4M3 bytes).
//  * Exact decode: cvt.rn.f16x2.e2m1x2 / .e4m3x2 are exact, and an E2M1 value
//    times an E4M3 scale has at most 6 significant bits and magnitude in
//    [2^-10, 2688], so the group scale is folded into the fp16 weight with no
//    rounding. The per-tensor scale (NVFP4) or the row scale (FP8) multiplies
//    the fp32 result once.
//  * fp32 accumulation inside mma.sync.m16n8k16 (f16 x f16 -> f32): no fp16
//    partial sums, so activation outliers up to 65504 cannot overflow (the
//    page's failure mode and the reason for its per-16 fp32 flush).
//  * The weights are the A operand (16 output rows per warp), the M <= 8
//    activation rows the B operand (n = 8). A dot product does not depend on
//    the order of k, so each lane takes a contiguous 32-byte run of its row
//    (one 128-byte line per four lanes: full-line, coalesced loads) and the
//    activation fragment is gathered in the same k order.
//  * Split K: a CTA owns 16 rows; its 8 warps take interleaved 128-byte steps
//    of the rows (adjacent lines in flight together), then reduce in shared memory.
#include "qmv_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kRowsPerCta = 16;
constexpr int kStepBytes = 128;   // bytes of one weight row per warp step

// kFp4: NVFP4 (256 k per step, E4M3 group scales); else FP8 (128 k per step, row scale).
template <bool kFp4>
__global__ void __launch_bounds__(kThreads) wq_mma_kernel(const uint8_t *__restrict__ codes,
                                                         const uint8_t *__restrict__ scales,
                                                         const float *__restrict__ row_scale, float g,
                                                         const uint16_t *__restrict__ x, float *__restrict__ y,
                                                         int M, int64_t N, int64_t K)
{
    __shared__ float red[kWarps][kRowsPerCta][9];
    constexpr int kStepK = kFp4 ? 2 * kStepBytes : kStepBytes;
    constexpr int kXWords = kStepK / 8;    // this lane's activation words per step (4 k per 2 words)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kRowsPerCta;
    // Rows past N read row 0 (valid memory); their results are discarded.
    const int64_t ra = row0 + gid < N ? row0 + gid : 0;
    const int64_t rb = row0 + gid + 8 < N ? row0 + gid + 8 : 0;
    const int64_t row_bytes = kFp4 ? K / 2 : K;
    const uint8_t *pa = codes + ra * row_bytes + 32 * t;
    const uint8_t *pb = codes + rb * row_bytes + 32 * t;
    const uint8_t *sa_ptr = kFp4 ? scales + ra * (K / 16) + 4 * t : nullptr;
    const uint8_t *sb_ptr = kFp4 ? scales + rb * (K / 16) + 4 * t : nullptr;
    const bool has_x = gid < M;
    const uint16_t *xp = x + (has_x ? gid : 0) * K + (kStepK / 4) * t;
    const int64_t nsteps = K / kStepK;
    const uint64_t pol = policy_evict_first();

    grid_launch_dependents();
    grid_dependency_wait();

    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int64_t s = warp; s < nsteps; s += kWarps) {
        const int64_t off = s * kStepBytes;
        const uint4 a0 = ld_stream_v4(pa + off, pol), a1 = ld_stream_v4(pa + off + 16, pol);
        const uint4 b0 = ld_stream_v4(pb + off, pol), b1 = ld_stream_v4(pb + off + 16, pol);
        const uint32_t cwa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t cwb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        uint32_t xw[kXWords];
        if (has_x) {
#pragma unroll
            for (int i = 0; i < kXWords / 4; ++i) {
                const uint4 v = ld_shared_v4(xp + s * kStepK + 8 * i);
                xw[4 * i] = v.x;
                xw[4 * i + 1] = v.y;
                xw[4 * i + 2] = v.z;
                xw[4 * i + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < kXWords; ++i) xw[i] = 0u;
        }
        if (kFp4) {
            // 4 scale bytes: group q covers this lane's codes bytes 8q..8q+7 (k 64t+16q ..).
            const uint32_t sa = ld_stream_u32(sa_ptr + s * 16, pol);
            const uint32_t sb = ld_stream_u32(sb_ptr + s * 16, pol);
            const uint32_t sa01 = e4m3x2_to_f16x2(sa & 0xffffu), sa23 = e4m3x2_to_f16x2(sa >> 16);
            const uint32_t sb01 = e4m3x2_to_f16x2(sb & 0xffffu), sb23 = e4m3x2_to_f16x2(sb >> 16);
            const uint32_t sca[4] = {dup_lo16(sa01), dup_hi16(sa01), dup_lo16(sa23), dup_hi16(sa23)};
            const uint32_t scb[4] = {dup_lo16(sb01), dup_hi16(sb01), dup_lo16(sb23), dup_hi16(sb23)};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                // word i = codes bytes 4i..4i+3 = k 8i..8i+7 of this lane's run; group i/2
                uint32_t ha[4], hb[4];
                e2m1x8_to_f16x2(cwa[i], ha);
                e2m1x8_to_f16x2(cwb[i], hb);
                const uint32_t ga = sca[i >> 1], gb = scb[i >> 1];
                mma_16816(d, hmul2_u32(ha[0], ga), hmul2_u32(hb[0], gb), hmul2_u32(ha[1], ga),
                          hmul2_u32(hb[1], gb), xw[4 * i], xw[4 * i + 1]);
                mma_16816(d, hmul2_u32(ha[2], ga), hmul2_u32(hb[2], gb), hmul2_u32(ha[3], ga),
                          hmul2_u32(hb[3], gb), xw[4 * i + 2], xw[4 * i + 3]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                // word j = codes bytes 4j..4j+3 = k 4j..4j+3 of this lane's run
                mma_16816(d, e4m3x2_to_f16x2(cwa[j] & 0xffffu), e4m3x2_to_f16x2(cwb[j] & 0xffffu),
                          e4m3x2_to_f16x2(cwa[j] >> 16), e4m3x2_to_f16x2(cwb[j] >> 16), xw[2 * j],
                          xw[2 * j + 1]);
            }
        }
    }

    red[warp][gid][2 * t] = d[0];
    red[warp][gid][2 * t + 1] = d[1];
    red[warp][gid + 8][2 * t] = d[2];
    red[warp][gid + 8][2 * t + 1] = d[3];
    __syncthreads();
    if (tid < kRowsPerCta * 8) {
        const int r = tid >> 3, m = tid & 7;
        const int64_t n = row0 + r;
        if (m < M && n < N) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s += red[w][r][m];
            y[m * N + n] = s * (kFp4 ? g : row_scale[n]);
        }
    }
}

// Any K % 16 == 0 (NVFP4) or any K (FP8), any alignment of the byte arrays:
// one warp per weight row, lanes over k, fp32 multiply-add.
template <bool kFp4>
__global__ void __launch_bounds__(kThreads) wq_generic_kernel(const uint8_t *__restrict__ codes,
                                                             const uint8_t *__restrict__ scales,
                                                             const float *__restrict__ row_scale, float g,
                                                             const uint16_t *__restrict__ x,
                                                             float *__restrict__ y, int M, int64_t N, int64_t K)
{
    grid_launch_dependents();
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (n >= N) return;
    float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    for (int64_t k = lane; k < K; k += 32) {
        float wv;
        if (kFp4) {
            const uint32_t byte = __ldg(codes + n * (K / 2) + k / 2);
            const uint32_t h = e2m1x2_to_f16x2(byte);
            const uint32_t c = (k & 1) ? (h >> 16) : (h & 0xffffu);
            const uint32_t sh = e4m3x2_to_f16x2(__ldg(scales + n * (K / 16) + k / 16));
            wv = f16_bits_to_float(c) * f16_bits_to_float(sh & 0xffffu);   // exact
        } else {
            wv = f16_bits_to_float(e4m3x2_to_f16x2(__ldg(codes + n * K + k)) & 0xffffu);
        }
#pragma unroll
        for (int m = 0; m < 8; ++m)
            if (m < M) acc[m] = fmaf(wv, f16_bits_to_float(__ldg(x + m * K + k)), acc[m]);
    }
    const float scale = kFp4 ? g : row_scale[n];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        if (m >= M) break;
        float v = acc[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) y[m * N + n] = v * scale;
    }
}

template <bool kFp4>
cudaError_t launch_wq(Route r, const uint8_t *codes, const uint8_t *scales, const float *rs, float g,
                      const uint16_t *x, float *y, int M, int64_t N, int64_t K, cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = set_launch_overlap_attr(attr);
    route_hit(r);
    const bool mma = (r == kRouteNvfp4Mma || r == kRouteFp8Mma);
    const int64_t grid = mma ? (N + kRowsPerCta - 1) / kRowsPerCta : (N + kWarps - 1) / kWarps;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    auto kern = mma ? wq_mma_kernel<kFp4> : wq_generic_kernel<kFp4>;
    // activations are re-read through L1: keep the default L1/shared split
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), 0, -1);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, kern, codes, scales, rs, g, x, y, M, N, K);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

Route plan_nvfp4(const uint8_t *codes, const uint8_t *scales, const uint16_t *x, int64_t K)
{
    const bool scales4 = (reinterpret_cast<uintptr_t>(scales) & 3u) == 0;
    return (K % 256 == 0 && aligned16(codes) && aligned16(x) && scales4) ? kRouteNvfp4Mma : kRouteNvfp4Generic;
}

Route plan_fp8(const uint8_t *w, const uint16_t *x, int64_t K)
{
    return (K % 128 == 0 && aligned16(w) && aligned16(x)) ? kRouteFp8Mma : kRouteFp8Generic;
}

cudaError_t launch_nvfp4(Route r, const DeviceInfo &, const uint8_t *codes, const uint8_t *scales, float g,
                         const uint16_t *x, float *y, int M, int64_t N, int64_t K, cudaStream_t s)
{
    return launch_wq<true>(r, codes, scales, nullptr, g, x, y, M, N, K, s);
}

cudaError_t launch_fp8(Route r, const DeviceInfo &, const uint8_t *w, const float *rs, const uint16_t *x, float *y,
                       int M, int64_t N, int64_t K, cudaStream_t s)
{
    return launch_wq<false>(r, w, nullptr, rs, 0.0f, x, y, M, N, K, s);
}

}  // namespace qmv
