// q4_0_q8_1.cu -- Q4_0 x Q8_1 mat-vec (MMVQ) for M = 1..8 activation rows.
//
// The quantized mat x vec of llama.cpp decode ("Machine Learning on NVIDIA CMP",
// sections "TL;DR" and "The DP2A patch"): per 32-weight block the integer dot of
// unsigned nibbles with int8 activations (one dp4a per 4 bytes, int32 sum), then
// one fp32 scale per block:
//     y[m][n] = sum_b (d4[n][b] * d8[m][b]) * (S[n][m][b] - 8 T[m][b]),
//     S = sum_j q4_j q8_j,  T = sum_j q8_j   (exact integers).
// The page's PRMT+DP2A rewrite exists because DP4A is throttled on mining cards;
// dp4a is a full-rate instruction here, so the dot stays one dp4a per word.
//
// Streaming kernel (K % 256 == 0, 16-byte aligned rows): a row is K/32 blocks of
// 18 bytes, a multiple of 144 = 9 x 16 bytes, so tiles of whole rows are one
// contiguous, 16-byte aligned span. Each CTA streams its tiles with 1-D bulk
// copies into a ring of shared-memory stages (mbarrier completion, evict-first
// L2 hint), after staging the Q8_1 activations once in shared memory. A thread
// consumes block pairs (36 bytes, always 4-byte aligned); lanes stride by one
// pair, so its nine 32-bit reads are bank-conflict free, and the activation
// pairs are padded to 80 bytes so the 16-byte activation reads are too.
#include <algorithm>

#include "qmv_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

__device__ uint32_t g_q4_error;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPairBytes = 36;        // two Q4_0 blocks
constexpr int kActPairStride = 80;    // 64 int8 activations + 16 bytes of padding

struct ActBlock {
    float d8;   // Q8_1 scale as fp32
    int t8;     // 8 * sum(q8)
};

struct Q4Layout {
    uint32_t rowbytes, tilebytes;
    uint32_t off_act, act_m_stride, off_dt, off_red, off_bar, total;
};

__host__ __device__ inline Q4Layout q4_layout(int M, int64_t K, int R, int S)
{
    Q4Layout L;
    const uint32_t nb = static_cast<uint32_t>(K / 32), np = static_cast<uint32_t>(K / 64);
    L.rowbytes = nb * 18u;
    L.tilebytes = static_cast<uint32_t>(R) * L.rowbytes;
    L.off_act = static_cast<uint32_t>(S) * L.tilebytes;
    L.act_m_stride = np * kActPairStride;
    L.off_dt = L.off_act + static_cast<uint32_t>(M) * L.act_m_stride;
    L.off_red = L.off_dt + static_cast<uint32_t>(M) * nb * static_cast<uint32_t>(sizeof(ActBlock));
    const uint32_t red_rows = static_cast<uint32_t>(R > kWarps ? R : kWarps);
    L.off_bar = (L.off_red + red_rows * static_cast<uint32_t>(M) * 4u + 7u) & ~7u;
    L.total = L.off_bar + static_cast<uint32_t>(S) * 8u;
    return L;
}

// Dot of one block pair of a weight row against M staged activation rows.
// wp: the pair's 36 bytes in shared memory (4-byte aligned).
// act: the pair's activations of row 0 (stride act_stride per row).
// dt:  ActBlock of block 2p of row 0 (stride nb per row).
template <int M, bool kDots>
__device__ __forceinline__ void q4_pair(const uint8_t *wp8, const uint8_t *act, uint32_t act_stride,
                                        const ActBlock *dt, int nb, float (&acc)[M], int32_t *dots,
                                        int64_t dots_m_stride)
{
    const uint32_t *wp = reinterpret_cast<const uint32_t *>(wp8);
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = wp[i];
    // block A = bytes 0..17: d4 in bytes 0..1, qs in bytes 2..17 (2 mod 4: realign)
    // block B = bytes 18..35: d4 in bytes 18..19, qs in bytes 20..35 (aligned)
    const float d4a = f16_bits_to_float(w[0] & 0xffffu);
    const float d4b = f16_bits_to_float(w[4] >> 16);
    uint32_t la[4], ha[4], lb[4], hb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t qa = __byte_perm(w[i], w[i + 1], 0x5432);
        la[i] = qa & 0x0f0f0f0fu;          // elements 4i..4i+3
        ha[i] = (qa >> 4) & 0x0f0f0f0fu;   // elements 16+4i..16+4i+3
        lb[i] = w[5 + i] & 0x0f0f0f0fu;
        hb[i] = (w[5 + i] >> 4) & 0x0f0f0f0fu;
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 *a = reinterpret_cast<const uint4 *>(act + m * act_stride);
        const uint4 a0 = a[0], a1 = a[1], a2 = a[2], a3 = a[3];
        int sa = 0, sb = 0;
        sa = dp4a_us(la[0], a0.x, sa);
        sa = dp4a_us(la[1], a0.y, sa);
        sa = dp4a_us(la[2], a0.z, sa);
        sa = dp4a_us(la[3], a0.w, sa);
        sa = dp4a_us(ha[0], a1.x, sa);
        sa = dp4a_us(ha[1], a1.y, sa);
        sa = dp4a_us(ha[2], a1.z, sa);
        sa = dp4a_us(ha[3], a1.w, sa);
        sb = dp4a_us(lb[0], a2.x, sb);
        sb = dp4a_us(lb[1], a2.y, sb);
        sb = dp4a_us(lb[2], a2.z, sb);
        sb = dp4a_us(lb[3], a2.w, sb);
        sb = dp4a_us(hb[0], a3.x, sb);
        sb = dp4a_us(hb[1], a3.y, sb);
        sb = dp4a_us(hb[2], a3.z, sb);
        sb = dp4a_us(hb[3], a3.w, sb);
        const ActBlock ba = dt[m * nb], bb = dt[m * nb + 1];
        const int da = sa - ba.t8, db = sb - bb.t8;
        if (kDots) {
            dots[m * dots_m_stride] = da;
            dots[m * dots_m_stride + 1] = db;
        } else {
            acc[m] += (d4a * ba.d8) * static_cast<float>(da) + (d4b * bb.d8) * static_cast<float>(db);
        }
    }
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int M, bool kDots>
__global__ void __launch_bounds__(kThreads) q4_0_stream_kernel(const uint8_t *__restrict__ w,
                                                              const uint8_t *__restrict__ xq,
                                                              float *__restrict__ y, int32_t *__restrict__ dots,
                                                              int64_t N, int64_t K, int R, int S)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const Q4Layout L = q4_layout(M, K, R, S);
    const int nb = static_cast<int>(K >> 5), np = static_cast<int>(K >> 6);
    const int64_t ntiles = (N + R - 1) / R;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.off_bar);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncthreads();

    const uint64_t pol = policy_evict_first();
    auto issue = [&](int64_t tile, int slot) {
        const int64_t row0 = tile * R;
        const uint32_t rows = static_cast<uint32_t>(min(static_cast<int64_t>(R), N - row0));
        const uint32_t bytes = rows * L.rowbytes;
        mbar_arrive_expect_tx(&bars[slot], bytes);
        bulk_copy_g2s(smem + static_cast<uint32_t>(slot) * L.tilebytes, w + row0 * L.rowbytes, bytes, &bars[slot],
                      pol);
    };
    // Weights do not depend on the preceding kernel: start streaming before waiting on it.
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            const int64_t tile = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (tile < ntiles) issue(tile, s);
        }
    }
    grid_launch_dependents();
    grid_dependency_wait();

    // Stage the Q8_1 activations: padded int8 pairs + (d8, 8T) per block.
    ActBlock *dts = reinterpret_cast<ActBlock *>(smem + L.off_dt);
    for (int i = tid; i < M * nb; i += kThreads) {
        const int m = i / nb, b = i - m * nb;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + static_cast<int64_t>(i) * 36);
        uint32_t q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = __ldg(src + 1 + j);
        int t = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) t = __dp4a(static_cast<int>(q[j]), 0x01010101, t);
        dts[i].d8 = f16_bits_to_float(__ldg(src) & 0xffffu);
        dts[i].t8 = 8 * t;
        uint4 *dst = reinterpret_cast<uint4 *>(smem + L.off_act + m * L.act_m_stride + (b >> 1) * kActPairStride +
                                               (b & 1) * 32);
        dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
        dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
    }
    __syncthreads();

    const int wpr = (R >= kWarps) ? 1 : kWarps / R;   // warps sharing one row
    const int rows_par = kWarps / wpr;                  // rows in flight per pass
    const int sub = warp % wpr;
    float *red = reinterpret_cast<float *>(smem + L.off_red);

    int64_t local = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++local) {
        const int slot = static_cast<int>(local % S);
        const uint32_t parity = static_cast<uint32_t>((local / S) & 1);
        const bool ok = mbar_wait(&bars[slot], parity);
        if (!__syncthreads_and(ok)) {
            if (tid == 0) {
                atomicOr(&g_q4_error, kErrWaitTimeout);
                // let copies still in flight land before the CTA's shared memory is released
                for (int s = 1; s < S; ++s) {
                    const int64_t lt = local + s;
                    if (blockIdx.x + lt * gridDim.x < ntiles)
                        (void)mbar_wait(&bars[lt % S], static_cast<uint32_t>((lt / S) & 1));
                }
            }
            return;
        }
        const uint8_t *tb = smem + static_cast<uint32_t>(slot) * L.tilebytes;
        const int64_t row0 = tile * R;
        const int rows_here = static_cast<int>(min(static_cast<int64_t>(R), N - row0));

        for (int rr = warp / wpr; rr < rows_here; rr += rows_par) {
            float acc[M];
#pragma unroll
            for (int m = 0; m < M; ++m) acc[m] = 0.0f;
            const uint8_t *wrow = tb + rr * L.rowbytes;
            int32_t *drow = kDots ? dots + (row0 + rr) * nb : nullptr;
            for (int p = sub * 32 + lane; p < np; p += 32 * wpr) {
                q4_pair<M, kDots>(wrow + kPairBytes * p, smem + L.off_act + kActPairStride * p, L.act_m_stride,
                                  dts + 2 * p, nb, acc, kDots ? drow + 2 * p : nullptr, N * nb);
            }
            if (!kDots) {
#pragma unroll
                for (int m = 0; m < M; ++m) acc[m] = warp_sum(acc[m]);
                if (lane == 0) {
#pragma unroll
                    for (int m = 0; m < M; ++m) red[(rr * wpr + sub) * M + m] = acc[m];
                }
            }
        }
        __syncthreads();   // every thread is done with this stage
        if (tid == 0) {
            const int64_t next = tile + static_cast<int64_t>(S) * gridDim.x;
            if (next < ntiles) issue(next, slot);
        }
        if (!kDots) {
            for (int i = tid; i < rows_here * M; i += kThreads) {
                const int r = i / M, m = i - r * M;
                float s = 0.0f;
                for (int j = 0; j < wpr; ++j) s += red[(r * wpr + j) * M + m];
                y[m * N + row0 + r] = s;
            }
        }
    }
}

// Any K % 32 == 0 and 2-byte aligned rows: one warp per weight row, lanes over blocks.
template <int M, bool kDots>
__global__ void __launch_bounds__(kThreads) q4_0_generic_kernel(const uint8_t *__restrict__ w,
                                                               const uint8_t *__restrict__ xq,
                                                               float *__restrict__ y, int32_t *__restrict__ dots,
                                                               int64_t N, int64_t K)
{
    grid_launch_dependents();
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (n >= N) return;
    const int64_t nb = K >> 5;
    float acc[M];
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] = 0.0f;
    for (int64_t b = lane; b < nb; b += 32) {
        const uint16_t *wb = reinterpret_cast<const uint16_t *>(w + (n * nb + b) * 18);
        const float d4 = f16_bits_to_float(__ldg(wb));
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t q = static_cast<uint32_t>(__ldg(wb + 1 + 2 * i)) |
                               (static_cast<uint32_t>(__ldg(wb + 2 + 2 * i)) << 16);
            lo[i] = q & 0x0f0f0f0fu;
            hi[i] = (q >> 4) & 0x0f0f0f0fu;
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint32_t *xb = reinterpret_cast<const uint32_t *>(xq + (m * nb + b) * 36);
            uint32_t a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) a[j] = __ldg(xb + 1 + j);
            int s = 0, t = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                s = dp4a_us(lo[i], a[i], s);
                s = dp4a_us(hi[i], a[4 + i], s);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) t = __dp4a(static_cast<int>(a[j]), 0x01010101, t);
            const int d = s - 8 * t;
            if (kDots) {
                dots[(m * N + n) * nb + b] = d;
            } else {
                acc[m] += (d4 * f16_bits_to_float(__ldg(xb) & 0xffffu)) * static_cast<float>(d);
            }
        }
    }
    if (!kDots) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const float s = warp_sum(acc[m]);
            if (lane == 0) y[m * N + n] = s;
        }
    }
}

// ---------------------------------------------------------------- host side

template <int M, bool kDots>
cudaError_t launch_m(const Q4Plan &p, const uint8_t *w, const uint8_t *xq, float *y, int32_t *dots, int64_t N,
                     int64_t K, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    if (p.route == kRouteQ4_0Stream) {
        auto kern = q4_0_stream_kernel<M, kDots>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
        if (e != cudaSuccess) return e;
        cfg.dynamicSmemBytes = static_cast<size_t>(p.smem_bytes);
        return cudaLaunchKernelEx(&cfg, kern, w, xq, y, dots, N, K, p.rows_per_tile, p.stages);
    }
    return cudaLaunchKernelEx(&cfg, q4_0_generic_kernel<M, kDots>, w, xq, y, dots, N, K);
}

template <bool kDots>
cudaError_t launch_dispatch(const Q4Plan &p, const uint8_t *w, const uint8_t *xq, float *y, int32_t *dots, int M,
                            int64_t N, int64_t K, cudaStream_t s)
{
    switch (M) {
    case 1: return launch_m<1, kDots>(p, w, xq, y, dots, N, K, s);
    case 2: return launch_m<2, kDots>(p, w, xq, y, dots, N, K, s);
    case 3: return launch_m<3, kDots>(p, w, xq, y, dots, N, K, s);
    case 4: return launch_m<4, kDots>(p, w, xq, y, dots, N, K, s);
    case 5: return launch_m<5, kDots>(p, w, xq, y, dots, N, K, s);
    case 6: return launch_m<6, kDots>(p, w, xq, y, dots, N, K, s);
    case 7: return launch_m<7, kDots>(p, w, xq, y, dots, N, K, s);
    case 8: return launch_m<8, kDots>(p, w, xq, y, dots, N, K, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t plan_q4_0(const DeviceInfo &dev, const void *w, const void *xq, int M, int64_t N, int64_t K,
                      Q4Plan *plan)
{
    (void)xq;
    const bool aligned = (reinterpret_cast<uintptr_t>(w) & 15u) == 0;
    plan->route = kRouteQ4_0Generic;
    plan->rows_per_tile = 0;
    plan->stages = 0;
    plan->smem_bytes = 0;
    plan->grid = static_cast<int>((N + kWarps - 1) / kWarps);
    if (!aligned || K % 256 != 0) return cudaSuccess;

    const int64_t rowbytes = K / 32 * 18;
    // Tile: whole rows, at most ~20 KB per stage; fewer rows when the matrix is
    // short so every CTA gets several tiles.
    int R = 1;
    while (R < 64 && (2 * R) * rowbytes <= 20 * 1024) R *= 2;
    while (R > 1 && (N + R - 1) / R < 4LL * dev.sm_count) R /= 2;
    int S = 4;
    Q4Layout L = q4_layout(M, K, R, S);
    while (L.total > static_cast<uint32_t>(dev.smem_optin) && S > 2) L = q4_layout(M, K, R, --S);
    while (L.total > static_cast<uint32_t>(dev.smem_optin) && R > 1) L = q4_layout(M, K, R /= 2, S);
    if (L.total > static_cast<uint32_t>(dev.smem_optin)) return cudaSuccess;   // generic kernel

    const int per_sm = std::max(1, std::min(kWarps, dev.smem_per_sm / static_cast<int>(L.total + 1024)));
    const int64_t ntiles = (N + R - 1) / R;
    plan->route = kRouteQ4_0Stream;
    plan->rows_per_tile = R;
    plan->stages = S;
    plan->smem_bytes = static_cast<int>(L.total);
    plan->grid = static_cast<int>(std::min<int64_t>(ntiles, static_cast<int64_t>(dev.sm_count) * per_sm));
    return cudaSuccess;
}

cudaError_t launch_q4_0(const Q4Plan &plan, const void *w, const void *xq, float *y, int32_t *dots, int M,
                        int64_t N, int64_t K, cudaStream_t s)
{
    const uint8_t *wb = static_cast<const uint8_t *>(w);
    const uint8_t *xb = static_cast<const uint8_t *>(xq);
    route_hit(plan.route);
    if (dots) return launch_dispatch<true>(plan, wb, xb, y, dots, M, N, K, s);
    return launch_dispatch<false>(plan, wb, xb, y, dots, M, N, K, s);
}

cudaError_t read_error_word_q4_0(uint32_t *out, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_q4_error, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_q4_error, &zero, sizeof(uint32_t));
}

}  // namespace qmv
