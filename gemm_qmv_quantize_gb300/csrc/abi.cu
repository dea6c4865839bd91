// abi.cu -- the C ABI of include/qmv.h: argument validation (before any CUDA
// call), the per-(M, N, K) kernel choice, the route census and the error word.
#include <atomic>
#include <cstdlib>
#include <mutex>

#include "qmv.h"
#include "qmv_device.cuh"
#include "qmv_internal.h"

namespace qmv {

namespace {

std::atomic<int64_t> g_route_launches[kRouteCount];

constexpr const char *kRouteNames[kRouteCount] = {
    "quantize_q8_1", "q4_0_stream_dp4a", "q4_0_generic", "q4_0_stream_fused_quantize", "nvfp4_mma_m16n8k16",
    "nvfp4_generic",
    "fp8_mma_m16n8k16", "fp8_generic", "zero_fill", "q4_0_mma_m16n8k32", "q4_0_mma_fused_quantize",
    "q4_k_stream_dp4a", "q4_k_stream_fused_quantize", "q4_k_mma_m16n8k32", "q4_k_mma_fused_quantize",
    "nvfp4_tcgen05", "fp8_tcgen05",
};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_valid[kMaxDevices];

constexpr int64_t kMaxDim = 0x7fffffffLL;
constexpr int kMaxRowsW = 96;   // activation rows of the NVFP4 / FP8 entry points (chunks of <= 16 above 16)

bool misaligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

qmv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QMV_OK : QMV_ERR_CUDA; }

// Shared shape checks: M in 0..max_m, 0 <= N, K <= 2^31-1, K a multiple of `kblock`.
qmv_status check_shape(int M, int64_t N, int64_t K, int64_t kblock, int max_m = 8)
{
    if (M < 0 || M > max_m || N < 0 || K < 0 || N > kMaxDim || K > kMaxDim) return QMV_ERR_SHAPE;
    if (kblock > 1 && K % kblock != 0) return QMV_ERR_SHAPE;
    return QMV_OK;
}

// Error word of the wait-bound self-checks below (OR-ed into qmv_error_flags).
__device__ uint32_t g_abi_error;

// One thread waits, with the bounded wait of the streaming kernels, on an mbarrier
// that expects one arrival nobody makes: the wait must give up, flag the error word
// and return. out[0] = 1 if the wait completed (never expected), else 0; out[1] =
// nanoseconds spent in the wait.
__global__ void wait_bound_kernel(int64_t *out)
{
    __shared__ __align__(8) uint64_t bar;
    mbar_init(&bar, 1);
    fence_barrier_init();
    const uint64_t t0 = globaltimer_ns();
    const bool done = mbar_wait_bounded(&bar, 0);
    const uint64_t t1 = globaltimer_ns();
    out[0] = done ? 1 : 0;
    out[1] = static_cast<int64_t>(t1 - t0);
    if (!done) atomicOr(&g_abi_error, kErrWaitTimeout);
}

// Source of the self-check's real copies (its contents are never used).
__device__ __align__(16) uint8_t g_probe_src[64];

constexpr int kProbeWarps = 8, kProbeSlots = 2, kProbeBytes = 16;

// The tensor-core kernels' way of giving up, in one CTA of 8 warps: every warp fills
// a 2-slot ring, warp `stuck` arms its mbarriers but issues no copy, so its bounded
// wait runs out while the other warps consume real copies and go on to the CTA-wide
// barrier that ends the round. The stuck warp must flag the error word and the CTA's
// abort word and reach that barrier too; after it every warp sees the abort, lets its
// copies land and returns. out int64 [8][4], per warp: 1 if its wait gave up; 1 if
// it passed the barrier and saw the abort; copies still outstanding when it left the
// round; nanoseconds from the first wait to the barrier.
__global__ void cta_abort_kernel(int64_t *out, int stuck)
{
    __shared__ __align__(128) uint8_t ring[kProbeWarps][kProbeSlots][kProbeBytes];
    __shared__ __align__(8) uint64_t bars[kProbeWarps][kProbeSlots];
    __shared__ uint32_t cta_abort;
    const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
    if (threadIdx.x == 0) cta_abort = 0u;
    int outstanding = 0;
    if (lane == 0) {
        for (int s = 0; s < kProbeSlots; ++s) mbar_init(&bars[warp][s], 1);
        fence_barrier_init();
        const uint64_t pol = policy_evict_first();
        for (int s = 0; s < kProbeSlots; ++s) {
            mbar_arrive_expect_tx(&bars[warp][s], kProbeBytes);
            if (warp != stuck) bulk_copy_g2s(ring[warp][s], g_probe_src + kProbeBytes * s, kProbeBytes, &bars[warp][s], pol);
            ++outstanding;
        }
    }
    __syncthreads();   // the prologue's barrier
    int slot = 0;
    uint32_t phase = 0;
    bool failed = false;
    const uint64_t t0 = globaltimer_ns();
    for (int i = 0; i < kProbeSlots; ++i) {
        if (!mbar_wait_bounded(&bars[warp][slot], phase)) {
            if (lane == 0) note_wait_timeout(&g_abi_error, &cta_abort);
            failed = true;
            break;
        }
        --outstanding;
        if (++slot == kProbeSlots) {
            slot = 0;
            phase ^= 1u;
        }
    }
    __syncthreads();   // the round's barrier
    const uint64_t t1 = globaltimer_ns();
    const bool abort = cta_abort != 0u;
    if (lane == 0) {
        out[4 * warp] = failed ? 1 : 0;
        out[4 * warp + 1] = abort ? 1 : 0;
        out[4 * warp + 2] = outstanding;
        out[4 * warp + 3] = static_cast<int64_t>(t1 - t0);
    }
    if (abort) {
        if (lane == 0) drain_ring(bars[warp], kProbeSlots, slot, phase, outstanding);
        return;
    }
}

qmv_status zero_fill(float *y, int M, int64_t N, cudaStream_t s)
{
    route_hit(kRouteZeroFill);
    return from_cuda(cudaMemsetAsync(y, 0, static_cast<size_t>(M) * static_cast<size_t>(N) * sizeof(float), s));
}

}  // namespace

namespace {
std::atomic<int> g_launch_overlap{0};

struct SmemAttrEntry {
    const void *kernel;
    int device;
    int bytes;
};
std::mutex g_attr_mutex;
SmemAttrEntry g_attr_cache[256];
int g_attr_count = 0;
}  // namespace

int env_int(const char *name, int fallback)
{
    const char *v = std::getenv(name);
    if (!v || !*v) return fallback;
    char *end = nullptr;
    const long x = std::strtol(v, &end, 10);
    return (end && *end == 0) ? static_cast<int>(x) : fallback;
}

int set_launch_overlap_attr(cudaLaunchAttribute *attr)
{
    if (!g_launch_overlap.load(std::memory_order_relaxed)) return 0;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    return 1;
}

cudaError_t ensure_smem_attr(const void *kernel, int bytes, int carveout)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    for (int i = 0; i < g_attr_count; ++i) {
        SmemAttrEntry &c = g_attr_cache[i];
        if (c.kernel == kernel && c.device == dev) {
            if (c.bytes >= bytes) return cudaSuccess;
            if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) == cudaSuccess)
                c.bytes = bytes;
            return e;
        }
    }
    if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
        return e;
    if (carveout >= 0 &&
        (e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carveout)) != cudaSuccess)
        return e;
    if (g_attr_count < 256) g_attr_cache[g_attr_count++] = SmemAttrEntry{kernel, dev, bytes};
    return cudaSuccess;
}

const char *route_name(int r) { return (r >= 0 && r < kRouteCount) ? kRouteNames[r] : "unknown"; }

void route_hit(Route r) { g_route_launches[r].fetch_add(1, std::memory_order_relaxed); }

cudaError_t current_device_info(DeviceInfo *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_valid[dev]) {
        DeviceInfo d{};
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess)
            return e;
        g_dev[dev] = d;
        g_dev_valid[dev] = true;
    }
    *out = g_dev[dev];
    return cudaSuccess;
}

}  // namespace qmv

using namespace qmv;

extern "C" {

const char *qmv_status_string(qmv_status status)
{
    switch (status) {
    case QMV_OK: return "QMV_OK";
    case QMV_ERR_NULL: return "QMV_ERR_NULL: a required pointer is NULL";
    case QMV_ERR_SHAPE: return "QMV_ERR_SHAPE: M outside 0..8, a negative or oversized N/K, or K not a multiple of the block";
    case QMV_ERR_ALIGN: return "QMV_ERR_ALIGN: a pointer is not aligned to its element type";
    case QMV_ERR_CUDA: return "QMV_ERR_CUDA: a CUDA runtime call failed";
    case QMV_ERR_TIMEOUT: return "QMV_ERR_TIMEOUT: a bounded device-side wait gave up";
    default: return "unknown qmv status";
    }
}

qmv_status qmv_quantize_q8_1(const float *x, void *xq, int M, int64_t K, qmv_stream_t stream)
{
    qmv_status st = check_shape(M, 1, K, 32);
    if (st != QMV_OK) return st;
    if (M == 0 || K == 0) return QMV_OK;
    if (!x || !xq) return QMV_ERR_NULL;
    if (misaligned(x, 4) || misaligned(xq, 4)) return QMV_ERR_ALIGN;
    return from_cuda(launch_quantize_q8_1(x, xq, M, K, stream));
}

static Q4Group single_group(const void *w, const void *x, float *y, int64_t N)
{
    Q4Group g{};
    g.count = 1;
    g.nx = 1;
    g.xslot[0] = 0;
    g.w[0] = static_cast<const uint8_t *>(w);
    g.x[0] = x;
    g.y[0] = y;
    g.row_start[0] = 0;
    g.row_start[1] = N;
    return g;
}

static qmv_status q4_0_common(const void *w, const void *xq, float *y, int32_t *dots, int M, int64_t N, int64_t K,
                              qmv_stream_t stream)
{
    qmv_status st = check_shape(M, N, K, 32);
    if (st != QMV_OK) return st;
    if (M == 0 || N == 0) return QMV_OK;
    if (!dots && !y) return QMV_ERR_NULL;
    if (K == 0) return dots ? QMV_OK : zero_fill(y, M, N, stream);
    if (!w || !xq) return QMV_ERR_NULL;
    if (misaligned(w, 2) || misaligned(xq, 4) || misaligned(y, 4) || misaligned(dots, 4)) return QMV_ERR_ALIGN;
    DeviceInfo dev;
    cudaError_t e = current_device_info(&dev);
    if (e != cudaSuccess) return QMV_ERR_CUDA;
    const Q4Group grp = single_group(w, xq, y, N);
    Q4Plan plan;
    if ((e = plan_q4_0(dev, grp, M, K, &plan)) != cudaSuccess) return QMV_ERR_CUDA;
    return from_cuda(launch_q4_0(plan, grp, dots, M, K, false, stream));
}

qmv_status qmv_q4_0_q8_1(const void *w, const void *xq, float *y, int M, int64_t N, int64_t K, qmv_stream_t stream)
{
    return q4_0_common(w, xq, y, nullptr, M, N, K, stream);
}

qmv_status qmv_debug_q4_0_block_dots(const void *w, const void *xq, int32_t *dots, int M, int64_t N, int64_t K,
                                     qmv_stream_t stream)
{
    if (!dots && M > 0 && N > 0 && K > 0) return QMV_ERR_NULL;
    return q4_0_common(w, xq, nullptr, dots, M, N, K, stream);
}

// Grouped launch of `count` matrices with the same M and K: fused, x[i] are fp32
// [M][K] (16-byte aligned); else Q8_1 [M][K/32] (4-byte aligned).
static qmv_status q4_0_group(int count, const void *const *w, const void *const *x, float *const *y,
                             const int64_t *N, int M, int64_t K, bool fused, qmv_stream_t stream, bool q4k = false,
                             int32_t *dots = nullptr)
{
    if (count < 1 || count > kMaxGroup) return QMV_ERR_SHAPE;
    if (!w || !x || !y || !N) return QMV_ERR_NULL;
    Q4Group grp{};
    grp.count = count;
    grp.row_start[0] = 0;
    for (int i = 0; i < count; ++i) {
        qmv_status st = check_shape(M, N[i], K, 256);
        if (st != QMV_OK) return st;
        grp.row_start[i + 1] = grp.row_start[i] + N[i];
    }
    if (grp.row_start[count] > kMaxDim) return QMV_ERR_SHAPE;
    if (M == 0 || grp.row_start[count] == 0) return QMV_OK;
    for (int i = 0; i < count; ++i) {
        if (N[i] > 0 && !y[i] && !dots) return QMV_ERR_NULL;
        if (misaligned(y[i], 4) || misaligned(dots, 4)) return QMV_ERR_ALIGN;
    }
    if (K == 0) {
        if (dots) return QMV_OK;
        for (int i = 0; i < count; ++i) {
            if (N[i] == 0) continue;
            qmv_status st = zero_fill(y[i], M, N[i], stream);
            if (st != QMV_OK) return st;
        }
        return QMV_OK;
    }
    for (int i = 0; i < count; ++i) {
        if (!w[i] || !x[i]) return QMV_ERR_NULL;
        if (misaligned(w[i], 16) || misaligned(x[i], fused ? 16 : 4)) return QMV_ERR_ALIGN;
        grp.w[i] = static_cast<const uint8_t *>(w[i]);
        grp.y[i] = y[i];
        // matrices given the same activation stage (and quantize) it once
        int j = 0;
        while (j < grp.nx && grp.x[j] != x[i]) ++j;
        if (j == grp.nx) grp.x[grp.nx++] = x[i];
        grp.xslot[i] = j;
    }
    DeviceInfo dev;
    cudaError_t e = current_device_info(&dev);
    if (e != cudaSuccess) return QMV_ERR_CUDA;
    Q4Plan plan;
    if ((e = plan_q4_0(dev, grp, M, K, &plan, q4k)) != cudaSuccess) return QMV_ERR_CUDA;
    if (plan.route != kRouteQ4_0Stream && plan.route != kRouteQ4_0Mma)
        return QMV_ERR_SHAPE;   // the activations do not fit in shared memory
    return from_cuda(launch_q4_0(plan, grp, dots, M, K, fused, stream, q4k));
}

qmv_status qmv_q4_0_q8_1_fused_group(int count, const void *const *w, const float *const *x, float *const *y,
                                     const int64_t *N, int M, int64_t K, qmv_stream_t stream)
{
    return q4_0_group(count, w, reinterpret_cast<const void *const *>(x), y, N, M, K, true, stream);
}

qmv_status qmv_q4_0_q8_1_group(int count, const void *const *w, const void *const *xq, float *const *y,
                               const int64_t *N, int M, int64_t K, qmv_stream_t stream)
{
    return q4_0_group(count, w, xq, y, N, M, K, false, stream);
}

qmv_status qmv_q4_0_q8_1_fused(const void *w, const float *x, float *y, int M, int64_t N, int64_t K,
                               qmv_stream_t stream)
{
    return qmv_q4_0_q8_1_fused_group(1, &w, &x, &y, &N, M, K, stream);
}

// ---- Q4_K: the grouped streaming path for every call (K % 256, 16-byte aligned rows)

qmv_status qmv_q4_k_q8_1(const void *w, const void *xq, float *y, int M, int64_t N, int64_t K, qmv_stream_t stream)
{
    return q4_0_group(1, &w, &xq, &y, &N, M, K, false, stream, true);
}

qmv_status qmv_q4_k_q8_1_group(int count, const void *const *w, const void *const *xq, float *const *y,
                               const int64_t *N, int M, int64_t K, qmv_stream_t stream)
{
    return q4_0_group(count, w, xq, y, N, M, K, false, stream, true);
}

qmv_status qmv_q4_k_q8_1_fused(const void *w, const float *x, float *y, int M, int64_t N, int64_t K,
                               qmv_stream_t stream)
{
    const void *xv = x;
    return q4_0_group(1, &w, &xv, &y, &N, M, K, true, stream, true);
}

qmv_status qmv_q4_k_q8_1_fused_group(int count, const void *const *w, const float *const *x, float *const *y,
                                     const int64_t *N, int M, int64_t K, qmv_stream_t stream)
{
    return q4_0_group(count, w, reinterpret_cast<const void *const *>(x), y, N, M, K, true, stream, true);
}

qmv_status qmv_debug_q4_k_block_dots(const void *w, const void *xq, int32_t *dots, int M, int64_t N, int64_t K,
                                     qmv_stream_t stream)
{
    if (!dots && M > 0 && N > 0 && K > 0) return QMV_ERR_NULL;
    float *no_y = nullptr;
    return q4_0_group(1, &w, &xq, &no_y, &N, M, K, false, stream, true, dots);
}

qmv_status qgemm_nvfp4_w4a16(const uint8_t *codes, const uint8_t *scales_e4m3, float global_scale,
                             const uint16_t *x, float *y, int M, int64_t N, int64_t K, qmv_stream_t stream)
{
    qmv_status st = check_shape(M, N, K, 16, kMaxRowsW);
    if (st != QMV_OK) return st;
    if (M == 0 || N == 0) return QMV_OK;
    if (!y) return QMV_ERR_NULL;
    if (misaligned(y, 4)) return QMV_ERR_ALIGN;
    if (K == 0) return zero_fill(y, M, N, stream);
    if (!codes || !scales_e4m3 || !x) return QMV_ERR_NULL;
    if (misaligned(x, 2)) return QMV_ERR_ALIGN;
    DeviceInfo dev;
    if (current_device_info(&dev) != cudaSuccess) return QMV_ERR_CUDA;
    const Route r = plan_nvfp4(codes, scales_e4m3, x, K);
    WqGroup grp{};
    grp.count = 1;
    grp.codes[0] = codes;
    grp.scales[0] = scales_e4m3;
    grp.g[0] = global_scale;
    grp.y[0] = y;
    grp.N[0] = N;
    return from_cuda(launch_nvfp4(r, dev, grp, x, M, K, stream));
}

qmv_status qgemm_fp8_w8a16(const uint8_t *w, const float *row_scale, const uint16_t *x, float *y, int M, int64_t N,
                           int64_t K, qmv_stream_t stream)
{
    qmv_status st = check_shape(M, N, K, 1, kMaxRowsW);
    if (st != QMV_OK) return st;
    if (M == 0 || N == 0) return QMV_OK;
    if (!y) return QMV_ERR_NULL;
    if (misaligned(y, 4)) return QMV_ERR_ALIGN;
    if (K == 0) return zero_fill(y, M, N, stream);
    if (!w || !row_scale || !x) return QMV_ERR_NULL;
    if (misaligned(x, 2) || misaligned(row_scale, 4)) return QMV_ERR_ALIGN;
    DeviceInfo dev;
    if (current_device_info(&dev) != cudaSuccess) return QMV_ERR_CUDA;
    const Route r = plan_fp8(w, x, K);
    WqGroup grp{};
    grp.count = 1;
    grp.codes[0] = w;
    grp.row_scale[0] = row_scale;
    grp.y[0] = y;
    grp.N[0] = N;
    return from_cuda(launch_fp8(r, dev, grp, x, M, K, stream));
}

// Grouped NVFP4 / FP8 launches (fp4: codes + E4M3 scales + global scales; else E4M3
// weights + row scales), all matrices reading x: the tensor-core kernel only.
static qmv_status wq_group(bool fp4, int count, const uint8_t *const *codes, const uint8_t *const *scales,
                           const float *g, const float *const *row_scale, const uint16_t *x, float *const *y,
                           const int64_t *N, int M, int64_t K, qmv_stream_t stream)
{
    if (count < 1 || count > kMaxGroup) return QMV_ERR_SHAPE;
    if (!codes || !y || !N || (fp4 ? (!scales || !g) : !row_scale)) return QMV_ERR_NULL;
    WqGroup grp{};
    grp.count = count;
    int64_t total = 0;
    for (int i = 0; i < count; ++i) {
        qmv_status st = check_shape(M, N[i], K, fp4 ? 256 : 128, kMaxRowsW);
        if (st != QMV_OK) return st;
        total += N[i];
    }
    if (total > kMaxDim) return QMV_ERR_SHAPE;
    if (M == 0 || total == 0) return QMV_OK;
    for (int i = 0; i < count; ++i) {
        if (N[i] > 0 && !y[i]) return QMV_ERR_NULL;
        if (misaligned(y[i], 4)) return QMV_ERR_ALIGN;
    }
    if (K == 0) {
        for (int i = 0; i < count; ++i) {
            if (N[i] == 0) continue;
            qmv_status st = zero_fill(y[i], M, N[i], stream);
            if (st != QMV_OK) return st;
        }
        return QMV_OK;
    }
    if (!x) return QMV_ERR_NULL;
    if (misaligned(x, 16)) return QMV_ERR_ALIGN;
    for (int i = 0; i < count; ++i) {
        if (!codes[i] || (fp4 ? !scales[i] : !row_scale[i])) return QMV_ERR_NULL;
        if (misaligned(codes[i], 16) || (fp4 ? misaligned(scales[i], 4) : misaligned(row_scale[i], 4)))
            return QMV_ERR_ALIGN;
        grp.codes[i] = codes[i];
        grp.scales[i] = fp4 ? scales[i] : nullptr;
        grp.row_scale[i] = fp4 ? nullptr : row_scale[i];
        grp.g[i] = fp4 ? g[i] : 0.0f;
        grp.y[i] = y[i];
        grp.N[i] = N[i];
    }
    DeviceInfo dev;
    if (current_device_info(&dev) != cudaSuccess) return QMV_ERR_CUDA;
    return fp4 ? from_cuda(launch_nvfp4(kRouteNvfp4Mma, dev, grp, x, M, K, stream))
               : from_cuda(launch_fp8(kRouteFp8Mma, dev, grp, x, M, K, stream));
}

qmv_status qgemm_nvfp4_w4a16_group(int count, const uint8_t *const *codes, const uint8_t *const *scales_e4m3,
                                   const float *global_scale, const uint16_t *x, float *const *y, const int64_t *N,
                                   int M, int64_t K, qmv_stream_t stream)
{
    return wq_group(true, count, codes, scales_e4m3, global_scale, nullptr, x, y, N, M, K, stream);
}

qmv_status qgemm_fp8_w8a16_group(int count, const uint8_t *const *w, const float *const *row_scale,
                                 const uint16_t *x, float *const *y, const int64_t *N, int M, int64_t K,
                                 qmv_stream_t stream)
{
    return wq_group(false, count, w, nullptr, nullptr, row_scale, x, y, N, M, K, stream);
}

void qmv_set_launch_overlap(int enable) { g_launch_overlap.store(enable ? 1 : 0, std::memory_order_relaxed); }

int qmv_get_launch_overlap(void) { return g_launch_overlap.load(std::memory_order_relaxed); }

int qmv_route_count(void) { return kRouteCount; }

const char *qmv_route_name(int route) { return route_name(route); }

int64_t qmv_route_launches(int route)
{
    return (route >= 0 && route < kRouteCount) ? g_route_launches[route].load(std::memory_order_relaxed) : -1;
}

void qmv_route_reset(void)
{
    for (auto &c : g_route_launches) c.store(0, std::memory_order_relaxed);
}

qmv_status qmv_error_flags(uint32_t *flags, int clear)
{
    if (!flags) return QMV_ERR_NULL;
    if (cudaDeviceSynchronize() != cudaSuccess) return QMV_ERR_CUDA;
    uint32_t w = 0, w2 = 0, w3 = 0, w4 = 0, w5 = 0;
    if (read_error_word_q4_0(&w, clear != 0) != cudaSuccess) return QMV_ERR_CUDA;
    if (read_error_word_umma(&w5, clear != 0) != cudaSuccess) return QMV_ERR_CUDA;
    if (read_error_word_wq(&w2, clear != 0) != cudaSuccess) return QMV_ERR_CUDA;
    if (read_error_word_q4_0_mma(&w3, clear != 0) != cudaSuccess) return QMV_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&w4, g_abi_error, sizeof(uint32_t)) != cudaSuccess) return QMV_ERR_CUDA;
    if (clear) {
        const uint32_t zero = 0;
        if (cudaMemcpyToSymbol(g_abi_error, &zero, sizeof(uint32_t)) != cudaSuccess) return QMV_ERR_CUDA;
    }
    *flags = w | w2 | w3 | w4 | w5;
    return QMV_OK;
}

qmv_status qmv_debug_plan_q4(int q4k, int M, int64_t N, int64_t K, int n_inputs, int w_align16, int sm_count,
                             int smem_optin, int smem_per_sm, int64_t *out)
{
    if (!out) return QMV_ERR_NULL;
    qmv_status st = check_shape(M, N, K, q4k ? 256 : 32);
    if (st != QMV_OK) return st;
    if (M < 1 || N < 1 || K < 1 || n_inputs < 1 || n_inputs > kMaxGroup || N < n_inputs || sm_count < 1 ||
        smem_optin < 1 || smem_per_sm < 1)
        return QMV_ERR_SHAPE;
    const DeviceInfo dev{0, sm_count, smem_optin, smem_per_sm};
    // n_inputs matrices of N / n_inputs rows, each reading its own activation; the
    // plan looks only at the weights' alignment, the rows and the distinct inputs
    Q4Group g{};
    g.count = n_inputs;
    g.nx = n_inputs;
    const uintptr_t base = w_align16 ? 0x10000u : 0x10002u;
    for (int i = 0; i <= n_inputs; ++i) g.row_start[i] = N * i / n_inputs;
    for (int i = 0; i < n_inputs; ++i) {
        g.xslot[i] = i;
        g.w[i] = reinterpret_cast<const uint8_t *>(base);
    }
    Q4Plan plan{};
    if (plan_q4_0(dev, g, M, K, &plan, q4k != 0) != cudaSuccess) return QMV_ERR_CUDA;
    int route = plan.route;
    if (q4k && route == kRouteQ4_0Stream) route = kRouteQ4KStream;
    if (q4k && route == kRouteQ4_0Mma) route = kRouteQ4KMma;
    const int64_t v[8] = {route, plan.warps, plan.stages, plan.grid, plan.smem_bytes, plan.act_regs ? 1 : 0,
                          plan.pair ? 1 : 0, plan.chunk_units};
    for (int i = 0; i < 8; ++i) out[i] = v[i];
    return QMV_OK;
}

qmv_status qmv_debug_plan_wq(int fp4, int M, int64_t K, int count, const int64_t *N, int aligned16, int sm_count,
                             int smem_optin, int smem_per_sm, const int *ctas_by_regs, int64_t *out)
{
    if (!out || !N) return QMV_ERR_NULL;
    if (count < 1 || count > kMaxGroup || M < 1 || M > kMaxRowsW || K < 1 || sm_count < 1 || smem_optin < 1 ||
        smem_per_sm < 1)
        return QMV_ERR_SHAPE;
    for (int i = 0; i < count; ++i) {
        qmv_status st = check_shape(M, N[i], K, count > 1 ? (fp4 ? 256 : 128) : (fp4 ? 16 : 1), kMaxRowsW);
        if (st != QMV_OK) return st;
    }
    static const int kLaunchBoundsCtas[3] = {3, 2, 1};   // the kernels' minimum CTAs per SM
    const int *regs = ctas_by_regs ? ctas_by_regs : kLaunchBoundsCtas;
    for (int i = 0; i < 3; ++i)
        if (regs[i] < 1) return QMV_ERR_SHAPE;
    const DeviceInfo dev{0, sm_count, smem_optin, smem_per_sm};
    const cudaError_t e = debug_plan_wq(fp4 != 0, dev, M, K, count, N, aligned16 != 0, regs, out);
    return e == cudaSuccess ? QMV_OK : (e == cudaErrorInvalidValue ? QMV_ERR_SHAPE : QMV_ERR_CUDA);
}

qmv_status qmv_debug_wait_bound(int64_t *out, qmv_stream_t stream)
{
    if (!out) return QMV_ERR_NULL;
    if (misaligned(out, alignof(int64_t))) return QMV_ERR_ALIGN;
    wait_bound_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(out);
    return from_cuda(cudaGetLastError());
}

qmv_status qmv_debug_cta_abort(int64_t *out, int stuck_warp, qmv_stream_t stream)
{
    if (!out) return QMV_ERR_NULL;
    if (misaligned(out, alignof(int64_t))) return QMV_ERR_ALIGN;
    if (stuck_warp < 0 || stuck_warp >= kProbeWarps) return QMV_ERR_SHAPE;
    cta_abort_kernel<<<1, 32 * kProbeWarps, 0, static_cast<cudaStream_t>(stream)>>>(out, stuck_warp);
    return from_cuda(cudaGetLastError());
}

}  // extern "C"
