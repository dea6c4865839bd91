// qmv_internal.h -- host-side interface between the C ABI layer (abi.cu) and the
// kernel translation units. Not installed; not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qmv {

// Kernel choices, counted per launch (the route census).
enum Route : int {
    kRouteQuantizeQ8_1 = 0,
    kRouteQ4_0Stream,     // Q4_0: bulk-copy staged rows, dp4a
    kRouteQ4_0Generic,    // Q4_0: any K % 32 == 0, 2-byte aligned rows
    kRouteQ4_0StreamFused,  // Q4_0 with the Q8_1 quantize in the prologue
    kRouteNvfp4Mma,       // NVFP4: register-fed m16n8k16, K % 256 == 0
    kRouteNvfp4Generic,   // NVFP4: any K % 16 == 0
    kRouteFp8Mma,         // FP8: register-fed m16n8k16, K % 128 == 0
    kRouteFp8Generic,     // FP8: any K
    kRouteZeroFill,       // K == 0: y = 0
    kRouteQ4_0Mma,        // Q4_0: tensor cores (m16n8k32 int8), larger M
    kRouteQ4_0MmaFused,   // ... with the Q8_1 quantize in the prologue
    kRouteQ4KStream,      // Q4_K: the Q4_0 streaming kernel's machinery, K-quant super-blocks
    kRouteQ4KStreamFused, // ... with the Q8_1 quantize in the prologue
    kRouteQ4KMma,         // Q4_K: the Q4_0 tensor-core kernel's machinery (m16n8k32 int8), larger M
    kRouteQ4KMmaFused,    // ... with the Q8_1 quantize in the prologue
    kRouteNvfp4Umma,      // NVFP4: tcgen05.mma (TMEM accumulators), M <= 96 in one weight pass
    kRouteFp8Umma,        // FP8: the same kernel with a byte-wide decode
    kRouteCount
};

const char *route_name(int r);
void route_hit(Route r);

struct DeviceInfo {
    int device;
    int sm_count;
    int smem_optin;     // max dynamic shared memory per block (opt-in)
    int smem_per_sm;
};
// Properties of the current device, cached after the first query.
cudaError_t current_device_info(DeviceInfo *out);

// ---- launchers (arguments already validated by the ABI layer)
cudaError_t launch_quantize_q8_1(const float *x, void *xq, int M, int64_t K, cudaStream_t s);

// Q4_0 plan: which kernel, warps per CTA, ring slots per warp, grid.
struct Q4Plan {
    Route route;
    int warps;         // streaming kernel: warps per CTA
    int stages;        // streaming kernel: ring slots per warp
    int chunk_units;   // 144-byte units per ring slot
    int prefetch;      // streaming kernel: chunks per CTA requested before the programmatic-dependency wait
    int round;         // tensor-core kernel: tiles per reduction round
    int grid;
    int smem_bytes;
    bool act_regs;     // streaming kernel, M <= 2: activation records in registers (rows of U | 32 units)
    bool pair;         // streaming kernel, Q4_0 M = 2..4, rows of 16 units: lane pairs share records
};

// Programmatic dependent launch (opt-in, qmv_set_launch_overlap): fills attr[0]
// and returns 1 when enabled, else returns 0.
int set_launch_overlap_attr(cudaLaunchAttribute *attr);
// Integer from the environment (plan overrides for sweeps), else `fallback`.
int env_int(const char *name, int fallback);
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize = bytes, and the preferred
// shared-memory carveout in percent unless negative) once per kernel and device.
cudaError_t ensure_smem_attr(const void *kernel, int bytes, int carveout = cudaSharedmemCarveoutMaxShared);
// A group of Q4_0 matrices with the same K launched together (count 1 for a
// single call): rows are concatenated in order, each matrix with its own
// activations and outputs. Passed to the kernel by value.
constexpr int kMaxGroup = 8;
struct Q4Group {
    int count;
    const uint8_t *w[kMaxGroup];
    int nx;                        // distinct activations: matrices reading the same one share it
    int xslot[kMaxGroup];          // matrix i reads activation x[xslot[i]]
    const void *x[kMaxGroup];      // fp32 [M][K] (fused) or Q8_1 [M][K/32], x[0 .. nx)
    float *y[kMaxGroup];           // fp32 [M][N_i]
    int64_t row_start[kMaxGroup + 1];
    int cta_start[kMaxGroup + 1];   // streaming kernel: warps of matrix i are [cta_start[i], cta_start[i+1])
};

// q4k: the weights are Q4_K super-blocks (streaming kernel only; route
// kRouteQ4_0Stream when it applies, else kRouteQ4_0Generic = not supported).
cudaError_t plan_q4_0(const DeviceInfo &dev, const Q4Group &grp, int M, int64_t K, Q4Plan *plan, bool q4k = false);
// The tensor-core kernel's plan (route kRouteQ4_0Mma), or route kRouteQ4_0Generic
// when it does not apply.
cudaError_t plan_q4_0_mma(const DeviceInfo &dev, const Q4Group &grp, int M, int64_t K, Q4Plan *plan,
                          bool q4k = false);
cudaError_t launch_q4_0_mma(const Q4Plan &plan, const Q4Group &grp, int32_t *dots, int M, int64_t K, bool fused,
                            cudaStream_t s, bool q4k = false);
cudaError_t launch_q4_0(const Q4Plan &plan, const Q4Group &grp, int32_t *dots, int M, int64_t K, bool fused,
                        cudaStream_t s, bool q4k = false);

// NVFP4 / FP8: a group of matrices with the same K reading the same activations
// (count 1 for a single call). codes: NVFP4 [N][K/2] or FP8 [N][K]; scales: NVFP4
// [N][K/16] E4M3; g: NVFP4 per-tensor scale; row_scale: FP8 [N].
struct WqGroup {
    int count;
    const uint8_t *codes[kMaxGroup];
    const uint8_t *scales[kMaxGroup];
    const float *row_scale[kMaxGroup];
    float g[kMaxGroup];
    float *y[kMaxGroup];
    int64_t N[kMaxGroup];
};

Route plan_nvfp4(const uint8_t *codes, const uint8_t *scales, const uint16_t *x, int64_t K);
cudaError_t launch_nvfp4(Route r, const DeviceInfo &dev, const WqGroup &grp, const uint16_t *x, int M, int64_t K,
                         cudaStream_t s);

Route plan_fp8(const uint8_t *w, const uint16_t *x, int64_t K);
cudaError_t launch_fp8(Route r, const DeviceInfo &dev, const WqGroup &grp, const uint16_t *x, int M, int64_t K,
                       cudaStream_t s);

// The NVFP4 / FP8 plan of one call (count matrices of N[i] rows) on a device given by
// its limits, with CTAs per SM from an occupancy model instead of the device (no CUDA
// call): ctas_by_regs = what the registers of the (8 warps, 1 row tile), (8 warps, 2
// row tiles) and 16-warp kernels allow. out: route, chunks, rows of the first chunk,
// warps, slots, staged, passes, tiles per round, CTAs per SM, grid, shared memory.
cudaError_t debug_plan_wq(bool fp4, const DeviceInfo &dev, int M, int64_t K, int count, const int64_t *N,
                          bool aligned16, const int ctas_by_regs[3], int64_t out[14]);

// Device error words of each translation unit (read synchronously; optionally cleared).
cudaError_t read_error_word_q4_0(uint32_t *out, bool clear);
cudaError_t read_error_word_wq(uint32_t *out, bool clear);
cudaError_t read_error_word_q4_0_mma(uint32_t *out, bool clear);

// Row-major byte matrix [rows][cols] (row stride = cols, a multiple of 16) as a 2-D
// tensor map with a box of box_cols bytes x box_rows rows; zero fill outside.
cudaError_t encode_map_2d(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, uint32_t box_cols,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle);
// Tensor map of `rank` dimensions (dims[0] innermost), strides in bytes of dims 1..rank-1,
// zero fill outside.
cudaError_t encode_map_nd(CUtensorMap *map, CUtensorMapDataType dtype, int rank, const void *base, const uint64_t *dims,
                          const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swizzle);

// NVFP4 / FP8 on the 5th-generation tensor cores (tcgen05, TMEM accumulators): a group
// with M <= 96 rows in one weight pass. K a multiple of 256 (NVFP4) / 128 (FP8), codes,
// NVFP4 scales and x 16-byte aligned.
struct UmmaPlan {
    int n_pad = 0;        // activation rows padded to a multiple of 16 (the MMA's N)
    int T = 0, S = 0, Q = 0, R = 0;   // issuing threads, weight stages, A buffers, activation slices
    int splits = 1;       // CTAs (a cluster) sharing a tile, each a range of K
    int grid = 0;
    uint32_t smem = 0, tmem_cols = 0;
};
// The tcgen05 kernel's plan for `tiles` 128-row tiles (no CUDA call).
cudaError_t plan_umma(bool fp4, const DeviceInfo &dev, int64_t tiles, int M, int64_t K, UmmaPlan *out);
// First M the tcgen05 kernel takes for a launch of `tiles` 128-row tiles: 17, or 9 when
// the tiles fill at most a third of the SMs (QMV_WQ_UMMA_MIN_M / QMV_WQ_UMMA_FEW_TILES_MIN_M
// override; QMV_WQ_UMMA_MIN_M = 0: never).
int umma_min_m(bool fp4, const DeviceInfo &dev, int64_t tiles);
cudaError_t launch_nvfp4_umma(const DeviceInfo &dev, const WqGroup &grp, const uint16_t *x, int M, int64_t K,
                              cudaStream_t s);
cudaError_t launch_fp8_umma(const DeviceInfo &dev, const WqGroup &grp, const uint16_t *x, int M, int64_t K,
                            cudaStream_t s);
cudaError_t read_error_word_umma(uint32_t *out, bool clear);

}  // namespace qmv
