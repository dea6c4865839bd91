// qmv_internal.h -- host-side interface between the C ABI layer (abi.cu) and the
// kernel translation units. Not installed; not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qmv {

// Kernel choices, counted per launch (the route census).
enum Route : int {
    kRouteQuantizeQ8_1 = 0,
    kRouteQ4_0Stream,     // Q4_0: bulk-copy staged rows, dp4a
    kRouteQ4_0Generic,    // Q4_0: any K % 32 == 0, 2-byte aligned rows
    kRouteNvfp4Mma,       // NVFP4: register-fed m16n8k16, K % 256 == 0
    kRouteNvfp4Generic,   // NVFP4: any K % 16 == 0
    kRouteFp8Mma,         // FP8: register-fed m16n8k16, K % 128 == 0
    kRouteFp8Generic,     // FP8: any K
    kRouteZeroFill,       // K == 0: y = 0
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

// Q4_0 plan: which kernel, tile rows, pipeline stages, grid.
struct Q4Plan {
    Route route;
    int rows_per_tile;
    int stages;
    int grid;
    int smem_bytes;
};
cudaError_t plan_q4_0(const DeviceInfo &dev, const void *w, const void *xq, int M, int64_t N, int64_t K,
                      Q4Plan *plan);
cudaError_t launch_q4_0(const Q4Plan &plan, const void *w, const void *xq, float *y, int32_t *dots, int M,
                        int64_t N, int64_t K, cudaStream_t s);

Route plan_nvfp4(const uint8_t *codes, const uint8_t *scales, const uint16_t *x, int64_t K);
cudaError_t launch_nvfp4(Route r, const DeviceInfo &dev, const uint8_t *codes, const uint8_t *scales, float g,
                         const uint16_t *x, float *y, int M, int64_t N, int64_t K, cudaStream_t s);

Route plan_fp8(const uint8_t *w, const uint16_t *x, int64_t K);
cudaError_t launch_fp8(Route r, const DeviceInfo &dev, const uint8_t *w, const float *rs, const uint16_t *x,
                       float *y, int M, int64_t N, int64_t K, cudaStream_t s);

// Device error words of each translation unit (read synchronously; optionally cleared).
cudaError_t read_error_word_q4_0(uint32_t *out, bool clear);

}  // namespace qmv
