// wq_umma.cu -- NVFP4 W4A16 and FP8 W8A16 skinny GEMM on the 5th-generation tensor
// cores (tcgen05), M = 1..96 activation rows in one pass over the weights.
//
// QPN2 / QPN8 of "v100-skinny README", section "How QPN works": packed weights are
// streamed once and decoded on chip into the operands of a tensor-core product
// against fp16 activations, with fp32 accumulation. The page's Volta kernels decode
// into mma registers lane by lane; here the product is tcgen05.mma issued by one
// thread per CTA, so the warps only decode:
//  * A tile = 128 weight rows x K of one matrix (TMEM lane = weight row); B = the M
//    activation rows, padded with zero rows to N = 16 ceil(M / 16) <= 96; D (fp32,
//    128 x N) accumulates over all of K in tensor memory. The whole activation
//    width rides one weight pass: the README's M = 9..16 and 17..96 bands need no
//    second pass over the weights and no chunking.
//  * Exact decode, as in the mma.sync kernel: an E2M1 code times its E4M3 group
//    scale is exact in fp16 (at most 6 significant bits, magnitude 2^-10 .. 2688),
//    so the scale is folded into the fp16 weight; E4M3 to fp16 is exact; the
//    per-tensor scale (NVFP4) or the row scale (FP8) multiplies the fp32 result.
//  * Roles (warp specialisation): warp 0 streams, per K step, the codes (a 128-row
//    box with the 128-byte swizzle), the group scales and the activation slice (a
//    3-D box that lands in the tensor cores' K-major core-matrix layout, rows past M
//    zero-filled) with TMA into a ring of stages; warps 2..5 decode one weight row
//    per thread into fp16 core matrices of a 64-k A buffer (double-buffered); warp 1
//    allocates tensor memory and one of its threads issues the MMAs (4 per 64 k);
//    the decode warps read the accumulators back (tcgen05.ld) and store y. The
//    accumulator is double-buffered across tiles, so a tile's read-back overlaps the
//    next tile's MMAs.
//  * Every mbarrier wait is bounded; a thread whose wait gives up flags the error
//    word and the CTA's abort word and leaves its loop; all threads meet at the final
//    barrier, the producer lets its copies land, the MMA thread waits for its
//    products to complete and the tensor memory is released before the CTA exits.
#include <algorithm>
#include <cstdio>

#include <cuda.h>

#include "qmv_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

__device__ uint32_t g_umma_error;

constexpr int kTileRows = 128;         // MMA M: weight rows per tile = TMEM lanes
constexpr int kQuarterK = 64;          // k per A buffer (8 core matrices of 8 k)
constexpr int kCodesBox = kTileRows * 128;   // one step's codes: 128 rows x 128 bytes
constexpr int kScalesBox = kTileRows * 16;   // NVFP4: 128 rows x 16 E4M3 scales
constexpr int kABytes = kTileRows * kQuarterK * 2;   // 16 KB of fp16 per A buffer
constexpr int kDecodeWarps = 8;        // two threads per weight row, each half of a 64-k buffer
constexpr int kFirstDecodeWarp = 3;    // warp 0 weight producer, 1 tensor memory, 2 activation producer, 3..10 decode
constexpr int kMaxIssuers = 8;         // warps 11 .. 11 + T - 1: one MMA-issuing thread each
constexpr int kFirstIssuerWarp = kFirstDecodeWarp + kDecodeWarps;
constexpr int kThreadsUmma = 32 * (kFirstIssuerWarp + kMaxIssuers);
constexpr int kMaxStages = 8;          // weight stages (one K step of codes and scales each)
constexpr int kMaxABufs = 8;           // 64-k A buffers and 64-k activation slices

__host__ __device__ constexpr int step_k(bool fp4) { return fp4 ? 256 : 128; }   // 128 code bytes per row

struct UmmaLayout {
    uint32_t off_codes, off_scales, off_b, off_a, off_bar, off_misc, total;
    uint32_t b_bytes;   // one 64-k activation slice: 64 x N fp16
};

// Dynamic shared memory (base aligned to 1024 bytes): S weight stages of codes
// (1024-aligned for the 128-byte swizzle) and scales, R 64-k activation slices, Q 64-k
// A buffers, the mbarriers, the tensor-memory address and the abort word.
__host__ __device__ inline UmmaLayout umma_layout(bool fp4, int S, int R, int Q, int n_pad)
{
    UmmaLayout L;
    L.b_bytes = static_cast<uint32_t>(kQuarterK * n_pad * 2);
    L.off_codes = 0;
    L.off_scales = L.off_codes + static_cast<uint32_t>(S * kCodesBox);
    L.off_b = (L.off_scales + (fp4 ? static_cast<uint32_t>(S * kScalesBox) : 0u) + 1023u) & ~1023u;
    L.off_a = (L.off_b + static_cast<uint32_t>(R) * L.b_bytes + 1023u) & ~1023u;
    L.off_bar = L.off_a + static_cast<uint32_t>(Q) * kABytes;
    // w_full, w_free: S each; b_full, b_free: R each; a_full, a_free: Q each; acc_full, acc_free, done
    L.off_misc = L.off_bar + static_cast<uint32_t>(2 * S + 2 * R + 2 * Q + 3) * 8u;
    L.total = L.off_misc + 16u;
    return L;
}

// Group of matrices with the same K reading the same activations: tensor maps of each
// matrix's codes (and NVFP4 scales), its first tile, scale and output.
struct UmmaParams {
    CUtensorMap codes[kMaxGroup];
    CUtensorMap scales[kMaxGroup];
    CUtensorMap x;                       // activations: {K, M} fp16, 64 x n_pad boxes
    const float *row_scale[kMaxGroup];   // FP8
    float g[kMaxGroup];                  // NVFP4
    float *y[kMaxGroup];
    int64_t N[kMaxGroup];
    int tile_start[kMaxGroup + 1];
    int count;
};

// ---------------------------------------------------------------- tcgen05 helpers (inline PTX)

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzled
// layout: rows of 64 fp16 (128 bytes) at a 128-byte pitch, 8-row groups 1024 bytes
// apart (sbo), the 16-byte chunk c of row r stored at chunk c ^ (r % 8) from a
// 1024-byte aligned base -- the layout a TMA box with the 128-byte swizzle lands in.
// A K step of 16 within the 64-k row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (1ull << 16) |   // leading offset: unused (1)
           (static_cast<uint64_t>(1024u >> 4) << 32) | (1ull << 46) |       // sbo = 1024; bits 46..48 = 0b001
           (2ull << 61);                                                    // swizzle mode: 128 bytes
}

// Instruction descriptor of kind::f16: fp16 A and B (both K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n)
{
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The mbarrier completes (one arrival) when every earlier tcgen05 operation of this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's TMEM lane (warp-wide, .sync.aligned).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- the kernel

// T MMA-issuing threads (one per warp) take the 64-k quarters round robin, each into
// its own accumulator: one thread's products that are tracked by commits complete
// about one per 150 ns on this part, and several threads' streams overlap (measured:
// 2 / 4 / 8 threads -> 77 / 38 / 21 ns per 128 x 16 x 16 product). The read-back sums
// the T accumulators in a fixed order, so results do not depend on the interleaving.
template <bool kFp4>
__global__ void __launch_bounds__(kThreadsUmma, 1)
    wq_umma_kernel(const __grid_constant__ UmmaParams p, int M, int64_t K, int n_pad, int S, int R, int Q, int T,
                   uint32_t tmem_cols)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const UmmaLayout L = umma_layout(kFp4, S, R, Q, n_pad);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kStepK = step_k(kFp4);
    constexpr int kQuarters = kStepK / kQuarterK;
    const int nsteps = static_cast<int>(K / kStepK);
    const int tile_quarters = nsteps * kQuarters;
    const int ntiles = p.tile_start[p.count];
    const int nt = (ntiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                   static_cast<int>(gridDim.x);   // tiles of this CTA: blockIdx.x + gridDim.x * lt
    const int total_steps = nt * nsteps, total_quarters = total_steps * kQuarters;
    const int used = min(T, tile_quarters);   // accumulators a tile writes

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.off_bar);
    uint64_t *w_full = bars, *w_free = bars + S, *b_full = bars + 2 * S, *b_free = b_full + R;
    uint64_t *a_full = b_free + R, *a_free = a_full + Q, *acc_full = a_free + Q, *acc_free = acc_full + 1;
    uint64_t *done = acc_free + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile uint32_t *abort_word = reinterpret_cast<volatile uint32_t *>(smem + L.off_misc + 4);
    uint8_t *codes_ring = smem + L.off_codes, *scales_ring = smem + L.off_scales;
    uint8_t *b_ring = smem + L.off_b, *a_buf = smem + L.off_a;

    auto locate = [&](int tile, int &mi, int &row0) {
        mi = 0;
#pragma unroll
        for (int i = 1; i < kMaxGroup; ++i)
            if (i < p.count && tile >= p.tile_start[i]) mi = i;
        row0 = (tile - p.tile_start[mi]) * kTileRows;
    };
    auto fail = [&]() { note_wait_timeout(&g_umma_error, abort_word); };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_free[s], kDecodeWarps);
        }
        for (int j = 0; j < R; ++j) {
            mbar_init(&b_full[j], 1);
            mbar_init(&b_free[j], 1);
        }
        for (int j = 0; j < Q; ++j) {
            mbar_init(&a_full[j], kDecodeWarps);
            mbar_init(&a_free[j], 1);
        }
        mbar_init(acc_full, used);
        mbar_init(acc_free, kDecodeWarps);
        mbar_init(done, T);
        *abort_word = 0u;
        fence_barrier_init();
    }
    if (warp == 1) {   // tensor memory: T accumulators of n_pad columns x 128 lanes
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------ weight producer (one thread)
        // Weights do not depend on the preceding kernel: the ring fills before the
        // dependency wait (this thread never waits for it: it touches no activation).
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const uint32_t tx = kCodesBox + (kFp4 ? kScalesBox : 0);
            int issued = 0;
            for (int g = 0; g < total_steps && !*abort_word; ++g) {
                const int s = g % S;
                if (g >= S && !mbar_wait_bounded(&w_free[s], static_cast<uint32_t>((g / S) - 1) & 1u)) {
                    fail();
                    break;
                }
                const int lt = g / nsteps, st = g - lt * nsteps;
                int mi, row0;
                locate(static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) * lt, mi, row0);
                mbar_arrive_expect_tx(&w_full[s], tx);
                tma_load_2d(codes_ring + s * kCodesBox, &p.codes[mi], st * 128, row0, &w_full[s], pol);
                if (kFp4) tma_load_2d(scales_ring + s * kScalesBox, &p.scales[mi], st * 16, row0, &w_full[s], pol);
                issued = g + 1;
            }
            for (int g = max(0, issued - S); g < issued; ++g)   // every copy lands before the CTA can exit
                (void)mbar_wait_bounded(&w_full[g % S], static_cast<uint32_t>(g / S) & 1u);
        }
    } else if (warp == 2) {
        // ------------------------------------------------ activation producer (one thread): 64-k slices
        if (lane == 0) {
            grid_dependency_wait();
            const uint64_t pol_x = policy_evict_last();
            int issued = 0;
            for (int h = 0; h < total_quarters && !*abort_word; ++h) {
                const int j = h % R;
                if (h >= R && !mbar_wait_bounded(&b_free[j], static_cast<uint32_t>((h / R) - 1) & 1u)) {
                    fail();
                    break;
                }
                const int kq = h % tile_quarters;   // 64-k slice of K
                mbar_arrive_expect_tx(&b_full[j], L.b_bytes);
                tma_load_2d(b_ring + j * L.b_bytes, &p.x, kq * kQuarterK, 0, &b_full[j], pol_x);
                issued = h + 1;
            }
            for (int h = max(0, issued - R); h < issued; ++h)
                (void)mbar_wait_bounded(&b_full[h % R], static_cast<uint32_t>(h / R) & 1u);
        }
    } else if (warp >= kFirstIssuerWarp) {
        // ------------------------------------------------ MMA issue: thread t takes quarters t, t + T, ...
        const int t = warp - kFirstIssuerWarp;
        if (lane == 0 && t < T) {
            const uint32_t idesc = idesc_f16_f32(kTileRows, n_pad);
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(t * n_pad);
            bool ok = true, any = false;
            for (int lt = 0; lt < nt && ok; ++lt) {
                if (lt >= 1 && t < used &&   // the read-back of the previous tile is done
                    !mbar_wait_bounded(acc_free, static_cast<uint32_t>(lt - 1) & 1u)) {
                    fail();
                    break;
                }
                tc_fence_after();
                bool first = true;
                for (int kq = t; kq < tile_quarters && ok; kq += T) {
                    const int h = lt * tile_quarters + kq;
                    const int ja = h % Q, jb = h % R;
                    if (*abort_word || !mbar_wait_bounded(&b_full[jb], static_cast<uint32_t>(h / R) & 1u) ||
                        !mbar_wait_bounded(&a_full[ja], static_cast<uint32_t>(h / Q) & 1u)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_addr(a_buf + ja * kABytes);
                    const uint32_t b_base = smem_addr(b_ring + jb * L.b_bytes);
#pragma unroll
                    for (int kk = 0; kk < kQuarterK / 16; ++kk)
                        umma_f16(d_tmem, smem_desc_sw128(a_base + 32u * kk), smem_desc_sw128(b_base + 32u * kk), idesc,
                                 (first && kk == 0) ? 0u : 1u);
                    first = false;
                    any = true;
                    umma_commit(&a_free[ja]);   // the A buffer and the activation slice are free once
                    umma_commit(&b_free[jb]);   // these products are done
                }
                if (ok && t < used) umma_commit(acc_full);   // this thread's share of the tile is done
            }
            // every product this thread issued has completed before the tensor memory is released
            if (any) {
                umma_commit(done);
            } else {
                mbar_arrive(done);
            }
            (void)mbar_wait_bounded(done, 0u);
        }
        __syncwarp();
    } else if (warp >= kFirstDecodeWarp) {
        // ------------------------------------------------ decode, then read back
        // Two threads per weight row: warps 3..6 take k groups 0..3 of every 64-k
        // buffer, warps 7..10 groups 4..7; the row is this warp's TMEM lane quarter.
        const int r = 32 * (warp & 3) + lane;
        const int hf = (warp - kFirstDecodeWarp) >> 2;
        uint8_t *a_row = a_buf + r * 128;   // chunk c (k 8c .. 8c + 7) at 16 (c ^ (r % 8))
        const int sw = r & 7;
        int g = 0, h = 0;
        bool ok = true, waited = false;
        for (int lt = 0; lt < nt && ok; ++lt) {
            int mi, row0;
            locate(static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) * lt, mi, row0);
            for (int st = 0; st < nsteps && ok; ++st, ++g) {
                const int s = g % S;
                if (*abort_word || !mbar_wait_bounded(&w_full[s], static_cast<uint32_t>(g / S) & 1u)) {
                    fail();
                    ok = false;
                    break;
                }
                const uint8_t *crow = codes_ring + s * kCodesBox + r * 128;
                for (int q = 0; q < kQuarters; ++q, ++h) {
                    const int j = h % Q;
                    if (h >= Q && !mbar_wait_bounded(&a_free[j], static_cast<uint32_t>((h / Q) - 1) & 1u)) {
                        fail();
                        ok = false;
                        break;
                    }
                    uint8_t *dst = a_row + j * kABytes;
                    if (kFp4) {
                        // k 64q + 32hf .. + 31: code chunk 2q + hf (swizzled by row), groups 4q + 2hf, + 1
                        const uint4 c = *reinterpret_cast<const uint4 *>(crow + 16 * ((2 * q + hf) ^ sw));
                        const uint32_t s2 = *reinterpret_cast<const uint16_t *>(scales_ring + s * kScalesBox + r * 16 +
                                                                                 4 * q + 2 * hf);
                        const uint32_t s01 = e4m3x2_to_f16x2(s2);
                        const uint32_t sc0 = dup_lo16(s01), sc1 = dup_hi16(s01);
                        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                        for (int kg = 0; kg < 4; ++kg) {   // 8 k: one word of codes, group kg / 2
                            uint32_t hv[4];
                            e2m1x8_to_f16x2(cw[kg], hv);
                            const uint32_t gsc = kg < 2 ? sc0 : sc1;
                            *reinterpret_cast<uint4 *>(dst + 16 * ((4 * hf + kg) ^ sw)) =
                                make_uint4(hmul2_u32(hv[0], gsc), hmul2_u32(hv[1], gsc), hmul2_u32(hv[2], gsc),
                                           hmul2_u32(hv[3], gsc));
                        }
                    } else {
                        // k 64q + 32hf .. + 31: code chunks 4q + 2hf, + 1, 8 bytes per k8 group
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(crow + 16 * ((4 * q + 2 * hf + c) ^ sw));
                            *reinterpret_cast<uint4 *>(dst + 16 * ((4 * hf + 2 * c) ^ sw)) =
                                make_uint4(e4m3x2_to_f16x2(v.x & 0xffffu), e4m3x2_to_f16x2(v.x >> 16),
                                           e4m3x2_to_f16x2(v.y & 0xffffu), e4m3x2_to_f16x2(v.y >> 16));
                            *reinterpret_cast<uint4 *>(dst + 16 * ((4 * hf + 2 * c + 1) ^ sw)) =
                                make_uint4(e4m3x2_to_f16x2(v.z & 0xffffu), e4m3x2_to_f16x2(v.z >> 16),
                                           e4m3x2_to_f16x2(v.w & 0xffffu), e4m3x2_to_f16x2(v.w >> 16));
                        }
                    }
                    fence_proxy_async_shared();   // the generic writes of A before the tensor core reads it
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&a_full[j]);
                }
                if (ok && lane == 0) mbar_arrive(&w_free[s]);   // (the warp's reads fenced above)
            }
            if (!ok) break;
            // read back tile lt: row row0 + r of matrix mi, activation rows in 16-column
            // chunks (the two warps of a lane quarter take alternate chunks), the
            // accumulators of the issuing threads summed in a fixed order
            if (!waited) {   // outputs may be read by the preceding kernel until it has finished
                grid_dependency_wait();
                waited = true;
            }
            if (!mbar_wait_bounded(acc_full, static_cast<uint32_t>(lt) & 1u)) {
                fail();
                break;
            }
            tc_fence_after();
            const int64_t n = row0 + r, Nm = p.N[mi];
            const float scale = kFp4 ? p.g[mi] : (n < Nm ? __ldg(p.row_scale[mi] + n) : 0.0f);
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
            for (int c16 = 16 * hf; c16 < n_pad; c16 += 32) {
                float v[16];
                tmem_ld16(taddr + static_cast<uint32_t>(c16), v);
                for (int a = 1; a < used; ++a) {
                    float u[16];
                    tmem_ld16(taddr + static_cast<uint32_t>(a * n_pad + c16), u);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += u[i];
                }
                if (n < Nm) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (c16 + i < M) p.y[mi][static_cast<int64_t>(c16 + i) * Nm + n] = v[i] * scale;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
    }
}

// 2-D tensor map of fp16 activations x [M][K] with a box of 64 k x n_pad rows and the
// 128-byte swizzle: a box lands as the K-major swizzled B operand (rows of 128 bytes,
// rows past M zero-filled).
cudaError_t encode_x_map(CUtensorMap *map, const uint16_t *x, int M, int64_t K, int n_pad)
{
    const uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(K) * 2};
    const uint32_t box[2] = {static_cast<uint32_t>(kQuarterK), static_cast<uint32_t>(n_pad)};
    return encode_map_nd(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

cudaError_t plan_umma(bool fp4, const DeviceInfo &dev, int64_t tiles, int M, int64_t K, UmmaPlan *out)
{
    UmmaPlan pl;
    pl.n_pad = 16 * ((M + 15) / 16);
    // MMA-issuing threads T, each with one accumulator of n_pad columns (512 columns in
    // all), one 64-k A buffer and one activation slice: thread t takes quarters t, t + T,
    // ... and always the same buffers, so it waits for every phase of them in order (with
    // fewer buffers than threads a thread could reach a buffer's next phase while the
    // previous one is pending and pass its parity test on the phase before). Then as many
    // weight stages (the bytes in flight from HBM) as shared memory holds, at least 3.
    int T = std::max(1, std::min({kMaxIssuers, 512 / pl.n_pad, env_int("QMV_UMMA_ISSUERS", kMaxIssuers)}));
    auto fits = [&](int s_, int t_) {
        return umma_layout(fp4, s_, std::max(2, t_), std::max(2, t_), pl.n_pad).total + 1024 <=
               static_cast<uint32_t>(dev.smem_optin);
    };
    while (T > 1 && !fits(3, T)) --T;
    int S = std::max(2, std::min(kMaxStages, env_int("QMV_UMMA_STAGES", kMaxStages)));
    while (S > 2 && !fits(S, T)) --S;
    pl.T = T;
    pl.S = S;
    pl.Q = pl.R = std::max(2, T);
    pl.smem = umma_layout(fp4, pl.S, pl.R, pl.Q, pl.n_pad).total + 1024;
    if (pl.smem > static_cast<uint32_t>(dev.smem_optin) || K % step_k(fp4) != 0) return cudaErrorInvalidValue;
    pl.tmem_cols = 32;
    while (pl.tmem_cols < static_cast<uint32_t>(T * pl.n_pad)) pl.tmem_cols <<= 1;
    pl.grid = static_cast<int>(std::min<int64_t>(tiles, dev.sm_count));
    *out = pl;
    return cudaSuccess;
}

namespace {

template <bool kFp4>
cudaError_t launch_umma(const DeviceInfo &dev, const WqGroup &grp, const uint16_t *x, int M, int64_t K,
                        cudaStream_t s)
{
    int tiles = 0;
    for (int i = 0; i < grp.count; ++i) tiles += static_cast<int>((grp.N[i] + kTileRows - 1) / kTileRows);
    if (tiles == 0) return cudaSuccess;
    UmmaPlan pl;
    cudaError_t pe = plan_umma(kFp4, dev, tiles, M, K, &pl);
    if (pe != cudaSuccess) return pe;
    const int n_pad = pl.n_pad, S = pl.S, R = pl.R, Q = pl.Q, T = pl.T;
    const uint32_t smem = pl.smem, cols = pl.tmem_cols;
    UmmaParams p{};
    p.count = grp.count;
    int t = 0;
    for (int i = 0; i < grp.count; ++i) {
        p.tile_start[i] = t;
        t += static_cast<int>((grp.N[i] + kTileRows - 1) / kTileRows);
        p.row_scale[i] = grp.row_scale[i];
        p.g[i] = grp.g[i];
        p.y[i] = grp.y[i];
        p.N[i] = grp.N[i];
        if (grp.N[i] == 0) continue;
        cudaError_t e = encode_map_2d(&p.codes[i], grp.codes[i], grp.N[i], kFp4 ? K / 2 : K, 128, kTileRows,
                                      CU_TENSOR_MAP_SWIZZLE_128B);
        if (e != cudaSuccess) return e;
        if (kFp4) {
            e = encode_map_2d(&p.scales[i], grp.scales[i], grp.N[i], K / 16, 16, kTileRows, CU_TENSOR_MAP_SWIZZLE_NONE);
            if (e != cudaSuccess) return e;
        }
    }
    for (int i = grp.count; i <= kMaxGroup; ++i) p.tile_start[i] = t;
    cudaError_t e = encode_x_map(&p.x, x, M, K, n_pad);
    if (e != cudaSuccess) return e;
    auto kern = wq_umma_kernel<kFp4>;
    if ((e = ensure_smem_attr(reinterpret_cast<const void *>(kern), static_cast<int>(smem))) != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreadsUmma);
    cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = set_launch_overlap_attr(attr);
    if (env_int("QMV_PLAN_LOG", 0))
        std::fprintf(stderr,
                     "umma plan: fmt=%s M=%d n_pad=%d K=%lld tiles=%d S=%d R=%d Q=%d issuers=%d grid=%u smem=%u "
                     "tmem=%u\n",
                     kFp4 ? "nvfp4" : "fp8", M, n_pad, static_cast<long long>(K), tiles, S, R, Q, T, cfg.gridDim.x,
                     smem, cols);
    return cudaLaunchKernelEx(&cfg, kern, p, M, K, n_pad, S, R, Q, T, cols);
}

}  // namespace

cudaError_t launch_nvfp4_umma(const DeviceInfo &dev, const WqGroup &grp, const uint16_t *x, int M, int64_t K,
                              cudaStream_t s)
{
    route_hit(kRouteNvfp4Umma);
    return launch_umma<true>(dev, grp, x, M, K, s);
}

cudaError_t launch_fp8_umma(const DeviceInfo &dev, const WqGroup &grp, const uint16_t *x, int M, int64_t K,
                            cudaStream_t s)
{
    route_hit(kRouteFp8Umma);
    return launch_umma<false>(dev, grp, x, M, K, s);
}

cudaError_t read_error_word_umma(uint32_t *out, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_umma_error, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_umma_error, &zero, sizeof(uint32_t));
}

}  // namespace qmv
