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
//  * Split K: a persistent CTA walks its 16-row tiles in rounds of B tiles; the 8
//    warps take interleaved 128-byte steps of the round (adjacent lines of the same
//    rows in flight together, which keeps DRAM pages open), then reduce in shared
//    memory. B = 8 / gcd(steps per tile, 8), at most 4, makes the steps of a round
//    a multiple of 8, so every warp gets the same number of steps.
//  * Weight streaming: each step's 16 x 128-byte box of codes (and 16 x 16-byte box
//    of E4M3 scales) is one 2-D tensor copy (TMA) into the warp's ring of shared-
//    memory slots, with the hardware 128-byte swizzle so the fragment reads are
//    bank-conflict free and zero fill past the last row. Every warp keeps S steps in
//    flight across tile boundaries, and the first copies are issued before the
//    programmatic-dependency wait.
//  * Activations: staged once per CTA in shared memory when they fit, in an
//    XOR-swizzled layout (16-byte chunk c of a row stored at c ^ 2((c >> 3) & 3),
//    row stride 16 mod 32 bytes) that makes the fragment reads bank-conflict free;
//    when M x K does not fit, K is cut into P equal passes: the CTA walks all its
//    tiles over the first K range with that slice of x staged, restages the next
//    slice, walks them again and adds to the outputs it wrote (its own rows only,
//    so no other CTA is involved and the sum order is fixed). Read through L1
//    only where no pass count fits.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "qmv_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

cudaError_t encode_map_2d(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, uint32_t box_cols,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estride,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_map_nd(CUtensorMap *map, CUtensorMapDataType dtype, int rank, const void *base, const uint64_t *dims,
                          const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swizzle)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || rank < 1 || rank > 5) return cudaErrorNotSupported;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides_bytes[i];
    }
    const CUresult r = enc(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void *>(base), d, st, b, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


namespace {

__device__ uint32_t g_wq_error;

constexpr int kThreads = 256;   // the generic kernel; the tensor-core kernel runs 8 or 16 warps
constexpr int kWarps = 8;
constexpr int kRowsPerCta = 16;
constexpr int kStepBytes = 128;   // bytes of one weight row per warp step
constexpr int kMaxRound = 8;      // tiles per round at most

// Row stride of the staged activations (16 mod 32 bytes) and the chunk swizzle.
__host__ __device__ inline uint32_t xs_row_stride(int64_t K) { return static_cast<uint32_t>(K * 2 + 16); }
__device__ __forceinline__ uint32_t xs_chunk(uint32_t c) { return c ^ (2u * ((c >> 3) & 3u)); }

constexpr int kCodesBox = kRowsPerCta * kStepBytes;   // 2048 bytes: 16 rows x 128 bytes
constexpr int kScalesBox = kRowsPerCta * 16;          // 256 bytes: 16 rows x 16 scales

// floats per partial row of the reduction: 8 activation rows per row tile, + pad
__host__ __device__ constexpr int red_pitch(int mt) { return 8 * mt + 1; }

struct WqLayout {
    uint32_t off_codes, off_scales, off_bar, off_abort, off_red, off_x, total;
};

// Shared memory of W warps: per-warp rings of codes boxes (1024-byte aligned for the
// swizzle), of scale boxes, their mbarriers, the CTA's abort word, the round's
// partial sums [warp][B * 16 rows][8 mt + 1], then the staged activations.
__host__ __device__ inline WqLayout wq_layout(int S, int B, uint32_t xbytes, int mt, int W)
{
    WqLayout L;
    L.off_codes = 0;
    L.off_scales = static_cast<uint32_t>(W * S * kCodesBox);
    L.off_bar = L.off_scales + static_cast<uint32_t>(W * S * kScalesBox);
    L.off_abort = L.off_bar + static_cast<uint32_t>(W * S) * 8u;
    L.off_red = (L.off_abort + 4u + 15u) & ~15u;
    L.off_x = (L.off_red + static_cast<uint32_t>(W * B * kRowsPerCta * red_pitch(mt)) * 4u + 127u) & ~127u;
    L.total = L.off_x + xbytes;
    return L;
}

// A group of matrices with the same K reading the same activations (count 1 for a
// single call): tensor maps of their codes (and NVFP4 scales), scales, outputs, and
// the first tile of each (tiles of 16 rows, numbered over the matrices in order).
struct WqParams {
    CUtensorMap codes[kMaxGroup];
    CUtensorMap scales[kMaxGroup];
    const float *row_scale[kMaxGroup];   // FP8
    float g[kMaxGroup];                  // NVFP4
    float *y[kMaxGroup];
    int64_t N[kMaxGroup];
    int64_t tile_start[kMaxGroup + 1];
    int count;
};

// kFp4: NVFP4 (256 k per step, E4M3 group scales); else FP8 (128 k per step, row scale).
// kMT: 8-row tiles of activations per weight pass (M <= 8 kMT): the decoded weight
// fragments feed kMT mma each, so up to 16 rows share one weight stream.
// kXSmem: activations staged in shared memory.
// kW: warps per CTA (8, or 16 sharing one staged copy of large activations).
// P: passes over K (staged activations only; 1 otherwise), K / kStepK a multiple of P.
template <bool kFp4, bool kXSmem, int kMT, int kW>
__global__ void __launch_bounds__(32 * kW, kW == 16 ? 1 : (kMT == 1 ? 3 : 2))
    wq_mma_kernel(const __grid_constant__ WqParams p,
                                                            const uint16_t *__restrict__ x, int M, int64_t K, int S,
                                                            int B, int P)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte swizzle needs 1024-byte aligned boxes (1 KB extra is allocated)
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    constexpr int kStepK = kFp4 ? 2 * kStepBytes : kStepBytes;
    constexpr int kXWords = kStepK / 8;    // this lane's activation words per step (4 k per 2 words)
    constexpr int kXChunks = kXWords / 4;  // ... in 16-byte chunks

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int64_t ntiles = p.tile_start[p.count];
    const int nsteps = static_cast<int>(K / kStepK) / P;   // steps of one pass
    const int64_t Kp = static_cast<int64_t>(nsteps) * kStepK;
    // matrix of a tile (tiles are numbered over the group's matrices in order), and its first row
    auto locate = [&](int64_t tile, int &mi, int64_t &row0) {
        mi = 0;
#pragma unroll
        for (int i = 1; i < kMaxGroup; ++i)
            if (i < p.count && tile >= p.tile_start[i]) mi = i;
        row0 = (tile - p.tile_start[mi]) * kRowsPerCta;
    };
    constexpr int kPitch = red_pitch(kMT);
    const uint32_t RS = xs_row_stride(Kp);
    constexpr int kT = 32 * kW;   // threads
    const WqLayout L = wq_layout(S, B, kXSmem ? static_cast<uint32_t>(M) * RS : 0u, kMT, kW);
    uint8_t *codes_ring = smem + L.off_codes + warp * S * kCodesBox;
    uint8_t *scales_ring = smem + L.off_scales + warp * S * kScalesBox;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.off_bar) + warp * S;
    uint8_t *xs = smem + L.off_x;
    // partial sums of the round: red(w, row of the round, column)
    float *red_base = reinterpret_cast<float *>(smem + L.off_red);
    auto red = [&](int w, int rr, int m) -> float & {
        return red_base[(w * B * kRowsPerCta + rr) * kPitch + m];
    };
    const uint64_t pol = policy_evict_first();

    // This CTA's tiles blockIdx.x + gridDim.x * lt, lt < nt, in rounds of B tiles; a
    // round's items j = tb * nsteps + step (tile tb of the round), and this warp's
    // are j = warp, warp + kW, ... Lane 0 keeps S of them in flight.
    const int nt = static_cast<int>((ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x);
    // first item of a round for this warp: tile warp / nsteps, step warp % nsteps
    const int tb0 = warp / nsteps, s0 = warp - tb0 * nsteps;
    // producer: pass, local tile, step, end of its round
    int p_ps = 0, p_lt = tb0, p_step = s0, p_rend = min(B, nt);
    // past the end of a round: restart at this warp's first item of the next round,
    // or of the next pass's first round
    auto settle = [&]() {
        while (p_ps < P && p_lt >= p_rend) {
            if (p_rend >= nt) {
                ++p_ps;
                p_rend = 0;
            }
            p_lt = p_rend + tb0;
            p_step = s0;
            p_rend = min(p_rend + B, nt);
        }
    };
    settle();
    int64_t p_tile = -1, p_row0 = 0;   // the producer's last located tile
    int p_mi = 0;
    int outstanding = 0;   // lane 0: copies issued and not yet consumed
    auto issue = [&](int slot) {
        ++outstanding;
        const int64_t tile = blockIdx.x + static_cast<int64_t>(gridDim.x) * p_lt;
        if (tile != p_tile) {
            locate(tile, p_mi, p_row0);
            p_tile = tile;
        }
        const int y0 = static_cast<int>(p_row0);
        mbar_arrive_expect_tx(&bars[slot], kFp4 ? kCodesBox + kScalesBox : kCodesBox);
        const int gs = p_ps * nsteps + p_step;   // step over the whole of K
        tma_load_2d(codes_ring + slot * kCodesBox, &p.codes[p_mi], gs * kStepBytes, y0, &bars[slot], pol);
        if (kFp4) tma_load_2d(scales_ring + slot * kScalesBox, &p.scales[p_mi], gs * 16, y0, &bars[slot], pol);
        p_step += kW;
        while (p_step >= nsteps) {   // once when nsteps >= kW
            p_step -= nsteps;
            ++p_lt;
        }
        settle();
    };
    // rounds before the last hold a multiple of kW items, so a warp with an item in
    // one round has one in every round of the pass but perhaps the last
    auto pending = [&]() { return p_ps < P && p_lt < p_rend; };
    // set when a warp's bounded wait gave up; zeroed before the prologue's barrier
    volatile uint32_t &cta_abort = *reinterpret_cast<volatile uint32_t *>(smem + L.off_abort);
    if (tid == 0) cta_abort = 0u;
    if (lane == 0) {
        for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
        // weights do not depend on the preceding kernel: start streaming them now
        for (int i = 0; i < S && pending(); ++i) issue(i);
    }
    __syncwarp();
    grid_launch_dependents();
    grid_dependency_wait();

    // stage x[:, pass ps] as [M][Kp] fp16, 16-byte chunks, swizzled
    auto stage_x = [&](int ps) {
        const int chunks = static_cast<int>(Kp / 8);
        const uint16_t *src = x + ps * Kp;
        for (int i = tid; i < M * chunks; i += kT) {
            const int m = i / chunks, c = i - m * chunks;
            cp_async_16(xs + m * RS + 16 * xs_chunk(static_cast<uint32_t>(c)), src + static_cast<int64_t>(m) * K + 8 * c);
        }
        cp_async_wait_all();
    };
    if (kXSmem) stage_x(0);
    __syncthreads();

    int slot = 0;   // ring position of this warp's next item
    uint32_t phase = 0;
    for (int ps = 0; ps < P; ++ps) {
        if (ps > 0) {   // every warp is past the previous pass (the barrier ending its last round)
            stage_x(ps);
            __syncthreads();
        }
        for (int round = 0; round * B < nt; ++round) {
            const int bt = min(B, nt - round * B);
            // accumulators; with one row tile the two mma of a word go to d and e, two
            // independent chains (kMT = 2 has its tiles' chains already)
            constexpr bool kDual = kMT == 1 && kXSmem;   // (unstaged: no registers to spare)
            float d[kMT][4], e[kMT][4];
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
                for (int c = 0; c < 4; ++c) d[mt][c] = e[mt][c] = 0.0f;
            int cur = 0;   // tile of the round that d accumulates
            // zero the partials of this warp for tiles of the round it has no step of
            auto flush = [&](int upto) {   // store d as tile cur, zeros for cur+1 .. upto-1
                for (int tb = cur; tb < upto; ++tb) {
                    const bool mine = tb == cur;
#pragma unroll
                    for (int mt = 0; mt < kMT; ++mt) {
                        float v[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) v[c] = mine ? d[mt][c] + (kDual ? e[mt][c] : 0.0f) : 0.0f;
                        red(warp, tb * kRowsPerCta + gid, 8 * mt + 2 * t) = v[0];
                        red(warp, tb * kRowsPerCta + gid, 8 * mt + 2 * t + 1) = v[1];
                        red(warp, tb * kRowsPerCta + gid + 8, 8 * mt + 2 * t) = v[2];
                        red(warp, tb * kRowsPerCta + gid + 8, 8 * mt + 2 * t + 1) = v[3];
                    }
                }
#pragma unroll
                for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) d[mt][c] = e[mt][c] = 0.0f;
            };
            for (int tb = tb0, s = s0; tb < bt;) {
                if (tb != cur) {
                    flush(tb);
                    cur = tb;
                }
                if (!mbar_wait_bounded(&bars[slot], phase)) {
                    if (lane == 0) note_wait_timeout(&g_wq_error, &cta_abort);
                    break;   // skip the rest of the round, up to its barrier
                }
                --outstanding;
                // codes of rows gid and gid+8: 16-byte chunks 2t, 2t+1 of the row (swizzled by row & 7)
                const uint8_t *cb = codes_ring + slot * kCodesBox;
                const uint4 a0 = *reinterpret_cast<const uint4 *>(cb + gid * 128 + 16 * ((2 * t) ^ gid));
                const uint4 a1 = *reinterpret_cast<const uint4 *>(cb + gid * 128 + 16 * ((2 * t + 1) ^ gid));
                const uint4 b0 = *reinterpret_cast<const uint4 *>(cb + (gid + 8) * 128 + 16 * ((2 * t) ^ gid));
                const uint4 b1 = *reinterpret_cast<const uint4 *>(cb + (gid + 8) * 128 + 16 * ((2 * t + 1) ^ gid));
                uint32_t sa = 0, sb = 0;
                if (kFp4) {
                    const uint8_t *sbx = scales_ring + slot * kScalesBox;
                    sa = *reinterpret_cast<const uint32_t *>(sbx + gid * 16 + 4 * t);
                    sb = *reinterpret_cast<const uint32_t *>(sbx + (gid + 8) * 16 + 4 * t);
                }
                __syncwarp();   // the slot is in registers: refill it
                if (lane == 0 && pending()) {
                    fence_proxy_async_shared();   // the warp's reads of the slot before the copy's writes
                    issue(slot);
                }

                // B fragments: activation rows gid + 8 mt. Columns of D past M are never
                // stored, so their lanes need only finite values: from shared memory they
                // read row M - 1 (a broadcast, no divergence); from global memory they skip
                // the load and take zeros (8 lanes load instead of 32 at M = 1, through L1).
                uint32_t xw[kMT][kXWords];
#pragma unroll
                for (int mt = 0; mt < kMT; ++mt) {
                    const int xr = min(gid + 8 * mt, M - 1);
                    if (kXSmem) {
#pragma unroll
                        for (int i = 0; i < kXChunks; ++i) {
                            const uint32_t c = static_cast<uint32_t>(s) * (kStepK / 8) + kXChunks * t + i;
                            const uint4 v = *reinterpret_cast<const uint4 *>(xs + xr * RS + 16 * xs_chunk(c));
                            xw[mt][4 * i] = v.x;
                            xw[mt][4 * i + 1] = v.y;
                            xw[mt][4 * i + 2] = v.z;
                            xw[mt][4 * i + 3] = v.w;
                        }
                    } else if (gid + 8 * mt < M) {
#pragma unroll
                        for (int i = 0; i < kXChunks; ++i) {
                            const uint4 v = ld_shared_v4(x + xr * K + static_cast<int64_t>(ps * nsteps + s) * kStepK +
                                                         (kStepK / 4) * t + 8 * i);
                            xw[mt][4 * i] = v.x;
                            xw[mt][4 * i + 1] = v.y;
                            xw[mt][4 * i + 2] = v.z;
                            xw[mt][4 * i + 3] = v.w;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < kXWords; ++i) xw[mt][i] = 0u;
                    }
                }
                const uint32_t cwa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const uint32_t cwb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                if (kFp4) {
                    // 4 scale bytes: group q covers this lane's codes bytes 8q..8q+7 (k 64t+16q ..).
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
                        const uint32_t a00 = hmul2_u32(ha[0], ga), a01 = hmul2_u32(hb[0], gb);
                        const uint32_t a02 = hmul2_u32(ha[1], ga), a03 = hmul2_u32(hb[1], gb);
                        const uint32_t a10 = hmul2_u32(ha[2], ga), a11 = hmul2_u32(hb[2], gb);
                        const uint32_t a12 = hmul2_u32(ha[3], ga), a13 = hmul2_u32(hb[3], gb);
#pragma unroll
                        for (int mt = 0; mt < kMT; ++mt) {
                            mma_16816(d[mt], a00, a01, a02, a03, xw[mt][4 * i], xw[mt][4 * i + 1]);
                            mma_16816(kDual ? e[mt] : d[mt], a10, a11, a12, a13, xw[mt][4 * i + 2], xw[mt][4 * i + 3]);
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        // word j = codes bytes 4j..4j+3 = k 4j..4j+3 of this lane's run
                        const uint32_t a0 = e4m3x2_to_f16x2(cwa[j] & 0xffffu), a1 = e4m3x2_to_f16x2(cwb[j] & 0xffffu);
                        const uint32_t a2 = e4m3x2_to_f16x2(cwa[j] >> 16), a3 = e4m3x2_to_f16x2(cwb[j] >> 16);
#pragma unroll
                        for (int mt = 0; mt < kMT; ++mt)
                            mma_16816(kDual && (j & 1) ? e[mt] : d[mt], a0, a1, a2, a3, xw[mt][2 * j], xw[mt][2 * j + 1]);
                    }
                }
                if (++slot == S) {
                    slot = 0;
                    phase ^= 1u;
                }
                s += kW;
                while (s >= nsteps) {
                    s -= nsteps;
                    ++tb;
                }
            }
            flush(bt);
            __syncthreads();
            if (cta_abort) {   // a warp gave up waiting: the whole CTA leaves here, its copies landed
                if (lane == 0) drain_ring(bars, S, slot, phase, outstanding);
                return;
            }
            for (int e = tid; e < bt * kRowsPerCta * 8 * kMT; e += kT) {
                const int rr = e / (8 * kMT), m = e - rr * (8 * kMT), tb = rr / kRowsPerCta, r = rr - tb * kRowsPerCta;
                int mi;
                int64_t row0;
                locate(blockIdx.x + static_cast<int64_t>(gridDim.x) * (round * B + tb), mi, row0);
                const int64_t n = row0 + r, Nm = p.N[mi];
                if (m < M && n < Nm) {
                    float sum = 0.0f;
#pragma unroll
                    for (int w = 0; w < kW; ++w) sum += red(w, rr, m);
                    float *out = &p.y[mi][m * Nm + n];
                    // later passes add to what this thread wrote for the same element
                    const float v = sum * (kFp4 ? p.g[mi] : p.row_scale[mi][n]);
                    *out = ps > 0 ? *out + v : v;
                }
            }
            __syncthreads();   // red is reused by the next round
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

// The tensor-core kernel's launch plan for one call (or one chunk of <= 16 rows).
struct WqPlan {
    int W = 0, S = 0, B = 0, P = 1, occ = 0;
    bool xsmem = false;
    int64_t grid = 0;
    uint32_t smem = 0;   // dynamic shared memory, bytes
};

// Plan candidates (warps, ring slots, activations in shared memory), in order of preference.
struct WqCand {
    int W, S;
    bool xs;
};
constexpr WqCand kWqCands[] = {{8, 3, true}, {8, 4, true}, {8, 2, true}, {16, 3, true}, {16, 2, true},
                               {8, 4, false}, {8, 3, false}, {8, 2, false}};
constexpr int kWqCandCount = static_cast<int>(sizeof(kWqCands) / sizeof(kWqCands[0]));

// Chooses the plan of `ntiles` 16-row tiles at M <= 16 rows. occ_of(W, xs, dyn, &occ)
// gives the CTAs per SM of a candidate with `dyn` bytes of dynamic shared memory (the
// occupancy API on a device, a model in the introspection call). Returns
// cudaErrorInvalidValue when no candidate fits.
template <typename OccFn>
cudaError_t choose_wq_plan(bool fp4, const DeviceInfo &dev, int64_t ntiles, int M, int64_t K, OccFn occ_of,
                           WqPlan *out)
{
    const int mt = M > 8 ? 2 : 1;
    const int step_k = fp4 ? 2 * kStepBytes : kStepBytes;   // k per step
    const int64_t nsteps_all = K / step_k;
    // tiles per round for `ns` steps per pass and W warps: a multiple of W / gcd(ns, W),
    // so every warp gets the same number of steps, and enough for 8 steps per warp
    // between the round's barriers
    auto round_unit = [](int64_t ns, int W) {
        int gcd = W;
        while (ns % gcd) gcd >>= 1;   // gcd(ns, W): W is a power of two
        return static_cast<int>(W / gcd);
    };
    auto round_tiles = [&](int64_t ns, int W) {
        const int unit = round_unit(ns, W);
        int b = unit;
        while (b * ns < 8 * W && b + unit <= kMaxRound) b += unit;
        return b;
    };
    // Candidates scored by the tail they leave: whole tiles over `grid` CTAs take
    // ceil(tiles / grid) rounds, so the busiest CTA holds waves * grid / tiles times the
    // mean. Within 15 % of the mean a candidate scores 1, else its imbalance; fewer than
    // 16 resident warps per SM add 0.5 (too few to hide the decode latency), each pass
    // over K beyond the first adds 1 (a pass repeats the per-round reduction), every 8
    // resident warps take 0.05 off (the kernel is bound by latency, and more warps hide
    // more of it: at M = 1 three 8-warp CTAs with 2 slots beat two with 4 on balanced
    // shapes); ties keep the earlier candidate. Activations stay in shared memory
    // whenever they fit (re-read through L1 they thrash it at M = 8); 16 warps share one
    // staged copy where 8-warp CTAs would fit only one per SM. At M <= 2, where the
    // activations fit in L1, an unstaged candidate may win on balance.
    const uint32_t x_cap = static_cast<uint32_t>(env_int("QMV_WQ_XSMEM_MAX", 200 * 1024));
    const int p_env = env_int("QMV_WQ_PASSES", 0);
    const int s_env = env_int("QMV_WQ_SLOTS", 0);
    const int w_env = env_int("QMV_WQ_WARPS", 0);
    int best = -1;
    double best_score = 1e30;
    WqPlan bp;
    for (int c = 0; c < kWqCandCount; ++c) {
        const WqCand &cd = kWqCands[c];
        if (!cd.xs && best >= 0 && kWqCands[best].xs && (M > 2 || best_score <= 1.15)) break;
        if (w_env > 0 && cd.W != w_env) continue;
        const int Wc = cd.W;
        const int Sc = s_env > 0 ? std::min(8, s_env) : cd.S;
        // staged: the fewest passes (dividing the steps) whose slice of x fits, with
        // fewer tiles per round (a smaller reduction buffer) where that makes it fit
        int Pc = 0, Bc = 0;
        uint32_t dyn = 0;
        for (int pp = 1; pp <= (cd.xs ? 8 : 1) && Pc == 0; ++pp) {
            if (p_env > 0 && cd.xs && pp != p_env) continue;
            if (nsteps_all % pp) continue;
            const int64_t ns = nsteps_all / pp;
            const uint64_t xb = cd.xs ? static_cast<uint64_t>(M) * xs_row_stride(ns * step_k) : 0;
            if (xb > x_cap) continue;
            const int unit = round_unit(ns, Wc);
            if (unit > kMaxRound) continue;
            int b = round_tiles(ns, Wc);
            uint32_t d = wq_layout(Sc, b, static_cast<uint32_t>(xb), mt, Wc).total + 1024;
            while (d > static_cast<uint32_t>(dev.smem_optin) && b > unit) {
                b -= unit;
                d = wq_layout(Sc, b, static_cast<uint32_t>(xb), mt, Wc).total + 1024;
            }
            if (d > static_cast<uint32_t>(dev.smem_optin)) continue;
            Pc = pp;
            Bc = b;
            dyn = d;
        }
        if (Pc == 0) continue;
        int occ = 0;
        const cudaError_t e = occ_of(Wc, cd.xs, dyn, &occ);
        if (e != cudaSuccess) return e;
        occ = std::min(occ, 4);
        if (occ < 1) continue;
        const int64_t g = std::min<int64_t>(
            ntiles, std::max<int64_t>(1, static_cast<int64_t>(dev.sm_count) * occ - env_int("QMV_WQ_SPARE_CTAS", 0)));
        const double imb = static_cast<double>((ntiles + g - 1) / g * g) / static_cast<double>(ntiles);
        const double score =
            (imb <= 1.15 ? 1.0 : imb) + (occ * Wc < 16 ? 0.5 : 0.0) + (Pc - 1) - 0.05 * (occ * Wc / 8);
        if (score < best_score) {
            best_score = score;
            best = c;
            bp.W = Wc;
            bp.S = Sc;
            bp.xsmem = cd.xs;
            bp.B = Bc;
            bp.P = Pc;
            bp.occ = occ;
            bp.grid = g;
            bp.smem = dyn;
        }
    }
    if (best < 0) return cudaErrorInvalidValue;
    *out = bp;
    return cudaSuccess;
}

template <bool kFp4>
cudaError_t launch_wq(Route r, const DeviceInfo &dev, const WqGroup &grp, const uint16_t *x, int M, int64_t K,
                      cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = set_launch_overlap_attr(attr);
    if (r == kRouteNvfp4Mma || r == kRouteFp8Mma) {
        route_hit(r);
        // up to 8 activation rows per row tile; 9..16 rows take two tiles per weight pass
        using Kern = void (*)(WqParams, const uint16_t *, int, int64_t, int, int, int);
        const int mt = M > 8 ? 2 : 1;
        auto kernel_of = [mt](bool xs, int W) -> Kern {
            if (W == 16) return mt == 2 ? wq_mma_kernel<kFp4, true, 2, 16> : wq_mma_kernel<kFp4, true, 1, 16>;
            if (mt == 2) return xs ? wq_mma_kernel<kFp4, true, 2, 8> : wq_mma_kernel<kFp4, false, 2, 8>;
            return xs ? wq_mma_kernel<kFp4, true, 1, 8> : wq_mma_kernel<kFp4, false, 1, 8>;
        };
        int64_t ntiles = 0;
        for (int i = 0; i < grp.count; ++i) ntiles += (grp.N[i] + kRowsPerCta - 1) / kRowsPerCta;
        if (ntiles == 0) return cudaSuccess;
        auto occ_of = [&](int W, bool xs, uint32_t dyn, int *occ) -> cudaError_t {
            const Kern kc = kernel_of(xs, W);
            cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kc), dev.smem_optin,
                                             xs ? cudaSharedmemCarveoutMaxShared : -1);
            if (e != cudaSuccess) return e;
            return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, kc, 32 * W, dyn);
        };
        WqPlan plan;
        cudaError_t pe = choose_wq_plan(kFp4, dev, ntiles, M, K, occ_of, &plan);
        if (pe != cudaSuccess) return pe;
        const int W = plan.W, S = plan.S, B = plan.B, P = plan.P;
        const bool xsmem = plan.xsmem;
        const uint32_t xbytes = xsmem ? static_cast<uint32_t>(M) * xs_row_stride(K / P) : 0u;
        const WqLayout L = wq_layout(S, B, xbytes, mt, W);
        cfg.blockDim = dim3(static_cast<unsigned>(32 * W));
        cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
        WqParams p{};
        p.count = grp.count;
        int64_t t = 0;
        for (int i = 0; i < grp.count; ++i) {
            p.tile_start[i] = t;
            t += (grp.N[i] + kRowsPerCta - 1) / kRowsPerCta;
            p.row_scale[i] = grp.row_scale[i];
            p.g[i] = grp.g[i];
            p.y[i] = grp.y[i];
            p.N[i] = grp.N[i];
            if (grp.N[i] == 0) continue;
            cudaError_t e = encode_map_2d(&p.codes[i], grp.codes[i], grp.N[i], kFp4 ? K / 2 : K, kStepBytes,
                                          kRowsPerCta, CU_TENSOR_MAP_SWIZZLE_128B);
            if (e != cudaSuccess) return e;
            if (kFp4) {
                e = encode_map_2d(&p.scales[i], grp.scales[i], grp.N[i], K / 16, 16, kRowsPerCta,
                                  CU_TENSOR_MAP_SWIZZLE_NONE);
                if (e != cudaSuccess) return e;
            }
        }
        for (int i = grp.count; i <= kMaxGroup; ++i) p.tile_start[i] = t;
        const Kern kern = kernel_of(xsmem, W);
        cfg.dynamicSmemBytes = L.total + 1024;
        if (env_int("QMV_PLAN_LOG", 0))   // diagnostic: the chosen plan, one line per launch
            std::fprintf(stderr, "wq plan: fmt=%s M=%d K=%lld tiles=%lld W=%d S=%d xsmem=%d P=%d B=%d occ=%d grid=%u smem=%u\n",
                         kFp4 ? "nvfp4" : "fp8", M, static_cast<long long>(K), static_cast<long long>(ntiles), W, S,
                         xsmem ? 1 : 0, P, B, plan.occ, cfg.gridDim.x, static_cast<unsigned>(cfg.dynamicSmemBytes));
        return cudaLaunchKernelEx(&cfg, kern, p, x, M, K, S, B, P);
    }
    if (grp.count != 1) return cudaErrorInvalidValue;   // groups need the tensor-core kernel
    const int64_t N = grp.N[0];
    const int64_t grid = (N + kWarps - 1) / kWarps;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    auto kern = wq_generic_kernel<kFp4>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), 0, -1);
    if (e != cudaSuccess) return e;
    // 8 activation rows per launch
    for (int m0 = 0; m0 < M; m0 += 8) {
        route_hit(r);
        e = cudaLaunchKernelEx(&cfg, kern, grp.codes[0], grp.scales[0], grp.row_scale[0], grp.g[0], x + m0 * K,
                               grp.y[0] + m0 * N, std::min(8, M - m0), N, K);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t read_error_word_wq(uint32_t *out, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_wq_error, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_wq_error, &zero, sizeof(uint32_t));
}

Route plan_nvfp4(const uint8_t *codes, const uint8_t *scales, const uint16_t *x, int64_t K)
{
    const bool scales4 = (reinterpret_cast<uintptr_t>(scales) & 3u) == 0;
    return (K % 256 == 0 && aligned16(codes) && aligned16(x) && scales4) ? kRouteNvfp4Mma : kRouteNvfp4Generic;
}

Route plan_fp8(const uint8_t *w, const uint16_t *x, int64_t K)
{
    return (K % 128 == 0 && aligned16(w) && aligned16(x)) ? kRouteFp8Mma : kRouteFp8Generic;
}

namespace {

// More than 16 activation rows (up to 96: the chunked packed-FP8 band of the
// README's region-dispatch table, "Native mixed-precision checkpoint path"): M
// is cut into ceil(M / 16) balanced chunks of at most 16 rows, each one launch of
// the tensor-core kernel (one or two 8-row tiles per weight pass). Chunk c + 1
// reads the same weights right after chunk c, from L2 when the group's weights fit
// there. The generic kernel takes any M in 8-row launches already.
// The tcgen05 kernel takes a call from umma_min_m(fp4, tiles) activation rows on, when
// its operands suit TMA: K a multiple of the step, codes, scales and x 16-byte aligned
// (the tensor-core route already requires all but the scales).
bool umma_applies(bool fp4, const DeviceInfo &dev, const WqGroup &grp, int M)
{
    int64_t tiles = 0;
    for (int i = 0; i < grp.count; ++i) tiles += (grp.N[i] + 127) / 128;
    const int min_m = umma_min_m(fp4, dev, tiles);
    if (min_m <= 0 || M < min_m || M > 96) return false;
    for (int i = 0; i < grp.count; ++i)
        if (fp4 && grp.N[i] > 0 && !aligned16(grp.scales[i])) return false;
    return true;
}

template <bool kFp4>
cudaError_t launch_wq_chunked(Route r, const DeviceInfo &dev, const WqGroup &grp, const uint16_t *x, int M,
                              int64_t K, cudaStream_t s)
{
    if ((r == kRouteNvfp4Mma || r == kRouteFp8Mma) && umma_applies(kFp4, dev, grp, M))
        return kFp4 ? launch_nvfp4_umma(dev, grp, x, M, K, s) : launch_fp8_umma(dev, grp, x, M, K, s);
    if (M <= 16 || (r != kRouteNvfp4Mma && r != kRouteFp8Mma)) return launch_wq<kFp4>(r, dev, grp, x, M, K, s);
    const int nch = (M + 15) / 16;
    int m0 = 0;
    for (int c = 0; c < nch; ++c) {
        const int mc = (M - m0 + (nch - c) - 1) / (nch - c);   // ceil(rows left / chunks left) <= 16
        WqGroup g = grp;
        for (int i = 0; i < grp.count; ++i) g.y[i] = grp.y[i] + static_cast<int64_t>(m0) * grp.N[i];
        const cudaError_t e = launch_wq<kFp4>(r, dev, g, x + static_cast<int64_t>(m0) * K, mc, K, s);
        if (e != cudaSuccess) return e;
        m0 += mc;
    }
    return cudaSuccess;
}

}  // namespace

// Where the chunked mma.sync path would take several passes over the weights, the
// tcgen05 kernel's one pass wins (measured in chains of calls, GB/s, mma.sync / tcgen05:
// NVFP4 17408 x 5120 at M = 16: 1945 / 1818, 24: 1058 / 1817, 48: 693 / 1798, 96: 372 /
// 1633; FP8 7168 x 5120 at M = 16: 2595 / 1805, 24: 1395 / 1688, 32: 1336 / 1631, 96:
// 479 / 1282). A launch of at most a third of the SMs' worth of tiles splits K over
// three or more CTAs of a cluster on the tcgen05 kernel, which then wins from 9 rows
// (27B-class stack at M = 16, its 5120-row matrices split in three: 1295 -> 1747 GB/s;
// at M = 8 the mma.sync kernel stays ahead, 2645 / 2090; with only two CTAs per tile,
// FP8 7168 x 5120 at M = 16, it stays ahead too, 2567 / 1804).
// QMV_WQ_UMMA_MIN_M moves the threshold (0: the tcgen05 kernel is never taken);
// QMV_WQ_UMMA_FEW_TILES_MIN_M that of launches of few tiles.
int umma_min_m(bool fp4, const DeviceInfo &dev, int64_t tiles)
{
    (void)fp4;
    const int base = env_int("QMV_WQ_UMMA_MIN_M", 17);
    if (base <= 0) return 0;
    if (tiles * 3 <= dev.sm_count) return env_int("QMV_WQ_UMMA_FEW_TILES_MIN_M", std::min(base, 9));
    return base;
}

cudaError_t debug_plan_wq(bool fp4, const DeviceInfo &dev, int M, int64_t K, int count, const int64_t *N,
                          bool aligned16, const int ctas_by_regs[3], int64_t out[14])
{
    for (int i = 0; i < 14; ++i) out[i] = 0;
    const bool mma = aligned16 && K % (fp4 ? 256 : 128) == 0;
    if (!mma) {   // the generic kernel, 8 activation rows per launch
        if (count != 1) return cudaErrorInvalidValue;
        out[0] = fp4 ? kRouteNvfp4Generic : kRouteFp8Generic;
        out[1] = (M + 7) / 8;
        out[2] = std::min(8, M);
        return cudaSuccess;
    }
    int64_t ntiles = 0;
    for (int i = 0; i < count; ++i) ntiles += (N[i] + kRowsPerCta - 1) / kRowsPerCta;
    int64_t tiles = 0;
    for (int i = 0; i < count; ++i) tiles += (N[i] + 127) / 128;
    const int min_m = umma_min_m(fp4, dev, tiles);
    if (min_m > 0 && M >= min_m) {   // the tcgen05 kernel: 128-row tiles, one pass for all M rows
        UmmaPlan pl;
        const cudaError_t e = plan_umma(fp4, dev, std::max<int64_t>(tiles, 1), M, K, &pl);
        if (e != cudaSuccess) return e;
        const int64_t v[14] = {fp4 ? kRouteNvfp4Umma : kRouteFp8Umma, 1, M, pl.T, pl.S, 1, 1, 1, 1,
                               tiles ? pl.grid : 0, static_cast<int64_t>(pl.smem), pl.Q, pl.R, pl.splits};
        for (int i = 0; i < 14; ++i) out[i] = v[i];
        return cudaSuccess;
    }
    const int nch = M > 16 ? (M + 15) / 16 : 1;
    const int mc = (M + nch - 1) / nch;   // the first (largest) chunk
    out[0] = fp4 ? kRouteNvfp4Mma : kRouteFp8Mma;
    out[1] = nch;
    out[2] = mc;
    if (ntiles == 0) return cudaSuccess;
    const int mt = mc > 8 ? 2 : 1;
    // CTAs per SM: the registers' limit of the variant, the shared memory of the SM
    // less 1 KB reserved per CTA, and 64 resident warps
    auto occ_model = [&](int W, bool, uint32_t dyn, int *occ) -> cudaError_t {
        const int by_regs = ctas_by_regs[W == 16 ? 2 : (mt == 2 ? 1 : 0)];
        *occ = std::min({by_regs, dev.smem_per_sm / static_cast<int>(dyn + 1024), 64 / W});
        return cudaSuccess;
    };
    WqPlan plan;
    const cudaError_t e = choose_wq_plan(fp4, dev, ntiles, mc, K, occ_model, &plan);
    if (e != cudaSuccess) return e;
    const int64_t v[8] = {plan.W, plan.S, plan.xsmem ? 1 : 0, plan.P, plan.B, plan.occ, plan.grid,
                          static_cast<int64_t>(plan.smem)};
    for (int i = 0; i < 8; ++i) out[3 + i] = v[i];
    return cudaSuccess;
}

cudaError_t launch_nvfp4(Route r, const DeviceInfo &dev, const WqGroup &grp, const uint16_t *x, int M, int64_t K,
                         cudaStream_t s)
{
    return launch_wq_chunked<true>(r, dev, grp, x, M, K, s);
}

cudaError_t launch_fp8(Route r, const DeviceInfo &dev, const WqGroup &grp, const uint16_t *x, int M, int64_t K,
                       cudaStream_t s)
{
    return launch_wq_chunked<false>(r, dev, grp, x, M, K, s);
}

}  // namespace qmv
