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
// 18 bytes, a whole number of 144-byte units (8 blocks, 9 x 16 bytes). The grid is
// persistent and every warp owns a contiguous span of rows of one matrix, i.e. one
// contiguous, 16-byte aligned byte range, which it streams through its own ring
// of shared-memory slots with one 1-D bulk copy of up to 32 units (4608 bytes) per
// iteration (mbarrier completion, evict-first L2 hint): after the activation
// prologue no warp waits for another, and the cost of issuing a copy is spread
// over all warps of the SM. Per iteration a lane takes one unit -- nine
// conflict-free 16-byte shared-memory reads, 8 blocks of independent work -- and
// rows that end inside the chunk are closed with a warp segmented scan (a row may
// span chunks: its partial sum is carried). The high nibbles are summed under a
// 0xF0 mask (one shift per block, not per word). Weight copies are issued before
// the programmatic-dependency wait: with programmatic dependent launch the next
// call's weights stream in while the previous call finishes.
#include <algorithm>

#include "q8_1_block.cuh"
#include "qmv_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

__device__ uint32_t g_q4_error;

// Stage trace (profiling builds only, compiled with -DQMV_STAGE_TRACE): every warp of
// the streaming kernel records %globaltimer at its start, after the programmatic-
// dependency wait, after the activation prologue's barrier, when its first chunk has
// landed and at its end, with its SM, into a per-launch record the host assigns
// (qmv_stage_trace_set). gemm_qmv_quantize_gb300/stage_trace.py reads the records.
#ifdef QMV_STAGE_TRACE
constexpr int kTraceWarps = 16, kTraceFields = 8;   // per warp: 5 times, SM, chunks, valid
#define QMV_TRACE_PARAM , unsigned long long *trace
#define QMV_TRACE_STAMP(var) var = globaltimer_ns()
#else
#define QMV_TRACE_PARAM
#define QMV_TRACE_STAMP(var)
#endif

constexpr int kThreads = 256;        // generic kernel
constexpr int kWarps = kThreads / 32;
constexpr int kStreamThreads = 512;      // streaming kernel, M <= kWideFromM - 1: up to 16 warps
constexpr int kStreamThreadsWide = 256;  // streaming kernel, larger M: up to 8 warps
#ifndef QMV_Q4_WIDE_FROM_M
#define QMV_Q4_WIDE_FROM_M 3
#endif
constexpr int kWideFromM = QMV_Q4_WIDE_FROM_M;   // first M whose registers allow only 8 warps
__host__ __device__ constexpr int stream_threads(int M) { return M < kWideFromM ? kStreamThreads : kStreamThreadsWide; }
constexpr int kActRegsThreads = 512;     // streaming kernel with register-resident activations
// Staged activations, per activation row, one record per unit (8 blocks):
// q8[256] (bytes 0..255), d8[8] as fp32 (256..287), 8*sum(q8)[8] (288..319),
// padded to 336 bytes (21 x 16, odd) so 16-byte reads of consecutive records by
// eight lanes fall in distinct bank groups.
constexpr int kActUnitStride = 336;
constexpr int kActD8Off = 256, kActT8Off = 288;
constexpr int kUnitBytes = 144;      // 8 blocks: the 16-byte aligned unit of a row
constexpr int kChunkUnits = 32;      // units per ring slot: one per lane

struct Q4Layout {
    uint32_t rowbytes, units, slotbytes;
    uint32_t off_act, act_m_stride, off_ring, ring_warp_stride, off_bar, total;
};

// Shared memory: staged activations (act_rows = distinct activations x M rows), then one ring of
// S slots of 32 units per warp, then the warps' mbarriers.
__host__ __device__ inline Q4Layout q4_layout(int act_rows, int64_t K, int warps, int S)
{
    Q4Layout L;
    const uint32_t nb = static_cast<uint32_t>(K / 32);
    L.units = static_cast<uint32_t>(K / 256);
    L.rowbytes = nb * 18u;
    L.slotbytes = kChunkUnits * kUnitBytes;
    L.off_act = 0;
    L.act_m_stride = L.units * kActUnitStride;
    L.off_ring = (static_cast<uint32_t>(act_rows) * L.act_m_stride + 127u) & ~127u;
    L.ring_warp_stride = static_cast<uint32_t>(S) * L.slotbytes;
    L.off_bar = L.off_ring + static_cast<uint32_t>(warps) * L.ring_warp_stride;
    L.total = L.off_bar + static_cast<uint32_t>(warps * S) * 8u;
    return L;
}

// S - 8T of one block: qs (4 words of nibbles), its 8 activation words, and 8T.
// The high nibbles stay in place under a 0xF0 mask (bytes 0..240, exact), so their
// sum is 16x and is shifted once.
__device__ __forceinline__ int q4_block_dot(const uint32_t (&qs)[4], const uint4 &a0, const uint4 &a1, int t8)
{
    int lo = 0, hi = 0;
    lo = dp4a_us(qs[0] & 0x0f0f0f0fu, a0.x, lo);
    hi = dp4a_us(qs[0] & 0xf0f0f0f0u, a1.x, hi);
    lo = dp4a_us(qs[1] & 0x0f0f0f0fu, a0.y, lo);
    hi = dp4a_us(qs[1] & 0xf0f0f0f0u, a1.y, hi);
    lo = dp4a_us(qs[2] & 0x0f0f0f0fu, a0.z, lo);
    hi = dp4a_us(qs[2] & 0xf0f0f0f0u, a1.z, hi);
    lo = dp4a_us(qs[3] & 0x0f0f0f0fu, a0.w, lo);
    hi = dp4a_us(qs[3] & 0xf0f0f0f0u, a1.w, hi);
    return lo + (hi >> 4) - t8;
}

// Dot of one 8-block unit of a weight row against M staged activation rows.
// wu: the unit's 144 bytes in shared memory (16-byte aligned).
// act: the unit's activation record of row 0 (stride act_stride per row).
// dots: block dots of row 0 (stride dots_m_stride per row), kDots only.
template <int M, bool kDots>
__device__ __forceinline__ void q4_unit(const uint8_t *wu, const uint8_t *act, uint32_t act_stride, float (&acc)[M],
                                        int32_t *dots, int64_t dots_m_stride)
{
    const uint4 *wp = reinterpret_cast<const uint4 *>(wu);
    uint32_t w[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 v = wp[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    // block j starts at byte 18j: d4 in its first two bytes, qs in the next 16;
    // even blocks have their qs at 2 mod 4 and are realigned with byte permutes.
    float d4[8];
    uint32_t qs[8][4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        const int wa = (18 * j) / 4;           // word holding block j's first byte (aligned)
        d4[j] = f16_bits_to_float(w[wa] & 0xffffu);
        d4[j + 1] = f16_bits_to_float(w[wa + 4] >> 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            qs[j][i] = __byte_perm(w[wa + i], w[wa + i + 1], 0x5432);
            qs[j + 1][i] = w[wa + 5 + i];
        }
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint8_t *am = act + m * act_stride;
        const uint4 *a = reinterpret_cast<const uint4 *>(am);
        const float4 d8a = *reinterpret_cast<const float4 *>(am + kActD8Off);
        const float4 d8b = *reinterpret_cast<const float4 *>(am + kActD8Off + 16);
        const int4 t8a = *reinterpret_cast<const int4 *>(am + kActT8Off);
        const int4 t8b = *reinterpret_cast<const int4 *>(am + kActT8Off + 16);
        const float d8[8] = {d8a.x, d8a.y, d8a.z, d8a.w, d8b.x, d8b.y, d8b.z, d8b.w};
        const int t8[8] = {t8a.x, t8a.y, t8a.z, t8a.w, t8b.x, t8b.y, t8b.z, t8b.w};
        int sd[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) sd[j] = q4_block_dot(qs[j], a[2 * j], a[2 * j + 1], t8[j]);
        if (kDots) {
            int32_t *dm = dots + m * dots_m_stride;
#pragma unroll
            for (int j = 0; j < 8; ++j) dm[j] = sd[j];
        } else {
            float part = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) part = fmaf(d4[j] * d8[j], static_cast<float>(sd[j]), part);
            acc[m] += part;
        }
    }
}

// Dot of one Q4_K super-block (llama.cpp's K-quant layout, 144 bytes = 256
// weights, the same size as a Q4_0 unit) against M staged activation rows:
//   bytes 0..3 fp16 d and dmin; 4..15 eight packed 6-bit sub-block scales sc_j and
//   minimums mn_j; 16..143 nibbles, data byte 32c + e holding element e of
//   sub-block 2c (low nibble) and of sub-block 2c + 1 (high nibble).
//   sum_j d8_j (d sc_j S_j - dmin mn_j T_j),  S_j = sum q * q8, T_j = sum q8,
// with S_j, T_j exact integers and d sc_j, dmin mn_j exact in fp32.
// dots: the raw S_j (kDots only).
template <int M, bool kDots>
__device__ __forceinline__ void q4k_unit(const uint8_t *wu, const uint8_t *act, uint32_t act_stride, float (&acc)[M],
                                         int32_t *dots, int64_t dots_m_stride)
{
    const uint4 *wp = reinterpret_cast<const uint4 *>(wu);
    uint32_t w[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 v = wp[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    const float d = f16_bits_to_float(w[0] & 0xffffu), dmin = f16_bits_to_float(w[0] >> 16);
    // scale bytes p0..p3 = w[1], p4..p7 = w[2], p8..p11 = w[3]: sub-blocks 0..3 keep
    // their 6 bits in p0..3 (scales) and p4..7 (minimums); 4..7 their low 4 bits in
    // p8..11 (scale low, minimum high nibble) and their top 2 bits on top of p0..7.
    const uint32_t sc_lo = w[1] & 0x3f3f3f3fu, mn_lo = w[2] & 0x3f3f3f3fu;
    const uint32_t sc_hi = (w[3] & 0x0f0f0f0fu) | ((w[1] >> 2) & 0x30303030u);
    const uint32_t mn_hi = ((w[3] >> 4) & 0x0f0f0f0fu) | ((w[2] >> 2) & 0x30303030u);
    float dsc[8], dmn[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        dsc[j] = d * static_cast<float>((sc_lo >> (8 * j)) & 0xffu);
        dsc[j + 4] = d * static_cast<float>((sc_hi >> (8 * j)) & 0xffu);
        dmn[j] = dmin * static_cast<float>((mn_lo >> (8 * j)) & 0xffu);
        dmn[j + 4] = dmin * static_cast<float>((mn_hi >> (8 * j)) & 0xffu);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint8_t *am = act + m * act_stride;
        const uint4 *a = reinterpret_cast<const uint4 *>(am);
        const float4 d8a = *reinterpret_cast<const float4 *>(am + kActD8Off);
        const float4 d8b = *reinterpret_cast<const float4 *>(am + kActD8Off + 16);
        const int4 t8a = *reinterpret_cast<const int4 *>(am + kActT8Off);
        const int4 t8b = *reinterpret_cast<const int4 *>(am + kActT8Off + 16);
        const float d8[8] = {d8a.x, d8a.y, d8a.z, d8a.w, d8b.x, d8b.y, d8b.z, d8b.w};
        const int t8[8] = {t8a.x, t8a.y, t8a.z, t8a.w, t8b.x, t8b.y, t8b.z, t8b.w};
        int sd[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            // sub-blocks 2c (low nibbles) and 2c + 1 (high nibbles, summed 16x under a
            // 0xF0 mask) of data words 8c .. 8c + 7, against activation blocks 2c, 2c + 1
            const uint4 x0 = a[4 * c], x1 = a[4 * c + 1], x2 = a[4 * c + 2], x3 = a[4 * c + 3];
            const uint32_t lo_x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const uint32_t hi_x[8] = {x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
            int lo = 0, hi = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t q = w[4 + 8 * c + i];
                lo = dp4a_us(q & 0x0f0f0f0fu, lo_x[i], lo);
                hi = dp4a_us(q & 0xf0f0f0f0u, hi_x[i], hi);
            }
            sd[2 * c] = lo;
            sd[2 * c + 1] = hi >> 4;
        }
        if (kDots) {
            int32_t *dm = dots + m * dots_m_stride;
#pragma unroll
            for (int j = 0; j < 8; ++j) dm[j] = sd[j];
        } else {
            float part = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                part = fmaf(dsc[j] * d8[j], static_cast<float>(sd[j]), part);
                part = fmaf(-(dmn[j] * d8[j]), 0.125f * static_cast<float>(t8[j]), part);   // 8T / 8, exact
            }
            acc[m] += part;
        }
    }
}

// One activation row's record of one unit held in registers (M = 1, a lane that
// handles the same unit of every row it visits): q8 of the unit's 8 blocks, d8, 8 T.
struct ActRegs {
    uint4 q[16];
    float d8[8];
    int t8[8];
};

__device__ __forceinline__ void load_act_regs(const uint8_t *rec, ActRegs &r)
{
    const uint4 *a = reinterpret_cast<const uint4 *>(rec);
#pragma unroll
    for (int i = 0; i < 16; ++i) r.q[i] = a[i];
    const float4 d8a = *reinterpret_cast<const float4 *>(rec + kActD8Off);
    const float4 d8b = *reinterpret_cast<const float4 *>(rec + kActD8Off + 16);
    const int4 t8a = *reinterpret_cast<const int4 *>(rec + kActT8Off);
    const int4 t8b = *reinterpret_cast<const int4 *>(rec + kActT8Off + 16);
    r.d8[0] = d8a.x; r.d8[1] = d8a.y; r.d8[2] = d8a.z; r.d8[3] = d8a.w;
    r.d8[4] = d8b.x; r.d8[5] = d8b.y; r.d8[6] = d8b.z; r.d8[7] = d8b.w;
    r.t8[0] = t8a.x; r.t8[1] = t8a.y; r.t8[2] = t8a.z; r.t8[3] = t8a.w;
    r.t8[4] = t8b.x; r.t8[5] = t8b.y; r.t8[6] = t8b.z; r.t8[7] = t8b.w;
}

// q4_unit / q4k_unit for M = 1 against a register-resident activation record.
__device__ __forceinline__ float q4_unit_regs(const uint8_t *wu, const ActRegs &r)
{
    const uint4 *wp = reinterpret_cast<const uint4 *>(wu);
    uint32_t w[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 v = wp[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    float part = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        const int wa = (18 * j) / 4;
        uint32_t qa[4], qb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            qa[i] = __byte_perm(w[wa + i], w[wa + i + 1], 0x5432);
            qb[i] = w[wa + 5 + i];
        }
        const int sa = q4_block_dot(qa, r.q[2 * j], r.q[2 * j + 1], r.t8[j]);
        const int sb = q4_block_dot(qb, r.q[2 * j + 2], r.q[2 * j + 3], r.t8[j + 1]);
        part = fmaf(f16_bits_to_float(w[wa] & 0xffffu) * r.d8[j], static_cast<float>(sa), part);
        part = fmaf(f16_bits_to_float(w[wa + 4] >> 16) * r.d8[j + 1], static_cast<float>(sb), part);
    }
    return part;
}

// q4_unit for M = 2 against two register-resident activation records (the weight
// unit decoded once for both rows).
__device__ __forceinline__ void q4_unit_regs2(const uint8_t *wu, const ActRegs (&r)[2], float (&v)[2])
{
    const uint4 *wp = reinterpret_cast<const uint4 *>(wu);
    uint32_t w[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 x = wp[i];
        w[4 * i] = x.x;
        w[4 * i + 1] = x.y;
        w[4 * i + 2] = x.z;
        w[4 * i + 3] = x.w;
    }
    float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        const int wa = (18 * j) / 4;
        uint32_t qa[4], qb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            qa[i] = __byte_perm(w[wa + i], w[wa + i + 1], 0x5432);
            qb[i] = w[wa + 5 + i];
        }
        const float da = f16_bits_to_float(w[wa] & 0xffffu), db = f16_bits_to_float(w[wa + 4] >> 16);
        const int a0 = q4_block_dot(qa, r[0].q[2 * j], r[0].q[2 * j + 1], r[0].t8[j]);
        const int b0 = q4_block_dot(qb, r[0].q[2 * j + 2], r[0].q[2 * j + 3], r[0].t8[j + 1]);
        const int a1 = q4_block_dot(qa, r[1].q[2 * j], r[1].q[2 * j + 1], r[1].t8[j]);
        const int b1 = q4_block_dot(qb, r[1].q[2 * j + 2], r[1].q[2 * j + 3], r[1].t8[j + 1]);
        p0 = fmaf(da * r[0].d8[j], static_cast<float>(a0), p0);
        p0 = fmaf(db * r[0].d8[j + 1], static_cast<float>(b0), p0);
        p1 = fmaf(da * r[1].d8[j], static_cast<float>(a1), p1);
        p1 = fmaf(db * r[1].d8[j + 1], static_cast<float>(b1), p1);
    }
    v[0] = p0;
    v[1] = p1;
}

__device__ __forceinline__ float q4k_unit_regs(const uint8_t *wu, const ActRegs &r)
{
    const uint4 *wp = reinterpret_cast<const uint4 *>(wu);
    uint32_t w[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 v = wp[i];
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    const float d = f16_bits_to_float(w[0] & 0xffffu), dmin = f16_bits_to_float(w[0] >> 16);
    const uint32_t sc[2] = {w[1] & 0x3f3f3f3fu, (w[3] & 0x0f0f0f0fu) | ((w[1] >> 2) & 0x30303030u)};
    const uint32_t mn[2] = {w[2] & 0x3f3f3f3fu, ((w[3] >> 4) & 0x0f0f0f0fu) | ((w[2] >> 2) & 0x30303030u)};
    float part = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 x0 = r.q[4 * c], x1 = r.q[4 * c + 1], x2 = r.q[4 * c + 2], x3 = r.q[4 * c + 3];
        const uint32_t lo_x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const uint32_t hi_x[8] = {x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
        int lo = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t qw = w[4 + 8 * c + i];
            lo = dp4a_us(qw & 0x0f0f0f0fu, lo_x[i], lo);
            hi = dp4a_us(qw & 0xf0f0f0f0u, hi_x[i], hi);
        }
        const int sd[2] = {lo, hi >> 4};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = 2 * c + h;
            const float dsc = d * static_cast<float>((sc[j >> 2] >> (8 * (j & 3))) & 0xffu);
            const float dmn = dmin * static_cast<float>((mn[j >> 2] >> (8 * (j & 3))) & 0xffu);
            part = fmaf(dsc * r.d8[j], static_cast<float>(sd[h]), part);
            part = fmaf(-(dmn * r.d8[j]), 0.125f * static_cast<float>(r.t8[j]), part);
        }
    }
    return part;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Division by a kernel-wide divisor 0 < n: q = umulhi(u, ceil(2^32 / n)) equals
// u / n whenever u * n < 2^32 (the error u * (ceil - 2^32/n) / 2^32 stays below
// the distance 1/n from u/n to the next integer); the staging indices are bounded
// by the shared-memory size, far inside that range.
__device__ __forceinline__ uint32_t div_magic(int n) { return 0xffffffffu / static_cast<uint32_t>(n) + 1u; }
__device__ __forceinline__ int div_by(int u, uint32_t magic)
{
    return static_cast<int>(__umulhi(static_cast<uint32_t>(u), magic));
}

// Shared-memory record of the unit holding block b of activation row gm (= matrix * M + m).
__device__ __forceinline__ uint8_t *act_block(uint8_t *smem, const Q4Layout &L, int gm, int b)
{
    return smem + L.off_act + gm * L.act_m_stride + (b >> 3) * kActUnitStride;
}

// Quantize the group's fp32 activations to Q8_1 straight into the shared-memory
// staging layout, a quad of lanes per 32-value block (the quantizer's own code).
template <int M, typename AfterLoads>
__device__ __forceinline__ void stage_fused(const Q4Group &grp, int nb, uint8_t *smem, const Q4Layout &L,
                                            int nthreads, AfterLoads after_loads)
{
    constexpr int kPasses = 4;   // loads of up to 4 passes are issued before any is used
    const int part = threadIdx.x & 3;
    const int total = grp.nx * M * nb;   // blocks over (activation, row m, block b)
    const int quads = nthreads >> 2;
    const uint32_t inv_nb = div_magic(nb);
    for (int base = 0; base < total; base += kPasses * quads) {   // uniform trip count: whole warps shuffle
        float v[kPasses][8];
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
            const int u = base + ps * quads + static_cast<int>(threadIdx.x >> 2);
            const int uc = u < total ? u : 0;
            const int gm = div_by(uc, inv_nb), b = uc - gm * nb;
            const int gi = gm / M, m = gm - gi * M;
            const float *src = static_cast<const float *>(grp.x[gi]) + static_cast<int64_t>(m) * (nb * 32) + b * 32 +
                               8 * part;
            if (base + ps * quads < total) {
                const float4 a = __ldg(reinterpret_cast<const float4 *>(src));
                const float4 c = __ldg(reinterpret_cast<const float4 *>(src) + 1);
                v[ps][0] = a.x; v[ps][1] = a.y; v[ps][2] = a.z; v[ps][3] = a.w;
                v[ps][4] = c.x; v[ps][5] = c.y; v[ps][6] = c.z; v[ps][7] = c.w;
            }
        }
        if (base == 0) after_loads();
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
            if (base + ps * quads >= total) break;   // uniform over the CTA
            const int u = base + ps * quads + static_cast<int>(threadIdx.x >> 2);
            const Q8Quad r = q8_1_quantize_quad(v[ps]);
            if (u < total) {
                const int gm = div_by(u, inv_nb), b = u - gm * nb;
                uint8_t *rec = act_block(smem, L, gm, b);
                const int j = b & 7;
                *reinterpret_cast<uint2 *>(rec + 32 * j + 8 * part) = make_uint2(r.qlo, r.qhi);
                if (part == 0) {
                    reinterpret_cast<float *>(rec + kActD8Off)[j] = f16_bits_to_float(q8_1_d8_bits(r));
                    reinterpret_cast<int *>(rec + kActT8Off)[j] = 8 * r.sum;
                }
            }
        }
    }
}

// Copy the group's Q8_1 activations into the staging layout, adding 8 * sum(q) per block.
template <int M, typename AfterLoads>
__device__ __forceinline__ void stage_q8_1(const Q4Group &grp, int nb, uint8_t *smem, const Q4Layout &L,
                                           int nthreads, AfterLoads after_loads)
{
    const int total = grp.nx * M * nb;
    const uint32_t inv_nb = div_magic(nb);
    after_loads();
    for (int u = threadIdx.x; u < total; u += nthreads) {
        const int gm = div_by(u, inv_nb), b = u - gm * nb;
        const int gi = gm / M, m = gm - gi * M;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(grp.x[gi]) +
                                                                 (static_cast<int64_t>(m) * nb + b) * 36);
        uint32_t q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = __ldg(src + 1 + j);
        int t = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) t = __dp4a(static_cast<int>(q[j]), 0x01010101, t);
        uint8_t *rec = act_block(smem, L, gm, b);
        const int j = b & 7;
        reinterpret_cast<float *>(rec + kActD8Off)[j] = f16_bits_to_float(__ldg(src) & 0xffffu);
        reinterpret_cast<int *>(rec + kActT8Off)[j] = 8 * t;
        uint4 *dst = reinterpret_cast<uint4 *>(rec + 32 * j);
        dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
        dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
    }
}

// kFused: the group's activations are fp32 [M][K], quantized to Q8_1 in the
// prologue; else they are Q8_1 [M][K/32]. kDots: write the integer block dots of
// matrix 0 instead of y (a single-matrix group). kQ4K: the weights are Q4_K
// super-blocks (a row is K/256 of 144 bytes, the same units as Q4_0).
// kActRegs (M = 1, or Q4_0 at M = 2; rows of U units with 32 % U == 0): a lane
// handles unit lane % U of every row it visits, so its activation records are loaded
// into registers once instead of read from shared memory for every unit.
// kPair (Q4_0, M = 2..4, rows of 16 units): in a chunk of two whole rows, lanes l and
// l + 16 hold the same unit of the two rows; each computes both rows' unit against
// half of the M activation rows and they swap halves with one shuffle per output
// pair, so a lane reads ceil(M / 2) activation records from shared memory, not M.
template <int M, bool kDots, bool kFused, bool kQ4K, bool kActRegs = false, bool kPair = false>
__global__ void __launch_bounds__(kActRegs ? (M == 1 ? kActRegsThreads : kStreamThreadsWide) : stream_threads(M))
    q4_0_stream_kernel(
    const __grid_constant__ Q4Group grp, int32_t *__restrict__ dots, int64_t K, int S, int P QMV_TRACE_PARAM)
{
#ifdef QMV_STAGE_TRACE
    uint64_t t_start = globaltimer_ns(), t_rel = 0, t_sync = 0, t_first = 0;
#endif
    extern __shared__ __align__(128) uint8_t smem[];
    const int warps = blockDim.x >> 5;
    const Q4Layout L = q4_layout(M * grp.nx, K, warps, S);
    const int nb = static_cast<int>(K >> 5);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int U = static_cast<int>(L.units);
    uint8_t *ring = smem + L.off_ring + warp * L.ring_warp_stride;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.off_bar) + warp * S;

    // This warp's span: rows [r0, r1) of matrix mi (warps are split over the
    // matrices in proportion to their rows, then rows evenly over the warps).
    const int gw = blockIdx.x * warps + warp;
    int mi = 0;
#pragma unroll
    for (int i = 1; i < kMaxGroup; ++i)
        if (i < grp.count && gw >= grp.cta_start[i]) mi = i;
    const int64_t Nm = grp.row_start[mi + 1] - grp.row_start[mi];
    const int64_t wm = grp.cta_start[mi + 1] - grp.cta_start[mi];
    const int64_t j = gw - grp.cta_start[mi];
    const int64_t r0 = j < wm ? j * Nm / wm : Nm, r1 = j < wm ? (j + 1) * Nm / wm : Nm;
    const int TU = static_cast<int>((r1 - r0) * U);   // units in the span (< 2^31: checked by the host)
    const int nchunks = (TU + kChunkUnits - 1) / kChunkUnits;
    const uint8_t *span = grp.w[mi] + r0 * L.rowbytes;
    const uint64_t pol = policy_evict_first();
    const int pw = min(S, (P + warps - 1 - warp) / warps);   // this warp's share of the P early chunks

    auto issue = [&](int c, int slot) {   // chunk c into a free slot
        const uint32_t bytes = static_cast<uint32_t>(min(kChunkUnits, TU - c * kChunkUnits)) * kUnitBytes;
        mbar_arrive_expect_tx(&bars[slot], bytes);
        bulk_copy_g2s(ring + slot * L.slotbytes, span + static_cast<int64_t>(c) * (kChunkUnits * kUnitBytes), bytes,
                      &bars[slot], pol);
    };
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
        // weights do not depend on the preceding kernel: the CTA's first P chunks
        // (spread over its warps) are requested now
        for (int c = 0; c < pw && c < nchunks; ++c) issue(c, c);
    }
    __syncwarp();
    grid_launch_dependents();
    grid_dependency_wait();
    QMV_TRACE_STAMP(t_rel);

    // the rest of the ring is requested once the activation loads are in flight,
    // so that they do not queue behind a full ring of weight copies
    auto fill_ring = [&]() {
        if (lane == 0)
            for (int c = pw; c < S && c < nchunks; ++c) issue(c, c);
    };
    if (kFused)
        stage_fused<M>(grp, nb, smem, L, blockDim.x, fill_ring);
    else
        stage_q8_1<M>(grp, nb, smem, L, blockDim.x, fill_ring);
    __syncthreads();   // the only CTA-wide barrier
    QMV_TRACE_STAMP(t_sync);

    const uint8_t *act0 = smem + L.off_act + (grp.xslot[mi] * M) * L.act_m_stride;
    float *ym = grp.y[mi] + r0;
    // This lane's unit in the chunk: row rr of the span, unit uin of the row. Chunk
    // c + 1 starts 32 units later, i.e. dr rows and du units further on.
    int rr = lane / U, uin = lane - rr * U;
    const int dr = kChunkUnits / U, du = kChunkUnits - dr * U;
    float carry[M];   // partial sum of the row left open by the previous chunk
#pragma unroll
    for (int m = 0; m < M; ++m) carry[m] = 0.0f;
    // register-resident records: rows 0 .. kRegRows-1 (M = 3: rows 0, 1; row 2 from shared memory)
    constexpr int kRegRows = kActRegs ? (M < 3 ? M : 2) : 1;
    ActRegs ar[kRegRows];
    if (kActRegs) {   // uin never changes (du == 0)
#pragma unroll
        for (int m = 0; m < kRegRows; ++m) load_act_regs(act0 + m * L.act_m_stride + uin * kActUnitStride, ar[m]);
    }
    int slot = 0;
    uint32_t phase = 0;
    for (int c = 0; c < nchunks; ++c) {
        if (!mbar_wait_bounded(&bars[slot], phase)) {
            // chunks c .. c + S - 1 are in flight; no CTA-wide barrier follows the
            // prologue in this kernel, so the warp may leave once they have landed
            if (lane == 0) {
                note_wait_timeout(&g_q4_error, nullptr);
                drain_ring(bars, S, slot, phase, min(S, nchunks - c));
            }
            return;
        }
#ifdef QMV_STAGE_TRACE
        if (c == 0) t_first = globaltimer_ns();
#endif
        const bool live = c * kChunkUnits + lane < TU;
        float v[M];
#pragma unroll
        for (int m = 0; m < M; ++m) v[m] = 0.0f;
        // (kPair) a chunk of 32 live units: two whole rows
        const bool paired = kPair && c * kChunkUnits + kChunkUnits <= TU;
        if (paired) {
            constexpr int MA = (M + 1) / 2, MB = M - MA;
            const int h = lane >> 4;
            const uint8_t *w0 = ring + slot * L.slotbytes + (lane & 15) * kUnitBytes;   // the chunk's first row
            const uint8_t *w1 = w0 + 16 * kUnitBytes;                                   // its second row
            const uint8_t *ab = act0 + (h ? MA : 0) * L.act_m_stride + uin * kActUnitStride;
            // half 1 holds MB <= MA rows: its missing row re-reads its last one (discarded)
            const uint32_t ast = (h && MB < MA) ? 0u : L.act_m_stride;
            float p0[MA], p1[MA];
#pragma unroll
            for (int k = 0; k < MA; ++k) p0[k] = p1[k] = 0.0f;
            q4_unit<MA, false>(w0, ab, ast, p0, nullptr, 0);
            q4_unit<MA, false>(w1, ab, ast, p1, nullptr, 0);
            // half 0 keeps the first row's activation rows 0..MA-1 and receives MA..M-1;
            // half 1 keeps the second row's MA..M-1 and receives 0..MA-1
#pragma unroll
            for (int k = 0; k < MA; ++k) {
                const float got = __shfl_xor_sync(0xffffffffu, h ? p0[k] : p1[k], 16);
                if (h) {
                    v[k] = got;
                    if (k < MB) v[MA + k] = p1[k];
                } else {
                    v[k] = p0[k];
                    if (k < MB) v[MA + k] = got;
                }
            }
        } else if (live) {
            const uint8_t *wu = ring + slot * L.slotbytes + lane * kUnitBytes;
            int32_t *du = kDots ? dots + (r0 + rr) * nb + 8 * uin : nullptr;
            if constexpr (kActRegs && M == 3) {
                float v2[2];
                q4_unit_regs2(wu, ar, v2);
                v[0] = v2[0];
                v[1] = v2[1];
                float v3[1] = {0.0f};
                q4_unit<1, false>(wu, act0 + 2 * L.act_m_stride + uin * kActUnitStride, 0u, v3, nullptr, 0);
                v[2] = v3[0];
            } else if constexpr (kActRegs && M == 2)
                q4_unit_regs2(wu, ar, v);
            else if (kActRegs)
                v[0] = kQ4K ? q4k_unit_regs(wu, ar[0]) : q4_unit_regs(wu, ar[0]);
            else if (kQ4K)
                q4k_unit<M, kDots>(wu, act0 + uin * kActUnitStride, L.act_m_stride, v, du, Nm * nb);
            else
                q4_unit<M, kDots>(wu, act0 + uin * kActUnitStride, L.act_m_stride, v, du, Nm * nb);
        }
        __syncwarp();   // every lane is done with the slot
        if (lane == 0 && c + S < nchunks) {
            fence_proxy_async_shared();   // the warp's reads of the slot before the copy's writes
            issue(c + S, slot);
        }
        if (!kDots) {
            // Inclusive scan within the row: the lanes of one row are consecutive,
            // min(uin, lane) of them precede this lane in the chunk.
            const int before = min(uin, lane);
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const float o = __shfl_up_sync(0xffffffffu, v[m], d);
                    if (d <= before) v[m] += o;
                }
            }
            const bool row_end = live && uin == U - 1;
            // the row that began in an earlier chunk is closed (or carried on) by its last lane here
            if (live && (row_end || lane == 31) && uin >= lane) {
#pragma unroll
                for (int m = 0; m < M; ++m) v[m] += carry[m];
            }
            if (row_end) {
#pragma unroll
                for (int m = 0; m < M; ++m) ym[m * Nm + rr] = v[m];
            }
            const bool open = (__ballot_sync(0xffffffffu, row_end) >> 31) == 0;   // lane 31's row continues
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const float t = __shfl_sync(0xffffffffu, v[m], 31);
                carry[m] = open ? t : 0.0f;
            }
        }
        uin += du;
        rr += dr;
        if (uin >= U) {
            uin -= U;
            ++rr;
        }
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
    }
#ifdef QMV_STAGE_TRACE
    if (trace && lane == 0 && warp < kTraceWarps) {
        unsigned long long *tw = trace + (static_cast<size_t>(blockIdx.x) * kTraceWarps + warp) * kTraceFields;
        uint32_t sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        tw[0] = t_start; tw[1] = t_rel; tw[2] = t_sync; tw[3] = t_first; tw[4] = globaltimer_ns();
        tw[5] = sm; tw[6] = static_cast<unsigned long long>(nchunks); tw[7] = 1;
    }
#endif
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

#ifdef QMV_STAGE_TRACE
unsigned long long *g_trace_buf = nullptr;
int g_trace_records = 0, g_trace_next = 0, g_trace_ctas = 0;

// The record of the next streaming launch (records are used in launch order, cyclically).
unsigned long long *next_trace_record(int grid)
{
    if (!g_trace_buf || g_trace_records == 0 || grid > g_trace_ctas) return nullptr;
    const int r = g_trace_next++ % g_trace_records;
    return g_trace_buf + static_cast<size_t>(r) * g_trace_ctas * kTraceWarps * kTraceFields;
}
#endif

template <int M, bool kDots, bool kFused, bool kQ4K>
cudaError_t launch_m(const Q4Plan &p, const Q4Group &grp, int32_t *dots, int64_t K, cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    cfg.attrs = attr;
    cfg.numAttrs = set_launch_overlap_attr(attr);
    if (p.route == kRouteQ4_0Stream) {
        auto kern = q4_0_stream_kernel<M, kDots, kFused, kQ4K>;
        if constexpr ((M == 1 || ((M == 2 || M == 3) && !kQ4K)) && !kDots)
            if (p.act_regs) kern = q4_0_stream_kernel<M, kDots, kFused, kQ4K, true>;
        if constexpr (M >= 2 && M <= 4 && !kQ4K && !kDots)
            if (p.pair) kern = q4_0_stream_kernel<M, kDots, kFused, kQ4K, false, true>;
        cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), p.smem_bytes);
        if (e != cudaSuccess) return e;
        cfg.blockDim = dim3(static_cast<unsigned>(p.warps * 32));   // consumers + the producer
        cfg.dynamicSmemBytes = static_cast<size_t>(p.smem_bytes);
#ifdef QMV_STAGE_TRACE
        return cudaLaunchKernelEx(&cfg, kern, grp, dots, K, p.stages, p.prefetch, next_trace_record(p.grid));
#else
        return cudaLaunchKernelEx(&cfg, kern, grp, dots, K, p.stages, p.prefetch);
#endif
    }
    if (kQ4K || kFused || grp.count != 1) return cudaErrorInvalidValue;   // these need the streaming kernel
    cfg.blockDim = dim3(kThreads);
    auto gk = q4_0_generic_kernel<M, kDots>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(gk), 0);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, gk, grp.w[0], static_cast<const uint8_t *>(grp.x[0]), grp.y[0], dots,
                              grp.row_start[1], K);
}

template <bool kDots, bool kFused, bool kQ4K>
cudaError_t launch_dispatch(const Q4Plan &p, const Q4Group &grp, int32_t *dots, int M, int64_t K, cudaStream_t s)
{
    switch (M) {
    case 1: return launch_m<1, kDots, kFused, kQ4K>(p, grp, dots, K, s);
    case 2: return launch_m<2, kDots, kFused, kQ4K>(p, grp, dots, K, s);
    case 3: return launch_m<3, kDots, kFused, kQ4K>(p, grp, dots, K, s);
    case 4: return launch_m<4, kDots, kFused, kQ4K>(p, grp, dots, K, s);
    case 5: return launch_m<5, kDots, kFused, kQ4K>(p, grp, dots, K, s);
    case 6: return launch_m<6, kDots, kFused, kQ4K>(p, grp, dots, K, s);
    case 7: return launch_m<7, kDots, kFused, kQ4K>(p, grp, dots, K, s);
    case 8: return launch_m<8, kDots, kFused, kQ4K>(p, grp, dots, K, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t plan_q4_0(const DeviceInfo &dev, const Q4Group &grp, int M, int64_t K, Q4Plan *plan, bool q4k)
{
    bool aligned = true;
    for (int i = 0; i < grp.count; ++i) aligned = aligned && (reinterpret_cast<uintptr_t>(grp.w[i]) & 15u) == 0;
    const int64_t N = grp.row_start[grp.count];
    plan->route = kRouteQ4_0Generic;
    plan->warps = kWarps;
    plan->stages = 0;
    plan->prefetch = 0;
    plan->round = 0;
    plan->smem_bytes = 0;
    plan->act_regs = false;
    plan->pair = false;
    plan->grid = static_cast<int>((N + kWarps - 1) / kWarps);
    if (!aligned || K % 256 != 0) return cudaSuccess;
    // from a few activation rows on, the tensor cores
    if (M >= env_int(q4k ? "QMV_Q4K_MMA_MIN_M" : "QMV_Q4_MMA_MIN_M", 5)) {
        cudaError_t e = plan_q4_0_mma(dev, grp, M, K, plan, q4k);
        if (e != cudaSuccess || plan->route == kRouteQ4_0Mma) return e;
    }

    // Warps hide latency (each also issues its own copies); slots are the bytes in flight.
    const int act_rows = M * grp.nx;
    const int cap = stream_threads(M) / 32;
    int warps = std::max(1, std::min(cap, env_int("QMV_Q4_WARPS", cap)));
    int S = std::max(1, std::min(8, env_int("QMV_Q4_SLOTS", 2)));
    const int budget = env_int("QMV_Q4_PAIR_SMEM", 0) ? dev.smem_per_sm / 2 - 2048 : dev.smem_optin;
    while (warps > 1 && q4_layout(act_rows, K, warps, S).total > static_cast<uint32_t>(budget)) --warps;
    if (q4_layout(act_rows, K, warps, S).total > static_cast<uint32_t>(dev.smem_optin)) return cudaSuccess;
    // M = 1 with rows of U units, U dividing 32 (K = 4096: U = 16): every lane keeps
    // one unit of every row it visits, so its activation record lives in registers
    // (119 of them: 16 warps still fit) and the 20 shared-memory reads of the record
    // per 144-byte unit are gone (Llama-2-7B stack 3839 -> 3972 GB/s)
    bool act_regs = false;
    const int U = static_cast<int>(K / 256);
    // M = 2 (Q4_0): two records, 215 registers, 8 warps with 4-slot rings (Llama-3-8B
    // MLP 3218 -> 3264 GB/s). M = 3 (Q4_0): rows 0 and 1 in registers, row 2 read from
    // shared memory, 231 registers (Llama-3-8B MLP 2556 -> 2840 GB/s)
    const bool m2 = (M == 2 && !q4k && env_int("QMV_Q4_ACT_REGS_M2", 1) != 0) ||
                    (M == 3 && !q4k && env_int("QMV_Q4_ACT_REGS_M3", 1) != 0);
    if ((M == 1 || m2) && U <= 32 && 32 % U == 0 && env_int("QMV_Q4_ACT_REGS", 1) != 0) {
        const int wcap = M == 1 ? kActRegsThreads / 32 : kStreamThreadsWide / 32;
        int w2 = std::min(warps, std::max(1, std::min(wcap, env_int("QMV_Q4_ACT_REGS_WARPS", 16))));
        const int S2 = std::max(1, std::min(8, env_int("QMV_Q4_ACT_REGS_SLOTS", M == 1 ? S : 4)));
        while (w2 > 1 && q4_layout(act_rows, K, w2, S2).total > static_cast<uint32_t>(dev.smem_optin)) --w2;
        if (q4_layout(act_rows, K, w2, S2).total <= static_cast<uint32_t>(dev.smem_optin)) {
            act_regs = true;
            warps = w2;
            S = S2;
        }
    }
    // Q4_0 at M = 4 with rows of 16 units (K = 4096): lane pairs share activation
    // records, half the shared-memory reads of them (Llama-3-8B MLP 2116 -> 2401 GB/s).
    // At M = 3 the odd split adds a third more dot work and gains nothing; at M = 2 the
    // records fit in registers. QMV_Q4_PAIR=1 forces it at M = 2..3, 0 disables it.
    const int pair_env = env_int("QMV_Q4_PAIR", -1);
    const bool pair = !act_regs && !q4k && M >= 2 && M <= 4 && U == 16 &&
                      (pair_env < 0 ? M == 4 : pair_env != 0);
    // Spare SMs: the grid leaves about one SM in twelve without a CTA. In a chain of
    // calls with launch overlap the next call's CTAs take the SMs in the order they
    // free up, and its last CTA lands on the SM that finished the previous call last;
    // that CTA then starts after the others' early weight copies have landed, finishes
    // last, and hands the lateness on to the next call (globaltimer traces of the
    // Llama-2-7B stack: one CTA about 1 us behind the rest in every stage). With spare
    // SMs the previous call's stragglers get no CTA of the next call. Llama-2-7B stack:
    // 3935 GB/s with no spare SM, 4086 with 1, 4149 with 4, 4245 with 12, 4195 with 16,
    // 3894 with 32.
    const int per_sm = std::max(1, std::min(4, env_int("QMV_Q4_CTAS_PER_SM", 1)));
    const int spare = std::max(0, std::min(dev.sm_count - 1, env_int("QMV_Q4_SPARE_SMS", dev.sm_count / 12)));
    const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>((N + warps - 1) / warps,
                                                                 static_cast<int64_t>(dev.sm_count - spare) * per_sm));
    if ((N / (ctas * warps) + 1) * (K / 256) >= (int64_t(1) << 31)) return cudaSuccess;   // 32-bit unit counters
    plan->route = kRouteQ4_0Stream;
    plan->act_regs = act_regs;
    plan->pair = pair;
    plan->warps = warps;
    plan->stages = S;
    plan->prefetch = std::max(0, std::min(S * warps, env_int("QMV_Q4_PREFETCH", 4)));
    plan->chunk_units = kChunkUnits;
    plan->smem_bytes = static_cast<int>(q4_layout(act_rows, K, warps, S).total);
    plan->grid = static_cast<int>(ctas);
    return cudaSuccess;
}

// Split the grid's warps over the group's matrices in proportion to their rows
// (at least one warp per non-empty matrix when there are enough warps).
void assign_ctas(Q4Group &grp, int total)
{
    const int64_t N = grp.row_start[grp.count];
    int64_t acc = 0;
    grp.cta_start[0] = 0;
    for (int i = 0; i < grp.count; ++i) {
        const int64_t n = grp.row_start[i + 1] - grp.row_start[i];
        acc += n;
        int64_t end = (acc * total + N - 1) / N;   // ceil share of the CTAs so far
        const int64_t lo = grp.cta_start[i] + (n > 0 ? 1 : 0);
        const int64_t hi = total - (grp.count - 1 - i);
        end = std::max(lo, std::min(end, hi));
        if (i == grp.count - 1) end = total;
        grp.cta_start[i + 1] = static_cast<int>(end);
    }
    for (int i = grp.count + 1; i <= kMaxGroup; ++i) grp.cta_start[i] = total;
}

cudaError_t launch_q4_0(const Q4Plan &plan, const Q4Group &grp_in, int32_t *dots, int M, int64_t K, bool fused,
                        cudaStream_t s, bool q4k)
{
    if (plan.route == kRouteQ4_0Mma) return launch_q4_0_mma(plan, grp_in, dots, M, K, fused, s, q4k);
    if (fused && plan.route != kRouteQ4_0Stream) return cudaErrorInvalidValue;
    Q4Group grp = grp_in;
    if (plan.route == kRouteQ4_0Stream) assign_ctas(grp, plan.grid * plan.warps);   // per warp
    if (q4k) {
        if (plan.route != kRouteQ4_0Stream) return cudaErrorInvalidValue;   // Q4_K: the streaming kernels only
        route_hit(fused ? kRouteQ4KStreamFused : kRouteQ4KStream);
        if (dots) return launch_dispatch<true, false, true>(plan, grp, dots, M, K, s);
        if (fused) return launch_dispatch<false, true, true>(plan, grp, dots, M, K, s);
        return launch_dispatch<false, false, true>(plan, grp, dots, M, K, s);
    }
    route_hit(fused ? kRouteQ4_0StreamFused : plan.route);
    if (dots) return launch_dispatch<true, false, false>(plan, grp, dots, M, K, s);
    if (fused) return launch_dispatch<false, true, false>(plan, grp, dots, M, K, s);
    return launch_dispatch<false, false, false>(plan, grp, dots, M, K, s);
}

#ifdef QMV_STAGE_TRACE
// Profiling builds: records[r][cta < ctas][warp < 16][8] of the streaming kernel's launches, in
// launch order from the next launch on (NULL stops tracing). Not part of the product library.
extern "C" __attribute__((visibility("default"))) void qmv_stage_trace_set(unsigned long long *records, int count,
                                                                          int ctas)
{
    g_trace_buf = records;
    g_trace_records = records ? count : 0;
    g_trace_ctas = ctas;
    g_trace_next = 0;
}
#endif

cudaError_t read_error_word_q4_0(uint32_t *out, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_q4_error, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_q4_error, &zero, sizeof(uint32_t));
}

}  // namespace qmv
