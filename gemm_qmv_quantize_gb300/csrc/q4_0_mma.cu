// q4_0_mma.cu -- Q4_0 x Q8_1 (MMVQ) on the tensor cores, for M = 5..8 activation rows.
//
// The block dot of "Machine Learning on NVIDIA CMP" (sections "TL;DR" and "The DP2A
// patch") is an integer dot of 32 nibbles against 32 int8 activations, scaled once
// per block by d4 * d8. At M rows the CUDA-core path spends M times its dp4a work
// per weight byte and falls well short of the HBM stream from M = 5 on; here one
// mma.sync.m16n8k32 (s8 x s8 -> s32) takes 16 weight rows x one 32-weight block x
// 8 activation rows at once:
//  * A (16 x 32, weights): lane (g, t) needs k = 4t..4t+3 and 16+4t..16+4t+3 of rows
//    g and g+8, which are exactly the low and the high nibbles of qs word t of the
//    block. Each nibble becomes the byte 16 (q - 8) = ((q ^ 8) << 4) as int8, so the
//    product is 16 (S - 8 T) with S = sum q4 q8, T = sum q8: the offset-8 identity
//    of the format, exact in int32, with no separate sum of the activations.
//  * B (32 x 8, activations): the Q8_1 bytes of the M rows (rows M..7 are zero).
//  * Per block: y += (d4 * d8 / 16) * D in fp32 (d4 * d8 is exact in fp32).
// (An f16 m16n8k16 form on the exact integers q - 8 and q8 is as exact and spares
// the int8 tensor rate, but its operand decode costs more instructions than the
// int8 pipe costs time: measured slower.)
// Streaming: a 2-D tensor copy (TMA) of 16 rows x 144 bytes (8 blocks of each row)
// per warp step into a per-warp ring of shared-memory slots; the 144-byte row pitch
// in shared memory puts the 8 rows of a fragment read in distinct banks. The CTA
// walks its 16-row tiles in rounds of B tiles, its 8 warps taking interleaved steps
// (B a multiple of 8 / gcd(steps per tile, 8), so every warp gets the same number,
// and at least 8 steps per warp), then reduces the round in shared memory.
// Activations are staged once per CTA (quantized from fp32 in the prologue, or
// copied from Q8_1) in a layout whose fragment reads are 64-bit and conflict free.
#include <algorithm>

#include <cuda.h>

#include "q8_1_block.cuh"
#include "qmv_device.cuh"
#include "qmv_internal.h"

namespace qmv {
namespace {

__device__ uint32_t g_q4m_error;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 16;                       // weight rows per mma
constexpr int kUnitBytes = 144;                 // 8 blocks of one row
constexpr int kBox = kTile * kUnitBytes;        // 2304 bytes: one warp step
constexpr int kMaxRound = 8;
constexpr int kRedPitch = 9;                    // floats per partial row (8 columns + pad)
// Staged activations, per (distinct input, block): the q8 bytes of the M rows,
// 32 bytes each with the words in the order 0 4 1 5 2 6 3 7 (lane t's words t and
// 4 + t adjacent), then the scale of rows 0..7 as fp32 (zero from row M on): d8 / 16
// for Q4_0, d8 for Q4_K, which also stores d8 * T of rows 0..7 (T = sum q8).
__host__ __device__ inline int act_block_bytes(int M, bool q4k) { return 32 * M + (q4k ? 64 : 32); }

struct MmaParams {
    CUtensorMap tm[kMaxGroup];     // weights of matrix i: [N_i][K / 32 * 18] bytes, box 144 x 16
    int count, nx, M, S, B;
    int xslot[kMaxGroup];
    int tile_start[kMaxGroup + 1];  // tiles of matrix i: [tile_start[i], tile_start[i + 1])
    int64_t N[kMaxGroup];
    const void *x[kMaxGroup];
    float *y[kMaxGroup];
    int32_t *dots;                  // block dots of matrix 0 instead of y (a single matrix)
};

struct MmaLayout {
    uint32_t off_bar, off_abort, off_act, off_red, total;
};

// Shared memory: per-warp rings of boxes, their mbarriers, the CTA's abort word, the
// staged activations, the round's partial sums [warp][B * 16 rows][9].
__host__ __device__ inline MmaLayout mma_layout(int S, int B, int nx, int nb, int M, bool q4k)
{
    MmaLayout L;
    L.off_bar = static_cast<uint32_t>(kWarps * S * kBox);
    L.off_abort = L.off_bar + static_cast<uint32_t>(kWarps * S) * 8u;
    L.off_act = (L.off_abort + 4u + 15u) & ~15u;
    L.off_red = L.off_act + static_cast<uint32_t>(nx) * static_cast<uint32_t>(nb) * act_block_bytes(M, q4k);
    L.total = L.off_red + static_cast<uint32_t>(kWarps * B * kTile * kRedPitch) * 4u;
    return L;
}

// Position of q8 word w (bytes 4w..4w+3) in a staged row: 0 4 1 5 2 6 3 7.
__device__ __forceinline__ int act_word_pos(int w) { return 2 * (w & 3) + (w >> 2); }

// Stage the activations: fused, quantize fp32 [M][K] to Q8_1 with a quad of lanes per
// block (loads of four passes in flight before any is used); else copy Q8_1
// [M][K/32]. Rows M..7 of every record are zero.
template <bool kFused, bool kQ4K>
__device__ __forceinline__ void stage_act(const MmaParams &p, int nb, uint8_t *act)
{
    const int M = p.M, rb = act_block_bytes(M, kQ4K);
    const float dscale = kQ4K ? 1.0f : 0.0625f;   // Q4_0's product is 16 (S - 8 T)
    const int total = p.nx * M * nb;   // (input, row < M, block)
    if (kFused) {
        constexpr int kPasses = 4;
        constexpr int kQuads = kThreads / 4;
        const int part = threadIdx.x & 3;
        for (int base = 0; base < total; base += kPasses * kQuads) {   // uniform: whole warps shuffle
            float v[kPasses][8];
#pragma unroll
            for (int ps = 0; ps < kPasses; ++ps) {
                const int u = base + ps * kQuads + static_cast<int>(threadIdx.x >> 2);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[ps][i] = 0.0f;
                if (u < total) {
                    const int b = u % nb, gm = u / nb, gx = gm / M, m = gm - gx * M;
                    const float4 *src = reinterpret_cast<const float4 *>(
                        static_cast<const float *>(p.x[gx]) + static_cast<int64_t>(m) * nb * 32 + b * 32 + 8 * part);
                    const float4 a = __ldg(src), c = __ldg(src + 1);
                    v[ps][0] = a.x; v[ps][1] = a.y; v[ps][2] = a.z; v[ps][3] = a.w;
                    v[ps][4] = c.x; v[ps][5] = c.y; v[ps][6] = c.z; v[ps][7] = c.w;
                }
            }
#pragma unroll
            for (int ps = 0; ps < kPasses; ++ps) {
                if (base + ps * kQuads >= total) break;   // uniform over the CTA
                const int u = base + ps * kQuads + static_cast<int>(threadIdx.x >> 2);
                const Q8Quad r = q8_1_quantize_quad(v[ps]);
                if (u < total) {
                    const int b = u % nb, gm = u / nb, gx = gm / M, m = gm - gx * M;
                    uint8_t *rec = act + (static_cast<int64_t>(gx) * nb + b) * rb;
                    uint32_t *q = reinterpret_cast<uint32_t *>(rec + 32 * m);
                    q[act_word_pos(2 * part)] = r.qlo;
                    q[act_word_pos(2 * part + 1)] = r.qhi;
                    if (part == 0) {
                        const float d8 = f16_bits_to_float(q8_1_d8_bits(r));
                        reinterpret_cast<float *>(rec + 32 * M)[m] = d8 * dscale;
                        if (kQ4K) reinterpret_cast<float *>(rec + 32 * M + 32)[m] = d8 * static_cast<float>(r.sum);
                    }
                }
            }
        }
    } else {
        for (int u = threadIdx.x; u < total; u += kThreads) {
            const int b = u % nb, gm = u / nb, gx = gm / M, m = gm - gx * M;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(p.x[gx]) +
                                                                     (static_cast<int64_t>(m) * nb + b) * 36);
            uint32_t w[9];
#pragma unroll
            for (int i = 0; i < 9; ++i) w[i] = __ldg(src + i);
            uint8_t *rec = act + (static_cast<int64_t>(gx) * nb + b) * rb;
            uint32_t *q = reinterpret_cast<uint32_t *>(rec + 32 * m);
#pragma unroll
            for (int i = 0; i < 8; ++i) q[act_word_pos(i)] = w[1 + i];
            const float d8 = f16_bits_to_float(w[0] & 0xffffu);
            reinterpret_cast<float *>(rec + 32 * M)[m] = d8 * dscale;
            if (kQ4K) {
                int tsum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) tsum = __dp4a(static_cast<int>(w[1 + i]), 0x01010101, tsum);
                reinterpret_cast<float *>(rec + 32 * M + 32)[m] = d8 * static_cast<float>(tsum);   // exact
            }
        }
    }
    for (int u = threadIdx.x; u < p.nx * nb * (8 - M); u += kThreads) {   // d8 (and d8 T) of rows M..7
        const int rec_i = u / (8 - M), k = u - rec_i * (8 - M);
        reinterpret_cast<float *>(act + static_cast<int64_t>(rec_i) * rb + 32 * M)[M + k] = 0.0f;
        if (kQ4K) reinterpret_cast<float *>(act + static_cast<int64_t>(rec_i) * rb + 32 * M + 32)[M + k] = 0.0f;
    }
}

__device__ __forceinline__ void mma_16832_s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0), "r"(0), "r"(0), "r"(0));
}

// The A-operand words of qs word t of block j of a staged row: low nibbles (k 4t..)
// and high nibbles (k 16+4t..) as int8 16 (q - 8); and the block's d4.
struct WeightFrag {
    uint32_t lo, hi;
    float d4;
};

__device__ __forceinline__ WeightFrag weight_block(const uint8_t *row, int j, int t)
{
    const uint8_t *blk = row + 18 * j;
    uint32_t qs, dw;
    if ((j & 1) == 0) {   // block at 0 mod 4: d4 in the low half of its first word, qs at 2 mod 4
        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(blk + 4 * t);
        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(blk + 4 * t + 4);
        qs = __byte_perm(w0, w1, 0x5432);
        dw = *reinterpret_cast<const uint32_t *>(blk) & 0xffffu;
    } else {              // block at 2 mod 4: qs aligned, d4 in the high half of the word before
        qs = *reinterpret_cast<const uint32_t *>(blk + 2 + 4 * t);
        dw = *reinterpret_cast<const uint32_t *>(blk - 2) >> 16;
    }
    WeightFrag f;
    f.lo = ((qs << 4) & 0xf0f0f0f0u) ^ 0x80808080u;
    f.hi = (qs & 0xf0f0f0f0u) ^ 0x80808080u;
    f.d4 = f16_bits_to_float(dw);
    return f;
}

// kQ4K: the weights are Q4_K super-blocks (144 bytes per row per step, like eight
// Q4_0 blocks): per sub-block j one mma of the unsigned nibbles (D = S exactly),
// y += d8 (d sc_j S - dmin mn_j T) with d8 and d8 T from the staged record.
template <bool kFused, bool kDots, bool kQ4K>
__global__ void __launch_bounds__(kThreads, 1) q4_0_mma_kernel(const __grid_constant__ MmaParams p, int64_t K)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int S = p.S, B = p.B;
    const int nb = static_cast<int>(K >> 5);
    const int nsteps = nb >> 3;   // 8 blocks per step
    const int ntiles = p.tile_start[p.count];
    const MmaLayout L = mma_layout(S, B, p.nx, nb, p.M, kQ4K);
    const int rb = act_block_bytes(p.M, kQ4K);
    uint8_t *ring = smem + warp * S * kBox;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.off_bar) + warp * S;
    uint8_t *act = smem + L.off_act;
    float *red = reinterpret_cast<float *>(smem + L.off_red);
    const uint64_t pol = policy_evict_first();

    // matrix of a tile, and the tile's first row within it
    auto locate = [&](int tile, int &mi, int &row0) {
        mi = 0;
#pragma unroll
        for (int i = 1; i < kMaxGroup; ++i)
            if (i < p.count && tile >= p.tile_start[i]) mi = i;
        row0 = (tile - p.tile_start[mi]) * kTile;
    };

    // This CTA's tiles blockIdx.x + gridDim.x * lt (lt < nt) in rounds of B tiles; this
    // warp's steps of a round are items warp, warp + 8, ... (item = tile * nsteps + step).
    const int nt = (ntiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                   static_cast<int>(gridDim.x);
    const int tb0 = warp / nsteps, s0 = warp - tb0 * nsteps;
    int p_lt = tb0, p_step = s0, p_rend = min(B, nt);
    int outstanding = 0;   // lane 0: copies issued and not yet consumed
    auto issue = [&](int slot) {
        int mi, row0;
        locate(static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) * p_lt, mi, row0);
        ++outstanding;
        mbar_arrive_expect_tx(&bars[slot], kBox);
        tma_load_2d(ring + slot * kBox, &p.tm[mi], p_step * kUnitBytes, row0, &bars[slot], pol);
        p_step += kWarps;
        while (p_step >= nsteps) {
            p_step -= nsteps;
            ++p_lt;
        }
        if (p_lt >= p_rend) {   // next round: this warp's first item again
            p_lt = p_rend + tb0;
            p_step = s0;
            p_rend = min(p_rend + B, nt);
        }
    };
    auto pending = [&]() { return p_lt < p_rend; };
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
    stage_act<kFused, kQ4K>(p, nb, act);
    __syncthreads();

    int slot = 0;
    uint32_t phase = 0;
    for (int round = 0; round * B < nt; ++round) {
        const int bt = min(B, nt - round * B);
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        int cur = 0;   // tile of the round that acc holds
        // store acc as tile cur of this warp's partials, zeros for cur+1 .. upto-1
        auto flush = [&](int upto) {
            for (int tb = cur; tb < upto; ++tb) {
                const bool mine = tb == cur;
                float *pr = red + (warp * B + tb) * kTile * kRedPitch;
                pr[gid * kRedPitch + 2 * t] = mine ? acc[0] : 0.0f;
                pr[gid * kRedPitch + 2 * t + 1] = mine ? acc[1] : 0.0f;
                pr[(gid + 8) * kRedPitch + 2 * t] = mine ? acc[2] : 0.0f;
                pr[(gid + 8) * kRedPitch + 2 * t + 1] = mine ? acc[3] : 0.0f;
            }
            acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
        };
        int mi = 0, row0 = 0, tile_of = -1;
        const uint8_t *xa = act;
        bool failed = false;
        for (int tb = tb0, s = s0; tb < bt;) {
            if (tb != cur) {
                flush(tb);
                cur = tb;
            }
            const int tile = static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) * (round * B + tb);
            if (tile != tile_of) {
                locate(tile, mi, row0);
                tile_of = tile;
                xa = act + static_cast<int64_t>(p.xslot[mi]) * nb * rb;
            }
            if (!mbar_wait_bounded(&bars[slot], phase)) {
                if (lane == 0) note_wait_timeout(&g_q4m_error, &cta_abort);
                failed = true;
                break;   // skip the rest of the round, up to its barrier
            }
            --outstanding;
            const uint8_t *box = ring + slot * kBox;
            const uint8_t *rg = box + gid * kUnitBytes, *rh = box + (gid + 8) * kUnitBytes;
            if constexpr (kQ4K) {
                // super-block headers of rows gid, gid + 8 (16-byte aligned: 144-byte pitch)
                const uint4 hg = *reinterpret_cast<const uint4 *>(rg), hh = *reinterpret_cast<const uint4 *>(rh);
                const float dg = f16_bits_to_float(hg.x & 0xffffu), mg = f16_bits_to_float(hg.x >> 16);
                const float dh = f16_bits_to_float(hh.x & 0xffffu), mh = f16_bits_to_float(hh.x >> 16);
                // six-bit scales and minimums: sub-blocks 0..3 in the low bits of bytes 0..7,
                // 4..7 from a nibble of bytes 8..11 and the top two bits of bytes 0..7
                const uint32_t scg[2] = {hg.y & 0x3f3f3f3fu, (hg.w & 0x0f0f0f0fu) | ((hg.y >> 2) & 0x30303030u)};
                const uint32_t mng[2] = {hg.z & 0x3f3f3f3fu, ((hg.w >> 4) & 0x0f0f0f0fu) | ((hg.z >> 2) & 0x30303030u)};
                const uint32_t sch[2] = {hh.y & 0x3f3f3f3fu, (hh.w & 0x0f0f0f0fu) | ((hh.y >> 2) & 0x30303030u)};
                const uint32_t mnh[2] = {hh.z & 0x3f3f3f3fu, ((hh.w >> 4) & 0x0f0f0f0fu) | ((hh.z >> 2) & 0x30303030u)};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // data words t and 4 + t of sub-block pair c: k 4t.. and 16 + 4t.. of
                    // sub-block 2c (low nibbles) and 2c + 1 (high nibbles)
                    const uint32_t g0 = *reinterpret_cast<const uint32_t *>(rg + 16 + 32 * c + 4 * t);
                    const uint32_t g1 = *reinterpret_cast<const uint32_t *>(rg + 32 + 32 * c + 4 * t);
                    const uint32_t h0 = *reinterpret_cast<const uint32_t *>(rh + 16 + 32 * c + 4 * t);
                    const uint32_t h1 = *reinterpret_cast<const uint32_t *>(rh + 32 + 32 * c + 4 * t);
#pragma unroll
                    for (int hi = 0; hi < 2; ++hi) {
                        const int j = 2 * c + hi;
                        const int sh = 4 * hi;
                        const int b = s * 8 + j;
                        const uint8_t *rec = xa + static_cast<int64_t>(b) * rb;
                        const uint2 bw = gid < p.M ? *reinterpret_cast<const uint2 *>(rec + 32 * gid + 8 * t)
                                                   : make_uint2(0u, 0u);
                        int d[4];
                        mma_16832_s8(d, (g0 >> sh) & 0x0f0f0f0fu, (h0 >> sh) & 0x0f0f0f0fu, (g1 >> sh) & 0x0f0f0f0fu,
                                     (h1 >> sh) & 0x0f0f0f0fu, bw.x, bw.y);
                        if (kDots) {
                            const int64_t n0 = row0 + gid, n1 = n0 + 8, N0 = p.N[0];
                            const int m0 = 2 * t, m1 = m0 + 1;
                            if (m0 < p.M && n0 < N0) p.dots[(m0 * N0 + n0) * nb + b] = d[0];
                            if (m1 < p.M && n0 < N0) p.dots[(m1 * N0 + n0) * nb + b] = d[1];
                            if (m0 < p.M && n1 < N0) p.dots[(m0 * N0 + n1) * nb + b] = d[2];
                            if (m1 < p.M && n1 < N0) p.dots[(m1 * N0 + n1) * nb + b] = d[3];
                        } else {
                            const int wi = j >> 2, by = 8 * (j & 3);
                            const float dsg = dg * static_cast<float>((scg[wi] >> by) & 0xffu);
                            const float dmg = mg * static_cast<float>((mng[wi] >> by) & 0xffu);
                            const float dsh = dh * static_cast<float>((sch[wi] >> by) & 0xffu);
                            const float dmh = mh * static_cast<float>((mnh[wi] >> by) & 0xffu);
                            const float2 d8 = *reinterpret_cast<const float2 *>(rec + 32 * p.M + 8 * t);
                            const float2 d8t = *reinterpret_cast<const float2 *>(rec + 32 * p.M + 32 + 8 * t);
                            acc[0] = fmaf(static_cast<float>(d[0]), dsg * d8.x, fmaf(-dmg, d8t.x, acc[0]));
                            acc[1] = fmaf(static_cast<float>(d[1]), dsg * d8.y, fmaf(-dmg, d8t.y, acc[1]));
                            acc[2] = fmaf(static_cast<float>(d[2]), dsh * d8.x, fmaf(-dmh, d8t.x, acc[2]));
                            acc[3] = fmaf(static_cast<float>(d[3]), dsh * d8.y, fmaf(-dmh, d8t.y, acc[3]));
                        }
                    }
                }
            } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const WeightFrag fg = weight_block(rg, j, t), fh = weight_block(rh, j, t);
                const int b = s * 8 + j;
                const uint8_t *rec = xa + static_cast<int64_t>(b) * rb;
                // words t (k 4t..) and 4 + t (k 16 + 4t..) of activation row gid
                const uint2 bw = gid < p.M ? *reinterpret_cast<const uint2 *>(rec + 32 * gid + 8 * t)
                                           : make_uint2(0u, 0u);
                int d[4];
                mma_16832_s8(d, fg.lo, fh.lo, fg.hi, fh.hi, bw.x, bw.y);
                if (kDots) {
                    // 16 (S - 8T) -> S - 8T for rows row0 + gid (+8), activation rows 2t, 2t+1
                    const int64_t n0 = row0 + gid, n1 = n0 + 8, N0 = p.N[0];
                    const int m0 = 2 * t, m1 = m0 + 1;
                    if (m0 < p.M && n0 < N0) p.dots[(m0 * N0 + n0) * nb + b] = d[0] >> 4;
                    if (m1 < p.M && n0 < N0) p.dots[(m1 * N0 + n0) * nb + b] = d[1] >> 4;
                    if (m0 < p.M && n1 < N0) p.dots[(m0 * N0 + n1) * nb + b] = d[2] >> 4;
                    if (m1 < p.M && n1 < N0) p.dots[(m1 * N0 + n1) * nb + b] = d[3] >> 4;
                } else {
                    const float2 d8 = *reinterpret_cast<const float2 *>(rec + 32 * p.M + 8 * t);   // d8 / 16
                    acc[0] = fmaf(static_cast<float>(d[0]), fg.d4 * d8.x, acc[0]);
                    acc[1] = fmaf(static_cast<float>(d[1]), fg.d4 * d8.y, acc[1]);
                    acc[2] = fmaf(static_cast<float>(d[2]), fh.d4 * d8.x, acc[2]);
                    acc[3] = fmaf(static_cast<float>(d[3]), fh.d4 * d8.y, acc[3]);
                }
            }
            }
            __syncwarp();   // every lane is done with the box: refill the slot
            if (lane == 0 && pending()) {
                fence_proxy_async_shared();   // the warp's reads of the box before the copy's writes
                issue(slot);
            }
            if (++slot == S) {
                slot = 0;
                phase ^= 1u;
            }
            s += kWarps;
            while (s >= nsteps) {
                s -= nsteps;
                ++tb;
            }
        }
        if (kDots) {   // no reduction and no CTA-wide barrier: every block dot went out directly
            if (failed) {
                if (lane == 0) drain_ring(bars, S, slot, phase, outstanding);
                return;
            }
            continue;
        }
        flush(bt);
        __syncthreads();
        if (cta_abort) {   // a warp gave up waiting: the whole CTA leaves here, its copies landed
            if (lane == 0) drain_ring(bars, S, slot, phase, outstanding);
            return;
        }
        for (int e = tid; e < bt * kTile * 8; e += kThreads) {
            const int rr = e >> 3, m = e & 7, tb = rr / kTile, r = rr - tb * kTile;
            if (m >= p.M) continue;
            int emi, erow0;
            locate(static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) * (round * B + tb), emi, erow0);
            const int64_t n = erow0 + r;
            if (n < p.N[emi]) {
                float sum = 0.0f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) sum += red[((w * B) * kTile + rr) * kRedPitch + m];
                p.y[emi][m * p.N[emi] + n] = sum;
            }
        }
        __syncthreads();   // red is reused by the next round
    }
}

}  // namespace

cudaError_t plan_q4_0_mma(const DeviceInfo &dev, const Q4Group &grp, int M, int64_t K, Q4Plan *plan, bool q4k)
{
    plan->route = kRouteQ4_0Generic;   // "not planned"
    if (K % 256 != 0 || M < 1 || M > 8) return cudaSuccess;
    for (int i = 0; i < grp.count; ++i)
        if ((reinterpret_cast<uintptr_t>(grp.w[i]) & 15u) != 0) return cudaSuccess;
    const int64_t nb = K / 32, nsteps = nb / 8;
    int64_t ntiles = 0;
    for (int i = 0; i < grp.count; ++i) ntiles += (grp.row_start[i + 1] - grp.row_start[i] + kTile - 1) / kTile;
    if (ntiles == 0 || ntiles > 0x7fffffff || nb > 0x7fffffff / act_block_bytes(M, q4k)) return cudaSuccess;
    // tiles per round: a multiple of 8 / gcd(steps, 8), so every warp gets the same
    // number of steps, and enough for 8 steps per warp between the round's barriers
    int gcd = kWarps;
    while (nsteps % gcd) gcd >>= 1;
    const int unit = kWarps / gcd;
    int B = unit;
    while (B * nsteps < 8 * kWarps && B + unit <= kMaxRound) B += unit;
    // the most ring slots that let two CTAs share an SM, else the most that fit
    const int s_env = env_int("QMV_Q4_MMA_SLOTS", 0);
    const int cands[3] = {4, 3, 2};
    int best_s = 0, best_occ = 0;
    for (int c = 0; c < 3; ++c) {
        const int S = s_env > 0 ? std::min(8, s_env) : cands[c];
        const uint32_t dyn = mma_layout(S, B, grp.nx, static_cast<int>(nb), M, q4k).total;
        if (dyn > static_cast<uint32_t>(dev.smem_optin)) continue;
        auto k = q4k ? q4_0_mma_kernel<true, false, true> : q4_0_mma_kernel<true, false, false>;
        cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(k), dev.smem_optin);
        if (e != cudaSuccess) return e;
        int occ = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, dyn)) != cudaSuccess) return e;
        if (occ < 1) continue;
        if (best_s == 0) {
            best_s = S;
            best_occ = occ;
        }
        if (occ >= 2) {
            best_s = S;
            best_occ = occ;
            break;
        }
    }
    if (best_s == 0) return cudaSuccess;
    plan->route = kRouteQ4_0Mma;
    plan->warps = kWarps;
    plan->stages = best_s;
    plan->round = B;
    plan->prefetch = 0;
    plan->chunk_units = 1;
    plan->grid = static_cast<int>(std::min<int64_t>(ntiles, static_cast<int64_t>(dev.sm_count) * std::min(4, best_occ)));
    plan->smem_bytes = static_cast<int>(mma_layout(best_s, B, grp.nx, static_cast<int>(nb), M, q4k).total);
    return cudaSuccess;
}

cudaError_t launch_q4_0_mma(const Q4Plan &plan, const Q4Group &grp, int32_t *dots, int M, int64_t K, bool fused,
                            cudaStream_t s, bool q4k)
{
    MmaParams p{};
    p.count = grp.count;
    p.nx = grp.nx;
    p.M = M;
    p.S = plan.stages;
    p.B = plan.round;
    p.dots = dots;
    const int64_t rowbytes = K / 32 * 18;
    int tiles = 0;
    for (int i = 0; i < grp.count; ++i) {
        p.tile_start[i] = tiles;
        p.N[i] = grp.row_start[i + 1] - grp.row_start[i];
        p.xslot[i] = grp.xslot[i];
        p.y[i] = grp.y[i];
        tiles += static_cast<int>((p.N[i] + kTile - 1) / kTile);
        if (p.N[i] > 0) {
            cudaError_t e = encode_map_2d(&p.tm[i], grp.w[i], p.N[i], rowbytes, kUnitBytes, kTile,
                                          CU_TENSOR_MAP_SWIZZLE_NONE);
            if (e != cudaSuccess) return e;
        }
    }
    for (int i = grp.count; i <= kMaxGroup; ++i)
        if (i <= kMaxGroup) p.tile_start[i] = tiles;
    for (int i = 0; i < grp.nx; ++i) p.x[i] = grp.x[i];

    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(plan.smem_bytes);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = set_launch_overlap_attr(attr);
    auto kern = q4k ? (dots ? q4_0_mma_kernel<false, true, true>
                            : (fused ? q4_0_mma_kernel<true, false, true> : q4_0_mma_kernel<false, false, true>))
                    : (dots ? q4_0_mma_kernel<false, true, false>
                            : (fused ? q4_0_mma_kernel<true, false, false> : q4_0_mma_kernel<false, false, false>));
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(kern), plan.smem_bytes);
    if (e != cudaSuccess) return e;
    route_hit(q4k ? (fused ? kRouteQ4KMmaFused : kRouteQ4KMma) : (fused ? kRouteQ4_0MmaFused : kRouteQ4_0Mma));
    return cudaLaunchKernelEx(&cfg, kern, p, K);
}

cudaError_t read_error_word_q4_0_mma(uint32_t *out, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_q4m_error, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_q4m_error, &zero, sizeof(uint32_t));
}

}  // namespace qmv
