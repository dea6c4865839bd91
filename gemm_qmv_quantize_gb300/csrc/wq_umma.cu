// wq_umma.cu -- NVFP4 W4A16 and FP8 W8A16 skinny GEMM on the 5th-generation tensor
// cores (tcgen05), M = 1..96 activation rows in one pass over the weights.
//
// QPN2 / QPN8 of "v100-skinny README", section "How QPN works": packed weights are
// streamed once and decoded on chip into the operands of a tensor-core product
// against fp16 activations, with fp32 accumulation. The page's Volta kernels decode
// into mma registers lane by lane; here single threads issue tcgen05.mma, so most
// warps only decode:
//  * A tile = 128 weight rows x K of one matrix (TMEM lane = weight row); B = the M
//    activation rows, padded with zero rows to N = 16 ceil(M / 16) <= 96; D (fp32,
//    128 x N) accumulates over all of K in tensor memory. The whole activation
//    width rides one weight pass: the README's M = 9..16 and 17..96 bands need no
//    second pass over the weights and no chunking.
//  * The decoded A operand lives in tensor memory too: a decode thread owns one
//    weight row, which is one TMEM lane, and writes its fp16 pairs there with
//    tcgen05.st; the MMA reads A from TMEM and only B from shared memory, which then
//    holds the weight stages and activation slices alone.
//  * Exact decode, as in the mma.sync kernel: an E2M1 code times its E4M3 group
//    scale is exact in fp16 (at most 6 significant bits, magnitude 2^-10 .. 2688),
//    so the scale is folded into the fp16 weight; E4M3 to fp16 is exact; the
//    per-tensor scale (NVFP4) or the row scale (FP8) multiplies the fp32 result.
//  * Roles (warp specialisation): warps 0..2 each have one thread that streams every
//    third K step's codes (a 128-row box with the 128-byte swizzle) and group scales
//    with TMA into its own slots of the weight ring (warp 1 also allocates tensor
//    memory); warps 3..14, three groups of four, decode the 64-k quarters in turn (one
//    weight row per thread, all 64 k of the quarter) and at the end of a tile read the
//    accumulators back (tcgen05.ld) and store y; warps 15..18 each have one thread
//    that streams its own 64-k activation slices (the K-major B operand, a box with
//    the 128-byte swizzle, rows past M zero-filled) and issues four MMAs per quarter
//    into its own accumulator. A single thread sustains only a few TMA copies per
//    microsecond under load, hence the copies spread over seven threads.
//  * Launches of few tiles split K over the CTAs of a cluster: each CTA leaves its
//    partial sums in shared memory and the rank-0 CTA adds them in rank order through
//    distributed shared memory.
//  * Every mbarrier wait is bounded; a thread whose wait gives up flags the error
//    word and the CTA's abort word and leaves its loop; all threads meet at the final
//    barrier (and both cluster barriers), the producers let their copies land, the
//    issuing threads wait for their products and copies, and the tensor memory is
//    released before the CTA exits.
#include <algorithm>
#include <numeric>
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
constexpr int kACols = kQuarterK / 2;  // TMEM columns of one 64-k A buffer (fp16 pairs)
constexpr int kTmemCols = 512;         // the whole of tensor memory: accumulators and A buffers
constexpr int kWeightProducers = 3;    // warps 0, 1, 2: one thread each streams every third K step
#ifndef QMV_UMMA_DECODE_GROUPS
#define QMV_UMMA_DECODE_GROUPS 3
#endif
constexpr int kDecodeGroups = QMV_UMMA_DECODE_GROUPS;   // groups of four warps (one per TMEM lane
constexpr int kDecodeWarps = 4 * kDecodeGroups;         // quarter), quarter h to group h % groups
constexpr int kFirstDecodeWarp = 3;    // warps 0..2 weight producers (warp 1 also allocates TMEM), then decode
#ifndef QMV_UMMA_ISSUER_WARPS
#define QMV_UMMA_ISSUER_WARPS (16 - 4 * QMV_UMMA_DECODE_GROUPS)
#endif
constexpr int kMaxIssuers = QMV_UMMA_ISSUER_WARPS;   // the warps after the decode warps: one MMA-issuing thread each
constexpr int kFirstIssuerWarp = kFirstDecodeWarp + kDecodeWarps;
constexpr int kThreadsUmma = 32 * (kFirstIssuerWarp + kMaxIssuers);
constexpr int kMaxStages = 12;         // weight stages (one K step of codes and scales each), a multiple of 3
constexpr int kMaxSlicesPerIssuer = 12;
constexpr int kMaxABufs = 12;          // 64-k A buffers in TMEM

__host__ __device__ constexpr int step_k(bool fp4) { return fp4 ? 256 : 128; }   // 128 code bytes per row

struct UmmaLayout {
    uint32_t off_codes, off_scales, off_b, off_bar, off_misc, total;
    uint32_t b_bytes;   // one 64-k activation slice: 64 x N fp16
};

// Dynamic shared memory (base aligned to 1024 bytes): S weight stages of codes
// (1024-aligned for the 128-byte swizzle) and scales, R 64-k activation slices, the
// mbarriers (Q of each A-buffer kind), the tensor-memory address and the abort word.
__host__ __device__ inline UmmaLayout umma_layout(bool fp4, int S, int R, int Q, int n_pad)
{
    UmmaLayout L;
    L.b_bytes = static_cast<uint32_t>(kQuarterK * n_pad * 2);
    L.off_codes = 0;
    L.off_scales = L.off_codes + static_cast<uint32_t>(S * kCodesBox);
    L.off_b = (L.off_scales + (fp4 ? static_cast<uint32_t>(S * kScalesBox) : 0u) + 1023u) & ~1023u;
    L.off_bar = L.off_b + static_cast<uint32_t>(R) * L.b_bytes;
    // w_full, w_free: S each; b_full, b_free: R each; a_full, a_free: Q each; acc_full, acc_free, done
    L.off_misc = L.off_bar + static_cast<uint32_t>(2 * S + 2 * R + 2 * Q + 3) * 8u;
    L.total = L.off_misc + 16u;
    return L;
}

// First TMEM column of the A buffers: after the T accumulators of n_pad columns,
// 32-aligned. plan_umma keeps a_first_col + 32 Q <= 512.
__host__ __device__ constexpr uint32_t a_first_col(int T, int n_pad)
{
    return (static_cast<uint32_t>(T * n_pad) + 31u) & ~31u;
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

// D (+)= A x B with A in tensor memory (128 lanes = rows, fp16 pairs along columns).
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
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

// 16 consecutive 32-bit columns of this thread's TMEM lane from v (warp-wide,
// .sync.aligned); the stores are complete when tcgen05.wait::st returns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// All threads of every CTA of the cluster (release / acquire: shared-memory writes
// before it are visible to the cluster's reads after it).
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The float at the same shared-memory offset in the cluster's CTA `rank`.
__device__ __forceinline__ float ld_peer_f32(const float *local, int rank)
{
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

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
    wq_umma_kernel(const __grid_constant__ UmmaParams p, int M, int64_t K, int n_pad, int S, int rb, int Q, int T,
                   int splits, uint32_t tmem_cols)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int R = T * rb;   // activation slices: rb per issuing thread
    const UmmaLayout L = umma_layout(kFp4, S, R, Q, n_pad);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kStepK = step_k(kFp4);
    constexpr int kQuarters = kStepK / kQuarterK;
    // Split K (splits > 1): a cluster of `splits` CTAs shares one tile, CTA `rank` taking
    // the K steps [st0, st0 + nsteps); its partial sums meet in the rank-0 CTA.
    const int nsteps_all = static_cast<int>(K / kStepK);
    const int rank = splits > 1 ? static_cast<int>(blockIdx.x) % splits : 0;
    const int st0 = rank * nsteps_all / splits;
    const int nsteps = (rank + 1) * nsteps_all / splits - st0;   // K steps of this CTA per tile
    const int tile_quarters = nsteps * kQuarters;
    const int q0 = st0 * kQuarters;   // first 64-k quarter of K
    const int ntiles = p.tile_start[p.count];
    const int first_tile = static_cast<int>(blockIdx.x) / splits, tile_stride = static_cast<int>(gridDim.x) / splits;
    const int nt = (ntiles - first_tile + tile_stride - 1) / tile_stride;   // tiles first_tile + tile_stride * lt
    const int total_steps = nt * nsteps, total_quarters = total_steps * kQuarters;
    const int used = min(T, tile_quarters);   // accumulators a tile writes

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.off_bar);
    uint64_t *w_full = bars, *w_free = bars + S, *b_full = bars + 2 * S, *b_free = b_full + R;
    uint64_t *a_full = b_free + R, *a_free = a_full + Q, *acc_full = a_free + Q, *acc_free = acc_full + 1;
    uint64_t *done = acc_free + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile uint32_t *abort_word = reinterpret_cast<volatile uint32_t *>(smem + L.off_misc + 4);
    uint8_t *codes_ring = smem + L.off_codes, *scales_ring = smem + L.off_scales;
    uint8_t *b_ring = smem + L.off_b;
    const uint32_t a_col0 = a_first_col(T, n_pad);   // TMEM: accumulators, then the A buffers

    auto locate = [&](int tile, int &mi, int &row0) {
        mi = 0;
#pragma unroll
        for (int i = 1; i < kMaxGroup; ++i)
            if (i < p.count && tile >= p.tile_start[i]) mi = i;
        row0 = (tile - p.tile_start[mi]) * kTileRows;
    };
    auto fail = [&]() { note_wait_timeout(&g_umma_error, abort_word); };
    // K step g sits in slot (g % 3) + 3 ((g / 3) % (S / 3)): producer g % 3's own slots,
    // the (g / S)-th use of that slot
    auto stage_slot = [&](int g) {
        return g % kWeightProducers + kWeightProducers * ((g / kWeightProducers) % (S / kWeightProducers));
    };

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
            mbar_init(&a_full[j], kDecodeWarps / kDecodeGroups);
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

    if (warp < kWeightProducers) {
        // ------------------------------------------------ weight producers (one thread each)
        // Producer w loads the K steps g with g % 3 == w into its own slots. Weights do
        // not depend on the preceding kernel: the ring fills before the dependency wait
        // (these threads never wait for it: they touch no activation).
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const uint32_t tx = kCodesBox + (kFp4 ? kScalesBox : 0);
            int last = -1;
            for (int g = warp; g < total_steps && !*abort_word; g += kWeightProducers) {
                const int s = stage_slot(g);
                if (g >= S && !mbar_wait_bounded(&w_free[s], static_cast<uint32_t>((g / S) - 1) & 1u)) {
                    fail();
                    break;
                }
                const int lt = g / nsteps, st = g - lt * nsteps;
                int mi, row0;
                locate(first_tile + tile_stride * lt, mi, row0);
                mbar_arrive_expect_tx(&w_full[s], tx);
                tma_load_2d(codes_ring + s * kCodesBox, &p.codes[mi], (st0 + st) * 128, row0, &w_full[s], pol);
                if (kFp4) tma_load_2d(scales_ring + s * kScalesBox, &p.scales[mi], (st0 + st) * 16, row0, &w_full[s], pol);
                last = g;
            }
            // every copy lands before the CTA can exit (the slot of a step within the last S
            // has not been reused, so its phase is the one that step's copy completes)
            for (int g = warp; g <= last; g += kWeightProducers)
                if (g > last - S) (void)mbar_wait_bounded(&w_full[stage_slot(g)], static_cast<uint32_t>(g / S) & 1u);
        }
    } else if (warp >= kFirstIssuerWarp) {
        // ------------------------------------------------ MMA issue: thread t takes quarters t, t + T, ...
        // of every tile, and streams their activation slices itself through its own rb
        // slots (slot t + T (i % rb) for its i-th quarter): a single thread sustains only
        // a few TMA copies per microsecond under load, so the copies are spread over the
        // T issuing threads.
        const int t = warp - kFirstIssuerWarp;
        if (lane == 0 && t < T) {
            const uint32_t idesc = idesc_f16_f32(kTileRows, n_pad);
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(t * n_pad);
            const int per_tile = t < tile_quarters ? (tile_quarters - t + T - 1) / T : 0;
            const int nmine = nt * per_tile;
            auto bslot = [&](int i) { return t + T * (i % rb); };
            grid_dependency_wait();   // the activations may be written by the preceding kernel
            const uint64_t pol_x = policy_evict_last();
            auto load_b = [&](int i) {
                const int jb = bslot(i), kq = t + T * (i % per_tile);
                mbar_arrive_expect_tx(&b_full[jb], L.b_bytes);
                tma_load_2d(b_ring + jb * L.b_bytes, &p.x, (q0 + kq) * kQuarterK, 0, &b_full[jb], pol_x);
            };
            int loaded = 0;
            for (; loaded < rb && loaded < nmine; ++loaded) load_b(loaded);
            bool ok = true, any = false;
            int i = 0;   // this thread's quarters so far
            for (int lt = 0; lt < nt && ok; ++lt) {
                if (lt >= 1 && t < used &&   // the read-back of the previous tile is done
                    !mbar_wait_bounded(acc_free, static_cast<uint32_t>(lt - 1) & 1u)) {
                    fail();
                    break;
                }
                tc_fence_after();
                bool first = true;
                for (int kq = t; kq < tile_quarters && ok; kq += T, ++i) {
                    const int h = lt * tile_quarters + kq;
                    const int ja = h % Q, jb = bslot(i);
                    // refill the slot of the previous quarter (loaded == i - 1 + rb) once its
                    // products are done
                    if (i >= 1 && loaded < nmine) {
                        if (*abort_word || !mbar_wait_bounded(&b_free[bslot(i - 1)], static_cast<uint32_t>((i - 1) / rb) & 1u)) {
                            fail();
                            ok = false;
                            break;
                        }
                        load_b(loaded++);
                    }
                    if (*abort_word || !mbar_wait_bounded(&b_full[jb], static_cast<uint32_t>(i / rb) & 1u) ||
                        !mbar_wait_bounded(&a_full[ja], static_cast<uint32_t>(h / Q) & 1u)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_tmem = tmem + a_col0 + static_cast<uint32_t>(ja * kACols);
                    const uint32_t b_base = smem_addr(b_ring + jb * L.b_bytes);
#pragma unroll
                    for (int kk = 0; kk < kQuarterK / 16; ++kk)   // k 16 kk ..: A columns 8 kk .., B bytes 32 kk ..
                        umma_f16_ta(d_tmem, a_tmem + 8u * kk, smem_desc_sw128(b_base + 32u * kk), idesc,
                                    (first && kk == 0) ? 0u : 1u);
                    first = false;
                    any = true;
                    umma_commit(&a_free[ja]);   // the A buffer and the activation slice are free once
                    umma_commit(&b_free[jb]);   // these products are done
                }
                if (ok && t < used) umma_commit(acc_full);   // this thread's share of the tile is done
            }
            // every product this thread issued has completed before the tensor memory is
            // released, and every activation copy it started has landed
            if (any) {
                umma_commit(done);
            } else {
                mbar_arrive(done);
            }
            (void)mbar_wait_bounded(done, 0u);
            for (int k = i; k < loaded; ++k) (void)mbar_wait_bounded(&b_full[bslot(k)], static_cast<uint32_t>(k / rb) & 1u);
        }
        __syncwarp();
    } else if (warp >= kFirstDecodeWarp) {
        // ------------------------------------------------ decode, then read back
        // Groups of four warps take turns on the 64-k quarters (group gq the quarters h
        // with h % groups == gq; every decode warp takes and releases every K step). In
        // a group, warp w decodes the rows of its TMEM lane quarter 32 (w % 4) .. + 31,
        // one row per thread, all 64 k of the quarter: 32 TMEM columns of fp16 pairs.
        // Waits are made warp-uniform, since the tensor-memory accesses that follow them
        // are .sync.aligned.
        const int r = 32 * (warp & 3) + lane;
        const int gq = (warp - kFirstDecodeWarp) >> 2;
        const uint32_t a_lane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + a_col0;
        const int sw = r & 7;   // the codes box's 128-byte swizzle: chunk c of row r at c ^ (r % 8)
        auto wait_all = [&](uint64_t *bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity) ? 1 : 0) != 0;
        };
        int g = 0, h = 0;
        bool ok = true, waited = false;
        for (int lt = 0; lt < nt && ok; ++lt) {
            int mi, row0;
            locate(first_tile + tile_stride * lt, mi, row0);
            for (int st = 0; st < nsteps && ok; ++st, ++g) {
                const int s = stage_slot(g);
                if (*abort_word || !wait_all(&w_full[s], static_cast<uint32_t>(g / S) & 1u)) {
                    fail();
                    ok = false;
                    break;
                }
                const uint8_t *crow = codes_ring + s * kCodesBox + r * 128;
                for (int q = 0; q < kQuarters; ++q) {
                    const int hq = h + q, j = hq % Q;
                    if (hq % kDecodeGroups != gq) continue;
                    if (hq >= Q && !wait_all(&a_free[j], static_cast<uint32_t>((hq / Q) - 1) & 1u)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tc_fence_after();   // the products that read this buffer before are complete
                    uint32_t av[32];    // k pairs (2i, 2i + 1) of the quarter: TMEM column i
                    if (kFp4) {
                        // k 64q .. + 63: code chunks 2q, 2q + 1 (swizzled by row), groups 4q .. 4q + 3
                        const uint32_t s4 =
                            *reinterpret_cast<const uint32_t *>(scales_ring + s * kScalesBox + r * 16 + 4 * q);
                        const uint32_t s01 = e4m3x2_to_f16x2(s4 & 0xffffu), s23 = e4m3x2_to_f16x2(s4 >> 16);
                        const uint32_t sc[4] = {dup_lo16(s01), dup_hi16(s01), dup_lo16(s23), dup_hi16(s23)};
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const uint4 cv = *reinterpret_cast<const uint4 *>(crow + 16 * ((2 * q + c) ^ sw));
                            const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                            for (int kg = 0; kg < 4; ++kg) {   // 8 k: one word of codes, group 2c + kg / 2
                                uint32_t hv[4];
                                e2m1x8_to_f16x2(cw[kg], hv);
                                const uint32_t gsc = sc[2 * c + (kg >> 1)];
#pragma unroll
                                for (int i = 0; i < 4; ++i) av[16 * c + 4 * kg + i] = hmul2_u32(hv[i], gsc);
                            }
                        }
                    } else {
                        // k 64q .. + 63: code chunks 4q .. 4q + 3 (16 k each)
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(crow + 16 * ((4 * q + c) ^ sw));
                            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                av[8 * c + 2 * i] = e4m3x2_to_f16x2(wv[i] & 0xffffu);
                                av[8 * c + 2 * i + 1] = e4m3x2_to_f16x2(wv[i] >> 16);
                            }
                        }
                    }
                    const uint32_t ta = a_lane + static_cast<uint32_t>(j * kACols);
                    tmem_st16(ta, *reinterpret_cast<const uint32_t(*)[16]>(av));
                    tmem_st16(ta + 16u, *reinterpret_cast<const uint32_t(*)[16]>(av + 16));
                    tmem_wait_st();
                    tc_fence_before();   // the stores before the arrival the MMA thread waits on
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&a_full[j]);
                }
                h += kQuarters;
                // Release the slot. No cross-proxy fence is needed before the next copy's
                // async-proxy writes: every value this warp read from the slot has been
                // consumed -- converted, stored to tensor memory and waited for with
                // tcgen05.wait::st -- so the reads are complete. (A fence here waits for
                // the CTA's copies in flight and cost 7 % at M = 32.)
                if (ok) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&w_free[s]);
                }
            }
            if (!ok) break;
            // read back tile lt: row row0 + r of matrix mi, activation rows in 16-column
            // chunks (the two warps of a lane quarter take alternate chunks), the
            // accumulators of the issuing threads summed in a fixed order
            if (!waited) {   // outputs may be read by the preceding kernel until it has finished
                grid_dependency_wait();
                waited = true;
            }
            if (!wait_all(acc_full, static_cast<uint32_t>(lt) & 1u)) {
                fail();
                break;
            }
            tc_fence_after();
            const int64_t n = row0 + r, Nm = p.N[mi];
            const float scale = kFp4 ? p.g[mi] : (n < Nm ? __ldg(p.row_scale[mi] + n) : 0.0f);
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
            // split K: this CTA's partial sums go to its weight ring (idle now: every stage
            // has been consumed) as [column][128 rows] fp32, for the rank-0 CTA to add up
            float *part = reinterpret_cast<float *>(codes_ring);
            for (int c16 = 16 * gq; c16 < n_pad; c16 += 16 * kDecodeGroups) {
                float v[16];
                tmem_ld16(taddr + static_cast<uint32_t>(c16), v);
                for (int a = 1; a < used; ++a) {
                    float u[16];
                    tmem_ld16(taddr + static_cast<uint32_t>(a * n_pad + c16), u);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += u[i];
                }
                if (splits > 1) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) part[(c16 + i) * kTileRows + r] = v[i];
                } else if (n < Nm) {
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
    if (splits > 1) {
        // every CTA of the cluster has its partial sums in shared memory; the rank-0 CTA's
        // decode threads (past the dependency wait, like every writer of y) add them up
        // in rank order and store y; the second barrier keeps the other CTAs' shared
        // memory alive until then
        cluster_sync_all();
        if (rank == 0 && warp >= kFirstDecodeWarp && warp < kFirstIssuerWarp) {
            grid_dependency_wait();   // (done already unless this warp gave up early)
            int mi, row0;
            locate(first_tile, mi, row0);
            const int64_t Nm = p.N[mi];
            const float *part = reinterpret_cast<const float *>(codes_ring);
            for (int idx = tid - 32 * kFirstDecodeWarp; idx < kTileRows * M; idx += 32 * kDecodeWarps) {
                const int rr = idx % kTileRows, c = idx / kTileRows;
                const int64_t n = row0 + rr;
                float v = part[c * kTileRows + rr];
                for (int k = 1; k < splits; ++k) v += ld_peer_f32(&part[c * kTileRows + rr], k);
                if (n < Nm) p.y[mi][static_cast<int64_t>(c) * Nm + n] = v * (kFp4 ? p.g[mi] : __ldg(p.row_scale[mi] + n));
            }
        }
        cluster_sync_all();
    }
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
    // Tensor memory (512 columns) holds T accumulators of n_pad columns, one per
    // MMA-issuing thread, and Q 64-k A buffers of 32 columns. Q is a multiple of the
    // decode groups (each A buffer is then written by one group only) and of T: thread
    // t takes quarters t, t + T, ..., so the quarter that last used buffer h % Q,
    // h - Q, is one of its own earlier quarters, whose phase it has waited for. Any
    // other Q lets a thread meet a buffer two phases behind -- the decode groups drift
    // against each other -- and pass its parity test on the phase before (seen as
    // timeouts with 7 threads and 9 buffers). T is as large as allows such a Q of at
    // least 6 (the decode runs up to Q quarters ahead of the products). Each issuing
    // thread streams its activation slices through rb slots: enough for about 12
    // quarters of the CTA in flight. Shared memory then takes as many weight stages as
    // fit, a multiple of the 3 producers, 3 .. 12. QMV_UMMA_ISSUERS / QMV_UMMA_ABUFS /
    // QMV_UMMA_STAGES cap T, Q and S; QMV_UMMA_BBUFS sets rb.
    const int t_cap = std::max(1, std::min(kMaxIssuers, env_int("QMV_UMMA_ISSUERS", kMaxIssuers)));
    const int q_cap = std::min(kMaxABufs, env_int("QMV_UMMA_ABUFS", kMaxABufs));
    auto q_room = [&](int t_) {
        return (kTmemCols - static_cast<int>(a_first_col(t_, pl.n_pad))) / kACols;
    };
    // the largest multiple of lcm(groups, t) that fits, or 0
    auto q_for = [&](int t_, int cap) {
        const int l = kDecodeGroups / std::gcd(kDecodeGroups, t_) * t_;
        return std::min(cap, q_room(t_)) / l * l;
    };
    int T = t_cap;
    while (T > 1 && q_for(T, kMaxABufs) < 6) --T;
    if (q_for(T, kMaxABufs) == 0) return cudaErrorInvalidValue;
    const int Q = std::max(q_for(T, q_cap), kDecodeGroups / std::gcd(kDecodeGroups, T) * T);
    int rb = std::max(2, std::min(kMaxSlicesPerIssuer, env_int("QMV_UMMA_BBUFS", (12 + T - 1) / T)));
    auto fits = [&](int s_, int rb_) {
        return umma_layout(fp4, s_, T * rb_, Q, pl.n_pad).total + 1024 <= static_cast<uint32_t>(dev.smem_optin);
    };
    while (rb > 2 && !fits(kWeightProducers, rb)) --rb;
    int S = std::max(kWeightProducers, std::min(kMaxStages, env_int("QMV_UMMA_STAGES", kMaxStages))) /
            kWeightProducers * kWeightProducers;
    while (S > kWeightProducers && !fits(S, rb)) S -= kWeightProducers;
    pl.T = T;
    pl.S = S;
    pl.Q = Q;
    pl.R = T * rb;
    pl.smem = umma_layout(fp4, pl.S, pl.R, pl.Q, pl.n_pad).total + 1024;
    if (pl.smem > static_cast<uint32_t>(dev.smem_optin) || K % step_k(fp4) != 0) return cudaErrorInvalidValue;
    pl.tmem_cols = kTmemCols;
    // Split K when the tiles leave half the SMs idle: clusters of up to 4 CTAs, each
    // with a range of K steps (a CTA streams at a fixed rate, so a launch of few tiles
    // needs more CTAs per tile to fill the device). QMV_UMMA_SPLITS overrides (1: off).
    const int64_t nsteps = K / step_k(fp4);
    int splits = env_int("QMV_UMMA_SPLITS", tiles * 2 <= dev.sm_count ? static_cast<int>(dev.sm_count / std::max<int64_t>(tiles, 1)) : 1);
    splits = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({splits, 4, nsteps})));
    while (splits > 1 && tiles * splits > dev.sm_count) --splits;
    pl.splits = splits;
    pl.grid = splits > 1 ? static_cast<int>(tiles * splits) : static_cast<int>(std::min<int64_t>(tiles, dev.sm_count));
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
    const int n_pad = pl.n_pad, S = pl.S, R = pl.R, Q = pl.Q, T = pl.T, rb = R / T;
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
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreadsUmma);
    cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = set_launch_overlap_attr(attr);
    if (pl.splits > 1) {   // the CTAs of a tile form a cluster
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = static_cast<unsigned>(pl.splits);
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    if (env_int("QMV_PLAN_LOG", 0))
        std::fprintf(stderr,
                     "umma plan: fmt=%s M=%d n_pad=%d K=%lld tiles=%d S=%d R=%d Q=%d issuers=%d splits=%d grid=%u "
                     "smem=%u tmem=%u\n",
                     kFp4 ? "nvfp4" : "fp8", M, n_pad, static_cast<long long>(K), tiles, S, R, Q, T, pl.splits,
                     cfg.gridDim.x, smem, cols);
    return cudaLaunchKernelEx(&cfg, kern, p, M, K, n_pad, S, rb, Q, T, pl.splits, cols);
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
