// ffn_prefill.cu -- expert FFN for prefill-sized batches: a grouped GEMM on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory), fed by
// in-register int4 dequantisation.
//
// Sources: "Public Colibri Observation and Revision Ledger", "Exact
// Architecture and Data-Flow Reconstruction" (three-matrix experts at int4, a
// shared expert always used; the union groups the batch's tokens by expert).
// With ~128 tokens per routed expert the FFN is a real dense contraction.
//
// Design (GB300, sm_103a), one CTA per SM, persistent over work items:
//  * item = (expert unit, tile of output rows, tile of <= 160 tokens).
//    D[rows][tokens] = W[rows][K] * X[tokens][K]^T ("swap AB": the weights
//    are the M = 128 operand, the tokens the N operand).  Gate/up stacks 64
//    gate rows over the same 64 up rows in one A tile (an item is 64 rows of
//    h; one MMA per k16 serves both matrices; each TMEM subpartition holds 16
//    gate rows and the same 16 up rows); down takes 128 rows.  Every CTA builds the unit table
//    (expert, first sorted row, tokens, prefix of token tiles) in shared
//    memory once, so items are decoded without global loads.
//  * warp 0 (weight producer): TMA loads of the packed int4 rows + fp32 scales
//    (raw ring, 256 elements of a row per stage), running ahead of everything
//    else; warp 14 (token producer): TMA loads of the 16-bit token rows (operand
//    ring, 128 elements per stage, 128-byte swizzle).
//  * warps 6-13 (dequant: two groups of four warps, each taking one of the two
//    op stages of every raw stage, thread = row of the A tile):
//    nibbles -> fp16 (q * s) with an exact magic-exponent conversion
//    (0x6400|(n^8) = 1032 + q, then subtract) and one multiply, written straight
//    into tensor memory: the MMA reads A from there, so shared memory carries
//    only the raw nibbles and the token rows (the operand traffic that bounded
//    the kernel when A went through shared memory).  Nibble pairs come out as
//    (k, k+4); the token rows are stored with the same within-8 permutation,
//    so no reshuffle is needed.
//  * warp 1: allocates tensor memory; one lane issues tcgen05.mma (M = 128,
//    N = tokens rounded up to 16, K = 16 per instruction) into an fp32
//    accumulator, and commits stage releases.  The 512 TMEM columns hold two
//    accumulator buffers (so the MMAs of the next item run while the epilogue
//    drains the previous one) and three A stages.  Issuing an MMA, waiting for
//    a stage and committing its release each cost the single issuing thread
//    tens of cycles whatever N is, so stages are made long (8 MMAs each) and
//    N as large as the token tile allows.
//  * warps 2-5 (epilogue, one TMEM subpartition each): gate/up -> a gate lane
//    and its up lane swap one value per token pair with a shuffle and form
//    h = silu(g) * u in fp32; down -> y in fp32.
//  * precision: both GEMMs run on fp16 operands, weights fp16(q * s * 2^-e_r)
//    with e_r the binary exponent of the first group scale of weight row r (so
//    the row's first group has |s * 2^-e_r| in [1, 2) whatever the absolute
//    size of the scales), and activations scaled per row by a power of two so
//    that |v| < 2^14; both factors are applied to the fp32 result.  A group
//    scale more than 2^13 above or 2^14 below its row's first scale would
//    overflow or lose bits in fp16: it sets MOE_DEVERR_SCALE_RANGE.  fp32
//    accumulation, round to nearest even.  h is written in fp32, then a small kernel finds each
//    row's max |h| and writes the scaled fp16 rows the down GEMM reads.
//    (bf16 h and weights for the down GEMM would skip that pass, but their
//    rounding alone uses up the prefill tolerance of 2e-2 of the output RMS.)
//  * every wait is bounded; a timeout sets MOE_DEVERR_TIMEOUT, the roles stop
//    working but keep their loop structure, and tensor memory is freed.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

enum { kPGateUp = 0, kPDown = 1 };

constexpr int kPThreads = 480;                 // 15 warps
constexpr int kProdWarp = 0, kMmaWarp = 1, kEpiWarp0 = 2, kDeqWarp0 = 6, kBProdWarp = 14;
constexpr int kDeqThreads = 256;               // warps 6-13: two groups of 128 (A row each), alternate op stages
constexpr int kTileM = 128;                    // rows of the MMA's A tile
constexpr int kTileN = 160;                    // tokens per item
constexpr uint32_t kTmemCols = 512;
// Tensor memory: two accumulator buffers of kTileN columns, then the A tiles of
// the op stages (128 lanes x kOpK / 2 columns of packed fp16 each).
constexpr int kAccStride = kTileN;
constexpr int kACol0 = 2 * kTileN;

// Gate/up: the A tile stacks 64 rows of gate over the same 64 rows of up (one
// MMA per k16 computes both), so an item covers 64 rows of h and the
// accumulator needs only N columns.  Down: 128 rows of the down matrix.
// RAWK: elements of a row per raw stage -- 256 (128-byte row segments, 128B
// swizzle) when the reduction length allows it, else 128 (64 bytes, 64B swizzle).
// A raw stage feeds two op stages of RAWK / 2 elements, one per dequant group.
template <int MODE, int RAWK, int GS>
struct PCfg {
    static constexpr int kRawK = RAWK;
    static constexpr int kRowB = RAWK / 2;                     // packed bytes of a row per raw stage
    static constexpr int kChunks = RAWK / 32;                  // 16-byte chunks (= groups) per row
    static constexpr int kOpK = RAWK / 2;                      // reduction elements per op stage
    static constexpr int kOpPerRaw = 2;
    static constexpr int kCPO = kOpK / 32;                     // groups (16-byte chunks) per op stage
    static constexpr int kACols = kOpK / 2;                    // TMEM columns of one A stage
    static constexpr int kBChunks = kOpK / 64;                 // 128-byte token-row chunks per op stage
    static constexpr int kRawMats = MODE == kPGateUp ? 2 : 1;
    static constexpr int kRowsPerMat = kTileM / kRawMats;      // weight rows of one matrix per item
    static constexpr int kRawQ = kRowsPerMat * kRawK / 2;      // packed nibbles per matrix per raw stage
    static constexpr int kSpr = kRawK / GS;                     // scales of a row per raw stage
    static constexpr int kRawS = kRowsPerMat * kSpr * 4;
    static_assert(kSpr * 4 % 16 == 0, "a scale box row is a multiple of 16 bytes");
    static constexpr int kRawStage = kRawMats * (kRawQ + kRawS);   // 20 KB (RAWK 256) or 10 KB
    static constexpr int kRawStages = RAWK == 256 ? 4 : 6;
    static constexpr int kOpB = kTileN * kOpK * 2;             // fp16 token rows of a stage (A is in TMEM)
    static constexpr int kOpStage = kOpB;
    static constexpr int kOpStages = 3;
    static_assert(kACol0 + kOpStages * kACols <= (int)kTmemCols, "tensor memory budget");
    static constexpr int kRing = kRawStages * kRawStage + kOpStages * kOpStage;
    static_assert(kRawStage % 1024 == 0 && kOpStage % 1024 == 0, "alignment");
};

// Unit table in shared memory: unit 0 = shared expert (T tokens) when the
// launch includes it, then the uniq list; cum = prefix of token tiles over the
// units; zq = block of the layer view holding a routed expert's weights.
struct PUnit {
    int expert, row0, m, cum, zq;
};

__host__ __device__ constexpr size_t prefill_smem(int ring, int max_units)
{
    return 1024 + (size_t)ring + (size_t)(max_units + 1) * sizeof(PUnit);
}

struct PMaps {
    CUtensorMap q[2];   // packed weights: routed, shared; gate/up maps carry the matrix as a dimension
    CUtensorMap s[2];   // scales, same order
    CUtensorMap b;      // fp16 token rows (X_sorted or H_sorted), [rows][K]
};

struct PParams {
    const int32_t *offsets, *uniq, *n_uniq;
    // first-group scale of each weight row, read by the epilogue for the row's power-of-two
    // factor: expert block base + s_off0 + matrix * s_mat + row * s_row
    const float *s_routed, *s_shared;
    uint64_t s_expert, s_off0, s_mat;
    int s_row;
    const float *row_scale;       // power-of-two factor of each sorted activation row (x or h)
    float *h32;                   // gate/up: h [rows][f] fp32, natural order
    float *y_pair, *y_shared;     // down outputs
    uint16_t *y_pair16;           // down: routed outputs as bf16 instead of y_pair, when set
    const int32_t *slot_of;       // when set: routed expert e's weights are block slot_of[e] of the layer view
    int with_shared;              // 1: unit 0 is the shared expert; 0: the units are the uniq list only
    int32_t *err;
    int T, k, K, mtiles, out_rows;
    int n_experts, n_view;        // routed experts of the routing; expert blocks of the weight view
    int max_uniq;                 // capacity of the unit table beyond the shared expert: n_uniq is clamped to it
};

__device__ __forceinline__ int frag_pos8(int o) { return 2 * (o & 3) + (o >> 2); }

struct PItem {
    int expert;   // -1 = shared
    int zq;       // block of the layer view holding its weights (routed)
    int mtile;
    int tok0;     // first token of the tile within the unit
    int ntok;     // tokens in this tile (1..N)
    int row0;     // first row of the unit in the sorted activation rows
    int m;
};

// Build the unit table and the prefix of token tiles (N tokens per tile) for
// units 0 .. units - 1; tab[units].cum = total tiles.  All threads of the block.
template <int N>
__device__ void build_units(const PParams &p, int units, PUnit *tab)
{
    constexpr int kPer = 4;   // units per thread (blockDim.x * 4 >= E + 1)
    __shared__ int wsum[kPThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int tiles[kPer], tot = 0;
#pragma unroll
    for (int j = 0; j < kPer; j++) {
        const int u = tid * kPer + j;
        tiles[j] = 0;
        if (u < units) {
            PUnit t;
            if (u < p.with_shared) {
                t.expert = -1;
                t.row0 = p.T * p.k;
                t.m = p.T;
                t.zq = 0;
            } else {
                const int e = p.uniq[u - p.with_shared];
                t.expert = e;
                if (MOE_IN_BOUNDS(e >= 0 && e < p.n_experts, p.err)) {
                    t.row0 = p.offsets[e];
                    t.m = p.offsets[e + 1] - t.row0;
                    t.zq = p.slot_of ? p.slot_of[e] : e;
                    // a unit outside the pairs or the weight view gets no tokens
                    if (!MOE_IN_BOUNDS(t.row0 >= 0 && t.m >= 0 && t.row0 + t.m <= p.T * p.k && t.zq >= 0 &&
                                           t.zq < p.n_view,
                                       p.err))
                        t.m = 0;
                } else {
                    t.expert = 0;
                    t.row0 = t.m = t.zq = 0;
                }
            }
            tiles[j] = (t.m + N - 1) / N;
            tab[u] = t;
        }
        tot += tiles[j];
    }
    int inc = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off)
            inc += v;
    }
    if (lane == 31)
        wsum[warp] = inc;
    __syncthreads();
    int base = 0, all = 0;
    for (int w = 0; w < kPThreads / 32; w++) {
        base += w < warp ? wsum[w] : 0;
        all += wsum[w];
    }
    int run = base + inc - tot;
#pragma unroll
    for (int j = 0; j < kPer; j++) {
        const int u = tid * kPer + j;
        if (u < units)
            tab[u].cum = run;
        run += tiles[j];
    }
    if (tid == 0)
        tab[units].cum = all;
    __syncthreads();
}

template <int N>
__device__ __forceinline__ PItem decode_pitem(const PParams &p, const PUnit *tab, int units, int i)
{
    PItem it;
    const int ntg = i / p.mtiles;
    it.mtile = i - ntg * p.mtiles;
    // unit u: largest u with cum[u] <= ntg
    int lo = 0, hi = units;   // tab[hi].cum > ntg
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tab[mid].cum <= ntg)
            lo = mid;
        else
            hi = mid;
    }
    const PUnit t = tab[lo];
    it.expert = t.expert;
    it.zq = t.zq;
    it.row0 = t.row0;
    it.m = t.m;
    // the unit's tokens in ceil(m / N) balanced tiles (each <= N)
    const int nt = tab[lo + 1].cum - t.cum, j = ntg - t.cum;
    it.tok0 = j * t.m / nt;
    it.ntok = (j + 1) * t.m / nt - it.tok0;
    return it;
}

// Exact (q, q') from nibbles at bits 0-3 and 16-19: bf16 pair (136 + q, 136 + q')
// or fp16 pair (1032 + q, 1032 + q'), then the magic subtracted.
template <bool F16>
__device__ __forceinline__ uint32_t nib_q2(uint32_t w)
{
    uint32_t v, r;
    if (F16) {
        asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(v) : "r"(w), "r"(0x000F000Fu), "r"(0x64086408u));
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x64086408u));
    } else {
        asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(v) : "r"(w), "r"(0x000F000Fu), "r"(0x43084308u));
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x43084308u));
    }
    return r;
}

template <bool F16>
__device__ __forceinline__ uint32_t mul_x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    if (F16)
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    else
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Power-of-two shift of a weight row: s0 * 2^shift in [1, 2) for the row's first group scale s0,
// read from its fp32 exponent field (0 when s0 is 0 or not finite; clamped to [-126, 126] so that
// 2^shift and 2^-shift are normal fp32; subnormal s0 take 126).
__device__ __forceinline__ int row_shift(float s0)
{
    const uint32_t bits = __float_as_uint(s0) & 0x7fffffffu;
    const int biased = (int)(bits >> 23);
    if (bits == 0u || biased == 255)
        return 0;
    return min(max(127 - biased, -126), 126);
}

// 2^n for n in [-126, 127], exactly.
__device__ __forceinline__ float pow2i(int n) { return __uint_as_float((uint32_t)(127 + n) << 23); }

template <bool F16>
__device__ __forceinline__ uint32_t pack_scale(float s)
{
    if (F16) {
        const __half2 h = __float2half2_rn(s);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    const __nv_bfloat162 b = __float2bfloat162_rn(s);
    return *reinterpret_cast<const uint32_t *>(&b);
}

template <int MODE, int RAWK, int GS>
__global__ void __launch_bounds__(kPThreads, 1)
ffn_prefill_kernel(const __grid_constant__ PMaps maps, const PParams p)
{
    using C = PCfg<MODE, RAWK, GS>;
    constexpr int N = kTileN;
    constexpr bool kF16 = true;   // operand type of both GEMMs
    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t raw_full[C::kRawStages], raw_empty[C::kRawStages];
    __shared__ __align__(8) uint64_t op_full[C::kOpStages], op_empty[C::kOpStages];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const uint32_t raw_base = (smem_addr(dyn_smem) + 1023u) & ~1023u;
    const uint8_t *gen_base = dyn_smem + (raw_base - smem_addr(dyn_smem));
    const uint32_t op_base = raw_base + C::kRawStages * C::kRawStage;
    PUnit *tab = reinterpret_cast<PUnit *>(const_cast<uint8_t *>(gen_base) + C::kRing);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kRawStages; s++) {
            mbar_init(smem_addr(&raw_full[s]), 1);
            mbar_init(smem_addr(&raw_empty[s]), kDeqThreads);
        }
        for (int s = 0; s < C::kOpStages; s++) {
            mbar_init(smem_addr(&op_full[s]), kDeqThreads / 2 + 1);   // one dequant group + the token load
            mbar_init(smem_addr(&op_empty[s]), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(smem_addr(&acc_full[b]), 1);
            mbar_init(smem_addr(&acc_empty[b]), 128);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(&tmem_base_sh), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_sh;
    griddep_launch_dependents();
    griddep_wait();   // union and sorted activation rows come from earlier kernels

    const int units = min(max(*p.n_uniq, 0), p.max_uniq) + p.with_shared;
    build_units<N>(p, units, tab);
    const int n_items = tab[units].cum * p.mtiles;
    const int nraw = p.K / RAWK;

    if (warp == kProdWarp) {
        // ------------------------------------------------- weight producer
        if (lane == 0) {
            int rs = 0;
            uint32_t rph = 0;
            for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
                const PItem it = decode_pitem<N>(p, tab, units, i);
                const int z = it.expert < 0 ? 0 : it.zq;
                const int w = it.expert < 0 ? 1 : 0;
                const int wrow0 = it.mtile * C::kRowsPerMat;
                for (int r = 0; r < nraw; r++) {
                    if (!abort_flag && !mbar_wait(smem_addr(&raw_empty[rs]), rph ^ 1u)) {
                        atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                        abort_flag = 1;
                    }
                    if (!abort_flag) {
                        const uint32_t sb = raw_base + rs * C::kRawStage;
                        const uint32_t fb = smem_addr(&raw_full[rs]);
                        mbar_arrive_expect_tx(fb, C::kRawStage);
                        if (MODE == kPGateUp) {   // both matrices in one load each
                            tma_load_4d(sb, &maps.q[w], r * C::kRowB, wrow0, 0, z, fb);
                            tma_load_4d(sb + 2 * C::kRawQ, &maps.s[w], r * C::kSpr, wrow0, 0, z, fb);
                        } else {
                            tma_load_3d(sb, &maps.q[w], r * C::kRowB, wrow0, z, fb);
                            tma_load_3d(sb + C::kRawQ, &maps.s[w], r * C::kSpr, wrow0, z, fb);
                        }
                    }
                    if (++rs == C::kRawStages) {
                        rs = 0;
                        rph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == kBProdWarp) {
        // -------------------------------------------------- token producer
        if (lane == 0) {
            int os = 0;
            uint32_t oph = 0;
            for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
                const PItem it = decode_pitem<N>(p, tab, units, i);
                for (int kb = 0; kb < C::kOpPerRaw * nraw; kb++) {
                    if (!abort_flag && !mbar_wait(smem_addr(&op_empty[os]), oph ^ 1u)) {
                        atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                        abort_flag = 1;
                    }
                    if (!abort_flag) {
                        const uint32_t fb = smem_addr(&op_full[os]);
                        mbar_arrive_expect_tx(fb, C::kOpB);
                        tma_load_3d(op_base + os * C::kOpStage, &maps.b, 0, it.row0 + it.tok0, kb * C::kBChunks,
                                    fb);
                    }
                    if (++os == C::kOpStages) {
                        os = 0;
                        oph ^= 1u;
                    }
                }
            }
        }
    } else if (warp >= kDeqWarp0) {
        // -------------------------------------------------- dequantisation
        // two groups of four warps take alternate op stages (group g: op stage g of every raw
        // stage, i.e. its chunks g * kCPO .. g * kCPO + kCPO - 1), so each has two stage periods for
        // its work; a warp writes the 32 TMEM lanes of its subpartition: A rows 32 * (warp % 4) + lane
        // Gate/up: subpartition s holds gate rows 16s .. 16s + 15 in its lanes 0-15 and the same
        // up rows in lanes 16-31, so the epilogue pairs them with a shuffle.
        const int ar = ((warp & 3) << 5) | lane;        // row of the A tile
        const int g = (warp - kDeqWarp0) >> 2;          // 0 or 1
        const int mat = C::kRawMats == 2 ? ((lane >> 4) & 1) : 0;
        const int r = C::kRawMats == 2 ? (((warp & 3) << 4) | (lane & 15)) : ar;   // row within the matrix's tile
        const uint32_t tlane = tmem_base + ((uint32_t)((warp & 3) << 5) << 16);
        int rs = 0;
        uint32_t rph = 0;
        uint32_t kop = g;   // global index of this group's next op stage
        float rowfac = 1.0f;   // 2^shift of this thread's weight row (set from the item's first raw stage)
        bool range_bad = false;
        for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
            for (int rr = 0; rr < nraw; rr++) {
                if (!abort_flag && !mbar_wait(smem_addr(&raw_full[rs]), rph)) {
                    atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
                const uint8_t *rsb = gen_base + rs * C::kRawStage;
                // this row's packed bytes, swizzled (128B: 16-byte chunk c at c ^ (r & 7); 64B: at
                // c ^ ((r >> 1) & 3)); chunk c = group c of the raw stage
                const uint8_t *qrow = rsb + mat * C::kRawQ + r * C::kRowB;
                const float *srow = reinterpret_cast<const float *>(rsb + C::kRawMats * C::kRawQ + mat * C::kRawS +
                                                                    r * C::kSpr * 4);
                const int sw = RAWK == 256 ? (r & 7) : ((r >> 1) & 3);
                uint4 wv[C::kCPO];
                float sg[C::kCPO];
                if (rr == 0)
                    rowfac = pow2i(row_shift(srow[0]));
#pragma unroll
                for (int q = 0; q < C::kCPO; q++) {
                    const int c = g * C::kCPO + q;
                    wv[q] = *reinterpret_cast<const uint4 *>(qrow + ((c ^ sw) << 4));
                    sg[q] = srow[c * 32 / GS] * rowfac;   // exact: a power of two
                    const float a = fabsf(sg[q]);
                    range_bad |= a > 0.f && (a < 0x1p-14f || a > 8192.0f);
                }
                if (!abort_flag)
                    mbar_arrive(smem_addr(&raw_empty[rs]));   // the raw stage is in registers now
                if (++rs == C::kRawStages) {
                    rs = 0;
                    rph ^= 1u;
                }
                const int os = (int)(kop % C::kOpStages);
                const uint32_t oph = (kop / C::kOpStages) & 1u;
                kop += 2;
                if (!abort_flag && !mbar_wait(smem_addr(&op_empty[os]), oph ^ 1u)) {
                    atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
                if (!abort_flag) {
                    tc_fence_after();
#pragma unroll
                    for (int q = 0; q < C::kCPO; q++) {
                        const uint4 w4 = wv[q];
                        const uint32_t sfac = pack_scale<kF16>(sg[q]);
                        const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
                        uint32_t out[16];
#pragma unroll
                        for (int j = 0; j < 4; j++) {   // word j: elements 8j .. 8j+7 of the group
                            const uint32_t w = ws[j];
                            out[4 * j + 0] = mul_x2<kF16>(nib_q2<kF16>(w), sfac);          // (e0, e4)
                            out[4 * j + 1] = mul_x2<kF16>(nib_q2<kF16>(w >> 4), sfac);     // (e1, e5)
                            out[4 * j + 2] = mul_x2<kF16>(nib_q2<kF16>(w >> 8), sfac);     // (e2, e6)
                            out[4 * j + 3] = mul_x2<kF16>(nib_q2<kF16>(w >> 12), sfac);    // (e3, e7)
                        }
                        // k pairs of this group = columns q * 16 .. + 15 of the stage's A tile
                        tmem_st16(tlane + kACol0 + os * C::kACols + q * 16, out);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(smem_addr(&op_full[os]));
                }
            }
        }
        if (range_bad)
            atomicOr(p.err, MOE_DEVERR_SCALE_RANGE);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------ MMA issue
        // The whole warp runs the loop and one elected lane issues each MMA and commit: the
        // operands stay warp-uniform, which keeps the issue cost per instruction low.  The
        // next stage's readiness is tested before this stage's MMAs are issued, so the test's
        // latency overlaps them; only a stage found not ready is waited for (lane 0, then the
        // result is broadcast).  After a timeout (here or in another role) the warp stops
        // waiting and runs its loop to the end on whatever the stages hold.
        int os = 0, j = 0;
        uint32_t oph = 0, eph[2] = {0u, 0u};
        int stop = 0, rdy = 0;   // warp-uniform
        const int nkb = C::kOpPerRaw * nraw;
        for (int i = blockIdx.x; i < n_items; i += gridDim.x, j++) {
            const PItem it = decode_pitem<N>(p, tab, units, i);
            const int b = j & 1;
            const int n_mma = (it.ntok + 15) & ~15;
            const uint32_t idesc = kF16 ? idesc_f16_f32(kTileM, n_mma) : idesc_bf16_f32(kTileM, n_mma);
            stop |= abort_flag;
            int ok = 1;
            if (lane == 0 && !stop)
                ok = mbar_wait_or_abort(smem_addr(&acc_empty[b]), eph[b] ^ 1u, &abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
                stop = 1;
            }
            eph[b] ^= 1u;
            tc_fence_after();
            const uint32_t dcol = tmem_base + b * kAccStride;
            for (int kb = 0; kb < nkb; kb++) {
                if (!rdy && !stop) {
                    ok = lane == 0 ? (mbar_wait_or_abort(smem_addr(&op_full[os]), oph, &abort_flag) ? 1 : 0) : 1;
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) {
                        if (lane == 0) {
                            atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                            abort_flag = 1;
                        }
                        stop = 1;
                    }
                }
                tc_fence_after();
                const int nos = os + 1 == C::kOpStages ? 0 : os + 1;
                const uint32_t noph = nos == 0 ? oph ^ 1u : oph;
                const int nrdy = mbar_test(smem_addr(&op_full[nos]), noph) ? 1 : 0;   // the next stage
                const uint64_t bd = smem_desc_sw128(op_base + os * C::kOpStage);
                const uint32_t acol = tmem_base + kACol0 + os * C::kACols;
                // B: 128-byte chunk c of the token rows at c * kTileN * 128 bytes; k16 step
                // within it +32 bytes (descriptor units of 16 bytes)
#pragma unroll
                for (int k16 = 0; k16 < C::kOpK / 16; k16++)
                    umma_f16_ts_elect(dcol, acol + 8 * k16,
                                      bd + (uint64_t)((k16 >> 2) * (kTileN * 128 / 16) + 2 * (k16 & 3)), idesc,
                                      (kb > 0 || k16 > 0) ? 1u : 0u);
                umma_commit_elect(smem_addr(&op_empty[os]));
                os = nos;
                oph = noph;
                rdy = __shfl_sync(0xffffffffu, nrdy, 0);
            }
            umma_commit_elect(smem_addr(&acc_full[b]));
        }
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------- epilogue
        const int sub = warp & 3;                 // TMEM lanes 32*sub .. 32*sub+31 = A rows
        // the row factors of an item's tokens, loaded into this warp's slice before the item's
        // accumulator is waited for (one global round trip per item instead of one per chunk)
        __shared__ float epi_scale[4][kTileN];
        float *rsc = epi_scale[warp - kEpiWarp0];
        uint32_t fph[2] = {0u, 0u};
        int j = 0;
        for (int i = blockIdx.x; i < n_items; i += gridDim.x, j++) {
            const PItem it = decode_pitem<N>(p, tab, units, i);
            const int b = j & 1;
            __syncwarp();
            for (int q = lane; q < it.ntok; q += 32)
                rsc[q] = p.row_scale[it.row0 + it.tok0 + q];
            __syncwarp();
            // this lane's weight row and the power of two its dequantised weights were scaled by
            const int wrow = MODE == kPGateUp ? it.mtile * 64 + sub * 16 + (lane & 15) : it.mtile * kTileM + sub * 32 + lane;
            const int wmat = MODE == kPGateUp ? (lane >> 4) : 0;
            const float *sbase = it.expert < 0 ? p.s_shared : p.s_routed + (size_t)it.zq * p.s_expert;
            const float ef = pow2i(-row_shift(__ldg(sbase + p.s_off0 + (size_t)wmat * p.s_mat +
                                                    (size_t)wrow * p.s_row)));
            if (!abort_flag && !mbar_wait(smem_addr(&acc_full[b]), fph[b])) {
                atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                abort_flag = 1;
            }
            fph[b] ^= 1u;
            tc_fence_after();
            const uint32_t tl = tmem_base + ((uint32_t)(sub * 32) << 16) + b * kAccStride;
            for (int c0 = 0; c0 < it.ntok; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tl + c0, v);
                const int nj = min(16, it.ntok - c0);
                if (MODE == kPGateUp) {
                    // lane l < 16: gate row 16 sub + l; lane l + 16: the same up row.  Pair q of
                    // tokens (2q, 2q + 1): the gate lane forms h of token 2q, the up lane token 2q + 1,
                    // each taking the other's value with one shuffle.
                    tmem_wait_ld();
                    const int hi = lane >> 4;
                    const int hr = it.mtile * 64 + sub * 16 + (lane & 15);   // column of h
#pragma unroll
                    for (int q = 0; q < 8; q++) {
                        const float mine = __uint_as_float(hi ? v[2 * q + 1] : v[2 * q]) * ef;
                        const float other = __shfl_xor_sync(0xffffffffu,
                                                            __uint_as_float(hi ? v[2 * q] : v[2 * q + 1]) * ef, 16);
                        const int jj = 2 * q + hi;
                        if (jj < nj) {
                            const float rf = rsc[c0 + jj];
                            const float gv = (hi ? other : mine) * rf;
                            const float uv = (hi ? mine : other) * rf;
                            const float hv = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                            p.h32[(size_t)(it.row0 + it.tok0 + c0 + jj) * p.out_rows + hr] = hv;
                        }
                    }
                } else {
                    tmem_wait_ld();
                    const int orow = it.mtile * kTileM + sub * 32 + lane;
#pragma unroll
                    for (int jj = 0; jj < 16; jj++) {
                        if (jj >= nj)
                            break;
                        const float rf = rsc[c0 + jj];
                        const int tok = it.tok0 + c0 + jj;
                        const float yv = __uint_as_float(v[jj]) * ef * rf;
                        if (it.expert < 0)
                            p.y_shared[(size_t)tok * p.out_rows + orow] = yv;
                        else if (p.y_pair16)
                            p.y_pair16[(size_t)(it.row0 + tok) * p.out_rows + orow] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(yv));
                        else
                            p.y_pair[(size_t)(it.row0 + tok) * p.out_rows + orow] = yv;
                    }
                }
            }
            tc_fence_before();
            if (!abort_flag)
                mbar_arrive(smem_addr(&acc_empty[b]));
        }
    }

    // all roles done: free tensor memory (the MMA warp owns the allocation)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------- helpers ---

// Token rows in expert order as fp16, permuted within each 8 like the weights
// and scaled per row by a power of two 2^(14-e) (|value| < 2^14; row_scale
// keeps 2^(e-14)): row p < T*k is x[sorted_pair[p] / k], row T*k + t is x[t].
// pair_pos_kernel inverts sorted_pair over its n_valid = offsets[E] valid
// positions (pos[q] = p for q = sorted_pair[p]); token_rows_kernel then
// converts each token once (one block of 256 threads) and writes the result to
// the token's pair rows and its shared-expert row.  A slot that joined no
// group (an empty slot, id -1, or a bad id) has no valid position: pos[q] is
// then whatever an earlier call left there, so a slot counts as placed only
// when pos[q] is a valid position whose sorted_pair entry is q itself.
__global__ void __launch_bounds__(256)
pair_pos_kernel(const int32_t *__restrict__ sorted_pair, const int32_t *__restrict__ offsets, int E,
                int32_t *__restrict__ pos, int n_pairs, int32_t *err)
{
    griddep_launch_dependents();
    griddep_wait();
    const int p = blockIdx.x * 256 + threadIdx.x;
    if (p < offsets[E]) {
        const int q = sorted_pair[p];
        if (MOE_IN_BOUNDS(q >= 0 && q < n_pairs && p < n_pairs, err))
            pos[q] = p;
    }
    (void)n_pairs;
    (void)err;
}

__global__ void __launch_bounds__(256)
token_rows_kernel(const float *__restrict__ x, const int32_t *__restrict__ pos,
                  const int32_t *__restrict__ sorted_pair, const int32_t *__restrict__ offsets, int E, int T,
                  int k, int K, uint16_t *__restrict__ out, float *__restrict__ row_scale)
{
    __shared__ float wmax[8];
    __shared__ int dst[33];
    griddep_launch_dependents();
    griddep_wait();
    const int t = blockIdx.x;
    if (threadIdx.x < k) {
        const int q = t * k + threadIdx.x;
        const int v = pos[q];
        dst[threadIdx.x] = (v >= 0 && v < offsets[E] && sorted_pair[v] == q) ? v : -1;
    } else if (threadIdx.x == k) {
        dst[k] = T * k + t;
    }
    const float *xr = x + (size_t)t * K;
    float mx = 0.f;
    for (int i = threadIdx.x; i < K / 4; i += 256) {
        const float4 v = reinterpret_cast<const float4 *>(xr)[i];
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0)
        wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0.f;
#pragma unroll
    for (int w = 0; w < 8; w++)
        mx = fmaxf(mx, wmax[w]);
    int e = 0;
    frexpf(mx, &e);
    const float up = mx > 0.f ? ldexpf(1.0f, 14 - e) : 1.0f;
    if (threadIdx.x <= k && dst[threadIdx.x] >= 0)
        row_scale[dst[threadIdx.x]] = mx > 0.f ? ldexpf(1.0f, e - 14) : 1.0f;
    for (int c = threadIdx.x; c < K / 8; c += 256) {
        const float4 *sp = reinterpret_cast<const float4 *>(xr + c * 8);
        const float4 a = sp[0], b = sp[1];
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        __align__(16) uint16_t o[8];
#pragma unroll
        for (int el = 0; el < 8; el++)
            o[frag_pos8(el)] = __half_as_ushort(__float2half_rn(v[el] * up));
        const uint4 ov = *reinterpret_cast<const uint4 *>(o);
        for (int j = 0; j <= k; j++)
            if (dst[j] >= 0)
                *reinterpret_cast<uint4 *>(out + (size_t)dst[j] * K + c * 8) = ov;
    }
}

// h rows (fp32) -> fp16 rows scaled by 2^(14-e), e from the row's max |h|,
// permuted within each 8 like the weights; h_scale keeps 2^(e-14).  One block
// of 256 threads per row: a pass for the max, a pass to convert (the row is
// then in L1).
__global__ void __launch_bounds__(256)
h_to_f16_kernel(const float *__restrict__ h32, int K, uint16_t *__restrict__ out, float *__restrict__ h_scale)
{
    __shared__ float wmax[8];
    griddep_launch_dependents();
    griddep_wait();
    const int r = blockIdx.x;
    const float *hr = h32 + (size_t)r * K;
    float mx = 0.f;
    for (int i = threadIdx.x; i < K / 4; i += 256) {
        const float4 v = reinterpret_cast<const float4 *>(hr)[i];
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0)
        wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0.f;
#pragma unroll
    for (int w = 0; w < 8; w++)
        mx = fmaxf(mx, wmax[w]);
    int e = 0;
    frexpf(mx, &e);
    const float up = mx > 0.f ? ldexpf(1.0f, 14 - e) : 1.0f;
    if (threadIdx.x == 0)
        h_scale[r] = mx > 0.f ? ldexpf(1.0f, e - 14) : 1.0f;
    for (int c = threadIdx.x; c < K / 8; c += 256) {
        const float4 *sp = reinterpret_cast<const float4 *>(hr + c * 8);
        const float4 a = sp[0], b = sp[1];
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        __align__(16) uint16_t o[8];
#pragma unroll
        for (int el = 0; el < 8; el++)
            o[frag_pos8(el)] = __half_as_ushort(__float2half_rn(v[el] * up));
        *reinterpret_cast<uint4 *>(out + (size_t)r * K + c * 8) = *reinterpret_cast<const uint4 *>(o);
    }
}

// 16-bit token rows [rows][K] as (64 elements, row, 128-byte chunk): one load
// brings kTileN rows x `chunks` chunks, chunk-major, 128-byte swizzled.
int make_tmap_rows(CUtensorMap *m, const uint16_t *base, int K, size_t rows, int chunks)
{
    const uint64_t dim[3] = {64, (uint64_t)rows, (uint64_t)K / 64};
    const uint64_t str[2] = {(uint64_t)K * 2, 128};
    const uint32_t box[3] = {64, (uint32_t)kTileN, (uint32_t)chunks};
    return make_tmap_nd(m, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, dim, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int MODE, int RAWK, int GS>
int launch_prefill_one(const PMaps &maps, const PParams &prm, int max_units, cudaStream_t s)
{
    using C = PCfg<MODE, RAWK, GS>;
    auto kern = ffn_prefill_kernel<MODE, RAWK, GS>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return MOE_ERR_CUDA;
    // per device and instantiation, once (several host threads may get here together: a second
    // attribute call is harmless, and the flag is atomic)
    static std::atomic<int> configured[64];
    if (!configured[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)prefill_smem(C::kRing, 1025)) != cudaSuccess)
            return MOE_ERR_CUDA;
        configured[dev].store(1, std::memory_order_release);
    }
    return launch_pdl(kern, sm_count(dev), kPThreads, prefill_smem(C::kRing, max_units), s, maps, prm);
}

}  // namespace

namespace {

struct PrefillScratch {
    uint16_t *x16, *h16;   // scaled fp16 x and h rows
    float *x_scale, *h_scale, *h32;
    int32_t *pos;          // pair position of each (token, slot)
};

size_t prefill_layout(int T, int k, int d, int f, uint8_t *base, PrefillScratch *o)
{
    const size_t rows = (size_t)T * k + T;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + off : nullptr;
        off += (bytes + 255) & ~(size_t)255;
        return p;
    };
    PrefillScratch s{};
    s.x16 = reinterpret_cast<uint16_t *>(take(rows * d * 2));
    s.h16 = reinterpret_cast<uint16_t *>(take(rows * f * 2));
    s.h32 = reinterpret_cast<float *>(take(rows * f * 4));
    s.x_scale = reinterpret_cast<float *>(take(rows * 4));
    s.h_scale = reinterpret_cast<float *>(take(rows * 4));
    s.pos = reinterpret_cast<int32_t *>(take((size_t)T * k * 4));
    if (o)
        *o = s;
    return off;
}

}  // namespace

size_t prefill_scratch_bytes(int T, int k, int d, int f) { return prefill_layout(T, k, d, f, nullptr, nullptr); }

int launch_ffn_prefill(const PrefillFfnArgs &a, cudaStream_t s)
{
    const moe_layer_int4 &w = *a.w;
    const int d = w.d, f = w.f, E = w.E, G = w.G, T = a.T, k = a.k;
    const uint64_t qb = (uint64_t)moe_expert_q_bytes(d, f);
    const uint64_t sc = (uint64_t)moe_expert_s_count(d, f, G);
    const size_t rows = (size_t)T * k + T;
    PrefillScratch ps{};
    prefill_layout(T, k, d, f, static_cast<uint8_t *>(a.scratch), &ps);
    uint16_t *x_sorted = ps.x16;
    uint16_t *h_sorted = ps.h16;
    float *row_scale = ps.x_scale;
    int rc = MOE_OK;

    // fp16 token rows: each token converted once and written to its pair rows and shared row
    const int E_off = a.n_experts > 0 ? a.n_experts : E;   // offsets[E_off] = the placed pairs
    rc = launch_pdl(pair_pos_kernel, (T * k + 255) / 256, 256, 0, s, a.sorted_pair, a.offsets, E_off, ps.pos, T * k,
                    a.err);
    if (rc == MOE_OK)
        rc = launch_pdl(token_rows_kernel, T, 256, 0, s, a.x, (const int32_t *)ps.pos, a.sorted_pair, a.offsets,
                        E_off, T, k, d, x_sorted, row_scale);
    if (rc != MOE_OK)
        return rc;

    const uint8_t *qs[2] = {w.q_base, w.shared_q};
    const float *ss[2] = {w.s_base, w.shared_s};
    const uint64_t outer[2] = {(uint64_t)E, 1};

    // ---- gate / up: (row bytes, row, matrix, expert) maps, both matrices per load
    PMaps gm{};
    for (int i = 0; i < 2 && rc == MOE_OK; i++) {
        const uint64_t q_dim[4] = {(uint64_t)d / 2, (uint64_t)f, 2, outer[i]};
        const uint64_t q_str[3] = {(uint64_t)d / 2, (uint64_t)f * d / 2, qb};
        const uint32_t q_box[4] = {128, (uint32_t)PCfg<kPGateUp, 256, 32>::kRowsPerMat, 2, 1};
        const uint64_t s_dim[4] = {(uint64_t)d / G, (uint64_t)f, 2, outer[i]};
        const uint64_t s_str[3] = {(uint64_t)(d / G) * 4, (uint64_t)f * (d / G) * 4, sc * 4};
        const uint32_t s_box[4] = {(uint32_t)(256 / G), (uint32_t)PCfg<kPGateUp, 256, 32>::kRowsPerMat, 2, 1};
        rc |= make_tmap_nd(&gm.q[i], qs[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, q_dim, q_str, q_box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
        rc |= make_tmap_nd(&gm.s[i], ss[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, s_dim, s_str, s_box,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    rc |= make_tmap_rows(&gm.b, x_sorted, d, rows, PCfg<kPGateUp, 256, 32>::kBChunks);
    if (rc != MOE_OK)
        return MOE_ERR_INVALID_ARG;
    PParams pg{};
    pg.offsets = a.offsets;
    pg.uniq = a.uniq;
    pg.n_uniq = a.n_uniq;
    pg.s_routed = w.s_base;
    pg.s_shared = w.shared_s;
    pg.s_expert = sc;
    pg.s_off0 = 0;
    pg.s_mat = (uint64_t)f * (d / G);
    pg.s_row = d / G;
    pg.row_scale = row_scale;
    pg.h32 = ps.h32;
    pg.slot_of = a.slot_of;
    pg.with_shared = a.with_shared;
    pg.err = a.err;
    pg.T = T;
    pg.k = k;
    pg.K = d;
    pg.mtiles = f / PCfg<kPGateUp, 256, 32>::kRowsPerMat;
    pg.out_rows = f;
    pg.n_experts = E_off;
    pg.n_view = E;
    const int max_units = (E < T * k ? E : T * k) + 1;
    pg.max_uniq = max_units - 1;
    // d is a multiple of 256
    rc = G == 64 ? launch_prefill_one<kPGateUp, 256, 64>(gm, pg, max_units, s)
                 : launch_prefill_one<kPGateUp, 256, 32>(gm, pg, max_units, s);
    if (rc == MOE_OK)
        rc = launch_pdl(h_to_f16_kernel, (int)rows, 256, 0, s, (const float *)ps.h32, f, h_sorted, ps.h_scale);
    if (rc != MOE_OK)
        return rc;

    // ---- down
    const int dn_rawk = f % 256 == 0 ? 256 : 128;
    if (dn_rawk / G * 4 % 16 != 0)
        return MOE_ERR_UNSUPPORTED;   // G = 64 needs f a multiple of 256 (a scale box row of 16 bytes)
    PMaps dm{};
    for (int i = 0; i < 2 && rc == MOE_OK; i++) {
        rc |= make_tmap_3d(&dm.q[i], qs[i] + (size_t)f * d, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, f / 2, d, outer[i],
                           f / 2, qb, dn_rawk / 2, kTileM,
                           dn_rawk == 256 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
        rc |= make_tmap_3d(&dm.s[i], ss[i] + (size_t)2 * f * d / G, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, f / G, d,
                           outer[i], (uint64_t)(f / G) * 4, sc * 4, dn_rawk / G, kTileM, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    rc |= make_tmap_rows(&dm.b, h_sorted, f, rows, dn_rawk == 256 ? PCfg<kPDown, 256, 32>::kBChunks
                                                                   : PCfg<kPDown, 128, 32>::kBChunks);
    if (rc != MOE_OK)
        return MOE_ERR_INVALID_ARG;
    PParams pd = pg;
    pd.s_off0 = (uint64_t)2 * f * (d / G);
    pd.s_mat = 0;
    pd.s_row = f / G;
    pd.h32 = nullptr;
    pd.row_scale = ps.h_scale;
    pd.y_pair = a.y_pair;
    pd.y_pair16 = a.y_pair16;
    pd.y_shared = a.y_shared;
    pd.K = f;
    pd.mtiles = d / kTileM;
    pd.out_rows = d;
    if (dn_rawk == 256)
        return G == 64 ? launch_prefill_one<kPDown, 256, 64>(dm, pd, max_units, s)
                       : launch_prefill_one<kPDown, 256, 32>(dm, pd, max_units, s);
    return launch_prefill_one<kPDown, 128, 32>(dm, pd, max_units, s);
}

}  // namespace moe
