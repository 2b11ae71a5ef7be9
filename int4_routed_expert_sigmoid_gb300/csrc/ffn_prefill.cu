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
//  * item = (expert unit, 128-row tile of the output matrix, tile of <= 256
//    tokens).  D[rows][tokens] = W[rows][K] * X[tokens][K]^T ("swap AB": the
//    weights are the M = 128 operand, the tokens the N <= 256 operand).
//  * warp 0 (producer): TMA loads of the packed int4 rows + fp32 scales
//    (raw ring, k-blocks of 128) and of the bf16 token rows (operand ring,
//    k-blocks of 64, 128-byte swizzle).
//  * warps 6-9 (dequant, thread = weight row): nibbles -> fp16 / bf16 (q * s)
//    with an exact magic-exponent conversion (fp16: 0x6400|(n^8) = 1032 + q;
//    bf16: 0x4300|(n^8) = 136 + q; then subtract) and one multiply, written into the operand stage in the 128B-swizzled K-major
//    layout the MMA reads.  Nibble pairs come out as (k, k+4); the token rows
//    are stored with the same within-8 permutation, so no reshuffle is needed.
//  * warp 1: allocates tensor memory; one lane issues tcgen05.mma (M = 128,
//    N = tokens rounded up to 16, K = 16 per instruction) into fp32
//    accumulators (gate and up: two), and commits stage releases.
//  * warps 2-5 (epilogue, one TMEM subpartition each): gate/up ->
//    h = silu(g) * u in fp32 plus the per-token max |h|; down -> y in fp32.
//  * precision: both GEMMs run on fp16 operands, weights fp16(q * s) and
//    activations scaled per row by a power of two so that |v| < 2^14 (the
//    factor is applied to the fp32 result); fp32 accumulation, round to
//    nearest even.  h is written in fp32 with a per-token max, then turned
//    into scaled fp16 rows by a small kernel before the down GEMM.
//  * every wait is bounded; a timeout sets MOE_DEVERR_TIMEOUT, the roles stop
//    working but keep their loop structure, and tensor memory is freed.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

enum { kPGateUp = 0, kPDown = 1 };

constexpr int kPThreads = 320;                 // 10 warps
constexpr int kProdWarp = 0, kMmaWarp = 1, kEpiWarp0 = 2, kDeqWarp0 = 6;
constexpr int kTileM = 128, kTileN = 256;
constexpr int kRawK = 128, kOpK = 64;
constexpr uint32_t kTmemCols = 512;

template <int MODE>
struct PCfg {
    static constexpr int kMats = MODE == kPGateUp ? 2 : 1;
    static constexpr int kRawQ = kTileM * kRawK / 2;        // 8 KB of packed nibbles per matrix
    static constexpr int kRawS = kTileM * (kRawK / 32) * 4; // 2 KB of scales per matrix
    static constexpr int kRawStage = kMats * (kRawQ + kRawS);
    static constexpr int kRawStages = MODE == kPGateUp ? 3 : 4;
    static constexpr int kOpA = kTileM * kOpK * 2;          // 16 KB bf16 per matrix
    static constexpr int kOpB = kTileN * kOpK * 2;          // 32 KB bf16 of token rows
    static constexpr int kOpStage = kMats * kOpA + kOpB;
    static constexpr int kOpStages = MODE == kPGateUp ? 2 : 3;
    static constexpr int kSmem = 1024 + kRawStages * kRawStage + kOpStages * kOpStage;
    static_assert(kRawStage % 1024 == 0 && kOpStage % 1024 == 0, "alignment");
};

struct PMaps {
    CUtensorMap q[4];   // packed weights: routed mat0, routed mat1, shared mat0, shared mat1
    CUtensorMap s[4];   // scales, same order
    CUtensorMap b;      // bf16 token rows (X_sorted or H_sorted), [rows][K]
};

struct PParams {
    const int32_t *offsets, *uniq, *n_uniq;
    const float *row_scale;       // power-of-two factor of each sorted activation row (x or h)
    const int32_t *cum;           // [n_uniq + 2] prefix of token tiles per unit (unit 0 = shared)
    float *h32;                   // gate/up: h [rows][f] fp32, natural order
    unsigned int *hmax;           // gate/up: per-row max |h| (fp32 bits)
    float *y_pair, *y_shared;     // down outputs
    int32_t *err;
    int T, k, K, mtiles, out_rows;
};

__device__ __forceinline__ int frag_pos8(int o) { return 2 * (o & 3) + (o >> 2); }

struct PItem {
    int expert;   // -1 = shared
    int mtile;
    int tok0;     // first token of the tile within the unit
    int ntok;     // tokens in this tile (1..256)
    int row0;     // first row of the unit in the sorted activation rows
    int m;
};

__device__ __forceinline__ PItem decode_pitem(const PParams &p, int i)
{
    PItem it;
    const int ntg = i / p.mtiles;
    it.mtile = i - ntg * p.mtiles;
    // unit u: largest u with cum[u] <= ntg
    int lo = 0, hi = *p.n_uniq + 1;   // cum[hi] > ntg
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.cum[mid] <= ntg)
            lo = mid;
        else
            hi = mid;
    }
    const int u = lo;
    if (u == 0) {
        it.expert = -1;
        it.m = p.T;
        it.row0 = p.T * p.k;
    } else {
        it.expert = p.uniq[u - 1];
        it.row0 = p.offsets[it.expert];
        it.m = p.offsets[it.expert + 1] - it.row0;
    }
    it.tok0 = (ntg - p.cum[u]) * kTileN;
    it.ntok = min(kTileN, it.m - it.tok0);
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

template <int MODE>
__global__ void __launch_bounds__(kPThreads, 1)
ffn_prefill_kernel(const __grid_constant__ PMaps maps, const PParams p)
{
    using C = PCfg<MODE>;
    constexpr bool kF16 = true;   // operand type of both GEMMs
    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t raw_full[C::kRawStages], raw_empty[C::kRawStages];
    __shared__ __align__(8) uint64_t op_full[C::kOpStages], op_empty[C::kOpStages];
    __shared__ __align__(8) uint64_t acc_full, acc_empty;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const uint32_t raw_base = (smem_addr(dyn_smem) + 1023u) & ~1023u;
    const uint8_t *gen_base = dyn_smem + (raw_base - smem_addr(dyn_smem));
    const uint32_t op_base = raw_base + C::kRawStages * C::kRawStage;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kRawStages; s++) {
            mbar_init(smem_addr(&raw_full[s]), 1);
            mbar_init(smem_addr(&raw_empty[s]), 128);
        }
        for (int s = 0; s < C::kOpStages; s++) {
            mbar_init(smem_addr(&op_full[s]), 128 + 1);
            mbar_init(smem_addr(&op_empty[s]), 1);
        }
        mbar_init(smem_addr(&acc_full), 1);
        mbar_init(smem_addr(&acc_empty), 128);
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
    griddep_wait();   // union, plan and sorted activation rows come from earlier kernels

    const int n_units_tiles = p.cum[*p.n_uniq + 1];
    const int n_items = n_units_tiles * p.mtiles;
    const int nraw = p.K / kRawK;

    if (warp == kProdWarp) {
        // -------------------------------------------------------- producer
        if (lane == 0) {
            int rs = 0, os = 0;
            uint32_t rph = 0, oph = 0;
            for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
                const PItem it = decode_pitem(p, i);
                const int z = it.expert < 0 ? 0 : it.expert;
                const int mb = it.expert < 0 ? 2 : 0;
                const int wrow0 = it.mtile * kTileM;
                for (int r = 0; r < nraw; r++) {
                    if (!abort_flag && !mbar_wait(smem_addr(&raw_empty[rs]), rph ^ 1u)) {
                        atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                        abort_flag = 1;
                    }
                    if (!abort_flag) {
                        const uint32_t sb = raw_base + rs * C::kRawStage;
                        const uint32_t fb = smem_addr(&raw_full[rs]);
                        mbar_arrive_expect_tx(fb, C::kRawStage);
                        for (int mat = 0; mat < C::kMats; mat++) {
                            tma_load_3d(sb + mat * C::kRawQ, &maps.q[mb + mat], r * (kRawK / 2), wrow0, z, fb);
                            tma_load_3d(sb + C::kMats * C::kRawQ + mat * C::kRawS, &maps.s[mb + mat],
                                        r * (kRawK / 32), wrow0, z, fb);
                        }
                    }
                    if (++rs == C::kRawStages) {
                        rs = 0;
                        rph ^= 1u;
                    }
                    for (int h = 0; h < 2; h++) {
                        if (!abort_flag && !mbar_wait(smem_addr(&op_empty[os]), oph ^ 1u)) {
                            atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                            abort_flag = 1;
                        }
                        if (!abort_flag) {
                            const uint32_t fb = smem_addr(&op_full[os]);
                            mbar_arrive_expect_tx(fb, C::kOpB);
                            tma_load_2d(op_base + os * C::kOpStage + C::kMats * C::kOpA, &maps.b,
                                        (2 * r + h) * kOpK, it.row0 + it.tok0, fb);
                        }
                        if (++os == C::kOpStages) {
                            os = 0;
                            oph ^= 1u;
                        }
                    }
                }
            }
        }
    } else if (warp >= kDeqWarp0) {
        // -------------------------------------------------- dequantisation
        const int row = threadIdx.x - kDeqWarp0 * 32;   // 0..127
        int rs = 0, os = 0;
        uint32_t rph = 0, oph = 0;
        for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
            for (int r = 0; r < nraw; r++) {
                if (!abort_flag && !mbar_wait(smem_addr(&raw_full[rs]), rph)) {
                    atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
                const uint8_t *rsb = gen_base + rs * C::kRawStage;
                for (int h = 0; h < 2; h++) {
                    if (!abort_flag && !mbar_wait(smem_addr(&op_empty[os]), oph ^ 1u)) {
                        atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                        abort_flag = 1;
                    }
                    if (!abort_flag) {
                        uint8_t *osb = const_cast<uint8_t *>(gen_base) + (op_base - raw_base) + os * C::kOpStage;
#pragma unroll
                        for (int mat = 0; mat < C::kMats; mat++) {
                            // this row's 64 packed bytes, 64B-swizzled: 16-byte chunk c at (c ^ ((row >> 1) & 3))
                            const uint8_t *qrow = rsb + mat * C::kRawQ + row * 64;
                            const float4 sc = *reinterpret_cast<const float4 *>(rsb + C::kMats * C::kRawQ +
                                                                               mat * C::kRawS + row * 16);
                            const float s_lo = h ? sc.z : sc.x, s_hi = h ? sc.w : sc.y;
                            const uint32_t sbl = pack_scale<kF16>(s_lo), sbh = pack_scale<kF16>(s_hi);
                            uint8_t *arow = osb + mat * C::kOpA + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
                            for (int cc = 0; cc < 2; cc++) {   // two 16-byte chunks = 32 elements = one group
                                const int c = 2 * h + cc;
                                const uint4 wv = *reinterpret_cast<const uint4 *>(qrow + ((c ^ ((row >> 1) & 3)) << 4));
                                const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
                                const uint32_t sfac = cc ? sbh : sbl;
#pragma unroll
                                for (int j = 0; j < 4; j++) {   // word j: elements 8j .. 8j+7 of the group
                                    const uint32_t w = ws[j];
                                    uint4 out;
                                    out.x = mul_x2<kF16>(nib_q2<kF16>(w), sfac);          // (e0, e4)
                                    out.y = mul_x2<kF16>(nib_q2<kF16>(w >> 4), sfac);     // (e1, e5)
                                    out.z = mul_x2<kF16>(nib_q2<kF16>(w >> 8), sfac);     // (e2, e6)
                                    out.w = mul_x2<kF16>(nib_q2<kF16>(w >> 12), sfac);    // (e3, e7)
                                    const int chunk = cc * 4 + j;                   // 8-element chunk of the 64
                                    *reinterpret_cast<uint4 *>(arow + ((chunk ^ (row & 7)) << 4)) = out;
                                }
                            }
                        }
                        fence_proxy_async_smem();
                        mbar_arrive(smem_addr(&op_full[os]));
                    }
                    if (++os == C::kOpStages) {
                        os = 0;
                        oph ^= 1u;
                    }
                }
                if (!abort_flag)
                    mbar_arrive(smem_addr(&raw_empty[rs]));
                if (++rs == C::kRawStages) {
                    rs = 0;
                    rph ^= 1u;
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------ MMA issue
        if (lane == 0) {
            int os = 0;
            uint32_t oph = 0, aph = 0;
            for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
                const PItem it = decode_pitem(p, i);
                const int n_mma = (it.ntok + 15) & ~15;
                const uint32_t idesc = kF16 ? idesc_f16_f32(kTileM, n_mma) : idesc_bf16_f32(kTileM, n_mma);
                if (!abort_flag && !mbar_wait(smem_addr(&acc_empty), aph ^ 1u)) {
                    atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
                aph ^= 1u;
                tc_fence_after();
                for (int kb = 0; kb < 2 * nraw; kb++) {
                    if (!abort_flag && !mbar_wait(smem_addr(&op_full[os]), oph)) {
                        atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                        abort_flag = 1;
                    }
                    tc_fence_after();
                    if (!abort_flag) {
                        const uint32_t sb = op_base + os * C::kOpStage;
#pragma unroll
                        for (int k16 = 0; k16 < kOpK / 16; k16++) {
                            const uint64_t bd = smem_desc_sw128(sb + C::kMats * C::kOpA + k16 * 32);
                            const uint32_t acc = (kb > 0 || k16 > 0) ? 1u : 0u;
#pragma unroll
                            for (int mat = 0; mat < C::kMats; mat++)
                                umma_f16(tmem_base + mat * kTileN, smem_desc_sw128(sb + mat * C::kOpA + k16 * 32), bd,
                                         idesc, acc);
                        }
                        umma_commit(smem_addr(&op_empty[os]));
                    }
                    if (++os == C::kOpStages) {
                        os = 0;
                        oph ^= 1u;
                    }
                }
                if (!abort_flag)
                    umma_commit(smem_addr(&acc_full));
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------- epilogue
        const int sub = warp & 3;                 // TMEM lanes 32*sub .. 32*sub+31
        const int row = sub * 32 + lane;          // output row within the tile
        uint32_t aph = 0;
        for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
            const PItem it = decode_pitem(p, i);
            if (!abort_flag && !mbar_wait(smem_addr(&acc_full), aph)) {
                atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                abort_flag = 1;
            }
            aph ^= 1u;
            tc_fence_after();
            if (!abort_flag) {
                const int orow = it.mtile * kTileM + row;
                const uint32_t tl = tmem_base + ((uint32_t)(sub * 32) << 16);
                for (int c0 = 0; c0 < it.ntok; c0 += 16) {
                    uint32_t g[16], u[16];
                    tmem_ld16(tl + c0, g);
                    if (MODE == kPGateUp)
                        tmem_ld16(tl + kTileN + c0, u);
                    tmem_wait_ld();
                    const int nj = min(16, it.ntok - c0);
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        if (j >= nj)
                            break;
                        const int tok = it.tok0 + c0 + j;
                        const float rf = p.row_scale[it.row0 + tok];
                        const float gv = __uint_as_float(g[j]) * rf;
                        if (MODE == kPGateUp) {
                            const float uv = __uint_as_float(u[j]) * rf;
                            const float hv = gv / (1.0f + expf(-gv)) * uv;
                            p.h32[(size_t)(it.row0 + tok) * p.out_rows + orow] = hv;
                            float mx = fabsf(hv);
#pragma unroll
                            for (int off = 16; off > 0; off >>= 1)
                                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                            if (lane == 0)
                                atomicMax(p.hmax + it.row0 + tok, __float_as_uint(mx));
                        } else {
                            float *dst = it.expert < 0 ? p.y_shared + (size_t)tok * p.out_rows
                                                       : p.y_pair + (size_t)(it.row0 + tok) * p.out_rows;
                            dst[orow] = gv;
                        }
                    }
                }
            }
            tc_fence_before();
            if (!abort_flag)
                mbar_arrive(smem_addr(&acc_empty));
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
// One block of 256 threads per row.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const float *__restrict__ x, const int32_t *__restrict__ sorted_pair, int T, int k, int K,
                   uint16_t *__restrict__ out, float *__restrict__ row_scale, unsigned int *__restrict__ hmax)
{
    __shared__ float wmax[8];
    griddep_launch_dependents();
    griddep_wait();
    const int r = blockIdx.x;
    const int src = r < T * k ? sorted_pair[r] / k : r - T * k;
    const float *xr = x + (size_t)src * K;
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
    if (threadIdx.x == 0) {
        row_scale[r] = mx > 0.f ? ldexpf(1.0f, e - 14) : 1.0f;
        hmax[r] = 0u;
    }
    for (int c = threadIdx.x; c < K / 8; c += 256) {
        const float4 *sp = reinterpret_cast<const float4 *>(xr + c * 8);
        const float4 a = sp[0], b = sp[1];
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        __align__(16) uint16_t o[8];
#pragma unroll
        for (int el = 0; el < 8; el++)
            o[frag_pos8(el)] = __half_as_ushort(__float2half_rn(v[el] * up));
        *reinterpret_cast<uint4 *>(out + (size_t)r * K + c * 8) = *reinterpret_cast<const uint4 *>(o);
    }
}

// h rows (fp32) -> fp16 rows scaled by 2^(14-e), e from the row's max |h|,
// permuted within each 8; h_scale keeps 2^(e-14).  One block per row.
__global__ void __launch_bounds__(256)
h_to_f16_kernel(const float *__restrict__ h32, const unsigned int *__restrict__ hmax, int K,
                uint16_t *__restrict__ out, float *__restrict__ h_scale)
{
    griddep_launch_dependents();
    griddep_wait();
    const int r = blockIdx.x;
    const float mx = __uint_as_float(hmax[r]);
    int e = 0;
    frexpf(mx, &e);
    const float up = mx > 0.f ? ldexpf(1.0f, 14 - e) : 1.0f;
    if (threadIdx.x == 0)
        h_scale[r] = mx > 0.f ? ldexpf(1.0f, e - 14) : 1.0f;
    const float *hr = h32 + (size_t)r * K;
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

// Prefix of 256-token tiles per unit (unit 0 = shared expert with T tokens,
// unit u >= 1 = uniq[u-1]); cum has n_uniq + 2 entries.
__global__ void prefill_plan_kernel(const int32_t *__restrict__ offsets, const int32_t *__restrict__ uniq,
                                    const int32_t *__restrict__ n_uniq, int T, int32_t *__restrict__ cum)
{
    griddep_wait();
    if (threadIdx.x >= 32)
        return;
    const int lane = threadIdx.x;
    const int nu = *n_uniq + 1;
    int carry = 0;
    for (int u0 = 0; u0 < nu; u0 += 32) {
        const int u = u0 + lane;
        int nt = 0;
        if (u < nu) {
            const int m = u == 0 ? T : offsets[uniq[u - 1] + 1] - offsets[uniq[u - 1]];
            nt = (m + kTileN - 1) / kTileN;
        }
        int inc = nt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off)
                inc += v;
        }
        if (u < nu)
            cum[u] = carry + inc - nt;
        carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0)
        cum[nu] = carry;
}

template <int MODE>
int launch_prefill_one(const PMaps &maps, const PParams &prm, cudaStream_t s)
{
    using C = PCfg<MODE>;
    auto kern = ffn_prefill_kernel<MODE>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return MOE_ERR_CUDA;
    static int configured[64] = {0};
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
            return MOE_ERR_CUDA;
        configured[dev] = 1;
    }
    return launch_pdl(kern, sm_count(dev), kPThreads, (size_t)C::kSmem, s, maps, prm);
}

}  // namespace

namespace {

struct PrefillScratch {
    uint16_t *x16, *h16;
    float *x_scale, *h_scale, *h32;
    unsigned int *hmax;
    int32_t *cum;
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
    s.hmax = reinterpret_cast<unsigned int *>(take(rows * 4));
    s.cum = reinterpret_cast<int32_t *>(take(((size_t)T * k + 2) * 4));
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
    int32_t *cum = ps.cum;
    float *row_scale = ps.x_scale;
    int rc = MOE_OK;

    // plan + gathered bf16 token rows
    rc = launch_pdl(prefill_plan_kernel, 1, 32, 0, s, a.offsets, a.uniq, a.n_uniq, T, cum);
    if (rc != MOE_OK)
        return rc;
    rc = launch_pdl(gather_rows_kernel, (int)rows, 256, 0, s, a.x, a.sorted_pair, T, k, d, x_sorted, row_scale,
                    ps.hmax);
    if (rc != MOE_OK)
        return rc;

    const uint8_t *qs[2] = {w.q_base, w.shared_q};
    const float *ss[2] = {w.s_base, w.shared_s};
    const uint64_t outer[2] = {(uint64_t)E, 1};

    // ---- gate / up
    PMaps gm{};
    for (int i = 0; i < 2 && rc == MOE_OK; i++)
        for (int mat = 0; mat < 2; mat++) {
            rc |= make_tmap_3d(&gm.q[2 * i + mat], qs[i] + (size_t)mat * f * d / 2, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                               1, d / 2, f, outer[i], d / 2, qb, kRawK / 2, kTileM, CU_TENSOR_MAP_SWIZZLE_64B);
            rc |= make_tmap_3d(&gm.s[2 * i + mat], ss[i] + (size_t)mat * f * d / G,
                               CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d / G, f, outer[i], (uint64_t)(d / G) * 4,
                               sc * 4, kRawK / 32, kTileM, CU_TENSOR_MAP_SWIZZLE_NONE);
        }
    rc |= make_tmap_2d(&gm.b, x_sorted, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, d, rows, (uint64_t)d * 2, kOpK, kTileN,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != MOE_OK)
        return MOE_ERR_INVALID_ARG;
    PParams pg{};
    pg.offsets = a.offsets;
    pg.uniq = a.uniq;
    pg.n_uniq = a.n_uniq;
    pg.cum = cum;
    pg.row_scale = row_scale;
    pg.h32 = ps.h32;
    pg.hmax = ps.hmax;
    pg.err = a.err;
    pg.T = T;
    pg.k = k;
    pg.K = d;
    pg.mtiles = f / kTileM;
    pg.out_rows = f;
    rc = launch_prefill_one<kPGateUp>(gm, pg, s);
    if (rc == MOE_OK)
        rc = launch_pdl(h_to_f16_kernel, (int)rows, 256, 0, s, (const float *)ps.h32,
                        (const unsigned int *)ps.hmax, f, h_sorted, ps.h_scale);
    if (rc != MOE_OK)
        return rc;

    // ---- down
    PMaps dm{};
    for (int i = 0; i < 2 && rc == MOE_OK; i++) {
        rc |= make_tmap_3d(&dm.q[2 * i], qs[i] + (size_t)f * d, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, f / 2, d,
                           outer[i], f / 2, qb, kRawK / 2, kTileM, CU_TENSOR_MAP_SWIZZLE_64B);
        rc |= make_tmap_3d(&dm.s[2 * i], ss[i] + (size_t)2 * f * d / G, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                           f / G, d, outer[i], (uint64_t)(f / G) * 4, sc * 4, kRawK / 32, kTileM,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
        dm.q[2 * i + 1] = dm.q[2 * i];
        dm.s[2 * i + 1] = dm.s[2 * i];
    }
    rc |= make_tmap_2d(&dm.b, h_sorted, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, f, rows, (uint64_t)f * 2, kOpK, kTileN,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != MOE_OK)
        return MOE_ERR_INVALID_ARG;
    PParams pd = pg;
    pd.h32 = nullptr;
    pd.hmax = nullptr;
    pd.row_scale = ps.h_scale;
    pd.y_pair = a.y_pair;
    pd.y_shared = a.y_shared;
    pd.K = f;
    pd.mtiles = d / kTileM;
    pd.out_rows = d;
    return launch_prefill_one<kPDown>(dm, pd, s);
}

}  // namespace moe
