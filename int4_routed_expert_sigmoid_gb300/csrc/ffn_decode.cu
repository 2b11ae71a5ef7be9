// ffn_decode.cu -- expert FFN for decode-sized batches: an int4 grouped GEMV
// over the batch union, streaming each selected expert's packed weights from
// HBM once per pass through a TMA-fed shared-memory ring.
//
// Sources: "Public Colibri Observation and Revision Ledger", "Exact
// Architecture and Data-Flow Reconstruction" (each selected expert is a
// three-matrix MLP stored contiguously at int4; a shared expert is always
// used) and the batch-union of "Cache/Prefetch Design Comparison" (each unique
// expert read once per batch).  SwiGLU (h = silu(gate x) * up x, y = down h)
// and the group-32 fp32 scales are readings of the pages.
//
// Design (GB300, sm_103a)
//  * Work item = (expert of the union or the shared expert, tile of output
//    rows).  A persistent grid walks the items; warp 8 of every CTA is a TMA
//    producer that streams the item's weight rows (packed nibbles + scales)
//    through an 8-stage mbarrier ring, k-chunks of 256 elements, 128B-swizzled.
//  * Eight consumer warps turn nibbles into bf16 *exactly* (magic-exponent
//    trick: 0x4300|(n^8) is 136+q as bf16, minus 136) and run m16n8k16 MMAs
//    whose B operand is the activation split into bf16 hi + lo columns, so each
//    product is exact and the fp32 accumulation gives fp32-grade results.  The
//    per-group scale multiplies each group's MMA result in fp32.
//    A plain fp32 CUDA-core GEMV would need ~2 integer ops per weight for the
//    unpacking (integer pipe at half rate) plus the FMA, which caps it below
//    the HBM roofline; here the unpacking costs ~1 op per weight and the
//    multiply-add runs on the tensor pipe.
//  * Gate/up pass: rows of gate and up for a 32-row tile; the epilogue forms
//    h = silu(g) * u in fp32 and stores it as hi/lo bf16 fragments (the B
//    operand of the down pass).  Down pass: 64-row tiles of the down matrix,
//    output y in fp32.
//  * Every mbarrier wait is bounded; a timeout sets MOE_DEVERR_TIMEOUT and the
//    CTA finishes without further waits.
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kProducerWarp = kConsumerWarps;

enum { kGateUp = 0, kDown = 1 };

template <int MODE, int KC>
struct Cfg {
    static constexpr int kRowsPerMat = MODE == kGateUp ? 32 : 64;   // output rows per item
    static constexpr int kMats = MODE == kGateUp ? 2 : 1;
    static constexpr int kRowBytes = KC / 2;                        // packed bytes per row per stage
    static constexpr int kGps = KC / 32;                            // scale groups per stage
    static constexpr int kGph = kGps / 2;                           // groups per k-half
    static constexpr int kQBytes = kRowsPerMat * kRowBytes;         // per matrix
    static constexpr int kSBytes = kRowsPerMat * kGps * 4;          // per matrix
    static constexpr int kStageBytes = kMats * (kQBytes + kSBytes);
    static constexpr int kStages = KC == 256 ? 8 : 16;
    static_assert(kStageBytes % 1024 == 0, "stage must keep 1 KiB alignment");
};

struct Maps {
    CUtensorMap m[8];   // gate/up: gq, uq, gs, us (routed) then the shared expert's
                        // down:    dq, ds (routed), dq, ds (shared)
};

struct Params {
    const int32_t *offsets, *sorted_pair, *uniq, *n_uniq;
    const uint16_t *act;   // activation fragments, row stride 2*K bf16
    uint16_t *h_out;       // gate/up output fragments, row stride 2*f bf16
    float *y_pair, *y_shared;
    int32_t *err;
    int T, k, K, tiles, out_rows;   // K: reduction length; out_rows: rows of the output matrix
};

// Packed nibble pair (bits 0-3 and 16-19 of w) -> two exact bf16 values.
__device__ __forceinline__ uint32_t nib2_to_bf16x2(uint32_t w)
{
    const uint32_t v = (w & 0x000F000Fu) ^ 0x43084308u;   // bf16 136 + q in each half
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x43084308u));
    return r;
}

template <int KC>
__device__ __forceinline__ int swz(int r)
{
    return KC == 256 ? (r & 7) : ((r >> 1) & 3);
}

struct Item {
    int expert;   // routed expert id, or -1 for the shared expert
    int tile;     // row tile
    int m;        // tokens of this expert
    int pos0;     // first pair position (routed) of the expert's group
};

__device__ __forceinline__ Item decode_item(const Params &p, int i)
{
    Item it;
    const int u = i / p.tiles;
    it.tile = i - u * p.tiles;
    if (u == 0) {
        it.expert = -1;
        it.m = p.T;
        it.pos0 = 0;
    } else {
        const int e = p.uniq[u - 1];
        it.expert = e;
        it.pos0 = p.offsets[e];
        it.m = p.offsets[e + 1] - it.pos0;
    }
    return it;
}

template <int MODE, int NT, int KC>
__global__ void __launch_bounds__(kThreads, NT <= 4 ? 2 : 1)
ffn_decode_kernel(const __grid_constant__ Maps maps, const Params p)
{
    using C = Cfg<MODE, KC>;
    constexpr int kTokPerPass = 4 * NT;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t full_bar[C::kStages];
    __shared__ __align__(8) uint64_t empty_bar[C::kStages];
    __shared__ volatile int abort_flag;

    const uint32_t raw = smem_addr(dyn_smem);
    const uint32_t stage0 = (raw + 1023u) & ~1023u;
    const uint8_t *stage_ptr = dyn_smem + (stage0 - raw);
    float *red = reinterpret_cast<float *>(dyn_smem + (stage0 - raw) + C::kStages * C::kStageBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; s++) {
            mbar_init(smem_addr(&full_bar[s]), 1);
            mbar_init(smem_addr(&empty_bar[s]), kConsumerWarps);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int n_items = (*p.n_uniq + 1) * p.tiles;
    const int nchunks = p.K / KC;

    if (warp == kProducerWarp) {
        if (lane != 0)
            return;
        for (int i = 0; i < 8; i++)
            prefetch_tmap(&maps.m[i]);
        int stage = 0;
        uint32_t phase = 0;
        int issued[C::kStages];
        for (int s = 0; s < C::kStages; s++)
            issued[s] = 0;
        for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
            const Item it = decode_item(p, i);
            const int npass = (it.m + kTokPerPass - 1) / kTokPerPass;
            const int mbase = it.expert < 0 ? 4 : 0;   // shared expert's maps follow
            const int z = it.expert < 0 ? 0 : it.expert;
            const int row0 = it.tile * C::kRowsPerMat;
            for (int pass = 0; pass < npass; pass++)
                for (int c = 0; c < nchunks; c++) {
                    if (!abort_flag) {
                        if (!mbar_wait(smem_addr(&empty_bar[stage]), phase ^ 1u)) {
                            atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                            abort_flag = 1;
                        }
                    }
                    if (!abort_flag) {
                        const uint32_t sb = stage0 + stage * C::kStageBytes;
                        const uint32_t fb = smem_addr(&full_bar[stage]);
                        mbar_arrive_expect_tx(fb, C::kStageBytes);
                        if (MODE == kGateUp) {
                            tma_load_3d(sb, &maps.m[mbase + 0], c * C::kRowBytes, row0, z, fb);
                            tma_load_3d(sb + C::kQBytes, &maps.m[mbase + 1], c * C::kRowBytes, row0, z, fb);
                            tma_load_3d(sb + 2 * C::kQBytes, &maps.m[mbase + 2], c * C::kGps, row0, z, fb);
                            tma_load_3d(sb + 2 * C::kQBytes + C::kSBytes, &maps.m[mbase + 3], c * C::kGps,
                                        row0, z, fb);
                        } else {
                            const int mb = it.expert < 0 ? 2 : 0;
                            tma_load_3d(sb, &maps.m[mb + 0], c * C::kRowBytes, row0, z, fb);
                            tma_load_3d(sb + C::kQBytes, &maps.m[mb + 1], c * C::kGps, row0, z, fb);
                        }
                        issued[stage] = 1;
                    }
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
        }
        // Let every copy this thread issued land before the CTA may exit.
        // Stage s last used phase (phase of its last issue); walk back one round.
        for (int s = 0; s < C::kStages; s++) {
            if (!issued[s])
                continue;
            const uint32_t last_phase = s < stage ? phase : phase ^ 1u;
            if (!mbar_wait(smem_addr(&full_bar[s]), last_phase))
                atomicOr(p.err, MOE_DEVERR_TIMEOUT);
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int mt = warp & 3, khalf = warp >> 2;
    const int mat = MODE == kGateUp ? (mt >> 1) : 0;
    const int mtile = MODE == kGateUp ? (mt & 1) : mt;
    const int g = lane >> 2, t4 = lane & 3;
    const int ra = mtile * 16 + g, rb = ra + 8;
    const uint32_t q_off_a = mat * C::kQBytes + ra * C::kRowBytes + 4 * t4;
    const uint32_t q_off_b = mat * C::kQBytes + rb * C::kRowBytes + 4 * t4;
    const uint32_t s_off = C::kMats * C::kQBytes + mat * C::kSBytes;
    const int swa = swz<KC>(ra), swb = swz<KC>(rb);
    int stage = 0;
    uint32_t phase = 0;
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};

    for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
        const Item it = decode_item(p, i);
        const int npass = (it.m + kTokPerPass - 1) / kTokPerPass;
        for (int pass = 0; pass < npass; pass++) {
            // activation rows feeding this lane's B column in each n-tile
            const uint4 *brow[NT];
#pragma unroll
            for (int n = 0; n < NT; n++) {
                const int tt = pass * kTokPerPass + n * 4 + (g >> 1);
                brow[n] = nullptr;
                if (tt < it.m) {
                    int row;
                    if (MODE == kGateUp)
                        row = it.expert < 0 ? tt : p.sorted_pair[it.pos0 + tt] / p.k;
                    else
                        row = it.expert < 0 ? p.T * p.k + tt : it.pos0 + tt;
                    brow[n] = reinterpret_cast<const uint4 *>(p.act + (size_t)row * 2 * p.K +
                                                              (size_t)(g & 1) * p.K) + t4;
                }
            }
            float acc[NT][4];
#pragma unroll
            for (int n = 0; n < NT; n++)
#pragma unroll
                for (int j = 0; j < 4; j++)
                    acc[n][j] = 0.f;

            for (int c = 0; c < nchunks; c++) {
                if (!abort_flag) {
                    if (!mbar_wait(smem_addr(&full_bar[stage]), phase)) {
                        if (lane == 0)
                            atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                        abort_flag = 1;
                    }
                }
                __syncwarp();
                if (!abort_flag) {
                    const uint8_t *sb = stage_ptr + stage * C::kStageBytes;
                    const float *sc = reinterpret_cast<const float *>(sb + s_off);
#pragma unroll
                    for (int gi = 0; gi < C::kGph; gi++) {
                        const int gl = khalf * C::kGph + gi;
                        const uint32_t wa = *reinterpret_cast<const uint32_t *>(sb + q_off_a + ((gl ^ swa) << 4));
                        const uint32_t wb = *reinterpret_cast<const uint32_t *>(sb + q_off_b + ((gl ^ swb) << 4));
                        const float sa = sc[ra * C::kGps + gl];
                        const float sbv = sc[rb * C::kGps + gl];
                        uint32_t a0[4], a1[4];
                        a0[0] = nib2_to_bf16x2(wa);
                        a0[1] = nib2_to_bf16x2(wb);
                        a0[2] = nib2_to_bf16x2(wa >> 4);
                        a0[3] = nib2_to_bf16x2(wb >> 4);
                        a1[0] = nib2_to_bf16x2(wa >> 8);
                        a1[1] = nib2_to_bf16x2(wb >> 8);
                        a1[2] = nib2_to_bf16x2(wa >> 12);
                        a1[3] = nib2_to_bf16x2(wb >> 12);
                        const int gg = c * C::kGps + gl;
#pragma unroll
                        for (int n = 0; n < NT; n++) {
                            uint4 bv = make_uint4(0u, 0u, 0u, 0u);
                            if (brow[n])
                                bv = __ldg(brow[n] + gg * 4);
                            float d[4];
                            mma_bf16_16816(d, a0, bv.x, bv.y, zero4);
                            mma_bf16_16816(d, a1, bv.z, bv.w, d);
                            acc[n][0] = fmaf(sa, d[0], acc[n][0]);
                            acc[n][1] = fmaf(sa, d[1], acc[n][1]);
                            acc[n][2] = fmaf(sbv, d[2], acc[n][2]);
                            acc[n][3] = fmaf(sbv, d[3], acc[n][3]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0 && !abort_flag)
                    mbar_arrive(smem_addr(&empty_bar[stage]));
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }

            // ---- epilogue: reduce the two k-halves, then SwiGLU or store y
            float4 *my_red = reinterpret_cast<float4 *>(red) + (warp * NT) * 32 + lane;
#pragma unroll
            for (int n = 0; n < NT; n++)
                my_red[n * 32] = make_float4(acc[n][0], acc[n][1], acc[n][2], acc[n][3]);
            named_bar_sync(1, kConsumerWarps * 32);
            const float4 *R = reinterpret_cast<const float4 *>(red);
            auto part = [&](int w, int n) { return R[(w * NT + n) * 32 + lane]; };
            if (!abort_flag) {
                if (MODE == kGateUp && (warp == 2 || warp == 3)) {
                    // up warps of k-half 0 finish rows 16*mtile + g (+8)
                    const int f = p.out_rows;
#pragma unroll
                    for (int n = 0; n < NT; n++) {
                        const int tt = pass * kTokPerPass + n * 4 + t4;
                        if (tt >= it.m)
                            continue;
                        const float4 g0 = part(warp - 2, n), g1 = part(warp + 2, n);
                        const float4 u0 = part(warp, n), u1 = part(warp + 4, n);
                        const float gva = (g0.x + g1.x) + (g0.y + g1.y);
                        const float gvb = (g0.z + g1.z) + (g0.w + g1.w);
                        const float uva = (u0.x + u1.x) + (u0.y + u1.y);
                        const float uvb = (u0.z + u1.z) + (u0.w + u1.w);
                        const float ha = gva / (1.0f + expf(-gva)) * uva;
                        const float hb = gvb / (1.0f + expf(-gvb)) * uvb;
                        const int pos = it.expert < 0 ? p.T * p.k + tt : it.pos0 + tt;
                        uint16_t *hrow = p.h_out + (size_t)pos * 2 * f;
                        const int grp = it.tile;                 // 32 rows = one group of the down input
                        const int ia = (grp * 4 + 2 * mtile) * 8 + frag_pos(g);
                        const int ib = ia + 8;                   // row + 8 -> next quad
                        const __nv_bfloat16 ha_hi = __float2bfloat16_rn(ha);
                        const __nv_bfloat16 hb_hi = __float2bfloat16_rn(hb);
                        hrow[ia] = __bfloat16_as_ushort(ha_hi);
                        hrow[ib] = __bfloat16_as_ushort(hb_hi);
                        hrow[f + ia] = __bfloat16_as_ushort(__float2bfloat16_rn(ha - __bfloat162float(ha_hi)));
                        hrow[f + ib] = __bfloat16_as_ushort(__float2bfloat16_rn(hb - __bfloat162float(hb_hi)));
                    }
                } else if (MODE == kDown && warp < 4) {
                    const int d = p.out_rows;
                    const int row_a = it.tile * 64 + mtile * 16 + g;
#pragma unroll
                    for (int n = 0; n < NT; n++) {
                        const int tt = pass * kTokPerPass + n * 4 + t4;
                        if (tt >= it.m)
                            continue;
                        const float4 y0 = part(warp, n), y1 = part(warp + 4, n);
                        float *yrow = it.expert < 0 ? p.y_shared + (size_t)tt * d
                                                    : p.y_pair + (size_t)(it.pos0 + tt) * d;
                        yrow[row_a] = (y0.x + y1.x) + (y0.y + y1.y);
                        yrow[row_a + 8] = (y0.z + y1.z) + (y0.w + y1.w);
                    }
                }
            }
            named_bar_sync(1, kConsumerWarps * 32);
        }
    }
}

template <int MODE, int NT, int KC>
int launch_one(const Maps &maps, const Params &prm, int max_items, cudaStream_t s)
{
    using C = Cfg<MODE, KC>;
    const size_t smem = 1024 + (size_t)C::kStages * C::kStageBytes + (size_t)kConsumerWarps * NT * 32 * 16;
    auto kern = ffn_decode_kernel<MODE, NT, KC>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return MOE_ERR_CUDA;
    // per device, once: opt in to the dynamic shared memory and cache the occupancy
    static int per_sm_cache[64] = {0};
    int per_sm = per_sm_cache[dev];
    if (per_sm == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        per_sm_cache[dev] = per_sm;
    }
    int grid = per_sm * sm_count(dev);
    if (grid > max_items)
        grid = max_items;
    if (grid < 1)
        grid = 1;
    kern<<<grid, kThreads, smem, s>>>(maps, prm);
    return cuda_status(cudaGetLastError());
}

template <int MODE, int KC>
int launch_nt(const Maps &maps, const Params &prm, int max_items, int T, cudaStream_t s)
{
    if (T <= 4)
        return launch_one<MODE, 1, KC>(maps, prm, max_items, s);
    if (T <= 8)
        return launch_one<MODE, 2, KC>(maps, prm, max_items, s);
    return launch_one<MODE, 4, KC>(maps, prm, max_items, s);
}

}  // namespace

int launch_ffn_decode(const DecodeFfnArgs &a, cudaStream_t s)
{
    const moe_layer_int4 &w = *a.w;
    const int d = w.d, f = w.f, E = w.E, G = w.G;
    const uint64_t qb = (uint64_t)moe_expert_q_bytes(d, f);
    const uint64_t sc = (uint64_t)moe_expert_s_count(d, f, G);
    const int kc_gu = 256;
    const int kc_dn = f % 256 == 0 ? 256 : 128;
    const CUtensorMapSwizzle sw_gu = CU_TENSOR_MAP_SWIZZLE_128B;
    const CUtensorMapSwizzle sw_dn = kc_dn == 256 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const int max_experts = (E < a.T * a.k ? E : a.T * a.k) + 1;
    int rc = MOE_OK;

    // ---- gate / up
    Maps gu{};
    const uint8_t *qs[2] = {w.q_base, w.shared_q};
    const float *ss[2] = {w.s_base, w.shared_s};
    const uint64_t outer[2] = {(uint64_t)E, 1};
    for (int i = 0; i < 2 && rc == MOE_OK; i++) {
        const uint8_t *q = qs[i];
        const float *sp = ss[i];
        rc |= make_tmap_3d(&gu.m[4 * i + 0], q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d / 2, f, outer[i],
                           d / 2, qb, kc_gu / 2, 32, sw_gu);
        rc |= make_tmap_3d(&gu.m[4 * i + 1], q + (size_t)f * d / 2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                           d / 2, f, outer[i], d / 2, qb, kc_gu / 2, 32, sw_gu);
        rc |= make_tmap_3d(&gu.m[4 * i + 2], sp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d / G, f,
                           outer[i], (uint64_t)(d / G) * 4, sc * 4, kc_gu / 32, 32,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
        rc |= make_tmap_3d(&gu.m[4 * i + 3], sp + (size_t)f * d / G, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                           d / G, f, outer[i], (uint64_t)(d / G) * 4, sc * 4, kc_gu / 32, 32,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (rc != MOE_OK)
        return MOE_ERR_INVALID_ARG;
    Params pg{};
    pg.offsets = a.offsets;
    pg.sorted_pair = a.sorted_pair;
    pg.uniq = a.uniq;
    pg.n_uniq = a.n_uniq;
    pg.act = a.x_frag;
    pg.h_out = a.h_frag;
    pg.err = a.err;
    pg.T = a.T;
    pg.k = a.k;
    pg.K = d;
    pg.tiles = f / 32;
    pg.out_rows = f;
    rc = launch_nt<kGateUp, 256>(gu, pg, max_experts * pg.tiles, a.T, s);
    if (rc != MOE_OK)
        return rc;

    // ---- down
    Maps dn{};
    for (int i = 0; i < 2 && rc == MOE_OK; i++) {
        rc |= make_tmap_3d(&dn.m[2 * i + 0], qs[i] + (size_t)f * d, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                           f / 2, d, outer[i], f / 2, qb, kc_dn / 2, 64, sw_dn);
        rc |= make_tmap_3d(&dn.m[2 * i + 1], ss[i] + (size_t)2 * f * d / G,
                           CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, f / G, d, outer[i],
                           (uint64_t)(f / G) * 4, sc * 4, kc_dn / 32, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (rc != MOE_OK)
        return MOE_ERR_INVALID_ARG;
    Params pd = pg;
    pd.act = a.h_frag;
    pd.h_out = nullptr;
    pd.y_pair = a.y_pair;
    pd.y_shared = a.y_shared;
    pd.K = f;
    pd.tiles = d / 64;
    pd.out_rows = d;
    if (kc_dn == 256)
        return launch_nt<kDown, 256>(dn, pd, max_experts * pd.tiles, a.T, s);
    return launch_nt<kDown, 128>(dn, pd, max_experts * pd.tiles, a.T, s);
}

}  // namespace moe
