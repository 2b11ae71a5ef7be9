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
//    rows).  A persistent grid walks the items.  Warp 8 of every CTA is the
//    producer: per k-chunk of 256 (or 128) elements it TMA-loads the item's
//    weight rows (packed nibbles, 128B/64B-swizzled, and fp32 scales) and, with
//    1-D bulk copies issued by one lane per token, the matching activation
//    fragments and their corrections, all into one stage of an mbarrier ring.
//    Consumers read every operand from shared memory.
//  * Eight consumer warps run m16n8k16 fp16 MMAs.  A packed nibble becomes
//    an fp16 *subnormal* with one logic op: (n ^ 8) in the mantissa is
//    (q + 8) * 2^-24 exactly (a nibble four bits higher gives 16 (q + 8) * 2^-24,
//    the 16 being undone in the activation operand).  The activation is split
//    into fp16 hi + lo columns, scaled by a power of two for range.  Products
//    are exact and accumulate in fp32; per group, 2^24 * D minus the
//    precomputed 8 * sum(activation) correction is the exact-integer dot
//    product, multiplied in fp32 by the group scale.  Unpacking costs 10
//    integer ops per 512 weights and no float op (the integer pipe, which runs
//    at half rate, is what bounds this loop).
//  * Gate/up pass: rows of gate and up for a 32-row tile; the epilogue forms
//    h = silu(g) * u in fp32 and stores it as fragments (one power-of-two
//    factor and one correction pair per 32 rows) for the down pass.  Down
//    pass: 64-row tiles of the down matrix, output y in fp32.
//  * Every mbarrier wait is bounded; a timeout sets MOE_DEVERR_TIMEOUT and the
//    CTA finishes without further waits.
//  * The kernels wait on their predecessor grid (griddepcontrol) only after
//    their prologue, so a programmatic-dependent launch overlaps the two.
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kProducerWarp = kConsumerWarps;

enum { kGateUp = 0, kDown = 1 };

// TOK: tokens per pass (1, 4, 8 or 16); NT = ceil(TOK / 4) MMA n-tiles of 4 tokens (hi + lo columns).
template <int MODE, int TOK, int KC>
struct Cfg {
    static constexpr int kRowsPerMat = MODE == kGateUp ? 32 : 64;   // output rows per item
    static constexpr int kMats = MODE == kGateUp ? 2 : 1;
    static constexpr int kRowBytes = KC / 2;                        // packed bytes per row per stage
    static constexpr int kGps = KC / 32;                            // scale groups per stage
    static constexpr int kGph = kGps / 2;                           // groups per k-half
    static constexpr int kTok = TOK;                                // tokens per pass
    static constexpr int kQBytes = kRowsPerMat * kRowBytes;         // per matrix
    static constexpr int kSBytes = kRowsPerMat * kGps * 4;          // per matrix
    static constexpr int kPlaneBytes = kGps * 64;                   // one token's hi (or lo) chunk
    static constexpr int kCBytes = kGps * 8;                        // one token's corrections (hi, lo)
    static constexpr int kFBytes = MODE == kDown ? kGps * 4 : 0;    // one token's group factors
    static constexpr int kQOff = 0;
    static constexpr int kSOff = kMats * kQBytes;
    static constexpr int kBOff = kSOff + kMats * kSBytes;
    static constexpr int kCOff = kBOff + kTok * 2 * kPlaneBytes;
    static constexpr int kFOff = kCOff + kTok * kCBytes;
    static constexpr int kUsed = kFOff + kTok * kFBytes;
    static constexpr int kStageBytes = (kUsed + 1023) / 1024 * 1024;   // keeps the swizzle atoms aligned
    static constexpr int kStages = (100 * 1024) / kStageBytes < 16 ? (100 * 1024) / kStageBytes : 16;
    static constexpr int kWeightBytes = kMats * (kQBytes + kSBytes);
    static constexpr int kTokBytes = 2 * kPlaneBytes + kCBytes + kFBytes;
    static_assert(kStages >= 3, "ring too shallow");
};

struct Maps {
    CUtensorMap m[8];   // gate/up: gq, uq, gs, us (routed) then the shared expert's
                        // down:    dq, ds (routed), dq, ds (shared)
};

struct Params {
    const int32_t *offsets, *sorted_pair, *uniq, *n_uniq;
    const uint16_t *act;        // activation fragments (fp16), row stride 2*K
    const float *act_scale;     // gate/up: per-row factor of x; down: per-(row, group) factor of h
    const float *act_corr;      // [rows][K/32][2] corrections
    uint16_t *h_out;            // gate/up output fragments, row stride 2*f
    float *h_scale;             // gate/up output factors [rows][f/32]
    float *h_corr;              // gate/up output corrections [rows][f/32][2]
    float *y_pair, *y_shared;
    int32_t *err;
    int T, k, K, tiles, out_rows;   // K: reduction length; out_rows: rows of the output matrix
};

// Packed nibbles -> fp16 subnormal pairs: lo takes the nibbles at bits 0-3 and
// 16-19 -> (q + 8) * 2^-24 each; hi those at bits 4-7 and 20-23 -> 16 (q + 8) * 2^-24.
// (w & m) ^ x as one three-input logic op: both constants are passed in
// registers (an instruction can carry only one immediate), LUT 0x6A.
struct NibConst {
    uint32_t m_lo, x_lo, m_hi, x_hi;
};

__device__ __forceinline__ uint32_t and_xor(uint32_t w, uint32_t m, uint32_t x)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(w), "r"(m), "r"(x));
    return r;
}

__device__ __forceinline__ uint32_t nib_lo(uint32_t w, const NibConst &k) { return and_xor(w, k.m_lo, k.x_lo); }
__device__ __forceinline__ uint32_t nib_hi(uint32_t w, const NibConst &k) { return and_xor(w, k.m_hi, k.x_hi); }

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

// Activation row of token tt (< m) of an item: x row (gate/up) or h row (down).
template <int MODE>
__device__ __forceinline__ int act_row(const Params &p, const Item &it, int tt)
{
    if (MODE == kGateUp)
        return it.expert < 0 ? tt : p.sorted_pair[it.pos0 + tt] / p.k;
    return it.expert < 0 ? p.T * p.k + tt : it.pos0 + tt;
}

template <int MODE, int TOK, int KC>
__global__ void __launch_bounds__(kThreads, 2)
ffn_decode_kernel(const __grid_constant__ Maps maps, const Params p)
{
    using C = Cfg<MODE, TOK, KC>;
    constexpr int NT = (TOK + 3) / 4;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t full_bar[C::kStages];
    __shared__ __align__(8) uint64_t empty_bar[C::kStages];
    __shared__ volatile int abort_flag;

    const uint32_t raw = smem_addr(dyn_smem);
    const uint32_t stage0 = (raw + 1023u) & ~1023u;
    const uint8_t *stage_ptr = dyn_smem + (stage0 - raw);
    float *red = reinterpret_cast<float *>(dyn_smem + (stage0 - raw) + C::kStages * C::kStageBytes);
    float *hbuf = red + kConsumerWarps * NT * 32 * 4;   // [kTok][32] h values of one item

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; s++) {
            mbar_init(smem_addr(&full_bar[s]), 1);
            mbar_init(smem_addr(&empty_bar[s]), kConsumerWarps);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kProducerWarp && lane == 0)
        for (int i = 0; i < 8; i++)
            prefetch_tmap(&maps.m[i]);
    __syncthreads();
    griddep_launch_dependents();
    griddep_wait();   // routing, union and activation fragments come from the previous kernels

    const int n_items = (*p.n_uniq + 1) * p.tiles;
    const int nchunks = p.K / KC;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------- producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0;   // bit s: stage s was filled at least once
        for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
            const Item it = decode_item(p, i);
            const int npass = (it.m + C::kTok - 1) / C::kTok;
            const int z = it.expert < 0 ? 0 : it.expert;
            const int row0 = it.tile * C::kRowsPerMat;
            for (int pass = 0; pass < npass; pass++) {
                const int ntok = min(C::kTok, it.m - pass * C::kTok);
                // lane j < ntok copies the activation data of token j of this pass
                const int my_row = lane < ntok ? act_row<MODE>(p, it, pass * C::kTok + lane) : 0;
                const uint16_t *my_act = p.act + (size_t)my_row * 2 * p.K;
                const float *my_corr = p.act_corr + (size_t)my_row * (p.K / 32) * 2;
                const float *my_fac = p.act_scale + (size_t)my_row * (p.K / 32);
                const uint32_t tx = C::kWeightBytes + ntok * C::kTokBytes;
                for (int c = 0; c < nchunks; c++) {
                    if (!abort_flag && lane == 0) {
                        if (!mbar_wait(smem_addr(&empty_bar[stage]), phase ^ 1u)) {
                            atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                            abort_flag = 1;
                        }
                    }
                    __syncwarp();
                    if (!abort_flag) {
                        const uint32_t sb = stage0 + stage * C::kStageBytes;
                        const uint32_t fb = smem_addr(&full_bar[stage]);
                        if (lane == 0) {
                            mbar_arrive_expect_tx(fb, tx);
                            if (MODE == kGateUp) {
                                const int mb = it.expert < 0 ? 4 : 0;   // shared expert's maps follow
                                tma_load_3d(sb + C::kQOff, &maps.m[mb + 0], c * C::kRowBytes, row0, z, fb);
                                tma_load_3d(sb + C::kQOff + C::kQBytes, &maps.m[mb + 1], c * C::kRowBytes,
                                            row0, z, fb);
                                tma_load_3d(sb + C::kSOff, &maps.m[mb + 2], c * C::kGps, row0, z, fb);
                                tma_load_3d(sb + C::kSOff + C::kSBytes, &maps.m[mb + 3], c * C::kGps, row0,
                                            z, fb);
                            } else {
                                const int mb = it.expert < 0 ? 2 : 0;
                                tma_load_3d(sb + C::kQOff, &maps.m[mb + 0], c * C::kRowBytes, row0, z, fb);
                                tma_load_3d(sb + C::kSOff, &maps.m[mb + 1], c * C::kGps, row0, z, fb);
                            }
                            issued |= 1u << stage;
                        }
                        __syncwarp();   // expect_tx is posted before any copy below can complete
                        if (lane < ntok) {
                            const uint16_t *src = my_act + (size_t)c * KC;
                            const uint32_t dst = sb + C::kBOff + lane * 2 * C::kPlaneBytes;
                            bulk_load(dst, src, C::kPlaneBytes, fb);                          // hi plane
                            bulk_load(dst + C::kPlaneBytes, src + p.K, C::kPlaneBytes, fb);     // lo plane
                            bulk_load(sb + C::kCOff + lane * C::kCBytes, my_corr + c * C::kGps * 2,
                                      C::kCBytes, fb);
                            if (MODE == kDown)
                                bulk_load(sb + C::kFOff + lane * C::kFBytes, my_fac + c * C::kGps,
                                          C::kFBytes, fb);
                        }
                    }
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        // Let every copy issued here land before the CTA may exit: stages below
        // `stage` were last filled in the current round, the rest in the
        // previous one.
        if (lane == 0) {
            for (int s = 0; s < C::kStages; s++) {
                if (!((issued >> s) & 1u))
                    continue;
                const uint32_t last_phase = s < stage ? phase : phase ^ 1u;
                if (!mbar_wait(smem_addr(&full_bar[s]), last_phase))
                    atomicOr(p.err, MOE_DEVERR_TIMEOUT);
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    // warp -> (matrix, 16-row m-tile, k-half of every stage)
    const int mt = warp & 3, khalf = warp >> 2;
    const int mat = MODE == kGateUp ? (mt >> 1) : 0;
    const int mtile = MODE == kGateUp ? (mt & 1) : mt;
    const int g = lane >> 2, t4 = lane & 3;
    const int ra = mtile * 16 + g;   // and ra + 8: same swizzle phase
    uint32_t qoff[C::kGph];          // byte offset of this lane's word of row ra, per group of the k-half
#pragma unroll
    for (int gi = 0; gi < C::kGph; gi++) {
        const int gl = khalf * C::kGph + gi;
        qoff[gi] = C::kQOff + mat * C::kQBytes + ra * C::kRowBytes + ((gl ^ swz<KC>(ra)) << 4) + 4 * t4;
    }
    constexpr uint32_t kRowB = 8 * C::kRowBytes;
    const uint32_t soff_a = C::kSOff + mat * C::kSBytes + (ra * C::kGps + khalf * C::kGph) * 4;
    const uint32_t soff_b = soff_a + 8 * C::kGps * 4;
    int stage = 0;
    uint32_t phase = 0;
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    constexpr float kTwo24 = 16777216.0f;
    const NibConst nk = {0x000F000Fu, 0x00080008u, 0x00F000F0u, 0x00800080u};

    for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
        const Item it = decode_item(p, i);
        const int npass = (it.m + C::kTok - 1) / C::kTok;
        for (int pass = 0; pass < npass; pass++) {
            const int ntok = min(C::kTok, it.m - pass * C::kTok);
            // stage offsets of this lane's B chunk (token g/2 of each n-tile, plane g&1) and of the
            // corrections / factors of the token whose D columns it holds (token t4); tokens past
            // ntok read token 0's data (finite, discarded)
            uint32_t boff[NT], coff[NT], foff[NT];
#pragma unroll
            for (int n = 0; n < NT; n++) {
                int jb = n * 4 + (g >> 1);
                jb = jb < ntok ? jb : 0;
                boff[n] = C::kBOff + (jb * 2 + (g & 1)) * C::kPlaneBytes + (khalf * C::kGph * 4 + t4) * 16;
                int jd = n * 4 + t4;
                jd = jd < ntok ? jd : 0;
                coff[n] = C::kCOff + jd * C::kCBytes + khalf * C::kGph * 8;
                foff[n] = C::kFOff + jd * C::kFBytes + khalf * C::kGph * 4;
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
#pragma unroll
                    for (int gi = 0; gi < C::kGph; gi++) {
                        const uint32_t wa = *reinterpret_cast<const uint32_t *>(sb + qoff[gi]);
                        const uint32_t wb = *reinterpret_cast<const uint32_t *>(sb + qoff[gi] + kRowB);
                        const float sa = reinterpret_cast<const float *>(sb + soff_a)[gi];
                        const float sbv = reinterpret_cast<const float *>(sb + soff_b)[gi];
                        const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
                        const uint32_t a0[4] = {nib_lo(wa, nk), nib_lo(wb, nk), nib_hi(wa, nk), nib_hi(wb, nk)};
                        const uint32_t a1[4] = {nib_lo(wa8, nk), nib_lo(wb8, nk), nib_hi(wa8, nk), nib_hi(wb8, nk)};
#pragma unroll
                        for (int n = 0; n < NT; n++) {
                            const uint4 bv = *reinterpret_cast<const uint4 *>(sb + boff[n] + gi * 64);
                            const float2 cc = *reinterpret_cast<const float2 *>(sb + coff[n] + gi * 8);
                            float d[4];
                            mma_f16_16816(d, a0, bv.x, bv.y, zero4);
                            mma_f16_16816(d, a1, bv.z, bv.w, d);
                            float fa = sa, fb = sbv;
                            if (MODE == kDown) {
                                const float hf = reinterpret_cast<const float *>(sb + foff[n])[gi];
                                fa *= hf;
                                fb *= hf;
                            }
                            acc[n][0] = fmaf(fa, fmaf(d[0], kTwo24, -cc.x), acc[n][0]);
                            acc[n][1] = fmaf(fa, fmaf(d[1], kTwo24, -cc.y), acc[n][1]);
                            acc[n][2] = fmaf(fb, fmaf(d[2], kTwo24, -cc.x), acc[n][2]);
                            acc[n][3] = fmaf(fb, fmaf(d[3], kTwo24, -cc.y), acc[n][3]);
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

            // ---- epilogue: reduce the two k-halves, then SwiGLU (+ fragments) or store y
            float4 *my_red = reinterpret_cast<float4 *>(red) + (warp * NT) * 32 + lane;
#pragma unroll
            for (int n = 0; n < NT; n++)
                my_red[n * 32] = make_float4(acc[n][0], acc[n][1], acc[n][2], acc[n][3]);
            named_bar_sync(1, kConsumerWarps * 32);
            const float4 *R = reinterpret_cast<const float4 *>(red);
            auto part = [&](int w, int n) { return R[(w * NT + n) * 32 + lane]; };
            if (MODE == kGateUp) {
                if (!abort_flag && (warp == 2 || warp == 3)) {
                    // up warps of k-half 0: h for rows 16*mtile + g (+8), token t4 of each n-tile
#pragma unroll
                    for (int n = 0; n < NT; n++) {
                        const int tl = n * 4 + t4;
                        if (tl >= ntok)
                            continue;
                        const float xf = p.act_scale[act_row<MODE>(p, it, pass * C::kTok + tl)];
                        const float4 g0 = part(warp - 2, n), g1 = part(warp + 2, n);
                        const float4 u0 = part(warp, n), u1 = part(warp + 4, n);
                        const float gva = ((g0.x + g1.x) + (g0.y + g1.y)) * xf;
                        const float gvb = ((g0.z + g1.z) + (g0.w + g1.w)) * xf;
                        const float uva = ((u0.x + u1.x) + (u0.y + u1.y)) * xf;
                        const float uvb = ((u0.z + u1.z) + (u0.w + u1.w)) * xf;
                        hbuf[tl * 32 + mtile * 16 + g] = gva / (1.0f + expf(-gva)) * uva;
                        hbuf[tl * 32 + mtile * 16 + g + 8] = gvb / (1.0f + expf(-gvb)) * uvb;
                    }
                }
                named_bar_sync(1, kConsumerWarps * 32);
                // one warp per token: the item's 32 rows form one group of the down input
                if (!abort_flag) {
                    const int f = p.out_rows;
                    for (int tl = warp; tl < ntok; tl += kConsumerWarps) {
                        const int tt = pass * C::kTok + tl;
                        float v = hbuf[tl * 32 + lane];
                        float mx = fabsf(v);
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1)
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                        int e = 0;
                        frexpf(mx, &e);
                        const float up = mx > 0.f ? ldexpf(1.0f, 14 - e) : 1.0f;
                        v *= up;
                        if (lane & 1)
                            v *= 0.0625f;
                        const __half hi = __float2half_rn(v);
                        const __half lo = __float2half_rn(v - __half2float(hi));
                        const float wgt = (lane & 1) ? 128.0f : 8.0f;
                        float chi = wgt * __half2float(hi), clo = wgt * __half2float(lo);
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) {
                            chi += __shfl_xor_sync(0xffffffffu, chi, off);
                            clo += __shfl_xor_sync(0xffffffffu, clo, off);
                        }
                        const int pos = it.expert < 0 ? p.T * p.k + tt : it.pos0 + tt;
                        uint16_t *hrow = p.h_out + (size_t)pos * 2 * f;
                        const int idx = (it.tile * 4 + (lane >> 3)) * 8 + frag_pos(lane & 7);
                        hrow[idx] = __half_as_ushort(hi);
                        hrow[f + idx] = __half_as_ushort(lo);
                        if (lane == 0) {
                            const size_t gidx = (size_t)pos * (f / 32) + it.tile;
                            p.h_scale[gidx] = mx > 0.f ? ldexpf(1.0f, e - 14) : 1.0f;
                            p.h_corr[gidx * 2 + 0] = chi;
                            p.h_corr[gidx * 2 + 1] = clo;
                        }
                    }
                }
            } else if (!abort_flag && warp < 4) {
                const int d = p.out_rows;
                const int row_a = it.tile * 64 + mtile * 16 + g;
#pragma unroll
                for (int n = 0; n < NT; n++) {
                    const int tl = n * 4 + t4;
                    if (tl >= ntok)
                        continue;
                    const int tt = pass * C::kTok + tl;
                    const float4 y0 = part(warp, n), y1 = part(warp + 4, n);
                    float *yrow = it.expert < 0 ? p.y_shared + (size_t)tt * d
                                                : p.y_pair + (size_t)(it.pos0 + tt) * d;
                    yrow[row_a] = (y0.x + y1.x) + (y0.y + y1.y);
                    yrow[row_a + 8] = (y0.z + y1.z) + (y0.w + y1.w);
                }
            }
            named_bar_sync(1, kConsumerWarps * 32);
        }
    }
}

template <int MODE, int TOK, int KC>
int launch_one(const Maps &maps, const Params &prm, int max_items, cudaStream_t s)
{
    using C = Cfg<MODE, TOK, KC>;
    constexpr int NT = (TOK + 3) / 4;
    const size_t smem = 1024 + (size_t)C::kStages * C::kStageBytes + (size_t)kConsumerWarps * NT * 32 * 16 +
                        (size_t)C::kTok * 32 * 4;
    auto kern = ffn_decode_kernel<MODE, TOK, KC>;
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
    return launch_pdl(kern, grid, kThreads, smem, s, maps, prm);
}

template <int MODE, int KC>
int launch_nt(const Maps &maps, const Params &prm, int max_items, int T, cudaStream_t s)
{
    if (T == 1)
        return launch_one<MODE, 1, KC>(maps, prm, max_items, s);
    if (T <= 4)
        return launch_one<MODE, 4, KC>(maps, prm, max_items, s);
    if (T <= 8)
        return launch_one<MODE, 8, KC>(maps, prm, max_items, s);
    return launch_one<MODE, 16, KC>(maps, prm, max_items, s);
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
    pg.act_scale = a.x_scale;
    pg.act_corr = a.x_corr;
    pg.h_out = a.h_frag;
    pg.h_scale = a.h_scale;
    pg.h_corr = a.h_corr;
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
    pd.act_scale = a.h_scale;
    pd.act_corr = a.h_corr;
    pd.h_out = nullptr;
    pd.h_scale = nullptr;
    pd.h_corr = nullptr;
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
