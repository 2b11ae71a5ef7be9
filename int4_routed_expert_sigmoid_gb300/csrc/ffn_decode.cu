// ffn_decode.cu -- expert FFN for decode-sized batches: an int4 grouped GEMV
// over the batch union, streaming each selected expert's packed weights from
// HBM once per pass through a TMA-fed shared-memory ring.
//
// Sources: "Public Colibri Observation and Revision Ledger", "Exact
// Architecture and Data-Flow Reconstruction" (a routed expert is an MLP of
// three int4 matrices kept side by side; the shared expert runs for every
// token) and the batch union of "Cache/Prefetch Design Comparison" (one fetch
// of a selected expert serves the whole batch).  SwiGLU (h = silu(gate x) * up x, y = down h)
// and the group-32 fp32 scales are readings of the pages.
//
// Design (GB300, sm_103a)
//  * Work item = (expert of the union or the shared expert, tile of output
//    rows: 32 rows of gate and of up, or 64 rows of down).  A persistent grid
//    walks the items; CTA c starts with item c.  For batches of more than one
//    token each CTA's producer then takes the next unclaimed item from a
//    global counter (zeroed by the kernel that precedes the FFN): units of
//    very different token counts make items of very different lengths, and
//    CTAs that finish early take more of them (at 64 tokens this shortened the
//    FFN by 6 %).  At T = 1 all items are equal and CTA c takes c, c + G, ...
//    (claiming was 2 us slower there).  The producer tags every ring stage
//    with its item, so the consumers follow without knowing the schedule.  An
//    item's tokens are taken in passes of at most TOK tokens (balanced), each
//    pass streaming the item's weights once (a second pass finds them in L2).
//  * Warp 8 of every CTA is the producer: per stage (one or two k-chunks of
//    32 * GPC elements) it TMA-loads the item's packed rows (swizzled) and
//    scales and, with one bulk copy per token, that token's activation
//    fragment blocks, all into one stage of an mbarrier ring.
//  * Eight consumer warps (matrix x 16-row m-tile x half of the stage's
//    groups) run m16n8k16 fp16 MMAs.  A packed nibble pair becomes two fp16
//    subnormals (q + 8) * 2^-24 with one three-input logic op (exact; the
//    tensor cores multiply subnormals exactly).  The activation is split into
//    fp16 hi + lo planes (power-of-two scaled), the B columns being (token,
//    plane) pairs.  The accumulator of every group starts at the fragment's
//    -2^-24 * 8 * sum(activation) (the +8 of the nibble encoding), so after the
//    group's two MMAs it holds 2^-24 * sum q v, and one FMA per output row and
//    token applies the group scale: acc += s * (D_hi + D_lo).
//  * Gate/up epilogue: the two k-halves are reduced through shared memory,
//    h = silu(g) * u is formed in fp32 and packed as the down pass's fragment
//    blocks (one power-of-two factor per 32 rows).  Down: y in fp32.
//  * Every mbarrier wait is bounded; a timeout sets MOE_DEVERR_TIMEOUT and the
//    CTA's roles stop waiting (results are then invalid, nothing hangs).
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
constexpr int kRingBytes = 96 * 1024;   // two CTAs per SM

enum { kGateUp = 0, kDown = 1 };

// TOK: tokens per pass (1, 4, 8 or 16); CPS: k-chunks per stage; GPC: groups per chunk (8 or 4).
template <int MODE, int TOK, int CPS, int GPC, int GS>
struct Cfg {
    static constexpr int kRows = MODE == kGateUp ? 32 : 64;   // output rows per matrix per item
    static constexpr int kMats = MODE == kGateUp ? 2 : 1;
    static constexpr int kNTM = (TOK + 3) / 4;                 // n-tiles (4 tokens each) at most
    static constexpr int kRowB = 16 * GPC;                     // packed bytes of a row per chunk
    static constexpr int kQSub = kRows * kRowB;                // one (matrix, chunk) tile of nibbles
    static constexpr int kSpr = GPC * 32 / GS;                 // scales of a row per chunk (group size GS)
    static constexpr int kSSub = kRows * kSpr * 4;             // one (matrix, chunk) tile of scales
    static constexpr int kBlk = frag_blk(GPC);
    static constexpr int kGpw = CPS * GPC / 2;                 // groups per warp per stage
    static constexpr int kSOff = kMats * CPS * kQSub;
    static constexpr int kBOff = kSOff + kMats * CPS * kSSub;
    static constexpr int kTokBytes = CPS * kBlk;               // one token's fragment blocks per stage
    static constexpr int kUsed = kBOff + TOK * kTokBytes;
    static constexpr int kStageBytes = (kUsed + 1023) / 1024 * 1024;   // keeps the swizzle atoms aligned
    static constexpr int kStages = kRingBytes / kStageBytes < 12 ? kRingBytes / kStageBytes : 12;
    static constexpr int kWeightBytes = kMats * CPS * (kQSub + kSSub);
    static constexpr int kRedBytes = kConsumerWarps * kNTM * 32 * 8;
    static constexpr int kHBufBytes = TOK * 32 * 4;
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kRedBytes + kHBufBytes;   // + unit table
    static_assert(kStages >= 3, "ring too shallow");
    static constexpr int kSpw = kGpw * 32 / GS;                // scales per warp per stage
    static_assert(GS == 32 || GS == 64, "group sizes");
    static_assert(kSpr * 4 % 16 == 0, "a scale box row is a multiple of 16 bytes");
    static_assert(kSpw == 1 || kSpw == 2 || kSpw % 4 == 0, "scale vector loads");
    static_assert(kBOff % 16 == 0 && kTokBytes % 16 == 0, "bulk copy alignment");
};

// Tensor maps of one half of the FFN: packed rows and scales, [0] routed
// experts, [1] the shared expert.  A stage's box lands in shared memory as
// [chunk][matrix][row][bytes of the chunk].  With `merged`, the chunk is a
// dimension of the map, so one load per stage moves all nibbles (and one all
// scales); otherwise one load per chunk.
struct Maps {
    CUtensorMap q[2], s[2];
    int merged;
    int cps;   // k-chunks one merged box spans: the kernel's stage layout must hold exactly that many
};

struct Params {
    const int32_t *offsets, *sorted_pair, *uniq, *n_uniq;
    const uint8_t *act;         // activation fragment rows (x for gate/up, h for down)
    size_t act_row_bytes;
    const float *x_scale;       // gate/up: per-row factor of x
    uint8_t *h_out;             // gate/up: fragment rows of h
    size_t h_row_bytes;
    int gpc_h;                  // groups per block of the h fragments
    float *y_pair, *y_shared;
    int32_t *work;              // items claimed beyond the first one per CTA; zero on entry
    const int32_t *slot_of;     // when set: routed expert e's weights are block slot_of[e] of the layer view
    int with_shared;            // 1: unit 0 is the shared expert; 0: the units are the uniq list only
    int32_t *err;
    int T, k, nchunks, tiles, out_rows;   // nchunks: k-chunks of the reduction; out_rows: d (down)
    int dynamic;                // 1: items after the first from the counter; 0: CTA c takes c, c + G, ...
    int n_experts, n_view;      // routed experts of the routing; expert blocks of the weight view
    int max_uniq;               // capacity of the unit table beyond the shared expert: n_uniq is clamped to it
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

// 16-byte unit of packed row r that holds logical unit u after the TMA swizzle
// (128-byte rows: 128B swizzle; 64-byte rows: 64B swizzle).
template <int GPC>
__device__ __forceinline__ int swz(int r)
{
    return GPC == 8 ? (r & 7) : ((r >> 1) & 3);
}

struct Item {
    int expert;   // routed expert id, or -1 for the shared expert
    int zq;       // block of the layer view holding its weights (routed)
    int tile;     // row tile
    int m;        // tokens of this expert
    int pos0;     // first pair position (routed) of the expert's group
};

// Unit table: unit 0 is the shared expert (all T tokens), unit u >= 1 the
// union's expert uniq[u - 1]; built once per CTA in shared memory so that
// walking the items needs no dependent global loads.
struct Unit {
    int expert, pos0, m, zq;
};

// (L2 loads: the down kernel reads the table before its grid wait, when the
// union is complete but this SM's L1 may hold an older launch's copy)
__device__ __forceinline__ void load_units(const Params &p, int units, Unit *tab)
{
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
        Unit t;
        if (u < p.with_shared) {
            t.expert = -1;
            t.pos0 = 0;
            t.m = p.T;
            t.zq = 0;
        } else {
            const int e = __ldcg(p.uniq + u - p.with_shared);
            t.expert = e;
            if (MOE_IN_BOUNDS(e >= 0 && e < p.n_experts, p.err)) {
                t.pos0 = __ldcg(p.offsets + e);
                t.m = __ldcg(p.offsets + e + 1) - t.pos0;
                t.zq = p.slot_of ? __ldcg(p.slot_of + e) : e;
                // a unit outside the pairs or the weight view gets no tokens (its items do nothing)
                if (!MOE_IN_BOUNDS(t.pos0 >= 0 && t.m >= 0 && t.pos0 + t.m <= p.T * p.k && t.zq >= 0 &&
                                       t.zq < p.n_view,
                                   p.err))
                    t.m = 0;
            } else {
                t.expert = 0;
                t.pos0 = t.m = t.zq = 0;
            }
        }
        tab[u] = t;
    }
}

__device__ __forceinline__ Item decode_item(const Params &p, const Unit *tab, int i)
{
    Item it;
    const int u = i / p.tiles;
    it.tile = i - u * p.tiles;
    const Unit t = tab[u];
    it.expert = t.expert;
    it.zq = t.zq;
    it.pos0 = t.pos0;
    it.m = t.m;
    return it;
}

// Activation row of token tt (< m) of an item: x row (gate/up) or h row (down).
template <int MODE>
__device__ __forceinline__ int act_row(const Params &p, const Item &it, int tt)
{
    if (MODE == kGateUp) {
        if (it.expert < 0)
            return tt;
        const int sp = p.sorted_pair[it.pos0 + tt];
        return MOE_IN_BOUNDS(sp >= 0 && sp < p.T * p.k, p.err) ? sp / p.k : 0;
    }
    return it.expert < 0 ? p.T * p.k + tt : it.pos0 + tt;
}

// Tokens [t0, t0 + ntok) of pass `pass` of `npass` over m tokens (balanced).
__device__ __forceinline__ void pass_range(int m, int npass, int pass, int &t0, int &ntok)
{
    t0 = pass * m / npass;
    ntok = (pass + 1) * m / npass - t0;
}

// Shared state of the consumer warps of one CTA.
struct Consumer {
    const uint8_t *base;     // stage 0
    uint64_t *full, *empty;
    volatile int *abort;
    float2 *red;             // [warp][n-tile][lane]
    float *hbuf;             // [token][32]
    int warp, lane, g, t4, mtile;
    int stage;
    uint32_t phase;
};

// One pass over an item's tokens [t0, t0 + ntok), NT = ceil(ntok / 4) n-tiles.
template <int MODE, int TOK, int CPS, int GPC, int GS, int NT>
__device__ __forceinline__ void run_pass(const Params &p, const Item &it, int t0, int ntok, Consumer &cs,
                                         const uint32_t (&qoff)[Cfg<MODE, TOK, CPS, GPC, GS>::kGpw], uint32_t soff,
                                         uint32_t kb, uint32_t kbc, uint32_t kbf, uint32_t plane_off)
{
    using C = Cfg<MODE, TOK, CPS, GPC, GS>;
    constexpr int kGpw = C::kGpw;
    const int g = cs.g, t4 = cs.t4, lane = cs.lane, warp = cs.warp;
    // stage offsets of this lane's B chunk (token g/2 of each n-tile, plane g&1) and of the
    // accumulator inputs / factors of the token whose D columns it holds (token t4).  Columns of
    // tokens past ntok are computed and discarded; when the stage has room for all 4 * NT token
    // blocks they read whatever the stage holds there, so the offsets are a base plus a fixed
    // stride per n-tile (no per-tile registers); a stage with fewer token blocks (TOK < 4 NT) has
    // those columns read token 0 instead.
    constexpr bool kClamp = TOK < 4 * NT;
    constexpr uint32_t kNStride = 4 * C::kTokBytes;
    uint32_t boff[kClamp ? NT : 1], coff[kClamp ? NT : 1], foff[kClamp ? NT : 1];
#pragma unroll
    for (int n = 0; n < (kClamp ? NT : 1); n++) {
        int jb = n * 4 + (g >> 1);
        jb = (!kClamp || jb < ntok) ? jb : 0;
        boff[n] = C::kBOff + jb * C::kTokBytes + kb + plane_off;
        int jd = n * 4 + t4;
        jd = (!kClamp || jd < ntok) ? jd : 0;
        coff[n] = C::kBOff + jd * C::kTokBytes + kbc;
        foff[n] = C::kBOff + jd * C::kTokBytes + kbf;
    }
    auto bo = [&](int n) { return kClamp ? boff[n] : boff[0] + n * kNStride; };
    auto co = [&](int n) { return kClamp ? coff[n] : coff[0] + n * kNStride; };
    auto fo = [&](int n) { return kClamp ? foff[n] : foff[0] + n * kNStride; };
    float acc[NT][2];
#pragma unroll
    for (int n = 0; n < NT; n++)
        acc[n][0] = acc[n][1] = 0.f;
    // gate/up: the x factor of token t4 of each n-tile (every group's factor slot of an x fragment
    // block holds it), read from the first stage and used in the epilogue
    float xfac[NT];
#pragma unroll
    for (int n = 0; n < NT; n++)
        xfac[n] = 0.f;
    const NibConst nk = {0x000F000Fu, 0x00080008u, 0x00F000F0u, 0x00800080u};
    const int nstages = p.nchunks / CPS;

    for (int c = 0; c < nstages; c++) {
        const uint32_t fbar = smem_addr(&cs.full[cs.stage]);
        if (!mbar_wait_or_abort(fbar, cs.phase, cs.abort)) {
            if (lane == 0)
                atomicOr(p.err, MOE_DEVERR_TIMEOUT);
            *cs.abort = 1;
        }
        const uint8_t *sb = cs.base + cs.stage * C::kStageBytes;
        if (MODE == kGateUp && c == 0) {
#pragma unroll
            for (int n = 0; n < NT; n++)
                xfac[n] = *reinterpret_cast<const float *>(sb + fo(n));
        }
        // group scales of rows ra and ra + 8 for this warp's groups (one per GS elements)
        constexpr int kSpw = C::kSpw;
        float sa[kSpw], sc[kSpw];
        if (kSpw == 1) {
            sa[0] = *reinterpret_cast<const float *>(sb + soff);
            sc[0] = *reinterpret_cast<const float *>(sb + soff + 8 * C::kSpr * 4);
        } else if (kSpw == 2) {
            const float2 va = *reinterpret_cast<const float2 *>(sb + soff);
            const float2 vb = *reinterpret_cast<const float2 *>(sb + soff + 8 * C::kSpr * 4);
            sa[0] = va.x; sa[1 % kSpw] = va.y;
            sc[0] = vb.x; sc[1 % kSpw] = vb.y;
        } else {
#pragma unroll
            for (int v = 0; v < kSpw / 4; v++) {
                const float4 va = *reinterpret_cast<const float4 *>(sb + soff + 16 * v);
                const float4 vb = *reinterpret_cast<const float4 *>(sb + soff + 8 * C::kSpr * 4 + 16 * v);
                sa[4 * v + 0] = va.x; sa[(4 * v + 1) % kSpw] = va.y;
                sa[(4 * v + 2) % kSpw] = va.z; sa[(4 * v + 3) % kSpw] = va.w;
                sc[4 * v + 0] = vb.x; sc[(4 * v + 1) % kSpw] = vb.y;
                sc[(4 * v + 2) % kSpw] = vb.z; sc[(4 * v + 3) % kSpw] = vb.w;
            }
        }
        // one-token passes: the stage's group corrections (and, down, the h factors) of each
        // n-tile's tokens are read with 16-byte loads before the group loop, not one per group
        constexpr bool kHoist = TOK == 1 && kGpw % 2 == 0;
        float2 ccv[kHoist ? NT : 1][kHoist ? kGpw : 1];
        float hfv[kHoist ? NT : 1][kHoist ? kGpw : 1];
        if (kHoist) {
#pragma unroll
            for (int n = 0; n < NT; n++) {
#pragma unroll
                for (int v = 0; v < kGpw / 2; v++) {
                    const float4 c4 = *reinterpret_cast<const float4 *>(sb + co(n) + 16 * v);
                    ccv[n][2 * v] = make_float2(c4.x, c4.y);
                    ccv[n][2 * v + 1] = make_float2(c4.z, c4.w);
                }
                if (MODE == kDown) {
#pragma unroll
                    for (int v = 0; v < kGpw; v += 4) {
                        if (kGpw - v >= 4) {
                            const float4 h4 = *reinterpret_cast<const float4 *>(sb + fo(n) + 4 * v);
                            hfv[n][v] = h4.x; hfv[n][(v + 1) % kGpw] = h4.y;
                            hfv[n][(v + 2) % kGpw] = h4.z; hfv[n][(v + 3) % kGpw] = h4.w;
                        } else {
                            for (int u = v; u < kGpw; u++)
                                hfv[n][u] = *reinterpret_cast<const float *>(sb + fo(n) + 4 * u);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int gi = 0; gi < kGpw; gi++) {
            const uint32_t wa = *reinterpret_cast<const uint32_t *>(sb + qoff[gi]);
            const uint32_t wb = *reinterpret_cast<const uint32_t *>(sb + qoff[gi] + 8 * C::kRowB);
            const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
            const uint32_t a0[4] = {nib_lo(wa, nk), nib_lo(wb, nk), nib_hi(wa, nk), nib_hi(wb, nk)};
            const uint32_t a1[4] = {nib_lo(wa8, nk), nib_lo(wb8, nk), nib_hi(wa8, nk), nib_hi(wb8, nk)};
#pragma unroll
            for (int n = 0; n < NT; n++) {
                const uint4 bv = *reinterpret_cast<const uint4 *>(sb + bo(n) + gi * 64);
                const float2 cc = kHoist ? ccv[n][gi] : *reinterpret_cast<const float2 *>(sb + co(n) + gi * 8);
                const float cin[4] = {cc.x, cc.y, cc.x, cc.y};
                float d[4];
                mma_f16_16816(d, a0, bv.x, bv.y, cin);
                mma_f16_16816(d, a1, bv.z, bv.w, d);
                float fa = sa[gi * 32 / GS], fb = sc[gi * 32 / GS];
                if (MODE == kDown) {
                    const float hf = kHoist ? hfv[n][gi] : *reinterpret_cast<const float *>(sb + fo(n) + gi * 4);
                    fa *= hf;
                    fb *= hf;
                }
                acc[n][0] = fmaf(fa, d[0] + d[1], acc[n][0]);
                acc[n][1] = fmaf(fb, d[2] + d[3], acc[n][1]);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&cs.empty[cs.stage]));
        if (++cs.stage == C::kStages) {
            cs.stage = 0;
            cs.phase ^= 1u;
        }
    }

    // ---- epilogue: reduce the two k-halves, then SwiGLU (+ fragments) or store y
    constexpr float kTwo24 = 16777216.0f;
    float2 *my_red = cs.red + (warp * C::kNTM) * 32 + lane;
#pragma unroll
    for (int n = 0; n < NT; n++)
        my_red[n * 32] = make_float2(acc[n][0], acc[n][1]);
    named_bar_sync(1, kConsumerWarps * 32);
    auto part = [&](int w, int n) { return cs.red[(w * C::kNTM + n) * 32 + lane]; };
    if (MODE == kGateUp) {
        const bool hw = warp == 2 || warp == 3;   // up warps of k-half 0: rows 16 * mtile + g (+ 8)
        const int rg = cs.mtile * 16 + g;
        if (hw) {
            // h for rows rg (+ 8), token t4 of each n-tile
#pragma unroll
            for (int n = 0; n < NT; n++) {
                const int tl = n * 4 + t4;
                if (tl >= ntok)
                    continue;
                const float xf = xfac[n] * kTwo24;
                const float2 g0 = part(warp - 2, n), g1 = part(warp + 2, n);
                const float2 u0 = part(warp, n), u1 = part(warp + 4, n);
                const float gva = (g0.x + g1.x) * xf, gvb = (g0.y + g1.y) * xf;
                const float uva = (u0.x + u1.x) * xf, uvb = (u0.y + u1.y) * xf;
                cs.hbuf[tl * 32 + rg] = gva / (1.0f + expf(-gva)) * uva;
                cs.hbuf[tl * 32 + rg + 8] = gvb / (1.0f + expf(-gvb)) * uvb;
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);
        // one warp per token: the item's 32 rows are one group of the down pass's reduction
        const int gpc_h = p.gpc_h;
        const int hblk = frag_blk(gpc_h);
        for (int tl = warp; tl < ntok; tl += kConsumerWarps) {
            const int tt = t0 + tl;
            float v = cs.hbuf[tl * 32 + lane];
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
            uint8_t *blk = p.h_out + (size_t)pos * p.h_row_bytes + (size_t)(it.tile / gpc_h) * hblk;
            const int gl = it.tile % gpc_h;
            const int off = gl * 64 + (lane >> 3) * 16 + frag_pos(lane & 7) * 2;
            *reinterpret_cast<uint16_t *>(blk + off) = __half_as_ushort(hi);
            *reinterpret_cast<uint16_t *>(blk + frag_lo(gpc_h) + off) = __half_as_ushort(lo);
            if (lane == 0) {
                float *cr = reinterpret_cast<float *>(blk + frag_corr(gpc_h)) + gl * 2;
                cr[0] = -chi * 0x1p-24f;
                cr[1] = -clo * 0x1p-24f;
                reinterpret_cast<float *>(blk + frag_fac(gpc_h))[gl] = mx > 0.f ? ldexpf(1.0f, e - 14) : 1.0f;
            }
        }
    } else if (warp < 4) {
        const int d = p.out_rows;
        const int row_a = it.tile * 64 + cs.mtile * 16 + g;
#pragma unroll
        for (int n = 0; n < NT; n++) {
            const int tl = n * 4 + t4;
            if (tl >= ntok)
                continue;
            const int tt = t0 + tl;
            const float2 y0 = part(warp, n), y1 = part(warp + 4, n);
            float *yrow = it.expert < 0 ? p.y_shared + (size_t)tt * d : p.y_pair + (size_t)(it.pos0 + tt) * d;
            yrow[row_a] = (y0.x + y1.x) * kTwo24;
            yrow[row_a + 8] = (y0.y + y1.y) * kTwo24;
        }
    }
    named_bar_sync(1, kConsumerWarps * 32);   // red and hbuf are reused by the next pass
}

// Weight loads (packed rows and scales) of stage `c` of an item into ring slot sb.
template <int MODE, int TOK, int CPS, int GPC, int GS>
__device__ __forceinline__ void issue_weights(const Maps &maps, const Item &it, int c, uint32_t sb, uint32_t fb,
                                              uint64_t pol)
{
    using C = Cfg<MODE, TOK, CPS, GPC, GS>;
    const int z = it.expert < 0 ? 0 : it.zq;
    const int w = it.expert < 0 ? 1 : 0;
    const int row0 = it.tile * C::kRows;
    const void *mq = &maps.q[w], *ms = &maps.s[w];
    if (maps.merged) {
        if (MODE == kGateUp) {
            tma_load_5d_hint(sb, mq, 0, row0, 0, c * CPS, z, fb, pol);
            tma_load_5d_hint(sb + C::kSOff, ms, 0, row0, 0, c * CPS, z, fb, pol);
        } else {
            tma_load_4d_hint(sb, mq, 0, row0, c * CPS, z, fb, pol);
            tma_load_4d_hint(sb + C::kSOff, ms, 0, row0, c * CPS, z, fb, pol);
        }
        return;
    }
#pragma unroll
    for (int ch = 0; ch < CPS; ch++) {
        const int cg = c * CPS + ch;
        if (MODE == kGateUp) {
            tma_load_4d_hint(sb + ch * C::kMats * C::kQSub, mq, cg * C::kRowB, row0, 0, z, fb, pol);
            tma_load_4d_hint(sb + C::kSOff + ch * C::kMats * C::kSSub, ms, cg * C::kSpr, row0, 0, z, fb, pol);
        } else {
            tma_load_3d_hint(sb + ch * C::kQSub, mq, cg * C::kRowB, row0, z, fb, pol);
            tma_load_3d_hint(sb + C::kSOff + ch * C::kSSub, ms, cg * C::kSpr, row0, z, fb, pol);
        }
    }
}

// L2 policy of an item's weights: evict_first when one pass over its tokens reads them once;
// an item taken in several passes reads them again from L2, so they are cached normally.
template <int TOK>
__device__ __forceinline__ uint64_t weight_policy(int m)
{
    return m <= TOK ? l2_policy_evict_first() : l2_policy_evict_normal();
}

template <int MODE, int TOK, int CPS, int GPC, int GS>
__global__ void __launch_bounds__(kThreads, 2)
ffn_decode_kernel(const __grid_constant__ Maps maps, const Params p)
{
    using C = Cfg<MODE, TOK, CPS, GPC, GS>;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t full_bar[C::kStages];
    __shared__ __align__(8) uint64_t empty_bar[C::kStages];
    __shared__ int stage_item[C::kStages];   // item of the stage in each slot (-1: no more items)
    __shared__ volatile int abort_flag;

    const uint32_t raw = smem_addr(dyn_smem);
    const uint32_t stage0 = (raw + 1023u) & ~1023u;
    uint8_t *base = dyn_smem + (stage0 - raw);

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
        for (int i = 0; i < 2; i++) {
            prefetch_tmap(&maps.q[i]);
            prefetch_tmap(&maps.s[i]);
        }
    __syncthreads();
    const int nstages = p.nchunks / CPS;
    Unit *tab = reinterpret_cast<Unit *>(base + C::kStages * C::kStageBytes + C::kRedBytes + C::kHBufBytes);

    // Before waiting on the previous kernel, start the weight loads of the first stages of this
    // CTA's first item when that item is already known: every down item (the union was complete
    // before the gate/up kernel released this one), and a gate/up item of the shared expert
    // (items 0 .. tiles - 1, whatever the union).  Weights do not depend on the previous kernel.
    int units = 0;
    if (MODE == kDown) {
        units = min(max(__ldcg(p.n_uniq), 0), p.max_uniq) + p.with_shared;
        load_units(p, units, tab);
        __syncthreads();
    }
    int pre = 0;   // producer: stages of the first item's first pass already holding their weights
    if (warp == kProducerWarp) {
        const bool known = MODE == kDown ? (int)blockIdx.x < units * p.tiles
                                         : (p.with_shared && (int)blockIdx.x < p.tiles);
        if (known) {
            Item it0;
            if (MODE == kDown) {
                it0 = decode_item(p, tab, blockIdx.x);
            } else {
                it0.expert = -1;
                it0.zq = 0;
                it0.tile = blockIdx.x;
                it0.m = p.T;
                it0.pos0 = 0;
            }
            // an item without tokens (a unit the bounds checks of a MOE_DEBUG_BOUNDS build emptied) has
            // no pass: nothing to pre-issue, and the main loop below skips it the same way
            if (it0.m > 0) {
                int t0, ntok;
                pass_range(it0.m, (it0.m + TOK - 1) / TOK, 0, t0, ntok);
                pre = nstages < C::kStages ? nstages : C::kStages;
                if (lane == 0) {
                    const uint64_t pol = weight_policy<TOK>(it0.m);
                    for (int c = 0; c < pre; c++) {
                        const uint32_t fb = smem_addr(&full_bar[c]);
                        stage_item[c] = blockIdx.x;
                        mbar_arrive_expect_tx(fb, C::kWeightBytes + ntok * C::kTokBytes);
                        issue_weights<MODE, TOK, CPS, GPC, GS>(maps, it0, c, stage0 + c * C::kStageBytes, fb, pol);
                    }
                }
            }
        }
    }
    if (MODE == kGateUp) {
        // the down kernel reads the union before its own grid wait: release it only after ours
        griddep_wait();   // routing, union and activation fragments come from the previous kernels
        griddep_launch_dependents();
        units = min(max(*p.n_uniq, 0), p.max_uniq) + p.with_shared;
        load_units(p, units, tab);
        __syncthreads();
    } else {
        griddep_launch_dependents();
        griddep_wait();   // h comes from the gate/up kernel
    }
    const int n_items = units * p.tiles;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------- producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = (1u << pre) - 1u;   // bit s: stage s was filled at least once
        bool first = true;
        int i = blockIdx.x;
        while (i < n_items) {
            // claim the next item now: the atomic's round trip overlaps this item's loads
            int next = i + (int)gridDim.x;
            if (lane == 0 && p.dynamic)
                next = (int)gridDim.x + atomicAdd(p.work, 1);
            const Item it = decode_item(p, tab, i);
            const int npass = (it.m + TOK - 1) / TOK;
            const uint64_t pol = weight_policy<TOK>(it.m);
            for (int pass = 0; pass < npass; pass++) {
                int t0, ntok;
                pass_range(it.m, npass, pass, t0, ntok);
                // lane j < ntok copies the fragment blocks of token j of this pass; its row is looked up
                // after the first stage's weight loads are issued, so the lookup overlaps them
                const uint8_t *src = p.act;
                const uint32_t tx = C::kWeightBytes + ntok * C::kTokBytes;
                for (int c = 0; c < nstages; c++) {
                    const bool pre_issued = first && pass == 0 && c < pre;
                    if (lane == 0 && !abort_flag && !pre_issued) {
                        if (!mbar_wait_or_abort(smem_addr(&empty_bar[stage]), phase ^ 1u, &abort_flag)) {
                            atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                            abort_flag = 1;
                        }
                    }
                    __syncwarp();
                    if (!abort_flag) {
                        const uint32_t sb = stage0 + stage * C::kStageBytes;
                        const uint32_t fb = smem_addr(&full_bar[stage]);
                        if (lane == 0 && !pre_issued) {
                            stage_item[stage] = i;   // published to the consumers by the arrive below
                            mbar_arrive_expect_tx(fb, tx);
                            issue_weights<MODE, TOK, CPS, GPC, GS>(maps, it, c, sb, fb, pol);
                            issued |= 1u << stage;
                        }
                        if (c == 0 && lane < ntok)
                            src += (size_t)act_row<MODE>(p, it, t0 + lane) * p.act_row_bytes;
                        __syncwarp();   // expect_tx is posted before any copy below can complete
                        if (lane < ntok)
                            bulk_load(sb + C::kBOff + lane * C::kTokBytes, src + (size_t)c * C::kTokBytes,
                                      C::kTokBytes, fb);
                    }
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            first = false;
            i = __shfl_sync(0xffffffffu, next, 0);
        }
        // no more items: one more slot, tagged -1 and completed without data, stops the consumers
        // (only when they follow the tags; in the fixed order they know where to stop)
        if (p.dynamic && lane == 0 && !abort_flag) {
            if (!mbar_wait_or_abort(smem_addr(&empty_bar[stage]), phase ^ 1u, &abort_flag)) {
                atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                abort_flag = 1;
            } else {
                stage_item[stage] = -1;
                mbar_arrive(smem_addr(&full_bar[stage]));
                issued |= 1u << stage;
            }
        }
        __syncwarp();
        if (p.dynamic && ++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
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
    // warp -> (matrix, 16-row m-tile, half of every stage's groups)
    Consumer cs;
    cs.base = base;
    cs.full = full_bar;
    cs.empty = empty_bar;
    cs.abort = &abort_flag;
    cs.red = reinterpret_cast<float2 *>(base + C::kStages * C::kStageBytes);
    cs.hbuf = reinterpret_cast<float *>(base + C::kStages * C::kStageBytes + C::kRedBytes);
    cs.warp = warp;
    cs.lane = lane;
    cs.g = lane >> 2;
    cs.t4 = lane & 3;
    cs.stage = 0;
    cs.phase = 0;
    const int mt = warp & 3, khalf = warp >> 2;
    const int mat = MODE == kGateUp ? (mt >> 1) : 0;
    cs.mtile = MODE == kGateUp ? (mt & 1) : mt;
    const int ra = cs.mtile * 16 + cs.g;   // and ra + 8: same swizzle phase
    // this warp's groups of a stage: chunk ch0, groups gl0 .. gl0 + kGpw - 1
    const int ch0 = CPS == 2 ? khalf : 0;
    const int gl0 = CPS == 2 ? 0 : khalf * C::kGpw;
    uint32_t qoff[C::kGpw];
#pragma unroll
    for (int gi = 0; gi < C::kGpw; gi++)
        qoff[gi] = (ch0 * C::kMats + mat) * C::kQSub + ra * C::kRowB + (((gl0 + gi) ^ swz<GPC>(ra)) << 4) +
                   4 * cs.t4;
    const uint32_t soff = C::kSOff + (ch0 * C::kMats + mat) * C::kSSub + (ra * C::kSpr + gl0 * 32 / GS) * 4;
    const uint32_t kb = ch0 * C::kBlk + gl0 * 64;
    const uint32_t kbc = ch0 * C::kBlk + frag_corr(GPC) + gl0 * 8;
    const uint32_t kbf = ch0 * C::kBlk + frag_fac(GPC) + gl0 * 4;
    const uint32_t plane_off = (cs.g & 1) * frag_lo(GPC) + cs.t4 * 16;

    for (int ii = blockIdx.x;; ii += gridDim.x) {
        int i = ii;
        if (p.dynamic) {
            // the next slot's tag names its item (the first stage of that item: the passes below then
            // wait on this slot again, which returns at once)
            if (!mbar_wait_or_abort(smem_addr(&full_bar[cs.stage]), cs.phase, &abort_flag)) {
                if (lane == 0)
                    atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                abort_flag = 1;
                break;
            }
            i = stage_item[cs.stage];
            if (i < 0)
                break;
        } else if (i >= n_items) {
            break;   // fixed order: CTA c takes c, c + G, ...
        }
        const Item it = decode_item(p, tab, i);
        const int npass = (it.m + TOK - 1) / TOK;
        for (int pass = 0; pass < npass; pass++) {
            int t0, ntok;
            pass_range(it.m, npass, pass, t0, ntok);
            const int nt = (ntok + 3) >> 2;
            if (nt <= 1)
                run_pass<MODE, TOK, CPS, GPC, GS, 1>(p, it, t0, ntok, cs, qoff, soff, kb, kbc, kbf, plane_off);
            else if (C::kNTM >= 2 && nt == 2)
                run_pass<MODE, TOK, CPS, GPC, GS, (C::kNTM >= 2 ? 2 : 1)>(p, it, t0, ntok, cs, qoff, soff, kb, kbc,
                                                                      kbf, plane_off);
            else if (C::kNTM >= 3 && nt == 3)
                run_pass<MODE, TOK, CPS, GPC, GS, (C::kNTM >= 3 ? 3 : 1)>(p, it, t0, ntok, cs, qoff, soff, kb, kbc,
                                                                      kbf, plane_off);
            else
                run_pass<MODE, TOK, CPS, GPC, GS, C::kNTM>(p, it, t0, ntok, cs, qoff, soff, kb, kbc, kbf, plane_off);
        }
    }
}

template <int MODE, int TOK, int CPS, int GPC, int GS>
int launch_one(const Maps &maps, const Params &prm, int max_items, int max_units, cudaStream_t s)
{
    // a merged box spans maps.cps chunks and lands in one stage: a kernel laid out for another count
    // would take more bytes into a stage than it holds
    if (maps.merged && maps.cps != CPS)
        return MOE_ERR_INVALID_ARG;
    using C = Cfg<MODE, TOK, CPS, GPC, GS>;
    auto kern = ffn_decode_kernel<MODE, TOK, CPS, GPC, GS>;
    const size_t smem = C::kSmem + ((size_t)max_units * sizeof(Unit) + 15) / 16 * 16;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return MOE_ERR_CUDA;
    // per device: opt in to the largest dynamic shared memory once; cache the occupancy of the last
    // shared-memory size as one atomic word (smem << 8 | blocks per SM), so host threads calling
    // together at worst repeat the query
    static std::atomic<int> opted[64];
    static std::atomic<uint64_t> occ[64];
    if (!opted[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(C::kSmem + 1025 * sizeof(Unit) + 16)) != cudaSuccess)
            return MOE_ERR_CUDA;
        opted[dev].store(1, std::memory_order_release);
    }
    const uint64_t oc = occ[dev].load(std::memory_order_relaxed);
    int per_sm = (oc >> 8) == (uint64_t)smem ? (int)(oc & 0xff) : 0;
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        if (per_sm > 255)
            per_sm = 255;
        occ[dev].store(((uint64_t)smem << 8) | (uint64_t)per_sm, std::memory_order_relaxed);
    }
    int grid = per_sm * sm_count(dev);
    if (grid > max_items)
        grid = max_items;
    if (grid < 1)
        grid = 1;
    return launch_pdl(kern, grid, kThreads, smem, s, maps, prm);
}

// Pass width by batch size: one token per pass for T = 1 (two k-chunks per
// stage when the chunk count is even), else up to 4, 8 or 16 tokens.
template <int MODE, int GPC, int GS>
int launch_tok(const Maps &maps, const Params &prm, int max_units, int T, cudaStream_t s)
{
    const int mi = max_units * prm.tiles;
    if (T == 1)
        return prm.nchunks % 2 == 0 ? launch_one<MODE, 1, 2, GPC, GS>(maps, prm, mi, max_units, s)
                                    : launch_one<MODE, 1, 1, GPC, GS>(maps, prm, mi, max_units, s);
    if (T <= 4)
        return launch_one<MODE, 4, 1, GPC, GS>(maps, prm, mi, max_units, s);
    // 8 tokens per pass up to T = 32 (measured faster than 16 at T = 16 and 32: fewer registers,
    // no spills); above, 16 for gate/up, so that an expert taken by many tokens is streamed fewer
    // times, and still 8 for down, whose items are a third as long (a 64-token Zipf batch: 4.2 %
    // faster than 16 for both, 3 % faster than 8 for both)
    if constexpr (MODE == kDown) {
        return launch_one<MODE, 8, 1, GPC, GS>(maps, prm, mi, max_units, s);
    } else {
        if (T <= 32)
            return launch_one<MODE, 8, 1, GPC, GS>(maps, prm, mi, max_units, s);
        return launch_one<MODE, 16, 1, GPC, GS>(maps, prm, mi, max_units, s);
    }
}

}  // namespace

int launch_ffn_decode(const DecodeFfnArgs &a, cudaStream_t s)
{
    const moe_layer_int4 &w = *a.w;
    const int d = w.d, f = w.f, E = w.E, G = w.G;
    const uint64_t qb = (uint64_t)moe_expert_q_bytes(d, f);
    const uint64_t sc = (uint64_t)moe_expert_s_count(d, f, G);
    const int gpc_h = frag_gpc_h(f);
    const CUtensorMapSwizzle sw_dn = gpc_h == 8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const int max_experts = (E < a.T * a.k ? E : a.T * a.k) + 1;
    int rc = MOE_OK;

    // ---- tensor maps: merged (chunk as a map dimension) when the driver accepts them, else per chunk
    const uint8_t *qs[2] = {w.q_base, w.shared_q};
    const float *ss[2] = {w.s_base, w.shared_s};
    const uint64_t outer[2] = {(uint64_t)E, 1};
    const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8, F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int cps_gu = (a.T == 1 && (d / 256) % 2 == 0) ? 2 : 1;
    const int cps_dn = (a.T == 1 && (f / (32 * gpc_h)) % 2 == 0) ? 2 : 1;
    // scales per row of a chunk: a gate/up chunk is 256 elements, a down chunk 32 * gpc_h
    const uint32_t spr_gu = 256 / G, spr_dn = 32 * gpc_h / G;
    if (spr_dn * 4 % 16 != 0)
        return MOE_ERR_UNSUPPORTED;   // a scale box row must be a multiple of 16 bytes
    Maps gu{}, dn{};
    gu.merged = dn.merged = 1;
    gu.cps = cps_gu;
    dn.cps = cps_dn;
    for (int i = 0; i < 2 && rc == MOE_OK; i++) {
        // gate/up: (bytes of a chunk, row, matrix, chunk, expert)
        const uint64_t gq_dim[5] = {128, (uint64_t)f, 2, (uint64_t)d / 256, outer[i]};
        const uint64_t gq_str[4] = {(uint64_t)d / 2, (uint64_t)f * d / 2, 128, qb};
        const uint32_t gq_box[5] = {128, 32, 2, (uint32_t)cps_gu, 1};
        const uint64_t gs_dim[5] = {spr_gu, (uint64_t)f, 2, (uint64_t)d / 256, outer[i]};
        const uint64_t gs_str[4] = {(uint64_t)(d / G) * 4, (uint64_t)f * (d / G) * 4, spr_gu * 4, sc * 4};
        const uint32_t gs_box[5] = {spr_gu, 32, 2, (uint32_t)cps_gu, 1};
        // down: (bytes of a chunk, row, chunk, expert)
        const uint64_t dq_dim[4] = {(uint64_t)16 * gpc_h, (uint64_t)d, (uint64_t)f / (32 * gpc_h), outer[i]};
        const uint64_t dq_str[3] = {(uint64_t)f / 2, (uint64_t)16 * gpc_h, qb};
        const uint32_t dq_box[4] = {(uint32_t)16 * gpc_h, 64, (uint32_t)cps_dn, 1};
        const uint64_t ds_dim[4] = {spr_dn, (uint64_t)d, (uint64_t)f / (32 * gpc_h), outer[i]};
        const uint64_t ds_str[3] = {(uint64_t)(f / G) * 4, (uint64_t)spr_dn * 4, sc * 4};
        const uint32_t ds_box[4] = {spr_dn, 64, (uint32_t)cps_dn, 1};
        if (gu.merged)
            gu.merged = make_tmap_nd(&gu.q[i], qs[i], U8, 5, gq_dim, gq_str, gq_box, CU_TENSOR_MAP_SWIZZLE_128B) ==
                            MOE_OK &&
                        make_tmap_nd(&gu.s[i], ss[i], F32, 5, gs_dim, gs_str, gs_box, CU_TENSOR_MAP_SWIZZLE_NONE) ==
                            MOE_OK;
        if (dn.merged)
            dn.merged = make_tmap_nd(&dn.q[i], qs[i] + (size_t)f * d, U8, 4, dq_dim, dq_str, dq_box, sw_dn) ==
                            MOE_OK &&
                        make_tmap_nd(&dn.s[i], ss[i] + (size_t)2 * f * d / G, F32, 4, ds_dim, ds_str, ds_box,
                                     CU_TENSOR_MAP_SWIZZLE_NONE) == MOE_OK;
    }
    for (int i = 0; i < 2 && !gu.merged && rc == MOE_OK; i++) {
        // per chunk: (row bytes, row, matrix, expert)
        const uint64_t q_dim[4] = {(uint64_t)d / 2, (uint64_t)f, 2, outer[i]};
        const uint64_t q_str[3] = {(uint64_t)d / 2, (uint64_t)f * d / 2, qb};
        const uint32_t q_box[4] = {128, 32, 2, 1};
        const uint64_t s_dim[4] = {(uint64_t)d / G, (uint64_t)f, 2, outer[i]};
        const uint64_t s_str[3] = {(uint64_t)(d / G) * 4, (uint64_t)f * (d / G) * 4, sc * 4};
        const uint32_t s_box[4] = {spr_gu, 32, 2, 1};
        rc |= make_tmap_nd(&gu.q[i], qs[i], U8, 4, q_dim, q_str, q_box, CU_TENSOR_MAP_SWIZZLE_128B);
        rc |= make_tmap_nd(&gu.s[i], ss[i], F32, 4, s_dim, s_str, s_box, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    for (int i = 0; i < 2 && !dn.merged && rc == MOE_OK; i++) {
        rc |= make_tmap_3d(&dn.q[i], qs[i] + (size_t)f * d, U8, 1, f / 2, d, outer[i], f / 2, qb, 16 * gpc_h, 64,
                           sw_dn);
        rc |= make_tmap_3d(&dn.s[i], ss[i] + (size_t)2 * f * d / G, F32, 4, f / G, d, outer[i],
                           (uint64_t)(f / G) * 4, sc * 4, spr_dn, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (rc != MOE_OK)
        return MOE_ERR_INVALID_ARG;
    Params pg{};
    pg.offsets = a.offsets;
    pg.sorted_pair = a.sorted_pair;
    pg.uniq = a.uniq;
    pg.n_uniq = a.n_uniq;
    pg.act = a.x_frag;
    pg.act_row_bytes = frag_row_bytes(d, 8);
    pg.x_scale = a.x_scale;
    pg.h_out = a.h_frag;
    pg.h_row_bytes = frag_row_bytes(f, gpc_h);
    pg.gpc_h = gpc_h;
    pg.work = a.work;
    pg.slot_of = a.slot_of;
    pg.with_shared = a.with_shared;
    // T = 1: every unit has one token and the items are equal, so the fixed order c, c + G, ...
    // balances them as well as claiming would (and saves the atomics, measured 2 us faster per
    // layer); larger batches give units of very different lengths: claim dynamically
    pg.dynamic = a.T > 1 ? 1 : 0;
    pg.err = a.err;
    pg.T = a.T;
    pg.k = a.k;
    pg.nchunks = d / 256;
    pg.tiles = f / 32;
    pg.out_rows = f;
    pg.n_experts = a.n_experts > 0 ? a.n_experts : E;
    pg.n_view = E;
    pg.max_uniq = max_experts - 1;
    // pass width from the most tokens a listed expert can have (the hybrid's decode half: at most 8)
    const int tsel = a.max_tokens > 0 && a.max_tokens < a.T ? a.max_tokens : a.T;
    rc = G == 64 ? launch_tok<kGateUp, 8, 64>(gu, pg, max_experts, tsel, s)
                 : launch_tok<kGateUp, 8, 32>(gu, pg, max_experts, tsel, s);
    if (rc != MOE_OK)
        return rc;

    Params pd = pg;
    pd.act = a.h_frag;
    pd.act_row_bytes = frag_row_bytes(f, gpc_h);
    pd.x_scale = nullptr;
    pd.h_out = nullptr;
    pd.y_pair = a.y_pair;
    pd.y_shared = a.y_shared;
    pd.work = a.work + 1;

    pd.nchunks = f / (32 * gpc_h);
    pd.tiles = d / 64;
    pd.out_rows = d;
    if (gpc_h == 8)
        return G == 64 ? launch_tok<kDown, 8, 64>(dn, pd, max_experts, tsel, s)
                       : launch_tok<kDown, 8, 32>(dn, pd, max_experts, tsel, s);
    return launch_tok<kDown, 4, 32>(dn, pd, max_experts, tsel, s);   // G = 64 needs gpc_h = 8 (checked above)
}

}  // namespace moe
