// router.cu -- Route stage: fp32 router logits, sigmoid + bias-keyed top-k with
// score weights, and the activation fragments the decode FFN consumes.
//
// Source: "Public Colibri Observation and Revision Ledger", "Exact Architecture
// and Data-Flow Reconstruction": a trained sigmoid gate (n_group = 1, fp32
// parameters) scores every expert of the layer for each token and the top
// experts are selected.
#include <cuda_fp16.h>
#include <cfloat>
#include <climits>

#include "moe_internal.h"
#include "ptx.cuh"
#include "route_common.cuh"

namespace moe {
namespace {

constexpr int kFragThreads = 256;   // threads of act_frag_kernel
constexpr int kXGpc = 8;            // scale groups per fragment block of x

__device__ __forceinline__ void frag_quad(const float *__restrict__ xr, float mx, int id, bool act,
                                          uint8_t *__restrict__ row);
__device__ __forceinline__ float absmax4(float4 v)
{
    return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// ----------------------------------------------------------------- logits ---
// Small T: each CTA owns kEB experts x kTB tokens and splits the reduction
// over d across its 256 threads (float4 loads), then reduces in a fixed order.
constexpr int kEB = 2, kTB = 8, kSkinnyThreads = 256;
constexpr int kSkinnyIt = 8;   // d up to 8192: the weight slice of a thread stays in registers

__global__ void __launch_bounds__(kSkinnyThreads)
logits_skinny_kernel(const float *__restrict__ x, const float *__restrict__ wg, int T, int d, int E,
                     float *__restrict__ logits, uint8_t *frag, float *row_scale, int32_t *zero, int nzero)
{
    griddep_launch_dependents();
    const int e0 = blockIdx.x * kEB;
    const int t0 = blockIdx.y * kTB;
    const int nt = min(kTB, T - t0);
    const int ne = min(kEB, E - e0);
    const int d4 = d / 4;
    float acc[kEB][kTB];
#pragma unroll
    for (int a = 0; a < kEB; a++)
#pragma unroll
        for (int b = 0; b < kTB; b++)
            acc[a][b] = 0.f;
    const float4 *w4 = reinterpret_cast<const float4 *>(wg);
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    auto fma4 = [&](const float4 &xv, const float4 &wv, float &a) {
        a = fmaf(xv.x, wv.x, a);
        a = fmaf(xv.y, wv.y, a);
        a = fmaf(xv.z, wv.z, a);
        a = fmaf(xv.w, wv.w, a);
    };
    // per-thread max |x| of each token (the fused path's fragments need the row maxima)
    float xmax[kTB];
#pragma unroll
    for (int b = 0; b < kTB; b++)
        xmax[b] = 0.f;
    if (d4 <= kSkinnyIt * kSkinnyThreads) {
        // the router weights do not depend on the previous kernel: all of this thread's loads are
        // issued before waiting on it
        // read once per call when one block of tokens covers the batch: evict_first (see
        // l2_policy_evict_first); several token blocks read the same slice, so it stays cached
        const uint64_t pol = gridDim.y == 1 ? l2_policy_evict_first() : l2_policy_evict_normal();
        float4 wv[kSkinnyIt][kEB];
#pragma unroll
        for (int it = 0; it < kSkinnyIt; it++) {
            const int i = threadIdx.x + it * kSkinnyThreads;
#pragma unroll
            for (int a = 0; a < kEB; a++)
                wv[it][a] = (i < d4 && a < ne) ? ldg_hint(w4 + (size_t)(e0 + a) * d4 + i, pol)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        griddep_wait();   // x may come from the previous kernel in the stream
        // a token's whole slice of x is loaded before any of it is used: one round trip per token
#pragma unroll
        for (int b = 0; b < kTB; b++) {
            if (b >= nt)
                continue;
            float4 xv[kSkinnyIt];
#pragma unroll
            for (int it = 0; it < kSkinnyIt; it++) {
                const int i = threadIdx.x + it * kSkinnyThreads;
                xv[it] = i < d4 ? __ldg(x4 + (size_t)(t0 + b) * d4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int it = 0; it < kSkinnyIt; it++) {
                const int i = threadIdx.x + it * kSkinnyThreads;
                if (i < d4) {
#pragma unroll
                    for (int a = 0; a < kEB; a++)
                        fma4(xv[it], wv[it][a], acc[a][b]);
                    xmax[b] = fmaxf(xmax[b], absmax4(xv[it]));
                }
            }
        }
    } else {
        griddep_wait();
        for (int i = threadIdx.x; i < d4; i += kSkinnyThreads) {
            float4 wv[kEB];
#pragma unroll
            for (int a = 0; a < kEB; a++)
                wv[a] = a < ne ? __ldg(w4 + (size_t)(e0 + a) * d4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int b = 0; b < kTB; b++)
                if (b < nt) {
                    const float4 xv = __ldg(x4 + (size_t)(t0 + b) * d4 + i);
#pragma unroll
                    for (int a = 0; a < kEB; a++)
                        fma4(xv, wv[a], acc[a][b]);
                    xmax[b] = fmaxf(xmax[b], absmax4(xv));
                }
        }
    }
    __shared__ float part[kSkinnyThreads / 32][kEB * kTB];
    __shared__ float pmax[kSkinnyThreads / 32][kTB];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int b = 0; b < kTB; b++) {
        if (b >= nt)
            continue;
#pragma unroll
        for (int a = 0; a < kEB; a++) {
            float v = acc[a][b];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0)
                part[warp][a * kTB + b] = v;
        }
        if (frag != nullptr) {
            float m = xmax[b];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (lane == 0)
                pmax[warp][b] = m;
        }
    }
    __syncthreads();
    if (threadIdx.x < kEB * kTB) {
        const int a = threadIdx.x / kTB, b = threadIdx.x % kTB;
        if (a < ne && b < nt) {
            float v = 0.f;
            for (int w = 0; w < kSkinnyThreads / 32; w++)
                v += part[w][threadIdx.x];
            logits[(size_t)(t0 + b) * E + e0 + a] = v;
        }
    }
    // fused path: block (0, 0) zeroes the FFN's counters (this is after the grid wait: the previous
    // layer's FFN, which used them, has finished), and the blocks build the FFN's fragments of x:
    // every block has the row maxima, and each converts an equal share of the (token, group) units,
    // four threads (one per quad of 8 elements) per unit
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < nzero; i += blockDim.x)
            zero[i] = 0;
    if (frag != nullptr && blockIdx.y == 0) {
        const int G = d / 32;
        const int nu = nt * G;
        const int per = (nu + gridDim.x - 1) / gridDim.x;
        const int u0 = min(nu, (int)blockIdx.x * per), u1 = min(nu, u0 + per);
        if (blockIdx.x == 0 && threadIdx.x < nt) {
            float mx = 0.f;
            for (int w = 0; w < kSkinnyThreads / 32; w++)
                mx = fmaxf(mx, pmax[w][threadIdx.x]);
            int e = 0;
            frexpf(mx, &e);
            row_scale[t0 + threadIdx.x] = mx > 0.f ? ldexpf(1.0f, e - 14) : 1.0f;
        }
        for (int base = u0; base < u1; base += kSkinnyThreads / 4) {   // uniform over the block
            const int u = base + (int)(threadIdx.x >> 2);
            const bool act = u < u1;
            const int b = act ? u / G : 0, g = act ? u - b * G : 0;
            float mx = 0.f;
            for (int w = 0; w < kSkinnyThreads / 32; w++)
                mx = fmaxf(mx, pmax[w][b]);
            frag_quad(x + (size_t)(t0 + b) * d, mx, g * 4 + (int)(threadIdx.x & 3), act,
                      frag + (size_t)(t0 + b) * frag_row_bytes(d, kXGpc));
        }
    }
}

// Large T: register-tiled fp32 GEMM, C[T][E] = X[T][d] * Wg[E][d]^T.
// 64 x 64 tile per CTA, 256 threads x (4 x 4), k-slabs of 16 staged in shared
// memory (transposed so both operands are read as float4 broadcasts).
constexpr int kBM = 64, kBN = 64, kBK = 16;
constexpr int kTcMinTokens = 128;   // from here on the tensor-core kernel below is used

__global__ void __launch_bounds__(256)
logits_tiled_kernel(const float *__restrict__ x, const float *__restrict__ wg, int T, int d, int E,
                    float *__restrict__ logits)
{
    __shared__ __align__(16) float As[2][kBK][kBM];
    __shared__ __align__(16) float Bs[2][kBK][kBN];
    const int tid = threadIdx.x;
    const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
    const int lr = tid >> 2, lk = (tid & 3) * 4;   // loader: row within tile, k offset
    const int tm = (tid >> 4) * 4, tn = (tid & 15) * 4;
    float acc[4][4] = {};
    const bool a_ok = m0 + lr < T, b_ok = n0 + lr < E;
    const float *ap = x + (size_t)(m0 + lr) * d + lk;
    const float *bp = wg + (size_t)(n0 + lr) * d + lk;
    float4 ra = a_ok ? __ldg(reinterpret_cast<const float4 *>(ap)) : make_float4(0, 0, 0, 0);
    float4 rb = b_ok ? __ldg(reinterpret_cast<const float4 *>(bp)) : make_float4(0, 0, 0, 0);
    const int nk = d / kBK;
    for (int kt = 0; kt < nk; kt++) {
        const int buf = kt & 1;
        As[buf][lk + 0][lr] = ra.x; As[buf][lk + 1][lr] = ra.y;
        As[buf][lk + 2][lr] = ra.z; As[buf][lk + 3][lr] = ra.w;
        Bs[buf][lk + 0][lr] = rb.x; Bs[buf][lk + 1][lr] = rb.y;
        Bs[buf][lk + 2][lr] = rb.z; Bs[buf][lk + 3][lr] = rb.w;
        __syncthreads();
        if (kt + 1 < nk) {
            ra = a_ok ? __ldg(reinterpret_cast<const float4 *>(ap + (kt + 1) * kBK)) : make_float4(0, 0, 0, 0);
            rb = b_ok ? __ldg(reinterpret_cast<const float4 *>(bp + (kt + 1) * kBK)) : make_float4(0, 0, 0, 0);
        }
#pragma unroll
        for (int kk = 0; kk < kBK; kk++) {
            const float4 av = *reinterpret_cast<const float4 *>(&As[buf][kk][tm]);
            const float4 bv = *reinterpret_cast<const float4 *>(&Bs[buf][kk][tn]);
            const float a4[4] = {av.x, av.y, av.z, av.w}, b4[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++)
                    acc[i][j] = fmaf(a4[i], b4[j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++)
            if (m0 + tm + i < T && n0 + tn + j < E)
                logits[(size_t)(m0 + tm + i) * E + n0 + tn + j] = acc[i][j];
}

// Large T on the tensor cores: split-tf32 GEMM.  Every fp32 operand is split
// into hi = tf32(v) and lo = tf32(v - hi) (together within about 2^-22 of v,
// with fp32's range, so no scaling is needed), and
//   x . w = x_hi w_hi + x_hi w_lo + x_lo w_hi (+ x_lo w_lo, below 2^-22, dropped)
// takes three kind::tf32 MMAs per k8 step.  The tensor cores' fp32
// accumulation does not round to nearest, and its error grows with the number
// of accumulation steps, so tensor memory holds only the partial sum of a
// short run of k (kRChunk stages, 24 MMAs); drain warps add the partials in
// fp32 registers, rounding to nearest, while the MMAs of the next run go to
// the other accumulator.
// A cluster of two CTAs covers 128 tokens x 128 experts: each CTA one half of
// the reduction, the second CTA's sums added to the first's through distributed
// shared memory (in a fixed order: the result does not depend on timing).
// 32 reduction elements per stage (one 128-byte
// swizzled row of fp32 per token/expert).  Two rings: the raw ring takes the
// TMA loads (fp32 x and w), the operand ring the split values (x hi, w hi,
// x lo, w lo in the same swizzled layout); a raw stage is free again as soon
// as the split warps hold it in registers, so the loads run ahead of the MMAs
// by the whole raw ring.  Warp 0: TMA producer; warp 1: MMA issue (whole
// warp, one elected lane) and tensor-memory owner; warps 2-5: split; warps
// 6-9: drain the partials (one TMEM subpartition each) and write the logits.
// Waits are bounded; a CTA that timed out writes NaN logits (the routing call
// has no error word).
constexpr int kRM = 128, kRN = 128, kRK = 32, kRThreads = 320, kRChunk = 2, kRSplit = 2;
constexpr int kRRaw = 3, kROps = 2;                           // raw and operand stages
constexpr int kRXB = kRM * kRK * 4, kRWB = kRN * kRK * 4;   // 16 KB, 16 KB
constexpr int kRRawStage = kRXB + kRWB;                       // x, w
constexpr int kROpStage = 2 * (kRXB + kRWB);                  // x hi, w hi, x lo, w lo
constexpr size_t kRSmem = 1024 + (size_t)kRRaw * kRRawStage + (size_t)kROps * kROpStage;

__global__ void __launch_bounds__(kRThreads, 1)
logits_tc_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw, int T, int d,
                 int E, float *__restrict__ logits)
{
    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t full[kRRaw], rfree[kRRaw], conv[kROps], empty[kROps], accf[2], acce[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;
    const uint32_t base = (smem_addr(dyn_smem) + 1023u) & ~1023u;
    uint8_t *gbase = dyn_smem + (base - smem_addr(dyn_smem));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRRaw; s++) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&rfree[s]), 128);
        }
        for (int s = 0; s < kROps; s++) {
            mbar_init(smem_addr(&conv[s]), 128);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(smem_addr(&accf[b]), 1);
            mbar_init(smem_addr(&acce[b]), 128);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&tmem_base_sh), 2 * kRN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const uint32_t rank = cluster_rank();           // which half of the reduction
    const int m0 = blockIdx.y * kRM, n0 = (blockIdx.x / kRSplit) * kRN;
    const int nk = d / kRK / kRSplit;               // stages of this CTA
    const int k0 = (int)rank * nk * kRK;            // first reduction element
    const int nchunk = (nk + kRChunk - 1) / kRChunk;
    const uint32_t opbase = base + kRRaw * kRRawStage;

    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < nk; kb++) {
                const int s = kb % kRRaw;
                const uint32_t ph = (uint32_t)(kb / kRRaw) & 1u;
                if (!abort_flag && !mbar_wait(smem_addr(&rfree[s]), ph ^ 1u))
                    abort_flag = 1;
                if (!abort_flag) {
                    const uint32_t sb = base + s * kRRawStage;
                    mbar_arrive_expect_tx(smem_addr(&full[s]), kRXB + kRWB);
                    tma_load_2d(sb, &mx, k0 + kb * kRK, m0, smem_addr(&full[s]));
                    tma_load_2d(sb + kRXB, &mw, k0 + kb * kRK, n0, smem_addr(&full[s]));
                }
            }
        }
    } else if (warp == 1) {
        constexpr uint32_t idesc = idesc_tf32_f32(kRM, kRN);
        for (int ch = 0; ch < nchunk; ch++) {
            const int b = ch & 1;
            int ok = 1;
            if (lane == 0)
                ok = (!abort_flag &&
                      mbar_wait_or_abort(smem_addr(&acce[b]), ((uint32_t)(ch >> 1) & 1u) ^ 1u, &abort_flag)) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok && lane == 0)
                abort_flag = 1;
            tc_fence_after();
            const uint32_t dcol = tmem + b * kRN;
            const int kb1 = min(nk, (ch + 1) * kRChunk);
            for (int kb = ch * kRChunk; kb < kb1; kb++) {
                const int s = kb % kROps;
                const uint32_t ph = (uint32_t)(kb / kROps) & 1u;
                ok = 1;
                if (lane == 0)
                    ok = (!abort_flag && mbar_wait_or_abort(smem_addr(&conv[s]), ph, &abort_flag)) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok && lane == 0)
                    abort_flag = 1;
                tc_fence_after();
                const uint32_t sb = opbase + s * kROpStage;
                const uint64_t xh = smem_desc_sw128(sb), wh = smem_desc_sw128(sb + kRXB);
                const uint64_t xl = smem_desc_sw128(sb + kRXB + kRWB), wl = smem_desc_sw128(sb + 2 * kRXB + kRWB);
#pragma unroll
                for (int j = 0; j < kRK / 8; j++) {   // k8 step j: +32 bytes = +2 in the descriptors
                    umma_tf32_elect(dcol, xh + 2 * j, wh + 2 * j, idesc, (kb > ch * kRChunk || j > 0) ? 1u : 0u);
                    umma_tf32_elect(dcol, xh + 2 * j, wl + 2 * j, idesc, 1u);
                    umma_tf32_elect(dcol, xl + 2 * j, wh + 2 * j, idesc, 1u);
                }
                umma_commit_elect(smem_addr(&empty[s]));
            }
            umma_commit_elect(smem_addr(&accf[b]));
        }
    } else if (warp < 6) {
        // split: the raw stage into registers (then free for the next load), hi and lo into the
        // operand stage at the same offsets (the swizzle is a property of the offset)
        constexpr int kV = kRRawStage / 16 / 128;   // float4 per thread per stage
        const int c = threadIdx.x - 64;   // 0 .. 127
        for (int kb = 0; kb < nk; kb++) {
            const int s = kb % kRRaw;
            const uint32_t ph = (uint32_t)(kb / kRRaw) & 1u;
            if (!abort_flag && !mbar_wait(smem_addr(&full[s]), ph))
                abort_flag = 1;
            const float4 *raw = reinterpret_cast<const float4 *>(gbase + s * kRRawStage);
            float4 v[kV];
#pragma unroll
            for (int q = 0; q < kV; q++)
                v[q] = raw[c + 128 * q];
            mbar_arrive(smem_addr(&rfree[s]));
            const int os = kb % kROps;
            const uint32_t oph = (uint32_t)(kb / kROps) & 1u;
            if (!abort_flag && !mbar_wait(smem_addr(&empty[os]), oph ^ 1u))
                abort_flag = 1;
            float4 *hi = reinterpret_cast<float4 *>(gbase + kRRaw * kRRawStage + os * kROpStage);
            float4 *lo = hi + kRRawStage / 16;
#pragma unroll
            for (int q = 0; q < kV; q++) {
                float4 h, l;
                h.x = to_tf32(v[q].x); l.x = to_tf32(v[q].x - h.x);
                h.y = to_tf32(v[q].y); l.y = to_tf32(v[q].y - h.y);
                h.z = to_tf32(v[q].z); l.z = to_tf32(v[q].z - h.z);
                h.w = to_tf32(v[q].w); l.w = to_tf32(v[q].w - h.w);
                hi[c + 128 * q] = h;
                lo[c + 128 * q] = l;
            }
            fence_proxy_async_smem();   // generic-proxy writes, read next by the tensor cores
            mbar_arrive(smem_addr(&conv[os]));
        }
    } else {
        // drain: TMEM lane = token row of the tile, columns = experts
        const int sub = warp & 3;
        float sum[kRN];
#pragma unroll
        for (int q = 0; q < kRN; q++)
            sum[q] = 0.f;
        bool ok = true;
        for (int ch = 0; ch < nchunk; ch++) {
            const int b = ch & 1;
            ok = ok && !abort_flag && mbar_wait_or_abort(smem_addr(&accf[b]), (uint32_t)(ch >> 1) & 1u, &abort_flag);
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < kRN; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(sub * 32) << 16) + b * kRN + c0, v);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 16; q++)
                    sum[c0 + q] += __uint_as_float(v[q]);
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&acce[b]));
        }
        // the second CTA leaves its sums (row = TMEM lane) in its raw ring, which is idle now
        const int row = sub * 32 + lane;
        if (rank != 0) {
            float4 *xs = reinterpret_cast<float4 *>(gbase) + (size_t)row * (kRN / 4);
#pragma unroll
            for (int q = 0; q < kRN / 4; q++)
                xs[q] = make_float4(sum[4 * q], sum[4 * q + 1], sum[4 * q + 2], sum[4 * q + 3]);
            reinterpret_cast<int *>(gbase + (size_t)kRM * kRN * 4)[row] = ok ? 1 : 0;
        }
        cluster_sync();
        if (rank == 0) {
            const uint32_t peer = map_to_rank(base, 1);
            const uint32_t prow = peer + (uint32_t)row * kRN * 4;
            const bool pok = ld_cluster_s32(peer + (uint32_t)kRM * kRN * 4 + row * 4) != 0;
            const int t = m0 + row;
            float4 *dst = reinterpret_cast<float4 *>(logits + (size_t)t * E + n0);
#pragma unroll
            for (int q = 0; q < kRN / 4; q++) {
                const float4 o = ld_cluster_f4(prow + q * 16);
                const float4 v = make_float4(sum[4 * q] + o.x, sum[4 * q + 1] + o.y, sum[4 * q + 2] + o.z,
                                             sum[4 * q + 3] + o.w);
                if (t < T)
                    dst[q] = (ok && pok) ? v : make_float4(NAN, NAN, NAN, NAN);
            }
        }
        cluster_sync();   // the peer's shared memory stays until it has been read
    }
    if (warp < 6)
        cluster_sync(), cluster_sync();   // the other roles take part in both cluster barriers
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, 2 * kRN);
    }
}

// ------------------------------------------------------------------ top-k ---
// One block per 8 tokens (topk_warp for E <= 256, else topk_block).
__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const float *__restrict__ logits, const float *__restrict__ bias, int T, int E, int k,
            int normalize, float route_scale, float top_p, int32_t *__restrict__ idx, float *__restrict__ w)
{
    extern __shared__ __align__(16) uint8_t tk_smem[];
    const int t0 = blockIdx.x * kTopkTokens;
    const int nt = min(kTopkTokens, T - t0);
    if (E <= 32 * kWarpTopkPer)
        topk_warp(logits, bias, t0, nt, E, k, normalize, route_scale, top_p, idx, w, nullptr);
    else
        topk_block(logits, bias, t0, nt, E, k, normalize, route_scale, top_p, idx, w, nullptr, tk_smem);
}

// --------------------------------------------------------- act fragments ---
// One CTA per row: the row's max |x| picks a power of two 2^(14-e) that brings
// every element below 2^14 (exact scaling); elements at odd offsets within
// each 8 are further divided by 16.  Each value becomes hi = fp16(v),
// lo = fp16(v - hi); row_scale[r] = 2^(e-14) undoes the scaling.  The row is
// written as fragment blocks of 8 groups (layout in moe_internal.h), with the
// accumulator inputs -2^-24 * 8 * sum (16 at odd offsets, else 1) * value and,
// in every group's factor slot, the row factor 2^(e-14).

// Fragments of one (group, quad) id of a row xr of x whose max |x| is mx: the
// 8 elements 32 * group + 8 * quad .. + 7 become hi/lo fp16 values in the
// fragment block, and the quad's share of the group's accumulator inputs is
// summed over the group's four quads with two shuffles, so the four quads of
// a group must sit in lanes 4j .. 4j + 3 of one warp and the whole warp calls
// this (act = false for lanes without an id).  The group's first quad writes
// the corrections and, in the group's factor slot, the row factor.
__device__ __forceinline__ void frag_quad(const float *__restrict__ xr, float mx, int id, bool act,
                                          uint8_t *__restrict__ row)
{
    int e = 0;
    frexpf(mx, &e);
    const float up = mx > 0.f ? ldexpf(1.0f, 14 - e) : 1.0f;
    const int g = id >> 2, q = id & 3;
    uint8_t *blk = row + (size_t)(g / kXGpc) * frag_blk(kXGpc);
    const int gl = g % kXGpc;
    float chi = 0.f, clo = 0.f;
    if (act) {
        const float4 *src = reinterpret_cast<const float4 *>(xr + 32 * g + 8 * q);
        const float4 v0 = src[0], v1 = src[1];
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        __align__(16) uint16_t hi[8], lo[8];
#pragma unroll
        for (int o = 0; o < 8; o++) {
            float sv = v[o] * up;
            if (o & 1)
                sv *= 0.0625f;
            const __half h = __float2half_rn(sv);
            const __half l = __float2half_rn(sv - __half2float(h));
            hi[frag_pos(o)] = __half_as_ushort(h);
            lo[frag_pos(o)] = __half_as_ushort(l);
            const float wgt = (o & 1) ? 128.0f : 8.0f;
            chi += wgt * __half2float(h);
            clo += wgt * __half2float(l);
        }
        *reinterpret_cast<uint4 *>(blk + gl * 64 + q * 16) = *reinterpret_cast<const uint4 *>(hi);
        *reinterpret_cast<uint4 *>(blk + frag_lo(kXGpc) + gl * 64 + q * 16) = *reinterpret_cast<const uint4 *>(lo);
    }
    chi += __shfl_xor_sync(0xffffffffu, chi, 1);
    clo += __shfl_xor_sync(0xffffffffu, clo, 1);
    chi += __shfl_xor_sync(0xffffffffu, chi, 2);
    clo += __shfl_xor_sync(0xffffffffu, clo, 2);
    if (act && q == 0) {
        float *c = reinterpret_cast<float *>(blk + frag_corr(kXGpc)) + gl * 2;
        c[0] = -chi * 0x1p-24f;
        c[1] = -clo * 0x1p-24f;
        // every group's factor slot holds the row factor, so it reaches the FFN with each stage
        reinterpret_cast<float *>(blk + frag_fac(kXGpc))[gl] = mx > 0.f ? ldexpf(1.0f, e - 14) : 1.0f;
    }
}

// Fragments of the whole row r of x by one 256-thread block: the row's max |x|
// (all of the row's loads issued before the reduction), then every (group,
// quad) id; the row factor goes to row_scale[r].
__device__ void act_frag_row(const float *__restrict__ x, int r, int K, uint8_t *__restrict__ frag,
                             float *__restrict__ row_scale)
{
    __shared__ float wmax[kFragThreads / 32];
    const float *xr = x + (size_t)r * K;
    const float4 *x4 = reinterpret_cast<const float4 *>(xr);
    float mx = 0.f;
    constexpr int kU = 8;
    for (int i0 = 0; i0 < K / 4; i0 += kU * kFragThreads) {
        float4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; u++) {
            const int i = i0 + u * kFragThreads + threadIdx.x;
            v[u] = i < K / 4 ? x4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kU; u++)
            mx = fmaxf(mx, absmax4(v[u]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((threadIdx.x & 31) == 0)
        wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0.f;
#pragma unroll
    for (int w = 0; w < kFragThreads / 32; w++)
        mx = fmaxf(mx, wmax[w]);
    if (threadIdx.x == 0) {
        int e = 0;
        frexpf(mx, &e);
        row_scale[r] = mx > 0.f ? ldexpf(1.0f, e - 14) : 1.0f;
    }
    uint8_t *row = frag + (size_t)r * frag_row_bytes(K, kXGpc);
    const int n_id = (K / 32) * 4;
    const int n_pad = (n_id + 31) / 32 * 32;   // whole warps take part in the shuffles
    for (int id = threadIdx.x; id < n_pad; id += kFragThreads)
        frag_quad(xr, mx, id, id < n_id, row);
}

__global__ void __launch_bounds__(kFragThreads)
act_frag_kernel(const float *__restrict__ x, int K, uint8_t *__restrict__ frag, float *__restrict__ row_scale,
                int32_t *__restrict__ zero, int nzero, const int32_t *__restrict__ gate)
{
    // launched as a programmatic dependent: resident while the previous kernel finishes, but x may
    // come from that kernel and the fragments and counters are still read by the previous FFN, so
    // everything waits for it
    griddep_launch_dependents();
    griddep_wait();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < nzero; i += blockDim.x)
            zero[i] = 0;
    if (gate != nullptr && *gate == 0)
        return;   // no expert will read the fragments (the hybrid's decode half is empty)
    act_frag_row(x, blockIdx.x, K, frag, row_scale);
}

}  // namespace

int launch_router_logits(const float *x, const float *wg, int T, int d, int E, float *logits,
                         cudaStream_t s)
{
    if (T >= kTcMinTokens && d % (kRK * kRSplit) == 0 && E % kRN == 0 && ((uintptr_t)x & 15) == 0 &&
        ((uintptr_t)wg & 15) == 0 && ((uintptr_t)logits & 15) == 0) {
        CUtensorMap mx, mw;
        int rc = make_tmap_2d(&mx, x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, d, T, (uint64_t)d * 4, kRK, kRM,
                              CU_TENSOR_MAP_SWIZZLE_128B);
        rc |= make_tmap_2d(&mw, wg, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, d, E, (uint64_t)d * 4, kRK, kRN,
                           CU_TENSOR_MAP_SWIZZLE_128B);
        if (rc != MOE_OK)
            return MOE_ERR_INVALID_ARG;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
            return MOE_ERR_CUDA;
        // per device, once (several host threads may get here together: a second attribute call is
        // harmless, and the flag is atomic)
        static std::atomic<int> configured[64];
        if (!configured[dev].load(std::memory_order_acquire)) {
            if (cudaFuncSetAttribute(logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmem) !=
                cudaSuccess)
                return MOE_ERR_CUDA;
            configured[dev].store(1, std::memory_order_release);
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(E / kRN * kRSplit), (unsigned)((T + kRM - 1) / kRM));
        cfg.blockDim = dim3(kRThreads);
        cfg.dynamicSmemBytes = kRSmem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kRSplit;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cuda_status(cudaLaunchKernelEx(&cfg, logits_tc_kernel, mx, mw, T, d, E, logits));
    } else if (T >= 128 && d % kBK == 0) {
        dim3 grid((E + kBN - 1) / kBN, (T + kBM - 1) / kBM);
        logits_tiled_kernel<<<grid, 256, 0, s>>>(x, wg, T, d, E, logits);
    } else {
        dim3 grid((E + kEB - 1) / kEB, (T + kTB - 1) / kTB);
        logits_skinny_kernel<<<grid, kSkinnyThreads, 0, s>>>(x, wg, T, d, E, logits, nullptr, nullptr, nullptr, 0);
    }
    return cuda_status(cudaGetLastError());
}

int launch_router_logits_frag(const float *x, const float *wg, int T, int d, int E, float *logits,
                              uint8_t *frag, float *row_scale, int32_t *zero, int nzero, cudaStream_t s)
{
    const int grid = (E + kEB - 1) / kEB;
    if (T > kTB)
        return MOE_ERR_UNSUPPORTED;
    return launch_pdl(logits_skinny_kernel, grid, kSkinnyThreads, 0, s, x, wg, T, d, E, logits, frag,
                      row_scale, zero, nzero);
}

int launch_router_topk(const float *logits, const float *bias, int T, int E, int k, int normalize,
                       float route_scale, float top_p, int32_t *idx, float *w, cudaStream_t s)
{
    // the warp form (E <= 256) keeps everything in registers: no shared memory to reserve
    const size_t smem = E <= 32 * kWarpTopkPer ? 0 : topk_smem_bytes(E, k);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MOE_ERR_CUDA;
    topk_kernel<<<(T + kTopkTokens - 1) / kTopkTokens, kTopkThreads, smem, s>>>(logits, bias, T, E, k, normalize,
                                                                               route_scale, top_p, idx, w);
    return cuda_status(cudaGetLastError());
}

int launch_act_frag(const float *x, int rows, int K, uint8_t *frag, float *row_scale, int32_t *zero, int nzero,
                    cudaStream_t s, const int32_t *gate)
{
    if (rows <= 0)
        return MOE_OK;
    return launch_pdl(act_frag_kernel, rows, kFragThreads, 0, s, x, K, frag, row_scale, zero, nzero, gate);
}

}  // namespace moe
