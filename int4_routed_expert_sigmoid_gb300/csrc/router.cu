// router.cu -- Route stage: fp32 router logits, sigmoid + bias-keyed top-k with
// score weights, and the activation fragments the decode FFN consumes.
//
// Source: "Public Colibri Observation and Revision Ledger", "Exact Architecture
// and Data-Flow Reconstruction": a trained sigmoid gate (n_group = 1, fp32
// parameters) scores every expert of the layer for each token and the top
// experts are selected.
#include <cuda_bf16.h>
#include <cfloat>
#include <climits>

#include "moe_internal.h"

namespace moe {
namespace {

// ----------------------------------------------------------------- logits ---
// Small T: each CTA owns kEB experts x kTB tokens and splits the reduction
// over d across its 256 threads (float4 loads), then reduces in a fixed order.
constexpr int kEB = 2, kTB = 8, kSkinnyThreads = 256;

__global__ void __launch_bounds__(kSkinnyThreads)
logits_skinny_kernel(const float *__restrict__ x, const float *__restrict__ wg, int T, int d, int E,
                     float *__restrict__ logits)
{
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
    for (int i = threadIdx.x; i < d4; i += kSkinnyThreads) {
        float4 wv[kEB];
#pragma unroll
        for (int a = 0; a < kEB; a++)
            wv[a] = a < ne ? __ldg(w4 + (size_t)(e0 + a) * d4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int b = 0; b < kTB; b++) {
            if (b < nt) {
                const float4 xv = __ldg(x4 + (size_t)(t0 + b) * d4 + i);
#pragma unroll
                for (int a = 0; a < kEB; a++) {
                    acc[a][b] = fmaf(xv.x, wv[a].x, acc[a][b]);
                    acc[a][b] = fmaf(xv.y, wv[a].y, acc[a][b]);
                    acc[a][b] = fmaf(xv.z, wv[a].z, acc[a][b]);
                    acc[a][b] = fmaf(xv.w, wv[a].w, acc[a][b]);
                }
            }
        }
    }
    __shared__ float part[kSkinnyThreads / 32][kEB * kTB];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int a = 0; a < kEB; a++)
#pragma unroll
        for (int b = 0; b < kTB; b++) {
            float v = acc[a][b];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0)
                part[warp][a * kTB + b] = v;
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
}

// Large T: register-tiled fp32 GEMM, C[T][E] = X[T][d] * Wg[E][d]^T.
// 64 x 64 tile per CTA, 256 threads x (4 x 4), k-slabs of 16 staged in shared
// memory (transposed so both operands are read as float4 broadcasts).
constexpr int kBM = 64, kBN = 64, kBK = 16;

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

// ------------------------------------------------------------------ top-k ---
// One warp per token.  Lane l holds experts l, l+32, ...; k rounds of a warp
// arg-max on (key desc, id asc) pick the experts in order.
template <int EPL>
__global__ void __launch_bounds__(256)
topk_kernel(const float *__restrict__ logits, const float *__restrict__ bias, int T, int E, int k,
            int normalize, float route_scale, int32_t *__restrict__ idx, float *__restrict__ w)
{
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T)
        return;
    float key[EPL], score[EPL];
    uint32_t live = 0;
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        const int e = lane + 32 * i;
        if (e < E) {
            const float l = logits[(size_t)t * E + e];
            score[i] = 1.0f / (1.0f + expf(-l));
            key[i] = score[i] + (bias ? bias[e] : 0.0f);
            live |= 1u << i;
        } else {
            score[i] = 0.f;
            key[i] = -FLT_MAX;
        }
    }
    float my_score = 0.f;   // lane j keeps the score of slot j
    for (int j = 0; j < k; j++) {
        float bk = -INFINITY, bs = 0.f;
        int be = INT_MAX;
#pragma unroll
        for (int i = 0; i < EPL; i++) {
            const int e = lane + 32 * i;
            if ((live >> i) & 1u) {
                if (key[i] > bk || (key[i] == bk && e < be)) {
                    bk = key[i];
                    be = e;
                    bs = score[i];
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            const float os = __shfl_xor_sync(0xffffffffu, bs, off);
            if (ok > bk || (ok == bk && oe < be)) {
                bk = ok;
                be = oe;
                bs = os;
            }
        }
        if ((be & 31) == lane)
            live &= ~(1u << (be >> 5));
        if (lane == j)
            my_score = bs;
        if (lane == 0)
            idx[(size_t)t * k + j] = be;
    }
    float scale = 1.0f;
    if (normalize) {
        float sum = 0.f;
        for (int j = 0; j < k; j++)
            sum += __shfl_sync(0xffffffffu, my_score, j);
        scale = route_scale / sum;
    }
    if (lane < k)
        w[(size_t)t * k + lane] = normalize ? my_score * scale : my_score;
}

// --------------------------------------------------------- act fragments ---
// One thread per (row, group, quad): 8 fp32 -> hi/lo bf16 in fragment order.
__global__ void act_frag_kernel(const float *__restrict__ x, int rows, int K,
                                uint16_t *__restrict__ frag)
{
    const int groups = K / 32;
    const long long id = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (id >= (long long)rows * groups * 4)
        return;
    const int q = (int)(id & 3);
    const int g = (int)((id >> 2) % groups);
    const int r = (int)(id / (4LL * groups));
    const float4 *src = reinterpret_cast<const float4 *>(x + (size_t)r * K + 32 * g + 8 * q);
    const float4 v0 = src[0], v1 = src[1];
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    __align__(16) uint16_t hi[8], lo[8];
#pragma unroll
    for (int o = 0; o < 8; o++) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v[o]);
        const __nv_bfloat16 l = __float2bfloat16_rn(v[o] - __bfloat162float(h));
        hi[frag_pos(o)] = __bfloat16_as_ushort(h);
        lo[frag_pos(o)] = __bfloat16_as_ushort(l);
    }
    uint16_t *row = frag + (size_t)r * 2 * K;
    *reinterpret_cast<uint4 *>(row + (size_t)(g * 4 + q) * 8) = *reinterpret_cast<const uint4 *>(hi);
    *reinterpret_cast<uint4 *>(row + K + (size_t)(g * 4 + q) * 8) = *reinterpret_cast<const uint4 *>(lo);
}

}  // namespace

int launch_router_logits(const float *x, const float *wg, int T, int d, int E, float *logits,
                         cudaStream_t s)
{
    if (T >= 128 && d % kBK == 0) {
        dim3 grid((E + kBN - 1) / kBN, (T + kBM - 1) / kBM);
        logits_tiled_kernel<<<grid, 256, 0, s>>>(x, wg, T, d, E, logits);
    } else {
        dim3 grid((E + kEB - 1) / kEB, (T + kTB - 1) / kTB);
        logits_skinny_kernel<<<grid, kSkinnyThreads, 0, s>>>(x, wg, T, d, E, logits);
    }
    return cuda_status(cudaGetLastError());
}

int launch_router_topk(const float *logits, const float *bias, int T, int E, int k, int normalize,
                       float route_scale, int32_t *idx, float *w, cudaStream_t s)
{
    const int blocks = (T + 7) / 8;
    const int epl = (E + 31) / 32;
#define MOE_TOPK(N)                                                                                \
    topk_kernel<N><<<blocks, 256, 0, s>>>(logits, bias, T, E, k, normalize, route_scale, idx, w)
    if (epl <= 1) MOE_TOPK(1);
    else if (epl <= 2) MOE_TOPK(2);
    else if (epl <= 4) MOE_TOPK(4);
    else if (epl <= 8) MOE_TOPK(8);
    else if (epl <= 16) MOE_TOPK(16);
    else MOE_TOPK(32);
#undef MOE_TOPK
    return cuda_status(cudaGetLastError());
}

int launch_act_frag(const float *x, int rows, int K, uint16_t *frag, cudaStream_t s)
{
    const long long n = (long long)rows * (K / 32) * 4;
    if (n == 0)
        return MOE_OK;
    act_frag_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(x, rows, K, frag);
    return cuda_status(cudaGetLastError());
}

}  // namespace moe
