// route_common.cuh -- top-k of up to 8 tokens' router logits by one block
// (a warp per token in registers for E <= 256, a rank-based block form above),
// shared by the stand-alone top-k kernel and the fused select+union kernel.
//
// Source: "Public Colibri Observation and Revision Ledger", "Exact Architecture
// and Data-Flow Reconstruction" (sigmoid router scores every expert; the top
// experts are selected).  Key = sigmoid(l) + bias (bias selects only), order
// key descending with ties to the lower expert id; weights are the sigmoid
// scores, optionally renormalised to route_scale.  top_p < 1 keeps only the
// shortest prefix of the k chosen slots whose scores reach top_p times the
// scores of all k (the lossy top-p gating of the Ledger's "Exact-Versus-Lossy
// Mode Table", the `--topp` setting of the summary page's "Configuration");
// the other slots are emptied (id -1, weight 0).
#pragma once
#include <cfloat>
#include <climits>
#include <cstdint>

namespace moe {

constexpr int kTopkThreads = 256;   // threads of a block running topk_block
constexpr int kTopkTokens = 8;      // tokens per block

// sigmoid(l) = 1 / (1 + e^-l); the reciprocal is correctly rounded, as a division would be.
__device__ __forceinline__ float router_score(float l) { return __frcp_rn(1.0f + expf(-l)); }

// (key, id) ranks before (key', id') in selection order.
__device__ __forceinline__ bool key_before(float ka, int ea, float kb, int eb)
{
    return ka > kb || (ka == kb && ea < eb);
}

// Dynamic shared memory of topk_block: keys and scores [8][E]; per token, the
// candidates followed by the k result slots, and the candidates' keys.
__host__ __device__ constexpr int topk_cand_cap(int E, int k) { return ((E + 31) / 32) * (k < 32 ? k : 32); }
__host__ __device__ constexpr int topk_cand_stride(int E, int k) { return topk_cand_cap(E, k) + 32; }
__host__ __device__ constexpr size_t topk_smem_bytes(int E, int k)
{
    return (size_t)kTopkTokens * E * 4 * 2 + (size_t)kTopkTokens * topk_cand_stride(E, k) * 4 * 2;
}

// The last step of both top-k forms, by the token's warp: lane j < k holds
// slot j (expert my_e, score my_s); lanes from k on hold (0, 0).  With
// top_p < 1 the slots are cut: slot j stays when the scores of slots 0 .. j-1
// add up to less than top_p times the scores of all k.  Then the weights
// (renormalised to route_scale when normalize) and the idx / w rows; the ids
// also go to sel[t * k + j] when sel is not null.
__device__ __forceinline__ void topk_finish(int t0, int t, int lane, int k, int my_e, float my_s, int normalize,
                                            float route_scale, float top_p, int32_t *__restrict__ idx,
                                            float *__restrict__ w, int *sel)
{
    if (top_p < 1.0f) {
        // exclusive prefix of the scores in slot order, and their total
        float inc = my_s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float v = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off)
                inc += v;
        }
        const float total = __shfl_sync(0xffffffffu, inc, 31);
        float excl = __shfl_up_sync(0xffffffffu, inc, 1);
        excl = lane == 0 ? 0.0f : excl;
        if (!(excl < top_p * total)) {   // slots from the first one past the cut
            my_e = -1;
            my_s = 0.0f;
        }
    }
    float scale = 1.0f;
    if (normalize) {
        float sum = my_s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            sum += __shfl_xor_sync(0xffffffffu, sum, off);
        scale = route_scale / sum;
    }
    if (lane < k) {
        idx[(size_t)(t0 + t) * k + lane] = my_e;
        w[(size_t)(t0 + t) * k + lane] = normalize ? my_s * scale : my_s;
        if (sel)
            sel[t * k + lane] = my_e;
    }
}

// Top-k of tokens t0 .. t0 + nt - 1 (nt <= 8) by the whole block (256 threads):
//  1. every (token, expert) score and key into shared memory (one thread each);
//  2. per 32-expert block, each expert's rank within the block; the block's
//     first k (at most) become candidates, stored with their keys -- every
//     expert of the overall top-k is among its block's top-k;
//  3. every candidate is ranked among its token's candidates (one thread
//     each, reading the candidates' ids and keys side by side); rank j < k
//     fills slot j; one warp per token forms the weights (and, with top_p < 1,
//     cuts the slots: slot j stays when the scores of slots 0 .. j-1 add up to
//     less than top_p times the scores of all k).
// Writes idx/w rows of the tokens and, when sel is not null, the ids to
// sel[(t - t0) * k + j].  Called by all threads of the block (it synchronises).
__device__ __forceinline__ void topk_block(const float *__restrict__ logits, const float *__restrict__ bias,
                                           int t0, int nt, int E, int k, int normalize, float route_scale,
                                           float top_p, int32_t *__restrict__ idx, float *__restrict__ w,
                                           int *sel, uint8_t *smem)
{
    const int stride = topk_cand_stride(E, k);
    float *keys = reinterpret_cast<float *>(smem);                                   // [8][E]
    float *scores = keys + kTopkTokens * E;                                          // [8][E]
    int *cand = reinterpret_cast<int *>(scores + kTopkTokens * E);                   // [8][stride]
    float *ckey = reinterpret_cast<float *>(cand + kTopkTokens * stride);            // [8][stride]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kU = 8;   // logits (and biases) of kU elements per thread loaded before any is used
    for (int i0 = 0; i0 < nt * E; i0 += kU * kTopkThreads) {
        float l[kU], bb[kU];
#pragma unroll
        for (int u = 0; u < kU; u++) {
            const int i = i0 + u * kTopkThreads + tid;
            const int t = i / E, e = i - t * E;
            l[u] = i < nt * E ? logits[(size_t)(t0 + t) * E + e] : 0.0f;
            bb[u] = (i < nt * E && bias) ? bias[e] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kU; u++) {
            const int i = i0 + u * kTopkThreads + tid;
            if (i < nt * E) {
                const float sc = router_score(l[u]);
                scores[i] = sc;
                keys[i] = sc + bb[u];
            }
        }
    }
    __syncthreads();
    const int nblk = (E + 31) / 32;
    const int kb = k < 32 ? k : 32;
    for (int task = warp; task < nt * nblk; task += kTopkThreads / 32) {
        const int t = task / nblk, b = task - t * nblk;
        const int n_in = E - b * 32 < 32 ? E - b * 32 : 32;
        const float *kr = keys + t * E + b * 32;
        if (lane < n_in) {
            const float kv = kr[lane];
            int r = 0;
            for (int j = 0; j < n_in; j++)
                r += key_before(kr[j], j, kv, lane) ? 1 : 0;
            if (r < kb) {
                cand[t * stride + b * kb + r] = b * 32 + lane;
                ckey[t * stride + b * kb + r] = kv;
            }
        }
        // a block with fewer than k experts leaves its remaining slots empty
        if (lane >= n_in && lane < kb) {
            cand[t * stride + b * kb + lane] = -1;
            ckey[t * stride + b * kb + lane] = 0.0f;
        }
    }
    __syncthreads();
    const int nc = nblk * kb;
    for (int i = tid; i < nt * nc; i += kTopkThreads) {
        const int t = i / nc, c = i - t * nc;
        const int *cr = cand + t * stride;
        const float *kc = ckey + t * stride;
        const int e = cr[c];
        if (e < 0)
            continue;
        const float kv = kc[c];
        int r = 0;
#pragma unroll 8
        for (int j = 0; j < nc; j++) {
            const int ej = cr[j];
            const float kj = kc[j];
            r += (ej >= 0 && key_before(kj, ej, kv, e)) ? 1 : 0;
        }
        if (r < k)
            cand[t * stride + nc + r] = e;
    }
    __syncthreads();
    if (warp < nt) {
        const int t = warp;
        const int my_e = lane < k ? cand[t * stride + nc + lane] : 0;
        const float my_s = lane < k ? scores[t * E + my_e] : 0.0f;
        topk_finish(t0, t, lane, k, my_e, my_s, normalize, route_scale, top_p, idx, w, sel);
    }
    __syncthreads();
}

// Top-k of tokens t0 .. t0 + nt - 1 (nt <= 8) for E <= 32 * kWarpTopkPer, one
// warp per token, all in registers: lane l holds the keys of experts l, l + 32,
// ..., and the k slots are filled one per round by a warp maximum of the key
// (keys mapped to unsigned integers in the same order, -0 as +0) followed by a
// warp minimum of the id among the lanes holding that key -- key descending,
// equal keys by ascending id, as topk_block.  Same outputs as topk_block.
// Called by all threads of a 256-thread block (it synchronises at the end).
constexpr int kWarpTopkPer = 8;
__device__ __forceinline__ void topk_warp(const float *__restrict__ logits, const float *__restrict__ bias, int t0,
                                          int nt, int E, int k, int normalize, float route_scale, float top_p,
                                          int32_t *__restrict__ idx, float *__restrict__ w, int *sel)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp < nt) {
        const int t = warp;
        float l[kWarpTopkPer], bb[kWarpTopkPer];
#pragma unroll
        for (int i = 0; i < kWarpTopkPer; i++) {
            const int e = lane + 32 * i;
            l[i] = e < E ? logits[(size_t)(t0 + t) * E + e] : 0.0f;
            bb[i] = (e < E && bias) ? bias[e] : 0.0f;
        }
        float sc[kWarpTopkPer];
        uint32_t ku[kWarpTopkPer];
        uint32_t taken = 0;
#pragma unroll
        for (int i = 0; i < kWarpTopkPer; i++) {
            sc[i] = router_score(l[i]);
            const float key = sc[i] + bb[i];
            const uint32_t b = __float_as_uint(key);
            ku[i] = key == 0.0f ? 0x80000000u : ((b & 0x80000000u) ? ~b : (b | 0x80000000u));
            if (key != key)
                ku[i] = 0u;   // NaN keys come last
            if (lane + 32 * i >= E)
                taken |= 1u << i;
        }
        int my_e = 0;
        float my_s = 0.0f;
        for (int j = 0; j < k; j++) {
            uint32_t bu = 0u;
            int bi = -1;
            float bs = 0.0f;
#pragma unroll
            for (int i = 0; i < kWarpTopkPer; i++)
                if (!((taken >> i) & 1u) && (bi < 0 || ku[i] > bu)) {
                    bu = ku[i];
                    bi = i;
                    bs = sc[i];
                }
            const uint32_t m = __reduce_max_sync(0xffffffffu, bi >= 0 ? bu : 0u);
            const uint32_t cid = (bi >= 0 && bu == m) ? (uint32_t)(lane + 32 * bi) : 0xffffffffu;
            const uint32_t win = __reduce_min_sync(0xffffffffu, cid);
            const int wl = (int)(win & 31u);
            if (lane == wl)
                taken |= 1u << (win >> 5);
            const float ws = __shfl_sync(0xffffffffu, bs, wl);
            if (lane == j) {
                my_e = (int)win;
                my_s = ws;
            }
        }
        topk_finish(t0, t, lane, k, my_e, my_s, normalize, route_scale, top_p, idx, w, sel);
    }
    __syncthreads();
}

}  // namespace moe
