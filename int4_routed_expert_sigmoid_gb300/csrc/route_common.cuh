// route_common.cuh -- warp-level top-k of one token's router logits, shared by
// the stand-alone top-k kernel and the fused select+union kernel.
//
// Source: "Public Colibri Observation and Revision Ledger", "Exact Architecture
// and Data-Flow Reconstruction" (sigmoid router scores every expert; the top
// experts are selected).  Key = sigmoid(l) + bias (bias selects only), order
// key descending with ties to the lower expert id; weights are the sigmoid
// scores, optionally renormalised to route_scale.
#pragma once
#include <cfloat>
#include <climits>
#include <cstdint>

namespace moe {

// One warp: lane l holds experts l, l+32, ...; k rounds of a warp arg-max on
// (key desc, id asc) pick the experts in order.  Writes idx[0..k) and w[0..k).
template <int EPL>
__device__ __forceinline__ void topk_warp(const float *__restrict__ lrow, const float *__restrict__ bias,
                                          int E, int k, int normalize, float route_scale,
                                          int32_t *__restrict__ idx, float *__restrict__ w)
{
    const int lane = threadIdx.x & 31;
    float key[EPL], score[EPL];
    uint32_t live = 0;
#pragma unroll
    for (int i = 0; i < EPL; i++) {
        const int e = lane + 32 * i;
        if (e < E) {
            const float l = lrow[e];
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
            idx[j] = be;
    }
    float scale = 1.0f;
    if (normalize) {
        float sum = 0.f;
        for (int j = 0; j < k; j++)
            sum += __shfl_sync(0xffffffffu, my_score, j);
        scale = route_scale / sum;
    }
    if (lane < k)
        w[lane] = normalize ? my_score * scale : my_score;
}


}  // namespace moe
