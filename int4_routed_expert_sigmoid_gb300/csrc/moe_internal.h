// moe_internal.h -- launchers shared between the translation units of libmoe.
// Internal: not part of the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// Activation fragment layout ("frag"): the B operand of the decode FFN's
// m16n8k16 MMAs, precomputed once per activation row.
//
// A row of K fp32 values v becomes two planes (hl = 0: hi = bf16(v),
// hl = 1: lo = bf16(v - hi)), each [K/32 groups][4 quads][8 bf16].  Quad t of
// group g holds elements 32g + 8t + kFragPerm[i], i = 0..7, kFragPerm =
// {0,4,1,5,2,6,3,7}: the order in which the MMA's k index meets the nibbles of
// a packed 32-bit weight word (see ffn_decode.cu).  Row stride = 2*K bf16.
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int frag_pos(int o) { return 2 * (o & 3) + (o >> 2); }

// Error propagation helper for launchers.
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// router.cu
int launch_router_logits(const float *x, const float *wg, int T, int d, int E, float *logits,
                         cudaStream_t s);
int launch_router_topk(const float *logits, const float *bias, int T, int E, int k, int normalize,
                       float route_scale, int32_t *idx, float *w, cudaStream_t s);
int launch_act_frag(const float *x, int rows, int K, uint16_t *frag, cudaStream_t s);

// union.cu
int launch_union(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
                 int32_t *perm, int32_t *sorted_pair, int32_t *uniq, int32_t *n_uniq,
                 uint64_t *hits, int32_t *err, cudaStream_t s);
int launch_hits(const int32_t *counts, int E, uint64_t *hits, cudaStream_t s);

// ffn_decode.cu
struct DecodeFfnArgs {
    const moe_layer_int4 *w;
    const int32_t *offsets, *sorted_pair, *uniq, *n_uniq;
    int T, k;
    const uint16_t *x_frag;   // [T][2*d] bf16 frag layout
    uint16_t *h_frag;         // [T*k + T][2*f] bf16 frag layout (scratch)
    float *y_pair, *y_shared;
    int32_t *err;
};
int launch_ffn_decode(const DecodeFfnArgs &a, cudaStream_t s);

// combine.cu
int launch_combine(const float *y_pair, const float *y_shared, const float *w, const int32_t *perm,
                   const float *res, int T, int k, int d, float *out, cudaStream_t s);

// tmap.cu
// 3-D tiled tensor map over `outer` equally strided blocks of a [rows][inner] matrix.
int make_tmap_3d(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                 uint64_t inner, uint64_t rows, uint64_t outer, uint64_t row_stride_bytes,
                 uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle);

// device properties cached per device
int sm_count(int device);

}  // namespace moe
