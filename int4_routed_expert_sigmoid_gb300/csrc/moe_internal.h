// moe_internal.h -- launchers shared between the translation units of libmoe.
// Internal: not part of the C ABI.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

#ifndef MOE_NO_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace moe {

// Bounds checks of a MOE_DEBUG_BOUNDS build: MOE_IN_BOUNDS(ok, err) is true when ok, else sets
// MOE_DEVERR_BOUNDS in the error word (when there is one) and is false, so the caller skips the
// access; in a normal build it is the constant true and costs nothing.
#ifdef MOE_DEBUG_BOUNDS
#ifdef __CUDACC__
__device__ __forceinline__ bool in_bounds_check(bool ok, int32_t *err)
{
    if (!ok && err != nullptr)
        atomicOr(err, MOE_DEVERR_BOUNDS);
    return ok;
}
#endif
#define MOE_IN_BOUNDS(ok, err) ::moe::in_bounds_check((ok), (err))
#else
#define MOE_IN_BOUNDS(ok, err) true
#endif

// Host-side NVTX range over one entry point's launches (a profiler's timeline shows where each
// stage's kernels were enqueued); compiled out with MOE_NO_NVTX.  Costs a few nanoseconds when
// no tool is attached.
struct NvtxRange {
#ifndef MOE_NO_NVTX
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
#else
    explicit NvtxRange(const char *) {}
#endif
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

// ---------------------------------------------------------------------------
// Activation fragment layout ("frag"): the B operand of the decode FFN's
// m16n8k16 fp16 MMAs, precomputed once per activation row.
//
// A row of K fp32 values is scaled by a power of two (per row for x, per
// 32-element group for h; the inverse is kept as a factor) so that
// |v| < 2^14, and split into two planes, hi = fp16(v) and lo = fp16(v - hi).
// Within a plane, quad t of group g holds elements 32g + 8t + o at position
// frag_pos(o), o = 0..7, i.e. in the order {0,4,1,5,2,6,3,7}: the order in
// which the MMA's k index meets the nibbles of a packed 32-bit weight word.
// Elements with odd o are stored divided by 16, because their weights enter
// the MMA multiplied by 16.
//
// The weights enter the MMA as fp16 subnormals (q + 8) * 2^-24 (times 16 at
// odd o).  With corr = 8 * sum_k w_k B_k (w_k = 16 at odd o, else 1; B the
// stored fp16 values) per (row, group, plane), an MMA whose accumulator
// starts at -2^-24 * corr ends at 2^-24 * sum_k q_k v_k.  The fragments keep
// -2^-24 * corr, so it can be the accumulator input directly.
//
// A row is stored as blocks of GPC groups (a "chunk" of 32 * GPC elements),
// each block holding, at byte offsets:
//   0                 hi plane  [GPC groups][4 quads][8 fp16]
//   frag_lo(GPC)      lo plane  (64 bytes after hi: the two planes then fall
//                               in different shared-memory banks)
//   frag_corr(GPC)    [GPC][2] fp32: -2^-24 * corr of hi and lo
//   frag_fac(GPC)     [GPC] fp32: per-group factor (h), or the row factor in every
//                     slot (x), so the factor travels with the stage's data
// so one stage of the pipeline copies one token's blocks with a single bulk
// copy.  x rows use GPC = 8; h rows GPC = 8 when f is a multiple of 256, else 4.
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int frag_lo(int gpc) { return gpc * 64 + 64; }
__host__ __device__ constexpr int frag_corr(int gpc) { return 2 * gpc * 64 + 64; }
__host__ __device__ constexpr int frag_fac(int gpc) { return frag_corr(gpc) + gpc * 8; }
__host__ __device__ constexpr int frag_blk(int gpc) { return frag_fac(gpc) + gpc * 4; }
__host__ __device__ constexpr int frag_gpc_h(int f) { return f % 256 == 0 ? 8 : 4; }
static_assert(frag_blk(8) % 16 == 0 && frag_blk(4) % 16 == 0, "bulk copies move 16-byte multiples");
// Bytes of one fragment row of K elements with GPC groups per block.
__host__ __device__ constexpr size_t frag_row_bytes(int K, int gpc) { return (size_t)(K / (32 * gpc)) * frag_blk(gpc); }
__host__ __device__ constexpr int frag_pos(int o) { return 2 * (o & 3) + (o >> 2); }

// Error propagation helper for launchers.
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream finishes; it must execute
// griddepcontrol.wait before it reads that kernel's results.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kern)(KArgs...), int grid, int block, size_t smem, cudaStream_t s, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...));
}

// router.cu
int launch_router_logits(const float *x, const float *wg, int T, int d, int E, float *logits,
                         cudaStream_t s);
// logits plus the FFN fragments of x in one kernel (T <= 8); also zeroes the nzero counters of the
// decode FFN (after its grid wait, so no earlier kernel still uses them)
int launch_router_logits_frag(const float *x, const float *wg, int T, int d, int E, float *logits,
                              uint8_t *frag, float *row_scale, int32_t *zero, int nzero, cudaStream_t s);
// top_p >= 1: plain top-k; below, the pruned slots get id -1 and weight 0
int launch_router_topk(const float *logits, const float *bias, int T, int E, int k, int normalize,
                       float route_scale, float top_p, int32_t *idx, float *w, cudaStream_t s);
// fragments (GPC = 8) of `rows` rows of x [rows][K], K a multiple of 256; also zeroes the nzero
// counters of the decode FFN.  With `gate` set, the fragments are skipped when *gate is 0 (a device
// count of the experts that would read them).
int launch_act_frag(const float *x, int rows, int K, uint8_t *frag, float *row_scale, int32_t *zero, int nzero,
                    cudaStream_t s, const int32_t *gate = nullptr);

// union.cu (an id of -1 is an empty slot: no group, perm -1, no hit, no error)
int launch_union(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
                 int32_t *perm, int32_t *sorted_pair, int32_t *uniq, int32_t *n_uniq,
                 uint64_t *hits, int32_t *err, cudaStream_t s);
int launch_hits(const int32_t *counts, int E, uint64_t *hits, cudaStream_t s);
// Hybrid FFN: the union's expert list split, in its order, into the experts with at most max_cold
// pairs (uniq_cold, *n_cold) and the rest (uniq_hot, *n_hot); an id outside [0, E) goes to neither
// list and sets MOE_DEVERR_BAD_EXPERT.  *n_uniq is clamped to min(E, pairs), the length of each
// list.  One block; E <= 1024.
int launch_split_units(const int32_t *offsets, const int32_t *uniq, const int32_t *n_uniq, int E, int pairs,
                       int max_cold, int32_t *uniq_cold, int32_t *n_cold, int32_t *uniq_hot, int32_t *n_hot,
                       int32_t *err, cudaStream_t s);
constexpr int kHybridColdMax = 8;   // pairs of an expert up to which the hybrid FFN takes the decode path
// top-k + union + hits in one block (T <= 8, T*k <= 64)
int launch_select_union(const float *logits, const float *bias, int T, int E, int k, int normalize,
                        float route_scale, float top_p, int32_t *idx, float *w, int32_t *counts, int32_t *offsets,
                        int32_t *perm, int32_t *sorted_pair, int32_t *uniq, int32_t *n_uniq,
                        uint64_t *hits, int32_t *err, cudaStream_t s);

// ffn_decode.cu
struct DecodeFfnArgs {
    const moe_layer_int4 *w;
    const int32_t *offsets, *sorted_pair, *uniq, *n_uniq;
    int T, k;
    const uint8_t *x_frag;    // [T] rows of frag_row_bytes(d, 8)
    const float *x_scale;     // [T] per-row factor of x_frag
    uint8_t *h_frag;          // [T*k + T] rows of frag_row_bytes(f, frag_gpc_h(f)) (scratch)
    float *y_pair, *y_shared;
    int32_t *work;            // kDecodeCounters item counters, zeroed by the kernel before (scratch)
    const int32_t *slot_of = nullptr;   // [E] block of w holding expert e (expert tier), or null: block e
    int with_shared = 1;                // 0: only the uniq list's experts (a second launch of the tier)
    int32_t *err;
    int n_experts = 0;                  // routed experts of the routing (offsets has n_experts + 1); 0: w->E
    int max_tokens = 0;                 // most tokens any listed expert has, when known (0: T); sets the pass width
};
constexpr int kDecodeCounters = 2;   // items claimed by the gate/up and the down kernel
int launch_ffn_decode(const DecodeFfnArgs &a, cudaStream_t s);

// ffn_prefill.cu
struct PrefillFfnArgs {
    const moe_layer_int4 *w;
    const float *x;                      // [T][d] fp32
    const int32_t *offsets, *sorted_pair, *uniq, *n_uniq;
    int T, k;
    void *scratch;                       // prefill_scratch_bytes(T, k, d, f) bytes, 256-aligned
    float *y_pair, *y_shared;
    uint16_t *y_pair16;                  // when set: routed outputs as bf16 here instead of y_pair (fp32)
    const int32_t *slot_of = nullptr;    // as in DecodeFfnArgs
    int n_experts = 0;                   // experts the union's offsets cover (0: w->E)
    int with_shared = 1;
    int32_t *err;
};
size_t prefill_scratch_bytes(int T, int k, int d, int f);
int launch_ffn_prefill(const PrefillFfnArgs &a, cudaStream_t s);

// combine.cu
int launch_combine(const float *y_pair, const float *y_shared, const float *w, const int32_t *perm,
                   const float *res, int T, int k, int d, float *out, cudaStream_t s, int32_t *err = nullptr);
// the same with the routed outputs in bf16
int launch_combine_bf16(const uint16_t *y_pair, const float *y_shared, const float *w, const int32_t *perm,
                        const float *res, int T, int k, int d, float *out, cudaStream_t s, int32_t *err = nullptr);
int launch_rms_norm(const float *x, int T, int d, float eps, float *out, cudaStream_t s);
// n floats (a multiple of 4, 16-byte aligned) from host rows the GPU addresses directly into device
// memory, as a programmatic dependent launch (the host-buffer entry point's input)
int launch_copy_rows(const float *src, float *dst, long long n, cudaStream_t s);
// the combine (fp32 y_pair, or bf16 y_pair16 when set) and RMSNorm(out) into out_normed, as the two
// separate kernels would compute them
int launch_combine_norm(const float *y_pair, const uint16_t *y_pair16, const float *y_shared, const float *w,
                        const int32_t *perm, const float *res, int T, int k, int d, float *out, float *out_normed,
                        float eps, cudaStream_t s, int32_t *err);

// tmap.cu
// 3-D tiled tensor map over `outer` equally strided blocks of a [rows][inner] matrix.
int make_tmap_3d(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                 uint64_t inner, uint64_t rows, uint64_t outer, uint64_t row_stride_bytes,
                 uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle);

int make_tmap_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, uint64_t inner, uint64_t rows,
                 uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle);

// Tiled tensor map of rank 1..5: dims and box innermost first, strides_bytes[i] the
// byte stride of dimension i + 1 (any order of strides).
int make_tmap_nd(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, int rank, const uint64_t *dims,
                 const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swizzle);

// device properties cached per device
int sm_count(int device);

// moe_api.cu: the FFN path a mode resolves to at T tokens (MOE_MODE_DECODE, _PREFILL or _HYBRID;
// resolve_mode_plain never gives _HYBRID: AUTO takes prefill from 128 tokens), and the workspace
// layouts of the FFN and of the whole layer (base may be null to size them).
int resolve_mode(int mode, int T);
int resolve_mode_plain(int mode, int T);
size_t ffn_scratch_bytes_mode(int T, int k, int d, int f, int mode);

// Scratch of the decode FFN: activation fragments of x (with a factor per row) and of h (factors
// inside the fragment blocks), and the item counters.
struct FfnScratch {
    uint8_t *x_frag, *h_frag;
    float *x_scale;
    int32_t *work;
};
size_t ffn_scratch_layout(int T, int k, int d, int f, uint8_t *base, FfnScratch *out);

// Scratch of the hybrid FFN: the decode path's, the prefill path's, and the two expert lists.
struct HybridScratch {
    FfnScratch dec;
    void *pre;
    int32_t *uniq_cold, *uniq_hot, *n_cold, *n_hot;
};
size_t hybrid_scratch_layout(int T, int k, int d, int f, uint8_t *base, HybridScratch *out);
// The hybrid FFN over a union (both paths, fp32 routed outputs), on stream s.
int run_ffn_hybrid(const moe_layer_int4 *w, const float *x, const int32_t *offsets, const int32_t *sorted_pair,
                   const int32_t *uniq, const int32_t *n_uniq, int T, int k, void *scratch, float *y_pair,
                   float *y_shared, int32_t *err, cudaStream_t s);

struct LayerScratch {
    float *logits;
    int32_t *idx;
    float *w;
    int32_t *counts, *offsets, *perm, *sorted_pair, *uniq, *n_uniq;
    float *y_pair, *y_shared;
    uint8_t *ffn;
};
size_t layer_scratch_layout(int T, int k, int E, int d, int f, int mode, uint8_t *base, LayerScratch *o);

}  // namespace moe
