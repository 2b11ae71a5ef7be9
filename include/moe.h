/*
 * moe.h -- C ABI of libmoe: one MoE layer of the Colibri GLM-5.2 engine on one
 * GB300 GPU (sm_103a): Route -> Union -> expert FFN (int4 SwiGLU, routed +
 * shared) -> score-weighted combine -> Learn (hit counters).
 *
 * The five per-layer stages come from "Public Colibri Observation and Revision
 * Ledger", section "Exact Architecture and Data-Flow Reconstruction" (Route,
 * Union, Place, Overlap, Learn).  The layer calls take every expert resident
 * in device memory, where Place and Overlap have no work; the expert tier
 * (moe_tier_*, moe_layer_forward_tier, at the end of this file) keeps the
 * routed experts in host memory with a device cache of some of them, placing
 * the missing ones on demand and overlapping those copies with the FFN of the
 * cached ones.  The usage file (moe_usage_*) persists the Learn stage's counts.
 *
 * Conventions shared by every entry point
 *  - Pointers are CUDA device pointers owned by the caller, unless a comment
 *    says "host".  Arrays are dense, row-major, with no padding; every pointer
 *    must be 16-byte aligned.  The library allocates no device memory: scratch
 *    comes from a caller workspace whose size the *_workspace_bytes queries
 *    return (an expert tier keeps its own small host-side tables).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call only enqueues work on that stream and returns; nothing is
 *    synchronised and nothing is read back to the host.  The calls keep no
 *    global state and are safe to issue from several host threads.
 *  - The kernels are programmatic dependent launches: each may start while
 *    the kernel before it in the stream finishes, and waits for it before it
 *    reads activations, routing or scratch.  Weights (router, bias, experts)
 *    are read before that wait, to start their streaming early: they must
 *    not be written by work still running in the stream when a call starts.
 *  - Return value: MOE_OK, or a negative MOE_ERR_* code when an argument is
 *    invalid or unsupported (nothing is enqueued then) or a launch failed.
 *    The library never exits, traps or prints.
 *  - Errors found by the kernels themselves (an expert id out of range, a
 *    pipeline wait that ran out of time) are OR-ed into a caller-owned device
 *    word `err` (int32, the caller zeroes it); the offending item is skipped.
 *    Copy it to the host after the stream has finished and decode it with
 *    moe_device_error().
 *
 * Data formats
 *  - int4 weights: symmetric two's complement in [-8, 7], no zero point; in a
 *    row of `cols` elements, element 2i is the low nibble of byte i and element
 *    2i+1 its high nibble; a matrix is [rows][cols/2] bytes.
 *  - scales: fp32, one per G consecutive elements of a row along the input
 *    (reduction) axis, G = 32 or 64: [rows][cols/G].
 *    deq(W)[r][i] = q[r][i] * s[r][i/G].
 *  - expert block: gate [f][d], up [f][d], down [d][f]: first the packed bytes
 *    of the three matrices in that order (moe_expert_q_bytes bytes), then their
 *    scales in the same order (moe_expert_s_count floats).  Expert e of a layer
 *    starts at q_base + e * moe_expert_q_bytes(d, f) and
 *    s_base + e * moe_expert_s_count(d, f, G).  (Same page and section: an
 *    expert's three weight matrices lie next to one another, about 19 MB per
 *    expert at int4.)
 *  - FFN_e(x) = down_e( silu(gate_e x) * (up_e x) ), silu(g) = g * sigmoid(g).
 *
 * Supported shapes: G = 32 or 64 (the colibri README, "2. Get the model":
 * group-scaled int4 containers, gs64 among them); d a multiple of 256; f a
 * multiple of 128 (of 256 when G = 64); 1 <= k <= min(E, 32); 1 <= E <= 1024;
 * 1 <= T.  A G, d or f outside these returns MOE_ERR_UNSUPPORTED; a T, k or E
 * outside them (an empty batch, T = 0, included) MOE_ERR_INVALID_ARG, before
 * anything is launched.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status ---- */
enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,   /* NULL pointer, misaligned pointer, size out of range */
    MOE_ERR_UNSUPPORTED = -2,   /* a shape or mode this build does not implement */
    MOE_ERR_WORKSPACE = -3,     /* workspace smaller than the matching *_workspace_bytes */
    MOE_ERR_CUDA = -4,          /* a CUDA runtime call or kernel launch failed */
    MOE_ERR_STALE = -5          /* a usage file written for another model or shape (not used) */
};

/* Bits of the device error word `err`. */
#define MOE_DEVERR_BAD_EXPERT 0x1   /* an expert id in topk_idx was outside [0, E) */
#define MOE_DEVERR_TIMEOUT 0x2      /* a bounded pipeline wait gave up; outputs are incomplete */
#define MOE_DEVERR_SCALE_RANGE 0x4  /* prefill path: a group scale lies more than 2^13 above or 2^14
                                       below the first group scale of its weight row, beyond what
                                       the path's fp16 weights hold; that row's outputs lose
                                       precision (the decode path has no such limit) */
#define MOE_DEVERR_BOUNDS 0x8       /* only in a library built with MOE_DEBUG_BOUNDS: an index (expert
                                       id, pair position, token or row) was outside its range; the
                                       access was skipped */

/* FFN execution modes. */
enum {
    MOE_MODE_AUTO = 0,     /* decode path when T < 128, else hybrid.  The paths differ in
                              precision (decode within 1e-4 of the output RMS of the exact
                              result, prefill and hybrid within 2e-2), so under this mode the
                              same token's output can move by up to 2e-2 * RMS when the batch
                              around it crosses 128 tokens.  Pass MOE_MODE_DECODE to keep the
                              decode path's precision at every batch size.  (The expert tier
                              has no hybrid: there AUTO takes prefill from 128 tokens.) */
    MOE_MODE_DECODE = 1,   /* fp32-accurate grouped GEMV: exact int4 against activations split
                              into fp16 hi + lo parts, fp32 accumulation */
    MOE_MODE_PREFILL = 2,  /* tcgen05 grouped GEMM on 16-bit operands (fp16 q*s weights scaled
                              per weight row by a power of two, fp16 activations scaled per
                              row by a power of two), fp32 accumulate.  Scale magnitudes are
                              free; within one weight row, group scales must stay within
                              2^-14 .. 2^13 of the row's first group scale (else
                              MOE_DEVERR_SCALE_RANGE) */
    MOE_MODE_HYBRID = 3    /* per expert of the union: one with at most 8 tokens of the batch
                              takes the decode path, one with more (and the shared expert) the
                              prefill path, so the tensor cores run only where an expert's
                              tokens make a dense contraction (a choice of this library: the
                              pages name no GPU paths).  Each expert's outputs are bitwise those
                              of its path; routed outputs in fp32.  Precision: the prefill
                              path's bound. */
};

/* Human-readable name of a status code (static string). */
MOE_API const char *moe_status_str(int status);

/* Decode a device error word copied to the host: MOE_OK when zero, else
 * MOE_ERR_CUDA for a timeout, MOE_ERR_INVALID_ARG for a bad expert id or (in a
 * MOE_DEBUG_BOUNDS build) an index out of range, MOE_ERR_UNSUPPORTED for scales
 * outside the prefill path's range. */
MOE_API int moe_device_error(int32_t err_word_host);

/* Packed bytes / fp32 scale count of one expert block (layout above). */
MOE_API size_t moe_expert_q_bytes(int d, int f);
MOE_API size_t moe_expert_s_count(int d, int f, int G);

/* One MoE layer's int4 experts (device pointers).  The shared expert has the
 * same block layout as a routed one. */
typedef struct {
    const uint8_t *q_base;    /* [E][moe_expert_q_bytes(d, f)] */
    const float *s_base;      /* [E][moe_expert_s_count(d, f, G)] */
    const uint8_t *shared_q;  /* [moe_expert_q_bytes(d, f)] */
    const float *shared_s;    /* [moe_expert_s_count(d, f, G)] */
    int E, d, f, G;
} moe_layer_int4;

/*
 * Route: sigmoid gate and top-k selection.
 * Source: "Public Colibri Observation and Revision Ledger", "Exact Architecture
 * and Data-Flow Reconstruction": the trained sigmoid router (n_group = 1)
 * scores all experts of the layer with fp32 gate parameters; colibri README,
 * "The idea": ~11 GB of routed experts per token, i.e. k = 8 for GLM-5.2.
 *
 *   l[t][e]  = sum_i x[t][i] * w_gate[e][i]               (fp32)
 *   s[t][e]  = 1 / (1 + exp(-l[t][e]))
 *   key      = s[t][e] + bias[e]       (bias selects only; NULL means 0)
 *   topk_idx[t][j], j < k: experts by key descending, equal keys -> lower id
 *   topk_w[t][j] = s of that expert            if normalize == 0
 *                = route_scale * s / sum_j s   if normalize != 0
 *
 * x [T][d] fp32; w_gate [E][d] fp32; bias [E] fp32 or NULL.
 * Outputs: topk_idx [T][k] int32, topk_w [T][k] fp32, logits [T][E] fp32
 * (the raw l, written as a by-product; caller-owned).
 * Errors: MOE_ERR_INVALID_ARG for NULL/misaligned pointers or T < 1, d < 1,
 * E > 1024, k < 1, k > min(E, 32).
 */
MOE_API int moe_route(const float *x, const float *w_gate, const float *bias, int T, int d,
              int E, int k, int normalize, float route_scale, int32_t *topk_idx,
              float *topk_w, float *logits, void *stream);

/*
 * moe_route with top-p pruning of the selection (a lossy mode).
 * Source: "Public Colibri Observation and Revision Ledger", "Exact-Versus-Lossy
 * Mode Table" (top-p gating restricts a layer to fewer experts and changes
 * the output); "Colibri is an open-source, lightweight Mixture-of-Experts",
 * "Configuration" (the --topp setting reads fewer experts).  The pages give no
 * formula; the cut taken here:
 *   s_1 .. s_k  the scores of the k chosen experts in selection order
 *   m = min { m >= 1 : s_1 + ... + s_m >= top_p * (s_1 + ... + s_k) }
 *   slots 1..m keep their expert; slots m+1..k get topk_idx = -1, topk_w = 0
 *   normalize != 0: topk_w = route_scale * s_j / (s_1 + ... + s_m) over kept slots
 * The sums are fp32 (a warp scan, not left to right), so a token whose cut
 * falls within rounding of top_p * total may keep one expert more or fewer
 * than an exact evaluation.  top_p >= 1 gives exactly moe_route's result.
 * An id of -1 in topk_idx is an empty slot for moe_union and moe_combine.
 * Errors: as moe_route; MOE_ERR_INVALID_ARG when top_p <= 0 or not finite.
 */
MOE_API int moe_route_topp(const float *x, const float *w_gate, const float *bias, int T, int d,
                           int E, int k, int normalize, float route_scale, float top_p,
                           int32_t *topk_idx, float *topk_w, float *logits, void *stream);

/*
 * Union: merge the routed (token, slot) pairs of the batch so each unique
 * expert is read once, and group the pairs by expert.
 * Source: same page and section (the Union stage combines the expert requests
 * of all tokens in the batch); same page, "Cache/Prefetch Design Comparison"
 * figure caption (with the batch union, a unique expert's weights are fetched
 * a single time per batch).
 *
 * Pair p = t*k + j.  Outputs (all int32, caller-owned):
 *   counts [E]        number of pairs routed to each expert
 *   offsets [E+1]     exclusive scan of counts over ascending expert id
 *   sorted_pair [T*k] pairs ordered by (expert, p): expert e's pairs occupy
 *                     positions offsets[e] .. offsets[e+1]-1, tokens ascending;
 *                     positions from offsets[E] on (left when slots are empty
 *                     or bad) are unspecified
 *   perm [T*k]        perm[p] = position of pair p in sorted_pair
 *   uniq [E]          experts with counts > 0, ascending; entries >= n_uniq unspecified
 *   n_uniq [1]        number of such experts
 * hits [E] uint64 or NULL: when given, hits[e] += counts[e] (the Learn stage,
 * fused; see moe_hits).  An id of -1 is an empty slot (pruned by
 * moe_route_topp): perm[p] = -1, no group, no hit, no error.  Any other id
 * outside [0, E) sets MOE_DEVERR_BAD_EXPERT in *err, gets perm[p] = -1 and is
 * left out.
 * Runs in one thread block; T*k <= 1<<22.
 */
MOE_API int moe_union(const int32_t *topk_idx, int T, int k, int E, int32_t *counts,
              int32_t *offsets, int32_t *perm, int32_t *sorted_pair, int32_t *uniq,
              int32_t *n_uniq, uint64_t *hits, int32_t *err, void *stream);

/*
 * Learn: per-expert hit counters, hits[e] += counts[e] (uint64, cumulative
 * across calls; one count per routed (token, slot) pair).
 * Source: "Public Colibri Observation and Revision Ledger", "Exact
 * Architecture and Data-Flow Reconstruction", Learn stage (the engine counts,
 * per expert, how often the router picked it).
 */
MOE_API int moe_hits(const int32_t *counts, int E, uint64_t *hits, void *stream);

/*
 * Expert FFN over the batch union: each expert in uniq (and the shared expert)
 * is streamed once and applied to all of its grouped tokens.
 * Source: same section (a routed expert is an MLP of three int4 matrices
 * kept side by side; a small shared expert runs for every token); the SwiGLU
 * form is a reading of the pages.
 *
 * x [T][d] fp32; w: the layer's experts; offsets/sorted_pair/uniq/n_uniq from
 * moe_union (device).  Outputs:
 *   y_pair [T*k][d] fp32: row q = FFN_e(x_t) for the pair sorted_pair[q]
 *                         (t = sorted_pair[q] / k, e its expert)
 *   y_shared [T][d] fp32: FFN_shared(x_t)
 * mode: MOE_MODE_*.  workspace: at least moe_ffn_workspace_bytes(T, k, d, f,
 * mode) bytes of device memory, 256-byte aligned; its contents on entry do not
 * matter.  Calls that share a workspace must not overlap in time.  The union
 * arrays must be moe_union's: *n_uniq is clamped to min(E, T*k) (the kernels'
 * unit tables hold no more), the rest is trusted (a MOE_DEBUG_BOUNDS build
 * checks every index and skips what is out of range).
 */
MOE_API int moe_expert_ffn_int4(const float *x, const moe_layer_int4 *w, const int32_t *offsets,
                        const int32_t *sorted_pair, const int32_t *uniq,
                        const int32_t *n_uniq, int T, int k, int mode, float *y_pair,
                        float *y_shared, void *workspace, size_t ws_bytes, int32_t *err,
                        void *stream);

MOE_API size_t moe_ffn_workspace_bytes(int T, int k, int d, int f, int mode);

/*
 * moe_expert_ffn_int4_noalloc: moe_expert_ffn_int4 without a caller workspace.
 * The pages have no counterpart of this call; it exists for callers that
 * cannot allocate device memory: code inside a host framework that owns all
 * device memory and forbids other allocations, or code on a latency-critical
 * path that cannot afford cudaMalloc/cudaFree (both may synchronise the
 * device).  Inputs and outputs are as for moe_expert_ffn_int4 and are still
 * passed by the caller.
 *
 * Scratch: a static device array of MOE_NOALLOC_SCRATCH_BYTES (8 MiB) that
 * every GPU which loads the library holds until the process exits.  The first
 * call made on a device looks up that array's device address (once per
 * device, with the device current); make that first call before any stream
 * capture.  No call allocates memory.  A batch whose scratch need
 * (moe_ffn_workspace_bytes) exceeds the array returns MOE_ERR_WORKSPACE and
 * enqueues nothing.  All calls on a device share the array, which keeps the
 * last call's contents: calls that overlap on the GPU race, so order them on
 * one stream.
 */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
MOE_API int moe_expert_ffn_int4_noalloc(const float *x, const moe_layer_int4 *w,
                                        const int32_t *offsets, const int32_t *sorted_pair,
                                        const int32_t *uniq, const int32_t *n_uniq, int T, int k,
                                        int mode, float *y_pair, float *y_shared, int32_t *err,
                                        void *stream);

/*
 * Score-weighted combine (+ residual):
 *   out[t][c] = residual[t][c] + y_shared[t][c] + sum_{j<k} topk_w[t][j] * y_pair[perm[t*k+j]][c]
 * summed left to right in slot order j.  residual may be NULL (taken as 0) and
 * may alias out.  A pair with perm < 0 is skipped.
 * Source: the weighted sum of the selected experts' outputs with the router's
 * scores and the always-on shared branch ("Public Colibri Observation and
 * Revision Ledger", "Exact Architecture and Data-Flow Reconstruction").
 */
MOE_API int moe_combine(const float *y_pair, const float *y_shared, const float *topk_w,
                const int32_t *perm, const float *residual, int T, int k, int d,
                float *out, void *stream);

/*
 * RMS normalisation of each row (unit weight), the input of a stacked layer:
 *   out[t][i] = x[t][i] / sqrt( (1/d) sum_i x[t][i]^2 + eps )
 * x, out: [T][d] fp32 (out may alias x); d a multiple of 4; eps >= 0.
 * fp32 sum of squares, IEEE square root and division.
 * Source: the dense part keeps its norms in fp32 ("Public Colibri Observation
 * and Revision Ledger", "Exact Architecture and Data-Flow Reconstruction").
 * A stack of MoE layers with nothing between them overflows fp32 within a few
 * layers (the SwiGLU is quadratic in x); stacked layers therefore take the
 * normalised residual stream, out_l = x_l + MoE(norm(x_l)), the pre-norm
 * placement of the model family (a reading: the pages do not place the norm).
 */
MOE_API int moe_rms_norm(const float *x, int T, int d, float eps, float *out, void *stream);

/*
 * The whole layer in one call: route -> union (+ hits) -> FFN -> combine, all
 * enqueued on `stream` with no host synchronisation.  Scratch (logits, union
 * arrays, activation fragments, y_pair, y_shared) is carved from `workspace`
 * (at least moe_layer_workspace_bytes(T, k, E, d, f, mode) bytes).
 * topk_idx [T][k] and topk_w [T][k] may be NULL (then kept in the workspace);
 * hits may be NULL (no Learn update).  residual may be NULL or alias out.
 */
MOE_API int moe_layer_forward(const float *x, const float *w_gate, const float *bias,
                      const moe_layer_int4 *w, const float *residual, int T, int k,
                      int normalize, float route_scale, int mode, float *out,
                      int32_t *topk_idx, float *topk_w, uint64_t *hits, void *workspace,
                      size_t ws_bytes, int32_t *err, void *stream);

/* moe_layer_forward with moe_route_topp's pruning (top_p >= 1: identical to
 * moe_layer_forward).  Empty slots add nothing to the output or the hits. */
MOE_API int moe_layer_forward_topp(const float *x, const float *w_gate, const float *bias,
                                   const moe_layer_int4 *w, const float *residual, int T, int k,
                                   int normalize, float route_scale, float top_p, int mode,
                                   float *out, int32_t *topk_idx, float *topk_w, uint64_t *hits,
                                   void *workspace, size_t ws_bytes, int32_t *err, void *stream);

MOE_API size_t moe_layer_workspace_bytes(int T, int k, int E, int d, int f, int mode);

/*
 * moe_layer_forward_topp, and the next layer's input of a pre-norm stack from
 * the same pass over the output: out_normed [T][d] = moe_rms_norm(out, eps)
 * (unit weight), bitwise equal to calling moe_rms_norm on out afterwards.  The
 * combine forms each output row in one block, so the separate normalisation
 * kernel and its launch are saved.  out_normed may not alias out or x.
 * Workspace: moe_layer_workspace_bytes.  Errors: as moe_layer_forward_topp;
 * MOE_ERR_INVALID_ARG for a bad out_normed or eps (negative or not finite).
 */
MOE_API int moe_layer_forward_norm(const float *x, const float *w_gate, const float *bias,
                                   const moe_layer_int4 *w, const float *residual, int T, int k,
                                   int normalize, float route_scale, float top_p, int mode,
                                   float *out, float *out_normed, float eps, int32_t *topk_idx,
                                   float *topk_w, uint64_t *hits, void *workspace, size_t ws_bytes,
                                   int32_t *err, void *stream);

/*
 * The layer with its token rows and its result in HOST memory: x_host [T][d]
 * is brought to the device, moe_layer_forward_topp runs on that copy, and its
 * out [T][d] lands in out_host -- all enqueued on `stream`.  When both buffers
 * are page-locked and mapped (cudaHostAlloc or cudaHostRegister on a system
 * with unified addressing) and 16-byte aligned, a kernel reads x_host over the
 * host link and the combine writes out_host directly, so the call is kernels
 * only and overlaps the previous one in the stream; otherwise one
 * cudaMemcpyAsync each way (pageable buffers make those synchronous).  Either
 * way the call returns before the work finishes: the caller synchronises the
 * stream before reading out_host or rewriting x_host.  The device copy of the
 * rows (and, on the copy route, of the result) sits in the workspace after the
 * layer's scratch: moe_layer_host_workspace_bytes(T, k, E, d, f, mode) bytes.
 * residual, topk_idx, topk_w, hits and err are device pointers as in
 * moe_layer_forward (residual may be NULL).
 * Errors: as moe_layer_forward; MOE_ERR_INVALID_ARG for a NULL host pointer;
 * MOE_ERR_CUDA when a copy cannot be enqueued.
 */
MOE_API int moe_layer_forward_host(const float *x_host, const float *w_gate, const float *bias,
                                   const moe_layer_int4 *w, const float *residual, int T, int k,
                                   int normalize, float route_scale, float top_p, int mode,
                                   float *out_host, int32_t *topk_idx, float *topk_w, uint64_t *hits,
                                   void *workspace, size_t ws_bytes, int32_t *err, void *stream);
MOE_API size_t moe_layer_host_workspace_bytes(int T, int k, int E, int d, int f, int mode);

/* --------------------------------------------- usage file (Learn, kept) ---- */
/*
 * The per-expert hit counters of `layers` layers (hits [layers][E], host)
 * saved to a file and loaded back, and the most used experts of a layer.
 * Source: "Public Colibri Observation and Revision Ledger", "Exact Architecture
 * and Data-Flow Reconstruction" (a learning cache of the most used experts,
 * persisted between runs) and "Failure, Corruption, and Restart Behavior" (the
 * usage file decides what is pinned on restart and is not checked against the
 * model).  The file holds a caller-chosen model id (e.g. a hash of the
 * weights), the shape, the counts and a checksum; it is written to
 * "<path>.tmp" and renamed over path.
 *   moe_usage_save: MOE_OK, or MOE_ERR_INVALID_ARG when it cannot be written.
 *   moe_usage_load: MOE_OK (hits filled); MOE_ERR_STALE when the file is sound
 *     but for another model id, layer count or E (hits untouched);
 *     MOE_ERR_INVALID_ARG when missing, of another version, cut short or
 *     corrupted (hits untouched).
 *   moe_usage_top: the n most used experts of one layer's hits [E], count
 *     descending, equal counts by ascending id (experts: host [n]).
 */
MOE_API int moe_usage_save(const char *path, const uint64_t *hits, int layers, int E, uint64_t model_id);
MOE_API int moe_usage_load(const char *path, uint64_t *hits, int layers, int E, uint64_t model_id);
MOE_API int moe_usage_top(const uint64_t *hits, int E, int n, int32_t *experts);

/* ------------------------------------------------- expert tier (Place) ---- */
/*
 * Place and Overlap: a layer whose routed experts live in host memory, with a
 * cache of n_slots expert blocks in device memory.
 * Source: "Public Colibri Observation and Revision Ledger", "Exact Architecture
 * and Data-Flow Reconstruction" (Place loads the experts a batch needs into
 * fast memory; Overlap computes on the experts already there while the loads
 * run); colibri README, "How it works" (where an expert is placed changes
 * only the speed: which experts are chosen and how precisely they are
 * computed do not depend on it).
 *
 * A tier belongs to one layer and one device (the current device at
 * creation).  It keeps host-side tables, two events and a small page-locked
 * staging buffer, all freed by moe_tier_destroy; device memory is the
 * caller's: slot_q [n_slots][moe_expert_q_bytes(d, f)] and slot_s
 * [n_slots][moe_expert_s_count(d, f, G)].  host_q/host_s hold all E expert
 * blocks in the layout of moe_layer_int4 and must be page-locked
 * (cudaHostAlloc or cudaHostRegister) and stay valid for the tier's life.
 * A tier is used by one host thread and one stream at a time (calls on it are
 * serialised by a lock).  Errors: MOE_ERR_INVALID_ARG for bad sizes or
 * pointers, MOE_ERR_UNSUPPORTED for shapes the FFN does not support,
 * MOE_ERR_CUDA when a runtime call fails.
 */
typedef struct moe_tier_s *moe_tier;

MOE_API int moe_tier_create(int E, int d, int f, int G, const uint8_t *host_q, const float *host_s,
                            uint8_t *slot_q, float *slot_s, int n_slots, moe_tier *out);
MOE_API void moe_tier_destroy(moe_tier tier);

/*
 * Pin experts (host array of n ids) in slots: they are loaded now (copies on
 * copy_stream, which this call waits for) and never evicted until
 * moe_tier_unpin_all.  At least one slot always stays unpinned.  This is how
 * a learned hot set (moe_usage_top) is kept resident.  Call it when no layer
 * call on this tier is still running on the device (its slots may be
 * rewritten).
 */
MOE_API int moe_tier_pin(moe_tier tier, const int32_t *experts, int n, void *copy_stream);
/* Load experts (host array of n ids) into slots without pinning them (a warm start, e.g. from
 * moe_usage_top): empty slots first, then the least recently used unpinned ones; once every
 * unpinned slot holds an expert of the list, the rest of the list is left out.  The copies go on
 * copy_stream, which this call waits for; the same rule as moe_tier_pin applies. */
MOE_API int moe_tier_prefetch(moe_tier tier, const int32_t *experts, int n, void *copy_stream);
MOE_API int moe_tier_unpin_all(moe_tier tier);

/* stats (host [4]): resident hits, misses (experts copied), bytes copied, layer calls. */
MOE_API int moe_tier_stats(moe_tier tier, uint64_t *stats);
/* The expert in each slot (-1: empty) and its pin flag (host [n_slots] each; either may be NULL). */
MOE_API int moe_tier_slots(moe_tier tier, int32_t *expert_in_slot, uint8_t *pinned);

MOE_API size_t moe_tier_workspace_bytes(int T, int k, int E, int d, int f, int mode);

/*
 * moe_layer_forward_topp over a tier (top_p = 1: plain top-k).  Steps:
 *   route and union on `stream`; the union's expert list is copied to the
 *   host and this call WAITS for it (the only call of this library that
 *   synchronises with the device, so it cannot be captured in a CUDA graph);
 *   experts already in a slot are hits, each missing one takes the least
 *   recently used unpinned slot not needed by this batch and is copied there
 *   (one cudaMemcpyAsync per block, on copy_stream); the FFN runs over the
 *   hits and the shared expert while the copies proceed, then, after the
 *   copies (an event), over the copied experts; then the combine.
 * Once every expert has a slot (n_slots = E, each used once) no call can
 * miss: calls then skip the host round trip and run one FFN over the union
 * (they count as calls in the stats, not as hits).
 * The output is bit-identical to moe_layer_forward_topp on the same weights
 * resident in device memory, at any residency.  A batch whose union has more
 * experts than unpinned slots returns MOE_ERR_INVALID_ARG (nothing is copied).
 * The shared expert (shared_q, shared_s) is in device memory.  workspace:
 * moe_tier_workspace_bytes(T, k, E, d, f, mode) bytes, 256-byte aligned.
 * mode: MOE_MODE_AUTO (decode below 128 tokens, prefill from 128), _DECODE or
 * _PREFILL; MOE_MODE_HYBRID returns MOE_ERR_INVALID_ARG.  The bit-identity
 * above holds against moe_layer_forward_topp with the mode AUTO resolves to.
 */
MOE_API int moe_layer_forward_tier(const float *x, const float *w_gate, const float *bias, moe_tier tier,
                                   const uint8_t *shared_q, const float *shared_s, const float *residual,
                                   int T, int k, int normalize, float route_scale, float top_p, int mode,
                                   float *out, int32_t *topk_idx, float *topk_w, uint64_t *hits,
                                   void *workspace, size_t ws_bytes, int32_t *err, void *stream,
                                   void *copy_stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
