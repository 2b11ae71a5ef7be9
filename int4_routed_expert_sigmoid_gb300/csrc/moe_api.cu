// moe_api.cu -- the extern "C" entry points of libmoe: argument validation,
// workspace carving and launch sequencing.  See include/moe.h for the contract
// of each call.
#include <cstdint>

#include <cmath>

#include "moe_internal.h"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;

inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool ok_ptr(const void *p) { return p != nullptr && aligned16(p); }
inline bool ok_opt(const void *p) { return p == nullptr || aligned16(p); }
inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// top_p in (0, 1]; 1 (or more) keeps all k experts
bool ok_top_p(float top_p) { return top_p > 0.0f && top_p < 3.0e38f; }

bool ok_route_shape(int T, int d, int E, int k)
{
    return T >= 1 && d >= 4 && d % 4 == 0 && E >= 1 && E <= 1024 && k >= 1 && k <= 32 && k <= E;
}

int check_layer(const moe_layer_int4 *w)
{
    if (w == nullptr || !ok_ptr(w->q_base) || !ok_ptr(w->s_base) || !ok_ptr(w->shared_q) ||
        !ok_ptr(w->shared_s))
        return MOE_ERR_INVALID_ARG;
    if (w->E < 1 || w->E > 1024 || w->d < 1 || w->f < 1)
        return MOE_ERR_INVALID_ARG;
    // group sizes 32 and 64 (the README's group-scaled container); with 64, f must be a multiple of
    // 256 so that every scale tile row the kernels load is a whole 16 bytes
    if ((w->G != 32 && w->G != 64) || w->d % 256 != 0 || w->f % 128 != 0 || (w->G == 64 && w->f % 256 != 0))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace

namespace moe {

// From 128 tokens the hybrid path is faster than either plain path on the measured batches (a
// Zipf-routed 256-expert layer at 128-512 tokens; at 4096 tokens with ~128 per expert it is the
// prefill path); below, the decode path keeps its 1e-4 precision.
int resolve_mode(int mode, int T)
{
    if (mode == MOE_MODE_AUTO)
        return T < 128 ? MOE_MODE_DECODE : MOE_MODE_HYBRID;
    return mode;
}

int resolve_mode_plain(int mode, int T)
{
    if (mode == MOE_MODE_AUTO)
        return T < 128 ? MOE_MODE_DECODE : MOE_MODE_PREFILL;   // measured crossover of the two plain paths
    return mode;
}

bool valid_mode(int mode)
{
    return mode == MOE_MODE_AUTO || mode == MOE_MODE_DECODE || mode == MOE_MODE_PREFILL || mode == MOE_MODE_HYBRID;
}

size_t ffn_scratch_layout(int T, int k, int d, int f, uint8_t *base, FfnScratch *out)
{
    size_t off = 0;
    const size_t rows_h = (size_t)T * k + T;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + off : nullptr;
        off = align_up(off + bytes);
        return p;
    };
    FfnScratch s{};
    s.x_frag = take((size_t)T * frag_row_bytes(d, 8));
    s.x_scale = reinterpret_cast<float *>(take((size_t)T * sizeof(float)));
    s.h_frag = take(rows_h * frag_row_bytes(f, frag_gpc_h(f)));
    s.work = reinterpret_cast<int32_t *>(take(kDecodeCounters * sizeof(int32_t)));
    if (out)
        *out = s;
    return off;
}

size_t layer_scratch_layout(int T, int k, int E, int d, int f, int mode, uint8_t *base, LayerScratch *o)
{
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + off : nullptr;
        off = align_up(off + bytes);
        return p;
    };
    const size_t P = (size_t)T * k;
    LayerScratch s{};
    s.logits = reinterpret_cast<float *>(take((size_t)T * E * 4));
    s.idx = reinterpret_cast<int32_t *>(take(P * 4));
    s.w = reinterpret_cast<float *>(take(P * 4));
    s.counts = reinterpret_cast<int32_t *>(take((size_t)E * 4));
    s.offsets = reinterpret_cast<int32_t *>(take((size_t)(E + 1) * 4));
    s.perm = reinterpret_cast<int32_t *>(take(P * 4));
    s.sorted_pair = reinterpret_cast<int32_t *>(take(P * 4));
    s.uniq = reinterpret_cast<int32_t *>(take((size_t)E * 4));
    s.n_uniq = reinterpret_cast<int32_t *>(take(4));
    s.y_pair = reinterpret_cast<float *>(take(P * d * 4));
    s.y_shared = reinterpret_cast<float *>(take((size_t)T * d * 4));
    s.ffn = take(ffn_scratch_bytes_mode(T, k, d, f, mode));
    if (o)
        *o = s;
    return off;
}

size_t hybrid_scratch_layout(int T, int k, int d, int f, uint8_t *base, HybridScratch *o)
{
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + off : nullptr;
        off = align_up(off + bytes);
        return p;
    };
    HybridScratch h{};
    uint8_t *dec = take(ffn_scratch_layout(T, k, d, f, nullptr, nullptr));
    if (base)
        ffn_scratch_layout(T, k, d, f, dec, &h.dec);
    h.pre = take(prefill_scratch_bytes(T, k, d, f));
    const size_t list = (size_t)T * k * sizeof(int32_t);   // the union has at most T * k experts
    h.uniq_cold = reinterpret_cast<int32_t *>(take(list));
    h.uniq_hot = reinterpret_cast<int32_t *>(take(list));
    h.n_cold = reinterpret_cast<int32_t *>(take(sizeof(int32_t)));
    h.n_hot = reinterpret_cast<int32_t *>(take(sizeof(int32_t)));
    if (o)
        *o = h;
    return off;
}

size_t ffn_scratch_bytes_mode(int T, int k, int d, int f, int mode)
{
    switch (resolve_mode(mode, T)) {
    case MOE_MODE_PREFILL: return prefill_scratch_bytes(T, k, d, f);
    case MOE_MODE_HYBRID: return hybrid_scratch_layout(T, k, d, f, nullptr, nullptr);
    default: return ffn_scratch_layout(T, k, d, f, nullptr, nullptr);
    }
}

// The two FFN paths one after the other over their halves of the union: the decode grouped GEMV
// over the experts with at most kHybridColdMax pairs, then the tcgen05 grouped GEMM over the rest
// and the shared expert.  They write disjoint rows of y_pair (each expert's pair rows) and the
// prefill path writes y_shared.
int run_ffn_hybrid(const moe_layer_int4 *w, const float *x, const int32_t *offsets, const int32_t *sorted_pair,
                   const int32_t *uniq, const int32_t *n_uniq, int T, int k, void *scratch, float *y_pair,
                   float *y_shared, int32_t *err, cudaStream_t s)
{
    HybridScratch h{};
    hybrid_scratch_layout(T, k, w->d, w->f, static_cast<uint8_t *>(scratch), &h);
    int rc = launch_split_units(offsets, uniq, n_uniq, w->E, T * k, kHybridColdMax, h.uniq_cold, h.n_cold,
                                h.uniq_hot, h.n_hot, err, s);
    if (rc == MOE_OK)
        rc = launch_act_frag(x, T, w->d, h.dec.x_frag, h.dec.x_scale, h.dec.work, kDecodeCounters, s, h.n_cold);
    if (rc != MOE_OK)
        return rc;
    DecodeFfnArgs a{};
    a.w = w;
    a.offsets = offsets;
    a.sorted_pair = sorted_pair;
    a.uniq = h.uniq_cold;
    a.n_uniq = h.n_cold;
    a.T = T;
    a.k = k;
    a.x_frag = h.dec.x_frag;
    a.x_scale = h.dec.x_scale;
    a.h_frag = h.dec.h_frag;
    a.y_pair = y_pair;
    a.y_shared = y_shared;   // not written: the shared expert is the prefill half's
    a.work = h.dec.work;
    a.with_shared = 0;
    a.max_tokens = kHybridColdMax;
    a.err = err;
    rc = launch_ffn_decode(a, s);
    if (rc != MOE_OK)
        return rc;
    PrefillFfnArgs pa{};
    pa.w = w;
    pa.x = x;
    pa.offsets = offsets;
    pa.sorted_pair = sorted_pair;
    pa.uniq = h.uniq_hot;
    pa.n_uniq = h.n_hot;
    pa.T = T;
    pa.k = k;
    pa.scratch = h.pre;
    pa.y_pair = y_pair;
    pa.y_shared = y_shared;
    pa.with_shared = 1;
    pa.err = err;
    return launch_ffn_prefill(pa, s);
}

}  // namespace moe

extern "C" {

const char *moe_status_str(int status)
{
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or mode";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_STALE: return "usage file of another model or shape";
    default: return "unknown status";
    }
}

int moe_device_error(int32_t err)
{
    if (err == 0)
        return MOE_OK;
    if (err & MOE_DEVERR_TIMEOUT)
        return MOE_ERR_CUDA;
    if (err & (MOE_DEVERR_BAD_EXPERT | MOE_DEVERR_BOUNDS))
        return MOE_ERR_INVALID_ARG;
    return MOE_ERR_UNSUPPORTED;
}

size_t moe_expert_q_bytes(int d, int f) { return (size_t)3 * d * f / 2; }

size_t moe_expert_s_count(int d, int f, int G) { return G > 0 ? (size_t)3 * d * f / G : 0; }

int moe_route_topp(const float *x, const float *w_gate, const float *bias, int T, int d, int E, int k,
                   int normalize, float route_scale, float top_p, int32_t *topk_idx, float *topk_w,
                   float *logits, void *stream)
{
    NvtxRange nvtx("moe.route");
    if (!ok_ptr(x) || !ok_ptr(w_gate) || !ok_opt(bias) || !ok_ptr(topk_idx) || !ok_ptr(topk_w) ||
        !ok_ptr(logits) || !ok_route_shape(T, d, E, k) || !ok_top_p(top_p))
        return MOE_ERR_INVALID_ARG;
    const cudaStream_t s = as_stream(stream);
    int rc = launch_router_logits(x, w_gate, T, d, E, logits, s);
    if (rc == MOE_OK)
        rc = launch_router_topk(logits, bias, T, E, k, normalize, route_scale, top_p, topk_idx, topk_w, s);
    return rc;
}

int moe_route(const float *x, const float *w_gate, const float *bias, int T, int d, int E, int k,
              int normalize, float route_scale, int32_t *topk_idx, float *topk_w, float *logits,
              void *stream)
{
    return moe_route_topp(x, w_gate, bias, T, d, E, k, normalize, route_scale, 1.0f, topk_idx, topk_w, logits,
                          stream);
}

int moe_union(const int32_t *topk_idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
              int32_t *perm, int32_t *sorted_pair, int32_t *uniq, int32_t *n_uniq, uint64_t *hits,
              int32_t *err, void *stream)
{
    NvtxRange nvtx("moe.union");
    if (!ok_ptr(topk_idx) || !ok_ptr(counts) || !ok_ptr(offsets) || !ok_ptr(perm) ||
        !ok_ptr(sorted_pair) || !ok_ptr(uniq) || !ok_ptr(n_uniq) || !ok_opt(hits) || !ok_ptr(err))
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || k < 1 || k > 32 || E < 1 || E > 1024 || (long long)T * k > (1LL << 22))
        return MOE_ERR_INVALID_ARG;
    return launch_union(topk_idx, T, k, E, counts, offsets, perm, sorted_pair, uniq, n_uniq, hits,
                        err, as_stream(stream));
}

int moe_hits(const int32_t *counts, int E, uint64_t *hits, void *stream)
{
    NvtxRange nvtx("moe.hits");
    if (!ok_ptr(counts) || !ok_ptr(hits) || E < 1 || E > (1 << 20))
        return MOE_ERR_INVALID_ARG;
    return launch_hits(counts, E, hits, as_stream(stream));
}

size_t moe_ffn_workspace_bytes(int T, int k, int d, int f, int mode)
{
    if (T < 1 || k < 1 || d < 1 || f < 1 || !valid_mode(mode))
        return 0;
    return ffn_scratch_bytes_mode(T, k, d, f, mode);
}

int moe_expert_ffn_int4(const float *x, const moe_layer_int4 *w, const int32_t *offsets,
                        const int32_t *sorted_pair, const int32_t *uniq, const int32_t *n_uniq,
                        int T, int k, int mode, float *y_pair, float *y_shared, void *workspace,
                        size_t ws_bytes, int32_t *err, void *stream)
{
    NvtxRange nvtx("moe.expert_ffn");
    int rc = check_layer(w);
    if (rc != MOE_OK)
        return rc;
    if (!ok_ptr(x) || !ok_ptr(offsets) || !ok_ptr(sorted_pair) || !ok_ptr(uniq) ||
        !ok_ptr(n_uniq) || !ok_ptr(y_pair) || !ok_ptr(y_shared) || !ok_ptr(err) ||
        workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || k < 1 || k > 32 || k > w->E || (long long)T * (k + 1) > (1LL << 24))
        return MOE_ERR_INVALID_ARG;
    if (!valid_mode(mode))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_ffn_workspace_bytes(T, k, w->d, w->f, mode))
        return MOE_ERR_WORKSPACE;
    mode = resolve_mode(mode, T);
    if (mode == MOE_MODE_HYBRID)
        return run_ffn_hybrid(w, x, offsets, sorted_pair, uniq, n_uniq, T, k, workspace, y_pair, y_shared, err,
                              as_stream(stream));
    if (mode == MOE_MODE_PREFILL) {
        PrefillFfnArgs pa{};
        pa.w = w;
        pa.x = x;
        pa.offsets = offsets;
        pa.sorted_pair = sorted_pair;
        pa.uniq = uniq;
        pa.n_uniq = n_uniq;
        pa.T = T;
        pa.k = k;
        pa.scratch = workspace;
        pa.y_pair = y_pair;
        pa.y_shared = y_shared;
        pa.err = err;
        return launch_ffn_prefill(pa, as_stream(stream));
    }
    FfnScratch sc{};
    ffn_scratch_layout(T, k, w->d, w->f, static_cast<uint8_t *>(workspace), &sc);
    const cudaStream_t s = as_stream(stream);
    rc = launch_act_frag(x, T, w->d, sc.x_frag, sc.x_scale, sc.work, kDecodeCounters, s);
    if (rc != MOE_OK)
        return rc;
    DecodeFfnArgs a{};
    a.w = w;
    a.offsets = offsets;
    a.sorted_pair = sorted_pair;
    a.uniq = uniq;
    a.n_uniq = n_uniq;
    a.T = T;
    a.k = k;
    a.x_frag = sc.x_frag;
    a.x_scale = sc.x_scale;
    a.h_frag = sc.h_frag;
    a.y_pair = y_pair;
    a.y_shared = y_shared;
    a.work = sc.work;
    a.err = err;
    return launch_ffn_decode(a, s);
}

int moe_combine(const float *y_pair, const float *y_shared, const float *topk_w,
                const int32_t *perm, const float *residual, int T, int k, int d, float *out,
                void *stream)
{
    NvtxRange nvtx("moe.combine");
    if (!ok_ptr(y_pair) || !ok_ptr(y_shared) || !ok_ptr(topk_w) || !ok_ptr(perm) ||
        !ok_opt(residual) || !ok_ptr(out) || T < 1 || k < 1 || k > 32 || d < 4 || d % 4 != 0)
        return MOE_ERR_INVALID_ARG;
    return launch_combine(y_pair, y_shared, topk_w, perm, residual, T, k, d, out, as_stream(stream));
}

int moe_rms_norm(const float *x, int T, int d, float eps, float *out, void *stream)
{
    NvtxRange nvtx("moe.rms_norm");
    if (!ok_ptr(x) || !ok_ptr(out) || T < 1 || T > (1 << 24) || d < 4 || d % 4 != 0 || d > (1 << 20) ||
        !(eps >= 0.0f) || !(eps < 1e30f))
        return MOE_ERR_INVALID_ARG;
    return launch_rms_norm(x, T, d, eps, out, as_stream(stream));
}

size_t moe_layer_workspace_bytes(int T, int k, int E, int d, int f, int mode)
{
    if (T < 1 || k < 1 || E < 1 || d < 1 || f < 1 || !valid_mode(mode))
        return 0;
    return layer_scratch_layout(T, k, E, d, f, mode, nullptr, nullptr);
}

int moe_layer_forward(const float *x, const float *w_gate, const float *bias,
                      const moe_layer_int4 *w, const float *residual, int T, int k, int normalize,
                      float route_scale, int mode, float *out, int32_t *topk_idx, float *topk_w,
                      uint64_t *hits, void *workspace, size_t ws_bytes, int32_t *err, void *stream)
{
    return moe_layer_forward_topp(x, w_gate, bias, w, residual, T, k, normalize, route_scale, 1.0f, mode, out,
                                  topk_idx, topk_w, hits, workspace, ws_bytes, err, stream);
}

}  // extern "C"

namespace {

// The layer (moe_layer_forward_topp); with out_normed set, the combine also writes RMSNorm(out)
// there (moe_layer_forward_norm).
int layer_forward(const float *x, const float *w_gate, const float *bias, const moe_layer_int4 *w,
                  const float *residual, int T, int k, int normalize, float route_scale, float top_p, int mode,
                  float *out, float *out_normed, float eps, int32_t *topk_idx, float *topk_w, uint64_t *hits,
                  void *workspace, size_t ws_bytes, int32_t *err, void *stream)
{
    int rc = check_layer(w);
    if (rc != MOE_OK)
        return rc;
    const int E = w->E, d = w->d, f = w->f;
    if (!ok_ptr(x) || !ok_ptr(w_gate) || !ok_opt(bias) || !ok_opt(residual) || !ok_ptr(out) ||
        !ok_opt(topk_idx) || !ok_opt(topk_w) || !ok_opt(hits) || !ok_ptr(err) ||
        workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return MOE_ERR_INVALID_ARG;
    if (!ok_route_shape(T, d, E, k) || (long long)T * (k + 1) > (1LL << 22) || !ok_top_p(top_p))
        return MOE_ERR_INVALID_ARG;
    if (!valid_mode(mode))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_layer_workspace_bytes(T, k, E, d, f, mode))
        return MOE_ERR_WORKSPACE;
    LayerScratch sc{};
    layer_scratch_layout(T, k, E, d, f, mode, static_cast<uint8_t *>(workspace), &sc);
    mode = resolve_mode(mode, T);
    int32_t *idx = topk_idx ? topk_idx : sc.idx;
    float *wt = topk_w ? topk_w : sc.w;
    const cudaStream_t s = as_stream(stream);
    if (mode == MOE_MODE_HYBRID) {
        rc = launch_router_logits(x, w_gate, T, d, E, sc.logits, s);
        if (rc == MOE_OK)
            rc = launch_router_topk(sc.logits, bias, T, E, k, normalize, route_scale, top_p, idx, wt, s);
        if (rc == MOE_OK)
            rc = launch_union(idx, T, k, E, sc.counts, sc.offsets, sc.perm, sc.sorted_pair, sc.uniq,
                              sc.n_uniq, hits, err, s);
        if (rc == MOE_OK)
            rc = run_ffn_hybrid(w, x, sc.offsets, sc.sorted_pair, sc.uniq, sc.n_uniq, T, k, sc.ffn, sc.y_pair,
                                sc.y_shared, err, s);
        if (rc != MOE_OK)
            return rc;
        if (out_normed != nullptr)
            return launch_combine_norm(sc.y_pair, nullptr, sc.y_shared, wt, sc.perm, residual, T, k, d, out,
                                       out_normed, eps, s, err);
        return launch_combine(sc.y_pair, sc.y_shared, wt, sc.perm, residual, T, k, d, out, s, err);
    }
    if (mode == MOE_MODE_PREFILL) {
        rc = launch_router_logits(x, w_gate, T, d, E, sc.logits, s);
        if (rc == MOE_OK)
            rc = launch_router_topk(sc.logits, bias, T, E, k, normalize, route_scale, top_p, idx, wt, s);
        if (rc == MOE_OK)
            rc = launch_union(idx, T, k, E, sc.counts, sc.offsets, sc.perm, sc.sorted_pair, sc.uniq,
                              sc.n_uniq, hits, err, s);
        if (rc != MOE_OK)
            return rc;
        PrefillFfnArgs pa{};
        pa.w = w;
        pa.x = x;
        pa.offsets = sc.offsets;
        pa.sorted_pair = sc.sorted_pair;
        pa.uniq = sc.uniq;
        pa.n_uniq = sc.n_uniq;
        pa.T = T;
        pa.k = k;
        pa.scratch = sc.ffn;
        // the routed outputs only feed the combine here: bf16 halves their traffic (the layer's
        // prefill tolerance, 2e-2 of the output RMS, is far above bf16's 2^-9 rounding)
        pa.y_pair = nullptr;
        pa.y_pair16 = reinterpret_cast<uint16_t *>(sc.y_pair);
        pa.y_shared = sc.y_shared;
        pa.err = err;
        rc = launch_ffn_prefill(pa, s);
        if (rc != MOE_OK)
            return rc;
        if (out_normed != nullptr)
            return launch_combine_norm(nullptr, reinterpret_cast<const uint16_t *>(sc.y_pair), sc.y_shared, wt,
                                       sc.perm, residual, T, k, d, out, out_normed, eps, s, err);
        return launch_combine_bf16(reinterpret_cast<const uint16_t *>(sc.y_pair), sc.y_shared, wt, sc.perm,
                                   residual, T, k, d, out, s, err);
    }
    FfnScratch fs{};
    ffn_scratch_layout(T, k, d, f, sc.ffn, &fs);
    // Small batches: logits + fragments of x in one grid, then top-k + union +
    // hits in one block; the kernels are chained with programmatic dependent
    // launches.  Larger batches use the separate stage kernels.
    const bool small = T <= 8 && T * k <= 64;
    if (small) {
        rc = launch_router_logits_frag(x, w_gate, T, d, E, sc.logits, fs.x_frag, fs.x_scale, fs.work,
                                       kDecodeCounters, s);
        if (rc == MOE_OK)
            rc = launch_select_union(sc.logits, bias, T, E, k, normalize, route_scale, top_p, idx, wt, sc.counts,
                                     sc.offsets, sc.perm, sc.sorted_pair, sc.uniq, sc.n_uniq, hits, err, s);
    } else {
        rc = launch_router_logits(x, w_gate, T, d, E, sc.logits, s);
        if (rc == MOE_OK)
            rc = launch_router_topk(sc.logits, bias, T, E, k, normalize, route_scale, top_p, idx, wt, s);
        if (rc == MOE_OK)
            rc = launch_union(idx, T, k, E, sc.counts, sc.offsets, sc.perm, sc.sorted_pair, sc.uniq,
                              sc.n_uniq, hits, err, s);
        if (rc == MOE_OK)
            rc = launch_act_frag(x, T, d, fs.x_frag, fs.x_scale, fs.work, kDecodeCounters, s);
    }
    if (rc != MOE_OK)
        return rc;
    DecodeFfnArgs a{};
    a.w = w;
    a.offsets = sc.offsets;
    a.sorted_pair = sc.sorted_pair;
    a.uniq = sc.uniq;
    a.n_uniq = sc.n_uniq;
    a.T = T;
    a.k = k;
    a.x_frag = fs.x_frag;
    a.x_scale = fs.x_scale;
    a.h_frag = fs.h_frag;
    a.y_pair = sc.y_pair;
    a.y_shared = sc.y_shared;
    a.work = fs.work;
    a.err = err;
    rc = launch_ffn_decode(a, s);
    if (rc != MOE_OK)
        return rc;
    if (out_normed != nullptr)
        return launch_combine_norm(sc.y_pair, nullptr, sc.y_shared, wt, sc.perm, residual, T, k, d, out, out_normed,
                                   eps, s, err);
    return launch_combine(sc.y_pair, sc.y_shared, wt, sc.perm, residual, T, k, d, out, s, err);
}

}  // namespace

extern "C" {

int moe_layer_forward_topp(const float *x, const float *w_gate, const float *bias,
                           const moe_layer_int4 *w, const float *residual, int T, int k, int normalize,
                           float route_scale, float top_p, int mode, float *out, int32_t *topk_idx,
                           float *topk_w, uint64_t *hits, void *workspace, size_t ws_bytes, int32_t *err,
                           void *stream)
{
    NvtxRange nvtx("moe.layer_forward");
    return layer_forward(x, w_gate, bias, w, residual, T, k, normalize, route_scale, top_p, mode, out, nullptr,
                         0.0f, topk_idx, topk_w, hits, workspace, ws_bytes, err, stream);
}

int moe_layer_forward_norm(const float *x, const float *w_gate, const float *bias,
                           const moe_layer_int4 *w, const float *residual, int T, int k, int normalize,
                           float route_scale, float top_p, int mode, float *out, float *out_normed, float eps,
                           int32_t *topk_idx, float *topk_w, uint64_t *hits, void *workspace, size_t ws_bytes,
                           int32_t *err, void *stream)
{
    NvtxRange nvtx("moe.layer_forward_norm");
    if (!ok_ptr(out_normed) || out_normed == out || out_normed == x || !(eps >= 0.0f) || !std::isfinite(eps))
        return MOE_ERR_INVALID_ARG;
    return layer_forward(x, w_gate, bias, w, residual, T, k, normalize, route_scale, top_p, mode, out, out_normed,
                         eps, topk_idx, topk_w, hits, workspace, ws_bytes, err, stream);
}

}  // extern "C"

namespace {

// The device address of a host buffer that kernels can read and write directly (page-locked and
// mapped: cudaHostAlloc, cudaHostRegister, on a system with unified addressing), else null.
void *mapped_host(const void *p)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();   // a pointer the runtime does not know: not an error of the call
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

}  // namespace

extern "C" {

size_t moe_layer_host_workspace_bytes(int T, int k, int E, int d, int f, int mode)
{
    const size_t layer = moe_layer_workspace_bytes(T, k, E, d, f, mode);
    if (layer == 0)
        return 0;
    return align_up(layer) + 2 * align_up((size_t)T * d * sizeof(float));
}

int moe_layer_forward_host(const float *x_host, const float *w_gate, const float *bias,
                           const moe_layer_int4 *w, const float *residual, int T, int k, int normalize,
                           float route_scale, float top_p, int mode, float *out_host, int32_t *topk_idx,
                           float *topk_w, uint64_t *hits, void *workspace, size_t ws_bytes, int32_t *err,
                           void *stream)
{
    NvtxRange nvtx("moe.layer_forward_host");
    if (x_host == nullptr || out_host == nullptr || w == nullptr || workspace == nullptr)
        return MOE_ERR_INVALID_ARG;
    const size_t layer = moe_layer_workspace_bytes(T, k, w->E, w->d, w->f, mode);
    if (layer == 0)
        return MOE_ERR_INVALID_ARG;
    const size_t rows = (size_t)T * w->d * sizeof(float);
    if (ws_bytes < moe_layer_host_workspace_bytes(T, k, w->E, w->d, w->f, mode))
        return MOE_ERR_WORKSPACE;
    uint8_t *base = static_cast<uint8_t *>(workspace);
    float *x_dev = reinterpret_cast<float *>(base + align_up(layer));
    float *out_dev = reinterpret_cast<float *>(base + align_up(layer) + align_up(rows));
    const cudaStream_t s = as_stream(stream);
    // Page-locked, mapped host buffers (the GPU addresses them over the host link): a kernel pulls the
    // rows and the combine writes the result straight into out_host, so the call is kernels only and
    // each launch still overlaps the end of the previous one.  Other host memory: one copy each way.
    const float *x_map = static_cast<const float *>(mapped_host(x_host));
    float *out_map = static_cast<float *>(mapped_host(out_host));
    if (x_map != nullptr && out_map != nullptr && aligned16(x_map) && aligned16(out_map)) {
        int rc = launch_copy_rows(x_map, x_dev, (long long)T * w->d, s);
        if (rc == MOE_OK)
            rc = moe_layer_forward_topp(x_dev, w_gate, bias, w, residual, T, k, normalize, route_scale, top_p, mode,
                                        out_map, topk_idx, topk_w, hits, workspace, layer, err, stream);
        return rc;
    }
    if (cudaMemcpyAsync(x_dev, x_host, rows, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int rc = moe_layer_forward_topp(x_dev, w_gate, bias, w, residual, T, k, normalize, route_scale, top_p,
                                          mode, out_dev, topk_idx, topk_w, hits, workspace, layer, err, stream);
    if (rc != MOE_OK)
        return rc;
    if (cudaMemcpyAsync(out_host, out_dev, rows, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // extern "C"
