// tier.cu -- Place and Overlap on GB300: a layer whose routed experts live in
// host memory, with a cache of expert blocks in device memory.
//
// Source: "Public Colibri Observation and Revision Ledger", "Exact Architecture
// and Data-Flow Reconstruction" (per layer: Route, Union, Place -- bring the
// missing experts to fast memory --, Overlap -- compute on the experts already
// there while the transfers run --, Learn); colibri README, "How it works"
// (the weights are spread over the levels of the memory hierarchy instead of
// all having to fit in one; where an expert sits changes how fast a token
// goes, never what it computes).
//
// On a GB300 the hierarchy is HBM3e and the Grace CPU's memory behind
// NVLink-C2C.  A tier holds, for one layer, n_slots expert blocks in device
// memory; every other expert stays in page-locked host memory.  A layer call:
//  1. routes and forms the union on the GPU, then copies the union's expert
//     list to the host and waits for it (the one host synchronisation);
//  2. plans: experts already in a slot are hits; each missing expert takes the
//     least recently used slot that is neither pinned nor used by this call,
//     and is copied there with one cudaMemcpyAsync per block (packed bytes,
//     scales) on the caller's copy stream;
//  3. runs the FFN over the resident experts and the shared expert at once,
//     while the copies proceed (Overlap), then waits for the copies (an event)
//     and runs the FFN over the copied experts; then the combine.
// The FFN kernels read routed expert e from slot slot_of[e] of the slot array;
// each output row is computed exactly as in the all-resident layer, so the
// results are the same bits whatever is resident.
//
// One stream of copies is used: on the GB300 machines measured, host-to-device
// copies from page-locked Grace memory reached about 190 GB/s on one stream
// and no more on 2 to 8 streams (a kernel reading host memory directly: 210
// GB/s).  Once every expert has a slot (n_slots = E, after each has been used
// once) nothing can miss: a call then skips the host round trip and runs the
// FFN once over the union with the full slot map, like a resident layer.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "moe_internal.h"

using namespace moe;

struct moe_tier_s {
    int E = 0, d = 0, f = 0, G = 0, n_slots = 0;
    const uint8_t *host_q = nullptr;
    const float *host_s = nullptr;
    uint8_t *slot_q = nullptr;
    float *slot_s = nullptr;
    size_t qb = 0, sc = 0;              // packed bytes and scale count of one expert block
    std::vector<int32_t> slot_of;       // [E]: the expert's slot, or -1
    std::vector<int32_t> expert_in;     // [n_slots]: the slot's expert, or -1
    std::vector<uint64_t> last_use;     // [n_slots]: call number of the last use
    std::vector<uint8_t> pinned;        // [n_slots]
    uint64_t clock = 0;                 // calls so far
    uint64_t stats[4] = {0, 0, 0, 0};   // hits, misses, bytes copied, calls
    int32_t *stage_in = nullptr;        // page-locked: n_uniq then the uniq list (device -> host)
    int32_t *stage_out = nullptr;       // page-locked: the upload image (host -> device)
    cudaEvent_t ev_route = nullptr, ev_copy = nullptr;
    int device = -1;
    int n_loaded = 0;                   // experts with a slot
    int32_t *stage_map = nullptr;       // page-locked: the full slot map, once every expert has a slot
    bool map_uploaded = false;          // stage_map is filled (every expert has a slot, none can miss)
    std::mutex mu;
};

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The upload image, ints: n1, n2, kTierCounters zeroed counters of the second FFN launch, then
// list1 [E] (resident experts), list2 [E] (copied experts), slot map [E].
constexpr int kTierHead = 8;
static_assert(kTierHead >= 2 + kDecodeCounters, "upload image head");
inline size_t tier_image_ints(int E) { return kTierHead + 3 * (size_t)E; }

// Plan one call: the n experts of uniq (ascending, distinct) are split into those in a slot
// (resident) and those to copy (missing, with their new slots in dst).  Tables are updated.
int tier_plan(moe_tier_s &t, const int32_t *uniq, int n, std::vector<int32_t> &resident,
              std::vector<int32_t> &missing, std::vector<int32_t> &dst)
{
    resident.clear();
    missing.clear();
    dst.clear();
    if (n < 0 || n > t.E)
        return MOE_ERR_INVALID_ARG;
    const uint64_t now = ++t.clock;
    for (int i = 0; i < n; i++) {
        const int e = uniq[i];
        if (e < 0 || e >= t.E)
            return MOE_ERR_INVALID_ARG;
        const int sl = t.slot_of[e];
        if (sl >= 0) {
            resident.push_back(e);
            t.last_use[sl] = now;
        } else {
            missing.push_back(e);
        }
    }
    int free_slots = 0;   // slots a missing expert may take: not pinned, not used by this call
    for (int sl = 0; sl < t.n_slots; sl++)
        free_slots += (!t.pinned[sl] && t.last_use[sl] != now) ? 1 : 0;
    if ((int)missing.size() > free_slots)
        return MOE_ERR_INVALID_ARG;   // more unique experts in this call than the tier can hold at once
    for (int e : missing) {
        // the least recently used slot that is not pinned and not used by this call
        int v = -1;
        for (int sl = 0; sl < t.n_slots; sl++) {
            if (t.pinned[sl] || t.last_use[sl] == now)
                continue;
            if (v < 0 || t.last_use[sl] < t.last_use[v])
                v = sl;
        }
        if (t.expert_in[v] >= 0)
            t.slot_of[t.expert_in[v]] = -1;
        else
            t.n_loaded++;
        t.expert_in[v] = e;
        t.slot_of[e] = v;
        t.last_use[v] = now;
        dst.push_back(v);
    }
    return MOE_OK;
}

// Copy the blocks of experts src[i] (host) to slots dst[i] on stream s: one copy per block of
// packed bytes and one per block of scales.
int tier_copy(moe_tier_s &t, const std::vector<int32_t> &src, const std::vector<int32_t> &dst, cudaStream_t s)
{
    for (size_t i = 0; i < src.size(); i++) {
        const int e = src[i], v = dst[i];
        if (cudaMemcpyAsync(t.slot_q + (size_t)v * t.qb, t.host_q + (size_t)e * t.qb, t.qb, cudaMemcpyHostToDevice,
                            s) != cudaSuccess ||
            cudaMemcpyAsync(t.slot_s + (size_t)v * t.sc, t.host_s + (size_t)e * t.sc, t.sc * sizeof(float),
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

void tier_free(moe_tier_s *t)
{
    if (t == nullptr)
        return;
    if (t->stage_in)
        cudaFreeHost(t->stage_in);
    if (t->stage_out)
        cudaFreeHost(t->stage_out);
    if (t->stage_map)
        cudaFreeHost(t->stage_map);
    if (t->ev_route)
        cudaEventDestroy(t->ev_route);
    if (t->ev_copy)
        cudaEventDestroy(t->ev_copy);
    delete t;
}

}  // namespace

extern "C" {

int moe_tier_create(int E, int d, int f, int G, const uint8_t *host_q, const float *host_s, uint8_t *slot_q,
                    float *slot_s, int n_slots, moe_tier *out)
{
    if (out == nullptr)
        return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    if (E < 1 || E > 1024 || n_slots < 1 || n_slots > E || d < 256 || f < 128 || host_q == nullptr ||
        host_s == nullptr || !aligned16(slot_q) || !aligned16(slot_s) || slot_q == nullptr || slot_s == nullptr)
        return MOE_ERR_INVALID_ARG;
    if ((G != 32 && G != 64) || d % 256 != 0 || f % 128 != 0 || (G == 64 && f % 256 != 0))
        return MOE_ERR_UNSUPPORTED;
    moe_tier_s *t = new (std::nothrow) moe_tier_s;
    if (t == nullptr)
        return MOE_ERR_INVALID_ARG;
    t->E = E;
    t->d = d;
    t->f = f;
    t->G = G;
    t->n_slots = n_slots;
    t->host_q = host_q;
    t->host_s = host_s;
    t->slot_q = slot_q;
    t->slot_s = slot_s;
    t->qb = moe_expert_q_bytes(d, f);
    t->sc = moe_expert_s_count(d, f, G);
    t->slot_of.assign(E, -1);
    t->expert_in.assign(n_slots, -1);
    t->last_use.assign(n_slots, 0);
    t->pinned.assign(n_slots, 0);
    if (cudaGetDevice(&t->device) != cudaSuccess ||
        cudaHostAlloc(reinterpret_cast<void **>(&t->stage_in), (E + 1) * sizeof(int32_t), cudaHostAllocDefault) !=
            cudaSuccess ||
        cudaHostAlloc(reinterpret_cast<void **>(&t->stage_out), tier_image_ints(E) * sizeof(int32_t),
                      cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(reinterpret_cast<void **>(&t->stage_map), E * sizeof(int32_t), cudaHostAllocDefault) !=
            cudaSuccess ||
        cudaEventCreateWithFlags(&t->ev_route, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&t->ev_copy, cudaEventDisableTiming) != cudaSuccess) {
        tier_free(t);
        return MOE_ERR_CUDA;
    }
    *out = t;
    return MOE_OK;
}

void moe_tier_destroy(moe_tier t) { tier_free(t); }

}  // extern "C"

namespace {

// Load experts into slots (least recently used unpinned slots first), optionally pinning them;
// the copies go on copy_stream, which is waited for.
int tier_load(moe_tier_s &t, const int32_t *experts, int n, bool pin, cudaStream_t cs)
{
    int npin = 0;
    for (int sl = 0; sl < t.n_slots; sl++)
        npin += t.pinned[sl];
    std::vector<int32_t> src, dst;
    std::vector<uint8_t> taken(t.n_slots, 0);   // slots filled by this call: not evicted by it
    for (int i = 0; i < n; i++) {
        const int e = experts[i];
        if (e < 0 || e >= t.E)
            return MOE_ERR_INVALID_ARG;
        int sl = t.slot_of[e];
        if (sl >= 0 && (t.pinned[sl] || !pin))
            continue;
        if (pin && npin + 1 >= t.n_slots)
            return MOE_ERR_INVALID_ARG;   // at least one slot stays free for the experts of a call
        if (sl < 0) {
            // an empty slot if there is one, else the least recently used one (neither pinned nor
            // filled by this call)
            for (int c = 0; c < t.n_slots && sl < 0; c++)
                if (t.expert_in[c] < 0 && !t.pinned[c] && !taken[c])
                    sl = c;
            if (sl < 0)
                for (int c = 0; c < t.n_slots; c++) {
                    if (t.pinned[c] || taken[c])
                        continue;
                    if (sl < 0 || t.last_use[c] < t.last_use[sl])
                        sl = c;
                }
            if (sl < 0)
                break;   // every slot is pinned or filled by this call: the rest of the list stays out
            if (t.expert_in[sl] >= 0)
                t.slot_of[t.expert_in[sl]] = -1;
            else
                t.n_loaded++;
            t.expert_in[sl] = e;
            t.slot_of[e] = sl;
            t.last_use[sl] = t.clock;   // as recent as the last call
            taken[sl] = 1;
            src.push_back(e);
            dst.push_back(sl);
            t.stats[2] += t.qb + t.sc * sizeof(float);
        }
        if (pin) {
            t.pinned[sl] = 1;
            npin++;
        }
    }
    int rc = tier_copy(t, src, dst, cs);
    if (rc != MOE_OK)
        return rc;
    if (t.n_loaded == t.E && !t.map_uploaded) {
        std::memcpy(t.stage_map, t.slot_of.data(), (size_t)t.E * sizeof(int32_t));
        t.map_uploaded = true;
    }
    // the next layer call treats these experts as resident: their copies must be complete
    return cudaStreamSynchronize(cs) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

extern "C" {

int moe_tier_pin(moe_tier t, const int32_t *experts, int n, void *copy_stream)
{
    NvtxRange nvtx("moe.tier_pin");
    if (t == nullptr || n < 0 || (n > 0 && experts == nullptr))
        return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(t->mu);
    return tier_load(*t, experts, n, true, reinterpret_cast<cudaStream_t>(copy_stream));
}

int moe_tier_prefetch(moe_tier t, const int32_t *experts, int n, void *copy_stream)
{
    NvtxRange nvtx("moe.tier_prefetch");
    if (t == nullptr || n < 0 || (n > 0 && experts == nullptr))
        return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(t->mu);
    return tier_load(*t, experts, n, false, reinterpret_cast<cudaStream_t>(copy_stream));
}

int moe_tier_unpin_all(moe_tier t)
{
    if (t == nullptr)
        return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(t->mu);
    for (int sl = 0; sl < t->n_slots; sl++)
        t->pinned[sl] = 0;
    return MOE_OK;
}

int moe_tier_stats(moe_tier t, uint64_t *stats)
{
    if (t == nullptr || stats == nullptr)
        return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(t->mu);
    std::memcpy(stats, t->stats, sizeof(t->stats));
    return MOE_OK;
}

int moe_tier_slots(moe_tier t, int32_t *expert_in_slot, uint8_t *pinned)
{
    if (t == nullptr)
        return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(t->mu);
    for (int sl = 0; sl < t->n_slots; sl++) {
        if (expert_in_slot)
            expert_in_slot[sl] = t->expert_in[sl];
        if (pinned)
            pinned[sl] = t->pinned[sl];
    }
    return MOE_OK;
}

size_t moe_tier_workspace_bytes(int T, int k, int E, int d, int f, int mode)
{
    const size_t layer = moe_layer_workspace_bytes(T, k, E, d, f, mode);
    if (layer == 0)
        return 0;
    return align_up(layer) + align_up(tier_image_ints(E) * sizeof(int32_t));
}

int moe_layer_forward_tier(const float *x, const float *w_gate, const float *bias, moe_tier tier,
                           const uint8_t *shared_q, const float *shared_s, const float *residual, int T, int k,
                           int normalize, float route_scale, float top_p, int mode, float *out, int32_t *topk_idx,
                           float *topk_w, uint64_t *hits, void *workspace, size_t ws_bytes, int32_t *err,
                           void *stream, void *copy_stream)
{
    NvtxRange nvtx("moe.layer_forward_tier");
    if (tier == nullptr)
        return MOE_ERR_INVALID_ARG;
    moe_tier_s &t = *tier;
    const int E = t.E, d = t.d, f = t.f;
    if (x == nullptr || w_gate == nullptr || out == nullptr || err == nullptr || shared_q == nullptr ||
        shared_s == nullptr || !aligned16(x) || !aligned16(w_gate) || !aligned16(out) || !aligned16(err) ||
        !aligned16(shared_q) || !aligned16(shared_s) || !aligned16(bias) || !aligned16(residual) ||
        !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(hits) || workspace == nullptr ||
        (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || k < 1 || k > 32 || k > E || (long long)T * (k + 1) > (1LL << 22) || !(top_p > 0.0f) ||
        !(top_p < 3.0e38f) || (mode != MOE_MODE_AUTO && mode != MOE_MODE_DECODE && mode != MOE_MODE_PREFILL))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_tier_workspace_bytes(T, k, E, d, f, mode))
        return MOE_ERR_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != t.device)
        return MOE_ERR_INVALID_ARG;   // the tier's events and staging belong to the device it was made on
    std::lock_guard<std::mutex> lock(t.mu);

    uint8_t *base = static_cast<uint8_t *>(workspace);
    LayerScratch sc{};
    const size_t layer_bytes = layer_scratch_layout(T, k, E, d, f, mode, base, &sc);
    int32_t *img = reinterpret_cast<int32_t *>(base + align_up(layer_bytes));
    int32_t *n1 = img, *n2 = img + 1, *work2 = img + 2, *list1 = img + kTierHead, *list2 = list1 + E,
            *map = list2 + E;
    mode = resolve_mode_plain(mode, T);   // the tier has no hybrid path
    int32_t *idx = topk_idx ? topk_idx : sc.idx;
    float *wt = topk_w ? topk_w : sc.w;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(copy_stream);

    // ---- Route and Union on the GPU, then the union's expert list to the host
    int rc = launch_router_logits(x, w_gate, T, d, E, sc.logits, s);
    if (rc == MOE_OK)
        rc = launch_router_topk(sc.logits, bias, T, E, k, normalize, route_scale, top_p, idx, wt, s);
    if (rc == MOE_OK)
        rc = launch_union(idx, T, k, E, sc.counts, sc.offsets, sc.perm, sc.sorted_pair, sc.uniq, sc.n_uniq, hits,
                          err, s);
    if (rc != MOE_OK)
        return rc;
    moe_layer_int4 view{t.slot_q, t.slot_s, shared_q, shared_s, t.n_slots, d, f, t.G};
    if (t.map_uploaded) {
        // every expert has a slot: no host round trip, one FFN launch over the union
        if (cudaMemcpyAsync(map, t.stage_map, (size_t)E * sizeof(int32_t), cudaMemcpyHostToDevice, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        t.stats[3] += 1;
        if (mode == MOE_MODE_PREFILL) {
            PrefillFfnArgs pa{};
            pa.w = &view;
            pa.x = x;
            pa.offsets = sc.offsets;
            pa.sorted_pair = sc.sorted_pair;
            pa.uniq = sc.uniq;
            pa.n_uniq = sc.n_uniq;
            pa.T = T;
            pa.k = k;
            pa.scratch = sc.ffn;
            pa.y_pair = nullptr;
            pa.y_pair16 = reinterpret_cast<uint16_t *>(sc.y_pair);
            pa.y_shared = sc.y_shared;
            pa.slot_of = map;
            pa.n_experts = E;
            pa.err = err;
            rc = launch_ffn_prefill(pa, s);
            if (rc != MOE_OK)
                return rc;
            return launch_combine_bf16(reinterpret_cast<const uint16_t *>(sc.y_pair), sc.y_shared, wt, sc.perm,
                                       residual, T, k, d, out, s, err);
        }
        FfnScratch fs{};
        ffn_scratch_layout(T, k, d, f, sc.ffn, &fs);
        rc = launch_act_frag(x, T, d, fs.x_frag, fs.x_scale, fs.work, kDecodeCounters, s);
        DecodeFfnArgs a{};
        a.w = &view;
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
        a.slot_of = map;
        a.n_experts = E;
        a.err = err;
        if (rc == MOE_OK)
            rc = launch_ffn_decode(a, s);
        if (rc != MOE_OK)
            return rc;
        return launch_combine(sc.y_pair, sc.y_shared, wt, sc.perm, residual, T, k, d, out, s, err);
    }
    if (cudaMemcpyAsync(t.stage_in, sc.n_uniq, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(t.stage_in + 1, sc.uniq, (size_t)E * sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaEventRecord(t.ev_route, s) != cudaSuccess || cudaEventSynchronize(t.ev_route) != cudaSuccess)
        return MOE_ERR_CUDA;
    // (every earlier kernel of this stream, the previous layer call's FFN included, has finished: the
    // slots can be rewritten)

    // ---- Place: plan, and start the copies of the missing experts
    std::vector<int32_t> resident, missing, dst;
    const int n = t.stage_in[0];
    rc = tier_plan(t, t.stage_in + 1, n, resident, missing, dst);
    if (rc != MOE_OK)
        return rc;
    rc = tier_copy(t, missing, dst, cs);
    if (rc != MOE_OK) {
        for (size_t i = 0; i < missing.size(); i++) {   // their slots hold nothing usable now
            t.slot_of[missing[i]] = -1;
            t.expert_in[dst[i]] = -1;
        }
        return rc;
    }
    if (!missing.empty() && cudaEventRecord(t.ev_copy, cs) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (t.n_loaded == E && !t.map_uploaded) {   // from the next call on, nothing can miss
        std::memcpy(t.stage_map, t.slot_of.data(), (size_t)E * sizeof(int32_t));
        t.map_uploaded = true;
    }
    t.stats[0] += resident.size();
    t.stats[1] += missing.size();
    t.stats[2] += missing.size() * (t.qb + t.sc * sizeof(float));
    t.stats[3] += 1;

    // ---- the upload image: list sizes, zeroed counters, lists, slot map
    int32_t *o = t.stage_out;
    std::memset(o, 0, kTierHead * sizeof(int32_t));
    o[0] = (int32_t)resident.size();
    o[1] = (int32_t)missing.size();
    std::memcpy(o + kTierHead, resident.data(), resident.size() * sizeof(int32_t));
    std::memcpy(o + kTierHead + E, missing.data(), missing.size() * sizeof(int32_t));
    std::memcpy(o + kTierHead + 2 * (size_t)E, t.slot_of.data(), (size_t)E * sizeof(int32_t));
    if (cudaMemcpyAsync(img, o, tier_image_ints(E) * sizeof(int32_t), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;

    // ---- Overlap: the FFN over the resident experts (and the shared expert) now, over the copied
    // ones once their copies are done
    if (mode == MOE_MODE_PREFILL) {
        PrefillFfnArgs pa{};
        pa.w = &view;
        pa.x = x;
        pa.offsets = sc.offsets;
        pa.sorted_pair = sc.sorted_pair;
        pa.uniq = list1;
        pa.n_uniq = n1;
        pa.T = T;
        pa.k = k;
        pa.scratch = sc.ffn;
        // routed outputs in bf16, as moe_layer_forward keeps them on this path (they only feed the combine)
        pa.y_pair = nullptr;
        pa.y_pair16 = reinterpret_cast<uint16_t *>(sc.y_pair);
        pa.y_shared = sc.y_shared;
        pa.slot_of = map;
        pa.n_experts = E;   // the union's offsets cover all E experts, the view only the slots
        pa.with_shared = 1;
        pa.err = err;
        rc = launch_ffn_prefill(pa, s);
        if (rc == MOE_OK && !missing.empty()) {
            if (cudaStreamWaitEvent(s, t.ev_copy, 0) != cudaSuccess)
                return MOE_ERR_CUDA;
            pa.uniq = list2;
            pa.n_uniq = n2;
            pa.with_shared = 0;
            rc = launch_ffn_prefill(pa, s);
        }
    } else {
        FfnScratch fs{};
        ffn_scratch_layout(T, k, d, f, sc.ffn, &fs);
        rc = launch_act_frag(x, T, d, fs.x_frag, fs.x_scale, fs.work, kDecodeCounters, s);
        DecodeFfnArgs a{};
        a.w = &view;
        a.offsets = sc.offsets;
        a.sorted_pair = sc.sorted_pair;
        a.uniq = list1;
        a.n_uniq = n1;
        a.T = T;
        a.k = k;
        a.x_frag = fs.x_frag;
        a.x_scale = fs.x_scale;
        a.h_frag = fs.h_frag;
        a.y_pair = sc.y_pair;
        a.y_shared = sc.y_shared;
        a.work = fs.work;
        a.slot_of = map;
        a.n_experts = E;
        a.with_shared = 1;
        a.err = err;
        if (rc == MOE_OK)
            rc = launch_ffn_decode(a, s);
        if (rc == MOE_OK && !missing.empty()) {
            if (cudaStreamWaitEvent(s, t.ev_copy, 0) != cudaSuccess)
                return MOE_ERR_CUDA;
            a.uniq = list2;
            a.n_uniq = n2;
            a.with_shared = 0;
            a.work = work2;
            rc = launch_ffn_decode(a, s);
        }
    }
    if (rc != MOE_OK)
        return rc;
    if (mode == MOE_MODE_PREFILL)
        return launch_combine_bf16(reinterpret_cast<const uint16_t *>(sc.y_pair), sc.y_shared, wt, sc.perm, residual,
                                   T, k, d, out, s, err);
    return launch_combine(sc.y_pair, sc.y_shared, wt, sc.perm, residual, T, k, d, out, s, err);
}

}  // extern "C"
