// union.cu -- Union and Learn stages: group the batch's (token, slot) pairs by
// expert so that every unique expert is read once, and bump the per-expert hit
// counters.
//
// Sources: "Public Colibri Observation and Revision Ledger", "Exact
// Architecture and Data-Flow Reconstruction" (the Union stage combines the
// batch's expert requests; the Learn stage counts per expert how often it was
// picked), and the figure caption of "Cache/Prefetch Design Comparison" (with
// the batch union, a selected expert's weights are fetched a single time).
//
// One thread block: a shared-memory histogram (atomics only count), a block
// scan for the offsets, then a stable placement pass over the pairs in chunks
// of the block size, where a pair's rank among equal experts is its rank in
// its warp (match_any) plus the counts of earlier warps and earlier chunks.
// The result is deterministic and independent of scheduling.
#include "moe_internal.h"
#include "ptx.cuh"
#include "route_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxE = 1024;

// Exclusive block scan of one int per thread (kThreads threads); returns the
// exclusive prefix and writes the total to *total.
__device__ int block_exclusive_scan(int v, int *warp_sums, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off)
            inc += n;
    }
    if (lane == 31)
        warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int ws = warp_sums[lane];
        int wi = ws;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off)
                wi += n;
        }
        warp_sums[lane] = wi - ws;   // exclusive prefix of warp totals
        if (lane == 31)
            *total = wi;
    }
    __syncthreads();
    const int r = warp_sums[warp] + inc - v;
    __syncthreads();
    return r;
}

__device__ void union_chunked(const int32_t *__restrict__ idx, int P, int E, int32_t *__restrict__ counts,
                              int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                              int32_t *__restrict__ sorted_pair, int32_t *__restrict__ uniq,
                              int32_t *__restrict__ n_uniq, uint64_t *__restrict__ hits, int32_t *__restrict__ err,
                              int *dyn)
{
    int *cnt = dyn;                 // [E] pairs per expert
    int *base = dyn + E;            // [E] next free position per expert
    unsigned short *wcnt = reinterpret_cast<unsigned short *>(dyn + 2 * E);   // [kWarps][E]
    __shared__ int warp_sums[32];
    __shared__ int total;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int e = tid; e < E; e += kThreads)
        cnt[e] = 0;
    __syncthreads();
    int bad = 0;
    for (int p = tid; p < P; p += kThreads) {
        const int e = idx[p];
        if (e >= 0 && e < E)
            atomicAdd(&cnt[e], 1);
        else if (e != -1)   // -1: an empty slot
            bad = 1;
    }
    if (__syncthreads_or(bad) && tid == 0)
        atomicOr(err, MOE_DEVERR_BAD_EXPERT);

    // offsets (exclusive scan over ascending expert id) and uniq list
    for (int e0 = 0; e0 < E; e0 += kThreads) {
        const int e = e0 + tid;
        const int c = e < E ? cnt[e] : 0;
        const int carry = e0 == 0 ? 0 : base[e0 - 1] + cnt[e0 - 1];
        const int ex = block_exclusive_scan(c, warp_sums, &total) + carry;
        if (e < E) {
            base[e] = ex;
            offsets[e] = ex;
            counts[e] = c;
            if (hits && c > 0)
                atomicAdd(reinterpret_cast<unsigned long long *>(hits + e), (unsigned long long)c);   // no read back
        }
        __syncthreads();
    }
    if (tid == 0)
        offsets[E] = E > 0 ? base[E - 1] + cnt[E - 1] : 0;
    {
        int carry = 0;
        for (int e0 = 0; e0 < E; e0 += kThreads) {
            const int e = e0 + tid;
            const int flag = (e < E && cnt[e] > 0) ? 1 : 0;
            const int ex = block_exclusive_scan(flag, warp_sums, &total) + carry;
            if (flag)
                uniq[ex] = e;
            carry += total;
            __syncthreads();
        }
        if (tid == 0)
            *n_uniq = carry;
    }

    // stable placement, one chunk of kThreads pairs at a time
    for (int c0 = 0; c0 < P; c0 += kThreads) {
        for (int i = tid; i < kWarps * E; i += kThreads)
            wcnt[i] = 0;
        __syncthreads();
        const int p = c0 + tid;
        int e = -1;
        if (p < P) {
            e = idx[p];
            if (e < 0 || e >= E)
                e = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rank_in_warp == 0)
            wcnt[warp * E + e] = (unsigned short)__popc(peers);
        __syncthreads();
        int pos = -1;
        if (e >= 0) {
            int before = 0;
            for (int w = 0; w < warp; w++)
                before += wcnt[w * E + e];
            pos = base[e] + before + rank_in_warp;
        }
        if (p < P) {
            perm[p] = pos;
            if (pos >= 0)
                sorted_pair[pos] = p;
        }
        __syncthreads();
        // advance the per-expert bases by this chunk's counts
        for (int x = tid; x < E; x += kThreads) {
            int s = 0;
            for (int w = 0; w < kWarps; w++)
                s += wcnt[w * E + x];
            base[x] += s;
        }
        __syncthreads();
    }
}

size_t union_smem_bytes(int E)
{
    return (size_t)E * 2 * sizeof(int) + (size_t)kWarps * E * sizeof(unsigned short);
}

// Bitmap union for batches whose (expert x token) bitmap fits in shared memory.
// The top-k gives every token distinct experts, so the pairs of expert e are
// the set bits of row e of a bitmap over tokens, and a pair's rank inside its
// expert's group is the number of set bits before its token: a per-word prefix
// of bit counts plus one masked popcount.  Every step is one pass over the
// pairs or the bitmap, all threads in parallel.  A token that names an expert
// twice (not a top-k result, but a caller may pass any ids) sends the whole
// call to the chunked algorithm above, which ranks pairs by position.
__host__ __device__ constexpr size_t union_bitmap_smem_bytes(int E, int T)
{
    return (size_t)E * ((T + 31) / 32) * (4 + 2) + (size_t)E * 4 + 16;
}
constexpr size_t kBitmapSmemMax = 200 * 1024;

__global__ void __launch_bounds__(kThreads)
union_kernel(const int32_t *__restrict__ idx, int T, int k, int E, int use_bitmap, int32_t *__restrict__ counts,
             int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
             int32_t *__restrict__ sorted_pair, int32_t *__restrict__ uniq,
             int32_t *__restrict__ n_uniq, uint64_t *__restrict__ hits, int32_t *__restrict__ err)
{
    extern __shared__ int dyn[];
    __shared__ int warp_sums[32];
    __shared__ int total;
    const int P = T * k;
    if (!use_bitmap) {
        union_chunked(idx, P, E, counts, offsets, perm, sorted_pair, uniq, n_uniq, hits, err, dyn);
        return;
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int W = (T + 31) / 32;                                      // bitmap words per expert
    // word-major layouts (word w of expert e at w * E + e): the lanes of a warp touch different
    // experts of the same word, i.e. different banks
    uint32_t *bits = reinterpret_cast<uint32_t *>(dyn);                 // [W][E]
    int *base = dyn + (size_t)E * W;                                    // [E] first position of the expert
    unsigned short *pre = reinterpret_cast<unsigned short *>(base + E); // [W][E] set bits before the word
    for (int i = tid; i < E * W; i += kThreads)
        bits[i] = 0u;
    __syncthreads();
    int bad = 0, dup = 0;
    for (int p = tid; p < P; p += kThreads) {
        const int e = idx[p];
        if (e < 0 || e >= E) {
            bad |= e != -1 ? 1 : 0;   // -1: an empty slot
            continue;
        }
        const int t = p / k;
        const uint32_t b = 1u << (t & 31);
        if (atomicOr(&bits[(t >> 5) * E + e], b) & b)
            dup = 1;
    }
    bad = __syncthreads_or(bad);
    if (__syncthreads_or(dup)) {   // the same expert twice in one token: rank by position instead
        union_chunked(idx, P, E, counts, offsets, perm, sorted_pair, uniq, n_uniq, hits, err, dyn);
        return;
    }
    if (bad && tid == 0)
        atomicOr(err, MOE_DEVERR_BAD_EXPERT);
    // per expert (one thread each): prefix of bit counts over the words
    for (int e = tid; e < E; e += kThreads) {
        int run = 0;
        for (int w = 0; w < W; w++) {
            pre[(size_t)w * E + e] = (unsigned short)run;
            run += __popc(bits[(size_t)w * E + e]);
        }
        base[e] = run;   // the expert's count, turned into its first position below
    }
    __syncthreads();
    // offsets (exclusive scan over ascending expert id), counts, hits, uniq
    int carry = 0, ucarry = 0;
    for (int e0 = 0; e0 < E; e0 += kThreads) {
        const int e = e0 + tid;
        const int c = e < E ? base[e] : 0;
        const int ex = block_exclusive_scan(c, warp_sums, &total) + carry;
        const int add = total;
        const int flag = c > 0 ? 1 : 0;
        const int ux = block_exclusive_scan(flag, warp_sums, &total) + ucarry;
        if (e < E) {
            base[e] = ex;
            offsets[e] = ex;
            counts[e] = c;
            if (hits && c > 0)
                atomicAdd(reinterpret_cast<unsigned long long *>(hits + e), (unsigned long long)c);   // no read back
            if (flag)
                uniq[ux] = e;
        }
        carry += add;
        ucarry += total;
        __syncthreads();
    }
    if (tid == 0) {
        offsets[E] = carry;
        *n_uniq = ucarry;
    }
    // placement: rank = set bits of the expert's row before the token
    for (int p = tid; p < P; p += kThreads) {
        const int e = idx[p];
        int pos = -1;
        if (e >= 0 && e < E) {
            const int t = p / k, w = t >> 5;
            const uint32_t below = bits[(size_t)w * E + e] & ((1u << (t & 31)) - 1u);
            pos = base[e] + pre[(size_t)w * E + e] + __popc(below);
            sorted_pair[pos] = p;
        }
        perm[p] = pos;
    }
}

// ------------------------------------------------- small-batch select+union
// One block of 256 threads for batches of at most 8 tokens and 64 pairs:
// warp t selects token t's experts (the same top-k as topk_kernel), then the
// block forms the union as above (histogram, exclusive scans over ascending
// expert id, stable placement by counting earlier pairs of the same expert)
// and bumps the hit counters.
constexpr int kSelThreads = 256;
static_assert(kSelThreads == kTopkThreads, "the select kernel runs topk_block");
constexpr int kSelMaxPairs = 64;

__global__ void __launch_bounds__(kSelThreads)
select_union_kernel(const float *__restrict__ logits, const float *__restrict__ bias, int T, int E, int k,
                    int normalize, float route_scale, float top_p, int32_t *__restrict__ idx,
                    float *__restrict__ w,
                    int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                    int32_t *__restrict__ sorted_pair, int32_t *__restrict__ uniq,
                    int32_t *__restrict__ n_uniq, uint64_t *__restrict__ hits, int32_t *__restrict__ err)
{
    __shared__ int se[kSelMaxPairs];      // expert of pair p (INT_MAX when out of range)
    __shared__ int sfirst[kSelMaxPairs];  // 1 when pair p is the first pair of its expert
    extern __shared__ __align__(16) uint8_t tk_smem[];
    const int tid = threadIdx.x;
    griddep_launch_dependents();
    griddep_wait();   // logits come from the previous kernel
    if (E <= 32 * kWarpTopkPer)
        topk_warp(logits, bias, 0, T, E, k, normalize, route_scale, top_p, idx, w, se);
    else
        topk_block(logits, bias, 0, T, E, k, normalize, route_scale, top_p, idx, w, se, tk_smem);
    const int P = T * k;
    if (tid < P) {
        const int e = se[tid];
        if (e < 0 || e >= E) {
            if (e != -1)   // -1: a slot emptied by top-p
                atomicOr(err, MOE_DEVERR_BAD_EXPERT);
            se[tid] = INT_MAX;
        }
    }
    __syncthreads();
    if (tid < P) {
        const int e = se[tid];
        int first = e != INT_MAX ? 1 : 0;
        for (int q = 0; q < tid; q++)
            first = se[q] == e ? 0 : first;
        sfirst[tid] = first;
    }
    __syncthreads();
    // pairs: position = (#pairs of smaller experts) + (#earlier pairs of the same expert)
    if (tid < P) {
        const int e = se[tid];
        int pos = -1;
        if (e != INT_MAX) {
            pos = 0;
            for (int q = 0; q < P; q++) {
                const int eq = se[q];
                pos += (eq < e || (eq == e && q < tid)) ? 1 : 0;
            }
            sorted_pair[pos] = tid;
        }
        perm[tid] = pos;
    }
    // experts: count, exclusive offset, rank among the distinct experts, hits
    for (int e = tid; e <= E; e += kSelThreads) {
        int cnt = 0, before = 0, ubefore = 0;
        for (int q = 0; q < P; q++) {
            const int eq = se[q];
            cnt += eq == e ? 1 : 0;
            before += eq < e ? 1 : 0;
            ubefore += (eq < e && sfirst[q]) ? 1 : 0;
        }
        offsets[e] = before;
        if (e == E) {
            *n_uniq = ubefore;
            continue;
        }
        counts[e] = cnt;
        if (cnt > 0) {
            uniq[ubefore] = e;
            if (hits)
                atomicAdd(reinterpret_cast<unsigned long long *>(hits + e), (unsigned long long)cnt);   // no read back
        }
    }
}

// Split of the union's expert list for the hybrid FFN: a stable compaction of the flags
// "at most max_cold pairs" and "more", one block of up to 1024 threads (warp ballots, then a scan
// of the 32 warp counts), looping when the list is longer than the block.
constexpr int kSplitThreads = 1024;

__global__ void __launch_bounds__(kSplitThreads)
split_units_kernel(const int32_t *__restrict__ offsets, const int32_t *__restrict__ uniq,
                   const int32_t *__restrict__ n_uniq, int E, int cap, int max_cold, int32_t *__restrict__ uniq_cold,
                   int32_t *__restrict__ n_cold, int32_t *__restrict__ uniq_hot, int32_t *__restrict__ n_hot,
                   int32_t *__restrict__ err)
{
    __shared__ int wcold[kSplitThreads / 32], whot[kSplitThreads / 32];
    griddep_launch_dependents();
    griddep_wait();   // the union comes from the previous kernel
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = max(0, min(*n_uniq, cap));   // cap: min(E, pairs), the lists' length
    int cold_base = 0, hot_base = 0;
    for (int base = 0; base < n; base += kSplitThreads) {
        const int i = base + (int)threadIdx.x;
        int e = -1;
        bool cold = false, hot = false;
        if (i < n) {
            e = uniq[i];
            if (e >= 0 && e < E) {
                const int m = offsets[e + 1] - offsets[e];
                cold = m <= max_cold;
                hot = !cold;
            } else {
                atomicOr(err, MOE_DEVERR_BAD_EXPERT);
            }
        }
        const unsigned bc = __ballot_sync(0xffffffffu, cold), bh = __ballot_sync(0xffffffffu, hot);
        if (lane == 0) {
            wcold[warp] = __popc(bc);
            whot[warp] = __popc(bh);
        }
        __syncthreads();
        int pc = cold_base, ph = hot_base, tc = 0, th = 0;
        for (int w = 0; w < kSplitThreads / 32; w++) {
            pc += w < warp ? wcold[w] : 0;
            ph += w < warp ? whot[w] : 0;
            tc += wcold[w];
            th += whot[w];
        }
        const unsigned below = (1u << lane) - 1u;
        if (cold)
            uniq_cold[pc + __popc(bc & below)] = e;
        if (hot)
            uniq_hot[ph + __popc(bh & below)] = e;
        cold_base += tc;
        hot_base += th;
        __syncthreads();   // the warp counts are rewritten by the next round
    }
    if (threadIdx.x == 0) {
        *n_cold = cold_base;
        *n_hot = hot_base;
    }
}

__global__ void hits_kernel(const int32_t *__restrict__ counts, int E, uint64_t *__restrict__ hits)
{
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e < E)
        hits[e] += (uint64_t)counts[e];
}

}  // namespace

int launch_union(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
                 int32_t *perm, int32_t *sorted_pair, int32_t *uniq, int32_t *n_uniq,
                 uint64_t *hits, int32_t *err, cudaStream_t s)
{
    const size_t bm = union_bitmap_smem_bytes(E, T);
    // one chunk of the chunked path is cheaper than the bitmap's passes; beyond that the bitmap wins
    const int use_bitmap = (bm <= kBitmapSmemMax && T * k > kThreads) ? 1 : 0;
    const size_t chunked = union_smem_bytes(E);
    const size_t smem = use_bitmap && bm > chunked ? bm : chunked;   // the bitmap path may fall back
    static thread_local int configured_for = -1;   // per host thread, per device attribute set once
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        const size_t most = kBitmapSmemMax > union_smem_bytes(kMaxE) ? kBitmapSmemMax : union_smem_bytes(kMaxE);
        if (cudaFuncSetAttribute(union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
        configured_for = dev;
    }
    union_kernel<<<1, kThreads, smem, s>>>(idx, T, k, E, use_bitmap, counts, offsets, perm, sorted_pair, uniq,
                                        n_uniq, hits, err);
    return cuda_status(cudaGetLastError());
}

int launch_split_units(const int32_t *offsets, const int32_t *uniq, const int32_t *n_uniq, int E, int pairs,
                       int max_cold, int32_t *uniq_cold, int32_t *n_cold, int32_t *uniq_hot, int32_t *n_hot,
                       int32_t *err, cudaStream_t s)
{
    if (E < 1 || E > kMaxE || pairs < 1)
        return MOE_ERR_UNSUPPORTED;
    const int cap = E < pairs ? E : pairs;
    return launch_pdl(split_units_kernel, 1, kSplitThreads, 0, s, offsets, uniq, n_uniq, E, cap, max_cold,
                      uniq_cold, n_cold, uniq_hot, n_hot, err);
}

int launch_select_union(const float *logits, const float *bias, int T, int E, int k, int normalize,
                        float route_scale, float top_p, int32_t *idx, float *w, int32_t *counts, int32_t *offsets,
                        int32_t *perm, int32_t *sorted_pair, int32_t *uniq, int32_t *n_uniq,
                        uint64_t *hits, int32_t *err, cudaStream_t s)
{
    if (T > kTopkTokens || T * k > kSelMaxPairs || E > kMaxE)
        return MOE_ERR_UNSUPPORTED;
    // the warp form (E <= 256) keeps everything in registers: no shared memory to reserve
    const size_t smem = E <= 32 * kWarpTopkPer ? 0 : topk_smem_bytes(E, k);
    if (smem > 48 * 1024 && cudaFuncSetAttribute(select_union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  (int)smem) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_pdl(select_union_kernel, 1, kSelThreads, smem, s, logits, bias, T, E, k, normalize, route_scale,
                      top_p, idx, w, counts, offsets, perm, sorted_pair, uniq, n_uniq, hits, err);
}

int launch_hits(const int32_t *counts, int E, uint64_t *hits, cudaStream_t s)
{
    hits_kernel<<<(E + 255) / 256, 256, 0, s>>>(counts, E, hits);
    return cuda_status(cudaGetLastError());
}

}  // namespace moe
