// combine.cu -- score-weighted combine of the routed experts' outputs with the
// always-on shared expert and the residual stream:
//   out[t][c] = res[t][c] + y_shared[t][c] + sum_{j<k} w[t][j] * y_pair[perm[t*k+j]][c]
// in slot order j (deterministic).  Source: "Public Colibri Observation and
// Revision Ledger", "Exact Architecture and Data-Flow Reconstruction" (selected
// experts weighted by the router; the shared branch is always used).
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float4 load4(const float4 *p, size_t i) { return p[i]; }
__device__ __forceinline__ float4 load4(const uint2 *p, size_t i)   // 4 bf16
{
    const uint2 u = p[i];
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
}

// One thread per 4 consecutive columns of one token.  Y: float4 (fp32 y_pair)
// or uint2 (four bf16).
template <typename Y>
__global__ void __launch_bounds__(256)
combine_kernel(const Y *__restrict__ y_pair, const float4 *__restrict__ y_shared,
               const float *__restrict__ w, const int32_t *__restrict__ perm,
               const float4 *res, int T, int k, int d4, float4 *out, int32_t *err)
{
    griddep_launch_dependents();
    griddep_wait();   // y_pair / y_shared come from the previous kernel
    const long long id = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (id >= (long long)T * d4)
        return;
    const int t = (int)(id / d4), c = (int)(id % d4);
    float4 acc = res ? res[id] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 ys = y_shared[id];
    acc.x += ys.x; acc.y += ys.y; acc.z += ys.z; acc.w += ys.w;
    // slots in groups of 8: the group's positions and weights, then all of its rows, are loaded
    // before the first is added (two round trips per group instead of two per slot); the sum
    // still runs in slot order
    constexpr int kG = 8;
    for (int j0 = 0; j0 < k; j0 += kG) {
        int q[kG];
        float wj[kG];
#pragma unroll
        for (int u = 0; u < kG; u++) {
            const int j = j0 + u;
            q[u] = j < k ? perm[(size_t)t * k + j] : -1;
            if (!MOE_IN_BOUNDS(q[u] < T * k, err))
                q[u] = -1;
            wj[u] = j < k ? w[(size_t)t * k + j] : 0.f;
        }
        float4 y[kG];
#pragma unroll
        for (int u = 0; u < kG; u++)
            y[u] = q[u] >= 0 ? load4(y_pair, (size_t)q[u] * d4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kG; u++)
            if (q[u] >= 0) {
                acc.x = fmaf(wj[u], y[u].x, acc.x);
                acc.y = fmaf(wj[u], y[u].y, acc.y);
                acc.z = fmaf(wj[u], y[u].z, acc.z);
                acc.w = fmaf(wj[u], y[u].w, acc.w);
            }
    }
    out[id] = acc;
}

// The combine and, for the next layer of a pre-norm stack, the RMS normalisation
// of the combined row, one CTA of kCNThreads per token row.  Each thread forms
// float4 c = tid, tid + kCNThreads of the row exactly as combine_kernel does and
// parks it in shared memory; the first 256 threads then reduce the squares in
// rms_norm_kernel's order (thread i: float4s i, i + 256, ...; warp tree; the
// eight warp sums in order) and every thread scales its float4s, so out and
// out_normed are bitwise those of the two separate kernels.  Rows up to
// kCNMaxD4 float4 (8192 elements).
constexpr int kCNThreads = 1024, kCNPer = 2, kCNMaxD4 = kCNThreads * kCNPer, kCNMaxRows = 64;

template <typename Y>
__global__ void __launch_bounds__(kCNThreads)
combine_norm_kernel(const Y *__restrict__ y_pair, const float4 *__restrict__ y_shared,
                    const float *__restrict__ w, const int32_t *__restrict__ perm, const float4 *res, int T, int k,
                    int d4, float4 *out, float4 *out_normed, float eps, int32_t *err)
{
    __shared__ float4 row[kCNMaxD4];
    __shared__ float part[8];
    __shared__ float rscale;
    griddep_launch_dependents();
    griddep_wait();   // y_pair / y_shared come from the previous kernel
    const int t = blockIdx.x;
    float4 acc[kCNPer];
#pragma unroll
    for (int j = 0; j < kCNPer; j++) {
        const int c = threadIdx.x + j * kCNThreads;
        const size_t id = (size_t)t * d4 + c;
        acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < d4) {
            acc[j] = res ? res[id] : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 ys = y_shared[id];
            acc[j].x += ys.x; acc[j].y += ys.y; acc[j].z += ys.z; acc[j].w += ys.w;
        }
    }
    constexpr int kG = 8;
    for (int j0 = 0; j0 < k; j0 += kG) {
        int q[kG];
        float wj[kG];
#pragma unroll
        for (int u = 0; u < kG; u++) {
            const int jj = j0 + u;
            q[u] = jj < k ? perm[(size_t)t * k + jj] : -1;
            if (!MOE_IN_BOUNDS(q[u] < T * k, err))
                q[u] = -1;
            wj[u] = jj < k ? w[(size_t)t * k + jj] : 0.f;
        }
        float4 y[kCNPer][kG];
#pragma unroll
        for (int j = 0; j < kCNPer; j++) {
            const int c = threadIdx.x + j * kCNThreads;
#pragma unroll
            for (int u = 0; u < kG; u++)
                y[j][u] = (q[u] >= 0 && c < d4) ? load4(y_pair, (size_t)q[u] * d4 + c)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kCNPer; j++)
#pragma unroll
            for (int u = 0; u < kG; u++)
                if (q[u] >= 0) {
                    acc[j].x = fmaf(wj[u], y[j][u].x, acc[j].x);
                    acc[j].y = fmaf(wj[u], y[j][u].y, acc[j].y);
                    acc[j].z = fmaf(wj[u], y[j][u].z, acc[j].z);
                    acc[j].w = fmaf(wj[u], y[j][u].w, acc[j].w);
                }
    }
#pragma unroll
    for (int j = 0; j < kCNPer; j++) {
        const int c = threadIdx.x + j * kCNThreads;
        if (c < d4) {
            out[(size_t)t * d4 + c] = acc[j];
            row[c] = acc[j];
        }
    }
    __syncthreads();
    if (threadIdx.x < 256) {
        float ss = 0.f;
        for (int c = threadIdx.x; c < d4; c += 256) {
            const float4 v = row[c];
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if ((threadIdx.x & 31) == 0)
            part[threadIdx.x >> 5] = ss;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < 8; w8++)
            tot += part[w8];
        rscale = 1.0f / sqrtf(tot / (float)(4 * d4) + eps);
    }
    __syncthreads();
    const float r = rscale;
#pragma unroll
    for (int j = 0; j < kCNPer; j++) {
        const int c = threadIdx.x + j * kCNThreads;
        if (c < d4) {
            float4 v = acc[j];
            v.x *= r;
            v.y *= r;
            v.z *= r;
            v.w *= r;
            out_normed[(size_t)t * d4 + c] = v;
        }
    }
}

// RMS normalisation of one row per CTA: fp32 sum of squares (per-thread, then
// warp and CTA tree), one IEEE square root and division, then x * r.  Each
// thread reads only its own elements before and after the reduction, so out
// may alias x.
__global__ void __launch_bounds__(256)
rms_norm_kernel(const float4 *x, int d4, float eps, float4 *out)
{
    __shared__ float part[8];
    griddep_launch_dependents();
    griddep_wait();   // x comes from the previous kernel
    const float4 *xr = x + (size_t)blockIdx.x * d4;
    float ss = 0.f;
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
        const float4 v = xr[c];
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0)
        part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; w++)
        tot += part[w];
    const float r = 1.0f / sqrtf(tot / (float)(4 * d4) + eps);
    float4 *orow = out + (size_t)blockIdx.x * d4;
    for (int c = threadIdx.x; c < d4; c += blockDim.x) {
        float4 v = xr[c];
        v.x *= r;
        v.y *= r;
        v.z *= r;
        v.w *= r;
        orow[c] = v;
    }
}

// n4 float4 from memory the GPU reaches over the host link (page-locked host rows, mapped) into device
// memory, one per thread.  The source does not depend on earlier work in the stream and is read before
// the grid wait, fetched again rather than from a line an earlier call left in this SM's L1 (ld.cv);
// the destination may still be read by the previous kernel, so the stores wait for it.
__global__ void __launch_bounds__(256)
copy_rows_kernel(const float4 *src, float4 *__restrict__ dst, long long n4)
{
    griddep_launch_dependents();
    const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < n4)
        v = __ldcv(src + i);
    griddep_wait();
    if (i < n4)
        dst[i] = v;
}

}  // namespace

int launch_copy_rows(const float *src, float *dst, long long n, cudaStream_t s)
{
    const long long n4 = n / 4;
    if (n4 <= 0)
        return MOE_OK;
    return launch_pdl(copy_rows_kernel, (int)((n4 + 255) / 256), 256, 0, s, reinterpret_cast<const float4 *>(src),
                      reinterpret_cast<float4 *>(dst), n4);
}

int launch_combine_norm(const float *y_pair, const uint16_t *y_pair16, const float *y_shared, const float *w,
                        const int32_t *perm, const float *res, int T, int k, int d, float *out, float *out_normed,
                        float eps, cudaStream_t s, int32_t *err)
{
    const int d4 = d / 4;
    // one CTA per row pays off while rows are few; with many rows the two kernels' wider grids
    // are faster (measured on an 8-layer d = 6144 stack: T <= 64 gained, T = 256 lost), as
    // they are for rows wider than the shared-memory copy holds
    if (d4 > kCNMaxD4 || T > kCNMaxRows) {
        const int rc = y_pair16 ? launch_combine_bf16(y_pair16, y_shared, w, perm, res, T, k, d, out, s, err)
                                : launch_combine(y_pair, y_shared, w, perm, res, T, k, d, out, s, err);
        return rc != MOE_OK ? rc : launch_rms_norm(out, T, d, eps, out_normed, s);
    }
    if (y_pair16)
        return launch_pdl(combine_norm_kernel<uint2>, T, kCNThreads, 0, s, reinterpret_cast<const uint2 *>(y_pair16),
                          reinterpret_cast<const float4 *>(y_shared), w, perm, reinterpret_cast<const float4 *>(res),
                          T, k, d4, reinterpret_cast<float4 *>(out), reinterpret_cast<float4 *>(out_normed), eps, err);
    return launch_pdl(combine_norm_kernel<float4>, T, kCNThreads, 0, s, reinterpret_cast<const float4 *>(y_pair),
                      reinterpret_cast<const float4 *>(y_shared), w, perm, reinterpret_cast<const float4 *>(res), T,
                      k, d4, reinterpret_cast<float4 *>(out), reinterpret_cast<float4 *>(out_normed), eps, err);
}

int launch_rms_norm(const float *x, int T, int d, float eps, float *out, cudaStream_t s)
{
    return launch_pdl(rms_norm_kernel, T, 256, 0, s, reinterpret_cast<const float4 *>(x), d / 4, eps,
                      reinterpret_cast<float4 *>(out));
}

int launch_combine(const float *y_pair, const float *y_shared, const float *w, const int32_t *perm,
                   const float *res, int T, int k, int d, float *out, cudaStream_t s, int32_t *err)
{
    const int d4 = d / 4;
    const long long n = (long long)T * d4;
    return launch_pdl(combine_kernel<float4>, (int)((n + 255) / 256), 256, 0, s,
                      reinterpret_cast<const float4 *>(y_pair), reinterpret_cast<const float4 *>(y_shared), w,
                      perm, reinterpret_cast<const float4 *>(res), T, k, d4, reinterpret_cast<float4 *>(out), err);
}

int launch_combine_bf16(const uint16_t *y_pair, const float *y_shared, const float *w, const int32_t *perm,
                        const float *res, int T, int k, int d, float *out, cudaStream_t s, int32_t *err)
{
    const int d4 = d / 4;
    const long long n = (long long)T * d4;
    return launch_pdl(combine_kernel<uint2>, (int)((n + 255) / 256), 256, 0, s,
                      reinterpret_cast<const uint2 *>(y_pair), reinterpret_cast<const float4 *>(y_shared), w,
                      perm, reinterpret_cast<const float4 *>(res), T, k, d4, reinterpret_cast<float4 *>(out), err);
}

}  // namespace moe
