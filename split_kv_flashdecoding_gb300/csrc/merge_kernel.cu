// merge_kernel.cu -- stage 2 of split-KV decode attention on sm_103a.
//
// "FlashDecoding++: sequence-dimension KV split parallelism for LLM serving"
// (techknowgenie.com), §3 stage 2 ("global reduction"): one block per head
// reads all of the head's chunk statistics, takes the global maximum, rescales
// each chunk by exp(local - global), sums the rescaled denominators and
// outputs, and divides.  With the partials stored as (O_i, LSE_i) the local
// statistic is LSE_i and each chunk's rescaled denominator is its weight
// w_i = exp(LSE_i - M); the output LSE is M + ln sum_i w_i.
//
// One CTA (4 warps) per (request, query head).  Warp w accumulates splits
// w, w+4, ... with a running maximum (8 rows of loads in flight), lane = 4
// output columns (one float4 of a 512-byte partial row); the four warp states
// are combined with the same rescaling.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace fd {
namespace {

constexpr int kMergeWarps = 4;
constexpr int kBatch = 8;   // partial rows a warp loads at once

__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeParams p)
{
    __shared__ int32_t s_info[3];   // prefix, splits, ok
    __shared__ float s_m[kMergeWarps];
    __shared__ float s_den[kMergeWarps];
    __shared__ float4 s_acc[kMergeWarps][32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / p.num_qo_heads;
    const int hq = blockIdx.x % p.num_qo_heads;

    if (warp == 0) {
        SplitCoord c{};
        const KeyIndex ki{p.kv_indptr, p.kv_last_len, p.page_size};
        const bool found = derive_split(ki, p.batch, p.chunk, b, true, c);
        if (lane == 0) {
            const bool ok = found && (c.splits == 0 ||
                                      partial_row(c.prefix, p.num_qo_heads, p.num_qo_heads - 1,
                                                  c.splits, c.splits - 1) < p.num_partial_rows);
            s_info[0] = c.prefix;
            s_info[1] = c.splits;
            s_info[2] = ok;
            if (!ok)
                report(p.status, FD_ERR_DEVICE_BOUNDS);
        }
    }
    // Partials are written by the preceding split grid: wait for it here.
    griddep_wait();
    __syncthreads();
    if (!s_info[2])
        return;
    const int n = s_info[1];
    float *o_row = p.o + (int64_t)blockIdx.x * kHeadDim;
    if (p.only_empty && n > 0)
        return;
    if (n == 0) {   // a request with no keys
        if (warp == 0) {
            reinterpret_cast<float4 *>(o_row)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (lane == 0)
                p.lse[blockIdx.x] = -INFINITY;
        }
        return;
    }
    const int64_t base = partial_row(s_info[0], p.num_qo_heads, hq, n, 0);
    const float *lse_in = p.partial_lse + base;
    const float4 *o_in = reinterpret_cast<const float4 *>(p.partial_o + base * kHeadDim) + lane;

    // Warp w reduces rows w, w + 4, ... with a running maximum, kBatch rows of
    // loads in flight at a time.
    float m = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = warp; i0 < n; i0 += kMergeWarps * kBatch) {
        float l[kBatch];
        float4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + u * kMergeWarps;
            if (i < n) {
                l[u] = __ldg(lse_in + i);
                v[u] = __ldg(o_in + (int64_t)i * (kHeadDim / 4));
            } else {
                l[u] = -INFINITY;
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float bm = l[0];
#pragma unroll
        for (int u = 1; u < kBatch; ++u)
            bm = fmaxf(bm, l[u]);
        const float m_new = fmaxf(m, bm);   // finite: row i0 exists
        const float f = expf(m - m_new);
        den *= f;
        acc.x *= f;
        acc.y *= f;
        acc.z *= f;
        acc.w *= f;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const float w = expf(l[u] - m_new);
            den += w;
            acc.x = fmaf(w, v[u].x, acc.x);
            acc.y = fmaf(w, v[u].y, acc.y);
            acc.z = fmaf(w, v[u].z, acc.z);
            acc.w = fmaf(w, v[u].w, acc.w);
        }
        m = m_new;
    }
    s_acc[warp][lane] = acc;
    if (lane == 0) {
        s_m[warp] = m;
        s_den[warp] = den;
    }
    __syncthreads();
    if (warp == 0) {
        float mx = s_m[0];
#pragma unroll
        for (int w = 1; w < kMergeWarps; ++w)
            mx = fmaxf(mx, s_m[w]);
        float d = 0.f;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) {
            const float f = expf(s_m[w] - mx);   // 0 for a warp that had no rows
            d = fmaf(f, s_den[w], d);
            const float4 t = s_acc[w][lane];
            a.x = fmaf(f, t.x, a.x);
            a.y = fmaf(f, t.y, a.y);
            a.z = fmaf(f, t.z, a.z);
            a.w = fmaf(f, t.w, a.w);
        }
        const float inv = 1.f / d;
        reinterpret_cast<float4 *>(o_row)[lane] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
        if (lane == 0)
            p.lse[blockIdx.x] = mx + logf(d);
    }
}

}  // namespace

namespace {

// Merge of R attention states per row (the sequence-sharded exchange): for
// row r, M = max_s LSE_s, w_s = exp(LSE_s - M), O = sum_s w_s O_s / sum_s w_s,
// LSE = M + ln sum_s w_s; a row whose states are all empty (LSE = -inf) gets
// O = 0, LSE = -inf.  One warp per row, lane = 4 columns (one float4).
constexpr int kStatesWarps = 4;

__global__ void __launch_bounds__(kStatesWarps * 32)
    merge_states_kernel(int num_states, int rows, const float *__restrict__ o_states,
                        const float *__restrict__ lse_states, float *__restrict__ o,
                        float *__restrict__ lse)
{
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kStatesWarps + (threadIdx.x >> 5);
    if (row < rows) {
        float m = -INFINITY;
        for (int s = 0; s < num_states; ++s)
            m = fmaxf(m, __ldg(lse_states + (int64_t)s * rows + row));
        float den = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m != -INFINITY) {
            for (int s = 0; s < num_states; ++s) {
                const int64_t r = (int64_t)s * rows + row;
                const float w = expf(__ldg(lse_states + r) - m);
                const float4 v = __ldg(reinterpret_cast<const float4 *>(o_states + r * kHeadDim) + lane);
                den += w;
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        reinterpret_cast<float4 *>(o + (int64_t)row * kHeadDim)[lane] =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (lane == 0)
            lse[row] = den > 0.f ? m + logf(den) : -INFINITY;
    }
    griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_merge_states(int num_states, int rows, const float *o_states,
                                const float *lse_states, float *o, float *lse, cudaStream_t stream)
{
    if (rows == 0)
        return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + kStatesWarps - 1) / kStatesWarps));
    cfg.blockDim = dim3(kStatesWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_states_kernel, num_states, rows, o_states, lse_states, o, lse);
}

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream)
{
    const int64_t ctas = (int64_t)p.batch * p.num_qo_heads;
    if (ctas == 0)
        return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_kernel, p);
}

}  // namespace fd
