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
// w, w+4, ...; lane = 4 output columns (one float4 of a 512-byte partial row).
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace fd {
namespace {

constexpr int kMergeWarps = 4;

__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeParams p)
{
    __shared__ int32_t s_info[3];   // prefix, splits, ok
    __shared__ float s_max[kMergeWarps];
    __shared__ float s_den[kMergeWarps];
    __shared__ float4 s_acc[kMergeWarps][32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / p.num_qo_heads;
    const int hq = blockIdx.x % p.num_qo_heads;

    if (warp == 0) {
        SplitCoord c{};
        const bool found = derive_split(p.kv_indptr, p.batch, p.chunk, b, true, c);
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
    __syncthreads();
    if (!s_info[2])
        return;
    const int n = s_info[1];
    float *o_row = p.o + (int64_t)blockIdx.x * kHeadDim;
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

    // global max of the chunk statistics
    float mx = -INFINITY;
    for (int i = tid; i < n; i += kMergeWarps * 32)
        mx = fmaxf(mx, lse_in[i]);
    mx = warp_max(mx);
    if (lane == 0)
        s_max[warp] = mx;
    __syncthreads();
    mx = s_max[0];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w)
        mx = fmaxf(mx, s_max[w]);

    // rescaled sums
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = warp; i < n; i += kMergeWarps) {
        const float w = expf(lse_in[i] - mx);
        const float4 v = reinterpret_cast<const float4 *>(p.partial_o + (base + i) * kHeadDim)[lane];
        den += w;
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    s_acc[warp][lane] = acc;
    if (lane == 0)
        s_den[warp] = den;
    __syncthreads();
    if (warp == 0) {
        float d = 0.f;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) {
            d += s_den[w];
            const float4 t = s_acc[w][lane];
            a.x += t.x;
            a.y += t.y;
            a.z += t.z;
            a.w += t.w;
        }
        const float inv = 1.f / d;
        reinterpret_cast<float4 *>(o_row)[lane] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
        if (lane == 0)
            p.lse[blockIdx.x] = mx + logf(d);
    }
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream)
{
    const int64_t ctas = (int64_t)p.batch * p.num_qo_heads;
    if (ctas == 0)
        return cudaSuccess;
    merge_kernel<<<(unsigned)ctas, kMergeWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace fd
