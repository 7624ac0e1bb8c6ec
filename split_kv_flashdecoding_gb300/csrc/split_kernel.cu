// split_kernel.cu -- stage 1 of split-KV decode attention on sm_103a.
//
// "FlashDecoding++: sequence-dimension KV split parallelism for LLM serving"
// (techknowgenie.com), §2 (each block keeps the query on chip and copies only
// its own chunk of K/V from HBM into shared memory) and §3 stage 1 (per chunk:
// logits, local max, exp, local sum, probability-weighted V; the block stores
// the partial and exits).
//
// One CTA = one (split, KV head).  All G query heads that share the KV head
// are served from the same shared-memory tiles, so every K/V byte is read
// from HBM once per step.
//
// Warp roles:
//   warp NC (producer): one lane issues 2-D TMA loads of 32-key tiles of K and
//     V (each tile = two 64-column boxes per tensor, 128-byte swizzle) into an
//     NS-stage ring guarded by full/empty mbarriers.
//   warps 0..NC-1 (consumers): warp w takes tiles w, w+NC, ...  NS is a
//     multiple of NC, so every stage always goes to the same warp and a warp
//     never waits on a barrier more than one phase ahead (parity waits can only
//     tell two phases apart).  Each warp keeps its own online-softmax state (running max m, partial sums l, accumulator) for
//     the G heads.  Scores: lane = key, q from shared memory (broadcast),
//     packed fp32x2 FMAs.  P.V: lane = 4 consecutive output columns, p values
//     broadcast from shared memory.  At the end the NC warp states are merged
//     in shared memory (the same rescaling as stage 2) and the normalised
//     partial (O_i, LSE_i) is written.
// Logits are kept in base 2 (q pre-multiplied by scale * log2 e); the stored
// LSE is converted back to the natural log.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace fd {
namespace {

constexpr int kHalfBytes = kTile * 128;        // 32 keys x 64 bf16 (one swizzled box)
constexpr int kStageBytes = 4 * kHalfBytes;    // K lo, K hi, V lo, V hi

enum Misc { kB, kPrefix, kSplits, kS, kT0, kT1, kOk, kAbort, kIssued, kMiscCount };

template <int G, int NC, int NS>
struct Layout {
    static_assert(NS % NC == 0, "each stage must belong to one consumer warp");
    static constexpr int kOffQ = NS * kStageBytes;
    static constexpr int kOffP = kOffQ + G * kHeadDim * 4;
    static constexpr int kOffBar = kOffP + NC * kTile * G * 8;
    static constexpr int kOffMisc = kOffBar + 2 * NS * 8;
    static constexpr int kBytes = kOffMisc + kMiscCount * 4;
    static constexpr int kAlloc = kBytes + 1024;   // room to align the base to 1024 B
    // End-of-kernel merge of the consumer warps, placed over the stage ring.
    static constexpr int kOffCombM = NC * G * kHeadDim * 4;
    static constexpr int kOffCombL = kOffCombM + NC * G * 4;
    static_assert(kOffCombL + NC * G * 4 <= NS * kStageBytes, "combine area must fit the ring");
};

// One key row of P.V for all G heads: acc[g] += p[g] * v (4 columns per lane).
template <int G>
__device__ __forceinline__ void pv_step(const uint8_t *v_half, int cc, int sub, int r,
                                        const float2 *__restrict__ p_row, float2 (&acc)[G][2])
{
    const uint2 vw =
        *reinterpret_cast<const uint2 *>(v_half + r * 128 + ((cc ^ (r & 7)) << 4) + sub);
    const float2 v0 = bf16x2_to_float2(vw.x);
    const float2 v1 = bf16x2_to_float2(vw.y);
    if constexpr (G == 1) {
        const float2 pp = p_row[0];
        acc[0][0] = __ffma2_rn(v0, pp, acc[0][0]);
        acc[0][1] = __ffma2_rn(v1, pp, acc[0][1]);
    } else {
#pragma unroll
        for (int g = 0; g < G; g += 2) {
            const float4 pq = *reinterpret_cast<const float4 *>(p_row + g);
            const float2 p0 = make_float2(pq.x, pq.y), p1 = make_float2(pq.z, pq.w);
            acc[g][0] = __ffma2_rn(v0, p0, acc[g][0]);
            acc[g][1] = __ffma2_rn(v1, p0, acc[g][1]);
            acc[g + 1][0] = __ffma2_rn(v0, p1, acc[g + 1][0]);
            acc[g + 1][1] = __ffma2_rn(v1, p1, acc[g + 1][1]);
        }
    }
}

template <int G, int NC, int NS, int MIN_CTAS>
__global__ void __launch_bounds__((NC + 1) * 32, MIN_CTAS)
    split_kv_kernel(const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const SplitParams p)
{
    using L = Layout<G, NC, NS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float *q_s = reinterpret_cast<float *>(smem + L::kOffQ);
    float2 *p_s = reinterpret_cast<float2 *>(smem + L::kOffP);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    volatile int *misc = reinterpret_cast<volatile int *>(smem + L::kOffMisc);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = blockIdx.x % p.num_kv_heads;
    const int32_t j = blockIdx.x / p.num_kv_heads;

    // ---- locate this CTA's split (same rule as the host planner)
    if (warp == 0) {
        SplitCoord c{};
        bool ok = derive_split(p.kv_indptr, p.batch, p.chunk, j, false, c);
        if (lane == 0) {
            int32_t t0 = 0, t1 = 0;
            if (ok) {
                const int32_t len = split_len_for(c.end - c.beg, c.splits);
                t0 = c.beg + c.s * len;
                t1 = min(t0 + len, c.end);
                ok = t0 < t1 && t1 <= p.total_tokens &&
                     partial_row(c.prefix, p.num_qo_heads, p.num_qo_heads - 1, c.splits,
                                 c.splits - 1) < p.num_partial_rows;
            }
            misc[kB] = c.b;
            misc[kPrefix] = c.prefix;
            misc[kSplits] = c.splits;
            misc[kS] = c.s;
            misc[kT0] = t0;
            misc[kT1] = t1;
            misc[kOk] = ok;
            misc[kAbort] = 0;
            misc[kIssued] = 0;
            if (!ok)
                report(p.status, FD_ERR_DEVICE_BOUNDS);
        }
    }
    if (warp == NC && lane == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_addr(&bars[s]), 1);        // full: producer arrive + TMA bytes
            mbar_init(smem_addr(&bars[NS + s]), 1);   // empty: consumer warp releases
        }
        fence_mbar_init();
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
    }
    __syncthreads();
    if (!misc[kOk])
        return;
    const int32_t t0 = misc[kT0], t1 = misc[kT1];
    const int n_tiles = (t1 - t0 + kTile - 1) / kTile;
    const int b = misc[kB];

    // ---- q of the G heads -> shared memory, fp32, times scale*log2(e)
    if (warp < NC) {
        for (int i = tid; i < G * 16; i += NC * 32) {
            const int g = i >> 4, c = i & 15;
            const uint4 w = *reinterpret_cast<const uint4 *>(
                p.q + ((int64_t)b * p.num_qo_heads + kvh * G + g) * kHeadDim + c * 8);
            float *dst = q_s + g * kHeadDim + c * 8;
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = bf16x2_to_float2(ws[e]);
                dst[2 * e] = f.x * p.q_scale;
                dst[2 * e + 1] = f.y * p.q_scale;
            }
        }
    }
    __syncthreads();

    float m_run[G], l_part[G];
    float2 acc[G][2];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
        l_part[g] = 0.f;
        acc[g][0] = acc[g][1] = make_float2(0.f, 0.f);
    }

    if (warp == NC) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            const int32_t x = kvh * kHeadDim;
            int issued = 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % NS;
                if (i >= NS &&
                    !mbar_wait(smem_addr(&bars[NS + s]), ((i / NS) - 1) & 1, p.timeout_ns)) {
                    misc[kAbort] = 1;
                    report(p.status, FD_ERR_TIMEOUT);
                    break;
                }
                if (misc[kAbort])
                    break;
                const uint32_t full = smem_addr(&bars[s]);
                const uint32_t dst = smem_addr(smem + s * kStageBytes);
                const int32_t y = t0 + i * kTile;
                mbar_arrive_expect_tx(full, kStageBytes);
                tma_load_2d(dst, &tm_k, x, y, full, pol);
                tma_load_2d(dst + kHalfBytes, &tm_k, x + 64, y, full, pol);
                tma_load_2d(dst + 2 * kHalfBytes, &tm_v, x, y, full, pol);
                tma_load_2d(dst + 3 * kHalfBytes, &tm_v, x + 64, y, full, pol);
                issued = i + 1;
            }
            misc[kIssued] = issued;
        }
    } else {
        // ---------------------------------------------------------- consumers
        float2 *p_w = p_s + warp * kTile * G;       // [key][g] pairs (p, p)
        const int sw = lane & 7;
        const int cc = (lane & 15) >> 1, sub = (lane & 1) * 8;
        for (int i = warp; i < n_tiles; i += NC) {
            const int s = i % NS;
            if (!mbar_wait(smem_addr(&bars[s]), (i / NS) & 1, p.timeout_ns)) {
                misc[kAbort] = 1;
                report(p.status, FD_ERR_TIMEOUT);
                break;
            }
            const uint8_t *st = smem + s * kStageBytes;
            const int n_valid = min(kTile, t1 - (t0 + i * kTile));

            // scores: lane = key (row `lane` of the tile)
            float sc[G];
            {
                const uint8_t *k_lo = st + lane * 128;
                const uint8_t *k_hi = st + kHalfBytes + lane * 128;
                float2 a0[G], a1[G];
#pragma unroll
                for (int g = 0; g < G; ++g)
                    a0[g] = a1[g] = make_float2(0.f, 0.f);
#pragma unroll 4
                for (int c = 0; c < 16; ++c) {
                    const uint8_t *kr = c < 8 ? k_lo : k_hi;
                    const uint4 kw = *reinterpret_cast<const uint4 *>(kr + (((c & 7) ^ sw) << 4));
                    const float2 k0 = bf16x2_to_float2(kw.x), k1 = bf16x2_to_float2(kw.y);
                    const float2 k2 = bf16x2_to_float2(kw.z), k3 = bf16x2_to_float2(kw.w);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float4 qa = *reinterpret_cast<const float4 *>(q_s + g * kHeadDim + c * 8);
                        const float4 qb =
                            *reinterpret_cast<const float4 *>(q_s + g * kHeadDim + c * 8 + 4);
                        a0[g] = __ffma2_rn(k0, make_float2(qa.x, qa.y), a0[g]);
                        a1[g] = __ffma2_rn(k1, make_float2(qa.z, qa.w), a1[g]);
                        a0[g] = __ffma2_rn(k2, make_float2(qb.x, qb.y), a0[g]);
                        a1[g] = __ffma2_rn(k3, make_float2(qb.z, qb.w), a1[g]);
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g)
                    sc[g] = lane < n_valid ? (a0[g].x + a0[g].y) + (a1[g].x + a1[g].y) : -INFINITY;
            }

            // online softmax over this tile (running max is warp-uniform)
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float mn = fmaxf(m_run[g], warp_max(sc[g]));
                const float alpha = exp2f(m_run[g] - mn);
                const float pv = exp2f(sc[g] - mn);
                l_part[g] = fmaf(l_part[g], alpha, pv);
                const float2 a2 = make_float2(alpha, alpha);
                acc[g][0] = __fmul2_rn(acc[g][0], a2);
                acc[g][1] = __fmul2_rn(acc[g][1], a2);
                m_run[g] = mn;
                p_w[lane * G + g] = make_float2(pv, pv);
            }
            __syncwarp();

            // P.V: lane = output columns 4*lane .. 4*lane+3
            const uint8_t *v_half = st + 2 * kHalfBytes + (lane >> 4) * kHalfBytes;
            if (n_valid == kTile) {
#pragma unroll 8
                for (int r = 0; r < kTile; ++r)
                    pv_step<G>(v_half, cc, sub, r, p_w + r * G, acc);
            } else {
                for (int r = 0; r < n_valid; ++r)
                    pv_step<G>(v_half, cc, sub, r, p_w + r * G, acc);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&bars[NS + s]));
        }
    }

    __syncthreads();
    if (misc[kAbort]) {
        // Let every copy this CTA issued land before the CTA exits.
        if (warp == NC && lane == 0) {
            const int issued = misc[kIssued];
            for (int i = max(0, issued - NS); i < issued; ++i)
                if (!mbar_wait(smem_addr(&bars[i % NS]), (i / NS) & 1, kDrainTimeoutNs))
                    report(p.status, FD_ERR_TIMEOUT);
        }
        __syncthreads();
        return;
    }

    // ---- merge the consumer warps' states (the ring is free now)
    float *comb_acc = reinterpret_cast<float *>(smem);
    float *comb_m = reinterpret_cast<float *>(smem + L::kOffCombM);
    float *comb_l = reinterpret_cast<float *>(smem + L::kOffCombL);
    if (warp < NC) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float l_tot = warp_sum(l_part[g]);
            *reinterpret_cast<float4 *>(comb_acc + (warp * G + g) * kHeadDim + 4 * lane) =
                make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
            if (lane == 0) {
                comb_m[warp * G + g] = m_run[g];
                comb_l[warp * G + g] = l_tot;
            }
        }
    }
    __syncthreads();

    const int prefix = misc[kPrefix], splits = misc[kSplits], split = misc[kS];
    for (int idx = tid; idx < G * 32; idx += (NC + 1) * 32) {
        const int g = idx >> 5, c4 = idx & 31;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < NC; ++w)
            mx = fmaxf(mx, comb_m[w * G + g]);
        float den = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < NC; ++w) {
            const float e = exp2f(comb_m[w * G + g] - mx);
            den = fmaf(e, comb_l[w * G + g], den);
            const float4 a = *reinterpret_cast<const float4 *>(comb_acc + (w * G + g) * kHeadDim + 4 * c4);
            o.x = fmaf(e, a.x, o.x);
            o.y = fmaf(e, a.y, o.y);
            o.z = fmaf(e, a.z, o.z);
            o.w = fmaf(e, a.w, o.w);
        }
        const float inv = 1.f / den;
        o.x *= inv;
        o.y *= inv;
        o.z *= inv;
        o.w *= inv;
        const int64_t row = partial_row(prefix, p.num_qo_heads, kvh * G + g, splits, split);
        *reinterpret_cast<float4 *>(p.partial_o + row * kHeadDim + 4 * c4) = o;
        if (c4 == 0)
            p.partial_lse[row] = (mx + log2f(den)) * kLn2;
    }
}

// Launch shape per group size: consumer warps, stages, resident CTAs per SM.
template <int G> struct Shape { static constexpr int NC = 6, NS = 6, MIN_CTAS = 2; };
template <> struct Shape<8> { static constexpr int NC = 4, NS = 4, MIN_CTAS = 2; };

template <int G>
cudaError_t launch_g(const CUtensorMap &tk, const CUtensorMap &tv, const SplitParams &p,
                     int num_work, cudaStream_t stream)
{
    constexpr int NC = Shape<G>::NC, NS = Shape<G>::NS;
    using L = Layout<G, NC, NS>;
    static_assert(2 * (L::kAlloc + 1024) <= 233472 || Shape<G>::MIN_CTAS == 1,
                  "two CTAs per SM must fit in shared memory");
    auto kern = split_kv_kernel<G, NC, NS, Shape<G>::MIN_CTAS>;
    // The shared-memory opt-in is per device; remember it for the first 64.
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            configured[dev] = true;
    }
    kern<<<num_work, (NC + 1) * 32, L::kAlloc, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_split(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const SplitParams &p,
                         int group, int num_work, cudaStream_t stream)
{
    switch (group) {
    case 1: return launch_g<1>(tm_k, tm_v, p, num_work, stream);
    case 2: return launch_g<2>(tm_k, tm_v, p, num_work, stream);
    case 4: return launch_g<4>(tm_k, tm_v, p, num_work, stream);
    case 8: return launch_g<8>(tm_k, tm_v, p, num_work, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fd
