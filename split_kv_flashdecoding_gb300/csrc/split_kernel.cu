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
//   warp NC (producer): one lane issues TMA loads of 32-key tiles of K and V
//     into an NS-stage ring guarded by full/empty mbarriers.  A tile is one
//     3-D box per tensor holding both 64-column halves of the head's 32 rows
//     (128-byte swizzle), or, for a paged cache whose pages are not a
//     multiple of 32 keys, two such boxes of 16 rows.
//   warps 0..NC-1 (consumers): warp w takes tiles w, w+NC, ...  NS is a
//     multiple of NC, so every stage always goes to the same warp and a warp
//     never waits on a barrier more than one phase ahead (parity waits can only
//     tell two phases apart).  Each warp keeps its own online-softmax state and
//     at the end the NC states are merged in shared memory with the same
//     rescaling as stage 2.
//
// Arithmetic per tile (warp-level mma.sync m16n8k16, bf16 in, fp32 accumulate):
//   S = Q K^T    A = the G query rows (rows >= G are zero), kept in registers;
//                B = K rows read with ldmatrix straight from the swizzled tile.
//   online softmax on the fp32 accumulator fragments (base-2 logits: S is
//                scaled by scale * log2 e; the running max and sum are per row).
//   O += P V     A = P split into bf16 hi + lo parts: rows 0-7 carry hi, rows
//                8-15 (padding in the score product) carry lo = P - hi, so the
//                weights keep ~16 mantissa bits; O rows g and g+8 are added at
//                the end.  B = V rows read with ldmatrix.trans.
// The tensor cores are used here because the CUDA-core version of the same
// loop was limited by shared-memory wavefronts (broadcast reads of q and p)
// and instruction issue, not by HBM; the contraction itself stays tiny
// (m = G <= 8 rows).
#include <cuda/atomic>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace fd {
namespace {

constexpr int kHalfBytes = kTile * 128;        // 32 keys x 64 bf16
constexpr int kStageBytes = 4 * kHalfBytes;    // K lo, K hi, V lo, V hi

// How K/V rows are found and how a stage is laid out.  A stage holds K then
// V (kStageBytes / 2 each); key row r (0..31), column half h (64 columns of
// 128 bytes, 16-byte chunks XOR-swizzled by r % 8) of a tensor sits at
//   h * HalfStride + (r / 16) * BlockStride + (r % 16) * 128.
//   kKvRagged, kKvPaged:  [half][32 rows]            HalfStride 4096, BlockStride 2048
//   kKvPaged16:           [16-row block][half][16]   HalfStride 2048, BlockStride 4096
// (kKvPaged16 is what one 16-row box of both halves per page lands as.)
enum KvLayout { kKvRagged = 0, kKvPaged = 1, kKvPaged16 = 2 };

template <int KV>
struct StageLayout {
    static constexpr int kHalfStride = KV == kKvPaged16 ? 2048 : kHalfBytes;
    static constexpr int kBlockStride = KV == kKvPaged16 ? 4096 : 2048;
    static constexpr int kBoxRows = KV == kKvPaged16 ? 16 : kTile;
};
constexpr int kMaxGroup = 8;                   // rows 8-15 of the MMA carry the lo part of P

enum Misc { kB, kPrefix, kSplits, kS, kT0, kT1, kOk, kAbort, kIssued, kLast, kMiscCount };

template <int G, int NC, int NS>
struct Layout {
    static_assert(NS % NC == 0, "each stage must belong to one consumer warp");
    static_assert(G >= 1 && G <= kMaxGroup, "group size");
    static constexpr int kOffBar = NS * kStageBytes;
    static constexpr int kOffMisc = kOffBar + 2 * NS * 8;
    static constexpr int kBytes = kOffMisc + kMiscCount * 4;
    static constexpr int kAlloc = kBytes + 1024;   // room to align the base to 1024 B
    // End-of-kernel merge of the consumer warps, placed over the stage ring.
    static constexpr int kOffCombM = NC * G * kHeadDim * 4;
    static constexpr int kOffCombL = kOffCombM + NC * G * 4;
    static_assert(kOffCombL + NC * G * 4 <= NS * kStageBytes, "combine area must fit the ring");
    // The fused stage-2 merge of the last CTA also works over the drained ring.
    static_assert((NC + 1) * G * (kHeadDim + 2) * 4 <= NS * kStageBytes, "merge area must fit the ring");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D (+)= A B for one m16n8k16 tile, bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> packed bf16x2 (first argument in the low half), round to nearest.
__device__ __forceinline__ uint32_t pack_bf16(float lo_elem, float hi_elem)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo_elem, hi_elem);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float bf16_round(float x)
{
    return __bfloat162float(__float2bfloat16_rn(x));
}

// Stage 2 for one (request, KV head) group, run by the CTA that finished the
// group last: for each of its G heads, M = max_i LSE_i, w_i = exp(LSE_i - M),
// O = sum_i w_i O_i / sum_i w_i, LSE = M + ln sum_i w_i over the group's splits.
// Warp w of the NW warps takes splits w, w + NW, ... (U splits of loads in
// flight per batch, lane = 4 output columns, all G heads), keeps a running
// maximum per head, and the NW warp states are combined through shared memory
// (`scratch`, free once the stage ring has drained).  The other CTAs' partials
// are read through L2 (ld.global.cg).
template <int G, int NW>
__device__ __forceinline__ void merge_group(const SplitParams &p, int prefix, int splits, int b,
                                            int kvh, int warp, int lane, float *scratch)
{
    constexpr int U = (16 / G) > 1 ? 16 / G : 1;   // splits per batch: 16 float4 in flight
    float m[G], den[G];
    float4 acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        den[g] = 0.f;
        acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int64_t row0 = partial_row(prefix, p.num_qo_heads, kvh * G, splits, 0);
    for (int s0 = warp; s0 < splits; s0 += NW * U) {
        float l[U][G];
        float4 v[U][G];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + u * NW;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                // rows of head kvh*G + g are splits apart
                const int64_t row = row0 + (int64_t)g * splits + s;
                if (s < splits) {
                    l[u][g] = __ldcg(p.partial_lse + row);
                    v[u][g] = __ldcg(reinterpret_cast<const float4 *>(p.partial_o + row * kHeadDim) + lane);
                } else {
                    l[u][g] = -INFINITY;
                    v[u][g] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float bm = l[0][g];
#pragma unroll
            for (int u = 1; u < U; ++u)
                bm = fmaxf(bm, l[u][g]);
            const float m_new = fmaxf(m[g], bm);
            if (m_new == -INFINITY)   // only empty partials so far (none in practice)
                continue;
            const float f = expf(m[g] - m_new);
            den[g] *= f;
            acc[g].x *= f;
            acc[g].y *= f;
            acc[g].z *= f;
            acc[g].w *= f;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float w = expf(l[u][g] - m_new);
                den[g] += w;
                acc[g].x = fmaf(w, v[u][g].x, acc[g].x);
                acc[g].y = fmaf(w, v[u][g].y, acc[g].y);
                acc[g].z = fmaf(w, v[u][g].z, acc[g].z);
                acc[g].w = fmaf(w, v[u][g].w, acc[g].w);
            }
            m[g] = m_new;
        }
    }
    float *s_acc = scratch;                       // [NW][G][128]
    float *s_m = scratch + NW * G * kHeadDim;     // [NW][G]
    float *s_den = s_m + NW * G;                  // [NW][G]
#pragma unroll
    for (int g = 0; g < G; ++g) {
        reinterpret_cast<float4 *>(s_acc + (warp * G + g) * kHeadDim)[lane] = acc[g];
        if (lane == 0) {
            s_m[warp * G + g] = m[g];
            s_den[warp * G + g] = den[g];
        }
    }
    __syncthreads();
    for (int idx = warp * 32 + lane; idx < G * 32; idx += NW * 32) {
        const int g = idx >> 5, c4 = idx & 31;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w)
            mx = fmaxf(mx, s_m[w * G + g]);
        float d = 0.f;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float f = expf(s_m[w * G + g] - mx);   // 0 for a warp with no splits
            d = fmaf(f, s_den[w * G + g], d);
            const float4 t = reinterpret_cast<const float4 *>(s_acc + (w * G + g) * kHeadDim)[c4];
            a.x = fmaf(f, t.x, a.x);
            a.y = fmaf(f, t.y, a.y);
            a.z = fmaf(f, t.z, a.z);
            a.w = fmaf(f, t.w, a.w);
        }
        const float inv = 1.f / d;
        const int64_t row = (int64_t)b * p.num_qo_heads + kvh * G + g;
        reinterpret_cast<float4 *>(p.o + row * kHeadDim)[c4] =
            make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
        if (c4 == 0)
            p.lse[row] = mx + logf(d);
    }
}

template <int G, int NC, int NS, int MIN_CTAS, int KV>
__global__ void __launch_bounds__((NC + 1) * 32, MIN_CTAS)
    split_kv_kernel(const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ SplitParams p)
{
    using L = Layout<G, NC, NS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    volatile int *misc = reinterpret_cast<volatile int *>(smem + L::kOffMisc);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = blockIdx.x % p.num_kv_heads;
    const int32_t j = blockIdx.x / p.num_kv_heads;
    // The inputs may come from the preceding grid in the stream: wait for it
    // before touching global memory (the launch itself overlaps its tail).
    // When kv_indptr is in the launch parameters, the producer warp locates
    // its split before that wait.
    const bool early_derive = p.indptr_in_params && warp == NC;
    if (!early_derive)
        griddep_wait();

    // ---- the producer warp locates this CTA's split (same rule as the host
    // planner), sets up the barriers and puts the first NS tiles in flight
    // before the block synchronises, so the loads start as early as possible.
    // With the paged layout the whole warp runs the issue loop (it shares a
    // window of page ids); lane 0 issues the barrier operations and the
    // copies.  The ragged layout needs lane 0 alone.  Key positions t0, t1 are
    // relative to the request's first key.
    constexpr bool paged = KV != kKvRagged;
    using SL = StageLayout<KV>;
    uint64_t pol = 0;
    int issued = 0;
    int32_t t0 = 0, t1 = 0, req_base = 0, req_len = 0, req_pages = 0;
    // paged: lane l holds the page id of page win_first + l, and nxt_id that
    // of page win_first + 32 + l, loaded one window ahead so that moving on to
    // the next window never waits for a global load.  The window starts far
    // below page 0 so the first lookup always fills it.
    int32_t win_first = -(1 << 30), win_id = 0, nxt_id = 0;
    auto fetch_ids = [&](int32_t first) -> int32_t {
        return first + lane < req_pages ? __ldg(p.page_indices + req_base + first + lane) : 0;
    };

    // Warp-collective: physical page of the request's page `pg` (paged layout).
    auto page_id = [&](int32_t pg) -> int32_t {
        if (pg < win_first || pg >= win_first + 32) {
            win_id = pg == win_first + 32 ? nxt_id : fetch_ids(pg);
            win_first = pg;
            nxt_id = fetch_ids(pg + 32);
        }
        int32_t id = __shfl_sync(0xffffffffu, win_id, pg - win_first);
        if (id < 0 || id >= p.num_pages) {   // a page outside the pool
            if (lane == 0)
                report(p.status, FD_ERR_DEVICE_BOUNDS);
            id = 0;
        }
        return id;
    };
    // paged: the next box starts at row cur_off of the request's page cur_pg.
    // Tiles are issued in order, so the cursor only moves forward.
    int32_t cur_pg = 0, cur_off = 0;
    auto next_box_row = [&]() -> int32_t {
        // Rows past the request's last key read whatever its last page holds
        // there; the consumers mask them.
        const int32_t y = page_id(min(cur_pg, req_pages - 1)) * p.page_size + cur_off;
        cur_off += SL::kBoxRows;
        if (cur_off >= p.page_size) {
            cur_off -= p.page_size;
            ++cur_pg;
        }
        return y;
    };
    // First rows (in K/V, or in the page pool) of tile i's boxes: ya, and yb
    // for the second 16-row box of a paged tile.  Warp-collective for the
    // paged layout.  The producer computes these before it waits for the
    // tile's stage, so that only the copies remain once the stage is free.
    auto tile_rows = [&](int i, int32_t &ya, int32_t &yb) {
        if constexpr (!paged) {
            ya = req_base + t0 + i * kTile;
        } else {
            ya = next_box_row();
            if constexpr (SL::kBoxRows < kTile)
                yb = next_box_row();
        }
    };
    // Lane 0: put tile i into stage i % NS: one 3-D box of both 64-column
    // halves per tensor and per box of rows (one box, or two of 16 rows).
    auto issue_tile = [&](int i, int32_t ya, int32_t yb) {
        const int s = i % NS;
        const uint32_t full = smem_addr(&bars[s]);
        const uint32_t dst = smem_addr(smem + s * kStageBytes);
        mbar_arrive_expect_tx(full, kStageBytes);
        tma_load_3d(dst, &tm_k, 0, ya, 2 * kvh, full, pol);
        tma_load_3d(dst + 2 * kHalfBytes, &tm_v, 0, ya, 2 * kvh, full, pol);
        if constexpr (SL::kBoxRows < kTile) {
            tma_load_3d(dst + SL::kBlockStride, &tm_k, 0, yb, 2 * kvh, full, pol);
            tma_load_3d(dst + 2 * kHalfBytes + SL::kBlockStride, &tm_v, 0, yb, 2 * kvh, full, pol);
        }
    };

    if (warp == NC) {
        const KeyIndex ki = p.indptr_in_params
                                ? KeyIndex{p.indptr_param, paged ? p.last_len_param : nullptr,
                                           p.page_size}
                                : KeyIndex{p.kv_indptr, p.kv_last_len, p.page_size};
        SplitCoord c{};
        bool ok = derive_split(ki, p.batch, p.chunk, j, false, c);
        if (early_derive)
            griddep_wait();
        if (ok) {
            const int32_t len = split_len_for(c.len, c.splits);
            t0 = c.s * len;
            t1 = min(t0 + len, c.len);
            req_base = c.base;
            req_len = c.len;
            req_pages = c.pages;
            ok = t0 < t1 && c.base >= 0 &&
                 (paged ? c.base + c.pages <= p.num_page_entries
                        : c.base + c.len <= p.total_tokens) &&
                 partial_row(c.prefix, p.num_qo_heads, p.num_qo_heads - 1, c.splits,
                             c.splits - 1) < p.num_partial_rows;
        }
        if (lane == 0) {
            misc[kB] = c.b;
            misc[kPrefix] = c.prefix;
            misc[kSplits] = c.splits;
            misc[kS] = c.s;
            misc[kT0] = t0;
            misc[kT1] = t1;
            misc[kOk] = ok;
            misc[kAbort] = 0;
            for (int s = 0; s < NS; ++s) {
                mbar_init(smem_addr(&bars[s]), 1);        // full: producer arrive + TMA bytes
                mbar_init(smem_addr(&bars[NS + s]), 1);   // empty: consumer warp releases
            }
            fence_mbar_init();
            if (!ok)
                report(p.status, FD_ERR_DEVICE_BOUNDS);
        }
        __syncwarp();
        if (ok && (paged || lane == 0)) {
            pol = l2_evict_first_policy();
            if constexpr (paged) {
                cur_pg = t0 / p.page_size;
                cur_off = t0 % p.page_size;
            }
            const int first = min(NS, (t1 - t0 + kTile - 1) / kTile);
            for (; issued < first; ++issued) {
                int32_t ya = 0, yb = 0;
                tile_rows(issued, ya, yb);
                if (lane == 0)
                    issue_tile(issued, ya, yb);
            }
        }
        if (lane == 0)
            misc[kIssued] = issued;
    }
    (void)req_len;
    __syncthreads();
    if (!misc[kOk])
        return;
    if (warp != NC) {
        t0 = misc[kT0];
        t1 = misc[kT1];
    }
    const int n_tiles = (t1 - t0 + kTile - 1) / kTile;
    const int b = misc[kB];

    // Per-thread fragment coordinates: row g = lane / 4 of the MMA tiles,
    // column pair 2 * (lane % 4).
    const int g_row = lane >> 2, t4 = lane & 3;
    float m_run = -INFINITY, l_part = 0.f;
    float o_acc[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n)
        o_acc[n][0] = o_acc[n][1] = o_acc[n][2] = o_acc[n][3] = 0.f;

    if (warp == NC) {
        // ---------------------------------------------------------- producer
        if (paged || lane == 0) {
            for (int i = issued; i < n_tiles; ++i) {
                const int s = i % NS;
                int32_t ya = 0, yb = 0;
                tile_rows(i, ya, yb);
                int go = 0;
                if (lane == 0) {
                    go = mbar_wait(smem_addr(&bars[NS + s]), ((i / NS) - 1) & 1, p.timeout_ns);
                    if (!go) {
                        misc[kAbort] = 1;
                        report(p.status, FD_ERR_TIMEOUT);
                    } else if (misc[kAbort]) {
                        go = 0;
                    }
                }
                if constexpr (paged)
                    go = __shfl_sync(0xffffffffu, go, 0);
                if (!go)
                    break;
                if (lane == 0)
                    issue_tile(i, ya, yb);
                issued = i + 1;
            }
            if (lane == 0)
                misc[kIssued] = issued;
        }
    } else {
        // ---------------------------------------------------------- consumers
        // Q fragments (A operand of S = Q K^T) for the 8 k-steps of 16 columns;
        // rows g >= G and the padding rows 8-15 are zero.
        uint32_t qa[8][2];
        {
            const bool valid = g_row < G;
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                p.q + ((int64_t)b * p.num_qo_heads + kvh * G + (valid ? g_row : 0)) * kHeadDim);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                qa[kk][0] = valid ? __ldg(qrow + kk * 8 + t4) : 0u;       // cols 16kk + 2t4 (+1)
                qa[kk][1] = valid ? __ldg(qrow + kk * 8 + 4 + t4) : 0u;   // cols 16kk + 8 + 2t4 (+1)
            }
        }
        const float qk_scale = p.q_scale;
        // ldmatrix: lane supplies row lr of matrix lm.  The 128-byte swizzle XORs
        // the 16-byte chunk index with the row index mod 8, which is lr here.
        const int lr = lane & 7, lm = lane >> 3;
        const uint32_t ring = smem_addr(smem);

        for (int i = warp; i < n_tiles; i += NC) {
            const int s = i % NS;
            if (!mbar_wait(smem_addr(&bars[s]), (i / NS) & 1, p.timeout_ns)) {
                misc[kAbort] = 1;
                report(p.status, FD_ERR_TIMEOUT);
                break;
            }
            const uint32_t st = ring + s * kStageBytes;
            const int n_valid = min(kTile, t1 - (t0 + i * kTile));

            // ---- S = Q K^T : 4 key groups (n-tiles) of 8, 8 k-steps of 16 columns
            float sc[4][4];
#pragma unroll
            for (int jn = 0; jn < 4; ++jn)
                sc[jn][0] = sc[jn][1] = sc[jn][2] = sc[jn][3] = 0.f;
#pragma unroll
            for (int kp = 0; kp < 4; ++kp) {           // 32 columns per ldmatrix.x4
                const uint32_t half = st + (kp >> 1) * SL::kHalfStride;
                const int chunk = 4 * (kp & 1) + lm;   // matrix lm = columns 8*lm .. +7
#pragma unroll
                for (int jn = 0; jn < 4; ++jn) {
                    // key row 8 jn + lr: block jn / 2, row 8 (jn % 2) + lr in it
                    const uint32_t row_off = (jn >> 1) * SL::kBlockStride + (8 * (jn & 1) + lr) * 128;
                    uint32_t kb[4];
                    ldsm_x4(half + row_off + ((chunk ^ lr) << 4), kb);
                    mma_bf16(sc[jn], qa[2 * kp][0], 0u, qa[2 * kp][1], 0u, kb[0], kb[1]);
                    mma_bf16(sc[jn], qa[2 * kp + 1][0], 0u, qa[2 * kp + 1][1], 0u, kb[2], kb[3]);
                }
            }

            // ---- online softmax on row g_row (this thread's 8 scores of the tile)
            float x[8];
            float mt = -INFINITY;
#pragma unroll
            for (int jn = 0; jn < 4; ++jn)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = 8 * jn + 2 * t4 + e;
                    const float v = key < n_valid ? sc[jn][e] * qk_scale : -INFINITY;
                    x[2 * jn + e] = v;
                    mt = fmaxf(mt, v);
                }
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
            const float m_new = fmaxf(m_run, mt);
            const float alpha = exp2f(m_run - m_new);
            m_run = m_new;
            float psum = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                x[e] = exp2f(x[e] - m_new);
                psum += x[e];
            }
            l_part = fmaf(l_part, alpha, psum);
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    o_acc[n][0] *= alpha;
                    o_acc[n][1] *= alpha;
                    o_acc[n][2] *= alpha;
                    o_acc[n][3] *= alpha;
                }
            }
            // P as the A operand: k-step ks covers keys 16ks .. 16ks+15 (n-tiles
            // 2ks, 2ks+1); rows 0-7 hi, rows 8-15 lo.
            uint32_t pa[2][4];
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const float p0 = x[4 * ks], p1 = x[4 * ks + 1];
                const float p2 = x[4 * ks + 2], p3 = x[4 * ks + 3];
                const float h0 = bf16_round(p0), h1 = bf16_round(p1);
                const float h2 = bf16_round(p2), h3 = bf16_round(p3);
                pa[ks][0] = pack_bf16(h0, h1);
                pa[ks][1] = pack_bf16(p0 - h0, p1 - h1);
                pa[ks][2] = pack_bf16(h2, h3);
                pa[ks][3] = pack_bf16(p2 - h2, p3 - h3);
            }

            // ---- O += P V : 2 k-steps of 16 keys, 16 n-tiles of 8 columns
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                // matrix lm: keys 16 ks + 8 (lm & 1) + lr = block ks, row 8 (lm & 1) + lr
                const uint32_t row_off = ks * SL::kBlockStride + (8 * (lm & 1) + lr) * 128;
#pragma unroll
                for (int np = 0; np < 8; ++np) {                // 16 columns per ldmatrix.x4
                    const uint32_t half = st + 2 * kHalfBytes + (np >> 2) * SL::kHalfStride;
                    const int chunk = 2 * (np & 3) + (lm >> 1);  // columns 8*(lm>>1) ..
                    uint32_t vb[4];
                    ldsm_x4_trans(half + row_off + ((chunk ^ lr) << 4), vb);
                    mma_bf16(o_acc[2 * np], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], vb[0], vb[1]);
                    mma_bf16(o_acc[2 * np + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], vb[2],
                             vb[3]);
                }
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
        float l_tot = l_part;
        l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 1);
        l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 2);
        if (g_row < G) {
            float *dst = comb_acc + (warp * G + g_row) * kHeadDim + 2 * t4;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                *reinterpret_cast<float2 *>(dst + 8 * n) =
                    make_float2(o_acc[n][0] + o_acc[n][2], o_acc[n][1] + o_acc[n][3]);
            if (t4 == 0) {
                comb_m[warp * G + g_row] = m_run;
                comb_l[warp * G + g_row] = l_tot;
            }
        }
    }
    __syncthreads();

    const int prefix = misc[kPrefix], splits = misc[kSplits], split = misc[kS];
    // A request with one split needs no stage 2 when it is fused: write O/LSE.
    const bool direct = p.fuse_merge && splits == 1;
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
            const float e = mx == -INFINITY ? 0.f : exp2f(comb_m[w * G + g] - mx);
            den = fmaf(e, comb_l[w * G + g], den);
            const float4 a = *reinterpret_cast<const float4 *>(comb_acc + (w * G + g) * kHeadDim + 4 * c4);
            o.x = fmaf(e, a.x, o.x);
            o.y = fmaf(e, a.y, o.y);
            o.z = fmaf(e, a.z, o.z);
            o.w = fmaf(e, a.w, o.w);
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        o.x *= inv;
        o.y *= inv;
        o.z *= inv;
        o.w *= inv;
        const float lse_nat = den > 0.f ? (mx + log2f(den)) * kLn2 : -INFINITY;
        if (direct) {
            const int64_t row = (int64_t)b * p.num_qo_heads + kvh * G + g;
            *reinterpret_cast<float4 *>(p.o + row * kHeadDim + 4 * c4) = o;
            if (c4 == 0)
                p.lse[row] = lse_nat;
        } else {
            const int64_t row = partial_row(prefix, p.num_qo_heads, kvh * G + g, splits, split);
            *reinterpret_cast<float4 *>(p.partial_o + row * kHeadDim + 4 * c4) = o;
            if (c4 == 0)
                p.partial_lse[row] = lse_nat;
        }
    }

    if (p.fuse_merge && splits > 1) {
        // Ticket: the last CTA of the (request, KV head) group to finish merges
        // the group (stage 2).  The ticket add is acquire-release at GPU scope:
        // it publishes this CTA's partials (made visible to thread 0 by the
        // barrier) and lets the last CTA see everyone else's; that CTA also
        // resets the ticket for the next call.
        __syncthreads();
        if (tid == 0) {
            cuda::atomic_ref<int, cuda::thread_scope_device> ticket(
                p.counters[(int64_t)b * p.num_kv_heads + kvh]);
            const int prev = ticket.fetch_add(1, cuda::memory_order_acq_rel);
            const bool last = prev == splits - 1;
            if (last)
                ticket.store(0, cuda::memory_order_relaxed);
            misc[kLast] = last;
        }
        __syncthreads();
        if (misc[kLast])
            merge_group<G, NC + 1>(p, prefix, splits, b, kvh, warp, lane,
                                   reinterpret_cast<float *>(smem));
    }
    // This CTA's outputs are written: a dependent grid may launch.
    __syncthreads();
    griddep_launch_dependents();
}

// Launch shape: consumer warps, stages, resident CTAs per SM (compile-time;
// the defaults are the measured best on GB300).
#ifndef FD_SPLIT_CONSUMER_WARPS
#define FD_SPLIT_CONSUMER_WARPS 4
#endif
#ifndef FD_SPLIT_STAGES
#define FD_SPLIT_STAGES 4
#endif
#ifndef FD_SPLIT_CTAS_PER_SM
#define FD_SPLIT_CTAS_PER_SM 2
#endif
constexpr int kNC = FD_SPLIT_CONSUMER_WARPS;
constexpr int kNS = FD_SPLIT_STAGES;
constexpr int kMinCtas = FD_SPLIT_CTAS_PER_SM;

template <int G, int KV>
cudaError_t launch_g(const CUtensorMap &tk, const CUtensorMap &tv, const SplitParams &p,
                     int num_work, cudaStream_t stream)
{
    using L = Layout<G, kNC, kNS>;
    static_assert(kMinCtas * (L::kAlloc + 1024) <= 233472,
                  "the resident CTAs must fit in shared memory");
    auto kern = split_kv_kernel<G, kNC, kNS, kMinCtas, KV>;
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_work);
    cfg.blockDim = dim3((kNC + 1) * 32);
    cfg.dynamicSmemBytes = L::kAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace

int split_ctas_per_sm()
{
    return kMinCtas;
}

cudaError_t launch_split(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const SplitParams &p,
                         int group, int num_work, cudaStream_t stream)
{
    const int kv = p.kv_last_len == nullptr ? kKvRagged
                   : p.box_rows == kTile    ? kKvPaged
                                            : kKvPaged16;
    auto by_layout = [&](auto g) -> cudaError_t {
        constexpr int G = decltype(g)::value;
        switch (kv) {
        case kKvRagged: return launch_g<G, kKvRagged>(tm_k, tm_v, p, num_work, stream);
        case kKvPaged: return launch_g<G, kKvPaged>(tm_k, tm_v, p, num_work, stream);
        default: return launch_g<G, kKvPaged16>(tm_k, tm_v, p, num_work, stream);
        }
    };
    switch (group) {
    case 1: return by_layout(std::integral_constant<int, 1>{});
    case 2: return by_layout(std::integral_constant<int, 2>{});
    case 4: return by_layout(std::integral_constant<int, 4>{});
    case 8: return by_layout(std::integral_constant<int, 8>{});
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fd
