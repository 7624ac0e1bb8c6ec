// split_kernel.cuh -- stage 1 of split-KV decode attention on sm_103a (the
// kernel templates; split_kernel.cu instantiates them for bf16 K/V and
// split_kernel_fp8.cu for FP8 E4M3 K/V).
//
// "FlashDecoding++: sequence-dimension KV split parallelism for LLM serving"
// (techknowgenie.com), §2 (each block keeps the query on chip and copies only
// its own chunk of K/V from HBM into shared memory) and §3 stage 1 (per chunk:
// logits, local max, exp, local sum, probability-weighted V; the block stores
// the partial and exits).
//
// Work item = one (split, KV head).  All G query heads that share the KV head
// are served from the same shared-memory tiles, so every K/V byte is read
// from HBM once per step.  The kernel is persistent: a grid of at most
// (SMs x resident CTAs per SM) CTAs, CTA c taking items c, c + grid, ... in
// order.  Its tiles form one stream through the stage ring, so while the
// consumer warps finish one item (combine, partial write, stage-2 ticket and
// merge) the producer is already loading the next; a CTA's start-up and
// epilogue costs are paid once per CTA rather than once per item.
//
// Warp roles:
//   warp NC (producer): one lane issues TMA loads of 32-key tiles of K and V
//     into an NS-stage ring guarded by full/empty mbarriers.  A tile is one
//     3-D box per tensor holding both 64-column halves of the head's 32 rows
//     (128-byte swizzle), or, for a paged cache whose pages are not a
//     multiple of 32 keys, two such boxes of 16 rows.
//     It hands each item to the consumers through a ring of kDescSlots
//     descriptors (full/empty mbarriers of their own).
//   warps 0..NC-1 (consumers): warp w takes stream tiles w, w+NC, ...  NS is a
//     multiple of NC, so every stage always goes to the same warp and a warp
//     never waits on a barrier more than one phase ahead (parity waits can only
//     tell two phases apart).  Each warp keeps its own online-softmax state per
//     item and at the item's end the NC states are merged in shared memory
//     with the same rescaling as stage 2.
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
#pragma once

#include <cuda/atomic>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace fd {
namespace {

constexpr int kHalfBytes = kTile * 128;   // 32 keys x 64 bf16

enum KvLayout { kKvRagged = 0, kKvPaged = 1, kKvPaged16 = 2 };
enum KvType { kKvBf16 = 0, kKvFp8 = 1, kKvInt4 = 2 };

// One pipeline stage holds K then V for kTile = 32 keys of one KV head.
//  bf16: a tensor's key row r (0..31), column half h (64 columns of 128 bytes,
//    16-byte chunks XOR-swizzled by r % 8) sits at
//      h * HalfStride + (r / 16) * BlockStride + (r % 16) * 128:
//      ragged, paged:  [half][32 rows]            HalfStride 4096, BlockStride 2048
//      paged16:        [16-row block][half][16]   HalfStride 2048, BlockStride 4096
//    (paged16 is what one 16-row box of both halves per page lands as).
//  FP8: a tensor is [32 rows][128 bytes] (a key row of the head is 128 one-byte
//    values), 16-byte chunks XOR-swizzled by r % 8; a second 16-row page box
//    lands 16 rows further.
//  INT4: a tensor is [32 rows][64 bytes] (128 four-bit values), 16-byte chunks
//    XOR-swizzled by (r / 2) % 4, then the rows' K scales and V scales (fp32,
//    32 each).  INT4 stages are filled by 16-byte cp.async copies (kDirect;
//    a consumer warp's own lanes on ragged one-item calls, the producer warp's
//    otherwise): with 64-byte rows and per-row scales, TMA boxes cost more
//    copy-engine time per byte than the copies do.
template <int KV, int DT>
struct Stage {
    static constexpr bool kFp8 = DT == kKvFp8;
    static constexpr bool kInt4 = DT == kKvInt4;
    static constexpr bool kDirect = kInt4;
    static constexpr int kRowBytes = kInt4 ? kHeadDim / 2 : kFp8 ? kHeadDim : 2 * kHeadDim;
    static constexpr int kFullArrivals = kDirect ? 32 : 1;   // full barrier: arrivals per phase
    static constexpr int kTensorBytes = kTile * kRowBytes;
    static constexpr int kBoxRows = KV == kKvPaged16 ? 16 : kTile;
    static constexpr int kKsOff = 2 * kTensorBytes;            // INT4 scales
    static constexpr int kVsOff = kKsOff + kTile * 4;
    static constexpr int kBytes = kInt4 ? kVsOff + kTile * 4 : 2 * kTensorBytes;
    static constexpr int kHalfStride = KV == kKvPaged16 ? 2048 : kHalfBytes;
    static constexpr int kBlockStride = KV == kKvPaged16 ? 4096 : 2048;
    // a TMA copy's shared-memory destination must be 128-byte aligned
    static_assert(kDirect || kTensorBytes % 1024 == 0, "stage copies on 128-byte boundaries");

    // Offset in a tensor's part of the stage of 16-byte chunk c of key row r
    // (the bf16 and FP8 layouts are those of the TMA boxes' 128-byte swizzle,
    // which XORs the chunk index with address bits 7-9).
    static __device__ __forceinline__ uint32_t chunk_offset(int r, int c)
    {
        if constexpr (kInt4)
            return r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
        else if constexpr (kFp8)
            return r * 128 + ((c ^ (r & 7)) << 4);
        else
            return (c >> 3) * kHalfStride + (r >> 4) * kBlockStride + (r & 15) * 128 +
                   (((c & 7) ^ (r & 7)) << 4);
    }
};
constexpr int kMaxGroup = 8;                   // rows 8-15 of the MMA carry the lo part of P
constexpr int kNoExp = -1000;                  // INT4 V-scale exponent before any nonzero scale

// 2^k as a float, exactly, for k in [-126, 127]; 0 below, +inf above.
__device__ __forceinline__ float pow2i(int k)
{
    return k < -126 ? 0.f : k > 127 ? INFINITY : __int_as_float((127 + k) << 23);
}

enum Misc { kAbort, kIssued, kDescs, kLast, kFinalK, kMiscCount };

// An item (one split of one KV head) as the producer hands it to the other
// warps: request, its split prefix and count, split, key range [t0, t1)
// relative to the request's first key, KV head, index of the item's first
// tile in the CTA's stream of tiles, the head's K and V scales (FP8 K/V; float
// bits), the request's first key row or page-list entry, and a state:
// kItemOk, kItemBad (outside the plan: the CTA stops) or kItemEnd (no further
// item; the previous one was the CTA's last).
enum Desc { kDB, kDPrefix, kDSplits, kDS, kDT0, kDT1, kDKvh, kDGt0, kDState, kDKs, kDVs, kDBase, kDescInts };
enum ItemState { kItemBad = 0, kItemOk = 1, kItemEnd = 2 };
constexpr int kDescSlots = 4;

struct Item {
    int32_t b, prefix, splits, s, t0, t1, kvh, gt0, state, ks, vs, base;
};

__device__ __forceinline__ Item read_item(const volatile int *d)
{
    return Item{d[kDB], d[kDPrefix], d[kDSplits], d[kDS], d[kDT0], d[kDT1],
                d[kDKvh], d[kDGt0], d[kDState], d[kDKs], d[kDVs], d[kDBase]};
}

// Shared memory of the one-item kernel: [stage ring | full[NS] empty[NS] |
// item descriptor | misc].  The consumer-state combine and the stage-2 merge
// of the CTA's item work over the drained ring.
template <int G, int NC, int NS, int SB>
struct SingleLayout {
    static_assert(NS % NC == 0, "each stage must belong to one consumer warp");
    static_assert(G >= 1 && G <= kMaxGroup, "group size");
    static constexpr int kWarps = NC + 1;
    static_assert(kWarps * G * (kHeadDim + 2) * 4 <= NS * SB, "the merge fits the ring");
    static constexpr int kOffBar = NS * SB;
    static constexpr int kOffDesc = kOffBar + 2 * NS * 8;
    static constexpr int kOffMisc = kOffDesc + kDescInts * 4;
    static constexpr int kOffFills = kOffMisc + kMiscCount * 4;   // copies issued into each stage
    static constexpr int kBytes = kOffFills + NS * 4;
    static constexpr int kAlloc = kBytes + 1024;   // room to align the base to 1024 B
};

// Shared memory of the persistent kernel (warps: 0..NC-1 consumers, NC
// producer, NC+1 epilogue): [stage ring | Q of each item slot | 2 consumer-
// state buffers | mbarriers | item descriptors | misc].  Barriers: full[NS],
// empty[NS] (stages), item_full[4] (descriptor written and its Q landed),
// item_empty[4] (consumers and epilogue warp are done with the slot),
// state_full[2], state_empty[2] (a finished item's consumer states, handed to
// the epilogue warp).
template <int G, int NC, int NS, int SB>
struct PersistentLayout {
    static_assert(NS % NC == 0, "each stage must belong to one consumer warp");
    static_assert(G >= 1 && G <= kMaxGroup, "group size");
    static constexpr int kWarps = NC + 2;
    static constexpr int kQBytes = G * kHeadDim * 2;                    // the item's G query rows
    static constexpr int kQSlot = (kQBytes + 127) / 128 * 128;
    // [NC][G][128] acc, then m, l; rounded up so that the second buffer's
    // float4 rows stay 16-byte aligned for any NC and G
    static constexpr int kStateBytes = (NC * G * (kHeadDim + 2) * 4 + 127) / 128 * 128;
    static_assert(kWarps * G * (kHeadDim + 2) * 4 <= NS * SB,
                  "the last item's merge works over the drained ring");
    static constexpr int kOffQ = NS * SB;
    static constexpr int kOffState = kOffQ + kDescSlots * kQSlot;
    static constexpr int kOffBar = kOffState + 2 * kStateBytes;
    static constexpr int kNumBars = 2 * NS + 2 * kDescSlots + 4;
    static constexpr int kOffDesc = kOffBar + kNumBars * 8;
    static constexpr int kOffMisc = kOffDesc + kDescSlots * kDescInts * 4;
    static constexpr int kBytes = kOffMisc + kMiscCount * 4;
    static constexpr int kAlloc = kBytes + 1024;   // room to align the base to 1024 B
    static_assert(kOffBar % 8 == 0, "mbarriers are 8-byte aligned");
};

// Barrier of a group: BAR 0 = the whole CTA (__syncthreads), BAR -1 = one warp.
template <int BAR>
__device__ __forceinline__ void group_sync()
{
    static_assert(BAR == 0 || BAR == -1, "barrier");
    if constexpr (BAR == 0)
        __syncthreads();
    else
        __syncwarp();
}

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

// The warp's 8x8 matrix of 16-bit elements (lane (g, t4) holds row g,
// columns 2t4 and 2t4 + 1) transposed, in the same fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a)
{
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
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

// D (+)= A B for one m16n8k16 tile, f16 inputs, fp32 accumulator.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> packed f16x2 (first argument in the low half), round to nearest.
__device__ __forceinline__ uint32_t pack_f16(float lo_elem, float hi_elem)
{
    const __half2 h = __floats2half2_rn(lo_elem, hi_elem);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float f16_round(float x)
{
    return __half2float(__float2half_rn(x));
}

// Four E4M3 values (bytes 0..3 of x) -> two f16x2: lo = bytes 0, 1 and
// hi = bytes 2, 3 (the lower byte in the lower half).  Every E4M3 value is an
// f16 value, so this is exact.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t &lo, uint32_t &hi)
{
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
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

// Eight 4-bit two's-complement values (nibble j of each 16-bit half of x; the
// low nibble first) -> four f16x2: r[j] = (nibble j of the low half, nibble j
// of the high half).  Per half, the nibbles at bits 0-3 and 4-7 are taken in
// place: one lop3 keeps the nibble, flips its sign bit (u = n + 8) and sets
// the exponent of 1024, which gives the f16 1024 + u (bits 0-3, where the unit
// in the last place is 1) or 1024 + 16 u (bits 4-7); subtracting 1032, or a
// multiply-add by 1/16 and -72, leaves n.  Nibbles 2 and 3 do the same after
// one shift by 8.  Every step is exact.
__device__ __forceinline__ void int4x8_to_f16x2x4(uint32_t x, uint32_t (&r)[4])
{
    // lop3 0x6A = (b & (a ^ c)) | (~b & c): a nibble of a under mask b with
    // its sign bit flipped by c, and c's exponent bits elsewhere
    auto pick = [](uint32_t a, uint32_t mask, uint32_t c) {
        uint32_t d;
        asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(mask), "r"(c));
        return d;
    };
    const uint32_t y = x >> 8;
    const uint32_t t0 = pick(x, 0x000F000Fu, 0x64086408u), t1 = pick(x, 0x00F000F0u, 0x64806480u);
    const uint32_t t2 = pick(y, 0x000F000Fu, 0x64086408u), t3 = pick(y, 0x00F000F0u, 0x64806480u);
    constexpr uint32_t k1032 = 0x64086408u, kSixteenth = 0x2C002C00u, kMinus72 = 0xD480D480u;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r[0]) : "r"(t0), "r"(k1032));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r[1]) : "r"(t1), "r"(kSixteenth), "r"(kMinus72));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r[2]) : "r"(t2), "r"(k1032));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r[3]) : "r"(t3), "r"(kSixteenth), "r"(kMinus72));
}

// 16 zero bytes to shared memory (32-bit shared address, 16-byte aligned).
__device__ __forceinline__ void sts_zero16(uint32_t addr)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One fp32 from shared memory (32-bit shared address).
__device__ __forceinline__ float lds_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Stage 2 for one (request, KV head) group, run by the CTA that finished the
// group last: for each of its G heads, M = max_i LSE_i, w_i = exp(LSE_i - M),
// O = sum_i w_i O_i / sum_i w_i, LSE = M + ln sum_i w_i over the group's splits.
// Warp w of the first NW warps takes splits w, w + NW, ... (U splits of loads
// in flight per batch, lane = 4 output columns, all G heads), keeps a running
// maximum per head, and the NW warp states are combined through `scratch`
// behind barrier BAR (a single warp writes O / LSE from its registers).  The
// other CTAs' partials are read through L2 (ld.global.cg).
template <int G, int NW, int BAR>
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
    if constexpr (NW == 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float inv = 1.f / den[g];
            const int64_t row = (int64_t)b * p.num_qo_heads + kvh * G + g;
            reinterpret_cast<float4 *>(p.o + row * kHeadDim)[lane] =
                make_float4(acc[g].x * inv, acc[g].y * inv, acc[g].z * inv, acc[g].w * inv);
            if (lane == 0)
                p.lse[row] = m[g] + logf(den[g]);
        }
        return;
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
    group_sync<BAR>();
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

// One consumer warp's work on one staged tile of 32 keys (stage at shared
// address st, the first n_valid keys real): S = Q K^T on the tensor cores,
// the online-softmax update of the running max m_run / row sum l_part (base 2,
// logits = S * qk_scale), and O += P V.  qa: the Q fragments (A operand) of
// the 8 k-steps of 16 head dimensions.
//  bf16: mma.sync bf16; B fragments straight from the tile via ldmatrix.
//  FP8: mma.sync f16; the E4M3 bytes are widened to f16 (exact) in registers.
//    An ldmatrix of the 128-byte key rows read as 16-bit pairs gives lane
//    (g, t4) dims 16c + 4t4 .. +3 of key g, which feed k positions 2t4, 2t4+1
//    (dims +0, +1) and 2t4+8, 2t4+9 (dims +2, +3) of k-step c; qa holds q in the
//    same order.  For P V, ldmatrix.trans gives lane (g, t4) dims 16c + 2g and
//    +1 of keys 2t4 and 2t4+1, so one tile of columns takes the even dims and
//    one the odd: o_acc[2c + e] holds dims 16c + 4t4 + e (and + 2).
//  INT4: mma.sync f16; the four-bit codes are widened to f16 (exact) in
//    registers.  An ldmatrix of the 64-byte key rows gives lane (g, t4) dims
//    32c + 8t4 .. +7 of key g in one word; nibbles j and j + 4 pair up, so
//    k-step 2c + h takes dims 32c + 8t4 + 2h (+4) at k 2t4 (+1) and + 2h + 1
//    (+4) at k 2t4 + 8 (+9); qa holds q in that order.  Each key's K scale
//    multiplies its logit, and its V scale its probability in P V (the row sum
//    takes the probability alone).  ldmatrix.trans of V gives lane (g, t4) dims
//    32c + 4g .. +3 of keys 2t4 and 2t4 + 1, so o_acc[4c + j] holds dims
//    32c + 8t4 + j (and + 4).
template <int KV, int DT>
__device__ __forceinline__ void consume_tile(uint32_t st, int n_valid, const uint32_t (&qa)[8][2],
                                             float qk_scale, int lane, float &m_run, float &l_part,
                                             float (&o_acc)[16][4], int &v_exp)
{
    using S = Stage<KV, DT>;
    const int t4 = lane & 3;
    // ldmatrix: lane supplies row lr of matrix lm.  The 128-byte swizzle XORs
    // the 16-byte chunk index with the row index mod 8, which is lr here.
    const int lr = lane & 7, lm = lane >> 3;

    // ---- rows past the last key (the rest of a page, another request's keys)
    // get P = 0, but 0 * NaN would still reach O: a tile that ends early has
    // its V rows from n_valid on zeroed (the stage is this warp's alone).  The
    // proxy fence orders these writes before the stage's next TMA refill.
    // INT4 needs none: its codes are finite, and a masked key's V scale is
    // replaced by 0 before P V.
    if constexpr (!S::kInt4) {
        if (n_valid < kTile) {
            constexpr int kChunks = S::kRowBytes / 16;
            const uint32_t vt = st + S::kTensorBytes;
            for (int idx = lane; idx < (kTile - n_valid) * kChunks; idx += 32)
                sts_zero16(vt + S::chunk_offset(n_valid + idx / kChunks, idx % kChunks));
            fence_proxy_async_shared();
            __syncwarp();
        }
    }

    // ---- S = Q K^T : 4 key groups (n-tiles) of 8, 8 k-steps of 16 dims
    float sc[4][4];
#pragma unroll
    for (int jn = 0; jn < 4; ++jn)
        sc[jn][0] = sc[jn][1] = sc[jn][2] = sc[jn][3] = 0.f;
    if constexpr (S::kInt4) {
#pragma unroll
        for (int jn = 0; jn < 4; ++jn) {
            // matrix lm = chunk lm of key rows 8 jn .. +7 (64-byte swizzle)
            const int r = 8 * jn + lr;
            uint32_t kb[4];
            ldsm_x4(st + r * 64 + ((lm ^ ((r >> 1) & 3)) << 4), kb);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t b[4];   // b[j]: dims 32c + 8t4 + j and + 4 of key 8 jn + g
                int4x8_to_f16x2x4(kb[c], b);
                mma_f16(sc[jn], qa[2 * c][0], 0u, qa[2 * c][1], 0u, b[0], b[1]);
                mma_f16(sc[jn], qa[2 * c + 1][0], 0u, qa[2 * c + 1][1], 0u, b[2], b[3]);
            }
        }
    } else if constexpr (S::kFp8) {
#pragma unroll
        for (int jn = 0; jn < 4; ++jn) {
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {         // chunks 4hc .. 4hc+3 (64 dims)
                uint32_t kb[4];
                ldsm_x4(st + (8 * jn + lr) * 128 + (((4 * hc + lm) ^ lr) << 4), kb);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int c = 4 * hc + m;
                    uint32_t b0, b1;   // dims 16c + 4t4 (+1), 16c + 4t4 + 2 (+3)
                    e4m3x4_to_f16x2x2(kb[m], b0, b1);
                    mma_f16(sc[jn], qa[c][0], 0u, qa[c][1], 0u, b0, b1);
                }
            }
        }
    } else {
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {             // 32 columns per ldmatrix.x4
            const uint32_t half = st + (kp >> 1) * S::kHalfStride;
            const int chunk = 4 * (kp & 1) + lm;      // matrix lm = columns 8*lm .. +7
#pragma unroll
            for (int jn = 0; jn < 4; ++jn) {
                // key row 8 jn + lr: block jn / 2, row 8 (jn % 2) + lr in it
                const uint32_t row_off = (jn >> 1) * S::kBlockStride + (8 * (jn & 1) + lr) * 128;
                uint32_t kb[4];
                ldsm_x4(half + row_off + ((chunk ^ lr) << 4), kb);
                mma_bf16(sc[jn], qa[2 * kp][0], 0u, qa[2 * kp][1], 0u, kb[0], kb[1]);
                mma_bf16(sc[jn], qa[2 * kp + 1][0], 0u, qa[2 * kp + 1][1], 0u, kb[2], kb[3]);
            }
        }
    }

    // ---- online softmax on row g_row (this thread's 8 scores of the tile)
    float x[8];
    float mt = -INFINITY;
    const uint32_t ks_base = st + S::kKsOff, vs_base = st + S::kVsOff;
#pragma unroll
    for (int jn = 0; jn < 4; ++jn)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int key = 8 * jn + 2 * t4 + e;
            float logit = sc[jn][e] * qk_scale;
            if constexpr (S::kInt4)
                logit = sc[jn][e] * lds_f32(ks_base + 4 * key) * qk_scale;
            const float v = key < n_valid ? logit : -INFINITY;
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
    // INT4: the tile's V scales (0 for masked keys: another request's row or
    // past the end is never read).  P V runs in f16, so the weights enter it as
    // p * v_scale * 2^-v_exp, where 2^v_exp bounds every V scale seen so far
    // by this warp: the products stay in [-1, 1], far from f16's overflow and
    // subnormal range, whatever the scales.  When v_exp grows, O is rescaled
    // by the same exact power of two, together with the softmax rescale;
    // write_state multiplies 2^v_exp back.
    float vs[2][4] = {};
    float oscale = alpha;
    if constexpr (S::kInt4) {
        float vmax = 0.f;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const int k0 = 16 * ks + 2 * t4;   // keys k0 (+1) and k0 + 8 (+9)
            const uint32_t vk = vs_base + 4 * k0;
            vs[ks][0] = k0 < n_valid ? lds_f32(vk) : 0.f;
            vs[ks][1] = k0 + 1 < n_valid ? lds_f32(vk + 4) : 0.f;
            vs[ks][2] = k0 + 8 < n_valid ? lds_f32(vk + 32) : 0.f;
            vs[ks][3] = k0 + 9 < n_valid ? lds_f32(vk + 36) : 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                vmax = fmaxf(vmax, fabsf(vs[ks][j]));
        }
        // lanes of one t4 hold the same keys: the warp's 32 keys in 2 steps
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 1));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));
        if (!(vmax <= 0.f)) {   // a nonzero, inf or NaN scale: vmax < 2^e
            const int e = ((__float_as_int(vmax) >> 23) & 0xFF) - 126;
            if (e > v_exp) {
                oscale *= pow2i(v_exp - e);   // 0 when v_exp is still kNoExp
                v_exp = e;
            }
        }
    }
    if (__any_sync(0xffffffffu, oscale != 1.f)) {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            o_acc[n][0] *= oscale;
            o_acc[n][1] *= oscale;
            o_acc[n][2] *= oscale;
            o_acc[n][3] *= oscale;
        }
    }
    // P as the A operand: k-step ks covers keys 16ks .. 16ks+15 (n-tiles
    // 2ks, 2ks+1); rows 0-7 hi, rows 8-15 lo = P - hi, in the MMA's type.
    uint32_t pa[2][4];
    // INT4: 2^-v_exp (NaN-propagating 0 once an infinite or NaN scale was seen)
    const float vinv = S::kInt4 ? (v_exp == kNoExp ? 1.f : pow2i(-v_exp)) : 1.f;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        float p0 = x[4 * ks], p1 = x[4 * ks + 1];
        float p2 = x[4 * ks + 2], p3 = x[4 * ks + 3];
        if constexpr (S::kInt4) {
            // keys 16ks + 2t4 (+1) and 16ks + 8 + 2t4 (+1)
            p0 *= vs[ks][0] * vinv;
            p1 *= vs[ks][1] * vinv;
            p2 *= vs[ks][2] * vinv;
            p3 *= vs[ks][3] * vinv;
        }
        if constexpr (S::kFp8 || S::kInt4) {
            const float h0 = f16_round(p0), h1 = f16_round(p1);
            const float h2 = f16_round(p2), h3 = f16_round(p3);
            pa[ks][0] = pack_f16(h0, h1);
            pa[ks][1] = pack_f16(p0 - h0, p1 - h1);
            pa[ks][2] = pack_f16(h2, h3);
            pa[ks][3] = pack_f16(p2 - h2, p3 - h3);
        } else {
            const float h0 = bf16_round(p0), h1 = bf16_round(p1);
            const float h2 = bf16_round(p2), h3 = bf16_round(p3);
            pa[ks][0] = pack_bf16(h0, h1);
            pa[ks][1] = pack_bf16(p0 - h0, p1 - h1);
            pa[ks][2] = pack_bf16(h2, h3);
            pa[ks][3] = pack_bf16(p2 - h2, p3 - h3);
        }
    }

    // ---- O += P V : 2 k-steps of 16 keys, 16 n-tiles of 8 columns
    if constexpr (S::kInt4) {
        const uint32_t vt = st + S::kTensorBytes;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            // matrix lm: keys 16 ks + 8 (lm & 1) .. +7, chunk 2 cp + (lm >> 1)
            const int r = 16 * ks + 8 * (lm & 1) + lr;
#pragma unroll
            for (int cp = 0; cp < 2; ++cp) {
                uint32_t vb[4];
                ldsm_x4_trans(vt + r * 64 + (((2 * cp + (lm >> 1)) ^ ((r >> 1) & 3)) << 4), vb);
#pragma unroll
                for (int h = 0; h < 2; ++h) {         // chunk c = 2 cp + h: vb[2h] keys +0..7, vb[2h+1] +8..15
                    const int c = 2 * cp + h;
                    uint32_t lo[4], hi[4];            // [j]: dim 32c + 4g + j of keys 2t4, 2t4 + 1
                    int4x8_to_f16x2x4(vb[2 * h], lo);
                    int4x8_to_f16x2x4(vb[2 * h + 1], hi);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_f16(o_acc[4 * c + j], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], lo[j],
                                hi[j]);
                }
            }
        }
    } else if constexpr (S::kFp8) {
        const uint32_t vt = st + S::kTensorBytes;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            // matrix lm: keys 16 ks + 8 (lm & 1) .. +7, chunk 2 cp + (lm >> 1)
            const uint32_t row = vt + (16 * ks + 8 * (lm & 1) + lr) * 128;
#pragma unroll
            for (int cp = 0; cp < 4; ++cp) {
                uint32_t vb[4];
                ldsm_x4_trans(row + (((2 * cp + (lm >> 1)) ^ lr) << 4), vb);
#pragma unroll
                for (int h = 0; h < 2; ++h) {         // chunk c = 2 cp + h: vb[2h] keys +0..7, vb[2h+1] +8..15
                    const int c = 2 * cp + h;
                    // bytes of vb: key 2t4 (dim 2g, 2g+1), key 2t4+1 (dim 2g, 2g+1);
                    // regrouped as (key 2t4, key 2t4+1) of dim 2g, then of dim 2g+1
                    uint32_t lo_even, lo_odd, hi_even, hi_odd;
                    e4m3x4_to_f16x2x2(__byte_perm(vb[2 * h], 0u, 0x3120), lo_even, lo_odd);
                    e4m3x4_to_f16x2x2(__byte_perm(vb[2 * h + 1], 0u, 0x3120), hi_even, hi_odd);
                    mma_f16(o_acc[2 * c], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], lo_even, hi_even);
                    mma_f16(o_acc[2 * c + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], lo_odd,
                            hi_odd);
                }
            }
        }
    } else {
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            // matrix lm: keys 16 ks + 8 (lm & 1) + lr = block ks, row 8 (lm & 1) + lr
            const uint32_t row_off = ks * S::kBlockStride + (8 * (lm & 1) + lr) * 128;
#pragma unroll
            for (int np = 0; np < 8; ++np) {          // 16 columns per ldmatrix.x4
                const uint32_t half = st + 2 * kHalfBytes + (np >> 2) * S::kHalfStride;
                const int chunk = 2 * (np & 3) + (lm >> 1);   // columns 8*(lm>>1) ..
                uint32_t vb[4];
                ldsm_x4_trans(half + row_off + ((chunk ^ lr) << 4), vb);
                mma_bf16(o_acc[2 * np], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], vb[0], vb[1]);
                mma_bf16(o_acc[2 * np + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], vb[2],
                         vb[3]);
            }
        }
    }
}

// The producer warp's side of the stage ring, one item at a time: where each
// tile's rows are (in K/V, or through the page table in the page pool) and
// how a tile is put into a stage.  page_id, next_box_row and tile_rows are
// warp-collective in the paged layout (the warp shares a window of page ids);
// issue is lane 0's.
template <int NS, int KV, int DT>
struct TileSource {
    using SL = Stage<KV, DT>;
    static constexpr bool kPaged = KV != kKvRagged;
    const SplitParams &p;
    const CUtensorMap *tm_k, *tm_v;
    uint8_t *ring;
    uint64_t *full;   // full[NS]
    uint64_t pol;
    int lane;
    int32_t t0 = 0, req_base = 0, req_pages = 0;
    // paged: lane l holds the page id of page win_first + l, and nxt_id that
    // of page win_first + 32 + l, loaded one window ahead so that moving on to
    // the next window never waits for a global load.
    int32_t win_first = 0, win_id = 0, nxt_id = 0;
    // paged: the next box starts at row cur_off of the request's page cur_pg;
    // the cursor only moves forward within an item.
    int32_t cur_pg = 0, cur_off = 0;

    __device__ __forceinline__ TileSource(const SplitParams &p_, const CUtensorMap *k,
                                          const CUtensorMap *v, uint8_t *ring_, uint64_t *full_,
                                          int lane_)
        : p(p_), tm_k(k), tm_v(v), ring(ring_), full(full_), pol(l2_evict_first_policy()), lane(lane_)
    {
    }

    // An item of keys t0.. (relative to its request's first key); base and
    // pages locate the request (first key row, or first page-list entry).
    __device__ __forceinline__ void begin_item(int32_t t0_, int32_t base, int32_t pages)
    {
        t0 = t0_;
        req_base = base;
        req_pages = pages;
        if constexpr (kPaged) {
            win_first = -(1 << 30);   // far below page 0: the first lookup fills the window
            cur_pg = t0 / p.page_size;
            cur_off = t0 % p.page_size;
        }
    }

    __device__ __forceinline__ int32_t fetch_ids(int32_t first) const
    {
        return first + lane < req_pages ? __ldg(p.page_indices + req_base + first + lane) : 0;
    }

    // Physical page of the request's page `pg`; a page outside the pool is
    // reported (FD_ERR_DEVICE_BOUNDS) and page 0 read instead.
    __device__ __forceinline__ int32_t page_id(int32_t pg)
    {
        if (pg < win_first || pg >= win_first + 32) {
            win_id = pg == win_first + 32 ? nxt_id : fetch_ids(pg);
            win_first = pg;
            nxt_id = fetch_ids(pg + 32);
        }
        int32_t id = __shfl_sync(0xffffffffu, win_id, pg - win_first);
        if (id < 0 || id >= p.num_pages) {
            if (lane == 0)
                report(p.status, FD_ERR_DEVICE_BOUNDS);
            id = 0;
        }
        return id;
    }

    __device__ __forceinline__ int32_t next_box_row()
    {
        // Rows past the request's last key read whatever its last page holds
        // there; the consumers mask them.
        const int32_t y = page_id(min(cur_pg, req_pages - 1)) * p.page_size + cur_off;
        cur_off += SL::kBoxRows;
        if (cur_off >= p.page_size) {
            cur_off -= p.page_size;
            ++cur_pg;
        }
        return y;
    }

    // First rows (in K/V, or in the page pool) of the item's tile i: ya, and
    // yb for the second 16-row box of a paged tile.  The producer computes them
    // before it waits for the tile's stage, so that only the copies remain
    // once the stage is free.
    __device__ __forceinline__ void tile_rows(int i, int32_t &ya, int32_t &yb)
    {
        if constexpr (!kPaged) {
            ya = req_base + t0 + i * kTile;
        } else {
            ya = next_box_row();
            if constexpr (SL::kBoxRows < kTile)
                yb = next_box_row();
        }
    }

    // cp.async (INT4, every lane): the lane's share of the 16-byte chunks of
    // a tile's rows ya.. (yb.. for the second 16 rows of a paged tile) in both
    // tensors (rows past the end of K/V zero-filled) and the K and V scale of
    // row `lane`, into the stage at shared address dst.
    __device__ __forceinline__ void copy_direct(uint32_t dst, int kvh, int32_t ya, int32_t yb) const
    {
        constexpr int kChunks = SL::kRowBytes / 16;   // per key row
        const int64_t row_stride = (int64_t)p.num_kv_heads * SL::kRowBytes;
        const uint8_t *kb = p.k_data + kvh * SL::kRowBytes;
        const uint8_t *vb = p.v_data + kvh * SL::kRowBytes;
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
            const int idx = lane + 32 * i, r = idx / kChunks, c = idx % kChunks;
            const int32_t row = SL::kBoxRows == kTile || r < 16 ? ya + r : yb + (r - 16);
            const bool in = row < p.kv_rows;
            const int64_t off = (int64_t)(in ? row : 0) * row_stride + c * 16;
            const uint32_t so = SL::chunk_offset(r, c);
            cp_async_16(dst + so, kb + off, in ? 16 : 0, pol);
            cp_async_16(dst + SL::kTensorBytes + so, vb + off, in ? 16 : 0, pol);
        }
        const int32_t row = SL::kBoxRows == kTile || lane < 16 ? ya + lane : yb + (lane - 16);
        const bool in = row < p.kv_rows;
        const int64_t si = (int64_t)kvh * p.kv_rows + (in ? row : 0);
        cp_async_4(dst + SL::kKsOff + 4 * lane, p.k_scale + si, in ? 4 : 0);
        cp_async_4(dst + SL::kVsOff + 4 * lane, p.v_scale + si, in ? 4 : 0);
    }

    // Put stream tile g (KV head kvh) into stage g % NS.
    //  TMA (lane 0): per tensor and per box of rows -- bf16, one 3-D box of
    //    both 64-column halves; FP8, one 2-D box of the rows' 128 bytes.
    //  cp.async (INT4, every lane): the lane's share of the 16-byte chunks of
    //    both tensors (rows past the end of K/V zero-filled) and the K and V
    //    scale of row `lane`, then one arrival once its copies have landed.
    __device__ __forceinline__ void issue(int g, int kvh, int32_t ya, int32_t yb) const
    {
        const int s = g % NS;
        const uint32_t bar = smem_addr(&full[s]);
        const uint32_t dst = smem_addr(ring + s * SL::kBytes);
        if constexpr (SL::kDirect) {
            copy_direct(dst, kvh, ya, yb);
            cp_async_mbar_arrive(bar);
        } else {
            mbar_arrive_expect_tx(bar, SL::kBytes);
            if constexpr (SL::kFp8) {
                const int32_t x = kvh * kHeadDim;
                tma_load_2d(dst, tm_k, x, ya, bar, pol);
                tma_load_2d(dst + SL::kTensorBytes, tm_v, x, ya, bar, pol);
                if constexpr (SL::kBoxRows < kTile) {
                    tma_load_2d(dst + 16 * 128, tm_k, x, yb, bar, pol);
                    tma_load_2d(dst + SL::kTensorBytes + 16 * 128, tm_v, x, yb, bar, pol);
                }
            } else {
                tma_load_3d(dst, tm_k, 0, ya, 2 * kvh, bar, pol);
                tma_load_3d(dst + SL::kTensorBytes, tm_v, 0, ya, 2 * kvh, bar, pol);
                if constexpr (SL::kBoxRows < kTile) {
                    tma_load_3d(dst + SL::kBlockStride, tm_k, 0, yb, 2 * kvh, bar, pol);
                    tma_load_3d(dst + SL::kTensorBytes + SL::kBlockStride, tm_v, 0, yb, 2 * kvh, bar,
                                pol);
                }
            }
        }
    }
};

// Locate split j of the plan (warp-collective) and check it against the
// buffers: key range [t0, t1) relative to the request's first key.
template <bool PAGED>
__device__ __forceinline__ bool item_range(const SplitParams &p, const SplitCoord &c, bool found,
                                           int32_t &t0, int32_t &t1)
{
    t0 = t1 = 0;
    if (!found)
        return false;
    const int32_t len = split_len_for(c.len, c.splits);
    t0 = c.s * len;
    t1 = min(t0 + len, c.len);
    // under the device-side plan an empty request is one split of no keys
    const bool empty_item = p.device_plan && c.len == 0 && c.splits == 1;
    return (t0 < t1 || empty_item) && c.base >= 0 &&
           (PAGED ? c.base + c.pages <= p.num_page_entries : c.base + c.len <= p.total_tokens) &&
           partial_row(c.prefix, p.num_qo_heads, p.num_qo_heads - 1, c.splits, c.splits - 1) <
               p.num_partial_rows;
}

__device__ __forceinline__ void write_desc(volatile int *d, const SplitCoord &c, int32_t t0,
                                           int32_t t1, int kvh, int gt0, int state, float ks = 1.f,
                                           float vs = 1.f)
{
    d[kDKs] = __float_as_int(ks);
    d[kDVs] = __float_as_int(vs);
    d[kDB] = c.b;
    d[kDPrefix] = c.prefix;
    d[kDSplits] = c.splits;
    d[kDS] = c.s;
    d[kDT0] = t0;
    d[kDT1] = t1;
    d[kDKvh] = kvh;
    d[kDGt0] = gt0;
    d[kDBase] = c.base;
    d[kDState] = state;
}

__device__ __forceinline__ KeyIndex key_index(const SplitParams &p, bool paged)
{
    return p.indptr_in_params ? KeyIndex{p.indptr_param, paged ? p.last_len_param : nullptr, p.page_size}
                              : KeyIndex{p.kv_indptr, p.kv_last_len, p.page_size};
}

// Q fragments (A operand of S = Q K^T) for the 8 k-steps of 16 dims from the
// G bf16 query rows at `qrows` (global or shared); rows g >= G and the padding
// rows 8-15 are zero.  Returns the factor the logits must be multiplied by.
// COLS: the same registers as the B operand of S^T = K Q^T, column g holding
// query row g mod G (every column filled).
//  bf16: qa[c] = dims 16c + 2t4 (+1) and 16c + 8 + 2t4 (+1), as stored; 1.
//  FP8 (f16 MMA): qa[c] = dims 16c + 4t4 (+1) and 16c + 4t4 + 2 (+3), the order
//    consume_tile reads K in.  Each row is first scaled by the power of two
//    that puts its largest magnitude in [2^8, 2^9), so every bf16 value of the
//    row converts to f16 exactly (values below 2^-22 of the row's maximum
//    round in f16's subnormal range); returns the inverse power.
//  INT4 (f16 MMA): qa[2c + h] = dims 32c + 8t4 + 2h (+4) and 32c + 8t4 + 2h + 1
//    (+4), the order consume_tile reads K in, each row scaled into f16 as for
//    FP8; returns the inverse power.
template <int G, int DT, bool GLOBAL, bool COLS = false>
__device__ __forceinline__ float load_q(const uint16_t *qrows, int lane, uint32_t (&qa)[8][2])
{
    const int g_row = COLS ? (lane >> 2) & (G - 1) : lane >> 2, t4 = lane & 3;
    const bool valid = COLS || g_row < G;
    if constexpr (DT == kKvInt4) {
        const uint4 *row = reinterpret_cast<const uint4 *>(qrows + (valid ? g_row : 0) * kHeadDim);
        uint4 raw[4];
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            raw[c] = make_uint4(0u, 0u, 0u, 0u);   // dims 32c + 8t4 .. +7
            if constexpr (GLOBAL) {
                if (valid)
                    raw[c] = __ldg(row + 4 * c + t4);
            } else {
                if (valid)
                    raw[c] = row[4 * c + t4];
            }
            const uint32_t w[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 a = bf16x2_to_float2(w[i]);
                amax = fmaxf(amax, fmaxf(fabsf(a.x), fabsf(a.y)));
            }
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        int sh = 0;
        if (amax > 0.f) {
            int e;
            frexpf(amax, &e);
            sh = min(max(9 - e, -100), 100);
        }
        const float up = __int_as_float((127 + sh) << 23);
        auto f16pair = [&](uint32_t pair) {   // a bf16x2 pair -> f16x2, times 2^sh (exact)
            const float2 a = bf16x2_to_float2(pair);
            return pack_f16(a.x * up, a.y * up);
        };
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            qa[2 * c][0] = f16pair(__byte_perm(raw[c].x, raw[c].z, 0x5410));       // dims +0, +4
            qa[2 * c][1] = f16pair(__byte_perm(raw[c].x, raw[c].z, 0x7632));       // dims +1, +5
            qa[2 * c + 1][0] = f16pair(__byte_perm(raw[c].y, raw[c].w, 0x5410));   // dims +2, +6
            qa[2 * c + 1][1] = f16pair(__byte_perm(raw[c].y, raw[c].w, 0x7632));   // dims +3, +7
        }
        return __int_as_float((127 - sh) << 23);
    } else if constexpr (DT == kKvFp8) {
        const uint2 *row = reinterpret_cast<const uint2 *>(qrows + (valid ? g_row : 0) * kHeadDim);
        uint2 raw[8];
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if constexpr (GLOBAL)
                raw[c] = valid ? __ldg(row + 4 * c + t4) : make_uint2(0u, 0u);
            else
                raw[c] = valid ? row[4 * c + t4] : make_uint2(0u, 0u);
            const float2 a = bf16x2_to_float2(raw[c].x), b = bf16x2_to_float2(raw[c].y);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y))));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        int sh = 0;
        if (amax > 0.f) {
            int e;
            frexpf(amax, &e);   // amax in [2^(e-1), 2^e)
            sh = min(max(9 - e, -100), 100);
        }
        const float up = __int_as_float((127 + sh) << 23);   // 2^sh, exact
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float2 a = bf16x2_to_float2(raw[c].x), b = bf16x2_to_float2(raw[c].y);
            qa[c][0] = pack_f16(a.x * up, a.y * up);
            qa[c][1] = pack_f16(b.x * up, b.y * up);
        }
        return __int_as_float((127 - sh) << 23);   // 2^-sh
    } else {
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(qrows) + (valid ? g_row : 0) * (kHeadDim / 2);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            if constexpr (GLOBAL) {
                qa[kk][0] = valid ? __ldg(qrow + kk * 8 + t4) : 0u;       // cols 16kk + 2t4 (+1)
                qa[kk][1] = valid ? __ldg(qrow + kk * 8 + 4 + t4) : 0u;   // cols 16kk + 8 + 2t4 (+1)
            } else {
                qa[kk][0] = valid ? qrow[kk * 8 + t4] : 0u;
                qa[kk][1] = valid ? qrow[kk * 8 + 4 + t4] : 0u;
            }
        }
        return 1.f;
    }
}

// Consumer warp `warp`: put its online-softmax state for one item (O rows g
// and g+8 summed and multiplied by vscale, running max, row sum) into a state
// buffer, O in dim order (consume_tile's FP8 and INT4 column orders are undone
// here).
template <int G, int NC, int DT>
__device__ __forceinline__ void write_state(uint8_t *state, int warp, int lane,
                                            const float (&o_acc)[16][4], float m_run, float l_part,
                                            float vscale)
{
    float *comb_acc = reinterpret_cast<float *>(state);
    float *comb_m = comb_acc + NC * G * kHeadDim;
    float *comb_l = comb_m + NC * G;
    const int g_row = lane >> 2, t4 = lane & 3;
    float l_tot = l_part;
    l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 1);
    l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 2);
    if (g_row < G) {
        if constexpr (DT == kKvInt4) {
            float *dst = comb_acc + (warp * G + g_row) * kHeadDim + 8 * t4;
#pragma unroll
            for (int c = 0; c < 4; ++c) {   // dims 32c + 8t4 + (0..3), then + (4..7)
                const int n = 4 * c;
                *reinterpret_cast<float4 *>(dst + 32 * c) = make_float4(
                    (o_acc[n][0] + o_acc[n][2]) * vscale, (o_acc[n + 1][0] + o_acc[n + 1][2]) * vscale,
                    (o_acc[n + 2][0] + o_acc[n + 2][2]) * vscale, (o_acc[n + 3][0] + o_acc[n + 3][2]) * vscale);
                *reinterpret_cast<float4 *>(dst + 32 * c + 4) = make_float4(
                    (o_acc[n][1] + o_acc[n][3]) * vscale, (o_acc[n + 1][1] + o_acc[n + 1][3]) * vscale,
                    (o_acc[n + 2][1] + o_acc[n + 2][3]) * vscale, (o_acc[n + 3][1] + o_acc[n + 3][3]) * vscale);
            }
        } else if constexpr (DT == kKvFp8) {
            float *dst = comb_acc + (warp * G + g_row) * kHeadDim + 4 * t4;
#pragma unroll
            for (int c = 0; c < 8; ++c)   // dims 16c + 4t4 + (0, 1, 2, 3)
                *reinterpret_cast<float4 *>(dst + 16 * c) = make_float4(
                    (o_acc[2 * c][0] + o_acc[2 * c][2]) * vscale,
                    (o_acc[2 * c + 1][0] + o_acc[2 * c + 1][2]) * vscale,
                    (o_acc[2 * c][1] + o_acc[2 * c][3]) * vscale,
                    (o_acc[2 * c + 1][1] + o_acc[2 * c + 1][3]) * vscale);
        } else {
            float *dst = comb_acc + (warp * G + g_row) * kHeadDim + 2 * t4;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                *reinterpret_cast<float2 *>(dst + 8 * n) =
                    make_float2(o_acc[n][0] + o_acc[n][2], o_acc[n][1] + o_acc[n][3]);
        }
        if (t4 == 0) {
            comb_m[warp * G + g_row] = m_run;
            comb_l[warp * G + g_row] = l_tot;
        }
    }
}

// A consumer warp's online-softmax state for one item in the row form
// (S = Q K^T, the query rows in the MMA's rows; every K/V type and group
// size): begin() resets it with the logit factor of the lane's query row,
// tile() takes one stage, write() hands the state to the CTA's combine.
template <int G, int KV, int DT>
struct RowConsumer {
    float o_acc[16][4];
    float m_run, l_part, qk;
    int v_exp;   // INT4: see consume_tile

    __device__ __forceinline__ void begin(float qk_row, int)
    {
        qk = qk_row;
        m_run = -INFINITY;
        l_part = 0.f;
        v_exp = kNoExp;
#pragma unroll
        for (int n = 0; n < 16; ++n)
            o_acc[n][0] = o_acc[n][1] = o_acc[n][2] = o_acc[n][3] = 0.f;
    }
    __device__ __forceinline__ void tile(uint32_t st, int n_valid, const uint32_t (&qa)[8][2], int lane)
    {
        consume_tile<KV, DT>(st, n_valid, qa, qk, lane, m_run, l_part, o_acc, v_exp);
    }
    // fp8_vscale: the head's V scale (FP8 K/V; ignored otherwise)
    template <int NC>
    __device__ __forceinline__ void write(uint8_t *state, int warp, int lane, float fp8_vscale) const
    {
        const float vscale = DT == kKvInt4 ? (v_exp == kNoExp ? 1.f : pow2i(v_exp)) : fp8_vscale;
        write_state<G, NC, DT>(state, warp, lane, o_acc, m_run, l_part, vscale);
    }
};

// The column form for FP8 and INT4 K/V with G <= 4: S^T = K Q^T and
// O^T = V^T P^T, the tile's keys (scores) and the head's dims (output) in the
// MMA's 16 rows and the query heads in its 8 columns, so every MMA row carries
// data: half the MMAs and half the output accumulators of the row form, whose
// padding rows 8-15 carry nothing in Q K^T.  Column n < G is head n with the
// hi part of its P V weights, column G + n the same head with the lo part (the
// f16 weights keep about 22 bits, as in the row form), columns >= 2G repeat
// heads and are dropped.  Q fills every column (load_q<..., COLS>), so a lo
// column computes the same scores, maxima and sums as its hi column in its
// own lanes and needs no exchange until write().
//  Lane (g, t4) holds scores of keys g, g + 8, 16 + g, 24 + g for columns
//  2t4 and 2t4 + 1 (m[e], l[e], qk[e]: column 2t4 + e).  P^T as the B operand
//  is the transpose of the score fragments (movmatrix).  Output m-block n
//  holds, for the lane's two columns, dims dim0(n, g) (c0, c1) and
//  dim0(n, g) + 1 (c2, c3): INT4 n = 2c + jp -> 32c + 4g + 2jp, FP8 n = c ->
//  16c + 2g (the orders ldmatrix.trans and the widenings give).
template <int G, int KV, int DT>
struct ColumnConsumer {
    static_assert(G == 1 || G == 2 || G == 4, "column form: two columns per head");
    static_assert(DT == kKvFp8 || DT == kKvInt4, "column form: FP8 or INT4 K/V");
    static constexpr bool kInt4 = DT == kKvInt4;
    float o[8][4];
    float m[2], l[2], qk[2], lo[2];
    int v_exp;   // INT4: see consume_tile

    static __device__ __forceinline__ int dim0(int n, int g)
    {
        return kInt4 ? 32 * (n >> 1) + 4 * g + 2 * (n & 1) : 16 * n + 2 * g;
    }

    __device__ __forceinline__ void begin(float qk_row, int lane)
    {
        const int t4 = lane & 3;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = 2 * t4 + e;   // this lane's column: head n mod G, from lane 4 (n mod G)
            qk[e] = __shfl_sync(0xffffffffu, qk_row, (n & (G - 1)) * 4);
            lo[e] = n >= G && n < 2 * G ? 1.f : 0.f;
            m[e] = -INFINITY;
            l[e] = 0.f;
        }
        v_exp = kNoExp;
#pragma unroll
        for (int n = 0; n < 8; ++n)
            o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    }

    __device__ __forceinline__ void tile(uint32_t st, int n_valid, const uint32_t (&qa)[8][2], int lane)
    {
        using S = Stage<KV, DT>;
        const int g = lane >> 2, lr = lane & 7, lm = lane >> 3;

        // FP8: V rows past the last key zeroed, as in consume_tile
        if constexpr (!kInt4) {
            if (n_valid < kTile) {
                constexpr int kChunks = S::kRowBytes / 16;
                const uint32_t vt = st + S::kTensorBytes;
                for (int idx = lane; idx < (kTile - n_valid) * kChunks; idx += 32)
                    sts_zero16(vt + S::chunk_offset(n_valid + idx / kChunks, idx % kChunks));
                fence_proxy_async_shared();
                __syncwarp();
            }
        }

        // ---- S^T = K Q^T: m-block mb = keys 16 mb + g (rows g), 16 mb + 8 + g
        // (rows g + 8); ldmatrix gives lane (g, t4) word t4 of each 16-byte
        // chunk of a key row, widened in the dim order load_q puts Q in.
        float s[2][4];
#pragma unroll
        for (int mb = 0; mb < 2; ++mb) {
            s[mb][0] = s[mb][1] = s[mb][2] = s[mb][3] = 0.f;
            const int r0 = 16 * mb + lr, r1 = r0 + 8;
            if constexpr (kInt4) {
                // chunk c = dims 32c .. +31; k-step 2c + h takes dims
                // 32c + 8t4 + 2h (+4) at k 2t4 (+1) and + 2h + 1 (+4) at k 2t4 + 8 (+9)
                uint32_t k0[4], k1[4];
                ldsm_x4(st + r0 * 64 + ((lm ^ ((r0 >> 1) & 3)) << 4), k0);
                ldsm_x4(st + r1 * 64 + ((lm ^ ((r1 >> 1) & 3)) << 4), k1);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t a[4], b[4];   // [j]: dims 32c + 8t4 + j and + 4 of keys 16mb + g, + 8
                    int4x8_to_f16x2x4(k0[c], a);
                    int4x8_to_f16x2x4(k1[c], b);
                    mma_f16(s[mb], a[0], b[0], a[1], b[1], qa[2 * c][0], qa[2 * c][1]);
                    mma_f16(s[mb], a[2], b[2], a[3], b[3], qa[2 * c + 1][0], qa[2 * c + 1][1]);
                }
            } else {
                // chunk c = dims 16c .. +15 = k-step c: dims 16c + 4t4 (+1) at
                // k 2t4 (+1), 16c + 4t4 + 2 (+3) at k 2t4 + 8 (+9)
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                    uint32_t k0[4], k1[4];
                    ldsm_x4(st + r0 * 128 + (((4 * hc + lm) ^ lr) << 4), k0);
                    ldsm_x4(st + r1 * 128 + (((4 * hc + lm) ^ lr) << 4), k1);
#pragma unroll
                    for (int mc = 0; mc < 4; ++mc) {
                        uint32_t a0, a1, a2, a3;
                        e4m3x4_to_f16x2x2(k0[mc], a0, a2);
                        e4m3x4_to_f16x2x2(k1[mc], a1, a3);
                        mma_f16(s[mb], a0, a1, a2, a3, qa[4 * hc + mc][0], qa[4 * hc + mc][1]);
                    }
                }
            }
        }

        // ---- online softmax per column over the warp's 32 keys (the 8 lanes
        // of a t4 hold them: reductions over g); INT4: the lane's 4 keys' K
        // and V scales, and the V exponent as in the row form (consume_tile)
        const uint32_t ks_base = st + S::kKsOff, vs_base = st + S::kVsOff;
        float x[2][4], vs[2][2];
        float mt0 = -INFINITY, mt1 = -INFINITY, vmax = 0.f;
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int key = 16 * mb + 8 * hf + g;
                const bool ok = key < n_valid;
                const float ksc = kInt4 ? lds_f32(ks_base + 4 * key) : 1.f;
                const float v0 = ok ? s[mb][2 * hf] * ksc * qk[0] : -INFINITY;
                const float v1 = ok ? s[mb][2 * hf + 1] * ksc * qk[1] : -INFINITY;
                x[mb][2 * hf] = v0;
                x[mb][2 * hf + 1] = v1;
                mt0 = fmaxf(mt0, v0);
                mt1 = fmaxf(mt1, v1);
                if constexpr (kInt4) {
                    vs[mb][hf] = ok ? lds_f32(vs_base + 4 * key) : 0.f;
                    vmax = fmaxf(vmax, fabsf(vs[mb][hf]));
                }
            }
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, sh));
            mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, sh));
            if constexpr (kInt4)
                vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, sh));
        }
        const float m0 = fmaxf(m[0], mt0), m1 = fmaxf(m[1], mt1);
        float os0 = exp2f(m[0] - m0), os1 = exp2f(m[1] - m1);
        m[0] = m0;
        m[1] = m1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                x[mb][2 * hf] = exp2f(x[mb][2 * hf] - m0);
                x[mb][2 * hf + 1] = exp2f(x[mb][2 * hf + 1] - m1);
                ps0 += x[mb][2 * hf];
                ps1 += x[mb][2 * hf + 1];
            }
        l[0] = fmaf(l[0], os0, ps0);
        l[1] = fmaf(l[1], os1, ps1);
        if constexpr (kInt4) {
            if (!(vmax <= 0.f)) {   // a nonzero, inf or NaN scale: vmax < 2^e
                const int e = ((__float_as_int(vmax) >> 23) & 0xFF) - 126;
                if (e > v_exp) {
                    const float f = pow2i(v_exp - e);   // 0 when v_exp is still kNoExp
                    os0 *= f;
                    os1 *= f;
                    v_exp = e;
                }
            }
        }
        if (__any_sync(0xffffffffu, os0 != 1.f || os1 != 1.f)) {
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                o[n][0] *= os0;
                o[n][1] *= os1;
                o[n][2] *= os0;
                o[n][3] *= os1;
            }
        }

        // ---- P^T (B operand of k-step mb: keys 16 mb + 2t4 (+1) in b0,
        // + 8 in b1, column g): the weights (INT4: p * v_scale * 2^-v_exp) as
        // f16 (hi columns) or their remainder after f16 (lo columns), packed
        // per key row and transposed
        const float vinv = kInt4 && v_exp != kNoExp ? pow2i(-v_exp) : 1.f;
        uint32_t pt[2][2];
#pragma unroll
        for (int mb = 0; mb < 2; ++mb)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float p0 = x[mb][2 * hf], p1 = x[mb][2 * hf + 1];
                if constexpr (kInt4) {
                    const float w = vs[mb][hf] * vinv;
                    p0 *= w;
                    p1 *= w;
                }
                p0 = fmaf(-lo[0], f16_round(p0), p0);
                p1 = fmaf(-lo[1], f16_round(p1), p1);
                pt[mb][hf] = movmatrix_trans(pack_f16(p0, p1));
            }

        // ---- O^T += V^T P^T: k-step ks = keys 16 ks .. +15.  ldmatrix.trans
        // matrix lm = keys 16 ks + 8 (lm & 1) .. +7 of chunk 2 cp + (lm >> 1)
        const uint32_t vt = st + S::kTensorBytes;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const int r = 16 * ks + 8 * (lm & 1) + lr;
            if constexpr (kInt4) {
                // lane (g, t4): dims 32c + 4g .. +3 of keys 2t4, 2t4 + 1 in one
                // word, widened to (key 2t4, key 2t4 + 1) pairs per dim;
                // m-block 2c + jp = dims + 2jp (rows g), + 2jp + 1 (rows g + 8)
#pragma unroll
                for (int cp = 0; cp < 2; ++cp) {
                    uint32_t vb[4];
                    ldsm_x4_trans(vt + r * 64 + (((2 * cp + (lm >> 1)) ^ ((r >> 1) & 3)) << 4), vb);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {   // chunk c = 2 cp + h
                        const int c = 2 * cp + h;
                        uint32_t a[4], b[4];        // [j]: dim 32c + 4g + j of keys 2t4, 2t4 + 1 (+8 in b)
                        int4x8_to_f16x2x4(vb[2 * h], a);
                        int4x8_to_f16x2x4(vb[2 * h + 1], b);
#pragma unroll
                        for (int jp = 0; jp < 2; ++jp)
                            mma_f16(o[2 * c + jp], a[2 * jp], a[2 * jp + 1], b[2 * jp], b[2 * jp + 1],
                                    pt[ks][0], pt[ks][1]);
                    }
                }
            } else {
                // lane (g, t4): dims 16c + 2g, + 1 of keys 2t4, 2t4 + 1,
                // regrouped per dim; m-block c = dims 16c + 2g (rows g), + 1
                // (rows g + 8)
#pragma unroll
                for (int cp = 0; cp < 4; ++cp) {
                    uint32_t vb[4];
                    ldsm_x4_trans(vt + r * 128 + (((2 * cp + (lm >> 1)) ^ lr) << 4), vb);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {   // chunk c = 2 cp + h
                        uint32_t a0, a1, a2, a3;
                        e4m3x4_to_f16x2x2(__byte_perm(vb[2 * h], 0u, 0x3120), a0, a1);
                        e4m3x4_to_f16x2x2(__byte_perm(vb[2 * h + 1], 0u, 0x3120), a2, a3);
                        mma_f16(o[2 * cp + h], a0, a1, a2, a3, pt[ks][0], pt[ks][1]);
                    }
                }
            }
        }
    }

    // O of head n = hi column n + lo column G + n (lane ^ G/2, or the lane's
    // other column for G = 1), times the V scale (INT4: 2^v_exp; FP8: the
    // head's); the row sums summed over g.
    template <int NC>
    __device__ __forceinline__ void write(uint8_t *state, int warp, int lane, float fp8_vscale) const
    {
        float *comb_acc = reinterpret_cast<float *>(state);
        float *comb_m = comb_acc + NC * G * kHeadDim;
        float *comb_l = comb_m + NC * G;
        const int g = lane >> 2, t4 = lane & 3;
        const float vscale = !kInt4 ? fp8_vscale : v_exp == kNoExp ? 1.f : pow2i(v_exp);
        float lt[2] = {l[0], l[1]};
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            lt[0] += __shfl_xor_sync(0xffffffffu, lt[0], sh);
            lt[1] += __shfl_xor_sync(0xffffffffu, lt[1], sh);
        }
        if constexpr (G == 1) {
            if (t4 == 0) {
                float *dst = comb_acc + warp * kHeadDim;
#pragma unroll
                for (int n = 0; n < 8; ++n)
                    *reinterpret_cast<float2 *>(dst + dim0(n, g)) =
                        make_float2((o[n][0] + o[n][1]) * vscale, (o[n][2] + o[n][3]) * vscale);
                if (g == 0) {
                    comb_m[warp] = m[0];
                    comb_l[warp] = lt[0];
                }
            }
        } else {
            float tot[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    tot[n][i] = o[n][i] + __shfl_xor_sync(0xffffffffu, o[n][i], G / 2);
            if (t4 < G / 2) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {   // head 2t4 + e
                    float *dst = comb_acc + (warp * G + 2 * t4 + e) * kHeadDim;
#pragma unroll
                    for (int n = 0; n < 8; ++n)
                        *reinterpret_cast<float2 *>(dst + dim0(n, g)) =
                            make_float2(tot[n][e] * vscale, tot[n][2 + e] * vscale);
                    if (g == 0) {
                        comb_m[warp * G + 2 * t4 + e] = m[e];
                        comb_l[warp * G + 2 * t4 + e] = lt[e];
                    }
                }
            }
        }
    }
};

// FP8 and INT4 K/V with G <= 4 take the column form.
template <int G, int DT>
constexpr bool kColumnForm = (DT == kKvFp8 || DT == kKvInt4) && G <= 4;
template <int G, int KV, int DT>
using Consumer = std::conditional_t<kColumnForm<G, DT>, ColumnConsumer<G, KV, DT>, RowConsumer<G, KV, DT>>;

// Combine the NC consumer states in `state` (NW warps, thread `tid` of
// NW * 32) into the item's normalised partial rows, or, when `direct`, into
// the request's O / LSE rows (stage 2 fused and the request has one split).
template <int G, int NC, int NW>
__device__ __forceinline__ void combine_states(const SplitParams &p, const Item &it, const uint8_t *state,
                                               int tid, bool direct)
{
    const float *comb_acc = reinterpret_cast<const float *>(state);
    const float *comb_m = comb_acc + NC * G * kHeadDim;
    const float *comb_l = comb_m + NC * G;
    for (int idx = tid; idx < G * 32; idx += NW * 32) {
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
            const int64_t row = (int64_t)it.b * p.num_qo_heads + it.kvh * G + g;
            *reinterpret_cast<float4 *>(p.o + row * kHeadDim + 4 * c4) = o;
            if (c4 == 0)
                p.lse[row] = lse_nat;
        } else {
            const int64_t row = partial_row(it.prefix, p.num_qo_heads, it.kvh * G + g, it.splits, it.s);
            *reinterpret_cast<float4 *>(p.partial_o + row * kHeadDim + 4 * c4) = o;
            if (c4 == 0)
                p.partial_lse[row] = lse_nat;
        }
    }
}

// End of one item, run by NW warps (thread `tid` of NW * 32) behind barrier
// BAR: NW = 1, BAR = -1 is the epilogue warp while the others stream the next
// items; NW = all warps, BAR = 0 is the whole CTA after its last item.
// Combines the NC consumer states in `state` into the item's normalised
// partial -- or O / LSE directly when stage 2 is fused and the request has one
// split -- calls combined() once the state buffer has been read, then takes
// the group's ticket and, as the group's last CTA, runs stage 2 (using
// `merge_scratch` when NW > 1).
template <int G, int NC, int NW, int BAR, typename Combined>
__device__ __forceinline__ void finish_item(const SplitParams &p, const Item &it, const uint8_t *state,
                                            uint8_t *merge_scratch, volatile int *misc, int tid,
                                            Combined combined)
{
    combine_states<G, NC, NW>(p, it, state, tid, p.fuse_merge && it.splits == 1);
    combined();

    if (p.fuse_merge && it.splits > 1) {
        // Ticket: the last CTA of the (request, KV head) group to finish merges
        // the group (stage 2).  The ticket add is acquire-release at GPU scope:
        // it publishes this item's partials (made visible to thread 0 by the
        // barrier) and lets the last CTA see everyone else's; that CTA also
        // resets the ticket for the next call.
        group_sync<BAR>();
        if (tid == 0) {
            cuda::atomic_ref<int, cuda::thread_scope_device> ticket(
                p.counters[(int64_t)it.b * p.num_kv_heads + it.kvh]);
            const int prev = ticket.fetch_add(1, cuda::memory_order_acq_rel);
            const bool last = prev == it.splits - 1;
            if (last)
                ticket.store(0, cuda::memory_order_relaxed);
            misc[kLast] = last;
        }
        group_sync<BAR>();
        if (misc[kLast])
            merge_group<G, NW, BAR>(p, it.prefix, it.splits, it.b, it.kvh, tid >> 5, tid & 31,
                                    reinterpret_cast<float *>(merge_scratch));
    }
    group_sync<BAR>();
}

// The one-item kernel's end of a split of a request with several splits, on
// host-planned fused calls (p.flags set), run by the whole CTA (NW warps).
// Stage 2 is spread over the group's last min(G, splits) CTAs to arrive, one
// or more heads each, so that no single SM pulls the whole group's partials
// from L2: `ticket` is this CTA's arrival order in the group (a relaxed add
// taken by thread `ticket_tid` when its stream ended).  Every CTA writes its partial rows and
// publishes them by a release store of the call's token into its flag; a
// merging CTA waits (bounded by the plan's timeout) until every split of the
// group has published -- the CTAs that arrived before it are running, and at
// most G CTAs of a group wait -- then merges heads k, k + mergers, ... in the
// same fixed split order as a single merger would.  The last arrival resets
// the ticket for the next call; the flags need no reset (tokens differ).
template <int G, int NC, int NW>
__device__ __forceinline__ void finish_item_spread(const SplitParams &p, const Item &it, const uint8_t *state,
                                                   uint8_t *merge_scratch, volatile int *misc, int tid,
                                                   int ticket, int ticket_tid)
{
    combine_states<G, NC, NW>(p, it, state, tid, false);
    __syncthreads();
    const int total_splits = p.num_work / p.num_kv_heads;
    int *flags = p.flags + (int64_t)it.kvh * total_splits + it.prefix;
    if (tid == ticket_tid) {
        if (ticket == it.splits - 1)   // every CTA of the group has taken its ticket
            cuda::atomic_ref<int, cuda::thread_scope_device>(
                p.counters[(int64_t)it.b * p.num_kv_heads + it.kvh])
                .store(0, cuda::memory_order_relaxed);
        st_release_gpu(flags + it.s, p.token);   // this split's partial rows are written
        misc[kLast] = ticket;
    }
    __syncthreads();
    const int mergers = min(G, it.splits);
    const int k = it.splits - 1 - misc[kLast];
    if (k < 0 || k >= mergers)
        return;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        int ready = 1;
        for (int s = tid; s < it.splits; s += NW * 32)
            ready &= ld_acquire_gpu(flags + s) == p.token;
        if (__syncthreads_and(ready))
            break;
        const bool late = (int64_t)(global_timer_ns() - t0) > p.timeout_ns;
        if (__syncthreads_or(late)) {
            if (tid == 0)
                report(p.status, FD_ERR_TIMEOUT);
            return;
        }
    }
    for (int h = k; h < G; h += mergers) {
        // head h of the group: its split rows are consecutive, as for G = 1
        merge_group<1, NW, 0>(p, it.prefix, it.splits, it.b, it.kvh * G + h, tid >> 5, tid & 31,
                              reinterpret_cast<float *>(merge_scratch));
        __syncthreads();   // the scratch is reused by the next head
    }
}

// L2 prefetch of one TMA box of K and one of V (KV head kvh) from row y:
// the rows one stage copy of that box would read.
template <class SG>
__device__ __forceinline__ void prefetch_box(const CUtensorMap *tm_k, const CUtensorMap *tm_v, int kvh,
                                             int32_t y)
{
    if constexpr (SG::kFp8) {
        tma_prefetch_l2_2d(tm_k, kvh * kHeadDim, y);
        tma_prefetch_l2_2d(tm_v, kvh * kHeadDim, y);
    } else {
        tma_prefetch_l2_3d(tm_k, 0, y, 2 * kvh);
        tma_prefetch_l2_3d(tm_v, 0, y, 2 * kvh);
    }
}

// One item per CTA: the grid is the items, all resident at once (the plan
// fits one wave).  Warp NC produces, warps 0..NC-1 consume, and the whole CTA
// closes the item.
template <int G, int NC, int NS, int MIN_CTAS, int KV, int DT>
__global__ void __launch_bounds__((NC + 1) * 32, MIN_CTAS)
    split_kv_kernel(const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ SplitParams p)
{
    using SG = Stage<KV, DT>;
    using L = SingleLayout<G, NC, NS, SG::kBytes>;
    constexpr bool paged = KV != kKvRagged;
    constexpr bool warp_loop = paged || SG::kDirect;   // the whole producer warp runs the issue loop
    // Ragged FP8 and INT4: each consumer warp refills its own stages (see the
    // consumers); INT4 also makes its first copies itself.
    constexpr bool self_fill = !paged && DT == kKvInt4;
    constexpr bool self_refill = !paged && DT != kKvBf16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    volatile int *desc = reinterpret_cast<volatile int *>(smem + L::kOffDesc);
    volatile int *misc = reinterpret_cast<volatile int *>(smem + L::kOffMisc);
    volatile int *fills = reinterpret_cast<volatile int *>(smem + L::kOffFills);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = blockIdx.x % p.num_kv_heads;
    // The inputs may come from the preceding grid in the stream: wait for it
    // before touching global memory (the launch itself overlaps its tail).
    // When kv_indptr is in the launch parameters, the producer warp locates
    // its split before that wait.
    const bool early_derive = p.indptr_in_params && warp == NC;
    if (!early_derive)
        griddep_wait();

    float vscale = 1.f;              // FP8: the head's V scale
    Consumer<G, KV, DT> cs;          // consumer warps: set up by begin()

    if (warp == NC) {
        // ---------------------------------------------------------- producer
        // Set up the barriers (shared memory only, so before the wait for the
        // preceding grid), locate the split (the host planner's rule) and put
        // the first NS tiles in flight before the CTA barrier.  With the paged
        // layout the whole warp runs the issue loop; lane 0 issues the barrier
        // operations and the copies.
        if (lane == 0) {
            for (int s = 0; s < NS; ++s) {
                mbar_init(smem_addr(&bars[s]), SG::kFullArrivals);   // full: producer arrive(s) + bytes
                mbar_init(smem_addr(&bars[NS + s]), 1);   // empty: the stage's consumer warp
            }
            fence_mbar_init();
        }
        SplitCoord c{};
        const bool found = derive_split(key_index(p, paged), p.batch, p.chunk,
                                        blockIdx.x / p.num_kv_heads, false, c, p.device_plan);
        // Prologue for a split longer than the ring, while the preceding grid
        // may still run: the first kPrologueBytes of the split are prefetched
        // into L2, and the next grid may launch now.  Back to back, a call's
        // CTAs then take the SM slots of this call's finished CTAs and pull
        // their first tiles into L2 while this call's stream ends and its
        // stragglers merge -- DRAM time that would otherwise sit idle -- and
        // their own stream starts from L2 once the wait returns.  Every byte is
        // still read from DRAM once per call.  A short split (the ring holds
        // all of it) does neither: its copies follow at once, and the
        // prefetches would only delay them.  Measured (interleaved A/B): 64k
        // step 43.7 -> 40.0 us, 128k 79.7 -> 76.5 us, FP8 64k 27.4 -> 26.0 us;
        // 192 KB and 384 KB per CTA were each worse on some workload.
        //  Paged: the lanes share the boxes of the prologue's keys, each looking
        // up its box's page.  The page list is read through L2 only: the
        // preceding grid may still be writing it, so a page id read here can
        // be stale -- it then only misdirects a hint, and no stale line is
        // left in L1 for the producer's own lookups after the wait.  Ids
        // outside the pool are skipped.
        constexpr int kPrologueBytes = 256 * 1024;
        constexpr int kPrefetchTiles = kPrologueBytes / SG::kBytes;   // per CTA
        // FP8 in a paged cache runs none: with 2 KB page boxes the prologue's
        // prefetches only queue ahead of the stage copies (measured, P = 16:
        // 64k 38.6 -> 35.7 us without it, 128k 67.8 -> 63.9 us, cold 64k
        // 44.6 -> 40.5 us; P = 32: 30.3 -> 29.4 us).
        if constexpr (!SG::kDirect && !(paged && SG::kFp8)) {
            if (early_derive && found && c.len > 0) {   // warp-uniform
                const int32_t len = split_len_for(c.len, c.splits);
                const int32_t t0p = c.s * len;
                const int32_t t1p = min(t0p + len, c.len);
                const int n_split = (t1p - t0p + kTile - 1) / kTile;
                if (n_split > NS) {
                    if constexpr (!paged) {
                        if (lane == 0)
                            for (int i = 0; i < min(kPrefetchTiles, n_split); ++i)
                                prefetch_box<SG>(&tm_k, &tm_v, kvh, c.base + t0p + i * kTile);
                    } else if (c.base >= 0 && c.base + c.pages <= p.num_page_entries) {
                        constexpr int kBox = SG::kBoxRows;
                        // boxes per lane: all of a lane's page ids are loaded
                        // before its first prefetch, so one L2 round trip (not
                        // one per box) delays the early launch
                        constexpr int kPerLane = (kPrefetchTiles * (kTile / kBox) + 31) / 32;
                        const int32_t t_end = min(t1p, t0p + kPrefetchTiles * kTile);
                        int32_t ids[kPerLane];
#pragma unroll
                        for (int j = 0; j < kPerLane; ++j) {
                            const int32_t t = t0p + (lane + 32 * j) * kBox;
                            const int32_t pg = t / p.page_size;
                            ids[j] = t < t_end && pg < c.pages ? __ldcg(p.page_indices + c.base + pg) : -1;
                        }
#pragma unroll
                        for (int j = 0; j < kPerLane; ++j) {
                            const int32_t t = t0p + (lane + 32 * j) * kBox;
                            if (ids[j] >= 0 && ids[j] < p.num_pages)
                                prefetch_box<SG>(&tm_k, &tm_v, kvh, ids[j] * p.page_size + t % p.page_size);
                        }
                    }
                    __syncwarp();
                    if (lane == 0)
                        griddep_launch_dependents();
                }
            }
        }
        if (early_derive)
            griddep_wait();
        int32_t t0, t1;
        const bool ok = item_range<paged>(p, c, found, t0, t1);
        // the device-side plan launches a CTA per item of its capacity; those
        // past the batch's items have nothing to do
        const bool none = !found && p.device_plan;
        if (lane == 0) {
            write_desc(desc, c, t0, t1, kvh, 0, ok ? kItemOk : (none ? kItemEnd : kItemBad));
            misc[kAbort] = ok || none ? 0 : 1;
            misc[kLast] = 0;
            if (!ok && !none)
                report(p.status, FD_ERR_DEVICE_BOUNDS);
        }
        __syncwarp();
        TileSource<NS, KV, DT> src(p, &tm_k, &tm_v, smem, bars, lane);
        const int n_tiles = ok && !self_fill ? (t1 - t0 + kTile - 1) / kTile : 0;
        const int first = min(NS, n_tiles);
        if (ok && (warp_loop || lane == 0)) {
            src.begin_item(t0, c.base, c.pages);
            for (int i = 0; i < first; ++i) {
                int32_t ya = 0, yb = 0;
                src.tile_rows(i, ya, yb);
                if (SG::kDirect || lane == 0)
                    src.issue(i, kvh, ya, yb);
            }
        }
        // fills[s]: copies issued into stage s, for the drain after an error
        if (lane == 0)
            for (int s = 0; s < NS; ++s)
                fills[s] = s < first ? 1 : 0;
        __syncthreads();   // the barriers are initialised
        if (ok && (warp_loop || lane == 0) && !self_refill) {
            // The producer refills in order (paged K/V: its cursor only moves
            // forward; bf16 K/V: bound by HBM, every warp as fast as its data,
            // in-order refills measured faster than out-of-order ones).
            int issued = first;
            for (int i = first; i < n_tiles; ++i) {
                int32_t ya = 0, yb = 0;
                src.tile_rows(i, ya, yb);
                int go = 0;
                if (lane == 0) {
                    go = mbar_wait(smem_addr(&bars[NS + i % NS]), ((i / NS) - 1) & 1, p.timeout_ns);
                    if (!go) {
                        misc[kAbort] = 1;
                        report(p.status, FD_ERR_TIMEOUT);
                    } else if (misc[kAbort]) {
                        go = 0;
                    }
                    if (go && !SG::kDirect)
                        src.issue(i, kvh, ya, yb);
                }
                if constexpr (warp_loop)
                    go = __shfl_sync(0xffffffffu, go, 0);
                if (!go)
                    break;
                if constexpr (SG::kDirect)
                    src.issue(i, kvh, ya, yb);
                issued = i + 1;
            }
            if (lane == 0)
                for (int s = 0; s < NS; ++s)
                    fills[s] = issued > s ? (issued - 1 - s) / NS + 1 : 0;
        }
    } else {
        // ---------------------------------------------------------- consumers
        __syncthreads();   // the barriers are initialised
        const Item it = read_item(desc);
        if (it.state == kItemOk) {
            uint32_t qa[8][2];
            float qk = p.q_scale * load_q<G, DT, true, kColumnForm<G, DT>>(
                                       p.q + ((int64_t)it.b * p.num_qo_heads + kvh * G) * kHeadDim, lane, qa);
            if constexpr (DT == kKvFp8) {   // the head's dequantisation scales
                qk *= __ldg(p.k_scale + kvh);
                vscale = __ldg(p.v_scale + kvh);
            }
            cs.begin(qk, lane);
            const uint32_t ring = smem_addr(smem);
            const int n_tiles = (it.t1 - it.t0 + kTile - 1) / kTile;
            if constexpr (self_fill) {
                // The warp's own pipeline over its stages warp + NC j (j < D):
                // its k-th tile (warp + NC k) goes to stage (warp + NC k) % NS,
                // one cp.async group per tile (an empty group past the last),
                // so that waiting for all but the D - 1 newest groups waits for
                // the tile about to be consumed.  No producer hop and no
                // mbarrier between a freed stage and its refill, and nothing
                // to time out: every wait is for this warp's own copies.
                // Measured against out-of-order refills by the producer warp
                // (back to back): 64k 24.82 -> 24.19 us, 128k 41.53 -> 41.00
                // us, 2048 keys 6.51 -> 6.28 us; three or four stages per warp
                // were slower.
                constexpr int D = NS / NC;
                static_assert(NS % NC == 0, "self-filled stages: D per consumer warp");
                const TileSource<NS, KV, DT> fsrc(p, &tm_k, &tm_v, smem, bars, lane);
                const int32_t y0 = it.base + it.t0;
                auto fill = [&](int k) {
                    const int i = warp + NC * k;
                    if (i < n_tiles)
                        fsrc.copy_direct(ring + (i % NS) * SG::kBytes, kvh, y0 + i * kTile, 0);
                    cp_async_commit();
                };
#pragma unroll
                for (int k = 0; k < D; ++k)
                    fill(k);
                for (int k = 0; warp + NC * k < n_tiles; ++k) {
                    const int i = warp + NC * k;
                    cp_async_wait_group<D - 1>();
                    __syncwarp();   // every lane's copies of the tile have landed
                    cs.tile(ring + (i % NS) * SG::kBytes, min(kTile, it.t1 - (it.t0 + i * kTile)), qa, lane);
                    __syncwarp();   // every lane is done reading the stage
                    fill(k + D);
                }
                cp_async_wait_group<0>();
            } else {
                const TileSource<NS, KV, DT> rsrc(p, &tm_k, &tm_v, smem, bars, lane);
                int i = warp;
                for (; i < n_tiles; i += NC) {
                    const int s = i % NS;
                    if (!mbar_wait(smem_addr(&bars[s]), (i / NS) & 1, p.timeout_ns)) {
                        misc[kAbort] = 1;
                        if (lane == 0)
                            report(p.status, FD_ERR_TIMEOUT);
                        break;
                    }
                    cs.tile(ring + s * SG::kBytes, min(kTile, it.t1 - (it.t0 + i * kTile)), qa, lane);
                    __syncwarp();
                    if constexpr (self_refill) {
                        // FP8: lane 0 refills the stage it just freed with the
                        // warp's tile after next (the producer issued the first
                        // two); the proxy fence orders the warp's reads of the
                        // stage before the TMA's writes.  Measured against
                        // out-of-order refills by the producer warp (64k keys,
                        // back to back): 22.85 -> 22.41 us, 128k 41.25 -> 40.40
                        // us, 2048 keys 6.45 -> 6.31 us.
                        if (lane == 0 && i + NS < n_tiles) {
                            fence_proxy_async_shared();
                            rsrc.issue(i + NS, kvh, it.base + it.t0 + (i + NS) * kTile, 0);
                        }
                    } else if (lane == 0) {
                        mbar_arrive(smem_addr(&bars[NS + s]));
                    }
                }
                if constexpr (self_refill) {
                    // copies issued into the warp's D stages, for the drain
                    // after an error: its first min(mine, done + D) tiles,
                    // done = the tiles it consumed (tile i stopped the loop);
                    // its k-th tile went to stage warp + NC (k mod D)
                    constexpr int D = NS / NC;
                    static_assert(NS % NC == 0, "self-refilled stages: D per consumer warp");
                    if (lane == 0) {
                        const int mine = n_tiles > warp ? (n_tiles - warp + NC - 1) / NC : 0;
                        const int done = (i - warp) / NC;
                        const int issued = min(mine, done + D);
#pragma unroll
                        for (int j = 0; j < D; ++j)
                            fills[warp + NC * j] = issued > j ? (issued - 1 - j) / D + 1 : 0;
                    }
                }
            }
        }
    }

    __syncthreads();
    if (misc[kAbort]) {
        // Let every copy this CTA issued land before the CTA exits: the last
        // fill of each stage completes that stage's phase fills - 1.
        if (warp == NC && lane == 0) {
            for (int s = 0; s < NS; ++s)
                if (fills[s] > 0 &&
                    !mbar_wait(smem_addr(&bars[s]), (fills[s] - 1) & 1, kDrainTimeoutNs))
                    report(p.status, FD_ERR_TIMEOUT);
        }
        __syncthreads();
        return;
    }
    // ---- close the item: consumer states over the drained ring, then the
    // whole CTA combines them (and runs stage 2 as the group's last CTA)
    const Item it = read_item(desc);
    if (it.state != kItemOk) {   // a CTA without an item (device-side plan)
        griddep_launch_dependents();
        return;
    }
    // Host-planned fused calls with several heads per group spread stage 2
    // over the group's last CTAs (with one head, a single merger is faster:
    // its acquire-release ticket needs no second round trip to see the
    // others' flags); the arrival ticket is taken now, so its round trip
    // overlaps the combine.  Measured (back to back, interleaved): 64k keys
    // 40.1 -> 39.7 us, FP8 26.1 -> 25.3 us, 128k FP8 43.9 -> 42.9 us.
    // The producer warp's lane takes it: it has no consumer state to write,
    // and a warp with the atomic in flight was measured to run its shuffles
    // about 100 ns each (warp 0 taking it: 64k INT4 column form +4.5 us).
    const bool spread = G > 1 && p.fuse_merge && p.flags != nullptr && it.splits > 1;
    constexpr int kTicketTid = NC * 32;
    int ticket = 0;
    if (spread && tid == kTicketTid)
        ticket = atomicAdd(p.counters + (int64_t)it.b * p.num_kv_heads + it.kvh, 1);
    if (warp < NC)
        cs.template write<NC>(smem, warp, lane, vscale);
    __syncthreads();
    if (spread)
        finish_item_spread<G, NC, NC + 1>(p, it, smem, smem, misc, tid, ticket, kTicketTid);
    else
        finish_item<G, NC, NC + 1, 0>(p, it, smem, smem, misc, tid, [] {});
    // This CTA's outputs are written: a dependent grid may launch.
    griddep_launch_dependents();
}

// Persistent (the plan needs more than one wave): at most one wave of resident
// CTAs.  CTA c starts with item c (item w = split w / Hkv of KV head w % Hkv,
// the planner's order) and then claims its next items from a counter, one item
// ahead so that the claim's latency hides behind the current item; that keeps
// a ragged batch balanced the way block scheduling would.  A CTA's tiles form
// one stream through the stage ring: the producer loads the next item while
// the consumers finish the current one and the epilogue warp closes the one
// before (combine, partial write, ticket, stage 2 as the group's last CTA);
// the CTA's last item is closed by the whole CTA.
template <int G, int NC, int NS, int MIN_CTAS, int KV, int DT>
__global__ void __launch_bounds__((NC + 2) * 32, MIN_CTAS)
    split_kv_persistent_kernel(const __grid_constant__ CUtensorMap tm_k,
                               const __grid_constant__ CUtensorMap tm_v,
                               const __grid_constant__ SplitParams p)
{
    using SG = Stage<KV, DT>;
    using L = PersistentLayout<G, NC, NS, SG::kBytes>;
    constexpr bool paged = KV != kKvRagged;
    constexpr bool warp_loop = paged || SG::kDirect;   // the whole producer warp runs the issue loop
    constexpr int kProducer = NC;   // the epilogue warp is NC + 1
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *qslots = smem + L::kOffQ;
    uint8_t *states = smem + L::kOffState;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint64_t *item_full = bars + 2 * NS;
    uint64_t *item_empty = item_full + kDescSlots;
    uint64_t *state_full = item_empty + kDescSlots;
    uint64_t *state_empty = state_full + 2;
    volatile int *desc = reinterpret_cast<volatile int *>(smem + L::kOffDesc);
    volatile int *misc = reinterpret_cast<volatile int *>(smem + L::kOffMisc);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t grid = (int32_t)gridDim.x;
    const bool early_derive = p.indptr_in_params && warp == kProducer;
    if (!early_derive)
        griddep_wait();

    if (warp == kProducer) {
        // ---------------------------------------------------------- producer
        // The whole warp locates each item (and, paged, runs the issue loop);
        // lane 0 issues the barrier operations, the claims and the copies.  It
        // sets up the barriers and puts the first tiles in flight before the
        // CTA barrier.
        if (lane == 0) {
            misc[kAbort] = 0;
            misc[kIssued] = 0;
            misc[kDescs] = 0;
            misc[kLast] = 0;
            misc[kFinalK] = -1;   // set to the last item's index; stays -1 for no items
            for (int s = 0; s < NS; ++s) {
                mbar_init(smem_addr(&bars[s]), SG::kFullArrivals);   // full: producer arrive(s) + bytes
                mbar_init(smem_addr(&bars[NS + s]), 1);   // empty: the stage's consumer warp
            }
            for (int s = 0; s < kDescSlots; ++s) {
                mbar_init(smem_addr(&item_full[s]), 1);        // producer arrive (+ Q bytes)
                mbar_init(smem_addr(&item_empty[s]), NC + 1);  // consumer warps + epilogue warp
            }
            for (int s = 0; s < 2; ++s) {
                mbar_init(smem_addr(&state_full[s]), NC);   // every consumer warp wrote its state
                mbar_init(smem_addr(&state_empty[s]), 1);   // the epilogue warp read it
            }
            fence_mbar_init();
        }
        __syncwarp();
        bool synced = false;
        auto cta_sync = [&]() {
            if (!synced) {
                __syncthreads();   // the barriers are initialised
                synced = true;
            }
        };
        const KeyIndex ki = key_index(p, paged);
        SplitCursor cursor;
        cursor.empty_split = p.device_plan;
        TileSource<NS, KV, DT> src(p, &tm_k, &tm_v, smem, bars, lane);
        int gt = 0;      // tiles issued so far (index of the stream's next tile)
        int descs = 0;   // descriptors published (lane 0)

        // Issue the item's tiles i0 .. i1-1 (stream tiles from gt on); false if
        // the CTA stops (a wait ran out, or another warp gave up).
        auto issue_range = [&](int i0, int i1, int kvh) -> bool {
            int stop = 0;
            if (warp_loop || lane == 0) {
                for (int i = i0; i < i1; ++i) {
                    int32_t ya = 0, yb = 0;
                    src.tile_rows(i, ya, yb);
                    int go = 0;
                    if (lane == 0) {
                        go = gt < NS ? 1
                                     : mbar_wait(smem_addr(&bars[NS + gt % NS]), ((gt / NS) - 1) & 1,
                                                 p.timeout_ns);
                        if (!go) {
                            misc[kAbort] = 1;
                            report(p.status, FD_ERR_TIMEOUT);
                        } else if (misc[kAbort]) {
                            go = 0;
                        }
                        if (go && !SG::kDirect)
                            src.issue(gt, kvh, ya, yb);
                    }
                    if constexpr (warp_loop)
                        go = __shfl_sync(0xffffffffu, go, 0);
                    if (!go) {
                        stop = 1;
                        break;
                    }
                    if constexpr (SG::kDirect)
                        src.issue(gt, kvh, ya, yb);
                    ++gt;
                }
            }
            stop = __shfl_sync(0xffffffffu, stop, 0);
            gt = __shfl_sync(0xffffffffu, gt, 0);
            return !stop;
        };
        // Lane 0: wait until descriptor slot k's previous item is closed;
        // false if the CTA stops.
        auto slot_free = [&](int k) -> bool {
            int go = 1;
            if (k >= kDescSlots)
                go = mbar_wait(smem_addr(&item_empty[k % kDescSlots]), ((k / kDescSlots) - 1) & 1,
                               p.timeout_ns);
            if (!go) {
                misc[kAbort] = 1;
                report(p.status, FD_ERR_TIMEOUT);
            } else if (misc[kAbort]) {
                go = 0;
            }
            return go;
        };

        // Lane 0: this CTA makes no more claims.  The CTA that completes the
        // count resets both counters for the next call; the count is
        // acquire-release, so every CTA's claims come before the reset.
        auto stop_claiming = [&]() {
            cuda::atomic_ref<int, cuda::thread_scope_device> done(*p.done);
            if (done.fetch_add(1, cuda::memory_order_acq_rel) == grid - 1) {
                cuda::atomic_ref<int, cuda::thread_scope_device>(*p.claim).store(
                    0, cuda::memory_order_relaxed);
                done.store(0, cuda::memory_order_relaxed);
            }
        };

        int k = 0;
        int32_t w = blockIdx.x;   // this item
        int32_t nxt = 0;          // the CTA's next item (lane 0; claimed during this one)
        for (;;) {
            const int kvh = w % p.num_kv_heads;
            SplitCoord c{};
            const bool found = cursor.find(ki, p.batch, p.chunk, w / p.num_kv_heads, c);
            if (k == 0 && early_derive)
                griddep_wait();
            if (!found) {
                // past the last item: the end of the CTA's stream (before its
                // first item when the plan has fewer items than CTAs)
                if (lane == 0) {
                    stop_claiming();
                    if (slot_free(k)) {
                        desc[(k % kDescSlots) * kDescInts + kDState] = kItemEnd;
                        ++descs;
                        mbar_arrive(smem_addr(&item_full[k % kDescSlots]));
                    }
                }
                break;
            }
            if (lane == 0)
                nxt = grid + atomicAdd(p.claim, 1);
            int32_t t0, t1;
            const bool ok = item_range<paged>(p, c, found, t0, t1);
            // hand the item (descriptor + its Q rows) to the other warps
            const int slot = k % kDescSlots;
            int go = 0;
            if (lane == 0) {
                go = slot_free(k);
                if (go) {
                    float ks = 1.f, vs = 1.f;
                    if constexpr (DT == kKvFp8) {   // the head's dequantisation scales
                        ks = __ldg(p.k_scale + kvh);
                        vs = __ldg(p.v_scale + kvh);
                    }
                    write_desc(desc + slot * kDescInts, c, t0, t1, kvh, gt, ok ? kItemOk : kItemBad,
                               ks, vs);
                    ++descs;
                    const uint32_t fb = smem_addr(&item_full[slot]);
                    if (ok) {
                        mbar_arrive_expect_tx(fb, L::kQBytes);
                        bulk_load(smem_addr(qslots + slot * L::kQSlot),
                                  p.q + ((int64_t)c.b * p.num_qo_heads + kvh * G) * kHeadDim,
                                  L::kQBytes, fb);
                    } else {
                        report(p.status, FD_ERR_DEVICE_BOUNDS);
                        misc[kAbort] = 1;
                        mbar_arrive(fb);
                    }
                }
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            if (!go || !ok)
                break;
            src.begin_item(t0, c.base, c.pages);
            const int n_tiles = (t1 - t0 + kTile - 1) / kTile;
            const int first = k == 0 ? min(NS, n_tiles) : n_tiles;
            if (!issue_range(0, first, kvh))
                break;
            cta_sync();
            if (!issue_range(first, n_tiles, kvh))
                break;
            w = __shfl_sync(0xffffffffu, nxt, 0);   // the next item
            ++k;
        }
        cta_sync();
        if (lane == 0) {
            misc[kIssued] = gt;
            misc[kDescs] = descs;
        }
    } else if (warp < NC) {
        // ---------------------------------------------------------- consumers
        __syncthreads();   // the barriers are initialised
        const uint32_t ring = smem_addr(smem);
        int k = 0;
        bool ok = mbar_wait(smem_addr(&item_full[0]), 0, p.timeout_ns);
        if (!ok) {
            misc[kAbort] = 1;
            if (lane == 0)
                report(p.status, FD_ERR_TIMEOUT);
        }
        Item it = read_item(desc);
        while (ok && it.state == kItemOk) {
            const int slot = k % kDescSlots;
            uint32_t qa[8][2];
            Consumer<G, KV, DT> cs;
            cs.begin(p.q_scale * __int_as_float(it.ks) *
                         load_q<G, DT, false, kColumnForm<G, DT>>(
                             reinterpret_cast<const uint16_t *>(qslots + slot * L::kQSlot), lane, qa),
                     lane);
            const int n_tiles = (it.t1 - it.t0 + kTile - 1) / kTile;
            // this warp's tiles of the item: stream tiles g = warp (mod NC)
            const int first = it.gt0 + ((warp - it.gt0 % NC) + NC) % NC;
            for (int g = first; g < it.gt0 + n_tiles; g += NC) {
                const int i = g - it.gt0;
                const int s = g % NS;
                if (!mbar_wait(smem_addr(&bars[s]), (g / NS) & 1, p.timeout_ns)) {
                    misc[kAbort] = 1;
                    if (lane == 0)
                        report(p.status, FD_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                cs.tile(ring + s * SG::kBytes, min(kTile, it.t1 - (it.t0 + i * kTile)), qa, lane);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&bars[NS + s]));
            }
            if (!ok)
                break;
            // The next descriptor tells whether this was the CTA's last item.
            const int nslot = (k + 1) % kDescSlots;
            ok = mbar_wait(smem_addr(&item_full[nslot]), ((k + 1) / kDescSlots) & 1, p.timeout_ns);
            if (!ok) {
                misc[kAbort] = 1;
                if (lane == 0)
                    report(p.status, FD_ERR_TIMEOUT);
                break;
            }
            const Item nx = read_item(desc + nslot * kDescInts);
            // state buffer k % 2: the epilogue warp must have read item k - 2's
            const int sb = k & 1;
            if (k >= 2 && !mbar_wait(smem_addr(&state_empty[sb]), ((k >> 1) - 1) & 1, p.timeout_ns)) {
                misc[kAbort] = 1;
                if (lane == 0)
                    report(p.status, FD_ERR_TIMEOUT);
                break;
            }
            cs.template write<NC>(states + sb * L::kStateBytes, warp, lane, __int_as_float(it.vs));
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&state_full[sb]));
            if (nx.state != kItemOk) {
                // the CTA's last item: the whole CTA closes it below
                if (warp == 0 && lane == 0)
                    misc[kFinalK] = k;
                break;
            }
            if (lane == 0)
                mbar_arrive(smem_addr(&item_empty[slot]));
            it = nx;
            ++k;
        }
    } else {
        // ---------------------------------------------------------- epilogue
        // Closes every item but the CTA's last while the other warps stream on.
        __syncthreads();   // the barriers are initialised
        // does the CTA have an item at all?  (later items are known to exist
        // from the descriptor checked below)
        if (!mbar_wait(smem_addr(&item_full[0]), 0, p.timeout_ns)) {
            misc[kAbort] = 1;
            if (lane == 0)
                report(p.status, FD_ERR_TIMEOUT);
        }
        const bool has_items = !misc[kAbort] && desc[kDState] == kItemOk;   // item 0, slot 0
        for (int k = 0; has_items; ++k) {
            const int sb = k & 1;
            if (!mbar_wait(smem_addr(&state_full[sb]), (k >> 1) & 1, p.timeout_ns)) {
                misc[kAbort] = 1;
                if (lane == 0)
                    report(p.status, FD_ERR_TIMEOUT);
                break;
            }
            // the consumers read the next descriptor before handing item k over
            if (misc[kAbort] || desc[((k + 1) % kDescSlots) * kDescInts + kDState] != kItemOk)
                break;
            const Item it = read_item(desc + (k % kDescSlots) * kDescInts);
            finish_item<G, NC, 1, -1>(p, it, states + sb * L::kStateBytes, nullptr, misc, lane, [&] {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&state_empty[sb]));
            });
            if (lane == 0)
                mbar_arrive(smem_addr(&item_empty[k % kDescSlots]));
        }
    }

    __syncthreads();
    if (misc[kAbort]) {
        // Let every copy this CTA issued land before the CTA exits: the tiles
        // (stage barriers) and each item's Q rows (descriptor barriers).
        if (warp == kProducer && lane == 0) {
            const int issued = misc[kIssued];
            for (int g = max(0, issued - NS); g < issued; ++g)
                if (!mbar_wait(smem_addr(&bars[g % NS]), (g / NS) & 1, kDrainTimeoutNs))
                    report(p.status, FD_ERR_TIMEOUT);
            const int descs = misc[kDescs];
            for (int kk = max(0, descs - kDescSlots); kk < descs; ++kk)
                if (!mbar_wait(smem_addr(&item_full[kk % kDescSlots]), (kk / kDescSlots) & 1,
                               kDrainTimeoutNs))
                    report(p.status, FD_ERR_TIMEOUT);
        }
        __syncthreads();
        return;
    }

    // ---- the CTA's last item, closed by the whole CTA (its consumer states
    // are in state buffer k % 2; the drained ring is the merge scratch)
    const int k_last = misc[kFinalK];
    if (k_last >= 0)
        finish_item<G, NC, NC + 2, 0>(p, read_item(desc + (k_last % kDescSlots) * kDescInts),
                                      states + (k_last & 1) * L::kStateBytes, smem, misc, tid,
                                      [] {});
    // This CTA's outputs are written: a dependent grid may launch.
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

// Launch one kernel with programmatic stream serialisation, opting in to its
// dynamic shared memory once per device (for the first 64 devices).
template <typename Kernel>
cudaError_t launch_kernel(Kernel kern, bool (&configured)[64], int smem_bytes, int threads,
                          int num_ctas, const KvMaps &m, const SplitParams &p, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess)
            return e;
        if (dev < 64)
            configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_ctas);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, m.k, m.v, p);
}

// Consumer warps (and stages, two per warp) for INT4 K/V, whose consumers
// are the bound (codes widened in registers).  Row form (G = 8), one-item
// kernel: a fifth consumer warp still fits the register file at two CTAs per
// SM (12 warps x 168 registers; 64k step -2 %, 128k -4.5 %; FP8 was slower
// with 5).  Column form (G <= 4, ~40 registers fewer), with the consumers
// filling their own stages: four in the one-item kernel (64k 22.0 us with
// four, 24.2 with five, 26.0 with three, 34.8 with two; 128k 35.9 against
// 41.1 with five; three stages per warp were slower) and three in the
// persistent kernel (ragged batch 168.4 us; four 185.4, six 182.7, two 221.3):
// the consumer warps then spread evenly over the SM's four schedulers.
constexpr int kNCInt4 = 5;
#ifndef FD_SPLIT_INT4_COLUMN_WARPS
#define FD_SPLIT_INT4_COLUMN_WARPS 4
#endif
#ifndef FD_SPLIT_INT4_COLUMN_PWARPS
#define FD_SPLIT_INT4_COLUMN_PWARPS 3
#endif
constexpr int kNCInt4Cols = FD_SPLIT_INT4_COLUMN_WARPS;     // one-item kernel, column form
constexpr int kNCInt4ColsP = FD_SPLIT_INT4_COLUMN_PWARPS;   // persistent kernel, column form
// FP8, column form: four consumer warps in the one-item kernel (with the
// consumers refilling their own stages: 64k 22.41 us with four, 22.38 with
// five, but 128k 40.40 against 41.27), four in the persistent kernel (ragged
// batch 164.7 us; five: 170.5; six do not fit two CTAs' shared memory).
#ifndef FD_SPLIT_FP8_COLUMN_WARPS
#define FD_SPLIT_FP8_COLUMN_WARPS 4
#endif
#ifndef FD_SPLIT_FP8_COLUMN_PWARPS
#define FD_SPLIT_FP8_COLUMN_PWARPS 4
#endif
constexpr int kNCFp8Cols = FD_SPLIT_FP8_COLUMN_WARPS;
constexpr int kNCFp8ColsP = FD_SPLIT_FP8_COLUMN_PWARPS;

// One wave of items: one item per CTA.  More: the persistent kernel on
// num_ctas CTAs.
template <int G, int KV, int DT>
cudaError_t launch_g(const KvMaps &m, const SplitParams &p, int num_ctas, cudaStream_t stream)
{
    constexpr bool cols = kColumnForm<G, DT>;
    // consumer warps of the one-item and the persistent kernel; FP8 and INT4
    // tiles are half the bytes or less, so their rings hold two stages per
    // consumer warp
    constexpr int NC1 = DT == kKvInt4 ? (cols ? kNCInt4Cols : kNCInt4) : DT == kKvFp8 && cols ? kNCFp8Cols : kNC;
    constexpr int NCP = DT == kKvInt4 && cols ? kNCInt4ColsP : DT == kKvFp8 && cols ? kNCFp8ColsP : kNC;
    constexpr int NS1 = DT == kKvBf16 ? kNS : 2 * NC1;
    constexpr int NS = DT == kKvBf16 ? kNS : 2 * NCP;
    using SG = Stage<KV, DT>;
    using LS = SingleLayout<G, NC1, NS1, SG::kBytes>;
    using LP = PersistentLayout<G, NCP, NS, SG::kBytes>;
    static_assert(kMinCtas * (LS::kAlloc + 1024) <= 233472 && kMinCtas * (LP::kAlloc + 1024) <= 233472,
                  "the resident CTAs must fit in shared memory");
    if (num_ctas >= p.num_work) {   // one wave: one item (or, device-side plan, at most one) per CTA
        static bool configured[64] = {};
        return launch_kernel(split_kv_kernel<G, NC1, NS1, kMinCtas, KV, DT>, configured, LS::kAlloc,
                             LS::kWarps * 32, p.num_work, m, p, stream);
    }
    static bool configured[64] = {};
    return launch_kernel(split_kv_persistent_kernel<G, NCP, NS, kMinCtas, KV, DT>, configured,
                         LP::kAlloc, LP::kWarps * 32, num_ctas, m, p, stream);
}

// Stage 1 for K/V elements of type DT: dispatch on the group size and the KV
// layout.
template <int DT>
cudaError_t launch_split_dt(const KvMaps &m, const SplitParams &p, int group, int num_ctas,
                            cudaStream_t stream)
{
    if (num_ctas < 1 || num_ctas > p.num_work)
        return cudaErrorInvalidValue;
    const int kv = p.kv_last_len == nullptr ? kKvRagged
                   : p.box_rows == kTile    ? kKvPaged
                                            : kKvPaged16;
    auto by_layout = [&](auto g) -> cudaError_t {
        constexpr int G = decltype(g)::value;
        switch (kv) {
        case kKvRagged: return launch_g<G, kKvRagged, DT>(m, p, num_ctas, stream);
        case kKvPaged: return launch_g<G, kKvPaged, DT>(m, p, num_ctas, stream);
        default: return launch_g<G, kKvPaged16, DT>(m, p, num_ctas, stream);
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

}  // namespace
}  // namespace fd
