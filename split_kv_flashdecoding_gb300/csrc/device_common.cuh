// device_common.cuh -- sm_103a building blocks shared by the libfd kernels:
// mbarrier and TMA (cp.async.bulk.tensor) wrappers in inline PTX, bounded
// waits, bf16 unpacking, warp reductions, and the on-device derivation of a
// CTA's split from kv_indptr (the same rule as the host planner).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fd.h"
#include "plan_rule.h"

namespace fd {

constexpr int kHeadDim = 128;
constexpr int kTile = FD_TILE_TOKENS;   // keys per pipeline stage
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// A wait that drains copies still in flight after an error always gets this
// long, whatever the plan's timeout (the copies target valid addresses and end).
constexpr int64_t kDrainTimeoutNs = 200000000LL;

// ------------------------------------------------------------------ status

// Record the first error a kernel hits in the workspace status word.
__device__ __forceinline__ void report(int *status, int code)
{
    atomicCAS(status, 0, code);
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete; give up after
// timeout_ns (timeout_ns <= 0 gives up at once).  Returns false on give-up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int64_t timeout_ns)
{
    if (timeout_ns <= 0)
        return false;
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((int64_t)(global_timer_ns() - t0) > timeout_ns)
            return false;
    }
}

// --------------------------------------------------------------------- TMA

__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2-D tiled TMA load of box (x, y) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t x,
                                            int32_t y, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// 16-byte asynchronous copy global -> shared (L2 only), the bytes past
// src_bytes (0 or 16) zero-filled, with an L2 eviction policy.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes,
                                            uint64_t policy)
{
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst),
                 "l"(src), "r"(src_bytes), "l"(policy)
                 : "memory");
}

// 4-byte asynchronous copy global -> shared, zero-filled past src_bytes (0 or 4).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// Close this thread's group of cp.async copies issued since the last commit.
__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's committed cp.async groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One arrival on `bar` once every cp.async this thread issued before has
// landed (the barrier's expected count includes it).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Prefetch a tiled TMA box into L2.  A hint: it changes no value, so it may
// run before the wait for a preceding grid that writes the same memory (L2 is
// where global memory is coherent).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int32_t x, int32_t y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *map, int32_t x, int32_t y,
                                                   int32_t z)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// 3-D tiled TMA load of box (x, y, z) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int32_t x,
                                            int32_t y, int32_t z, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// Untiled bulk copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// ------------------------------------------------ flags between CTAs

__device__ __forceinline__ int ld_acquire_gpu(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(int *p, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ------------------------------------------- programmatic dependent launch

// Allow the next grid in the stream (launched with programmatic stream
// serialisation) to start launching; its griddep_wait() still waits for this
// grid to finish and its writes to be visible.
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the preceding grid in the stream has completed (no-op when this
// grid was not launched as a programmatic dependent).
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------ arithmetic

// Two packed bf16 (low half = first element) widened exactly to fp32.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// ------------------------------------------------------- split derivation

// Where each request's keys live.
//   ragged: indptr = key-row prefix [B+1]; request b's keys are the rows
//           indptr[b] .. indptr[b+1]-1 of K/V [T, Hkv, D].
//   paged:  indptr = page-list prefix [B+1]; request b's keys fill, in order,
//           the pages page_indices[indptr[b] .. indptr[b+1]-1] of the page pool
//           [num_pages, page_size, Hkv, D], the last one up to last_len[b] keys.
struct KeyIndex {
    const int32_t *indptr;
    const int32_t *last_len;   // null: ragged
    int32_t page_size;

    // base: first key row (ragged) or first page-list entry (paged); len: keys;
    // pages: page-list entries (paged) or 0.
    __device__ __forceinline__ void at(int b, int32_t &base, int32_t &len, int32_t &pages) const
    {
        // plain loads: the arrays may live in global or in parameter space
        const int32_t a = indptr[b], e = indptr[b + 1];
        base = a;
        if (!last_len) {
            len = e - a;
            pages = 0;
        } else {
            pages = e - a;
            len = pages > 0 ? (pages - 1) * page_size + last_len[b] : 0;
        }
    }
};

struct SplitCoord {
    int32_t b;        // request
    int32_t prefix;   // splits of requests before b
    int32_t splits;   // splits_b
    int32_t s;        // split within the request (when derived from a split index)
    int32_t base;     // first key row (ragged) or first page-list entry (paged)
    int32_t len;      // keys of the request
    int32_t pages;    // page-list entries of the request (paged)
};

// Warp-collective: locate global split `j` (if by_request is false) or request
// `j` (if true) by scanning the requests' key counts.  All lanes return the
// same result; returns false if j is out of range.  empty_split: an empty
// request counts as one split (the device-side plan).
__device__ __forceinline__ bool derive_split(const KeyIndex &ki, int batch, int32_t chunk, int32_t j,
                                             bool by_request, SplitCoord &out,
                                             bool empty_split = false)
{
    const int lane = threadIdx.x & 31;
    int32_t carry = 0;
    for (int b0 = 0; b0 < batch; b0 += 32) {
        const int b = b0 + lane;
        int32_t base = 0, len = 0, pages = 0, n = 0;
        if (b < batch) {
            ki.at(b, base, len, pages);
            n = len > 0 ? splits_for(len, chunk) : (empty_split ? 1 : 0);
        }
        int32_t incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += t;
        }
        incl += carry;
        const int32_t excl = incl - n;
        const bool hit = b < batch && (by_request ? b == j : (j >= excl && j < incl));
        const unsigned mask = __ballot_sync(0xffffffffu, hit);
        if (mask) {
            const int src = __ffs(mask) - 1;
            out.b = __shfl_sync(0xffffffffu, b, src);
            out.prefix = __shfl_sync(0xffffffffu, excl, src);
            out.splits = __shfl_sync(0xffffffffu, n, src);
            out.base = __shfl_sync(0xffffffffu, base, src);
            out.len = __shfl_sync(0xffffffffu, len, src);
            out.pages = __shfl_sync(0xffffffffu, pages, src);
            out.s = by_request ? 0 : j - out.prefix;
            return true;
        }
        carry = __shfl_sync(0xffffffffu, incl, 31);
    }
    return false;
}

// Warp-collective cursor over all requests' splits for a sequence of split
// indices that never decreases (the items of one persistent CTA).  Lane l holds
// request b0 + l of the current window of 32 requests and the inclusive prefix
// of the split counts; moving on to the next window costs one load per lane,
// so a batch of at most 32 requests is read once per CTA.  empty_split: an
// empty request counts as one split of no keys (the device-side plan, where
// that split writes the request's O = 0, LSE = -inf rows).
struct SplitCursor {
    int32_t b0 = 0;      // first request of the window
    int32_t carry = 0;   // splits of the requests before b0
    int32_t base = 0, len = 0, pages = 0, n = 0, incl = 0;
    bool loaded = false;
    bool empty_split = false;

    __device__ __forceinline__ void load(const KeyIndex &ki, int batch, int32_t chunk)
    {
        const int lane = threadIdx.x & 31;
        const int b = b0 + lane;
        base = len = pages = n = 0;
        if (b < batch) {
            ki.at(b, base, len, pages);
            n = len > 0 ? splits_for(len, chunk) : (empty_split ? 1 : 0);
        }
        incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += t;
        }
        incl += carry;
        loaded = true;
    }

    // Locate global split j (not below any j asked before); false if j is
    // past the last split.
    __device__ __forceinline__ bool find(const KeyIndex &ki, int batch, int32_t chunk, int32_t j,
                                         SplitCoord &out)
    {
        const int lane = threadIdx.x & 31;
        while (b0 < batch) {
            if (!loaded)
                load(ki, batch, chunk);
            const int32_t excl = incl - n;
            const unsigned mask = __ballot_sync(0xffffffffu, b0 + lane < batch && j >= excl && j < incl);
            if (mask) {
                const int src = __ffs(mask) - 1;
                out.b = b0 + src;
                out.prefix = __shfl_sync(0xffffffffu, excl, src);
                out.splits = __shfl_sync(0xffffffffu, n, src);
                out.base = __shfl_sync(0xffffffffu, base, src);
                out.len = __shfl_sync(0xffffffffu, len, src);
                out.pages = __shfl_sync(0xffffffffu, pages, src);
                out.s = j - out.prefix;
                return true;
            }
            carry = __shfl_sync(0xffffffffu, incl, 31);
            b0 += 32;
            loaded = false;
        }
        return false;
    }
};

}  // namespace fd
