// plan_rule.h -- the split rule shared by the host planner and the kernels.
//
// "FlashDecoding++: sequence-dimension KV split parallelism for LLM serving"
// (techknowgenie.com), §2: each request's keys are cut into chunks along the
// sequence and every (chunk, head) becomes its own thread block.  The plan
// fixes one chunk length C per step; request b with L_b keys then gets
//     splits_b = ceil(L_b / C)
// splits of length roundup(ceil(L_b / splits_b), FD_TILE_TOKENS) (equalised
// within the request, last split ragged).  Because C is a multiple of the tile
// and splits_b - 1 < L_b / C, no split is ever empty.
#pragma once

#include <stdint.h>

#include "fd.h"

#if defined(__CUDACC__)
#define FD_HD __host__ __device__ __forceinline__
#else
#define FD_HD inline
#endif

namespace fd {

FD_HD int32_t splits_for(int32_t len, int32_t chunk)
{
    return len > 0 ? (len + chunk - 1) / chunk : 0;
}

FD_HD int32_t split_len_for(int32_t len, int32_t splits)
{
    const int32_t even = (len + splits - 1) / splits;
    return (even + FD_TILE_TOKENS - 1) / FD_TILE_TOKENS * FD_TILE_TOKENS;
}

// Row of (request with split prefix `prefix` and `splits` splits, query head hq,
// split s) in the partial buffers.
FD_HD int64_t partial_row(int32_t prefix, int32_t num_qo_heads, int32_t hq,
                          int32_t splits, int32_t s)
{
    return (int64_t)prefix * num_qo_heads + (int64_t)hq * splits + s;
}

}  // namespace fd
