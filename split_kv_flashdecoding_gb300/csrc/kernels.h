// kernels.h -- parameters and launchers of the libfd kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fd {

// Small batches carry kv_indptr in the launch parameters as well, so a CTA
// finds its key range without a dependent global load before its first copy.
constexpr int kParamIndptr = 33;   // batch <= 32

struct SplitParams {
    const uint16_t *q;          // bf16 [B, Hq, D]
    const int32_t *kv_indptr;   // device [B+1]: key-row prefix (ragged) or page-list prefix (paged)
    float *partial_o;           // [rows, D]
    float *partial_lse;         // [rows]
    int *status;                // workspace status word
    int32_t batch;
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t chunk;
    int32_t num_partial_rows;
    int32_t num_work;           // items: total splits x KV heads
    int32_t total_tokens;
    float q_scale;              // softmax scale * log2(e): logits are kept in base 2
    int64_t timeout_ns;
    // Fused stage 2 (fd_decode): the last CTA of each (request, KV head) group
    // merges the group's partials into o/lse; a request with a single split
    // writes o/lse directly.  counters: [B * Hkv] zero-initialised tickets.
    int32_t fuse_merge;
    float *o;                   // [B, Hq, D]
    float *lse;                 // [B, Hq]
    int *counters;
    // One-item kernel, host-planned fd_decode calls: each split publishes its
    // partial rows by writing `token` (unique per call) into its flag
    // (flags [Hkv][total_splits], kvh-major), and the last min(G, splits)
    // CTAs of a group to arrive merge one or more of its heads each.  Null
    // under the device-side plan: there the group's last CTA merges all heads.
    int *flags;
    int32_t token;
    // Persistent grid: items past the first wave are claimed from `claim`;
    // every CTA adds one to `done` when it stops claiming, and the CTA that
    // completes `done` resets both (zero-initialised, in the workspace header).
    int *claim;
    int *done;
    // Device-side plan (graph-capturable calls): the kernel finds the items
    // from the device kv_indptr alone, num_work is only an upper bound, and an
    // empty request is one split of no keys (it writes O = 0, LSE = -inf).
    int32_t device_plan;
    int32_t indptr_in_params;   // 1: indptr_param (and last_len_param) hold the device arrays
    int32_t indptr_param[kParamIndptr];
    // Paged KV (kv_last_len non-null): K/V are page pools [num_pages, page_size,
    // Hkv, D]; request b's pages are page_indices[kv_indptr[b] .. kv_indptr[b+1]).
    const int32_t *kv_last_len; // [B] valid keys in each request's last page
    const int32_t *page_indices;
    int32_t page_size;
    int32_t box_rows;           // rows per TMA box: 32, or 16 when pages are 16-row aligned only
    int32_t num_pages;
    int32_t num_page_entries;   // kv_indptr[B]
    int32_t last_len_param[kParamIndptr];
    // Element type of K/V (kKvTypeBf16, kKvTypeFp8, kKvTypeInt4), dequantised in
    // registers.  FP8 (E4M3): one byte per element; k_scale, v_scale [Hkv]
    // (device) multiply the head's K and V values.  INT4: two four-bit codes
    // per byte, and one scale per key row and head (k_scale, v_scale
    // [Hkv][kv_rows] fp32), loaded without tensor maps from k_data / v_data.
    int32_t kv_type;
    int32_t kv_rows;            // rows of K/V: T keys, or num_pages * page_size
    const uint8_t *k_data;      // K and V themselves
    const uint8_t *v_data;
    const float *k_scale;
    const float *v_scale;
};

constexpr int kKvTypeBf16 = 0;
constexpr int kKvTypeFp8 = 1;
constexpr int kKvTypeInt4 = 2;

// The split kernel's TMA descriptors of K and V (INT4 K/V: not read).
struct KvMaps {
    CUtensorMap k, v;
};

struct MergeParams {
    const int32_t *kv_indptr;
    const float *partial_o;
    const float *partial_lse;
    float *o;                   // [B, Hq, D]
    float *lse;                 // [B, Hq]
    int *status;
    int32_t batch;
    int32_t num_qo_heads;
    int32_t chunk;
    int32_t num_partial_rows;
    int32_t only_empty;         // write only the rows of requests with no keys
    const int32_t *kv_last_len; // paged layout (see SplitParams), or null
    int32_t page_size;
};

// Stage 1: p.num_work items (split, KV head) on a persistent grid of num_ctas
// CTAs (1 <= num_ctas <= p.num_work), CTA c taking items c, c + num_ctas, ...
// Launched as a programmatic dependent of the preceding grid (it waits for
// that grid before touching global memory).
cudaError_t launch_split(const KvMaps &maps, const SplitParams &p, int group, int num_ctas,
                         cudaStream_t stream);

// The same for FP8 and INT4 K/V (p.kv_type); launch_split dispatches to them.
cudaError_t launch_split_fp8(const KvMaps &maps, const SplitParams &p, int group, int num_ctas,
                             cudaStream_t stream);
cudaError_t launch_split_int4(const KvMaps &maps, const SplitParams &p, int group, int num_ctas,
                              cudaStream_t stream);

// Resident split-kernel CTAs per SM the launch shape is built for.
int split_ctas_per_sm();

// Stage 2: one CTA per (request, query head), launched as a programmatic
// dependent of the preceding grid so its launch overlaps that grid's tail.
cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream);

// Merge of num_states attention states per row (o_states [num_states][rows][D],
// lse_states [num_states][rows]) into o [rows][D], lse [rows].
cudaError_t launch_merge_states(int num_states, int rows, const float *o_states,
                                const float *lse_states, float *o, float *lse, cudaStream_t stream);

}  // namespace fd
