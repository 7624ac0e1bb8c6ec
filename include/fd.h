/*
 * fd.h -- C ABI of libfd: split-KV ("flash-decoding") decode attention for
 * NVIDIA GB300 (sm_103a).
 *
 * Method: "FlashDecoding++: sequence-dimension KV split parallelism for LLM
 * serving" (techknowgenie.com).  §2 adds the sequence axis to the grid so a
 * batch-1 decode step fills every SM; §3 computes a partial softmax per chunk
 * (stage 1) and merges the partials by their log-sum-exp (stage 2); §6 (chunk
 * size tuning guide) sizes the chunks from the SM count.
 *
 * What one decode step computes (for each request b and query head hq, with
 * G = Hq / Hkv and KV head kvh = hq / G):
 *     s_j   = scale * <q[b,hq,:], K[j,kvh,:]>      j in [kv_indptr[b], kv_indptr[b+1])
 *     O     = sum_j softmax(s)_j * V[j,kvh,:]
 *     LSE   = ln sum_j exp(s_j)
 *
 * Tensor layouts (all row-major, contiguous, device memory unless noted):
 *     q          bf16  [B, Hq, D]
 *     k, v       bf16  [T, Hkv, D]   ragged "packed" KV cache, T = kv_indptr[B]
 *     kv_indptr  int32 [B+1]         0 = kv_indptr[0] <= ... <= kv_indptr[B] = T
 *     o          fp32  [B, Hq, D]
 *     lse        fp32  [B, Hq]       natural log; -inf for a request with no keys
 *     partial_o  fp32  [num_partial_rows, D]
 *     partial_lse fp32 [num_partial_rows]
 * Partial row of (request b, query head hq, split s):
 *     split_prefix[b] * Hq + hq * splits_b + s
 * where splits_b is request b's split count and split_prefix[b] is the sum of
 * splits_b' over b' < b.
 *
 * Supported: D = 128; G = Hq / Hkv in {1, 2, 4, 8}.  Others return
 * FD_ERR_UNSUPPORTED.  q, k, v, o, partial_o must be 16-byte aligned.
 *
 * Ownership: the caller owns every buffer.  The library allocates no device
 * memory and keeps no state between calls besides a cached SM count per device,
 * with one exception: fd_decode_static_workspace keeps its scratch in a fixed
 * device array of FD_STATIC_WORKSPACE_BYTES inside the library (present on
 * every GPU that loads it, holding the last such call's contents) and caches
 * that array's device address per device.
 * All device work is asynchronous on the given stream (a cudaStream_t passed as
 * void*; NULL = legacy default stream).
 *
 * Errors: every entry point returns an fd_status (0 = FD_OK, negative =
 * error) and never throws.  Arguments are validated on the host before any
 * launch; launch failures return FD_ERR_CUDA.  Errors the kernels detect
 * (a bounded wait that ran out, a derived index outside the plan) are written
 * to a status word in the workspace and read by fd_get_device_status().
 *
 * Workspace: a caller-owned device buffer, zero-filled before its first use.
 * Its first FD_WORKSPACE_HEADER_BYTES hold the device status word and the
 * work counter of the split kernel (used when a plan has more split items than
 * one wave of resident CTAs: the kernel then runs persistent CTAs that claim
 * items from the counter); fd_decode also keeps in it one merge ticket per
 * (request, KV head) and the split partials (size:
 * fd_plan_info.workspace_bytes).  The counter and the tickets return to zero
 * at the end of every successful call; after a call that reported an error
 * status, zero the workspace again before reusing it.  Calls that share one
 * workspace must be ordered on one stream.
 *
 * Launches: the kernels are launched with programmatic stream serialisation:
 * each may begin launching while the previous grid in the stream finishes,
 * and waits for that grid to complete before it reads or writes global
 * memory, so stream order is kept.  The one exception changes no result:
 * before that wait, the split kernel of a long split may prefetch the split's
 * first K/V rows into L2 (a hint), and the paged one reads the page list
 * through L2 to aim those prefetches.  Every value a kernel computes is read
 * after the wait.
 */
#ifndef FD_H
#define FD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fd_status {
    FD_OK = 0,
    FD_ERR_INVALID_ARG = -1,   /* bad pointer, size, layout or indptr */
    FD_ERR_UNSUPPORTED = -2,   /* head_dim or group size not built */
    FD_ERR_WORKSPACE = -3,     /* workspace missing or too small */
    FD_ERR_CUDA = -4,          /* a CUDA runtime call or launch failed */
    FD_ERR_TIMEOUT = -5,       /* an in-kernel wait ran past its limit */
    FD_ERR_DEVICE_BOUNDS = -6  /* a kernel derived an index outside the plan */
} fd_status;

/* Keys per pipeline stage; every chunk length is a multiple of it. */
#define FD_TILE_TOKENS 32
/* Bytes at the start of every workspace reserved for the device status. */
#define FD_WORKSPACE_HEADER_BYTES 256
/* Default bound on each in-kernel wait, in nanoseconds. */
#define FD_DEFAULT_TIMEOUT_NS 1000000000LL

/*
 * A decode plan (plain data; fill it with fd_plan).
 *
 * The plan fixes one chunk length C for the step.  Request b (L_b keys) is cut
 * into splits_b = ceil(L_b / C) splits of equal length rounded up to a
 * multiple of FD_TILE_TOKENS (the last one ragged); each (split, KV head) is
 * one CTA of the split kernel.  The kernels re-derive each CTA's key range
 * from kv_indptr on the device with this same rule, so no per-step work list
 * is copied to the GPU.
 */
typedef struct fd_plan_info {
    int32_t batch;
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t group_size;        /* num_qo_heads / num_kv_heads */
    int32_t chunk;             /* max keys per split, multiple of FD_TILE_TOKENS */
    int32_t total_splits;      /* sum over requests of splits_b */
    int32_t max_splits;        /* max over requests of splits_b */
    int32_t num_work;          /* split-kernel CTAs = total_splits * num_kv_heads */
    int32_t num_partial_rows;  /* total_splits * num_qo_heads */
    int32_t num_sms;           /* SM count the chunk was chosen for */
    int32_t ctas_per_sm;       /* target CTAs per SM the chunk was chosen for */
    int64_t total_tokens;      /* kv_indptr[batch] */
    int64_t workspace_bytes;   /* workspace fd_decode needs for this plan */
    int64_t timeout_ns;        /* limit on each in-kernel wait; 0 makes every
                                  wait give up at once (a test hook: the call
                                  then reports FD_ERR_TIMEOUT) */
} fd_plan_info;

/* Human-readable name of a status code (static string). */
const char *fd_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int fd_version(void);

/* SM count of a CUDA device (cached after the first query). */
int fd_num_sms(int device, int *num_sms);

/*
 * fd_plan -- choose the chunk length and size the split grid (host only, no
 * CUDA call unless num_sms == 0).
 *
 * Article §2 (split grid = batch x heads x chunks) and §6 (chunk size tuning
 * guide: enough CTAs to fill the SMs, chunks not so small that the stage-2
 * reduction dominates, adapted to the load).  With chunk == 0 the plan tries
 *     C_w = max(FD_MIN_CHUNK, roundup(ceil(T * Hkv / (w * num_sms * ctas_per_sm)), FD_TILE_TOKENS))
 * for w = 1, 2, 4, 8 waves of resident CTAs, simulates how the hardware would
 * dispatch each grid in launch order onto num_sms * ctas_per_sm slots (per-CTA
 * cost = its 32-key tiles + a fixed overhead), and keeps the shortest.  Even
 * batches get one wave; ragged ones get smaller chunks that balance the
 * slots.  chunk > 0 forces C (must be a positive multiple of FD_TILE_TOKENS).
 *
 * kv_indptr_host: host int32 [batch+1].  num_sms: 0 = query the current
 * device.  ctas_per_sm: resident CTAs per SM; 0 = what the split kernel's
 * launch shape fits (2).  Writes *info; returns
 * FD_ERR_INVALID_ARG for a malformed indptr or head counts,
 * FD_ERR_UNSUPPORTED for an unsupported head_dim or group size.
 */
#define FD_MIN_CHUNK 128
int fd_plan(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
            const int32_t *kv_indptr_host, int num_sms, int ctas_per_sm, int chunk,
            fd_plan_info *info);

/*
 * fd_plan_work_items -- list the plan's CTAs in launch order (host only).
 * items: caller-owned host int32 [num_work][5] = (b, kv_head, split,
 * tok_begin, tok_end) with absolute key rows [tok_begin, tok_end).
 * capacity: rows available in items; FD_ERR_INVALID_ARG if too small.
 */
int fd_plan_work_items(const fd_plan_info *info, const int32_t *kv_indptr_host,
                       int32_t *items, int64_t capacity);

/*
 * fd_decode_split -- stage 1 (article §3, "local chunk computation"): one CTA
 * per (split, KV head) streams its keys once through shared memory (TMA,
 * multi-stage mbarrier pipeline), and for each of the G query heads that share
 * the KV head computes the local max, the local exp-sum and the local
 * probability-weighted sum of V.  It stores the partial in normalised form,
 *     partial_o   = (sum_j exp(s_j - m) V_j) / (sum_j exp(s_j - m))
 *     partial_lse = m + ln(sum_j exp(s_j - m)),
 * which carries the same information as the article's (output, max, sum).
 *
 * info: from fd_plan for this kv_indptr.  kv_indptr_dev: device copy of the
 * same indptr.  scale: softmax scale (applied to q.k).  workspace: device,
 * >= FD_WORKSPACE_HEADER_BYTES (status word, work counter).
 */
int fd_decode_split(const fd_plan_info *info, const void *q, const void *k,
                    const void *v, const int32_t *kv_indptr_dev, float scale,
                    float *partial_o, float *partial_lse, void *workspace,
                    int64_t workspace_bytes, void *stream);

/*
 * fd_merge -- stage 2 (article §3, "global reduction"): for each (b, hq) take
 * M = max_i partial_lse_i, weights w_i = exp(partial_lse_i - M), and write
 *     o = sum_i w_i partial_o_i / sum_i w_i,   lse = M + ln sum_i w_i.
 * A request with no keys gets o = 0, lse = -inf.
 */
int fd_merge(const fd_plan_info *info, const int32_t *kv_indptr_dev,
             const float *partial_o, const float *partial_lse, float *o, float *lse,
             void *workspace, int64_t workspace_bytes, void *stream);

/*
 * fd_decode -- plan (default chunking for the current device), stage 1 and
 * stage 2 in one call.  Stage 2 is fused into the split kernel: the CTA that
 * finishes a (request, KV head) group last (a ticket in the workspace) merges
 * the group's partials with the same arithmetic as fd_merge, and a request
 * with a single split writes O and LSE directly.  The partials live in the
 * workspace, which must hold fd_plan_info.workspace_bytes (FD_ERR_WORKSPACE
 * otherwise; query it with fd_plan for the same arguments).  Needs kv_indptr
 * on the host (for the plan) and on the device (for the kernels); the two must
 * hold the same values.
 */
int fd_decode(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
              const int32_t *kv_indptr_host, const int32_t *kv_indptr_dev,
              const void *q, const void *k, const void *v, float scale,
              float *o, float *lse, void *workspace, int64_t workspace_bytes,
              void *stream);

/*
 * Paged KV cache -- FD++ §6 ("vLLM and TensorRT-LLM integration"): the engine
 * keeps K/V in fixed-size physical pages from a page table, and each split
 * chunk streams the pages its keys fall in.
 *
 * Layout:
 *     k_pages, v_pages      bf16  [num_pages, page_size, Hkv, D]   page pools
 *     kv_page_indptr        int32 [B+1]   request b owns page-list entries
 *                                          kv_page_indptr[b] .. kv_page_indptr[b+1]-1
 *     kv_page_indices       int32 [kv_page_indptr[B]]   physical page of each entry
 *     kv_last_page_len      int32 [B]     keys in request b's last page, 1..page_size
 * Request b's keys are, in order, rows 0..page_size-1 of its pages, the last
 * page filled to kv_last_page_len[b]; it has (pages_b - 1) * page_size +
 * kv_last_page_len[b] keys (0 with no pages).  page_size must be a positive
 * multiple of 16 (FD_ERR_UNSUPPORTED otherwise).  A page index outside
 * [0, num_pages) sets FD_ERR_DEVICE_BOUNDS in the status word (the page is not
 * read).
 */

/*
 * fd_plan_paged -- fd_plan for a paged layout: the same chunking on the
 * requests' key counts (host only).  Sizes the fd_decode_paged workspace.
 */
int fd_plan_paged(int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                  const int32_t *kv_page_indptr_host, const int32_t *kv_last_page_len_host,
                  int num_sms, int ctas_per_sm, int chunk, fd_plan_info *info);

/*
 * fd_decode_paged -- fd_decode over a paged KV cache: plan, stage 1 with each
 * 32-key tile copied from the page it lies in (TMA boxes never cross a page),
 * stage 2 fused.  kv_page_indptr and kv_last_page_len are given on the host
 * (for the plan) and on the device (for the kernels) with the same values;
 * kv_page_indices on the device.  Workspace as fd_decode, sized by
 * fd_plan_paged.
 */
int fd_decode_paged(int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                    int num_pages, const int32_t *kv_page_indptr_host,
                    const int32_t *kv_last_page_len_host, const int32_t *kv_page_indptr_dev,
                    const int32_t *kv_last_page_len_dev, const int32_t *kv_page_indices_dev,
                    const void *q, const void *k_pages, const void *v_pages, float scale,
                    float *o, float *lse, void *workspace, int64_t workspace_bytes,
                    void *stream);

/*
 * FP8 (E4M3) KV cache -- FD++ §4 ("quantisation-friendly kernel fusion"): the
 * quantised K and V are read from HBM as they are and dequantised on chip, in
 * registers, straight into the tensor-core operands, so the stream moves half
 * the bytes of bf16.
 *
 * Layout: K and V hold one OCP FP8 E4M3 byte per value (1 sign, 4 exponent
 * bits with bias 7, 3 mantissa bits; no infinities) in the same shapes as the
 * bf16 entry points ([T, Hkv, D] ragged, [num_pages, page_size, Hkv, D]
 * paged).  k_scale and v_scale (device, fp32 [Hkv]) give each KV head's
 * scale: the value of a K byte is E4M3(byte) * k_scale[head], and likewise
 * for V.  q stays bf16 and O, LSE fp32.  The arithmetic matches the bf16 path
 * (every E4M3 value is exact in f16, the products accumulate in fp32); the
 * result is attention over the dequantised K and V.  Byte 0x7F / 0xFF (NaN)
 * propagates as NaN.  Workspace and plan as for fd_decode / fd_decode_paged.
 */
int fd_decode_fp8(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                  const int32_t *kv_indptr_host, const int32_t *kv_indptr_dev,
                  const void *q, const void *k_fp8, const void *v_fp8,
                  const float *k_scale, const float *v_scale, float scale,
                  float *o, float *lse, void *workspace, int64_t workspace_bytes,
                  void *stream);

int fd_decode_paged_fp8(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                        int page_size, int num_pages, const int32_t *kv_page_indptr_host,
                        const int32_t *kv_last_page_len_host, const int32_t *kv_page_indptr_dev,
                        const int32_t *kv_last_page_len_dev, const int32_t *kv_page_indices_dev,
                        const void *q, const void *k_pages_fp8, const void *v_pages_fp8,
                        const float *k_scale, const float *v_scale, float scale,
                        float *o, float *lse, void *workspace, int64_t workspace_bytes,
                        void *stream);

/*
 * INT4 KV cache -- FD++ §4 names INT4 beside FP8: the packed codes are read
 * from HBM as they are and widened on chip, in registers, into the
 * tensor-core operands, so the stream moves about a quarter of the bytes of
 * bf16.  The page fixes no INT4 format; this is the plainest one that keeps a
 * head's values on a common scale per key: symmetric codes, one scale per
 * (key row, KV head).
 *
 * Layout: K and V hold head_dim / 2 bytes per (row, KV head): [T, Hkv, D/2]
 * ragged, [num_pages, page_size, Hkv, D/2] paged.  Byte j of a row holds
 * element 2j in its low nibble and element 2j + 1 in its high nibble, each a
 * four-bit two's-complement code c in -8..7.  k_scale and v_scale (device,
 * fp32) are head-major: [Hkv][rows], rows = T (ragged) or
 * num_pages * page_size (paged; entry h * rows + p * page_size + r belongs to
 * row r of page p).  The value of a K element is c * k_scale[h][row], and
 * likewise for V.  q stays bf16 and O, LSE fp32; the result is attention over
 * the dequantised K and V (the codes widen to f16 exactly and each q row is
 * scaled into f16 by a power of two, as for FP8; each row's K scale multiplies
 * its logit in fp32, and its V scale its softmax weight, which enters P V as
 * an f16 hi + lo pair after division by a power of two that bounds the V
 * scales seen so far, so scales of any finite magnitude keep the path's
 * relative accuracy).  A scale of +-inf or NaN propagates (as NaN); the scales
 * of rows past a request's last key (the rest of its last page) are never
 * used.  Workspace and plan as for fd_decode / fd_decode_paged.
 */
int fd_decode_int4(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                   const int32_t *kv_indptr_host, const int32_t *kv_indptr_dev,
                   const void *q, const void *k_int4, const void *v_int4,
                   const float *k_scale, const float *v_scale, float scale,
                   float *o, float *lse, void *workspace, int64_t workspace_bytes,
                   void *stream);

int fd_decode_paged_int4(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                         int page_size, int num_pages, const int32_t *kv_page_indptr_host,
                         const int32_t *kv_last_page_len_host, const int32_t *kv_page_indptr_dev,
                         const int32_t *kv_last_page_len_dev, const int32_t *kv_page_indices_dev,
                         const void *q, const void *k_pages_int4, const void *v_pages_int4,
                         const float *k_scale, const float *v_scale, float scale,
                         float *o, float *lse, void *workspace, int64_t workspace_bytes,
                         void *stream);

/*
 * Graph-capturable decode -- for engines that run decode steps as CUDA graphs
 * with a fixed batch (FD++ §6 integration).  fd_decode plans on the host from
 * the host copy of kv_indptr on every call, which a graph replay cannot
 * repeat.  Here the plan is made once for a capacity, and each call takes
 * device data only, so it can be captured in a CUDA graph and replayed with
 * new lengths written to the device indptr between replays.
 *
 * fd_plan_graph -- host only.  Fixes the chunk length (`chunk`, or 0 for the
 * planner's choice for max_total_tokens keys spread evenly over the batch) and
 * sizes the plan for any kv_indptr with kv_indptr[batch] <= max_total_tokens:
 * at most floor(max_total_tokens / chunk) + batch splits.  info->workspace_bytes
 * is the workspace fd_decode_graph needs.
 *
 * fd_decode_graph -- plan + stage 1 with stage 2 fused, the split of every
 * request derived on the device from kv_indptr_dev (same split rule as
 * fd_plan for that chunk; an empty request gives O = 0, LSE = -inf).  Reads no
 * host memory and makes no host-synchronising call, so it may be captured.
 * K and V must hold at least max_total_tokens rows.  A device indptr beyond the
 * capacity sets FD_ERR_DEVICE_BOUNDS in the status word.  Workspace as
 * fd_decode (zero-filled once, reused across replays on one stream).
 */
int fd_plan_graph(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                  int64_t max_total_tokens, int num_sms, int chunk, fd_plan_info *info);

int fd_decode_graph(const fd_plan_info *info, const int32_t *kv_indptr_dev,
                    const void *q, const void *k, const void *v, float scale,
                    float *o, float *lse, void *workspace, int64_t workspace_bytes,
                    void *stream);

/*
 * fd_merge_states -- the merge of attention states computed over disjoint
 * parts of the same keys: the exchange step of sequence sharding (one
 * request's keys cut into contiguous shards on several GPUs, each running
 * fd_decode on its shard; the per-shard O and LSE are gathered and merged
 * here).  FD++ §3 stage 2: the same global reduction, now across shards.
 *
 * For each row r: M = max_s lse_states[s][r], w_s = exp(lse_states[s][r] - M),
 * o[r] = sum_s w_s o_states[s][r] / sum_s w_s, lse[r] = M + ln sum_s w_s; a
 * row whose states are all -inf (no keys in any shard) gets o = 0, lse = -inf.
 * o_states fp32 [num_states, rows, head_dim], lse_states fp32 [num_states,
 * rows], o [rows, head_dim], lse [rows], all on the device; rows = B * Hq.
 */
int fd_merge_states(int num_states, int rows, int head_dim, const float *o_states,
                    const float *lse_states, float *o, float *lse, void *stream);

/*
 * fd_decode_static_workspace -- fd_decode for callers that cannot allocate.
 *
 * The article has no counterpart: this is a library convenience.  Some
 * callers run decode attention where they must not allocate device memory:
 * the enqueue step of an inference-engine plugin, a runtime whose memory is
 * planned up front and owned by someone else, code that may not grow the
 * process's footprint.  This entry point needs only the inputs and outputs.
 * Its scratch (status word, merge tickets, split partials) is a fixed device
 * array of FD_STATIC_WORKSPACE_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits; it calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * Arguments and results as fd_decode, without the workspace.  Returns
 * FD_ERR_WORKSPACE, before touching the GPU, when the plan for these
 * arguments needs more than FD_STATIC_WORKSPACE_BYTES (fd_plan reports the
 * need in fd_plan_info.workspace_bytes); use fd_decode with a workspace then.
 * The first call on a device looks up the array's device address with that
 * device current and caches it for the life of the process; make that first
 * call before any stream capture.  The cached address does not survive
 * cudaDeviceReset (or any other teardown of the device's primary context):
 * after one, this entry point must not be called again in the process.  Each call
 * clears the workspace header and the merge tickets on its stream before it runs.
 * All calls share the one array, which keeps the last call's contents: calls
 * that can overlap on the GPU (other streams, other host threads, without
 * ordering between them) race and give wrong results.  The status word is
 * not reachable from outside the library, so errors the kernels detect are
 * not reported by this entry point.
 */
#define FD_STATIC_WORKSPACE_BYTES (16 << 20)
int fd_decode_static_workspace(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                               const int32_t *kv_indptr_host, const int32_t *kv_indptr_dev,
                               const void *q, const void *k, const void *v, float scale,
                               float *o, float *lse, void *stream);

/*
 * fd_get_device_status -- synchronise the stream, read and clear the status
 * word the kernels write into the workspace.  Returns FD_OK,
 * FD_ERR_TIMEOUT, FD_ERR_DEVICE_BOUNDS, or FD_ERR_CUDA if the read failed.
 */
int fd_get_device_status(void *workspace, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FD_H */
