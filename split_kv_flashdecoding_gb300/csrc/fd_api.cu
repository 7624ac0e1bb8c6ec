// fd_api.cu -- the C ABI of libfd: argument checks, TMA descriptors and the
// launches of the two kernels.  See include/fd.h for the contract of each
// entry point.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <algorithm>
#include <vector>

#include "fd.h"
#include "kernels.h"

namespace {

constexpr int kHeadDim = 128;
constexpr int kBoxCols = 64;     // one 128-byte swizzle span of bf16
// Workspace header: the status word at byte 0, the split kernel's item-claim
// counter at byte 64 and its done counter at byte 128 (sectors of their own).
constexpr int kClaimOffset = 64;
constexpr int kDoneOffset = 128;
constexpr int kBoxRows = FD_TILE_TOKENS;

bool aligned(const void *p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

int64_t round_up(int64_t x, int64_t m)
{
    return (x + m - 1) / m * m;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// K or V [rows, Hkv, 128] bf16 (rows = T keys, or num_pages * page_size for a
// page pool) as a 3-D tensor (64 columns, rows, Hkv * 2 blocks of 64 columns),
// 128-byte swizzle, zero fill past the last row.  One box (64, box_rows, 2)
// brings both 64-column halves of one head's box_rows rows (32, or 16 for
// pages that are not a multiple of 32 keys) in one copy, laid out in shared
// memory as [half][row][64].  The block dimension comes last with a 128-byte
// stride, smaller than the row stride: TMA takes any 16-byte-multiple strides.
int make_kv_map(CUtensorMap *map, const void *base, int64_t rows, int num_kv_heads,
                int box_rows = kBoxRows)
{
    auto encode = tensor_map_encoder();
    if (!encode)
        return FD_ERR_CUDA;
    const cuuint64_t dims[3] = {kBoxCols, (cuuint64_t)rows, (cuuint64_t)num_kv_heads * 2};
    const cuuint64_t strides[2] = {(cuuint64_t)num_kv_heads * kHeadDim * 2, kBoxCols * 2};
    const cuuint32_t box[3] = {kBoxCols, (cuuint32_t)box_rows, 2};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base),
                              dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FD_OK : FD_ERR_INVALID_ARG;
}

// FP8 K or V [rows, Hkv, 128] (one byte per value) as a 2-D tensor of rows x
// Hkv*128 bytes; one box = box_rows rows x the head's 128 bytes, 128-byte
// swizzle, zero fill past the last row.
int make_kv_map_fp8(CUtensorMap *map, const void *base, int64_t rows, int num_kv_heads, int box_rows)
{
    auto encode = tensor_map_encoder();
    if (!encode)
        return FD_ERR_CUDA;
    const cuuint64_t dims[2] = {(cuuint64_t)num_kv_heads * kHeadDim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)num_kv_heads * kHeadDim};
    const cuuint32_t box[2] = {kHeadDim, (cuuint32_t)box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                              strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FD_OK : FD_ERR_INVALID_ARG;
}

int check_info(const fd_plan_info *info)
{
    if (!info)
        return FD_ERR_INVALID_ARG;
    if (info->head_dim != kHeadDim)
        return FD_ERR_UNSUPPORTED;
    if (info->batch < 0 || info->num_qo_heads <= 0 || info->num_kv_heads <= 0 ||
        info->num_qo_heads % info->num_kv_heads != 0 ||
        info->group_size != info->num_qo_heads / info->num_kv_heads)
        return FD_ERR_INVALID_ARG;
    const int g = info->group_size;
    if (g != 1 && g != 2 && g != 4 && g != 8)
        return FD_ERR_UNSUPPORTED;
    if (info->chunk <= 0 || info->chunk % FD_TILE_TOKENS != 0 || info->total_splits < 0 ||
        (int64_t)info->num_work != (int64_t)info->total_splits * info->num_kv_heads ||
        (int64_t)info->num_partial_rows != (int64_t)info->total_splits * info->num_qo_heads ||
        info->total_tokens < 0 || info->total_tokens > INT32_MAX)
        return FD_ERR_INVALID_ARG;
    return FD_OK;
}

cudaStream_t as_stream(void *s)
{
    return reinterpret_cast<cudaStream_t>(s);
}

// A token unique to each fused call (never 0, the value of a zeroed flag):
// the split kernel's CTAs publish their partial rows by writing it into their
// flags, so flags left by earlier calls never match.
int32_t next_call_token()
{
    static std::atomic<uint32_t> counter{0};
    uint32_t t = counter.fetch_add(1, std::memory_order_relaxed) + 1;
    if (t == 0)
        t = counter.fetch_add(1, std::memory_order_relaxed) + 1;
    return static_cast<int32_t>(t);
}

// Where fd_decode keeps its scratch in a workspace of a plan:
// status header | tickets [B * Hkv] | partial LSE | partial O | flags [num_work].
struct WorkspaceLayout {
    int *counters;
    float *partial_lse;
    float *partial_o;
    int *flags;
};

WorkspaceLayout workspace_layout(void *workspace, int64_t batch, int64_t num_kv_heads,
                                 int64_t num_partial_rows)
{
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    WorkspaceLayout l;
    l.counters = reinterpret_cast<int *>(ws + FD_WORKSPACE_HEADER_BYTES);
    uint8_t *after = ws + FD_WORKSPACE_HEADER_BYTES + round_up(batch * num_kv_heads * 4, 256);
    l.partial_lse = reinterpret_cast<float *>(after);
    uint8_t *po = after + round_up(num_partial_rows * 4, 256);
    l.partial_o = reinterpret_cast<float *>(po);
    l.flags = reinterpret_cast<int *>(po + num_partial_rows * kHeadDim * 4);
    return l;
}

}  // namespace

extern "C" const char *fd_status_string(int status)
{
    switch (status) {
    case FD_OK: return "FD_OK";
    case FD_ERR_INVALID_ARG: return "FD_ERR_INVALID_ARG";
    case FD_ERR_UNSUPPORTED: return "FD_ERR_UNSUPPORTED";
    case FD_ERR_WORKSPACE: return "FD_ERR_WORKSPACE";
    case FD_ERR_CUDA: return "FD_ERR_CUDA";
    case FD_ERR_TIMEOUT: return "FD_ERR_TIMEOUT";
    case FD_ERR_DEVICE_BOUNDS: return "FD_ERR_DEVICE_BOUNDS";
    default: return "FD_ERR_UNKNOWN";
    }
}

extern "C" int fd_version(void)
{
    return 100;   // 0.1.0
}

extern "C" int fd_num_sms(int device, int *num_sms)
{
    static int cache[64] = {};
    if (!num_sms)
        return FD_ERR_INVALID_ARG;
    if (device < 0 && cudaGetDevice(&device) != cudaSuccess)
        return FD_ERR_CUDA;
    if (device < 64 && cache[device] > 0) {
        *num_sms = cache[device];
        return FD_OK;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0)
        return FD_ERR_CUDA;
    if (device < 64)
        cache[device] = n;
    *num_sms = n;
    return FD_OK;
}

namespace {

// Quantised K/V: the element type (fd::kKvTypeFp8 or fd::kKvTypeInt4) and the
// device scales -- FP8: [Hkv] each; INT4: [Hkv][rows] each.
struct QuantKV {
    int type;
    const float *k_scale;
    const float *v_scale;
};

// The page-pool description of a paged KV cache (see fd_decode_paged).
struct PagedKV {
    int32_t page_size;
    int32_t num_pages;
    const int32_t *last_len_dev;
    const int32_t *last_len_host;
    const int32_t *page_indices_dev;
    int32_t num_page_entries;   // kv_page_indptr[batch]
};

// Stage 1 launch shared by fd_decode_split (partials only), fd_decode and
// fd_decode_paged (stage 2 fused into the split kernel: o/lse/counters
// non-null).  kv_indptr_* is the key-row prefix, or the page-list prefix when
// `paged` is given.

int launch_stage1(const fd_plan_info *info, const void *q, const void *k, const void *v,
                  const int32_t *kv_indptr_dev, float scale, float *partial_o, float *partial_lse,
                  void *workspace, float *o, float *lse, int *counters,
                  const int32_t *kv_indptr_host, cudaStream_t stream,
                  const PagedKV *paged = nullptr, const QuantKV *quant = nullptr,
                  bool device_plan = false, int *flags = nullptr)
{
    if (!q || !k || !v || !kv_indptr_dev || !partial_o || !partial_lse)
        return FD_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(partial_o, 16) ||
        !aligned(partial_lse, 4) || !aligned(kv_indptr_dev, 4) || !aligned(workspace, 16))
        return FD_ERR_INVALID_ARG;
    if (!(scale == scale))
        return FD_ERR_INVALID_ARG;
    const int kv_type = quant ? quant->type : fd::kKvTypeBf16;
    if (quant && (!quant->k_scale || !quant->v_scale || !aligned(quant->k_scale, 4) ||
                  !aligned(quant->v_scale, 4)))
        return FD_ERR_INVALID_ARG;

    fd::KvMaps maps;
    memset(&maps, 0, sizeof maps);   // INT4: loaded without tensor maps
    int rc;
    const int64_t rows = paged ? (int64_t)paged->num_pages * paged->page_size : info->total_tokens;
    const int box_rows = paged && paged->page_size % kBoxRows != 0 ? 16 : kBoxRows;
    if (kv_type == fd::kKvTypeFp8) {
        if ((rc = make_kv_map_fp8(&maps.k, k, rows, info->num_kv_heads, box_rows)) != FD_OK ||
            (rc = make_kv_map_fp8(&maps.v, v, rows, info->num_kv_heads, box_rows)) != FD_OK)
            return rc;
    } else if (kv_type == fd::kKvTypeBf16) {
        if ((rc = make_kv_map(&maps.k, k, rows, info->num_kv_heads, box_rows)) != FD_OK ||
            (rc = make_kv_map(&maps.v, v, rows, info->num_kv_heads, box_rows)) != FD_OK)
            return rc;
    }

    fd::SplitParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.kv_indptr = kv_indptr_dev;
    p.partial_o = partial_o;
    p.partial_lse = partial_lse;
    p.status = static_cast<int *>(workspace);
    p.claim = reinterpret_cast<int *>(static_cast<uint8_t *>(workspace) + kClaimOffset);
    p.done = reinterpret_cast<int *>(static_cast<uint8_t *>(workspace) + kDoneOffset);
    p.device_plan = device_plan;
    p.batch = info->batch;
    p.num_qo_heads = info->num_qo_heads;
    p.num_kv_heads = info->num_kv_heads;
    p.chunk = info->chunk;
    p.num_partial_rows = info->num_partial_rows;
    p.total_tokens = (int32_t)info->total_tokens;
    p.q_scale = scale * 1.4426950408889634f;
    p.timeout_ns = info->timeout_ns;
    p.fuse_merge = counters != nullptr;
    p.o = o;
    p.lse = lse;
    p.counters = counters;
    p.flags = counters && !device_plan ? flags : nullptr;
    p.token = p.flags ? next_call_token() : 0;
    // kv_indptr_host is only known on the fd_decode path (the same values as
    // the device copy, by contract).
    p.indptr_in_params = kv_indptr_host && info->batch + 1 <= fd::kParamIndptr &&
                         (!paged || paged->last_len_host);
    memset(p.indptr_param, 0, sizeof p.indptr_param);
    memset(p.last_len_param, 0, sizeof p.last_len_param);
    if (p.indptr_in_params)
        memcpy(p.indptr_param, kv_indptr_host, (size_t)(info->batch + 1) * sizeof(int32_t));
    p.kv_last_len = paged ? paged->last_len_dev : nullptr;
    p.page_indices = paged ? paged->page_indices_dev : nullptr;
    p.page_size = paged ? paged->page_size : 0;
    p.box_rows = box_rows;
    p.num_pages = paged ? paged->num_pages : 0;
    p.num_page_entries = paged ? paged->num_page_entries : 0;
    if (paged && p.indptr_in_params)
        memcpy(p.last_len_param, paged->last_len_host, (size_t)info->batch * sizeof(int32_t));
    p.kv_type = kv_type;
    p.kv_rows = (int32_t)rows;
    p.k_data = static_cast<const uint8_t *>(k);
    p.v_data = static_cast<const uint8_t *>(v);
    p.k_scale = quant ? quant->k_scale : nullptr;
    p.v_scale = quant ? quant->v_scale : nullptr;
    // Persistent grid: at most one wave of resident CTAs on the plan's SMs.
    p.num_work = info->num_work;
    const int64_t slots = (int64_t)info->num_sms * fd::split_ctas_per_sm();
    const int num_ctas = slots > 0 && slots < info->num_work ? (int)slots : info->num_work;
    const cudaError_t e = fd::launch_split(maps, p, info->group_size, num_ctas, stream);
    return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

}  // namespace

extern "C" int fd_decode_split(const fd_plan_info *info, const void *q, const void *k,
                               const void *v, const int32_t *kv_indptr_dev, float scale,
                               float *partial_o, float *partial_lse, void *workspace,
                               int64_t workspace_bytes, void *stream)
{
    const int rc = check_info(info);
    if (rc != FD_OK)
        return rc;
    if (!workspace || workspace_bytes < FD_WORKSPACE_HEADER_BYTES)
        return FD_ERR_WORKSPACE;
    if (info->num_work == 0)
        return FD_OK;
    return launch_stage1(info, q, k, v, kv_indptr_dev, scale, partial_o, partial_lse, workspace,
                         nullptr, nullptr, nullptr, nullptr, as_stream(stream));
}

extern "C" int fd_merge(const fd_plan_info *info, const int32_t *kv_indptr_dev,
                        const float *partial_o, const float *partial_lse, float *o, float *lse,
                        void *workspace, int64_t workspace_bytes, void *stream)
{
    const int rc = check_info(info);
    if (rc != FD_OK)
        return rc;
    if (!workspace || workspace_bytes < FD_WORKSPACE_HEADER_BYTES)
        return FD_ERR_WORKSPACE;
    if (info->batch == 0)
        return FD_OK;
    if (!kv_indptr_dev || !o || !lse || (info->num_partial_rows > 0 && (!partial_o || !partial_lse)))
        return FD_ERR_INVALID_ARG;
    if (!aligned(o, 16) || !aligned(lse, 4) || !aligned(partial_o, 16) ||
        !aligned(partial_lse, 4) || !aligned(kv_indptr_dev, 4) || !aligned(workspace, 16))
        return FD_ERR_INVALID_ARG;
    fd::MergeParams p;
    p.kv_indptr = kv_indptr_dev;
    p.partial_o = partial_o;
    p.partial_lse = partial_lse;
    p.o = o;
    p.lse = lse;
    p.status = static_cast<int *>(workspace);
    p.batch = info->batch;
    p.num_qo_heads = info->num_qo_heads;
    p.chunk = info->chunk;
    p.num_partial_rows = info->num_partial_rows;
    p.only_empty = 0;
    p.kv_last_len = nullptr;
    p.page_size = 0;
    const cudaError_t e = fd::launch_merge(p, as_stream(stream));
    return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

namespace {

// fd_decode, fd_decode_fp8 and fd_decode_int4 (quant non-null).
int decode_ragged(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                  const int32_t *kv_indptr_host, const int32_t *kv_indptr_dev, const void *q,
                  const void *k, const void *v, float scale, float *o, float *lse, void *workspace,
                  int64_t workspace_bytes, void *stream, const QuantKV *quant)
{
    fd_plan_info info;
    int rc = fd_plan(batch, num_qo_heads, num_kv_heads, head_dim, kv_indptr_host, 0, 0, 0, &info);
    if (rc != FD_OK)
        return rc;
    if (!workspace || workspace_bytes < info.workspace_bytes)
        return FD_ERR_WORKSPACE;
    if (batch == 0)
        return FD_OK;
    if (!o || !lse || !aligned(o, 16) || !aligned(lse, 4) || !kv_indptr_dev)
        return FD_ERR_INVALID_ARG;
    const WorkspaceLayout wl = workspace_layout(workspace, batch, num_kv_heads, info.num_partial_rows);
    int *counters = wl.counters;
    float *partial_lse = wl.partial_lse;
    float *partial_o = wl.partial_o;
    cudaStream_t s = as_stream(stream);
    if (info.num_work > 0) {
        rc = launch_stage1(&info, q, k, v, kv_indptr_dev, scale, partial_o, partial_lse, workspace,
                           o, lse, counters, kv_indptr_host, s, nullptr, quant, false, wl.flags);
        if (rc != FD_OK)
            return rc;
    }
    // Stage 2 is fused into the split kernel; only requests with no keys (no
    // CTA of their own) still need their O = 0, LSE = -inf rows written.
    bool any_empty = false;
    for (int b = 0; b < batch && !any_empty; ++b)
        any_empty = kv_indptr_host[b + 1] == kv_indptr_host[b];
    if (!any_empty)
        return FD_OK;
    fd::MergeParams p;
    p.kv_indptr = kv_indptr_dev;
    p.partial_o = partial_o;
    p.partial_lse = partial_lse;
    p.o = o;
    p.lse = lse;
    p.status = static_cast<int *>(workspace);
    p.batch = info.batch;
    p.num_qo_heads = info.num_qo_heads;
    p.chunk = info.chunk;
    p.num_partial_rows = info.num_partial_rows;
    p.only_empty = 1;
    p.kv_last_len = nullptr;
    p.page_size = 0;
    return fd::launch_merge(p, s) == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

// Host checks of a paged layout; fills the logical key-row prefix (keys of
// request b = (pages_b - 1) * page_size + last_len_b) for the planner.
int paged_logical_indptr(int batch, int page_size, const int32_t *page_indptr,
                         const int32_t *last_len, std::vector<int32_t> &indptr)
{
    if (batch < 0 || !page_indptr || (batch > 0 && !last_len))
        return FD_ERR_INVALID_ARG;
    if (page_size <= 0 || page_size % 16 != 0)
        return FD_ERR_UNSUPPORTED;
    if (page_indptr[0] != 0)
        return FD_ERR_INVALID_ARG;
    indptr.assign((size_t)batch + 1, 0);
    int64_t total = 0;
    for (int b = 0; b < batch; ++b) {
        const int32_t pages = page_indptr[b + 1] - page_indptr[b];
        if (pages < 0)
            return FD_ERR_INVALID_ARG;
        if (pages > 0 && (last_len[b] < 1 || last_len[b] > page_size))
            return FD_ERR_INVALID_ARG;
        total += pages > 0 ? (int64_t)(pages - 1) * page_size + last_len[b] : 0;
        if (total > INT32_MAX)
            return FD_ERR_INVALID_ARG;
        indptr[b + 1] = (int32_t)total;
    }
    return FD_OK;
}

}  // namespace

extern "C" int fd_plan_paged(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                             int page_size, const int32_t *kv_page_indptr_host,
                             const int32_t *kv_last_page_len_host, int num_sms, int ctas_per_sm,
                             int chunk, fd_plan_info *info)
{
    std::vector<int32_t> indptr;
    const int rc = paged_logical_indptr(batch, page_size, kv_page_indptr_host,
                                        kv_last_page_len_host, indptr);
    if (rc != FD_OK)
        return rc;
    return fd_plan(batch, num_qo_heads, num_kv_heads, head_dim, indptr.data(), num_sms,
                   ctas_per_sm, chunk, info);
}

namespace {

// fd_decode_paged, fd_decode_paged_fp8 and fd_decode_paged_int4 (quant non-null).
int decode_paged(int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                 int num_pages, const int32_t *kv_page_indptr_host,
                 const int32_t *kv_last_page_len_host, const int32_t *kv_page_indptr_dev,
                 const int32_t *kv_last_page_len_dev, const int32_t *kv_page_indices_dev,
                 const void *q, const void *k_pages, const void *v_pages, float scale, float *o,
                 float *lse, void *workspace, int64_t workspace_bytes, void *stream,
                 const QuantKV *quant)
{
    fd_plan_info info;
    int rc = fd_plan_paged(batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                           kv_page_indptr_host, kv_last_page_len_host, 0, 0, 0, &info);
    if (rc != FD_OK)
        return rc;
    if (!workspace || workspace_bytes < info.workspace_bytes)
        return FD_ERR_WORKSPACE;
    if (batch == 0)
        return FD_OK;
    if (!o || !lse || !aligned(o, 16) || !aligned(lse, 4) || !kv_page_indptr_dev ||
        !kv_last_page_len_dev || !aligned(kv_last_page_len_dev, 4) ||
        (info.num_work > 0 && (!kv_page_indices_dev || !aligned(kv_page_indices_dev, 4))))
        return FD_ERR_INVALID_ARG;
    if (num_pages <= 0 || (int64_t)num_pages * page_size > INT32_MAX)
        return FD_ERR_INVALID_ARG;
    const WorkspaceLayout wl = workspace_layout(workspace, batch, num_kv_heads, info.num_partial_rows);
    int *counters = wl.counters;
    float *partial_lse = wl.partial_lse;
    float *partial_o = wl.partial_o;
    cudaStream_t s = as_stream(stream);
    if (info.num_work > 0) {
        const PagedKV pk{page_size, num_pages, kv_last_page_len_dev, kv_last_page_len_host,
                         kv_page_indices_dev, kv_page_indptr_host[batch]};
        rc = launch_stage1(&info, q, k_pages, v_pages, kv_page_indptr_dev, scale, partial_o,
                           partial_lse, workspace, o, lse, counters, kv_page_indptr_host, s, &pk,
                           quant, false, wl.flags);
        if (rc != FD_OK)
            return rc;
    }
    bool any_empty = false;
    for (int b = 0; b < batch && !any_empty; ++b)
        any_empty = kv_page_indptr_host[b + 1] == kv_page_indptr_host[b];
    if (!any_empty)
        return FD_OK;
    fd::MergeParams p;
    p.kv_indptr = kv_page_indptr_dev;
    p.partial_o = partial_o;
    p.partial_lse = partial_lse;
    p.o = o;
    p.lse = lse;
    p.status = static_cast<int *>(workspace);
    p.batch = info.batch;
    p.num_qo_heads = info.num_qo_heads;
    p.chunk = info.chunk;
    p.num_partial_rows = info.num_partial_rows;
    p.only_empty = 1;
    p.kv_last_len = kv_last_page_len_dev;
    p.page_size = page_size;
    return fd::launch_merge(p, s) == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

}  // namespace

extern "C" int fd_decode(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                         const int32_t *kv_indptr_host, const int32_t *kv_indptr_dev,
                         const void *q, const void *k, const void *v, float scale, float *o,
                         float *lse, void *workspace, int64_t workspace_bytes, void *stream)
{
    return decode_ragged(batch, num_qo_heads, num_kv_heads, head_dim, kv_indptr_host, kv_indptr_dev,
                         q, k, v, scale, o, lse, workspace, workspace_bytes, stream, nullptr);
}

extern "C" int fd_decode_fp8(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                             const int32_t *kv_indptr_host, const int32_t *kv_indptr_dev,
                             const void *q, const void *k_fp8, const void *v_fp8,
                             const float *k_scale, const float *v_scale, float scale, float *o,
                             float *lse, void *workspace, int64_t workspace_bytes, void *stream)
{
    const QuantKV f{fd::kKvTypeFp8, k_scale, v_scale};
    return decode_ragged(batch, num_qo_heads, num_kv_heads, head_dim, kv_indptr_host, kv_indptr_dev,
                         q, k_fp8, v_fp8, scale, o, lse, workspace, workspace_bytes, stream, &f);
}

extern "C" int fd_decode_int4(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                              const int32_t *kv_indptr_host, const int32_t *kv_indptr_dev,
                              const void *q, const void *k_int4, const void *v_int4,
                              const float *k_scale, const float *v_scale, float scale, float *o,
                              float *lse, void *workspace, int64_t workspace_bytes, void *stream)
{
    const QuantKV f{fd::kKvTypeInt4, k_scale, v_scale};
    return decode_ragged(batch, num_qo_heads, num_kv_heads, head_dim, kv_indptr_host, kv_indptr_dev,
                         q, k_int4, v_int4, scale, o, lse, workspace, workspace_bytes, stream, &f);
}

extern "C" int fd_decode_paged(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                               int page_size, int num_pages, const int32_t *kv_page_indptr_host,
                               const int32_t *kv_last_page_len_host,
                               const int32_t *kv_page_indptr_dev,
                               const int32_t *kv_last_page_len_dev,
                               const int32_t *kv_page_indices_dev, const void *q,
                               const void *k_pages, const void *v_pages, float scale, float *o,
                               float *lse, void *workspace, int64_t workspace_bytes, void *stream)
{
    return decode_paged(batch, num_qo_heads, num_kv_heads, head_dim, page_size, num_pages,
                        kv_page_indptr_host, kv_last_page_len_host, kv_page_indptr_dev,
                        kv_last_page_len_dev, kv_page_indices_dev, q, k_pages, v_pages, scale, o,
                        lse, workspace, workspace_bytes, stream, nullptr);
}

extern "C" int fd_decode_paged_fp8(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                                   int page_size, int num_pages, const int32_t *kv_page_indptr_host,
                                   const int32_t *kv_last_page_len_host,
                                   const int32_t *kv_page_indptr_dev,
                                   const int32_t *kv_last_page_len_dev,
                                   const int32_t *kv_page_indices_dev, const void *q,
                                   const void *k_pages_fp8, const void *v_pages_fp8,
                                   const float *k_scale, const float *v_scale, float scale,
                                   float *o, float *lse, void *workspace, int64_t workspace_bytes,
                                   void *stream)
{
    const QuantKV f{fd::kKvTypeFp8, k_scale, v_scale};
    return decode_paged(batch, num_qo_heads, num_kv_heads, head_dim, page_size, num_pages,
                        kv_page_indptr_host, kv_last_page_len_host, kv_page_indptr_dev,
                        kv_last_page_len_dev, kv_page_indices_dev, q, k_pages_fp8, v_pages_fp8,
                        scale, o, lse, workspace, workspace_bytes, stream, &f);
}

extern "C" int fd_decode_paged_int4(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                                    int page_size, int num_pages,
                                    const int32_t *kv_page_indptr_host,
                                    const int32_t *kv_last_page_len_host,
                                    const int32_t *kv_page_indptr_dev,
                                    const int32_t *kv_last_page_len_dev,
                                    const int32_t *kv_page_indices_dev, const void *q,
                                    const void *k_pages_int4, const void *v_pages_int4,
                                    const float *k_scale, const float *v_scale, float scale,
                                    float *o, float *lse, void *workspace, int64_t workspace_bytes,
                                    void *stream)
{
    const QuantKV f{fd::kKvTypeInt4, k_scale, v_scale};
    return decode_paged(batch, num_qo_heads, num_kv_heads, head_dim, page_size, num_pages,
                        kv_page_indptr_host, kv_last_page_len_host, kv_page_indptr_dev,
                        kv_last_page_len_dev, kv_page_indices_dev, q, k_pages_int4, v_pages_int4,
                        scale, o, lse, workspace, workspace_bytes, stream, &f);
}

extern "C" int fd_plan_graph(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                             int64_t max_total_tokens, int num_sms, int chunk, fd_plan_info *info)
{
    if (!info || batch < 0 || max_total_tokens < 0 || max_total_tokens > INT32_MAX)
        return FD_ERR_INVALID_ARG;
    // The chunk: the caller's, or the planner's choice for the capacity spread
    // evenly over the batch.
    std::vector<int32_t> even((size_t)batch + 1, 0);
    for (int b = 1; b <= batch; ++b)
        even[b] = (int32_t)(max_total_tokens * b / batch);
    fd_plan_info base;
    int rc = fd_plan(batch, num_qo_heads, num_kv_heads, head_dim, even.data(), num_sms, 0, chunk,
                     &base);
    if (rc != FD_OK)
        return rc;
    // Capacity: a request of L keys has ceil(L / C) < L / C + 1 splits and an
    // empty one has one (it writes O = 0, LSE = -inf), so a batch of at most T
    // keys has at most floor(T / C) + B splits.
    const int64_t splits = max_total_tokens / base.chunk + batch;
    if (splits * num_qo_heads > INT32_MAX)
        return FD_ERR_INVALID_ARG;
    *info = base;
    info->total_splits = (int32_t)splits;
    info->max_splits = (int32_t)std::max<int64_t>(1, (max_total_tokens + base.chunk - 1) / base.chunk);
    info->num_work = (int32_t)(splits * num_kv_heads);
    info->num_partial_rows = (int32_t)(splits * num_qo_heads);
    info->total_tokens = max_total_tokens;
    info->workspace_bytes = FD_WORKSPACE_HEADER_BYTES + round_up((int64_t)batch * num_kv_heads * 4, 256) +
                            round_up((int64_t)info->num_partial_rows * 4, 256) +
                            (int64_t)info->num_partial_rows * kHeadDim * 4;
    return FD_OK;
}

extern "C" int fd_decode_graph(const fd_plan_info *info, const int32_t *kv_indptr_dev,
                               const void *q, const void *k, const void *v, float scale, float *o,
                               float *lse, void *workspace, int64_t workspace_bytes, void *stream)
{
    int rc = check_info(info);
    if (rc != FD_OK)
        return rc;
    if (!workspace || workspace_bytes < info->workspace_bytes)
        return FD_ERR_WORKSPACE;
    if (info->batch == 0 || info->num_work == 0)
        return FD_OK;
    if (!o || !lse || !aligned(o, 16) || !aligned(lse, 4) || !kv_indptr_dev)
        return FD_ERR_INVALID_ARG;
    const WorkspaceLayout wl =
        workspace_layout(workspace, info->batch, info->num_kv_heads, info->num_partial_rows);
    return launch_stage1(info, q, k, v, kv_indptr_dev, scale, wl.partial_o, wl.partial_lse, workspace,
                         o, lse, wl.counters, nullptr, as_stream(stream), nullptr, nullptr, true);
}

extern "C" int fd_merge_states(int num_states, int rows, int head_dim, const float *o_states,
                               const float *lse_states, float *o, float *lse, void *stream)
{
    if (head_dim != kHeadDim)
        return FD_ERR_UNSUPPORTED;
    if (num_states < 1 || rows < 0 || (int64_t)num_states * rows > INT32_MAX)
        return FD_ERR_INVALID_ARG;
    if (rows == 0)
        return FD_OK;
    if (!o_states || !lse_states || !o || !lse || !aligned(o_states, 16) || !aligned(o, 16) ||
        !aligned(lse_states, 4) || !aligned(lse, 4))
        return FD_ERR_INVALID_ARG;
    const cudaError_t e =
        fd::launch_merge_states(num_states, rows, o_states, lse_states, o, lse, as_stream(stream));
    return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

extern "C" int fd_get_device_status(void *workspace, void *stream)
{
    if (!workspace)
        return FD_ERR_WORKSPACE;
    int status = 0;
    cudaStream_t s = as_stream(stream);
    if (cudaMemcpyAsync(&status, workspace, sizeof status, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return FD_ERR_CUDA;
    if (status != 0) {
        if (cudaMemsetAsync(workspace, 0, sizeof status, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return FD_ERR_CUDA;
    }
    return status;
}
