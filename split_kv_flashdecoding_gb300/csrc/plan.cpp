// plan.cpp -- host planner of libfd (no CUDA calls except the SM-count query).
//
// "FlashDecoding++: sequence-dimension KV split parallelism for LLM serving"
// (techknowgenie.com), §2 (sequence-split grid) and §6 (chunk size tuning
// guide: chunks small enough that the grid covers the SMs, large enough that
// stage 2 stays light).
#include <stdint.h>
#include <string.h>

#include "fd.h"
#include "plan_rule.h"

namespace fd {
int split_ctas_per_sm();   // resident CTAs per SM of the split kernel's launch shape
}

namespace {

bool supported_group(int g)
{
    return g == 1 || g == 2 || g == 4 || g == 8;
}

int64_t round_up(int64_t x, int64_t m)
{
    return (x + m - 1) / m * m;
}

}  // namespace

extern "C" int fd_plan(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                       const int32_t *kv_indptr_host, int num_sms, int ctas_per_sm,
                       int chunk, fd_plan_info *info)
{
    if (!info || batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || !kv_indptr_host)
        return FD_ERR_INVALID_ARG;
    if (num_qo_heads % num_kv_heads != 0)
        return FD_ERR_INVALID_ARG;
    if (ctas_per_sm < 0 || ctas_per_sm > 64 || num_sms < 0 || chunk < 0)
        return FD_ERR_INVALID_ARG;
    if (chunk > 0 && (chunk % FD_TILE_TOKENS != 0 || chunk > (1 << 30)))
        return FD_ERR_INVALID_ARG;
    if (kv_indptr_host[0] != 0)
        return FD_ERR_INVALID_ARG;
    for (int b = 0; b < batch; ++b)
        if (kv_indptr_host[b + 1] < kv_indptr_host[b])
            return FD_ERR_INVALID_ARG;
    const int group = num_qo_heads / num_kv_heads;
    if (head_dim != 128 || !supported_group(group))
        return FD_ERR_UNSUPPORTED;

    if (num_sms == 0) {
        const int rc = fd_num_sms(-1, &num_sms);
        if (rc != FD_OK)
            return rc;
    }
    if (ctas_per_sm == 0)
        ctas_per_sm = fd::split_ctas_per_sm();

    const int64_t total = kv_indptr_host[batch];
    int64_t c = chunk;
    if (c == 0) {
        const int64_t target = (int64_t)num_sms * ctas_per_sm;
        c = round_up((total * num_kv_heads + target - 1) / target, FD_TILE_TOKENS);
        if (c < FD_MIN_CHUNK)
            c = FD_MIN_CHUNK;
        if (c > (1 << 30))
            c = 1 << 30;
    }

    int64_t total_splits = 0;
    int32_t max_splits = 0;
    for (int b = 0; b < batch; ++b) {
        const int32_t n = fd::splits_for(kv_indptr_host[b + 1] - kv_indptr_host[b], (int32_t)c);
        total_splits += n;
        if (n > max_splits)
            max_splits = n;
    }
    const int64_t num_work = total_splits * num_kv_heads;
    const int64_t rows = total_splits * num_qo_heads;
    if (num_work > INT32_MAX || rows > INT32_MAX / head_dim)
        return FD_ERR_INVALID_ARG;

    memset(info, 0, sizeof *info);
    info->batch = batch;
    info->num_qo_heads = num_qo_heads;
    info->num_kv_heads = num_kv_heads;
    info->head_dim = head_dim;
    info->group_size = group;
    info->chunk = (int32_t)c;
    info->total_splits = (int32_t)total_splits;
    info->max_splits = max_splits;
    info->num_work = (int32_t)num_work;
    info->num_partial_rows = (int32_t)rows;
    info->num_sms = num_sms;
    info->ctas_per_sm = ctas_per_sm;
    info->total_tokens = total;
    info->workspace_bytes = FD_WORKSPACE_HEADER_BYTES + round_up(rows * 4, 256) +
                            rows * head_dim * 4;
    info->timeout_ns = FD_DEFAULT_TIMEOUT_NS;
    return FD_OK;
}

extern "C" int fd_plan_work_items(const fd_plan_info *info, const int32_t *kv_indptr_host,
                                  int32_t *items, int64_t capacity)
{
    if (!info || !kv_indptr_host || (!items && info->num_work > 0))
        return FD_ERR_INVALID_ARG;
    if (capacity < info->num_work || info->chunk <= 0)
        return FD_ERR_INVALID_ARG;
    // CTA w handles global split j = w / Hkv of KV head w % Hkv; global splits
    // are numbered request by request.
    int64_t w = 0;
    for (int b = 0; b < info->batch; ++b) {
        const int32_t beg = kv_indptr_host[b], end = kv_indptr_host[b + 1];
        const int32_t n = fd::splits_for(end - beg, info->chunk);
        if (n == 0)
            continue;
        const int32_t len = fd::split_len_for(end - beg, n);
        for (int32_t s = 0; s < n; ++s) {
            const int32_t t0 = beg + s * len;
            const int32_t t1 = t0 + len < end ? t0 + len : end;
            for (int h = 0; h < info->num_kv_heads; ++h, ++w) {
                if (w >= info->num_work)
                    return FD_ERR_INVALID_ARG;
                int32_t *it = items + 5 * w;
                it[0] = b;
                it[1] = h;
                it[2] = s;
                it[3] = t0;
                it[4] = t1;
            }
        }
    }
    return w == info->num_work ? FD_OK : FD_ERR_INVALID_ARG;
}
