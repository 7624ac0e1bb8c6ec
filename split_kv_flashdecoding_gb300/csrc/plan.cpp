// plan.cpp -- host planner of libfd (no CUDA calls except the SM-count query).
//
// "FlashDecoding++: sequence-dimension KV split parallelism for LLM serving"
// (techknowgenie.com), §2 (sequence-split grid) and §6 (chunk size tuning
// guide: chunks small enough that the grid covers the SMs, large enough that
// stage 2 stays light).
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <utility>
#include <vector>

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

// Fixed cost of one CTA (launch, pipeline fill, epilogue), in units of the
// time one 32-key tile takes per resident CTA.
constexpr int64_t kCtaOverheadTiles = 3;

int64_t chunk_for_target(int64_t total, int num_kv_heads, int64_t target)
{
    int64_t c = round_up((total * num_kv_heads + target - 1) / target, FD_TILE_TOKENS);
    if (c < FD_MIN_CHUNK)
        c = FD_MIN_CHUNK;
    if (c > (1 << 30))
        c = 1 << 30;
    return c;
}

struct GridCost {
    int64_t ctas;          // CTAs of the grid
    int64_t total;         // sum of CTA costs
    int64_t largest;       // largest CTA cost
};

GridCost grid_cost(int batch, const int32_t *indptr, int num_kv_heads, int32_t c)
{
    GridCost g{0, 0, 0};
    for (int b = 0; b < batch; ++b) {
        const int32_t len = indptr[b + 1] - indptr[b];
        const int32_t n = fd::splits_for(len, c);
        if (n == 0)
            continue;
        const int32_t split_len = fd::split_len_for(len, n);
        const int32_t tail = len - (n - 1) * split_len;
        const int64_t full_cost = (split_len + FD_TILE_TOKENS - 1) / FD_TILE_TOKENS + kCtaOverheadTiles;
        const int64_t tail_cost = (tail + FD_TILE_TOKENS - 1) / FD_TILE_TOKENS + kCtaOverheadTiles;
        g.ctas += (int64_t)n * num_kv_heads;
        g.total += ((int64_t)(n - 1) * full_cost + tail_cost) * num_kv_heads;
        g.largest = std::max(g.largest, std::max(n > 1 ? full_cost : 0, tail_cost));
    }
    return g;
}

// Makespan, in tile units, of the split grid for chunk c: CTAs in launch order
// (request by request, split by split, KV head fastest) go to the earliest free
// of `slots` resident-CTA slots, as the hardware block scheduler does.  The
// slots are kept as (free time -> count), so a run of equal CTAs costs a few
// map operations.
int64_t simulate_makespan(int batch, const int32_t *indptr, int num_kv_heads, int32_t c,
                          int64_t slots)
{
    std::map<int64_t, int64_t> free_at{{0, slots}};
    std::vector<std::pair<int64_t, int64_t>> taken;
    for (int b = 0; b < batch; ++b) {
        const int32_t len = indptr[b + 1] - indptr[b];
        const int32_t n = fd::splits_for(len, c);
        if (n == 0)
            continue;
        const int32_t split_len = fd::split_len_for(len, n);
        for (int32_t s = 0; s < n; ++s) {
            const int32_t keys = std::min(split_len, len - s * split_len);
            const int64_t cost = (keys + FD_TILE_TOKENS - 1) / FD_TILE_TOKENS + kCtaOverheadTiles;
            int64_t need = num_kv_heads;   // the KV heads of one split, in a row
            taken.clear();
            while (need > 0) {
                if (free_at.empty()) {   // more KV heads than slots: reuse the first ones
                    for (const auto &t : taken)
                        free_at[t.first] += t.second;
                    taken.clear();
                }
                auto it = free_at.begin();
                const int64_t k = std::min(need, it->second);
                taken.emplace_back(it->first + cost, k);
                need -= k;
                if ((it->second -= k) == 0)
                    free_at.erase(it);
            }
            for (const auto &t : taken)
                free_at[t.first] += t.second;
        }
    }
    return free_at.rbegin()->first;
}

// Choose the chunk length: for each candidate grid of about 1, 2, 4 or 8
// waves of resident CTAs, estimate the makespan and keep the shortest (the
// fewest waves on a tie).  A grid that fits the slots takes as long as its
// largest CTA; otherwise the dispatch is simulated, unless the lower bound
// total / slots already rules the candidate out.  One wave is best when the
// requests split evenly; ragged batches gain from smaller chunks that even
// out the per-slot load.
int64_t choose_chunk(int batch, const int32_t *indptr, int num_kv_heads, int64_t slots)
{
    const int64_t total = indptr[batch];
    int64_t best_c = chunk_for_target(total, num_kv_heads, slots);
    int64_t best_t = -1, last_c = -1;
    for (int waves : {1, 2, 4, 8}) {
        const int64_t c = chunk_for_target(total, num_kv_heads, slots * waves);
        if (c == last_c)
            continue;
        last_c = c;
        const GridCost g = grid_cost(batch, indptr, num_kv_heads, (int32_t)c);
        int64_t t;
        if (g.ctas <= slots) {
            t = g.largest;
        } else {
            const int64_t lower = std::max(g.largest, (g.total + slots - 1) / slots);
            if (best_t >= 0 && lower >= best_t)
                continue;
            t = simulate_makespan(batch, indptr, num_kv_heads, (int32_t)c, slots);
        }
        if (best_t < 0 || t < best_t) {
            best_t = t;
            best_c = c;
        }
    }
    return best_c;
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
    if (c == 0)
        c = choose_chunk(batch, kv_indptr_host, num_kv_heads, (int64_t)num_sms * ctas_per_sm);

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
    // fd_decode workspace: status header, one merge ticket per (request, KV
    // head), partial LSE, partial O, one publication flag per split item.
    info->workspace_bytes = FD_WORKSPACE_HEADER_BYTES +
                            round_up((int64_t)batch * num_kv_heads * 4, 256) +
                            round_up(rows * 4, 256) + rows * head_dim * 4 + round_up(num_work * 4, 256);
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
