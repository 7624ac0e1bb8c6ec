// split_kernel.cu -- stage 1 for bf16 K/V (the templates are in
// split_kernel.cuh), and the dtype dispatch of launch_split.
#include "split_kernel.cuh"

namespace fd {

int split_ctas_per_sm()
{
    return kMinCtas;
}

cudaError_t launch_split(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const SplitParams &p,
                         int group, int num_ctas, cudaStream_t stream)
{
    if (p.kv_fp8)
        return launch_split_fp8(tm_k, tm_v, p, group, num_ctas, stream);
    return launch_split_dt<kKvBf16>(tm_k, tm_v, p, group, num_ctas, stream);
}

}  // namespace fd
