// split_kernel.cu -- stage 1 for bf16 K/V (the templates are in
// split_kernel.cuh), and the K/V type dispatch of launch_split.
#include "split_kernel.cuh"

namespace fd {

int split_ctas_per_sm()
{
    return kMinCtas;
}

cudaError_t launch_split(const KvMaps &maps, const SplitParams &p, int group, int num_ctas,
                         cudaStream_t stream)
{
    switch (p.kv_type) {
    case kKvTypeBf16: return launch_split_dt<kKvBf16>(maps, p, group, num_ctas, stream);
    case kKvTypeFp8: return launch_split_fp8(maps, p, group, num_ctas, stream);
    case kKvTypeInt4: return launch_split_int4(maps, p, group, num_ctas, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace fd
