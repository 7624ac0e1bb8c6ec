// split_kernel_fp8.cu -- stage 1 for FP8 (E4M3) K/V: the split kernels of
// split_kernel.cuh with the K/V bytes widened to f16 in registers.
//
// "FlashDecoding++: sequence-dimension KV split parallelism for LLM serving"
// (techknowgenie.com), §4 (quantisation-friendly fusion): the quantised K and
// V are loaded from HBM as they are and dequantised on chip, in the register
// file, straight into tensor-core operands, so the stream moves half the
// bytes of bf16.  Here the per-KV-head scales of K and V are folded into the
// logit scale and into O; the E4M3 -> f16 widening itself is exact.
#include "split_kernel.cuh"

namespace fd {

cudaError_t launch_split_fp8(const KvMaps &maps, const SplitParams &p, int group, int num_ctas,
                             cudaStream_t stream)
{
    return launch_split_dt<kKvFp8>(maps, p, group, num_ctas, stream);
}

}  // namespace fd
