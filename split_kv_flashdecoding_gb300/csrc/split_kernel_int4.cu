// split_kernel_int4.cu -- stage 1 for INT4 K/V: the split kernels of
// split_kernel.cuh with the four-bit codes widened to f16 in registers.
//
// "FlashDecoding++: sequence-dimension KV split parallelism for LLM serving"
// (techknowgenie.com), §4 (quantisation-friendly fusion): INT4 K and V stay
// packed in HBM and are dequantised in the register file as they reach the
// tensor cores, so the stream moves about a quarter of the bytes of bf16.
// Each key row of each KV head carries its own K and V scale; the K scale
// multiplies the row's logit and the V scale its probability in P V, so the
// widening of the codes is the only dequantisation step on the operands, and
// it is exact (one lop3 and one f16 subtract or multiply-add per pair of codes;
// with the bf16 widening it replaced, which needed a shift per pair, the 64k
// step took 31.7 us instead of 26.8).  The stages are filled by 16-byte
// cp.async copies rather than TMA boxes (64-byte rows and 4-byte scales:
// measured faster on multi-wave plans, equal on one wave), made by the
// consumer warps themselves on ragged one-item calls and by the producer warp
// otherwise.
#include "split_kernel.cuh"

namespace fd {

cudaError_t launch_split_int4(const KvMaps &maps, const SplitParams &p, int group, int num_ctas,
                              cudaStream_t stream)
{
    return launch_split_dt<kKvInt4>(maps, p, group, num_ctas, stream);
}

}  // namespace fd
