// bfloat16-storage kernels of TD(lambda) and the fused value targets.
#include "dispatch.cuh"

namespace rlca {
template cudaError_t run_scan<TdLambdaEst<true, bf16>>(const TdLambdaEst<true, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<TdLambdaEst<false, bf16>>(const TdLambdaEst<false, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<ValueTargetsEst<true, bf16>>(const ValueTargetsEst<true, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<ValueTargetsEst<false, bf16>>(const ValueTargetsEst<false, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
cudaError_t status_values_bf16_b(unsigned int* word, bool clear) { return tu_status(word, clear); }
}  // namespace rlca
