// bfloat16-storage kernels of GAE and the discounted return.
#include "dispatch.cuh"

namespace rlca {
template cudaError_t run_scan<GaeEst<true, bf16>>(const GaeEst<true, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<GaeEst<false, bf16>>(const GaeEst<false, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<DiscEst<true, bf16>>(const DiscEst<true, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<DiscEst<false, bf16>>(const DiscEst<false, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
cudaError_t status_values_bf16_a(unsigned int* word, bool clear) { return tu_status(word, clear); }
}  // namespace rlca
