// bfloat16-storage kernels of the forward scans and the generic affine scan.
#include "dispatch.cuh"

namespace rlca {
template cudaError_t run_scan<EligEst<bf16>>(const EligEst<bf16>&, const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<PrefixSumEst<float, bf16>>(const PrefixSumEst<float, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<AffineEst<true, bf16>>(const AffineEst<true, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<AffineEst<false, bf16>>(const AffineEst<false, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
cudaError_t status_forward_bf16(unsigned int* word, bool clear) { return tu_status(word, clear); }
}  // namespace rlca
