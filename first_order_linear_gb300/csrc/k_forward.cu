// Kernels of the forward scans (eligibility trace, episodic prefix sums) and
// of the generic affine scan.
#include "dispatch.cuh"

namespace rlca {
template cudaError_t run_scan<EligEst<>>(const EligEst<>&, const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<PrefixSumEst<uint32_t>>(const PrefixSumEst<uint32_t>&, const Plan&, const Geom&,
                                                      cudaStream_t);
template cudaError_t run_scan<PrefixSumEst<float>>(const PrefixSumEst<float>&, const Plan&, const Geom&,
                                                   cudaStream_t);
template cudaError_t run_scan<AffineEst<true>>(const AffineEst<true>&, const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<AffineEst<false>>(const AffineEst<false>&, const Plan&, const Geom&, cudaStream_t);
cudaError_t status_forward(unsigned int* word, bool clear) { return tu_status(word, clear); }
}  // namespace rlca
