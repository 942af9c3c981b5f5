// Kernels of the value-target estimators: GAE, discounted return, TD(lambda),
// and the fused pass computing all three.
#include "dispatch.cuh"

namespace rlca {
template cudaError_t run_scan<GaeEst<true>>(const GaeEst<true>&, const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<GaeEst<false>>(const GaeEst<false>&, const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<DiscEst<true>>(const DiscEst<true>&, const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<DiscEst<false>>(const DiscEst<false>&, const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<TdLambdaEst<true>>(const TdLambdaEst<true>&, const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<TdLambdaEst<false>>(const TdLambdaEst<false>&, const Plan&, const Geom&,
                                                  cudaStream_t);
template cudaError_t run_scan<ValueTargetsEst<true>>(const ValueTargetsEst<true>&, const Plan&, const Geom&,
                                                     cudaStream_t);
template cudaError_t run_scan<ValueTargetsEst<false>>(const ValueTargetsEst<false>&, const Plan&, const Geom&,
                                                      cudaStream_t);
cudaError_t status_values(unsigned int* word, bool clear) { return tu_status(word, clear); }
}  // namespace rlca
