// Kernels of the off-policy estimators: V-Trace, Retrace(lambda).
#include "dispatch.cuh"

namespace rlca {
template cudaError_t run_scan<VtraceEst<true>>(const VtraceEst<true>&, const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<VtraceEst<false>>(const VtraceEst<false>&, const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<RetraceEst<true>>(const RetraceEst<true>&, const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<RetraceEst<false>>(const RetraceEst<false>&, const Plan&, const Geom&,
                                                 cudaStream_t);
cudaError_t status_offpolicy(unsigned int* word, bool clear) { return tu_status(word, clear); }
}  // namespace rlca
