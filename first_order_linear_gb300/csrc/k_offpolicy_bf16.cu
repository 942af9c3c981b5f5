// bfloat16-storage kernels of V-Trace and Retrace(lambda).
#include "dispatch.cuh"

namespace rlca {
template cudaError_t run_scan<VtraceEst<true, bf16>>(const VtraceEst<true, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<VtraceEst<false, bf16>>(const VtraceEst<false, bf16>&,
    const Plan&, const Geom&, cudaStream_t);
template cudaError_t run_scan<RetraceEst<true, bf16>>(const RetraceEst<true, bf16>&, const Plan&, const Geom&,
                                                     cudaStream_t);
template cudaError_t run_scan<RetraceEst<false, bf16>>(const RetraceEst<false, bf16>&, const Plan&, const Geom&,
                                                      cudaStream_t);
cudaError_t status_offpolicy_bf16(unsigned int* word, bool clear) { return tu_status(word, clear); }
}  // namespace rlca
