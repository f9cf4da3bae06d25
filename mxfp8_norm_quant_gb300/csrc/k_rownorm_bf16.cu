// The Gemma RMSNorm alone, rounded to BF16: the sequence-parallel path in
// which the norm output stays BF16 through the all-gather and is quantised
// after it (vLLM PR #65496, Overview and Details / Tradeoff).  Same kernels
// and row ownership as the quantising forms (row_common.cuh, row_lb.cuh);
// only the stores differ.
#include "row_lb.cuh"

namespace mxk {

cudaError_t launch_rmsnorm_bf16(const void* x, const void* w, float eps, void* y, int M, int H, int num_sms,
                                unsigned int* fault, cudaStream_t stream) {
  return dispatch_norm<OUT_BF16>(x, w, eps, static_cast<uint8_t*>(y), nullptr, M, H, num_sms, fault, stream);
}

}  // namespace mxk
