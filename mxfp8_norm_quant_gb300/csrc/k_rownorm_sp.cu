// The fused norm's two output forms for the sequence-parallel path (vLLM
// PR #65496, Details / Tradeoff): E4M3 codes with row-major scales, whose
// row shards concatenate after an all-gather and are swizzled once; and the
// norm alone rounded to BF16, quantised after the gather.  Same kernels and
// row ownership as the swizzled form (row_common.cuh); only the stores differ.
#include "row_common.cuh"

namespace mxk {

cudaError_t launch_rmsnorm_quant_rowmajor(const void* x, const void* w, float eps, uint8_t* q, uint8_t* sc, int M,
                                          int H, int num_sms, unsigned int* fault, cudaStream_t stream) {
  return dispatch_norm<OUT_MX_ROWMAJOR>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
}

cudaError_t launch_rmsnorm_bf16(const void* x, const void* w, float eps, void* y, int M, int H, int num_sms,
                                unsigned int* fault, cudaStream_t stream) {
  return dispatch_norm<OUT_BF16>(x, w, eps, static_cast<uint8_t*>(y), nullptr, M, H, num_sms, fault, stream);
}

}  // namespace mxk
