// The fused norm with row-major scales, for the sequence-parallel path (vLLM
// PR #65496, Details / Tradeoff): E4M3 codes with [M][H/32] scales, whose row
// shards concatenate after an all-gather and are swizzled once.  Same kernels
// and row ownership as the swizzled form (row_common.cuh, row_lb.cuh); only
// the scale stores differ.  One output form per translation unit, so the
// forms compile in parallel.
#include "row_lb.cuh"

namespace mxk {

cudaError_t launch_rmsnorm_quant_rowmajor(const void* x, const void* w, float eps, uint8_t* q, uint8_t* sc, int M,
                                          int H, int num_sms, unsigned int* fault, cudaStream_t stream) {
  return dispatch_norm<OUT_MX_ROWMAJOR>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
}

}  // namespace mxk
