// Internal launchers behind the C ABI (host code, not exported).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mxk {

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device; the CUDA call is made only when the limit grows.
cudaError_t set_smem_once(const void* kernel, int bytes);

// Launch attributes shared by every kernel of the library: programmatic
// stream serialisation (the kernel's set-up overlaps the previous kernel of
// the stream; the kernels wait on griddepcontrol before touching global
// memory) and, when cluster_x > 1, the cluster shape.
struct LaunchAttrs {
  cudaLaunchAttribute a[2];
  cudaLaunchConfig_t cfg;
  LaunchAttrs(dim3 grid, dim3 block, size_t smem, cudaStream_t stream, unsigned cluster_x = 1) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a[0].val.programmaticStreamSerializationAllowed = 1;
    int n = 1;
    if (cluster_x > 1) {
      a[1].id = cudaLaunchAttributeClusterDimension;
      a[1].val.clusterDim.x = cluster_x;
      a[1].val.clusterDim.y = 1;
      a[1].val.clusterDim.z = 1;
      n = 2;
    }
    cfg.attrs = a;
    cfg.numAttrs = n;
  }
};

cudaError_t launch_rmsnorm_quant(const void* x, const void* w, float eps, uint8_t* q, uint8_t* sc, int M, int H,
                                 int num_sms, unsigned int* fault, cudaStream_t stream);
// the lane-block norm with its row copies withheld, so that every wait for a
// row runs out after wait_ns (failure-handling self-test)
cudaError_t launch_rmsnorm_quant_stalled(const void* x, const void* w, float eps, uint8_t* q, uint8_t* sc, int M,
                                         int H, int num_sms, unsigned int* fault, unsigned long long wait_ns,
                                         cudaStream_t stream);
// the same norm with row-major [M][H/32] scales, and with a bf16 [M][H] output
cudaError_t launch_rmsnorm_quant_rowmajor(const void* x, const void* w, float eps, uint8_t* q, uint8_t* sc, int M,
                                          int H, int num_sms, unsigned int* fault, cudaStream_t stream);
cudaError_t launch_rmsnorm_bf16(const void* x, const void* w, float eps, void* y, int M, int H, int num_sms,
                                unsigned int* fault, cudaStream_t stream);
cudaError_t launch_quant(const void* x, uint8_t* q, uint8_t* sc, int rows, int cols, int num_sms,
                         unsigned int* fault, cudaStream_t stream);
// [rows][C] row-major scale bytes <-> the F8_128x4 layout (C = cols / 32)
cudaError_t launch_swizzle_scales(const uint8_t* in, uint8_t* out, int rows, int C, int num_sms, cudaStream_t stream);
cudaError_t launch_unswizzle_scales(const uint8_t* in, uint8_t* out, int rows, int C, int num_sms,
                                    cudaStream_t stream);
cudaError_t launch_e4m3_encode(const float* in, uint8_t* out, size_t n, int num_sms, cudaStream_t stream);

bool gemm_tile_supported(int tile_m, int tile_n);
int gemm_stages(int tile_m, int tile_n);
void gemm_pick_tile(int M, int N, int K, int num_sms, int* tile_m, int* tile_n);
int gemm_grid(int M, int N, int tile_m, int tile_n, int num_sms);
cudaError_t launch_gemm(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, void* out, int M,
                        int N, int K, int tile_m, int tile_n, int num_sms, unsigned int* fault, cudaStream_t stream);
// test hook: the GEMM launched with its producer issuing no copies, so that
// every bounded wait runs out after wait_ns and the kernel takes its give-up
// path (fault bits set, TMEM freed, clean exit); C is not written
cudaError_t launch_gemm_stalled(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, void* out,
                                int M, int N, int K, int tile_m, int tile_n, int num_sms, unsigned int* fault,
                                unsigned long long wait_ns, cudaStream_t stream);
// the same GEMM with C leaving as an MXFP8 operand (codes + F8_128x4 scales); N % 32 == 0
cudaError_t launch_gemm_quant(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, uint8_t* q,
                              uint8_t* qs, int M, int N, int K, int tile_m, int tile_n, int num_sms,
                              unsigned int* fault, cudaStream_t stream);

}  // namespace mxk
