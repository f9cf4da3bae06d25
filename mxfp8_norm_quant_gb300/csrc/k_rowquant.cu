// Plain MXFP8 quantisation of a bf16 operand, the swizzled-scale form of the
// fused norm, the standalone scale (un)swizzle kernels and the encoder probe.
// The norm kernels themselves are in row_common.cuh.
#include <cstdint>

#include "quant_lb.cuh"

namespace mxk {

namespace {

// --------------------------------------------------------------- plain quant

// A warp task is up to G consecutive chunks of one row.  SCALE_BYTES: each
// block's first lane stores its scale byte (as the norm kernels do while the
// launch is latency-bound) instead of one 4-byte store per 4 blocks.
template <int G, bool SCALE_BYTES>
__global__ void __launch_bounds__(ROW_THREADS, 2)
    k_quant(const uint16_t* __restrict__ x, uint8_t* __restrict__ q, uint8_t* __restrict__ sc, int rows,
            int cols) {
  const int nchunk = (cols + 255) >> 8;
  const int words = (cols / 32 + 3) / 4;
  const int Mp = ((rows + 127) / 128) * 128;
  const int tpr = (nchunk + G - 1) / G;
  const long long ntask = static_cast<long long>(rows) * tpr;
  const long long nall = ntask + (Mp - rows);
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * ROW_WARPS;
  pdl_wait();  // the previous kernel of the stream has finished with x, q and sc
  pdl_launch_dependents();
  for (long long task = static_cast<long long>(blockIdx.x) * ROW_WARPS + (threadIdx.x >> 5); task < nall;
       task += nwarps) {
    if (task >= ntask) {
      const int row = rows + static_cast<int>(task - ntask);
      for (int wd = lane; wd < words; wd += 32)
        *reinterpret_cast<uint32_t*>(sc + scale_word_off(row, wd, words)) = 0u;
      continue;
    }
    const int row = static_cast<int>(task / tpr);
    const int c0 = static_cast<int>(task % tpr) * G;
    const uint16_t* xr = x + static_cast<size_t>(row) * cols;
    uint4 xv[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int col = (c0 + j) * 256 + lane * 8;
      xv[j] = col < cols ? ldg_stream(xr + col) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int c = c0 + j;
      if (c >= nchunk) break;  // warp-uniform
      const uint4 v = xv[j];
      quantize_store<false, SCALE_BYTES>(make_float2(bf16lo(v.x), bf16hi(v.x)), make_float2(bf16lo(v.y), bf16hi(v.y)),
                     make_float2(bf16lo(v.z), bf16hi(v.z)), make_float2(bf16lo(v.w), bf16hi(v.w)),
                     c * 256 + lane * 8 < cols, lane, row, c, cols, words, q, sc);
    }
  }
}

// ------------------------------------------------------- scale (un)swizzle

// Row-major [rows][C] scale bytes -> F8_128x4 layout (padding bytes zero).
// A 128-row block of either layout is one contiguous span (128 * C bytes in,
// 128 * Cp bytes out), so one CTA permutes one block through shared memory:
// coalesced loads of the input span into rows of stride S = Cp + 4 bytes (an
// odd number of words, so the column reads below hit distinct banks), then
// 16-byte output vectors, each the 4-byte words of rows rl, rl+32, rl+64,
// rl+96 at one 4-column group, written in output order.
constexpr int SWZ_THREADS = 256;

__global__ void __launch_bounds__(SWZ_THREADS) k_swizzle_scales(const uint8_t* __restrict__ in,
                                                                uint8_t* __restrict__ out, int rows, int C) {
  extern __shared__ __align__(16) uint8_t tile[];
  const int words = (C + 3) / 4;
  const int S = words * 4 + 4;
  const int r0 = blockIdx.x * 128;
  const int nr = min(128, rows - r0);
  const uint8_t* src = in + static_cast<size_t>(r0) * C;
  pdl_wait();
  pdl_launch_dependents();
  const int span = nr * C;
  if ((C & 15) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
    for (int o = threadIdx.x * 16; o < span; o += SWZ_THREADS * 16) {
      const uint4 v = *reinterpret_cast<const uint4*>(src + o);
      uint32_t* d = reinterpret_cast<uint32_t*>(tile + (o / C) * S + o % C);
      d[0] = v.x;
      d[1] = v.y;
      d[2] = v.z;
      d[3] = v.w;
    }
  } else {
    for (int o = threadIdx.x; o < span; o += SWZ_THREADS) tile[(o / C) * S + o % C] = src[o];
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(blockIdx.x) * words * 512);
  for (int v = threadIdx.x; v < words * 32; v += SWZ_THREADS) {
    const int wd = v >> 5, rl = v & 31;
    uint32_t wv[4];
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      const int r = rl + 32 * qd;
      const uint8_t* t = tile + r * S + 4 * wd;
      if (r >= nr) {
        wv[qd] = 0u;
      } else if (4 * wd + 4 <= C) {
        wv[qd] = *reinterpret_cast<const uint32_t*>(t);
      } else {
        uint32_t b = 0;
        for (int j = 0; 4 * wd + j < C; ++j) b |= static_cast<uint32_t>(t[j]) << (8 * j);
        wv[qd] = b;
      }
    }
    dst[v] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
}

// F8_128x4 layout -> row-major [rows][C] scale bytes, one thread per output byte.
__global__ void __launch_bounds__(256) k_unswizzle_scales(const uint8_t* __restrict__ in, uint8_t* __restrict__ out,
                                                          int rows, int C) {
  const int words = (C + 3) / 4;
  const long long total = static_cast<long long>(rows) * C;
  pdl_wait();
  pdl_launch_dependents();
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / C), c = static_cast<int>(i % C);
    out[i] = in[scale_word_off(r, c >> 2, words) + (c & 3)];
  }
}

unsigned scale_grid(long long items, int num_sms) {
  long long blocks = (items + 255) / 256;
  const long long cap = 8LL * num_sms;
  if (blocks > cap) blocks = cap;
  return static_cast<unsigned>(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_rmsnorm_quant(const void* x, const void* w, float eps, uint8_t* q, uint8_t* sc, int M, int H,
                                 int num_sms, unsigned int* fault, cudaStream_t stream) {
  return dispatch_norm<OUT_MX_SWIZZLED>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
}

cudaError_t launch_rmsnorm_quant_stalled(const void* x, const void* w, float eps, uint8_t* q, uint8_t* sc, int M,
                                         int H, int num_sms, unsigned int* fault, unsigned long long wait_ns,
                                         cudaStream_t stream) {
  const NormPlan pl = plan_norm(OUT_MX_SWIZZLED, M, H, num_sms);
  if (pl.wpr == 0) return cudaErrorInvalidValue;  // the chunked kernels have no row copies to withhold
  return launch_norm_plan<OUT_MX_SWIZZLED>(pl, x, static_cast<const uint16_t*>(w), eps, q, sc, M, H, num_sms, fault,
                                           stream, wait_ns, 1);
}

cudaError_t launch_swizzle_scales(const uint8_t* in, uint8_t* out, int rows, int C, int /*num_sms*/,
                                  cudaStream_t stream) {
  const int smem = 128 * (((C + 3) / 4) * 4 + 4);
  cudaError_t err = set_smem_once(reinterpret_cast<const void*>(k_swizzle_scales), smem);
  if (err != cudaSuccess) return err;
  LaunchAttrs la(dim3((rows + 127) / 128), dim3(SWZ_THREADS), static_cast<size_t>(smem), stream);
  return cudaLaunchKernelEx(&la.cfg, k_swizzle_scales, in, out, rows, C);
}

cudaError_t launch_unswizzle_scales(const uint8_t* in, uint8_t* out, int rows, int C, int num_sms,
                                    cudaStream_t stream) {
  LaunchAttrs la(dim3(scale_grid(static_cast<long long>(rows) * C, num_sms)), dim3(256), 0, stream);
  return cudaLaunchKernelEx(&la.cfg, k_unswizzle_scales, in, out, rows, C);
}

namespace {

template <int G>
cudaError_t launch_quant_g(const uint16_t* x, uint8_t* q, uint8_t* sc, int rows, int cols, int num_sms,
                           cudaStream_t stream) {
  auto kern = rows <= SCALE_BYTE_STORES_MAX_ROWS ? k_quant<G, true> : k_quant<G, false>;
  const int nchunk = (cols + 255) / 256;
  const long long tasks = static_cast<long long>(rows) * ((nchunk + G - 1) / G) + 127;
  long long grid = 2LL * num_sms;
  const long long need = (tasks + ROW_WARPS - 1) / ROW_WARPS;
  if (grid > need) grid = need;
  LaunchAttrs la(dim3(static_cast<unsigned>(grid)), dim3(ROW_THREADS), 0, stream);
  return cudaLaunchKernelEx(&la.cfg, kern, x, q, sc, rows, cols);
}

}  // namespace

// The lane-block quantiser (one 1024-element chunk per warp task) once a
// launch has at least 10 such tasks per SM; below that, the chunked kernel,
// whose 256-element tasks spread a small launch over more SMs.  Same-box
// timings (CUDA graphs, inputs rotating beyond L2), us per launch, chunked /
// lane-block with 1, 2, 4 chunks per task:
//   128 x 2048    1.78 / 2.15  3.10  3.07      512 x 2048   2.29 / 2.40  3.31  3.24
//   512 x 3072    2.75 / 2.60  3.26  4.13     1024 x 2048   3.04 / 2.84  3.59  3.54
//   4096 x 3072   8.72 / 8.09  8.26  9.58    32768 x 3072  53.58 / 46.81 49.19 46.87
//   32768 x 6144 102.49 / 92.07 102.07 93.28
// Within the chunked kernel, chunks per warp task: the longest tasks that
// leave no warp idle (1024 x 2048: 2.9 / 3.0 / 3.9 us with 2 / 4 / 8 chunks
// per task; 1024 x 3072: 3.9 us with 4 vs 4.4 with 8).  Tasks of 8 chunks
// would need more than 4 per warp, i.e. launches the lane-block kernel takes.
cudaError_t launch_quant(const void* xv, uint8_t* q, uint8_t* sc, int rows, int cols, int num_sms,
                         unsigned int* /*fault*/, cudaStream_t stream) {
  const uint16_t* x = static_cast<const uint16_t*>(xv);
  if (static_cast<long long>(rows) * ((cols + 1023) / 1024) >= 10LL * num_sms)
    return launch_quant_lb_g<1>(x, q, sc, rows, cols, num_sms, stream);
  const long long warps = static_cast<long long>(num_sms) * ROW_WARPS;
  const long long nchunk = (cols + 255) / 256;
  const auto tasks = [&](long long g) { return static_cast<long long>(rows) * ((nchunk + g - 1) / g); };
  if (tasks(4) * 5 >= warps * 4) return launch_quant_g<4>(x, q, sc, rows, cols, num_sms, stream);
  if (tasks(2) * 5 >= warps * 4) return launch_quant_g<2>(x, q, sc, rows, cols, num_sms, stream);
  return launch_quant_g<1>(x, q, sc, rows, cols, num_sms, stream);
}

// ---------------------------------------------------------------- probe

__global__ void k_e4m3_encode(const float* __restrict__ in, uint8_t* __restrict__ out, size_t n) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x * 4;
  for (size_t i = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4; i < n; i += stride) {
    if (i + 4 <= n) {
      const float4 v = *reinterpret_cast<const float4*>(in + i);
      *reinterpret_cast<uint32_t*>(out + i) = cvt_e4m3x2(v.x, v.y) | (cvt_e4m3x2(v.z, v.w) << 16);
    } else {
      for (size_t j = i; j < n; ++j) out[j] = static_cast<uint8_t>(cvt_e4m3x2(in[j], 0.0f) & 0xFF);
    }
  }
}

cudaError_t launch_e4m3_encode(const float* in, uint8_t* out, size_t n, int num_sms, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  size_t blocks = (n / 4 + 255) / 256 + 1;
  const size_t cap = static_cast<size_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  k_e4m3_encode<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(in, out, n);
  return cudaGetLastError();
}

}  // namespace mxk
