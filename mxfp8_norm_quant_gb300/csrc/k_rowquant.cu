// Row kernels: fused Gemma RMSNorm + MXFP8 quantisation, and plain MXFP8
// quantisation of a bf16 operand.
//
// The operation is the norm of a decoder layer's input emitting E4M3 data and
// UE8M0 scales directly (vLLM PR #65496, Overview and Details / Root cause),
// with the scales in the F8_128x4 layout the GEMM consumes (PR #64659,
// Details / "GEMM-RS with a quantized input").
//
// Design (HBM-bound, ~3 bytes moved per element):
//   * persistent grid, one CTA per SM; warp 0 is a TMA producer that streams
//     whole rows (2*H bytes each) into a ring of shared-memory stages with
//     cp.async.bulk, so ~150 KB per SM is in flight;
//   * GROUPS groups of 8 consumer warps; a group owns one row at a time,
//     lane l of warp v handles the 8 elements [256*c + 8*l, +8) of each
//     256-element chunk c = v, v+8, ...;
//   * the sum of squares follows the pairwise tree exactly: an 8-leaf tree
//     inside the lane, a xor-butterfly over the 32 lanes (masks 1..16, i.e.
//     the next five tree levels of the chunk), then a tree over the chunk
//     sums (zero-padded to a power of two);
//   * 4 lanes hold one 32-element MX block: amax by two shuffles, the UE8M0
//     byte from the exponent field, one cvt per element pair, an 8-byte
//     store of codes per lane and one 4-byte store per 4 scales.
#include <cstdint>

#include "mx_kernels.h"
#include "mx_ptx.cuh"

namespace mxk {

namespace {

constexpr int CWARPS = 8;  // consumer warps per group

template <int CPW>
struct RowCfg {
  static constexpr int GROUPS = CPW <= 4 ? 2 : 1;
  static constexpr int THREADS = 32 + GROUPS * CWARPS * 32;
  static constexpr int MAXCHUNK = 8 * CPW;
  static constexpr int TREE = MAXCHUNK <= 8 ? 8 : MAXCHUNK <= 16 ? 16 : MAXCHUNK <= 32 ? 32 : 64;
};

struct SmemLayout {
  int stage_bytes, stages, red_off, bar_off, abort_off, total;
};

__host__ __device__ inline SmemLayout row_smem_layout(int H, int stages, int groups) {
  SmemLayout L;
  L.stage_bytes = ((H + 255) / 256) * 512;
  L.stages = stages;
  L.red_off = stages * L.stage_bytes;
  L.bar_off = L.red_off + groups * 2 * 64 * 4;
  L.abort_off = L.bar_off + (2 * stages + groups) * 8;
  L.total = L.abort_off + 16;
  return L;
}

// byte offset of the 4-scale word (r, 4*wd) in the F8_128x4 layout
__device__ __forceinline__ size_t scale_word_off(int r, int wd, int words) {
  return (static_cast<size_t>(r >> 7) * words + wd) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
}

__device__ __forceinline__ float tree8_squares(const uint4& v) {
  const float x0 = bf16lo(v.x), x1 = bf16hi(v.x), x2 = bf16lo(v.y), x3 = bf16hi(v.y);
  const float x4 = bf16lo(v.z), x5 = bf16hi(v.z), x6 = bf16lo(v.w), x7 = bf16hi(v.w);
  const float a = __fadd_rn(__fmul_rn(x0, x0), __fmul_rn(x1, x1));
  const float b = __fadd_rn(__fmul_rn(x2, x2), __fmul_rn(x3, x3));
  const float c = __fadd_rn(__fmul_rn(x4, x4), __fmul_rn(x5, x5));
  const float d = __fadd_rn(__fmul_rn(x6, x6), __fmul_rn(x7, x7));
  return __fadd_rn(__fadd_rn(a, b), __fadd_rn(c, d));
}

template <bool NORM, int CPW>
__global__ void __launch_bounds__(RowCfg<CPW>::THREADS, 1)
    k_row_quant(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w, float eps,
                uint8_t* __restrict__ q, uint8_t* __restrict__ sc, int M, int H, int stages,
                unsigned int* fault) {
  using Cfg = RowCfg<CPW>;
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemLayout L = row_smem_layout(H, stages, Cfg::GROUPS);
  const int nchunk = (H + 255) >> 8;
  const int words = (H / 32 + 3) / 4;  // 4-scale words per row (Cp / 4)
  const int Mp = ((M + 127) / 128) * 128;
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  const uint32_t bar_full = smem_u32(smem + L.bar_off);
  const uint32_t bar_empty = bar_full + 8 * stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, CWARPS);
    }
    for (int gi = 0; gi < Cfg::GROUPS; ++gi) mbar_init(bar_full + 8 * (2 * stages + gi), CWARPS);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t row_bytes = 2u * static_cast<uint32_t>(H);
      uint32_t it = 0;
      for (int row = blockIdx.x; row < Mp; row += gridDim.x, ++it) {
        const uint32_t s = it % stages, ph = (it / stages) & 1u;
        if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort_flag)) {
          if (*abort_flag == 0) atomicOr(fault, FAULT_ROWQ_PRODUCER);
          *abort_flag = 1;
          break;
        }
        if (row < M) {
          mbar_arrive_expect_tx(bar_full + 8 * s, row_bytes);
          bulk_g2s(smem_u32(smem + s * L.stage_bytes), x + static_cast<size_t>(row) * H, row_bytes,
                   bar_full + 8 * s);
        } else {
          mbar_arrive(bar_full + 8 * s);  // padding row: no data, scales only
        }
      }
      // Let every issued copy land before the CTA can exit (normally a no-op).
      const uint32_t issued = it;
      for (uint32_t s = 0; s < static_cast<uint32_t>(stages) && s < issued; ++s) {
        const uint32_t last = s + ((issued - 1 - s) / stages) * stages;
        if (!mbar_wait(bar_full + 8 * s, (last / stages) & 1u, nullptr, DRAIN_LIMIT_NS))
          atomicOr(fault, FAULT_DRAIN);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int gidx = (warp - 1) / CWARPS;
    const int v = (warp - 1) % CWARPS;

    float g[NORM ? CPW : 1][8];
    if constexpr (NORM) {
#pragma unroll
      for (int j = 0; j < CPW; ++j) {
        const int col = (v + 8 * j) * 256 + lane * 8;
        uint4 wv = make_uint4(0, 0, 0, 0);
        if (col < H) wv = *reinterpret_cast<const uint4*>(w + col);
        g[j][0] = __fadd_rn(1.0f, bf16lo(wv.x));
        g[j][1] = __fadd_rn(1.0f, bf16hi(wv.x));
        g[j][2] = __fadd_rn(1.0f, bf16lo(wv.y));
        g[j][3] = __fadd_rn(1.0f, bf16hi(wv.y));
        g[j][4] = __fadd_rn(1.0f, bf16lo(wv.z));
        g[j][5] = __fadd_rn(1.0f, bf16hi(wv.z));
        g[j][6] = __fadd_rn(1.0f, bf16lo(wv.w));
        g[j][7] = __fadd_rn(1.0f, bf16hi(wv.w));
      }
    }

    // group barrier: the group's 8 warps publish their chunk sums, then all
    // read them (an mbarrier rather than bar.sync, so that waiting on it is
    // bounded too)
    const uint32_t bar_group = bar_full + 8 * (2 * stages + gidx);
    uint32_t k = 0, nreal = 0;
    for (int row = blockIdx.x + gidx * gridDim.x, it = gidx; row < Mp;
         row += Cfg::GROUPS * gridDim.x, it += Cfg::GROUPS, ++k) {
      const uint32_t s = it % stages, ph = (it / stages) & 1u;
      if (!warp_wait(bar_full + 8 * s, ph, abort_flag)) {
        if (lane == 0) {
          if (*abort_flag == 0) atomicOr(fault, FAULT_ROWQ_CONSUMER);
          *abort_flag = 1;
        }
        break;
      }
      if (row >= M) {
        // padding row of the last 128-row block: its scale bytes are zero
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        for (int wd = v * 32 + lane; wd < words; wd += CWARPS * 32)
          *reinterpret_cast<uint32_t*>(sc + scale_word_off(row, wd, words)) = 0u;
        continue;
      }

      const uint8_t* stg = smem + s * L.stage_bytes;
      uint4 xv[CPW];
#pragma unroll
      for (int j = 0; j < CPW; ++j) {
        const int c = v + 8 * j;
        xv[j] = make_uint4(0, 0, 0, 0);
        if (c < nchunk && c * 256 + lane * 8 < H) xv[j] = *reinterpret_cast<const uint4*>(stg + c * 512 + lane * 16);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);  // this warp is done with the stage

      float r = 1.0f;
      if constexpr (NORM) {
        float* red_row = red + (gidx * 2 + (k & 1)) * 64;
#pragma unroll
        for (int j = 0; j < CPW; ++j) {
          float p = tree8_squares(xv[j]);
#pragma unroll
          for (int m = 1; m < 32; m <<= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, m));
          const int c = v + 8 * j;
          if (lane == 0 && c < nchunk) red_row[c] = p;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_group);
        if (!warp_wait(bar_group, nreal & 1u, abort_flag)) {
          if (lane == 0) {
            if (*abort_flag == 0) atomicOr(fault, FAULT_ROWQ_CONSUMER);
            *abort_flag = 1;
          }
          break;
        }
        ++nreal;
        float t[Cfg::TREE];
#pragma unroll
        for (int i = 0; i < Cfg::TREE; ++i) t[i] = i < nchunk ? red_row[i] : 0.0f;
#pragma unroll
        for (int width = Cfg::TREE / 2; width >= 1; width >>= 1) {
#pragma unroll
          for (int i = 0; i < width; ++i) t[i] = __fadd_rn(t[2 * i], t[2 * i + 1]);
        }
        const float ms = __fdiv_rn(t[0], static_cast<float>(H));
        r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
      }

#pragma unroll
      for (int j = 0; j < CPW; ++j) {
        const int c = v + 8 * j;
        if (c >= nchunk) continue;  // warp-uniform
        const int col = c * 256 + lane * 8;
        const bool valid = col < H;
        float y[8] = {bf16lo(xv[j].x), bf16hi(xv[j].x), bf16lo(xv[j].y), bf16hi(xv[j].y),
                      bf16lo(xv[j].z), bf16hi(xv[j].z), bf16lo(xv[j].w), bf16hi(xv[j].w)};
        if constexpr (NORM) {
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(y[e], r), g[j][e]);
        }
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(y[e]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const uint32_t byte = ue8m0_from_amax(amax);
        const float inv = inv_scale_from_ue8m0(byte);
        uint2 codes;
        codes.x = cvt_e4m3x2(__fmul_rn(y[0], inv), __fmul_rn(y[1], inv)) |
                  (cvt_e4m3x2(__fmul_rn(y[2], inv), __fmul_rn(y[3], inv)) << 16);
        codes.y = cvt_e4m3x2(__fmul_rn(y[4], inv), __fmul_rn(y[5], inv)) |
                  (cvt_e4m3x2(__fmul_rn(y[6], inv), __fmul_rn(y[7], inv)) << 16);
        if (valid) *reinterpret_cast<uint2*>(q + static_cast<size_t>(row) * H + col) = codes;
        // gather the four scale bytes of each 128-element word: block b = lane/4
        uint32_t wv = valid ? byte << (8 * ((lane >> 2) & 3)) : 0u;
        wv |= __shfl_xor_sync(0xffffffffu, wv, 4);
        wv |= __shfl_xor_sync(0xffffffffu, wv, 8);
        const int wd = 2 * c + (lane >> 4);
        if ((lane & 15) == 0 && wd < words)
          *reinterpret_cast<uint32_t*>(sc + scale_word_off(row, wd, words)) = wv;
      }
    }
  }
  __syncthreads();
}

template <bool NORM, int CPW>
cudaError_t launch_row(const uint16_t* x, const uint16_t* w, float eps, uint8_t* q, uint8_t* sc, int M, int H,
                       int num_sms, unsigned int* fault, cudaStream_t stream) {
  using Cfg = RowCfg<CPW>;
  const int stage_bytes = ((H + 255) / 256) * 512;
  int stages = (160 * 1024) / stage_bytes;
  if (stages > 16) stages = 16;
  if (stages < 2) stages = 2;
  const SmemLayout L = row_smem_layout(H, stages, Cfg::GROUPS);
  auto kern = k_row_quant<NORM, CPW>;
  cudaError_t err = set_smem_once(reinterpret_cast<const void*>(kern), L.total);
  if (err != cudaSuccess) return err;
  const int Mp = ((M + 127) / 128) * 128;
  int grid = num_sms;
  if (grid > Mp) grid = Mp;
  kern<<<grid, Cfg::THREADS, L.total, stream>>>(x, w, eps, q, sc, M, H, stages, fault);
  return cudaGetLastError();
}

template <bool NORM>
cudaError_t dispatch_row(const uint16_t* x, const uint16_t* w, float eps, uint8_t* q, uint8_t* sc, int M, int H,
                         int num_sms, unsigned int* fault, cudaStream_t stream) {
  const int cpw = ((H + 255) / 256 + 7) / 8;
  switch (cpw) {
    case 1: return launch_row<NORM, 1>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    case 2: return launch_row<NORM, 2>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    case 3: return launch_row<NORM, 3>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    case 4: return launch_row<NORM, 4>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    case 5: return launch_row<NORM, 5>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    case 6: return launch_row<NORM, 6>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    case 7: return launch_row<NORM, 7>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    case 8: return launch_row<NORM, 8>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_rmsnorm_quant(const void* x, const void* w, float eps, uint8_t* q, uint8_t* sc, int M, int H,
                                 int num_sms, unsigned int* fault, cudaStream_t stream) {
  return dispatch_row<true>(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(w), eps, q, sc, M, H,
                            num_sms, fault, stream);
}

cudaError_t launch_quant(const void* x, uint8_t* q, uint8_t* sc, int rows, int cols, int num_sms,
                         unsigned int* fault, cudaStream_t stream) {
  return dispatch_row<false>(static_cast<const uint16_t*>(x), nullptr, 0.0f, q, sc, rows, cols, num_sms, fault,
                             stream);
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
