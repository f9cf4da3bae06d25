// Plain MXFP8 quantisation with each lane owning whole MX blocks.
//
// The operand quantisation of the GEMM inputs (A and W; the BF16-input GEMM
// numbers of vLLM PR #64659, GEMM-RS microbenchmark table, include it) with
// the data layout of the lane-block norm: lane l of a warp owns the
// 32-element block [1024 c + 32 l, +32) of each 1024-element chunk c of a
// row, loads its 64 bytes with four 16-byte loads (the warp's four loads
// together read 2 KB contiguous; the L1 merges the two that share each
// 32-byte sector), takes the block's amax without shuffles, and stores its 32
// codes with one 32-byte store and its scale byte with one byte store.
#pragma once

#include "row_lb.cuh"

namespace mxk {

namespace {

__device__ __forceinline__ uint4 ldg_l1(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

constexpr int QLB_THREADS = 512;

// A warp task is G consecutive 1024-element chunks of one row (the last
// task of a row may hold fewer).  Tasks past the rows zero the scale bytes of
// the padding rows of the last 128-row block.
template <int G>
__global__ void __launch_bounds__(QLB_THREADS, G <= 2 ? 2 : 1)
    k_quant_lb(const uint16_t* __restrict__ x, uint8_t* __restrict__ q, uint8_t* __restrict__ sc, int rows, int cols,
               int out32) {
  const int blocks = cols >> 5;
  const int words = (blocks + 3) >> 2;
  const int nchunk = (cols + 1023) >> 10;
  const int tpr = (nchunk + G - 1) / G;
  const int Mp = ((rows + 127) / 128) * 128;
  const long long ntask = static_cast<long long>(rows) * tpr;
  const long long nall = ntask + (Mp - rows);
  const int lane = threadIdx.x & 31;
  constexpr int WPC = QLB_THREADS / 32;
  const long long nwarps = static_cast<long long>(gridDim.x) * WPC;
  pdl_wait();  // the previous kernel of the stream has finished with x, q and sc
  pdl_launch_dependents();
  for (long long task = static_cast<long long>(blockIdx.x) * WPC + (threadIdx.x >> 5); task < nall;
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
    uint4 v[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int b = (c0 + g) * 32 + lane;
#pragma unroll
      for (int j = 0; j < 4; ++j) v[g][j] = b < blocks ? ldg_l1(xr + b * 32 + 8 * j) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int c = c0 + g;
      if (c >= nchunk) break;  // warp-uniform
      const int b = c * 32 + lane;
      float amax = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&v[g][j]);
#pragma unroll
        for (int k = 0; k < 4; ++k) amax = max_abs2(amax, bf16lo(w[k]), bf16hi(w[k]));
      }
      const uint32_t byte = ue8m0_from_amax(amax);
      const float2 iv = make_float2(inv_scale_from_ue8m0(byte), inv_scale_from_ue8m0(byte));
      uint32_t codes[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&v[g][j]);
        const float2 t0 = __fmul2_rn(make_float2(bf16lo(w[0]), bf16hi(w[0])), iv);
        const float2 t1 = __fmul2_rn(make_float2(bf16lo(w[1]), bf16hi(w[1])), iv);
        const float2 t2 = __fmul2_rn(make_float2(bf16lo(w[2]), bf16hi(w[2])), iv);
        const float2 t3 = __fmul2_rn(make_float2(bf16lo(w[3]), bf16hi(w[3])), iv);
        codes[2 * j] = cvt_e4m3x4(t0.x, t0.y, t1.x, t1.y);
        codes[2 * j + 1] = cvt_e4m3x4(t2.x, t2.y, t3.x, t3.y);
      }
      if (b < blocks) stg256(q + static_cast<size_t>(row) * cols + static_cast<size_t>(b) * 32, codes, out32 != 0);
      // a block past the row's end inside the last 4-column group is padding (0)
      if (b < 4 * words)
        sc[scale_word_off(row, b >> 2, words) + (b & 3)] = b < blocks ? static_cast<uint8_t>(byte) : uint8_t{0};
    }
  }
}

template <int G>
cudaError_t launch_quant_lb_g(const uint16_t* x, uint8_t* q, uint8_t* sc, int rows, int cols, int num_sms,
                              cudaStream_t stream) {
  const int nchunk = (cols + 1023) / 1024;
  const long long tasks = static_cast<long long>(rows) * ((nchunk + G - 1) / G) + 127;
  constexpr int WPC = QLB_THREADS / 32;
  long long grid = 2LL * num_sms;
  const long long need = (tasks + WPC - 1) / WPC;
  if (grid > need) grid = need;
  const int out32 = (reinterpret_cast<uintptr_t>(q) & 31u) == 0 && cols % 32 == 0 ? 1 : 0;
  LaunchAttrs la(dim3(static_cast<unsigned>(grid)), dim3(QLB_THREADS), 0, stream);
  return cudaLaunchKernelEx(&la.cfg, k_quant_lb<G>, x, q, sc, rows, cols, out32);
}

}  // namespace

}  // namespace mxk
