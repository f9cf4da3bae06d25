// Row kernels of the fused Gemma RMSNorm, shared by the translation units
// that instantiate its output forms (one form per unit, so they compile in
// parallel).
//
// The operation is the norm of a decoder layer's input emitting E4M3 data and
// UE8M0 scales directly (vLLM PR #65496, Overview and Details / Root cause),
// with the scales in the F8_128x4 layout the GEMM consumes (PR #64659,
// Details / "GEMM-RS with a quantized input").  Two more output forms serve
// the sequence-parallel path, where rows are all-gathered after the norm and
// 128x4-swizzled scales cannot be concatenated by rows (PR #65496, Details /
// Tradeoff): scales in plain row-major order (swizzled after the gather), and
// the norm alone in BF16 (quantised after the gather).
//
// The kernels are HBM-bound (about 3 bytes per element: 2 read, 1 written;
// 4 for the BF16 form) and are built to spend few instructions per element
// and keep many bytes in flight:
//   * a row is owned by WPR warps (1, 2, 3, 4 or 6); each lane owns 8 consecutive
//     elements of every 256-element chunk it holds (one 16-byte load per
//     chunk), and the whole row is loaded into registers with back-to-back
//     16-byte loads before any arithmetic;
//   * fp32 arithmetic uses the packed f32x2 instructions (two independent
//     correctly rounded operations each);
//   * the sum of squares is the pairwise tree exactly: the 8 leaves of a
//     lane, then a xor-butterfly over the 32 lanes (masks 1..16 are the next
//     five tree levels of the chunk), then the tree over the chunks, built
//     incrementally as a binary counter and closed with zero subtrees; with
//     WPR > 1 every warp owns an aligned power-of-two run of chunks and the
//     warp subtotals are added in tree order (zero-padded to a power of two)
//     through shared memory;
//   * 4 lanes hold one 32-element MX block: amax by two shuffles, the UE8M0
//     byte from the exponent field, one cvt per element pair, an 8-byte
//     store of codes per lane and a byte store of the scale.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "mx_kernels.h"
#include "mx_ptx.cuh"
#include "norm_plan.h"

namespace mxk {

namespace {

constexpr int ROW_WARPS = 16;
constexpr int ROW_THREADS = ROW_WARPS * 32;

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// byte offset of the 4-scale word (r, 4*wd) in the F8_128x4 layout
__device__ __forceinline__ size_t scale_word_off(int r, int wd, int words) {
  return (static_cast<size_t>(r >> 7) * words + wd) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
}

// Pairwise tree of the 8 squares held by one lane:
// ((e0+e1)+(e2+e3)) + ((e4+e5)+(e6+e7)); the packed pairs (x0,x4), (x1,x5),
// (x2,x6), (x3,x7) make each packed add one level of the tree.
__device__ __forceinline__ float lane_square_tree(const uint4& v) {
  const float2 a = make_float2(bf16lo(v.x), bf16lo(v.z));
  const float2 b = make_float2(bf16hi(v.x), bf16hi(v.z));
  const float2 c = make_float2(bf16lo(v.y), bf16lo(v.w));
  const float2 d = make_float2(bf16hi(v.y), bf16hi(v.w));
  const float2 l1a = __fadd2_rn(__fmul2_rn(a, a), __fmul2_rn(b, b));  // (e0+e1, e4+e5)
  const float2 l1b = __fadd2_rn(__fmul2_rn(c, c), __fmul2_rn(d, d));  // (e2+e3, e6+e7)
  const float2 l2 = __fadd2_rn(l1a, l1b);
  return __fadd_rn(l2.x, l2.y);
}

// Tree over the 32 lanes of a warp (lane l holds leaf l); result in all lanes.
__device__ __forceinline__ float warp_tree(float p) {
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, m));
  return p;
}

// The sum of squares of a row of NCH = 8, 16 or 24 chunks (lane l holds
// elements [256c + 8l, +8) of chunk c), in the same pairwise tree as
// warp_tree per chunk followed by the chunk-level tree, but with 36 instead
// of 120 shuffles for NCH = 24: the three lane levels below 8 lanes are a
// reduce-scatter (at each level a lane keeps half of its chunk partials and
// adds its partner's half of the same chunks), so that lane l ends with the
// 64-element sums of chunks c = l % 8 (mod 8); two butterfly levels finish
// those chunks and three more combine chunks 8k .. 8k+7, whose lanes differ
// in bits 0-2.  Every node is the same two children added, so the result is
// bit-identical to the per-chunk butterflies.
template <int NCH>
__device__ __forceinline__ float row_square_tree_rs(const uint4 (&xv)[NCH], int lane) {
  static_assert(NCH == 8 || NCH == 16 || NCH == 24, "chunk runs of 8, 16 or 24");
  float v[NCH];
#pragma unroll
  for (int c = 0; c < NCH; ++c) v[c] = lane_square_tree(xv[c]);
  const bool b0 = lane & 1, b1 = (lane >> 1) & 1, b2 = (lane >> 2) & 1;
  float u1[NCH / 2];  // 16-element sums of chunks 2k + b0
#pragma unroll
  for (int k = 0; k < NCH / 2; ++k) {
    const float keep = b0 ? v[2 * k + 1] : v[2 * k];
    const float give = b0 ? v[2 * k] : v[2 * k + 1];
    u1[k] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, give, 1));
  }
  float u2[NCH / 4];  // 32-element sums of chunks 4k + 2 b1 + b0
#pragma unroll
  for (int k = 0; k < NCH / 4; ++k) {
    const float keep = b1 ? u1[2 * k + 1] : u1[2 * k];
    const float give = b1 ? u1[2 * k] : u1[2 * k + 1];
    u2[k] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, give, 2));
  }
  float u3[NCH / 8];  // 64-element sums of chunks 8k + (l & 7)
#pragma unroll
  for (int k = 0; k < NCH / 8; ++k) {
    const float keep = b2 ? u2[2 * k + 1] : u2[2 * k];
    const float give = b2 ? u2[2 * k] : u2[2 * k + 1];
    u3[k] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, give, 4));
  }
#pragma unroll
  for (int k = 0; k < NCH / 8; ++k) {
    u3[k] = __fadd_rn(u3[k], __shfl_xor_sync(0xffffffffu, u3[k], 8));   // 128 elements
    u3[k] = __fadd_rn(u3[k], __shfl_xor_sync(0xffffffffu, u3[k], 16));  // the chunk
    u3[k] = __fadd_rn(u3[k], __shfl_xor_sync(0xffffffffu, u3[k], 1));   // chunk pairs
    u3[k] = __fadd_rn(u3[k], __shfl_xor_sync(0xffffffffu, u3[k], 2));
    u3[k] = __fadd_rn(u3[k], __shfl_xor_sync(0xffffffffu, u3[k], 4));   // chunks 8k .. 8k+7
  }
  if constexpr (NCH == 8) return u3[0];
  if constexpr (NCH == 16) return __fadd_rn(u3[0], u3[1]);
  return __fadd_rn(__fadd_rn(u3[0], u3[1]), u3[2]);
}

// Quantises the 8 values a lane holds (4 lanes = one MX block) and stores
// their codes and the scales of the 256-element chunk c of row `row`:
// swizzled, lanes 0 and 16 store the chunk's two 4-scale words; row-major,
// the first lane of each block stores its byte.
template <bool ROWMAJOR, bool SCALE_BYTES>
__device__ __forceinline__ void quantize_store(float2 y01, float2 y23, float2 y45, float2 y67, bool valid,
                                               int lane, int row, int c, int H, int words, uint8_t* __restrict__ q,
                                               uint8_t* __restrict__ sc) {
  float amax = fmaxf(fmaxf(fmaxf(fabsf(y01.x), fabsf(y01.y)), fmaxf(fabsf(y23.x), fabsf(y23.y))),
                     fmaxf(fmaxf(fabsf(y45.x), fabsf(y45.y)), fmaxf(fabsf(y67.x), fabsf(y67.y))));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const uint32_t byte = ue8m0_from_amax(amax);
  const float inv = inv_scale_from_ue8m0(byte);
  const float2 iv = make_float2(inv, inv);
  const float2 t01 = __fmul2_rn(y01, iv), t23 = __fmul2_rn(y23, iv);
  const float2 t45 = __fmul2_rn(y45, iv), t67 = __fmul2_rn(y67, iv);
  uint2 codes;
  codes.x = cvt_e4m3x2(t01.x, t01.y) | (cvt_e4m3x2(t23.x, t23.y) << 16);
  codes.y = cvt_e4m3x2(t45.x, t45.y) | (cvt_e4m3x2(t67.x, t67.y) << 16);
  const int col = c * 256 + lane * 8;
  if (valid) *reinterpret_cast<uint2*>(q + static_cast<size_t>(row) * H + col) = codes;
  if constexpr (ROWMAJOR) {
    if (valid && (lane & 3) == 0) sc[static_cast<size_t>(row) * (H >> 5) + (col >> 5)] = static_cast<uint8_t>(byte);
  } else if constexpr (SCALE_BYTES) {
    // the first lane of each block stores its byte at its F8_128x4 place;
    // a block past the row's end inside the last 4-column group is padding (0)
    const int wd = 2 * c + (lane >> 4);
    if ((lane & 3) == 0 && wd < words)
      sc[scale_word_off(row, wd, words) + ((lane >> 2) & 3)] = valid ? static_cast<uint8_t>(byte) : uint8_t{0};
  } else {
    // the four scale bytes of each 128-element word gathered by two shuffles,
    // one 4-byte store (block b = lane / 4)
    uint32_t wv = valid ? byte << (8 * ((lane >> 2) & 3)) : 0u;
    wv |= __shfl_xor_sync(0xffffffffu, wv, 4);
    wv |= __shfl_xor_sync(0xffffffffu, wv, 8);
    const int wd = 2 * c + (lane >> 4);
    if ((lane & 15) == 0 && wd < words) *reinterpret_cast<uint32_t*>(sc + scale_word_off(row, wd, words)) = wv;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Writes the 8 normalised values a lane holds in the kernel's output form.
// For OUT_BF16, `q` is the [M][H] bf16 output and `sc` is unused.
template <int FORM, bool SCALE_BYTES = true>
__device__ __forceinline__ void emit(float2 y01, float2 y23, float2 y45, float2 y67, bool valid, int lane, int row,
                                     int c, int H, int words, uint8_t* __restrict__ q, uint8_t* __restrict__ sc) {
  if constexpr (FORM == OUT_BF16) {
    if (valid) {
      const uint4 v = make_uint4(pack_bf16x2(y01.x, y01.y), pack_bf16x2(y23.x, y23.y), pack_bf16x2(y45.x, y45.y),
                                 pack_bf16x2(y67.x, y67.y));
      *reinterpret_cast<uint4*>(q + (static_cast<size_t>(row) * H + c * 256 + lane * 8) * 2) = v;
    }
  } else {
    quantize_store<FORM == OUT_MX_ROWMAJOR, SCALE_BYTES>(y01, y23, y45, y67, valid, lane, row, c, H, words, q, sc);
  }
}

// Rows a norm kernel walks: the swizzled form also zeroes the scale bytes of
// the padding rows of the last 128-row block.
template <int FORM>
__device__ __forceinline__ int rows_walked(int M) {
  return FORM == OUT_MX_SWIZZLED ? ((M + 127) / 128) * 128 : M;
}

// (1 + w) lives in shared memory lane-interleaved: the 8 gains of lane l in
// chunk c are two float4 at ((2c + h) * 32 + l) * 4, h = 0, 1, so a warp's
// float4 load of them is one contiguous 512-byte run (element-order storage
// puts lanes 32 bytes apart and costs twice the shared-memory wavefronts).
__device__ __forceinline__ int gain_index(int i) {
  const int c = i >> 8, l = (i >> 3) & 31, e = i & 7;
  return ((2 * c + (e >> 2)) * 32 + l) * 4 + (e & 3);
}

// --------------------------------------------------------------- fused norm

// CTA shape for WPR warps per row: as many whole row groups as fit in 16 warps.
template <int WPR>
struct NormCta {
  static constexpr int GROUPS = ROW_WARPS / WPR;
  static constexpr int THREADS = GROUPS * WPR * 32;
};

// Sum of the WPR warp subtotals of a row, in tree order (padded with zeros
// to a power of two).
template <int WPR>
__device__ __forceinline__ float combine_subtotals(const float* t) {
  if constexpr (WPR == 1) return t[0];
  if constexpr (WPR == 2) return __fadd_rn(t[0], t[1]);
  if constexpr (WPR == 3) return __fadd_rn(__fadd_rn(t[0], t[1]), t[2]);
  if constexpr (WPR == 4) return __fadd_rn(__fadd_rn(t[0], t[1]), __fadd_rn(t[2], t[3]));
  if constexpr (WPR == 6)
    return __fadd_rn(__fadd_rn(__fadd_rn(t[0], t[1]), __fadd_rn(t[2], t[3])), __fadd_rn(t[4], t[5]));
  return 0.0f;
}

// WPR warps per row, NCH chunks of 256 elements per warp (a power of two when
// WPR > 1, so that every warp's chunks form an aligned subtree).
template <int WPR, int NCH, int FORM>
__global__ void __launch_bounds__(NormCta<WPR>::THREADS, 1)
    k_rmsnorm_quant(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w, float eps,
                    uint8_t* __restrict__ q, uint8_t* __restrict__ sc, int M, int H) {
  static_assert(WPR == 1 || (NCH & (NCH - 1)) == 0, "multi-warp rows need power-of-two chunk runs");
  static_assert(WPR == 1 || WPR == 2 || WPR == 3 || WPR == 4 || WPR == 6, "warps per row");
  constexpr int GROUPS = NormCta<WPR>::GROUPS;
  constexpr int THREADS = NormCta<WPR>::THREADS;
  extern __shared__ float g_s[];  // (1 + w) in fp32, zero-padded to whole chunks
  __shared__ float red[GROUPS][2][8];

  const int nchunk = (H + 255) >> 8;
  const int words = (H / 32 + 3) / 4;
  const int Mw = rows_walked<FORM>(M);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / WPR, wi = warp % WPR;
  const int c0 = wi * NCH;

  pdl_wait();  // the previous kernel of the stream has finished with x, w, q and sc
  pdl_launch_dependents();
  // the first row's loads go out before the gain set-up, whose latency they hide
  const int row0 = blockIdx.x + gridDim.x * grp;
  uint4 xv[NCH];
  if (row0 < M) {
    const uint16_t* xr = x + static_cast<size_t>(row0) * H;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int col = (c0 + j) * 256 + lane * 8;
      xv[j] = col < H ? ldg_stream(xr + col) : make_uint4(0, 0, 0, 0);
    }
  }
  for (int i = threadIdx.x; i < nchunk * 256; i += THREADS)
    g_s[gain_index(i)] = i < H ? __fadd_rn(1.0f, __uint_as_float(static_cast<uint32_t>(w[i]) << 16)) : 0.0f;
  __syncthreads();

  int it = 0;
  for (int row = row0; row < Mw; row += gridDim.x * GROUPS, ++it) {
    if (row >= M) {
      // padding row of the last 128-row block: its scale bytes are zero
      if (wi == 0)
        for (int wd = lane; wd < words; wd += 32)
          *reinterpret_cast<uint32_t*>(sc + scale_word_off(row, wd, words)) = 0u;
      continue;
    }
    if (row != row0) {
      const uint16_t* xr = x + static_cast<size_t>(row) * H;
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int col = (c0 + j) * 256 + lane * 8;
        xv[j] = col < H ? ldg_stream(xr + col) : make_uint4(0, 0, 0, 0);
      }
    }

    // pass 1: sum of squares, pairwise tree over the warp's chunks
    float lvl[6];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      float t = warp_tree(lane_square_tree(xv[j]));
      int k = 0;
#pragma unroll
      for (; k < 6; ++k) {
        if (((j >> k) & 1) == 0) break;
        t = __fadd_rn(lvl[k], t);
      }
      lvl[k] = t;
    }
    // close the tree with zero subtrees: fold the pending subtrees, smallest first
    float ss_w = 0.0f;
    bool first = true;
#pragma unroll
    for (int k = 0; k < 6; ++k) {
      if ((NCH >> k) & 1) {
        ss_w = first ? lvl[k] : __fadd_rn(lvl[k], ss_w);
        first = false;
      }
    }
    float ss = ss_w;
    if constexpr (WPR > 1) {
      if (lane == 0) red[grp][it & 1][wi] = ss_w;
      named_barrier_sync(1 + grp, WPR * 32);
      ss = combine_subtotals<WPR>(red[grp][it & 1]);
    }
    // the packed row stays live across the reduction; re-unpacking it in
    // pass 2 is cheaper than keeping every unpacked float alive
#pragma unroll
    for (int j = 0; j < NCH; ++j) asm volatile("" : "+r"(xv[j].x), "+r"(xv[j].y), "+r"(xv[j].z), "+r"(xv[j].w));
    const float ms = __fdiv_rn(ss, static_cast<float>(H));
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    const float2 rr2 = make_float2(r, r);

    // pass 2: y = (x * r) * (1 + w), then the output form
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = c0 + j;
      if (c >= nchunk) break;  // warp-uniform
      const int col = c * 256 + lane * 8;
      const float4 ga = *reinterpret_cast<const float4*>(g_s + ((2 * (col >> 8)) * 32 + lane) * 4);
      const float4 gb = *reinterpret_cast<const float4*>(g_s + ((2 * (col >> 8) + 1) * 32 + lane) * 4);
      const uint4 v = xv[j];
      const float2 y01 = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.x), bf16hi(v.x)), rr2), make_float2(ga.x, ga.y));
      const float2 y23 = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.y), bf16hi(v.y)), rr2), make_float2(ga.z, ga.w));
      const float2 y45 = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.z), bf16hi(v.z)), rr2), make_float2(gb.x, gb.y));
      const float2 y67 = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.w), bf16hi(v.w)), rr2), make_float2(gb.z, gb.w));
      emit<FORM>(y01, y23, y45, y67, col < H, lane, row, c, H, words, q, sc);
      // keep the next chunk's shared-memory loads from being hoisted above
      // this point (hoisting them all costs more registers than it hides)
      asm volatile("" ::: "memory");
    }
  }
}

// One warp per row, with the next row prefetched: each warp owns a
// shared-memory slot of one row; while it computes the row it holds in
// registers, a TMA bulk copy brings its next row into the slot, so memory
// and arithmetic overlap within the warp (the register-only kernel above
// loads, then computes, then loads again).  NCH * 256 >= H.  RS selects
// the reduce-scatter form of the sum of squares (same result, fewer
// shuffles; measured faster for launches of 1-4 rows per warp only).
template <int NCH, int FORM, bool SCALE_BYTES, bool RS>
__global__ void __launch_bounds__(ROW_THREADS, 1)
    k_rmsnorm_quant_pf(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w, float eps,
                       uint8_t* __restrict__ q, uint8_t* __restrict__ sc, int M, int H, unsigned int* fault) {
  extern __shared__ __align__(128) uint8_t smem_pf[];
  const int nchunk = (H + 255) >> 8;
  const int slot_bytes = nchunk * 512;
  float* g_s = reinterpret_cast<float*>(smem_pf);                  // nchunk * 256 floats
  uint8_t* slots = smem_pf + nchunk * 1024;                        // ROW_WARPS slots
  const uint32_t bars = smem_u32(slots + ROW_WARPS * slot_bytes);  // one mbarrier per warp
  const int words = (H / 32 + 3) / 4;
  const int Mw = rows_walked<FORM>(M);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* slot = slots + warp * slot_bytes;
  const uint32_t slot_s = smem_u32(slot);
  const uint32_t bar = bars + 8 * warp;
  const uint32_t row_bytes = 2u * static_cast<uint32_t>(H);

  if (lane == 0) mbar_init(bar, 1);
  fence_barrier_init();
  pdl_wait();  // the previous kernel of the stream has finished with x, w, q and sc
  pdl_launch_dependents();
  // Order of the first requests: this thread's gains, then the warp's first
  // row, then the gain table.  The gain loads go out before the burst of
  // row copies (issued after it, they queue behind it and hold every warp at
  // the barrier below), and the first row's copy goes out before the
  // table's set-up, whose latency it hides.
  constexpr int GAINS_PER_THREAD = (NCH * 256 + ROW_THREADS - 1) / ROW_THREADS;
  uint32_t wr[GAINS_PER_THREAD];
#pragma unroll
  for (int k = 0; k < GAINS_PER_THREAD; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    wr[k] = i < H ? static_cast<uint32_t>(w[i]) : 0u;
  }
  const int stride = gridDim.x * ROW_WARPS;
  int row = blockIdx.x + gridDim.x * warp;
  __syncwarp();
  if (lane == 0 && row < M) {
    mbar_arrive_expect_tx(bar, row_bytes);
    bulk_g2s(slot_s, x + static_cast<size_t>(row) * H, row_bytes, bar);
  }
#pragma unroll
  for (int k = 0; k < GAINS_PER_THREAD; ++k) {
    const int i = threadIdx.x + k * ROW_THREADS;
    if (i < nchunk * 256) g_s[gain_index(i)] = i < H ? __fadd_rn(1.0f, __uint_as_float(wr[k] << 16)) : 0.0f;
  }
  __syncthreads();
  uint32_t phase = 0;
  for (; row < Mw; row += stride) {
    if (row >= M) {
      // padding row of the last 128-row block: its scale bytes are zero
      for (int wd = lane; wd < words; wd += 32)
        *reinterpret_cast<uint32_t*>(sc + scale_word_off(row, wd, words)) = 0u;
      continue;
    }
    if (!warp_wait(bar, phase, nullptr)) {
      if (lane == 0) atomicOr(fault, FAULT_ROWQ_CONSUMER);
      break;
    }
    phase ^= 1u;
    uint4 xv[NCH];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int col = j * 256 + lane * 8;
      xv[j] = col < H ? *reinterpret_cast<const uint4*>(slot + j * 512 + lane * 16) : make_uint4(0, 0, 0, 0);
    }

    float ss;
    if constexpr (RS) {
      ss = row_square_tree_rs<NCH>(xv, lane);
    } else {
      // pass 1: sum of squares, pairwise tree over the row's chunks
      float lvl[6];
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        float t = warp_tree(lane_square_tree(xv[j]));
        int k = 0;
#pragma unroll
        for (; k < 6; ++k) {
          if (((j >> k) & 1) == 0) break;
          t = __fadd_rn(lvl[k], t);
        }
        lvl[k] = t;
      }
      ss = 0.0f;
      bool first = true;
#pragma unroll
      for (int k = 0; k < 6; ++k) {
        if ((NCH >> k) & 1) {
          ss = first ? lvl[k] : __fadd_rn(lvl[k], ss);
          first = false;
        }
      }
    }
    // every lane's reads of the slot are consumed: the slot may take the next row
#pragma unroll
    for (int j = 0; j < NCH; ++j) asm volatile("" : "+r"(xv[j].x), "+r"(xv[j].y), "+r"(xv[j].z), "+r"(xv[j].w));
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    const int next = row + stride;
    if (lane == 0 && next < M) {
      mbar_arrive_expect_tx(bar, row_bytes);
      bulk_g2s(slot_s, x + static_cast<size_t>(next) * H, row_bytes, bar);
    }

    const float ms = __fdiv_rn(ss, static_cast<float>(H));
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    const float2 rr2 = make_float2(r, r);
    // pass 2: y = (x * r) * (1 + w), then the output form
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      if (j >= nchunk) break;  // warp-uniform
      const int col = j * 256 + lane * 8;
      const float4 ga = *reinterpret_cast<const float4*>(g_s + ((2 * (col >> 8)) * 32 + lane) * 4);
      const float4 gb = *reinterpret_cast<const float4*>(g_s + ((2 * (col >> 8) + 1) * 32 + lane) * 4);
      const uint4 v = xv[j];
      const float2 y01 = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.x), bf16hi(v.x)), rr2), make_float2(ga.x, ga.y));
      const float2 y23 = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.y), bf16hi(v.y)), rr2), make_float2(ga.z, ga.w));
      const float2 y45 = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.z), bf16hi(v.z)), rr2), make_float2(gb.x, gb.y));
      const float2 y67 = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.w), bf16hi(v.w)), rr2), make_float2(gb.z, gb.w));
      emit<FORM, SCALE_BYTES>(y01, y23, y45, y67, col < H, lane, row, j, H, words, q, sc);
      asm volatile("" ::: "memory");
    }
  }
}

// Scale stores of the swizzled form: a byte per block from the block's first
// lane is fewer instructions and measured faster for up to ~10k rows; beyond,
// where the launch is bandwidth-bound, one 4-byte store per 4 blocks is
// (same-box timing at H = 6144, bytes vs words: 1024 rows 6.4 vs 6.9 us, 8192
// rows 31.9 vs 33.3 us, 16384 rows 54.7 vs 53.4 us, 32768 rows 109.7 vs 102.5).
constexpr int SCALE_BYTE_STORES_MAX_ROWS = 12288;

// The reduce-scatter sum of squares (bit-identical) is faster while a
// launch gives each warp 1-4 rows and slower with more (same-box timing at
// H = 6144, per-chunk butterflies vs reduce-scatter: 1024 rows 7.9 vs 8.05 us,
// 2048 rows 11.8 vs 11.3, 4096 rows 19.1 vs 18.3, 8192 rows 31.4 vs 31.0,
// 32768 rows 97.5 vs 107.7); measured for rows of 17-24 chunks only.
template <int NCH>
bool norm_pf_uses_rs(int M, int num_sms) {
  const long long warps = static_cast<long long>(num_sms) * ROW_WARPS;
  return NCH == 24 && 2LL * M > warps && M <= 4 * warps;
}

template <int NCH, int FORM>
cudaError_t launch_norm_pf(const uint16_t* x, const uint16_t* w, float eps, uint8_t* q, uint8_t* sc, int M, int H,
                           int num_sms, unsigned int* fault, cudaStream_t stream) {
  auto kern = norm_pf_uses_rs<NCH>(M, num_sms) ? k_rmsnorm_quant_pf<NCH, FORM, true, NCH == 24>
              : M <= SCALE_BYTE_STORES_MAX_ROWS ? k_rmsnorm_quant_pf<NCH, FORM, true, false>
                                                : k_rmsnorm_quant_pf<NCH, FORM, FORM != OUT_MX_SWIZZLED, false>;
  const int nchunk = (H + 255) / 256;
  const int smem = nchunk * 1024 + ROW_WARPS * nchunk * 512 + ROW_WARPS * 8;
  cudaError_t err = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  const int Mw = FORM == OUT_MX_SWIZZLED ? ((M + 127) / 128) * 128 : M;
  const int grid = Mw < num_sms ? Mw : num_sms;
  LaunchAttrs la(dim3(grid), dim3(ROW_THREADS), static_cast<size_t>(smem), stream);
  return cudaLaunchKernelEx(&la.cfg, kern, x, w, eps, q, sc, M, H, fault);
}

template <int WPR, int NCH, int FORM>
cudaError_t launch_norm(const uint16_t* x, const uint16_t* w, float eps, uint8_t* q, uint8_t* sc, int M, int H,
                        int num_sms, cudaStream_t stream) {
  auto kern = k_rmsnorm_quant<WPR, NCH, FORM>;
  const int smem = ((H + 255) / 256) * 256 * 4;
  cudaError_t err = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  const int Mw = FORM == OUT_MX_SWIZZLED ? ((M + 127) / 128) * 128 : M;
  const int grid = Mw < num_sms ? Mw : num_sms;
  LaunchAttrs la(dim3(grid), dim3(NormCta<WPR>::THREADS), static_cast<size_t>(smem), stream);
  return cudaLaunchKernelEx(&la.cfg, kern, x, w, eps, q, sc, M, H);
}

}  // namespace

}  // namespace mxk
