// The fused Gemma RMSNorm with each lane owning whole MX blocks.
//
// Same operation, readings and output forms as the kernels of row_common.cuh
// (the norm of a decoder layer's input emitting E4M3 data and UE8M0 scales,
// vLLM PR #65496, Overview and Details / Root cause; scales in the F8_128x4
// layout, PR #64659, Details / "GEMM-RS with a quantized input"), with a data
// layout chosen to spend fewer instructions per element:
//   * a row is cut into 1024-element chunks; lane l owns elements
//     [1024 c + 32 l, +32) of every chunk c, i.e. one whole 32-element MX
//     block per chunk.  The block's amax needs no shuffles, its scale byte
//     and 2^-E are computed once per 32 elements, its 32 codes leave in one
//     32-byte store and its scale in one byte store;
//   * rows reach shared memory by a 3-D TMA tensor copy ([M][H/64][64] bf16,
//     128-byte swizzle), one slot per warp, the next row's copy issued as soon
//     as the current row is in registers.  The swizzle spreads the four
//     16-byte pieces of each lane's 64-byte run over distinct banks, so the
//     lane-contiguous reads are conflict free;
//   * the sum of squares is the same pairwise tree as everywhere else: each
//     lane's 32 leaves form a subtree (reduced with packed f32x2 adds, two
//     tree nodes of one level per add), a 5-level xor butterfly over the
//     lanes gives the chunk, the chunks are combined in tree order, and with
//     WPR warps per row the warps' aligned power-of-two chunk runs are added
//     in tree order through shared memory.
#pragma once

#include "row_common.cuh"

namespace mxk {

// 3-D tensor map of x viewed as [rows][H/64][64] bf16 with 128-byte swizzle;
// a box is {64, box_lines, 1}: box_lines 128-byte lines of one row.
cudaError_t make_row_tensor_map(CUtensorMap* map, const void* x, int rows, int H, int box_lines);

namespace {

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void stg256(void* p, const uint32_t (&w)[8], bool aligned32) {
  if (aligned32) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
  } else {
    reinterpret_cast<uint4*>(p)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(p)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// The 32-leaf pairwise tree of the squares of one lane's block (pieces
// p[0..3] hold elements 0-7, 8-15, 16-23, 24-31 as bf16 pairs).  Element k
// is paired with element k + 16, so each packed add computes two nodes of
// the same tree level.
__device__ __forceinline__ float block_square_tree(const uint4 (&p)[4]) {
  float2 s[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t wl = reinterpret_cast<const uint32_t*>(&p[k >> 3])[(k & 7) >> 1];
    const uint32_t wh = reinterpret_cast<const uint32_t*>(&p[2 + (k >> 3)])[(k & 7) >> 1];
    const float2 v = (k & 1) ? make_float2(bf16hi(wl), bf16hi(wh)) : make_float2(bf16lo(wl), bf16lo(wh));
    s[k] = __fmul2_rn(v, v);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) s[k] = __fadd2_rn(s[2 * k], s[2 * k + 1]);   // 2-leaf nodes
#pragma unroll
  for (int k = 0; k < 4; ++k) s[k] = __fadd2_rn(s[2 * k], s[2 * k + 1]);   // 4
#pragma unroll
  for (int k = 0; k < 2; ++k) s[k] = __fadd2_rn(s[2 * k], s[2 * k + 1]);   // 8
  s[0] = __fadd2_rn(s[0], s[1]);                                           // 16 | 16
  return __fadd_rn(s[0].x, s[0].y);
}

// The same tree from the block's values already unpacked as the pairs
// v[k] = (element k, element k + 16).
__device__ __forceinline__ float block_square_tree_f(const float2 (&v)[16]) {
  float2 s[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) s[k] = __fmul2_rn(v[k], v[k]);
#pragma unroll
  for (int k = 0; k < 8; ++k) s[k] = __fadd2_rn(s[2 * k], s[2 * k + 1]);
#pragma unroll
  for (int k = 0; k < 4; ++k) s[k] = __fadd2_rn(s[2 * k], s[2 * k + 1]);
#pragma unroll
  for (int k = 0; k < 2; ++k) s[k] = __fadd2_rn(s[2 * k], s[2 * k + 1]);
  s[0] = __fadd2_rn(s[0], s[1]);
  return __fadd_rn(s[0].x, s[0].y);
}

// The pairs (element k, element k + 16), k = 0..15, of a lane's block.
__device__ __forceinline__ void unpack_block(const uint4 (&p)[4], float2 (&v)[16]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t wl = reinterpret_cast<const uint32_t*>(&p[k >> 3])[(k & 7) >> 1];
    const uint32_t wh = reinterpret_cast<const uint32_t*>(&p[2 + (k >> 3)])[(k & 7) >> 1];
    v[k] = (k & 1) ? make_float2(bf16hi(wl), bf16hi(wh)) : make_float2(bf16lo(wl), bf16lo(wh));
  }
}

// Byte offset, inside a warp's slot, of piece j (elements 8j..8j+7 of the
// lane's block) of chunk 0: 128-byte line l/2, 16-byte unit 4(l&1) + j,
// swizzled by the line index (the TMA 128-byte pattern; slots are 1 KB
// aligned).  Chunk c adds 2048 bytes (16 lines: the pattern repeats).
__device__ __forceinline__ uint32_t piece_offset(int lane, int j) {
  const int line = lane >> 1;
  const int unit = ((lane & 1) * 4 + j) ^ (line & 7);
  return static_cast<uint32_t>(line * 128 + unit * 16);
}

// Index (in floats) of gain element e (0..3) of half h of piece j of lane l in
// global chunk c: a warp's float4 load of one (c, j, h) is one 512-byte run.
__device__ __forceinline__ int lb_gain_index(int c, int l, int j, int h) {
  return (((c * 4 + j) * 2 + h) * 32 + l) * 4;
}

// The gain table for kernels that keep the row unpacked as pairs
// (element k, element k + 16): float4 q of lane l in chunk c holds the gains
// of elements 2q, 2q + 16, 2q + 1, 2q + 17 of the lane's block, so a warp's
// float4 load of one (c, q) is again one 512-byte run.  Element e of the
// block sits at float (e % 2) * 2 + e / 16 of float4 (e % 16) / 2.
__device__ __forceinline__ int lb_gain_index_pairs(int c, int l, int e) {
  const int k = e & 15;
  return ((c * 8 + (k >> 1)) * 32 + l) * 4 + (k & 1) * 2 + (e >> 4);
}

template <int WPR, int NCW, int GROUPS>
struct LbCfg {
  static constexpr int WARPS = GROUPS * WPR;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int NCH = WPR * NCW;             // chunks the gain table covers
  static constexpr int SLOT = NCW * 2048;           // one warp's part of a row, bf16
  static constexpr int OFF_SLOTS = 0;
  static constexpr int OFF_GAINS = OFF_SLOTS + WARPS * SLOT;
  static constexpr int OFF_BARS = OFF_GAINS + NCH * 1024 * 4;
  static constexpr int OFF_RED = OFF_BARS + WARPS * 8;
  static constexpr int SMEM = OFF_RED + GROUPS * 2 * WPR * 8 + 1024;   // + slack to align the base to 1 KB
  static_assert(WPR == 1 || (NCW & (NCW - 1)) == 0, "multi-warp rows need power-of-two chunk runs");
  static_assert(WPR == 1 || WPR == 2 || WPR == 3 || WPR == 4 || WPR == 6 || WPR == 8, "warps per row");
  static_assert(WPR == 1 || GROUPS <= 15, "one named barrier per row group");
};

// WPR warps per row, NCW 1024-element chunks per warp, GROUPS rows in flight
// per CTA.  Requires H % 64 == 0 and H <= WPR * NCW * 1024.
// KEEP: the row stays in registers unpacked (twice the registers of the
// packed row), so pass 2 does not unpack it again: about one instruction per
// element fewer, for the configurations whose row groups leave the registers.
template <int WPR, int NCW, int GROUPS, int FORM, bool KEEP>
__global__ void __launch_bounds__(LbCfg<WPR, NCW, GROUPS>::THREADS, 1)
    k_rmsnorm_lb(const __grid_constant__ CUtensorMap tmap_x, const uint16_t* __restrict__ w, float eps,
                 uint8_t* __restrict__ q, uint8_t* __restrict__ sc, int M, int H, int out32,
                 unsigned int* fault, unsigned long long wait_ns, int withhold) {
  using C = LbCfg<WPR, NCW, GROUPS>;
  extern __shared__ uint8_t lb_smem_raw[];
  const uint32_t raw_u32 = smem_u32(lb_smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* smem = lb_smem_raw + (base - raw_u32);
  float* gains = reinterpret_cast<float*>(smem + C::OFF_GAINS);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);            // [GROUPS][2][WPR] subtotals
  int* red_ok = reinterpret_cast<int*>(smem + C::OFF_RED) + GROUPS * 2 * WPR;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / WPR, wi = warp % WPR;
  const int blocks = H >> 5;                         // logical scale columns
  const int words = (blocks + 3) >> 2;
  const int Mw = rows_walked<FORM>(M);
  const uint32_t slot = base + C::OFF_SLOTS + warp * C::SLOT;
  const uint32_t bar = base + C::OFF_BARS + 8 * warp;
  const int cw0 = wi * NCW;                          // this warp's first global chunk
  // chunks of this warp that hold any element of the row (warp-uniform)
  const int nch_row = (H + 1023) >> 10;
  const int nc = nch_row - cw0 < 0 ? 0 : (nch_row - cw0 > NCW ? NCW : nch_row - cw0);

  if (lane == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  pdl_wait();  // the previous kernel of the stream has finished with x, w, q and sc
  pdl_launch_dependents();
  if (threadIdx.x == 0) prefetch_tensormap(&tmap_x);
  // this thread's gains first (they would queue behind the burst of row
  // copies), then the warp's first row copy, then the gain table
  constexpr int PIECES = C::NCH * 128;                // 8-element pieces of the table
  constexpr int PPT = (PIECES + C::THREADS - 1) / C::THREADS;
  uint4 wv[PPT];
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    const int pc = threadIdx.x + k * C::THREADS;
    wv[k] = pc < PIECES && pc * 8 < H ? *reinterpret_cast<const uint4*>(w + pc * 8) : make_uint4(0, 0, 0, 0);
  }
  const int stride = gridDim.x * GROUPS;
  int row = blockIdx.x + gridDim.x * grp;
  // withhold (failure-handling self-test): no row copy is issued, so every
  // wait for a row runs out after wait_ns
  if (lane == 0 && row < M && nc > 0 && !withhold) {
    mbar_arrive_expect_tx(bar, C::SLOT);
    tma_load_3d(slot, &tmap_x, 0, cw0 * 16, row, bar);
  }
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    const int pc = threadIdx.x + k * C::THREADS;
    if (pc < PIECES) {
      // piece pc = elements 8 pc .. 8 pc + 7: chunk pc / 128, lane (pc / 4) % 32, piece pc % 4
      const int c = pc >> 7, l = (pc >> 2) & 31, j = pc & 3;
      const bool in = pc * 8 < H;
      const uint4 v = wv[k];
      float4 g0, g1;
      g0.x = in ? __fadd_rn(1.0f, bf16lo(v.x)) : 0.0f;
      g0.y = in ? __fadd_rn(1.0f, bf16hi(v.x)) : 0.0f;
      g0.z = in ? __fadd_rn(1.0f, bf16lo(v.y)) : 0.0f;
      g0.w = in ? __fadd_rn(1.0f, bf16hi(v.y)) : 0.0f;
      g1.x = in ? __fadd_rn(1.0f, bf16lo(v.z)) : 0.0f;
      g1.y = in ? __fadd_rn(1.0f, bf16hi(v.z)) : 0.0f;
      g1.z = in ? __fadd_rn(1.0f, bf16lo(v.w)) : 0.0f;
      g1.w = in ? __fadd_rn(1.0f, bf16hi(v.w)) : 0.0f;
      if constexpr (KEEP) {
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) gains[lb_gain_index_pairs(c, l, 8 * j + t)] = g[t];
      } else {
        *reinterpret_cast<float4*>(gains + lb_gain_index(c, l, j, 0)) = g0;
        *reinterpret_cast<float4*>(gains + lb_gain_index(c, l, j, 1)) = g1;
      }
    }
  }
  __syncthreads();

  uint32_t off[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) off[j] = slot + piece_offset(lane, j);
  uint32_t phase = 0;
  int it = 0;
  bool own_ok = true;     // this warp's last wait succeeded
  bool issued = false;    // this warp has a copy in flight for the next row
  for (; row < Mw; row += stride, ++it) {
    if (row >= M) {
      // padding row of the last 128-row block: its scale bytes are zero
      if (wi == 0)
        for (int wd = lane; wd < words; wd += 32)
          *reinterpret_cast<uint32_t*>(sc + scale_word_off(row, wd, words)) = 0u;
      continue;
    }
    bool ok = true;
    uint4 xv[NCW][4];
    if (nc > 0) {
      ok = warp_wait(bar, phase, nullptr, wait_ns);
      own_ok = ok;
      phase ^= 1u;
#pragma unroll
      for (int c = 0; c < NCW; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j) xv[c][j] = lds128(off[j] + c * 2048);
    } else {
#pragma unroll
      for (int c = 0; c < NCW; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j) xv[c][j] = make_uint4(0, 0, 0, 0);
    }

    // pass 1: the warp's subtree of squares (chunks beyond the row are zeros)
    float2 xf[KEEP ? NCW : 1][16];
    float lvl[4];
#pragma unroll
    for (int c = 0; c < NCW; ++c) {
      float t;
      if constexpr (KEEP) {
        unpack_block(xv[c], xf[c]);
        t = warp_tree(block_square_tree_f(xf[c]));
      } else {
        t = warp_tree(block_square_tree(xv[c]));
      }
      int k = 0;
#pragma unroll
      for (; k < 4; ++k) {
        if (((c >> k) & 1) == 0) break;
        t = __fadd_rn(lvl[k], t);
      }
      lvl[k] = t;
    }
    float ss = 0.0f;
    {
      bool first = true;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if ((NCW >> k) & 1) {
          ss = first ? lvl[k] : __fadd_rn(lvl[k], ss);
          first = false;
        }
      }
    }
    // the row is in registers: the slot may take this warp's part of the next row
    if constexpr (KEEP) {
#pragma unroll
      for (int c = 0; c < NCW; ++c)
#pragma unroll
        for (int k = 0; k < 16; ++k) asm volatile("" : "+f"(xf[c][k].x), "+f"(xf[c][k].y));
    } else {
#pragma unroll
      for (int c = 0; c < NCW; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          asm volatile("" : "+r"(xv[c][j].x), "+r"(xv[c][j].y), "+r"(xv[c][j].z), "+r"(xv[c][j].w));
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    const int next = row + stride;
    issued = ok && next < M && nc > 0 && !withhold;
    if (issued && lane == 0) {
      mbar_arrive_expect_tx(bar, C::SLOT);
      tma_load_3d(slot, &tmap_x, 0, cw0 * 16, next, bar);
    }
    if constexpr (WPR > 1) {
      if (lane == 0) {
        red[(grp * 2 + (it & 1)) * WPR + wi] = ss;
        red_ok[(grp * 2 + (it & 1)) * WPR + wi] = ok ? 1 : 0;
      }
      named_barrier_sync(1 + grp, WPR * 32);
      const float* t = red + (grp * 2 + (it & 1)) * WPR;
      const int* o = red_ok + (grp * 2 + (it & 1)) * WPR;
      if constexpr (WPR == 2) ss = __fadd_rn(t[0], t[1]);
      if constexpr (WPR == 3) ss = __fadd_rn(__fadd_rn(t[0], t[1]), t[2]);
      if constexpr (WPR == 4) ss = __fadd_rn(__fadd_rn(t[0], t[1]), __fadd_rn(t[2], t[3]));
      if constexpr (WPR == 6)
        ss = __fadd_rn(__fadd_rn(__fadd_rn(t[0], t[1]), __fadd_rn(t[2], t[3])), __fadd_rn(t[4], t[5]));
      if constexpr (WPR == 8)
        ss = __fadd_rn(__fadd_rn(__fadd_rn(t[0], t[1]), __fadd_rn(t[2], t[3])),
                       __fadd_rn(__fadd_rn(t[4], t[5]), __fadd_rn(t[6], t[7])));
#pragma unroll
      for (int k = 0; k < WPR; ++k) ok = ok && o[k] != 0;
    }
    if (!ok) {
      // a row copy never landed: report it and stop the whole row group
      // (every warp of the group saw the same flags), after a bounded wait
      // for this warp's own copy in flight: the row it waited for, or the
      // next row's when its own wait succeeded and it issued that copy
      if (lane == 0) {
        atomicOr(fault, FAULT_ROWQ_CONSUMER);
        if (!own_ok && !withhold) {
          if (!mbar_wait(bar, phase ^ 1u, nullptr, DRAIN_LIMIT_NS)) atomicOr(fault, FAULT_DRAIN);
        } else if (issued) {
          if (!mbar_wait(bar, phase, nullptr, DRAIN_LIMIT_NS)) atomicOr(fault, FAULT_DRAIN);
        }
      }
      break;
    }
    const float ms = __fdiv_rn(ss, static_cast<float>(H));
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    const float2 rr = make_float2(r, r);
    // this lane's output addresses in chunk 0 of the row; chunk c adds 1024
    // codes (2048 bytes of y), 32 row-major scale bytes, or 8 scale words
    // (4096 bytes) of the F8_128x4 layout
    uint8_t* q_row = q + (static_cast<size_t>(row) * H + lane * 32) * (FORM == OUT_BF16 ? 2 : 1);
    uint8_t* sc_row = nullptr;
    if constexpr (FORM == OUT_MX_ROWMAJOR) sc_row = sc + static_cast<size_t>(row) * blocks + lane;
    if constexpr (FORM == OUT_MX_SWIZZLED) sc_row = sc + scale_word_off(row, lane >> 2, words) + (lane & 3);

    // pass 2: y = (x * r) * (1 + w) block by block, then the output form
#pragma unroll
    for (int c = 0; c < NCW; ++c) {
      if (c >= nc) break;  // warp-uniform
      const int cg = cw0 + c;
      const int b = cg * 32 + lane;          // this lane's MX block of the row
      // y[k]: elements (2k, 2k + 1) of the block; with KEEP, (k, k + 16)
      float2 y[16];
      if constexpr (KEEP) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 g = *reinterpret_cast<const float4*>(gains + ((cg * 8 + q) * 32 + lane) * 4);
          y[2 * q] = __fmul2_rn(__fmul2_rn(xf[c][2 * q], rr), make_float2(g.x, g.y));
          y[2 * q + 1] = __fmul2_rn(__fmul2_rn(xf[c][2 * q + 1], rr), make_float2(g.z, g.w));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 ga = *reinterpret_cast<const float4*>(gains + lb_gain_index(cg, lane, j, 0));
          const float4 gb = *reinterpret_cast<const float4*>(gains + lb_gain_index(cg, lane, j, 1));
          const uint4 v = xv[c][j];
          y[4 * j + 0] = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.x), bf16hi(v.x)), rr), make_float2(ga.x, ga.y));
          y[4 * j + 1] = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.y), bf16hi(v.y)), rr), make_float2(ga.z, ga.w));
          y[4 * j + 2] = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.z), bf16hi(v.z)), rr), make_float2(gb.x, gb.y));
          y[4 * j + 3] = __fmul2_rn(__fmul2_rn(make_float2(bf16lo(v.w), bf16hi(v.w)), rr), make_float2(gb.z, gb.w));
        }
      }
      // element e of the block: y[e / 2] component e % 2, or with KEEP y[e % 16] component e / 16
      auto elem = [&](int e) -> float {
        if constexpr (KEEP) return (e < 16) ? y[e].x : y[e - 16].y;
        return (e & 1) ? y[e >> 1].y : y[e >> 1].x;
      };
      if constexpr (FORM == OUT_BF16) {
        if (b < blocks) {
          uint32_t o[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) o[k] = pack_bf16x2(elem(2 * k), elem(2 * k + 1));
          uint8_t* dst = q_row + cg * 2048;
          const uint32_t lo[8] = {o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]};
          const uint32_t hi[8] = {o[8], o[9], o[10], o[11], o[12], o[13], o[14], o[15]};
          stg256(dst, lo, out32 != 0);
          stg256(dst + 32, hi, out32 != 0);
        }
      } else {
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; ++k) amax = max_abs2(amax, y[k].x, y[k].y);
        const uint32_t byte = ue8m0_from_amax(amax);
        const float inv = inv_scale_from_ue8m0(byte);
        const float2 iv = make_float2(inv, inv);
#pragma unroll
        for (int k = 0; k < 16; ++k) y[k] = __fmul2_rn(y[k], iv);
        uint32_t codes[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) codes[w] = cvt_e4m3x4(elem(4 * w), elem(4 * w + 1), elem(4 * w + 2), elem(4 * w + 3));
        if (b < blocks) stg256(q_row + cg * 1024, codes, out32 != 0);
        if constexpr (FORM == OUT_MX_ROWMAJOR) {
          if (b < blocks) sc_row[cg * 32] = static_cast<uint8_t>(byte);
        } else {
          // a block past the row's end inside the last 4-column group is padding (0)
          if (b < 4 * words) sc_row[cg * 8 * 512] = b < blocks ? static_cast<uint8_t>(byte) : uint8_t{0};
        }
      }
    }
  }
}

template <int WPR, int NCW, int GROUPS, int FORM, bool KEEP = false>
cudaError_t launch_norm_lb(const void* x, const uint16_t* w, float eps, uint8_t* q, uint8_t* sc, int M, int H,
                           int num_sms, unsigned int* fault, cudaStream_t stream,
                           unsigned long long wait_ns = WAIT_LIMIT_NS, int withhold = 0) {
  using C = LbCfg<WPR, NCW, GROUPS>;
  CUtensorMap tmap;
  cudaError_t err = make_row_tensor_map(&tmap, x, M, H, NCW * 16);
  if (err != cudaSuccess) return err;
  auto kern = k_rmsnorm_lb<WPR, NCW, GROUPS, FORM, KEEP>;
  err = set_smem_once(reinterpret_cast<const void*>(kern), C::SMEM);
  if (err != cudaSuccess) return err;
  const int Mw = FORM == OUT_MX_SWIZZLED ? ((M + 127) / 128) * 128 : M;
  const int grid = Mw < num_sms ? Mw : num_sms;
  // 32-byte vector stores: the row pitch (H or 2H bytes, H % 64 == 0) and the
  // block offsets are multiples of 32, so the base alone decides
  const int out32 = (reinterpret_cast<uintptr_t>(q) & 31u) == 0 ? 1 : 0;
  LaunchAttrs la(dim3(grid), dim3(C::THREADS), static_cast<size_t>(C::SMEM), stream);
  return cudaLaunchKernelEx(&la.cfg, kern, tmap, w, eps, q, sc, M, H, out32, fault, wait_ns, withhold);
}

// The chunked kernels of row_common.cuh, for the widths the lane-block
// kernels do not take (H % 64 != 0) and for rows of at most 512 elements in
// launches of up to 16 rows per SM.  Row ownership: a
// warp owns a run of 256-element chunks (at most 24 in registers); rows wider
// than one warp's run, and rows in launches with few rows per warp, are split
// over several warps so that more loads are in flight and each warp's chain
// is shorter.  The row counts below were measured at H = 6144.
template <int FORM>
cudaError_t dispatch_norm_chunked(const void* xv, const void* wv, float eps, uint8_t* q, uint8_t* sc, int M, int H,
                          int num_sms, unsigned int* fault, cudaStream_t stream) {
  const uint16_t* x = static_cast<const uint16_t*>(xv);
  const uint16_t* w = static_cast<const uint16_t*>(wv);
  const int nchunk = (H + 255) / 256;
  const long long warps = static_cast<long long>(num_sms) * ROW_WARPS;
  const long long rows_per_warp = M / (warps > 0 ? warps : 1);
  if (nchunk <= 24 && M > warps) {
    // more than one row per warp: prefetch the next row while computing
    if (nchunk <= 8) return launch_norm_pf<8, FORM>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    if (nchunk <= 16) return launch_norm_pf<16, FORM>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    return launch_norm_pf<24, FORM>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
  }
  if (nchunk > 16 && nchunk <= 24) {
    // rows of 4097..6144 elements, at most one row per warp.  A register
    // kernel is best while its rows fit one round (6 warps per row: 2 rows
    // per CTA; 3 warps: 5 rows per CTA); past that the prefetching kernel.
    // Measured on GB300 at H = 6144 (CUDA-graph timing, inputs rotating
    // beyond L2; swizzled / row-major / bf16 forms, us):
    //   M = 128: 6 warps per row 3.3 / 3.1 / 2.9, prefetching 5.5 / 6.1 / 4.4;
    //   M = 704: 3 warps per row 6.3 / 6.0 / 5.9, 6 warps 7.8 / 7.5 / 7.3,
    //            prefetching 6.9 / 7.6 / 6.2;
    //   M = 768: 3 warps (two rounds) 8.3 / 7.9 / 7.3, 6 warps 7.9 / 7.5 / 7.4,
    //            prefetching 7.2 / 7.9 / 6.3;
    //   M = 1024: prefetching 7.8 / 8.4 / 7.0.
    if (M >= 896) return launch_norm_pf<24, FORM>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    if (M > 256 && M <= NormCta<3>::GROUPS * num_sms)
      return launch_norm<3, 8, FORM>(x, w, eps, q, sc, M, H, num_sms, stream);
    if (M > 256 && FORM != OUT_MX_ROWMAJOR)
      return launch_norm_pf<24, FORM>(x, w, eps, q, sc, M, H, num_sms, fault, stream);
    return launch_norm<6, 4, FORM>(x, w, eps, q, sc, M, H, num_sms, stream);
  }
  // (rows of 17..24 chunks have returned above)
  if (nchunk <= 16 && (M >= 512 || rows_per_warp > 0)) {
    if (nchunk <= 4) return launch_norm<1, 4, FORM>(x, w, eps, q, sc, M, H, num_sms, stream);
    if (nchunk <= 8) return launch_norm<1, 8, FORM>(x, w, eps, q, sc, M, H, num_sms, stream);
    return launch_norm<1, 16, FORM>(x, w, eps, q, sc, M, H, num_sms, stream);
  }
  // a few hundred rows: split each row over several warps to shorten the chain
  if (nchunk <= 8) return launch_norm<2, 4, FORM>(x, w, eps, q, sc, M, H, num_sms, stream);
  if (nchunk <= 24) return launch_norm<6, 4, FORM>(x, w, eps, q, sc, M, H, num_sms, stream);
  if (nchunk <= 32) return launch_norm<4, 8, FORM>(x, w, eps, q, sc, M, H, num_sms, stream);
  return launch_norm<4, 16, FORM>(x, w, eps, q, sc, M, H, num_sms, stream);
}

// The lane-block kernel `pl` names (norm_plan.h), for the output form FORM.
// Every shape the plan can choose for FORM is instantiated here; any other
// is an error.
template <int FORM>
cudaError_t launch_norm_plan(const NormPlan& pl, const void* x, const uint16_t* w, float eps, uint8_t* q,
                             uint8_t* sc, int M, int H, int num_sms, unsigned int* fault, cudaStream_t stream,
                             unsigned long long wait_ns = WAIT_LIMIT_NS, int withhold = 0) {
  constexpr bool BF = FORM == OUT_BF16;
#define MX_NORM_CASE(W, N, G, K, FORMS_OK)                                                                   \
  case norm_plan_key(W, N, G, K):                                                                            \
    if constexpr (FORMS_OK)                                                                                  \
      return launch_norm_lb<W, N, G, FORM, (K) != 0>(x, w, eps, q, sc, M, H, num_sms, fault, stream, wait_ns, \
                                                     withhold);                                              \
    break;
  switch (norm_plan_key(pl.wpr, pl.ncw, pl.groups, pl.keep)) {
    // 4097..6144 elements
    MX_NORM_CASE(6, 1, 2, 0, true)
    MX_NORM_CASE(3, 2, 5, 1, !BF)
    MX_NORM_CASE(3, 2, 5, 0, BF)
    MX_NORM_CASE(3, 2, 8, 0, true)
    MX_NORM_CASE(3, 2, 6, 1, !BF)
    MX_NORM_CASE(6, 1, 4, 0, BF)
    // up to 1024 elements
    MX_NORM_CASE(1, 1, 8, 0, true)
    MX_NORM_CASE(1, 1, 16, 0, true)
    MX_NORM_CASE(1, 1, 32, 0, true)
    // 1025..2048
    MX_NORM_CASE(2, 1, 4, 0, true)
    MX_NORM_CASE(2, 1, 8, 0, true)
    MX_NORM_CASE(1, 2, 16, 0, true)
    MX_NORM_CASE(1, 2, 24, 0, true)
    // 2049..3072
    MX_NORM_CASE(3, 1, 2, 0, true)
    MX_NORM_CASE(3, 1, 4, 0, true)
    MX_NORM_CASE(3, 1, 8, 0, true)
    MX_NORM_CASE(1, 4, 16, 0, true)
    // 3073..4096
    MX_NORM_CASE(4, 1, 2, 0, true)
    MX_NORM_CASE(4, 1, 4, 0, true)
    MX_NORM_CASE(2, 2, 8, 0, true)
    MX_NORM_CASE(1, 4, 12, 0, true)
    // 6145..8192
    MX_NORM_CASE(8, 1, 2, 0, true)
    MX_NORM_CASE(4, 2, 4, 0, true)
    MX_NORM_CASE(4, 2, 6, 0, !BF)
    MX_NORM_CASE(4, 2, 3, 0, BF)
    // 8193..16384
    MX_NORM_CASE(8, 2, 2, 0, true)
    MX_NORM_CASE(8, 2, 3, 0, true)
    MX_NORM_CASE(4, 4, 3, 0, !BF)
    default: break;
  }
#undef MX_NORM_CASE
  return cudaErrorInvalidValue;
}

// The norm in output form FORM: the kernel plan_norm chooses.
template <int FORM>
cudaError_t dispatch_norm(const void* xv, const void* wv, float eps, uint8_t* q, uint8_t* sc, int M, int H,
                          int num_sms, unsigned int* fault, cudaStream_t stream) {
  const NormPlan pl = plan_norm(FORM, M, H, num_sms);
  if (pl.wpr == 0) return dispatch_norm_chunked<FORM>(xv, wv, eps, q, sc, M, H, num_sms, fault, stream);
  return launch_norm_plan<FORM>(pl, xv, static_cast<const uint16_t*>(wv), eps, q, sc, M, H, num_sms, fault,
                                stream);
}

}  // namespace

}  // namespace mxk
