// MXFP8 block-scaled GEMM on the 5th-generation tensor cores:
//   C[M][N] (bf16) = A[M][K] . B[N][K]^T, E4M3 operands, one UE8M0 scale per
//   32 K-elements of every row of A and B, fp32 accumulation in TMEM.
//
// This is the local GEMM of the o_proj (K=2048) and dense down_proj (K=3072)
// projections at N=6144 (vLLM PR #64659, GEMM-RS microbenchmark table), fed
// with operands whose scales are already in the F8_128x4 layout (PR #64659,
// Details / "GEMM-RS with a quantized input").
//
// One kernel template, two tile families:
//   * PAIR = false: 128 x BN tiles, one CTA per tile;
//   * PAIR = true:  256 x BN tiles, a cluster of two CTAs running one
//     cta_group::2 MMA; CTA r stages rows [128 r, +128) of the A tile and
//     rows [BN/2 r, +BN/2) of the B tile, i.e. half of B per SM.
// Persistent grid (one CTA per SM), 10 warps per CTA:
//   warp 0     TMA producer: per K step of 128, the E4M3 tiles of A and B
//              (tensor maps, 128-byte swizzle) and the 512-byte F8_128x4 scale
//              blocks of A (one) and B (two consecutive) into a ring of
//              STAGES shared-memory stages;
//   warps 6-9  scales into TMEM: one CTA, four scale warps (one per TMEM lane
//              quarter) move a stage's scale blocks from shared memory into
//              its TMEM scale slot with tcgen05.st; a pair, one thread of the
//              leader copies both CTAs' blocks with tcgen05.cp.cta_group::2
//              and commits to the stage's sf_ready barrier.  Either way the
//              MMA issuer does not issue the scale moves;
//   warp 1     TMEM owner and (leader CTA) MMA issuer: once a stage's scales
//              are in TMEM (in both CTAs of a pair), four
//              tcgen05.mma.kind::mxf8f6f4.block_scale (K=32 each, scale byte
//              k of each 4-byte TMEM cell) into one of two TMEM accumulators;
//              tcgen05.commit frees the stage (in both CTAs of a pair);
//   warps 2-5  epilogue: TMEM -> registers (tcgen05.ld 32x32b), fp32 -> bf16
//              (RNE), 32-byte stores; then hand the accumulator back.  In the
//              MXFP8-output form each thread's 32 columns of one row are one
//              MX block: the bf16-rounded values are quantised in registers
//              and stored as 32 E4M3 codes and one UE8M0 byte at its F8_128x4
//              place, so C leaves the kernel as an MXFP8 operand for the next
//              GEMM (the quantised-activation output of vLLM PR #64659,
//              Details / "GEMM-RS with a quantized input").  When a CTA has
//              more than one tile, warps 6-9 (idle by then) drain the second
//              half of the columns of its last tile.
// The single threads that issue copies, scale moves and MMAs are
// instruction-bound, so their loops keep descriptors as 32-bit words and ring
// positions as counters.  Two accumulators let the epilogue of one tile
// overlap the main loop of the next.  Tiles are dealt round-robin, N-tile
// fastest, so concurrently running CTAs share A rows and all of B in L2.  In
// a pair both CTAs' copies complete on the leader's barriers, and both CTAs'
// epilogues hand their accumulator back to it.
//
// F8_128x4 and TMEM: the MMA reads row r's scales from TMEM column
// (slot + r/32) of lane r%32 in the lane quarters, scale column c in byte c
// of the cell: exactly a 512-byte scale block (byte (r%32)*16 + (r/32)*4 + c)
// whose 16-byte line j is written to lane j of every quarter.  A B tile
// starting 64 rows into a block therefore reads its scales from column
// offset 2 (tile widths are multiples of 64: an odd column offset is not a
// valid scale address).  With cta_group::2 each CTA's TMEM holds the A scales
// of its own rows and the B scales of the whole tile.
#include <atomic>
#include <cmath>
#include <mutex>

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "mx_kernels.h"
#include "mx_ptx.cuh"

namespace mxk {

namespace {

constexpr int BM = 128;  // rows of A per CTA
constexpr int BK = 128;  // K elements (= bytes) per pipeline stage
constexpr int GEMM_THREADS = 320;
constexpr int TMEM_COLS = 512;
constexpr int SMEM_BUDGET = 220 * 1024;
constexpr int SF_COLS = 12;  // TMEM columns per stage: 4 for A's scales, 8 for two blocks of B's

template <int BN, bool PAIR>
struct Cfg {
  // TMEM accumulators: two (the epilogue of one tile overlaps the main loop
  // of the next), or one for the 256-column tile, whose two would leave no
  // TMEM columns for the scales
  static constexpr int ACCS = BN <= 192 ? 2 : 1;
  static constexpr int TM = PAIR ? 2 * BM : BM;      // output tile rows
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // B rows staged per CTA
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = B_ROWS * BK;
  static constexpr int SFA_BYTES = 512;
  static constexpr int SFB_BYTES = 1024;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int STAGES_SMEM = SMEM_BUDGET / STAGE_BYTES;
  static constexpr int STAGES_TMEM = (TMEM_COLS - ACCS * BN) / SF_COLS;
  static constexpr int STAGES_MIN = STAGES_SMEM < STAGES_TMEM ? STAGES_SMEM : STAGES_TMEM;
  static constexpr int STAGES = STAGES_MIN > 10 ? 10 : STAGES_MIN;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
  // full[STAGES], empty[STAGES], sf_ready[STAGES], tmem_full[2], tmem_empty[2], final[2], last
  static constexpr int NUM_BARS = 3 * STAGES + 7;
  static constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_ABORT = OFF_SLOT + 8;
  static constexpr int SMEM_BYTES = OFF_ABORT + 8 + 1024;  // + slack to align the base to 1 KB
  static constexpr int TMEM_SF = ACCS * BN;
  static_assert(STAGES >= 3, "pipeline too shallow");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "tile width");
  static_assert(BN <= 192 || PAIR, "the 256-column tile is a CTA pair's");
  static_assert(B_BYTES % 1024 == 0, "B tiles keep the 1 KB swizzle-atom alignment");
};

// Output forms of the kernel.
enum GemmOut : int {
  GEMM_OUT_BF16 = 0,   // C as bf16
  GEMM_OUT_MXFP8 = 1,  // C rounded to bf16, then E4M3 codes + F8_128x4 UE8M0 scales
};

struct GemmArgs {
  uint16_t* out;     // GEMM_OUT_BF16: [M][N] bf16
  uint8_t* q;        // GEMM_OUT_MXFP8: [M][N] E4M3 codes
  uint8_t* qs;       // GEMM_OUT_MXFP8: F8_128x4 scales of C, (M, N) operand
  int M, N, K;
  int tiles_m, tiles_n, k_tiles;  // tiles_m counts output tiles of Cfg::TM rows
  int out_32b_aligned;            // 32-byte vector stores are allowed
  int withhold;                   // test hook: the producer issues no copies, so every wait runs out
  unsigned long long wait_ns;     // limit of each bounded wait
  unsigned int* fault;
};

// Instruction descriptor of tcgen05.mma.kind::mxf8f6f4.block_scale:
// bits 4-5 B scale id, 7-9 A type (0 = E4M3), 10-12 B type, 15/16 K-major,
// 17-22 N>>3, 23 scale type (1 = UE8M0), 24-28 M>>4, 29-30 A scale id.
__host__ __device__ constexpr uint32_t idesc_mxf8(int m, int n, int sf_id) {
  return (static_cast<uint32_t>(sf_id) << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(m >> 4) << 24) | (static_cast<uint32_t>(sf_id) << 29);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void st_global_32B(void* p, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
               "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

// One MX block of the output: the 32 accumulators of columns [col, col+32)
// of `row` rounded to bf16 (RNE), then the shared exponent from their
// absolute maximum and the 32 E4M3 codes, as the quantisers of the row
// kernels compute them.  Stores the codes; returns the scale byte.
__device__ __forceinline__ uint32_t quantize_block_store(const uint32_t (&v)[32], int row, int col, const GemmArgs& p) {
  float y[32];
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const uint32_t b = pack_bf16x2(v[i], v[i + 1]);
    y[i] = __uint_as_float(b << 16);
    y[i + 1] = __uint_as_float(b & 0xFFFF0000u);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(y[i]));
  const uint32_t byte = ue8m0_from_amax(amax);
  const float inv = inv_scale_from_ue8m0(byte);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = cvt_e4m3x2(__fmul_rn(y[4 * i], inv), __fmul_rn(y[4 * i + 1], inv)) |
           (cvt_e4m3x2(__fmul_rn(y[4 * i + 2], inv), __fmul_rn(y[4 * i + 3], inv)) << 16);
  uint8_t* dst = p.q + static_cast<size_t>(row) * p.N + col;
  const uint4 lo = make_uint4(w[0], w[1], w[2], w[3]), hi = make_uint4(w[4], w[5], w[6], w[7]);
  if (p.out_32b_aligned) {
    st_global_32B(dst, lo, hi);
  } else {
    reinterpret_cast<uint4*>(dst)[0] = lo;
    reinterpret_cast<uint4*>(dst)[1] = hi;
  }
  return byte;
}

// Byte offset of the scale of (row, 32-column block cb) in the F8_128x4 layout.
__device__ __forceinline__ size_t out_scale_off(int row, int cb, int words) {
  return (static_cast<size_t>(row >> 7) * words + (cb >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (cb & 3);
}

// Epilogue of one warp: columns [c_begin, c_end) of the tile's accumulator
// rows held in this warp's TMEM lane quarter (t_row: the row's first column),
// converted to bf16 (or to MXFP8) and stored; `row` is the C row of this lane.
template <int OUT>
__device__ __forceinline__ void drain_chunks(const GemmArgs& p, uint32_t t_row, int row, int n0, int c_begin,
                                             int c_end) {
  uint16_t* out_row = p.out + static_cast<size_t>(row) * p.N;
#pragma unroll 1
  for (int c = c_begin; c < c_end; c += 32) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(t_row + c, v);
    tmem_ld_wait();
    const int col = n0 + c;
    if constexpr (OUT == GEMM_OUT_MXFP8) {
      // N % 32 == 0: a 32-column chunk is in C entirely or not at all
      const int Mp = (p.M + 127) & ~127;
      const int blocks = p.N >> 5, words = (blocks + 3) >> 2;
      if (col < p.N && row < Mp) {
        const int cb = col >> 5;
        // a padding row of the last 128-row block gets a zero scale byte
        const uint32_t byte = row < p.M ? quantize_block_store(v, row, col, p) : 0u;
        p.qs[out_scale_off(row, cb, words)] = static_cast<uint8_t>(byte);
        if (cb == blocks - 1)  // padding scale columns of the last 4-column group
          for (int pc = blocks; pc < 4 * words; ++pc) p.qs[out_scale_off(row, pc, words)] = 0;
      }
      continue;
    }
    if (row < p.M && col < p.N) {
      uint4 pk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        pk[i].x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
        pk[i].y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
        pk[i].z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
        pk[i].w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
      }
      uint16_t* dst = out_row + col;
      if (col + 32 <= p.N && p.out_32b_aligned) {
        st_global_32B(dst, pk[0], pk[1]);
        st_global_32B(dst + 16, pk[2], pk[3]);
      } else if (col + 32 <= p.N) {
#pragma unroll
        for (int i = 0; i < 4; ++i) reinterpret_cast<uint4*>(dst)[i] = pk[i];
      } else {
        for (int i = 0; i < 4 && col + 8 * i < p.N; ++i) reinterpret_cast<uint4*>(dst)[i] = pk[i];
      }
    }
  }
}

template <int BN, bool PAIR, int OUT>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm_mxf8(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                const GemmArgs p) {
  using C = Cfg<BN, PAIR>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_u32);

  const uint32_t sA = base + C::OFF_A, sB = base + C::OFF_B;
  const uint32_t sSFA = base + C::OFF_SFA, sSFB = base + C::OFF_SFB;
  const uint32_t bar_full = base + C::OFF_BAR;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_sfready = bar_empty + 8 * STAGES;
  const uint32_t bar_tfull = bar_sfready + 8 * STAGES;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_final = bar_tempty + 16;
  const uint32_t bar_last = bar_final + 16;  // the epilogue warps have reached the CTA's last tile
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  // tiles the epilogue warps of this CTA have drained (helpers' stall clock)
  volatile uint32_t* progress = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_ABORT + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int nunits = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int num_tiles = p.tiles_m * p.tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_sfready + 8 * s, PAIR ? 1 : 4);  // the leader's scale-copy commit, or the 4 scale warps
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, PAIR ? 8 : 4);  // the epilogue warps of every CTA of the tile
    }
    mbar_init(bar_final, 1);
    mbar_init(bar_final + 8, 1);
    mbar_init(bar_last, 4);
    *abort_flag = 0;
    *progress = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR) {
    cluster_sync();  // both CTAs' barriers initialised, TMEM allocated in both
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the previous kernel of the stream has finished with A, B, their scales and C
  pdl_launch_dependents();

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&tmap_a);
      prefetch_tensormap(&tmap_b);
      prefetch_tensormap(&tmap_sfa);
      prefetch_tensormap(&tmap_sfb);
      const uint32_t lead_full = PAIR ? mapa_shared(bar_full, 0) : bar_full;
      // stage s and its phase parity ph advance together; `it` counts stages issued
      uint32_t it = 0, s = 0, ph = 0;
      bool ok = true;
      for (int tile = unit; tile < num_tiles && ok && !p.withhold; tile += nunits) {
        const int mt = tile / p.tiles_n, nt = tile % p.tiles_n;
        const int m0 = mt * C::TM + static_cast<int>(rank) * BM;
        const int n0 = nt * BN;
        const int b0 = n0 + static_cast<int>(rank) * C::B_ROWS;
        for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort_flag, p.wait_ns)) {
            if (*abort_flag == 0) atomicOr(p.fault, FAULT_GEMM_PRODUCER);
            *abort_flag = 1;
            ok = false;
            break;
          }
          if constexpr (PAIR) {
            // both CTAs' copies complete on the leader's barrier
            if (leader) mbar_arrive_expect_tx(bar_full + 8 * s, 2 * C::STAGE_BYTES);
            const uint32_t fb = lead_full + 8 * s;
            tma_load_2d_pair(sA + s * C::A_BYTES, &tmap_a, kt * BK, m0, fb);
            tma_load_2d_pair(sB + s * C::B_BYTES, &tmap_b, kt * BK, b0, fb);
            tma_load_4d_pair(sSFA + s * C::SFA_BYTES, &tmap_sfa, 0, 0, kt, m0 >> 7, fb);
            tma_load_4d_pair(sSFB + s * C::SFB_BYTES, &tmap_sfb, 0, 0, kt, n0 >> 7, fb);
          } else {
            const uint32_t fb = bar_full + 8 * s;
            mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
            tma_load_2d(sA + s * C::A_BYTES, &tmap_a, kt * BK, m0, fb);
            tma_load_2d(sB + s * C::B_BYTES, &tmap_b, kt * BK, b0, fb);
            tma_load_4d(sSFA + s * C::SFA_BYTES, &tmap_sfa, 0, 0, kt, m0 >> 7, fb);
            tma_load_4d(sSFB + s * C::SFB_BYTES, &tmap_sfb, 0, 0, kt, n0 >> 7, fb);
          }
          if (++s == static_cast<uint32_t>(STAGES)) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // every issued copy must land before the CTA may exit (normally a no-op);
      // in a pair the leader's barriers count the copies of both CTAs
      if (leader) {
        for (uint32_t s = 0; s < static_cast<uint32_t>(STAGES) && s < it; ++s) {
          const uint32_t last = s + ((it - 1 - s) / STAGES) * STAGES;
          if (!mbar_wait(bar_full + 8 * s, (last / STAGES) & 1u, nullptr, DRAIN_LIMIT_NS))
            atomicOr(p.fault, FAULT_DRAIN);
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (leader && lane == 0) {
      // the single issuing thread is instruction-bound: descriptors are kept
      // as 32-bit words advanced by adds, stage and phase by counters
      const uint32_t a_lo0 = static_cast<uint32_t>(smem_desc(sA, 16, 1024, SWIZZLE_128B));
      const uint32_t b_lo0 = static_cast<uint32_t>(smem_desc(sB, 16, 1024, SWIZZLE_128B));
      const uint32_t d_hi = static_cast<uint32_t>(smem_desc(sA, 16, 1024, SWIZZLE_128B) >> 32);
      uint32_t s = 0, ph = 0, tc = 0;
      bool ok = true;
      for (int tile = unit; tile < num_tiles && ok; tile += nunits, ++tc) {
        const int nt = tile % p.tiles_n;
        const uint32_t sfb_col = static_cast<uint32_t>(((nt * BN) & 127) >> 5);
        if ((sfb_col & 1u) != 0) {  // unreachable for BN % 64 == 0; never issue such an MMA
          atomicOr(p.fault, FAULT_GEMM_MMA);
          *abort_flag = 1;
          break;
        }
        const uint32_t acc = C::ACCS == 2 ? (tc & 1u) : 0u;
        const uint32_t aph = C::ACCS == 2 ? ((tc >> 1) & 1u) : (tc & 1u);
        if (!mbar_wait(bar_tempty + 8 * acc, aph ^ 1u, abort_flag, p.wait_ns)) {
          if (*abort_flag == 0) atomicOr(p.fault, FAULT_GEMM_MMA);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          // the stage's operands have landed and its scales are in TMEM (every CTA of the tile)
          if (!mbar_wait(bar_sfready + 8 * s, ph, abort_flag, p.wait_ns)) {
            if (*abort_flag == 0) atomicOr(p.fault, FAULT_GEMM_MMA);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem + C::TMEM_SF + s * SF_COLS;
          const uint32_t sfb_t = sfa_t + 4 + sfb_col;
          const uint32_t a_lo = a_lo0 + s * (C::A_BYTES >> 4), b_lo = b_lo0 + s * (C::B_BYTES >> 4);
          // K advances 32 bytes (2 descriptor units) per MMA inside the 128-byte swizzled rows
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            mma_mxf8_w<PAIR>(d_tmem, a_lo + 2 * k, d_hi, b_lo + 2 * k, d_hi, idesc_mxf8(C::TM, BN, k), sfa_t, sfb_t,
                             (kt | k) != 0 ? 1u : 0u);
          if constexpr (PAIR) {
            tc_commit_pair_mc(bar_empty + 8 * s, 3);  // stage s is free in both CTAs
          } else {
            tc_commit(bar_empty + 8 * s);
          }
          if (++s == static_cast<uint32_t>(STAGES)) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR) {
          tc_commit_pair_mc(bar_tfull + 8 * acc, 3);  // accumulators ready in both CTAs
        } else {
          tc_commit(bar_tfull + 8 * acc);
        }
      }
      // no MMA may still be running when TMEM is released
      if constexpr (PAIR) {
        tc_commit_pair_mc(bar_final, 1);
      } else {
        tc_commit(bar_final);
      }
      if (!mbar_wait(bar_final, 0, nullptr, DRAIN_LIMIT_NS)) atomicOr(p.fault, FAULT_DRAIN);
    }
  } else if (warp >= 6 && PAIR) {
    // -------------------------------------------------------------- scale copies (pair)
    // one thread of the leader copies each stage's scale blocks from both
    // CTAs' shared memory into both TMEMs (tcgen05.cp.cta_group::2), apart
    // from the MMA issuer, and commits to the stage's sf_ready barrier
    if (leader && warp == 6 && lane == 0) {
      uint32_t s = 0, ph = 0;
      bool ok = true;
      for (int tile = unit; tile < num_tiles && ok; tile += nunits) {
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (!mbar_wait(bar_full + 8 * s, ph, abort_flag, p.wait_ns)) {
            if (*abort_flag == 0) atomicOr(p.fault, FAULT_GEMM_SCALES);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t slot = tmem + C::TMEM_SF + s * SF_COLS;
          tc_cp_32x128b_x4_pair(slot, smem_desc(sSFA + s * C::SFA_BYTES, 0, 128, SWIZZLE_NONE));
          tc_cp_32x128b_x4_pair(slot + 4, smem_desc(sSFB + s * C::SFB_BYTES, 0, 128, SWIZZLE_NONE));
          tc_cp_32x128b_x4_pair(slot + 8, smem_desc(sSFB + s * C::SFB_BYTES + 512, 0, 128, SWIZZLE_NONE));
          tc_commit_pair_mc(bar_sfready + 8 * s, 1);
          if (++s == static_cast<uint32_t>(STAGES)) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      tc_commit_pair_mc(bar_final + 8, 1);
      if (!mbar_wait(bar_final + 8, 0, nullptr, DRAIN_LIMIT_NS)) atomicOr(p.fault, FAULT_DRAIN);
    }
  } else if (warp >= 6) {
    // -------------------------------------------------------------- scale warps
    // lane j of lane quarter q writes the 16-byte line j of each scale block
    // to TMEM lane 32q + j: the four quarters hold identical copies
    const int quad = warp & 3;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint8_t* gSFA = smem + C::OFF_SFA + lane * 16;
    const uint8_t* gSFB = smem + C::OFF_SFB + lane * 16;
    uint32_t s = 0, ph = 0;
    for (int tile = unit; tile < num_tiles; tile += nunits) {
      bool ok = true;
      for (int kt = 0; kt < p.k_tiles; ++kt) {
        if (!warp_wait(bar_full + 8 * s, ph, abort_flag, p.wait_ns)) {
          if (lane == 0) {
            if (*abort_flag == 0) atomicOr(p.fault, FAULT_GEMM_SCALES);
            *abort_flag = 1;
          }
          ok = false;
          break;
        }
        const uint4 va = *reinterpret_cast<const uint4*>(gSFA + s * C::SFA_BYTES);
        const uint4 vb0 = *reinterpret_cast<const uint4*>(gSFB + s * C::SFB_BYTES);
        const uint4 vb1 = *reinterpret_cast<const uint4*>(gSFB + s * C::SFB_BYTES + 512);
        const uint32_t slot = lane_base + C::TMEM_SF + s * SF_COLS;
        tmem_st_32x32b_x4(slot, va);
        tmem_st_32x32b_x4(slot + 4, vb0);
        tmem_st_32x32b_x4(slot + 8, vb1);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sfready + 8 * s);
        if (++s == static_cast<uint32_t>(STAGES)) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
    }
  }

  if (warp >= 2) {
    // -------------------------------------------------------------- epilogue
    // Warps 2-5 drain every tile.  When a CTA has more than one tile, warps
    // 6-9, whose own work is over by then, drain the second half of the
    // columns of its last tile, through the same code (so that it is not
    // cold in the instruction cache).  Measured: 3-5 % faster at M >= 4096;
    // for CTAs of a single tile (M = 128) the split was 3-5 % slower.
    const bool helper = warp >= 6;
    const int quad = warp & 3;  // the TMEM lane quarter this warp may access
    const uint32_t lead_tempty = PAIR ? mapa_shared(bar_tempty, 0) : bar_tempty;
    uint32_t tc = 0;
    for (int tile = unit; tile < num_tiles; tile += nunits, ++tc) {
      const bool split = tile + nunits >= num_tiles && tile != unit;  // last tile, not the first
      if (helper && !split) continue;
      const uint32_t acc = C::ACCS == 2 ? (tc & 1u) : 0u;
      const uint32_t aph = C::ACCS == 2 ? ((tc >> 1) & 1u) : (tc & 1u);
      // a helper waits until the epilogue warps have reached the last tile:
      // then that tile's phase is the last one bar_tfull completes, and the
      // parity wait cannot be satisfied by an earlier phase.  That wait spans
      // the CTA's whole run, so its limit bounds a stall of the epilogue
      // warps' progress, not the run's length.
      bool ok = !helper || warp_wait_progress(bar_last, 0, abort_flag, progress, p.wait_ns);
      ok = ok && warp_wait(bar_tfull + 8 * acc, aph, abort_flag, p.wait_ns);
      if (!ok) {
        if (lane == 0) {
          if (*abort_flag == 0) atomicOr(p.fault, FAULT_GEMM_EPILOGUE);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const int mt = tile / p.tiles_n, nt = tile % p.tiles_n;
      const int row = mt * C::TM + static_cast<int>(rank) * BM + quad * 32 + lane;
      const uint32_t t_row = tmem + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      int c_begin = 0, c_end = BN;
      if (split) {
        if (helper) {
          c_begin = BN / 2;
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_last);
          c_end = BN / 2;
        }
      }
      drain_chunks<OUT>(p, t_row, row, nt * BN, c_begin, c_end);
      if (!helper) {
        tc_fence_before();
        __syncwarp();
        if (warp == 2 && lane == 0) *progress = tc + 1;
        if (lane == 0) {
          if constexpr (PAIR) {
            mbar_arrive_cluster(lead_tempty + 8 * acc);
          } else {
            mbar_arrive(bar_tempty + 8 * acc);
          }
        }
      }
    }
  }

  tc_fence_before();
  if constexpr (PAIR) {
    cluster_sync();  // both CTAs done with TMEM and with the leader's barriers
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) {
      tmem_dealloc_pair(tmem, TMEM_COLS);
    } else {
      tmem_dealloc(tmem, TMEM_COLS);
    }
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// K-contiguous E4M3 operand [rows][K] -> tensor map with a box of
// box_rows x 128 bytes, 128-byte swizzle (the tcgen05 K-major SW128 layout).
cudaError_t make_operand_map(CUtensorMap* map, const uint8_t* ptr, int rows, int K, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// F8_128x4 scale buffer of a (blocks*128) x K operand as a 4-D byte tensor
// [block][k_tile][4][128]: one box {128, 4, 1, atoms} is `atoms` consecutive
// 512-byte scale blocks of the same K step (blocks past the end read as 0).
cudaError_t make_scale_map(CUtensorMap* map, const uint8_t* ptr, int blocks, int k_tiles, int atoms) {
  auto fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {128, 4, static_cast<cuuint64_t>(k_tiles), static_cast<cuuint64_t>(blocks)};
  const cuuint64_t strides[3] = {128, 512, static_cast<cuuint64_t>(k_tiles) * 512};
  const cuuint32_t box[4] = {128, 4, 1, static_cast<cuuint32_t>(atoms)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Clusters of two that can be resident at once (cached per device and width;
// concurrent first calls compute the same value, and the atomic makes the
// publication race-free).
template <int BN>
int pair_max_clusters(int num_sms) {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  const int known = cached[dev].load(std::memory_order_acquire);
  if (known > 0) return known;
  // both output forms have the same shared memory and block: one answer serves both
  auto kern = k_gemm_mxf8<BN, true, GEMM_OUT_BF16>;
  using C = Cfg<BN, true>;
  if (set_smem_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES) != cudaSuccess) return num_sms / 2;
  LaunchAttrs la(dim3(static_cast<unsigned>(num_sms & ~1)), dim3(GEMM_THREADS), C::SMEM_BYTES, nullptr, 2);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kern), &la.cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = num_sms / 2;
  }
  cached[dev].store(n, std::memory_order_release);
  return n;
}

template <int BN, bool PAIR, int OUT>
cudaError_t launch_tile(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, void* out,
                        uint8_t* q, uint8_t* qs, int M, int N, int K, int num_sms, unsigned int* fault,
                        cudaStream_t stream, int withhold, unsigned long long wait_ns) {
  using C = Cfg<BN, PAIR>;
  CUtensorMap ta, tb, tsa, tsb;
  const int k_tiles = (K + BK - 1) / BK;
  cudaError_t err = make_operand_map(&ta, aq, M, K, BM);
  if (err == cudaSuccess) err = make_operand_map(&tb, bq, N, K, C::B_ROWS);
  if (err == cudaSuccess) err = make_scale_map(&tsa, as, (M + 127) / 128, k_tiles, 1);
  if (err == cudaSuccess) err = make_scale_map(&tsb, bs, (N + 127) / 128, k_tiles, 2);
  if (err != cudaSuccess) return err;
  GemmArgs p;
  p.out = static_cast<uint16_t*>(out);
  p.q = q;
  p.qs = qs;
  p.M = M;
  p.N = N;
  p.K = K;
  p.tiles_m = (M + C::TM - 1) / C::TM;
  p.tiles_n = (N + BN - 1) / BN;
  p.k_tiles = k_tiles;
  // bf16: row pitch 2N is a multiple of 32 (N % 16 == 0) and tile columns
  // start at multiples of 64 bytes; codes: row pitch N and chunk columns are
  // multiples of 32 (N % 32 == 0).  So the base alone decides.
  const void* vec_base = OUT == GEMM_OUT_MXFP8 ? static_cast<const void*>(q) : out;
  p.out_32b_aligned = (reinterpret_cast<uintptr_t>(vec_base) & 31u) == 0 ? 1 : 0;
  p.withhold = withhold;
  p.wait_ns = wait_ns;
  p.fault = fault;
  auto kern = k_gemm_mxf8<BN, PAIR, OUT>;
  err = set_smem_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  const int tiles = p.tiles_m * p.tiles_n;
  if constexpr (PAIR) {
    const int clusters = pair_max_clusters<BN>(num_sms);
    const int pairs = tiles < clusters ? tiles : clusters;
    LaunchAttrs la(dim3(static_cast<unsigned>(2 * pairs)), dim3(GEMM_THREADS), C::SMEM_BYTES, stream, 2);
    return cudaLaunchKernelEx(&la.cfg, kern, ta, tb, tsa, tsb, p);
  } else {
    const int grid = tiles < num_sms ? tiles : num_sms;
    LaunchAttrs la(dim3(static_cast<unsigned>(grid)), dim3(GEMM_THREADS), C::SMEM_BYTES, stream);
    return cudaLaunchKernelEx(&la.cfg, kern, ta, tb, tsa, tsb, p);
  }
}

}  // namespace

// x [rows][H] bf16 viewed as [rows][H/64][64] (128-byte lines), 128-byte
// swizzle; a box is box_lines lines of one row.  Used by the row kernels
// whose lanes read 64-byte runs of a row from shared memory.
cudaError_t make_row_tensor_map(CUtensorMap* map, const void* x, int rows, int H, int box_lines) {
  auto fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(H / 64), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(H) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_lines), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tile shapes: tile_m 128 (one CTA) with tile_n 64/128/192, or tile_m 256 (a
// CTA pair, cta_group::2) with tile_n 128/192.
bool gemm_tile_supported(int tile_m, int tile_n) {
  if (tile_m == 128) return tile_n == 64 || tile_n == 128 || tile_n == 192;
  if (tile_m == 256) return tile_n == 128 || tile_n == 192 || tile_n == 256;
  return false;
}

int gemm_stages(int tile_m, int tile_n) {
  if (tile_m == 256)
    return tile_n == 128   ? Cfg<128, true>::STAGES
           : tile_n == 192 ? Cfg<192, true>::STAGES
           : tile_n == 256 ? Cfg<256, true>::STAGES
                           : 0;
  switch (tile_n) {
    case 64: return Cfg<64, false>::STAGES;
    case 128: return Cfg<128, false>::STAGES;
    case 192: return Cfg<192, false>::STAGES;
    default: return 0;
  }
}

// Tile shape from a cost model of this kernel measured on GB300: the SM
// cycles one K step of 128 takes in steady state for each tile family (the
// pair's deeper pipeline makes its steps cheaper per output), tiles dealt in
// waves over the SMs (or SM pairs), and a fixed per-tile cost for the
// pipeline fill and the last epilogue.
void gemm_pick_tile(int M, int N, int K, int num_sms, int* tile_m, int* tile_n) {
  // one 128-row tile of A: every CTA reads all of A, so the narrowest B
  // slice per CTA spreads the weights over the most SMs (same-box, N = 6144:
  // M = 128, K = 2048 takes 8.43 us with 128 x 64 against 9.23 with the pair
  // 256 x 128; K = 3072 10.47 against 11.30)
  if (M <= BM) {
    *tile_m = BM;
    *tile_n = 64;
    return;
  }
  // the 256 x 256 pair tile has one accumulator, so a CTA's second tile
  // waits for the first one's epilogue; it pays where its tiles fit one wave
  // of pairs and the 256 x 192 ones need two (same-box, N = 6144: M = 768,
  // K = 2048 takes 11.73 us against 14.67 for 256 x 128 and 14.97 for
  // 256 x 192; K = 3072 14.44 against 18.63 and 19.28; with more tiles than
  // pairs it is slower: M = 4096, K = 2048 51.8 against 38.1 us)
  {
    const long long pairs = num_sms / 2, mt = (M + 255) / 256;
    const long long t256 = mt * ((N + 255) / 256), t192 = mt * ((N + 191) / 192);
    if (t256 <= pairs && t192 > pairs) {
      *tile_m = 256;
      *tile_n = 256;
      return;
    }
  }
  struct Cand {
    int tm, tn;
    double step;  // cycles per K step of 128, measured
  };
  // SM cycles per K step of one tile, from M = 32768, K = 2048 runs on GB300
  static const Cand cands[] = {{256, 192, 612.0}, {128, 192, 746.0}, {256, 128, 457.0},
                               {128, 128, 611.0}, {128, 64, 602.0}};
  const double kt = (K + BK - 1) / BK;
  double best = -1;
  int bm = 128, bn = 192;
  for (const Cand& c : cands) {
    const int units = c.tm == 256 ? num_sms / 2 : num_sms;
    const double tiles = static_cast<double>((M + c.tm - 1) / c.tm) * ((N + c.tn - 1) / c.tn);
    const double waves = std::ceil(tiles / units);
    const double cost = waves * (kt * c.step + 1500.0);
    if (best < 0 || cost < best * 0.999) {
      best = cost;
      bm = c.tm;
      bn = c.tn;
    }
  }
  *tile_m = bm;
  *tile_n = bn;
}

int gemm_grid(int M, int N, int tile_m, int tile_n, int num_sms) {
  if (tile_m == 256) {
    const int tiles = ((M + 255) / 256) * ((N + tile_n - 1) / tile_n);
    const int clusters = tile_n == 128   ? pair_max_clusters<128>(num_sms)
                         : tile_n == 192 ? pair_max_clusters<192>(num_sms)
                                         : pair_max_clusters<256>(num_sms);
    return 2 * (tiles < clusters ? tiles : clusters);
  }
  const int tiles = ((M + BM - 1) / BM) * ((N + tile_n - 1) / tile_n);
  return tiles < num_sms ? tiles : num_sms;
}

namespace {

template <int OUT>
cudaError_t dispatch_tile(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, void* out,
                          uint8_t* q, uint8_t* qs, int M, int N, int K, int tile_m, int tile_n, int num_sms,
                          unsigned int* fault, cudaStream_t stream, int withhold = 0,
                          unsigned long long wait_ns = WAIT_LIMIT_NS) {
  if (tile_m == 256) {
    switch (tile_n) {
      case 128:
        return launch_tile<128, true, OUT>(aq, as, bq, bs, out, q, qs, M, N, K, num_sms, fault, stream, withhold,
                                           wait_ns);
      case 192:
        return launch_tile<192, true, OUT>(aq, as, bq, bs, out, q, qs, M, N, K, num_sms, fault, stream, withhold,
                                           wait_ns);
      case 256:
        return launch_tile<256, true, OUT>(aq, as, bq, bs, out, q, qs, M, N, K, num_sms, fault, stream, withhold,
                                           wait_ns);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (tile_n) {
    case 64:
      return launch_tile<64, false, OUT>(aq, as, bq, bs, out, q, qs, M, N, K, num_sms, fault, stream, withhold,
                                         wait_ns);
    case 128:
      return launch_tile<128, false, OUT>(aq, as, bq, bs, out, q, qs, M, N, K, num_sms, fault, stream, withhold,
                                          wait_ns);
    case 192:
      return launch_tile<192, false, OUT>(aq, as, bq, bs, out, q, qs, M, N, K, num_sms, fault, stream, withhold,
                                          wait_ns);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemm(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, void* out, int M,
                        int N, int K, int tile_m, int tile_n, int num_sms, unsigned int* fault, cudaStream_t stream) {
  return dispatch_tile<GEMM_OUT_BF16>(aq, as, bq, bs, out, nullptr, nullptr, M, N, K, tile_m, tile_n, num_sms, fault,
                                      stream);
}

cudaError_t launch_gemm_stalled(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, void* out,
                                int M, int N, int K, int tile_m, int tile_n, int num_sms, unsigned int* fault,
                                unsigned long long wait_ns, cudaStream_t stream) {
  return dispatch_tile<GEMM_OUT_BF16>(aq, as, bq, bs, out, nullptr, nullptr, M, N, K, tile_m, tile_n, num_sms, fault,
                                      stream, 1, wait_ns);
}

cudaError_t launch_gemm_quant(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, uint8_t* q,
                              uint8_t* qs, int M, int N, int K, int tile_m, int tile_n, int num_sms,
                              unsigned int* fault, cudaStream_t stream) {
  return dispatch_tile<GEMM_OUT_MXFP8>(aq, as, bq, bs, nullptr, q, qs, M, N, K, tile_m, tile_n, num_sms, fault,
                                       stream);
}

}  // namespace mxk
