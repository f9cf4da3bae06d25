// MXFP8 block-scaled GEMM on the 5th-generation tensor cores:
//   C[M][N] (bf16) = A[M][K] . B[N][K]^T, E4M3 operands, one UE8M0 scale per
//   32 K-elements of every row of A and B, fp32 accumulation in TMEM.
//
// This is the local GEMM of the o_proj (K=2048) and dense down_proj (K=3072)
// projections at N=6144 (vLLM PR #64659, GEMM-RS microbenchmark table), fed
// with operands whose scales are already in the F8_128x4 layout (PR #64659,
// Details / "GEMM-RS with a quantized input").
//
// Kernel structure (one persistent CTA per SM, 6 warps):
//   warp 0       TMA producer: per 128-wide K step, a 128x128 E4M3 tile of A
//                and a BNx128 tile of B (tensor maps, 128-byte swizzle), plus
//                the 512-byte F8_128x4 scale blocks of A and B (bulk copies)
//                into a ring of STAGES shared-memory stages;
//   warp 1       TMEM owner and MMA issuer: copies the stage's scales into
//                TMEM (tcgen05.cp 32x128b.warpx4) and issues four
//                tcgen05.mma.kind::mxf8f6f4.block_scale (K=32 each, scale
//                byte k of each 4-byte TMEM cell) into one of two TMEM
//                accumulators; tcgen05.commit frees the stage;
//   warps 2-5    epilogue: TMEM -> registers (tcgen05.ld 32x32b), fp32 ->
//                bf16 (RNE), stores; then hand the accumulator back.
// Two accumulators let the epilogue of tile i overlap the main loop of
// tile i+1.  Tiles are dealt round-robin over the persistent CTAs, N-tile
// fastest, so concurrently running CTAs share A rows and all of B in L2.
//
// F8_128x4 and TMEM: a 512-byte scale block (128 rows x 4 scale columns,
// byte (r%32)*16 + (r/32)*4 + c) copied with 32x128b.warpx4 puts rows
// 32j..32j+31 in TMEM column j, scale column c in byte c of the cell.  A
// tile whose first row is 32*o rows into a block therefore reads its scales
// from column offset o, which is how B tiles narrower than 128 rows or not
// aligned to 128 rows address their scales.
#include <mutex>

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "mx_kernels.h"
#include "mx_ptx.cuh"

namespace mxk {

namespace {

constexpr int BM = 128;
constexpr int BK = 128;
constexpr int GEMM_THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr int SMEM_BUDGET = 220 * 1024;

template <int BN>
struct GemmCfg {
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int SFA_BYTES = 512;
  static constexpr int SFB_BYTES = 2 * 512;  // up to two 128-row scale blocks
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int SF_COLS = 12;  // TMEM columns per stage: 4 for A, 8 for B
  static constexpr int STAGES_SMEM = SMEM_BUDGET / STAGE_BYTES;
  static constexpr int STAGES_TMEM = (TMEM_COLS - 2 * BN) / SF_COLS;
  static constexpr int STAGES_MIN = STAGES_SMEM < STAGES_TMEM ? STAGES_SMEM : STAGES_TMEM;
  static constexpr int STAGES = STAGES_MIN > 8 ? 8 : STAGES_MIN;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
  // full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2], final
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_ABORT = OFF_SLOT + 8;
  static constexpr int SMEM_BYTES = OFF_ABORT + 8 + 1024;  // + slack to align the base to 1 KB
  static constexpr int TMEM_SF = 2 * BN;
  static_assert(STAGES >= 2, "pipeline too shallow");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 192, "tile width");
  static_assert(B_BYTES % 1024 == 0, "B tiles keep the 1 KB swizzle-atom alignment");
};

struct GemmArgs {
  const uint8_t* sfa;
  const uint8_t* sfb;
  uint16_t* out;
  int M, N, K;
  int tiles_m, tiles_n, k_tiles;
  int sfb_blocks;  // ceil(N / 128)
  unsigned int* fault;
};

// Instruction descriptor of tcgen05.mma.kind::mxf8f6f4.block_scale:
// bits 4-5 B scale id, 7-9 A type (0 = E4M3), 10-12 B type, 15/16 K-major,
// 17-22 N>>3, 23 scale type (1 = UE8M0), 24-28 M>>4, 29-30 A scale id.
__host__ __device__ constexpr uint32_t idesc_mxf8(int bn, int sf_id) {
  return (static_cast<uint32_t>(sf_id) << 4) | (static_cast<uint32_t>(bn >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(BM >> 4) << 24) | (static_cast<uint32_t>(sf_id) << 29);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ int sfb_atoms(int n0, int bn, int sfb_blocks) {
  const int need = ((n0 & 127) + bn + 127) >> 7;
  const int have = sfb_blocks - (n0 >> 7);
  return need < have ? need : have;
}

template <int BN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm_mxf8(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                const GemmArgs p) {
  using Cfg = GemmCfg<BN>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_u32);

  const uint32_t sA = base + Cfg::OFF_A, sB = base + Cfg::OFF_B;
  const uint32_t sSFA = base + Cfg::OFF_SFA, sSFB = base + Cfg::OFF_SFB;
  const uint32_t bar_full = base + Cfg::OFF_BAR;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_tfull = bar_empty + 8 * STAGES;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_final = bar_tempty + 16;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_SLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_ABORT);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = p.tiles_m * p.tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 4);
    }
    mbar_init(bar_final, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&tmap_a);
      prefetch_tensormap(&tmap_b);
      const size_t rb = static_cast<size_t>(p.k_tiles) * 512;  // bytes per 128-row scale block
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int mt = tile / p.tiles_n, nt = tile % p.tiles_n;
        const int m0 = mt * BM, n0 = nt * BN;
        const int atom0 = n0 >> 7;
        const int nat = sfb_atoms(n0, BN, p.sfb_blocks);
        const uint32_t bytes = Cfg::A_BYTES + Cfg::B_BYTES + 512u + 512u * nat;
        for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(bar_empty + 8 * s, ph ^ 1u, abort_flag)) {
            if (*abort_flag == 0) atomicOr(p.fault, FAULT_GEMM_PRODUCER);
            *abort_flag = 1;
            ok = false;
            break;
          }
          const uint32_t fb = bar_full + 8 * s;
          mbar_arrive_expect_tx(fb, bytes);
          tma_load_2d(sA + s * Cfg::A_BYTES, &tmap_a, kt * BK, m0, fb);
          tma_load_2d(sB + s * Cfg::B_BYTES, &tmap_b, kt * BK, n0, fb);
          bulk_g2s(sSFA + s * Cfg::SFA_BYTES, p.sfa + mt * rb + kt * 512, 512, fb);
          for (int a = 0; a < nat; ++a)
            bulk_g2s(sSFB + s * Cfg::SFB_BYTES + a * 512, p.sfb + (atom0 + a) * rb + kt * 512, 512, fb);
        }
      }
      // every issued copy must land before the CTA may exit (normally a no-op)
      for (uint32_t s = 0; s < static_cast<uint32_t>(STAGES) && s < it; ++s) {
        const uint32_t last = s + ((it - 1 - s) / STAGES) * STAGES;
        if (!mbar_wait(bar_full + 8 * s, (last / STAGES) & 1u, nullptr, DRAIN_LIMIT_NS))
          atomicOr(p.fault, FAULT_DRAIN);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, tc = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++tc) {
        const int nt = tile % p.tiles_n;
        const int n0 = nt * BN;
        const int nat = sfb_atoms(n0, BN, p.sfb_blocks);
        const uint32_t sfb_col = static_cast<uint32_t>((n0 & 127) >> 5);
        if ((sfb_col & 1u) != 0 || nat > 2) {  // unreachable for BN % 64 == 0; never issue such an MMA
          atomicOr(p.fault, FAULT_GEMM_MMA);
          *abort_flag = 1;
          break;
        }
        const uint32_t acc = tc & 1u, aph = (tc >> 1) & 1u;
        if (!mbar_wait(bar_tempty + 8 * acc, aph ^ 1u, abort_flag)) {
          if (*abort_flag == 0) atomicOr(p.fault, FAULT_GEMM_MMA);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        for (int kt = 0; kt < p.k_tiles; ++kt, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(bar_full + 8 * s, ph, abort_flag)) {
            if (*abort_flag == 0) atomicOr(p.fault, FAULT_GEMM_MMA);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem + Cfg::TMEM_SF + s * Cfg::SF_COLS;
          const uint32_t sfb_t = sfa_t + 4;
          tc_cp_32x128b_x4(sfa_t, smem_desc(sSFA + s * Cfg::SFA_BYTES, 0, 128, SWIZZLE_NONE));
          for (int a = 0; a < nat; ++a)
            tc_cp_32x128b_x4(sfb_t + 4 * a, smem_desc(sSFB + s * Cfg::SFB_BYTES + a * 512, 0, 128, SWIZZLE_NONE));
          const uint32_t a_base = sA + s * Cfg::A_BYTES, b_base = sB + s * Cfg::B_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) {
            const uint64_t ad = smem_desc(a_base + 32 * k, 16, 1024, SWIZZLE_128B);
            const uint64_t bd = smem_desc(b_base + 32 * k, 16, 1024, SWIZZLE_128B);
            mma_mxf8(d_tmem, ad, bd, idesc_mxf8(BN, k), sfa_t, sfb_t + sfb_col, (kt | k) != 0 ? 1u : 0u);
          }
          tc_commit(bar_empty + 8 * s);  // stage s is free once these MMAs are done
        }
        if (!ok) break;
        tc_commit(bar_tfull + 8 * acc);  // accumulator ready for the epilogue
      }
      // no MMA may still be running when TMEM is released
      tc_commit(bar_final);
      if (!mbar_wait(bar_final, 0, nullptr, DRAIN_LIMIT_NS)) atomicOr(p.fault, FAULT_DRAIN);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lanes this warp may access
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tc) {
      const uint32_t acc = tc & 1u, aph = (tc >> 1) & 1u;
      if (!warp_wait(bar_tfull + 8 * acc, aph, abort_flag)) {
        if (lane == 0) {
          if (*abort_flag == 0) atomicOr(p.fault, FAULT_GEMM_EPILOGUE);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const int mt = tile / p.tiles_n, nt = tile % p.tiles_n;
      const int row = mt * BM + quad * 32 + lane;
      const int n0 = nt * BN;
      const uint32_t t_row = tmem + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      uint16_t* out_row = p.out + static_cast<size_t>(row) * p.N;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_row + c, v);
        tmem_ld_wait();
        const int col = n0 + c;
        if (row < p.M && col < p.N) {
          uint4 pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            pk[i].x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
            pk[i].y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
            pk[i].z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
            pk[i].w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
          }
          uint4* dst = reinterpret_cast<uint4*>(out_row + col);
          if (col + 32 <= p.N) {
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = pk[i];
          } else {
            for (int i = 0; i < 4 && col + 8 * i < p.N; ++i) dst[i] = pk[i];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * acc);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
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

template <int BN>
cudaError_t launch_bn(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, void* out, int M,
                      int N, int K, int num_sms, unsigned int* fault, cudaStream_t stream) {
  using Cfg = GemmCfg<BN>;
  CUtensorMap ta, tb;
  cudaError_t err = make_operand_map(&ta, aq, M, K, BM);
  if (err != cudaSuccess) return err;
  err = make_operand_map(&tb, bq, N, K, BN);
  if (err != cudaSuccess) return err;
  GemmArgs p;
  p.sfa = as;
  p.sfb = bs;
  p.out = static_cast<uint16_t*>(out);
  p.M = M;
  p.N = N;
  p.K = K;
  p.tiles_m = (M + BM - 1) / BM;
  p.tiles_n = (N + BN - 1) / BN;
  p.k_tiles = (K + BK - 1) / BK;
  p.sfb_blocks = (N + 127) / 128;
  p.fault = fault;
  auto kern = k_gemm_mxf8<BN>;
  err = set_smem_once(reinterpret_cast<const void*>(kern), Cfg::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  const int tiles = p.tiles_m * p.tiles_n;
  const int grid = tiles < num_sms ? tiles : num_sms;
  kern<<<grid, GEMM_THREADS, Cfg::SMEM_BYTES, stream>>>(ta, tb, p);
  return cudaGetLastError();
}

template <int BN>
int stages_of() {
  return GemmCfg<BN>::STAGES;
}

}  // namespace

// Tile widths are multiples of 64 so that a tile starts 0 or 64 rows into a
// 128-row scale block: the B-scale TMEM address is then shifted by 0 or 2
// columns (an odd column shift is not a valid scale address).
bool gemm_block_n_supported(int bn) { return bn == 64 || bn == 128 || bn == 192; }

int gemm_stages(int bn) {
  switch (bn) {
    case 64: return stages_of<64>();
    case 128: return stages_of<128>();
    case 192: return stages_of<192>();
    default: return 0;
  }
}

// Tile width from a simple cost model: a 128 x BN x 128 step costs
// max(2*BN tensor cycles, 128 + BN shared-memory cycles); tiles are dealt in
// waves of num_sms; a fixed per-tile overhead covers pipeline fill and the
// last epilogue.
int gemm_pick_block_n(int M, int N, int K, int num_sms) {
  static const int cands[] = {64, 128, 192};
  const long long kt = (K + BK - 1) / BK;
  long long best = -1;
  int best_bn = 128;
  for (int bn : cands) {
    const long long tiles = static_cast<long long>((M + BM - 1) / BM) * ((N + bn - 1) / bn);
    const long long waves = (tiles + num_sms - 1) / num_sms;
    const long long step = 2 * bn > 128 + bn ? 2 * bn : 128 + bn;
    const long long cost = waves * (kt * step + 800);
    if (best < 0 || cost < best) {
      best = cost;
      best_bn = bn;
    }
  }
  return best_bn;
}

int gemm_grid(int M, int N, int bn, int num_sms) {
  const int tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  return tiles < num_sms ? tiles : num_sms;
}

cudaError_t launch_gemm(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, void* out, int M,
                        int N, int K, int bn, int num_sms, unsigned int* fault, cudaStream_t stream) {
  switch (bn) {
    case 64: return launch_bn<64>(aq, as, bq, bs, out, M, N, K, num_sms, fault, stream);
    case 128: return launch_bn<128>(aq, as, bq, bs, out, M, N, K, num_sms, fault, stream);
    case 192: return launch_bn<192>(aq, as, bq, bs, out, M, N, K, num_sms, fault, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mxk
