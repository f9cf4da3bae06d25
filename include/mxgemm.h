/*
 * libmxgemm -- MXFP8 Gemma-RMSNorm quantisation and block-scaled GEMM for
 * NVIDIA GB300 (sm_103a).  Plain C ABI: device pointers, sizes and a CUDA
 * stream; no C++ or framework types cross it.
 *
 * What the operations are (sources: the vLLM pull-request pages for
 * MiniMax-M3 serving):
 *
 *   - The input RMSNorm of each decoder layer emits its output directly as
 *     MXFP8 -- a "QuantizedActivation" holding E4M3 data and UE8M0 scales --
 *     whenever the following qkv_proj GEMM can consume it (vLLM PR #65496,
 *     Overview; Details / Root cause).  The norm is the Gemma variant
 *     (PR #64659, Details / Fusions: "AR + Gemma RMSNorm fusions").
 *   - The GEMMs take MXFP8 operands whose scales are already in the
 *     F8_128x4 swizzled layout (PR #64659, Details / "GEMM-RS with a
 *     quantized input"); the 128x4-swizzled scales cannot be concatenated
 *     by rows (PR #65496, Details / Tradeoff).
 *   - Shapes: N = 6144, K = 2048 (o_proj) and K = 3072 (dense down_proj),
 *     BF16 output (PR #64659, GEMM-RS microbenchmark table).
 *
 * The pages print no formula.  The arithmetic implemented here is:
 *
 *   y[i]   = (x[i] * r) * (1 + w[i]),   r = 1 / sqrt(ss / H + eps)
 *   ss     = sum of x[i]^2 in fp32, as a pairwise tree (row padded with
 *            zeros to a power of two, sibling pairs added level by level)
 *   scale  = per 32 consecutive elements of a row: E = floor(log2(amax)) - 8,
 *            stored as the UE8M0 byte max(E + 127, 0)
 *   q[i]   = E4M3(y[i] * 2^-E), round to nearest even, |.| > 448 -> 448
 *   C      = A . B^T accumulated in fp32, rounded to BF16 (RNE)
 *
 * Every fp32 step above is one correctly rounded IEEE operation, so the
 * quantised bytes are reproducible bit for bit on any conforming machine.
 *
 * F8_128x4 scale layout.  A rows x cols operand has the logical scale matrix
 * S[rows][C], C = cols / 32.  It is stored padded to Rp = ceil(rows/128)*128
 * rows and Cp = ceil(C/4)*4 columns, zero-filled, at byte
 *
 *   off(r, c) = ((r / 128) * (Cp / 4) + c / 4) * 512
 *               + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4)
 *
 * i.e. 512-byte blocks of 128 rows x 4 scale columns.  mx_scale_bytes()
 * returns Rp * Cp.  The functions below write every byte of that buffer,
 * padding included.
 *
 * Conventions for every entry point
 *   - All buffers are caller-owned DEVICE memory; the library allocates
 *     nothing on the call path and keeps no per-call state.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *     and never synchronise the host.
 *   - Arguments are validated before anything is launched; on error nothing
 *     is launched and the status says why.  A failed launch returns
 *     MX_ERR_CUDA (mx_last_cuda_error() gives the CUDA error code).
 *   - Every pointer must be 16-byte aligned (the kernels move data with
 *     TMA bulk copies and 16-byte vector accesses).
 *   - Row-major everywhere.  Sizes are element counts.
 *   - Thread-safe: calls may come from several host threads and streams.
 *   - No exceptions cross the ABI.
 */
#ifndef MXGEMM_H
#define MXGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, spelled so this header needs no CUDA header. */
typedef struct CUstream_st* mx_stream_t;

typedef enum mx_status {
  MX_OK = 0,
  MX_ERR_NULL = 1,          /* a required pointer is NULL                        */
  MX_ERR_ALIGN = 2,         /* a pointer is not 16-byte aligned                  */
  MX_ERR_SHAPE = 3,         /* a size is negative, not a multiple of 32 where    */
                            /* required, or above the supported maximum          */
  MX_ERR_ARCH = 4,          /* the current device is not a compute 10.x part     */
  MX_ERR_CUDA = 5,          /* a CUDA runtime or driver call failed              */
  MX_ERR_DEVICE_TIMEOUT = 6 /* a kernel gave up a bounded wait (mx_device_fault) */
} mx_status;

/* Bytes of the F8_128x4 scale buffer for a rows x cols operand:
 * ceil(rows/128)*128 * ceil(cols/32/4)*4.  Returns 0 if rows < 0, cols < 0
 * or cols % 32 != 0. */
size_t mx_scale_bytes(int64_t rows, int64_t cols);

/* Fused Gemma RMSNorm + MXFP8 quantisation of M rows of width H.
 *
 *   x           [M][H] bf16, read only
 *   w           [H] bf16 gain; the norm multiplies by (1 + w)
 *   eps         added to mean(x^2) inside the square root (fp32)
 *   out_q       [M][H] E4M3 codes (one byte per element), written
 *   out_scales  mx_scale_bytes(M, H) bytes of UE8M0 scales in the F8_128x4
 *               layout, written in full (padding rows/columns set to 0)
 *   M >= 0 (M == 0 is a no-op that returns MX_OK), H % 32 == 0,
 *   32 <= H <= 16384.
 * Inputs must be finite; NaN or Inf inputs give unspecified codes. */
mx_status mx_rmsnorm_quant(const void* x, const void* w, float eps,
                           uint8_t* out_q, uint8_t* out_scales,
                           int64_t M, int64_t H, mx_stream_t stream);

/* Scale layouts of mx_rmsnorm_quant_ex. */
enum {
  MX_SCALES_F8_128X4 = 0, /* mx_scale_bytes(M, H) bytes, swizzled, as mx_rmsnorm_quant */
  MX_SCALES_ROW_MAJOR = 1 /* M * (H / 32) bytes, [M][H/32] row-major, no padding      */
};

/* mx_rmsnorm_quant with the scale layout chosen.  MX_SCALES_ROW_MAJOR serves
 * sequence parallelism: each rank normalises its own token rows, and the
 * 128x4-swizzled scales cannot be concatenated by rows after the all-gather,
 * while row-major ones can; the gathered scales are swizzled once with
 * mx_swizzle_scales (vLLM PR #65496, Details / Tradeoff).  Codes and scale
 * values are bit-identical to mx_rmsnorm_quant's.  A row-major scale buffer
 * needs no alignment (it is written byte by byte); the other pointers must
 * be 16-byte aligned.  Any other scale_layout: MX_ERR_SHAPE. */
mx_status mx_rmsnorm_quant_ex(const void* x, const void* w, float eps,
                              uint8_t* out_q, uint8_t* out_scales,
                              int64_t M, int64_t H, int scale_layout,
                              mx_stream_t stream);

/* The Gemma RMSNorm alone: out[M][H] = bf16(y), y as above, rounded to
 * nearest even.  The path for sequence parallelism in which the norm output
 * stays BF16 through the all-gather and is quantised afterwards
 * (mx_quant_weights) (vLLM PR #65496, Overview and Details / Tradeoff).
 * Same size limits as mx_rmsnorm_quant; out is caller-owned, 16-byte aligned. */
mx_status mx_rmsnorm_bf16(const void* x, const void* w, float eps, void* out,
                          int64_t M, int64_t H, mx_stream_t stream);

/* Output forms of the norm, for mx_rmsnorm_plan. */
enum {
  MX_NORM_SWIZZLED = 0,  /* mx_rmsnorm_quant                                   */
  MX_NORM_ROW_MAJOR = 1, /* mx_rmsnorm_quant_ex with MX_SCALES_ROW_MAJOR         */
  MX_NORM_BF16 = 2       /* mx_rmsnorm_bf16                                    */
};

/* The kernel the norm entry points launch for an M x H input in output form
 * `form` on a GPU of num_sms SMs; no device is touched, so it answers on a
 * machine without a GPU.  plan[4] is written: {warps per row, 1024-element
 * chunks per warp, rows in flight per CTA, 1 if the row stays unpacked in
 * registers between the sum of squares and the quantisation} for the
 * lane-block kernels, or {0, 0, 0, 0} for the chunked kernels (which take
 * odd multiples of 32 and short rows).  M >= 1, H as for mx_rmsnorm_quant,
 * num_sms >= 1, form one of the above: else MX_ERR_SHAPE; plan NULL:
 * MX_ERR_NULL.  The rows-per-SM limits of the choice are same-box timings
 * of every candidate on a 152-SM GB300. */
mx_status mx_rmsnorm_plan(int64_t M, int64_t H, int form, int num_sms, int plan[4]);

/* Row-major [rows][cols/32] UE8M0 scales -> the F8_128x4 layout
 * (mx_scale_bytes(rows, cols) bytes, padding written as 0), and back.
 * These are the swizzle that runs after the all-gather of row-major scales
 * (vLLM PR #65496, Details / Tradeoff) and its inverse.  cols is the width of
 * the quantised operand in elements (cols % 32 == 0, 32 <= cols <= 16384),
 * rows >= 0.  The row-major buffer needs no alignment; the swizzled one must
 * be 16-byte aligned.  Input and output must not overlap. */
mx_status mx_swizzle_scales(const uint8_t* in_row_major, uint8_t* out_swizzled,
                            int64_t rows, int64_t cols, mx_stream_t stream);
mx_status mx_unswizzle_scales(const uint8_t* in_swizzled, uint8_t* out_row_major,
                              int64_t rows, int64_t cols, mx_stream_t stream);

/* Plain MXFP8 quantisation (no norm) of a rows x cols bf16 operand: the
 * activation A (M x K) or the weight W (N x K) of mx_gemm.  Same element and
 * scale rules and the same outputs as mx_rmsnorm_quant with y = x.
 *   rows >= 0, cols % 32 == 0, 32 <= cols <= 16384. */
mx_status mx_quant_weights(const void* x, uint8_t* out_q, uint8_t* out_scales,
                           int64_t rows, int64_t cols, mx_stream_t stream);

/* MXFP8 block-scaled GEMM, C = A . B^T, fp32 accumulation, BF16 output.
 *
 *   a_q [M][K] E4M3, a_s = F8_128x4 scales of A (mx_scale_bytes(M, K) bytes)
 *   b_q [N][K] E4M3, b_s = F8_128x4 scales of B (mx_scale_bytes(N, K) bytes)
 *   out [M][N] bf16, written
 *   M >= 0 (M == 0 is a no-op), N % 16 == 0, N >= 16, K % 32 == 0, K >= 32,
 *   M, N, K <= 2^20.
 * The output tile shape is chosen from (M, N, K, SM count); see
 * mx_gemm_ex to force one. */
mx_status mx_gemm(const uint8_t* a_q, const uint8_t* a_s,
                  const uint8_t* b_q, const uint8_t* b_s,
                  void* out, int64_t M, int64_t N, int64_t K, mx_stream_t stream);

/* mx_gemm with the output tile forced.  (tile_m, tile_n) = (0, 0) picks
 * automatically; otherwise tile_m = 128 (one CTA per tile, tile_n 64, 128 or
 * 192) or tile_m = 256 (a cluster of two CTAs sharing one tcgen05 MMA, each
 * staging half of the B tile; tile_n 128, 192 or 256 -- the 256-column tile
 * has one TMEM accumulator, so a CTA's next tile waits for its epilogue).
 * MX_ERR_SHAPE otherwise. */
mx_status mx_gemm_ex(const uint8_t* a_q, const uint8_t* a_s,
                     const uint8_t* b_q, const uint8_t* b_s,
                     void* out, int64_t M, int64_t N, int64_t K,
                     int tile_m, int tile_n, mx_stream_t stream);

/* The GEMM with its output quantised in the epilogue: C = A . B^T (fp32
 * accumulation) is rounded to bf16 (RNE) and leaves the kernel as an MXFP8
 * operand -- E4M3 codes and UE8M0 scales in the F8_128x4 layout, by the same
 * rules as mx_quant_weights applied to the bf16 C -- ready to be the A
 * operand of the next mx_gemm.  This is the shape of a dense GEMM whose
 * consumer takes a quantized activation (vLLM PR #64659, Details / "GEMM-RS
 * with a quantized input"; PR #65496, Overview).
 *
 *   out_q       [M][N] E4M3 codes, written
 *   out_scales  mx_scale_bytes(M, N) bytes, written in full (padding 0)
 *   N % 32 == 0 in addition to mx_gemm's limits; (tile_m, tile_n) as for
 *   mx_gemm_ex ((0, 0) = automatic).  For a given tile the accumulators, and
 *   hence the bytes, are those the bf16 mx_gemm_ex of that tile rounds. */
mx_status mx_gemm_quant(const uint8_t* a_q, const uint8_t* a_s,
                        const uint8_t* b_q, const uint8_t* b_s,
                        uint8_t* out_q, uint8_t* out_scales,
                        int64_t M, int64_t N, int64_t K,
                        int tile_m, int tile_n, mx_stream_t stream);

/* Self-test of the norm's failure handling.  Launches the lane-block kernel
 * mx_rmsnorm_quant would launch (H % 64 == 0, else MX_ERR_SHAPE) with its
 * row copies withheld, so that every warp's bounded wait for a row runs out
 * after wait_ns nanoseconds (100 us <= wait_ns <= 1 s, else MX_ERR_SHAPE;
 * M >= 1).  The warps of each row group then stop together and set
 * FAULT bit 1 (a consumer gave up) in the device fault word (read it with
 * mx_device_fault); no thread is left waiting.  out_q is not written; scale
 * bytes of padding rows may be.  Arguments as for mx_rmsnorm_quant.  For
 * tests only. */
mx_status mx_rmsnorm_selftest_stall(const void* x, const void* w, float eps,
                                    uint8_t* out_q, uint8_t* out_scales,
                                    int64_t M, int64_t H, uint64_t wait_ns,
                                    mx_stream_t stream);

/* Self-test of the GEMM's failure handling.  Launches mx_gemm_ex's kernel
 * with its producer issuing no copies, so that every bounded wait in it runs
 * out after wait_ns nanoseconds (100 us <= wait_ns <= 1 s, else
 * MX_ERR_SHAPE; M >= 1).  The kernel then takes the path a real stall would:
 * it sets bits in the device fault word (read them with mx_device_fault),
 * frees its tensor memory and exits; no thread is left waiting.  out is not
 * written.  Arguments are validated as for mx_gemm_ex and must describe real
 * buffers of those sizes.  For tests only: it exercises the give-up path
 * without a broken device. */
mx_status mx_gemm_selftest_stall(const uint8_t* a_q, const uint8_t* a_s,
                                 const uint8_t* b_q, const uint8_t* b_s,
                                 void* out, int64_t M, int64_t N, int64_t K,
                                 int tile_m, int tile_n, uint64_t wait_ns,
                                 mx_stream_t stream);

/* The output tile mx_gemm chooses for an M x N x K product on a GPU of
 * num_sms SMs (>= 2); no device is touched, so it answers on a machine
 * without a GPU.  Shapes as for mx_gemm (else MX_ERR_SHAPE), out-pointers
 * non-NULL (else MX_ERR_NULL). */
mx_status mx_gemm_tile_for(int64_t M, int64_t N, int64_t K, int num_sms,
                           int* tile_m, int* tile_n);

/* The launch configuration mx_gemm would use on the current device: output
 * tile, pipeline stages and grid size (CTAs).  Any out-pointer may be NULL. */
mx_status mx_gemm_plan(int64_t M, int64_t N, int64_t K, int* tile_m,
                       int* tile_n, int* stages, int* grid);

/* Conformance probe for the element encoder the kernels use: out[i] =
 * E4M3(in[i]) with round-to-nearest-even and saturation at +-448, for n
 * fp32 values (device buffers).  Used by tests to compare the hardware
 * conversion with the oracle over all fp32 bit patterns. */
mx_status mx_e4m3_encode_f32(const float* in, uint8_t* out, int64_t n,
                             mx_stream_t stream);

/* Reads and clears this library's device fault word on the current device.
 * A kernel that gives up a bounded wait (about one second; only a bug or a
 * broken device can cause it) sets a bit here and exits cleanly instead of
 * hanging.  *code receives the bits (0 = no fault).  Synchronises the
 * current device first (cudaDeviceSynchronize: kernels on every stream,
 * blocking or not), so the word is read after every kernel launched before
 * the call has finished.  Calls from several host threads, or launches
 * racing this call, may see or clear each other's bits.  Returns
 * MX_ERR_DEVICE_TIMEOUT if a bit was set. */
mx_status mx_device_fault(uint32_t* code);

/* The cudaError_t of the most recent failing CUDA call on this host thread. */
int mx_last_cuda_error(void);

/* Human-readable name of a status value (static storage). */
const char* mx_status_string(mx_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
int mx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXGEMM_H */
