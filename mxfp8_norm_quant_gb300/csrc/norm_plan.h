// Kernel choice of the fused Gemma RMSNorm (+ MXFP8 quantisation): which
// kernel, and in which shape, the norm entry points launch for an M x H
// input in a given output form on a GPU of a given SM count.  Host-only
// logic with no CUDA dependency, shared by the launchers (row_lb.cuh) and by
// mx_rmsnorm_plan, which lets tests check the table on a machine without a
// GPU.
#pragma once

namespace mxk {

// Output forms of the norm kernels.
enum RowOutForm : int {
  OUT_MX_SWIZZLED = 0,  // E4M3 codes + F8_128x4 scales (padding rows zeroed)
  OUT_MX_ROWMAJOR = 1,  // E4M3 codes + [M][H/32] row-major scales
  OUT_BF16 = 2,         // the normalised rows rounded to BF16
};

// A lane-block kernel k_rmsnorm_lb<wpr, ncw, groups, form, keep>: wpr warps
// per row, ncw 1024-element chunks per warp, `groups` rows in flight per CTA,
// keep = the row stays unpacked in registers between the sum of squares and
// the quantisation.  wpr == 0: the chunked kernels of row_common.cuh (which
// choose their own shape).
struct NormPlan {
  int wpr, ncw, groups, keep;
};

constexpr int norm_plan_key(int wpr, int ncw, int groups, int keep) {
  return ((wpr * 8 + ncw) * 64 + groups) * 2 + keep;
}

// Rows of 4097..6144 elements (H % 64 == 0, the width of the pages' models),
// by rows per SM, from same-box timings of the candidates at H = 6144 on 152
// SMs (CUDA graphs of launches cycling over inputs larger than 2x L2; us per
// launch, swizzled form; row-major within 1-4 % of it):
//   M      <6,1,2> <3,2,5> <3,2,8> <3,2,6>
//   256     3.22    3.29    3.41    3.39
//   512     4.60    4.22    4.33    4.30
//   1024    7.09    6.34    5.89    6.76
//   1280    8.31    6.88    7.48    7.25
//   2048   11.11    9.06    9.10    9.83
//   4096   19.77   14.68   14.16   14.86
//   8192   36.48   25.49   24.96   25.19
//   32768 137.46   91.72   97.83   89.66
// (the chunked kernels of row_common.cuh: 3.23, 5.58, 7.87, 8.66, 10.81,
// 17.56, 30.56, 101.35).  The BF16 form stores twice the bytes and prefers
// <6,1,4> from 6144 rows (8192: 31.6 against 33.3 for <3,2,8>; 32768: 118.4
// against 131.2).  A kernel whose row groups fill the SMs in one round is
// best while the rows fit; <3,2,5> takes the second round's remainder better
// between 8 and 16 rows per SM.  The quantising forms keep the row unpacked
// where the row groups leave the registers for it (<3,2,5> and <3,2,6>: 5 %
// fewer instructions at 32768 rows, 63.4 M -> 60.2 M; same-box time equal
// unthrottled, 1-2 % faster at 1024-2048 rows); the BF16 form keeps it
// packed (<3,2,6> would spill).
inline NormPlan plan_norm_6144(int form, long long m, long long s) {
  const int keep = form != OUT_BF16 ? 1 : 0;
  if (10 * m <= 17 * s) return {6, 1, 2, 0};
  if (100 * m <= 465 * s) return {3, 2, 5, keep};
  if (m <= 8 * s) return {3, 2, 8, 0};
  if (m <= 16 * s) return {3, 2, 5, keep};
  if (form == OUT_BF16) {
    if (5 * m < 202 * s) return {3, 2, 8, 0};
    return {6, 1, 4, 0};
  }
  if (m < 64 * s) return {3, 2, 8, 0};
  return {3, 2, 6, keep};
}

// The other widths the lane-block kernels take (H % 64 == 0, up to 4096 and
// 6145..16384 elements), by width class and rows per SM, from same-box
// timings on 152 SMs (CUDA graphs of launches cycling over more than 2x L2
// of input; us per launch, swizzled form, the chunked kernels of
// row_common.cuh in brackets; the row-major form follows the swizzled one):
//   H = 256..512: chunked up to 16 rows per SM; 4096 rows <1,1,32> 3.41
//       (3.74), 16384 rows 8.55 (9.79) at H = 256
//   H = 1024: 128 rows <1,1,8> 2.03 (2.43); 2048 <1,1,16> 3.11 (3.79);
//       16384 <1,1,32> 10.4 (13.3)
//   H = 2048: 512 rows <2,1,4> 2.70 (3.07); 1024 <2,1,8> 3.27 (3.80);
//       2048 <1,2,16> 4.42 (5.47); 16384 <1,2,24> 17.3 (19.3)
//   H = 2112 / 3072 (three chunks; WPR = 3 is balanced there): 512 rows
//       <3,1,4> 2.87 / 3.07 (3.53 / 4.26); 1024 <3,1,8> 3.71 / 4.11;
//       16384 <1,4,16> 21.6 / 24.9 (23.8 / 27.9)
//   H = 3136 / 4096: 128 rows <4,1,2> 2.42 / 2.48 (2.84 / 3.29); 2048
//       <2,2,8> 6.30 / 6.62 (7.99 / 8.85); 16384 <1,4,12> 26.0 / 32.9
//       (29.2 / 34.2)
//   H = 7168 / 8192: 128 rows <8,1,2> 2.90 / 3.03 (4.10 / 3.95); 2048
//       <4,2,4> 10.3 / 11.1 (16.2 / 17.0); 16384 <4,2,6> 53.1 / 63.5
//       (89.8 / 91.6)
//   H = 8256 / 12288 / 16384: 512 rows <8,2,2> 5.92 / 6.77 / 7.74 (8.77 /
//       9.85 / 11.0); 16384 <4,4,3> 88.7 / 93.0, <8,2,3> 123 at 16384
//       (146 / 155 / 165)
// The BF16 form stores twice the bytes and prefers fewer rows in flight for
// its largest launches (16384 rows: H = 8192 <4,2,3> 80.6 against <4,2,6>
// 89.8, chunked 86.3; H = 12288 <8,2,2> 122 against <4,4,3> 135, chunked
// 129).
inline NormPlan plan_norm_other(int form, long long m, int H, long long s) {
  const bool bf16 = form == OUT_BF16;
  if (H <= 1024) {
    if (m > 16 * s) return {1, 1, 32, 0};
    if (H <= 512) return {0, 0, 0, 0};
    if (m <= 8 * s) return {1, 1, 8, 0};
    return {1, 1, 16, 0};
  }
  if (H <= 2048) {
    if (m <= 4 * s) return {2, 1, 4, 0};
    if (m <= 8 * s) return {2, 1, 8, 0};
    if (m <= 64 * s) return {1, 2, 16, 0};
    return {1, 2, 24, 0};
  }
  if (H <= 3072) {
    if (m <= 2 * s) return {3, 1, 2, 0};
    if (m <= 4 * s) return {3, 1, 4, 0};
    if (m <= 8 * s) return {3, 1, 8, 0};
    return {1, 4, 16, 0};
  }
  if (H <= 4096) {
    if (m <= 2 * s) return {4, 1, 2, 0};
    if (m <= 4 * s) return {4, 1, 4, 0};
    if (m <= 16 * s) return {2, 2, 8, 0};
    return {1, 4, 12, 0};
  }
  if (H <= 8192) {
    if (2 * m <= 3 * s) return {8, 1, 2, 0};
    if (bf16) return m <= 64 * s ? NormPlan{4, 2, 4, 0} : NormPlan{4, 2, 3, 0};
    return m <= 16 * s ? NormPlan{4, 2, 4, 0} : NormPlan{4, 2, 6, 0};
  }
  if (m <= 4 * s) return {8, 2, 2, 0};
  if (bf16) return (H <= 9216 || (H <= 12288 && m <= 64 * s)) ? NormPlan{8, 2, 3, 0} : NormPlan{8, 2, 2, 0};
  return H <= 12288 ? NormPlan{4, 4, 3, 0} : NormPlan{8, 2, 3, 0};
}

// Rows whose width is a multiple of 64 go to the lane-block kernels (the
// models' 4097..6144 by their own table, the other widths by the table
// above); widths that are an odd multiple of 32 to the chunked kernels.
// Valid for 32 <= H <= 16384, H % 32 == 0, m >= 1, s >= 1.
inline NormPlan plan_norm(int form, long long m, int H, int num_sms) {
  const long long s = num_sms;
  if (H % 64 != 0 || H > 16384) return {0, 0, 0, 0};
  if (H > 4096 && H <= 6144) return plan_norm_6144(form, m, s);
  return plan_norm_other(form, m, H, s);
}

}  // namespace mxk
