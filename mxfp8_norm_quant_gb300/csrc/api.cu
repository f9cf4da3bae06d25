// C ABI of libmxgemm: argument validation, per-device set-up and dispatch.
// Declarations and the contract of every entry point are in include/mxgemm.h.
#include <climits>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "mx_kernels.h"
#include "mxgemm.h"
#include "norm_plan.h"

#define MX_API extern "C" __attribute__((visibility("default")))

static_assert(MX_NORM_SWIZZLED == mxk::OUT_MX_SWIZZLED && MX_NORM_ROW_MAJOR == mxk::OUT_MX_ROWMAJOR &&
                  MX_NORM_BF16 == mxk::OUT_BF16,
              "the header's norm forms are the kernels' output forms");

// The library's device fault word.  Kernels that give up a bounded wait set a
// bit here (see mx_device_fault) instead of hanging the GPU.
__device__ unsigned int g_mx_fault_word;

namespace {

constexpr int MAX_DEVICES = 64;
constexpr int64_t MAX_ROW_WIDTH = 16384;
constexpr int64_t MAX_ROWS = int64_t(1) << 28;
constexpr int64_t MAX_GEMM_DIM = int64_t(1) << 20;

struct DeviceInfo {
  cudaError_t err = cudaSuccess;
  int major = 0, minor = 0, num_sms = 0;
  unsigned int* fault = nullptr;
};

DeviceInfo g_devices[MAX_DEVICES];
std::once_flag g_device_once[MAX_DEVICES];
thread_local int t_last_cuda_error = 0;

mx_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return MX_ERR_CUDA;
}

// Per-device set-up, done once with the device current: compute capability,
// SM count and the device address of the fault word.
mx_status current_device(const DeviceInfo** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= MAX_DEVICES) return cuda_fail(cudaErrorInvalidDevice);
  std::call_once(g_device_once[dev], [dev] {
    DeviceInfo& d = g_devices[dev];
    cudaError_t r = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    if (r == cudaSuccess) r = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (r == cudaSuccess) r = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (r == cudaSuccess && d.major == 10 && d.minor == 3)
      r = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.fault), g_mx_fault_word);
    d.err = r;
  });
  const DeviceInfo& d = g_devices[dev];
  if (d.err != cudaSuccess) return cuda_fail(d.err);
  // the kernels are built for sm_103a only
  if (d.major != 10 || d.minor != 3) return MX_ERR_ARCH;
  *out = &d;
  return MX_OK;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

mx_status launched(cudaError_t e) { return e == cudaSuccess ? MX_OK : cuda_fail(e); }

mx_status check_row_op(int64_t rows, int64_t cols) {
  if (rows < 0 || rows > MAX_ROWS) return MX_ERR_SHAPE;
  if (cols < 32 || cols > MAX_ROW_WIDTH || cols % 32 != 0) return MX_ERR_SHAPE;
  return MX_OK;
}

mx_status check_gemm(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || M > MAX_GEMM_DIM) return MX_ERR_SHAPE;
  if (N < 16 || N > MAX_GEMM_DIM || N % 16 != 0) return MX_ERR_SHAPE;
  if (K < 32 || K > MAX_GEMM_DIM || K % 32 != 0) return MX_ERR_SHAPE;
  return MX_OK;
}

}  // namespace

namespace mxk {

// The table remembers the limit set per (kernel, device); once it is full
// (more than TABLE kernel-device pairs, far beyond this library's ~40
// kernels on 8 devices) the attribute is simply set on every call, which is
// correct but slower.
cudaError_t set_smem_once(const void* kernel, int bytes) {
  struct Entry {
    const void* fn;
    int dev;
    int bytes;
  };
  constexpr int TABLE = 1024;
  static std::mutex mu;
  static Entry table[TABLE];
  static int used = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (table[i].fn == kernel && table[i].dev == dev) {
      if (table[i].bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) table[i].bytes = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && used < TABLE) table[used++] = Entry{kernel, dev, bytes};
  return e;
}

}  // namespace mxk

MX_API size_t mx_scale_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0 || cols % 32 != 0) return 0;
  const int64_t c = cols / 32;
  return static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>((c + 3) / 4 * 4);
}

MX_API mx_status mx_rmsnorm_quant(const void* x, const void* w, float eps, uint8_t* out_q, uint8_t* out_scales,
                                  int64_t M, int64_t H, mx_stream_t stream) {
  mx_status st = check_row_op(M, H);
  if (st != MX_OK) return st;
  if (M == 0) return MX_OK;
  if (!x || !w || !out_q || !out_scales) return MX_ERR_NULL;
  if (misaligned(x) || misaligned(w) || misaligned(out_q) || misaligned(out_scales)) return MX_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = current_device(&d);
  if (st != MX_OK) return st;
  return launched(mxk::launch_rmsnorm_quant(x, w, eps, out_q, out_scales, static_cast<int>(M), static_cast<int>(H),
                                            d->num_sms, d->fault, reinterpret_cast<cudaStream_t>(stream)));
}

MX_API mx_status mx_rmsnorm_quant_ex(const void* x, const void* w, float eps, uint8_t* out_q, uint8_t* out_scales,
                                     int64_t M, int64_t H, int scale_layout, mx_stream_t stream) {
  if (scale_layout == MX_SCALES_F8_128X4) return mx_rmsnorm_quant(x, w, eps, out_q, out_scales, M, H, stream);
  if (scale_layout != MX_SCALES_ROW_MAJOR) return MX_ERR_SHAPE;
  mx_status st = check_row_op(M, H);
  if (st != MX_OK) return st;
  if (M == 0) return MX_OK;
  if (!x || !w || !out_q || !out_scales) return MX_ERR_NULL;
  if (misaligned(x) || misaligned(w) || misaligned(out_q)) return MX_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = current_device(&d);
  if (st != MX_OK) return st;
  return launched(mxk::launch_rmsnorm_quant_rowmajor(x, w, eps, out_q, out_scales, static_cast<int>(M),
                                                     static_cast<int>(H), d->num_sms, d->fault,
                                                     reinterpret_cast<cudaStream_t>(stream)));
}

MX_API mx_status mx_rmsnorm_bf16(const void* x, const void* w, float eps, void* out, int64_t M, int64_t H,
                                 mx_stream_t stream) {
  mx_status st = check_row_op(M, H);
  if (st != MX_OK) return st;
  if (M == 0) return MX_OK;
  if (!x || !w || !out) return MX_ERR_NULL;
  if (misaligned(x) || misaligned(w) || misaligned(out)) return MX_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = current_device(&d);
  if (st != MX_OK) return st;
  return launched(mxk::launch_rmsnorm_bf16(x, w, eps, out, static_cast<int>(M), static_cast<int>(H), d->num_sms,
                                           d->fault, reinterpret_cast<cudaStream_t>(stream)));
}

MX_API mx_status mx_swizzle_scales(const uint8_t* in_row_major, uint8_t* out_swizzled, int64_t rows, int64_t cols,
                                   mx_stream_t stream) {
  mx_status st = check_row_op(rows, cols);
  if (st != MX_OK) return st;
  if (rows == 0) return MX_OK;
  if (!in_row_major || !out_swizzled) return MX_ERR_NULL;
  if (misaligned(out_swizzled)) return MX_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = current_device(&d);
  if (st != MX_OK) return st;
  return launched(mxk::launch_swizzle_scales(in_row_major, out_swizzled, static_cast<int>(rows),
                                             static_cast<int>(cols / 32), d->num_sms,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

MX_API mx_status mx_unswizzle_scales(const uint8_t* in_swizzled, uint8_t* out_row_major, int64_t rows, int64_t cols,
                                     mx_stream_t stream) {
  mx_status st = check_row_op(rows, cols);
  if (st != MX_OK) return st;
  if (rows == 0) return MX_OK;
  if (!in_swizzled || !out_row_major) return MX_ERR_NULL;
  if (misaligned(in_swizzled)) return MX_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = current_device(&d);
  if (st != MX_OK) return st;
  return launched(mxk::launch_unswizzle_scales(in_swizzled, out_row_major, static_cast<int>(rows),
                                               static_cast<int>(cols / 32), d->num_sms,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

MX_API mx_status mx_quant_weights(const void* x, uint8_t* out_q, uint8_t* out_scales, int64_t rows, int64_t cols,
                                  mx_stream_t stream) {
  mx_status st = check_row_op(rows, cols);
  if (st != MX_OK) return st;
  if (rows == 0) return MX_OK;
  if (!x || !out_q || !out_scales) return MX_ERR_NULL;
  if (misaligned(x) || misaligned(out_q) || misaligned(out_scales)) return MX_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = current_device(&d);
  if (st != MX_OK) return st;
  return launched(mxk::launch_quant(x, out_q, out_scales, static_cast<int>(rows), static_cast<int>(cols), d->num_sms,
                                    d->fault, reinterpret_cast<cudaStream_t>(stream)));
}

MX_API mx_status mx_gemm_ex(const uint8_t* a_q, const uint8_t* a_s, const uint8_t* b_q, const uint8_t* b_s,
                            void* out, int64_t M, int64_t N, int64_t K, int tile_m, int tile_n,
                            mx_stream_t stream) {
  mx_status st = check_gemm(M, N, K);
  if (st != MX_OK) return st;
  const bool autotile = tile_m == 0 && tile_n == 0;
  if (!autotile && !mxk::gemm_tile_supported(tile_m, tile_n)) return MX_ERR_SHAPE;
  if (M == 0) return MX_OK;
  if (!a_q || !a_s || !b_q || !b_s || !out) return MX_ERR_NULL;
  if (misaligned(a_q) || misaligned(a_s) || misaligned(b_q) || misaligned(b_s) || misaligned(out))
    return MX_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = current_device(&d);
  if (st != MX_OK) return st;
  if (autotile)
    mxk::gemm_pick_tile(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), d->num_sms, &tile_m, &tile_n);
  return launched(mxk::launch_gemm(a_q, a_s, b_q, b_s, out, static_cast<int>(M), static_cast<int>(N),
                                   static_cast<int>(K), tile_m, tile_n, d->num_sms, d->fault,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

MX_API mx_status mx_rmsnorm_selftest_stall(const void* x, const void* w, float eps, uint8_t* out_q,
                                           uint8_t* out_scales, int64_t M, int64_t H, uint64_t wait_ns,
                                           mx_stream_t stream) {
  mx_status st = check_row_op(M, H);
  if (st != MX_OK) return st;
  if (M == 0 || H % 64 != 0 || wait_ns < 100000ull || wait_ns > 1000000000ull) return MX_ERR_SHAPE;
  if (!x || !w || !out_q || !out_scales) return MX_ERR_NULL;
  if (misaligned(x) || misaligned(w) || misaligned(out_q) || misaligned(out_scales)) return MX_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = current_device(&d);
  if (st != MX_OK) return st;
  if (mxk::plan_norm(MX_NORM_SWIZZLED, M, static_cast<int>(H), d->num_sms).wpr == 0) return MX_ERR_SHAPE;
  return launched(mxk::launch_rmsnorm_quant_stalled(x, w, eps, out_q, out_scales, static_cast<int>(M),
                                                    static_cast<int>(H), d->num_sms, d->fault, wait_ns,
                                                    reinterpret_cast<cudaStream_t>(stream)));
}

MX_API mx_status mx_gemm_selftest_stall(const uint8_t* a_q, const uint8_t* a_s, const uint8_t* b_q,
                                        const uint8_t* b_s, void* out, int64_t M, int64_t N, int64_t K, int tile_m,
                                        int tile_n, uint64_t wait_ns, mx_stream_t stream) {
  mx_status st = check_gemm(M, N, K);
  if (st != MX_OK) return st;
  if (M == 0 || wait_ns < 100000ull || wait_ns > 1000000000ull) return MX_ERR_SHAPE;
  const bool autotile = tile_m == 0 && tile_n == 0;
  if (!autotile && !mxk::gemm_tile_supported(tile_m, tile_n)) return MX_ERR_SHAPE;
  if (!a_q || !a_s || !b_q || !b_s || !out) return MX_ERR_NULL;
  if (misaligned(a_q) || misaligned(a_s) || misaligned(b_q) || misaligned(b_s) || misaligned(out))
    return MX_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = current_device(&d);
  if (st != MX_OK) return st;
  if (autotile)
    mxk::gemm_pick_tile(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), d->num_sms, &tile_m, &tile_n);
  return launched(mxk::launch_gemm_stalled(a_q, a_s, b_q, b_s, out, static_cast<int>(M), static_cast<int>(N),
                                           static_cast<int>(K), tile_m, tile_n, d->num_sms, d->fault, wait_ns,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

MX_API mx_status mx_gemm_quant(const uint8_t* a_q, const uint8_t* a_s, const uint8_t* b_q, const uint8_t* b_s,
                               uint8_t* out_q, uint8_t* out_scales, int64_t M, int64_t N, int64_t K, int tile_m,
                               int tile_n, mx_stream_t stream) {
  mx_status st = check_gemm(M, N, K);
  if (st != MX_OK) return st;
  if (N % 32 != 0) return MX_ERR_SHAPE;
  const bool autotile = tile_m == 0 && tile_n == 0;
  if (!autotile && !mxk::gemm_tile_supported(tile_m, tile_n)) return MX_ERR_SHAPE;
  if (M == 0) return MX_OK;
  if (!a_q || !a_s || !b_q || !b_s || !out_q || !out_scales) return MX_ERR_NULL;
  if (misaligned(a_q) || misaligned(a_s) || misaligned(b_q) || misaligned(b_s) || misaligned(out_q) ||
      misaligned(out_scales))
    return MX_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = current_device(&d);
  if (st != MX_OK) return st;
  if (autotile)
    mxk::gemm_pick_tile(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), d->num_sms, &tile_m, &tile_n);
  return launched(mxk::launch_gemm_quant(a_q, a_s, b_q, b_s, out_q, out_scales, static_cast<int>(M),
                                         static_cast<int>(N), static_cast<int>(K), tile_m, tile_n, d->num_sms,
                                         d->fault, reinterpret_cast<cudaStream_t>(stream)));
}

MX_API mx_status mx_gemm(const uint8_t* a_q, const uint8_t* a_s, const uint8_t* b_q, const uint8_t* b_s, void* out,
                         int64_t M, int64_t N, int64_t K, mx_stream_t stream) {
  return mx_gemm_ex(a_q, a_s, b_q, b_s, out, M, N, K, 0, 0, stream);
}

MX_API mx_status mx_rmsnorm_plan(int64_t M, int64_t H, int form, int num_sms, int plan[4]) {
  mx_status st = check_row_op(M, H);
  if (st != MX_OK) return st;
  if (M < 1 || num_sms < 1 || form < MX_NORM_SWIZZLED || form > MX_NORM_BF16) return MX_ERR_SHAPE;
  if (!plan) return MX_ERR_NULL;
  const mxk::NormPlan pl = mxk::plan_norm(form, M, static_cast<int>(H), num_sms);
  plan[0] = pl.wpr;
  plan[1] = pl.ncw;
  plan[2] = pl.groups;
  plan[3] = pl.keep;
  return MX_OK;
}

MX_API mx_status mx_gemm_tile_for(int64_t M, int64_t N, int64_t K, int num_sms, int* tile_m, int* tile_n) {
  mx_status st = check_gemm(M, N, K);
  if (st != MX_OK) return st;
  if (num_sms < 2) return MX_ERR_SHAPE;
  if (!tile_m || !tile_n) return MX_ERR_NULL;
  mxk::gemm_pick_tile(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), num_sms, tile_m, tile_n);
  return MX_OK;
}

MX_API mx_status mx_gemm_plan(int64_t M, int64_t N, int64_t K, int* tile_m, int* tile_n, int* stages, int* grid) {
  mx_status st = check_gemm(M, N, K);
  if (st != MX_OK) return st;
  const DeviceInfo* d = nullptr;
  st = current_device(&d);
  if (st != MX_OK) return st;
  int tm = 0, tn = 0;
  mxk::gemm_pick_tile(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), d->num_sms, &tm, &tn);
  if (tile_m) *tile_m = tm;
  if (tile_n) *tile_n = tn;
  if (stages) *stages = mxk::gemm_stages(tm, tn);
  if (grid) *grid = M == 0 ? 0 : mxk::gemm_grid(static_cast<int>(M), static_cast<int>(N), tm, tn, d->num_sms);
  return MX_OK;
}

MX_API mx_status mx_e4m3_encode_f32(const float* in, uint8_t* out, int64_t n, mx_stream_t stream) {
  if (n < 0) return MX_ERR_SHAPE;
  if (n == 0) return MX_OK;
  if (!in || !out) return MX_ERR_NULL;
  if (misaligned(in) || misaligned(out)) return MX_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  mx_status st = current_device(&d);
  if (st != MX_OK) return st;
  return launched(
      mxk::launch_e4m3_encode(in, out, static_cast<size_t>(n), d->num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

MX_API mx_status mx_device_fault(uint32_t* code) {
  if (!code) return MX_ERR_NULL;
  const DeviceInfo* d = nullptr;
  mx_status st = current_device(&d);
  if (st != MX_OK) return st;
  // every kernel of the device, on every stream (non-blocking ones included),
  // has finished before the word is read and cleared
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_mx_fault_word, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e);
  if (v != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_mx_fault_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  *code = v;
  return v == 0 ? MX_OK : MX_ERR_DEVICE_TIMEOUT;
}

MX_API int mx_last_cuda_error(void) { return t_last_cuda_error; }

MX_API const char* mx_status_string(mx_status status) {
  switch (status) {
    case MX_OK: return "MX_OK";
    case MX_ERR_NULL: return "MX_ERR_NULL: a required pointer is NULL";
    case MX_ERR_ALIGN: return "MX_ERR_ALIGN: a pointer is not 16-byte aligned";
    case MX_ERR_SHAPE: return "MX_ERR_SHAPE: unsupported size";
    case MX_ERR_ARCH: return "MX_ERR_ARCH: the current device is not sm_103";
    case MX_ERR_CUDA: return "MX_ERR_CUDA: a CUDA call failed";
    case MX_ERR_DEVICE_TIMEOUT: return "MX_ERR_DEVICE_TIMEOUT: a kernel gave up a bounded wait";
  }
  return "unknown mx_status";
}

MX_API int mx_version(void) { return 100; }
