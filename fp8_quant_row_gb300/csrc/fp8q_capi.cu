// fp8q_capi.cu -- host side of libfp8q: argument validation, device checks, launch shapes.
//
// Every entry point validates synchronously and returns a status before anything is
// enqueued; it then launches exactly one kernel on the caller's stream. Nothing here
// allocates device memory or synchronises, so the calls can be captured in CUDA graphs
// once the per-device launch caches below are warm (first call on a device queries
// attributes).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "fp8q.h"
#include "elementwise_kernels.cuh"
#include "nss_kernels.cuh"
#include "nss_ws_kernels.cuh"
#include "nvfp4_kernels.cuh"
#include "qkv_kernels.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxLnCols = 32768;
constexpr int64_t kMaxEwCols = int64_t(1) << 30;

thread_local int g_last_cuda_error = 0;
thread_local char g_last_detail[160] = "";

struct DeviceInfo {
  int major = 0, minor = 0, sms = 0, smem_optin = 0;
  bool ok = false;
};

DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

// Records which runtime call failed (thread-local) and returns FP8Q_ERR_CUDA.
fp8q_status cuda_fail(cudaError_t e, const char* site, long long arg = -1) {
  g_last_cuda_error = int(e);
  std::snprintf(g_last_detail, sizeof g_last_detail, "%s(%lld): %s", site, arg,
                cudaGetErrorName(e));
  return FP8Q_ERR_CUDA;
}

// Current device, checked to be compute capability 10.3.
fp8q_status current_device(const DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return FP8Q_ERR_UNSUPPORTED;
  std::call_once(g_dev_once[dev], [dev] {
    DeviceInfo& d = g_dev[dev];
    d.ok = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
           cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
           cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
           cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ==
               cudaSuccess;
  });
  const DeviceInfo& d = g_dev[dev];
  if (!d.ok) return cuda_fail(cudaErrorInvalidDevice, "cudaDeviceGetAttribute", dev);
  if (d.major != 10 || d.minor != 3) return FP8Q_ERR_UNSUPPORTED;
  *out = &d;
  return FP8Q_OK;
}

// Resident CTAs per SM of a kernel at a dynamic shared-memory size, cached per device.
struct OccEntry {
  int dev;
  const void* fn;
  size_t smem;
  int blocks;
};
OccEntry g_occ[256];
int g_occ_n = 0;
// Dynamic shared-memory limit set on each (device, function): the limit is a property of the
// function, not of a launch, so it only ever grows to the largest size launched (a launch
// above the current limit is rejected; a smaller size seen later must not lower it).
struct SmemLimit {
  int dev;
  const void* fn;
  size_t limit;
};
SmemLimit g_lim[256];
int g_lim_n = 0;
std::mutex g_occ_mu;

fp8q_status raise_smem_limit(int dev, const void* fn, size_t smem) {
  SmemLimit* entry = nullptr;
  for (int i = 0; i < g_lim_n; ++i)
    if (g_lim[i].dev == dev && g_lim[i].fn == fn) entry = &g_lim[i];
  if (entry && entry->limit >= smem) return FP8Q_OK;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)", (long long)smem);
  if (entry) {
    entry->limit = smem;
  } else if (g_lim_n < 256) {
    g_lim[g_lim_n++] = SmemLimit{dev, fn, smem};
  }
  return FP8Q_OK;
}

fp8q_status blocks_per_sm(const void* fn, int threads, size_t smem, int* blocks) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_occ_mu);
  // Checked on every call: the cached occupancy below says nothing about the current limit.
  if (smem > 48 * 1024) {
    const fp8q_status st = raise_smem_limit(dev, fn, smem);
    if (st != FP8Q_OK) return st;
  }
  for (int i = 0; i < g_occ_n; ++i)
    if (g_occ[i].dev == dev && g_occ[i].fn == fn && g_occ[i].smem == smem) {
      *blocks = g_occ[i].blocks;
      return FP8Q_OK;
    }
  int b = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor", (long long)smem);
  if (g_occ_n < 256) g_occ[g_occ_n++] = OccEntry{dev, fn, smem, b};
  *blocks = b;
  return FP8Q_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// Bytes spanned by `tokens` rows of `width` BF16 values at a stride of `ld` values.
size_t strided_bytes(int64_t tokens, int64_t ld, int64_t width) {
  return tokens > 0 ? size_t((tokens - 1) * ld + width) * 2 : 0;
}

struct Range {
  const void* p;
  size_t bytes;
};

bool overlap(Range a, Range b) {
  if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

bool same(Range a, Range b) { return a.p == b.p && a.bytes == b.bytes; }

// One launch; the status is this launch's own (cudaLaunchKernelEx's return value), so an
// unrelated pending error of another library on the same thread is never reported as ours.
// Launches allow programmatic dependent launch: a kernel may be scheduled while the previous
// kernel in the stream drains, and every kernel executes griddepcontrol.wait before its first
// global-memory access, so producer -> consumer ordering is unchanged.
template <typename... Args>
fp8q_status launch(void (*fn)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                   Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, args...);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelEx", (long long)smem);
  return FP8Q_OK;
}

// ------------------------------------------------------------------------------------------
// LayerNorm family
// ------------------------------------------------------------------------------------------

template <int V, int WPR, bool RESID, bool HAS_BIAS>
fp8q_status launch_tuned(const fp8q::NssParams& p, const DeviceInfo& dev, int64_t n_mod,
                         cudaStream_t stream, bool* launched) {
  using L = fp8q::TunedLayout<V, WPR, RESID>;
  auto* fn = fp8q::nss_tuned_kernel<V, WPR, RESID, HAS_BIAS>;
  *launched = false;
  // As many warps per CTA (one CTA per SM) as the shared-memory ring allows, up to 24 where
  // the kernel is built for it; below 16 rows per SM at most 16 (width 3072, two warps per
  // row, 16 -> 24 warps: 2048 rows 10.41 -> 10.70 us, 3072 rows 13.25 -> 13.06 us, 4608 rows
  // 16.85 -> 16.59 us).
  int nw = fp8q::tuned_threads<V, WPR, RESID>() / 32;
  if (p.rows < 16 * int64_t(dev.sms) && nw > fp8q::kTunedMaxThreads / 32)
    nw = fp8q::kTunedMaxThreads / 32;
  while (nw >= WPR && L::smem_bytes(nw) > size_t(dev.smem_optin)) nw -= WPR;
  nw -= nw % WPR;
  if (nw < WPR) return FP8Q_OK;
  if (fp8q::kMaxTableUnitsPerThread * nw * 32 < WPR * V * 32) return FP8Q_OK;
  const size_t smem = L::smem_bytes(nw);
  int bps = 0;
  fp8q_status st = blocks_per_sm(reinterpret_cast<const void*>(fn), nw * 32, smem, &bps);
  if (st != FP8Q_OK) return st;
  if (bps <= 0) return FP8Q_OK;
  const int rows_per_iter = nw / WPR;
  int64_t need = (p.rows + rows_per_iter - 1) / rows_per_iter;
  // Fewer rows than a full wave: spread them over all SMs rather than filling a few CTAs, so
  // each SM's rows finish sooner (a warp or a warp pair computes a whole row).
  if (need < dev.sms) need = p.rows < dev.sms ? p.rows : dev.sms;
  const int64_t cap = int64_t(dev.sms) * bps;
  int64_t grid = need > n_mod ? need : n_mod;
  if (grid > cap) grid = cap;
  // Every CTA must sit inside one modulation group (single-row table).
  if (n_mod > grid) return FP8Q_OK;
  *launched = true;
  return launch(fn, dim3(unsigned(grid)), dim3(nw * 32), smem, stream, p, n_mod);
}

// Warp-specialised kernel: one CTA per SM (never more CTAs than rows), each owning a block
// of rows that it streams through a ring of WsLayout::kStages row stages.
constexpr int kWsDepth = 1 << 30;  // rows in flight per CTA (no limit beyond the ring)

template <int C, int NS, int NO>
fp8q_status launch_ws(const fp8q::NssParams& p, const DeviceInfo& dev, int64_t n_mod,
                      cudaStream_t stream, bool* launched) {
  using L = fp8q::WsLayout<C, NS, NO>;
  auto* fn = fp8q::nss_ws_kernel<C, NS, NO>;
  *launched = false;
  int64_t grid = std::min<int64_t>(dev.sms, p.rows);
  if (n_mod > grid) return FP8Q_OK;  // every CTA must sit inside one modulation group
  if (L::kSmemBytes > size_t(dev.smem_optin)) return FP8Q_OK;
  int bps = 0;
  fp8q_status st = blocks_per_sm(reinterpret_cast<const void*>(fn), L::kThreads, L::kSmemBytes, &bps);
  if (st != FP8Q_OK) return st;
  if (bps <= 0) return FP8Q_OK;
  *launched = true;
  return launch(fn, dim3(unsigned(grid)), dim3(L::kThreads), L::kSmemBytes, stream, p, n_mod,
                kWsDepth);
}

template <bool RESID, bool HAS_BIAS>
fp8q_status launch_generic(const fp8q::NssParams& p, const DeviceInfo& dev, cudaStream_t stream) {
  auto* fn = fp8q::nss_generic_kernel<RESID, HAS_BIAS>;
  const size_t smem = size_t(p.cols) * 2;
  int bps = 0;
  fp8q_status st = blocks_per_sm(reinterpret_cast<const void*>(fn), fp8q::kNssThreads, smem, &bps);
  if (st != FP8Q_OK) return st;
  if (bps <= 0) return cuda_fail(cudaErrorInvalidConfiguration, "occupancy", (long long)smem);
  int64_t grid = int64_t(dev.sms) * bps;
  if (grid > p.rows) grid = p.rows;
  return launch(fn, dim3(unsigned(grid)), dim3(fp8q::kNssThreads), smem, stream, p);
}

template <bool RESID, bool HAS_BIAS>
fp8q_status dispatch_ln(const fp8q::NssParams& p, const DeviceInfo& dev, int64_t n_mod,
                        cudaStream_t stream) {
  bool launched = false;
  fp8q_status st = FP8Q_OK;
  // Up to two rows per SM the CTA-per-row kernel (eight warps share a row) has the lower
  // latency (width 3072, against the tuned kernel with two warps per row: 4.19 vs 4.58 us at
  // 153 rows, 4.53 vs 4.83 at 256; above, 4.91 vs 5.25 at 400, 5.26 vs 6.12 at 512).
  // At width 3072 two warps share a row up to 48 rows per SM: each warp's chain of per-row
  // work is half as long, which pays while a warp has few rows (width 3072, one vs two warps
  // per row: 1024 rows 9.02 -> 7.44 us, 4608 rows 16.97 -> 16.74 us, 6144 rows 21.16 ->
  // 20.54 us, but 9216 rows 27.47 -> 28.14 us). The residual variant always uses two: its
  // ring stages hold two rows' worth of input (x and residual), and half rows per warp let
  // twice as many warps fit in shared memory.
  if (p.rows <= 2 * int64_t(dev.sms)) return launch_generic<RESID, HAS_BIAS>(p, dev, stream);
  if (!RESID && p.cols == 3072) {
    st = launch_ws<3072, 7, 3>(p, dev, n_mod, stream, &launched);
    if (st != FP8Q_OK || launched) return st;
  }
  if (p.cols == 3072 && (RESID || p.rows <= 48 * int64_t(dev.sms)))
    st = launch_tuned<6, 2, RESID, HAS_BIAS>(p, dev, n_mod, stream, &launched);
  else if (p.cols == 3072)
    st = launch_tuned<12, 1, RESID, HAS_BIAS>(p, dev, n_mod, stream, &launched);
  else if (p.cols == 6144)
    st = launch_tuned<12, 2, RESID, HAS_BIAS>(p, dev, n_mod, stream, &launched);
  if (st != FP8Q_OK || launched) return st;
  return launch_generic<RESID, HAS_BIAS>(p, dev, stream);
}

fp8q_status check_ln_shape(int64_t rows, int64_t cols, int64_t mod_rows, float eps) {
  if (rows < 0 || mod_rows < 0) return FP8Q_ERR_SHAPE;
  if (cols < 8 || cols > kMaxLnCols || cols % 8 != 0) return FP8Q_ERR_SHAPE;
  if (!std::isfinite(eps) || eps < 0.0f) return FP8Q_ERR_VALUE;
  return FP8Q_OK;
}

int64_t mod_count(int64_t rows, int64_t mod_rows) {
  return mod_rows > 0 ? (rows + mod_rows - 1) / mod_rows : 1;
}

}  // namespace

extern "C" {

fp8q_status fp8q_nss_fp8(void* y_bf16, uint8_t* q_e4m3, const void* x_bf16,
                         const void* scale_bf16, const void* shift_bf16, int64_t mod_rows,
                         const float* input_scale, int64_t rows, int64_t cols, float eps,
                         cudaStream_t stream) {
  fp8q_status st = check_ln_shape(rows, cols, mod_rows, eps);
  if (st != FP8Q_OK || rows == 0) return st;
  if (!y_bf16 || !q_e4m3 || !x_bf16 || !scale_bf16 || !shift_bf16 || !input_scale)
    return FP8Q_ERR_NULL;
  if (!aligned16(y_bf16) || !aligned16(q_e4m3) || !aligned16(x_bf16) || !aligned16(scale_bf16) ||
      !aligned16(shift_bf16))
    return FP8Q_ERR_ALIGN;
  const int64_t n_mod = mod_count(rows, mod_rows);
  const size_t n = size_t(rows) * size_t(cols);
  const Range y{y_bf16, n * 2}, q{q_e4m3, n}, x{x_bf16, n * 2};
  const Range sc{scale_bf16, size_t(n_mod) * cols * 2}, sh{shift_bf16, size_t(n_mod) * cols * 2};
  const Range is{input_scale, 4};
  for (Range out : {y, q})
    for (Range in : {x, sc, sh, is})
      if (overlap(out, in)) return FP8Q_ERR_ALIAS;
  if (overlap(y, q)) return FP8Q_ERR_ALIAS;
  const DeviceInfo* dev = nullptr;
  st = current_device(&dev);
  if (st != FP8Q_OK) return st;
  fp8q::NssParams p{};
  p.x = static_cast<const uint16_t*>(x_bf16);
  p.scale = static_cast<const uint16_t*>(scale_bf16);
  p.shift = static_cast<const uint16_t*>(shift_bf16);
  p.y = static_cast<uint16_t*>(y_bf16);
  p.q = q_e4m3;
  p.input_scale = input_scale;
  p.rows = rows;
  p.mod_rows = mod_rows;
  p.cols = int(cols);
  p.eps = eps;
  return dispatch_ln<false, false>(p, *dev, n_mod, stream);
}

fp8q_status fp8q_scale_residual_nss_fp8(void* residual_out, void* y_bf16, uint8_t* q_e4m3,
                                        const void* x_bf16, const void* residual_bf16,
                                        const void* bias_bf16, const void* gate_bf16,
                                        const void* scale_bf16, const void* shift_bf16,
                                        int64_t mod_rows, const float* input_scale,
                                        int64_t rows, int64_t cols, float eps,
                                        cudaStream_t stream) {
  fp8q_status st = check_ln_shape(rows, cols, mod_rows, eps);
  if (st != FP8Q_OK || rows == 0) return st;
  if (!residual_out || !y_bf16 || !q_e4m3 || !x_bf16 || !residual_bf16 || !gate_bf16 ||
      !scale_bf16 || !shift_bf16 || !input_scale)
    return FP8Q_ERR_NULL;
  if (!aligned16(residual_out) || !aligned16(y_bf16) || !aligned16(q_e4m3) ||
      !aligned16(x_bf16) || !aligned16(residual_bf16) || !aligned16(gate_bf16) ||
      !aligned16(scale_bf16) || !aligned16(shift_bf16) || (bias_bf16 && !aligned16(bias_bf16)))
    return FP8Q_ERR_ALIGN;
  const int64_t n_mod = mod_count(rows, mod_rows);
  const size_t n = size_t(rows) * size_t(cols);
  const size_t mod_bytes = size_t(n_mod) * cols * 2;
  const Range ro{residual_out, n * 2}, y{y_bf16, n * 2}, q{q_e4m3, n};
  const Range x{x_bf16, n * 2}, res{residual_bf16, n * 2}, b{bias_bf16, size_t(cols) * 2};
  const Range g{gate_bf16, mod_bytes}, sc{scale_bf16, mod_bytes}, sh{shift_bf16, mod_bytes};
  const Range is{input_scale, 4};
  for (Range out : {ro, y, q})
    for (Range in : {x, res, b, g, sc, sh, is}) {
      if (out.p == ro.p && same(ro, res) && in.p == res.p) continue;  // in-place residual
      if (overlap(out, in)) return FP8Q_ERR_ALIAS;
    }
  if (overlap(ro, y) || overlap(ro, q) || overlap(y, q)) return FP8Q_ERR_ALIAS;
  const DeviceInfo* dev = nullptr;
  st = current_device(&dev);
  if (st != FP8Q_OK) return st;
  fp8q::NssParams p{};
  p.x = static_cast<const uint16_t*>(x_bf16);
  p.residual = static_cast<const uint16_t*>(residual_bf16);
  p.bias = static_cast<const uint16_t*>(bias_bf16);
  p.gate = static_cast<const uint16_t*>(gate_bf16);
  p.scale = static_cast<const uint16_t*>(scale_bf16);
  p.shift = static_cast<const uint16_t*>(shift_bf16);
  p.residual_out = static_cast<uint16_t*>(residual_out);
  p.y = static_cast<uint16_t*>(y_bf16);
  p.q = q_e4m3;
  p.input_scale = input_scale;
  p.rows = rows;
  p.mod_rows = mod_rows;
  p.cols = int(cols);
  p.eps = eps;
  if (bias_bf16) return dispatch_ln<true, true>(p, *dev, n_mod, stream);
  return dispatch_ln<true, false>(p, *dev, n_mod, stream);
}

fp8q_status fp8q_bias_mul_add(void* y_bf16, const void* x_bf16, const void* bias_bf16,
                              const void* gate_bf16, const void* residual_bf16, int64_t rows,
                              int64_t cols, cudaStream_t stream) {
  if (rows < 0 || cols < 8 || cols % 8 != 0 || cols > kMaxEwCols) return FP8Q_ERR_SHAPE;
  if (rows == 0) return FP8Q_OK;
  if (!y_bf16 || !x_bf16 || !bias_bf16 || !gate_bf16 || !residual_bf16) return FP8Q_ERR_NULL;
  if (!aligned16(y_bf16) || !aligned16(x_bf16) || !aligned16(bias_bf16) ||
      !aligned16(gate_bf16) || !aligned16(residual_bf16))
    return FP8Q_ERR_ALIGN;
  const size_t n = size_t(rows) * size_t(cols);
  const Range y{y_bf16, n * 2}, x{x_bf16, n * 2}, res{residual_bf16, n * 2};
  const Range b{bias_bf16, size_t(cols) * 2}, g{gate_bf16, size_t(cols) * 2};
  // Elementwise: y may be exactly x or exactly residual; partial overlaps are rejected.
  if ((overlap(y, x) && !same(y, x)) || (overlap(y, res) && !same(y, res)) || overlap(y, b) ||
      overlap(y, g))
    return FP8Q_ERR_ALIAS;
  const DeviceInfo* dev = nullptr;
  fp8q_status st = current_device(&dev);
  if (st != FP8Q_OK) return st;
  const int chunks = int(cols / 8);
  const int per_cta = fp8q::kEwThreads * fp8q::kBmaUnroll;
  const unsigned gy = unsigned((chunks + per_cta - 1) / per_cta);
  if (gy > 65535u) return FP8Q_ERR_SHAPE;
  // Two rows per CTA once one row per CTA would need more than one wave of resident CTAs.
  auto* fn1 = fp8q::bias_mul_add_kernel<1>;
  auto* fn2 = fp8q::bias_mul_add_kernel<2>;
  int bps = 0;
  st = blocks_per_sm(reinterpret_cast<const void*>(fn2), fp8q::kEwThreads, 0, &bps);
  if (st != FP8Q_OK) return st;
  const int64_t wave = int64_t(dev->sms) * (bps > 0 ? bps : 1);
  const bool two = rows * int64_t(gy) > wave;
  const int64_t gx64 = two ? (rows + 1) / 2 : rows;
  const unsigned gx = unsigned(gx64 < 0x7FFFFFFF ? gx64 : 0x7FFFFFFF);
  auto* yp = static_cast<uint16_t*>(y_bf16);
  auto* xp = static_cast<const uint16_t*>(x_bf16);
  auto* bp = static_cast<const uint16_t*>(bias_bf16);
  auto* gp = static_cast<const uint16_t*>(gate_bf16);
  auto* rp = static_cast<const uint16_t*>(residual_bf16);
  if (two)
    return launch(fn2, dim3(gx, gy), dim3(fp8q::kEwThreads), 0, stream, yp, xp, bp, gp, rp, rows,
                  int(cols));
  return launch(fn1, dim3(gx, gy), dim3(fp8q::kEwThreads), 0, stream, yp, xp, bp, gp, rp, rows,
                int(cols));
}

fp8q_status fp8q_token_cat_fp8(uint8_t* q_e4m3, const void* a_bf16, int64_t a_cols,
                               const void* m_bf16, int64_t m_cols, const float* input_scale,
                               int64_t rows, cudaStream_t stream) {
  if (rows < 0 || a_cols < 16 || m_cols < 16 || a_cols % 16 != 0 || m_cols % 16 != 0 ||
      a_cols + m_cols > kMaxEwCols)
    return FP8Q_ERR_SHAPE;
  if (rows == 0) return FP8Q_OK;
  if (!q_e4m3 || !a_bf16 || !m_bf16 || !input_scale) return FP8Q_ERR_NULL;
  if (!aligned16(q_e4m3) || !aligned16(a_bf16) || !aligned16(m_bf16)) return FP8Q_ERR_ALIGN;
  const Range q{q_e4m3, size_t(rows) * size_t(a_cols + m_cols)};
  const Range a{a_bf16, size_t(rows) * size_t(a_cols) * 2};
  const Range m{m_bf16, size_t(rows) * size_t(m_cols) * 2};
  const Range is{input_scale, 4};
  if (overlap(q, a) || overlap(q, m) || overlap(q, is)) return FP8Q_ERR_ALIAS;
  const DeviceInfo* dev = nullptr;
  fp8q_status st = current_device(&dev);
  if (st != FP8Q_OK) return st;
  const int chunks = int((a_cols + m_cols) / 8);
  const int per_cta = fp8q::kEwThreads * fp8q::kCatUnroll;
  const unsigned gy = unsigned((chunks + per_cta - 1) / per_cta);
  const unsigned gx = unsigned(rows < 0x7FFFFFFF ? rows : 0x7FFFFFFF);
  if (gy > 65535u) return FP8Q_ERR_SHAPE;
  return launch(fp8q::token_cat_fp8_kernel, dim3(gx, gy), dim3(fp8q::kEwThreads), 0, stream,
                q_e4m3, static_cast<const uint16_t*>(a_bf16), int(a_cols),
                static_cast<const uint16_t*>(m_bf16), int(m_cols), input_scale, rows);
}

int64_t fp8q_nvfp4_scale_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 16 || cols % 16 != 0 || cols > kMaxEwCols) return -1;
  const int64_t groups = cols / 16;
  return (rows + 127) / 128 * 128 * ((groups + 3) / 4 * 4);
}

fp8q_status fp8q_token_cat_nvfp4(uint8_t* q_fp4, uint8_t* sf_e4m3, const void* a_bf16,
                                 int64_t a_cols, const void* m_bf16, int64_t m_cols,
                                 const float* global_scale, int64_t rows, cudaStream_t stream) {
  if (rows < 0 || a_cols < 64 || m_cols < 64 || a_cols % 64 != 0 || m_cols % 64 != 0 ||
      a_cols + m_cols > kMaxEwCols)
    return FP8Q_ERR_SHAPE;
  if (rows == 0) return FP8Q_OK;
  if (!q_fp4 || !sf_e4m3 || !a_bf16 || !m_bf16 || !global_scale) return FP8Q_ERR_NULL;
  if (!aligned32(q_fp4) || !aligned32(a_bf16) || !aligned32(m_bf16) || !aligned16(sf_e4m3))
    return FP8Q_ERR_ALIGN;
  const int64_t cols = a_cols + m_cols;
  const int64_t rows_pad = (rows + 127) / 128 * 128;
  const Range q{q_fp4, size_t(rows) * size_t(cols / 2)};
  const Range sf{sf_e4m3, size_t(fp8q_nvfp4_scale_bytes(rows, cols))};
  const Range a{a_bf16, size_t(rows) * size_t(a_cols) * 2};
  const Range m{m_bf16, size_t(rows) * size_t(m_cols) * 2};
  const Range gs{global_scale, 4};
  if (overlap(q, a) || overlap(q, m) || overlap(q, gs) || overlap(sf, a) || overlap(sf, m) ||
      overlap(sf, gs) || overlap(q, sf))
    return FP8Q_ERR_ALIAS;
  const DeviceInfo* dev = nullptr;
  fp8q_status st = current_device(&dev);
  if (st != FP8Q_OK) return st;
  const int64_t units = cols / 64;
  const int64_t items = rows_pad / 8 * ((units + 3) / 4);  // warp items (see the kernel)
  const int64_t warps_per_cta = fp8q::kFp4Threads / 32;
  int bps = 0;
  st = blocks_per_sm(reinterpret_cast<const void*>(fp8q::token_cat_nvfp4_kernel),
                     fp8q::kFp4Threads, 0, &bps);
  if (st != FP8Q_OK) return st;
  // One item per warp (short CTAs, one after another) unless that is under two waves of
  // resident CTAs: then a persistent grid of exactly one wave spreads the items evenly over
  // all warps (FLUX.2 widths: 512 tokens 8.16 -> 7.69 us; at 4096 tokens and above one item
  // per warp is faster, 42.5 against 47.7 us persistent).
  const int64_t blocks = (items + warps_per_cta - 1) / warps_per_cta;
  const int64_t wave = int64_t(dev->sms) * std::max(bps, 1);
  const int64_t grid = blocks < 2 * wave ? std::min(blocks, wave) : blocks;
  if (grid > 0x7FFFFFFF) return FP8Q_ERR_SHAPE;
  return launch(fp8q::token_cat_nvfp4_kernel, dim3(unsigned(grid)), dim3(fp8q::kFp4Threads), 0,
                stream, q_fp4, sf_e4m3, static_cast<const uint16_t*>(a_bf16), int(a_cols / 64),
                static_cast<const uint16_t*>(m_bf16), int(m_cols / 64), global_scale, rows,
                rows_pad);
}

fp8q_status fp8q_qkv_epilogue(void* joint_q, void* joint_k, void* joint_v,
                              const fp8q_qkv_stream* txt, const fp8q_qkv_stream* img,
                              int64_t heads, cudaStream_t stream) {
  if (!txt || !img) return FP8Q_ERR_NULL;
  if (heads < 1 || heads > 4096) return FP8Q_ERR_SHAPE;
  const int64_t width = heads * fp8q::kHeadDim;
  const fp8q_qkv_stream* st[2] = {txt, img};
  for (const fp8q_qkv_stream* s : st) {
    if (s->tokens < 0 || (s->tokens > 0 && (s->ld < width || s->ld % 16 != 0)))
      return FP8Q_ERR_SHAPE;
  }
  const int64_t total = txt->tokens + img->tokens;
  if (total == 0) return FP8Q_OK;
  for (const fp8q_qkv_stream* s : st) {
    if (s->tokens == 0) continue;
    if (!(s->eps > 0.0f) || !std::isfinite(s->eps)) return FP8Q_ERR_VALUE;
  }
  if (!joint_q || !joint_k || !joint_v) return FP8Q_ERR_NULL;
  for (const fp8q_qkv_stream* s : st) {
    if (s->tokens == 0) continue;
    if (!s->q || !s->k || !s->v || !s->q_weight || !s->k_weight || !s->cos_sin)
      return FP8Q_ERR_NULL;
    if (!aligned32(s->q) || !aligned32(s->k) || !aligned32(s->v) || !aligned32(s->q_weight) ||
        !aligned32(s->k_weight) || !aligned32(s->cos_sin))
      return FP8Q_ERR_ALIGN;
  }
  if (!aligned32(joint_q) || !aligned32(joint_k) || !aligned32(joint_v)) return FP8Q_ERR_ALIGN;
  const size_t out_bytes = size_t(total) * size_t(width) * 2;
  const Range outs[3] = {{joint_q, out_bytes}, {joint_k, out_bytes}, {joint_v, out_bytes}};
  for (int i = 0; i < 3; ++i) {
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i], outs[j])) return FP8Q_ERR_ALIAS;
    for (const fp8q_qkv_stream* s : st) {
      if (s->tokens == 0) continue;
      const Range ins[6] = {{s->q, strided_bytes(s->tokens, s->ld, width)},
                            {s->k, strided_bytes(s->tokens, s->ld, width)},
                            {s->v, strided_bytes(s->tokens, s->ld, width)},
                            {s->q_weight, size_t(fp8q::kHeadDim) * 2},
                            {s->k_weight, size_t(fp8q::kHeadDim) * 2},
                            {s->cos_sin, size_t(s->tokens) * fp8q::kHeadDim * 4}};
      for (const Range& r : ins)
        if (overlap(outs[i], r)) return FP8Q_ERR_ALIAS;
    }
  }
  const DeviceInfo* dev = nullptr;
  fp8q_status stt = current_device(&dev);
  if (stt != FP8Q_OK) return stt;
  fp8q::QkvParams p;
  p.jq = static_cast<uint16_t*>(joint_q);
  p.jk = static_cast<uint16_t*>(joint_k);
  p.jv = static_cast<uint16_t*>(joint_v);
  fp8q::QkvStream* dstp[2] = {&p.txt, &p.img};
  for (int i = 0; i < 2; ++i) {
    dstp[i]->q = static_cast<const uint16_t*>(st[i]->q);
    dstp[i]->k = static_cast<const uint16_t*>(st[i]->k);
    dstp[i]->v = static_cast<const uint16_t*>(st[i]->v);
    dstp[i]->wq = static_cast<const uint16_t*>(st[i]->q_weight);
    dstp[i]->wk = static_cast<const uint16_t*>(st[i]->k_weight);
    dstp[i]->cos_sin = st[i]->cos_sin;
    dstp[i]->ld = st[i]->ld;
    dstp[i]->tokens = st[i]->tokens;
    dstp[i]->eps = st[i]->eps;
  }
  p.heads = int(heads);
  if (heads <= fp8q::kQkvMaxWsHeads) {
    // warp-specialised: one CTA per SM (never more CTAs than tokens), a ring of whole tokens
    const size_t per_stage = fp8q::qws_stage_bytes(int(heads)) + 20;
    const int64_t fit = (int64_t(dev->smem_optin) - fp8q::kQkvWeightBytes - 16) / int64_t(per_stage);
    const int stages = int(std::min<int64_t>(fit, fp8q::kQwsMaxStages));
    if (stages >= 2) {
      const size_t smem = fp8q::qws_smem_bytes(int(heads), stages);
      const int nw = fp8q::qws_qk_warps(int(heads));
      auto* fn = nw == 16 ? fp8q::qkv_ws_kernel<16> : fp8q::qkv_ws_kernel<13>;
      const int threads = fp8q::qws_threads(nw);
      int bps = 0;
      stt = blocks_per_sm(reinterpret_cast<const void*>(fn), threads, smem, &bps);
      if (stt != FP8Q_OK) return stt;
      if (bps > 0) {
        const int64_t grid = std::min<int64_t>(total, dev->sms);
        return launch(fn, dim3(unsigned(grid)), dim3(threads), smem, stream, p, stages);
      }
    }
  }
  const unsigned gx = unsigned(total < 0x7FFFFFFF ? total : 0x7FFFFFFF);
  return launch(fp8q::qkv_epilogue_kernel, dim3(gx), dim3(fp8q::kQkvWarps * 32), 0, stream, p);
}

fp8q_status fp8q_device_error(unsigned int* bits) {
  if (!bits) return FP8Q_ERR_NULL;
  const DeviceInfo* dev = nullptr;
  fp8q_status st = current_device(&dev);
  if (st != FP8Q_OK) return st;
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, fp8q::g_device_error, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol(g_device_error)");
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(fp8q::g_device_error, &zero, sizeof zero);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol(g_device_error)");
  *bits = v;
  return FP8Q_OK;
}

const char* fp8q_status_string(int status) {
  switch (status) {
    case FP8Q_OK: return "ok";
    case FP8Q_ERR_NULL: return "null pointer";
    case FP8Q_ERR_ALIGN: return "pointer not aligned (16 bytes; 32 for NVFP4 and QKV data)";
    case FP8Q_ERR_SHAPE: return "unsupported shape";
    case FP8Q_ERR_UNSUPPORTED: return "device is not compute capability 10.3 (GB300)";
    case FP8Q_ERR_ALIAS: return "an output overlaps an input or another output";
    case FP8Q_ERR_CUDA: return "CUDA runtime error";
    case FP8Q_ERR_VALUE: return "scalar argument out of range";
    default: return "unknown status";
  }
}

int fp8q_last_cuda_error(void) { return g_last_cuda_error; }

const char* fp8q_last_error_detail(void) { return g_last_detail; }

int fp8q_version(void) { return 0x000300; }

}  // extern "C"
