// dd_lmhead_select_noalloc: the LM head + confidence select for callers that
// must not allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine): code that
// runs under a host framework's memory pool or a fixed device-memory budget
// it must not bypass, and latency-critical loops that cannot afford the
// implicit device synchronisation an allocation may cause.  They still own
// their inputs and outputs; only the kernel's scratch (the per-vocab-tile
// partials of the fused select) has to come from somewhere else.  Here it
// comes from a file-scope device array that every GPU loading this library
// holds until the process exits.
//
// The array's name is only a host-side stand-in in host code, so the first
// call on each device looks up its device address with
// cudaGetSymbolAddress (with that device current) and caches it.  With lazy
// module loading (CUDA's default) that lookup is also what loads the module
// and creates the array, so the first call may allocate and synchronise: it
// is a warm-up, to be made before any stream capture and outside any region
// that must not allocate.  The cached address is not refreshed, so a device
// reset after the first call is not supported.  Every call shares the array
// and it keeps the previous call's contents; calls that overlap on the GPU
// (on different streams, or from different threads) race on it.
//
// A bounded wait inside the GEMM that expires sets the status word at the
// start of the array; a last kernel reads it and, when it is set, overwrites
// every output with conf = NaN and arg = -1, so an expired wait never leaves
// plausible-looking results behind.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/dd.h"
#include "kernels.h"

namespace {

// Capacity: 256 bytes of status word plus three arrays of
// rows * (vocab / 256) four-byte entries (max, sum of exp, argmax).
constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr size_t kStatusBytes = 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

dd_status error(dd_status s, const char* msg) {
  dd::set_error_message(msg);
  return s;
}

// Device address of the scratch array on the current device (looked up once).
dd_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return error(DD_ERR_CUDA, "dd_lmhead_select_noalloc: no usable current device");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return error(DD_ERR_CUDA, "dd_lmhead_select_noalloc: cudaGetSymbolAddress of the scratch array failed");
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return DD_OK;
}

// Runs after the select: if the GEMM recorded an expired wait, no output of
// this call is valid.
__global__ void k_noalloc_status_outputs(const int* status, float* conf, int* arg, int rows) {
  if (*status == 0) return;
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows; r += gridDim.x * blockDim.x) {
    conf[r] = __int_as_float(0x7fc00000);
    arg[r] = -1;
  }
}

}  // namespace

extern "C" dd_status dd_lmhead_select_noalloc(int32_t rows, int32_t hidden, int32_t vocab, const void* x,
                                              const void* w, float* conf, int32_t* arg, void* stream) {
  if (rows < 1 || hidden < 64 || hidden % 64 || vocab < 256 || vocab % 256)
    return error(DD_ERR_UNSUPPORTED, "dd_lmhead_select_noalloc: need rows >= 1, hidden % 64 == 0, vocab % 256 == 0");
  if (!x || !w || !conf || !arg) return error(DD_ERR_INVALID_ARG, "dd_lmhead_select_noalloc: null pointer");
  const size_t tiles = (size_t)(vocab / 256);
  const size_t part = round256(tiles * (size_t)rows * 4);
  if (kStatusBytes + 3 * part > kScratchBytes)
    return error(DD_ERR_INVALID_ARG,
                 "dd_lmhead_select_noalloc: rows * (vocab / 256) exceeds the built-in scratch "
                 "(8 MiB: rows * (vocab / 256) must be at most 698944)");
  void* scratch = nullptr;
  dd_status s = scratch_address(&scratch);
  if (s != DD_OK) return s;
  if (dd::prepare_kernels() != cudaSuccess)
    return error(DD_ERR_CUDA, "dd_lmhead_select_noalloc: kernel set-up failed");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  dd::GemmPlan p = dd::plan_gemm(dd::kEpiSelect, rows, vocab, hidden);
  CUtensorMap mx, mw;
  if (!dd::make_map_2d(&mx, x, rows, hidden, 128) || !dd::make_map_2d(&mw, w, vocab, hidden, p.BN))
    return error(DD_ERR_CUDA, "dd_lmhead_select_noalloc: tensor map encoding failed");
  unsigned char* base = static_cast<unsigned char*>(scratch);
  // The status word is the only state that must start at zero; the partials
  // are fully overwritten by every call.
  if (cudaMemsetAsync(base, 0, kStatusBytes, st) != cudaSuccess)
    return error(DD_ERR_CUDA, "dd_lmhead_select_noalloc: clearing the status word failed");
  dd::GemmOut o{};
  o.rows_valid = rows;
  o.sel_m = reinterpret_cast<float*>(base + kStatusBytes);
  o.sel_s = reinterpret_cast<float*>(base + kStatusBytes + part);
  o.sel_a = reinterpret_cast<int*>(base + kStatusBytes + 2 * part);
  const int* status = reinterpret_cast<const int*>(base);
  if (dd::launch_gemm(p, mx, mw, o, reinterpret_cast<int*>(base), dd::kDefaultTimeoutNs, st) != cudaSuccess ||
      dd::launch_select_combine(o.sel_m, o.sel_s, o.sel_a, p.n_tiles, rows, conf, arg, st) != cudaSuccess)
    return error(DD_ERR_CUDA, "dd_lmhead_select_noalloc: kernel launch failed");
  const int threads = 256, blocks = (rows + threads - 1) / threads < 148 ? (rows + threads - 1) / threads : 148;
  k_noalloc_status_outputs<<<blocks, threads, 0, st>>>(status, conf, arg, rows);
  if (cudaGetLastError() != cudaSuccess)
    return error(DD_ERR_CUDA, "dd_lmhead_select_noalloc: status kernel launch failed");
  return DD_OK;
}
