// noalloc.cu -- a context projection that performs no device allocation.
//
// dflash_ctx_project() grows layer-owned scratch buffers with cudaMalloc the
// first time it meets a larger request.  Some callers cannot allow that:
// serving processes that plan all device memory at start-up and treat any
// later allocation as a fault, and hosts that hand the GPU to a custom pool
// and must not see a library take memory behind its back.
// dflash_ctx_project_noalloc() gives them the same computation with its
// scratch (the fp32 fc output, the split-K partial tiles and their counters)
// carved from one fixed array in the library's device image, sized
// kScratchBytes.  The array exists on every GPU that
// loads the library, for the life of the process.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "handles.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = 16u << 20;  // 16 MiB, also stated in the header
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on `dev` (the current device), looked up once
// per device, at the first call on that device.  The first lookup may load
// the library's device code on that device, which is why that first call
// should come before any stream capture.
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

int dflash_noalloc_fail(int code, const char* msg);

extern "C" int dflash_ctx_project_noalloc(dflash_attn* a, const void* x, int rows,
                                          void* y, dflash_stream stream) {
  if (a == nullptr) return dflash_noalloc_fail(DFLASH_ERR_ARG, "null layer handle");
  if (a->nL == 0)
    return dflash_noalloc_fail(DFLASH_ERR_UNSUPPORTED, "layer was created without fc");
  if (rows < 0) return dflash_noalloc_fail(DFLASH_ERR_ARG, "rows must be >= 0");
  if (rows == 0) return DFLASH_OK;
  if (x == nullptr || y == nullptr) return dflash_noalloc_fail(DFLASH_ERR_ARG, "null tensor");
  const bool bf = a->dt == DFLASH_BF16;
  if (bf && (((uintptr_t)x | (uintptr_t)y) & 15) != 0)
    return dflash_noalloc_fail(DFLASH_ERR_ARG, "bf16 tensors must be 16-byte aligned");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != a->device)
    return dflash_noalloc_fail(DFLASH_ERR_ARG,
                               "the layer's device must be the current device");
  if (dev < 0 || dev >= kMaxDevices)
    return dflash_noalloc_fail(DFLASH_ERR_UNSUPPORTED, "device index above 63");

  // carve [z | partial tiles | counters] out of the fixed array
  const int K = a->nL * a->H;
  const size_t z_bytes = round256((size_t)rows * a->H * sizeof(float));
  size_t part_bytes = 0;
  int n_counters = 0;
  if (bf)
    part_bytes = round256(df::gemm_scratch_bytes(df::EPI_F32, rows, 0, a->H, K, 0, a->num_sms,
                                                 &n_counters));
  const size_t cnt_bytes = round256((size_t)std::max(n_counters, 1) * sizeof(int));
  const size_t need = z_bytes + part_bytes + cnt_bytes;
  if (need > kScratchBytes) {
    char buf[256];
    snprintf(buf, sizeof(buf),
             "ctx_project_noalloc: %d rows need %zu bytes of scratch, above the fixed "
             "%zu-byte limit; use fewer rows per call",
             rows, need, kScratchBytes);
    return dflash_noalloc_fail(DFLASH_ERR_CAPACITY, buf);
  }
  void* base = nullptr;
  cudaError_t e = scratch_address(dev, &base);
  if (e != cudaSuccess)
    return dflash_noalloc_fail(DFLASH_ERR_CUDA, cudaGetErrorString(e));
  char* p = static_cast<char*>(base);
  float* z = reinterpret_cast<float*>(p);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (bf) {
    df::GemmScratch scr;
    scr.partial = reinterpret_cast<float*>(p + z_bytes);
    scr.partial_bytes = part_bytes;
    scr.counters = reinterpret_cast<int*>(p + z_bytes + part_bytes);
    scr.n_counters = n_counters;
    // the split-K counters must start at zero; the array keeps whatever the
    // previous call left, so clear them on this stream first
    e = cudaMemsetAsync(scr.counters, 0, cnt_bytes, s);
    if (e == cudaSuccess) {
      df::GemmShape gs{x, rows, nullptr, 0, &a->tm_fc, &a->tm_fc256, a->H, K, 0};
      e = (cudaError_t)df::launch_gemm_bf16(gs, df::EPI_F32, z, a->H, nullptr, nullptr, scr,
                                            a->num_sms, a->err, s);
    }
  } else {
    e = (cudaError_t)df::launch_gemm_f32(static_cast<const float*>(x), rows,
                                         static_cast<const float*>(a->w_fc), a->H, K, z,
                                         a->H, s);
  }
  if (e == cudaSuccess)
    e = (cudaError_t)df::launch_row_rmsnorm(z, rows, a->H, a->hidden_norm, a->cfg.rms_eps,
                                            y, bf, 1, 0, s);
  if (e != cudaSuccess) return dflash_noalloc_fail(DFLASH_ERR_CUDA, cudaGetErrorString(e));
  return DFLASH_OK;
}
