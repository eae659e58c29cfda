// misc.cu -- small kernels around the projections and the attention.
#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

// (cos, sin) of p * f_j for every position p < max_pos, j < half.  The
// frequencies arrive as fp32 values ("nemo_automodel...draft_qwen3",
// Qwen3DFlashDraftModel._apply: inv_freq stays fp32); the angle and its sine
// and cosine are evaluated in double and stored as float.
__global__ void rope_table_kernel(float2* tab, int max_pos, int half,
                                  const float* freqs) {
  const size_t n = (size_t)max_pos * half;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int p = (int)(i / half), j = (int)(i % half);
    double s, c;
    sincos((double)p * (double)freqs[j], &s, &c);
    tab[i] = make_float2((float)c, (float)s);
  }
}

// out[r] = w * x / sqrt(mean(x^2) + eps) with x = z[r] summed over the
// slices in slice order (the K splits of the fc projection): one CTA per
// row, the row held in registers (up to kNormVec float4 per thread), one
// reduction.
constexpr int kNormThreads = 512;
constexpr int kNormVec = 8;  // cols <= 512 * 4 * 8 = 16384
constexpr int kNormMaxSlices = 8;

// VEC float4 per thread and at most MAXS slices: the smallest instance that
// covers the call, so that the registers of a thread (the row's values, the
// slices' loads in flight, the gains) let two CTAs share an SM
template <int VEC, int MAXS>
__global__ void __launch_bounds__(kNormThreads)
    row_rmsnorm_kernel(const float* z, int cols, const float* w, float eps, void* out,
                       int out_bf16, int n_slices, size_t slice_stride) {
  const int n4 = cols / 4;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  // the gains do not depend on the previous kernel: read before its wait
  const float4* w4 = reinterpret_cast<const float4*>(w);
  float4 gv[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const int c = threadIdx.x + i * kNormThreads;
    gv[i] = c < n4 ? __ldg(w4 + c) : zero;
  }
  grid_dep_sync();
  const float4* zr = reinterpret_cast<const float4*>(z + (size_t)blockIdx.x * cols);
  float4 x[VEC];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const int c = threadIdx.x + i * kNormThreads;
    // every slice's load issued before the first is used; summed in order
    float4 t[MAXS];
#pragma unroll
    for (int sl = 0; sl < MAXS; ++sl)
      t[sl] = c < n4 && sl < n_slices ? __ldcg(zr + sl * (slice_stride / 4) + c) : zero;
    x[i] = t[0];
#pragma unroll
    for (int sl = 1; sl < MAXS; ++sl) {
      if (sl < n_slices) {
        x[i].x += t[sl].x;
        x[i].y += t[sl].y;
        x[i].z += t[sl].z;
        x[i].w += t[sl].w;
      }
    }
    ss += x[i].x * x[i].x + x[i].y * x[i].y + x[i].z * x[i].z + x[i].w * x[i].w;
  }
  __shared__ float red[kNormThreads / 32];
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += red[i];
  const float inv = rsqrtf(tot / cols + eps);
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const int c = threadIdx.x + i * kNormThreads;
    if (c >= n4) break;
    const float4 g = gv[i];
    const float4 y = make_float4(x[i].x * inv * g.x, x[i].y * inv * g.y,
                                 x[i].z * inv * g.z, x[i].w * inv * g.w);
    if (out_bf16) {
      uint2 pk;
      pk.x = pack_bf16x2(y.x, y.y);
      pk.y = pack_bf16x2(y.z, y.w);
      reinterpret_cast<uint2*>(out)[(size_t)blockIdx.x * n4 + c] = pk;
    } else {
      reinterpret_cast<float4*>(out)[(size_t)blockIdx.x * n4 + c] = y;
    }
  }
}

// Residual add + RMSNorm of a decoder layer, one CTA per row: r = a (+ b)
// in fp32, stored bf16 (the residual stream; sum_out may alias a or b: each
// element is read before it is written, by the same thread), and
// w * r / sqrt(mean(r^2) + eps) of the fp32 r, stored bf16.  Each thread
// holds up to kAddNormVec groups of 8 columns.
constexpr int kAddNormThreads = 256;
constexpr int kAddNormVec = 4;  // cols <= 256 * 8 * 4 = 8192

__global__ void __launch_bounds__(kAddNormThreads)
    add_rmsnorm_kernel(const uint4* a, const uint4* b, int cols,
                       const float* __restrict__ w, float eps, uint4* sum_out,
                       uint4* __restrict__ norm_out) {
  grid_dep_sync();
  const int n8 = cols / 8;
  const size_t row = (size_t)blockIdx.x * n8;
  float x[kAddNormVec][8];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kAddNormVec; ++i) {
    const int c = threadIdx.x + i * kAddNormThreads;
    if (c < n8) {
      uint4 va = a[row + c];
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&va);
      float f[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        f[2 * e] = __low2float(pa[e]);
        f[2 * e + 1] = __high2float(pa[e]);
      }
      if (b != nullptr) {
        uint4 vb = b[row + c];
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&vb);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          f[2 * e] += __low2float(pb[e]);
          f[2 * e + 1] += __high2float(pb[e]);
        }
      }
      // the residual stream is stored in bf16; the norm takes the fp32 sum
      // (one rounding fewer on the path into the projections)
      uint4 vr;
      uint32_t* pr = reinterpret_cast<uint32_t*>(&vr);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pr[e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
        x[i][2 * e] = f[2 * e];
        x[i][2 * e + 1] = f[2 * e + 1];
        ss += x[i][2 * e] * x[i][2 * e] + x[i][2 * e + 1] * x[i][2 * e + 1];
      }
      sum_out[row + c] = vr;
    }
  }
  __shared__ float red[kAddNormThreads / 32];
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kAddNormThreads / 32; ++i) tot += red[i];
  const float inv = rsqrtf(tot / cols + eps);
#pragma unroll
  for (int i = 0; i < kAddNormVec; ++i) {
    const int c = threadIdx.x + i * kAddNormThreads;
    if (c >= n8) break;
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(w) + 2 * c);
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(w) + 2 * c + 1);
    uint4 vo;
    vo.x = pack_bf16x2(x[i][0] * inv * g0.x, x[i][1] * inv * g0.y);
    vo.y = pack_bf16x2(x[i][2] * inv * g0.z, x[i][3] * inv * g0.w);
    vo.z = pack_bf16x2(x[i][4] * inv * g1.x, x[i][5] * inv * g1.y);
    vo.w = pack_bf16x2(x[i][6] * inv * g1.z, x[i][7] * inv * g1.w);
    norm_out[row + c] = vo;
  }
}

__global__ void to_f32_kernel(const void* src, int src_bf16, float* dst, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(src)[i])
                      : reinterpret_cast<const float*>(src)[i];
}

// positions of the packed training layout: context row j at j, row t of
// block k at anchors[k] + t (anchors outside [0, seq] are clamped and
// reported)
__global__ void packed_positions_kernel(const int* anchors, int seq, int n_blocks,
                                        int block_size, int* pos, int* err) {
  const int b = blockIdx.y;
  const int per = seq + n_blocks * block_size;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < per;
       i += gridDim.x * blockDim.x) {
    int v;
    if (i < seq) {
      v = i;
    } else {
      const int k = (i - seq) / block_size, t = (i - seq) % block_size;
      int a = anchors[b * n_blocks + k];
      if (a < 0 || a > seq) {
        record_error(err, 3 /* DFLASH_DEV_ANCHOR */);
        a = min(max(a, 0), seq);
      }
      v = a + t;
    }
    pos[(size_t)b * per + i] = v;
  }
}

// Check of the bounded pipeline wait: one thread waits on an mbarrier with
// the same wait routine every kernel uses, for at most limit_ns.  With
// `arrive` set, the barrier's one expected arrival is made first and the wait
// returns at once; without it nothing ever arrives, so the wait runs out,
// records DFLASH_DEV_WAIT_TIMEOUT in `err` and the kernel returns normally.
__global__ void wait_probe_kernel(int* err, unsigned long long limit_ns, int arrive) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (arrive) mbar_arrive(&bar);
    mbar_wait_for(&bar, 0, &abort_flag, err, limit_ns);
  }
  __syncthreads();
}


// Read-stream probe: streams a rows x cols bf16 row-major matrix once through
// TMA in the boxes the GEMMs read their weights in (128 rows x 64 columns,
// 128-byte swizzle).  Box b is (row block b / (cols / 64), column block
// b % (cols / 64)); CTA c takes boxes [c * total / G, (c + 1) * total / G)
// and keeps `stages` of them in flight, reusing a slot as soon as its box has
// landed.  The data is discarded: the kernel measures how fast TMA alone
// moves the bytes.
constexpr int kProbeBox = 128 * 64 * 2;
constexpr int kProbeMaxStages = 12;

__global__ void __launch_bounds__(32, 1)
    read_stream_kernel(const __grid_constant__ CUtensorMap tm, int n_row_blocks, int n_col_blocks,
                       int stages, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)stages * kProbeBox);
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  const long long total = (long long)n_row_blocks * n_col_blocks;
  const long long b0 = (long long)blockIdx.x * total / gridDim.x;
  const int n = (int)((long long)(blockIdx.x + 1) * total / gridDim.x - b0);
  abort_flag = 0;
  for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
  fence_mbar_init();
  const uint64_t pol = policy_evict_first();
  for (int i = 0; i < n; ++i) {
    const int s = i % stages;
    // slot s is free once its previous box (i - stages) has landed
    if (i >= stages && !mbar_wait(&full[s], ((i / stages) - 1) & 1, &abort_flag, err)) return;
    mbar_arrive_expect_tx(&full[s], kProbeBox);
    const long long b = b0 + i;
    tma_load_2d(smem + (size_t)s * kProbeBox, &tm, &full[s], (int)(b % n_col_blocks) * 64,
                (int)(b / n_col_blocks) * 128, pol);
  }
  for (int i = n > stages ? n - stages : 0; i < n; ++i)
    if (!mbar_wait(&full[i % stages], (i / stages) & 1, &abort_flag, err)) return;
}
}  // namespace

int launch_rope_table(float2* tab, int max_pos, int half, float theta,
                      cudaStream_t st) {
  // fp32 frequencies: the float nearest theta^(-2j/d)
  float h_f[256];
  if (half > 256) return cudaErrorInvalidValue;
  for (int j = 0; j < half; ++j)
    h_f[j] = (float)pow((double)theta, -2.0 * j / (2.0 * half));
  float* d_f = nullptr;
  cudaError_t e = cudaMalloc(&d_f, half * sizeof(float));
  if (e != cudaSuccess) return e;
  e = cudaMemcpy(d_f, h_f, half * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    count_launch();
    rope_table_kernel<<<1024, 256, 0, st>>>(tab, max_pos, half, d_f);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaFree(d_f);
  return e;
}

int launch_row_rmsnorm(const float* z, int rows, int cols, const float* w,
                       float eps, void* out, int out_bf16, int n_slices,
                       size_t slice_stride, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (cols % 4 != 0 || cols > kNormThreads * 4 * kNormVec || n_slices < 1 ||
      n_slices > kNormMaxSlices || (n_slices > 1 && slice_stride % 4 != 0))
    return cudaErrorInvalidValue;
  const int per = (cols / 4 + kNormThreads - 1) / kNormThreads;  // float4 per thread
  auto go = [&](auto kernel) {
    return launch_pdl(kernel, dim3(rows), dim3(kNormThreads), 0, st, z, cols, w, eps, out,
                      out_bf16, n_slices, slice_stride);
  };
  const bool few = n_slices <= 4;
  if (per <= 1) return few ? go(row_rmsnorm_kernel<1, 4>) : go(row_rmsnorm_kernel<1, 8>);
  if (per <= 2) return few ? go(row_rmsnorm_kernel<2, 4>) : go(row_rmsnorm_kernel<2, 8>);
  if (per <= 4) return few ? go(row_rmsnorm_kernel<4, 4>) : go(row_rmsnorm_kernel<4, 8>);
  return few ? go(row_rmsnorm_kernel<8, 4>) : go(row_rmsnorm_kernel<8, 8>);
}

int launch_add_rmsnorm(const void* a, const void* b, int rows, int cols, const float* w,
                       float eps, void* sum_out, void* norm_out, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (cols % 8 != 0 || cols > kAddNormThreads * 8 * kAddNormVec) return cudaErrorInvalidValue;
  return launch_pdl(add_rmsnorm_kernel, dim3(rows), dim3(kAddNormThreads), 0, st,
                    static_cast<const uint4*>(a), static_cast<const uint4*>(b), cols, w, eps,
                    static_cast<uint4*>(sum_out), static_cast<uint4*>(norm_out));
}

int launch_to_f32(const void* src, int src_bf16, float* dst, size_t n,
                  cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  count_launch();
  to_f32_kernel<<<(unsigned)std::min<size_t>((n + 255) / 256, 4096), 256, 0, st>>>(
      src, src_bf16, dst, n);
  return cudaGetLastError();
}

int launch_packed_positions(const int* anchors, int batch, int seq, int n_blocks,
                            int block_size, int* pos, int* err, cudaStream_t st) {
  const int per = seq + n_blocks * block_size;
  dim3 grid((per + 255) / 256, batch);
  count_launch();
  packed_positions_kernel<<<grid, 256, 0, st>>>(anchors, seq, n_blocks, block_size,
                                                pos, err);
  return cudaGetLastError();
}

int launch_wait_probe(int* err, unsigned long long limit_ns, int arrive, cudaStream_t st) {
  count_launch();
  wait_probe_kernel<<<1, 32, 0, st>>>(err, limit_ns, arrive);
  return cudaGetLastError();
}


int launch_read_stream(const void* src, long long rows, long long cols, int ctas, int stages,
                       int* err, cudaStream_t st) {
  if (rows <= 0 || cols <= 0 || rows % 128 != 0 || cols % 64 != 0 || cols > (1 << 30) ||
      rows / 128 > (1 << 30) || stages < 1 || stages > kProbeMaxStages || ctas < 1)
    return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> attr_done{0};
  if (!done_on_device(attr_done)) {
    cudaFuncSetAttribute(read_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kProbeMaxStages * kProbeBox + 2048);
    mark_device(attr_done);
  }
  CUtensorMap tm;
  if (make_tmap_bf16_rows(&tm, src, rows, cols, 128) != 0) return cudaErrorInvalidValue;
  count_launch();
  read_stream_kernel<<<ctas, 32, (size_t)stages * kProbeBox + 2048, st>>>(
      tm, (int)(rows / 128), (int)(cols / 64), stages, err);
  return cudaGetLastError();
}
}  // namespace df
