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

// out[r] = w * z[r] / sqrt(mean(z[r]^2) + eps), one CTA per row
__global__ void row_rmsnorm_kernel(const float* z, int cols, const float* w,
                                   float eps, void* out, int out_bf16) {
  const float* zr = z + (size_t)blockIdx.x * cols;
  float ss = 0.f;
  for (int c = threadIdx.x; c < cols; c += blockDim.x) ss = fmaf(zr[c], zr[c], ss);
  __shared__ float red[32];
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / cols + eps);
  for (int c = threadIdx.x; c < cols; c += blockDim.x) {
    const float y = zr[c] * inv * w[c];
    if (out_bf16)
      reinterpret_cast<__nv_bfloat16*>(out)[(size_t)blockIdx.x * cols + c] =
          __float2bfloat16_rn(y);
    else
      reinterpret_cast<float*>(out)[(size_t)blockIdx.x * cols + c] = y;
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
    rope_table_kernel<<<1024, 256, 0, st>>>(tab, max_pos, half, d_f);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaFree(d_f);
  return e;
}

int launch_row_rmsnorm(const float* z, int rows, int cols, const float* w,
                       float eps, void* out, int out_bf16, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  row_rmsnorm_kernel<<<rows, 256, 0, st>>>(z, cols, w, eps, out, out_bf16);
  return cudaGetLastError();
}

int launch_to_f32(const void* src, int src_bf16, float* dst, size_t n,
                  cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  to_f32_kernel<<<(unsigned)std::min<size_t>((n + 255) / 256, 4096), 256, 0, st>>>(
      src, src_bf16, dst, n);
  return cudaGetLastError();
}

int launch_packed_positions(const int* anchors, int batch, int seq, int n_blocks,
                            int block_size, int* pos, int* err, cudaStream_t st) {
  const int per = seq + n_blocks * block_size;
  dim3 grid((per + 255) / 256, batch);
  packed_positions_kernel<<<grid, 256, 0, st>>>(anchors, seq, n_blocks, block_size,
                                                pos, err);
  return cudaGetLastError();
}

}  // namespace df
