// handles.h -- definitions of the opaque C-ABI handles, shared by the files
// that implement entry points.
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "../../include/dflash_attn.h"
#include "internal.h"

namespace df {

// device buffer that only grows
struct Buf {
  void* p = nullptr;
  size_t bytes = 0;
  cudaError_t ensure(size_t need, bool zero = false) {
    if (need <= bytes) return cudaSuccess;
    if (p) {
      cudaDeviceSynchronize();
      cudaFree(p);
      p = nullptr;
      bytes = 0;
    }
    need = (need + 255) & ~size_t(255);
    cudaError_t e = cudaMalloc(&p, need);
    if (e != cudaSuccess) return e;
    bytes = need;
    if (zero) {
      // the memset runs on the legacy default stream, which a non-blocking
      // caller stream does not wait for: finish it before any launch
      e = cudaMemset(p, 0, need);
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
    }
    return e;
  }
  void release() {
    if (p) cudaFree(p);
    p = nullptr;
    bytes = 0;
  }
};

}  // namespace df

struct dflash_attn {
  dflash_attn_config cfg;
  int device = 0, num_sms = 0;
  int H = 0, d = 0, nq = 0, nkv = 0, g = 0, nL = 0, max_pos = 0, dt = 0;
  void* w_qkv = nullptr;  // [(nq + 2 nkv) d, H]
  void* w_o = nullptr;    // [H, nq d]
  void* w_fc = nullptr;   // [H, nL H]
  float* q_norm = nullptr;
  float* k_norm = nullptr;
  float* hidden_norm = nullptr;
  float2* rope = nullptr;
  int* err = nullptr;
  CUtensorMap tm_qkv, tm_o, tm_fc, tm_qkv256, tm_o256, tm_fc256;
  // launch trace
  bool trace = false;
  struct Rec { int kind; cudaEvent_t e0, e1; };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> event_pool;
  // scratch
  df::Buf qbuf, attn_out, gemm_partial, gemm_counters, part_o, part_ml, attn_counters,
      zbuf, proj_noise, proj_ctx, packed_k, packed_v, packed_pos, bwd_do, bwd_stats;
};

// Context K/V of several layers from one projection: the layers' K and V
// weights stacked as [layer][K rows | V rows][H] bf16.
struct dflash_kv_group {
  int n_layers = 0, device = 0, num_sms = 0;
  dflash_attn* layers[df::kMaxGroupLayers] = {};
  void* w_kv = nullptr;
  CUtensorMap tm, tm256;
  df::Buf gemm_partial, gemm_counters;
};

// The rest of a draft decoder layer: norms and the Qwen3 MLP.  gate and up
// rows interleaved in 64-row chunks ([g 0..63][u 0..63][g 64..127]...), so
// one 128-row weight tile feeds 64 SwiGLU outputs.
struct dflash_mlp {
  int H = 0, I = 0, device = 0, num_sms = 0;
  float eps = 0.f;
  void* w_gu = nullptr;  // [2I][H] bf16
  void* w_d = nullptr;   // [H][I] bf16
  float* in_norm = nullptr;
  float* post_norm = nullptr;
  CUtensorMap tm_gu, tm_gu256, tm_d, tm_d256;
  df::Buf y, attn_out, act, gemm_partial, gemm_counters;
};

struct dflash_cache {
  int batch = 0, cap = 0, nkv = 0, d = 0, dt = 0, device = 0;
  void* k = nullptr;
  void* v = nullptr;
  std::vector<int> len;
};

// Paged draft KV cache: pages of page_size rows, K and V each
// [n_pages][nkv][page_size][d] bf16; lengths, slots and block tables belong
// to the caller.
struct dflash_paged_cache {
  int n_pages = 0, page_size = 0, nkv = 0, d = 0, dt = 0, device = 0;
  void* k = nullptr;
  void* v = nullptr;
};
