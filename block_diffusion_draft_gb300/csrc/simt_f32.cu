// simt_f32.cu -- the fp32 path of the layer on CUDA cores.
//
// Layers created with DFLASH_FP32 keep fp32 weights, activations and cache
// and run these plain kernels: a tiled SIMT GEMM, a per-(row, head) norm +
// RoPE + scatter kernel, and a warp-per-query-row attention.  They serve the
// small fp32 configurations where the tolerance is tighter than bf16 allows;
// the production path is the bf16 tcgen05 one.
#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

constexpr int TS = 16;

// C[rows, n] = A[rows, k] * B[n, k]^T
__global__ void gemm_f32_kernel(const float* a, int rows, const float* b, int n,
                                int k, float* c, int ldc) {
  __shared__ float as[TS][TS + 1];
  __shared__ float bs[TS][TS + 1];
  const int r = blockIdx.y * TS + threadIdx.y;
  const int col = blockIdx.x * TS + threadIdx.x;
  float acc = 0.f;
  for (int k0 = 0; k0 < k; k0 += TS) {
    const int ka = k0 + threadIdx.x;
    as[threadIdx.y][threadIdx.x] = (r < rows && ka < k) ? a[(size_t)r * k + ka] : 0.f;
    const int bn = blockIdx.x * TS + threadIdx.y;
    bs[threadIdx.y][threadIdx.x] = (bn < n && ka < k) ? b[(size_t)bn * k + ka] : 0.f;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < TS; ++i) acc = fmaf(as[threadIdx.y][i], bs[threadIdx.x][i], acc);
    __syncthreads();
  }
  if (r < rows && col < n) c[(size_t)r * ldc + col] = acc;
}

// one CTA per (row, head slot); slots: n_heads Q heads, n_kv K heads,
// n_kv V heads for noise rows, n_kv K + n_kv V heads for context rows
__global__ void qkv_post_f32_kernel(const float* qkv_noise, int rows_noise,
                                    const float* kv_ctx, const QkvOut o,
                                    const SeqTable st, int d, int* err) {
  const int row = blockIdx.x;
  const int slot = blockIdx.y;
  const bool noise = row < rows_noise;
  const int nq = o.n_heads, nkv = o.n_kv;
  int kind, h;  // 0 = Q, 1 = K, 2 = V
  const float* src;
  int grow, b, t = 0, pos_idx, crow;
  if (noise) {
    if (slot < nq) { kind = 0; h = slot; }
    else if (slot < nq + nkv) { kind = 1; h = slot - nq; }
    else { kind = 2; h = slot - nq - nkv; }
    grow = row;
    src = qkv_noise + (size_t)grow * (nq + 2 * nkv) * d + (size_t)slot * d;
    b = grow / st.q_len;
    t = grow - b * st.q_len;
    const int nb = st.ctx_off[b + 1] - st.ctx_off[b];
    pos_idx = st.ctx_off[b + 1] + b * st.q_len + t;
    crow = st.cache_len[b] + nb + t;
  } else {
    if (slot >= 2 * nkv) return;
    kind = slot < nkv ? 1 : 2;
    h = slot < nkv ? slot : slot - nkv;
    grow = row - rows_noise;
    src = kv_ctx + (size_t)grow * 2 * nkv * d + (size_t)slot * d;
    int lo = 0, hi = st.n;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (st.ctx_off[mid] <= grow) lo = mid; else hi = mid;
    }
    b = lo;
    const int rr = grow - st.ctx_off[b];
    pos_idx = st.ctx_off[b] + b * st.q_len + rr;
    crow = st.cache_len[b] + rr;
  }
  extern __shared__ float xs[];
  __shared__ float red[32];
  const int half = d / 2;
  for (int j = threadIdx.x; j < d; j += blockDim.x) xs[j] = src[j];
  __syncthreads();
  float* dst;
  if (kind == 2) {
    dst = reinterpret_cast<float*>(o.cache_v) + (((size_t)b * nkv + h) * o.cap + crow) * d;
    for (int j = threadIdx.x; j < d; j += blockDim.x) dst[j] = xs[j];
    return;
  }
  float ss = 0.f;
  for (int j = threadIdx.x; j < d; j += blockDim.x) ss = fmaf(xs[j], xs[j], ss);
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
  const float inv = rsqrtf(tot / d + o.eps);
  const float* w = kind == 0 ? o.q_norm : o.k_norm;
  int pos = o.positions[pos_idx];
  if (pos < 0 || pos >= o.max_pos) {
    if (threadIdx.x == 0) record_error(err, 2 /* DFLASH_DEV_POSITION */);
    pos = 0;
  }
  const float2* rr = o.rope + (size_t)pos * half;
  const float scale = kind == 0 ? o.q_scale : 1.f;
  if (kind == 0) {
    const int hh = h / o.groups, gi = h - hh * o.groups;
    const int nblk = st.q_len / o.q_block;
    const int blk = t / o.q_block, tt = t - blk * o.q_block;
    const size_t qrow =
        ((((size_t)b * nkv + hh) * nblk + blk) * o.groups + gi) * o.q_block + tt;
    dst = reinterpret_cast<float*>(o.qbuf) + qrow * d;
  } else {
    dst = reinterpret_cast<float*>(o.cache_k) + (((size_t)b * nkv + h) * o.cap + crow) * d;
  }
  for (int j = threadIdx.x; j < half; j += blockDim.x) {
    const float x1 = xs[j] * inv * w[j];
    const float x2 = xs[j + half] * inv * w[j + half];
    const float2 cs = rr[j];
    dst[j] = (x1 * cs.x - x2 * cs.y) * scale;
    dst[j + half] = (x2 * cs.x + x1 * cs.y) * scale;
  }
}

// one warp per (sequence, query head, query row): online softmax over the
// allowed keys, one key at a time, lanes split head_dim
__global__ void attn_f32_kernel(const AttnArgs a, const AttnSeqs sq,
                                const float* qbuf, const float* kst,
                                const float* vst) {
  const int warps = blockDim.x >> 5;
  const int gw = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int nq = a.n_kv * a.groups;
  const int total = a.batch * nq * a.q_len;
  if (gw >= total) return;
  const int d = a.head_dim;
  const int b = gw / (nq * a.q_len);
  const int rem = gw - b * nq * a.q_len;
  const int hq = rem / a.q_len;
  const int tg = rem - hq * a.q_len;  // row within the sequence's queries
  const int h = hq / a.groups, gi = hq - h * a.groups;
  const int blk = tg / a.q_block, t = tg - blk * a.q_block;
  const size_t qrow =
      ((((size_t)b * a.n_kv + h) * a.n_blocks + blk) * a.groups + gi) * a.q_block + t;
  const float* qv = qbuf + qrow * d;
  int lo1, hi1, lo2 = 0, hi2 = 0;
  if (a.mode == 0) {
    const int len = sq.len[b];
    lo1 = 0;
    hi1 = len;
    const int qi = len - a.q_len + tg;  // the row's own key index
    if (a.window > 0) {
      lo1 = max(0, qi - a.window + 1);
      hi1 = min(len, qi + a.window);
    }
    if (a.causal) hi1 = min(hi1, qi + 1);
  } else {
    int an = a.anchors[b * a.n_blocks + blk];
    if (an < 0 || an > a.seq) {
      if (lane == 0) record_error(a.err, 3 /* DFLASH_DEV_ANCHOR */);
      an = min(max(an, 0), a.seq);
    }
    lo1 = 0;
    hi1 = an;
    lo2 = a.seq + blk * a.q_block;
    hi2 = lo2 + a.q_block;
  }
  const float* kb = kst + ((size_t)b * a.n_kv + h) * a.cap * d;
  const float* vb = vst + ((size_t)b * a.n_kv + h) * a.cap * d;
  constexpr int MAXD = 8;  // head_dim <= 256
  float acc[MAXD];
  float ql[MAXD];
#pragma unroll
  for (int i = 0; i < MAXD; ++i) {
    acc[i] = 0.f;
    const int e = lane + 32 * i;
    ql[i] = e < d ? qv[e] : 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int seg = 0; seg < 2; ++seg) {
    const int klo = seg == 0 ? lo1 : lo2, khi = seg == 0 ? hi1 : hi2;
    for (int key = klo; key < khi; ++key) {
      const float* kr = kb + (size_t)key * d;
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < MAXD; ++i) {
        const int e = lane + 32 * i;
        if (e < d) s = fmaf(ql[i], kr[e], s);
      }
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      const float mn = fmaxf(m, s);
      const float alpha = expf(m - mn);
      const float p = expf(s - mn);
      l = l * alpha + p;
      const float* vr = vb + (size_t)key * d;
#pragma unroll
      for (int i = 0; i < MAXD; ++i) {
        const int e = lane + 32 * i;
        acc[i] = acc[i] * alpha + (e < d ? p * vr[e] : 0.f);
      }
      m = mn;
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float* out = reinterpret_cast<float*>(a.out) +
               ((size_t)b * a.q_len + tg) * (size_t)nq * d + (size_t)hq * d;
#pragma unroll
  for (int i = 0; i < MAXD; ++i) {
    const int e = lane + 32 * i;
    if (e < d) out[e] = acc[i] * inv;
  }
}

}  // namespace

int launch_gemm_f32(const float* a, int rows, const float* b, int n, int k,
                    float* c, int ldc, cudaStream_t st) {
  if (rows <= 0 || n <= 0) return cudaSuccess;
  dim3 grid((n + TS - 1) / TS, (rows + TS - 1) / TS), block(TS, TS);
  count_launch();
  gemm_f32_kernel<<<grid, block, 0, st>>>(a, rows, b, n, k, c, ldc);
  return cudaGetLastError();
}

int launch_qkv_post_f32(const float* qkv_noise, int rows_noise, const float* kv_ctx,
                        int rows_ctx, const QkvOut& o, const SeqTable* seqs,
                        int head_dim, int* err, cudaStream_t st) {
  const int rows = rows_noise + rows_ctx;
  if (rows <= 0) return cudaSuccess;
  dim3 grid(rows, o.n_heads + 2 * o.n_kv);
  count_launch();
  qkv_post_f32_kernel<<<grid, 128, head_dim * sizeof(float), st>>>(
      qkv_noise, rows_noise, kv_ctx, o, *seqs, head_dim, err);
  return cudaGetLastError();
}

int launch_attn_f32(const AttnArgs& a, const AttnSeqs* seqs, const float* qbuf,
                    const float* k, const float* v, cudaStream_t st) {
  if (a.head_dim > 256) return cudaErrorInvalidValue;
  const int total = a.batch * a.n_kv * a.groups * a.q_len;
  if (total == 0) return cudaSuccess;
  static AttnSeqs zero_seqs{};
  count_launch();
  attn_f32_kernel<<<(total + 3) / 4, 128, 0, st>>>(a, seqs ? *seqs : zero_seqs, qbuf,
                                                  k, v);
  return cudaGetLastError();
}

}  // namespace df
