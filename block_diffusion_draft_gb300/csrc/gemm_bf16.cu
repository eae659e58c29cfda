// gemm_bf16.cu -- tcgen05 projection GEMM for the bf16 path.
//
// C = A * B^T where A holds token rows (bf16, K contiguous) and B the weight
// rows of an nn.Linear (bf16, [N, K]).  One CTA computes one 128 x BN output
// tile over one slice of K:
//   warp 0      TMA producer: A and B boxes of 64 K-columns, 128-byte swizzle,
//               an mbarrier ring of as many stages as shared memory holds
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer (M=128,
//               N=BN, K=16 per instruction), fp32 accumulator in TMEM
//   warps 2..5  epilogue: one accumulator row (token) per thread, read with
//               tcgen05.ld
// Token rows are few in decode-sized calls, so the A box covers only the rows
// that exist (16, 32, 64 ...) and each pipeline stage is mostly weight bytes;
// the MMA still runs M = 128 and rows past the box are don't-care rows that no
// epilogue stores.  When block rows and context rows together fit one tile
// they share it (two boxes into one A stage), so the K/V weights are streamed
// once.  Tiles are 128 columns wide (the QKV epilogue needs whole heads, and
// 16 KB weight boxes keep TMA requests few), and K is split when the tiles
// are too few to fill the GPU; then every CTA writes the valid rows of
// its fp32 partial, and the last CTA of a tile (atomic counter) sums all
// partials in split order (deterministic), spreading the loads over all its
// epilogue threads and staging the sums through shared memory.  It resets the
// counter for the next launch.
// Kernels launch with programmatic stream serialization: the producer starts
// streaming weights (which no kernel writes) before waiting for the previous
// kernel, so the weight fetch overlaps that kernel's tail.
//
// Epilogues:
//   EPI_BF16  plain bf16 store (o_proj)
//   EPI_F32   plain fp32 store (fc, before hidden_norm)
//   EPI_QKV   the fused QKV projection of the draft layer: per-head RMSNorm
//             (q_norm / k_norm), NeoX RoPE at the row's position, Q scaled by
//             head_dim^-0.5*log2(e) into the Q buffer, K and V appended to the
//             draft cache.  ("vllm.model_executor.models.qwen3_dflash",
//             DFlashQwen3Attention.forward: qkv_proj -> split -> per-head
//             RMSNorm -> rotary; "DFlash源码导读（二）", steps 1-4.)
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

constexpr int BM = 128, BK = 64, MAX_STAGES = 32;
constexpr int MAX_SPLITS = 8;               // K splits of the decode-size kernel
constexpr int kThreads = 192;
constexpr uint32_t A_FULL = BM * BK * 2;   // 16 KB: what one MMA reads of A
constexpr size_t SMEM_LIMIT = 232448;      // per-CTA opt-in maximum
constexpr size_t SMEM_FIXED = 1024 + 1024; // alignment slack + barriers
constexpr int HD = 128;                    // head_dim of the bf16 path
constexpr int M_GROUP = 16;                // m-tiles sharing one pass over N

struct Plan {
  int a0_rows, a1_rows, n_m0, n_m1;
  int merged;          // 1: one tile holds A0 rows then A1 rows
  int cluster;         // decode-size kernel: splits merge inside a cluster
  int box0, box1;      // rows of the A0 / A1 boxes
  int n_tiles, n_q_tiles, n_kb, splits;
  int stages;
  uint32_t a_bytes;    // bytes per A stage (all boxes of one stage)
  int units_q;
  int grid;            // persistent kernel: CTAs
  int ldc;
  float* partial;
  int* counters;
  void* c;
  int* err;
  int slices;           // EPI_F32: split `sp` writes its partial to slice sp of c
  size_t slice_stride;  // floats between slices
  int n_tile0;          // decode-size kernel: first n-tile of this launch
};

// Units of one region (M_r m-tiles x N_r n-tiles x splits), ordered by
// groups of M_GROUP m-tiles, then n-tile, then split, then m-tile: CTAs
// running together share weight tiles and a bounded set of activation rows.
DF_DEV void decode_region(int u, int M_r, int N_r, int splits, int& m, int& n,
                          int& split) {
  const int full = M_GROUP * N_r * splits;
  int mb = u / full;
  const int n_mb = (M_r + M_GROUP - 1) / M_GROUP;
  if (mb > n_mb - 1) mb = n_mb - 1;
  const int rem = u - mb * full;
  const int rows = min(M_GROUP, M_r - mb * M_GROUP);
  n = rem / (splits * rows);
  const int r2 = rem - n * splits * rows;
  split = r2 / rows;
  m = mb * M_GROUP + (r2 - split * rows);
}

DF_DEV void decode_unit(const Plan& p, int u, int& m_tile, int& n_tile, int& split) {
  if (u < p.units_q) {
    decode_region(u, p.n_m0, p.n_q_tiles, p.splits, m_tile, n_tile, split);
  } else {
    decode_region(u - p.units_q, p.n_m0 + p.n_m1, p.n_tiles - p.n_q_tiles, p.splits,
                  m_tile, n_tile, split);
    n_tile += p.n_q_tiles;
  }
}

// Decode-size kernel: unit u is split (u % splits) of tile (u / splits), so
// the splits of one tile are consecutive blocks (one cluster); tiles follow
// the grouped order.
DF_DEV void decode_tile_split(const Plan& p, int u, int& m_tile, int& n_tile, int& split) {
  split = u % p.splits;
  const int t = u / p.splits, tq = p.n_q_tiles * p.n_m0;
  int dummy;
  if (t < tq) {
    decode_region(t, p.n_m0, p.n_q_tiles, 1, m_tile, n_tile, dummy);
  } else {
    decode_region(t - tq, p.n_m0 + p.n_m1, p.n_tiles - p.n_q_tiles, 1, m_tile, n_tile, dummy);
    n_tile += p.n_q_tiles;
  }
}

// Which source row accumulator row r of tile m_tile holds: src 0 = A0
// (block rows), 1 = A1 (context rows), -1 = no row.
DF_DEV void row_source(const Plan& p, int m_tile, int r, int& src, int& row) {
  if (p.merged) {
    if (r < p.box0) {
      src = r < p.a0_rows ? 0 : -1;
      row = r;
    } else {
      row = r - p.box0;
      src = row < p.a1_rows ? 1 : -1;
    }
  } else if (m_tile < p.n_m0) {
    row = m_tile * BM + r;
    src = row < p.a0_rows ? 0 : -1;
  } else {
    row = (m_tile - p.n_m0) * BM + r;
    src = row < p.a1_rows ? 1 : -1;
  }
}

DF_DEV void store_bf16(void* dst, const float* v, int n) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (int i = 0; i < n / 8; ++i) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    w.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    w.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    w.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    d4[i] = w;
  }
}

// per-head RMSNorm over the 128 values, then NeoX rotation (pairs j, j+64)
// with the row's (cos, sin) table, then an optional scale
DF_DEV void norm_rope(float* v, const float* w, float eps, const float2* rope_row,
                      float scale) {
  // the sum of squares as 4 interleaved chains (one chain over 128 values is
  // a latency chain of 128 dependent FMAs)
  float ps[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) ps[e] = v[e] * v[e];
#pragma unroll
  for (int j = 4; j < HD; ++j) ps[j & 3] = fmaf(v[j], v[j], ps[j & 3]);
  const float ss = (ps[0] + ps[1]) + (ps[2] + ps[3]);
  const float inv = rsqrtf(ss * (1.f / HD) + eps);
#pragma unroll
  for (int j = 0; j < HD; ++j) v[j] *= inv * __ldg(w + j);
  const float4* r4 = reinterpret_cast<const float4*>(rope_row);
#pragma unroll
  for (int jj = 0; jj < HD / 4; ++jj) {
    const float4 cs = __ldg(r4 + jj);  // cos_j, sin_j, cos_j+1, sin_j+1
    const int j = 2 * jj;
    const float a0 = v[j], b0 = v[j + HD / 2];
    const float a1 = v[j + 1], b1 = v[j + 1 + HD / 2];
    v[j] = (a0 * cs.x - b0 * cs.y) * scale;
    v[j + HD / 2] = (b0 * cs.x + a0 * cs.y) * scale;
    v[j + 1] = (a1 * cs.z - b1 * cs.w) * scale;
    v[j + 1 + HD / 2] = (b1 * cs.z + a1 * cs.w) * scale;
  }
}

// Where one accumulator row of a QKV tile goes.  kind: 0 = nowhere (a
// context row of a query tile: queries exist for block rows only), 1 = Q
// (per-head RMSNorm + RoPE + scale), 2 = K (RMSNorm + RoPE), 3 = V (copy).
struct QkvTarget {
  int kind;
  int pos_idx;             // index into the positions array
  __nv_bfloat16* dst;      // the 128-value bf16 destination row
  const float* norm;       // RMSNorm gains of the row's head (null for V)
};

// RMSNorm gains of the head starting at output column n0 (null for V)
DF_DEV const float* qkv_col_norm(const QkvOut& qo, int n0) {
  const int kv_cols = qo.n_kv * HD;
  if (qo.n_layers > 0) {
    const int l = n0 / (2 * kv_cols);
    return n0 - l * 2 * kv_cols < kv_cols ? qo.g_k_norm[l] : nullptr;
  }
  const int q_cols = qo.n_heads * HD;
  return n0 < q_cols ? qo.q_norm : (n0 < q_cols + kv_cols ? qo.k_norm : nullptr);
}

DF_DEV QkvTarget qkv_target(const QkvOut& qo, const SeqTable& st, int src, int srow,
                            int n0) {
  int b, pos_idx, crow, t = 0;
  if (src == 0 && qo.n_layers == 0) {  // noise (block) row
    b = srow / st.q_len;
    t = srow - b * st.q_len;
    const int nb = st.ctx_off[b + 1] - st.ctx_off[b];
    pos_idx = st.ctx_off[b + 1] + b * st.q_len + t;
    crow = st.cache_len[b] + nb + t;
  } else {  // new context row: find its sequence
    int lo = 0, hi = st.n;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (st.ctx_off[mid] <= srow) lo = mid; else hi = mid;
    }
    b = lo;
    const int rr = srow - st.ctx_off[b];
    pos_idx = st.ctx_off[b] + b * st.q_len + rr;
    crow = st.cache_len[b] + rr;
  }
  const int q_cols = qo.n_heads * HD, kv_cols = qo.n_kv * HD;
  QkvTarget g;
  g.pos_idx = pos_idx;
  g.norm = qkv_col_norm(qo, n0);
  if (qo.n_layers > 0) {
    // layer group: column n0 is K or V head h of layer l
    const int l = n0 / (2 * kv_cols);
    const int c = n0 - l * 2 * kv_cols;
    const bool is_k = c < kv_cols;
    const int h = (is_k ? c : c - kv_cols) / HD;
    g.kind = is_k ? 2 : 3;
    g.dst = reinterpret_cast<__nv_bfloat16*>(is_k ? qo.g_cache_k[l] : qo.g_cache_v[l]) +
            (((size_t)b * qo.n_kv + h) * qo.g_cap[l] + crow) * HD;
    return g;
  }
  if (n0 < q_cols) {
    if (src != 0) {
      g.kind = 0;
      g.dst = nullptr;
      return g;
    }
    const int hq = n0 / HD;
    const int h = hq / qo.groups, gi = hq - h * qo.groups;
    const int nblk = st.q_len / qo.q_block;
    const int blk = t / qo.q_block, tt = t - blk * qo.q_block;
    const size_t qrow =
        ((((size_t)b * qo.n_kv + h) * nblk + blk) * qo.groups + gi) * qo.q_block + tt;
    g.kind = 1;
    g.dst = reinterpret_cast<__nv_bfloat16*>(qo.qbuf) + qrow * HD;
  } else {
    const bool is_k = n0 < q_cols + kv_cols;
    const int h = (n0 - q_cols - (is_k ? 0 : kv_cols)) / HD;
    size_t row = ((size_t)b * qo.n_kv + h) * qo.cap + crow;
    if (qo.slot_mapping != nullptr) {  // paged cache: the caller's slot for the row
      const int sl = qo.slot_mapping[pos_idx];
      const int page = sl >= 0 ? sl / qo.page_size : -1;
      if (page < 0 || page >= qo.n_pages) {
        record_error(qo.err, 4 /* DFLASH_DEV_SLOT */);
        g.kind = 0;
        g.dst = nullptr;
        return g;
      }
      row = ((size_t)page * qo.n_kv + h) * qo.page_size + (sl - page * qo.page_size);
    }
    g.kind = is_k ? 2 : 3;
    g.dst = reinterpret_cast<__nv_bfloat16*>(is_k ? qo.cache_k : qo.cache_v) + row * HD;
  }
  return g;
}

// the row's rotary position, out-of-range positions reported and read as 0
DF_DEV int checked_position(const QkvOut& qo, int pos_idx, int* err) {
  int pos = qo.positions[pos_idx];
  if (pos < 0 || pos >= qo.max_pos) {
    record_error(err, 2 /* DFLASH_DEV_POSITION */);
    pos = 0;
  }
  return pos;
}

// Final epilogue of one accumulator row held by one thread: `v` holds 128
// columns starting at output column n0 for source row (src, srow).
template <int EPI>
DF_DEV void finish_row(const Plan& p, const QkvOut& qo, const SeqTable& st, float* v,
                       int src, int srow, int n0, size_t c_off = 0) {
  constexpr int BN = HD;
  constexpr int C4 = BN / 4;
  if constexpr (EPI == EPI_SWIGLU) {
    // columns 0..63 gate, 64..127 up of the same 64 outputs
    float act[HD / 2];
#pragma unroll
    for (int c = 0; c < HD / 2; ++c) {
      const float gt = v[c];
      act[c] = gt / (1.f + __expf(-gt)) * v[HD / 2 + c];
    }
    store_bf16(reinterpret_cast<__nv_bfloat16*>(p.c) + (size_t)srow * p.ldc + n0 / 2, act,
               HD / 2);
  } else if constexpr (EPI == EPI_BF16 || EPI == EPI_F32) {
    if constexpr (EPI == EPI_BF16) {
      store_bf16(reinterpret_cast<__nv_bfloat16*>(p.c) + (size_t)srow * p.ldc + n0, v, BN);
    } else {
      float4* d4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.c) + c_off +
                                             (size_t)srow * p.ldc + n0);
#pragma unroll
      for (int c4 = 0; c4 < C4; ++c4)
        d4[c4] = make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
    }
  } else {
    // fused QKV epilogue: one head (128 columns) per tile
    const QkvTarget g = qkv_target(qo, st, src, srow, n0);
    if (g.kind == 0) return;
    if (g.kind != 3) {
      const int pos = checked_position(qo, g.pos_idx, p.err);
      norm_rope(v, g.norm, qo.eps,
                qo.rope + (size_t)pos * (HD / 2), g.kind == 1 ? qo.q_scale : 1.f);
    }
    store_bf16(g.dst, v, HD);
  }
}

// The QKV epilogue of one row held by one thread, with its destination and
// position worked out beforehand (while the main loop ran).
DF_DEV void qkv_apply(const QkvOut& qo, const QkvTarget& g, int pos, float* v) {
  if (g.kind == 0) return;
  if (g.kind != 3)
    norm_rope(v, g.norm, qo.eps, qo.rope + (size_t)pos * (HD / 2),
              g.kind == 1 ? qo.q_scale : 1.f);
  store_bf16(g.dst, v, HD);
}

// The same epilogue for a row still in TMEM (128 accumulator columns at
// `col`, this thread's lane), read twice in 32-column pieces: once for the
// sum of squares, then column pairs (j, j + 64) a piece of each at a time,
// so that few values, gains and (cos, sin) pairs are live at once.  The
// gains `w4` and the row's (cos, sin) pairs `r4` are generic pointers
// (global memory, or copies in shared memory).  Warp-collective (TMEM
// loads): every lane calls it.
DF_DEV void qkv_apply_tmem(const QkvOut& qo, const QkvTarget& g, uint32_t col, const float4* w4,
                           const float4* r4) {
  const bool live = g.kind != 0;
  float inv = 1.f;
  if (__any_sync(0xffffffffu, live && g.kind != 3)) {
    float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      float t[32];
      tmem_ld32(col + c * 32, t);
#pragma unroll
      for (int i = 0; i < 32; ++i) ps[i & 3] = fmaf(t[i], t[i], ps[i & 3]);
    }
    inv = rsqrtf(((ps[0] + ps[1]) + (ps[2] + ps[3])) * (1.f / HD) + qo.eps);
  }
  const bool rot = live && g.kind != 3;
  const float scale = g.kind == 1 ? qo.q_scale : 1.f;
#pragma unroll 1
  for (int c = 0; c < HD / 64; ++c) {  // columns 32c.. and 64 + 32c..
    float a[32], b[32];
    tmem_ld32(col + c * 32, a);
    tmem_ld32(col + HD / 2 + c * 32, b);
    if (!live) continue;
    if (rot) {
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 ga = w4[c * 8 + q4], gb = w4[HD / 8 + c * 8 + q4];
        const float4 cs0 = r4[c * 16 + 2 * q4], cs1 = r4[c * 16 + 2 * q4 + 1];
        const float ga_[4] = {ga.x, ga.y, ga.z, ga.w}, gb_[4] = {gb.x, gb.y, gb.z, gb.w};
        const float co[4] = {cs0.x, cs0.z, cs1.x, cs1.z}, si[4] = {cs0.y, cs0.w, cs1.y, cs1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = 4 * q4 + e;
          const float x = a[i] * (inv * ga_[e]), y = b[i] * (inv * gb_[e]);
          a[i] = (x * co[e] - y * si[e]) * scale;
          b[i] = (y * co[e] + x * si[e]) * scale;
        }
      }
    }
    store_bf16(g.dst + c * 32, a, 32);
    store_bf16(g.dst + HD / 2 + c * 32, b, 32);
  }
}

// The same epilogue with one row spread over a warp: lane l holds columns
// 4l .. 4l+3.  The RMSNorm sum is a butterfly over the warp, and the RoPE
// partner of column j < 64 (column j + 64) sits 16 lanes away.
DF_DEV float4 warp_norm_rope(float4 x, float4 w4, float eps, const float2* rope_row,
                             float scale, int lane) {
  float ss = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss * (1.f / HD) + eps);
  x.x *= inv * w4.x;
  x.y *= inv * w4.y;
  x.z *= inv * w4.z;
  x.w *= inv * w4.w;
  float4 y;
  y.x = __shfl_xor_sync(0xffffffffu, x.x, 16);
  y.y = __shfl_xor_sync(0xffffffffu, x.y, 16);
  y.z = __shfl_xor_sync(0xffffffffu, x.z, 16);
  y.w = __shfl_xor_sync(0xffffffffu, x.w, 16);
  // (cos, sin) of pairs 4(l % 16) .. 4(l % 16) + 3
  const float4* r4 = reinterpret_cast<const float4*>(rope_row) + 2 * (lane & 15);
  const float4 c0 = __ldg(r4), c1 = __ldg(r4 + 1);
  // first half: a' = a cos - b sin; second half: b' = b cos + a sin
  const float sg = lane < 16 ? -1.f : 1.f;
  float4 o;
  o.x = (x.x * c0.x + sg * y.x * c0.y) * scale;
  o.y = (x.y * c0.z + sg * y.y * c0.w) * scale;
  o.z = (x.z * c1.x + sg * y.z * c1.y) * scale;
  o.w = (x.w * c1.z + sg * y.w * c1.w) * scale;
  return o;
}

// Warp wq of the decode-size kernel's QKV epilogue finishes rows wq, wq + 4,
// wq + 8 ... of the tile, four at a time so that their loads overlap.  A row
// is read from the shared-memory tile (one split) or summed over the splits'
// global partials in split order.  Lane l holds the target of row wq + 4l
// (`lk` kind, `ld` destination, `lp` position), worked out while the main
// loop ran; the rows' targets are broadcast from there.
DF_DEV void qkv_finish_warp(const Plan& p, const QkvOut& qo, int wq, int lane, float4 w4,
                            int lk, __nv_bfloat16* ld, int lp, const float4* stile,
                            const float* tile_part, uint32_t cl_base = 0, int cl_rank = 0,
                            int cl_n = 1) {
  constexpr int C4 = HD / 4;
  const int last_j = __reduce_max_sync(0xffffffffu, lk != 0 ? lane : -1);
  // rows wq + 4j; with a cluster source (cl_base: the same offset of every
  // rank's shared memory) this rank takes j = cl_rank, cl_rank + cl_n, ...
  for (int k0 = 0; cl_rank + cl_n * k0 <= last_j; k0 += 4) {
    int kind[4], jv[4];
    float4 x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      jv[i] = cl_rank + cl_n * (k0 + i);
      const int rr = wq + 4 * jv[i];
      kind[i] = __shfl_sync(0xffffffffu, lk, jv[i] & 31);
      if (jv[i] >= 32) kind[i] = 0;
      x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kind[i] != 0 && stile != nullptr) x[i] = stile[rr * C4 + (lane ^ (rr & (C4 - 1)))];
    }
    if (cl_base != 0) {
      // the rows summed over the cluster's ranks, in rank order
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (kind[i] == 0) continue;
        const int rr = wq + 4 * jv[i];
        const uint32_t off = cl_base + (uint32_t)(rr * C4 + (lane ^ (rr & (C4 - 1)))) * 16;
        float4 t[MAX_SPLITS];
#pragma unroll
        for (int c = 0; c < MAX_SPLITS; ++c)
          if (c < cl_n) t[c] = ld_cluster_f4(cluster_map(off, (uint32_t)c));
#pragma unroll
        for (int c = 0; c < MAX_SPLITS; ++c) {
          if (c < cl_n) {
            x[i].x += t[c].x;
            x[i].y += t[c].y;
            x[i].z += t[c].z;
            x[i].w += t[c].w;
          }
        }
      }
    } else if (stile == nullptr) {
#pragma unroll
      for (int sp = 0; sp < MAX_SPLITS; ++sp) {
        if (sp < p.splits) {
          const float4* part = reinterpret_cast<const float4*>(tile_part + (size_t)sp * (BM * HD));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (kind[i] != 0) {
              const float4 t = __ldcg(part + (wq + 4 * jv[i]) * C4 + lane);
              x[i].x += t.x;
              x[i].y += t.y;
              x[i].z += t.z;
              x[i].w += t.w;
            }
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int src_lane = jv[i] & 31;
      const int pos_raw = __shfl_sync(0xffffffffu, lp, src_lane);
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(ld), src_lane));
      if (kind[i] == 0) continue;
      float4 o = x[i];
      if (kind[i] != 3) {
        int pos = pos_raw;
        if (pos < 0 || pos >= qo.max_pos) {
          if (lane == 0) record_error(p.err, 2 /* DFLASH_DEV_POSITION */);
          pos = 0;
        }
        o = warp_norm_rope(o, w4, qo.eps, qo.rope + (size_t)pos * (HD / 2),
                           kind[i] == 1 ? qo.q_scale : 1.f, lane);
      }
      uint2 pk;
      pk.x = pack_bf16x2(o.x, o.y);
      pk.y = pack_bf16x2(o.z, o.w);
      reinterpret_cast<uint2*>(dst)[lane] = pk;
    }
  }
}

// Split-K merge of a plain epilogue inside a thread-block cluster of SPLITS
// CTAs, each of which parked its fp32 rows in its own shared memory
// ([row][column chunk], swizzled).  Warp wq of rank c takes the valid rows
// r = c + SPLITS (wq + 4i); lane l reads columns 4l .. 4l+3 of row r from every
// rank, sums them in rank order and stores them (coalesced across the warp).
template <int EPI, int SPLITS>
DF_DEV void cluster_sum_rows(const Plan& p, int m_tile, int n0, const uint8_t* smem, int wq,
                             int lane) {
  constexpr int C4 = HD / 4;
  const int rank = (int)cluster_ctarank();
  const uint32_t base = smem_u32(smem);
  for (int r = rank + SPLITS * wq; r < BM; r += SPLITS * 4) {
    int src, srow;
    row_source(p, m_tile, r, src, srow);
    if (src < 0) continue;
    const uint32_t off = base + (uint32_t)(r * C4 + (lane ^ (r & (C4 - 1)))) * 16;
    float4 t[SPLITS];
#pragma unroll
    for (int c = 0; c < SPLITS; ++c) t[c] = ld_cluster_f4(cluster_map(off, (uint32_t)c));
    float4 acc = t[0];
#pragma unroll
    for (int c = 1; c < SPLITS; ++c) {
      acc.x += t[c].x;
      acc.y += t[c].y;
      acc.z += t[c].z;
      acc.w += t[c].w;
    }
    if constexpr (EPI == EPI_F32) {
      reinterpret_cast<float4*>(reinterpret_cast<float*>(p.c) + (size_t)srow * p.ldc + n0)[lane] =
          acc;
    } else if constexpr (EPI == EPI_SWIGLU) {
      // lanes 0..15 hold gate columns 4l.., lanes 16..31 the matching up columns
      float4 up;
      up.x = __shfl_down_sync(0xffffffffu, acc.x, 16);
      up.y = __shfl_down_sync(0xffffffffu, acc.y, 16);
      up.z = __shfl_down_sync(0xffffffffu, acc.z, 16);
      up.w = __shfl_down_sync(0xffffffffu, acc.w, 16);
      if (lane < 16) {
        uint2 pk;
        pk.x = pack_bf16x2(acc.x / (1.f + __expf(-acc.x)) * up.x,
                           acc.y / (1.f + __expf(-acc.y)) * up.y);
        pk.y = pack_bf16x2(acc.z / (1.f + __expf(-acc.z)) * up.z,
                           acc.w / (1.f + __expf(-acc.w)) * up.w);
        reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.c) + (size_t)srow * p.ldc +
                                 n0 / 2)[lane] = pk;
      }
    } else {
      uint2 pk;
      pk.x = pack_bf16x2(acc.x, acc.y);
      pk.y = pack_bf16x2(acc.z, acc.w);
      reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.c) + (size_t)srow * p.ldc +
                               n0)[lane] = pk;
    }
  }
}

template <int EPI, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA0,
                     const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ Plan p,
                     const __grid_constant__ QkvOut qo,
                     const __grid_constant__ SeqTable st) {
  static_assert(EPI != EPI_QKV || BN == HD, "QKV tiles are one head wide");
  constexpr uint32_t B_BYTES = BN * BK * 2;
  constexpr int C4 = BN / 4;  // float4 chunks per row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  // A stage holds two 64-column k-blocks, each [A rows (a_bytes) | B tile
  // (B_BYTES)], so that one wait and one commit of the MMA thread cover eight
  // MMAs (with four, the synchronisation is not hidden behind the MMAs).
  // The MMA reads 128 A rows; the rows past the box fall into the stage's own
  // B tile, which no copy writes while that MMA runs.
  const size_t half = (size_t)p.a_bytes + B_BYTES;
  const size_t stride = 2 * half;
  uint8_t* sA = smem;
  uint8_t* sB = smem + p.a_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * stride);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* accb = empty + MAX_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int m_tile, n_tile, split;
  decode_tile_split(p, blockIdx.x, m_tile, n_tile, split);
  n_tile += p.n_tile0;
  const int tile_id = n_tile * (p.n_m0 + p.n_m1) + m_tile;
  const int kb0 = (int)((long long)split * p.n_kb / p.splits);
  const int kb1 = (int)((long long)(split + 1) * p.n_kb / p.splits);
  const int nkb = kb1 - kb0;
  const int n_st = (nkb + 1) / 2;  // stages of two k-blocks (the last may hold one)
  const bool from_a0 = m_tile < p.n_m0;
  const int a_row0 = (from_a0 ? m_tile : m_tile - p.n_m0) * BM;
  const int n0 = n_tile * BN;
  // QKV epilogue: the tile's norm gains and, per lane, the target of the
  // row its warp finishes (set by the epilogue warps during the main loop)
  float4 qk_w4 = make_float4(0.f, 0.f, 0.f, 0.f);
  int qk_kind = 0, qk_pos = 0;
  __nv_bfloat16* qk_dst = nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accb, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA0);
    if (p.merged || !from_a0) prefetch_tmap(&tmA1);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const CUtensorMap* ma = from_a0 ? &tmA0 : &tmA1;
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      // weights first: they do not depend on the previous kernel
      const int pre = min(S, n_st);
      for (int i = 0; i < pre; ++i) {
        const int hk = min(2, nkb - 2 * i);
        mbar_arrive_expect_tx(&full[i], (uint32_t)(hk * half));
        for (int h = 0; h < hk; ++h)
          tma_load_2d(sB + (size_t)i * stride + h * half, &tmB, &full[i],
                      (kb0 + 2 * i + h) * BK, n0, pol_w);
      }
      grid_dep_sync();
      // slot s and its pass over the ring (phase bit ph) advance with i: the
      // ring depth is a run-time value, and a division per stage would sit
      // on this thread's issue path
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < n_st; ++i, s = s + 1 == S ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
        const int hk = min(2, nkb - 2 * i);
        if (i >= pre) {
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.err)) break;
          mbar_arrive_expect_tx(&full[s], (uint32_t)(hk * half));
          for (int h = 0; h < hk; ++h)
            tma_load_2d(sB + (size_t)s * stride + h * half, &tmB, &full[s],
                        (kb0 + 2 * i + h) * BK, n0, pol_w);
        }
        for (int h = 0; h < hk; ++h) {
          const int kx = (kb0 + 2 * i + h) * BK;
          uint8_t* a_dst = sA + (size_t)s * stride + h * half;
          tma_load_2d(a_dst, ma, &full[s], kx, a_row0, pol_a);
          if (p.merged)
            tma_load_2d(a_dst + (size_t)p.box0 * BK * 2, &tmA1, &full[s], kx, 0, pol_a);
        }
      }
    }
  } else if (warp == 1) {
    grid_dep_sync();
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN, false);
      // descriptors of stage 0, k-block 0; the others are address offsets
      // (the start address field holds address / 16)
      const uint64_t a_desc0 = sdesc_sw128(smem_u32(sA), 16, 1024);
      const uint64_t b_desc0 = sdesc_sw128(smem_u32(sB), 16, 1024);
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < n_st; ++i, s = s + 1 == S ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
        const int hk = min(2, nkb - 2 * i);
        if (!mbar_wait(&full[s], ph, abort_flag, p.err)) break;
        tc_fence_after();
        for (int h = 0; h < hk; ++h) {
          const uint32_t off = (uint32_t)(((size_t)s * stride + h * half) >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16(tmem, a_desc0 + off + kk * 2, b_desc0 + off + kk * 2, idesc,
                        (i > 0 || h > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&empty[s]);
      }
      tc_commit(accb);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    grid_dep_sync();
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    int src, srow;
    row_source(p, m_tile, r, src, srow);
    if constexpr (EPI == EPI_QKV) {
      // While the main loop runs: this tile's norm weights into registers,
      // and lane l looks up the position of row q + 4l (the rows warp q
      // finishes) and warms L2 with its RoPE row.
      const float* norm = qkv_col_norm(qo, n0);
      const float4 w4 = norm != nullptr ? __ldg(reinterpret_cast<const float4*>(norm) + lane)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
      int lane_kind = 0, lane_pos = 0;
      __nv_bfloat16* lane_dst = nullptr;
      {
        int s2, r2;
        row_source(p, m_tile, q + 4 * lane, s2, r2);
        if (s2 >= 0) {
          const QkvTarget g = qkv_target(qo, st, s2, r2, n0);
          lane_kind = g.kind;
          lane_dst = g.dst;
          if (g.kind == 1 || g.kind == 2) {
            lane_pos = qo.positions[g.pos_idx];
            if (lane_pos >= 0 && lane_pos < qo.max_pos) {
              const char* rp = reinterpret_cast<const char*>(qo.rope + (size_t)lane_pos * (HD / 2));
#pragma unroll
              for (int i = 0; i < HD * 4; i += 128) prefetch_l2(rp + i);
            }
          }
        }
      }
      qk_w4 = w4;
      qk_kind = lane_kind;
      qk_dst = lane_dst;
      qk_pos = lane_pos;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(accb, 0, abort_flag, p.err));
      tc_fence_after();
      const int et = threadIdx.x - 64;
      float* tile_part = p.partial + (size_t)tile_id * p.splits * (BM * HD);
      float4* stile = reinterpret_cast<float4*>(smem);
      bool finish = true;
      if (p.splits > 1 && p.cluster) {
        // the tile's splits are one cluster: the rows wait in this CTA's
        // idle stage buffers (as the one-split tile) for the merge below
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          float t[32];
          tmem_ld32(trow + c * 32, t);
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4)
            stile[r * C4 + ((c * 8 + i4) ^ (r & (C4 - 1)))] =
                ok ? make_float4(t[4 * i4], t[4 * i4 + 1], t[4 * i4 + 2], t[4 * i4 + 3])
                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        finish = false;
      } else if (p.splits == 1) {
        // accumulator row -> shared tile ([row][column chunk], swizzled)
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          float t[32];
          tmem_ld32(trow + c * 32, t);
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4)
            stile[r * C4 + ((c * 8 + i4) ^ (r & (C4 - 1)))] =
                ok ? make_float4(t[4 * i4], t[4 * i4 + 1], t[4 * i4 + 2], t[4 * i4 + 3])
                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        named_bar_sync(1, 128);
      } else {
        // every split writes the valid rows of its fp32 partial ([row][128]);
        // the last CTA of the tile (atomic counter) sums them in split order
        // (tcgen05.ld is warp-collective: every lane loads, valid rows store)
        float4* mine = reinterpret_cast<float4*>(tile_part + (size_t)split * (BM * HD) +
                                                 (size_t)r * HD);
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          float t[32];
          tmem_ld32(trow + c * 32, t);
          if (src >= 0) {
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4)
              __stcg(mine + c * 8 + i4,
                     ok ? make_float4(t[4 * i4], t[4 * i4 + 1], t[4 * i4 + 2], t[4 * i4 + 3])
                        : make_float4(0.f, 0.f, 0.f, 0.f));
          }
        }
        named_bar_sync(1, 128);
        if (et == 0) {
          const int old = atomic_add_acq_rel_gpu(p.counters + tile_id, 1);
          *last_flag = (old == p.splits - 1) ? 1 : 0;
        }
        named_bar_sync(1, 128);
        finish = *last_flag != 0;
      }
      if (finish) {
        qkv_finish_warp(p, qo, q, lane, w4, lane_kind, lane_dst, lane_pos,
                        p.splits == 1 ? stile : nullptr, tile_part);
        if (p.splits > 1 && et == 0) p.counters[tile_id] = 0;
      }
    } else {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(accb, 0, abort_flag, p.err));
      tc_fence_after();
      float v[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        float t[32];
        tmem_ld32(trow + c * 32, t);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[c * 32 + i] = ok ? t[i] : 0.f;
      }
      if (p.splits == 1 || p.slices) {
        if (src >= 0)
          finish_row<EPI>(p, qo, st, v, src, srow, n0, p.slices ? split * p.slice_stride : 0);
      } else if (src >= 0) {
        // park the valid rows in this CTA's (now idle) stage buffers, swizzled
        float4* red = reinterpret_cast<float4*>(smem);
#pragma unroll
        for (int c4 = 0; c4 < C4; ++c4)
          red[r * C4 + (c4 ^ (r & (C4 - 1)))] =
              make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
      }
    }
  }

  if (p.splits > 1 && p.cluster && !p.slices) {
    // The splits of this tile are one thread-block cluster.  Rank c sums the
    // valid rows r with r % splits == c from every rank's shared memory, in
    // rank order (so the result does not depend on timing), one row per warp.
    cluster_sync();
    if (warp >= 2) {
      if constexpr (EPI == EPI_QKV) {
        // rank c finishes the rows wq + 4j, j = c mod splits, of every warp wq
        qkv_finish_warp(p, qo, warp & 3, lane, qk_w4, qk_kind, qk_dst, qk_pos, nullptr, nullptr,
                        smem_u32(smem), (int)cluster_ctarank(), p.splits);
      } else {
        switch (p.splits) {
          case 2: cluster_sum_rows<EPI, 2>(p, m_tile, n0, smem, warp & 3, lane); break;
          case 3: cluster_sum_rows<EPI, 3>(p, m_tile, n0, smem, warp & 3, lane); break;
          case 4: cluster_sum_rows<EPI, 4>(p, m_tile, n0, smem, warp & 3, lane); break;
          case 5: cluster_sum_rows<EPI, 5>(p, m_tile, n0, smem, warp & 3, lane); break;
          case 6: cluster_sum_rows<EPI, 6>(p, m_tile, n0, smem, warp & 3, lane); break;
          case 7: cluster_sum_rows<EPI, 7>(p, m_tile, n0, smem, warp & 3, lane); break;
          default: cluster_sum_rows<EPI, 8>(p, m_tile, n0, smem, warp & 3, lane); break;
        }
      }
    }
    cluster_sync();  // no CTA leaves while the others still read its rows
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, BN);
  }
}

// ---------------------------------------------------------------- swapped operands
// 129 .. 384 token rows from one source (the context projection and o_proj of
// mid-size batches).  The MMA takes a 128-row weight tile as A and the token
// rows as B: N = the rows rounded up to 16, in one or two MMAs of at most 256,
// so no tensor work goes to padding rows (the persistent kernel would compute
// whole 128-row tiles).  D^T (weight rows x token rows) accumulates in TMEM.
// The K splits of a weight tile form one thread-block cluster: each parks D^T
// in its idle stage buffers as [token][column] rows, and every rank sums a
// share of the tokens from all ranks, in rank order.
constexpr int SWAP_MAX_ROWS = 384;

struct SwapPlan {
  int rows;          // token rows
  int rb;            // rows rounded up to 16 (the MMA N, both chunks)
  int xb0, xb1;      // rows of the two X boxes (xb1 = 0: one box)
  int n_kb, splits, stages;
  uint32_t x_bytes;  // X bytes per stage
  uint32_t tmem_cols;
  int ldc;
  void* c;
  int* err;
};

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_swap_kernel(const __grid_constant__ CUtensorMap tmX0,
                     const __grid_constant__ CUtensorMap tmX1,
                     const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ SwapPlan p) {
  constexpr uint32_t W_BYTES = BM * BK * 2;
  constexpr int C4 = BM / 4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  uint8_t* sW = smem;
  uint8_t* sX = smem + (size_t)S * W_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sX + (size_t)S * p.x_bytes);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* accb = empty + MAX_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
  const int kb0 = (int)((long long)split * p.n_kb / p.splits);
  const int kb1 = (int)((long long)(split + 1) * p.n_kb / p.splits);
  const int nkb = kb1 - kb0;
  const int n0 = n_tile * BM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accb, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmX0);
    if (p.xb1 > 0) prefetch_tmap(&tmX1);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      // weights first: they do not depend on the previous kernel
      const int pre = min(S, nkb);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], W_BYTES + p.x_bytes);
        tma_load_2d(sW + (size_t)i * W_BYTES, &tmW, &full[i], (kb0 + i) * BK, n0, pol_w);
      }
      grid_dep_sync();
      int s = 0;  // slot and phase bit advance with i (no division per stage)
      uint32_t ph = 0;
      for (int i = 0; i < nkb; ++i, s = s + 1 == S ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
        const int kx = (kb0 + i) * BK;
        if (i >= pre) {
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.err)) break;
          mbar_arrive_expect_tx(&full[s], W_BYTES + p.x_bytes);
          tma_load_2d(sW + (size_t)s * W_BYTES, &tmW, &full[s], kx, n0, pol_w);
        }
        uint8_t* x_dst = sX + (size_t)s * p.x_bytes;
        tma_load_2d(x_dst, &tmX0, &full[s], kx, 0, pol_x);
        if (p.xb1 > 0) tma_load_2d(x_dst + (size_t)p.xb0 * BK * 2, &tmX1, &full[s], kx, p.xb0, pol_x);
      }
    }
  } else if (warp == 1) {
    grid_dep_sync();
    if (lane == 0) {
      const uint32_t idesc0 = idesc_bf16(BM, p.xb0, false);
      const uint32_t idesc1 = idesc_bf16(BM, p.xb1 > 0 ? p.xb1 : 16, false);
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nkb; ++i, s = s + 1 == S ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
        if (!mbar_wait(&full[s], ph, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t w_base = smem_u32(sW + (size_t)s * W_BYTES);
        const uint32_t x_base = smem_u32(sX + (size_t)s * p.x_bytes);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(w_base + kk * 32, 16, 1024);
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          tc_mma_bf16(tmem, ad, sdesc_sw128(x_base + kk * 32, 16, 1024), idesc0, acc);
          if (p.xb1 > 0)
            tc_mma_bf16(tmem + (uint32_t)p.xb0, ad,
                        sdesc_sw128(x_base + (uint32_t)p.xb0 * BK * 2 + kk * 32, 16, 1024),
                        idesc1, acc);
        }
        tc_commit(&empty[s]);
      }
      tc_commit(accb);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    grid_dep_sync();
    const int q = warp & 3;
    const int j = q * 32 + lane;  // weight row of the tile = output column n0 + j
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(accb, 0, abort_flag, p.err));
    tc_fence_after();
    float* park = reinterpret_cast<float*>(smem);
    for (int t0 = 0; t0 < p.rb; t0 += 32) {
      float v[32];
      tmem_ld32(trow + (uint32_t)t0, v);
      if (p.splits == 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int t = t0 + i;
          if (t >= p.rows) break;
          const float y = ok ? v[i] : 0.f;
          if constexpr (EPI == EPI_F32)
            reinterpret_cast<float*>(p.c)[(size_t)t * p.ldc + n0 + j] = y;
          else
            reinterpret_cast<__nv_bfloat16*>(p.c)[(size_t)t * p.ldc + n0 + j] =
                __float2bfloat16_rn(y);
        }
      } else {
        // token t's row in the park area: 32 float4 chunks, swizzled by t
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int t = t0 + i;
          if (t >= p.rb) break;
          park[(t * C4 + ((j >> 2) ^ (t & (C4 - 1)))) * 4 + (j & 3)] = ok ? v[i] : 0.f;
        }
      }
    }
  }

  if (p.splits > 1) {
    cluster_sync();
    if (warp >= 2) {
      const int rank = (int)cluster_ctarank();
      const uint32_t base = smem_u32(smem);
      for (int t = rank + p.splits * (warp & 3); t < p.rows; t += p.splits * 4) {
        const uint32_t off = base + (uint32_t)(t * C4 + (lane ^ (t & (C4 - 1)))) * 16;
        float4 acc = ld_cluster_f4(cluster_map(off, 0u));
        for (int c = 1; c < p.splits; ++c) {
          const float4 u = ld_cluster_f4(cluster_map(off, (uint32_t)c));
          acc.x += u.x;
          acc.y += u.y;
          acc.z += u.z;
          acc.w += u.w;
        }
        if constexpr (EPI == EPI_F32) {
          reinterpret_cast<float4*>(reinterpret_cast<float*>(p.c) + (size_t)t * p.ldc + n0)[lane] =
              acc;
        } else {
          uint2 pk;
          pk.x = pack_bf16x2(acc.x, acc.y);
          pk.y = pack_bf16x2(acc.z, acc.w);
          reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.c) + (size_t)t * p.ldc +
                                   n0)[lane] = pk;
        }
      }
    }
    cluster_sync();  // no CTA leaves while the others still read its rows
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// ---------------------------------------------------------------- swapped, multicast
// The fp32 fc output of 129 .. 384 token rows, written as per-split slices
// that the following row norm sums.  Weights are the M = 128 operand and the
// token rows N, as in gemm_swap_kernel.  MC weight tiles with the same K range
// form a thread-block cluster.  Each CTA loads 1/MC of the token tile (P rows)
// and multicasts it to the cluster, so an SM issues W + X / MC bytes per
// k-block instead of W + X.  A stage is free again once every CTA of the
// cluster has consumed it (its MMA commit arrives on the stage's empty barrier
// in all of them).  No split merge: split sp writes slice sp of the output.
struct SwapMcPlan {
  int rows, rb, xb0, xb1;  // token rows, rows rounded to 16, the two MMA chunks
  int part;                // token rows each CTA loads (a multiple of 8)
  int tiles, n_kb, splits, stages;
  uint32_t x_bytes;        // MC * part * 128 bytes of tokens per stage
  uint32_t tmem_cols;
  int ldc;
  size_t slice_stride;
  float* c;
  int* err;
};

template <int MC>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_swapmc_kernel(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ SwapMcPlan p) {
  constexpr uint32_t W_BYTES = BM * BK * 2;
  constexpr uint16_t kMask = (uint16_t)((1u << MC) - 1u);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages;
  uint8_t* sW = smem;
  uint8_t* sX = smem + (size_t)S * W_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sX + (size_t)S * p.x_bytes);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* accb = empty + MAX_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tile = blockIdx.x % p.tiles, split = blockIdx.x / p.tiles;
  const int rank = n_tile % MC;  // cluster rank: clusters are MC consecutive tiles
  const int kb0 = (int)((long long)split * p.n_kb / p.splits);
  const int kb1 = (int)((long long)(split + 1) * p.n_kb / p.splits);
  const int nkb = kb1 - kb0;
  const int n0 = n_tile * BM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], MC);
    }
    mbar_init(accb, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every CTA's barriers exist before any multicast copy or commit reaches them
  if (MC > 1) cluster_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      const uint32_t stage_bytes = W_BYTES + p.x_bytes;
      // weights first: they do not depend on the previous kernel
      const int pre = min(S, nkb);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], stage_bytes);
        tma_load_2d(sW + (size_t)i * W_BYTES, &tmW, &full[i], (kb0 + i) * BK, n0, pol_w);
      }
      grid_dep_sync();
      int s = 0;  // slot and phase bit advance with i (no division per stage)
      uint32_t ph = 0;
      for (int i = 0; i < nkb; ++i, s = s + 1 == S ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
        const int kx = (kb0 + i) * BK;
        if (i >= pre) {
          // every CTA of the cluster is done with stage s
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.err)) break;
          mbar_arrive_expect_tx(&full[s], stage_bytes);
          tma_load_2d(sW + (size_t)s * W_BYTES, &tmW, &full[s], kx, n0, pol_w);
        }
        uint8_t* x_dst = sX + (size_t)s * p.x_bytes + (size_t)rank * p.part * (BK * 2);
        if (MC > 1)
          tma_load_2d_mc(x_dst, &tmX, &full[s], kx, rank * p.part, kMask, pol_x);
        else
          tma_load_2d(x_dst, &tmX, &full[s], kx, 0, pol_x);
      }
    }
  } else if (warp == 1) {
    grid_dep_sync();
    if (lane == 0) {
      const uint32_t idesc0 = idesc_bf16(BM, p.xb0, false);
      const uint32_t idesc1 = idesc_bf16(BM, p.xb1 > 0 ? p.xb1 : 16, false);
      const uint64_t w_desc0 = sdesc_sw128(smem_u32(sW), 16, 1024);
      const uint64_t x_desc0 = sdesc_sw128(smem_u32(sX), 16, 1024);
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < nkb; ++i, s = s + 1 == S ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
        if (!mbar_wait(&full[s], ph, abort_flag, p.err)) break;
        tc_fence_after();
        const uint64_t wd = w_desc0 + (((size_t)s * W_BYTES) >> 4);
        const uint64_t xd = x_desc0 + (((size_t)s * p.x_bytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          tc_mma_bf16(tmem, wd + kk * 2, xd + kk * 2, idesc0, acc);
          if (p.xb1 > 0)
            tc_mma_bf16(tmem + (uint32_t)p.xb0, wd + kk * 2,
                        xd + ((uint32_t)p.xb0 * BK * 2 >> 4) + kk * 2, idesc1, acc);
        }
        if (MC > 1)
          tc_commit_mc(&empty[s], kMask);
        else
          tc_commit(&empty[s]);
      }
      tc_commit(accb);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    grid_dep_sync();
    const int q = warp & 3;
    const int j = q * 32 + lane;  // weight row of the tile = output column n0 + j
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(accb, 0, abort_flag, p.err));
    tc_fence_after();
    float* out = p.c + (size_t)split * p.slice_stride + n0 + j;
    for (int t0 = 0; t0 < p.rb; t0 += 32) {
      float v[32];
      tmem_ld32(trow + (uint32_t)t0, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = t0 + i;
        if (t >= p.rows) break;
        out[(size_t)t * p.ldc] = ok ? v[i] : 0.f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // no CTA leaves while a peer's copies or commits may still reach it (each
  // CTA has seen its own last commit complete)
  if (MC > 1) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// ---------------------------------------------------------------- large M
// Persistent variant for calls with many token rows: one CTA per SM walks
// its share of 128 x 256 output tiles (round-robin over the grouped order).
// Two TMEM accumulators (2 x 256 fp32 columns) let the epilogue of one tile
// run while the MMA warp accumulates the next; 256-wide tiles halve the
// shared-memory traffic of A per flop.  K is never split.
constexpr int BNB = 256, STAGES_BIG = 4;
constexpr uint32_t B_BIG = BNB * BK * 2;  // 32 KB
constexpr size_t SMEM_BIG = 1024 + STAGES_BIG * (A_FULL + B_BIG) + 512;

// Work unit u of the persistent kernel: (m, n) tile and split of K.  Units
// are ordered as in the decode-size kernel (groups of m-tiles, then n, then
// split, then m), so the CTAs running at the same time share weight tiles.
DF_DEV void big_unit(const Plan& p, int u, int& m, int& n, int& split, int& k0, int& k1,
                     int& tile_id) {
  decode_unit(p, u, m, n, split);
  k0 = (int)((long long)split * p.n_kb / p.splits);
  k1 = (int)((long long)(split + 1) * p.n_kb / p.splits);
  tile_id = n * (p.n_m0 + p.n_m1) + m;
}

// MC = 2: CTAs 2c and 2c+1 form a cluster and take units 2j and 2j+1 (the
// same weight tile and K split, m-tiles m and m+1; m-tile counts are padded
// to even, a padded tile's rows store nothing).  Each loads its own A tile and
// half of the 256-row weight tile, multicast to both, so an SM issues 32 KB
// of the 48 KB a k-block needs; a stage is free once both have consumed it.
template <int EPI, int MC>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_big_kernel(const __grid_constant__ CUtensorMap tmA0,
                    const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBh,
                    const __grid_constant__ Plan p,
                    const __grid_constant__ QkvOut qo,
                    const __grid_constant__ SeqTable st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES_BIG * A_FULL;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES_BIG * B_BIG);
  uint64_t* empty = full + STAGES_BIG;
  uint64_t* acc_full = empty + STAGES_BIG;  // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2]
  uint64_t* rope_bar = acc_empty + 2;       // QKV, one unit per CTA: staged RoPE rows
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rope_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = p.units_q + (p.n_tiles - p.n_q_tiles) * (p.n_m0 + p.n_m1) * p.splits;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES_BIG; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], MC);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    mbar_init(rope_bar, 128);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA0);
    prefetch_tmap(&tmA1);
    prefetch_tmap(MC > 1 ? &tmBh : &tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // both CTAs' barriers exist before any multicast copy or commit reaches them
  if (MC > 1) cluster_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_last();
      const uint64_t pol_a = policy_evict_last();
      const int rk = MC > 1 ? (int)(blockIdx.x & 1) : 0;
      // this CTA's share of a weight k-block: half of the 256-row tile
      // (multicast to the pair), or all of it
      auto load_b = [&](int s, int n, int kb) {
        if (MC > 1)
          tma_load_2d_mc(sB + s * B_BIG + rk * (B_BIG / 2), &tmBh, &full[s], kb * BK,
                         n * BNB + rk * (BNB / 2), (uint16_t)3, pol_w);
        else
          tma_load_2d(sB + s * B_BIG, &tmB, &full[s], kb * BK, n * BNB, pol_w);
      };
      // The weights do not depend on the previous kernel: the first stages
      // get their weight boxes before the dependency wait.
      int pre = 0;
      if (blockIdx.x < units) {
        int m, n, sp, k0, k1, tid;
        big_unit(p, blockIdx.x, m, n, sp, k0, k1, tid);
        pre = min(STAGES_BIG, k1 - k0);
        for (int i = 0; i < pre; ++i) {
          mbar_arrive_expect_tx(&full[i], A_FULL + B_BIG);
          load_b(i, n, k0 + i);
        }
      }
      grid_dep_sync();
      uint32_t it = 0;
      bool alive = true;
      for (int u = blockIdx.x; alive && u < units; u += gridDim.x) {
        int m, n, sp, k0, k1, tid;
        big_unit(p, u, m, n, sp, k0, k1, tid);
        const bool a0 = m < p.n_m0;
        const CUtensorMap* ma = a0 ? &tmA0 : &tmA1;
        const int a_row0 = (a0 ? m : m - p.n_m0) * BM;
        for (int kb = k0; kb < k1; ++kb, ++it) {
          const int s = it % STAGES_BIG;
          if (it >= (uint32_t)pre) {
            const uint32_t ph = (it / STAGES_BIG) & 1;
            if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, p.err)) {
              alive = false;
              break;
            }
            mbar_arrive_expect_tx(&full[s], A_FULL + B_BIG);
            load_b(s, n, kb);
          }
          tma_load_2d(sA + s * A_FULL, ma, &full[s], kb * BK, a_row0, pol_a);
        }
      }
    } else {
      grid_dep_sync();
    }
  } else if (warp == 1) {
    grid_dep_sync();
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BNB, false);
      uint32_t it = 0, tc = 0;
      bool alive = true;
      for (int u = blockIdx.x; alive && u < units; u += gridDim.x, ++tc) {
        int m, n, sp, k0, k1, tid;
        big_unit(p, u, m, n, sp, k0, k1, tid);
        const uint32_t buf = tc & 1, use = tc >> 1;
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * BNB;
        for (int kb = k0; kb < k1; ++kb, ++it) {
          const int s = it % STAGES_BIG;
          const uint32_t ph = (it / STAGES_BIG) & 1;
          if (!mbar_wait(&full[s], ph, abort_flag, p.err)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + s * A_FULL);
          const uint32_t b_base = smem_u32(sB + s * B_BIG);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16(d, sdesc_sw128(a_base + kk * 32, 16, 1024),
                        sdesc_sw128(b_base + kk * 32, 16, 1024), idesc,
                        (kb > k0 || kk > 0) ? 1u : 0u);
          if (MC > 1)
            tc_commit_mc(&empty[s], (uint16_t)3);
          else
            tc_commit(&empty[s]);
        }
        tc_commit(&acc_full[buf]);
      }
    }
  } else {
    grid_dep_sync();
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int et = threadIdx.x - 64;
    uint32_t tc = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++tc) {
      int m, n, sp, k0, k1, tid;
      big_unit(p, u, m, n, sp, k0, k1, tid);
      const uint32_t buf = tc & 1, use = tc >> 1;
      int src, srow;
      row_source(p, m, r, src, srow);
      // QKV: the row's destinations and positions for both heads of the tile
      // (a search over the sequences and a global load), and its RoPE rows
      // warmed in L2, while the accumulator is still being computed
      QkvTarget tg[BNB / HD];
      int tpos[BNB / HD];
      if constexpr (EPI == EPI_QKV) {
#pragma unroll
        for (int h = 0; h < BNB / HD; ++h) {
          tg[h].kind = 0;
          tpos[h] = 0;
          if (src >= 0) {
            tg[h] = qkv_target(qo, st, src, srow, n * BNB + h * HD);
            if (tg[h].kind == 1 || tg[h].kind == 2) {
              tpos[h] = checked_position(qo, tg[h].pos_idx, p.err);
              const char* rp = reinterpret_cast<const char*>(qo.rope + (size_t)tpos[h] * (HD / 2));
#pragma unroll
              for (int i = 0; i < HD * 4; i += 128) prefetch_l2(rp + i);
            }
          }
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], use & 1, abort_flag, p.err)))
        break;
      tc_fence_after();
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + buf * BNB;
      const bool whole = p.splits == 1 || p.slices;
      if constexpr (EPI == EPI_QKV) {
        if (whole) {
          // norm, RoPE and stores straight from TMEM, then the accumulator
          // goes back to the MMA warp.  The tile's two heads share the row's
          // position and gains.  A CTA with a single unit has idle stage
          // buffers now (every MMA has completed): the rows' (cos, sin)
          // pairs and the gains are copied there in one round of bulk
          // copies rather than read piece by piece from L2 in the epilogue.
          const float* gains = qkv_col_norm(qo, n * BNB);
          const bool rot = src >= 0 && (tg[0].kind == 1 || tg[0].kind == 2);
          const float4* w4 = reinterpret_cast<const float4*>(gains);
          const float4* r4 = reinterpret_cast<const float4*>(qo.rope + (size_t)tpos[0] * (HD / 2));
          if ((int)gridDim.x >= units) {
            // HD / 2 (cos, sin) pairs = HD / 4 float4 = 512 B a row, rows 528 B
            // apart (a warp's 16-byte reads of 32 rows then spread over all
            // banks), then the gains
            constexpr int RS = HD / 4 + 1;
            float4* s_rope = reinterpret_cast<float4*>(smem) + r * RS;
            float4* s_gain = reinterpret_cast<float4*>(smem) + BM * RS;
            const uint32_t bytes = (rot ? 512u : 0u) + (et == 0 && gains != nullptr ? 512u : 0u);
            if (bytes > 0) {
              mbar_arrive_expect_tx(rope_bar, bytes);
              if (rot) bulk_load_1d(s_rope, r4, 512, rope_bar);
              if (et == 0 && gains != nullptr) bulk_load_1d(s_gain, gains, 512, rope_bar);
            } else {
              mbar_arrive(rope_bar);
            }
            mbar_wait(rope_bar, 0, abort_flag, p.err);
            w4 = s_gain;
            r4 = s_rope;
          }
#pragma unroll 1
          for (int half = 0; half < BNB / HD; ++half) {
            QkvTarget g = tg[half];
            if (src < 0) g.kind = 0;
            qkv_apply_tmem(qo, g, trow + half * HD, w4, r4);
          }
          tc_fence_before();
          mbar_arrive(&acc_empty[buf]);
          continue;
        }
      }
      // split units: sums of the valid rows go to the (tile, split) slot,
      // laid out [column chunk of 4][row] so a warp's access is contiguous
      float4* my_part =
          reinterpret_cast<float4*>(p.partial) + ((size_t)tid * p.splits + sp) * (BM * BNB / 4);
#pragma unroll 1
      for (int half = 0; half < BNB / HD; ++half) {
        float v[HD];
        uint32_t raw[HD / 32][32];
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) tmem_ld32_nowait(trow + half * HD + c * 32, raw[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < HD / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) v[c * 32 + i] = __uint_as_float(raw[c][i]);
        if (half == BNB / HD - 1) {
          // the accumulator is fully read: hand it back to the MMA warp
          tc_fence_before();
          mbar_arrive(&acc_empty[buf]);
        }
        if (whole) {
          if constexpr (EPI == EPI_QKV) {
            if (src >= 0) qkv_apply(qo, tg[half], tpos[half], v);
          } else if (src >= 0) {
            finish_row<EPI>(p, qo, st, v, src, srow, n * BNB + half * HD,
                            p.slices ? sp * p.slice_stride : 0);
          }
        } else if (src >= 0) {
#pragma unroll
          for (int c4 = 0; c4 < HD / 4; ++c4)
            __stcg(my_part + (half * (HD / 4) + c4) * BM + r,
                   make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]));
        }
      }
      if (whole) continue;
      // the CTA that finishes a tile's last split sums every split in order
      // (deterministic) and runs the epilogue
      named_bar_sync(1, 128);
      if (et == 0) {
        const int old = atomic_add_acq_rel_gpu(p.counters + tid, 1);
        *last_flag = (old == p.splits - 1) ? 1 : 0;
      }
      named_bar_sync(1, 128);
      const bool last = *last_flag != 0;
      named_bar_sync(1, 128);  // everyone has read the flag before it is reused
      if (!last) continue;
#pragma unroll 1
      for (int half = 0; half < BNB / HD; ++half) {
        float v[HD];
#pragma unroll
        for (int i = 0; i < HD; ++i) v[i] = 0.f;
        if (src >= 0) {
          for (int c = 0; c < p.splits; ++c) {
            const float4* pc = reinterpret_cast<const float4*>(p.partial) +
                               ((size_t)tid * p.splits + c) * (BM * BNB / 4) +
                               (size_t)half * (HD / 4) * BM + r;
#pragma unroll
            for (int c4 = 0; c4 < HD / 4; ++c4) {
              const float4 w4 = __ldcg(pc + c4 * BM);
              v[4 * c4] += w4.x;
              v[4 * c4 + 1] += w4.y;
              v[4 * c4 + 2] += w4.z;
              v[4 * c4 + 3] += w4.w;
            }
          }
          if constexpr (EPI == EPI_QKV)
            qkv_apply(qo, tg[half], tpos[half], v);
          else
            finish_row<EPI>(p, qo, st, v, src, srow, n * BNB + half * HD);
        }
      }
      if (et == 0) p.counters[tid] = 0;
    }
  }

  tc_fence_before();
  __syncthreads();
  // no CTA leaves while its peer's copies or commits may still reach it
  if (MC > 1) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                  void*, const cuuint64_t*, const cuuint64_t*,
                                  const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  // looked up once (thread-safe static initialisation); null if the driver
  // does not provide it
  static const EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

// Split count minimising (waves) x (per-unit time), per-unit time in
// k-block units plus a fixed cost per CTA and a cost for the cluster merge.
// At most 8 splits (a portable cluster).
int choose_splits(int tiles, int n_kb, int num_sms) {
  if (tiles >= num_sms) return 1;
  const double c_cta = 6.0, c_part = 2.0;
  int best = 1;
  double best_t = 1e30;
  const int max_s = std::max(1, std::min(8, n_kb / 2));
  for (int s = 1; s <= max_s; ++s) {
    const int waves = (tiles * s + num_sms - 1) / num_sms;
    const double t = waves * ((double)n_kb / s + c_cta + (s > 1 ? c_part : 0.0));
    if (t < best_t - 1e-9) {
      best_t = t;
      best = s;
    }
  }
  return best;
}

int round8(int x) { return (x + 7) / 8 * 8; }

struct Geometry {
  int bn, merged, box0, box1;
  int n_m0, n_m1, n_tiles, n_q_tiles, n_kb, tiles, splits;
  size_t a_bytes;
  int stages;
};

Geometry geometry(int epi, int rows0, int rows1, int n, int k, int q_cols, int num_sms) {
  Geometry g;
  // 128-wide tiles: 16 KB weight boxes (narrower boxes multiply the TMA
  // requests per byte, which caps per-SM bandwidth below the HBM share)
  g.bn = 128;
  (void)epi;
  g.merged = rows1 > 0 && round8(rows0) + round8(rows1) <= BM;
  if (g.merged) {
    g.box0 = std::max(8, round8(rows0));
    g.box1 = std::max(8, round8(rows1));
    g.n_m0 = 1;
    g.n_m1 = 0;
    g.a_bytes = (size_t)(g.box0 + g.box1) * BK * 2;
  } else {
    const int most = std::min(BM, std::max(rows0, rows1));
    g.box0 = g.box1 = std::min(BM, std::max(8, round8(most)));
    g.n_m0 = (rows0 + BM - 1) / BM;
    g.n_m1 = (rows1 + BM - 1) / BM;
    g.a_bytes = (size_t)g.box0 * BK * 2;
  }
  g.n_tiles = n / g.bn;
  g.n_q_tiles = q_cols / g.bn;
  g.n_kb = k / BK;
  g.tiles = g.n_q_tiles * g.n_m0 + (g.n_tiles - g.n_q_tiles) * (g.n_m0 + g.n_m1);
  g.splits = choose_splits(g.tiles, g.n_kb, num_sms);
  const size_t b_bytes = (size_t)g.bn * BK * 2;
  // a stage holds two k-blocks
  g.stages = (int)std::min<size_t>(MAX_STAGES,
                                   (SMEM_LIMIT - SMEM_FIXED) / (2 * (b_bytes + g.a_bytes)));
  return g;
}

size_t smem_bytes(const Geometry& g) {
  return SMEM_FIXED + (size_t)g.stages * 2 * ((size_t)g.bn * BK * 2 + g.a_bytes);
}

template <int EPI, int BN>
void set_smem_attr() {
  cudaFuncSetAttribute(gemm_bf16_kernel<EPI, BN>,
                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_LIMIT);
}

// one source of 129 .. 384 rows, plain epilogue: the swapped-operand kernel
bool use_swap(int epi, int rows0, int rows1, int n) {
  return (epi == EPI_F32 || epi == EPI_BF16) && rows1 == 0 && rows0 > BM &&
         rows0 <= SWAP_MAX_ROWS && n % BM == 0;
}

// many token rows and 256-aligned column regions: the persistent kernel
bool use_big(int rows0, int rows1, int n, int q_cols) {
  return rows0 + rows1 > BM && n % BNB == 0 && q_cols % BNB == 0;
}

int launch_swap(const GemmShape& s, int epi, void* c, int ldc, int num_sms, int* err,
                cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  if (!done_on_device(attr_done)) {
    cudaFuncSetAttribute(gemm_swap_kernel<EPI_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)SMEM_LIMIT);
    cudaFuncSetAttribute(gemm_swap_kernel<EPI_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)SMEM_LIMIT);
    mark_device(attr_done);
  }
  SwapPlan p{};
  p.rows = s.a0_rows;
  p.rb = (s.a0_rows + 15) / 16 * 16;
  // above 256 rows: two MMA chunks of near-equal width (an MMA costs about
  // max(N / 2, 64) cycles, so 144 + 128 beats 256 + 16)
  p.xb0 = p.rb <= 256 ? p.rb : (p.rb / 2 + 15) / 16 * 16;
  p.xb1 = p.rb - p.xb0;
  p.n_kb = s.k / BK;
  const int tiles = s.n / BM;
  p.splits = choose_splits(tiles, p.n_kb, num_sms);
  p.x_bytes = (uint32_t)p.rb * BK * 2;
  const size_t stage = (size_t)BM * BK * 2 + p.x_bytes;
  p.stages = (int)std::min<size_t>(MAX_STAGES, (SMEM_LIMIT - SMEM_FIXED) / stage);
  // the split merge parks [rb][128] fp32 in the stage buffers
  if (p.stages < 2 || (p.splits > 1 && (size_t)p.stages * stage < (size_t)p.rb * BM * 4))
    return cudaErrorInvalidValue;
  p.tmem_cols = p.rb <= 256 ? 256u : 512u;
  p.ldc = ldc;
  p.c = c;
  p.err = err;
  CUtensorMap mx0, mx1;
  if (make_tmap_bf16_rows(&mx0, s.a0, s.a0_rows, s.k, p.xb0) != 0)
    return cudaErrorInvalidValue;
  if (p.xb1 > 0) {
    if (make_tmap_bf16_rows(&mx1, s.a0, s.a0_rows, s.k, p.xb1) != 0)
      return cudaErrorInvalidValue;
  } else {
    mx1 = mx0;
  }
  const size_t smem = SMEM_FIXED + (size_t)p.stages * stage;
  const dim3 grid(tiles * p.splits), block(kThreads);
  const unsigned cl = p.splits > 1 ? (unsigned)p.splits : 1u;
  cudaError_t e;
  if (epi == EPI_F32)
    e = launch_pdl_cluster(gemm_swap_kernel<EPI_F32>, grid, block, smem, stream, cl, mx0, mx1,
                           *s.b_map, p);
  else
    e = launch_pdl_cluster(gemm_swap_kernel<EPI_BF16>, grid, block, smem, stream, cl, mx0, mx1,
                           *s.b_map, p);
  return (int)e;
}

// the multicast fc kernel takes one-source F32 calls of 129 .. 384 rows whose
// weight tiles pair up into clusters
bool use_swapmc(int epi, int rows0, int rows1, int n, bool slices) {
  return slices && epi == EPI_F32 && use_swap(epi, rows0, rows1, n) && (n / BM) % 2 == 0;
}

int launch_swapmc(const GemmShape& s, float* c, int ldc, size_t slice_stride, int num_sms,
                  int* err, cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  if (!done_on_device(attr_done)) {
    cudaFuncSetAttribute(gemm_swapmc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)SMEM_LIMIT);
    cudaFuncSetAttribute(gemm_swapmc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)SMEM_LIMIT);
    mark_device(attr_done);
  }
  SwapMcPlan p{};
  p.rows = s.a0_rows;
  p.rb = (s.a0_rows + 15) / 16 * 16;
  p.xb0 = p.rb <= 256 ? p.rb : (p.rb / 2 + 15) / 16 * 16;
  p.xb1 = p.rb - p.xb0;
  p.tiles = s.n / BM;
  p.n_kb = s.k / BK;
  p.splits = choose_splits(p.tiles, p.n_kb, num_sms);
  const int mc = p.tiles % 4 == 0 ? 4 : 2;
  p.part = ((p.rb + mc - 1) / mc + 7) / 8 * 8;
  p.x_bytes = (uint32_t)(mc * p.part * BK * 2);
  const size_t stage = (size_t)BM * BK * 2 + p.x_bytes;
  p.stages = (int)std::min<size_t>(MAX_STAGES, (SMEM_LIMIT - SMEM_FIXED) / stage);
  if (p.stages < 2 || p.part > 256) return cudaErrorInvalidValue;
  p.tmem_cols = p.rb <= 256 ? 256u : 512u;
  p.ldc = ldc;
  p.slice_stride = slice_stride;
  p.c = c;
  p.err = err;
  CUtensorMap mx;
  if (make_tmap_bf16_rows(&mx, s.a0, s.a0_rows, s.k, p.part) != 0) return cudaErrorInvalidValue;
  const size_t smem = SMEM_FIXED + (size_t)p.stages * stage;
  const dim3 grid(p.tiles * p.splits), block(kThreads);
  if (mc == 4)
    return (int)launch_pdl_cluster(gemm_swapmc_kernel<4>, grid, block, smem, stream, 4u, mx,
                                   *s.b_map, p);
  return (int)launch_pdl_cluster(gemm_swapmc_kernel<2>, grid, block, smem, stream, 2u, mx,
                                 *s.b_map, p);
}

// m-tiles of the persistent kernel's two sources, padded so that both of its
// regions (block-row tiles; all tiles) hold an even count: the kernel's CTA
// pairs take m-tiles two at a time
void big_m_tiles(int rows0, int rows1, int* m0, int* m1) {
  *m0 = (rows0 + BM - 1) / BM;
  *m1 = (rows1 + BM - 1) / BM;
  if (*m0 % 2) ++*m0;
  if ((*m0 + *m1) % 2) ++*m1;
}

int big_tiles(int rows0, int rows1, int n, int q_cols) {
  int m0, m1;
  big_m_tiles(rows0, rows1, &m0, &m1);
  return (q_cols / BNB) * m0 + (n / BNB - q_cols / BNB) * (m0 + m1);
}

// Splits of K for the persistent kernel: fill the SMs in whole waves, with
// a small per-unit cost (no relaunch); the last CTA of a tile reads every
// split's 128 KB partial back, a cost that grows with the split count.
int big_splits(int tiles, int n_kb, int num_sms) {
  if (tiles >= 2 * num_sms) return 1;
  const double c_unit = 2.0, c_merge = 8.0;
  int best = 1;
  double best_t = 1e30;
  const int max_s = std::max(1, std::min(4, n_kb / 4));
  for (int sp = 1; sp <= max_s; ++sp) {
    const int waves = (tiles * sp + num_sms - 1) / num_sms;
    const double t = waves * ((double)n_kb / sp + c_unit) + (sp > 1 ? c_merge * sp : 0.0);
    if (t < best_t - 1e-9) {
      best_t = t;
      best = sp;
    }
  }
  return best;
}

int launch_big(const GemmShape& s, int epi, void* c, int ldc, const QkvOut* qkv,
               const SeqTable* seqs, const GemmScratch& scr, int num_sms, int* err,
               cudaStream_t stream);

}  // namespace

int make_tmap_bf16_rows(CUtensorMap* map, const void* ptr, long long rows,
                        int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return -1;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) != 0 || (cols % 8) != 0 || rows <= 0)
    return -2;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
                  dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -3;
}

size_t gemm_scratch_bytes(int epi, int rows0, int rows1, int n, int k, int q_cols,
                          int num_sms, int* n_counters) {
  if (use_swap(epi, rows0, rows1, n)) {  // cluster merge, no scratch
    if (n_counters) *n_counters = 0;
    return 0;
  }
  if (use_big(rows0, rows1, n, q_cols)) {
    const int tiles = big_tiles(rows0, rows1, n, q_cols);
    const int splits = big_splits(tiles, k / BK, num_sms);
    int m0, m1;
    big_m_tiles(rows0, rows1, &m0, &m1);
    const int dense = (n / BNB) * (m0 + m1);
    if (n_counters) *n_counters = dense;
    if (splits == 1) return 0;
    return (size_t)dense * splits * BM * BNB * sizeof(float);
  }
  // plain epilogues merge their splits inside a cluster (no scratch); the
  // QKV epilogue merges through global partials
  Geometry g = geometry(epi, rows0, rows1, n, k, q_cols, num_sms);
  const int dense_tiles = g.n_tiles * (g.n_m0 + g.n_m1);
  if (epi != EPI_QKV || g.splits <= 1) {
    if (n_counters) *n_counters = 0;
    return 0;
  }
  if (n_counters) *n_counters = dense_tiles;
  return (size_t)dense_tiles * g.splits * BM * g.bn * sizeof(float);
}

int gemm_f32_slices(int rows, int n, int k, int num_sms) {
  if (use_swapmc(EPI_F32, rows, 0, n, true)) return choose_splits(n / BM, k / BK, num_sms);
  if (use_swap(EPI_F32, rows, 0, n)) return 1;
  if (use_big(rows, 0, n, 0)) return big_splits(big_tiles(rows, 0, n, 0), k / BK, num_sms);
  return geometry(EPI_F32, rows, 0, n, k, 0, num_sms).splits;
}

int launch_gemm_bf16(const GemmShape& s, int epi, void* c, int ldc,
                     const QkvOut* qkv, const SeqTable* seqs,
                     const GemmScratch& scr, int num_sms, int* err,
                     cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  if (!done_on_device(attr_done)) {
    set_smem_attr<EPI_BF16, 128>();
    set_smem_attr<EPI_F32, 128>();
    set_smem_attr<EPI_QKV, 128>();
    set_smem_attr<EPI_SWIGLU, 128>();
    mark_device(attr_done);
  }
  if (s.k % BK != 0) return cudaErrorInvalidValue;
  if (use_swapmc(epi, s.a0_rows, s.a1_rows, s.n, scr.f32_slices != 0))
    return launch_swapmc(s, static_cast<float*>(c), ldc, scr.slice_stride, num_sms, err, stream);
  if (use_swap(epi, s.a0_rows, s.a1_rows, s.n))
    return launch_swap(s, epi, c, ldc, num_sms, err, stream);
  if (use_big(s.a0_rows, s.a1_rows, s.n, s.q_cols))
    return launch_big(s, epi, c, ldc, qkv, seqs, scr, num_sms, err, stream);
  Geometry g = geometry(epi, s.a0_rows, s.a1_rows, s.n, s.k, s.q_cols, num_sms);
  if (s.n % g.bn != 0 || s.q_cols % g.bn != 0) return cudaErrorInvalidValue;
  if (g.tiles == 0) return cudaSuccess;
  Plan p;
  p.a0_rows = s.a0_rows;
  p.a1_rows = s.a1_rows;
  p.n_m0 = g.n_m0;
  p.n_m1 = g.n_m1;
  p.merged = g.merged;
  // plain epilogues merge splits in a cluster (or, F32 with slices, write
  // one slice per split).  The QKV epilogue of block and context rows takes
  // two splits in a 2-CTA cluster when the tiles allow one wave of them
  // (3-CTA clusters schedule poorly behind the previous kernel); with block
  // rows only, or more tiles, its splits merge through global partials
  // (measured: the 2-CTA clusters sped up the single-sequence and
  // band-layer steps and the per-layer five-layer schedule, and slowed the
  // layers that follow a grouped context projection).
  p.slices = epi == EPI_F32 && scr.f32_slices && g.splits > 1;
  p.slice_stride = scr.slice_stride;
  p.cluster = epi != EPI_QKV && !p.slices;
  if (epi == EPI_QKV && g.splits > 1 && 2 * g.tiles <= num_sms && s.a1_rows > 0) {
    g.splits = 2;
    p.cluster = 1;
  }
  if (g.splits > 1 && !p.cluster && !p.slices) {
    const size_t need = (size_t)g.n_tiles * (g.n_m0 + g.n_m1) * g.splits * BM * g.bn * 4;
    if (scr.partial == nullptr || scr.partial_bytes < need ||
        scr.n_counters < g.n_tiles * (g.n_m0 + g.n_m1))
      return cudaErrorInvalidValue;
  }
  p.box0 = g.box0;
  p.box1 = g.box1;
  p.n_tiles = g.n_tiles;
  p.n_q_tiles = g.n_q_tiles;
  p.n_kb = g.n_kb;
  p.splits = g.splits;
  p.stages = g.stages;
  p.a_bytes = (uint32_t)g.a_bytes;
  p.units_q = g.n_q_tiles * g.splits * g.n_m0;
  p.ldc = ldc;
  p.c = c;
  p.err = err;
  p.partial = scr.partial;
  p.counters = scr.counters;
  CUtensorMap ma0, ma1;
  if (make_tmap_bf16_rows(&ma0, s.a0, s.a0_rows, s.k, g.box0) != 0)
    return cudaErrorInvalidValue;
  if (s.a1_rows > 0) {
    if (make_tmap_bf16_rows(&ma1, s.a1, s.a1_rows, s.k, g.box1) != 0)
      return cudaErrorInvalidValue;
  } else {
    ma1 = ma0;
  }
  static QkvOut zero_q{};
  static SeqTable zero_st{};
  const QkvOut& qo = qkv ? *qkv : zero_q;
  const SeqTable& st = seqs ? *seqs : zero_st;
  const size_t smem = smem_bytes(g);
  if (g.bn != 128) return cudaErrorInvalidValue;
  auto launch = [&](const Plan& pl, int ctas) {
    const dim3 grid(ctas), block(kThreads);
    const unsigned cl = pl.cluster && pl.splits > 1 ? (unsigned)pl.splits : 1u;
    if (epi == EPI_QKV)
      return launch_pdl_cluster(gemm_bf16_kernel<EPI_QKV, 128>, grid, block, smem, stream, cl,
                                ma0, ma1, *s.b_map, pl, qo, st);
    if (epi == EPI_BF16)
      return launch_pdl_cluster(gemm_bf16_kernel<EPI_BF16, 128>, grid, block, smem, stream, cl,
                                ma0, ma1, *s.b_map, pl, qo, st);
    if (epi == EPI_SWIGLU)
      return launch_pdl_cluster(gemm_bf16_kernel<EPI_SWIGLU, 128>, grid, block, smem, stream,
                                cl, ma0, ma1, *s.b_map, pl, qo, st);
    return launch_pdl_cluster(gemm_bf16_kernel<EPI_F32, 128>, grid, block, smem, stream, cl,
                              ma0, ma1, *s.b_map, pl, qo, st);
  };
  p.n_tile0 = 0;
  // Between one and two waves of whole tiles (e.g. the MLP's gate/up
  // projection at decode size, 192 tiles): the tiles past the first wave
  // would run alone as a thin second wave, far below the HBM rate.  Those
  // go to a second launch with their K split over a cluster (2 to 4 CTAs),
  // which starts on the SMs the first wave frees.
  const int rem = g.n_tiles - num_sms;
  if (p.cluster && g.splits == 1 && g.n_m0 + g.n_m1 == 1 && g.n_q_tiles == 0 && rem > 0 &&
      rem < num_sms) {
    // (at most about 15/16 of the SMs hold 3- or 4-CTA clusters at once)
    const int cap = num_sms - num_sms / 16;
    const int s2 = rem * 4 <= cap ? 4 : rem * 3 <= cap ? 3 : rem * 2 <= num_sms ? 2 : 1;
    Plan p1 = p;
    p1.n_tiles = num_sms;
    const cudaError_t e = launch(p1, num_sms);
    if (e != cudaSuccess) return (int)e;
    Plan p2 = p;
    p2.n_tile0 = num_sms;
    p2.n_tiles = rem;
    p2.splits = s2;
    return (int)launch(p2, rem * s2);
  }
  return (int)launch(p, g.tiles * g.splits);
}

}  // namespace df

namespace df {
namespace {

int launch_big(const GemmShape& s, int epi, void* c, int ldc, const QkvOut* qkv,
               const SeqTable* seqs, const GemmScratch& scr, int num_sms, int* err,
               cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  if (!done_on_device(attr_done)) {
    cudaFuncSetAttribute(gemm_big_kernel<EPI_BF16, 2>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BIG);
    cudaFuncSetAttribute(gemm_big_kernel<EPI_F32, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)SMEM_BIG);
    cudaFuncSetAttribute(gemm_big_kernel<EPI_QKV, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)SMEM_BIG);
    cudaFuncSetAttribute(gemm_big_kernel<EPI_SWIGLU, 2>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BIG);
    mark_device(attr_done);
  }
  if (s.b_map256 == nullptr || s.b_map == nullptr) return cudaErrorInvalidValue;
  Plan p{};
  p.a0_rows = s.a0_rows;
  p.a1_rows = s.a1_rows;
  big_m_tiles(s.a0_rows, s.a1_rows, &p.n_m0, &p.n_m1);
  p.merged = 0;
  p.box0 = p.box1 = BM;
  p.n_tiles = s.n / BNB;
  p.n_q_tiles = s.q_cols / BNB;
  p.n_kb = s.k / BK;
  p.stages = STAGES_BIG;
  p.a_bytes = A_FULL;
  p.ldc = ldc;
  p.c = c;
  p.err = err;
  const int tiles = p.n_q_tiles * p.n_m0 + (p.n_tiles - p.n_q_tiles) * (p.n_m0 + p.n_m1);
  p.splits = big_splits(tiles, p.n_kb, num_sms);
  p.units_q = p.n_q_tiles * p.splits * p.n_m0;
  const int units = tiles * p.splits;  // even: the m-tile counts are
  p.grid = std::min(units, num_sms) & ~1;
  p.slices = epi == EPI_F32 && scr.f32_slices && p.splits > 1;
  p.slice_stride = scr.slice_stride;
  if (p.splits > 1 && !p.slices) {
    const int dense = p.n_tiles * (p.n_m0 + p.n_m1);
    if (scr.partial == nullptr || scr.n_counters < dense ||
        scr.partial_bytes < (size_t)dense * p.splits * BM * BNB * sizeof(float))
      return cudaErrorInvalidValue;
    p.partial = scr.partial;
    p.counters = scr.counters;
  }
  CUtensorMap ma0, ma1;
  if (make_tmap_bf16_rows(&ma0, s.a0, s.a0_rows, s.k, BM) != 0) return cudaErrorInvalidValue;
  if (s.a1_rows > 0) {
    if (make_tmap_bf16_rows(&ma1, s.a1, s.a1_rows, s.k, BM) != 0) return cudaErrorInvalidValue;
  } else {
    ma1 = ma0;
  }
  static QkvOut zero_q{};
  static SeqTable zero_st{};
  const QkvOut& qo = qkv ? *qkv : zero_q;
  const SeqTable& st = seqs ? *seqs : zero_st;
  if (p.grid < 2) return cudaErrorInvalidValue;
  const dim3 grid(p.grid), block(kThreads);
  cudaError_t e;
  if (epi == EPI_QKV)
    e = launch_pdl_cluster(gemm_big_kernel<EPI_QKV, 2>, grid, block, SMEM_BIG, stream, 2u, ma0,
                           ma1, *s.b_map256, *s.b_map, p, qo, st);
  else if (epi == EPI_BF16)
    e = launch_pdl_cluster(gemm_big_kernel<EPI_BF16, 2>, grid, block, SMEM_BIG, stream, 2u, ma0,
                           ma1, *s.b_map256, *s.b_map, p, qo, st);
  else if (epi == EPI_SWIGLU)
    e = launch_pdl_cluster(gemm_big_kernel<EPI_SWIGLU, 2>, grid, block, SMEM_BIG, stream, 2u,
                           ma0, ma1, *s.b_map256, *s.b_map, p, qo, st);
  else
    e = launch_pdl_cluster(gemm_big_kernel<EPI_F32, 2>, grid, block, SMEM_BIG, stream, 2u, ma0,
                           ma1, *s.b_map256, *s.b_map, p, qo, st);
  return (int)e;
}

}  // namespace
}  // namespace df
