// Backward of the packed training layout's attention core
// ("nemo_automodel.components.speculative.dflash.draft_qwen3", module
// docstring: block k's queries see the context strictly before its anchor and
// their own block; training backpropagates through that masked attention).
//
// Given Q, K, V, the forward output O and its per-row log-sum-exp, and dO:
//   P = exp(scale * Q K^T - lse) on visible keys (0 elsewhere)
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - rowsum(dO * O))
//   dQ = scale * dS K,  dK = scale * dS^T Q
// (rowsum(dO * O) equals each softmax row's rowsum(P * dP)).
//
// Layout and work split (GB300: one CTA per SM, 512 TMEM columns):
//  - a prep kernel writes Q' = Q * scale * log2(e) and dO in the tile layout
//    [B][n_kv][n_blocks][groups][block][d] (a block's groups x block = 64
//    query rows of one kv head are contiguous), rowsum(dO * O) and lse in
//    log2 units per tile row;
//  - one launch holds two kinds of CTA.  dK/dV CTAs keep a 128-key tile of K
//    and V in shared memory and stream the blocks that see it, 64 query rows
//    at a time: S^T = K Q'^T and dP^T = V dO^T (M 128 keys, N 64 queries) into
//    TMEM, eight compute warps (two per TMEM lane quarter, one key row and 32
//    query columns per thread) turn them into P^T and dS^T as bf16 pairs
//    written back over the first 16 of their columns, and dV += P^T dO,
//    dK += dS^T Q' run with A read from TMEM.  dQ CTAs keep two
//    blocks' Q' and dO (128 query rows) in TMEM as the A operands and stream
//    the keys those blocks see, 64 at a time: S = Q' K^T, dP = dO V^T, dS in
//    TMEM, dQ += dS K.  S/dP
//    buffers are double-buffered, so the tensor core computes step i+1 while
//    the compute warps work on step i.  No atomics: every output row is
//    written by exactly one CTA.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

constexpr int HD = 128;              // head_dim
constexpr int QB = 64;               // query rows of one block (groups x block)
constexpr int KT = 128;              // key rows of a dK/dV CTA
constexpr int KS = 64;               // key rows of a dQ step
constexpr int NST = 4;               // pipeline stages
constexpr int kThreads = 320;        // producer, MMA issuer, eight compute warps
constexpr int kCompute = 256;        // two warps per TMEM lane quarter, 32 columns each
constexpr uint32_t TMEM_COLS = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// shared memory (both CTA kinds use the same size):
//   dK/dV: K 32 KB | V 32 KB | Q' stages 4 x 16 KB | dO stages 4 x 16 KB |
//          stats stages 4 x 512 B | barriers
//   dQ:    K stages 6 x 16 KB | V stages 6 x 16 KB | barriers (Q' and dO
//          live in TMEM)
constexpr uint32_t T128 = 128 * HD * 2;  // 32 KB: 128 rows
constexpr uint32_t T64 = 64 * HD * 2;    // 16 KB: 64 rows
constexpr uint32_t STATS_BYTES = 2 * QB * 4;
constexpr size_t SMEM_BYTES = 1024 + 2 * T128 + 2 * NST * T64 + NST * STATS_BYTES + 512;

// TMEM columns (dK/dV CTAs)
constexpr uint32_t C_S0 = 0, C_DP0 = 64, C_S1 = 128, C_DP1 = 192, C_ACC0 = 256, C_ACC1 = 384;
// TMEM columns (dQ CTAs): Q' and dO rows as bf16 pairs (the A operands of
// S and dP), double-buffered S / dP, the dQ accumulator
constexpr uint32_t Q_QA = 0, Q_DOA = 64, Q_S0 = 128, Q_DP0 = 192, Q_S1 = 256, Q_DP1 = 320,
                   Q_ACC = 384;
constexpr int NKS = 6;               // dQ CTAs: K/V stages of 64 rows

// a shared-memory descriptor moved `bytes` further (the start address field
// holds address / 16 in its low 14 bits; no carry within one operand tile)
DF_DEV uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

DF_DEV int clamp_anchor(const PackedBwdArgs& a, int b, int k) {
  int an = a.anchors[b * a.n_blocks + k];
  return min(max(an, 0), a.seq);
}

// ------------------------------------------------------------------ prep
// One warp per (sequence, token, head) row; lane j holds elements 4j..4j+3.
__global__ void __launch_bounds__(256)
    packed_prep_kernel(const __nv_bfloat16* __restrict__ q,
                       const __nv_bfloat16* __restrict__ d_o,
                       const __nv_bfloat16* __restrict__ o, const float* __restrict__ lse,
                       int batch, int n_blocks, int block_size, int n_kv, int groups, float c,
                       __nv_bfloat16* __restrict__ qs, __nv_bfloat16* __restrict__ do_tile,
                       float* __restrict__ dsum, float* __restrict__ lse2) {
  const int nq = n_kv * groups;
  const int T = n_blocks * block_size;
  const long long rows = (long long)batch * T * nq;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  grid_dep_sync();
  if (row >= rows) return;
  const int head = (int)(row % nq);
  const long long bt = row / nq;
  const int token = (int)(bt % T);
  const int b = (int)(bt / T);
  const int h = head / groups, gi = head - h * groups;
  const int k = token / block_size, t = token - k * block_size;
  const long long trow =
      (((long long)b * n_kv + h) * n_blocks + k) * (groups * block_size) + gi * block_size + t;
  const uint2 qv = reinterpret_cast<const uint2*>(q + row * HD)[lane];
  float f[4];
  {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&qv);
    const float2 a0 = __bfloat1622float2(p[0]), a1 = __bfloat1622float2(p[1]);
    f[0] = a0.x * c; f[1] = a0.y * c; f[2] = a1.x * c; f[3] = a1.y * c;
  }
  uint2 out;
  out.x = pack_bf16x2(f[0], f[1]);
  out.y = pack_bf16x2(f[2], f[3]);
  reinterpret_cast<uint2*>(qs + trow * HD)[lane] = out;
  if (d_o == nullptr) return;
  const uint2 dv = reinterpret_cast<const uint2*>(d_o + row * HD)[lane];
  const uint2 ov = reinterpret_cast<const uint2*>(o + row * HD)[lane];
  reinterpret_cast<uint2*>(do_tile + trow * HD)[lane] = dv;
  const __nv_bfloat162* pd = reinterpret_cast<const __nv_bfloat162*>(&dv);
  const __nv_bfloat162* po = reinterpret_cast<const __nv_bfloat162*>(&ov);
  const float2 d0 = __bfloat1622float2(pd[0]), d1 = __bfloat1622float2(pd[1]);
  const float2 o0 = __bfloat1622float2(po[0]), o1 = __bfloat1622float2(po[1]);
  float s = d0.x * o0.x + d0.y * o0.y + d1.x * o1.x + d1.y * o1.y;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) {  // negated: the compute warps add them
    dsum[trow] = -s;
    lse2[trow] = -lse[row] * kLog2e;
  }
}

// ---------------------------------------------------------- dK / dV CTA
struct KvUnit {
  int b, h;
  int k0;          // first key row of the tile within its (sequence, kv head)
  bool own;        // a tile of the blocks' own rows (else context rows)
  int blk_lo, blk_hi;  // candidate blocks [lo, hi)
  int rows_valid;  // tile rows inside the unit's segment
};

// key tile j of pair `pair`: context rows (own = false) or the blocks' rows
DF_DEV KvUnit kv_unit(const PackedBwdArgs& a, int pair, int j, bool own) {
  KvUnit w;
  w.b = pair / a.n_kv;
  w.h = pair - w.b * a.n_kv;
  w.own = own;
  if (!own) {
    w.k0 = j * KT;
    w.blk_lo = 0;
    w.blk_hi = a.n_blocks;
    w.rows_valid = min(KT, a.seq - w.k0);
  } else {
    const int r0 = j * KT;  // first row of the tile in the blocks' region
    w.k0 = a.seq + r0;
    w.blk_lo = r0 / a.block_size;
    w.blk_hi = min(a.n_blocks, (r0 + KT + a.block_size - 1) / a.block_size);
    w.rows_valid = min(KT, a.n_blocks * a.block_size - r0);
  }
  return w;
}

// The blocks that see a key of the tile, walked from the last candidate
// down (every role of the CTA walks the same list): the context tiles of a
// pair differ in where their lists stop, not where they start, so the tiles
// dispatched together read each block's Q'/dO at about the same time and
// it is fetched from HBM about once.  kv_prev returns the largest block
// <= k that sees the tile, below blk_lo if none.
DF_DEV int kv_prev(const PackedBwdArgs& a, const KvUnit& w, int k) {
  if (w.own) return k;
  while (k >= w.blk_lo && clamp_anchor(a, w.b, k) <= w.k0) --k;
  return k;
}

DF_DEV void dkdv_body(uint8_t* smem, const CUtensorMap* tmQ, const CUtensorMap* tmDO,
                      const CUtensorMap* tmK, const CUtensorMap* tmV, const PackedBwdArgs& a,
                      const KvUnit& w) {
  uint8_t* sK = smem;
  uint8_t* sV = sK + T128;
  uint8_t* sQ = sV + T128;         // [NST] Q' of one block
  uint8_t* sDO = sQ + NST * T64;   // [NST] dO of one block
  float* sStat = reinterpret_cast<float*>(sDO + NST * T64);  // [NST][lse2 64 | dsum 64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sDO + NST * T64 + NST * STATS_BYTES);
  uint64_t* kv_full = bars;
  uint64_t* q_full = kv_full + 1;    // [NST]
  uint64_t* q_empty = q_full + NST;  // [NST]
  uint64_t* s_full = q_empty + NST;  // [2]
  uint64_t* p_full = s_full + 2;     // [2]
  uint64_t* acc_done = p_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kCompute);
    }
    mbar_init(acc_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(tmQ);
    prefetch_tmap(tmDO);
    prefetch_tmap(tmK);
    prefetch_tmap(tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_sync();
  const long long pair_blk = ((long long)w.b * a.n_kv + w.h) * a.n_blocks;
  const int first = kv_prev(a, w, w.blk_hi - 1);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();  // a block's rows serve many key tiles
      const int y = (int)(((long long)w.b * a.n_kv + w.h) * a.per + w.k0);
      mbar_arrive_expect_tx(kv_full, 2 * T128);
      tma_load_2d(sK, tmK, kv_full, 0, y, pol_kv);
      tma_load_2d(sK + T128 / 2, tmK, kv_full, 64, y, pol_kv);
      tma_load_2d(sV, tmV, kv_full, 0, y, pol_kv);
      tma_load_2d(sV + T128 / 2, tmV, kv_full, 64, y, pol_kv);
      int i = 0;
      for (int k = first; k >= w.blk_lo; k = kv_prev(a, w, k - 1), ++i) {
        const int s = i % NST;
        if (!mbar_wait(&q_empty[s], ((i / NST) & 1) ^ 1, abort_flag, a.err)) break;
        const int qrow = (int)((pair_blk + k) * QB);
        mbar_arrive_expect_tx(&q_full[s], 2 * T64 + STATS_BYTES);
        tma_load_2d(sQ + s * T64, tmQ, &q_full[s], 0, qrow, pol_q);
        tma_load_2d(sQ + s * T64 + T64 / 2, tmQ, &q_full[s], 64, qrow, pol_q);
        tma_load_2d(sDO + s * T64, tmDO, &q_full[s], 0, qrow, pol_q);
        tma_load_2d(sDO + s * T64 + T64 / 2, tmDO, &q_full[s], 64, qrow, pol_q);
        bulk_load_1d(sStat + s * 2 * QB, a.lse2 + (size_t)qrow, QB * 4, &q_full[s]);
        bulk_load_1d(sStat + s * 2 * QB + QB, a.dsum + (size_t)qrow, QB * 4, &q_full[s]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, QB, false);
      constexpr uint32_t idesc_acc = idesc_bf16(128, HD, true);
      const uint64_t d_k = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t d_v = sdesc_sw128(smem_u32(sV), 16, 1024);
      bool alive = mbar_wait(kv_full, 0, abort_flag, a.err);
      // S^T = K Q'^T and dP^T = V dO^T of step i into buffer i & 1
      auto issue_s = [&](int i) {
        const int s = i % NST;
        if (!mbar_wait(&q_full[s], (i / NST) & 1, abort_flag, a.err)) return false;
        tc_fence_after();
        const uint64_t d_q = sdesc_sw128(smem_u32(sQ + s * T64), 16, 1024);
        const uint64_t d_do = sdesc_sw128(smem_u32(sDO + s * T64), 16, 1024);
        const uint32_t cs = tmem + ((i & 1) ? C_S1 : C_S0);
        const uint32_t cdp = tmem + ((i & 1) ? C_DP1 : C_DP0);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t oa = (kk >> 2) * (T128 / 2) + (kk & 3) * 32;
          const uint32_t ob = (kk >> 2) * (T64 / 2) + (kk & 3) * 32;
          tc_mma_bf16(cs, desc_add(d_k, oa), desc_add(d_q, ob), idesc_s, kk > 0 ? 1u : 0u);
          tc_mma_bf16(cdp, desc_add(d_v, oa), desc_add(d_do, ob), idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[i & 1]);
        return true;
      };
      int k = first, i = 0;
      if (alive && k >= w.blk_lo) alive = issue_s(0);
      while (alive && k >= w.blk_lo) {
        const int kn = kv_prev(a, w, k - 1);
        if (kn >= w.blk_lo && !issue_s(i + 1)) break;
        if (!mbar_wait(&p_full[i & 1], (i >> 1) & 1, abort_flag, a.err)) break;
        tc_fence_after();
        const int s = i % NST;
        const uint64_t m_q = sdesc_sw128(smem_u32(sQ + s * T64), T64 / 2, 1024);
        const uint64_t m_do = sdesc_sw128(smem_u32(sDO + s * T64), T64 / 2, 1024);
        const uint32_t cs = tmem + ((i & 1) ? C_S1 : C_S0);
        const uint32_t cdp = tmem + ((i & 1) ? C_DP1 : C_DP0);
        // dV += P^T dO and dK += dS^T Q' (A from TMEM: the pairs of queries
        // 0..31 in columns 0..15, of queries 32..63 in columns 32..47)
#pragma unroll
        for (int kk = 0; kk < QB / 16; ++kk) {
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          const uint32_t ac = kk * 8 + (kk >= 2 ? 16 : 0);
          tc_mma_bf16_ta(tmem + C_ACC0, cs + ac, desc_add(m_do, kk * 16 * 128), idesc_acc, acc);
          tc_mma_bf16_ta(tmem + C_ACC1, cdp + ac, desc_add(m_q, kk * 16 * 128), idesc_acc, acc);
        }
        tc_commit(&q_empty[s]);
        k = kn;
        ++i;
      }
      tc_commit(acc_done);
    }
  } else {
    // ------------------------------------------------------- compute warps
    const int qd = warp & 3;                   // TMEM lane quarter
    const int hf = (warp - 2) >> 2;            // half: query columns hf*32 .. +31
    const int r = qd * 32 + lane;              // key row of the tile
    const uint32_t lrow = tmem + ((uint32_t)(qd * 32) << 16);
    const int key = w.k0 + r;                  // key index in the (sequence, head)
    const int brow = key - a.seq;              // own tiles: row in the blocks' region
    int i = 0;
    bool ok = true;
    for (int k = first; k >= w.blk_lo; k = kv_prev(a, w, k - 1), ++i) {
      const int s = i % NST;
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[i & 1], (i >> 1) & 1, abort_flag, a.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool vis = w.own ? (brow < a.n_blocks * a.block_size && brow / a.block_size == k)
                             : key < clamp_anchor(a, w.b, k);
      const uint32_t cs = lrow + ((i & 1) ? C_S1 : C_S0) + hf * 32;
      const uint32_t cdp = lrow + ((i & 1) ? C_DP1 : C_DP0) + hf * 32;
      // -lse2 and -rowsum(dO*O) of this half's 32 query rows
      const float2* nl = reinterpret_cast<const float2*>(sStat + s * 2 * QB + hf * 32);
      const float2* nd = reinterpret_cast<const float2*>(sStat + s * 2 * QB + QB + hf * 32);
      uint32_t rs[32], rd[32];
      tmem_ld32_nowait(cs, rs);
      tmem_ld32_nowait(cdp, rd);
      tmem_ld_wait();
      uint32_t pw[16], dw[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float2 p = make_float2(0.f, 0.f), g = make_float2(0.f, 0.f);
        if (vis) {
          const float2 x = add_f32x2(
              make_float2(__uint_as_float(rs[2 * e]), __uint_as_float(rs[2 * e + 1])), nl[e]);
          p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          g = mul_f32x2(p, add_f32x2(make_float2(__uint_as_float(rd[2 * e]),
                                                 __uint_as_float(rd[2 * e + 1])),
                                     nd[e]));
        }
        pw[e] = pack_bf16x2(p.x, p.y);
        dw[e] = pack_bf16x2(g.x, g.y);
      }
      // over the first 16 of this half's columns (already read)
      tmem_st16_nowait(cs, pw);
      tmem_st16_nowait(cdp, dw);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[i & 1]);
    }
    // ------------------------------------------------ epilogue (half 0: dV,
    // half 1: dK = ln2 * dS^T Q', Q' carrying scale * log2 e)
    const bool have = ok && i > 0;
    bool done = false;
    if (have) done = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag, a.err));
    tc_fence_after();
    const bool row_ok = r < w.rows_valid;
    const size_t grow = ((size_t)w.b * a.n_kv + w.h) * a.per + w.k0 + r;
    const float f = hf == 0 ? 1.f : kLn2;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(hf == 0 ? a.dv : a.dk) +
                                          grow * HD);
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      float o[32];
      if (done) {
        tmem_ld32(lrow + (hf == 0 ? C_ACC0 : C_ACC1) + c * 32, o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0.f;
      }
      if (row_ok) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint4 pk;
          pk.x = pack_bf16x2(o[8 * e] * f, o[8 * e + 1] * f);
          pk.y = pack_bf16x2(o[8 * e + 2] * f, o[8 * e + 3] * f);
          pk.z = pack_bf16x2(o[8 * e + 4] * f, o[8 * e + 5] * f);
          pk.w = pack_bf16x2(o[8 * e + 6] * f, o[8 * e + 7] * f);
          dst[c * 4 + e] = pk;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- dQ CTA
DF_DEV void dq_body(uint8_t* smem, const CUtensorMap* tmK, const CUtensorMap* tmV,
                    const PackedBwdArgs& a, int pair, int idx) {
  uint8_t* sK = smem;              // [NKS] 64 key rows
  uint8_t* sV = sK + NKS * T64;    // [NKS]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NKS * T64);
  uint64_t* q_full = bars;            // Q' and dO rows in TMEM (compute warps)
  uint64_t* kv_full = q_full + 1;     // [NKS]
  uint64_t* kv_empty = kv_full + NKS;  // [NKS]
  uint64_t* s_full = kv_empty + NKS;  // [2]
  uint64_t* p_full = s_full + 2;      // [2]
  uint64_t* acc_done = p_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // unit: two blocks of one (sequence, kv head); idx 0 = the latest blocks
  // (largest anchors, longest key ranges)
  const int n_qt = (a.n_blocks + 1) / 2;
  const int qt = n_qt - 1 - idx;
  const int b = pair / a.n_kv, h = pair - (pair / a.n_kv) * a.n_kv;
  const int blk0 = 2 * qt;
  const int nbk = min(2, a.n_blocks - blk0);
  const int rows = nbk * QB;

  if (threadIdx.x == 0) {
    mbar_init(q_full, kCompute);
    for (int s = 0; s < NKS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kCompute);
    }
    mbar_init(acc_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(tmK);
    prefetch_tmap(tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_sync();
  int amax = 0;
  for (int kb = 0; kb < nbk; ++kb) amax = max(amax, clamp_anchor(a, b, blk0 + kb));
  const int n_ctx = (amax + KS - 1) / KS;                  // context steps
  const int n_own = (nbk * a.block_size + KS - 1) / KS;    // the blocks' own rows
  const int T = n_ctx + n_own;
  const int own0 = a.seq + blk0 * a.block_size;
  auto key0 = [&](int j) { return j < n_ctx ? j * KS : own0 + (j - n_ctx) * KS; };
  const long long kv_pair = ((long long)b * a.n_kv + h) * a.per;
  const long long q_row0 = (((long long)b * a.n_kv + h) * a.n_blocks + blk0) * QB;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_last();  // context rows serve many CTAs
      for (int j = 0; j < T; ++j) {
        const int s = j % NKS;
        if (!mbar_wait(&kv_empty[s], ((j / NKS) & 1) ^ 1, abort_flag, a.err)) break;
        const int y = (int)(kv_pair + key0(j));
        mbar_arrive_expect_tx(&kv_full[s], 2 * T64);
        tma_load_2d(sK + s * T64, tmK, &kv_full[s], 0, y, pol_kv);
        tma_load_2d(sK + s * T64 + T64 / 2, tmK, &kv_full[s], 64, y, pol_kv);
        tma_load_2d(sV + s * T64, tmV, &kv_full[s], 0, y, pol_kv);
        tma_load_2d(sV + s * T64 + T64 / 2, tmV, &kv_full[s], 64, y, pol_kv);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, KS, false);
      constexpr uint32_t idesc_acc = idesc_bf16(128, HD, true);
      bool alive = mbar_wait(q_full, 0, abort_flag, a.err);
      tc_fence_after();
      // S = Q' K^T and dP = dO V^T of step j into buffer j & 1 (A from TMEM:
      // a K step of 16 head-dim elements is 8 columns)
      auto issue_s = [&](int j) {
        const int s = j % NKS;
        if (!mbar_wait(&kv_full[s], (j / NKS) & 1, abort_flag, a.err)) return false;
        tc_fence_after();
        const uint64_t d_k = sdesc_sw128(smem_u32(sK + s * T64), 16, 1024);
        const uint64_t d_v = sdesc_sw128(smem_u32(sV + s * T64), 16, 1024);
        const uint32_t cs = tmem + ((j & 1) ? Q_S1 : Q_S0);
        const uint32_t cdp = tmem + ((j & 1) ? Q_DP1 : Q_DP0);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t ob = (kk >> 2) * (T64 / 2) + (kk & 3) * 32;
          tc_mma_bf16_ta(cs, tmem + Q_QA + kk * 8, desc_add(d_k, ob), idesc_s, kk > 0 ? 1u : 0u);
          tc_mma_bf16_ta(cdp, tmem + Q_DOA + kk * 8, desc_add(d_v, ob), idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[j & 1]);
        return true;
      };
      if (alive && T > 0) alive = issue_s(0);
      for (int j = 0; j < T && alive; ++j) {
        if (j + 1 < T && !issue_s(j + 1)) break;
        if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1, abort_flag, a.err)) break;
        tc_fence_after();
        const int s = j % NKS;
        const uint64_t m_k = sdesc_sw128(smem_u32(sK + s * T64), T64 / 2, 1024);
        const uint32_t cdp = tmem + ((j & 1) ? Q_DP1 : Q_DP0);
        // dQ += dS K (A from TMEM: the pairs of keys 0..31 in columns 0..15,
        // of keys 32..63 in columns 32..47; K as MN-major B)
#pragma unroll
        for (int kk = 0; kk < KS / 16; ++kk)
          tc_mma_bf16_ta(tmem + Q_ACC, cdp + kk * 8 + (kk >= 2 ? 16 : 0),
                         desc_add(m_k, kk * 16 * 128), idesc_acc,
                         (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&kv_empty[s]);
      }
      tc_commit(acc_done);
    }
  } else {
    // ------------------------------------------------------- compute warps
    const int qd = warp & 3;
    const int hf = (warp - 2) >> 2;  // half: key columns hf*32 .. +31
    const int r = qd * 32 + lane;    // query row of the tile
    const uint32_t lrow = tmem + ((uint32_t)(qd * 32) << 16);
    const bool real = r < rows;
    const int kl = r / QB;
    const int blk = blk0 + kl;
    const int within = r - kl * QB;
    const int gi = within / a.block_size;
    const int t = within - gi * a.block_size;
    const int an = real ? clamp_anchor(a, b, blk) : 0;
    const int own_lo = a.seq + blk * a.block_size, own_hi = own_lo + a.block_size;
    const float nl = real ? a.lse2[q_row0 + r] : 0.f;   // -lse2
    const float nd = real ? a.dsum[q_row0 + r] : 0.f;   // -rowsum(dO*O)
    const float2 nl2 = make_float2(nl, nl), nd2 = make_float2(nd, nd);
    {
      // this row of Q' (half 0) or dO (half 1) into TMEM: the A operand of S
      // or dP, the row's 128 elements as 64 bf16 pairs (zeros past the rows)
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(hf == 0 ? a.qs : a.do_tile) +
          (size_t)(q_row0 + (real ? r : 0)) * HD);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t wv[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint4 x = real ? __ldg(src + c * 8 + e) : make_uint4(0u, 0u, 0u, 0u);
          wv[4 * e] = x.x;
          wv[4 * e + 1] = x.y;
          wv[4 * e + 2] = x.z;
          wv[4 * e + 3] = x.w;
        }
        tmem_st32_nowait(lrow + (hf == 0 ? Q_QA : Q_DOA) + c * 32, wv);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(q_full);
    }
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, a.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int k0 = key0(j) + hf * 32;
      const bool ctx = j < n_ctx;
      const int lo = ctx ? 0 : own_lo, hi = ctx ? an : own_hi;
      const bool all_vis = real && k0 >= lo && k0 + 32 <= hi;
      const uint32_t cs = lrow + ((j & 1) ? Q_S1 : Q_S0) + hf * 32;
      const uint32_t cdp = lrow + ((j & 1) ? Q_DP1 : Q_DP0) + hf * 32;
      uint32_t rs[32], rd[32];
      tmem_ld32_nowait(cs, rs);
      tmem_ld32_nowait(cdp, rd);
      tmem_ld_wait();
      uint32_t dw[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float2 x = add_f32x2(
            make_float2(__uint_as_float(rs[2 * e]), __uint_as_float(rs[2 * e + 1])), nl2);
        float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
        if (!all_vis) {
          const int key = k0 + 2 * e;
          if (!(real && key >= lo && key < hi)) p.x = 0.f;
          if (!(real && key + 1 >= lo && key + 1 < hi)) p.y = 0.f;
        }
        const float2 g = mul_f32x2(
            p, add_f32x2(make_float2(__uint_as_float(rd[2 * e]), __uint_as_float(rd[2 * e + 1])),
                         nd2));
        dw[e] = pack_bf16x2(g.x, g.y);
      }
      tmem_st16_nowait(cdp, dw);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
    }
    // ------------------------------------- epilogue (half h: columns 64h..)
    bool done = false;
    if (ok && T > 0) done = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag, a.err));
    tc_fence_after();
    const int nq = a.n_kv * a.groups;
    const size_t token = (size_t)b * a.n_blocks * a.block_size + (size_t)blk * a.block_size + t;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dq) +
                                          (token * nq + (size_t)h * a.groups + gi) * HD) +
                 hf * 8;
    const float f = a.dq_scale;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float o[32];
      if (done) {
        tmem_ld32(lrow + Q_ACC + hf * 64 + c * 32, o);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0.f;
      }
      if (real) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint4 pk;
          pk.x = pack_bf16x2(o[8 * e] * f, o[8 * e + 1] * f);
          pk.y = pack_bf16x2(o[8 * e + 2] * f, o[8 * e + 3] * f);
          pk.z = pack_bf16x2(o[8 * e + 4] * f, o[8 * e + 5] * f);
          pk.w = pack_bf16x2(o[8 * e + 6] * f, o[8 * e + 7] * f);
          dst[c * 4 + e] = pk;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// One launch.  The (sequence, kv head) pairs are taken kv_group at a time;
// for each group three runs of CTAs: dK/dV over context key tiles (longest
// first), dQ over block pairs (longest first), dK/dV over the blocks' own
// rows (short), each run interleaving the group's pairs.  The CTAs resident
// at a time then work on about one group, whose Q'/dO and K/V L2 holds, so
// every kind of CTA reads them from HBM about once.
__global__ void __launch_bounds__(kThreads, 1)
    packed_bwd_kernel(const __grid_constant__ CUtensorMap tmQ64,
                      const __grid_constant__ CUtensorMap tmDO64,
                      const __grid_constant__ CUtensorMap tmK128,
                      const __grid_constant__ CUtensorMap tmV128,
                      const __grid_constant__ CUtensorMap tmK64,
                      const __grid_constant__ CUtensorMap tmV64,
                      const __grid_constant__ PackedBwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int pairs = a.batch * a.n_kv;
  const int nt = a.n_kv_ctx_units / pairs, nq = a.n_q_units / pairs,
            no = a.n_kv_own_units / pairs;
  const int G = max(1, a.kv_group);
  const int g = (int)blockIdx.x / (G * (nt + nq + no));
  const int p0 = g * G, gsz = min(G, pairs - p0);
  int r = (int)blockIdx.x - g * G * (nt + nq + no);
  if (r < gsz * nt) {
    dkdv_body(smem, &tmQ64, &tmDO64, &tmK128, &tmV128, a,
              kv_unit(a, p0 + r % gsz, r / gsz, false));
  } else if ((r -= gsz * nt) < gsz * nq) {
    dq_body(smem, &tmK64, &tmV64, a, p0 + r % gsz, r / gsz);
  } else {
    r -= gsz * nq;
    dkdv_body(smem, &tmQ64, &tmDO64, &tmK128, &tmV128, a,
              kv_unit(a, p0 + r % gsz, r / gsz, true));
  }
}

}  // namespace

cudaError_t launch_packed_prep(const void* q, const void* d_o, const void* o, const float* lse,
                               int batch, int n_blocks, int block_size, int n_kv, int groups,
                               float c, void* qs, void* do_tile, float* dsum, float* lse2,
                               cudaStream_t stream) {
  const long long rows = (long long)batch * n_blocks * block_size * n_kv * groups;
  if (rows <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)((rows + 7) / 8);
  return launch_pdl(packed_prep_kernel, dim3(grid), dim3(256), 0, stream,
                    static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(d_o),
                    static_cast<const __nv_bfloat16*>(o), lse, batch, n_blocks, block_size, n_kv,
                    groups, c, static_cast<__nv_bfloat16*>(qs),
                    static_cast<__nv_bfloat16*>(do_tile), dsum, lse2);
}

cudaError_t launch_packed_bwd(const PackedBwdArgs& a, const void* qs, const void* do_tile,
                              const void* k, const void* v, cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_set{0};
  if (!done_on_device(attr_set)) {
    cudaError_t e = cudaFuncSetAttribute(packed_bwd_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    mark_device(attr_set);
  }
  const long long q_rows = (long long)a.batch * a.n_kv * a.n_blocks * QB;
  const long long kv_rows = (long long)a.batch * a.n_kv * a.per;
  CUtensorMap mq64, mdo64, mk128, mv128, mk64, mv64;
  if (make_tmap_bf16_rows(&mq64, qs, q_rows, HD, 64) != 0 ||
      make_tmap_bf16_rows(&mdo64, do_tile, q_rows, HD, 64) != 0 ||
      make_tmap_bf16_rows(&mk128, k, kv_rows, HD, 128) != 0 ||
      make_tmap_bf16_rows(&mv128, v, kv_rows, HD, 128) != 0 ||
      make_tmap_bf16_rows(&mk64, k, kv_rows, HD, 64) != 0 ||
      make_tmap_bf16_rows(&mv64, v, kv_rows, HD, 64) != 0)
    return cudaErrorInvalidValue;
  const int units = a.n_kv_ctx_units + a.n_q_units + a.n_kv_own_units;
  if (units <= 0) return cudaSuccess;
  PackedBwdArgs args = a;
  args.qs = qs;
  args.do_tile = do_tile;
  return launch_pdl(packed_bwd_kernel, dim3(units), dim3(kThreads), SMEM_BYTES, stream, mq64,
                    mdo64, mk128, mv128, mk64, mv64, args);
}

}  // namespace df
