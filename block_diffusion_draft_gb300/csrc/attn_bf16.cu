// attn_bf16.cu -- non-causal GQA attention of the draft layer on tcgen05.
//
// One CTA owns one work unit: a (sequence, kv head) pair and a range of its
// 128-key tiles.
// Its Q tile stacks every query head of the KV group times the block rows
// (groups * q_len rows), so each K/V row is read once for all heads of the
// group ("DFlash源码导读（二）" step 1: GQA with num_key_value_groups).
//
//   warp 0      TMA producer: Q tile once, then K and V tiles of 128 keys
//               (two 64-column boxes each, 128-byte swizzle) into a 3-stage ring
//   warp 1      TMEM allocator + MMA issuer:
//                 S(j) = Q K(j)^T          -> TMEM columns [128*(j&1), +128)
//                 O   += P(j) V(j)         -> TMEM columns [256, 384)
//               S(j+1) is issued before waiting for P(j) so the tensor core
//               overlaps the softmax of tile j.
//   warps 2..5  softmax, one TMEM lane (accumulator row) per thread: mask,
//               running max in log2 units (Q is pre-scaled by
//               head_dim^-0.5*log2 e), exp2, bf16 P written into the K slot of
//               the same stage (K(j) is dead once S(j) completed), lazy O
//               rescale (only when the max grows by more than 2^8), final
//               normalisation or split partials.
// The MMA is always M = 128.  An inference block has groups * q_len <= 64
// query rows (64 for 4 heads per KV head x 16); then the Q tile holds every
// row twice ("dual" mode): lane r and lane r + 64 see the same query, lane r
// takes keys 0..63 and lane r + 64 keys 64..127 of every tile as two
// independent online-softmax streams (the other half of each P row is zero),
// and the two are merged at the end.  All four softmax warps work and each
// thread handles 64 columns per tile.  Blocks of more than 64 query rows use
// the same kernel with one row per lane.  The packed training layout has its
// own kernel below (attn_pk2_kernel).
//
// Masks ("nemo_automodel...draft_qwen3", _sliding_window_mask): a row's
// allowed keys are the unit's key range, on a band layer cut to
// |query index - key| < W.
// Work split (plan_decode_attention): with many (sequence, kv head) pairs,
// every pair's tiles are split into units of near-equal size, dispatched
// largest first, so that the SMs finish together; with few pairs, C splits of
// a pair form a thread-block cluster and k clusters share a pair, so that
// every SM gets a unit.  A split leaves an unnormalised partial (O, running
// max, running sum) in its slot in L2; the split that finishes a pair last
// (an arrival counter) merges the pair's partials with the log-sum-exp
// rescaling, in split order.  In a cluster, one cluster barrier orders the
// partials and each rank merges a share of the rows; the clusters' merged row
// blocks are merged the same way by the last cluster to finish.
#include <algorithm>
#include <atomic>
#include <queue>
#include <utility>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

constexpr int HD = 128;
constexpr int BKEY = 128;    // keys per tile
constexpr int NST = 3;       // K/V stages
constexpr int kThreads = 192;
constexpr uint32_t TILE_BYTES = 128 * HD * 2;   // 32 KB: 128 rows x 128 bf16
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;  // one 64-column box
constexpr size_t SMEM_BYTES = 1024 + TILE_BYTES * (1 + 2 * NST) + 512;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t O_COL = 256;
constexpr float kRescaleThreshold = 8.f;  // log2 units

struct Unit {
  int b, h;
  int q_row0;         // first row of the Q tile in the Q buffer
  int rows;           // real query rows in the tile
  long long kv_row0;  // first K/V storage row of (b, h)
  int s0_lo, s0_hi;   // the unit's keys
  int len;            // keys of the sequence after this call
  int ns, c;          // splits of the (sequence, kv head) pair, this unit's split
  int pair_unit0;     // unit of the pair's split 0 (its units are consecutive)
};

// Inference work unit u: split c of the key tiles of (sequence b, kv head h).
DF_DEV Unit decode(const AttnArgs& a, const AttnSeqs& sq, int u) {
  Unit w;
  int lo = 0, hi = a.batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sq.unit_off[mid] <= u) lo = mid; else hi = mid;
  }
  w.b = sq.order[lo];
  w.ns = sq.n_split[w.b];
  const int r = u - sq.unit_off[lo];
  w.h = r / w.ns;
  w.c = r - w.h * w.ns;
  w.pair_unit0 = sq.unit_off[lo] + w.h * w.ns;
  w.len = sq.len[w.b];
  const int k_lo = sq.lo[w.b];
  const int n_t = (w.len - k_lo + BKEY - 1) / BKEY;
  const int t0 = (int)((long long)w.c * n_t / w.ns);
  const int t1 = (int)((long long)(w.c + 1) * n_t / w.ns);
  w.s0_lo = k_lo + t0 * BKEY;
  w.s0_hi = min(w.len, k_lo + t1 * BKEY);
  w.rows = a.groups * a.q_block;
  w.q_row0 = (w.b * a.n_kv + w.h) * w.rows;
  w.kv_row0 = ((long long)w.b * a.n_kv + w.h) * a.cap;
  return w;
}

DF_DEV int n_tiles_of(const Unit& w) {
  return w.s0_hi > w.s0_lo ? (w.s0_hi - w.s0_lo + BKEY - 1) / BKEY : 0;
}

DF_DEV int tile_start(const Unit& w, int j) { return w.s0_lo + j * BKEY; }

// the bf16 output row of query row `row` of the unit's Q tile
DF_DEV __nv_bfloat16* out_row(const AttnArgs& a, const Unit& w, int row) {
  const int gi = row / a.q_len, t = row - gi * a.q_len;
  const size_t token = (size_t)w.b * a.q_len + t;
  return reinterpret_cast<__nv_bfloat16*>(a.out) + token * (size_t)(a.n_kv * a.groups * HD) +
         (size_t)(w.h * a.groups + gi) * HD;
}

// One thread's unnormalised partial row (O, running max, running sum) into
// partial slot `slot` (fp32 [slot][row][d] and [slot][2][row]).
DF_DEV void write_partial(const AttnArgs& a, int slot, int row, const float (&o)[HD], float m,
                          float l) {
  float4* dst = reinterpret_cast<float4*>(a.part_o + ((size_t)slot * 128 + row) * HD);
#pragma unroll
  for (int c4 = 0; c4 < HD / 4; ++c4)
    __stcg(dst + c4, make_float4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]));
  __stcg(a.part_ml + (size_t)slot * 256 + row, m);
  __stcg(a.part_ml + (size_t)slot * 256 + 128 + row, l);
}

// Log-sum-exp merge of rows [r0, r1) over the n partial slots slot0 + i *
// stride, by the 128 softmax threads: thread et takes items et, et + 128, ...
// of (row, chunk of NC4 * 4 columns), so that every row advances at once (one
// round trip to L2 per source, not per source and row).  Sources are summed
// in slot order (the result does not depend on which CTA merges, nor when),
// each rescaled to the largest running max.  The merged row goes to the
// output as the normalised bf16 row, or (block_slot >= 0) unnormalised with
// its max and sum into that slot.
template <int NC4>
DF_DEV void merge_rows_t(const AttnArgs& a, const Unit& w, int slot0, int stride, int n,
                         int r0, int r1, int block_slot, int et) {
  constexpr int CH = HD / (4 * NC4);  // chunks per row
  for (int item = et; item < (r1 - r0) * CH; item += 128) {
    const int row = r0 + item / CH, ch = item % CH;
    float M = -INFINITY;
    for (int i = 0; i < n; ++i)
      M = fmaxf(M, __ldcg(a.part_ml + (size_t)(slot0 + i * stride) * 256 + row));
    float L = 0.f;
    float4 acc[NC4];
#pragma unroll
    for (int c = 0; c < NC4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int i = 0; i < n; ++i) {
        const size_t sl = (size_t)(slot0 + i * stride);
        const float m = __ldcg(a.part_ml + sl * 256 + row);
        const float l = __ldcg(a.part_ml + sl * 256 + 128 + row);
        const float4* src =
            reinterpret_cast<const float4*>(a.part_o + (sl * 128 + row) * HD) + ch * NC4;
        float4 t[NC4];
#pragma unroll
        for (int c = 0; c < NC4; ++c) t[c] = __ldcg(src + c);
        const float f = m == -INFINITY ? 0.f : fast_exp2(m - M);
        L += f * l;
#pragma unroll
        for (int c = 0; c < NC4; ++c) {
          acc[c].x += f * t[c].x;
          acc[c].y += f * t[c].y;
          acc[c].z += f * t[c].z;
          acc[c].w += f * t[c].w;
        }
      }
    }
    if (block_slot >= 0) {
      float4* dst = reinterpret_cast<float4*>(a.part_o + ((size_t)block_slot * 128 + row) * HD) +
                    ch * NC4;
#pragma unroll
      for (int c = 0; c < NC4; ++c) __stcg(dst + c, acc[c]);
      if (ch == 0) {
        __stcg(a.part_ml + (size_t)block_slot * 256 + row, M);
        __stcg(a.part_ml + (size_t)block_slot * 256 + 128 + row, L);
      }
    } else {
      const float inv = L > 0.f ? 1.f / L : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(out_row(a, w, row) + ch * NC4 * 4);
#pragma unroll
      for (int c = 0; c < NC4 / 2; ++c) {
        uint4 pk;
        pk.x = pack_bf16x2(acc[2 * c].x * inv, acc[2 * c].y * inv);
        pk.y = pack_bf16x2(acc[2 * c].z * inv, acc[2 * c].w * inv);
        pk.z = pack_bf16x2(acc[2 * c + 1].x * inv, acc[2 * c + 1].y * inv);
        pk.w = pack_bf16x2(acc[2 * c + 1].z * inv, acc[2 * c + 1].w * inv);
        dst[c] = pk;
      }
    }
  }
}

// the chunk width that keeps the 128 threads busy for the given row count
DF_DEV void merge_rows(const AttnArgs& a, const Unit& w, int slot0, int stride, int n, int r0,
                       int r1, int block_slot, int et) {
  const int rows = r1 - r0;
  if (rows >= 64)
    merge_rows_t<16>(a, w, slot0, stride, n, r0, r1, block_slot, et);
  else if (rows >= 32)
    merge_rows_t<8>(a, w, slot0, stride, n, r0, r1, block_slot, et);
  else if (rows >= 16)
    merge_rows_t<4>(a, w, slot0, stride, n, r0, r1, block_slot, et);
  else
    merge_rows_t<2>(a, w, slot0, stride, n, r0, r1, block_slot, et);
}

// The same merge for splits that are the C CTAs of one cluster, reading the
// partials from the CTAs' shared memory instead of L2: each CTA keeps its
// partial rows in its idle V stages ([row][HD] fp32, 16-byte chunk c of row r
// at position c ^ (r & 31)) followed by the rows' max and sum ([2][128]).
// Every load of an item (all C sources) is issued before any is used.
constexpr uint32_t SMEM_PART_ML = 128 * HD * 4;  // offset of (max, sum) in the partial area

DF_DEV void write_partial_smem(uint8_t* part, int row, const float (&o)[HD], float m, float l) {
  float4* dst = reinterpret_cast<float4*>(part) + row * (HD / 4);
#pragma unroll
  for (int c4 = 0; c4 < HD / 4; ++c4)
    dst[c4 ^ (row & 31)] = make_float4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
  float* ml = reinterpret_cast<float*>(part + SMEM_PART_ML);
  ml[row] = m;
  ml[128 + row] = l;
}

template <int C, int NC4>
DF_DEV void merge_rows_cluster_t(const AttnArgs& a, const Unit& w, uint32_t part, int r0, int r1,
                                 int et) {
  constexpr int CH = HD / (4 * NC4);  // chunks per row
  for (int item = et; item < (r1 - r0) * CH; item += 128) {
    const int row = r0 + item / CH, ch = item % CH;
    float mv[C], lv[C];
    float4 t[C][NC4];
#pragma unroll
    for (int i = 0; i < C; ++i) {
      mv[i] = ld_cluster_f32(cluster_map(part + SMEM_PART_ML + row * 4, (uint32_t)i));
      lv[i] = ld_cluster_f32(cluster_map(part + SMEM_PART_ML + (128 + row) * 4, (uint32_t)i));
#pragma unroll
      for (int c = 0; c < NC4; ++c) {
        const int c4 = ch * NC4 + c;
        t[i][c] = ld_cluster_f4(
            cluster_map(part + (uint32_t)((row * (HD / 4) + (c4 ^ (row & 31))) * 16), (uint32_t)i));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < C; ++i) M = fmaxf(M, mv[i]);
    float L = 0.f;
    float4 acc[NC4];
#pragma unroll
    for (int c = 0; c < NC4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int i = 0; i < C; ++i) {
        const float f = mv[i] == -INFINITY ? 0.f : fast_exp2(mv[i] - M);
        L += f * lv[i];
#pragma unroll
        for (int c = 0; c < NC4; ++c) {
          acc[c].x += f * t[i][c].x;
          acc[c].y += f * t[i][c].y;
          acc[c].z += f * t[i][c].z;
          acc[c].w += f * t[i][c].w;
        }
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(out_row(a, w, row) + ch * NC4 * 4);
#pragma unroll
    for (int c = 0; c < NC4 / 2; ++c) {
      uint4 pk;
      pk.x = pack_bf16x2(acc[2 * c].x * inv, acc[2 * c].y * inv);
      pk.y = pack_bf16x2(acc[2 * c].z * inv, acc[2 * c].w * inv);
      pk.z = pack_bf16x2(acc[2 * c + 1].x * inv, acc[2 * c + 1].y * inv);
      pk.w = pack_bf16x2(acc[2 * c + 1].z * inv, acc[2 * c + 1].w * inv);
      dst[c] = pk;
    }
  }
}

// chunk width by row count, with at most 16 chunks of 16 bytes in flight per
// thread (C sources x NC4)
DF_DEV void merge_rows_cluster(const AttnArgs& a, const Unit& w, uint32_t part, int C, int r0,
                               int r1, int et) {
  const int rows = r1 - r0;
  if (C == 8) {
    merge_rows_cluster_t<8, 2>(a, w, part, r0, r1, et);
  } else if (C == 4) {
    if (rows >= 16)
      merge_rows_cluster_t<4, 4>(a, w, part, r0, r1, et);
    else
      merge_rows_cluster_t<4, 2>(a, w, part, r0, r1, et);
  } else {
    if (rows >= 32)
      merge_rows_cluster_t<2, 8>(a, w, part, r0, r1, et);
    else if (rows >= 16)
      merge_rows_cluster_t<2, 4>(a, w, part, r0, r1, et);
    else
      merge_rows_cluster_t<2, 2>(a, w, part, r0, r1, et);
  }
}

// Called by the 128 softmax threads after their partial stores: counts this
// CTA in at `counter` (one thread, acquire-release at GPU scope, after a
// barrier that orders every thread's stores before it) and returns, to every
// one of them, whether it was the n-th arrival.  The n-th arrival resets the
// counter for the next launch.
DF_DEV bool last_arrival(int* counter, int n, int et, volatile int* flag) {
  __threadfence();
  named_bar_sync(1, 128);
  if (et == 0) {
    const int old = atomic_add_acq_rel_gpu(counter, 1);
    const bool last = old == n - 1;
    if (last) *counter = 0;
    *flag = last ? 1 : 0;
  }
  named_bar_sync(1, 128);
  const bool last = *flag != 0;
  if (last) __threadfence();
  return last;
}

template <bool DUAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ AttnArgs a,
                     const __grid_constant__ AttnSeqs sq) {
  constexpr int NC = DUAL ? 64 : 128;  // S columns one thread handles per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + TILE_BYTES;                  // [NST] K / P slots
  uint8_t* sV = sK + NST * TILE_BYTES;              // [NST] V slots
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + NST * TILE_BYTES);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + NST;
  uint64_t* kv_empty = v_full + NST;
  uint64_t* s_full = kv_empty + NST;  // [2]
  uint64_t* p_full = s_full + 2;      // [2]
  uint64_t* o_done = p_full + 2;      // [2]: PV(j) completes o_done[j & 1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Unit w = decode(a, sq, blockIdx.x);
  const int T = n_tiles_of(w);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
    }
    mbar_init(&o_done[0], 1);
    mbar_init(&o_done[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_kv = policy_evict_first();
    const uint64_t pol_q = policy_evict_first();
    // The whole warp runs the loop: lane 0 takes the waits and issues the
    // contiguous tile's boxes; on a paged cache lane i < 128 / P issues the
    // boxes of the tile's i-th page, its block-table entry read by the warp
    // 32 entries at a time (entries past the sequence or out of range read
    // page 0: keys the masks drop).
    const int P = a.page_size;
    const int npt = a.block_table != nullptr ? BKEY / P : 0;  // pages per tile
    const int* bt = a.block_table != nullptr ? a.block_table + (size_t)w.b * a.bt_stride
                                             : nullptr;
    int bt_base = -(1 << 30), my_page = 0;  // lane l holds entry bt_base + l
    auto load_kv = [&](int j) {
      const int s = j % NST;
      const int k0 = tile_start(w, j);
      int page = 0;
      if (bt != nullptr) {
        const int slot0 = k0 / P;
        if (slot0 < bt_base || slot0 + npt > bt_base + 32) {
          bt_base = slot0;
          const int e = bt_base + lane;
          my_page = e < a.bt_stride ? __ldg(bt + e) : 0;
          if (my_page < 0 || my_page >= a.n_pages) {
            // a page holding keys of the sequence must be a page of the cache
            if (e * P < w.len && e < a.bt_stride) record_error(a.err, 4 /* DFLASH_DEV_SLOT */);
            my_page = 0;
          }
        }
        page = __shfl_sync(0xffffffffu, my_page, min(slot0 - bt_base + lane, 31));
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&k_full[s], TILE_BYTES);
        mbar_arrive_expect_tx(&v_full[s], TILE_BYTES);
      }
      __syncwarp();
      if (bt == nullptr) {
        if (lane == 0) {
          const int y = (int)(w.kv_row0 + k0);
          tma_load_2d(sK + s * TILE_BYTES, &tmK, &k_full[s], 0, y, pol_kv);
          tma_load_2d(sK + s * TILE_BYTES + HALF_BYTES, &tmK, &k_full[s], 64, y, pol_kv);
          tma_load_2d(sV + s * TILE_BYTES, &tmV, &v_full[s], 0, y, pol_kv);
          tma_load_2d(sV + s * TILE_BYTES + HALF_BYTES, &tmV, &v_full[s], 64, y, pol_kv);
        }
      } else if (lane < npt) {
        const int y = (page * a.n_kv + w.h) * P;
        const uint32_t off = (uint32_t)(lane * P * 128);
        tma_load_2d(sK + s * TILE_BYTES + off, &tmK, &k_full[s], 0, y, pol_kv);
        tma_load_2d(sK + s * TILE_BYTES + HALF_BYTES + off, &tmK, &k_full[s], 64, y, pol_kv);
        tma_load_2d(sV + s * TILE_BYTES + off, &tmV, &v_full[s], 0, y, pol_kv);
        tma_load_2d(sV + s * TILE_BYTES + HALF_BYTES + off, &tmV, &v_full[s], 64, y, pol_kv);
      }
    };
    // Tiles made only of rows that were in the cache before this call were
    // written by kernels that have completed (every kernel here starts its
    // successor only after its own dependency wait): they fill the first
    // stages while the previous kernel (the one appending this call's rows
    // and writing Q) finishes.  The block table is the caller's input, in
    // place before the first kernel of the call.
    int pre = 0;
    {
      const int first_new = sq.first_new[w.b];
      for (; pre < T && pre < NST; ++pre) {
        if (tile_start(w, pre) + BKEY > first_new) break;
        load_kv(pre);
      }
    }
    grid_dep_wait();
    // A unit with no keys loads no Q either: nothing would wait for the copy,
    // and its softmax warps reuse the Q tile's shared memory to hand over
    // their (empty) row statistics, which a late TMA write would overwrite.
    if (lane == 0 && T > 0) {
      mbar_arrive_expect_tx(q_full, TILE_BYTES);
      if (DUAL) {  // the 64 query rows twice: smem rows 0..63 and 64..127
        for (int copy = 0; copy < 2; ++copy)
          for (int hf = 0; hf < 2; ++hf)
            tma_load_2d(sQ + hf * HALF_BYTES + copy * 64 * 128, &tmQ, q_full, 64 * hf,
                        w.q_row0, pol_q);
      } else {
        tma_load_2d(sQ, &tmQ, q_full, 0, w.q_row0, pol_q);
        tma_load_2d(sQ + HALF_BYTES, &tmQ, q_full, 64, w.q_row0, pol_q);
      }
    }
    for (int j = pre; j < T; ++j) {
      const int s = j % NST;
      const uint32_t ph = (j / NST) & 1;
      const bool ok = lane == 0 ? mbar_wait(&kv_empty[s], ph ^ 1, abort_flag, a.err) : true;
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      load_kv(j);
    }
    // Only once this CTA's last K/V tile has landed may the next kernel
    // start: its CTAs, on the SMs this grid leaves free, begin by streaming
    // their weights, and those copies would otherwise compete with our
    // tiles for HBM.  (Still after our own wait, as every kernel here.)
    if (T > 0 && lane == 0) {
      const int s = (T - 1) % NST;
      const uint32_t ph = ((T - 1) / NST) & 1;
      if (mbar_wait(&k_full[s], ph, abort_flag, a.err)) mbar_wait(&v_full[s], ph, abort_flag, a.err);
    }
    __syncwarp();
    grid_dep_launch();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    grid_dep_wait();
    if (lane == 0 && T > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, BKEY, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, HD, true);
      const uint32_t q_base = smem_u32(sQ);
      bool alive = mbar_wait(q_full, 0, abort_flag, a.err);
      auto issue_s = [&](int j) {
        const int s = j % NST;
        if (!mbar_wait(&k_full[s], (j / NST) & 1, abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t k_base = smem_u32(sK + s * TILE_BYTES);
        const uint32_t d_col = tmem + (uint32_t)((j & 1) * BKEY);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * HALF_BYTES + (kk & 3) * 32;
          tc_mma_bf16(d_col, sdesc_sw128(q_base + off, 16, 1024),
                      sdesc_sw128(k_base + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[j & 1]);
        return true;
      };
      if (alive) alive = issue_s(0);
      for (int j = 0; j < T && alive; ++j) {
        if (j + 1 < T && !issue_s(j + 1)) break;
        if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1, abort_flag, a.err)) break;
        const int s = j % NST;
        if (!mbar_wait(&v_full[s], (j / NST) & 1, abort_flag, a.err)) break;
        tc_fence_after();
        const uint32_t p_base = smem_u32(sK + s * TILE_BYTES);
        const uint32_t v_base = smem_u32(sV + s * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < BKEY / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(p_base + (kk >> 2) * HALF_BYTES + (kk & 3) * 32,
                                          16, 1024);
          const uint64_t bd = sdesc_sw128(v_base + kk * 16 * 128, HALF_BYTES, 1024);
          tc_mma_bf16(tmem + O_COL, ad, bd, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&o_done[j & 1]);
        tc_commit(&kv_empty[s]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int q = warp & 3;
    const int r = q * 32 + lane;                // TMEM lane (accumulator row)
    const int qr = DUAL ? (r & 63) : r;         // query row of the tile
    const int col0 = DUAL ? (r >> 6) * 64 : 0;  // first S column of this thread
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    const bool real = qr < w.rows;
    // this row's allowed keys: the unit's range, on a band layer cut to
    // |query index - key| < W, on a causal layer to keys <= the query index
    // (the query's index is len - q_len + t)
    int i1_lo = 0, i1_hi = 0;
    int out_token = 0, out_col = 0;
    {
      const int gi = qr / a.q_block;
      const int t = qr - gi * a.q_block;
      out_col = (w.h * a.groups + gi) * HD;
      out_token = w.b * a.q_len + t;
      i1_lo = w.s0_lo;
      i1_hi = w.s0_hi;
      const int qi = w.len - a.q_len + t;  // the row's own key index
      if (a.window > 0) {
        i1_lo = max(i1_lo, qi - a.window + 1);
        i1_hi = min(i1_hi, qi + a.window);
      }
      if (a.causal) i1_hi = min(i1_hi, qi + 1);
    }
    float m_run = -INFINITY, l_run = 0.f;
    // Pass -1 runs the tile body on whatever the S and O columns hold, with
    // every wait, store and state update left out and through the masking
    // and rescaling branches, before the dependency wait: the body's
    // instructions reach this SM's instruction cache while the previous
    // kernel finishes, instead of being fetched piece by piece during the
    // real tiles (its start is opaque to the compiler so that the pass stays
    // the same code as the real tiles).
    int j_first;
    asm volatile("mov.s32 %0, -1;" : "=r"(j_first));
    for (int jj = j_first; jj < T; ++jj) {
      const bool warm = jj < 0;
      const int j = warm ? 0 : jj;
      const int sb = j & 1;
      if (!__all_sync(0xffffffffu,
                      warm || mbar_wait(&s_full[sb], (j >> 1) & 1, abort_flag, a.err)))
        break;
      tc_fence_after();
      float s[NC];
      {
        uint32_t raw[NC / 32][32];
#pragma unroll
        for (int c = 0; c < NC / 32; ++c)
          tmem_ld32_nowait(trow + sb * BKEY + col0 + c * 32, raw[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < NC / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(raw[c][i]);
      }
      float alpha = 1.f;
      bool rescale = false;
      if (real) {
        const int k0 = tile_start(w, j) + col0;
        if (warm || !(k0 >= i1_lo && k0 + NC <= i1_hi)) {
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const int key = k0 + c;
            if (!(key >= i1_lo && key < i1_hi)) s[c] = -INFINITY;
          }
        }
        // row max and row sum as 8 interleaved partial chains (a single
        // chain over NC columns is a latency chain of NC dependent ops)
        // (three-input max: chain e takes columns e, e+8, e+16, ...)
        float pmax[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          pmax[e] = s[e];
#pragma unroll
          for (int k = 1; k < NC / 8; k += 2)
            pmax[e] = k + 1 < NC / 8 ? max3f(pmax[e], s[e + 8 * k], s[e + 8 * (k + 1)])
                                     : fmaxf(pmax[e], s[e + 8 * k]);
        }
        const float tmax = fmaxf(fmaxf(fmaxf(pmax[0], pmax[1]), fmaxf(pmax[2], pmax[3])),
                                 fmaxf(fmaxf(pmax[4], pmax[5]), fmaxf(pmax[6], pmax[7])));
        float m_new = m_run;
        if (m_run == -INFINITY || tmax > m_run + kRescaleThreshold) m_new = fmaxf(m_run, tmax);
        if (m_new != m_run) {
          alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
          rescale = j > 0;
        }
        const float mm = (m_new == -INFINITY) ? 0.f : m_new;
        // exponentials with paired fp32 subtract and sum
        const float2 neg_m = make_float2(-mm, -mm);
        float2 psum[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) psum[e] = make_float2(0.f, 0.f);
        uint8_t* prow = sK + (j % NST) * TILE_BYTES + r * 128;
        // this thread's NC columns are 16-byte chunks col0/8 .. col0/8+NC/8-1
        // of its P row (one 64-key atom per half); in dual mode the other
        // half of the row is zero
#pragma unroll
        for (int cc = 0; cc < NC / 8; ++cc) {
          float pv[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 d =
                add_f32x2(make_float2(s[cc * 8 + 2 * e], s[cc * 8 + 2 * e + 1]), neg_m);
            pv[2 * e] = fast_exp2(d.x);
            pv[2 * e + 1] = fast_exp2(d.y);
            psum[e] = add_f32x2(psum[e], make_float2(pv[2 * e], pv[2 * e + 1]));
          }
          uint4 pk;
          pk.x = pack_bf16x2(pv[0], pv[1]);
          pk.y = pack_bf16x2(pv[2], pv[3]);
          pk.z = pack_bf16x2(pv[4], pv[5]);
          pk.w = pack_bf16x2(pv[6], pv[7]);
          const int ch = col0 / 8 + cc;
          if (!warm)
            *reinterpret_cast<uint4*>(prow + (ch >> 3) * HALF_BYTES +
                                      (((ch & 7) ^ (r & 7)) * 16)) = pk;
        }
        if constexpr (DUAL) {
          const int other = col0 == 0 ? 1 : 0;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            if (!warm)
              *reinterpret_cast<uint4*>(prow + other * HALF_BYTES + ((cc ^ (r & 7)) * 16)) =
                  make_uint4(0u, 0u, 0u, 0u);
        }
        const float sum = ((psum[0].x + psum[0].y) + (psum[1].x + psum[1].y)) +
                          ((psum[2].x + psum[2].y) + (psum[3].x + psum[3].y));
        if (!warm) {
          l_run = l_run * alpha + sum;
          m_run = m_new;
        }
      }
      // O is touched only to rescale it, and only then must PV(j-1) be
      // complete.  Having seen S(j) complete, PV(j-2) and everything before
      // it are (one thread issues all MMAs, in order), so o_done[(j-1) & 1]
      // has at most the phase of PV(j-1) pending and a parity wait is exact.
      if (__any_sync(0xffffffffu, rescale) || warm) {
        if (!warm && !__all_sync(0xffffffffu, mbar_wait(&o_done[(j - 1) & 1],
                                                        ((j - 1) >> 1) & 1, abort_flag, a.err)))
          break;
        tc_fence_after();
        const float f = rescale ? alpha : 1.f;
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          float o[32];
          tmem_ld32(trow + O_COL + c * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          if (!warm) tmem_st32(trow + O_COL + c * 32, o);
        }
      }
      if (warm) {
        grid_dep_wait();
        continue;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[sb]);
    }
    // ------------------------------------------------------------ finish
    bool have_o = __all_sync(0xffffffffu, T > 0 && !*abort_flag);
    if (have_o) {
      have_o = __all_sync(0xffffffffu, mbar_wait(&o_done[(T - 1) & 1], ((T - 1) >> 1) & 1,
                                                 abort_flag, a.err));
      tc_fence_after();
    }
    float o[HD];
    {
      uint32_t raw[HD / 32][32];
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) tmem_ld32_nowait(trow + O_COL + c * 32, raw[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < HD / 32; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c * 32 + i] = have_o ? __uint_as_float(raw[c][i]) : 0.f;
    }
    if constexpr (DUAL) {
      // lanes 64..127 hand their half (keys 64..127 of every tile) to lanes
      // 0..63 through shared memory (K slot 0 and the Q tile are idle now)
      float4* xo = reinterpret_cast<float4*>(sK);
      float* xm = reinterpret_cast<float*>(sQ);
      if (r >= 64) {
#pragma unroll
        for (int c4 = 0; c4 < HD / 4; ++c4)
          xo[qr * 32 + (c4 ^ (qr & 31))] =
              make_float4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
        xm[qr] = m_run;
        xm[64 + qr] = l_run;
      }
      named_bar_sync(1, 128);
      if (r < 64) {
        const float mb = xm[qr], lb = xm[64 + qr];
        const float M = fmaxf(m_run, mb);
        const float fa = m_run == -INFINITY ? 0.f : fast_exp2(m_run - M);
        const float fb = mb == -INFINITY ? 0.f : fast_exp2(mb - M);
#pragma unroll
        for (int c4 = 0; c4 < HD / 4; ++c4) {
          const float4 t = xo[qr * 32 + (c4 ^ (qr & 31))];
          o[4 * c4] = fa * o[4 * c4] + fb * t.x;
          o[4 * c4 + 1] = fa * o[4 * c4 + 1] + fb * t.y;
          o[4 * c4 + 2] = fa * o[4 * c4 + 2] + fb * t.z;
          o[4 * c4 + 3] = fa * o[4 * c4 + 3] + fb * t.w;
        }
        l_run = fa * l_run + fb * lb;
        m_run = M;
      }
    }
    const bool writer = real && (!DUAL || r < 64);
    const int et = threadIdx.x - 64;
    if (a.cluster > 1 && a.k_clusters == 1) {
      // a split, and the pair's splits are the C CTAs of one cluster: the
      // unnormalised partial rows stay in this CTA's V stages (idle: the last
      // PV has completed and no copy is in flight); after one barrier each
      // rank merges its share of the rows from the C CTAs' shared memory, in
      // rank order, and a second barrier keeps every CTA resident until the
      // others have read its rows
      const int C = a.cluster;
      const int rank = w.c % C;
      if (writer) write_partial_smem(sV, qr, o, m_run, l_run);
      __syncwarp();
      cluster_sync();
      const int rpo = (w.rows + C - 1) / C;
      const int r0 = min(w.rows, rank * rpo), r1 = min(w.rows, r0 + rpo);
      merge_rows_cluster(a, w, smem_u32(sV), C, r0, r1, et);
      __syncwarp();
      cluster_sync();
    } else if (w.ns == 1) {
      // the unit covers every key of its rows: the normalised row
      if (writer) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const int ld_out = a.n_kv * a.groups * HD;
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                              (size_t)out_token * ld_out + out_col);
#pragma unroll
        for (int i = 0; i < HD / 8; ++i) {
          uint4 pk;
          pk.x = pack_bf16x2(o[8 * i] * inv, o[8 * i + 1] * inv);
          pk.y = pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
          pk.z = pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
          pk.w = pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
          dst[i] = pk;
        }
      }
    } else {
      // a split: the unnormalised partial rows go to the unit's slot, then
      // the rows are merged over the pair's splits
      if (writer) write_partial(a, (int)blockIdx.x, qr, o, m_run, l_run);
      if (a.cluster > 1) {
        // k clusters per pair: after one barrier each rank merges its share
        // of the rows from its cluster's C slots (through L2) into a block
        // slot, and the last cluster to finish a row block merges the
        // clusters' blocks
        __syncwarp();
        cluster_sync();
        const int C = a.cluster;
        const int rank = w.c % C, cl = w.c / C;
        const int rpo = (w.rows + C - 1) / C;
        const int r0 = min(w.rows, rank * rpo), r1 = min(w.rows, r0 + rpo);
        merge_rows(a, w, w.pair_unit0 + cl * C, 1, C, r0, r1, a.n_units + (int)blockIdx.x, et);
        int* cnt = a.counters + ((size_t)(w.b * a.n_kv + w.h) * C + rank);
        if (last_arrival(cnt, a.k_clusters, et, last_flag))
          merge_rows(a, w, a.n_units + w.pair_unit0 + rank, C, a.k_clusters, r0, r1, -1, et);
      } else if (last_arrival(a.counters + (w.b * a.n_kv + w.h), w.ns, et, last_flag)) {
        // the pair's last split to finish merges all of its rows
        merge_rows(a, w, w.pair_unit0, 1, w.ns, 0, w.rows, -1, et);
      }
    }
  }
  if (warp < 2 && a.cluster > 1) {
    // the producer and MMA warps take part in the cluster barriers
    __syncwarp();
    cluster_sync();
    if (a.k_clusters == 1) cluster_sync();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- packed, 2 Q tiles
// Packed training layout ("nemo_automodel...draft_qwen3", module docstring:
// a block sees the context strictly before its anchor and its own block).
// One CTA takes two Q tiles of the same (sequence, kv head) -- 2 x tile_blocks
// consecutive blocks -- and streams their common key range once:
// [0, largest anchor of its blocks) and the blocks' own rows.  Each K/V tile
// then feeds twice the tensor work, and the two softmax warpgroups take
// turns: while one works on its tile the tensor core runs the other's MMAs.
//
//   warp 0      TMA producer: Q0, Q1 once; K and V tiles of 128 keys into a
//               2-stage ring (K and V slots free separately)
//   warp 1      TMEM allocator + MMA issuer, per key tile j:
//                 PV0(j-1), S0(j), PV1(j-1), S1(j) (S_i(j) waits for the
//                 softmax of tile j-1 of Q tile i; PV_i(j-1) for its P)
//   warps 2-5   softmax of Q tile 0, one TMEM lane (row) per thread
//   warps 6-9   softmax of Q tile 1
// TMEM: S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512).  P_i(j) goes
// into the first 64 columns of S_i as bf16 pairs (S_i(j) is already in
// registers) and is the TMEM A operand of PV_i(j).  Because S_i(j+1) is
// issued after PV_i(j), seeing S_i(j+1) complete means PV_i(j) is complete:
// a rescale of O_i never waits.
constexpr int PK_NST = 2;
constexpr int PK_THREADS = 320;
constexpr size_t PK_SMEM = 1024 + TILE_BYTES * (2 + 2 * PK_NST) + 512;

struct PkUnit {
  int b, h, blk0;
  int rows[2];        // real query rows of Q tile 0 / 1
  int q_row0;         // first row of Q tile 0 in the Q buffer
  int s0_hi;          // context keys [0, s0_hi)
  int s1_lo, s1_hi;   // the blocks' own keys
  long long kv_row0;
};

DF_DEV PkUnit pk_decode(const AttnArgs& a, int u) {
  PkUnit w;
  const int rpb = a.groups * a.q_block;
  const int per_unit = 2 * a.tile_blocks;
  const int n_pu = (a.n_blocks + per_unit - 1) / per_unit;
  const int per = a.batch * a.n_kv;
  const int p_rev = u / per;
  const int rem = u - p_rev * per;
  w.b = rem / a.n_kv;
  w.h = rem - w.b * a.n_kv;
  const int p = n_pu - 1 - p_rev;  // latest anchors (longest key ranges) first
  w.blk0 = p * per_unit;
  const int nb = min(per_unit, a.n_blocks - w.blk0);
  const int nb0 = min(a.tile_blocks, nb);
  w.rows[0] = nb0 * rpb;
  w.rows[1] = (nb - nb0) * rpb;
  w.q_row0 = ((w.b * a.n_kv + w.h) * a.n_blocks + w.blk0) * rpb;
  int amax = 0;
  for (int k = 0; k < nb; ++k) {
    int an = a.anchors[w.b * a.n_blocks + w.blk0 + k];
    an = min(max(an, 0), a.seq);
    amax = max(amax, an);
  }
  w.s0_hi = amax;
  w.s1_lo = a.seq + w.blk0 * a.q_block;
  w.s1_hi = w.s1_lo + nb * a.q_block;
  w.kv_row0 = ((long long)w.b * a.n_kv + w.h) * a.cap;
  return w;
}

DF_DEV int pk_tiles(const PkUnit& w) {
  return (w.s0_hi + BKEY - 1) / BKEY + (w.s1_hi - w.s1_lo + BKEY - 1) / BKEY;
}

DF_DEV int pk_tile_start(const PkUnit& w, int j) {
  const int n0 = (w.s0_hi + BKEY - 1) / BKEY;
  return j < n0 ? j * BKEY : w.s1_lo + (j - n0) * BKEY;
}

__global__ void __launch_bounds__(PK_THREADS, 1)
    attn_pk2_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                              // [2] Q tiles
  uint8_t* sK = smem + 2 * TILE_BYTES;             // [PK_NST]
  uint8_t* sV = sK + PK_NST * TILE_BYTES;          // [PK_NST]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + PK_NST * TILE_BYTES);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* v_full = k_full + PK_NST;
  uint64_t* k_empty = v_full + PK_NST;
  uint64_t* v_empty = k_empty + PK_NST;
  uint64_t* s_full = v_empty + PK_NST;  // [2] per Q tile
  uint64_t* p_full = s_full + 2;        // [2]
  uint64_t* o_done = p_full + 2;        // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PkUnit w = pk_decode(a, blockIdx.x);
  const int T = pk_tiles(w);
  const int nqt = w.rows[1] > 0 ? 2 : 1;  // Q tiles with rows

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < PK_NST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    grid_dep_sync();
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_last();
      const uint64_t pol_q = policy_evict_first();
      mbar_arrive_expect_tx(q_full, (uint32_t)nqt * TILE_BYTES);
      for (int i = 0; i < nqt; ++i)
        for (int hf = 0; hf < 2; ++hf)
          tma_load_2d(sQ + i * TILE_BYTES + hf * HALF_BYTES, &tmQ, q_full, 64 * hf,
                      w.q_row0 + i * a.tile_blocks * a.groups * a.q_block, pol_q);
      for (int j = 0; j < T; ++j) {
        const int s = j % PK_NST;
        const uint32_t ph = ((j / PK_NST) & 1) ^ 1;
        const int y = (int)(w.kv_row0 + pk_tile_start(w, j));
        if (!mbar_wait(&k_empty[s], ph, abort_flag, a.err)) break;
        mbar_arrive_expect_tx(&k_full[s], TILE_BYTES);
        tma_load_2d(sK + s * TILE_BYTES, &tmK, &k_full[s], 0, y, pol_kv);
        tma_load_2d(sK + s * TILE_BYTES + HALF_BYTES, &tmK, &k_full[s], 64, y, pol_kv);
        if (!mbar_wait(&v_empty[s], ph, abort_flag, a.err)) break;
        mbar_arrive_expect_tx(&v_full[s], TILE_BYTES);
        tma_load_2d(sV + s * TILE_BYTES, &tmV, &v_full[s], 0, y, pol_kv);
        tma_load_2d(sV + s * TILE_BYTES + HALF_BYTES, &tmV, &v_full[s], 64, y, pol_kv);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    grid_dep_sync();
    if (lane == 0 && T > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, BKEY, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, HD, true);
      bool alive = mbar_wait(q_full, 0, abort_flag, a.err);
      // S_i(j) = Q_i K(j)^T into S_i; the last Q tile's S frees the K slot
      auto issue_s = [&](int i, int j) {
        const int s = j % PK_NST;
        if (!mbar_wait(&k_full[s], (j / PK_NST) & 1, abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t q_base = smem_u32(sQ + i * TILE_BYTES);
        const uint32_t k_base = smem_u32(sK + s * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * HALF_BYTES + (kk & 3) * 32;
          tc_mma_bf16(tmem + (uint32_t)(i * BKEY), sdesc_sw128(q_base + off, 16, 1024),
                      sdesc_sw128(k_base + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[i]);
        if (i == nqt - 1) tc_commit(&k_empty[s]);
        return true;
      };
      // O_i += P_i(j) V(j), P_i(j) from TMEM; the last Q tile's PV frees V
      auto issue_pv = [&](int i, int j) {
        const int s = j % PK_NST;
        if (!mbar_wait(&p_full[i], j & 1, abort_flag, a.err)) return false;
        if (!mbar_wait(&v_full[s], (j / PK_NST) & 1, abort_flag, a.err)) return false;
        tc_fence_after();
        const uint32_t v_base = smem_u32(sV + s * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < BKEY / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(v_base + kk * 16 * 128, HALF_BYTES, 1024);
          tc_mma_bf16_ta(tmem + O_COL + (uint32_t)(i * HD), tmem + (uint32_t)(i * BKEY) + kk * 8,
                         bd, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&o_done[i]);
        if (i == nqt - 1) tc_commit(&v_empty[s]);
        return true;
      };
      for (int i = 0; i < nqt && alive; ++i) alive = issue_s(i, 0);
      for (int j = 0; j < T && alive; ++j) {
        for (int i = 0; i < nqt && alive; ++i) {
          alive = issue_pv(i, j);
          if (alive && j + 1 < T) alive = issue_s(i, j + 1);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    grid_dep_sync();
    const int i = (warp - 2) >> 2;  // Q tile of this warpgroup
    if (i < nqt && T > 0) {
      const int q = warp & 3;
      const int r = q * 32 + lane;  // TMEM lane = row of Q tile i
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
      const uint32_t s_col = trow + (uint32_t)(i * BKEY);
      const uint32_t o_col = trow + O_COL + (uint32_t)(i * HD);
      const bool real = r < w.rows[i];
      const int rpb = a.groups * a.q_block;
      const int kb = r / rpb;
      const int within = r - kb * rpb;
      const int gi = within / a.q_block;
      const int t = within - gi * a.q_block;
      const int blk = w.blk0 + i * a.tile_blocks + kb;
      int i1_hi = 0, i2_lo = 0, i2_hi = 0;
      if (real) {
        int an = a.anchors[w.b * a.n_blocks + blk];
        if (an < 0 || an > a.seq) {
          record_error(a.err, 3 /* DFLASH_DEV_ANCHOR */);
          an = min(max(an, 0), a.seq);
        }
        i1_hi = an;
        i2_lo = a.seq + blk * a.q_block;
        i2_hi = i2_lo + a.q_block;
      }
      const int n_ctx_tiles = (w.s0_hi + BKEY - 1) / BKEY;
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < T; ++j) {
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[i], j & 1, abort_flag, a.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[BKEY];
        {
          uint32_t raw[BKEY / 32][32];
#pragma unroll
          for (int c = 0; c < BKEY / 32; ++c) tmem_ld32_nowait(s_col + c * 32, raw[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < BKEY / 32; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(raw[c][e]);
        }
        // a context tile may run past the context into block rows, which
        // the own-block tile covers: each tile admits only its segment's keys
        const int k0 = pk_tile_start(w, j);
        const bool ctx_tile = j < n_ctx_tiles;
        const int lo = ctx_tile ? 0 : i2_lo, hi = ctx_tile ? i1_hi : i2_hi;
        if (!real || !(k0 >= lo && k0 + BKEY <= hi)) {
#pragma unroll
          for (int c = 0; c < BKEY; ++c) {
            const int key = k0 + c;
            if (!(real && key >= lo && key < hi)) s[c] = -INFINITY;
          }
        }
        // row max as 8 interleaved three-input chains
        float pmax[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          pmax[e] = s[e];
#pragma unroll
          for (int k = 1; k < BKEY / 8; k += 2)
            pmax[e] = k + 1 < BKEY / 8 ? max3f(pmax[e], s[e + 8 * k], s[e + 8 * (k + 1)])
                                       : fmaxf(pmax[e], s[e + 8 * k]);
        }
        const float tmax = fmaxf(fmaxf(fmaxf(pmax[0], pmax[1]), fmaxf(pmax[2], pmax[3])),
                                 fmaxf(fmaxf(pmax[4], pmax[5]), fmaxf(pmax[6], pmax[7])));
        float m_new = m_run, alpha = 1.f;
        if (m_run == -INFINITY || tmax > m_run + kRescaleThreshold) m_new = fmaxf(m_run, tmax);
        bool rescale = false;
        if (m_new != m_run) {
          alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
          rescale = j > 0;
        }
        const float mm = (m_new == -INFINITY) ? 0.f : m_new;
        // P(j) = exp2(S - m) as bf16 pairs over the first 64 columns of S_i
        const float2 neg_m = make_float2(-mm, -mm);
        float2 psum[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) psum[e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int p0 = 0; p0 < BKEY; p0 += 64) {
          uint32_t pw[32];
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            float pv[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = p0 + cc * 8 + 2 * e;
              const float2 d = add_f32x2(make_float2(s[c], s[c + 1]), neg_m);
              pv[2 * e] = fast_exp2(d.x);
              pv[2 * e + 1] = fast_exp2(d.y);
              psum[e] = add_f32x2(psum[e], make_float2(pv[2 * e], pv[2 * e + 1]));
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) pw[cc * 4 + e] = pack_bf16x2(pv[2 * e], pv[2 * e + 1]);
          }
          tmem_st32_nowait(s_col + (uint32_t)(p0 / 2), pw);
        }
        const float sum = ((psum[0].x + psum[0].y) + (psum[1].x + psum[1].y)) +
                          ((psum[2].x + psum[2].y) + (psum[3].x + psum[3].y));
        l_run = l_run * alpha + sum;
        m_run = m_new;
        // S_i(j) complete implies PV_i(j-1) complete: O_i may be rescaled
        if (__any_sync(0xffffffffu, rescale)) {
          const float f = rescale ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            float o[32];
            tmem_ld32(o_col + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= f;
            tmem_st32(o_col + c * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[i]);
      }
      // ---------------------------------------------------------- finish
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_done[i], (T - 1) & 1, abort_flag, a.err));
      tc_fence_after();
      // normalised O row, 32 columns at a time (warp-collective loads)
      const float inv = ok && l_run > 0.f ? 1.f / l_run : 0.f;
      const int ld_out = a.n_kv * a.groups * HD;
      const size_t token = (size_t)w.b * a.q_len + (size_t)blk * a.q_block + t;
      if (a.lse != nullptr && real)  // natural log of the row's normaliser (S in log2 units)
        a.lse[token * (a.n_kv * a.groups) + w.h * a.groups + gi] =
            ok && l_run > 0.f ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) +
                                            token * ld_out + (size_t)(w.h * a.groups + gi) * HD);
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        float o[32];
        tmem_ld32(o_col + c * 32, o);
        if (real) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 pk;
            pk.x = pack_bf16x2(o[8 * e] * inv, o[8 * e + 1] * inv);
            pk.y = pack_bf16x2(o[8 * e + 2] * inv, o[8 * e + 3] * inv);
            pk.z = pack_bf16x2(o[8 * e + 4] * inv, o[8 * e + 5] * inv);
            pk.w = pack_bf16x2(o[8 * e + 6] * inv, o[8 * e + 7] * inv);
            dst[c * 4 + e] = pk;
          }
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

}  // namespace

namespace {

void set_attn_attrs() {
  static std::atomic<unsigned long long> done{0};
  if (done_on_device(done)) return;
  for (const void* f : {(const void*)attn_bf16_kernel<true>, (const void*)attn_bf16_kernel<false>}) {
    cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  }
  cudaFuncSetAttribute(attn_pk2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)PK_SMEM);
  mark_device(done);
}

// clusters of `c` decode-attention CTAs that can be resident at once
int max_active_clusters(int c, bool dual) {
  static std::atomic<int> cache[2][9];  // the count + 1; 0: not asked yet
  const int known = cache[dual][c].load(std::memory_order_acquire);
  if (known != 0) return known - 1;
  set_attn_attrs();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const void* f =
      dual ? (const void*)attn_bf16_kernel<true> : (const void*)attn_bf16_kernel<false>;
  if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[dual][c].store(n + 1, std::memory_order_release);
  return n;
}

}  // namespace

size_t decode_attention_slots(int batch, int n_kv, int num_sms) {
  // balanced plans: at most 4 units per SM plus one per pair; cluster plans:
  // at most one unit per SM, twice (the clusters' merged row blocks)
  return (size_t)4 * num_sms + (size_t)batch * n_kv;
}

size_t decode_attention_counters(int batch, int n_kv) { return (size_t)batch * n_kv * 8; }

int plan_decode_attention(AttnSeqs& sq, int batch, int n_kv, int num_sms, bool dual,
                          int* cluster, int* k_clusters) {
  const int pairs = batch * n_kv;
  std::vector<int> np(batch);
  int max_np = 1;
  long long tot = 0;
  for (int b = 0; b < batch; ++b) {
    np[b] = std::max(1, (sq.len[b] - sq.lo[b] + BKEY - 1) / BKEY);
    max_np = std::max(max_np, np[b]);
    tot += (long long)n_kv * np[b];
  }
  *cluster = 1;
  *k_clusters = 1;
  // Estimated makespans in tile times (about 1.2 us each at the HBM share of
  // an SM): a unit costs its tiles plus two for its start; a split pair's
  // merge costs about one round trip to L2 per merged source (~0.5 tile) plus
  // the arrival, done by the last split alone; a cluster's merge is spread
  // over its ranks (about three tiles whatever C).  The weights are fitted to
  // the measured single-sequence, serving and long-context steps.
  //
  // Few pairs: C splits per cluster, k clusters per pair, every cluster
  // resident at once, about one unit per SM and at least two tiles per unit.
  int best_C = 0, best_k = 1;
  double t_cluster = 1e300;
  for (int C = 8; C >= 2; C >>= 1) {
    if ((long long)pairs * C > num_sms || C > max_np) continue;
    const int fit = max_active_clusters(C, dual) / pairs;
    if (fit < 1) continue;
    const int k = std::max(1, std::min({fit, num_sms / (pairs * C), max_np / (2 * C)}));
    // several clusters per pair add a second merge through L2 after the
    // cluster merge (measured: eight tile times more than one cluster)
    const double t = (double)((max_np + C * k - 1) / (C * k)) + 2.0 + 3.0 + (k > 1 ? 8.0 : 0.0);
    if (t < t_cluster - 1e-9) {
      t_cluster = t;
      best_C = C;
      best_k = k;
    }
  }
  // Many pairs: units of at most U tiles for about m units per SM, dispatched
  // largest first; list scheduling gives the makespan of each m.
  std::vector<int> best_ns(batch, 1), ns(batch);
  double best_t = 1e300;
  for (int m = 1; m <= 4; ++m) {
    const long long U = std::max<long long>(1, (tot + (long long)m * num_sms - 1) /
                                                   ((long long)m * num_sms));
    long long units = 0;
    for (int b = 0; b < batch; ++b) {
      ns[b] = (int)std::min<long long>({(np[b] + U - 1) / U, (long long)np[b], 32});
      units += (long long)n_kv * ns[b];
    }
    if (units > (long long)decode_attention_slots(batch, n_kv, num_sms)) continue;
    std::vector<std::pair<double, int>> groups(batch);
    for (int b = 0; b < batch; ++b)
      groups[b] = {(double)np[b] / ns[b] + 2.0 + (ns[b] > 1 ? 1.0 + 0.5 * ns[b] : 0.0), b};
    std::sort(groups.begin(), groups.end(), [](const auto& x, const auto& y) {
      return x.first > y.first || (x.first == y.first && x.second < y.second);
    });
    std::priority_queue<double, std::vector<double>, std::greater<double>> load;
    for (int i = 0; i < num_sms; ++i) load.push(0.0);
    double t = 0.0;
    for (const auto& g : groups)
      for (int i = 0; i < n_kv * ns[g.second]; ++i) {
        const double l = load.top() + g.first;
        load.pop();
        load.push(l);
        t = std::max(t, l);
      }
    if (t < best_t - 1e-9) {
      best_t = t;
      best_ns = ns;
    }
  }
  if (best_C > 0 && t_cluster <= best_t) {
    *cluster = best_C;
    *k_clusters = best_k;
    sq.unit_off[0] = 0;
    for (int b = 0; b < batch; ++b) {
      sq.n_split[b] = best_C * best_k;
      sq.order[b] = b;
      sq.unit_off[b + 1] = sq.unit_off[b] + n_kv * best_C * best_k;
    }
    return sq.unit_off[batch];
  }
  std::vector<std::pair<double, int>> order(batch);
  for (int b = 0; b < batch; ++b) {
    sq.n_split[b] = best_ns[b];
    order[b] = {(double)np[b] / best_ns[b], b};
  }
  std::sort(order.begin(), order.end(), [](const auto& x, const auto& y) {
    return x.first > y.first || (x.first == y.first && x.second < y.second);
  });
  sq.unit_off[0] = 0;
  for (int i = 0; i < batch; ++i) {
    sq.order[i] = order[i].second;
    sq.unit_off[i + 1] = sq.unit_off[i] + n_kv * best_ns[order[i].second];
  }
  return sq.unit_off[batch];
}

int launch_attn_bf16(const AttnArgs& a, const AttnSeqs* seqs, const void* qbuf,
                     long long q_rows_total, const void* cache_k,
                     const void* cache_v, long long kv_rows_total,
                     cudaStream_t stream) {
  set_attn_attrs();
  if (a.n_units <= 0) return cudaSuccess;
  if (a.cluster > 1 && (a.mode != 0 || a.cluster > 8 || a.n_units % a.cluster != 0))
    return cudaErrorInvalidValue;
  if (a.mode == 0 && (a.part_o == nullptr || a.part_ml == nullptr || a.counters == nullptr))
    return cudaErrorInvalidValue;
  if (kv_rows_total >= (1LL << 31) || q_rows_total >= (1LL << 31))
    return cudaErrorInvalidValue;
  if (a.mode == 1) {
    // packed layout: two Q tiles per CTA sharing one pass over the keys
    CUtensorMap mq, mk, mv;
    if (make_tmap_bf16_rows(&mq, qbuf, q_rows_total, HD, 128) != 0 ||
        make_tmap_bf16_rows(&mk, cache_k, kv_rows_total, HD, 128) != 0 ||
        make_tmap_bf16_rows(&mv, cache_v, kv_rows_total, HD, 128) != 0)
      return cudaErrorInvalidValue;
    const int per_unit = 2 * a.tile_blocks;
    const int units = a.batch * a.n_kv * ((a.n_blocks + per_unit - 1) / per_unit);
    return (int)launch_pdl(attn_pk2_kernel, dim3(units), dim3(PK_THREADS), PK_SMEM, stream, mq,
                           mk, mv, a);
  }
  const bool dual = a.mode == 0 && a.groups * a.q_len <= 64;
  const int kv_box = a.block_table != nullptr ? a.page_size : 128;
  if (a.block_table != nullptr && (kv_box < 16 || kv_box > 128 || (kv_box & (kv_box - 1)) != 0))
    return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  if (make_tmap_bf16_rows(&mq, qbuf, q_rows_total, HD, dual ? 64 : 128) != 0 ||
      make_tmap_bf16_rows(&mk, cache_k, kv_rows_total, HD, kv_box) != 0 ||
      make_tmap_bf16_rows(&mv, cache_v, kv_rows_total, HD, kv_box) != 0)
    return cudaErrorInvalidValue;
  static AttnSeqs zero_seqs{};
  const AttnSeqs& sq = seqs ? *seqs : zero_seqs;
  const unsigned cl = a.cluster > 1 ? (unsigned)a.cluster : 1u;
  cudaError_t e =
      dual ? launch_pdl_cluster(attn_bf16_kernel<true>, dim3(a.n_units), dim3(kThreads),
                                SMEM_BYTES, stream, cl, mq, mk, mv, a, sq)
           : launch_pdl_cluster(attn_bf16_kernel<false>, dim3(a.n_units), dim3(kThreads),
                                SMEM_BYTES, stream, cl, mq, mk, mv, a, sq);
  return (int)e;
}

}  // namespace df
