// internal.h -- structures shared by the host API and the kernels, and the
// host-side launchers each kernel file exports.
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace df {

constexpr int kMaxBatch = 512;
constexpr int kMaxGroupLayers = 16;  // layers of one context K/V group

// Per-sequence bookkeeping of one forward call, passed to kernels by value.
struct SeqTable {
  int n;                       // sequences
  int q_len;                   // block rows per sequence
  int ctx_off[kMaxBatch + 1];  // prefix sums of new context rows
  int cache_len[kMaxBatch];    // rows cached before this call
};

// Where the QKV projection epilogue puts its results.
struct QkvOut {
  int n_heads, n_kv, groups;
  int q_block;       // rows of one block inside the Q buffer layout
  int cap;           // key rows per (sequence, kv head) in the K/V storage
  int max_pos;
  float eps;
  float q_scale;     // head_dim^-0.5 * log2(e), folded into Q
  const int* positions;
  const float2* rope;      // [max_pos][head_dim/2] (cos, sin)
  const float* q_norm;     // [head_dim] fp32
  const float* k_norm;     // [head_dim] fp32
  void* qbuf;              // [B][n_kv][n_blocks][groups][q_block][d]
  void* cache_k;           // [B][n_kv][cap][d]
  void* cache_v;
  // paged cache: the row at positions index i goes to slot slot_mapping[i]
  // (page slot / P, row slot % P) of storage [n_pages][n_kv][P][d]; null:
  // contiguous cache
  const int* slot_mapping;
  int page_size;
  int n_pages;
  int* err;
  // layer group (context K/V of several layers from one GEMM, no Q columns):
  // n_layers > 0, columns [layer][K heads | V heads], every row a context row
  int n_layers;
  void* g_cache_k[kMaxGroupLayers];
  void* g_cache_v[kMaxGroupLayers];
  const float* g_k_norm[kMaxGroupLayers];
  int g_cap[kMaxGroupLayers];
};

// Per-device one-time set-up (kernel attributes): bit d of `mask` is set once
// the set-up has run on device d.
inline bool done_on_device(const std::atomic<unsigned long long>& mask) {
  int dev = 0;
  cudaGetDevice(&dev);
  return (mask.load(std::memory_order_acquire) >> (dev & 63)) & 1ull;
}
inline void mark_device(std::atomic<unsigned long long>& mask) {
  int dev = 0;
  cudaGetDevice(&dev);
  mask.fetch_or(1ull << (dev & 63), std::memory_order_release);
}

// Kernels this library has launched in this process (every launch site
// counts itself; read through dflash_kernel_launches).
extern std::atomic<unsigned long long> g_kernel_launches;
inline void count_launch() { g_kernel_launches.fetch_add(1, std::memory_order_relaxed); }

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream finishes; it must call grid_dep_wait()
// before touching memory that kernel writes or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
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
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with a 1-D thread-block cluster of `cluster_x` CTAs (1 = none).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster_x > 1 ? 2 : 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ----------------------------------------------------------- bf16 GEMM
// C = A * B^T with A [rows, K] (token rows; two sources A0 then A1) and B
// [N, K] (weights), both bf16 K-contiguous; fp32 accumulation on tcgen05.
// EPI_SWIGLU: the weight rows are gate and up rows interleaved in 64-row
// chunks; each 128-column tile yields 64 outputs silu(gate) * up, bf16, at
// column n0 / 2
enum GemmEpi { EPI_BF16 = 0, EPI_F32 = 1, EPI_QKV = 2, EPI_SWIGLU = 3 };

struct GemmShape {
  const void* a0; int a0_rows;   // noise rows (or the only source)
  const void* a1; int a1_rows;   // context rows (may be 0)
  const CUtensorMap* b_map;      // weights, 128-row boxes, built at create
  const CUtensorMap* b_map256;   // the same weights, 256-row boxes
  int n, k;
  int q_cols;                    // leading columns computed from A0 only
};

struct GemmScratch {
  float* partial = nullptr; size_t partial_bytes = 0;
  int* counters = nullptr; int n_counters = 0;
  // EPI_F32 only: 1 = every K split writes its fp32 partial to its own slice
  // of the output (c + split * slice_stride floats) instead of merging them;
  // gemm_f32_slices() gives the number of slices
  int f32_slices = 0;
  size_t slice_stride = 0;
};

int launch_gemm_bf16(const GemmShape& s, int epi, void* c, int ldc,
                     const QkvOut* qkv, const SeqTable* seqs,
                     const GemmScratch& scr, int num_sms, int* err,
                     cudaStream_t st);
size_t gemm_scratch_bytes(int epi, int rows0, int rows1, int n, int k, int q_cols,
                          int num_sms, int* n_counters);
// slices an EPI_F32 launch of one source of `rows` rows writes when
// GemmScratch::f32_slices is set (1: it merges its splits itself)
int gemm_f32_slices(int rows, int n, int k, int num_sms);
int make_tmap_bf16_rows(CUtensorMap* map, const void* ptr, long long rows,
                        int cols, int box_rows);

// ----------------------------------------------------------- attention
// Per-sequence key ranges and the work split of an inference attention call.
// Each (sequence, kv head) pair's keys [lo, len) form ceil((len - lo) / 128)
// tiles, split into n_split units of near-equal tile counts.  Units follow
// the sequences in `order` (largest units first), kv head-major then split.
struct AttnSeqs {
  int len[kMaxBatch];          // keys of the sequence after this call's append
  int lo[kMaxBatch];           // first key any query of the block can see
  int first_new[kMaxBatch];    // first row this call appends (rows below it
                               // were written by earlier calls)
  int n_split[kMaxBatch];      // units per (sequence, kv head), by sequence
  int order[kMaxBatch];        // sequences in unit order
  int unit_off[kMaxBatch + 1]; // first unit of the i-th sequence of `order`
};

struct AttnArgs {
  int mode;          // 0 = inference (cache), 1 = packed training
  int batch, n_kv, groups, head_dim;
  int q_len;         // query rows per sequence (all blocks)
  int q_block;       // rows per block (q_len for inference)
  int n_blocks;      // blocks per sequence (1 for inference)
  int tile_blocks;   // blocks per 128-row Q tile
  int cap;           // key rows per (sequence, head) in the K/V storage
  int window;        // sliding window (0 = full)
  int causal;        // inference: block row t sees keys up to its own index
  // paged cache: a sequence's key row k lives in page block_table[b][k / P]
  // at offset k % P of storage [n_pages][n_kv][P][d] (cap = P); null:
  // contiguous [B][n_kv][cap][d]
  const int* block_table;
  int bt_stride;     // entries per sequence in block_table
  int page_size;     // P (16, 32, 64 or 128; a power of two)
  int n_pages;
  float* lse;        // packed core: per query row log-sum-exp (natural log), or null
  int seq;           // packed: context rows per sequence
  const int* anchors;  // packed: [B][n_blocks]
  int n_units;
  int cluster;       // inference: C > 1 = every C consecutive splits of a pair
                     // form a thread-block cluster (n_split = C * k_clusters)
  int k_clusters;    // clusters per (sequence, kv head)
  float* part_o;     // [slot][128 rows][d] fp32 partial outputs (slot = unit;
                     // cluster mode also [n_units + unit]: merged row blocks)
  float* part_ml;    // [slot][2][128] running max (log2 units) and sum
  int* counters;     // split merges: [B * n_kv] or [B * n_kv * C], zero
                     // between calls (the last arriver resets its counter)
  void* out;         // [B*q_len][n_heads*d]
  int* err;
};

// Work split of a decode-attention call (fills n_split, order, unit_off of
// `sq` from its len and lo): returns the number of units and sets the
// cluster size C (1 = none) and the clusters per pair.  Few (sequence, kv
// head) pairs: C = 8 (or fewer) splits per cluster, k clusters per pair;
// otherwise units of near-equal tile counts, largest first, so that the
// hardware's in-order dispatch balances the SMs.
int plan_decode_attention(AttnSeqs& sq, int batch, int n_kv, int num_sms, bool dual,
                          int* cluster, int* k_clusters);
// partial slots and merge counters a plan with these sizes can need
size_t decode_attention_slots(int batch, int n_kv, int num_sms);
size_t decode_attention_counters(int batch, int n_kv);

int launch_attn_bf16(const AttnArgs& a, const AttnSeqs* seqs, const void* qbuf,
                     long long q_rows_total, const void* cache_k,
                     const void* cache_v, long long kv_rows_total,
                     cudaStream_t st);

// ----------------------------------------------------------- small kernels
int launch_rope_table(float2* tab, int max_pos, int half, float theta,
                      cudaStream_t st);
// out = w * x / rms(x) per row, x = z[0] + z[1] + ... (n_slices slices of
// slice_stride floats, summed in slice order)
int launch_row_rmsnorm(const float* z, int rows, int cols, const float* w,
                       float eps, void* out, int out_bf16, int n_slices,
                       size_t slice_stride, cudaStream_t st);
int launch_to_f32(const void* src, int src_bf16, float* dst, size_t n,
                  cudaStream_t st);
// sum_out = a + b (b may be null), norm_out = w * sum / rms(sum); bf16 rows,
// cols % 8 == 0, cols <= 8192; w fp32
int launch_add_rmsnorm(const void* a, const void* b, int rows, int cols, const float* w,
                       float eps, void* sum_out, void* norm_out, cudaStream_t st);
int launch_packed_positions(const int* anchors, int batch, int seq,
                            int n_blocks, int block_size, int* pos, int* err,
                            cudaStream_t st);

// one thread waits on an mbarrier for at most limit_ns (a never-completed
// barrier unless `arrive`); on expiry DFLASH_DEV_WAIT_TIMEOUT goes to `err`
int launch_wait_probe(int* err, unsigned long long limit_ns, int arrive, cudaStream_t st);
int launch_read_stream(const void* src, long long rows, long long cols, int ctas, int stages,
                       int* err, cudaStream_t st);

// ----------------------------------------------------------- fp32 path
int launch_gemm_f32(const float* a, int rows, const float* b, int n, int k,
                    float* c, int ldc, cudaStream_t st);
int launch_qkv_post_f32(const float* qkv_noise, int rows_noise,
                        const float* qkv_ctx, int rows_ctx, const QkvOut& o,
                        const SeqTable* seqs, int head_dim, int* err,
                        cudaStream_t st);
int launch_attn_f32(const AttnArgs& a, const AttnSeqs* seqs, const float* qbuf,
                    const float* k, const float* v, cudaStream_t st);

// Packed-layout attention backward (attn_bwd.cu).  Query-side tensors are
// in the tile layout [B][n_kv][n_blocks][groups][block][d] (one block = 64
// rows), K/V and their gradients [B][n_kv][per][d] (context rows, then every
// block's rows).
struct PackedBwdArgs {
  int batch, seq, n_blocks, block_size, n_kv, groups;
  int per;                 // key rows per (sequence, kv head)
  const int* anchors;      // [B][n_blocks]
  const float* lse2;       // tile rows: minus the log-sum-exp in log2 units
  const float* dsum;       // tile rows: minus rowsum(dO * O)
  void* dq;                // [B][n_blocks * block][n_heads][d] bf16
  void* dk;
  void* dv;
  float dq_scale;          // softmax scale
  const void* qs;          // Q' (tile layout, bf16)
  const void* do_tile;     // dO (tile layout, bf16)
  int n_kv_ctx_units;      // dK/dV units over context key tiles
  int kv_group;            // (sequence, kv head) pairs whose units are dispatched together,
                           // so that their Q'/dO and K/V stay in L2 for every kind of CTA
  int n_q_units;           // dQ units
  int n_kv_own_units;      // dK/dV units over the blocks' own keys
  int* err;
};

// q (token-major [B][T][n_heads][d]) -> qs (tile layout, times c); with d_o
// and o: d_o -> do_tile, -rowsum(d_o * o) -> dsum, -lse * log2(e) -> lse2
// (tile rows).  d_o, o, lse and their outputs are null together.
cudaError_t launch_packed_prep(const void* q, const void* d_o, const void* o, const float* lse,
                               int batch, int n_blocks, int block_size, int n_kv, int groups,
                               float c, void* qs, void* do_tile, float* dsum, float* lse2,
                               cudaStream_t stream);
// dK/dV and dQ in one launch (units of both kinds); tensors as in PackedBwdArgs
cudaError_t launch_packed_bwd(const PackedBwdArgs& a, const void* qs, const void* do_tile,
                              const void* k, const void* v, cudaStream_t stream);

}  // namespace df
