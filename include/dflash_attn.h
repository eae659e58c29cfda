/*
 * dflash_attn.h -- C ABI of the GB300 DFlash draft attention library
 * (libdflash_attn.so).
 *
 * One draft attention layer of a DFlash block-diffusion drafter
 * (Qwen3DFlashAttention): queries from a block of noise tokens (one anchor
 * plus mask tokens), keys and values from the projected target-model context
 * followed by the block, per-head q/k RMSNorm, RoPE over the
 * [context | block] window, grouped KV heads, non-causal softmax (optionally
 * a symmetric sliding-window band), o_proj, and a draft KV cache that is
 * cropped back to the accepted prefix after verification.  Around it: the
 * context K/V of several layers from one projection, the rest of the draft
 * decoder layer (norms, residual stream, SwiGLU MLP), a paged cache with a
 * slot mapping and block tables, causal layers, and the attention core of
 * the packed training layout with its backward.
 *
 * Page citations name the page by title and the section or symbol on it:
 *   [P3] "DFlash源码导读（二）：Qwen3DFlashAttention注意力实现全解析"
 *   [P4] "nemo_automodel.components.speculative.dflash.draft_qwen3"
 *   [P5] "vllm.model_executor.models.qwen3_dflash"
 *
 * Conventions for every call:
 *  - Every entry point returns an int status: DFLASH_OK (0) or a negative
 *    DFLASH_ERR_* code; dflash_last_error() then returns a message for the
 *    calling thread.  No C++ exception crosses this boundary.
 *  - Arguments are checked on the host before anything is enqueued.  A call
 *    that fails a check enqueues no work and leaves every object unchanged.
 *  - "device" pointers are CUDA device memory of the device that was current
 *    when the layer was created; "host" pointers are ordinary CPU memory that
 *    is read only during the call.  The caller owns every pointer it passes.
 *    Device tensors handed to a bf16 layer must start on a 16-byte boundary.
 *  - Tensors are dense, row-major, in the layer's dtype (DFLASH_BF16 or
 *    DFLASH_FP32) unless stated otherwise; integer tensors are int32.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously; outputs are valid once the stream has
 *    reached that point.
 *  - Handles are not thread-safe: one thread (or external locking) per layer
 *    handle and per cache at a time.  One layer's calls share its scratch, so
 *    calls of one layer must not run concurrently on different streams.
 *  - Faults found on the device (a position outside [0, max_position), an
 *    anchor outside [0, seq], a paged-cache slot or block-table entry outside
 *    the cache, a bounded wait that ran out) do not stop the kernels: the
 *    offending value is clamped or the access skipped, a code is recorded in
 *    the layer's device error word, and dflash_device_error() reports it.
 */
#ifndef DFLASH_ATTN_H
#define DFLASH_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dflash_attn dflash_attn;   /* one layer: weights + scratch */
typedef struct dflash_cache dflash_cache; /* one draft KV cache */
typedef struct dflash_kv_group dflash_kv_group; /* context K/V of several layers */
typedef struct dflash_mlp dflash_mlp;     /* norms + MLP of a decoder layer */
typedef struct dflash_paged_cache dflash_paged_cache; /* paged KV storage */
typedef void* dflash_stream;              /* a cudaStream_t */

enum {
  DFLASH_OK = 0,
  DFLASH_ERR_ARG = -1,         /* null pointer, bad enum, non-positive size  */
  DFLASH_ERR_SHAPE = -2,       /* sizes inconsistent with the layer/cache    */
  DFLASH_ERR_CAPACITY = -3,    /* cache rows would exceed its capacity       */
  DFLASH_ERR_RANGE = -4,       /* crop length above the current length, ...  */
  DFLASH_ERR_CUDA = -5,        /* a CUDA runtime call failed                 */
  DFLASH_ERR_DEVICE = -6,      /* a kernel recorded a device-side fault      */
  DFLASH_ERR_UNSUPPORTED = -7, /* valid request the library does not handle */
  DFLASH_ERR_MEMORY = -8       /* device allocation failed                   */
};

enum { DFLASH_BF16 = 0, DFLASH_FP32 = 1 };

/* Device-side fault codes reported by dflash_device_error(). */
enum {
  DFLASH_DEV_OK = 0,
  DFLASH_DEV_WAIT_TIMEOUT = 1, /* a pipeline wait gave up (kernel returned)  */
  DFLASH_DEV_POSITION = 2,     /* position outside [0, max_position)         */
  DFLASH_DEV_ANCHOR = 3,       /* anchor outside [0, seq]                    */
  DFLASH_DEV_SLOT = 4          /* paged cache: a slot outside the cache (the
                                  row was not written), or a block-table entry
                                  of a page holding the sequence's keys outside
                                  the cache (page 0 read in its place)        */
};

/* Layer scalars.  [P3] step 1: head_dim is the explicit value, else
 * hidden / n_heads; num_key_value_groups = n_heads / n_kv_heads.
 * [P4] Qwen3DFlashAttention: scaling = head_dim^-0.5; sliding_window only on
 * sliding-attention layers ([P3] step 5).  [P5] DFlashQwen3Model: fc takes
 * n_target_layers * hidden concatenated features. */
typedef struct {
  int32_t hidden;          /* H                                              */
  int32_t n_heads;         /* query heads                                    */
  int32_t n_kv_heads;      /* key/value heads; divides n_heads               */
  int32_t head_dim;        /* d; 0 -> hidden / n_heads                       */
  int32_t n_target_layers; /* fc input width = n_target_layers * hidden; 0 = no fc */
  float rms_eps;           /* eps of q_norm, k_norm and hidden_norm          */
  float rope_theta;        /* RoPE base                                      */
  int32_t sliding_window;  /* 0 = full attention; W > 0 keeps keys with
                              |query key index - key index| < W ([P4]
                              _sliding_window_mask)                          */
  int32_t max_position;    /* positions must lie in [0, max_position);
                              0 -> 131072                                    */
  int32_t dtype;           /* DFLASH_BF16 or DFLASH_FP32                     */
  int32_t causal;          /* 1: block row t sees the keys at or before its
                              own key index (every cached and context row,
                              block rows 0..t), with the band on sliding
                              layers ([P5] _dflash_layer_causal); 0: the
                              block is bidirectional.  Inference only: the
                              packed training forward is _UNSUPPORTED on a
                              causal layer                                   */
} dflash_attn_config;

/* Message for the last failed call on this thread ("" if none). */
const char* dflash_last_error(void);

/* ABI version of this header (major * 100 + minor): 105. */
int dflash_abi_version(void);

/* Create one layer on the current CUDA device.
 * [P4] Qwen3DFlashAttention members q_proj, k_proj, v_proj, o_proj, q_norm,
 * k_norm; [P5] DFlashQwen3Attention (no biases); [P5] DFlashQwen3Model fc and
 * hidden_norm.
 *   wq [n_heads*d, H], wk [n_kv*d, H], wv [n_kv*d, H], wo [H, n_heads*d],
 *   q_norm_w [d], k_norm_w [d], fc_w [H, n_target_layers*H] (may be NULL when
 *   n_target_layers == 0), hidden_norm_w [H] (NULL iff fc_w is NULL).
 * All are device pointers in cfg->dtype, nn.Linear [out, in] layout.  They
 * are copied into library-owned memory before the call returns; the caller
 * may free them afterwards.
 * Errors: _ARG (null out/weights, bad dtype), _SHAPE (non-positive sizes,
 * n_heads % n_kv_heads != 0, odd head_dim; bf16 layers need head_dim 128 and
 * hidden % 128 == 0), _CUDA, _MEMORY.  On error *out is set to NULL. */
int dflash_attn_create(const dflash_attn_config* cfg, const void* wq,
                       const void* wk, const void* wv, const void* wo,
                       const void* q_norm_w, const void* k_norm_w,
                       const void* fc_w, const void* hidden_norm_w,
                       dflash_attn** out);

/* Free the layer and its scratch.  Waits for the device to finish the
 * layer's outstanding work.  NULL is accepted (no-op). */
int dflash_attn_destroy(dflash_attn* attn);

/* Optional: size the layer's scratch for calls up to these sizes now, so
 * that later calls of at most that size allocate nothing.
 * max_rows = largest (batch*q_len + total new context rows) of a forward, or
 * rows of a ctx_project; max_keys = largest total key rows of one sequence;
 * max_batch = largest batch. */
int dflash_attn_reserve(dflash_attn* attn, int max_batch, int max_rows,
                        int max_keys);

/* Draft KV cache for `batch` sequences of up to `capacity_rows` rows each.
 * [P3] step 4 (DynamicCache update/crop).  Layout of the device storage:
 * K and V each [batch][n_kv_heads][capacity_rows][head_dim] in the layer
 * dtype; K rows are stored after k_norm and RoPE, V rows raw.  Lengths start
 * at 0 and are mirrored on the host.  The cache may be used with any layer
 * whose n_kv_heads, head_dim and dtype match the one given here. */
int dflash_cache_create(const dflash_attn* attn, int batch, int capacity_rows,
                        dflash_cache** out);
int dflash_cache_destroy(dflash_cache* cache);

/* Copy the current row counts into host_len[batch] (host memory). */
int dflash_cache_lengths(const dflash_cache* cache, int32_t* host_len);

/* Device pointers to the K and V storage (layout above), and the geometry.
 * For inspection and tests; writing through them is the caller's risk. */
int dflash_cache_data(const dflash_cache* cache, void** k, void** v,
                      int32_t* batch, int32_t* n_kv_heads,
                      int32_t* capacity_rows, int32_t* head_dim);

/* Copy the whole K and V storage (layout above) into caller device buffers
 * k_dst and v_dst, each batch*n_kv_heads*capacity_rows*head_dim elements,
 * on `stream`.  For inspection and tests. */
int dflash_cache_read(const dflash_cache* cache, void* k_dst, void* v_dst,
                      dflash_stream stream);

/* Crop each sequence b to its first host_keep[b] rows (host memory).
 * [P3] step 4: after verification the cache is cut back to the accepted
 * prefix.  No data moves: rows at or beyond the new length are dead and are
 * overwritten by the next append.  keep == len is a no-op.
 * Errors: _RANGE if any keep < 0 or keep > current length (nothing changes). */
int dflash_cache_crop(dflash_cache* cache, const int32_t* host_keep);

/* Context projection ([P3] 看懂注意力数据流; [P5] combine_hidden_states and
 * precompute_and_store_context_kv's hidden_norm):
 *   target_hidden = hidden_norm(fc(target_layers))
 * target_layers [rows, n_target_layers*H] and target_hidden [rows, H] are
 * device tensors.  rows may be 0 (nothing is enqueued).
 * Errors: _UNSUPPORTED if the layer has no fc, _ARG, _SHAPE. */
int dflash_ctx_project(dflash_attn* attn, const void* target_layers, int rows,
                       void* target_hidden, dflash_stream stream);

/* The same context projection as dflash_ctx_project, for callers that must
 * not have device memory allocated on their behalf.  The pages have no
 * counterpart: this is a property of this library, not of the method.
 * Who needs it: serving processes that fix all device memory at start-up
 * and treat any later allocation as a failure, and hosts whose memory pool
 * must be the only allocator on the GPU.  dflash_ctx_project may grow
 * layer-owned scratch with cudaMalloc; this entry point never allocates and
 * never frees.
 * Its scratch (the fp32 fc output, the split-K partial tiles and their
 * counters) lives in one fixed 16 MiB array inside the library's device
 * image, present on every GPU that loads the library until the process
 * exits.  The scratch a request needs is rows * H * 4 bytes for the fc
 * output plus the split-K tiles of the projection kernel the row count
 * selects: up to 384 rows that kernel needs no split-K tiles, from 385 rows
 * the persistent kernel may split K and then needs 128 KB per (tile, split).
 * At H = 4096 (fc 20480 -> 4096) that admits up to 384 rows and rejects
 * 385 and more.  A request above 16 MiB is rejected with
 * DFLASH_ERR_CAPACITY and enqueues nothing.
 * The first call on a device looks up the array's device address (which may
 * load the library's device code on that device): make that first call
 * before any stream capture.  Every call on a device shares the one array
 * and the array keeps the previous call's contents; the call clears the
 * parts that must start at zero on `stream` itself.  Calls whose work can
 * overlap on the GPU (different streams, or other threads) race on the
 * array: serialise them.  Arguments, layouts and other errors are those of
 * dflash_ctx_project; the layer's device must be the current device. */
int dflash_ctx_project_noalloc(dflash_attn* attn, const void* target_layers,
                               int rows, void* target_hidden,
                               dflash_stream stream);

/* One inference step of the layer for `batch` sequences.
 * [P3] steps 1-4 and 关键设计; [P4] Qwen3DFlashAttention.forward,
 * apply_rotary_pos_emb, _sliding_window_mask; [P5] DFlashQwen3Attention.forward.
 *   noise_hidden  device [batch, q_len, H]: the block embeddings
 *   target_hidden device [sum_b n_ctx[b], H]: new context rows, sequence-major
 *                 (may be NULL when every n_ctx is 0)
 *   host_n_ctx    host   [batch]: new context rows per sequence (>= 0)
 *   positions     device [sum_b (n_ctx[b] + q_len)]: per sequence its context
 *                 rows' positions, then the block's q_len positions
 *   out           device [batch, q_len, H]
 * For sequence b with L_b cached rows, the call appends n_ctx[b] context rows
 * and then the q_len block rows (K after k_norm + RoPE, V raw) at cache rows
 * L_b .. L_b + n_ctx[b] + q_len - 1, sets its length to that sum, and attends
 * every block query to all rows of the sequence (non-causal; on a layer with
 * sliding_window W only to keys whose index is within W of the query's index
 * L_b + n_ctx[b] + t).  The block rows stay in the cache until a crop.
 * Requires batch == cache batch <= 512; bf16 layers also need
 * (n_heads/n_kv_heads) * q_len <= 128.
 * Errors: _ARG, _SHAPE, _CAPACITY (L_b + n_ctx[b] + q_len > capacity; nothing
 * is appended for any sequence), _CUDA. */
int dflash_attn_forward(dflash_attn* attn, dflash_cache* cache, int batch,
                        int q_len, const void* noise_hidden,
                        const void* target_hidden, const int32_t* host_n_ctx,
                        const int32_t* positions, void* out,
                        dflash_stream stream);

/* Paged draft KV cache ([P5] precompute_and_store_context_kv: the context
 * K/V go into the layer's paged cache through do_kv_cache_update with a
 * slot_mapping; the draft's attention reads the pages through the batch's
 * block table).  Storage: K and V each [n_pages][n_kv_heads][page_size]
 * [head_dim] bf16, zeroed at creation; page p row r is slot p*page_size + r.
 * page_size is 16, 32, 64 or 128.  The cache holds no lengths: which pages
 * belong to which sequence, their order and each sequence's length are the
 * caller's (block table, slot mapping, host_len_before), so crop and
 * reuse are the caller's bookkeeping.  bf16 layers only (else _UNSUPPORTED).
 * dflash_paged_cache_data returns the storage and its geometry (for
 * inspection and tests; writing through it is the caller's risk);
 * dflash_paged_cache_read copies the whole K and V storage into caller
 * device buffers of n_pages*n_kv_heads*page_size*head_dim elements each, on
 * `stream`. */
int dflash_paged_cache_create(const dflash_attn* attn, int n_pages,
                              int page_size, dflash_paged_cache** out);
int dflash_paged_cache_destroy(dflash_paged_cache* cache);
int dflash_paged_cache_data(const dflash_paged_cache* cache, void** k,
                            void** v, int32_t* n_pages, int32_t* n_kv_heads,
                            int32_t* page_size, int32_t* head_dim);
int dflash_paged_cache_read(const dflash_paged_cache* cache, void* k_dst,
                            void* v_dst, dflash_stream stream);

/* dflash_attn_forward over a paged cache.  Arguments, outputs and errors are
 * those of dflash_attn_forward, with the cache replaced by:
 *   host_len_before host   [batch]: rows each sequence already holds
 *   slot_mapping    device [sum_b (n_ctx[b] + q_len)]: the slot each new
 *                   row's K and V are written to, in the order of positions
 *   block_table     device [batch][bt_stride]: sequence b's key row k lives
 *                   in page block_table[b][k / page_size], row k % page_size
 * The new rows of sequence b take key indices len_before[b] .. len_before[b]
 * + n_ctx[b] + q_len - 1; the call attends over indices 0 .. that end
 * through the block table.  The slots must be the ones the block table gives
 * for those indices (the kernels trust it).  A slot outside the cache skips
 * that row's write and records DFLASH_DEV_SLOT; a block-table entry outside
 * the cache for a page that holds keys of the sequence reads page 0 in its
 * place and records DFLASH_DEV_SLOT.  Block-table entries past a sequence's
 * last row may hold anything.
 * Errors: _ARG, _SHAPE, _UNSUPPORTED, _CAPACITY (a sequence's rows exceed
 * bt_stride pages), _CUDA. */
int dflash_attn_forward_paged(dflash_attn* attn, dflash_paged_cache* cache,
                              int batch, int q_len, const void* noise_hidden,
                              const void* target_hidden,
                              const int32_t* host_n_ctx,
                              const int32_t* host_len_before,
                              const int32_t* positions,
                              const int32_t* slot_mapping,
                              const int32_t* block_table, int bt_stride,
                              void* out, dflash_stream stream);

/* Context K/V of several draft layers in one projection ([P5]
 * precompute_and_store_context_kv: the context K/V of all layers come from one
 * GEMM over their stacked k_proj/v_proj weights, then each layer's k_norm,
 * RoPE and cache insert).
 *
 * dflash_kv_group_create stacks the K and V weights of n_layers (1..16) bf16
 * layers that share hidden, n_kv_heads, head_dim, device, max_position,
 * rms_eps and rope_theta (else _SHAPE; fp32 layers _UNSUPPORTED).  The group
 * owns a copy of those weights; the layers must outlive it.
 *
 * dflash_kv_group_append projects the batch's new context rows once for all
 * layers and appends, for layer l, K = RoPE(k_norm_l(T Wk_l^T)) and
 * V = T Wv_l^T to caches[l] at its current lengths, exactly as
 * dflash_attn_forward appends context rows.  Afterwards call each layer's
 * dflash_attn_forward with host_n_ctx all zero (and positions for the block
 * rows only): it appends the block rows and attends over every cached row.
 *   caches          host array of n_layers cache handles (same batch and
 *                   lengths; geometry of the layers)
 *   target_hidden   device [sum n_i, H] bf16, sequence-major (may be NULL
 *                   when every n_i is 0)
 *   host_n_ctx      host [batch] new context rows per sequence
 *   positions       device [sum n_i] int32, the context rows' positions
 * Errors: _ARG (nulls, negative counts), _SHAPE (batch, geometry or lengths
 * differ between caches), _CAPACITY (a cache would overflow; nothing is
 * appended). */
int dflash_kv_group_create(dflash_attn* const* layers, int n_layers,
                           dflash_kv_group** out);
int dflash_kv_group_destroy(dflash_kv_group* group);
int dflash_kv_group_append(dflash_kv_group* group, dflash_cache* const* caches,
                           int batch, const void* target_hidden,
                           const int32_t* host_n_ctx, const int32_t* positions,
                           dflash_stream stream);

/* The rest of a draft decoder layer ([P4] Qwen3DFlashDecoderLayer:
 * input_layernorm, self_attn, post_attention_layernorm, mlp = Qwen3MLP; [P5]
 * stacks gate_proj/up_proj into gate_up_proj).  Reading taken (the pages name
 * Qwen3MLP without printing it): mlp(y) = down(silu(gate(y)) * up(y)).
 * Weights bf16 device, nn.Linear layout: gate_w, up_w [intermediate, hidden],
 * down_w [hidden, intermediate]; input_norm_w, post_norm_w [hidden] bf16.
 * hidden % 128 == 0 (<= 8192), intermediate % 128 == 0, else _SHAPE.  The
 * handle owns copies of the weights. */
int dflash_mlp_create(int hidden, int intermediate, float rms_eps,
                      const void* gate_w, const void* up_w, const void* down_w,
                      const void* input_norm_w, const void* post_norm_w,
                      dflash_mlp** out);
int dflash_mlp_destroy(dflash_mlp* mlp);

/* One draft decoder layer in the residual-stream form of [P5]'s draft model
 * (each layer returns (hidden_states, residual); the next one adds them):
 *   r1 = hidden_in + residual_in   (residual_in NULL: r1 = hidden_in)
 *   r2 = r1 + attn(input_norm(r1))   -- dflash_attn_forward on the normed rows
 *   hidden_out = mlp(post_norm(r2)),  residual_out = r2
 * hidden_in, residual_in, hidden_out, residual_out: device bf16
 * [batch, q_len, hidden] (residual_out may alias residual_in); the other
 * arguments and the cache update are those of dflash_attn_forward.  bf16
 * layers only (_UNSUPPORTED otherwise); the MLP's hidden must equal the
 * layer's (_SHAPE). */
int dflash_decoder_layer_forward(dflash_attn* attn, dflash_mlp* mlp,
                                 dflash_cache* cache, int batch, int q_len,
                                 const void* hidden_in, const void* residual_in,
                                 const void* target_hidden,
                                 const int32_t* host_n_ctx,
                                 const int32_t* positions, void* hidden_out,
                                 void* residual_out, dflash_stream stream);

/* Training-layout forward with no cache ([P4] module docstring: each block's
 * queries see the context strictly before its anchor plus their own block,
 * bidirectionally; training is one forward with no cache).
 *   noise_hidden  device [batch, n_blocks*block_size, H]
 *   target_hidden device [batch, seq, H]  (projected context)
 *   anchors       device [batch, n_blocks]  int32, each in [0, seq]
 *   out           device [batch, n_blocks*block_size, H]
 * Context row j sits at position j, row t of block k at anchors[k] + t.
 * Blocks may share positions; anchors need not be sorted (sorted anchors
 * balance the work best).  Layers with sliding_window > 0 are _UNSUPPORTED.
 * bf16 layers need (n_heads/n_kv_heads) * block_size <= 128. */
int dflash_attn_forward_packed(dflash_attn* attn, int batch, int seq,
                               int n_blocks, int block_size,
                               const void* noise_hidden,
                               const void* target_hidden,
                               const int32_t* anchors, void* out,
                               dflash_stream stream);

/* Kernel kinds of the per-launch event trace. */
enum {
  DFLASH_K_FC = 0,     /* fc projection GEMM of dflash_ctx_project        */
  DFLASH_K_NORM = 1,   /* hidden_norm row RMSNorm of dflash_ctx_project   */
  DFLASH_K_QKV = 2,    /* QKV projection + norm + RoPE + cache append     */
  DFLASH_K_ATTN = 3,   /* attention (with the split merge)                */
  DFLASH_K_OPROJ = 4,  /* o_proj GEMM                                     */
  DFLASH_K_MISC = 5,   /* packed-layout positions                         */
  DFLASH_K_MLP = 6,    /* decoder layer: add+norm kernels and MLP GEMMs    */
  DFLASH_K_BWD = 7,    /* packed attention core backward (dK/dV and dQ)   */
  DFLASH_K_COUNT = 8
};

/* Attention core of the packed training layout, forward and backward
 * ([P4] module docstring: block k's queries see the context strictly before
 * anchors[k] and their own block; the draft is trained by backpropagation
 * through that masked attention).  These take Q, K and V directly (after
 * the projections, norms and RoPE), so a training framework can run its own
 * projections and autograd around them.  The layer handle supplies
 * n_heads, n_kv_heads, head_dim and scratch; its weights are not used.
 *   q, out, d_out, dq  device [batch][n_blocks*block_size][n_heads][head_dim]
 *                      bf16 (block k's rows at k*block_size ..)
 *   k, v, dk, dv       device [batch][n_kv_heads][seq + n_blocks*block_size]
 *                      [head_dim] bf16: per (sequence, kv head) the seq
 *                      context rows, then every block's rows in block order
 *   lse                device [batch][n_blocks*block_size][n_heads] fp32:
 *                      natural log of each query row's softmax normaliser,
 *                      log(sum over visible keys of exp(q.k / sqrt(head_dim)))
 *   anchors            device [batch][n_blocks] int32 in [0, seq]
 * dflash_packed_attn_core writes out = softmax(q k^T / sqrt(d), masked) v and
 * lse.  dflash_packed_attn_core_backward takes the forward's q, k, v, out,
 * lse and the output gradient d_out and writes the gradients dq, dk, dv
 * (each KV head's gradient sums over the query heads that read it; key rows
 * no query sees get 0).  Every output element is written exactly once (no
 * atomics; reruns are bitwise identical).
 * Requires a bf16 layer without sliding window or causal flag, and
 * (n_heads / n_kv_heads) * block_size == 64.  An anchor outside [0, seq] is
 * clamped and recorded (DFLASH_DEV_ANCHOR) by the forward.
 * Errors: _ARG, _SHAPE, _UNSUPPORTED, _CUDA. */
int dflash_packed_attn_core(dflash_attn* attn, int batch, int seq,
                            int n_blocks, int block_size, const void* q,
                            const void* k, const void* v,
                            const int32_t* anchors, void* out, float* lse,
                            dflash_stream stream);
int dflash_packed_attn_core_backward(dflash_attn* attn, int batch, int seq,
                                     int n_blocks, int block_size,
                                     const void* q, const void* k,
                                     const void* v, const void* out,
                                     const float* lse, const void* d_out,
                                     const int32_t* anchors, void* dq,
                                     void* dk, void* dv,
                                     dflash_stream stream);

/* Kernels this library has launched in this process so far, over every
 * layer, cache and device (a launch that returned an error counts too).  A
 * caller reads it before and after a region to count that region's kernels. */
int dflash_kernel_launches(uint64_t* count);

/* Launch tracing for measurement: while enabled, every kernel launch of the
 * layer is bracketed by two CUDA events recorded on its own stream.
 * dflash_trace_enable(attn, 1) starts a fresh trace, (attn, 0) stops it.
 * dflash_trace_read waits for the recorded events and returns, for one
 * kernel kind, the summed device time in milliseconds and the launch count.
 * Not for use while a stream is being captured into a CUDA graph. */
int dflash_trace_enable(dflash_attn* attn, int enable);
int dflash_trace_read(dflash_attn* attn, int kind, double* total_ms,
                      int32_t* launches);

/* Wait for the device, then report and clear the layer's device error word
 * (DFLASH_DEV_*).  Returns DFLASH_ERR_DEVICE when the word was non-zero. */
int dflash_device_error(dflash_attn* attn, int32_t* code);

/* Check of the bounded device waits (no counterpart on the pages: failure
 * handling of this library).  Enqueues one kernel on `stream` in which one
 * thread waits on a shared-memory mbarrier with the same routine every
 * pipeline wait of the library uses, but for at most limit_ns nanoseconds of
 * GPU global time instead of the pipelines' 2 s.
 *   arrive = 1: the barrier's one expected arrival is made first; the wait
 *               completes at once and nothing is recorded.
 *   arrive = 0: nothing ever arrives; the wait runs out, records
 *               DFLASH_DEV_WAIT_TIMEOUT in the layer's device error word and
 *               the kernel returns normally (no trap, no fault): the context
 *               stays usable and dflash_device_error() reports the code.
 * limit_ns must lie in [1e3, 1e8].  Errors: _ARG, _CUDA. */
int dflash_wait_probe(dflash_attn* attn, int64_t limit_ns, int arrive,
                      dflash_stream stream);

/* Measurement aid (no counterpart on the pages): the rate at which TMA alone
 * reads a projection's weights.  Enqueues one kernel on `stream` that streams
 * the rows x cols bf16 row-major device matrix `matrix` (caller-owned, 16-byte
 * aligned) once into shared memory in the boxes the GEMMs read weights in
 * (128 rows x 64 columns, 128-byte swizzle) and discards it.  The boxes, in
 * (row block, column block) order, are split into `ctas` contiguous shares,
 * one per CTA; each CTA keeps `stages` boxes (16 KB each) in flight and
 * reuses a slot as soon as its box has landed.  Nothing is written.  Time it
 * with events on `stream`.  rows: a positive multiple of 128; cols: a
 * positive multiple of 64; stages in [1, 12]; ctas in [1, 2 x SMs], and at
 * most 6 stages when ctas exceeds the SM count (two CTAs per SM).  Its
 * bounded waits record DFLASH_DEV_WAIT_TIMEOUT in the layer's device error
 * word like every pipeline of the library.  Errors: _ARG, _CUDA. */
int dflash_read_stream_probe(dflash_attn* attn, const void* matrix, int64_t rows,
                             int64_t cols, int ctas, int stages, dflash_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_ATTN_H */
