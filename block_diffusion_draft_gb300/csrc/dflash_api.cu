// dflash_api.cu -- the C ABI (include/dflash_attn.h): handles, argument
// checks, scratch management and the launch sequence of each call.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/dflash_attn.h"
#include "handles.h"
#include "internal.h"

using namespace df;

namespace df {
std::atomic<unsigned long long> g_kernel_launches{0};
}  // namespace df

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(e == cudaErrorMemoryAllocation ? DFLASH_ERR_MEMORY : DFLASH_ERR_CUDA,
              "%s: %s", what, cudaGetErrorString(e));
}

#define DF_CUDA(call, what)                      \
  do {                                           \
    cudaError_t _e = (cudaError_t)(call);        \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)

size_t dtype_size(int dt) { return dt == DFLASH_BF16 ? 2 : 4; }

}  // namespace

namespace {

cudaEvent_t take_event(dflash_attn* a) {
  if (!a->event_pool.empty()) {
    cudaEvent_t e = a->event_pool.back();
    a->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// brackets one launch with events on its stream while tracing is on
struct TraceScope {
  dflash_attn* a;
  int kind;
  cudaStream_t s;
  cudaEvent_t e0 = nullptr;
  TraceScope(dflash_attn* a_, int kind_, cudaStream_t s_) : a(a_), kind(kind_), s(s_) {
    if (a->trace) {
      e0 = take_event(a);
      cudaEventRecord(e0, s);
    }
  }
  ~TraceScope() {
    if (a->trace && e0) {
      cudaEvent_t e1 = take_event(a);
      cudaEventRecord(e1, s);
      a->recs.push_back({kind, e0, e1});
    }
  }
};

int check_attn(const dflash_attn* a) {
  if (a == nullptr) return fail(DFLASH_ERR_ARG, "null layer handle");
  return DFLASH_OK;
}

// scratch needed by the bf16 GEMM for a given shape
int ensure_gemm_scratch(dflash_attn* a, int epi, int rows0, int rows1, int n, int k,
                        int q_cols) {
  int n_counters = 0;
  const size_t bytes =
      gemm_scratch_bytes(epi, rows0, rows1, n, k, q_cols, a->num_sms, &n_counters);
  DF_CUDA(a->gemm_partial.ensure(std::max<size_t>(bytes, 256)), "scratch allocation");
  DF_CUDA(a->gemm_counters.ensure((size_t)std::max(n_counters, 64) * sizeof(int), true),
          "scratch allocation");
  return DFLASH_OK;
}

// Scratch for every GEMM shape with up to max0 / max1 rows.  Split-K scratch
// is not monotonic in the row count (fewer row tiles take more K splits), so
// every count of 128-row tiles is tried.
int reserve_gemm_scratch(dflash_attn* a, int epi, int max0, int max1, int n, int k,
                         int q_cols) {
  const int m0 = (max0 + 127) / 128, m1 = (max1 + 127) / 128;
  for (int i = 1; i <= m0; ++i)
    for (int j = 0; j <= m1; ++j)
      if (int r = ensure_gemm_scratch(a, epi, std::min(max0, i * 128), std::min(max1, j * 128),
                                      n, k, q_cols))
        return r;
  return DFLASH_OK;
}

GemmScratch gemm_scratch(dflash_attn* a) {
  GemmScratch s;
  s.partial = static_cast<float*>(a->gemm_partial.p);
  s.partial_bytes = a->gemm_partial.bytes;
  s.counters = static_cast<int*>(a->gemm_counters.p);
  s.n_counters = (int)(a->gemm_counters.bytes / sizeof(int));
  return s;
}

QkvOut make_qkv_out(const dflash_attn* a, const int* positions, void* qbuf,
                    void* k, void* v, int cap, int q_block) {
  QkvOut o{};
  o.n_heads = a->nq;
  o.n_kv = a->nkv;
  o.groups = a->g;
  o.q_block = q_block;
  o.cap = cap;
  o.max_pos = a->max_pos;
  o.eps = a->cfg.rms_eps;
  const double scale = 1.0 / std::sqrt((double)a->d);
  // the bf16 path works in log2 units (exp2 softmax); the fp32 path in e
  o.q_scale = (float)(a->dt == DFLASH_BF16 ? scale * 1.4426950408889634 : scale);
  o.positions = positions;
  o.rope = a->rope;
  o.q_norm = a->q_norm;
  o.k_norm = a->k_norm;
  o.qbuf = qbuf;
  o.cache_k = k;
  o.cache_v = v;
  return o;
}

// Projections + norm + RoPE + append for `rows_noise` block rows and
// `rows_ctx` context rows whose bookkeeping is in `st`.
int run_qkv(dflash_attn* a, const void* noise, int rows_noise, const void* ctx,
            int rows_ctx, const QkvOut& o, const SeqTable& st, cudaStream_t s) {
  const int nqkv = (a->nq + 2 * a->nkv) * a->d;
  if (a->dt == DFLASH_BF16) {
    int r = ensure_gemm_scratch(a, EPI_QKV, rows_noise, rows_ctx, nqkv, a->H, a->nq * a->d);
    if (r) return r;
    GemmShape gs{noise, rows_noise, ctx, rows_ctx, &a->tm_qkv, &a->tm_qkv256, nqkv, a->H,
                 a->nq * a->d};
    TraceScope tr(a, DFLASH_K_QKV, s);
    DF_CUDA(launch_gemm_bf16(gs, EPI_QKV, nullptr, 0, &o, &st, gemm_scratch(a),
                             a->num_sms, a->err, s),
            "QKV projection launch");
  } else {
    const int nkv2 = 2 * a->nkv * a->d;
    DF_CUDA(a->proj_noise.ensure((size_t)std::max(rows_noise, 1) * nqkv * 4), "scratch");
    DF_CUDA(a->proj_ctx.ensure((size_t)std::max(rows_ctx, 1) * nkv2 * 4), "scratch");
    float* pn = static_cast<float*>(a->proj_noise.p);
    float* pc = static_cast<float*>(a->proj_ctx.p);
    const float* w = static_cast<const float*>(a->w_qkv);
    TraceScope tr(a, DFLASH_K_QKV, s);
    DF_CUDA(launch_gemm_f32(static_cast<const float*>(noise), rows_noise, w, nqkv, a->H,
                            pn, nqkv, s), "fp32 projection");
    if (rows_ctx > 0)
      DF_CUDA(launch_gemm_f32(static_cast<const float*>(ctx), rows_ctx,
                              w + (size_t)a->nq * a->d * a->H, nkv2, a->H, pc, nkv2, s),
              "fp32 projection");
    DF_CUDA(launch_qkv_post_f32(pn, rows_noise, pc, rows_ctx, o, &st, a->d, a->err, s),
            "fp32 norm/rope");
  }
  return DFLASH_OK;
}

int run_o_proj(dflash_attn* a, int rows, void* out, cudaStream_t s) {
  if (a->dt == DFLASH_BF16) {
    int r = ensure_gemm_scratch(a, EPI_BF16, rows, 0, a->H, a->nq * a->d, 0);
    if (r) return r;
    TraceScope tr(a, DFLASH_K_OPROJ, s);
    GemmShape gs{a->attn_out.p, rows, nullptr, 0, &a->tm_o, &a->tm_o256, a->H, a->nq * a->d, 0};
    DF_CUDA(launch_gemm_bf16(gs, EPI_BF16, out, a->H, nullptr, nullptr, gemm_scratch(a),
                             a->num_sms, a->err, s),
            "o_proj launch");
  } else {
    TraceScope tr(a, DFLASH_K_OPROJ, s);
    DF_CUDA(launch_gemm_f32(static_cast<const float*>(a->attn_out.p), rows,
                            static_cast<const float*>(a->w_o), a->H, a->nq * a->d,
                            static_cast<float*>(out), a->H, s),
            "fp32 o_proj");
  }
  return DFLASH_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The cache a forward appends to and reads: contiguous ([B][n_kv][cap][d])
// or paged ([n_pages][n_kv][P][d] with the caller's slots and block table).
struct KvView {
  void* k = nullptr;
  void* v = nullptr;
  int cap = 0;
  long long rows_total = 0;  // rows of the K (and V) storage
  const int* slot_mapping = nullptr;
  const int* block_table = nullptr;
  int bt_stride = 0, page_size = 0, n_pages = 0;
  static KvView of(const dflash_cache* c) {
    KvView v;
    v.k = c->k;
    v.v = c->v;
    v.cap = c->cap;
    v.rows_total = (long long)c->batch * c->nkv * c->cap;
    return v;
  }
};

// Projections, attention and o_proj of one forward (arguments checked by the
// caller); the caller updates its own lengths.
int forward_core(dflash_attn* a, const KvView& kv, int batch, int q_len, const void* noise,
                 const void* target_hidden, const int32_t* host_n_ctx, const int* len_before,
                 const int32_t* positions, void* out, dflash_stream stream) {
  const long long rows_noise = (long long)batch * q_len;
  long long total_ctx = 0;
  for (int b = 0; b < batch; ++b) total_ctx += host_n_ctx[b];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t es = dtype_size(a->dt);
  const size_t qd = (size_t)a->nq * a->d;

  SeqTable st;
  st.n = batch;
  st.q_len = q_len;
  st.ctx_off[0] = 0;
  for (int b = 0; b < batch; ++b) {
    st.ctx_off[b + 1] = st.ctx_off[b] + host_n_ctx[b];
    st.cache_len[b] = len_before[b];
  }
  DF_CUDA(a->qbuf.ensure(rows_noise * qd * es), "scratch allocation");
  DF_CUDA(a->attn_out.ensure(rows_noise * qd * es), "scratch allocation");
  QkvOut o = make_qkv_out(a, positions, a->qbuf.p, kv.k, kv.v, kv.cap, q_len);
  o.slot_mapping = kv.slot_mapping;
  o.page_size = kv.page_size;
  o.n_pages = kv.n_pages;
  o.err = a->err;
  if (int r = run_qkv(a, noise, (int)rows_noise, target_hidden, (int)total_ctx, o, st, s))
    return r;

  // attention work list: per sequence the visible key range, split in units
  AttnSeqs sq;
  for (int b = 0; b < batch; ++b) {
    sq.len[b] = len_before[b] + host_n_ctx[b] + q_len;
    sq.first_new[b] = len_before[b];
    sq.lo[b] = a->cfg.sliding_window > 0
                   ? std::max(0, sq.len[b] - q_len - a->cfg.sliding_window + 1)
                   : 0;
    // paged tiles gather whole pages: start the range on a tile boundary
    // (the band still cuts each row's keys)
    if (kv.block_table != nullptr) sq.lo[b] = sq.lo[b] / 128 * 128;
  }
  int cl = 1, kcl = 1, n_units = batch * a->nkv;
  if (a->dt == DFLASH_BF16)
    n_units = plan_decode_attention(sq, batch, a->nkv, a->num_sms, a->g * q_len <= 64, &cl,
                                    &kcl);
  AttnArgs aa{};
  aa.mode = 0;
  aa.batch = batch;
  aa.n_kv = a->nkv;
  aa.groups = a->g;
  aa.head_dim = a->d;
  aa.q_len = q_len;
  aa.q_block = q_len;
  aa.n_blocks = 1;
  aa.tile_blocks = 1;
  aa.cap = kv.cap;
  aa.block_table = kv.block_table;
  aa.bt_stride = kv.bt_stride;
  aa.page_size = kv.page_size;
  aa.n_pages = kv.n_pages;
  aa.window = a->cfg.sliding_window;
  aa.causal = a->cfg.causal != 0;
  aa.n_units = n_units;
  aa.cluster = cl;
  aa.k_clusters = kcl;
  aa.out = a->attn_out.p;
  aa.err = a->err;
  if (a->dt == DFLASH_BF16) {
    // partial slots: one per unit, twice in cluster mode with several
    // clusters per pair (the clusters' merged row blocks)
    const size_t slots = (size_t)n_units * (cl > 1 && kcl > 1 ? 2 : 1);
    DF_CUDA(a->part_o.ensure(slots * 128 * 128 * 4), "scratch allocation");
    DF_CUDA(a->part_ml.ensure(slots * 256 * 4), "scratch allocation");
    DF_CUDA(a->attn_counters.ensure(decode_attention_counters(batch, a->nkv) * sizeof(int), true),
            "scratch allocation");
    aa.part_o = static_cast<float*>(a->part_o.p);
    aa.part_ml = static_cast<float*>(a->part_ml.p);
    aa.counters = static_cast<int*>(a->attn_counters.p);
    TraceScope tr(a, DFLASH_K_ATTN, s);
    DF_CUDA(launch_attn_bf16(aa, &sq, a->qbuf.p, rows_noise * a->nq, kv.k, kv.v,
                             kv.rows_total, s),
            "attention launch");
  } else {
    TraceScope tr(a, DFLASH_K_ATTN, s);
    DF_CUDA(launch_attn_f32(aa, &sq, static_cast<const float*>(a->qbuf.p),
                            static_cast<const float*>(kv.k), static_cast<const float*>(kv.v),
                            s),
            "fp32 attention launch");
  }
  return run_o_proj(a, (int)rows_noise, out, s);
}


}  // namespace

// error reporting for the allocation-free entry point (noalloc.cu)
int dflash_noalloc_fail(int code, const char* msg) { return fail(code, "%s", msg); }

extern "C" {

const char* dflash_last_error(void) { return g_err.c_str(); }

int dflash_abi_version(void) { return 105; }

int dflash_attn_create(const dflash_attn_config* cfg_in, const void* wq, const void* wk,
                       const void* wv, const void* wo, const void* q_norm_w,
                       const void* k_norm_w, const void* fc_w, const void* hidden_norm_w,
                       dflash_attn** out) {
  if (out == nullptr) return fail(DFLASH_ERR_ARG, "out is null");
  *out = nullptr;
  if (cfg_in == nullptr) return fail(DFLASH_ERR_ARG, "config is null");
  dflash_attn_config cfg = *cfg_in;
  if (cfg.dtype != DFLASH_BF16 && cfg.dtype != DFLASH_FP32)
    return fail(DFLASH_ERR_ARG, "dtype must be DFLASH_BF16 or DFLASH_FP32");
  if (!wq || !wk || !wv || !wo || !q_norm_w || !k_norm_w)
    return fail(DFLASH_ERR_ARG, "a required weight pointer is null");
  if ((fc_w == nullptr) != (hidden_norm_w == nullptr))
    return fail(DFLASH_ERR_ARG, "fc_w and hidden_norm_w must both be given or both null");
  if (cfg.hidden <= 0 || cfg.n_heads <= 0 || cfg.n_kv_heads <= 0 || cfg.head_dim < 0 ||
      cfg.n_target_layers < 0 || cfg.sliding_window < 0 || cfg.max_position < 0 ||
      !(cfg.rms_eps >= 0.f) || !(cfg.rope_theta > 0.f))
    return fail(DFLASH_ERR_SHAPE, "non-positive or invalid layer scalar");
  if (cfg.causal != 0 && cfg.causal != 1) return fail(DFLASH_ERR_SHAPE, "causal must be 0 or 1");
  if (cfg.head_dim == 0) cfg.head_dim = cfg.hidden / cfg.n_heads;
  if (cfg.max_position == 0) cfg.max_position = 131072;
  if (cfg.n_heads % cfg.n_kv_heads != 0)
    return fail(DFLASH_ERR_SHAPE, "n_heads (%d) must be a multiple of n_kv_heads (%d)",
                cfg.n_heads, cfg.n_kv_heads);
  if (cfg.head_dim % 2 != 0 || cfg.head_dim <= 0)
    return fail(DFLASH_ERR_SHAPE, "head_dim must be even and positive");
  if ((fc_w != nullptr) != (cfg.n_target_layers > 0))
    return fail(DFLASH_ERR_SHAPE, "fc_w must be given exactly when n_target_layers > 0");
  if (cfg.dtype == DFLASH_BF16) {
    if (cfg.head_dim != 128)
      return fail(DFLASH_ERR_SHAPE, "bf16 layers need head_dim 128 (got %d)", cfg.head_dim);
    if (cfg.hidden % 128 != 0)
      return fail(DFLASH_ERR_SHAPE, "bf16 layers need hidden %% 128 == 0");
  } else if (cfg.head_dim > 256) {
    return fail(DFLASH_ERR_SHAPE, "fp32 layers need head_dim <= 256");
  }
  dflash_attn* a = new dflash_attn();
  a->cfg = cfg;
  cudaGetDevice(&a->device);
  cudaDeviceGetAttribute(&a->num_sms, cudaDevAttrMultiProcessorCount, a->device);
  a->H = cfg.hidden;
  a->d = cfg.head_dim;
  a->nq = cfg.n_heads;
  a->nkv = cfg.n_kv_heads;
  a->g = cfg.n_heads / cfg.n_kv_heads;
  a->nL = cfg.n_target_layers;
  a->max_pos = cfg.max_position;
  a->dt = cfg.dtype;
  const size_t es = dtype_size(a->dt);
  const size_t H = a->H, d = a->d, nq = a->nq, nkv = a->nkv;
  auto cleanup = [&](int code) {
    dflash_attn_destroy(a);
    return code;
  };
  cudaError_t e;
  e = cudaMalloc(&a->w_qkv, (nq + 2 * nkv) * d * H * es);
  if (e == cudaSuccess) e = cudaMalloc(&a->w_o, H * nq * d * es);
  if (e == cudaSuccess && fc_w) e = cudaMalloc(&a->w_fc, H * a->nL * H * es);
  if (e == cudaSuccess) e = cudaMalloc(&a->q_norm, d * 4);
  if (e == cudaSuccess) e = cudaMalloc(&a->k_norm, d * 4);
  if (e == cudaSuccess) e = cudaMalloc(&a->hidden_norm, H * 4);
  if (e == cudaSuccess) e = cudaMalloc(&a->rope, (size_t)a->max_pos * (d / 2) * sizeof(float2));
  if (e == cudaSuccess) e = cudaMalloc(&a->err, sizeof(int));
  if (e != cudaSuccess) return cleanup(cuda_fail(e, "weight allocation"));
  char* wqkv = static_cast<char*>(a->w_qkv);
  e = cudaMemcpy(wqkv, wq, nq * d * H * es, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(wqkv + nq * d * H * es, wk, nkv * d * H * es, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(wqkv + (nq + nkv) * d * H * es, wv, nkv * d * H * es,
                   cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(a->w_o, wo, H * nq * d * es, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess && fc_w)
    e = cudaMemcpy(a->w_fc, fc_w, H * a->nL * H * es, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess) e = cudaMemset(a->err, 0, sizeof(int));
  if (e != cudaSuccess) return cleanup(cuda_fail(e, "weight copy"));
  const int bf = a->dt == DFLASH_BF16;
  if ((e = (cudaError_t)launch_to_f32(q_norm_w, bf, a->q_norm, d, 0)) != cudaSuccess ||
      (e = (cudaError_t)launch_to_f32(k_norm_w, bf, a->k_norm, d, 0)) != cudaSuccess)
    return cleanup(cuda_fail(e, "norm weight conversion"));
  if (hidden_norm_w) {
    if ((e = (cudaError_t)launch_to_f32(hidden_norm_w, bf, a->hidden_norm, H, 0)) !=
        cudaSuccess)
      return cleanup(cuda_fail(e, "norm weight conversion"));
  }
  if ((e = (cudaError_t)launch_rope_table(a->rope, a->max_pos, (int)(d / 2), cfg.rope_theta,
                                          0)) != cudaSuccess)
    return cleanup(cuda_fail(e, "rope table"));
  if (bf) {
    if (make_tmap_bf16_rows(&a->tm_qkv, a->w_qkv, (nq + 2 * nkv) * d, (int)H, 128) != 0 ||
        make_tmap_bf16_rows(&a->tm_o, a->w_o, H, (int)(nq * d), 128) != 0 ||
        (fc_w && make_tmap_bf16_rows(&a->tm_fc, a->w_fc, H, (int)(a->nL * H), 128) != 0) ||
        make_tmap_bf16_rows(&a->tm_qkv256, a->w_qkv, (nq + 2 * nkv) * d, (int)H, 256) != 0 ||
        make_tmap_bf16_rows(&a->tm_o256, a->w_o, H, (int)(nq * d), 256) != 0 ||
        (fc_w && make_tmap_bf16_rows(&a->tm_fc256, a->w_fc, H, (int)(a->nL * H), 256) != 0))
      return cleanup(fail(DFLASH_ERR_CUDA, "tensor map encoding failed"));
  }
  if ((e = cudaDeviceSynchronize()) != cudaSuccess)
    return cleanup(cuda_fail(e, "layer set-up"));
  *out = a;
  return DFLASH_OK;
}

int dflash_attn_destroy(dflash_attn* a) {
  if (a == nullptr) return DFLASH_OK;
  cudaDeviceSynchronize();
  cudaFree(a->w_qkv);
  cudaFree(a->w_o);
  cudaFree(a->w_fc);
  cudaFree(a->q_norm);
  cudaFree(a->k_norm);
  cudaFree(a->hidden_norm);
  cudaFree(a->rope);
  cudaFree(a->err);
  for (auto& r : a->recs) {
    cudaEventDestroy(r.e0);
    cudaEventDestroy(r.e1);
  }
  for (cudaEvent_t e : a->event_pool) cudaEventDestroy(e);
  for (Buf* b : {&a->qbuf, &a->attn_out, &a->gemm_partial, &a->gemm_counters, &a->part_o,
                 &a->part_ml, &a->attn_counters, &a->zbuf, &a->proj_noise, &a->proj_ctx,
                 &a->packed_k, &a->packed_v, &a->packed_pos, &a->bwd_do, &a->bwd_stats})
    b->release();
  delete a;
  return DFLASH_OK;
}

int dflash_attn_reserve(dflash_attn* a, int max_batch, int max_rows, int max_keys) {
  if (int r = check_attn(a)) return r;
  if (max_batch <= 0 || max_rows <= 0 || max_keys <= 0 || max_batch > kMaxBatch)
    return fail(DFLASH_ERR_ARG, "reserve sizes must be positive (batch <= %d)", kMaxBatch);
  const size_t es = dtype_size(a->dt);
  const size_t qd = (size_t)a->nq * a->d;
  DF_CUDA(a->qbuf.ensure((size_t)max_rows * qd * es), "scratch allocation");
  DF_CUDA(a->attn_out.ensure((size_t)max_rows * qd * es), "scratch allocation");
  if (a->dt == DFLASH_BF16) {
    const int nqkv = (a->nq + 2 * a->nkv) * a->d;
    if (int r = reserve_gemm_scratch(a, EPI_QKV, max_rows, max_rows, nqkv, a->H, a->nq * a->d))
      return r;
    if (int r = reserve_gemm_scratch(a, EPI_BF16, max_rows, 0, a->H, a->nq * a->d, 0)) return r;
    if (a->nL > 0) {
      if (int r = reserve_gemm_scratch(a, EPI_F32, max_rows, 0, a->H, a->nL * a->H, 0)) return r;
    }
    // the decode attention's partial slots and merge counters
    const size_t slots = decode_attention_slots(max_batch, a->nkv, a->num_sms);
    DF_CUDA(a->part_o.ensure(slots * 128 * 128 * 4), "scratch allocation");
    DF_CUDA(a->part_ml.ensure(slots * 256 * 4), "scratch allocation");
    DF_CUDA(a->attn_counters.ensure(decode_attention_counters(max_batch, a->nkv) * sizeof(int),
                                    true),
            "scratch allocation");
  }
  if (a->nL > 0) {
    // the fc output slices of the largest row count that needs the most
    size_t zb = (size_t)max_rows * a->H * 4;
    if (a->dt == DFLASH_BF16)
      for (int r = 1; r <= max_rows; ++r)
        zb = std::max(zb, (size_t)gemm_f32_slices(r, a->H, a->nL * a->H, a->num_sms) * r *
                              a->H * 4);
    DF_CUDA(a->zbuf.ensure(zb), "scratch allocation");
  }
  return DFLASH_OK;
}

int dflash_cache_create(const dflash_attn* a, int batch, int capacity_rows,
                        dflash_cache** out) {
  if (out == nullptr) return fail(DFLASH_ERR_ARG, "out is null");
  *out = nullptr;
  if (int r = check_attn(a)) return r;
  if (batch <= 0 || capacity_rows <= 0)
    return fail(DFLASH_ERR_ARG, "batch and capacity_rows must be positive");
  if (batch > kMaxBatch) return fail(DFLASH_ERR_SHAPE, "batch above %d", kMaxBatch);
  dflash_cache* c = new dflash_cache();
  c->batch = batch;
  c->cap = capacity_rows;
  c->nkv = a->nkv;
  c->d = a->d;
  c->dt = a->dt;
  c->device = a->device;
  c->len.assign(batch, 0);
  const size_t bytes = (size_t)batch * a->nkv * capacity_rows * a->d * dtype_size(a->dt);
  cudaError_t e = cudaMalloc(&c->k, bytes);
  if (e == cudaSuccess) e = cudaMalloc(&c->v, bytes);
  if (e == cudaSuccess) e = cudaMemset(c->k, 0, bytes);
  if (e == cudaSuccess) e = cudaMemset(c->v, 0, bytes);
  if (e != cudaSuccess) {
    dflash_cache_destroy(c);
    return cuda_fail(e, "cache allocation");
  }
  *out = c;
  return DFLASH_OK;
}

int dflash_cache_destroy(dflash_cache* c) {
  if (c == nullptr) return DFLASH_OK;
  cudaDeviceSynchronize();
  cudaFree(c->k);
  cudaFree(c->v);
  delete c;
  return DFLASH_OK;
}

int dflash_cache_lengths(const dflash_cache* c, int32_t* host_len) {
  if (c == nullptr || host_len == nullptr) return fail(DFLASH_ERR_ARG, "null argument");
  for (int b = 0; b < c->batch; ++b) host_len[b] = c->len[b];
  return DFLASH_OK;
}

int dflash_cache_data(const dflash_cache* c, void** k, void** v, int32_t* batch,
                      int32_t* n_kv_heads, int32_t* capacity_rows, int32_t* head_dim) {
  if (c == nullptr) return fail(DFLASH_ERR_ARG, "null cache");
  if (k) *k = c->k;
  if (v) *v = c->v;
  if (batch) *batch = c->batch;
  if (n_kv_heads) *n_kv_heads = c->nkv;
  if (capacity_rows) *capacity_rows = c->cap;
  if (head_dim) *head_dim = c->d;
  return DFLASH_OK;
}

int dflash_cache_read(const dflash_cache* c, void* k_dst, void* v_dst,
                      dflash_stream stream) {
  if (c == nullptr || k_dst == nullptr || v_dst == nullptr)
    return fail(DFLASH_ERR_ARG, "null argument");
  const size_t bytes = (size_t)c->batch * c->nkv * c->cap * c->d * dtype_size(c->dt);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DF_CUDA(cudaMemcpyAsync(k_dst, c->k, bytes, cudaMemcpyDeviceToDevice, s), "cache copy");
  DF_CUDA(cudaMemcpyAsync(v_dst, c->v, bytes, cudaMemcpyDeviceToDevice, s), "cache copy");
  return DFLASH_OK;
}

int dflash_cache_crop(dflash_cache* c, const int32_t* host_keep) {
  if (c == nullptr || host_keep == nullptr) return fail(DFLASH_ERR_ARG, "null argument");
  for (int b = 0; b < c->batch; ++b)
    if (host_keep[b] < 0 || host_keep[b] > c->len[b])
      return fail(DFLASH_ERR_RANGE, "crop(%d) of sequence %d outside [0, %d]", host_keep[b],
                  b, c->len[b]);
  for (int b = 0; b < c->batch; ++b) c->len[b] = host_keep[b];
  return DFLASH_OK;
}

int dflash_ctx_project(dflash_attn* a, const void* x, int rows, void* y,
                       dflash_stream stream) {
  if (int r = check_attn(a)) return r;
  if (a->nL == 0) return fail(DFLASH_ERR_UNSUPPORTED, "layer was created without fc");
  if (rows < 0) return fail(DFLASH_ERR_ARG, "rows must be >= 0");
  if (rows == 0) return DFLASH_OK;
  if (x == nullptr || y == nullptr) return fail(DFLASH_ERR_ARG, "null tensor");
  if (a->dt == DFLASH_BF16 && (!aligned16(x) || !aligned16(y)))
    return fail(DFLASH_ERR_ARG, "bf16 tensors must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int K = a->nL * a->H;
  // bf16: the fc's K splits write one fp32 slice each, summed by the norm
  const int n_sl = a->dt == DFLASH_BF16 ? gemm_f32_slices(rows, a->H, K, a->num_sms) : 1;
  const size_t slice = (size_t)rows * a->H;
  DF_CUDA(a->zbuf.ensure(n_sl * slice * 4), "scratch allocation");
  float* z = static_cast<float*>(a->zbuf.p);
  if (a->dt == DFLASH_BF16) {
    if (int r = ensure_gemm_scratch(a, EPI_F32, rows, 0, a->H, K, 0)) return r;
    GemmShape gs{x, rows, nullptr, 0, &a->tm_fc, &a->tm_fc256, a->H, K, 0};
    GemmScratch scr = gemm_scratch(a);
    scr.f32_slices = 1;
    scr.slice_stride = slice;
    TraceScope tr(a, DFLASH_K_FC, s);
    DF_CUDA(launch_gemm_bf16(gs, EPI_F32, z, a->H, nullptr, nullptr, scr, a->num_sms, a->err, s),
            "fc launch");
  } else {
    TraceScope tr(a, DFLASH_K_FC, s);
    DF_CUDA(launch_gemm_f32(static_cast<const float*>(x), rows,
                            static_cast<const float*>(a->w_fc), a->H, K, z, a->H, s),
            "fp32 fc");
  }
  TraceScope tr(a, DFLASH_K_NORM, s);
  DF_CUDA(launch_row_rmsnorm(z, rows, a->H, a->hidden_norm, a->cfg.rms_eps, y,
                             a->dt == DFLASH_BF16, n_sl, slice, s),
          "hidden_norm launch");
  return DFLASH_OK;
}

int dflash_attn_forward(dflash_attn* a, dflash_cache* c, int batch, int q_len,
                        const void* noise, const void* target_hidden,
                        const int32_t* host_n_ctx, const int32_t* positions, void* out,
                        dflash_stream stream) {
  if (int r = check_attn(a)) return r;
  if (c == nullptr) return fail(DFLASH_ERR_ARG, "null cache");
  if (noise == nullptr || host_n_ctx == nullptr || positions == nullptr || out == nullptr)
    return fail(DFLASH_ERR_ARG, "null tensor");
  if (batch <= 0 || q_len <= 0) return fail(DFLASH_ERR_ARG, "batch and q_len must be positive");
  if (batch != c->batch)
    return fail(DFLASH_ERR_SHAPE, "batch %d differs from the cache batch %d", batch, c->batch);
  if (c->nkv != a->nkv || c->d != a->d || c->dt != a->dt)
    return fail(DFLASH_ERR_SHAPE, "cache geometry does not match the layer");
  if (a->dt == DFLASH_BF16 && a->g * q_len > 128)
    return fail(DFLASH_ERR_UNSUPPORTED, "groups * q_len = %d above 128", a->g * q_len);
  long long total_ctx = 0;
  for (int b = 0; b < batch; ++b) {
    if (host_n_ctx[b] < 0) return fail(DFLASH_ERR_ARG, "n_ctx[%d] < 0", b);
    total_ctx += host_n_ctx[b];
    if ((long long)c->len[b] + host_n_ctx[b] + q_len > c->cap)
      return fail(DFLASH_ERR_CAPACITY, "sequence %d: %d cached + %d + %d rows exceed capacity %d",
                  b, c->len[b], host_n_ctx[b], q_len, c->cap);
  }
  if (total_ctx > 0 && target_hidden == nullptr)
    return fail(DFLASH_ERR_ARG, "target_hidden is null but n_ctx is not all zero");
  const long long rows_noise = (long long)batch * q_len;
  if (rows_noise + total_ctx > (1LL << 30)) return fail(DFLASH_ERR_SHAPE, "too many rows");
  if (a->dt == DFLASH_BF16 &&
      (!aligned16(noise) || !aligned16(out) || (total_ctx > 0 && !aligned16(target_hidden))))
    return fail(DFLASH_ERR_ARG, "bf16 tensors must be 16-byte aligned");
  const int rc = forward_core(a, KvView::of(c), batch, q_len, noise, target_hidden, host_n_ctx,
                              c->len.data(), positions, out, stream);
  if (rc != DFLASH_OK) return rc;
  for (int b = 0; b < batch; ++b) c->len[b] += host_n_ctx[b] + q_len;
  return DFLASH_OK;
}

int dflash_paged_cache_create(const dflash_attn* a, int n_pages, int page_size,
                              dflash_paged_cache** out) {
  if (out == nullptr) return fail(DFLASH_ERR_ARG, "out is null");
  *out = nullptr;
  if (int r = check_attn(a)) return r;
  if (a->dt != DFLASH_BF16) return fail(DFLASH_ERR_UNSUPPORTED, "paged caches need a bf16 layer");
  if (n_pages <= 0) return fail(DFLASH_ERR_ARG, "n_pages must be positive");
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
    return fail(DFLASH_ERR_ARG, "page_size must be 16, 32, 64 or 128");
  if ((long long)n_pages * a->nkv * page_size >= (1LL << 31))
    return fail(DFLASH_ERR_SHAPE, "too many cache rows");
  dflash_paged_cache* c = new dflash_paged_cache();
  c->n_pages = n_pages;
  c->page_size = page_size;
  c->nkv = a->nkv;
  c->d = a->d;
  c->dt = a->dt;
  c->device = a->device;
  const size_t bytes = (size_t)n_pages * a->nkv * page_size * a->d * dtype_size(a->dt);
  cudaError_t e = cudaMalloc(&c->k, bytes);
  if (e == cudaSuccess) e = cudaMalloc(&c->v, bytes);
  // zeroed: keys past a sequence's end in its last tile are read (and masked)
  if (e == cudaSuccess) e = cudaMemset(c->k, 0, bytes);
  if (e == cudaSuccess) e = cudaMemset(c->v, 0, bytes);
  if (e != cudaSuccess) {
    dflash_paged_cache_destroy(c);
    return cuda_fail(e, "paged cache allocation");
  }
  *out = c;
  return DFLASH_OK;
}

int dflash_paged_cache_destroy(dflash_paged_cache* c) {
  if (c == nullptr) return DFLASH_OK;
  cudaDeviceSynchronize();
  cudaFree(c->k);
  cudaFree(c->v);
  delete c;
  return DFLASH_OK;
}

int dflash_paged_cache_data(const dflash_paged_cache* c, void** k, void** v, int32_t* n_pages,
                            int32_t* n_kv_heads, int32_t* page_size, int32_t* head_dim) {
  if (c == nullptr) return fail(DFLASH_ERR_ARG, "null cache");
  if (k) *k = c->k;
  if (v) *v = c->v;
  if (n_pages) *n_pages = c->n_pages;
  if (n_kv_heads) *n_kv_heads = c->nkv;
  if (page_size) *page_size = c->page_size;
  if (head_dim) *head_dim = c->d;
  return DFLASH_OK;
}

int dflash_paged_cache_read(const dflash_paged_cache* c, void* k_dst, void* v_dst,
                            dflash_stream stream) {
  if (c == nullptr || k_dst == nullptr || v_dst == nullptr)
    return fail(DFLASH_ERR_ARG, "null argument");
  const size_t bytes = (size_t)c->n_pages * c->nkv * c->page_size * c->d * dtype_size(c->dt);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DF_CUDA(cudaMemcpyAsync(k_dst, c->k, bytes, cudaMemcpyDeviceToDevice, s), "cache copy");
  DF_CUDA(cudaMemcpyAsync(v_dst, c->v, bytes, cudaMemcpyDeviceToDevice, s), "cache copy");
  return DFLASH_OK;
}

int dflash_attn_forward_paged(dflash_attn* a, dflash_paged_cache* c, int batch, int q_len,
                              const void* noise, const void* target_hidden,
                              const int32_t* host_n_ctx, const int32_t* host_len_before,
                              const int32_t* positions, const int32_t* slot_mapping,
                              const int32_t* block_table, int bt_stride, void* out,
                              dflash_stream stream) {
  if (int r = check_attn(a)) return r;
  if (c == nullptr) return fail(DFLASH_ERR_ARG, "null cache");
  if (noise == nullptr || host_n_ctx == nullptr || host_len_before == nullptr ||
      positions == nullptr || slot_mapping == nullptr || block_table == nullptr ||
      out == nullptr)
    return fail(DFLASH_ERR_ARG, "null tensor");
  if (batch <= 0 || q_len <= 0) return fail(DFLASH_ERR_ARG, "batch and q_len must be positive");
  if (batch > kMaxBatch) return fail(DFLASH_ERR_SHAPE, "batch above %d", kMaxBatch);
  if (c->nkv != a->nkv || c->d != a->d || c->dt != a->dt || c->device != a->device)
    return fail(DFLASH_ERR_SHAPE, "cache geometry does not match the layer");
  if (a->g * q_len > 128)
    return fail(DFLASH_ERR_UNSUPPORTED, "groups * q_len = %d above 128", a->g * q_len);
  if (bt_stride <= 0) return fail(DFLASH_ERR_ARG, "bt_stride must be positive");
  long long total_ctx = 0;
  std::vector<int> len_before(batch);
  for (int b = 0; b < batch; ++b) {
    if (host_n_ctx[b] < 0) return fail(DFLASH_ERR_ARG, "n_ctx[%d] < 0", b);
    if (host_len_before[b] < 0) return fail(DFLASH_ERR_ARG, "len_before[%d] < 0", b);
    total_ctx += host_n_ctx[b];
    const long long len = (long long)host_len_before[b] + host_n_ctx[b] + q_len;
    if (len > (long long)bt_stride * c->page_size)
      return fail(DFLASH_ERR_CAPACITY, "sequence %d: %lld rows exceed %d block-table pages",
                  b, len, bt_stride);
    len_before[b] = host_len_before[b];
  }
  if (total_ctx > 0 && target_hidden == nullptr)
    return fail(DFLASH_ERR_ARG, "target_hidden is null but n_ctx is not all zero");
  const long long rows_noise = (long long)batch * q_len;
  if (rows_noise + total_ctx > (1LL << 30)) return fail(DFLASH_ERR_SHAPE, "too many rows");
  if (!aligned16(noise) || !aligned16(out) || (total_ctx > 0 && !aligned16(target_hidden)))
    return fail(DFLASH_ERR_ARG, "bf16 tensors must be 16-byte aligned");
  KvView kv;
  kv.k = c->k;
  kv.v = c->v;
  kv.cap = c->page_size;
  kv.rows_total = (long long)c->n_pages * c->nkv * c->page_size;
  kv.slot_mapping = slot_mapping;
  kv.block_table = block_table;
  kv.bt_stride = bt_stride;
  kv.page_size = c->page_size;
  kv.n_pages = c->n_pages;
  return forward_core(a, kv, batch, q_len, noise, target_hidden, host_n_ctx, len_before.data(),
                      positions, out, stream);
}

int dflash_kv_group_create(dflash_attn* const* layers, int n_layers, dflash_kv_group** out) {
  if (out == nullptr || layers == nullptr) return fail(DFLASH_ERR_ARG, "null argument");
  *out = nullptr;
  if (n_layers < 1 || n_layers > kMaxGroupLayers)
    return fail(DFLASH_ERR_ARG, "n_layers must be in 1..%d", kMaxGroupLayers);
  const dflash_attn* a0 = layers[0];
  if (a0 == nullptr) return fail(DFLASH_ERR_ARG, "null layer handle");
  if (a0->dt != DFLASH_BF16) return fail(DFLASH_ERR_UNSUPPORTED, "layer groups need bf16 layers");
  for (int l = 0; l < n_layers; ++l) {
    const dflash_attn* a = layers[l];
    if (a == nullptr) return fail(DFLASH_ERR_ARG, "null layer handle %d", l);
    if (a->dt != a0->dt || a->H != a0->H || a->nkv != a0->nkv || a->d != a0->d ||
        a->device != a0->device || a->max_pos != a0->max_pos ||
        a->cfg.rms_eps != a0->cfg.rms_eps || a->cfg.rope_theta != a0->cfg.rope_theta)
      return fail(DFLASH_ERR_SHAPE,
                  "layer %d differs from layer 0 (dtype, hidden, kv heads, head_dim, device, "
                  "max_position, eps or rope_theta)", l);
  }
  dflash_kv_group* g = new dflash_kv_group();
  g->n_layers = n_layers;
  g->device = a0->device;
  g->num_sms = a0->num_sms;
  const size_t kv_rows = 2 * (size_t)a0->nkv * a0->d, H = a0->H;
  cudaError_t e = cudaMalloc(&g->w_kv, n_layers * kv_rows * H * 2);
  for (int l = 0; l < n_layers && e == cudaSuccess; ++l) {
    g->layers[l] = layers[l];
    // K and V rows follow the Q rows in the layer's stacked weight
    const char* src = static_cast<const char*>(layers[l]->w_qkv) + (size_t)layers[l]->nq *
                                                                          layers[l]->d * H * 2;
    e = cudaMemcpy(static_cast<char*>(g->w_kv) + l * kv_rows * H * 2, src, kv_rows * H * 2,
                   cudaMemcpyDeviceToDevice);
  }
  if (e != cudaSuccess) {
    dflash_kv_group_destroy(g);
    return cuda_fail(e, "layer group weights");
  }
  if (make_tmap_bf16_rows(&g->tm, g->w_kv, n_layers * kv_rows, (int)H, 128) != 0 ||
      make_tmap_bf16_rows(&g->tm256, g->w_kv, n_layers * kv_rows, (int)H, 256) != 0) {
    dflash_kv_group_destroy(g);
    return fail(DFLASH_ERR_CUDA, "tensor map encoding failed");
  }
  *out = g;
  return DFLASH_OK;
}

int dflash_kv_group_destroy(dflash_kv_group* g) {
  if (g == nullptr) return DFLASH_OK;
  cudaDeviceSynchronize();
  cudaFree(g->w_kv);
  g->gemm_partial.release();
  g->gemm_counters.release();
  delete g;
  return DFLASH_OK;
}

int dflash_kv_group_append(dflash_kv_group* g, dflash_cache* const* caches, int batch,
                           const void* target_hidden, const int32_t* host_n_ctx,
                           const int32_t* positions, dflash_stream stream) {
  if (g == nullptr || caches == nullptr || host_n_ctx == nullptr)
    return fail(DFLASH_ERR_ARG, "null argument");
  const dflash_attn* a0 = g->layers[0];
  if (batch <= 0) return fail(DFLASH_ERR_ARG, "batch must be positive");
  long long rows = 0;
  for (int b = 0; b < batch; ++b) {
    if (host_n_ctx[b] < 0) return fail(DFLASH_ERR_ARG, "n_ctx[%d] < 0", b);
    rows += host_n_ctx[b];
  }
  for (int l = 0; l < g->n_layers; ++l) {
    const dflash_cache* c = caches[l];
    if (c == nullptr) return fail(DFLASH_ERR_ARG, "null cache %d", l);
    if (c->batch != batch) return fail(DFLASH_ERR_SHAPE, "cache %d batch differs", l);
    if (c->nkv != a0->nkv || c->d != a0->d || c->dt != a0->dt)
      return fail(DFLASH_ERR_SHAPE, "cache %d geometry does not match the layers", l);
    for (int b = 0; b < batch; ++b) {
      if (c->len[b] != caches[0]->len[b])
        return fail(DFLASH_ERR_SHAPE, "caches 0 and %d hold different lengths (sequence %d)", l, b);
      if ((long long)c->len[b] + host_n_ctx[b] > c->cap)
        return fail(DFLASH_ERR_CAPACITY, "cache %d sequence %d: %d + %d rows exceed capacity %d",
                    l, b, c->len[b], host_n_ctx[b], c->cap);
    }
  }
  if (rows == 0) return DFLASH_OK;
  if (rows > (1LL << 30)) return fail(DFLASH_ERR_SHAPE, "too many rows");
  if (target_hidden == nullptr || positions == nullptr) return fail(DFLASH_ERR_ARG, "null tensor");
  if (!aligned16(target_hidden)) return fail(DFLASH_ERR_ARG, "bf16 tensors must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SeqTable st;
  st.n = batch;
  st.q_len = 0;  // context rows only: position index = row index
  st.ctx_off[0] = 0;
  for (int b = 0; b < batch; ++b) {
    st.ctx_off[b + 1] = st.ctx_off[b] + host_n_ctx[b];
    st.cache_len[b] = caches[0]->len[b];
  }
  QkvOut o{};
  o.n_heads = a0->nq;
  o.n_kv = a0->nkv;
  o.groups = a0->g;
  o.q_block = 1;
  o.max_pos = a0->max_pos;
  o.eps = a0->cfg.rms_eps;
  o.q_scale = 1.f;
  o.positions = positions;
  o.rope = a0->rope;
  o.n_layers = g->n_layers;
  for (int l = 0; l < g->n_layers; ++l) {
    o.g_cache_k[l] = caches[l]->k;
    o.g_cache_v[l] = caches[l]->v;
    o.g_k_norm[l] = g->layers[l]->k_norm;
    o.g_cap[l] = caches[l]->cap;
  }
  const int n = g->n_layers * 2 * a0->nkv * a0->d;
  int n_counters = 0;
  const size_t bytes = gemm_scratch_bytes(EPI_QKV, (int)rows, 0, n, a0->H, 0, g->num_sms,
                                          &n_counters);
  DF_CUDA(g->gemm_partial.ensure(std::max<size_t>(bytes, 256)), "scratch allocation");
  DF_CUDA(g->gemm_counters.ensure((size_t)std::max(n_counters, 64) * sizeof(int), true),
          "scratch allocation");
  GemmScratch scr;
  scr.partial = static_cast<float*>(g->gemm_partial.p);
  scr.partial_bytes = g->gemm_partial.bytes;
  scr.counters = static_cast<int*>(g->gemm_counters.p);
  scr.n_counters = (int)(g->gemm_counters.bytes / sizeof(int));
  GemmShape gs{target_hidden, (int)rows, nullptr, 0, &g->tm, &g->tm256, n, a0->H, 0};
  {
    TraceScope tr(g->layers[0], DFLASH_K_QKV, s);
    DF_CUDA(launch_gemm_bf16(gs, EPI_QKV, nullptr, 0, &o, &st, scr, g->num_sms, a0->err, s),
            "layer group projection launch");
  }
  for (int l = 0; l < g->n_layers; ++l)
    for (int b = 0; b < batch; ++b) caches[l]->len[b] += host_n_ctx[b];
  return DFLASH_OK;
}

int dflash_mlp_create(int hidden, int intermediate, float rms_eps, const void* gate_w,
                      const void* up_w, const void* down_w, const void* input_norm_w,
                      const void* post_norm_w, dflash_mlp** out) {
  if (out == nullptr) return fail(DFLASH_ERR_ARG, "null output handle");
  *out = nullptr;
  if (!gate_w || !up_w || !down_w || !input_norm_w || !post_norm_w)
    return fail(DFLASH_ERR_ARG, "a weight pointer is null");
  if (hidden <= 0 || hidden % 128 != 0 || hidden > 8192)
    return fail(DFLASH_ERR_SHAPE, "hidden must be a positive multiple of 128, at most 8192");
  if (intermediate <= 0 || intermediate % 128 != 0)
    return fail(DFLASH_ERR_SHAPE, "intermediate must be a positive multiple of 128");
  if (!(rms_eps >= 0.f)) return fail(DFLASH_ERR_SHAPE, "rms_eps must be >= 0");
  dflash_mlp* m = new dflash_mlp();
  m->H = hidden;
  m->I = intermediate;
  m->eps = rms_eps;
  cudaGetDevice(&m->device);
  cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device);
  const size_t H = hidden, I = intermediate;
  cudaError_t e = cudaMalloc(&m->w_gu, 2 * I * H * 2);
  if (e == cudaSuccess) e = cudaMalloc(&m->w_d, H * I * 2);
  if (e == cudaSuccess) e = cudaMalloc(&m->in_norm, H * 4);
  if (e == cudaSuccess) e = cudaMalloc(&m->post_norm, H * 4);
  // gate rows 64c .. 64c+63 -> rows 128c .., up rows -> rows 128c + 64 ..
  const size_t chunk = 64 * H * 2;
  if (e == cudaSuccess)
    e = cudaMemcpy2D(m->w_gu, 2 * chunk, gate_w, chunk, chunk, I / 64, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy2D(static_cast<char*>(m->w_gu) + chunk, 2 * chunk, up_w, chunk, chunk, I / 64,
                     cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(m->w_d, down_w, H * I * 2, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess) e = (cudaError_t)launch_to_f32(input_norm_w, 1, m->in_norm, H, 0);
  if (e == cudaSuccess) e = (cudaError_t)launch_to_f32(post_norm_w, 1, m->post_norm, H, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    dflash_mlp_destroy(m);
    return cuda_fail(e, "mlp weights");
  }
  if (make_tmap_bf16_rows(&m->tm_gu, m->w_gu, 2 * I, (int)H, 128) != 0 ||
      make_tmap_bf16_rows(&m->tm_gu256, m->w_gu, 2 * I, (int)H, 256) != 0 ||
      make_tmap_bf16_rows(&m->tm_d, m->w_d, H, (int)I, 128) != 0 ||
      make_tmap_bf16_rows(&m->tm_d256, m->w_d, H, (int)I, 256) != 0) {
    dflash_mlp_destroy(m);
    return fail(DFLASH_ERR_CUDA, "tensor map encoding failed");
  }
  *out = m;
  return DFLASH_OK;
}

int dflash_mlp_destroy(dflash_mlp* m) {
  if (m == nullptr) return DFLASH_OK;
  cudaDeviceSynchronize();
  cudaFree(m->w_gu);
  cudaFree(m->w_d);
  cudaFree(m->in_norm);
  cudaFree(m->post_norm);
  for (df::Buf* b : {&m->y, &m->attn_out, &m->act, &m->gemm_partial, &m->gemm_counters})
    b->release();
  delete m;
  return DFLASH_OK;
}

int dflash_decoder_layer_forward(dflash_attn* a, dflash_mlp* m, dflash_cache* c, int batch,
                                 int q_len, const void* hidden_in, const void* residual_in,
                                 const void* target_hidden, const int32_t* host_n_ctx,
                                 const int32_t* positions, void* hidden_out, void* residual_out,
                                 dflash_stream stream) {
  if (int r = check_attn(a)) return r;
  if (m == nullptr) return fail(DFLASH_ERR_ARG, "null mlp handle");
  if (a->dt != DFLASH_BF16) return fail(DFLASH_ERR_UNSUPPORTED, "decoder layers need bf16");
  if (m->H != a->H) return fail(DFLASH_ERR_SHAPE, "mlp hidden %d differs from the layer's %d",
                                m->H, a->H);
  if (hidden_in == nullptr || hidden_out == nullptr || residual_out == nullptr)
    return fail(DFLASH_ERR_ARG, "null tensor");
  if (batch <= 0 || q_len <= 0) return fail(DFLASH_ERR_ARG, "batch and q_len must be positive");
  if (!aligned16(hidden_in) || !aligned16(hidden_out) || !aligned16(residual_out) ||
      (residual_in && !aligned16(residual_in)))
    return fail(DFLASH_ERR_ARG, "bf16 tensors must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int rows = batch * q_len;
  const size_t H = m->H, I = m->I;
  DF_CUDA(m->y.ensure((size_t)rows * H * 2), "scratch allocation");
  DF_CUDA(m->attn_out.ensure((size_t)rows * H * 2), "scratch allocation");
  DF_CUDA(m->act.ensure((size_t)rows * I * 2), "scratch allocation");
  int n_counters = 0;
  size_t bytes = std::max(
      gemm_scratch_bytes(EPI_SWIGLU, rows, 0, (int)(2 * I), (int)H, 0, m->num_sms, &n_counters),
      gemm_scratch_bytes(EPI_BF16, rows, 0, (int)H, (int)I, 0, m->num_sms, nullptr));
  int n2 = 0;
  gemm_scratch_bytes(EPI_BF16, rows, 0, (int)H, (int)I, 0, m->num_sms, &n2);
  DF_CUDA(m->gemm_partial.ensure(std::max<size_t>(bytes, 256)), "scratch allocation");
  DF_CUDA(m->gemm_counters.ensure((size_t)std::max({n_counters, n2, 64}) * sizeof(int), true),
          "scratch allocation");
  GemmScratch scr;
  scr.partial = static_cast<float*>(m->gemm_partial.p);
  scr.partial_bytes = m->gemm_partial.bytes;
  scr.counters = static_cast<int*>(m->gemm_counters.p);
  scr.n_counters = (int)(m->gemm_counters.bytes / sizeof(int));
  // r1 = hidden (+ residual) -> residual_out; y = input_norm(r1)
  {
    TraceScope tr(a, DFLASH_K_MLP, s);
    DF_CUDA(launch_add_rmsnorm(hidden_in, residual_in, rows, (int)H, m->in_norm, m->eps,
                               residual_out, m->y.p, s),
            "add + norm launch");
  }
  if (int r = dflash_attn_forward(a, c, batch, q_len, m->y.p, target_hidden, host_n_ctx,
                                  positions, m->attn_out.p, stream))
    return r;
  // r2 = r1 + attention -> residual_out; y = post_norm(r2); out = mlp(y)
  TraceScope tr(a, DFLASH_K_MLP, s);
  DF_CUDA(launch_add_rmsnorm(residual_out, m->attn_out.p, rows, (int)H, m->post_norm, m->eps,
                             residual_out, m->y.p, s),
          "add + norm launch");
  GemmShape g1{m->y.p, rows, nullptr, 0, &m->tm_gu, &m->tm_gu256, (int)(2 * I), (int)H, 0};
  DF_CUDA(launch_gemm_bf16(g1, EPI_SWIGLU, m->act.p, (int)I, nullptr, nullptr, scr, m->num_sms,
                           a->err, s),
          "gate/up projection launch");
  GemmShape g2{m->act.p, rows, nullptr, 0, &m->tm_d, &m->tm_d256, (int)H, (int)I, 0};
  DF_CUDA(launch_gemm_bf16(g2, EPI_BF16, hidden_out, (int)H, nullptr, nullptr, scr, m->num_sms,
                           a->err, s),
          "down projection launch");
  return DFLASH_OK;
}

int dflash_attn_forward_packed(dflash_attn* a, int batch, int seq, int n_blocks,
                               int block_size, const void* noise, const void* target_hidden,
                               const int32_t* anchors, void* out, dflash_stream stream) {
  if (int r = check_attn(a)) return r;
  if (noise == nullptr || target_hidden == nullptr || anchors == nullptr || out == nullptr)
    return fail(DFLASH_ERR_ARG, "null tensor");
  if (batch <= 0 || seq <= 0 || n_blocks <= 0 || block_size <= 0)
    return fail(DFLASH_ERR_ARG, "sizes must be positive");
  if (batch > kMaxBatch) return fail(DFLASH_ERR_SHAPE, "batch above %d", kMaxBatch);
  if (a->cfg.sliding_window > 0)
    return fail(DFLASH_ERR_UNSUPPORTED, "packed layout on a sliding-window layer");
  if (a->cfg.causal) return fail(DFLASH_ERR_UNSUPPORTED, "packed layout on a causal layer");
  if (a->dt == DFLASH_BF16 && a->g * block_size > 128)
    return fail(DFLASH_ERR_UNSUPPORTED, "groups * block_size = %d above 128",
                a->g * block_size);
  const long long q_len = (long long)n_blocks * block_size;
  const long long per = seq + q_len;
  if ((long long)batch * per > (1LL << 30)) return fail(DFLASH_ERR_SHAPE, "too many rows");
  if (a->dt == DFLASH_BF16 && (!aligned16(noise) || !aligned16(out) || !aligned16(target_hidden)))
    return fail(DFLASH_ERR_ARG, "bf16 tensors must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t es = dtype_size(a->dt);
  const size_t qd = (size_t)a->nq * a->d;
  const long long rows_noise = batch * q_len;
  DF_CUDA(a->packed_pos.ensure((size_t)batch * per * 4), "scratch allocation");
  DF_CUDA(a->packed_k.ensure((size_t)batch * a->nkv * per * a->d * es), "scratch allocation");
  DF_CUDA(a->packed_v.ensure((size_t)batch * a->nkv * per * a->d * es), "scratch allocation");
  DF_CUDA(a->qbuf.ensure(rows_noise * qd * es), "scratch allocation");
  DF_CUDA(a->attn_out.ensure(rows_noise * qd * es), "scratch allocation");
  int* pos = static_cast<int*>(a->packed_pos.p);
  {
    TraceScope tr(a, DFLASH_K_MISC, s);
    DF_CUDA(launch_packed_positions(anchors, batch, seq, n_blocks, block_size, pos, a->err, s),
            "positions launch");
  }
  SeqTable st;
  st.n = batch;
  st.q_len = (int)q_len;
  for (int b = 0; b <= batch; ++b) st.ctx_off[b] = b * seq;
  for (int b = 0; b < batch; ++b) st.cache_len[b] = 0;
  QkvOut o = make_qkv_out(a, pos, a->qbuf.p, a->packed_k.p, a->packed_v.p, (int)per, block_size);
  if (int r = run_qkv(a, noise, (int)rows_noise, target_hidden, batch * seq, o, st, s)) return r;
  AttnArgs aa{};
  aa.mode = 1;
  aa.batch = batch;
  aa.n_kv = a->nkv;
  aa.groups = a->g;
  aa.head_dim = a->d;
  aa.q_len = (int)q_len;
  aa.q_block = block_size;
  aa.n_blocks = n_blocks;
  aa.tile_blocks = std::max(1, 128 / (a->g * block_size));
  aa.cap = (int)per;
  aa.window = 0;
  aa.seq = seq;
  aa.anchors = anchors;
  aa.out = a->attn_out.p;
  aa.err = a->err;
  if (a->dt == DFLASH_BF16) {
    const int n_tiles = (n_blocks + aa.tile_blocks - 1) / aa.tile_blocks;
    aa.n_units = batch * a->nkv * n_tiles;
    TraceScope tr(a, DFLASH_K_ATTN, s);
    DF_CUDA(launch_attn_bf16(aa, nullptr, a->qbuf.p, rows_noise * a->nq, a->packed_k.p,
                             a->packed_v.p, (long long)batch * a->nkv * per, s),
            "attention launch");
  } else {
    TraceScope tr(a, DFLASH_K_ATTN, s);
    DF_CUDA(launch_attn_f32(aa, nullptr, static_cast<const float*>(a->qbuf.p),
                            static_cast<const float*>(a->packed_k.p),
                            static_cast<const float*>(a->packed_v.p), s),
            "fp32 attention launch");
  }
  return run_o_proj(a, (int)rows_noise, out, s);
}

namespace {

// shared checks of the packed attention core entry points
int check_packed_core(const dflash_attn* a, int batch, int seq, int n_blocks, int block_size) {
  if (a->dt != DFLASH_BF16) return fail(DFLASH_ERR_UNSUPPORTED, "packed core needs a bf16 layer");
  if (a->cfg.sliding_window > 0 || a->cfg.causal)
    return fail(DFLASH_ERR_UNSUPPORTED, "packed core on a sliding-window or causal layer");
  if (batch <= 0 || seq <= 0 || n_blocks <= 0 || block_size <= 0)
    return fail(DFLASH_ERR_ARG, "sizes must be positive");
  if (a->g * block_size != 64)
    return fail(DFLASH_ERR_UNSUPPORTED, "packed core needs groups * block_size = 64 (got %d)",
                a->g * block_size);
  const long long per = seq + (long long)n_blocks * block_size;
  if ((long long)batch * a->nkv * per > (1LL << 30) ||
      (long long)batch * n_blocks * block_size * a->nq > (1LL << 30))
    return fail(DFLASH_ERR_SHAPE, "too many rows");
  return DFLASH_OK;
}

}  // namespace

int dflash_packed_attn_core(dflash_attn* a, int batch, int seq, int n_blocks, int block_size,
                            const void* q, const void* k, const void* v, const int32_t* anchors,
                            void* out, float* lse, dflash_stream stream) {
  if (int r = check_attn(a)) return r;
  if (q == nullptr || k == nullptr || v == nullptr || anchors == nullptr || out == nullptr ||
      lse == nullptr)
    return fail(DFLASH_ERR_ARG, "null tensor");
  if (int r = check_packed_core(a, batch, seq, n_blocks, block_size)) return r;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(DFLASH_ERR_ARG, "bf16 tensors must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long q_len = (long long)n_blocks * block_size;
  const long long per = seq + q_len;
  const long long q_rows = batch * q_len * a->nq;
  DF_CUDA(a->qbuf.ensure((size_t)q_rows * a->d * 2), "scratch allocation");
  const float c = (float)(1.0 / std::sqrt((double)a->d) * 1.4426950408889634);
  {
    TraceScope tr(a, DFLASH_K_MISC, s);
    DF_CUDA(launch_packed_prep(q, nullptr, nullptr, nullptr, batch, n_blocks, block_size, a->nkv,
                               a->g, c, a->qbuf.p, nullptr, nullptr, nullptr, s),
            "packed prep launch");
  }
  AttnArgs aa{};
  aa.mode = 1;
  aa.batch = batch;
  aa.n_kv = a->nkv;
  aa.groups = a->g;
  aa.head_dim = a->d;
  aa.q_len = (int)q_len;
  aa.q_block = block_size;
  aa.n_blocks = n_blocks;
  aa.tile_blocks = 128 / (a->g * block_size);
  aa.cap = (int)per;
  aa.seq = seq;
  aa.anchors = anchors;
  aa.out = out;
  aa.lse = lse;
  aa.err = a->err;
  aa.n_units = batch * a->nkv * ((n_blocks + aa.tile_blocks - 1) / aa.tile_blocks);
  TraceScope tr(a, DFLASH_K_ATTN, s);
  DF_CUDA(launch_attn_bf16(aa, nullptr, a->qbuf.p, q_rows, k, v, (long long)batch * a->nkv * per,
                           s),
          "attention launch");
  return DFLASH_OK;
}

int dflash_packed_attn_core_backward(dflash_attn* a, int batch, int seq, int n_blocks,
                                     int block_size, const void* q, const void* k, const void* v,
                                     const void* out, const float* lse, const void* d_out,
                                     const int32_t* anchors, void* dq, void* dk, void* dv,
                                     dflash_stream stream) {
  if (int r = check_attn(a)) return r;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || lse == nullptr ||
      d_out == nullptr || anchors == nullptr || dq == nullptr || dk == nullptr || dv == nullptr)
    return fail(DFLASH_ERR_ARG, "null tensor");
  if (int r = check_packed_core(a, batch, seq, n_blocks, block_size)) return r;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(d_out) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(DFLASH_ERR_ARG, "bf16 tensors must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long q_len = (long long)n_blocks * block_size;
  const long long per = seq + q_len;
  const long long q_rows = batch * q_len * a->nq;
  DF_CUDA(a->qbuf.ensure((size_t)q_rows * a->d * 2), "scratch allocation");
  DF_CUDA(a->bwd_do.ensure((size_t)q_rows * a->d * 2), "scratch allocation");
  DF_CUDA(a->bwd_stats.ensure((size_t)q_rows * 2 * sizeof(float)), "scratch allocation");
  float* lse2 = static_cast<float*>(a->bwd_stats.p);
  float* dsum = lse2 + q_rows;
  const double scale = 1.0 / std::sqrt((double)a->d);
  {
    TraceScope tr(a, DFLASH_K_MISC, s);
    DF_CUDA(launch_packed_prep(q, d_out, out, lse, batch, n_blocks, block_size, a->nkv, a->g,
                               (float)(scale * 1.4426950408889634), a->qbuf.p, a->bwd_do.p, dsum,
                               lse2, s),
            "packed prep launch");
  }
  PackedBwdArgs ba{};
  ba.batch = batch;
  ba.seq = seq;
  ba.n_blocks = n_blocks;
  ba.block_size = block_size;
  ba.n_kv = a->nkv;
  ba.groups = a->g;
  ba.per = (int)per;
  ba.anchors = anchors;
  ba.lse2 = lse2;
  ba.dsum = dsum;
  ba.dq = dq;
  ba.dk = dk;
  ba.dv = dv;
  ba.dq_scale = (float)scale;
  const int pairs = batch * a->nkv;
  ba.n_kv_ctx_units = pairs * ((seq + 127) / 128);
  ba.kv_group = std::max(1, std::min(pairs, a->num_sms / std::max(1, (seq + 127) / 128)));
  ba.n_q_units = pairs * ((n_blocks + 1) / 2);
  ba.n_kv_own_units = pairs * (int)((q_len + 127) / 128);
  ba.err = a->err;
  TraceScope tr(a, DFLASH_K_BWD, s);
  DF_CUDA(launch_packed_bwd(ba, a->qbuf.p, a->bwd_do.p, k, v, s), "backward launch");
  return DFLASH_OK;
}

int dflash_wait_probe(dflash_attn* a, int64_t limit_ns, int arrive, dflash_stream stream) {
  if (int r = check_attn(a)) return r;
  if (limit_ns < 1000 || limit_ns > 100000000)
    return fail(DFLASH_ERR_ARG, "limit_ns must be in [1e3, 1e8] (got %lld)", (long long)limit_ns);
  if (arrive != 0 && arrive != 1) return fail(DFLASH_ERR_ARG, "arrive must be 0 or 1");
  DF_CUDA(launch_wait_probe(a->err, (unsigned long long)limit_ns, arrive,
                            static_cast<cudaStream_t>(stream)),
          "wait probe launch");
  return DFLASH_OK;
}

int dflash_read_stream_probe(dflash_attn* a, const void* matrix, int64_t rows, int64_t cols,
                             int ctas, int stages, dflash_stream stream) {
  if (int r = check_attn(a)) return r;
  if (matrix == nullptr) return fail(DFLASH_ERR_ARG, "matrix is null");
  if ((reinterpret_cast<uintptr_t>(matrix) & 15) != 0)
    return fail(DFLASH_ERR_ARG, "matrix must be 16-byte aligned");
  if (rows <= 0 || cols <= 0 || rows % 128 != 0 || cols % 64 != 0 || cols > (1 << 30) ||
      rows / 128 > (1 << 30))
    return fail(DFLASH_ERR_ARG, "rows must be a positive multiple of 128 and cols of 64");
  if (stages < 1 || stages > 12) return fail(DFLASH_ERR_ARG, "stages must be in [1, 12]");
  if (ctas < 1 || ctas > 2 * a->num_sms)
    return fail(DFLASH_ERR_ARG, "ctas must be in [1, 2 x SMs]");
  if (ctas > a->num_sms && stages > 6)
    return fail(DFLASH_ERR_ARG, "more CTAs than SMs take at most 6 stages");
  DF_CUDA(launch_read_stream(matrix, rows, cols, ctas, stages, a->err,
                             static_cast<cudaStream_t>(stream)),
          "read stream probe launch");
  return DFLASH_OK;
}

int dflash_kernel_launches(uint64_t* count) {
  if (count == nullptr) return fail(DFLASH_ERR_ARG, "count is null");
  *count = df::g_kernel_launches.load(std::memory_order_relaxed);
  return DFLASH_OK;
}

int dflash_trace_enable(dflash_attn* a, int enable) {
  if (int r = check_attn(a)) return r;
  DF_CUDA(cudaDeviceSynchronize(), "device synchronize");
  for (auto& r : a->recs) {
    a->event_pool.push_back(r.e0);
    a->event_pool.push_back(r.e1);
  }
  a->recs.clear();
  a->trace = enable != 0;
  return DFLASH_OK;
}

int dflash_trace_read(dflash_attn* a, int kind, double* total_ms, int32_t* launches) {
  if (int r = check_attn(a)) return r;
  if (kind < 0 || kind >= DFLASH_K_COUNT) return fail(DFLASH_ERR_ARG, "bad kernel kind");
  double tot = 0.0;
  int n = 0;
  for (auto& r : a->recs) {
    if (r.kind != kind) continue;
    DF_CUDA(cudaEventSynchronize(r.e1), "event synchronize");
    float ms = 0.f;
    DF_CUDA(cudaEventElapsedTime(&ms, r.e0, r.e1), "event elapsed time");
    tot += ms;
    ++n;
  }
  if (total_ms) *total_ms = tot;
  if (launches) *launches = n;
  return DFLASH_OK;
}

int dflash_device_error(dflash_attn* a, int32_t* code) {
  if (int r = check_attn(a)) return r;
  DF_CUDA(cudaDeviceSynchronize(), "device synchronize");
  int h = 0;
  DF_CUDA(cudaMemcpy(&h, a->err, sizeof(int), cudaMemcpyDeviceToHost), "error word read");
  if (code) *code = h;
  if (h != 0) {
    // a kernel that gave up may have left split counters raised: clear them
    cudaMemset(a->err, 0, sizeof(int));
    if (a->gemm_counters.p) cudaMemset(a->gemm_counters.p, 0, a->gemm_counters.bytes);
    if (a->attn_counters.p) cudaMemset(a->attn_counters.p, 0, a->attn_counters.bytes);
    cudaDeviceSynchronize();
    return fail(DFLASH_ERR_DEVICE, "device-side fault code %d", h);
  }
  return DFLASH_OK;
}

}  // extern "C"
