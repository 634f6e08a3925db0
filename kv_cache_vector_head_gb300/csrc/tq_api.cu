// C ABI entry points of libtq: argument checks on the host, then launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "tq_internal.h"
#include "tq_launch.h"

namespace tq {

static thread_local char g_msg[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
}
void clear_error() { g_msg[0] = '\0'; }

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static int num_sms() {
  static int cached = -1;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  if (cached < 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      cached = n;
    else
      cached = 148;
  }
  return cached;
}

// Checks the layer parameters and fills the kernel-side copy.
static tq_status make_params(const tq_layer_params* p, KParams* K, bool need_device_ptrs) {
  if (!p) return fail(TQ_ERR_INVALID_ARG, "null tq_layer_params");
  if (p->d != 128 && p->d != 256) return fail(TQ_ERR_UNSUPPORTED, "d must be 128 or 256");
  if (p->n_kv_heads < 1 || p->n_q_heads < p->n_kv_heads || p->n_q_heads % p->n_kv_heads)
    return fail(TQ_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
  if (p->n_q_heads / p->n_kv_heads > TQ_MAX_GQA) return fail(TQ_ERR_UNSUPPORTED, "n_q_heads / n_kv_heads must be <= 8");
  if (p->page_size != TQ_PAGE_SIZE) return fail(TQ_ERR_UNSUPPORTED, "page_size must be 16");
  if (p->window < 0) return fail(TQ_ERR_INVALID_ARG, "window must be >= 0");
  if (p->key_bits < 1 || p->key_bits > TQ_MAX_BITS || p->value_bits < 1 || p->value_bits > TQ_MAX_BITS)
    return fail(TQ_ERR_UNSUPPORTED, "key_bits and value_bits must be 1..4");
  if (p->key_qjl < 0 || p->key_qjl > 3) return fail(TQ_ERR_INVALID_ARG, "key_qjl must be 0..3 (see tq_key_correction)");
  if (p->kind != TQ_DENSE && p->kind != TQ_FWHT) return fail(TQ_ERR_INVALID_ARG, "bad transform kind");
  if (p->head_dim != 0 && (p->head_dim % 8 != 0 || p->head_dim <= p->d / 2 || p->head_dim > p->d))
    return fail(TQ_ERR_INVALID_ARG, "head_dim must be 0 or a multiple of 8 in (d/2, d]");
  if (p->key_split != 0 && p->key_split != 1) return fail(TQ_ERR_INVALID_ARG, "key_split must be 0 or 1");
  if (p->key_split && p->key_bits + 1 > TQ_MAX_BITS)
    return fail(TQ_ERR_UNSUPPORTED, "key_split needs key_bits <= 3");
  if (p->key_split && p->key_qjl == TQ_KEY_QJL)
    return fail(TQ_ERR_UNSUPPORTED, "key_split does not combine with the QJL sketch");
  if (p->key_norm_u8 != 0 && p->key_norm_u8 != 1) return fail(TQ_ERR_INVALID_ARG, "key_norm_u8 must be 0 or 1");
  if (p->qjl_structured != 0 && p->qjl_structured != 1)
    return fail(TQ_ERR_INVALID_ARG, "qjl_structured must be 0 or 1");
  if (p->qjl_structured && p->key_qjl != TQ_KEY_QJL)
    return fail(TQ_ERR_INVALID_ARG, "qjl_structured needs key_qjl == TQ_KEY_QJL");
  if (p->kivi != 0 && p->kivi != 1) return fail(TQ_ERR_INVALID_ARG, "kivi must be 0 or 1");
  if (p->kivi) {
    auto kbits_ok = [](int b) { return b == 2 || b == 4; };
    if (!kbits_ok(p->key_bits) || !kbits_ok(p->value_bits))
      return fail(TQ_ERR_UNSUPPORTED, "kivi: key_bits and value_bits must be 2 or 4");
    if (p->key_qjl || p->key_split || p->key_norm_u8 || p->qjl_structured)
      return fail(TQ_ERR_INVALID_ARG, "kivi: key_qjl, key_split, key_norm_u8, qjl_structured must be 0");
    if (p->head_dim != 0 && p->head_dim != p->d) return fail(TQ_ERR_UNSUPPORTED, "kivi: head_dim must be d");
    if (p->window < 1) return fail(TQ_ERR_INVALID_ARG, "kivi: window must be >= 1 (pages are written whole)");
  }
  if (p->key_norm_u8 && !(std::isfinite(p->key_norm_log2_lo) && std::isfinite(p->key_norm_log2_hi) &&
                          p->key_norm_log2_lo < p->key_norm_log2_hi))
    return fail(TQ_ERR_INVALID_ARG, "key_norm_u8 needs finite key_norm_log2_lo < key_norm_log2_hi");
  if (need_device_ptrs && !p->kivi) {
    if (!p->k_rot || !p->v_rot) return fail(TQ_ERR_INVALID_ARG, "null k_rot / v_rot");
    if (p->key_qjl == TQ_KEY_QJL && !p->qjl_s) return fail(TQ_ERR_INVALID_ARG, "null qjl_s with key_qjl");
    if (!aligned(p->k_rot, 16) || !aligned(p->v_rot, 16) || (p->qjl_s && !aligned(p->qjl_s, 16)))
      return fail(TQ_ERR_INVALID_ARG, "transforms must be 16-byte aligned");
  }
  K->d = p->d;
  K->dh = p->head_dim ? p->head_dim : p->d;
  K->hkv = p->n_kv_heads;
  K->hq = p->n_q_heads;
  K->G = p->n_q_heads / p->n_kv_heads;
  K->window = p->window;
  K->kb = p->key_bits;
  K->kqjl = p->key_qjl;
  K->vb = p->value_bits;
  K->kind = p->kind;
  K->k_rot = p->k_rot;
  K->v_rot = p->v_rot;
  K->qjl_s = p->qjl_s;
  K->qjl_srht = p->qjl_structured;
  for (int i = 0; i < 16; ++i) {
    K->kc[i] = p->k_centroids[i];
    K->kt[i] = p->k_bounds[i];
    K->vc[i] = p->v_centroids[i];
    K->vt[i] = p->v_bounds[i];
  }
  // Walsh coefficients a_S = 2^-(b-1) sum_m c(m) (-1)^popcount(m & S), c(m) = C[half + m]
  auto walsh = [](const float* c, int bits, float* a) {
    const int half = 1 << (bits - 1);
    for (int S = 0; S < 8; ++S) {
      double acc = 0;
      if (S < half)
        for (int m = 0; m < half; ++m) acc += (double)c[half + m] * ((__builtin_popcount(m & S) & 1) ? -1.0 : 1.0);
      a[S] = S < half ? (float)(acc / half) : 0.f;
    }
  };
  walsh(p->k_centroids, p->key_bits, K->akw);
  walsh(p->v_centroids, p->value_bits, K->avw);
  K->ksplit = p->key_split;
  for (int i = 0; i < 16; ++i) {
    K->kc_hi[i] = p->key_split ? p->k_hi_centroids[i] : p->k_centroids[i];
    K->kt_hi[i] = p->key_split ? p->k_hi_bounds[i] : p->k_bounds[i];
  }
  if (p->key_split) walsh(p->k_hi_centroids, p->key_bits + 1, K->akw_hi);
  else for (int i = 0; i < 8; ++i) K->akw_hi[i] = K->akw[i];
  K->knu8 = p->key_norm_u8;
  K->kn_lo = p->key_norm_u8 ? p->key_norm_log2_lo : 0.f;
  K->kn_step = p->key_norm_u8 ? (float)(((double)p->key_norm_log2_hi - p->key_norm_log2_lo) / 254.0) : 1.f;
  K->kn_inv_step = p->key_norm_u8 ? (float)(254.0 / ((double)p->key_norm_log2_hi - p->key_norm_log2_lo)) : 1.f;
  K->xb1 = 0x3C003C00u;
  K->xb2 = 0x40004000u;
  K->kp = 1 << (p->key_bits - 1 + p->key_split);
  K->vp = 1 << (p->value_bits - 1);
  const int d = p->d, w = d / 32, P = TQ_PAGE_SIZE;
  int o = 0;
  K->off_knorm = o; o += (p->key_norm_u8 ? 1 : 4) * P;
  K->off_krnorm = o; o += p->key_qjl ? 4 * P : 0;
  K->off_kcodes = o; o += 4 * p->key_bits * P * w;
  K->off_kx = o; o += p->key_split ? 4 * P * (w / 2) : 0;
  K->off_ksigns = o; o += p->key_qjl == TQ_KEY_QJL ? 4 * P * w : 0;
  K->off_vnorm = o; o += 4 * P;
  K->off_vcodes = o; o += 2 * p->value_bits * d;
  K->sub_bytes = o;
  K->kivi = p->kivi;
  K->off_kscale = K->off_kzero = K->off_vscale = K->off_vzero = 0;
  if (p->kivi) {
    o = 0;
    K->off_kscale = o; o += 2 * d;
    K->off_kzero = o; o += 2 * d;
    K->off_kcodes = o; o += 4 * P * (d * p->key_bits / 32);
    K->off_vscale = o; o += 2 * P;
    K->off_vzero = o; o += 2 * P;
    K->off_vcodes = o; o += 4 * P * (d * p->value_bits / 32);
    K->sub_bytes = o;
    K->off_knorm = K->off_krnorm = K->off_kx = K->off_ksigns = K->off_vnorm = 0;
  }
  return TQ_OK;
}

static tq_status check_dtype(tq_dtype dt) {
  if (dt != TQ_F32 && dt != TQ_BF16 && dt != TQ_F16) return fail(TQ_ERR_INVALID_ARG, "bad dtype");
  return TQ_OK;
}

static tq_status cuda_status(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    set_error("%s: %s", what, cudaGetErrorString(e));
    return TQ_ERR_CUDA;
  }
  return ok();
}

// Rows (sequences, or a prefill chunk's queries) one decode launch can take: the page grid
// and the merge put them on a grid dimension of at most 65535, the query transform their
// (row, head) vectors in tiles of 4.
static bool decode_rows_ok(const KParams& K, long long rows) {
  return rows >= 1 && rows <= 65535 && rows * K.G <= 4LL * 65535;
}

static tq_status make_cache(const tq_cache* c, const KParams& K, KCache* C, bool need_window) {
  if (!c) return fail(TQ_ERR_INVALID_ARG, "null tq_cache");
  if (!c->page_pool || !aligned(c->page_pool, 16)) return fail(TQ_ERR_INVALID_ARG, "page_pool null or not 16-byte aligned");
  if (c->n_pages < 1 || c->batch < 1 || c->max_pages_per_seq < 1)
    return fail(TQ_ERR_INVALID_ARG, "n_pages, batch and max_pages_per_seq must be >= 1");
  if (!c->block_table || !c->seq_len || !c->n_compressed) return fail(TQ_ERR_INVALID_ARG, "null block_table / counters");
  if (need_window && K.window > 0 && (!c->win_k || !c->win_v))
    return fail(TQ_ERR_INVALID_ARG, "window > 0 needs win_k and win_v");
  C->pool = reinterpret_cast<unsigned char*>(c->page_pool);
  C->n_pages = c->n_pages;
  C->block_table = c->block_table;
  C->max_pages = c->max_pages_per_seq;
  C->seq_len = c->seq_len;
  C->n_compressed = c->n_compressed;
  C->win_k = reinterpret_cast<__half*>(c->win_k);
  C->win_v = reinterpret_cast<__half*>(c->win_v);
  C->batch = c->batch;
  C->ring = K.window > 0 ? K.window + TQ_PAGE_SIZE : 0;
  C->parent = nullptr;
  return TQ_OK;
}

// Prefill workspace: the virtual sequences' counters and parent rows, then a decode workspace
// for batch * n_query sequences.
static size_t prefill_layout(const KParams& K, int batch, int n_query, int max_ctx, WsLayout* L) {
  const size_t head = ((size_t)3 * batch * n_query * sizeof(int32_t) + 255) & ~(size_t)255;
  const int S = prefill_tiles_ok(K) ? prefill_tile_splits(K, batch, n_query, max_ctx, num_sms()) : 0;
  *L = decode_ws_layout(K, batch * n_query, max_ctx, S, num_sms());
  return head + L->total;
}

}  // namespace tq

using namespace tq;

extern "C" const char* tq_last_error(void) { return g_msg; }

extern "C" size_t tq_subblock_bytes(const tq_layer_params* p) {
  KParams K;
  if (make_params(p, &K, false) != TQ_OK) return 0;
  clear_error();
  return (size_t)K.sub_bytes;
}

extern "C" tq_status tq_quantize_keys(const tq_layer_params* p, const void* k, tq_dtype dtype, int64_t n_vec,
                                      uint32_t* code_planes, uint32_t* sign_planes, float* norms, float* rnorms,
                                      tq_stream_t stream) {
  KParams K;
  tq_status s = make_params(p, &K, true);
  if (s != TQ_OK) return s;
  if ((s = check_dtype(dtype)) != TQ_OK) return s;
  if (K.kivi) return fail(TQ_ERR_UNSUPPORTED, "kivi: keys are quantized into pages only");
  if (n_vec < 0) return fail(TQ_ERR_INVALID_ARG, "n_vec < 0");
  if (n_vec == 0) return ok();
  if (!k || !code_planes || !norms) return fail(TQ_ERR_INVALID_ARG, "null input or output");
  if (K.kqjl == TQ_KEY_QJL && (!sign_planes || !rnorms))
    return fail(TQ_ERR_INVALID_ARG, "key_qjl needs sign_planes and rnorms");
  if (K.kqjl >= TQ_KEY_EDEN && !rnorms) return fail(TQ_ERR_INVALID_ARG, "scaled keys need rnorms (the scale)");
  if (!aligned(k, 16)) return fail(TQ_ERR_INVALID_ARG, "k must be 16-byte aligned");
  return cuda_status(launch_quantize_flat(K, k, dtype, n_vec, true, code_planes, sign_planes, norms, rnorms,
                                          reinterpret_cast<cudaStream_t>(stream)),
                     "tq_quantize_keys");
}

extern "C" tq_status tq_quantize_values(const tq_layer_params* p, const void* v, tq_dtype dtype, int64_t n_vec,
                                        uint32_t* code_planes, float* norms, tq_stream_t stream) {
  KParams K;
  tq_status s = make_params(p, &K, true);
  if (s != TQ_OK) return s;
  if ((s = check_dtype(dtype)) != TQ_OK) return s;
  if (K.kivi) return fail(TQ_ERR_UNSUPPORTED, "kivi: values are quantized into pages only");
  if (n_vec < 0) return fail(TQ_ERR_INVALID_ARG, "n_vec < 0");
  if (n_vec == 0) return ok();
  if (!v || !code_planes || !norms) return fail(TQ_ERR_INVALID_ARG, "null input or output");
  if (!aligned(v, 16)) return fail(TQ_ERR_INVALID_ARG, "v must be 16-byte aligned");
  return cuda_status(launch_quantize_flat(K, v, dtype, n_vec, false, code_planes, nullptr, norms, nullptr,
                                          reinterpret_cast<cudaStream_t>(stream)),
                     "tq_quantize_values");
}

extern "C" tq_status tq_append_page(const tq_layer_params* p, tq_cache* cache, const void* k, const void* v,
                                    tq_dtype dtype, int64_t n_tok, const int64_t* slot_mapping, tq_stream_t stream) {
  KParams K;
  KCache C;
  tq_status s = make_params(p, &K, true);
  if (s != TQ_OK) return s;
  if ((s = check_dtype(dtype)) != TQ_OK) return s;
  if ((s = make_cache(cache, K, &C, slot_mapping == nullptr)) != TQ_OK) return s;
  if (n_tok < 0) return fail(TQ_ERR_INVALID_ARG, "n_tok < 0");
  if (n_tok == 0) return ok();
  if (!k || !v || !aligned(k, 16) || !aligned(v, 16)) return fail(TQ_ERR_INVALID_ARG, "k / v null or not 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (slot_mapping == nullptr) {
    if (n_tok != cache->batch) return fail(TQ_ERR_INVALID_ARG, "decode-step append needs n_tok == batch");
    return cuda_status(launch_append_step(K, C, k, v, dtype, st), "tq_append_page");
  }
  if (K.kivi && n_tok % TQ_PAGE_SIZE)
    return fail(TQ_ERR_INVALID_ARG, "kivi: direct appends write whole pages (n_tok a multiple of 16)");
  return cuda_status(launch_append_direct(K, C, k, v, dtype, n_tok, reinterpret_cast<const long long*>(slot_mapping), st),
                     "tq_append_page");
}

extern "C" tq_status tq_prefill_cache(const tq_layer_params* p, tq_cache* cache, const void* k, const void* v,
                                      tq_dtype dtype, int n_tok, tq_stream_t stream) {
  KParams K;
  KCache C;
  tq_status s = make_params(p, &K, true);
  if (s != TQ_OK) return s;
  if ((s = check_dtype(dtype)) != TQ_OK) return s;
  if ((s = make_cache(cache, K, &C, true)) != TQ_OK) return s;
  if (n_tok < 0) return fail(TQ_ERR_INVALID_ARG, "n_tok < 0");
  if (n_tok > 0 && (!k || !v || !aligned(k, 16) || !aligned(v, 16)))
    return fail(TQ_ERR_INVALID_ARG, "k / v null or not 16-byte aligned");
  // the window rule of the page format: whole pages of the tokens older than the last W;
  // without a window every token is in its page (the last one may be partly filled)
  const int n_c = K.window > 0 ? TQ_PAGE_SIZE * (std::max(0, n_tok - K.window) / TQ_PAGE_SIZE) : n_tok;
  if ((n_c + TQ_PAGE_SIZE - 1) / TQ_PAGE_SIZE > cache->max_pages_per_seq)
    return fail(TQ_ERR_CAPACITY, "tq_prefill_cache: n_tok needs more pages than max_pages_per_seq");
  if ((long long)cache->batch * n_c >= (1LL << 40)) return fail(TQ_ERR_INVALID_ARG, "tq_prefill_cache: too many tokens");
  return cuda_status(launch_prefill_cache(K, C, k, v, dtype, n_tok, n_c, reinterpret_cast<cudaStream_t>(stream)),
                     "tq_prefill_cache");
}

extern "C" size_t tq_decode_workspace_size(const tq_layer_params* p, int batch, int max_ctx, int n_splits) {
  KParams K;
  if (make_params(p, &K, false) != TQ_OK || batch < 1 || max_ctx < 0 || n_splits < 0) return 0;
  if (!decode_rows_ok(K, batch)) return 0;
  clear_error();
  return decode_ws_layout(K, batch, max_ctx, n_splits, num_sms()).total;
}

extern "C" tq_status tq_decode_attention(const tq_layer_params* p, const tq_cache* cache, const void* q, tq_dtype dtype,
                                         float scale, float* out, float* lse, float* scores, void* workspace,
                                         size_t workspace_bytes, int max_ctx, int n_splits, tq_stream_t stream) {
  KParams K;
  KCache C;
  tq_status s = make_params(p, &K, true);
  if (s != TQ_OK) return s;
  if ((s = check_dtype(dtype)) != TQ_OK) return s;
  if ((s = make_cache(cache, K, &C, true)) != TQ_OK) return s;
  if (!q || !out || !workspace) return fail(TQ_ERR_INVALID_ARG, "null q / out / workspace");
  if (!aligned(workspace, 256)) return fail(TQ_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (max_ctx < 0 || n_splits < 0) return fail(TQ_ERR_INVALID_ARG, "max_ctx and n_splits must be >= 0");
  if (!(scale == scale)) return fail(TQ_ERR_INVALID_ARG, "scale is NaN");
  if (!decode_rows_ok(K, cache->batch)) return fail(TQ_ERR_INVALID_ARG, "batch must be <= 65535 and batch * G <= 262140");
  const WsLayout L = decode_ws_layout(K, cache->batch, max_ctx, n_splits, num_sms());
  if (workspace_bytes < L.total) {
    set_error("workspace too small: %zu < %zu", workspace_bytes, L.total);
    return TQ_ERR_CAPACITY;
  }
  return cuda_status(launch_decode(K, C, q, dtype, scale, out, lse, scores, workspace, L, max_ctx,
                                   reinterpret_cast<cudaStream_t>(stream)),
                     "tq_decode_attention");
}

extern "C" size_t tq_prefill_workspace_size(const tq_layer_params* p, int batch, int n_query, int max_ctx) {
  KParams K;
  if (make_params(p, &K, false) != TQ_OK || batch < 1 || n_query < 1 || max_ctx < 0) return 0;
  if (!decode_rows_ok(K, (long long)batch * n_query)) return 0;
  clear_error();
  WsLayout L;
  return prefill_layout(K, batch, n_query, max_ctx, &L);
}

extern "C" tq_status tq_prefill_attention(const tq_layer_params* p, const tq_cache* cache, int n_query, const void* q,
                                          tq_dtype dtype, float scale, float* out, float* lse, void* workspace,
                                          size_t workspace_bytes, int max_ctx, tq_stream_t stream) {
  KParams K;
  KCache C;
  tq_status s = make_params(p, &K, true);
  if (s != TQ_OK) return s;
  if ((s = check_dtype(dtype)) != TQ_OK) return s;
  if ((s = make_cache(cache, K, &C, true)) != TQ_OK) return s;
  if (n_query < 1 || !decode_rows_ok(K, (long long)cache->batch * n_query))
    return fail(TQ_ERR_INVALID_ARG, "n_query must be >= 1, batch * n_query <= 65535 and batch * n_query * G <= 262140");
  if (!q || !out || !workspace) return fail(TQ_ERR_INVALID_ARG, "null q / out / workspace");
  if (!aligned(workspace, 256)) return fail(TQ_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (max_ctx < 0) return fail(TQ_ERR_INVALID_ARG, "max_ctx must be >= 0");
  if (!(scale == scale)) return fail(TQ_ERR_INVALID_ARG, "scale is NaN");
  WsLayout L;
  const size_t need = prefill_layout(K, cache->batch, n_query, max_ctx, &L);
  if (workspace_bytes < need) {
    set_error("workspace too small: %zu < %zu", workspace_bytes, need);
    return TQ_ERR_CAPACITY;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t nv = (size_t)cache->batch * n_query;
  int32_t* seq_v = reinterpret_cast<int32_t*>(workspace);
  int32_t* nc_v = seq_v + nv;
  int32_t* parent = nc_v + nv;
  unsigned char* dws = reinterpret_cast<unsigned char*>(workspace) + (need - L.total);
  cudaError_t e = launch_prefill_virtual(C, n_query, seq_v, nc_v, parent, st);
  if (e != cudaSuccess) return cuda_status(e, "tq_prefill_attention");
  KCache V = C;
  V.seq_len = seq_v;
  V.n_compressed = nc_v;
  V.parent = parent;
  V.batch = (int)nv;
  if (prefill_tiles_ok(K))
    return cuda_status(launch_prefill_tiles(K, V, n_query, cache->batch, q, dtype, scale, out, lse, dws, L, max_ctx, st),
                       "tq_prefill_attention");
  return cuda_status(launch_decode(K, V, q, dtype, scale, out, lse, nullptr, dws, L, max_ctx, st),
                     "tq_prefill_attention");
}

extern "C" tq_status tq_check_device_error(tq_stream_t stream, uint32_t* bits_out) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e, "tq_check_device_error: stream");
  unsigned a = 0, b = 0;
  if ((e = read_clear_quant_error(&a)) != cudaSuccess) return cuda_status(e, "tq_check_device_error");
  if ((e = read_clear_decode_error(&b)) != cudaSuccess) return cuda_status(e, "tq_check_device_error");
  if (bits_out) *bits_out = a | b;
  if (a | b) {
    set_error("device error word 0x%x", a | b);
    return TQ_ERR_DEVICE_CHECK;
  }
  return ok();
}

#ifdef TQ_TEST_HOOKS
// Test build only (libtq_testhooks.so; not part of the C ABI in include/tq.h): on = 1 makes
// the first chunk of every decode page split expect 16 bytes more than its copies deliver,
// so that split's bounded wait runs out and reports TQ_DEVERR_TIMEOUT; on = 0 restores
// normal decoding.
extern "C" tq_status tq_test_wait_fault(int on) {
  return cuda_status(set_test_wait_fault(on ? 1 : 0), "tq_test_wait_fault");
}
#endif

// ------------------------------------------------------------------ decode without a workspace argument

namespace tq {
namespace {
// Scratch for tq_decode_attention_static.  In host code this symbol is only a
// stand-in: its device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_static_scratch[TQ_STATIC_SCRATCH_BYTES];
std::mutex g_static_mu;
void* g_static_ptr[256] = {};
}  // namespace
}  // namespace tq

extern "C" tq_status tq_decode_attention_static(const tq_layer_params* p, const tq_cache* cache, const void* q,
                                                tq_dtype dtype, float scale, float* out, float* lse, float* scores,
                                                int max_ctx, int n_splits, tq_stream_t stream) {
  KParams K;
  tq_status s = make_params(p, &K, true);
  if (s != TQ_OK) return s;
  if (!cache || cache->batch < 1 || max_ctx < 0 || n_splits < 0)
    return fail(TQ_ERR_INVALID_ARG, "tq_decode_attention_static: bad cache, max_ctx or n_splits");
  if (!decode_rows_ok(K, cache->batch)) return fail(TQ_ERR_INVALID_ARG, "batch must be <= 65535 and batch * G <= 262140");
  const size_t need = decode_ws_layout(K, cache->batch, max_ctx, n_splits, num_sms()).total;
  if (need > (size_t)TQ_STATIC_SCRATCH_BYTES) {
    set_error("tq_decode_attention_static: this configuration needs %zu bytes of scratch, more than the %u-byte "
              "static array; use tq_decode_attention with a workspace", need, (unsigned)TQ_STATIC_SCRATCH_BYTES);
    return TQ_ERR_CAPACITY;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "tq_decode_attention_static: cudaGetDevice");
  if (dev < 0 || dev >= 256) return fail(TQ_ERR_UNSUPPORTED, "tq_decode_attention_static: device index >= 256");
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
      e = cudaGetSymbolAddress(&g_static_ptr[dev], g_static_scratch);
      if (e != cudaSuccess) {
        g_static_ptr[dev] = nullptr;
        return cuda_status(e, "tq_decode_attention_static: cudaGetSymbolAddress");
      }
    }
    ptr = g_static_ptr[dev];
  }
  return tq_decode_attention(p, cache, q, dtype, scale, out, lse, scores, ptr, (size_t)TQ_STATIC_SCRATCH_BYTES,
                             max_ctx, n_splits, stream);
}
