// The C ABI of the quantised KV cache: configuration checks, the arena
// carve-up, the per-layer counters (L, E) and segment bounds, kernel
// launches, statistics and canonical exports.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "kvq.h"
#include "kvq_internal.h"

using kvq::Geometry;
using kvq::kGroup;
using kvq::kMaxSinks;

namespace {

thread_local std::string g_last_error;
std::atomic<int64_t> g_launches{0};

kv_status fail(kv_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

kv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KV_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

struct LayerState {
  int64_t L = 0;
  int64_t E = 0;
  bool dyn_selected = false;
  int n_dyn_sel = 0;
};

}  // namespace

struct kv_cache {
  kv_cache_config cfg;
  Geometry geo;
  uint8_t* arena = nullptr;
  int device = 0;
  int sm_count = 0;
  int stream_ctas = 0;  // 0: SM count x occupancy
  std::vector<LayerState> layers;
  cudaEvent_t ev0 = nullptr, ev1 = nullptr;
};

namespace {

// Configuration rules (the cache's contract; see kvq.h).
kv_status check_config(const kv_cache_config* c) {
  if (!c) return fail(KV_ERR_INVALID_ARG, "config is NULL");
  if (c->n_layers < 1 || c->batch < 1 || c->n_kv_heads < 1 || c->n_q_heads < 1)
    return fail(KV_ERR_INVALID_ARG, "layers, batch and head counts must be positive");
  if (c->n_q_heads % c->n_kv_heads)
    return fail(KV_ERR_INVALID_ARG, "n_q_heads must be a multiple of n_kv_heads");
  if (c->n_q_heads / c->n_kv_heads > kvq::kMaxGqa)
    return fail(KV_ERR_UNSUPPORTED, "at most 4 query heads per KV head");
  if (c->head_dim != 64 && c->head_dim != 128) return fail(KV_ERR_INVALID_ARG, "head_dim must be 64 or 128");
  if (c->group_size != kGroup) return fail(KV_ERR_INVALID_ARG, "group_size must be 32");
  if (c->mode == KV_MODE_KIVI) {
    for (int b : {c->k_bits, c->v_bits})
      if (b != 2 && b != 3 && b != 4 && b != 8) return fail(KV_ERR_INVALID_ARG, "KIVI bits must be 2, 3, 4 or 8");
    if (c->residual != kGroup) return fail(KV_ERR_INVALID_ARG, "KIVI residual must be 32 (one group)");
  } else if (c->mode == KV_MODE_TURBOQUANT) {
    for (int b : {c->k_bits, c->v_bits})
      if (b != 2 && b != 3 && b != 4) return fail(KV_ERR_INVALID_ARG, "TurboQuant bits must be 2, 3 or 4");
    if (c->residual != 0) return fail(KV_ERR_INVALID_ARG, "TurboQuant residual must be 0");
    if (c->n_dyn_sinks) return fail(KV_ERR_INVALID_ARG, "KVSink sinks are defined on KIVI groups only");
  } else {
    return fail(KV_ERR_INVALID_ARG, "unknown mode");
  }
  if (c->n_sink < 0 || c->window < 0 || c->evict_window < 0 || c->n_dyn_sinks < 0)
    return fail(KV_ERR_INVALID_ARG, "negative size");
  if (c->n_sink > kMaxSinks) return fail(KV_ERR_INVALID_ARG, "at most 32 overlay sinks");
  if (c->n_dyn_sinks > kMaxSinks) return fail(KV_ERR_INVALID_ARG, "at most 32 dynamic sinks");
  if (c->n_dyn_sinks && (c->n_sink || c->window || c->evict_window))
    return fail(KV_ERR_INVALID_ARG, "KVSink sinks exclude the StreamingLLM overlay and eviction");
  if (c->evict_window && c->evict_window < std::max(c->window, kGroup))
    return fail(KV_ERR_INVALID_ARG, "evict_window must be >= max(window, 32)");
  if (c->act_dtype != KV_DT_F16 && c->act_dtype != KV_DT_BF16)
    return fail(KV_ERR_INVALID_ARG, "act_dtype must be F16 or BF16");
  if (c->max_tokens < kGroup) return fail(KV_ERR_INVALID_ARG, "max_tokens must be >= 32");
  if (c->max_tokens > (static_cast<int64_t>(1) << 40)) return fail(KV_ERR_INVALID_ARG, "max_tokens too large");
  if (!(c->rope_base >= 0.0)) return fail(KV_ERR_INVALID_ARG, "rope_base must be >= 0");
  if (c->rope_base > 0.0 && c->rope_max_pos < 1) return fail(KV_ERR_INVALID_ARG, "rope_max_pos must be >= 1");
  if (c->v_q4_0 && (c->mode != KV_MODE_KIVI || c->v_bits != 4))
    return fail(KV_ERR_INVALID_ARG, "v_q4_0 is a 4-bit KIVI V format");
  if (c->rope_reposition && !(c->rope_base > 0.0))
    return fail(KV_ERR_INVALID_ARG, "rope_reposition needs the cache to apply RoPE (rope_base > 0)");
  if (c->max_splits < 0 || c->max_splits > 4096) return fail(KV_ERR_INVALID_ARG, "max_splits out of range");
  if (c->k_pre_rope && (!(c->rope_base > 0.0) || c->mode != KV_MODE_KIVI || c->n_dyn_sinks))
    return fail(KV_ERR_INVALID_ARG, "k_pre_rope needs rope_base > 0, KIVI mode and no KVSink sinks");
  return KV_OK;
}

Geometry make_geometry(const kv_cache_config* c) {
  Geometry g{};
  g.B = c->batch;
  g.H = c->n_kv_heads;
  g.Hq = c->n_q_heads;
  g.D = c->head_dim;
  g.gqa = c->n_q_heads / c->n_kv_heads;
  g.mode_tq = c->mode == KV_MODE_TURBOQUANT;
  g.kb = c->k_bits;
  g.vb = c->v_bits;
  g.n_sink = c->n_sink;
  g.window = c->window;
  g.evict_window = c->evict_window;
  g.n_dyn = c->n_dyn_sinks;
  g.act_bf16 = c->act_dtype == KV_DT_BF16;
  g.max_tokens = c->max_tokens;
  g.n_slots = static_cast<int>((c->max_tokens + kGroup - 1) / kGroup);
  g.tail_cap = next_pow2(std::max(c->window, kGroup - 1) + 1);
  g.n_sink_slots = std::max(1, std::max(c->n_sink, c->n_dyn_sinks));
  g.max_splits = c->max_splits ? c->max_splits : 64;
  g.chunk = kvq::chunk_layout(g.mode_tq, g.D, g.kb, g.vb);
  g.rope_max_pos = c->rope_base > 0.0 ? c->rope_max_pos : 0;
  g.rope_repos = c->rope_reposition ? 1 : 0;
  g.v_q4_0 = c->v_q4_0 ? 1 : 0;
  g.k_pre_rope = c->k_pre_rope ? 1 : 0;

  const size_t B = g.B, H = g.H, D = g.D;
  size_t off = 0;
  g.off_err = off;
  off = align256(off + 256);
  g.off_rope = off;
  off = align256(off + static_cast<size_t>(g.rope_max_pos) * D * 4);
  g.off_signs = off;
  off = align256(off + D * 4);
  g.off_cbk = off;
  off = align256(off + 32 * 4);
  g.off_cbv = off;
  off = align256(off + 32 * 4);
  const size_t ns = g.max_splits + 1;
  g.off_part_o = off;
  off = align256(off + B * g.Hq * ns * D * 4);
  g.off_part_ml = off;
  off = align256(off + B * g.Hq * ns * 2 * 4);
  g.n_cand_chunks = g.n_dyn ? static_cast<size_t>((c->max_tokens + 1023) / 1024) : 0;
  g.off_norms = off;
  off = align256(off + (g.n_dyn ? B * static_cast<size_t>(c->max_tokens) * 4 : 0));
  g.off_cand_m = off;
  off = align256(off + B * g.n_cand_chunks * kMaxSinks * 4);
  g.off_cand_p = off;
  off = align256(off + B * g.n_cand_chunks * kMaxSinks * 8);
  g.off_layers = off;
  size_t lo = 0;
  g.l_chunks = lo;
  lo = align256(lo + B * H * g.n_slots * static_cast<size_t>(g.chunk.bytes));
  g.l_tail_k = lo;
  lo = align256(lo + B * H * g.tail_cap * D * 2);
  g.l_tail_v = lo;
  lo = align256(lo + B * H * g.tail_cap * D * 2);
  g.l_sink_k = lo;
  lo = align256(lo + B * H * g.n_sink_slots * D * 2);
  g.l_sink_v = lo;
  lo = align256(lo + B * H * g.n_sink_slots * D * 2);
  g.l_sink_pos = lo;
  lo = align256(lo + B * kMaxSinks * 8);
  g.l_sink_m = lo;
  lo = align256(lo + B * kMaxSinks * 4);
  g.l_sink_mask = lo;
  lo = align256(lo + B * static_cast<size_t>(g.n_slots) * 4);
  g.layer_bytes = lo;
  g.total = off + lo * c->n_layers;
  return g;
}

kvq::LayerDev layer_dev(const kv_cache* c, int layer) {
  const Geometry& g = c->geo;
  uint8_t* base = c->arena + g.off_layers + g.layer_bytes * layer;
  kvq::LayerDev d;
  d.chunks = base + g.l_chunks;
  d.tail_k = reinterpret_cast<uint16_t*>(base + g.l_tail_k);
  d.tail_v = reinterpret_cast<uint16_t*>(base + g.l_tail_v);
  d.sink_k = reinterpret_cast<uint16_t*>(base + g.l_sink_k);
  d.sink_v = reinterpret_cast<uint16_t*>(base + g.l_sink_v);
  d.sink_pos = reinterpret_cast<int64_t*>(base + g.l_sink_pos);
  d.sink_m = reinterpret_cast<float*>(base + g.l_sink_m);
  d.sink_mask = reinterpret_cast<uint32_t*>(base + g.l_sink_mask);
  return d;
}

kvq::TablesDev tables_dev(const kv_cache* c) {
  const Geometry& g = c->geo;
  kvq::TablesDev t;
  t.rope = g.rope_max_pos ? reinterpret_cast<const float*>(c->arena + g.off_rope) : nullptr;
  t.signs = reinterpret_cast<const float*>(c->arena + g.off_signs);
  t.cb_k = reinterpret_cast<const float*>(c->arena + g.off_cbk);
  t.cb_v = reinterpret_cast<const float*>(c->arena + g.off_cbv);
  t.err_flag = reinterpret_cast<int*>(c->arena + g.off_err);
  return t;
}

int64_t q_end_of(const Geometry& g, int64_t L) { return g.mode_tq ? L : kGroup * (L / kGroup); }

int64_t fp16_begin_of(const Geometry& g, int64_t L) {
  const int64_t a = L - g.window > g.n_sink ? L - g.window : g.n_sink;
  const int64_t q = q_end_of(g, L);
  return q < a ? q : a;
}

kv_status check_layer(const kv_cache* c, int layer) {
  if (!c) return fail(KV_ERR_INVALID_ARG, "cache is NULL");
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(KV_ERR_INVALID_ARG, "layer out of range");
  return KV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// kv_append and kv_prefill_quantize: one state change; the group flush
// quantises every group the call completes in one launch, however many.
kv_status do_append(kv_cache* c, int layer, const void* k, const void* v, int n, void* stream) {
  kv_status st = check_layer(c, layer);
  if (st != KV_OK) return st;
  if (!k || !v) return fail(KV_ERR_INVALID_ARG, "k/v is NULL");
  if (!aligned16(k) || !aligned16(v)) return fail(KV_ERR_INVALID_ARG, "k/v must be 16-byte aligned");
  if (n < 1) return fail(KV_ERR_INVALID_ARG, "n_new must be >= 1");
  const Geometry& g = c->geo;
  LayerState& ls = c->layers[layer];
  const int64_t L0 = ls.L, L1 = L0 + n;
  const int64_t first = kGroup * (ls.E / kGroup);
  if (L1 - first > g.max_tokens)
    return fail(KV_ERR_CAPACITY, "append exceeds max_tokens (evict first or raise max_tokens)");
  if (g.rope_max_pos && L1 > g.rope_max_pos) return fail(KV_ERR_CAPACITY, "position beyond rope_max_pos");
  // KVSink: every call (append or prefill) folds its tokens into the
  // running top-k before its groups are quantised
  const bool select = g.n_dyn > 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  kvq::AppendArgs a{};
  a.geo = g;
  a.lay = layer_dev(c, layer);
  a.tab = tables_dev(c);
  if (g.k_pre_rope) a.tab.rope = nullptr;  // keys are stored before RoPE
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.n = n;
  a.L0 = L0;
  a.tail_from = fp16_begin_of(g, L1);
  const int64_t q0 = q_end_of(g, L0), q1 = q_end_of(g, L1);
  a.g_first = q0 / kGroup;
  a.n_groups = g.mode_tq ? 0 : static_cast<int>((q1 - q0) / kGroup);
  int64_t launches = 0;
  cudaError_t e = cudaSuccess;
  int n_sel = ls.n_dyn_sel;
  if (select) {
    n_sel = static_cast<int>(std::min<int64_t>(g.n_dyn, L1));
    kvq::SinkSelectArgs sa{};
    sa.geo = g;
    sa.lay = a.lay;
    sa.tab = a.tab;
    sa.k = a.k;
    sa.v = a.v;
    sa.n = n;
    sa.norms = reinterpret_cast<float*>(c->arena + g.off_norms);
    sa.cand_m = reinterpret_cast<float*>(c->arena + g.off_cand_m);
    sa.cand_p = reinterpret_cast<int64_t*>(c->arena + g.off_cand_p);
    sa.n_chunks = (n + 1023) / 1024;
    sa.k_sel = std::min(g.n_dyn, n);
    sa.L0 = L0;
    sa.q0 = q0;
    sa.n_old = ls.n_dyn_sel;
    sa.k_total = n_sel;
    if (n <= kvq::kSinkSmallCallTokens) {  // decode-time appends: one launch
      e = kvq::launch_sink_admit_small(sa, s, &launches);
    } else {
      e = kvq::launch_sink_select(sa, s, &launches);
      if (e == cudaSuccess) {
        a.n_dyn_sel = n_sel;
        e = kvq::launch_sink_gather(a, s, &launches);
      }
    }
  }
  a.dyn_active = (select || ls.dyn_selected) ? 1 : 0;
  a.n_dyn_sel = n_sel;
  if (e == cudaSuccess) e = kvq::launch_append(a, s, &launches);
  g_launches += launches;
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  ls.L = L1;
  if (select) {
    ls.dyn_selected = true;
    ls.n_dyn_sel = n_sel;
  }
  return KV_OK;
}

size_t act_bytes() { return 2; }

}  // namespace

extern "C" {

kv_status kv_cache_required_bytes(const kv_cache_config* cfg, size_t* device_bytes) {
  kv_status st = check_config(cfg);
  if (st != KV_OK) return st;
  if (!device_bytes) return fail(KV_ERR_INVALID_ARG, "device_bytes is NULL");
  *device_bytes = make_geometry(cfg).total;
  return KV_OK;
}

kv_status kv_cache_create(const kv_cache_config* cfg, void* device_arena, size_t arena_bytes, kv_cache** out) {
  kv_status st = check_config(cfg);
  if (st != KV_OK) return st;
  if (!out) return fail(KV_ERR_INVALID_ARG, "out is NULL");
  if (!device_arena || (reinterpret_cast<uintptr_t>(device_arena) & 255u))
    return fail(KV_ERR_INVALID_ARG, "arena must be a 256-byte aligned device pointer");
  Geometry g = make_geometry(cfg);
  if (arena_bytes < g.total) return fail(KV_ERR_INVALID_ARG, "arena smaller than kv_cache_required_bytes");
  kv_cache* c = new (std::nothrow) kv_cache();
  if (!c) return fail(KV_ERR_INVALID_ARG, "out of host memory");
  c->cfg = *cfg;
  c->geo = g;
  c->arena = static_cast<uint8_t*>(device_arena);
  c->layers.assign(cfg->n_layers, LayerState());
  for (auto& l : c->layers) l.E = cfg->n_sink;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device);
  if (const char* env = std::getenv("KVQ_STREAM_CTAS")) c->stream_ctas = std::max(0, std::atoi(env));
  // host-built tables
  std::vector<float> tmp;
  if (e == cudaSuccess && g.rope_max_pos) {
    tmp.assign(static_cast<size_t>(g.rope_max_pos) * g.D, 0.0f);
    kvq::build_rope_table(tmp.data(), g.rope_max_pos, g.D, cfg->rope_base);
    e = cudaMemcpy(c->arena + g.off_rope, tmp.data(), tmp.size() * 4, cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) {
    tmp.assign(g.D, 0.0f);
    kvq::build_signs(tmp.data(), g.D, cfg->seed);
    e = cudaMemcpy(c->arena + g.off_signs, tmp.data(), g.D * 4, cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess && g.mode_tq) {
    for (int which = 0; which < 2 && e == cudaSuccess; ++which) {
      const int bits = which ? g.vb : g.kb;
      const int L = 1 << bits;
      std::vector<double> bd(L - 1), cd(L);
      kvq::build_beta_codebook(g.D / 2.0, bits, bd.data(), cd.data());
      std::vector<float> cb(32, 0.0f);
      for (int i = 0; i < L - 1; ++i) cb[i] = static_cast<float>(bd[i]);
      for (int i = 0; i < L; ++i) cb[L - 1 + i] = static_cast<float>(cd[i]);
      e = cudaMemcpy(c->arena + (which ? g.off_cbv : g.off_cbk), cb.data(), 32 * 4, cudaMemcpyHostToDevice);
    }
  }
  if (e == cudaSuccess) e = cudaMemset(c->arena + g.off_err, 0, 256);
  if (e == cudaSuccess) {
    for (int l = 0; l < cfg->n_layers && e == cudaSuccess; ++l) {
      kvq::LayerDev d = layer_dev(c, l);
      e = cudaMemset(d.sink_mask, 0, static_cast<size_t>(g.B) * g.n_slots * 4);
      if (e == cudaSuccess) e = cudaMemset(d.sink_pos, 0, static_cast<size_t>(g.B) * kMaxSinks * 8);
    }
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "kv_cache_create");
  }
  *out = c;
  return KV_OK;
}

kv_status kv_cache_destroy(kv_cache* cache) {
  if (!cache) return fail(KV_ERR_INVALID_ARG, "cache is NULL");
  delete cache;
  return KV_OK;
}

kv_status kv_cache_reset(kv_cache* cache) {
  if (!cache) return fail(KV_ERR_INVALID_ARG, "cache is NULL");
  for (auto& l : cache->layers) l = LayerState(), l.E = cache->cfg.n_sink;
  return KV_OK;
}

kv_status kv_append(kv_cache* cache, int layer, const void* k, const void* v, int n_new, void* cuda_stream) {
  return do_append(cache, layer, k, v, n_new, cuda_stream);
}

kv_status kv_prefill_quantize(kv_cache* cache, int layer, const void* k, const void* v, int n_tokens,
                              void* cuda_stream) {
  return do_append(cache, layer, k, v, n_tokens, cuda_stream);
}

kv_status kv_evict(kv_cache* cache, int layer, int64_t* evicted_begin, int64_t* evicted_end) {
  kv_status st = check_layer(cache, layer);
  if (st != KV_OK) return st;
  if (!evicted_begin || !evicted_end) return fail(KV_ERR_INVALID_ARG, "output pointer is NULL");
  LayerState& ls = cache->layers[layer];
  const int W = cache->geo.evict_window;
  if (W && ls.L - W > ls.E) {
    *evicted_begin = ls.E;
    *evicted_end = ls.L - W;
    ls.E = ls.L - W;
  } else {
    *evicted_begin = *evicted_end = ls.E;
  }
  return KV_OK;
}

}  // extern "C"

namespace kvq {

kv_status report(kv_status s, const char* msg) { return fail(s, msg); }

kv_status decode_attn_impl(kv_cache* cache, int layer, const void* q, float* out, float* lse_or_null,
                           void* cuda_stream, void* partials, size_t partial_bytes) {
  kv_status st = check_layer(cache, layer);
  if (st != KV_OK) return st;
  if (!q || !out) return fail(KV_ERR_INVALID_ARG, "q/out is NULL");
  if (reinterpret_cast<uintptr_t>(q) % 4 || reinterpret_cast<uintptr_t>(out) % 4)
    return fail(KV_ERR_INVALID_ARG, "q and out must be 4-byte aligned");
  const Geometry& g = cache->geo;
  const LayerState& ls = cache->layers[layer];
  if (ls.L == 0) return fail(KV_ERR_STATE, "decode on an empty layer");
  kvq::DecodeArgs a{};
  a.geo = g;
  a.lay = layer_dev(cache, layer);
  a.tab = tables_dev(cache);
  a.q = static_cast<const uint16_t*>(q);
  if (partials) {  // caller-given partial storage: [part_o | part_ml], each 256-byte aligned
    const size_t ns = static_cast<size_t>(g.max_splits) + 1, rows = static_cast<size_t>(g.B) * g.Hq;
    const size_t o_bytes = align256(rows * ns * g.D * 4);
    const size_t need = o_bytes + align256(rows * ns * 2 * 4);
    if (need > partial_bytes)
      return fail(KV_ERR_CAPACITY, "decode partials need " + std::to_string(need) +
                                       " bytes (batch * n_q_heads * (max_splits + 1) * (head_dim + 2) * 4, "
                                       "256-byte aligned); the scratch holds " +
                                       std::to_string(partial_bytes));
    a.part_o = static_cast<float*>(partials);
    a.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(partials) + o_bytes);
  } else {
    a.part_o = reinterpret_cast<float*>(cache->arena + g.off_part_o);
    a.part_ml = reinterpret_cast<float*>(cache->arena + g.off_part_ml);
  }
  a.out = out;
  a.lse = lse_or_null;
  a.L = ls.L;
  a.F = fp16_begin_of(g, ls.L);
  a.qlo = std::max<int64_t>(g.n_sink, ls.E);
  a.n_sink_read = static_cast<int>(std::min<int64_t>(std::min<int64_t>(g.n_sink, ls.L), a.F));
  a.n_dyn_sel = ls.n_dyn_sel;
  // re-positioning moves the query against the sinks by the evicted span
  a.sink_qpos = ls.L - 1 - (g.rope_repos ? ls.E - g.n_sink : 0);
  a.key_shift = (g.k_pre_rope && g.rope_repos) ? ls.E - g.n_sink : 0;
  a.q_pos = ls.L - 1 - a.key_shift;
  a.qscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(g.D)));
  const int64_t units = static_cast<int64_t>(g.B) * g.H;
  if (a.F > a.qlo) {
    a.g_begin = a.qlo / kGroup;
    const int64_t g_end = (a.F + kGroup - 1) / kGroup;
    a.n_groups = static_cast<int>(g_end - a.g_begin);
    a.work = units * a.n_groups;
  } else {
    a.g_begin = 0;
    a.n_groups = 0;
    a.work = 0;
  }
  a.n_ctas_hint = cache->stream_ctas;
  a.h2_magic = 0x64006400u;  // f16 1024.0 in both halves
  a.ns = g.max_splits + 1;
  int64_t launches = 0;
  cudaError_t e = kvq::launch_decode(a, static_cast<cudaStream_t>(cuda_stream), cache->ev0, cache->ev1,
                                     cache->sm_count, &launches);
  g_launches += launches;
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return KV_OK;
}

int cache_device(const kv_cache* cache) { return cache->device; }

}  // namespace kvq

extern "C" {

kv_status kv_decode_attn(kv_cache* cache, int layer, const void* q, float* out, float* lse_or_null,
                         void* cuda_stream) {
  return kvq::decode_attn_impl(cache, layer, q, out, lse_or_null, cuda_stream, nullptr, 0);
}

kv_status kv_cache_stats(kv_cache* cache, int layer, kv_cache_stats_t* out) {
  kv_status st = check_layer(cache, layer);
  if (st != KV_OK) return st;
  if (!out) return fail(KV_ERR_INVALID_ARG, "out is NULL");
  const Geometry& g = cache->geo;
  const LayerState& ls = cache->layers[layer];
  const int64_t B = g.B, H = g.H, D = g.D;
  const int64_t L = ls.L, E = ls.E, F = fp16_begin_of(g, L), Q = q_end_of(g, L);
  const int64_t lo = std::max<int64_t>(g.n_sink, E);
  int64_t n_sink = 0, n_sink_in_quant = 0;
  if (g.n_dyn) {
    if (ls.dyn_selected && ls.n_dyn_sel > 0) {
      std::vector<int64_t> pos(static_cast<size_t>(B) * kMaxSinks);
      cudaError_t e = cudaDeviceSynchronize();
      if (e == cudaSuccess)
        e = cudaMemcpy(pos.data(), layer_dev(cache, layer).sink_pos, pos.size() * 8, cudaMemcpyDeviceToHost);
      if (e != cudaSuccess) return cuda_fail(e, "kv_cache_stats");
      for (int64_t b = 0; b < B; ++b)
        for (int j = 0; j < ls.n_dyn_sel; ++j) {
          const int64_t p = pos[b * kMaxSinks + j];
          if (p < F) ++n_sink;
          if (p >= lo && p < F) ++n_sink_in_quant;
        }
    }
  } else {
    const int64_t ns = std::min<int64_t>(g.n_sink, L);
    for (int64_t p = 0; p < ns; ++p) {
      if (p < F) n_sink += B;
      if (p >= lo && p < F) n_sink_in_quant += B;
    }
  }
  out->length = L;
  out->evict_end = E;
  out->quant_end = Q;
  out->fp16_begin = F;
  out->n_sink = n_sink;
  out->n_quant = B * std::max<int64_t>(0, F - lo) - n_sink_in_quant;
  out->n_tail = B * (L - F);
  out->n_evicted = B * (E - g.n_sink);
  const int64_t row16 = 2 * D * 2;
  out->code_bytes = out->n_quant * H * (D * (g.kb + g.vb) / 8);
  if (!g.mode_tq) {
    const int64_t groups = F > lo ? (F + kGroup - 1) / kGroup - lo / kGroup : 0;
    out->kmeta_bytes = groups * B * H * 4 * D;
    out->vmeta_bytes = out->n_quant * H * (D / kGroup) * 4;
  } else {
    out->kmeta_bytes = out->n_quant * H * 4;
    out->vmeta_bytes = out->n_quant * H * 4;
  }
  out->sink_bytes = n_sink * H * row16;
  out->tail_bytes = out->n_tail * H * row16;
  return KV_OK;
}

namespace {

struct ExportPlan {
  int64_t T0, T1, n, G, S, R;
};

ExportPlan plan_of(const kv_cache* c, int layer) {
  const Geometry& g = c->geo;
  const LayerState& ls = c->layers[layer];
  ExportPlan p;
  p.T0 = kGroup * (ls.E / kGroup);
  p.T1 = q_end_of(g, ls.L);
  if (p.T1 < p.T0) p.T1 = p.T0;
  p.n = p.T1 - p.T0;
  p.G = p.n / kGroup;
  p.S = g.n_dyn ? ls.n_dyn_sel : std::min<int64_t>(g.n_sink, ls.L);
  p.R = ls.L - fp16_begin_of(g, ls.L);
  return p;
}

kv_status export_size(const kv_cache* c, int layer, int what, size_t* bytes) {
  const Geometry& g = c->geo;
  const ExportPlan p = plan_of(c, layer);
  const size_t B = g.B, H = g.H, D = g.D;
  const bool tq = g.mode_tq;
  switch (what) {
    case KV_EXPORT_K_CODES: *bytes = B * H * p.n * D * g.kb / 8; return KV_OK;
    case KV_EXPORT_V_CODES: *bytes = B * H * p.n * D * g.vb / 8; return KV_OK;
    case KV_EXPORT_K_SCALE:
    case KV_EXPORT_K_ZERO:
      if (tq) break;
      *bytes = B * H * p.G * D * 2;
      return KV_OK;
    case KV_EXPORT_V_SCALE:
    case KV_EXPORT_V_ZERO:
      if (tq) break;
      *bytes = B * H * p.n * (D / kGroup) * 2;
      return KV_OK;
    case KV_EXPORT_K_NORM:
    case KV_EXPORT_V_NORM:
      if (!tq) break;
      *bytes = B * H * p.n * 4;
      return KV_OK;
    case KV_EXPORT_SINK_POS: *bytes = B * p.S * 8; return KV_OK;
    case KV_EXPORT_SINK_K:
    case KV_EXPORT_SINK_V: *bytes = B * H * p.S * D * act_bytes(); return KV_OK;
    case KV_EXPORT_TAIL_K:
    case KV_EXPORT_TAIL_V: *bytes = B * H * p.R * D * act_bytes(); return KV_OK;
    case KV_EXPORT_SINK_MASK:
      if (tq) break;
      *bytes = B * p.G * 4;
      return KV_OK;
    case KV_EXPORT_CODEBOOK_K:
      if (!tq) break;
      *bytes = ((1u << g.kb) * 2 - 1) * 4;
      return KV_OK;
    case KV_EXPORT_CODEBOOK_V:
      if (!tq) break;
      *bytes = ((1u << g.vb) * 2 - 1) * 4;
      return KV_OK;
    case KV_EXPORT_TQ_SIGNS: *bytes = D * 4; return KV_OK;
    case KV_EXPORT_ROPE:
      *bytes = static_cast<size_t>(g.rope_max_pos) * D * 4;
      return KV_OK;
    default: return fail(KV_ERR_INVALID_ARG, "unknown export id");
  }
  return fail(KV_ERR_INVALID_ARG, "export id does not apply to this mode");
}

}  // namespace

kv_status kv_cache_export_bytes(kv_cache* cache, int layer, int what, size_t* bytes) {
  kv_status st = check_layer(cache, layer);
  if (st != KV_OK) return st;
  if (!bytes) return fail(KV_ERR_INVALID_ARG, "bytes is NULL");
  return export_size(cache, layer, what, bytes);
}

kv_status kv_cache_export(kv_cache* cache, int layer, int what, void* host_dst, size_t bytes, void* cuda_stream) {
  kv_status st = check_layer(cache, layer);
  if (st != KV_OK) return st;
  size_t need = 0;
  st = export_size(cache, layer, what, &need);
  if (st != KV_OK) return st;
  if (bytes != need) return fail(KV_ERR_INVALID_ARG, "bytes must equal kv_cache_export_bytes");
  if (need == 0) return KV_OK;
  if (!host_dst) return fail(KV_ERR_INVALID_ARG, "host_dst is NULL");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_cache_export");
  const Geometry& g = cache->geo;
  const ExportPlan p = plan_of(cache, layer);
  const kvq::LayerDev d = layer_dev(cache, layer);
  const int64_t B = g.B, H = g.H, D = g.D;
  uint8_t* dst = static_cast<uint8_t*>(host_dst);
  auto d2h = [&](void* h, const void* dv, size_t n) { return cudaMemcpy(h, dv, n, cudaMemcpyDeviceToHost); };

  // the sink slots of each sequence in position order (KVSink slots are
  // filled in admission order; overlay sink j sits in slot j)
  std::vector<int64_t> pos(static_cast<size_t>(B) * kMaxSinks);
  std::vector<int> order(static_cast<size_t>(B) * kMaxSinks);
  if (what == KV_EXPORT_SINK_POS || what == KV_EXPORT_SINK_K || what == KV_EXPORT_SINK_V) {
    if (g.n_dyn) {
      e = d2h(pos.data(), d.sink_pos, pos.size() * 8);
    } else {
      for (int64_t b = 0; b < B; ++b)
        for (int64_t j = 0; j < p.S; ++j) pos[b * kMaxSinks + j] = j;
    }
    for (int64_t b = 0; b < B; ++b) {
      int* ob = order.data() + b * kMaxSinks;
      for (int j = 0; j < p.S; ++j) ob[j] = j;
      const int64_t* pb = pos.data() + b * kMaxSinks;
      std::sort(ob, ob + p.S, [pb](int x, int y) { return pb[x] < pb[y]; });
    }
  }

  switch (what) {
    case KV_EXPORT_SINK_POS: {
      int64_t* o = reinterpret_cast<int64_t*>(dst);
      for (int64_t b = 0; b < B; ++b)
        for (int64_t j = 0; j < p.S; ++j) o[b * p.S + j] = pos[b * kMaxSinks + order[b * kMaxSinks + j]];
      break;
    }
    case KV_EXPORT_SINK_K:
    case KV_EXPORT_SINK_V: {
      const uint16_t* src = what == KV_EXPORT_SINK_K ? d.sink_k : d.sink_v;
      std::vector<uint16_t> rows(static_cast<size_t>(g.n_sink_slots) * D);
      for (int64_t bh = 0; bh < B * H && e == cudaSuccess; ++bh) {
        e = d2h(rows.data(), src + bh * g.n_sink_slots * D, rows.size() * 2);
        const int* ob = order.data() + (bh / H) * kMaxSinks;
        for (int64_t j = 0; j < p.S; ++j)
          std::memcpy(dst + (bh * p.S + j) * D * 2, rows.data() + static_cast<size_t>(ob[j]) * D, D * 2);
      }
      break;
    }
    case KV_EXPORT_TAIL_K:
    case KV_EXPORT_TAIL_V: {
      const uint16_t* src = what == KV_EXPORT_TAIL_K ? d.tail_k : d.tail_v;
      std::vector<uint16_t> ring(static_cast<size_t>(B) * H * g.tail_cap * D);
      e = d2h(ring.data(), src, ring.size() * 2);
      const int64_t F = cache->layers[layer].L - p.R;
      uint16_t* o = reinterpret_cast<uint16_t*>(dst);
      for (int64_t bh = 0; bh < B * H; ++bh)
        for (int64_t r = 0; r < p.R; ++r) {
          const int64_t slot = (F + r) & (g.tail_cap - 1);
          std::memcpy(o + (bh * p.R + r) * D, ring.data() + (bh * g.tail_cap + slot) * D, D * 2);
        }
      break;
    }
    case KV_EXPORT_CODEBOOK_K:
    case KV_EXPORT_CODEBOOK_V:
      e = d2h(dst, cache->arena + (what == KV_EXPORT_CODEBOOK_K ? g.off_cbk : g.off_cbv), need);
      break;
    case KV_EXPORT_TQ_SIGNS: e = d2h(dst, cache->arena + g.off_signs, need); break;
    case KV_EXPORT_ROPE: e = d2h(dst, cache->arena + g.off_rope, need); break;
    case KV_EXPORT_SINK_MASK: {
      std::vector<uint32_t> m(static_cast<size_t>(B) * g.n_slots);
      e = d2h(m.data(), d.sink_mask, m.size() * 4);
      uint32_t* o = reinterpret_cast<uint32_t*>(dst);
      for (int64_t b = 0; b < B; ++b)
        for (int64_t gi = 0; gi < p.G; ++gi) {
          const int64_t grp = p.T0 / kGroup + gi;
          o[b * p.G + gi] = g.n_dyn ? m[b * g.n_slots + grp % g.n_slots] : 0u;
        }
      break;
    }
    default: {
      // codes, scales, zeros and norms: fetch the stored groups chunk by chunk
      std::memset(dst, 0, need);
      const int CH = g.chunk.bytes;
      const int64_t g0 = p.T0 / kGroup, g1 = (p.T1 + kGroup - 1) / kGroup;
      std::vector<uint8_t> chunk(CH);
      for (int64_t bh = 0; bh < B * H && e == cudaSuccess; ++bh) {
        for (int64_t grp = g0; grp < g1 && e == cudaSuccess; ++grp) {
          const uint8_t* src = d.chunks + (static_cast<size_t>(bh) * g.n_slots + grp % g.n_slots) * CH;
          e = d2h(chunk.data(), src, CH);
          if (e != cudaSuccess) break;
          const int64_t gi = grp - g0;
          const int ntok = static_cast<int>(std::min<int64_t>(kGroup, p.T1 - grp * kGroup));
          if (what == KV_EXPORT_K_CODES || what == KV_EXPORT_V_CODES) {
            // canonical rows: D bits / 8 bytes, code c at bits c bits .. of
            // the row's little-endian bit string
            const bool isk = what == KV_EXPORT_K_CODES;
            const int bits = isk ? g.kb : g.vb;
            const int rowb = static_cast<int>(D) * bits / 8;
            uint8_t* o = dst + (bh * p.n + gi * kGroup) * rowb;
            const uint8_t* reg = chunk.data() + (isk ? g.chunk.kc_off : g.chunk.vc_off);
            auto put = [&](int tok, int ch, uint32_t code) {
              if (tok >= ntok) return;
              for (int k = 0; k < bits; ++k)
                if ((code >> k) & 1u) o[tok * rowb + (ch * bits + k) / 8] |= static_cast<uint8_t>(1u << ((ch * bits + k) % 8));
            };
            const int wpl = static_cast<int>(D) * bits / 32, pw = kvq::piece_words(wpl);
            auto lane_word = [&](int lane, int w) {
              uint32_t x;
              std::memcpy(&x, reg + kvq::code_word_offset(lane, w, pw), 4);
              return x;
            };
            const uint32_t fmask = (1u << (2 * bits)) - 1u;
            if (g.mode_tq && !isk) {  // token-pair rows
              const int rb = kvq::tq_vrow_bytes(static_cast<int>(D), bits);
              for (int pr = 0; pr < kGroup / 2; ++pr)
                for (int c = 0; c < D; ++c) {
                  const int fbit = kvq::tq_vfield_bit(static_cast<int>(D), bits, c);
                  uint32_t f = 0;
                  for (int k = 0; k < 2 * bits; ++k)
                    f |= ((reg[pr * rb + (fbit + k) / 8] >> ((fbit + k) % 8)) & 1u) << k;
                  put(2 * pr, c, f & ((1u << bits) - 1u));
                  put(2 * pr + 1, c, f >> bits);
                }
            } else if (g.mode_tq) {  // K fields in fragment order
              for (int lane = 0; lane < 32; ++lane) {
                std::vector<uint32_t> w(wpl + 1, 0u);
                for (int k = 0; k < wpl; ++k) w[k] = lane_word(lane, k);
                const int gg = lane >> 2, t = lane & 3;
                for (int b = 0; b < 4; ++b)
                  for (int j = 0; j < D / 8; ++j) {
                    const int fbit = kvq::tq_kfield_bit(static_cast<int>(D), bits, b, j);
                    const uint64_t two = w[fbit / 32] | (static_cast<uint64_t>(w[fbit / 32 + 1]) << 32);
                    const uint32_t f = static_cast<uint32_t>(two >> (fbit % 32)) & fmask;
                    const int tok = 16 * (b >> 1) + gg + 8 * (b & 1), c0 = 16 * (j >> 1) + 2 * t + 8 * (j & 1);
                    put(tok, c0, f & ((1u << bits) - 1u));
                    put(tok, c0 + 1, f >> bits);
                  }
              }
            } else {  // KIVI fragment order
              const uint32_t mask = (1u << bits) - 1;
              for (int lane = 0; lane < 32; ++lane)
                for (int f = 0; f < D; ++f) {
                  int tok, ch;
                  if (isk) kvq::k_frag_pos(static_cast<int>(D), lane, f, &tok, &ch, g.k_pre_rope != 0);
                  else kvq::v_frag_pos(static_cast<int>(D), lane, f, &tok, &ch);
                  uint32_t code;
                  if (bits == 3) {
                    const uint32_t blk[3] = {lane_word(lane, 3 * (f / 32)), lane_word(lane, 3 * (f / 32) + 1),
                                             lane_word(lane, 3 * (f / 32) + 2)};
                    code = kvq::frag3_get(blk, f % 32);
                  } else {
                    int w, bit;
                    kvq::frag_bits(bits, f, &w, &bit);
                    code = (lane_word(lane, w) >> bit) & mask;
                  }
                  put(tok, ch, code);
                }
            }
          } else if (what == KV_EXPORT_K_SCALE || what == KV_EXPORT_K_ZERO) {
            uint16_t* o = reinterpret_cast<uint16_t*>(dst) + (bh * p.G + gi) * D;
            const bool zero = what == KV_EXPORT_K_ZERO;
            for (int ch = 0; ch < D; ++ch) {
              const int pos = g.k_pre_rope ? (zero ? static_cast<int>(D) + ch : ch)
                              : zero       ? static_cast<int>(D) + kvq::kzero_pos(static_cast<int>(D), ch)
                                           : kvq::kmeta_pos(static_cast<int>(D), ch);
              std::memcpy(o + ch, chunk.data() + g.chunk.kmeta_off + pos * 2, 2);
            }
          } else if (what == KV_EXPORT_V_SCALE || what == KV_EXPORT_V_ZERO) {
            const int nv = static_cast<int>(D) / kGroup;
            uint16_t* o = reinterpret_cast<uint16_t*>(dst) + (bh * p.n + gi * kGroup) * nv;
            for (int r = 0; r < kGroup; ++r)
              for (int vg = 0; vg < nv; ++vg) {
                const int pos = what == KV_EXPORT_V_ZERO ? kvq::vzero_pos(nv, r, vg) : kvq::vscale_pos(nv, r, vg);
                std::memcpy(o + r * nv + vg, chunk.data() + g.chunk.vmeta_off + pos * 2, 2);
              }
          } else if (what == KV_EXPORT_K_NORM || what == KV_EXPORT_V_NORM) {
            float* o = reinterpret_cast<float*>(dst) + bh * p.n + gi * kGroup;
            const int off = what == KV_EXPORT_K_NORM ? g.chunk.kmeta_off : g.chunk.vmeta_off;
            std::memcpy(o, chunk.data() + off, static_cast<size_t>(ntok) * 4);
          }
        }
      }
      break;
    }
  }
  if (e != cudaSuccess) return cuda_fail(e, "kv_cache_export");
  return KV_OK;
}

kv_status kv_cache_check_device_error(kv_cache* cache, void* cuda_stream) {
  if (!cache) return fail(KV_ERR_INVALID_ARG, "cache is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  int flag = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&flag, cache->arena + cache->geo.off_err, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && flag) e = cudaMemset(cache->arena + cache->geo.off_err, 0, 4);
  if (e != cudaSuccess) return cuda_fail(e, "kv_cache_check_device_error");
  if (flag) return fail(KV_ERR_TIMEOUT, "a bounded device wait gave up");
  return KV_OK;
}

kv_status kv_cache_set_timing_events(kv_cache* cache, void* ev_begin, void* ev_end) {
  if (!cache) return fail(KV_ERR_INVALID_ARG, "cache is NULL");
  if ((ev_begin == nullptr) != (ev_end == nullptr)) return fail(KV_ERR_INVALID_ARG, "pass both events or neither");
  cache->ev0 = static_cast<cudaEvent_t>(ev_begin);
  cache->ev1 = static_cast<cudaEvent_t>(ev_end);
  return KV_OK;
}

kv_status kv_cache_test_bounded_wait(kv_cache* cache, int64_t budget_cycles, int64_t* host_result,
                                     void* cuda_stream) {
  if (!cache) return fail(KV_ERR_INVALID_ARG, "cache is NULL");
  if (!host_result) return fail(KV_ERR_INVALID_ARG, "host_result is NULL");
  if (budget_cycles < 1000 || budget_cycles > (int64_t{1} << 31))
    return fail(KV_ERR_INVALID_ARG, "budget_cycles must be in [1000, 2^31]");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  // the results go to the arena's error block, after the flag
  long long* res = reinterpret_cast<long long*>(cache->arena + cache->geo.off_err + 64);
  int64_t launches = 0;
  cudaError_t e = cudaMemsetAsync(res, 0xff, 5 * sizeof(long long), s);
  if (e == cudaSuccess)
    e = kvq::launch_wait_probe(reinterpret_cast<int*>(cache->arena + cache->geo.off_err), res, budget_cycles, s,
                               &launches);
  g_launches += launches;
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(host_result, res, 5 * sizeof(long long), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "kv_cache_test_bounded_wait");
  return KV_OK;
}

int64_t kv_launch_count(void) { return g_launches.load(); }

kv_status kv_copy_bandwidth_kernel(const void* src, void* dst, size_t bytes, void* cuda_stream) {
  if (!src || !dst) return fail(KV_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(src) || !aligned16(dst) || (bytes & 15u)) return fail(KV_ERR_INVALID_ARG, "16-byte alignment");
  int64_t launches = 0;
  cudaError_t e = kvq::launch_copy(src, dst, bytes, static_cast<cudaStream_t>(cuda_stream), &launches);
  g_launches += launches;
  if (e != cudaSuccess) return cuda_fail(e, "copy launch");
  return KV_OK;
}

const char* kv_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
