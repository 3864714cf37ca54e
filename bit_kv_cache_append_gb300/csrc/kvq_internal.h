// Kernel argument blocks and launchers of the library (internal).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "kvq.h"
#include "kvq_layout.h"

namespace kvq {

// Device pointers of one layer inside the arena.
struct LayerDev {
  uint8_t* chunks;      // [B][H][n_slots][chunk.bytes]
  uint16_t* tail_k;     // [B][H][tail_cap][D]  act dtype bits
  uint16_t* tail_v;
  uint16_t* sink_k;     // [B][H][n_sink_slots][D]
  uint16_t* sink_v;
  int64_t* sink_pos;    // [B][kMaxSinks] absolute positions of the sink set (slot order)
  float* sink_m;        // [B][kMaxSinks] their key norms
  uint32_t* sink_mask;  // [B][n_slots]
};

// Tables shared by every layer.
struct TablesDev {
  const float* rope;    // [rope_max_pos][D/2][2] or nullptr
  const float* signs;   // [D] TurboQuant +-1
  const float* cb_k;    // boundaries[2^kb - 1] then centroids[2^kb]
  const float* cb_v;
  int* err_flag;
};

// One append: tokens [L0, L0 + n) arrive in `k`, `v` ([B][H][n][D]).
struct AppendArgs {
  Geometry geo;
  LayerDev lay;
  TablesDev tab;
  const uint16_t* k;
  const uint16_t* v;
  int n;
  int64_t L0;           // L before the append
  int64_t tail_from;    // rows at positions >= tail_from go to the tail ring
  int64_t g_first;      // first group that completes in this append
  int n_groups;         // groups completing in this append (KIVI)
  int dyn_active;       // KVSink: sink positions valid for exclusion
  int n_dyn_sel;        // KVSink: number of selected sinks
};

// Decode attention of one layer.
struct DecodeArgs {
  Geometry geo;
  LayerDev lay;
  TablesDev tab;
  const uint16_t* q;    // [B][Hq][D] act dtype bits
  float* part_o;        // [B][Hq][ns][D]
  float* part_ml;       // [B][Hq][ns][2]  (max in log2 units, sum)
  float* out;           // [B][Hq][D]
  float* lse;           // [B][Hq] or nullptr
  int64_t L, F, qlo;    // quantised segment [qlo, F), tail [F, L)
  int64_t g_begin;      // first group of the quantised segment
  int n_groups;         // groups touching [qlo, F), per (sequence, KV head) unit
  int64_t work;         // units * n_groups: the quantised items the stream-K CTAs split
  int n_ctas;           // stream-K CTAs (set at launch)
  int n_ctas_hint;      // 0 = SM count x occupancy
  int ns;               // partial slot stride per (sequence, query head)
  int n_sink_read;      // overlay: sink slots [0, n) read from the sink buffer
  int n_dyn_sel;        // KVSink: selected sinks (read when pos < F)
  int64_t sink_qpos;    // RoPE position of the query against the sink rows
                        // (L - 1, or L - 1 - (E - n_sink) when re-positioning)
  int64_t key_shift;    // keys stored before RoPE: positions >= n_sink are
                        // rotated at p - key_shift (E - n_sink when
                        // re-positioning, else 0), the query at q_pos
  int64_t q_pos;
  float qscale;         // log2(e) / sqrt(D)
  // the f16x2 magic 1024.0 pair of the 8-bit code conversion, read from the
  // parameter bank so that the instruction needs no second immediate
  uint32_t h2_magic;
};

// KVSink selection scratch.
struct SinkSelectArgs {
  Geometry geo;
  LayerDev lay;
  TablesDev tab;
  const uint16_t* k;    // [B][H][n][D]
  const uint16_t* v;    // [B][H][n][D] (the single-kernel path copies new sink rows)
  int n;
  float* norms;         // [B][n]
  float* cand_m;        // [B][n_chunks][kMaxSinks]
  int64_t* cand_p;
  int n_chunks;
  int k_sel;            // candidates kept per chunk: min(k, n)
  int64_t L0;           // position of the call's first token
  int64_t q0;           // end of the quantised groups when the call began
  int n_old;            // members before the call (slots 0 .. n_old - 1)
  int k_total;          // members after the call: min(k, L0 + n)
};

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s, int64_t* launches);
// KIVI group quantisation of a.n_groups completed groups (flush_d*_k*.cu:
// head_dim 128 or 64, K codes of 2 or 3 bits, or of 4 or 8 bits).
void launch_flush_d128_k23(const AppendArgs& a, dim3 grid, cudaStream_t s);
void launch_flush_d128_k48(const AppendArgs& a, dim3 grid, cudaStream_t s);
void launch_flush_d64_k23(const AppendArgs& a, dim3 grid, cudaStream_t s);
void launch_flush_d64_k48(const AppendArgs& a, dim3 grid, cudaStream_t s);
cudaError_t launch_sink_select(const SinkSelectArgs& a, cudaStream_t s, int64_t* launches);
// KVSink calls of at most this many tokens take the single-launch path
// (norms, set update and new sink rows in one kernel per sequence).
constexpr int kSinkSmallCallTokens = 256;
cudaError_t launch_sink_admit_small(const SinkSelectArgs& a, cudaStream_t s, int64_t* launches);
cudaError_t launch_sink_gather(const AppendArgs& a, cudaStream_t s, int64_t* launches);
cudaError_t launch_decode(DecodeArgs& a, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1, int sm_count,
                          int64_t* launches);
cudaError_t launch_copy(const void* src, void* dst, size_t bytes, cudaStream_t s,
                        int64_t* launches);
// The decode kernels' bounded waits run out on barriers nobody completes
// (a test of the give-up path; res: 5 device int64).
cudaError_t launch_wait_probe(int* err_flag, long long* res, long long budget, cudaStream_t s,
                              int64_t* launches);

// Decode attention of one layer (the body of kv_decode_attn). With
// `partials` NULL the split partials live in the cache's arena; otherwise in
// `partials` (device, 256-byte aligned, `partial_bytes` long), and the call
// fails with KV_ERR_CAPACITY before any launch when they do not fit.
kv_status decode_attn_impl(kv_cache* cache, int layer, const void* q, float* out, float* lse_or_null,
                           void* cuda_stream, void* partials, size_t partial_bytes);
// Device ordinal the cache was created on.
int cache_device(const kv_cache* cache);
// Set the thread's last-error text and return `s`.
kv_status report(kv_status s, const char* msg);

// Host-built tables (independent of any other implementation).
void build_rope_table(float* out, int64_t max_pos, int D, double base);
void build_signs(float* out, int D, uint64_t seed);
// Lloyd-Max quantiser of Beta(a, a) on [0, 1] with 2^bits levels, by
// composite Gauss-Legendre quadrature of the density; double precision.
void build_beta_codebook(double a, int bits, double* boundaries, double* centroids);

}  // namespace kvq
