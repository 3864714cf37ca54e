// KVSink-style sink selection (VeloxQuant-MLX "KVSink-Adapted Sink
// Protection", "How it works" 1): the per-token key L2 norm averaged over the
// KV heads, folded call by call into a running top-k of positions per
// sequence (norm descending, ties to the lower position). A sink whose group
// is already quantised stays (the page never restores a quantised token, and
// its codes hold a substitute's values).
#include "kvq_device.cuh"

namespace kvq {
namespace {

// Key norm of token t (of the call) of sequence b, valid in lane 0: head
// norms by the fixed pairwise tree over k^2 (stride D/2, D/4, ..., 1), summed
// over heads in head order, divided by Hkv. Keys are rotated (and rounded to
// the activation dtype) first when the cache applies RoPE.
template <int D>
__device__ float token_key_norm(const SinkSelectArgs& a, int b, int t, int lane) {
  constexpr int NS = D / 32;
  const Geometry& G = a.geo;
  const int bf16 = G.act_bf16;
  float acc = 0.0f;
  for (int h = 0; h < G.H; ++h) {
    const size_t row = ((static_cast<size_t>(b) * G.H + h) * a.n + t) * D;
    float x[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) x[i] = act_to_float(a.k[row + i * 32 + lane], bf16);
    if (a.tab.rope) {
      const float* tr = a.tab.rope + static_cast<size_t>(a.L0 + t) * D;
#pragma unroll
      for (int i = 0; i < NS / 2; ++i) {
        const int c = i * 32 + lane;
        float rx, ry;
        rope_pair(x[i], x[i + NS / 2], tr[2 * c], tr[2 * c + 1], &rx, &ry);
        x[i] = act_to_float(float_to_act(rx, bf16), bf16);
        x[i + NS / 2] = act_to_float(float_to_act(ry, bf16), bf16);
      }
    }
    float sq[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) sq[i] = __fmul_rn(x[i], x[i]);
#pragma unroll
    for (int sl = NS / 2; sl >= 1; sl >>= 1) {
#pragma unroll
      for (int i = 0; i < sl; ++i) sq[i] = __fadd_rn(sq[i], sq[i + sl]);
    }
    float s = sq[0];
#pragma unroll
    for (int st = 16; st >= 1; st >>= 1) {
      const float o = __shfl_down_sync(0xffffffffu, s, st);
      if (lane < st) s = __fadd_rn(s, o);
    }
    const float nrm = __fsqrt_rn(s);
    acc = (h == 0) ? nrm : __fadd_rn(acc, nrm);
  }
  return __fdiv_rn(acc, static_cast<float>(G.H));
}

// One warp per (token, b).
template <int D>
__global__ void __launch_bounds__(128) keynorm_kernel(SinkSelectArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 4 + warp, b = blockIdx.y;
  if (t >= a.n) return;
  const float m = token_key_norm<D>(a, b, t, lane);
  if (lane == 0) a.norms[static_cast<size_t>(b) * a.n + t] = m;
}

__device__ __forceinline__ bool better(float m1, int64_t p1, float m2, int64_t p2) {
  return m1 > m2 || (m1 == m2 && p1 < p2);
}

constexpr int kTopkThreads = 256;
constexpr int kSinkSmallCall = kSinkSmallCallTokens;  // longest call of the single-launch path
constexpr int kTopkPer = 4;
constexpr int kChunk = kTopkThreads * kTopkPer;

// k rounds of a block-wide arg-best over candidates held 4 per thread;
// the winner of each round is taken out and written in rank order.
__device__ void block_topk(float (&m)[kTopkPer], int64_t (&p)[kTopkPer], int k, float* out_m,
                           int64_t* out_p) {
  __shared__ float wm[kTopkThreads / 32];
  __shared__ int64_t wp[kTopkThreads / 32];
  __shared__ float bm;
  __shared__ int64_t bp;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int round = 0; round < k; ++round) {
    float cm = -INFINITY;
    int64_t cp = INT64_MAX;
#pragma unroll
    for (int i = 0; i < kTopkPer; ++i)
      if (better(m[i], p[i], cm, cp)) { cm = m[i]; cp = p[i]; }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, cm, off);
      const int64_t op = __shfl_xor_sync(0xffffffffu, cp, off);
      if (better(om, op, cm, cp)) { cm = om; cp = op; }
    }
    if (lane == 0) { wm[warp] = cm; wp[warp] = cp; }
    __syncthreads();
    if (threadIdx.x == 0) {
      float xm = wm[0];
      int64_t xp = wp[0];
      for (int w = 1; w < kTopkThreads / 32; ++w)
        if (better(wm[w], wp[w], xm, xp)) { xm = wm[w]; xp = wp[w]; }
      bm = xm;
      bp = xp;
      out_m[round] = xm;
      out_p[round] = xp;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTopkPer; ++i)
      if (p[i] == bp && m[i] == bm) { m[i] = -INFINITY; p[i] = INT64_MAX; }
    __syncthreads();
  }
}

// Pass 1: the top k of each chunk of kChunk positions of one sequence.
__global__ void __launch_bounds__(kTopkThreads) topk_chunk_kernel(SinkSelectArgs a) {
  const int chunk = blockIdx.x, b = blockIdx.y;
  float m[kTopkPer];
  int64_t p[kTopkPer];
#pragma unroll
  for (int i = 0; i < kTopkPer; ++i) {
    const int64_t t = static_cast<int64_t>(chunk) * kChunk + i * kTopkThreads + threadIdx.x;
    if (t < a.n) { m[i] = a.norms[static_cast<size_t>(b) * a.n + t]; p[i] = t; }
    else { m[i] = -INFINITY; p[i] = INT64_MAX; }
  }
  const size_t o = (static_cast<size_t>(b) * a.n_chunks + chunk) * kMaxSinks;
  block_topk(m, p, a.k_sel, a.cand_m + o, a.cand_p + o);
}

// The running top-k of sequence b after the call, by one CTA. Members whose
// position lies below q0 (their group was quantised before the call) are
// locked and keep their slots. The other members and the call's candidates
// (cand(c, &m, &p) for c < n_call, absolute positions, false for an empty
// entry; strike(c) takes a winner out) compete for the remaining
// k_total - locked places by rounds of a block-wide arg-best: a member that
// wins keeps its slot, the call's winners take the freed slots and then the
// new ones, in rank order. Slots are not kept in position order; only the
// set matters to the readers. Ends with the block synchronised.
template <typename Cand, typename Strike>
__device__ void update_sinks(const SinkSelectArgs& a, int b, int n_call, Cand cand, Strike strike) {
  __shared__ int64_t win_p[kMaxSinks];
  __shared__ float win_m[kMaxSinks];
  __shared__ int64_t un_p[kMaxSinks];   // unlocked members: candidates (struck out in place)
  __shared__ float un_m[kMaxSinks];
  __shared__ int un_slot[kMaxSinks];
  __shared__ int keep[kMaxSinks];
  __shared__ int n_un, n_lock;
  __shared__ float wm[kTopkThreads / 32];
  __shared__ int64_t wp[kTopkThreads / 32];
  __shared__ int wc[kTopkThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t* spos = a.lay.sink_pos + static_cast<size_t>(b) * kMaxSinks;
  float* sm = a.lay.sink_m + static_cast<size_t>(b) * kMaxSinks;
  if (threadIdx.x == 0) {
    int nu = 0, nl = 0;
    for (int j = 0; j < a.n_old; ++j) {
      const bool locked = spos[j] < a.q0;
      keep[j] = locked ? 1 : 0;
      if (locked) {
        ++nl;
      } else {
        un_p[nu] = spos[j];
        un_m[nu] = sm[j];
        un_slot[nu] = j;
        ++nu;
      }
    }
    n_un = nu;
    n_lock = nl;
  }
  __syncthreads();
  const int budget = a.k_total - n_lock;
  for (int round = 0; round < budget; ++round) {
    float bm = -INFINITY;
    int64_t bp = INT64_MAX;
    int bc = -1;
    for (int c = threadIdx.x; c < n_call + n_un; c += blockDim.x) {
      float m;
      int64_t p;
      if (c < n_call) {
        if (!cand(c, &m, &p)) continue;
      } else {
        m = un_m[c - n_call];
        p = un_p[c - n_call];
      }
      if (better(m, p, bm, bp)) { bm = m; bp = p; bc = c; }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float om = __shfl_xor_sync(0xffffffffu, bm, off);
      const int64_t op = __shfl_xor_sync(0xffffffffu, bp, off);
      const int oc = __shfl_xor_sync(0xffffffffu, bc, off);
      if (better(om, op, bm, bp)) { bm = om; bp = op; bc = oc; }
    }
    if (lane == 0) { wm[warp] = bm; wp[warp] = bp; wc[warp] = bc; }
    __syncthreads();
    if (threadIdx.x == 0) {
      float xm = wm[0];
      int64_t xp = wp[0];
      int xc = wc[0];
      for (int w = 1; w < static_cast<int>(blockDim.x) / 32; ++w)
        if (better(wm[w], wp[w], xm, xp)) { xm = wm[w]; xp = wp[w]; xc = wc[w]; }
      win_m[round] = xm;
      win_p[round] = xp;
      if (xc >= 0 && xc < n_call) strike(xc);
      else if (xc >= n_call) { un_m[xc - n_call] = -INFINITY; un_p[xc - n_call] = INT64_MAX; }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    // winning members keep their slots
    for (int i = 0; i < n_un; ++i) {
      const int j = un_slot[i];
      const int64_t p = spos[j];
      for (int r = 0; r < budget; ++r)
        if (win_p[r] == p) {
          keep[j] = 1;
          win_p[r] = -1;
          break;
        }
    }
    // the call's winners fill the freed slots, then the new ones
    int r = 0;
    for (int j = 0; j < a.k_total; ++j) {
      if (j < a.n_old && keep[j]) continue;
      while (r < budget && win_p[r] < 0) ++r;
      if (r < budget) {
        spos[j] = win_p[r];
        sm[j] = win_m[r];
        ++r;
      }
    }
  }
  __syncthreads();
}

// Pass 2 of a long call, one CTA per sequence: the set update over the chunk
// winners (call-relative positions).
__global__ void __launch_bounds__(kTopkThreads) sink_update_kernel(SinkSelectArgs a) {
  const int b = blockIdx.x;
  const int n_cand = a.n_chunks * kMaxSinks;
  float* cm_base = a.cand_m + static_cast<size_t>(b) * n_cand;
  int64_t* cp_base = a.cand_p + static_cast<size_t>(b) * n_cand;
  update_sinks(
      a, b, n_cand,
      [&](int c, float* m, int64_t* p) {
        if (c % kMaxSinks >= a.k_sel || cp_base[c] == INT64_MAX) return false;
        *m = cm_base[c];
        *p = cp_base[c] + a.L0;
        return true;
      },
      [&](int c) { cm_base[c] = -INFINITY; cp_base[c] = INT64_MAX; });
}

// A short call (n <= kSinkSmallCall) in one launch per sequence: the call's
// key norms into shared memory, the set update over them, and the K/V rows
// of the call's new members into their sink slots (keys rotated like every
// stored key). The same arithmetic and order as the three-pass path.
template <int D>
__global__ void __launch_bounds__(kTopkThreads) sink_admit_small_kernel(SinkSelectArgs a) {
  const int b = blockIdx.x;
  const Geometry& G = a.geo;
  __shared__ float cm[kSinkSmallCall];
  __shared__ int64_t cp[kSinkSmallCall];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = warp; t < a.n; t += kTopkThreads / 32) {
    const float m = token_key_norm<D>(a, b, t, lane);
    if (lane == 0) {
      cm[t] = m;
      cp[t] = a.L0 + t;
    }
  }
  __syncthreads();
  update_sinks(
      a, b, a.n,
      [&](int c, float* m, int64_t* p) {
        if (cp[c] == INT64_MAX) return false;
        *m = cm[c];
        *p = cp[c];
        return true;
      },
      [&](int c) { cm[c] = -INFINITY; cp[c] = INT64_MAX; });
  // rows of the members this call brought in
  constexpr int HALF = D / 2, CPR = HALF / 8;
  const int64_t* spos = a.lay.sink_pos + static_cast<size_t>(b) * kMaxSinks;
  for (int idx = threadIdx.x; idx < a.k_total * G.H * CPR; idx += blockDim.x) {
    const int j = idx / (G.H * CPR), h = (idx / CPR) % G.H, c0 = (idx % CPR) * 8;
    const int64_t row = spos[j] - a.L0;
    if (row < 0 || row >= a.n) continue;
    const size_t bh = static_cast<size_t>(b) * G.H + h;
    const size_t in_row = (bh * a.n + row) * D;
    uint4 klo = *reinterpret_cast<const uint4*>(a.k + in_row + c0);
    uint4 khi = *reinterpret_cast<const uint4*>(a.k + in_row + HALF + c0);
    const uint4 vlo = *reinterpret_cast<const uint4*>(a.v + in_row + c0);
    const uint4 vhi = *reinterpret_cast<const uint4*>(a.v + in_row + HALF + c0);
    if (a.tab.rope) rotate8(klo, khi, a.tab.rope + static_cast<size_t>(spos[j]) * D, c0, G.act_bf16);
    const size_t o = (bh * G.n_sink_slots + j) * D;
    *reinterpret_cast<uint4*>(a.lay.sink_k + o + c0) = klo;
    *reinterpret_cast<uint4*>(a.lay.sink_k + o + HALF + c0) = khi;
    *reinterpret_cast<uint4*>(a.lay.sink_v + o + c0) = vlo;
    *reinterpret_cast<uint4*>(a.lay.sink_v + o + HALF + c0) = vhi;
  }
}

}  // namespace

cudaError_t launch_sink_admit_small(const SinkSelectArgs& a, cudaStream_t s, int64_t* launches) {
  if (a.geo.D == 128) sink_admit_small_kernel<128><<<a.geo.B, kTopkThreads, 0, s>>>(a);
  else sink_admit_small_kernel<64><<<a.geo.B, kTopkThreads, 0, s>>>(a);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_sink_select(const SinkSelectArgs& a, cudaStream_t s, int64_t* launches) {
  dim3 g1((a.n + 3) / 4, a.geo.B);
  if (a.geo.D == 128) keynorm_kernel<128><<<g1, 128, 0, s>>>(a);
  else keynorm_kernel<64><<<g1, 128, 0, s>>>(a);
  dim3 g2(a.n_chunks, a.geo.B);
  topk_chunk_kernel<<<g2, kTopkThreads, 0, s>>>(a);
  sink_update_kernel<<<a.geo.B, kTopkThreads, 0, s>>>(a);
  *launches += 3;
  return cudaGetLastError();
}

}  // namespace kvq
