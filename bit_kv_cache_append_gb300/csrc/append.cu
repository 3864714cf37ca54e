// Append-side kernels: exact tail ring and sink buffer writes, TurboQuant
// per-token quantisation and the KVSink sink-row gather; the launch of the
// KIVI group quantisation (flush.cuh).
#include <algorithm>

#include "kvq_device.cuh"

namespace kvq {
namespace {

// ---------------------------------------------------------------- tail ring
// Rows at positions >= tail_from go to the tail ring (slot pos mod tail_cap);
// positions < n_sink also go to the overlay sink buffer (slot = pos).
__global__ void tail_write_kernel(AppendArgs a, int row_begin, int n_rows) {
  const Geometry& G = a.geo;
  const int D = G.D, half = D / 2, cpr = half / 8;
  const int bh = blockIdx.y;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const int row = row_begin + idx / cpr;
  if (row >= row_begin + n_rows) return;
  const int c0 = (idx % cpr) * 8;
  const int64_t pos = a.L0 + row;
  const bool to_tail = pos >= a.tail_from;
  const bool to_sink = pos < G.n_sink;
  if (!to_tail && !to_sink) return;
  const size_t in_row = (static_cast<size_t>(bh) * a.n + row) * D;
  uint4 klo = *reinterpret_cast<const uint4*>(a.k + in_row + c0);
  uint4 khi = *reinterpret_cast<const uint4*>(a.k + in_row + half + c0);
  const uint4 vlo = *reinterpret_cast<const uint4*>(a.v + in_row + c0);
  const uint4 vhi = *reinterpret_cast<const uint4*>(a.v + in_row + half + c0);
  if (a.tab.rope) rotate8(klo, khi, a.tab.rope + static_cast<size_t>(pos) * D, c0, G.act_bf16);
  if (to_tail) {
    const size_t t = (static_cast<size_t>(bh) * G.tail_cap + (pos & (G.tail_cap - 1))) * D;
    *reinterpret_cast<uint4*>(a.lay.tail_k + t + c0) = klo;
    *reinterpret_cast<uint4*>(a.lay.tail_k + t + half + c0) = khi;
    *reinterpret_cast<uint4*>(a.lay.tail_v + t + c0) = vlo;
    *reinterpret_cast<uint4*>(a.lay.tail_v + t + half + c0) = vhi;
  }
  if (to_sink) {
    const size_t t = (static_cast<size_t>(bh) * G.n_sink_slots + pos) * D;
    *reinterpret_cast<uint4*>(a.lay.sink_k + t + c0) = klo;
    *reinterpret_cast<uint4*>(a.lay.sink_k + t + half + c0) = khi;
    *reinterpret_cast<uint4*>(a.lay.sink_v + t + c0) = vlo;
    *reinterpret_cast<uint4*>(a.lay.sink_v + t + half + c0) = vhi;
  }
}

// ---------------------------------------------------------------- TurboQuant
// Token pairs each warp of the quantiser takes in turn (the CTA's setup,
// the codebook boundaries and the warp's signs, is paid once for them).
constexpr int kTqPairsPerWarp = 8;
// The code search's guess table: w in [0, 1] falls in cell floor(kTqCells w)
// (kTqCells + 1 cells with w = 1); the cell's entry is the number of
// boundaries <= its start, valid while no cell holds two boundaries.
constexpr int kTqCells = 256;
constexpr float kMagicF = 12582912.0f;  // 1.5 * 2^23: x + kMagicF keeps floor / rint(x) in the low bits
constexpr uint32_t kMagicBitsF = 0x4B400000u;

// Builds the guess table of nb ascending boundaries (threads of the CTA in
// turn); returns, through ok (shared, set to 1 before), whether every cell
// holds at most one boundary.
__device__ __forceinline__ void tq_guess_table(const float* bnd, int nb, uint8_t* guess, int* ok) {
  for (int j = threadIdx.x; j <= kTqCells; j += blockDim.x) {
    const float lo = static_cast<float>(j) / kTqCells, hi = static_cast<float>(j + 1) / kTqCells;
    int below = 0, inside = 0;
    for (int k = 0; k < nb; ++k) {
      below += bnd[k] <= lo ? 1 : 0;
      inside += (bnd[k] > lo && bnd[k] < hi) ? 1 : 0;
    }
    guess[j] = static_cast<uint8_t>(below);
    if (inside > 1) *ok = 0;
  }
}

// One warp per (token, b, h): Foundry "TurboQuant KV Cache Compression - Spec",
// "Algorithm Detail" with the as-built order (signs, then the Walsh-Hadamard
// butterflies with stage length 1, 2, 4, ..., then 1/sqrt(d)); the norm is the
// fixed pairwise tree over x^2 (stride D/2, D/4, ..., 1) and its sqrt; each
// coordinate becomes w = (y/n + 1) * 0.5 and its code counts the boundaries
// <= w. Lane l holds channels i*32 + l.
template <int D>
__device__ __forceinline__ float tq_code_row(float (&x)[D / 32], const float (&sg)[D / 32], const float* bnd,
                                             const uint8_t* guess, int bits, float rsq, uint8_t* codes_smem) {
  constexpr int NS = D / 32;
  const int lane = threadIdx.x & 31;
  float y[NS], sq[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    y[i] = __fmul_rn(x[i], sg[i]);
    sq[i] = __fmul_rn(x[i], x[i]);
  }
#pragma unroll
  for (int len = 1; len < 32; len <<= 1) {
    // the upper lane of a butterfly takes o - y, the lower y + o: one FMA
    // with y times -1 or +1 (exact), rounded like the subtraction or sum
    const float sgn = (lane & len) ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, y[i], len);
      y[i] = __fmaf_rn(y[i], sgn, o);
    }
  }
#pragma unroll
  for (int sl = 1; sl < NS; sl <<= 1) {
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      if ((i & sl) == 0) {
        const float u = y[i], v = y[i + sl];
        y[i] = __fadd_rn(u, v);
        y[i + sl] = __fsub_rn(u, v);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NS; ++i) y[i] = __fmul_rn(y[i], rsq);
#pragma unroll
  for (int sl = NS / 2; sl >= 1; sl >>= 1) {
#pragma unroll
    for (int i = 0; i < sl; ++i) sq[i] = __fadd_rn(sq[i], sq[i + sl]);
  }
  float acc = sq[0];
#pragma unroll
  for (int st = 16; st >= 1; st >>= 1) {
    const float o = __shfl_down_sync(0xffffffffu, acc, st);
    if (lane < st) acc = __fadd_rn(acc, o);
  }
  const float n = __shfl_sync(0xffffffffu, __fsqrt_rn(acc), 0);
  // u = RN(y / n) by Markstein's correction step from RN(1 / n) (P.
  // Markstein, IBM J. Res. Dev. 34(1), 1990), exact like the division
  const float rn = n > 0.0f ? __frcp_rn(n) : 0.0f;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    float u = 0.0f;
    if (n > 0.0f) {
      const float q0 = __fmul_rn(y[i], rn);
      u = __fmaf_rn(__fmaf_rn(-q0, n, y[i]), rn, q0);
    }
    const float w = __fmul_rn(__fadd_rn(u, 1.0f), 0.5f);
    // the number of boundaries <= w (ascending, padded to 16 with 2.0,
    // above every w): from the guess of w's cell (w is in [0, 1]) and one
    // comparison, or a branchless binary search where a cell holds two
    // boundaries
    int code = 0;
    if (guess) {
      const float t = __fmaf_rd(w, static_cast<float>(kTqCells), kMagicF);  // kMagicF + floor(kTqCells w)
      const int g = guess[__float_as_uint(t) - kMagicBitsF];
      code = g + (w >= bnd[g] ? 1 : 0);
    } else {
#pragma unroll
      for (int step = 8; step >= 1; step >>= 1)
        if (step < (1 << bits)) code += (w >= bnd[code + step - 1]) ? step : 0;
    }
    codes_smem[i * 32 + lane] = static_cast<uint8_t>(code);
  }
  return n;
}

// One warp per token pair (2 pi, 2 pi + 1) of a group, for the tokens of
// the pair this call appends. Codes go to the decode's layouts
// (kvq_layout.h): K in fragment order (each token's fields are whole bytes
// of four lanes' strings, written as 16-bit halves), V in token-pair rows
// (a field holds both tokens' codes, so the warp writes the whole row; where
// only one token of the pair is in this call, the other's bits are kept).
// The norms go to the group's norm arrays.
template <int D>
__global__ void __launch_bounds__(128) tq_quantize_kernel(AppendArgs a, int64_t pair_begin, int n_pairs) {
  constexpr int NS = D / 32;
  __shared__ uint8_t codes[4][2][2][D];  // [warp][K, V][token of the pair][channel]
  __shared__ float s_bk[16], s_bv[16];
  __shared__ uint8_t s_gk[kTqCells + 1], s_gv[kTqCells + 1];
  __shared__ int s_ok[2];
  const Geometry& G = a.geo;
  if (threadIdx.x < 16) {
    s_bk[threadIdx.x] = (threadIdx.x < (1 << G.kb) - 1) ? a.tab.cb_k[threadIdx.x] : 2.0f;
    s_bv[threadIdx.x] = (threadIdx.x < (1 << G.vb) - 1) ? a.tab.cb_v[threadIdx.x] : 2.0f;
  }
  if (threadIdx.x < 2) s_ok[threadIdx.x] = 1;
  __syncthreads();
  tq_guess_table(s_bk, (1 << G.kb) - 1, s_gk, &s_ok[0]);
  tq_guess_table(s_bv, (1 << G.vb) - 1, s_gv, &s_ok[1]);
  __syncthreads();
  const uint8_t* gk = s_ok[0] ? s_gk : nullptr;
  const uint8_t* gv = s_ok[1] ? s_gv : nullptr;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float sg[NS];  // this lane's signs (channels i * 32 + lane)
#pragma unroll
  for (int i = 0; i < NS; ++i) sg[i] = a.tab.signs[i * 32 + lane];
  // the CTA's pairs [first, first + 4 kTqPairsPerWarp), warp w taking w, w + 4, ...
  const int first = blockIdx.x * 4 * kTqPairsPerWarp;
  const int last = min(n_pairs, first + 4 * kTqPairsPerWarp);
  for (int pi_idx = first + warp; pi_idx < last; pi_idx += 4) {
  __syncwarp();  // the previous pair's codes have been read
  const int64_t pi = pair_begin + pi_idx;
  const int bh = blockIdx.y;
  const int bf16 = G.act_bf16;
  const float rsq = static_cast<float>(1.0 / sqrt(static_cast<double>(D)));
  const int64_t p0 = 2 * pi;
  const int slot = static_cast<int>((p0 / kGroup) % G.n_slots);
  uint8_t* chunk = a.lay.chunks + (static_cast<size_t>(bh) * G.n_slots + slot) * G.chunk.bytes;
  const int kb = G.kb, vb = G.vb;
  // both tokens' rows first (a token not in this call reads the other's
  // row and stores nothing), so that their butterflies and searches overlap
  bool have[2];
  float xk[2][NS], xv[2][NS];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int64_t pos = p0 + e;
    have[e] = pos >= a.L0 && pos < a.L0 + a.n;
    const int64_t lp = have[e] ? pos : (have[e ^ 1] ? p0 + (e ^ 1) : a.L0);
    const size_t in_row = (static_cast<size_t>(bh) * a.n + (lp - a.L0)) * D;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      xk[e][i] = act_to_float(a.k[in_row + i * 32 + lane], bf16);
      xv[e][i] = act_to_float(a.v[in_row + i * 32 + lane], bf16);
    }
    if (a.tab.rope) {
      const float* tr = a.tab.rope + static_cast<size_t>(lp) * D;
#pragma unroll
      for (int i = 0; i < NS / 2; ++i) {
        const int c = i * 32 + lane;
        float rx, ry;
        rope_pair(xk[e][i], xk[e][i + NS / 2], tr[2 * c], tr[2 * c + 1], &rx, &ry);
        xk[e][i] = act_to_float(float_to_act(rx, bf16), bf16);
        xk[e][i + NS / 2] = act_to_float(float_to_act(ry, bf16), bf16);
      }
    }
  }
  float nk[2], nv[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    nk[e] = tq_code_row<D>(xk[e], sg, s_bk, gk, kb, rsq, codes[warp][0][e]);
    nv[e] = tq_code_row<D>(xv[e], sg, s_bv, gv, vb, rsq, codes[warp][1][e]);
  }
  __syncwarp();
  for (int e = 0; e < 2; ++e) {
    if (!have[e]) continue;
    const int r = static_cast<int>((p0 + e) % kGroup);
    if (lane == 0) {
      reinterpret_cast<float*>(chunk + G.chunk.kmeta_off)[r] = nk[e];
      reinterpret_cast<float*>(chunk + G.chunk.vmeta_off)[r] = nv[e];
    }
    // K: block b = 2 (r / 16) + (r / 8) % 2 of lanes 4 (r % 8) + t; lane
    // 2 BBK / 2 ... writes 16-bit half h of the block of lane t
    const int bbk = D * kb / 32;  // bytes per token block
    const int pw = piece_words(D * kb / 32);
    const int blk = 2 * (r >> 4) + ((r >> 3) & 1);
    if (lane < 2 * bbk) {
      const int t = lane / (bbk / 2), hw = lane % (bbk / 2);
      uint32_t half = 0;
      for (int j = (16 * hw) / (2 * kb); j * 2 * kb < 16 * hw + 16; ++j) {  // the fields that meet this half
        const int c0 = 16 * (j >> 1) + 2 * t + 8 * (j & 1);
        const uint32_t f = codes[warp][0][e][c0] | (static_cast<uint32_t>(codes[warp][0][e][c0 + 1]) << kb);
        const int sh = 2 * kb * j - 16 * hw;
        half |= sh >= 0 ? (f << sh) : (f >> -sh);
      }
      half &= 0xffffu;
      const int L = 4 * (r & 7) + t;
      *reinterpret_cast<uint16_t*>(chunk + G.chunk.kc_off + lane_byte_offset(L, blk * bbk + 2 * hw, pw)) =
          static_cast<uint16_t>(half);
    }
  }
  // V: the pair row, 16-bit halves; a token not in this call keeps its bits
  const int rb = tq_vrow_bytes(D, vb);
  uint16_t* row = reinterpret_cast<uint16_t*>(chunk + G.chunk.vc_off + static_cast<size_t>((p0 % kGroup) / 2) * rb);
  const uint32_t lo_mask = (1u << vb) - 1u;
  const uint32_t keep = (have[0] ? lo_mask : 0u) | (have[1] ? lo_mask << vb : 0u);  // bits of a field written here
  for (int hw = lane; hw < rb / 2; hw += 32) {
    uint32_t half = 0, mask = 0;
    for (int f = (16 * hw) / (2 * vb); f * 2 * vb < 16 * hw + 16; ++f) {  // the fields that meet this half
      const int c = 8 * (f % (D / 8)) + f / (D / 8);  // the channel of field position f
      const uint32_t v = (have[0] ? codes[warp][1][0][c] : 0u) | (have[1] ? static_cast<uint32_t>(codes[warp][1][1][c]) << vb : 0u);
      const int sh = 2 * vb * f - 16 * hw;
      half |= sh >= 0 ? (v << sh) : (v >> -sh);
      mask |= sh >= 0 ? (keep << sh) : (keep >> -sh);
    }
    mask &= 0xffffu;
    if (mask != 0xffffu) half = (row[hw] & ~mask) | (half & mask);
    row[hw] = static_cast<uint16_t>(half);
  }
  }
}

// ---------------------------------------------------------------- KVSink rows
// Copy the selected sink rows of the prefill input (keys rotated like every
// other key) into the sink buffer.
__global__ void sink_gather_kernel(AppendArgs a) {
  const Geometry& G = a.geo;
  const int D = G.D, half = D / 2, cpr = half / 8;
  const int j = blockIdx.x, bh = blockIdx.y, b = bh / G.H;
  const int64_t pos = a.lay.sink_pos[b * kMaxSinks + j];
  const int64_t row = pos - a.L0;
  if (row < 0 || row >= a.n) return;
  for (int idx = threadIdx.x; idx < cpr; idx += blockDim.x) {
    const int c0 = idx * 8;
    const size_t in_row = (static_cast<size_t>(bh) * a.n + row) * D;
    uint4 klo = *reinterpret_cast<const uint4*>(a.k + in_row + c0);
    uint4 khi = *reinterpret_cast<const uint4*>(a.k + in_row + half + c0);
    const uint4 vlo = *reinterpret_cast<const uint4*>(a.v + in_row + c0);
    const uint4 vhi = *reinterpret_cast<const uint4*>(a.v + in_row + half + c0);
    if (a.tab.rope) rotate8(klo, khi, a.tab.rope + static_cast<size_t>(pos) * D, c0, G.act_bf16);
    const size_t t = (static_cast<size_t>(bh) * G.n_sink_slots + j) * D;
    *reinterpret_cast<uint4*>(a.lay.sink_k + t + c0) = klo;
    *reinterpret_cast<uint4*>(a.lay.sink_k + t + half + c0) = khi;
    *reinterpret_cast<uint4*>(a.lay.sink_v + t + c0) = vlo;
    *reinterpret_cast<uint4*>(a.lay.sink_v + t + half + c0) = vhi;
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s, int64_t* launches) {
  const Geometry& G = a.geo;
  const int BH = G.B * G.H;
  if (!G.mode_tq && a.n_groups > 0) {
    dim3 grid(a.n_groups, BH);
    if (G.D == 128) (G.kb <= 3 ? launch_flush_d128_k23 : launch_flush_d128_k48)(a, grid, s);
    else (G.kb <= 3 ? launch_flush_d64_k23 : launch_flush_d64_k48)(a, grid, s);
    ++*launches;
  }
  if (G.mode_tq && a.n > 0) {  // token pairs (2 pi, 2 pi + 1) that meet [L0, L0 + n)
    const int64_t pair_begin = a.L0 / 2, pair_end = (a.L0 + a.n + 1) / 2;
    const int n_pairs = static_cast<int>(pair_end - pair_begin);
    dim3 grid((n_pairs + 4 * kTqPairsPerWarp - 1) / (4 * kTqPairsPerWarp), BH);
    if (G.D == 128) tq_quantize_kernel<128><<<grid, 128, 0, s>>>(a, pair_begin, n_pairs);
    else tq_quantize_kernel<64><<<grid, 128, 0, s>>>(a, pair_begin, n_pairs);
    ++*launches;
  }
  // rows [r0, r1) of the append that go to the sink buffer or the tail: the
  // overlay sinks at the front, then everything from tail_from on
  auto write_rows = [&](int64_t r0, int64_t r1) {
    if (r0 >= r1) return;
    const int rows = static_cast<int>(r1 - r0);
    const int cpr = G.D / 16;
    const int threads = 128;
    dim3 grid(static_cast<unsigned>((static_cast<int64_t>(rows) * cpr + threads - 1) / threads), BH);
    tail_write_kernel<<<grid, threads, 0, s>>>(a, static_cast<int>(r0), rows);
    ++*launches;
  };
  const int64_t n_front = a.L0 < G.n_sink ? std::min<int64_t>(a.n, G.n_sink - a.L0) : 0;
  const int64_t t0 = std::min<int64_t>(a.n, std::max<int64_t>(0, a.tail_from - a.L0));
  if (t0 <= n_front) {
    write_rows(0, t0 < a.n ? a.n : n_front);  // one run
  } else {
    write_rows(0, n_front);
    write_rows(t0, a.n);
  }
  return cudaGetLastError();
}

cudaError_t launch_sink_gather(const AppendArgs& a, cudaStream_t s, int64_t* launches) {
  if (a.n_dyn_sel <= 0) return cudaSuccess;
  dim3 grid(a.n_dyn_sel, a.geo.B * a.geo.H);
  sink_gather_kernel<<<grid, 32, 0, s>>>(a);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace kvq
