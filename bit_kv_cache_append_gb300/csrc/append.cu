// Append-side kernels: exact tail ring and sink buffer writes, TurboQuant
// per-token quantisation and the KVSink sink-row gather; the launch of the
// KIVI group quantisation (flush.cuh).
#include <algorithm>
#include <type_traits>

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
// (kTqCells + 1 cells with w = 1); the cell's entry is the number g of
// boundaries <= its start and the boundary g (the next one up, or the
// padding above every w), valid while no cell holds two boundaries.
constexpr int kTqCells = 256;
constexpr float kMagicF = 12582912.0f;  // 1.5 * 2^23: x + kMagicF keeps floor / rint(x) in the low bits
constexpr uint32_t kMagicBitsF = 0x4B400000u;

// Builds the guess table of nb ascending boundaries, padded with 2.0 (threads
// of the CTA in turn): entry (bits of boundary g, g); returns, through ok
// (shared, set to 1 before), whether every cell holds at most one boundary.
__device__ __forceinline__ void tq_guess_table(const float* bnd, int nb, uint2* guess, int* ok) {
  for (int j = threadIdx.x; j <= kTqCells; j += blockDim.x) {
    const float lo = static_cast<float>(j) / kTqCells, hi = static_cast<float>(j + 1) / kTqCells;
    int below = 0, inside = 0;
    for (int k = 0; k < nb; ++k) {
      below += bnd[k] <= lo ? 1 : 0;
      inside += (bnd[k] > lo && bnd[k] < hi) ? 1 : 0;
    }
    guess[j] = make_uint2(__float_as_uint(bnd[below]), static_cast<uint32_t>(below));
    if (inside > 1) *ok = 0;
  }
}

// How a row's codes are searched: the three 2-bit boundaries in registers,
// the guess table and one comparison, or a binary search over the padded
// boundaries in shared memory (where a guess cell holds two boundaries).
enum TqSearch { kTqRegs = 0, kTqGuess = 1, kTqBinary = 2 };

// One row (token, b, h) of a warp: Foundry "TurboQuant KV Cache Compression
// - Spec", "Algorithm Detail" with the as-built order (signs, then the
// Walsh-Hadamard butterflies with stage length 1, 2, 4, ..., then 1/sqrt(d));
// the norm is the fixed pairwise tree over x^2 (stride D/2, D/4, ..., 1) and
// its sqrt; each coordinate becomes w = (y/n + 1) * 0.5 and its code counts
// the boundaries <= w. Lane l holds channels i*32 + l; bs[k] is -1 on the
// lanes that take the upper end of a butterfly of length 2^k, else +1.
template <int D, int BITS, int SEARCH>
__device__ __forceinline__ float tq_code_row(const float (&x)[D / 32], const float (&sg)[D / 32], const float (&bs)[5],
                                             const float (&br)[3], const float* bnd, const uint2* guess, float rsq,
                                             uint32_t (&code)[D / 32]) {
  constexpr int NS = D / 32;
  float y[NS], sq[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    y[i] = __fmul_rn(x[i], sg[i]);
    sq[i] = __fmul_rn(x[i], x[i]);
  }
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    // the upper lane of a butterfly takes o - y, the lower y + o: one FMA
    // with y times -1 or +1 (exact), rounded like the subtraction or sum
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, y[i], 1 << k);
      y[i] = __fmaf_rn(y[i], bs[k], o);
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
  for (int sl = NS / 2; sl >= 1; sl >>= 1) {
#pragma unroll
    for (int i = 0; i < sl; ++i) sq[i] = __fadd_rn(sq[i], sq[i + sl]);
  }
  // the tree's cross-lane levels as xor butterflies: lanes l and l ^ st add
  // the same two partial sums (in either order: addition commutes), so
  // every lane ends with the tree's root
  float acc = sq[0];
#pragma unroll
  for (int st = 16; st >= 1; st >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, st));
  const float n = __fsqrt_rn(acc);
  // u = RN(y / n) by Markstein's correction step from RN(1 / n) (P.
  // Markstein, IBM J. Res. Dev. 34(1), 1990), exact like the division; a
  // zero norm takes 1/n = 0, which gives u = 0
  const float rn = n > 0.0f ? __frcp_rn(n) : 0.0f;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const float yr = __fmul_rn(y[i], rsq);
    const float q0 = __fmul_rn(yr, rn);
    const float u = __fmaf_rn(__fmaf_rn(-q0, n, yr), rn, q0);
    // RN(u / 2 + 1 / 2) = RN(u + 1) / 2: halving is exact for u + 1 in [0, 2]
    const float w = __fmaf_rn(u, 0.5f, 0.5f);
    uint32_t c;
    if constexpr (SEARCH == kTqRegs) {  // three ascending boundaries
      c = w >= br[1] ? 2u : 0u;
      c += w >= (c ? br[2] : br[0]) ? 1u : 0u;
    } else if constexpr (SEARCH == kTqGuess) {
      // kMagicF + floor(kTqCells w), w clamped to [0, 1] for the cell only: u
      // may stray past -1 or 1 by rounding, and a w outside [0, 1] is coded
      // right from cell 0 (guess 0) or cell kTqCells (every boundary but the
      // padding below it)
      const float t = __fmaf_rd(__saturatef(w), static_cast<float>(kTqCells), kMagicF);
      const uint2 cell = guess[__float_as_uint(t) - kMagicBitsF];
      c = cell.y + (w >= __uint_as_float(cell.x) ? 1u : 0u);
    } else {  // boundaries padded to 16 with 2.0, above every w
      c = 0;
#pragma unroll
      for (int step = 8; step >= 1; step >>= 1)
        if (step < (1 << BITS)) c += (w >= bnd[c + step - 1]) ? step : 0;
    }
    code[i] = c;
  }
  return n;
}

// ORs value v, placed at bit `bit` of a little-endian string of W words,
// into the string (v < 2^(32 - bit % 32) unless the string has a next word).
template <int W>
__device__ __forceinline__ void tq_place(uint32_t (&s)[W], int word, int shift, uint32_t v, bool straddle) {
  if (!straddle) {
    s[word] |= v << shift;
  } else {
    const uint64_t x = static_cast<uint64_t>(v) << shift;
    s[word] |= static_cast<uint32_t>(x);
    if (word + 1 < W) s[word + 1] |= static_cast<uint32_t>(x >> 32);
  }
}

// Word k of a string held in registers (k from the lane, a select chain).
template <int W>
__device__ __forceinline__ uint32_t tq_word(const uint32_t (&s)[W], int k) {
  uint32_t r = s[0];
#pragma unroll
  for (int j = 1; j < W; ++j)
    if (k == j) r = s[j];
  return r;
}

// One warp per token pair (2 pi, 2 pi + 1) of a group, for the tokens of
// the pair this call appends; KB and VB are the code widths. Codes go to the
// decode's layouts (kvq_layout.h), packed in registers and merged across
// lanes by shuffles:
//  * K in fragment order: string t (0..3) of a token holds the channels c
//    with (c mod 8) / 2 = t, channel c at bit KB (2 (c / 8) + c mod 2); the
//    lanes l with (l mod 8) / 2 = t hold them (channel i 32 + l at bit
//    KB (8 i + 2 (l / 8) + l mod 2)). The string is the token's block
//    (2 (r / 16) + (r / 8) mod 2, r its row in the group) of decode lane
//    4 (r mod 8) + t.
//  * V in token-pair rows: field f = (c mod 8) D / 8 + c / 8 holds both
//    tokens' codes of channel c; the lanes with l mod 8 = p hold the fields
//    of block p (channel i 32 + l at field p D / 8 + 4 i + l / 8). A token
//    not in this call keeps its bits of the row.
// The norms go to the group's norm arrays.
template <int D, int KB, int VB>
__global__ void __launch_bounds__(128) tq_quantize_kernel(AppendArgs a, int64_t pair_begin, int n_pairs) {
  constexpr int NS = D / 32;
  constexpr int KSB = D / 4 * KB;           // bits of a K string
  constexpr int KW = (KSB + 31) / 32;       // its words
  constexpr int BBK = D * KB / 32;          // bytes of a K string (a token block of a decode lane)
  constexpr bool KWORDS = BBK % 4 == 0;     // written as words, else as 16-bit halves
  constexpr int VSB = D / 8 * 2 * VB;       // bits of a V block (fields of one l mod 8)
  constexpr int VW = (VSB + 31) / 32;
  constexpr int VBB = VSB / 8;              // its bytes
  constexpr bool VWORDS = VBB % 4 == 0;
  __shared__ float s_bk[16], s_bv[16];
  __shared__ uint2 s_gk[kTqCells + 1], s_gv[kTqCells + 1];
  __shared__ int s_ok[2];
  const Geometry& G = a.geo;
  if (threadIdx.x < 16) {
    s_bk[threadIdx.x] = (threadIdx.x < (1 << KB) - 1) ? a.tab.cb_k[threadIdx.x] : 2.0f;
    s_bv[threadIdx.x] = (threadIdx.x < (1 << VB) - 1) ? a.tab.cb_v[threadIdx.x] : 2.0f;
  }
  if (threadIdx.x < 2) s_ok[threadIdx.x] = 1;
  __syncthreads();
  if (KB > 2) tq_guess_table(s_bk, (1 << KB) - 1, s_gk, &s_ok[0]);
  if (VB > 2) tq_guess_table(s_bv, (1 << VB) - 1, s_gv, &s_ok[1]);
  __syncthreads();
  const bool gk_ok = s_ok[0] != 0, gv_ok = s_ok[1] != 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float sg[NS];  // this lane's signs (channels i * 32 + lane)
#pragma unroll
  for (int i = 0; i < NS; ++i) sg[i] = a.tab.signs[i * 32 + lane];
  float bs[5];
#pragma unroll
  for (int k = 0; k < 5; ++k) bs[k] = (lane >> k) & 1 ? -1.0f : 1.0f;
  const float brk[3] = {s_bk[0], s_bk[1], s_bk[2]}, brv[3] = {s_bv[0], s_bv[1], s_bv[2]};
  const int bh = blockIdx.y;
  const int bf16 = G.act_bf16;
  const float rsq = static_cast<float>(1.0 / sqrt(static_cast<double>(D)));
  const int q8 = lane >> 3, lo = lane & 1;
  // the CTA's pairs [first, first + 4 kTqPairsPerWarp), warp w taking w, w + 4, ...
  const int first = blockIdx.x * 4 * kTqPairsPerWarp;
  const int last = min(n_pairs, first + 4 * kTqPairsPerWarp);
  for (int pi_idx = first + warp; pi_idx < last; pi_idx += 4) {
    const int64_t p0 = 2 * (pair_begin + pi_idx);
    const int slot = static_cast<int>((p0 / kGroup) % G.n_slots);
    uint8_t* chunk = a.lay.chunks + (static_cast<size_t>(bh) * G.n_slots + slot) * G.chunk.bytes;
    // both tokens' rows first (a token not in this call reads the other's
    // row and stores nothing), so that their butterflies and searches overlap
    bool have[2];
    float xk[2][NS], xv[2][NS];
    int64_t lp[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int64_t pos = p0 + e;
      have[e] = pos >= a.L0 && pos < a.L0 + a.n;
      lp[e] = have[e] ? pos : (have[e ^ 1] ? p0 + (e ^ 1) : a.L0);
    }
    auto load = [&](auto bf) {
      constexpr bool BF = decltype(bf)::value;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const size_t in_row = (static_cast<size_t>(bh) * a.n + (lp[e] - a.L0)) * D;
#pragma unroll
        for (int i = 0; i < NS; ++i) {
          const uint16_t kbits = a.k[in_row + i * 32 + lane], vbits = a.v[in_row + i * 32 + lane];
          xk[e][i] = BF ? __uint_as_float(static_cast<uint32_t>(kbits) << 16) : __half2float(__ushort_as_half(kbits));
          xv[e][i] = BF ? __uint_as_float(static_cast<uint32_t>(vbits) << 16) : __half2float(__ushort_as_half(vbits));
        }
      }
    };
    if (bf16) load(std::true_type{});
    else load(std::false_type{});
    if (a.tab.rope) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float* tr = a.tab.rope + static_cast<size_t>(lp[e]) * D;
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
    uint32_t ck[2][NS], cv[2][NS];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if constexpr (KB == 2) nk[e] = tq_code_row<D, KB, kTqRegs>(xk[e], sg, bs, brk, s_bk, s_gk, rsq, ck[e]);
      else if (gk_ok) nk[e] = tq_code_row<D, KB, kTqGuess>(xk[e], sg, bs, brk, s_bk, s_gk, rsq, ck[e]);
      else nk[e] = tq_code_row<D, KB, kTqBinary>(xk[e], sg, bs, brk, s_bk, s_gk, rsq, ck[e]);
      if constexpr (VB == 2) nv[e] = tq_code_row<D, VB, kTqRegs>(xv[e], sg, bs, brv, s_bv, s_gv, rsq, cv[e]);
      else if (gv_ok) nv[e] = tq_code_row<D, VB, kTqGuess>(xv[e], sg, bs, brv, s_bv, s_gv, rsq, cv[e]);
      else nv[e] = tq_code_row<D, VB, kTqBinary>(xv[e], sg, bs, brv, s_bv, s_gv, rsq, cv[e]);
    }
    const int r0 = static_cast<int>(p0 % kGroup);  // the pair's first row in the group
    if (lane < 2 && (lane ? have[1] : have[0])) {  // lane e stores token e's norms
      reinterpret_cast<float*>(chunk + G.chunk.kmeta_off)[r0 + lane] = lane ? nk[1] : nk[0];
      reinterpret_cast<float*>(chunk + G.chunk.vmeta_off)[r0 + lane] = lane ? nv[1] : nv[0];
    }

    // K: this lane's codes in both tokens' strings t = (lane mod 8) / 2, then
    // the strings merged over the eight lanes of each t: lane bit 4 picks the
    // token (the other token's words go to the partner), bits 3 and 0 merge
    uint32_t ks[2][KW];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
#pragma unroll
      for (int w = 0; w < KW; ++w) ks[e][w] = 0u;
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        const int bit0 = KB * 8 * i;  // the lane's bit is bit0 + KB (2 q8 + lo)
        tq_place<KW>(ks[e], bit0 / 32, bit0 % 32 + KB * (2 * q8 + lo), ck[e][i], KB == 3);
      }
    }
    const int ktok = (lane >> 4) & 1;
    uint32_t kstr[KW];
#pragma unroll
    for (int w = 0; w < KW; ++w) {
      const uint32_t send = ktok ? ks[0][w] : ks[1][w];
      kstr[w] = (ktok ? ks[1][w] : ks[0][w]) | __shfl_xor_sync(0xffffffffu, send, 16);
      kstr[w] |= __shfl_xor_sync(0xffffffffu, kstr[w], 8);
      kstr[w] |= __shfl_xor_sync(0xffffffffu, kstr[w], 1);
    }
    if (ktok ? have[1] : have[0]) {
      const int r = r0 + ktok;
      const int t = (lane & 7) >> 1, idx = 2 * (q8 & 1) + lo;  // idx: the writer among the four lanes
      const int L = 4 * (r & 7) + t, blk = 2 * (r >> 4) + ((r >> 3) & 1);
      constexpr int pw = piece_words(D * KB / 32);
      if constexpr (KWORDS) {
        if (idx < KW)
          *reinterpret_cast<uint32_t*>(chunk + G.chunk.kc_off + lane_byte_offset(L, blk * BBK + 4 * idx, pw)) =
              tq_word<KW>(kstr, idx);
      } else {
        if (idx < BBK / 2)
          *reinterpret_cast<uint16_t*>(chunk + G.chunk.kc_off + lane_byte_offset(L, blk * BBK + 2 * idx, pw)) =
              static_cast<uint16_t>(tq_word<KW>(kstr, idx >> 1) >> (16 * (idx & 1)));
      }
    }

    // V: the fields of block p = lane mod 8 (both tokens' codes), merged
    // over the four lanes of each p (lane bits 3 and 4)
    const uint32_t keep_lo = (have[0] ? (1u << VB) - 1u : 0u) | (have[1] ? ((1u << VB) - 1u) << VB : 0u);
    const bool whole = have[0] && have[1];
    uint32_t vs[VW], vm[VW];
#pragma unroll
    for (int w = 0; w < VW; ++w) vs[w] = vm[w] = 0u;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const int bit0 = 2 * VB * 4 * i;  // the lane's field is at bit0 + 2 VB q8
      const uint32_t f = (cv[0][i] | (cv[1][i] << VB)) & keep_lo;
      tq_place<VW>(vs, bit0 / 32, bit0 % 32 + 2 * VB * q8, f, VB == 3);
      if (!whole) tq_place<VW>(vm, bit0 / 32, bit0 % 32 + 2 * VB * q8, keep_lo, VB == 3);
    }
#pragma unroll
    for (int w = 0; w < VW; ++w) {
      vs[w] |= __shfl_xor_sync(0xffffffffu, vs[w], 8);
      vs[w] |= __shfl_xor_sync(0xffffffffu, vs[w], 16);
      if (!whole) {
        vm[w] |= __shfl_xor_sync(0xffffffffu, vm[w], 8);
        vm[w] |= __shfl_xor_sync(0xffffffffu, vm[w], 16);
      }
    }
    {
      const int p = lane & 7, idx = q8;  // idx: the writer among the four lanes
      uint8_t* row = chunk + G.chunk.vc_off + static_cast<size_t>(r0 / 2) * tq_vrow_bytes(D, VB) + p * VBB;
      if constexpr (VWORDS) {
        if (idx < VW) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(row + 4 * idx);
          uint32_t val = tq_word<VW>(vs, idx);
          if (!whole) {
            const uint32_t m = tq_word<VW>(vm, idx);
            val = (*dst & ~m) | (val & m);
          }
          *dst = val;
        }
      } else {
        if (idx < VBB / 2) {
          uint16_t* dst = reinterpret_cast<uint16_t*>(row + 2 * idx);
          uint32_t val = tq_word<VW>(vs, idx >> 1) >> (16 * (idx & 1));
          if (!whole) {
            const uint32_t m = tq_word<VW>(vm, idx >> 1) >> (16 * (idx & 1));
            val = (*dst & ~m) | (val & m);
          }
          *dst = static_cast<uint16_t>(val);
        }
      }
    }
  }
}

template <int D, int KB>
void launch_tq_kb(const AppendArgs& a, dim3 grid, cudaStream_t s, int64_t pair_begin, int n_pairs) {
  switch (a.geo.vb) {
    case 2: tq_quantize_kernel<D, KB, 2><<<grid, 128, 0, s>>>(a, pair_begin, n_pairs); break;
    case 3: tq_quantize_kernel<D, KB, 3><<<grid, 128, 0, s>>>(a, pair_begin, n_pairs); break;
    default: tq_quantize_kernel<D, KB, 4><<<grid, 128, 0, s>>>(a, pair_begin, n_pairs); break;
  }
}

template <int D>
void launch_tq(const AppendArgs& a, dim3 grid, cudaStream_t s, int64_t pair_begin, int n_pairs) {
  switch (a.geo.kb) {
    case 2: launch_tq_kb<D, 2>(a, grid, s, pair_begin, n_pairs); break;
    case 3: launch_tq_kb<D, 3>(a, grid, s, pair_begin, n_pairs); break;
    default: launch_tq_kb<D, 4>(a, grid, s, pair_begin, n_pairs); break;
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
    if (G.D == 128) launch_tq<128>(a, grid, s, pair_begin, n_pairs);
    else launch_tq<64>(a, grid, s, pair_begin, n_pairs);
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
