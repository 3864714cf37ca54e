// Append-side kernels: exact tail ring and sink buffer writes, KIVI group
// quantisation (with KVSink calibration exclusion), TurboQuant per-token
// quantisation, and the KVSink sink-row gather.
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

// ---------------------------------------------------------------- KIVI flush
// One CTA per (completed group, b, h); D threads. Quantisation follows
// posttrainllm "StreamingLLM + KIVI", "Affine quantisation formula", in the
// unsigned-code form: scale = max((max - min) / (2^b - 1), 1e-5) in fp32,
// scale and zero (= min) stored as fp16, code = rint((x - zero) / scale)
// clamped to [0, 2^b - 1], computed from the stored fp16 values promoted to
// fp32. K: one (scale, zero) per channel over the group's 32 tokens; V: one
// per token per 32-channel group (the KIVI group idea, same page, "Caveats").
// KVSink (VeloxQuant-MLX "KVSink-Adapted Sink Protection", "How it works" 3):
// before calibration every sink row of the group is replaced by its nearest
// non-sink row (ties to the earlier row); sink rows keep the substitute's
// codes and the group's mask bit tells attention to skip them.
__device__ __forceinline__ void quantize_slice_params(float mn, float mx, int bits, __half* sh,
                                                      __half* zh, float* s, float* z) {
  const float lb = static_cast<float>((1 << bits) - 1);
  const float s32 = fmaxf(__fdiv_rn(__fsub_rn(mx, mn), lb), 1e-5f);
  *sh = __float2half_rn(s32);
  *zh = __float2half_rn(mn);
  *s = __half2float(*sh);
  *z = __half2float(*zh);
}

// Code of x for a slice with stored scale s, zero z and reciprocal rs =
// 1/s (correctly rounded): rint of the correctly rounded quotient (x - z) / s
// (x - z rounded on its own), clamped to [0, LB]. The quotient is formed as
// (x - z) * rs, whose distance to the correctly rounded quotient is at most
// about 2^-22 of its magnitude (two roundings of 2^-24 each, plus the
// quotient's own): below 6.2e-5 while |q| <= 257. Away from a half-integer by
// more than 1e-4 the two round to the same integer, and beyond 257 the clamp
// decides; within 1e-4 of a half-integer the correctly rounded division is
// taken, so the code equals rint(fl((x - z) / s)) in every case.
// The correctly rounded quotient's integer, out of line: it runs only for
// quotients within 1e-4 of a half-integer, and inlined it would multiply the
// size of every quantisation loop.
__device__ __noinline__ float rint_of_quotient(float d, float s) { return rintf(__fdiv_rn(d, s)); }

template <int LB>
__device__ __forceinline__ uint32_t quantize_code(float x, float s, float z, float rs) {
  const float d = __fsub_rn(x, z);
  const float q = __fmul_rn(d, rs);
  float qr = rintf(q);
  if (fabsf(__fsub_rn(q, qr)) > 0.4999f) qr = rint_of_quotient(d, s);  // within 1e-4 of a half-integer
  qr = fminf(fmaxf(qr, 0.0f), static_cast<float>(LB));
  return static_cast<uint32_t>(qr);
}

// Bit position of the element i (0 .. 32/BITS - 1) of a packed word (the
// frag_bits layout: pair j = i / 2, element e = i % 2).
template <int BITS>
__device__ __forceinline__ int word_bit(int i) {
  const int j = i >> 1, e = i & 1;
  if (BITS == 2) return 8 * (j & 3) + 2 * (j >> 2) + 4 * e;
  if (BITS == 4) return 16 * (j & 1) + 4 * (j >> 1) + 8 * e;
  return 8 * j + 16 * e;
}

// Byte offset, from the lane's base (K: cs[g][t D / 4], V: cs[2t][g]), of
// the code of fragment element f of lane (g, t) (kvq_layout.h k_frag_pos,
// v_frag_pos): a constant, so that packing loads each code with one
// shared-memory byte load (rows are D + 4 bytes: the lanes' loads fall in
// distinct banks or share a word).
template <int D, bool IS_K, bool PR>
__device__ __forceinline__ constexpr int frag_code_offset(int f) {
  const int e = f & 1, r = (f >> 1) & 3, hi = f >> 3;
  if (IS_K) {
    const int mt = hi / (D / 16), s = hi % (D / 16);
    if (PR) return (16 * mt + 8 * (r & 1)) * (D + 4) + 2 * s + (r >> 1) + e * (D / 2);
    return (16 * mt + 8 * (r & 1)) * (D + 4) + 4 * s + 2 * (r >> 1) + e;
  }
  const int m = hi >> 1, kb = hi & 1;
  return (16 * kb + e + 8 * (r >> 1)) * (D + 4) + 16 * m + 8 * (r & 1);
}

// Words [W0, W0 + NW) of every lane's K (IS_K) or V fragment block, packed
// by this warp's thread `lane` for fragment lane `lane`; 3-bit codes in
// blocks of three words (W0, NW multiples of 3). PR: the K channel order of
// keys stored before RoPE (kvq_layout.h k_frag_pos).
template <int D, int BITS, bool IS_K, bool PR, int W0, int NW>
__device__ __forceinline__ void pack_words(const uint8_t (*cs)[D + 4], uint8_t* region, int lane) {
  constexpr int WPL = D * BITS / 32, PW = piece_words(WPL);
  const int g = lane >> 2, t = lane & 3;
  const uint8_t* base = IS_K ? &cs[g][t * (PR ? D / 8 : D / 4)] : &cs[2 * t][g];
  if constexpr (BITS == 3) {
#pragma unroll
    for (int blk = W0 / 3; blk < (W0 + NW) / 3; ++blk) {
      uint32_t w[3] = {0u, 0u, 0u};
#pragma unroll
      for (int i = 0; i < 32; ++i) frag3_put(w, i, base[frag_code_offset<D, IS_K, PR>(32 * blk + i)]);
#pragma unroll
      for (int q = 0; q < 3; ++q)
        *reinterpret_cast<uint32_t*>(region + code_word_offset(lane, 3 * blk + q, PW)) = w[q];
    }
  } else {
    constexpr int PER = 32 / BITS;
#pragma unroll
    for (int w = W0; w < W0 + NW; ++w) {
      uint32_t word = 0;
#pragma unroll
      for (int i = 0; i < PER; ++i)
        word |= static_cast<uint32_t>(base[frag_code_offset<D, IS_K, PR>(w * PER + i)]) << word_bit<BITS>(i);
      *reinterpret_cast<uint32_t*>(region + code_word_offset(lane, w, PW)) = word;
    }
  }
}

// The codes of one group (cs[token][channel]) in the decode kernel's
// fragment order: the D / 32 warps of the CTA take equal shares of the
// words of every lane's block.
template <int D, int BITS, bool IS_K, bool PR = false>
__device__ __forceinline__ void pack_fragments(const uint8_t (*cs)[D + 4], uint8_t* region, int tid) {
  constexpr int NWARP = D / 32, NW = D * BITS / 32 / NWARP;
  static_assert(NW * NWARP == D * BITS / 32 && (BITS != 3 || NW % 3 == 0), "equal shares");
  const int warp = tid >> 5, lane = tid & 31;
  if (warp == 0) pack_words<D, BITS, IS_K, PR, 0, NW>(cs, region, lane);
  else if (warp == 1) pack_words<D, BITS, IS_K, PR, NW, NW>(cs, region, lane);
  if constexpr (NWARP > 2) {
    if (warp == 2) pack_words<D, BITS, IS_K, PR, 2 * NW, NW>(cs, region, lane);
    else if (warp == 3) pack_words<D, BITS, IS_K, PR, 3 * NW, NW>(cs, region, lane);
  }
}

// KB, VB: code widths (levels 2^bits - 1), packed tight (3-bit codes in
// blocks of three words, kvq_layout.h frag3_put).
template <int D, int KB, int VB>
__global__ void __launch_bounds__(D) kivi_flush_kernel(AppendArgs a) {
  constexpr int HALF = D / 2, NV = D / 32, CPR = HALF / 8;
  constexpr int LK = (1 << KB) - 1, LV = (1 << VB) - 1;
  constexpr int SK = KB, SV = VB;
  // the group's rows as activation-dtype bits (rows padded by 16 bytes so
  // that 16-byte row stores stay aligned and column reads spread over banks)
  __shared__ __align__(16) uint16_t xk[32][D + 8];
  __shared__ __align__(16) uint16_t xv[32][D + 8];
  __shared__ __align__(16) uint8_t ck[32][D + 4];  // rows padded by a word: the packing gathers down columns
  __shared__ __align__(16) uint8_t cv[32][D + 4];
  __shared__ int sub[32];
  __shared__ uint32_t smask;
  const Geometry& G = a.geo;
  const int tid = threadIdx.x;
  const int bh = blockIdx.y, b = bh / G.H, h = bh % G.H;
  const int64_t g = a.g_first + blockIdx.x;
  const int64_t p0 = g * kGroup;
  const int slot = static_cast<int>(g % G.n_slots);
  const int bf16 = G.act_bf16;

  if (tid < 32) {  // KVSink: the nearest non-sink row of each row (ties to the earlier)
    uint32_t m = 0;
    if (a.dyn_active) {
      for (int j = 0; j < a.n_dyn_sel; ++j) {
        const int64_t p = a.lay.sink_pos[b * kMaxSinks + j];
        if (p >= p0 && p < p0 + kGroup) m |= 1u << (p - p0);
      }
    }
    const int r = tid;
    int sr = r;
    if (((m >> r) & 1u) && m != 0xFFFFFFFFu) {
      for (int d = 1; d < 32; ++d) {
        if (r - d >= 0 && !((m >> (r - d)) & 1u)) { sr = r - d; break; }
        if (r + d < 32 && !((m >> (r + d)) & 1u)) { sr = r + d; break; }
      }
    }
    sub[r] = sr;
    if (r == 0) smask = m;
  }
  __syncthreads();

#pragma unroll
  for (int idx = tid; idx < 32 * CPR; idx += D) {
    const int r = idx / CPR, c0 = (idx % CPR) * 8;
    const int64_t pos = p0 + sub[r];
    uint4 klo, khi, vlo, vhi;
    if (pos < a.L0) {
      const size_t t = (static_cast<size_t>(bh) * G.tail_cap + (pos & (G.tail_cap - 1))) * D;
      klo = *reinterpret_cast<const uint4*>(a.lay.tail_k + t + c0);
      khi = *reinterpret_cast<const uint4*>(a.lay.tail_k + t + HALF + c0);
      vlo = *reinterpret_cast<const uint4*>(a.lay.tail_v + t + c0);
      vhi = *reinterpret_cast<const uint4*>(a.lay.tail_v + t + HALF + c0);
    } else {
      const size_t t = (static_cast<size_t>(bh) * a.n + (pos - a.L0)) * D;
      klo = *reinterpret_cast<const uint4*>(a.k + t + c0);
      khi = *reinterpret_cast<const uint4*>(a.k + t + HALF + c0);
      vlo = *reinterpret_cast<const uint4*>(a.v + t + c0);
      vhi = *reinterpret_cast<const uint4*>(a.v + t + HALF + c0);
      if (a.tab.rope) rotate8(klo, khi, a.tab.rope + static_cast<size_t>(pos) * D, c0, bf16);
    }
    *reinterpret_cast<uint4*>(&xk[r][c0]) = klo;
    *reinterpret_cast<uint4*>(&xk[r][HALF + c0]) = khi;
    *reinterpret_cast<uint4*>(&xv[r][c0]) = vlo;
    *reinterpret_cast<uint4*>(&xv[r][HALF + c0]) = vhi;
  }
  __syncthreads();

  uint8_t* chunk = a.lay.chunks + (static_cast<size_t>(bh) * G.n_slots + slot) * G.chunk.bytes;
  // the first half of the threads quantise K (two channels each, over the
  // 32 tokens), the second half V (two (token, 32-channel group) slices
  // each); every value is read from shared memory once (32-bit and 16-byte
  // loads) and kept in registers between min/max and the codes
  if (tid < D / 2) {  // K: channels 2 tid, 2 tid + 1
    const int c = 2 * tid;
    auto kpair = [&](int r) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(&xk[r][c]);
      return make_float2(act_to_float(static_cast<uint16_t>(w & 0xffffu), bf16),
                         act_to_float(static_cast<uint16_t>(w >> 16), bf16));
    };
    float2 x = kpair(0);
    float mn0 = x.x, mx0 = x.x, mn1 = x.y, mx1 = x.y;
#pragma unroll 4
    for (int r = 1; r < 32; ++r) {
      x = kpair(r);
      mn0 = fminf(mn0, x.x), mx0 = fmaxf(mx0, x.x);
      mn1 = fminf(mn1, x.y), mx1 = fmaxf(mx1, x.y);
    }
    __half sh0, zh0, sh1, zh1;
    float s0, z0, s1, z1;
    quantize_slice_params(mn0, mx0, KB, &sh0, &zh0, &s0, &z0);
    quantize_slice_params(mn1, mx1, KB, &sh1, &zh1, &s1, &z1);
    const float rs0 = __frcp_rn(s0), rs1 = __frcp_rn(s1);
#pragma unroll 4
    for (int r = 0; r < 32; ++r) {
      x = kpair(r);
      const uint32_t q0 = quantize_code<LK>(x.x, s0, z0, rs0), q1 = quantize_code<LK>(x.y, s1, z1, rs1);
      *reinterpret_cast<uint16_t*>(&ck[r][c]) = static_cast<uint16_t>(q0 | (q1 << 8));
    }
    // K scales and zeros in the decode's B-operand orders (keys stored
    // before RoPE: the natural channel order)
    __half* km = reinterpret_cast<__half*>(chunk + G.chunk.kmeta_off);
    const bool pr = G.k_pre_rope;
    km[pr ? c : kmeta_pos(D, c)] = sh0;
    km[D + (pr ? c : kzero_pos(D, c))] = zh0;
    km[pr ? c + 1 : kmeta_pos(D, c + 1)] = sh1;
    km[D + (pr ? c + 1 : kzero_pos(D, c + 1))] = zh1;
  } else {  // V: two (token r, channel group vg) slices
#pragma unroll 1
    for (int k = 0; k < 2; ++k) {
      const int si = tid - D / 2 + k * (D / 2);
      const int r = si % 32, vg = si / 32, base = 32 * vg;  // a warp's lanes take 32 rows: no bank conflicts
      const uint4* row = reinterpret_cast<const uint4*>(&xv[r][base]);  // 4 x 8 values
      auto unpack8 = [&](const uint4& u, float (&o)[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[2 * i] = act_to_float(static_cast<uint16_t>(w[i] & 0xffffu), bf16);
          o[2 * i + 1] = act_to_float(static_cast<uint16_t>(w[i] >> 16), bf16);
        }
      };
      __half sh, zh;
      float o[8];
      if (VB == 4 && G.v_q4_0) {
        // the symmetric q4_0 form ([P3] "Summary"): d = m / -8 with m the value
        // of largest magnitude (the first in channel order on ties), code
        // min(15, floor(x / d + 8.5)) from the stored d, zero -8 d
        float m = 0.0f, am = -1.0f;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          unpack8(row[q], o);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (fabsf(o[i]) > am) am = fabsf(o[i]), m = o[i];
        }
        sh = __float2half_rn(__fdiv_rn(m, -8.0f));
        const float d = __half2float(sh);
        zh = __float2half_rn(__fmul_rn(d, -8.0f));  // exact: a power-of-two multiple
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          unpack8(row[q], o);
          uint32_t cw[2] = {0u, 0u};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float qv = 8.0f;
            if (d != 0.0f) qv = fminf(fmaxf(floorf(__fadd_rn(__fdiv_rn(o[i], d), 8.5f)), 0.0f), 15.0f);
            cw[i >> 2] |= static_cast<uint32_t>(qv) << (8 * (i & 3));
          }
          reinterpret_cast<uint32_t*>(&cv[r][base + 8 * q])[0] = cw[0];  // rows of D + 4 bytes: 4-byte aligned
          reinterpret_cast<uint32_t*>(&cv[r][base + 8 * q])[1] = cw[1];
        }
      } else {
        float mn = INFINITY, mx = -INFINITY;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          unpack8(row[q], o);
#pragma unroll
          for (int i = 0; i < 8; ++i) mn = fminf(mn, o[i]), mx = fmaxf(mx, o[i]);
        }
        float sv, zv;
        quantize_slice_params(mn, mx, VB, &sh, &zh, &sv, &zv);
        const float rs = __frcp_rn(sv);
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          unpack8(row[q], o);
          uint32_t cw[2] = {0u, 0u};
#pragma unroll
          for (int i = 0; i < 8; ++i) cw[i >> 2] |= quantize_code<LV>(o[i], sv, zv, rs) << (8 * (i & 3));
          reinterpret_cast<uint32_t*>(&cv[r][base + 8 * q])[0] = cw[0];  // rows of D + 4 bytes: 4-byte aligned
          reinterpret_cast<uint32_t*>(&cv[r][base + 8 * q])[1] = cw[1];
        }
      }
      __half* vm = reinterpret_cast<__half*>(chunk + G.chunk.vmeta_off);
      vm[vscale_pos(NV, r, vg)] = sh;
      vm[vzero_pos(NV, r, vg)] = zh;
    }
  }
  __syncthreads();

  // pack in the decode kernel's fragment order (kvq_layout.h)
  if (G.k_pre_rope) pack_fragments<D, SK, true, true>(ck, chunk + G.chunk.kc_off, tid);
  else pack_fragments<D, SK, true>(ck, chunk + G.chunk.kc_off, tid);
  pack_fragments<D, SV, false>(cv, chunk + G.chunk.vc_off, tid);
  if (G.n_dyn && h == 0 && tid == 0) a.lay.sink_mask[b * G.n_slots + slot] = smask;
}

template <int D>
void launch_flush(const AppendArgs& a, dim3 grid, cudaStream_t s) {
  const int kb = a.geo.kb, vb = a.geo.vb;
#define KVQ_FLUSH(K, V) \
  if (kb == K && vb == V) { kivi_flush_kernel<D, K, V><<<grid, D, 0, s>>>(a); return; }
  KVQ_FLUSH(2, 2) KVQ_FLUSH(2, 3) KVQ_FLUSH(2, 4) KVQ_FLUSH(2, 8)
  KVQ_FLUSH(3, 2) KVQ_FLUSH(3, 3) KVQ_FLUSH(3, 4) KVQ_FLUSH(3, 8)
  KVQ_FLUSH(4, 2) KVQ_FLUSH(4, 3) KVQ_FLUSH(4, 4) KVQ_FLUSH(4, 8)
  KVQ_FLUSH(8, 2) KVQ_FLUSH(8, 3) KVQ_FLUSH(8, 4) KVQ_FLUSH(8, 8)
#undef KVQ_FLUSH
}

// ---------------------------------------------------------------- TurboQuant
// One warp per (token, b, h): Foundry "TurboQuant KV Cache Compression - Spec",
// "Algorithm Detail" with the as-built order (signs, then the Walsh-Hadamard
// butterflies with stage length 1, 2, 4, ..., then 1/sqrt(d)); the norm is the
// fixed pairwise tree over x^2 (stride D/2, D/4, ..., 1) and its sqrt; each
// coordinate becomes w = (y/n + 1) * 0.5 and its code counts the boundaries
// <= w. Lane l holds channels i*32 + l.
template <int D>
__device__ __forceinline__ float tq_code_row(float (&x)[D / 32], const float* signs, const float* bnd,
                                             int bits, float rsq, uint8_t* codes_smem) {
  constexpr int NS = D / 32;
  const int lane = threadIdx.x & 31;
  float y[NS], sq[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    y[i] = __fmul_rn(x[i], signs[i * 32 + lane]);
    sq[i] = __fmul_rn(x[i], x[i]);
  }
#pragma unroll
  for (int len = 1; len < 32; len <<= 1) {
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, y[i], len);
      y[i] = (lane & len) ? __fsub_rn(o, y[i]) : __fadd_rn(y[i], o);
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
  const int nb = (1 << bits) - 1;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const float u = (n > 0.0f) ? __fdiv_rn(y[i], n) : 0.0f;
    const float w = __fmul_rn(__fadd_rn(u, 1.0f), 0.5f);
    int code = 0;
    for (int k = 0; k < nb; ++k) code += (w >= bnd[k]) ? 1 : 0;
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
  __shared__ float s_signs[D];
  __shared__ float s_bk[16], s_bv[16];
  const Geometry& G = a.geo;
  for (int i = threadIdx.x; i < D; i += blockDim.x) s_signs[i] = a.tab.signs[i];
  if (threadIdx.x < 16) {
    s_bk[threadIdx.x] = (threadIdx.x < (1 << G.kb) - 1) ? a.tab.cb_k[threadIdx.x] : 2.0f;
    s_bv[threadIdx.x] = (threadIdx.x < (1 << G.vb) - 1) ? a.tab.cb_v[threadIdx.x] : 2.0f;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pi_idx = blockIdx.x * 4 + warp;
  if (pi_idx >= n_pairs) return;
  const int64_t pi = pair_begin + pi_idx;
  const int bh = blockIdx.y;
  const int bf16 = G.act_bf16;
  const float rsq = static_cast<float>(1.0 / sqrt(static_cast<double>(D)));
  const int64_t p0 = 2 * pi;
  const int slot = static_cast<int>((p0 / kGroup) % G.n_slots);
  uint8_t* chunk = a.lay.chunks + (static_cast<size_t>(bh) * G.n_slots + slot) * G.chunk.bytes;
  const int kb = G.kb, vb = G.vb;
  bool have[2];
  for (int e = 0; e < 2; ++e) {
    const int64_t pos = p0 + e;
    have[e] = pos >= a.L0 && pos < a.L0 + a.n;
    if (!have[e]) continue;
    const size_t in_row = (static_cast<size_t>(bh) * a.n + (pos - a.L0)) * D;
    float xk[NS], xv[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      xk[i] = act_to_float(a.k[in_row + i * 32 + lane], bf16);
      xv[i] = act_to_float(a.v[in_row + i * 32 + lane], bf16);
    }
    if (a.tab.rope) {
      const float* tr = a.tab.rope + static_cast<size_t>(pos) * D;
#pragma unroll
      for (int i = 0; i < NS / 2; ++i) {
        const int c = i * 32 + lane;
        float rx, ry;
        rope_pair(xk[i], xk[i + NS / 2], tr[2 * c], tr[2 * c + 1], &rx, &ry);
        xk[i] = act_to_float(float_to_act(rx, bf16), bf16);
        xk[i + NS / 2] = act_to_float(float_to_act(ry, bf16), bf16);
      }
    }
    const int r = static_cast<int>(pos % kGroup);
    const float nk = tq_code_row<D>(xk, s_signs, s_bk, kb, rsq, codes[warp][0][e]);
    const float nv = tq_code_row<D>(xv, s_signs, s_bv, vb, rsq, codes[warp][1][e]);
    if (lane == 0) {
      reinterpret_cast<float*>(chunk + G.chunk.kmeta_off)[r] = nk;
      reinterpret_cast<float*>(chunk + G.chunk.vmeta_off)[r] = nv;
    }
    __syncwarp();
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
    __syncwarp();
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
    if (G.D == 128) launch_flush<128>(a, grid, s);
    else launch_flush<64>(a, grid, s);
    ++*launches;
  }
  if (G.mode_tq && a.n > 0) {  // token pairs (2 pi, 2 pi + 1) that meet [L0, L0 + n)
    const int64_t pair_begin = a.L0 / 2, pair_end = (a.L0 + a.n + 1) / 2;
    const int n_pairs = static_cast<int>(pair_end - pair_begin);
    dim3 grid((n_pairs + 3) / 4, BH);
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
