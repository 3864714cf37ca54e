// KIVI group quantisation: the flush of completed 32-token groups into the
// code chunks, as whole words of the decode kernel's fragment order
// (kvq_layout.h) built in registers; each thread's values wait in its own
// column of a shared-memory scratch between min/max and the per-word loop.
//
// One CTA per (group, b, h), D threads: the first D/2 quantise K, the rest V.
// Quantisation follows posttrainllm "StreamingLLM + KIVI", "Affine
// quantisation formula", in the unsigned-code form: scale = max((max - min) /
// (2^b - 1), 1e-5) in fp32, scale and zero (= min) stored as fp16, code =
// rint((x - zero) / scale) clamped to [0, 2^b - 1], computed from the stored
// fp16 values promoted to fp32. K: one (scale, zero) per channel over the
// group's 32 tokens; V: one per token per 32-channel group (the KIVI group
// idea, same page, "Caveats"). The symmetric q4_0 V form ([P3] "Summary"):
// d = m / -8 with m the value of largest magnitude (the first in channel
// order on ties), code min(15, floor(x / d + 8.5)) from the stored d, zero
// -8 d.
//
// KVSink (VeloxQuant-MLX "KVSink-Adapted Sink Protection", "How it works" 3):
// before calibration every sink row of the group is replaced by its nearest
// non-sink row (ties to the earlier row); sink rows keep the substitute's
// codes and the group's mask bit tells attention to skip them.
//
// Work split (each thread quantises 64 values and writes whole words):
//   K thread (cq, tq): channel quads 4 cq .. 4 cq + 3 and D/2 + 4 cq .. (the
//     RoPE partners), tokens 16 mt + g + 8 ts for the four g of its quarter
//     (mt = tq / 2, g in 4 (tq % 2) .. +3, ts in {0, 1}). The four tq lanes of
//     a quad are adjacent and reduce min / max with two shuffles. Every K
//     fragment word (kvq_layout.h k_frag_pos) covers tokens g, g + 8 of one
//     mt and channels inside one thread's quads, except the 2-bit words
//     (two quads: one shuffle joins the halves) and the 3-bit blocks (four
//     quads: the quad values of the fourth lane are shuffled to the other
//     three, which store).
//   V thread (m, t, kb): tokens 16 kb + 2 t + e + 8 h (e, h in {0, 1}) and
//     channels 16 m .. 16 m + 15. The two m of a 32-channel group are
//     adjacent lanes and reduce the per-token min / max with one shuffle.
//     A V fragment word (v_frag_pos) covers channels g, g + 8 of one m and
//     those four tokens of one kb (2-bit: both kb, 3-bit: both kb and both m
//     of the group), joined the same way as for K.
//
// Codes: the correctly rounded quotient fl(d / s) (d = x - z rounded) is
// formed without a division by Markstein's correction step (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): with r = RN(1/s), q0 = RN(d r),
// the residual e = RN(d - q0 s) is exact and RN(q0 + e r) = RN(d / s)
// (no underflow can occur here: a quotient that can round to a nonzero
// code has d >= s / 2 >= 5e-6). Adding 1.5 * 2^23 then rounds it half to
// even to an integer held in the low mantissa bits, which one integer
// multiply-add places in the word. Where the stored zero's and scale's fp16
// rounding could move a code out of [0, 2^b - 1] (checked per slice from its
// min and max) the thread's words take the exact path (a division per value
// and the clamp).
#pragma once

#include "kvq_device.cuh"
#include "kvq_layout.h"

namespace kvq {
namespace {

// 1.5 * 2^23: for |y| < 2^22, the float nearest y + kMagic is kMagic +
// rint(y) (ties to even, kMagic being even), so the integer sits in the low
// mantissa bits.
constexpr float kMagic = 12582912.0f;
constexpr uint32_t kMagicBits = 0x4B400000u;

template <bool BF16>
__device__ __forceinline__ float act_lo(uint32_t w) {
  if constexpr (BF16) return __uint_as_float(w << 16);
  else return __low2float(*reinterpret_cast<const __half2*>(&w));
}
template <bool BF16>
__device__ __forceinline__ float act_hi(uint32_t w) {
  if constexpr (BF16) return __uint_as_float(w & 0xffff0000u);
  else return __high2float(*reinterpret_cast<const __half2*>(&w));
}
template <bool BF16>
__device__ __forceinline__ float act_half(uint32_t w, int h) {
  return h ? act_hi<BF16>(w) : act_lo<BF16>(w);
}
// Elementwise min / max of two packed pairs (exact: the result is one of
// the inputs).
template <bool BF16>
__device__ __forceinline__ uint32_t act_min2(uint32_t a, uint32_t b) {
  uint32_t r;
  if constexpr (BF16) {
    const __nv_bfloat162 m = __hmin2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                     *reinterpret_cast<const __nv_bfloat162*>(&b));
    r = *reinterpret_cast<const uint32_t*>(&m);
  } else {
    const __half2 m = __hmin2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    r = *reinterpret_cast<const uint32_t*>(&m);
  }
  return r;
}
template <bool BF16>
__device__ __forceinline__ uint32_t act_max2(uint32_t a, uint32_t b) {
  uint32_t r;
  if constexpr (BF16) {
    const __nv_bfloat162 m = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                     *reinterpret_cast<const __nv_bfloat162*>(&b));
    r = *reinterpret_cast<const uint32_t*>(&m);
  } else {
    const __half2 m = __hmax2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    r = *reinterpret_cast<const uint32_t*>(&m);
  }
  return r;
}
// Two floats rounded to the activation dtype (nearest even), packed low |
// high << 16 (one conversion instruction for both).
template <bool BF16>
__device__ __forceinline__ uint32_t act_pack(float lo, float hi) {
  uint32_t r;
  if constexpr (BF16) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    r = *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __half2 v = __floats2half2_rn(lo, hi);
    r = *reinterpret_cast<const uint32_t*>(&v);
  }
  return r;
}

// RN(n / s) from r = RN(1 / s) (Markstein's correction step).
__device__ __forceinline__ float quotient(float n, float s, float r) {
  const float q0 = __fmul_rn(n, r);
  const float e = __fmaf_rn(-q0, s, n);
  return __fmaf_rn(e, r, q0);
}

// Stored scale and zero of one slice from its min and max: sh, zh the fp16
// values, zs = zh | sh << 16 (the bits), r the correctly rounded 1 / s. ok
// is cleared where a code of a value in [mn, mx] could leave [0, LB] (the
// zero's rounding moved it by more than 0.375 s), so the clamp is needed.
template <int LB>
__device__ __forceinline__ void slice_params(float mn, float mx, __half* sh, __half* zh, uint32_t* zs,
                                             float* r, bool* ok) {
  constexpr float lb = static_cast<float>(LB), inv_lb = 1.0f / lb;  // RN(1 / LB), folded by the compiler
  const float s32 = fmaxf(quotient(__fsub_rn(mx, mn), lb, inv_lb), 1e-5f);
  *sh = __float2half_rn(s32);
  *zh = __float2half_rn(mn);
  const float s = __half2float(*sh), z = __half2float(*zh);
  *zs = static_cast<uint32_t>(__half_as_ushort(*zh)) | (static_cast<uint32_t>(__half_as_ushort(*sh)) << 16);
  *r = __frcp_rn(s);
  const float dlo = __fsub_rn(mn, z), dhi = __fsub_rn(mx, z);
  *ok = *ok && dlo >= -0.375f * s && dhi <= (static_cast<float>(LB) + 0.375f) * s;
}

// The code of x with the correctly rounded division (the exact path).
__device__ __forceinline__ uint32_t exact_code(float x, uint32_t zs, int lb) {
  const float z = __half2float(__ushort_as_half(static_cast<unsigned short>(zs & 0xffffu)));
  const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(zs >> 16)));
  const float q = rintf(__fdiv_rn(__fsub_rn(x, z), s));
  return static_cast<uint32_t>(fminf(fmaxf(q, 0.0f), static_cast<float>(lb)));
}

// Per-slice constants of the fast path: zero, scale and RN(1 / scale).
struct Slice {
  float z, s, r;
};
__device__ __forceinline__ Slice make_slice(uint32_t zs, float r) {
  Slice q;
  q.z = __half2float(__ushort_as_half(static_cast<unsigned short>(zs & 0xffffu)));
  q.s = __half2float(__ushort_as_half(static_cast<unsigned short>(zs >> 16)));
  q.r = r;
  return q;
}

// Two slices' constants side by side for the packed FP32x2 instructions:
// -zero, -scale and RN(1 / scale).
struct Slice2 {
  float2 nz, ns, r;
};
__device__ __forceinline__ Slice2 pair_slices(const Slice& a, const Slice& b) {
  Slice2 q;
  q.nz = make_float2(-a.z, -b.z);
  q.ns = make_float2(-a.s, -b.s);
  q.r = make_float2(a.r, b.r);
  return q;
}

// The codes of two values of two slices, each accumulated as (kMagicBits +
// code) << bit into its word (corr collects the kMagicBits parts, constants
// after unrolling): d = RN(x - z), q0 = RN(d r), e = RN(d - q0 s), RN(q0 + e r)
// = RN(d / s), then + 1.5 * 2^23 rounds half to even; two values per
// instruction with Blackwell's FP32x2 add, multiply and FMA (each lane
// rounded as the scalar instruction would).
__device__ __forceinline__ void add_code2(float2 x, const Slice2& q, int bit0, int bit1, uint32_t& acc0,
                                          uint32_t& corr0, uint32_t& acc1, uint32_t& corr1) {
  const float2 d = __fadd2_rn(x, q.nz);
  const float2 q0 = __fmul2_rn(d, q.r);
  const float2 e = __ffma2_rn(q0, q.ns, d);
  const float2 t = __fadd2_rn(__ffma2_rn(e, q.r, q0), make_float2(kMagic, kMagic));
  acc0 += __float_as_uint(t.x) << bit0;
  corr0 += kMagicBits << bit0;
  acc1 += __float_as_uint(t.y) << bit1;
  corr1 += kMagicBits << bit1;
}

// q4_0: min(15, floor(RN(RN(x / d) + 8.5))) clamped at 0, d the stored scale
// (code 8 where d = 0); r = RN(1 / d).
__device__ __forceinline__ uint32_t q40_fast(float x, float d, float r) {
  const float y = __fadd_rn(quotient(x, d, r), 8.5f);
  const float t = __fadd_rd(fminf(fmaxf(y, -1.0f), 16.0f), kMagic);  // floor, in the low mantissa bits
  const int c = min(max(static_cast<int>(__float_as_uint(t) - kMagicBits), 0), 15);
  return d == 0.0f ? 8u : static_cast<uint32_t>(c);
}

// The three words of a 3-bit block from its eight quad values (four codes
// each, one per byte, kvq_layout.h frag3_put): quads 2w, 2w + 1 in word w
// for w < 3; quads 6 and 7 split into low bits (words 0, 1) and high bits
// (word 2). qa, qb are the two quads of word w, x, y the quads 6 and 7.
__device__ __forceinline__ uint32_t block3_word(int w, uint32_t qa, uint32_t qb, uint32_t x, uint32_t y) {
  const uint32_t base = qa | (qb << 3);
  if (w == 0) return base | ((x & 0x03030303u) << 6);
  if (w == 1) return base | ((y & 0x03030303u) << 6);
  return base | ((x & 0x04040404u) << 4) | ((y & 0x04040404u) << 5);
}

__device__ __forceinline__ void store_word(uint8_t* region, int lane, int w, int pw, uint32_t v) {
  *reinterpret_cast<uint32_t*>(region + code_word_offset(lane, w, pw)) = v;
}

// Where a K or V row of the group comes from: the tail ring for positions
// before the append, else the appended rows.
__device__ __forceinline__ const uint16_t* group_row(const AppendArgs& a, const uint16_t* tail, const uint16_t* in,
                                                    int bh, int64_t pos) {
  const Geometry& G = a.geo;
  if (pos < a.L0) return tail + (static_cast<size_t>(bh) * G.tail_cap + (pos & (G.tail_cap - 1))) * G.D;
  return in + (static_cast<size_t>(bh) * a.n + (pos - a.L0)) * G.D;
}

// ---------------------------------------------------------------- K
// Element (ts, k) of one g of a K thread (k: 0..3 low quad, 4..7 high quad)
// -> accumulator and bit (3-bit: quad value, bit 8 x byte).
template <int BITS, bool PR>
struct KMap {
  static constexpr int NQ = BITS == 8 ? 4 : BITS == 3 ? 4 : (BITS == 2 && PR) ? 1 : 2;
  __host__ __device__ static constexpr int acc(int ts, int k) {
    const int kk = k & 3;
    (void)ts;
    if (!PR) {
      if (BITS == 8 || BITS == 3) return 2 * (k >> 2) + (kk >> 1);
      return k >> 2;
    }
    if (BITS == 4) return kk >> 1;
    if (BITS == 2) return 0;
    return kk;  // 8, 3
  }
  __host__ __device__ static constexpr int bit(int ts, int k) {
    const int kk = k & 3;
    if (!PR) {
      if (BITS == 4) return 16 * ts + 4 * (kk >> 1) + 8 * (k & 1);
      if (BITS == 8) return 8 * ts + 16 * (k & 1);
      if (BITS == 2) return 8 * (ts + 2 * (kk >> 1)) + 4 * (k & 1);
      return 8 * (2 * ts + (k & 1));
    }
    const int e = k >> 2;
    if (BITS == 4) return 16 * ts + 4 * (kk & 1) + 8 * e;
    if (BITS == 8) return 8 * ts + 16 * e;
    if (BITS == 2) return 8 * (ts + 2 * (kk & 1)) + 2 * (kk >> 1) + 4 * e;
    return 8 * (2 * ts + e);
  }
};

// The exact path for one g of a K thread: the 16 values re-read from the
// rows (rotated again where the fast path rotated them) and coded with the
// correctly rounded division; zsk[c] holds channel c's stored zero | scale.
template <int D, int KB, bool BF16, bool PR>
__device__ __noinline__ uint4 k_exact_g(const uint16_t* row0, const uint16_t* row1, const float* tr0,
                                        const float* tr1, int cq, const uint32_t* zsk) {
  using M = KMap<KB, PR>;
  constexpr int LB = (1 << KB) - 1, HALF = D / 2;
  uint32_t acc[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int ts = 0; ts < 2; ++ts) {
    const uint16_t* row = ts ? row1 : row0;
    const float* tr = ts ? tr1 : tr0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = 4 * cq + (k & 3), c = k < 4 ? i : HALF + i;
      float xv = act_to_float(row[c], BF16);
      if (tr) {
        float rx, ry;
        rope_pair(act_to_float(row[i], BF16), act_to_float(row[HALF + i], BF16), tr[2 * i], tr[2 * i + 1], &rx, &ry);
        xv = act_to_float(float_to_act(k < 4 ? rx : ry, BF16), BF16);
      }
      acc[M::acc(ts, k)] |= exact_code(xv, zsk[c], LB) << M::bit(ts, k);
    }
  }
  return make_uint4(acc[0], acc[1], acc[2], acc[3]);
}

// lin: the group's first K row when its 32 rows are consecutive rows of the
// appended input (no sink substitution, nothing from the tail), else null.
template <int D, int KB, bool BF16, bool PR>
__device__ __forceinline__ void flush_k(const AppendArgs& a, const int* sub, int64_t p0, int bh, uint8_t* chunk,
                                        uint32_t* zsk, uint4 (*scratch)[D], const uint16_t* lin) {
  using M = KMap<KB, PR>;
  constexpr int LB = (1 << KB) - 1, HALF = D / 2, S = D / 16;
  constexpr int PW = piece_words(D * KB / 32);
  const Geometry& G = a.geo;
  const int tid = threadIdx.x, lane = tid & 31;
  const int cq = (tid >> 5) * 8 + (lane >> 2), tq = lane & 3, mt = tq >> 1, gb = 4 * (tq & 1);
  const float* rope = PR ? nullptr : a.tab.rope;
  // every load is issued before the first use: the rows, then (RoPE at
  // append) the table rows of the appended tokens
  uint32_t x[8][4];
  auto row_idx = [&](int i) { return 16 * mt + gb + (i >> 1) + 8 * (i & 1); };
  auto pos_of = [&](int i) {
    const int r = row_idx(i);
    return p0 + (sub ? sub[r] : r);
  };
  auto load_rows = [&](auto row_of) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint16_t* row = row_of(i);
      const uint2 lo = __ldg(reinterpret_cast<const uint2*>(row + 4 * cq));
      const uint2 hi = __ldg(reinterpret_cast<const uint2*>(row + HALF + 4 * cq));
      x[i][0] = lo.x, x[i][1] = lo.y, x[i][2] = hi.x, x[i][3] = hi.y;
    }
  };
  if (lin) load_rows([&](int i) { return lin + row_idx(i) * D; });  // the group's rows, in order, all appended
  else load_rows([&](int i) { return group_row(a, a.lay.tail_k, a.k, bh, pos_of(i)); });
  if (rope) {  // RoPE at the absolute position, rounded back to the activation dtype
#pragma unroll
    for (int i0 = 0; i0 < 8; i0 += 4) {  // four tokens' table rows in flight at a time
      float4 cs[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4* tr = reinterpret_cast<const float4*>(rope + static_cast<size_t>(pos_of(i0 + i)) * D + 8 * cq);
        cs[i][0] = __ldg(tr), cs[i][1] = __ldg(tr + 1);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t* xi = x[i0 + i];
        if (pos_of(i0 + i) < a.L0) continue;  // tail rows were rotated when they were appended
        const float c[8] = {cs[i][0].x, cs[i][0].y, cs[i][0].z, cs[i][0].w,
                            cs[i][1].x, cs[i][1].y, cs[i][1].z, cs[i][1].w};
        float rx[4], ry[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          rope_pair(act_half<BF16>(xi[kk >> 1], kk & 1), act_half<BF16>(xi[2 + (kk >> 1)], kk & 1), c[2 * kk],
                    c[2 * kk + 1], &rx[kk], &ry[kk]);
        xi[0] = act_pack<BF16>(rx[0], rx[1]), xi[1] = act_pack<BF16>(rx[2], rx[3]);
        xi[2] = act_pack<BF16>(ry[0], ry[1]), xi[3] = act_pack<BF16>(ry[2], ry[3]);
      }
    }
  }
  // per-channel min / max over the 32 tokens: 8 here, then the quad's 4 lanes
  uint32_t mn[4], mx[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    mn[p] = x[0][p], mx[p] = x[0][p];
#pragma unroll
    for (int i = 1; i < 8; ++i) mn[p] = act_min2<BF16>(mn[p], x[i][p]), mx[p] = act_max2<BF16>(mx[p], x[i][p]);
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      mn[p] = act_min2<BF16>(mn[p], __shfl_xor_sync(0xffffffffu, mn[p], o));
      mx[p] = act_max2<BF16>(mx[p], __shfl_xor_sync(0xffffffffu, mx[p], o));
    }
  }
  // the values wait in this thread's column of the scratch (conflict-free
  // 16-byte accesses) for the compact per-g loop below
#pragma unroll
  for (int i = 0; i < 8; ++i) scratch[i][tid] = make_uint4(x[i][0], x[i][1], x[i][2], x[i][3]);
  // lane tq computes the stored scale and zero of channels k = 2 tq, 2 tq + 1
  const uint32_t mnw = (tq & 2) ? ((tq & 1) ? mn[3] : mn[2]) : ((tq & 1) ? mn[1] : mn[0]);
  const uint32_t mxw = (tq & 2) ? ((tq & 1) ? mx[3] : mx[2]) : ((tq & 1) ? mx[1] : mx[0]);
  __half* km = reinterpret_cast<__half*>(chunk + G.chunk.kmeta_off);
  uint32_t zs[2];
  float rr[2];
  bool ok = true;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    __half sh, zh;
    slice_params<LB>(act_half<BF16>(mnw, h), act_half<BF16>(mxw, h), &sh, &zh, &zs[h], &rr[h], &ok);
    const int k = 2 * tq + h;
    const int c = k < 4 ? 4 * cq + k : HALF + 4 * cq + k - 4;
    km[PR ? c : kmeta_pos(D, c)] = sh;  // keys stored before RoPE: the natural order
    km[D + (PR ? c : kzero_pos(D, c))] = zh;
    zsk[c] = zs[h];
  }
  __syncwarp();
  Slice2 q[4];  // channels (2p, 2p + 1), from lane p of the quad
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int src = (lane & ~3) | p;
    q[p] = pair_slices(make_slice(__shfl_sync(0xffffffffu, zs[0], src), __shfl_sync(0xffffffffu, rr[0], src)),
                       make_slice(__shfl_sync(0xffffffffu, zs[1], src), __shfl_sync(0xffffffffu, rr[1], src)));
  }
  // a slice whose codes could leave [0, LB] sends the quad's words down the exact path
  const bool clamp = ((__ballot_sync(0xffffffffu, !ok) >> (lane & ~3)) & 0xfu) != 0;

  uint8_t* kc = chunk + G.chunk.kc_off;
  const int tA = cq / (D / 16), s = cq % (D / 16);        // plain order: quad cq = lane t, k-step s
  const int tP = cq / (D / 32), s0 = 2 * (cq % (D / 32));  // stored before RoPE
#pragma unroll 1
  for (int gl = 0; gl < 4; ++gl) {
    const int g = gb + gl;
    const uint4 u0 = scratch[2 * gl][tid], u1 = scratch[2 * gl + 1][tid];
    const uint32_t xg[2][4] = {{u0.x, u0.y, u0.z, u0.w}, {u1.x, u1.y, u1.z, u1.w}};
    uint32_t acc[M::NQ], corr[M::NQ];
#pragma unroll
    for (int j = 0; j < M::NQ; ++j) acc[j] = 0u, corr[j] = 0u;
#pragma unroll
    for (int ts = 0; ts < 2; ++ts) {
#pragma unroll
      for (int p = 0; p < 4; ++p) {  // channels 2p, 2p + 1: the two halves of one word
        const int j0 = M::acc(ts, 2 * p), j1 = M::acc(ts, 2 * p + 1);
        add_code2(make_float2(act_lo<BF16>(xg[ts][p]), act_hi<BF16>(xg[ts][p])), q[p], M::bit(ts, 2 * p),
                  M::bit(ts, 2 * p + 1), acc[j0], corr[j0], acc[j1], corr[j1]);
      }
    }
#pragma unroll
    for (int j = 0; j < M::NQ; ++j) acc[j] -= corr[j];
    if (clamp) {  // a slice that needs the clamp: the exact path
      const int r0 = 16 * mt + g, r1 = r0 + 8;
      const int64_t q0 = p0 + (sub ? sub[r0] : r0), q1 = p0 + (sub ? sub[r1] : r1);
      const float* t0 = rope && q0 >= a.L0 ? rope + static_cast<size_t>(q0) * D : nullptr;
      const float* t1 = rope && q1 >= a.L0 ? rope + static_cast<size_t>(q1) * D : nullptr;
      const uint4 e = k_exact_g<D, KB, BF16, PR>(group_row(a, a.lay.tail_k, a.k, bh, q0),
                                                  group_row(a, a.lay.tail_k, a.k, bh, q1), t0, t1, cq, zsk);
      const uint32_t ev[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
      for (int j = 0; j < M::NQ; ++j) acc[j] = ev[j];
    }
    const int ms_plain = mt * S + s, ms_pr = mt * S + s0;
    if constexpr (!PR) {
      if constexpr (KB == 4) {
#pragma unroll
        for (int j = 0; j < 2; ++j) store_word(kc, 4 * g + tA + 2 * j, ms_plain, PW, acc[j]);
      } else if constexpr (KB == 8) {
#pragma unroll
        for (int j = 0; j < 4; ++j) store_word(kc, 4 * g + tA + 2 * (j >> 1), 2 * ms_plain + (j & 1), PW, acc[j]);
      } else if constexpr (KB == 2) {  // quads cq, cq ^ 1 share a word: k-steps s, s ^ 1
        uint32_t w[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          w[j] = acc[j] << (2 * (s & 1));
          w[j] |= __shfl_xor_sync(0xffffffffu, w[j], 4);
        }
        const int j = s & 1;  // the even quad stores the low quads' word, the odd one the high quads'
        store_word(kc, 4 * g + tA + 2 * j, ms_plain >> 1, PW, j ? w[1] : w[0]);
      } else {  // 3-bit: quads of k-steps s % 4 = 0 .. 3 share a block; the fourth lane's quads go to the others
        const int sig = s & 3, l3 = lane | 12;
#pragma unroll
        for (int qd = 0; qd < 2; ++qd) {
          const uint32_t qa = acc[2 * qd], qb = acc[2 * qd + 1];
          const uint32_t xx = __shfl_sync(0xffffffffu, qa, l3), yy = __shfl_sync(0xffffffffu, qb, l3);
          if (sig < 3)
            store_word(kc, 4 * g + tA + 2 * qd, 3 * (ms_plain >> 2) + sig, PW, block3_word(sig, qa, qb, xx, yy));
        }
      }
    } else {
      if constexpr (KB == 4) {
#pragma unroll
        for (int j = 0; j < 2; ++j) store_word(kc, 4 * g + tP, ms_pr + j, PW, acc[j]);
      } else if constexpr (KB == 8) {
#pragma unroll
        for (int j = 0; j < 4; ++j) store_word(kc, 4 * g + tP, 2 * (ms_pr + (j >> 1)) + (j & 1), PW, acc[j]);
      } else if constexpr (KB == 2) {
        store_word(kc, 4 * g + tP, ms_pr >> 1, PW, acc[0]);
      } else {  // 3-bit: an even quad holds quads 0..3 of the block, the odd one 4..7
        const uint32_t xx = __shfl_xor_sync(0xffffffffu, acc[2], 4), yy = __shfl_xor_sync(0xffffffffu, acc[3], 4);
        const int blk = 3 * (ms_pr >> 2);
        if ((cq & 1) == 0) {
          store_word(kc, 4 * g + tP, blk, PW, block3_word(0, acc[0], acc[1], xx, yy));
          store_word(kc, 4 * g + tP, blk + 1, PW, block3_word(1, acc[2], acc[3], xx, yy));
        } else {
          store_word(kc, 4 * g + tP, blk + 2, PW, block3_word(2, acc[0], acc[1], acc[2], acc[3]));
        }
      }
    }
  }
}

// ---------------------------------------------------------------- V
// Element (i, h) of one g of a V thread (token i: e = i & 1, hh = i >> 1;
// channel g + 8 h of the thread's m block) -> accumulator, bit.
template <int BITS>
struct VMap {
  static constexpr int NQ = (BITS == 8 || BITS == 3) ? 2 : 1;
  __host__ __device__ static constexpr int acc(int i, int h) {
    (void)h;
    return (BITS == 8 || BITS == 3) ? (i >> 1) : 0;
  }
  __host__ __device__ static constexpr int bit(int i, int h) {
    if (BITS == 4) return 16 * h + 4 * (i >> 1) + 8 * (i & 1);
    if (BITS == 8) return 8 * h + 16 * (i & 1);
    if (BITS == 2) return 8 * (h + 2 * (i >> 1)) + 4 * (i & 1);
    return 8 * (2 * h + (i & 1));
  }
};

// The exact path for one g of a V thread (channels 16 m + g, +8 of the four
// token rows, zs the tokens' stored zero | scale).
template <int VB, bool BF16>
__device__ __noinline__ uint2 v_exact_g(const uint16_t* row0, const uint16_t* row1, const uint16_t* row2,
                                        const uint16_t* row3, uint4 zs) {
  using M = VMap<VB>;
  constexpr int LB = (1 << VB) - 1;
  const uint16_t* rows[4] = {row0, row1, row2, row3};
  const uint32_t z4[4] = {zs.x, zs.y, zs.z, zs.w};
  uint32_t acc[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float xv = act_to_float(rows[i][8 * h], BF16);
      acc[M::acc(i, h)] |= exact_code(xv, z4[i], LB) << M::bit(i, h);
    }
  }
  return make_uint2(acc[0], acc[1]);
}

// lin: as for flush_k, the group's first V row or null.
template <int D, int VB, bool BF16>
__device__ __forceinline__ void flush_v(const AppendArgs& a, const int* sub, int64_t p0, int bh, uint8_t* chunk,
                                        uint4 (*scratch)[D], const uint16_t* lin) {
  using M = VMap<VB>;
  constexpr int LB = (1 << VB) - 1, NV = D / 32;
  constexpr int PW = piece_words(D * VB / 32);
  const Geometry& G = a.geo;
  const int tid = threadIdx.x, lane = tid & 31, vt = tid - D / 2;
  const int m = vt % (D / 16), kb = (vt / (D / 16)) & 1, t = vt / (D / 8);
  const bool odd = m & 1;
  const uint16_t* rows[4];
  uint32_t x[4][8];
  auto load_rows = [&](auto row_of) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 16 * kb + 2 * t + (i & 1) + 8 * (i >> 1);
      rows[i] = row_of(r) + 16 * m;
      const uint4 u0 = __ldg(reinterpret_cast<const uint4*>(rows[i]));
      const uint4 u1 = __ldg(reinterpret_cast<const uint4*>(rows[i] + 8));
      x[i][0] = u0.x, x[i][1] = u0.y, x[i][2] = u0.z, x[i][3] = u0.w;
      x[i][4] = u1.x, x[i][5] = u1.y, x[i][6] = u1.z, x[i][7] = u1.w;
    }
  };
  if (lin) load_rows([&](int r) { return lin + r * D; });
  else load_rows([&](int r) { return group_row(a, a.lay.tail_v, a.v, bh, p0 + (sub ? sub[r] : r)); });
  // slot 2 g2 + hh of this thread's scratch column: the channel pairs
  // (2 g2, +1) and (2 g2 + 8, +9) of tokens 2 hh, 2 hh + 1, what the g = 2 g2,
  // 2 g2 + 1 steps of the compact loop below read
#pragma unroll
  for (int g2 = 0; g2 < 4; ++g2) {
    scratch[2 * g2][tid] = make_uint4(x[0][g2], x[0][g2 + 4], x[1][g2], x[1][g2 + 4]);
    scratch[2 * g2 + 1][tid] = make_uint4(x[2][g2], x[2][g2 + 4], x[3][g2], x[3][g2 + 4]);
  }
  __half* vm = reinterpret_cast<__half*>(chunk + G.chunk.vmeta_off);
  uint8_t* vc = chunk + G.chunk.vc_off;
  const int vg = m >> 1, mk = 2 * m + kb;
  const bool q40 = VB == 4 && G.v_q4_0;
  Slice q[4];
  Slice2 q2[2];  // tokens (0, 1) and (2, 3)
  uint32_t zsv[4] = {0u, 0u, 0u, 0u};
  float qd[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  bool clamp = false;
  if (q40) {
    // the value of largest magnitude, the first in channel order on ties
    // (the even m holds the lower 16 channels of the group)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float am = -1.0f, mv = 0.0f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float xv = act_half<BF16>(x[i][c >> 1], c & 1);
        if (fabsf(xv) > am) am = fabsf(xv), mv = xv;
      }
      const float am2 = __shfl_xor_sync(0xffffffffu, am, 1), mv2 = __shfl_xor_sync(0xffffffffu, mv, 1);
      if (odd ? am2 >= am : am2 > am) mv = mv2;
      const __half sh = __float2half_rn(__fmul_rn(mv, -0.125f));  // = RN(mv / -8): a power of two
      qd[i] = __half2float(sh);
      q[i].r = __frcp_rn(qd[i]);
      if ((i >> 1) == static_cast<int>(odd)) {  // each of the pair writes two tokens' meta
        const int r = 16 * kb + 2 * t + (i & 1) + 8 * (i >> 1);
        vm[vscale_pos(NV, r, vg)] = sh;
        vm[vzero_pos(NV, r, vg)] = __float2half_rn(__fmul_rn(qd[i], -8.0f));  // exact: a power-of-two multiple
      }
    }
  } else {
    float mnf[4], mxf[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo = x[i][0], hi = x[i][0];
#pragma unroll
      for (int w = 1; w < 8; ++w) lo = act_min2<BF16>(lo, x[i][w]), hi = act_max2<BF16>(hi, x[i][w]);
      lo = act_min2<BF16>(lo, __shfl_xor_sync(0xffffffffu, lo, 1));
      hi = act_max2<BF16>(hi, __shfl_xor_sync(0xffffffffu, hi, 1));
      mnf[i] = fminf(act_lo<BF16>(lo), act_hi<BF16>(lo));
      mxf[i] = fmaxf(act_lo<BF16>(hi), act_hi<BF16>(hi));
    }
    // the even m computes tokens i = 0, 1, the odd one i = 2, 3
    uint32_t zs[2];
    float rr[2];
    bool ok = true;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      __half sh, zh;
      slice_params<LB>(odd ? mnf[2 + e] : mnf[e], odd ? mxf[2 + e] : mxf[e], &sh, &zh, &zs[e], &rr[e], &ok);
      const int r = 16 * kb + 2 * t + e + 8 * static_cast<int>(odd);
      vm[vscale_pos(NV, r, vg)] = sh;
      vm[vzero_pos(NV, r, vg)] = zh;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t zo = __shfl_xor_sync(0xffffffffu, zs[e], 1);
      const float ro = __shfl_xor_sync(0xffffffffu, rr[e], 1);
      zsv[e] = odd ? zo : zs[e];
      zsv[2 + e] = odd ? zs[e] : zo;
      q[e] = make_slice(zsv[e], odd ? ro : rr[e]);
      q[2 + e] = make_slice(zsv[2 + e], odd ? rr[e] : ro);
    }
    q2[0] = pair_slices(q[0], q[1]);
    q2[1] = pair_slices(q[2], q[3]);
    // a slice whose codes could leave [0, LB] sends the pair's words down the exact path
    clamp = __shfl_xor_sync(0xffffffffu, static_cast<int>(!ok), 1) != 0 || !ok;
  }

#pragma unroll 1
  for (int g2 = 0; g2 < 4; ++g2) {
    const uint4 u0 = scratch[2 * g2][tid], u1 = scratch[2 * g2 + 1][tid];
    const uint32_t xg[4][2] = {{u0.x, u0.y}, {u0.z, u0.w}, {u1.x, u1.y}, {u1.z, u1.w}};
#pragma unroll
  for (int gg = 0; gg < 2; ++gg) {
    const int g = 2 * g2 + gg;
    uint32_t acc[M::NQ], corr[M::NQ];
#pragma unroll
    for (int j = 0; j < M::NQ; ++j) acc[j] = 0u, corr[j] = 0u;
    if (VB == 4 && q40) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          acc[M::acc(i, h)] |= q40_fast(act_half<BF16>(xg[i][h], gg), qd[i], q[i].r) << M::bit(i, h);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; i += 2) {  // tokens i, i + 1: two slices
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j0 = M::acc(i, h), j1 = M::acc(i + 1, h);
          add_code2(make_float2(act_half<BF16>(xg[i][h], gg), act_half<BF16>(xg[i + 1][h], gg)), q2[i >> 1],
                    M::bit(i, h), M::bit(i + 1, h), acc[j0], corr[j0], acc[j1], corr[j1]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < M::NQ; ++j) acc[j] -= corr[j];
    if (clamp) {  // a slice that needs the clamp: the exact path
      const uint2 e = v_exact_g<VB, BF16>(rows[0] + g, rows[1] + g, rows[2] + g, rows[3] + g,
                                          make_uint4(zsv[0], zsv[1], zsv[2], zsv[3]));
      acc[0] = e.x;
      if (M::NQ > 1) acc[M::NQ - 1] = e.y;
    }
    const int ln = 4 * g + t;
    if constexpr (VB == 4) {
      store_word(vc, ln, mk, PW, acc[0]);
    } else if constexpr (VB == 8) {
      store_word(vc, ln, 2 * mk, PW, acc[0]);
      store_word(vc, ln, 2 * mk + 1, PW, acc[1]);
    } else if constexpr (VB == 2) {  // kb 0 and 1 share a word
      uint32_t w = acc[0] << (2 * kb);
      w |= __shfl_xor_sync(0xffffffffu, w, D / 16);
      if ((g & 1) == kb) store_word(vc, ln, m, PW, w);
    } else {  // 3-bit: (m & 1, kb) = quad pair sigma of the block of the m pair
      const int sig = 2 * (m & 1) + kb, l3 = lane | 1 | (D / 16);
      const uint32_t xx = __shfl_sync(0xffffffffu, acc[0], l3), yy = __shfl_sync(0xffffffffu, acc[1], l3);
      if (sig < 3) store_word(vc, ln, 3 * (m >> 1) + sig, PW, block3_word(sig, acc[0], acc[1], xx, yy));
    }
  }
  }
}

template <int D, int KB, int VB, bool BF16>
__device__ __forceinline__ void flush_group(const AppendArgs& a, const int* sub, int64_t p0, int bh, uint8_t* chunk,
                                            uint32_t* zsk, uint4 (*scratch)[D]) {
  // the common prefill case: the group's 32 rows are consecutive appended rows
  const size_t lin_off = (!sub && p0 >= a.L0) ? (static_cast<size_t>(bh) * a.n + (p0 - a.L0)) * D : ~size_t{0};
  if (threadIdx.x < D / 2) {
    const uint16_t* lin = lin_off != ~size_t{0} ? a.k + lin_off : nullptr;
    if (a.geo.k_pre_rope) flush_k<D, KB, BF16, true>(a, sub, p0, bh, chunk, zsk, scratch, lin);
    else flush_k<D, KB, BF16, false>(a, sub, p0, bh, chunk, zsk, scratch, lin);
  } else {
    const uint16_t* lin = lin_off != ~size_t{0} ? a.v + lin_off : nullptr;
    flush_v<D, VB, BF16>(a, sub, p0, bh, chunk, scratch, lin);
  }
}

template <int D, int KB, int VB>
__global__ void __launch_bounds__(D, 768 / D) kivi_flush_kernel(AppendArgs a) {
  __shared__ int sub_rows[32];
  __shared__ uint32_t zsk[D];  // K: stored zero | scale << 16 per channel, for the exact path
  __shared__ uint4 scratch[8][D];  // each thread's 64 values, one column per thread
  const Geometry& G = a.geo;
  const int tid = threadIdx.x;
  const int bh = blockIdx.y, b = bh / G.H, h = bh % G.H;
  const int64_t g = a.g_first + blockIdx.x;
  const int64_t p0 = g * kGroup;
  const int slot = static_cast<int>(g % G.n_slots);
  uint32_t smask = 0;
  const int* sub = nullptr;
  if (a.dyn_active) {  // KVSink: the nearest non-sink row of each row (ties to the earlier)
    if (tid < 32) {
      uint32_t msk = 0;
      for (int j = 0; j < a.n_dyn_sel; ++j) {
        const int64_t p = a.lay.sink_pos[b * kMaxSinks + j];
        if (p >= p0 && p < p0 + kGroup) msk |= 1u << (p - p0);
      }
      const int r = tid;
      int sr = r;
      if (((msk >> r) & 1u) && msk != 0xFFFFFFFFu) {
        for (int d = 1; d < 32; ++d) {
          if (r - d >= 0 && !((msk >> (r - d)) & 1u)) { sr = r - d; break; }
          if (r + d < 32 && !((msk >> (r + d)) & 1u)) { sr = r + d; break; }
        }
      }
      sub_rows[r] = sr;
      smask = msk;
    }
    __syncthreads();
    sub = sub_rows;
  }
  uint8_t* chunk = a.lay.chunks + (static_cast<size_t>(bh) * G.n_slots + slot) * G.chunk.bytes;
  if (G.act_bf16) flush_group<D, KB, VB, true>(a, sub, p0, bh, chunk, zsk, scratch);
  else flush_group<D, KB, VB, false>(a, sub, p0, bh, chunk, zsk, scratch);
  if (G.n_dyn && h == 0 && tid == 0) a.lay.sink_mask[b * G.n_slots + slot] = smask;
}

// Launch for the K code width KB (V width from the geometry).
template <int D, int KB>
void launch_flush_kb(const AppendArgs& a, dim3 grid, cudaStream_t s) {
  switch (a.geo.vb) {
    case 2: kivi_flush_kernel<D, KB, 2><<<grid, D, 0, s>>>(a); break;
    case 3: kivi_flush_kernel<D, KB, 3><<<grid, D, 0, s>>>(a); break;
    case 4: kivi_flush_kernel<D, KB, 4><<<grid, D, 0, s>>>(a); break;
    default: kivi_flush_kernel<D, KB, 8><<<grid, D, 0, s>>>(a); break;
  }
}

}  // namespace
}  // namespace kvq
