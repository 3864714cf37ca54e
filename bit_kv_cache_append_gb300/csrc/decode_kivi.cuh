// Split-KV decode attention over the KIVI and TurboQuant caches (internal
// template; the instantiations live in decode_d{64,128}_{k2,k3,k4,k8,tq}.cu).
//
// Work decomposition (stream-K): the quantised segment of every (sequence,
// KV head) unit is a run of 32-token groups; all units' groups form one flat
// list cut into n_ctas equal contiguous ranges, one per persistent CTA
// (n_ctas = SM count x resident CTAs). A CTA walks its range unit by unit;
// for each unit it touches, its NP warp pairs (4, two CTAs per SM; in
// TurboQuant mode 8, one CTA per SM) take the unit's groups in runs of two
// consecutive groups (runs p, p+NP, ...; one group per run for TurboQuant
// and where a chunk exceeds 6 KB) and the CTA merges the pairs into one partial (max,
// sum, unnormalised output) per query head. The exact pools (sinks and tail)
// are left to the merge kernel, which combines them with every partial of a
// (sequence, query head).
//
// Warp specialisation: a pair is a QK warp and a PV warp working on the same
// group stream. The QK warp turns the K codes into scores and softmax
// weights and hands the weights (and the rescale factor of the running max)
// to the PV warp through a double-buffered shared-memory slot; the PV warp
// turns the V codes into the weighted sum and, being the last reader of each
// staged run, refills the stage with the next run (one 1-D bulk copy when
// its chunks are adjacent in the ring); three stages per pair where they
// leave room for the CTAs per SM, else two. Each role keeps only its own
// operands in registers, so more warps fit per SM and the two halves of a
// group's dependency chain overlap across groups.
//
// Per group, on the tensor cores (mma.sync m16n8k16, f16 in, f32 out):
//   scores^T [32 tokens x 8 cols] = zeros-row . q + codes_K [32 x D] . qt
//   out^T    [D x 8]             += codes_V^T [D x 32] . pt [32 x 8]
// with the KIVI scales folded into the small operand
//   qt[c][j]  = q_j[c] * sK[c]            (K scale per channel of the group)
//   pt[t][j]  = p_j[t] * sV[t][c / 32]    (V scale per token and 32 channels;
//                                          one pt per V channel group)
// and the zero points: the K zeros enter as a row of the MMA (sum_c zK[c]
// q_j[c]), the V zeros as fp32 sums sum_t p_j[t] zV[t][c/32].
// The codes enter the MMA exactly, as code * unit in f16 with a power-of-two
// unit undone on the fp32 sums (code_pair). In the score MMA the 8 columns
// hold, for query head j, column 2j = the f16 value of q * sK and column
// 2j+1 its f16 residual, formed exactly by an FMA (x * s - f16(x * s) has no
// rounding), so the product is carried at about 22 bits: a score error is
// amplified by the exponential. In the value MMA the weight p of a token is
// one f16 value in the even columns (the odd ones are zero) and p * sV one f16
// product, made on the transposed weights: the errors of the weights average
// over tokens. Thread (g, t) of a C fragment owns query head t.
//
// Every wait is bounded; a wait that gives up raises the CTA's abort flag so
// that every other wait of the CTA gives up at once.
#pragma once

#include <type_traits>

#include "decode_common.cuh"

namespace kvq {

constexpr uint32_t h2pow2(int e) {
  return (static_cast<uint32_t>(15 + e) << 10) | (static_cast<uint32_t>(15 + e) << 26);
}
constexpr uint32_t h2negpow2(int e) {
  return (0x8000u | (static_cast<uint32_t>(15 + e) << 10)) |
         ((0x8000u | (static_cast<uint32_t>(15 + e) << 10)) << 16);
}

__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}


__device__ __forceinline__ __half2 as_h2(uint32_t x) { return *reinterpret_cast<__half2*>(&x); }
__device__ __forceinline__ uint32_t as_u32(__half2 x) { return *reinterpret_cast<uint32_t*>(&x); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Packed codes become exact f16 operands by the hardware's narrow-float
// conversions, with the code bits laid out (kvq_layout.h) so that one mask
// exposes them in the right format:
//   2-bit: a code in the low two bits of an e2m1 nibble is the value code/2
//          (subnormal 0.5, then 1.0, 1.5), a byte gives an f16x2;
//   4-bit: a code in the low nibble of an e4m3 byte is code * 2^-9 (the
//          subnormal and first normal binade are evenly spaced), two bytes
//          give an f16x2;
//   8-bit: the code is OR-ed into the mantissa of 1024.0 and 1024 is
//          subtracted.
// kCodeInv is the factor that turns sums over these values back into sums
// over codes (a power of two, so the rescale is exact).
template <int BITS>
struct CodeConsts {
  static constexpr float kCodeInv = BITS == 2 ? 2.0f : (BITS == 3 ? 8.0f : (BITS == 4 ? 512.0f : 1.0f));
  uint32_t magic;
  __device__ __forceinline__ void load(const DecodeArgs& a) {
    if (BITS == 8) magic = pin(a.h2_magic);
  }
};

template <int BYTE>
__device__ __forceinline__ uint32_t cvt_e2m1x2(uint32_t m) {
  uint32_t d;
  if (BYTE == 0) asm("{.reg .b8 a, b, c, e; mov.b32 {a, b, c, e}, %1; cvt.rn.f16x2.e2m1x2 %0, a;}" : "=r"(d) : "r"(m));
  if (BYTE == 1) asm("{.reg .b8 a, b, c, e; mov.b32 {a, b, c, e}, %1; cvt.rn.f16x2.e2m1x2 %0, b;}" : "=r"(d) : "r"(m));
  if (BYTE == 2) asm("{.reg .b8 a, b, c, e; mov.b32 {a, b, c, e}, %1; cvt.rn.f16x2.e2m1x2 %0, c;}" : "=r"(d) : "r"(m));
  if (BYTE == 3) asm("{.reg .b8 a, b, c, e; mov.b32 {a, b, c, e}, %1; cvt.rn.f16x2.e2m1x2 %0, e;}" : "=r"(d) : "r"(m));
  return d;
}

template <int HALF>
__device__ __forceinline__ uint32_t cvt_e4m3x2(uint32_t m) {
  uint32_t d;
  if (HALF == 0) asm("{.reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e4m3x2 %0, l;}" : "=r"(d) : "r"(m));
  if (HALF == 1) asm("{.reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e4m3x2 %0, h;}" : "=r"(d) : "r"(m));
  return d;
}

template <int HALF>
__device__ __forceinline__ uint32_t cvt_e2m3x2(uint32_t m) {
  uint32_t d;
  if (HALF == 0) asm("{.reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e2m3x2 %0, l;}" : "=r"(d) : "r"(m));
  if (HALF == 1) asm("{.reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e2m3x2 %0, h;}" : "=r"(d) : "r"(m));
  return d;
}

// Pair j (0 .. 15) of a 3-bit block of three words w (kvq_layout.h
// frag3_put) as an exact f16x2 of code / 8: quad j / 2 holds four codes, one
// in the low three bits of each byte, which as e2m3 (exponent field 0) are
// the evenly spaced values code / 8.
__device__ __forceinline__ uint32_t code_pair3(const uint32_t* w, int j) {
  const int q = j >> 1;
  uint32_t m;
  if (q < 6) m = (w[q >> 1] >> (3 * (q & 1))) & 0x07070707u;
  else m = ((w[q - 6] >> 6) & 0x03030303u) | ((w[2] >> (4 + (q - 6))) & 0x04040404u);
  return (j & 1) ? cvt_e2m3x2<1>(m) : cvt_e2m3x2<0>(m);
}

// Pair j of a packed word (the lane's fragment elements 2P, 2P + 1 where
// P = word * pairs-per-word + j) as an exact f16x2 of code * unit. j is a
// constant after unrolling, so the selections below fold away.
template <int BITS>
__device__ __forceinline__ uint32_t code_pair(const CodeConsts<BITS>& k, uint32_t w, int j) {
  if (BITS == 2) {
    const uint32_t m = (j < 4 ? w : (w >> 2)) & 0x33333333u;
    switch (j & 3) {
      case 0: return cvt_e2m1x2<0>(m);
      case 1: return cvt_e2m1x2<1>(m);
      case 2: return cvt_e2m1x2<2>(m);
      default: return cvt_e2m1x2<3>(m);
    }
  } else if (BITS == 4) {
    const uint32_t m = (j < 2 ? w : (w >> 4)) & 0x0F0F0F0Fu;
    return (j & 1) ? cvt_e4m3x2<1>(m) : cvt_e4m3x2<0>(m);
  } else {
    const uint32_t hv = __byte_perm(w, k.magic, static_cast<uint32_t>(j | 0x50 | ((j + 2) << 8) | 0x7000));
    return as_u32(__hsub2(as_h2(hv), as_h2(k.magic)));
  }
}

// Pair P (fragment elements 2P, 2P + 1) of a lane's code words w (from the
// start of the lane's block) as an exact f16x2 of code * unit.
template <int BITS>
__device__ __forceinline__ uint32_t pair_at(const CodeConsts<BITS>& k, const uint32_t* w, int P) {
  if constexpr (BITS == 3) {
    return code_pair3(w + 3 * (P >> 4), P & 15);
  } else {
    constexpr int PPW = 16 / BITS;
    return code_pair<BITS>(k, w[P / PPW], P % PPW);
  }
}

#ifndef KVQ_LAZY_RESCALE
#define KVQ_LAZY_RESCALE 8.0f
#endif
// Headroom (log2 units) the running softmax max may lag behind the scores.
constexpr float kLazyRescale = KVQ_LAZY_RESCALE;

// CTA shape: KVQ_DECODE_PAIRS warp pairs per CTA, at least
// KVQ_DECODE_MIN_CTAS CTAs resident per SM (the register budget follows).
#ifndef KVQ_DECODE_PAIRS
#define KVQ_DECODE_PAIRS 4
#endif
#ifndef KVQ_DECODE_MIN_CTAS
#define KVQ_DECODE_MIN_CTAS (8 / KVQ_DECODE_PAIRS)
#endif
// TurboQuant: one CTA per SM of KVQ_TQ_PAIRS warp pairs, so that one copy of
// the 64 KB byte tables serves sixteen warps.
#ifndef KVQ_TQ_PAIRS
#define KVQ_TQ_PAIRS 8
#endif

template <int D, int KB, int VB, bool TQ = false, bool PR = false>
struct KiviTile {
  // chunk layout (kvq_layout.h): KIVI codes and meta, or TurboQuant K codes
  // in fragment order and V codes in token-pair rows, one f32 norm per token
  static constexpr int KC = 32 * D * KB / 8;
  static constexpr int KMETA = KC;
  static constexpr int VC = KMETA + (TQ ? 4 * 32 : 4 * D);
  static constexpr int VMETA = VC + 32 * D * VB / 8;
  static constexpr int CHUNK = VMETA + (TQ ? 4 * 32 : 4 * D);
  static constexpr int NP = TQ ? KVQ_TQ_PAIRS : KVQ_DECODE_PAIRS;  // warp pairs per CTA
  static constexpr int MIN_CTAS = TQ ? 8 / KVQ_TQ_PAIRS : KVQ_DECODE_MIN_CTAS;
  // groups per stage: a pair takes runs of GPB consecutive groups, so the
  // waits, hand-off and rescale decision are paid once per run (KIVI chunks
  // up to 6 KB); one for TurboQuant, whose tables leave less shared memory,
  // and for larger chunks
  static constexpr int GPB = (TQ || PR || CHUNK > 6144) ? 1 : 2;
  static constexpr int STAGE = GPB * CHUNK;
  static constexpr int PBUF = GPB * 32 * 8 + 16;         // weights (4 f16, 8 B per lane per group) + 4 rescale factors
  static constexpr int RED_FLOATS = NP * kMaxGqa * (D + 2);  // one merged state per pair
  // TurboQuant codebook tables: a field (two codes, low | high << bits) ->
  // f16x2 of their values 2 c[code] - 1, in NLUT = 32 interleaved copies,
  // lane l reading copy l (its own bank). 4-bit K codes are read by the
  // byte that holds their field: 256 blocks of 256 B, entry e of copy cp
  // at 256 e + 4 cp, so the address is the byte in bits 8..15 and the copy
  // offset in bits 0..7, one byte permute. Every other field (V, and K of 2
  // and 3 bits) is shifted to its scaled offset in a table of 2^(2 bits)
  // entries, entry e of copy cp at 4 (e NLUT + cp). (Byte lookups of the V
  // fields, 64 bits wide for 2-bit pairs, were measured slower.)
  static constexpr bool KBYTE = TQ && KB == 4;
  static constexpr int NLUT = 32;
  static constexpr int shift_lut_bytes(int bits) { return TQ ? (1 << (2 * bits)) * NLUT * 4 : 0; }
  static constexpr int LUTK = KBYTE ? 256 * 256 : shift_lut_bytes(KB), LUTV = shift_lut_bytes(VB);
  static constexpr int smem_for(int nst) {
    return NP * nst * STAGE + NP * 2 * PBUF + (D / 16) * 32 * 16 + (TQ ? kMaxGqa * D * 4 : 0) + LUTK + LUTV +
           RED_FLOATS * 4 + NP * (nst + 4) * 8 + 16;
  }
  // what one of MIN_CTAS CTAs may take of an SM's 228 KB (1 KB of each
  // CTA's share is reserved by the hardware)
  static constexpr int kCtaSmem = 228 * 1024 / MIN_CTAS - 1024;
  // bulk-copy stages per pair: three where they leave room for MIN_CTAS CTAs
  // per SM (runs of two groups up to 4 KB each; single groups), else two
#ifndef KVQ_DECODE_STAGES
  static constexpr int NST = smem_for(3) <= kCtaSmem ? 3 : 2;
#else
  static constexpr int NST = KVQ_DECODE_STAGES;
#endif
  // shared memory: stages | weight buffers | query operand | query scratch |
  // tables | red | barriers | abort flag
  static constexpr int OFF_PBUF = NP * NST * STAGE;
  static constexpr int OFF_Q = OFF_PBUF + NP * 2 * PBUF;  // [D/16 k-steps][32 lanes] x 16 B
  static constexpr int OFF_QF = OFF_Q + (D / 16) * 32 * 16;  // TurboQuant: rotated queries [kMaxGqa][D] f32
  static constexpr int OFF_LUTK = OFF_QF + (TQ ? kMaxGqa * D * 4 : 0);
  static constexpr int OFF_LUTV = OFF_LUTK + LUTK;
  static constexpr int OFF_RED = OFF_LUTV + LUTV;
  static constexpr int OFF_BAR = OFF_RED + RED_FLOATS * 4;
  static constexpr int NBAR = NP * (NST + 4);             // full[NST], pfull[2], pempty[2]
  static constexpr int OFF_ABORT = OFF_BAR + NBAR * 8;
  static constexpr size_t smem_bytes() { return OFF_ABORT + 16; }
  static_assert(smem_bytes() == static_cast<size_t>(smem_for(NST)), "layout and its size agree");
  static_assert(OFF_LUTK % 16 == 0, "tables 16-byte aligned");
  static_assert(OFF_BAR % 8 == 0, "mbarriers are 8-byte aligned");
  static_assert(!TQ || smem_bytes() <= static_cast<size_t>(kCtaSmem), "MIN_CTAS CTAs per SM");
};

// CTA that owns flattened item i under the equal split of `work` items into
// `n` ranges [floor(c work / n), floor((c+1) work / n)).
__device__ __forceinline__ int owner_cta(int64_t i, int64_t work, int n) {
  return static_cast<int>(((i + 1) * n - 1) / work);
}

// The W words of this lane's block of a code region whose lane blocks are
// interleaved in pieces of PW words (kvq_layout.h code_word_offset).
template <int W, int PW>
__device__ __forceinline__ void load_lane_words(const uint8_t* region, int lane, uint32_t* w) {
#pragma unroll
  for (int pc = 0; pc < W / PW; ++pc) {
    if constexpr (PW == 4) {
      const uint4 v = reinterpret_cast<const uint4*>(region)[pc * 32 + lane];
      w[4 * pc] = v.x, w[4 * pc + 1] = v.y, w[4 * pc + 2] = v.z, w[4 * pc + 3] = v.w;
    } else {
      const uint2 v = reinterpret_cast<const uint2*>(region)[pc * 32 + lane];
      w[2 * pc] = v.x, w[2 * pc + 1] = v.y;
    }
  }
}

// Words [first, first + N) of this lane's block (first a constant after
// unrolling), lane blocks interleaved in pieces of PW words.
template <int N, int PW>
__device__ __forceinline__ void load_lane_range(const uint8_t* region, int lane, int first, uint32_t* out) {
  const int p0 = first / PW, p1 = (first + N - 1) / PW;
#pragma unroll
  for (int pc = p0; pc <= p1; ++pc) {
    uint32_t tmp[PW];
    if constexpr (PW == 4) {
      const uint4 v = reinterpret_cast<const uint4*>(region)[pc * 32 + lane];
      tmp[0] = v.x, tmp[1] = v.y, tmp[2] = v.z, tmp[3] = v.w;
    } else {
      const uint2 v = reinterpret_cast<const uint2*>(region)[pc * 32 + lane];
      tmp[0] = v.x, tmp[1] = v.y;
    }
#pragma unroll
    for (int k = 0; k < PW; ++k) {
      const int w = pc * PW + k;
      if (w >= first && w < first + N) out[w - first] = tmp[k];
    }
  }
}

// The table entry of the field of 2 BITS bits at bit `bit` of a lane's bit
// string: entry e of copy cp sits at byte (e NLUT + cp) 4 of the table, so
// the field is taken out already scaled to e NLUT 4 (one shift, or a funnel
// shift where it straddles two words) and joined with cp4 = 4 cp by the
// mask's own instruction; the table's shared-memory base folds into the
// load's immediate.
template <int BITS, int NLUT>
__device__ __forceinline__ uint32_t table_entry(const uint32_t* table, const uint32_t* w, int bit, uint32_t cp4) {
  constexpr int SH = NLUT == 32 ? 7 : 6;
  static_assert(NLUT == 32 || NLUT == 16, "copies");
  constexpr uint32_t M = ((1u << (2 * BITS)) - 1u) << SH;
  const int wi = bit >> 5, sh = bit & 31;
  uint32_t x;
  if (sh + 2 * BITS <= 32) x = sh >= SH ? (w[wi] >> (sh - SH)) : (w[wi] << (SH - sh));
  else x = __funnelshift_r(w[wi], w[wi + 1], sh - SH);  // sh > 32 - 2 BITS >= SH here
  return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(table) + ((x & M) | cp4));
}

// Offset of byte k of a lane's code words w inside a byte table: the byte
// in bits 8..15, the lane's copy offset cpo (< 256) in bits 0..7, by one
// byte permute.
__device__ __forceinline__ uint32_t byte_offset(const uint32_t* w, int k, uint32_t cpo) {
  return __byte_perm(w[k >> 2], cpo, 0x6504u | (static_cast<uint32_t>(k & 3) << 4));
}
// The f16x2 of the field (4-bit codes: a whole byte) in byte k.
__device__ __forceinline__ uint32_t byte_entry(const uint8_t* table, const uint32_t* w, int k, uint32_t cpo) {
  return *reinterpret_cast<const uint32_t*>(table + byte_offset(w, k, cpo));
}

// Walks the runs of pair p inside its CTA's range [i0, i1): per unit (run of
// ng items), the unit's items from s on (s = the first item of the unit
// inside the range) are cut into runs of GPB consecutive items; the pair
// takes runs p, p + NP, ... The group index and its ring slot advance by
// additions; divisions happen only when the walk enters a new unit. The
// chunks of a run are consecutive ring slots (wrapping to the unit's first
// slot).
template <int NP, int GPB>
struct RunCursor {
  int64_t item;        // first item of the current run (-1: exhausted)
  int64_t seg_end;     // end of the current unit inside the range
  int64_t grp;         // absolute group index of `item`
  int slot;            // grp mod n_slots
  int cnt;             // items in the run (1 .. GPB)
  const uint8_t* base; // the unit's first chunk
  const uint8_t* ptr;  // chunk of `item`

  __device__ __forceinline__ void enter(int64_t s, int64_t i1, int64_t ng, int w, int64_t g_begin, int n_slots,
                                        const uint8_t* chunks, int chunk_bytes) {
    while (s < i1) {
      const int64_t u = s / ng;
      const int64_t e = (u + 1) * ng < i1 ? (u + 1) * ng : i1;
      if (s + GPB * w < e) {
        item = s + GPB * w;
        seg_end = e;
        grp = g_begin + (item - u * ng);
        slot = static_cast<int>(grp % n_slots);
        base = chunks + static_cast<size_t>(u) * n_slots * chunk_bytes;
        ptr = base + static_cast<size_t>(slot) * chunk_bytes;
        cnt = (e - item) < GPB ? static_cast<int>(e - item) : GPB;
        return;
      }
      s = e;
    }
    item = -1;
  }
  __device__ __forceinline__ void advance(int64_t i1, int64_t ng, int w, int64_t g_begin, int n_slots,
                                          const uint8_t* chunks, int chunk_bytes) {
    if (item + GPB * NP < seg_end) {
      item += GPB * NP;
      grp += GPB * NP;
      slot += GPB * NP;
      while (slot >= n_slots) slot -= n_slots;
      ptr = base + static_cast<size_t>(slot) * chunk_bytes;
      cnt = (seg_end - item) < GPB ? static_cast<int>(seg_end - item) : GPB;
    } else {
      enter(seg_end, i1, ng, w, g_begin, n_slots, chunks, chunk_bytes);
    }
  }
  // chunk q (< cnt) of the run
  __device__ __forceinline__ const uint8_t* chunk(int q, int n_slots, int chunk_bytes) const {
    return q == 0 ? ptr : base + static_cast<size_t>(slot + q < n_slots ? slot + q : slot + q - n_slots) * chunk_bytes;
  }
};

// QX (KIVI only): the query enters unscaled and unrotated, so each value is
// exact in f16 (an f16 or bf16 activation) and q sK splits into an f16
// product and its exact residual in two operations; the score scale is
// applied in the softmax. Otherwise (RoPE applied here, or TurboQuant) the
// query is an fp32 value carried as f16 value + residual with the scale in.
// PR: keys stored before RoPE (KIVI with RoPE in the cache): the QK warp
// dequantises each key, rotates it at its position and scores it in two
// MMAs (f16 value and residual of the rotated key).
template <int D, int KB, int VB, bool TQ, bool QX, bool PR = false>
__global__ void __launch_bounds__(64 * KiviTile<D, KB, VB, TQ, PR>::NP, KiviTile<D, KB, VB, TQ, PR>::MIN_CTAS)
    decode_kivi_kernel(DecodeArgs a) {
  using T = KiviTile<D, KB, VB, TQ, PR>;
  constexpr int NP = T::NP, NST = T::NST, CHUNK = T::CHUNK;
  constexpr int S = D / 16, MV = D / 16, NVG = D / 32;
  constexpr int KW = D * KB / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  float* red = reinterpret_cast<float*>(smem + T::OFF_RED);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_ABORT);

  pdl_launch_dependents();
  const Geometry& G = a.geo;
  const unsigned full = 0xffffffffu;
  const int cta = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = warp % NP;
  const bool is_pv = warp >= NP;
  const int g = lane >> 2, t = lane & 3;
  const int gq = G.gqa;
  const int64_t ng = a.n_groups, work = a.work;
  const int64_t i0 = cta * work / a.n_ctas, i1 = (cta + 1) * work / a.n_ctas;
  const int n_slots = G.n_slots;

  constexpr int GPB = T::GPB, STAGE = T::STAGE;
  uint8_t* stages = smem + pair * NST * STAGE;
  uint8_t* pbuf = smem + T::OFF_PBUF + pair * 2 * T::PBUF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR) + pair * (NST + 4);
  uint64_t* full_bar = bars;            // [NST] chunk landed (one arrival: the copy's issuer)
  uint64_t* pfull = bars + NST;         // [2] weights written (32 arrivals: the QK warp's lanes)
  uint64_t* pempty = bars + NST + 2;    // [2] weights read (32 arrivals: the PV warp's lanes)
  if (threadIdx.x == 0) *abort_flag = 0;
  if (is_pv && lane == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(&full_bar[i], 1);
    for (int i = 0; i < 4; ++i) mbar_init(&pfull[i], 32);
    mbar_fence_init();
  }
  uint8_t* lut_k = smem + T::OFF_LUTK;
  uint8_t* lut_v = smem + T::OFF_LUTV;
  if constexpr (TQ) {  // value of code c: 2 c[c] - 1 (Foundry TurboQuant spec, "Algorithm Detail")
    // a field is (low code | high code << bits); the codebooks have 2^bits levels
    auto field = [](const float* cb, int bits, int f) {
      const int n = 1 << bits;
      return f2_to_h2(2.0f * cb[n - 1 + (f & (n - 1))] - 1.0f, 2.0f * cb[n - 1 + (f >> bits)] - 1.0f);
    };
    auto build = [&](uint8_t* lut, const float* cb, auto bits_c, auto byte_c) {
      constexpr int BITS = decltype(bits_c)::value;
      if constexpr (decltype(byte_c)::value) {  // byte e = one field: 32 copies of 4 B in a 256-B block
        for (int i = threadIdx.x; i < 256 * 32; i += blockDim.x)
          *reinterpret_cast<uint32_t*>(lut + (i >> 5) * 256 + (i & 31) * 4) = field(cb, BITS, i >> 5);
      } else {  // fields of 2 BITS bits: 2^(2 BITS) entries in NLUT copies
        for (int i = threadIdx.x; i < (1 << (2 * BITS)) * T::NLUT; i += blockDim.x)
          reinterpret_cast<uint32_t*>(lut)[i] = field(cb, BITS, i / T::NLUT);
      }
    };
    build(lut_k, a.tab.cb_k, std::integral_constant<int, KB>{}, std::bool_constant<T::KBYTE>{});
    build(lut_v, a.tab.cb_v, std::integral_constant<int, VB>{}, std::false_type{});
  }
  __syncthreads();

  // producer state (the PV warp: every lane keeps the same cursor, lane 0
  // issues): the next run whose chunks are to be fetched
  RunCursor<NP, GPB> pc{};
  int issued = 0;
  auto fetch = [&](int st) {  // the cursor's run into stage st, then advance
    expect_tx_if(lane == 0, &full_bar[st], static_cast<uint32_t>(pc.cnt * CHUNK));
    if (GPB == 1 || pc.cnt == 1 || pc.slot + 1 < n_slots) {  // the run's chunks are adjacent: one copy
      copy_g2s_if(lane == 0, stages + st * STAGE, pc.ptr, pc.cnt * CHUNK, &full_bar[st]);
    } else {
#pragma unroll
      for (int q = 0; q < GPB; ++q)
        if (q < pc.cnt) copy_g2s_if(lane == 0, stages + st * STAGE + q * CHUNK, pc.chunk(q, n_slots, CHUNK), CHUNK,
                                    &full_bar[st]);
    }
    pc.advance(i1, ng, pair, a.g_begin, n_slots, a.lay.chunks, CHUNK);
    ++issued;
  };
  if (is_pv) {
    pc.enter(i0, i1, ng, pair, a.g_begin, n_slots, a.lay.chunks, CHUNK);
    for (int i = 0; i < NST && pc.item >= 0; ++i) fetch(i);
  }
  int n_t = 0;  // runs this pair has processed (stage and buffer phases)
  bool failed = false;

  int64_t seg = i0;
  while (seg < i1) {
    const int64_t unit = seg / ng, ubase = unit * ng;
    const int64_t seg_e = ubase + ng < i1 ? ubase + ng : i1;
    const int b = static_cast<int>(unit / G.H), h = static_cast<int>(unit % G.H);
    // this pair's runs of the segment: run j starts at item my0 + j GPB NP
    // and holds min(GPB, seg_e - start) items (n_my runs)
    const int64_t my0 = seg + GPB * pair;
    const int n_my = my0 < seg_e ? static_cast<int>((seg_e - my0 + GPB * NP - 1) / (GPB * NP)) : 0;

    if (!is_pv) {
      // ------------------------------------------------------------ QK warp
      // the query operand of the unit, shared by the CTA's QK warps: per
      // k-step s and lane, {qx, qa} of the lane's two k-pairs (fold_q turns
      // it into the B operand). QX: qa is the value and qx the value on "lo"
      // columns, zero on the others. Otherwise qa is the column's operand
      // (value, or residual on "lo" columns) and qx as before, so that
      // qa s + (qx s - f16(qx s)) is the column's folded operand
      uint4* qsm = reinterpret_cast<uint4*>(smem + T::OFF_Q);
      if constexpr (TQ) {
        // rotated queries R q = FWHT(signs q) / sqrt(D) (Foundry TurboQuant
        // spec, "Optimization: Fused dequant-dot"), one QK warp per query
        // head, then the operand in natural channel order: k-step s, lane
        // (g, t) holds channels 16 s + 2t (+1) and 16 s + 2t + 8 (+1) of
        // column g (query head g / 2, value or residual)
        float* qf = reinterpret_cast<float*>(smem + T::OFF_QF);
        constexpr int NS = D / 32;
        const float rsq = static_cast<float>(1.0 / sqrt(static_cast<double>(D)));
        for (int j = pair; j < kMaxGqa; j += NP) {
          float y[NS];
#pragma unroll
          for (int i = 0; i < NS; ++i)
            y[i] = (j < gq) ? query_value(a, b, h * gq + j, i * 32 + lane) * a.tab.signs[i * 32 + lane] : 0.0f;
          warp_fwht<D>(y);
#pragma unroll
          for (int i = 0; i < NS; ++i) qf[j * D + i * 32 + lane] = y[i] * rsq;
        }
        named_barrier_sync(1, NP * 32);
        const int jc = g >> 1;
        const bool col_lo = g & 1;
        for (int s = pair; s < S; s += NP) {
          uint32_t v[4];
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const int c0 = 16 * s + 2 * t + 8 * p;
            const float x0 = qf[jc * D + c0], x1 = qf[jc * D + c0 + 1];
            const uint32_t hi = f2_to_h2(x0, x1);
            const float2 hf = h2_to_f2(hi);
            v[2 * p] = 0u;
            v[2 * p + 1] = col_lo ? f2_to_h2(x0 - hf.x, x1 - hf.y) : hi;
          }
          qsm[s * 32 + lane] = make_uint4(v[0], v[1], v[2], v[3]);
        }
        named_barrier_sync(1, NP * 32);  // the QK warps only
      } else if constexpr (PR) {
        // keys stored before RoPE: k-step s of lane (g, t) holds the RoPE
        // partners c = t D/8 + 2s + p and c + D/2 (kvq_layout.h k_frag_pos);
        // the query is rotated at q_pos, scale in, value or residual by column
        const int jc = g >> 1;
        const bool col_lo = g & 1;
        for (int s = pair; s < S; s += NP) {
          uint32_t v[4];
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const int c0 = t * (D / 8) + 2 * s + p;
            const float x0 = jc < gq ? query_value(a, b, h * gq + jc, c0, a.q_pos) : 0.0f;
            const float x1 = jc < gq ? query_value(a, b, h * gq + jc, c0 + D / 2, a.q_pos) : 0.0f;
            v[2 * p] = 0u;
            v[2 * p + 1] = split_h2(x0, x1, col_lo);
          }
          qsm[s * 32 + lane] = make_uint4(v[0], v[1], v[2], v[3]);
        }
        named_barrier_sync(1, NP * 32);  // the QK warps only
      } else {
        const int jc = g >> 1;        // query head of this lane's B column
        const bool col_lo = g & 1;    // B column holds the residual part
        for (int s = pair; s < S; s += NP) {
          uint32_t v[4];
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const int c0 = t * (D / 4) + 4 * s + 2 * p;
            const float2 x = jc < gq ? query_pair(a, b, h * gq + jc, c0, QX ? 1.0f : a.qscale, a.L - 1)
                                     : make_float2(0.0f, 0.0f);
            const float x0 = x.x, x1 = x.y;
            const uint32_t hi = f2_to_h2(x0, x1);
            if constexpr (QX) {  // {qm, qv}: q on "lo" columns (else 0), q
              v[2 * p] = col_lo ? hi : 0u;
              v[2 * p + 1] = hi;
            } else {
              const float2 hf = h2_to_f2(hi);
              v[2 * p] = col_lo ? hi : 0u;
              v[2 * p + 1] = col_lo ? f2_to_h2(x0 - hf.x, x1 - hf.y) : hi;
            }
          }
          qsm[s * 32 + lane] = make_uint4(v[0], v[1], v[2], v[3]);
        }
        named_barrier_sync(1, NP * 32);  // the QK warps only
      }
      // the running max m_run is in score units; ks turns them into log2
      // units (the score scale when the scores arrive unscaled, else 1)
      float m_run = -INFINITY, l_run = 0.0f;
      const float ks = QX ? a.qscale : 1.0f;
      const float lazy = QX ? kLazyRescale / a.qscale : kLazyRescale;
      const bool n_dyn = G.n_dyn != 0;
      CodeConsts<KB> kc;
      kc.load(a);
      // the B operand of one k-step: the query operand {qx, qa} times the K
      // scales sK of its channels, as an f16 product on "value" columns and
      // the rest of the product on "lo" columns
      auto fold_q = [&](uint32_t qx, uint32_t qa, uint32_t sk) -> uint32_t {
        const __half2 sv = as_h2(sk);
        const __half2 x = __hmul2(as_h2(qx), sv);
        if constexpr (QX) {  // qv sK - (qm sK on lo columns): the product, or its exact residual
          return as_u32(__hfma2(as_h2(qa), sv, __hneg2(x)));
        } else {  // qa sK + the exact residual of qx sK
          const __half2 y = __hfma2(as_h2(qx), sv, __hneg2(x));
          return as_u32(__hfma2(as_h2(qa), sv, y));
        }
      };
      // scores of one group into the lane's C fragment
      auto qk_scores = [&](const uint8_t* tile, float (&sc)[2][4], int64_t kpos0) {
        if constexpr (TQ) {
          // scores in the rotated domain: the lane's K fields (fragment order,
          // kvq_layout.h tq_kfield_bit) from its own words of the tile, each
          // field turned into the f16x2 of its two codebook values by the
          // lane's copy of the table; the K norm of each token scales its row
          constexpr int KWT = D * KB / 32, PWT = piece_words(KWT);
          uint32_t kw[KWT + 1];
          load_lane_words<KWT, PWT>(tile, lane, kw);
          kw[KWT] = 0u;
          const uint32_t cpk = 4u * (lane % T::NLUT);
          float acc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
          for (int s = 0; s < S; ++s) {  // one read of the query operand per k-step serves both m-tiles
            const uint4 q4 = qsm[s * 32 + lane];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              // field (b, j) of the lane's string is at bit (b D / 8 + j) 2 KB
              uint32_t a0, a1, a2, a3;
              if constexpr (T::KBYTE) {  // one byte per field
                a0 = byte_entry(lut_k, kw, 2 * mt * (D / 8) + 2 * s, cpk);
                a1 = byte_entry(lut_k, kw, (2 * mt + 1) * (D / 8) + 2 * s, cpk);
                a2 = byte_entry(lut_k, kw, 2 * mt * (D / 8) + 2 * s + 1, cpk);
                a3 = byte_entry(lut_k, kw, (2 * mt + 1) * (D / 8) + 2 * s + 1, cpk);
              } else {
                const uint32_t* lk = reinterpret_cast<const uint32_t*>(lut_k);
                a0 = table_entry<KB, T::NLUT>(lk, kw, tq_kfield_bit(D, KB, 2 * mt, 2 * s), cpk);
                a1 = table_entry<KB, T::NLUT>(lk, kw, tq_kfield_bit(D, KB, 2 * mt + 1, 2 * s), cpk);
                a2 = table_entry<KB, T::NLUT>(lk, kw, tq_kfield_bit(D, KB, 2 * mt, 2 * s + 1), cpk);
                a3 = table_entry<KB, T::NLUT>(lk, kw, tq_kfield_bit(D, KB, 2 * mt + 1, 2 * s + 1), cpk);
              }
              mma_f16(acc[mt], a0, a1, a2, a3, q4.y, q4.w);
            }
          }
          const float* kn = reinterpret_cast<const float*>(tile + T::KMETA);
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const float n0 = kn[16 * mt + g], n1 = kn[16 * mt + g + 8];
            sc[mt][0] = acc[mt][0] * n0;
            sc[mt][1] = acc[mt][1] * n0;
            sc[mt][2] = acc[mt][2] * n1;
            sc[mt][3] = acc[mt][3] * n1;
          }
        } else if constexpr (PR) {
          // each key dequantised (code s + z, fp32), rotated at its position
          // kpos0 + token (the table, clamped: masked tokens may lie outside
          // it) and split into an f16 value and residual, two MMAs per k-step
          uint32_t kr[KW];
          load_lane_words<KW, piece_words(KW)>(tile, lane, kr);
          const __half* ksc = reinterpret_cast<const __half*>(tile + T::KMETA);
          const __half* kzr = ksc + D;
          const int i0 = t * (D / 8);
          const int64_t pmax = a.geo.rope_max_pos - 1;
          float acc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
          const float* rope_rows[2][2];  // table rows of tokens 16 mt + g (+ 8), clamped
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
              int64_t kp = kpos0 + 16 * mt + g + 8 * rh;
              kp = kp < 0 ? 0 : (kp > pmax ? pmax : kp);
              rope_rows[mt][rh] = a.tab.rope + static_cast<size_t>(kp) * D + 2 * i0;
            }
#pragma unroll
          for (int s = 0; s < S; ++s) {
            const uint4 q4 = qsm[s * 32 + lane];
            float sk[2][2], zk[2][2];  // scale (unit folded in) and zero of channels i0 + 2s + pp and + D/2
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int c = i0 + 2 * s + pp + hh * (D / 2);
                sk[pp][hh] = __half2float(ksc[c]) * CodeConsts<KB>::kCodeInv;
                zk[pp][hh] = __half2float(kzr[c]);
              }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              uint32_t ah[4], al[4];
#pragma unroll
              for (int reg = 0; reg < 4; ++reg) {
                const int pp = reg >> 1, rh = reg & 1;
                const float2 cs = *reinterpret_cast<const float2*>(rope_rows[mt][rh] + 2 * (2 * s + pp));
                const float2 cf = h2_to_f2(pair_at<KB>(kc, kr, (mt * S + s) * 4 + reg));
                float ra, rb;
                rope_pair(fmaf(cf.x, sk[pp][0], zk[pp][0]), fmaf(cf.y, sk[pp][1], zk[pp][1]), cs.x, cs.y, &ra, &rb);
                ah[reg] = f2_to_h2(ra, rb);
                const float2 hf = h2_to_f2(ah[reg]);
                al[reg] = f2_to_h2(ra - hf.x, rb - hf.y);
              }
              mma_f16(acc[mt], ah[0], ah[1], ah[2], ah[3], q4.y, q4.w);
              mma_f16(acc[mt], al[0], al[1], al[2], al[3], q4.y, q4.w);
            }
            asm volatile("" ::: "memory");  // keep the next k-step's loads from being hoisted here
          }
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[mt][e] = acc[mt][e];
        } else {
          uint32_t kr[KW];
          load_lane_words<KW, piece_words(KW)>(tile, lane, kr);
          const uint4* ks = reinterpret_cast<const uint4*>(tile + T::KMETA);
          // the zero-point operand: every row is the k-step's zero row
          const uint8_t* zrow = tile + T::KMETA + 2 * D + ((lane >> 4) & 1) * 16;
          float zb[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
          float sa[2][2][4] = {};
#pragma unroll
          for (int u = 0; u < S / 2; ++u) {
            const uint4 s4 = ks[u * 4 + t];
            const uint32_t sp[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
              const int s = 2 * u + hlf;
              const uint4 q4 = qsm[s * 32 + lane];
              const uint32_t qx[2] = {q4.x, q4.z}, qa[2] = {q4.y, q4.w};
              uint32_t bq[2];
#pragma unroll
              for (int p = 0; p < 2; ++p) bq[p] = fold_q(qx[p], qa[p], sp[2 * hlf + p]);
              uint32_t za[4];
              ldmatrix_x4(za, zrow + s * 32);
              mma_f16(zb[hlf], za[0], za[1], za[2], za[3], QX ? qx[0] : qa[0], QX ? qx[1] : qa[1]);
#pragma unroll
              for (int mt = 0; mt < 2; ++mt) {
                const int pbase = (mt * S + s) * 4;
                const uint32_t a0 = pair_at<KB>(kc, kr, pbase + 0);
                const uint32_t a1 = pair_at<KB>(kc, kr, pbase + 1);
                const uint32_t a2 = pair_at<KB>(kc, kr, pbase + 2);
                const uint32_t a3 = pair_at<KB>(kc, kr, pbase + 3);
                mma_f16(sa[mt][s & 1], a0, a1, a2, a3, bq[0], bq[1]);
              }
            }
          }
          const float2 ci = make_float2(CodeConsts<KB>::kCodeInv, CodeConsts<KB>::kCodeInv);
#pragma unroll
          for (int e = 0; e < 4; e += 2) {  // two accumulator elements per FP32x2 instruction
            const float2 z = __fadd2_rn(make_float2(zb[0][e], zb[0][e + 1]), make_float2(zb[1][e], zb[1][e + 1]));
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              const float2 r = __ffma2_rn(__fadd2_rn(make_float2(sa[mt][0][e], sa[mt][0][e + 1]),
                                                     make_float2(sa[mt][1][e], sa[mt][1][e + 1])),
                                          ci, z);
              sc[mt][e] = r.x, sc[mt][e + 1] = r.y;
            }
          }
        }
      };
      // scores of the two groups of a run, k-step by k-step: one read of
      // the query operand per k-step serves both, and their MMA chains are
      // independent (KIVI runs of two groups only)
      auto qk_scores_pair = [&](const uint8_t* t0, const uint8_t* t1, float (&sc)[2][2][4]) {
        const uint8_t* tl[2] = {t0, t1};
        uint32_t kr[2][KW];
#pragma unroll
        for (int q = 0; q < 2; ++q) load_lane_words<KW, piece_words(KW)>(tl[q], lane, kr[q]);
        float zb[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
        float sa[2][2][4] = {};
#pragma unroll
        for (int u = 0; u < S / 2; ++u) {
          uint32_t sp[2][4];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint4 s4 = reinterpret_cast<const uint4*>(tl[q] + T::KMETA)[u * 4 + t];
            sp[q][0] = s4.x;
            sp[q][1] = s4.y;
            sp[q][2] = s4.z;
            sp[q][3] = s4.w;
          }
#pragma unroll
          for (int hlf = 0; hlf < 2; ++hlf) {
            const int s = 2 * u + hlf;
            const uint4 q4 = qsm[s * 32 + lane];
            const uint32_t qx[2] = {q4.x, q4.z}, qa[2] = {q4.y, q4.w};
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              uint32_t bq[2];
#pragma unroll
              for (int p = 0; p < 2; ++p) bq[p] = fold_q(qx[p], qa[p], sp[q][2 * hlf + p]);
              uint32_t za[4];
              ldmatrix_x4(za, tl[q] + T::KMETA + 2 * D + ((lane >> 4) & 1) * 16 + s * 32);
              mma_f16(zb[q], za[0], za[1], za[2], za[3], QX ? qx[0] : qa[0], QX ? qx[1] : qa[1]);
#pragma unroll
              for (int mt = 0; mt < 2; ++mt) {
                const int pbase = (mt * S + s) * 4;
                const uint32_t a0 = pair_at<KB>(kc, kr[q], pbase + 0);
                const uint32_t a1 = pair_at<KB>(kc, kr[q], pbase + 1);
                const uint32_t a2 = pair_at<KB>(kc, kr[q], pbase + 2);
                const uint32_t a3 = pair_at<KB>(kc, kr[q], pbase + 3);
                mma_f16(sa[q][mt], a0, a1, a2, a3, bq[0], bq[1]);
              }
            }
          }
        }
        const float2 ci = make_float2(CodeConsts<KB>::kCodeInv, CodeConsts<KB>::kCodeInv);
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int e = 0; e < 4; e += 2) {  // two accumulator elements per FP32x2 FMA
            const float2 z = make_float2(zb[q][e], zb[q][e + 1]);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              const float2 r = __ffma2_rn(make_float2(sa[q][mt][e], sa[q][mt][e + 1]), ci, z);
              sc[q][mt][e] = r.x, sc[q][mt][e + 1] = r.y;
            }
          }
      };
      for (int k = 0; k < n_my && !failed; ++k, ++n_t) {
        const int st = n_t % NST, pb = n_t & 1;
        const int64_t f = my0 + static_cast<int64_t>(k) * GPB * NP;  // first item of the run
        const int cnt = (seg_e - f) < GPB ? static_cast<int>(seg_e - f) : GPB;
        if (!warp_wait(&full_bar[st], static_cast<uint32_t>((n_t / NST) & 1), abort_flag)) {
          failed = true;
          break;
        }
        float scr[GPB][2][4];
        if constexpr (GPB == 2) {  // a short run scores its one group twice (the copy is discarded)
          qk_scores_pair(stages + st * STAGE, stages + st * STAGE + (cnt > 1 ? CHUNK : 0), scr);
        } else {
          qk_scores(stages + st * STAGE, scr[0], (a.g_begin + (f - ubase)) * kGroup - a.key_shift);
        }
        float pr[GPB][2][2];
#pragma unroll
        for (int q = 0; q < GPB; ++q) {
          if (q >= cnt) {  // a short run: no group here
            pr[q][0][0] = pr[q][0][1] = pr[q][1][0] = pr[q][1][1] = -INFINITY;
            continue;
          }
          const float (&sc)[2][4] = scr[q];
          // valid tokens: inside [qlo, F) and not a KVSink sink of this group
          // (only the unit's first and last groups can be partial)
          const int64_t it = f + q;
          uint32_t vbits = 0xffffffffu;
          if (__any_sync(full, it == ubase || it == ubase + ng - 1) || n_dyn) {
            const int64_t grp = a.g_begin + (it - ubase);
            const int64_t p0 = grp * kGroup;
            if (p0 < a.qlo) vbits &= 0xffffffffu << static_cast<int>(a.qlo - p0);
            if (p0 + kGroup > a.F) vbits &= (1u << static_cast<int>(a.F - p0)) - 1u;
            if (n_dyn) vbits &= ~a.lay.sink_mask[b * n_slots + static_cast<int>(grp % n_slots)];
          }
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) pr[q][mt][r] = sc[mt][2 * r] + sc[mt][2 * r + 1];
          if (vbits != 0xffffffffu || gq < kMaxGqa) {  // uniform: only edge groups pay for masking
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                const int tok = 16 * mt + g + 8 * r;
                if (t >= gq || !((vbits >> tok) & 1u)) pr[q][mt][r] = -INFINITY;
              }
          }
        }
        // lazy rescaling: the running max only moves when some score exceeds
        // it by more than the headroom, so weights stay below 2^8 and the
        // common path needs one warp vote (per run) instead of a max reduction
        float al = 1.0f;
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < GPB; ++q) mx = fmaxf(mx, fmaxf(fmaxf(pr[q][0][0], pr[q][0][1]), fmaxf(pr[q][1][0], pr[q][1][1])));
        if (__any_sync(full, mx > m_run + lazy)) {
          mx = fmaxf(mx, __shfl_xor_sync(full, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(full, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(full, mx, 16));
          const float mn = mx > m_run + lazy ? mx : m_run;
          al = (m_run == -INFINITY) ? 0.0f : fast_exp2((m_run - mn) * ks);
          l_run *= al;
          m_run = mn;
        }
        const float nref = (m_run == -INFINITY) ? 0.0f : -m_run * ks;  // exponent offset
        // weights as (f16 value, 0) per token (the odd B columns stay zero),
        // tokens g and g + 8 of an m-tile in one f16x2 word; two tokens per
        // FP32x2 instruction
        uint32_t ph[GPB][2];
        const float2 ks2 = make_float2(ks, ks), nref2 = make_float2(nref, nref);
        float2 l2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < GPB; ++q)
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const float2 x2 = __ffma2_rn(make_float2(pr[q][mt][0], pr[q][mt][1]), ks2, nref2);
            const float2 p2 = make_float2(fast_exp2(x2.x), fast_exp2(x2.y));
            l2 = __fadd2_rn(l2, p2);
            float2 w = p2;
            if constexpr (TQ) {  // the V norm of the token folded in (rows past F hold no data: weight 0)
              const float* nv = reinterpret_cast<const float*>(stages + st * STAGE + q * CHUNK + T::VMETA);
              w.x = p2.x > 0.0f ? p2.x * nv[16 * mt + g] : 0.0f;
              w.y = p2.y > 0.0f ? p2.y * nv[16 * mt + g + 8] : 0.0f;
            }
            const __half2 wh = __floats2half2_rn(w.x, w.y);
            ph[q][mt] = *reinterpret_cast<const uint32_t*>(&wh);
          }
        l_run += l2.x + l2.y;
        // hand the weights to the PV warp
        if (!warp_wait(&pempty[pb], static_cast<uint32_t>(((n_t >> 1) & 1) ^ 1), abort_flag)) {
          failed = true;
          break;
        }
        uint8_t* pw = pbuf + pb * T::PBUF;
#pragma unroll
        for (int q = 0; q < GPB; ++q)
          *reinterpret_cast<uint2*>(pw + (q * 32 + lane) * 8) = make_uint2(ph[q][0], ph[q][1]);
        reinterpret_cast<float*>(pw + GPB * 32 * 8)[t] = al;  // the 8 lanes of query head t store the same value
        mbar_arrive(&pfull[pb]);
      }
      l_run += __shfl_xor_sync(full, l_run, 4);
      l_run += __shfl_xor_sync(full, l_run, 8);
      l_run += __shfl_xor_sync(full, l_run, 16);
      __syncthreads();  // (1) the previous unit's partial has been written
      if (t < gq && g == 0) {
        float* rj = red + (pair * kMaxGqa + t) * (D + 2);
        rj[D] = m_run * ks;  // log2 units
        rj[D + 1] = l_run;
      }
    } else {
      // ------------------------------------------------------------ PV warp
      float oacc[MV][4];
      // zero-point sums: rows = V channel groups (g < NVG), columns as oacc
      float zacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int m = 0; m < MV; ++m) oacc[m][0] = oacc[m][1] = oacc[m][2] = oacc[m][3] = 0.0f;
      CodeConsts<VB> vc;
      vc.load(a);
      // values of one group with its weights ph into oacc, zacc
      auto pv_values = [&](const uint8_t* tile, const uint32_t (&ph)[4]) {
        if constexpr (TQ) {
          // out^T += V^T (p n_v) with one B operand for every m-tile; the A
          // fragments come straight from the token-pair rows (kvq_layout.h):
          // lane (g, t) needs tokens 16 kb + 2t (+1) and 16 kb + 2t + 8 (+9),
          // i.e. pair rows 8 kb + t and 8 kb + t + 4, and in each the fields
          // of channels g + 8 j: block g of the row, whose fields are exactly
          // its A pairs (channel, two tokens); the lane's copy of the table
          // turns them into f16x2
          constexpr int RB = tq_vrow_bytes(D, VB), BB = D * VB / 32, BW = (BB + 3) / 4;
          const uint32_t cpv = 4u * (lane % T::NLUT);
          const uint8_t* vrows = tile + T::VC;
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            const uint32_t b0 = movmatrix_t(ph[2 * kb]);
            const uint32_t b1 = movmatrix_t(ph[2 * kb + 1]);
            // the words of block hh (pair row 8 kb + t + 4 hh, block g)
            auto load_block = [&](int hh, uint32_t (&bw)[BW + 1]) {
              const uint8_t* blk = vrows + (8 * kb + t + 4 * hh) * RB + g * BB;
              if constexpr (BB % 16 == 0) {
                const uint4 v = *reinterpret_cast<const uint4*>(blk);
                bw[0] = v.x, bw[1] = v.y, bw[2] = v.z, bw[3] = v.w;
              } else if constexpr (BB % 8 == 0) {
                const uint2 v = *reinterpret_cast<const uint2*>(blk);
                bw[0] = v.x, bw[1] = v.y;
              } else if constexpr (BB % 4 == 0) {
#pragma unroll
                for (int k = 0; k < BW; ++k) bw[k] = reinterpret_cast<const uint32_t*>(blk)[k];
              } else {  // 6-byte blocks (3-bit codes, head_dim 64)
                const uint16_t* h16 = reinterpret_cast<const uint16_t*>(blk);
                bw[0] = h16[0] | (static_cast<uint32_t>(h16[1]) << 16);
                bw[1] = h16[2];
              }
              bw[BW] = 0u;
            };
            const uint32_t* lv = reinterpret_cast<const uint32_t*>(lut_v);
            if constexpr (VB == 4) {
              uint32_t bw[2][BW + 1];
              load_block(0, bw[0]);
              load_block(1, bw[1]);
#pragma unroll
              for (int m = 0; m < MV; ++m)
                mma_f16(oacc[m], table_entry<VB, T::NLUT>(lv, bw[0], 4 * VB * m, cpv),
                        table_entry<VB, T::NLUT>(lv, bw[0], 4 * VB * m + 2 * VB, cpv),
                        table_entry<VB, T::NLUT>(lv, bw[1], 4 * VB * m, cpv),
                        table_entry<VB, T::NLUT>(lv, bw[1], 4 * VB * m + 2 * VB, cpv), b0, b1);
            } else {
              uint32_t A[MV][4];
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                uint32_t bw[BW + 1];
                load_block(hh, bw);
#pragma unroll
                for (int jj = 0; jj < 2 * MV; ++jj)
                  A[jj >> 1][2 * hh + (jj & 1)] = table_entry<VB, T::NLUT>(lv, bw, 2 * VB * jj, cpv);
              }
#pragma unroll
              for (int m = 0; m < MV; ++m) mma_f16(oacc[m], A[m][0], A[m][1], A[m][2], A[m][3], b0, b1);
            }
          }
        } else {
        // the weights as the B operand (column g, token pairs 2t + 8 kk,
        // + 1; the odd columns are zero), shared by the zero-point MMA and
        // every channel group
        uint32_t bT[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) bT[kk] = movmatrix_t(ph[kk]);
        // zero points: zsum[v][j] += sum_t zV[t][v] p_j[t] as one MMA per
        // 16 tokens with the groups as rows (the zeros are stored group-major)
        {
          const uint32_t* zw = reinterpret_cast<const uint32_t*>(tile + T::VMETA + 64 * NVG);
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            const uint32_t z0 = g < NVG ? zw[g * 16 + 8 * kb + t] : 0u;
            const uint32_t z2 = g < NVG ? zw[g * 16 + 8 * kb + t + 4] : 0u;
            mma_f16(zacc, z0, 0u, z2, 0u, bT[2 * kb], bT[2 * kb + 1]);
          }
        }
        // V scales in B order: 16 bytes per lane and group hold the scales
        // of the lane's token pairs 2t + 8 kk, + 1 (kk = 0..3)
        const uint4* vsc = reinterpret_cast<const uint4*>(tile + T::VMETA);
        const uint4* vcode = reinterpret_cast<const uint4*>(tile + T::VC);
#pragma unroll
        for (int v = 0; v < NVG; ++v) {
          // the VB code words of channel group v (m-tiles 2v, 2v + 1), loaded
          // when first needed to keep them live briefly
          uint32_t vr[VB];
          load_lane_range<VB, piece_words(D * VB / 32)>(reinterpret_cast<const uint8_t*>(vcode), lane, v * VB, vr);
          const uint4 s4 = vsc[v * 4 + t];
          const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            // p s of each token: one f16 product per weight
            const uint32_t b0 = as_u32(__hmul2(as_h2(bT[2 * kb]), as_h2(sw[2 * kb])));
            const uint32_t b1 = as_u32(__hmul2(as_h2(bT[2 * kb + 1]), as_h2(sw[2 * kb + 1])));
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int m = 2 * v + hh;
              const int pbase = (m * 2 + kb) * 4;
              const uint32_t a0 = pair_at<VB>(vc, vr, pbase + 0 - 16 * v);
              const uint32_t a1 = pair_at<VB>(vc, vr, pbase + 1 - 16 * v);
              const uint32_t a2 = pair_at<VB>(vc, vr, pbase + 2 - 16 * v);
              const uint32_t a3 = pair_at<VB>(vc, vr, pbase + 3 - 16 * v);
              mma_f16(oacc[m], a0, a1, a2, a3, b0, b1);
            }
          }
        }
        }
      };
      for (int k = 0; k < n_my && !failed; ++k, ++n_t) {
        const int st = n_t % NST, pb = n_t & 1;
        const int64_t f = my0 + static_cast<int64_t>(k) * GPB * NP;
        const int cnt = (seg_e - f) < GPB ? static_cast<int>(seg_e - f) : GPB;
        if (!warp_wait(&pfull[pb], static_cast<uint32_t>((n_t >> 1) & 1), abort_flag) ||
            !warp_wait(&full_bar[st], static_cast<uint32_t>((n_t / NST) & 1), abort_flag)) {
          failed = true;
          break;
        }
        const uint8_t* pw = pbuf + pb * T::PBUF;
        uint32_t ph[GPB][4];
#pragma unroll
        for (int q = 0; q < GPB; ++q) {
          // the four f16 weights, each back to (value, 0) for the transposes
          const uint2 pv2 = *reinterpret_cast<const uint2*>(pw + (q * 32 + lane) * 8);
          ph[q][0] = pv2.x & 0xffffu;
          ph[q][1] = pv2.x >> 16;
          ph[q][2] = pv2.y & 0xffffu;
          ph[q][3] = pv2.y >> 16;
        }
        const float al = reinterpret_cast<const float*>(pw + GPB * 32 * 8)[t];
        mbar_arrive(&pempty[pb]);
        if (__any_sync(full, al != 1.0f)) {
#pragma unroll
          for (int m = 0; m < MV; ++m) {
            oacc[m][0] *= al;
            oacc[m][1] *= al;
            oacc[m][2] *= al;
            oacc[m][3] *= al;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) zacc[e] *= al;
        }
#pragma unroll
        for (int q = 0; q < GPB; ++q)
          if (q < cnt) pv_values(stages + st * STAGE + q * CHUNK, ph[q]);
        // this pair is done with the stage: refill it with the next run
        __syncwarp();
        if (pc.item >= 0) fetch(st);
      }
      // zero sum of group v, query head t, is in lane (v, t)
      const float zt = TQ ? 0.0f : zacc[0] + zacc[1];
      __syncthreads();  // (1) the previous unit's partial has been written
#pragma unroll
      for (int m = 0; m < MV; ++m) {
        const float zg = __shfl_sync(full, zt, (m >> 1) * 4 + t);
        if (t < gq) {
          float* rj = red + (pair * kMaxGqa + t) * (D + 2);
          const float cu = TQ ? 1.0f : CodeConsts<VB>::kCodeInv;
          rj[16 * m + g] = fmaf(oacc[m][0] + oacc[m][1], cu, zg);
          rj[16 * m + g + 8] = fmaf(oacc[m][2] + oacc[m][3], cu, zg);
        }
      }
    }
    __syncthreads();  // (2) red complete
    write_partial<D, 2 * NP>(a, red, b, h, cta - owner_cta(ubase, work, a.n_ctas), NP);
    seg = seg_e;
  }
  if ((failed || *abort_flag) && lane == 0) set_error(a.tab.err_flag, kErrTimeout);
  // the copies this pair issued but never consumed must land before exit
  if (is_pv && lane == 0) {
    for (int i = n_t; i < issued; ++i)
      (void)mbar_wait_bounded(&full_bar[i % NST], static_cast<uint32_t>((i / NST) & 1));
  }
}

template <int D, int KB, int VB, bool TQ, bool QX, bool PR = false>
cudaError_t launch_kivi_instance(DecodeArgs& a, cudaStream_t s, int sm_count) {
  using T = KiviTile<D, KB, VB, TQ, PR>;
  const size_t smem = T::smem_bytes();
  static int occ_of[kMaxDevices] = {};  // per device: the attribute is per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int& occupancy = occ_of[dev];
  if (!occupancy) {
    e = cudaFuncSetAttribute(decode_kivi_kernel<D, KB, VB, TQ, QX, PR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occupancy, decode_kivi_kernel<D, KB, VB, TQ, QX, PR>, 64 * T::NP, smem);
    if (e != cudaSuccess) return e;
    if (occupancy < 1) occupancy = 1;
  }
  // stream-K CTAs: fill the machine, never more than one per group, and at
  // most max_splits per unit (partial slots per query head)
  int64_t n = a.n_ctas_hint > 0 ? a.n_ctas_hint : static_cast<int64_t>(sm_count) * occupancy;
  const int64_t units = static_cast<int64_t>(a.geo.B) * a.geo.H;
  if (n > a.work) n = a.work;
  if (n > units * (a.geo.max_splits - 1)) n = units * (a.geo.max_splits - 1);
  if (n < 1) n = 1;
  a.n_ctas = static_cast<int>(n);
  if (a.work <= 0) return cudaSuccess;  // nothing quantised to read: the merge does it all
  decode_kivi_kernel<D, KB, VB, TQ, QX, PR><<<a.n_ctas, 64 * T::NP, smem, s>>>(a);
  return cudaGetLastError();
}

// KIVI decode of K width K (the V width and the query form picked at run
// time): one translation unit per (head_dim, K width) keeps the build parallel.
template <int D, int K>
cudaError_t launch_kivi_k(DecodeArgs& a, cudaStream_t s, int sm_count) {
  // an exact query operand unless RoPE is applied to the query here
  const bool qx = a.tab.rope == nullptr;
#define KVQ_CASE(V)                                                                                       \
  if (a.geo.vb == V)                                                                                      \
    return a.geo.k_pre_rope ? launch_kivi_instance<D, K, V, false, false, true>(a, s, sm_count)          \
           : qx             ? launch_kivi_instance<D, K, V, false, true>(a, s, sm_count)                 \
                            : launch_kivi_instance<D, K, V, false, false>(a, s, sm_count);
  KVQ_CASE(2) KVQ_CASE(3) KVQ_CASE(4) KVQ_CASE(8)
#undef KVQ_CASE
  return cudaErrorInvalidValue;
}

// TurboQuant decode (K and V widths 2, 3 or 4).
template <int D>
cudaError_t launch_tq_d(DecodeArgs& a, cudaStream_t s, int sm_count) {
#define KVQ_CASE(K, V) \
  if (a.geo.kb == K && a.geo.vb == V) return launch_kivi_instance<D, K, V, true, false>(a, s, sm_count);
  KVQ_CASE(2, 2) KVQ_CASE(2, 3) KVQ_CASE(2, 4)
  KVQ_CASE(3, 2) KVQ_CASE(3, 3) KVQ_CASE(3, 4)
  KVQ_CASE(4, 2) KVQ_CASE(4, 3) KVQ_CASE(4, 4)
#undef KVQ_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kvq
