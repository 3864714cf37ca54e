// Internal layout of the cache arena: group chunks, the tail ring and the
// fragment-native order of the packed codes. Included by the host code and
// by the kernels of the library (and by nothing else).
//
// A "chunk" holds one 32-token group of one (layer, b, kv-head):
//   KIVI:       [K codes 32*D*kb/8][K scales D f16][K zeros D f16]
//               [V codes 32*D*vb/8][V scales 32 x D/32 f16][V zeros D/32 x 32 f16]
//               (both group-major, scales in lane order: vscale_pos, vzero_pos)
//   TurboQuant: [K codes 32*D*kb/8 in fragment order (tq_kfield_bit)][K norms 32 f32]
//               [V codes 32 x D*vb/8 row-major][V norms 32 f32]
// Chunk sizes are multiples of 16 bytes so one 1-D bulk copy moves a chunk.
// 3-bit codes are packed tight, eight to three bytes (Foundry spec, "Step 3:
// Packing", the no-waste form): a row-major code row is one little-endian
// bit string with code c at bits 3c .. 3c+2; the fragment-order forms are
// given below.
//
// KIVI codes are stored in the order the decode kernel's tensor-core
// fragments consume them (the canonical, page-defined order is produced by
// kv_cache_export). The 32 lanes of the consuming warp (lane = 4 g + t) own
// D codes each. Fragment element f = 0 .. D-1 of a lane maps to a (token,
// channel) of the group:
//   K (A operand of S^T = K Q^T, m16n8k16, rows = tokens, k = channels):
//     f = ((mt * S + s) * 4 + r) * 2 + e,  S = D/16, mt in {0,1}, r in 0..3
//     token = 16 mt + g + 8 (r & 1);  channel = t D/4 + 4 s + 2 (r >> 1) + e
//   V (A operand of O^T = V^T P^T, rows = channels, k = tokens):
//     f = ((m * 2 + kb) * 4 + r) * 2 + e,  m in [0, D/16), kb in {0,1}
//     channel = 16 m + g + 8 (r & 1);  token = 16 kb + 2 t + e + 8 (r >> 1)
// Element f sits in 32-bit word w = f / (32/bits) of its lane at the bit
// frag_bits gives: placed so that one mask turns a pair of codes into a pair
// of narrow floats (e2m1 for 2-bit, e4m3 for 4-bit) or, for 8-bit, into a
// pair of bytes 16 bits apart, each converted to an exact f16x2 by one
// instruction in the decode kernel. 3-bit elements go in blocks of 32 (f /
// 32) of three words each (frag3_bits), placed so that a mask or two turn
// four codes into four bytes, each an e2m3 value code / 8 (the subnormal
// binade, evenly spaced), converted two at a time. Words are interleaved across
// lanes in 16-byte pieces (word w of lane L at byte ((w/4) * 32 + L) * 16 +
// (w % 4) * 4) so that a warp's 16-byte loads are contiguous.
// K scales are kept in the order the B operand is built: f16 position
// (u * 4 + t) * 8 + e holds channel t D/4 + 8 u + e (u = pair of k-steps), so
// the four lanes t read one contiguous 64-byte run; K zeros are kept as one
// 16-value row per k-step in MMA k order (kzero_pos).
#pragma once

#include <cstddef>
#include <cstdint>

#if defined(__CUDACC__)
#define KVQ_HD __host__ __device__ __forceinline__
#else
#define KVQ_HD inline
#endif

namespace kvq {

constexpr int kGroup = 32;
constexpr int kMaxSinks = 32;
constexpr int kMaxGqa = 4;
constexpr int kMaxDevices = 64;  // device ordinals the per-device launch settings cover

struct Chunk {
  int kc_off, kmeta_off, vc_off, vmeta_off, bytes;
};

// kb, vb: code widths (2, 3, 4 or 8; codes packed tight).
KVQ_HD Chunk chunk_layout(int mode_tq, int D, int kb, int vb) {
  Chunk c;
  c.kc_off = 0;
  c.kmeta_off = kGroup * D * kb / 8;
  if (!mode_tq) {  // K meta: D scales then D zeros (f16); V meta per token: D/32 scales, D/32 zeros
    c.vc_off = c.kmeta_off + 4 * D;
    c.vmeta_off = c.vc_off + kGroup * D * vb / 8;
    c.bytes = c.vmeta_off + 4 * D;
  } else {
    c.vc_off = c.kmeta_off + 4 * kGroup;
    c.vmeta_off = c.vc_off + kGroup * D * vb / 8;
    c.bytes = c.vmeta_off + 4 * kGroup;
  }
  return c;
}

// (token, channel) of fragment element f of lane (g, t) for K. With keys
// stored before RoPE (pr) the two elements of a pair are RoPE partners:
// channel t D/8 + 2s + (r >> 1) and that + D/2, so one lane rotates them.
KVQ_HD void k_frag_pos(int D, int lane, int f, int* token, int* channel, bool pr = false) {
  const int g = lane >> 2, t = lane & 3, S = D / 16;
  const int e = f & 1, r = (f >> 1) & 3, ms = f >> 3;  // ms = mt * S + s
  const int mt = ms / S, s = ms % S;
  *token = 16 * mt + g + 8 * (r & 1);
  *channel = pr ? t * (D / 8) + 2 * s + (r >> 1) + e * (D / 2) : t * (D / 4) + 4 * s + 2 * (r >> 1) + e;
}

// (token, channel) of fragment element f of lane (g, t) for V.
KVQ_HD void v_frag_pos(int D, int lane, int f, int* token, int* channel) {
  (void)D;
  const int g = lane >> 2, t = lane & 3;
  const int e = f & 1, r = (f >> 1) & 3, mk = f >> 3;  // mk = m * 2 + kb
  const int m = mk >> 1, kb = mk & 1;
  *channel = 16 * m + g + 8 * (r & 1);
  *token = 16 * kb + 2 * t + e + 8 * (r >> 1);
}

// Words per interleaved piece of a lane block of `words` words: 16-byte
// pieces, or 8-byte ones where the block is not a whole number of 16-byte
// pieces (3-bit codes at head_dim 64: 6 words per lane).
KVQ_HD constexpr int piece_words(int words) { return words % 4 == 0 ? 4 : 2; }

// Byte offset of 32-bit word w of lane `lane` inside a code region whose
// lane blocks are interleaved in pieces of pw words.
KVQ_HD int code_word_offset(int lane, int w, int pw = 4) { return ((w / pw) * 32 + lane) * (4 * pw) + (w % pw) * 4; }

// f16 position of channel c inside the K scale array (keys stored before
// RoPE: the natural order, callers pass c itself).
KVQ_HD int kmeta_pos(int D, int c) {
  const int q = D / 4, t = c / q, r = c % q;
  return ((r >> 3) * 4 + t) * 8 + (r & 7);
}

// f16 position of channel c inside the K zero array: for k-step s the 16
// zeros of its MMA k-slots in k order (k = 2t + e + 8p holds channel
// t D/4 + 4s + 2p + e), so one row of 16 values is the zero-point operand.
KVQ_HD int kzero_pos(int D, int c) {
  const int q = D / 4, t = c / q, r = c % q;
  const int s = r >> 2, p = (r >> 1) & 1, e = r & 1;
  return s * 16 + 2 * t + e + 8 * p;
}

// f16 positions inside the V meta of token r, channel group vg (NV groups):
// the scales group by group, each group's 32 in the order the decode
// kernel's B operand wants them (token 8 kk + 2t + e at 8t + 2kk + e, so
// the lanes t of a group read 16 contiguous bytes holding the token pairs
// (2t, 2t + 1), (2t + 8, 2t + 9), ... in 32-bit words), then the zeros group
// by group in token order (one 32-bit word holds the zeros of two
// consecutive tokens of a group, the A operand of the zero-point MMA).
KVQ_HD int vscale_pos(int NV, int r, int vg) {
  (void)NV;
  return vg * 32 + 8 * ((r & 7) >> 1) + 2 * (r >> 3) + (r & 1);
}
KVQ_HD int vzero_pos(int NV, int r, int vg) { return 32 * NV + vg * 32 + r; }

// Word index and bit position of element f inside a lane block. Pair
// j = (f % per_word) / 2 of a word holds elements e = 0, 1 (f = 2P + e):
//   2-bit: byte j & 3, bits 2 (j >> 2) + 4 e   (an e2m1 nibble pair per byte
//          after masking with 0x33 at shift 0 or 2)
//   4-bit: half j & 1, bits 16 (j & 1) + 4 (j >> 1) + 8 e   (an e4m3 byte
//          pair per half after masking with 0x0F at shift 0 or 4)
//   8-bit: bits 8 j + 16 e
KVQ_HD void frag_bits(int bits, int f, int* word, int* bit) {
  const int per_word = 32 / bits;
  const int w = f / per_word, i = f % per_word, j = i >> 1, e = i & 1;
  *word = w;
  if (bits == 2) *bit = 8 * (j & 3) + 2 * (j >> 2) + 4 * e;
  else if (bits == 4) *bit = 16 * (j & 1) + 4 * (j >> 1) + 8 * e;
  else *bit = 8 * j + 16 * e;
}

// 3-bit fragment blocks: element i (0 .. 31) of a block of three words
// w0, w1, w2. Pair j = i / 2 (element e = i % 2) lies in quad q = j / 2 at
// byte k = 2 (j % 2) + e of the quad's 32-bit value, which holds one code in
// the low three bits of each byte:
//   q 0..5: word q / 2, bits 8k + 3 (q % 2) .. +2 (quad = (w >> 3 (q % 2)) & 0x07070707)
//   q 6:    low two bits at w0 bits 8k + 6, 7; high bit at w2 bit 8k + 6
//   q 7:    low two bits at w1 bits 8k + 6, 7; high bit at w2 bit 8k + 7
// (quads 6 and 7 = ((w0 or w1) >> 6 & 0x03030303) | (w2 >> 4 or 5 & 0x04040404)).
KVQ_HD void frag3_put(uint32_t* w, int i, uint32_t code) {
  const int j = i >> 1, e = i & 1, q = j >> 1, k = 2 * (j & 1) + e;
  if (q < 6) {
    w[q >> 1] |= (code & 7u) << (8 * k + 3 * (q & 1));
  } else {
    w[q - 6] |= (code & 3u) << (8 * k + 6);
    w[2] |= ((code >> 2) & 1u) << (8 * k + 6 + (q - 6));
  }
}
KVQ_HD uint32_t frag3_get(const uint32_t* w, int i) {
  const int j = i >> 1, e = i & 1, q = j >> 1, k = 2 * (j & 1) + e;
  if (q < 6) return (w[q >> 1] >> (8 * k + 3 * (q & 1))) & 7u;
  return ((w[q - 6] >> (8 * k + 6)) & 3u) | (((w[2] >> (8 * k + 6 + (q - 6))) & 1u) << 2);
}

// TurboQuant K codes in fragment order. The A operand of scores^T = K q^T
// (m16n8k16, rows = tokens, k = channels in natural order): lane (g, t) of
// m-tile mt holds at k-step s the channel pairs (16 s + 2 t + 8 p, +1) of
// the tokens 16 mt + g + 8 rh (p, rh in {0, 1}). One pair is one field (low
// code | high code << kb, 2 kb bits). A lane's fields form one bit string of
// D kb bits: four token blocks b = 2 mt + rh, each the D / 8 fields
// j = 2 s + p in order, so one token's fields in one lane are a run of whole
// bytes (D kb / 32 of them) and a writer of one token shares no byte with
// another token. The strings are interleaved across lanes in pieces like
// the KIVI words (byte k of lane L at lane_byte_offset(L, k, pw) with pw =
// piece_words(D kb / 32)).
KVQ_HD int tq_kfield_bit(int D, int kb, int b, int j) { return (b * (D / 8) + j) * 2 * kb; }
KVQ_HD int lane_byte_offset(int lane, int k, int pw) { return code_word_offset(lane, k >> 2, pw) + (k & 3); }

// TurboQuant V codes in token-pair rows: pair row pi (tokens 2 pi, 2 pi + 1
// of the group, 16 rows per group) holds for every channel c one field (code
// of token 2 pi | code of token 2 pi + 1 << vb, 2 vb bits): the A-operand
// pair (channel c, tokens 2 pi, 2 pi + 1) of out^T = V^T p. The fields are in
// the order c' = (c mod 8) D / 8 + c / 8 of one little-endian bit string of
// D vb / 4 bytes, so the fields a decode lane g needs (channels g + 8 j) are
// one block of D vb / 32 bytes at byte (c mod 8) D vb / 32, read as a whole.
KVQ_HD constexpr int tq_vrow_bytes(int D, int vb) { return D * vb / 4; }
KVQ_HD int tq_vfield_bit(int D, int vb, int c) { return 2 * vb * ((c % 8) * (D / 8) + c / 8); }

// Arena geometry shared by every layer.
struct Geometry {
  int B, H, Hq, D, gqa;
  int mode_tq, kb, vb;
  int n_sink, window, evict_window, n_dyn;
  int rope_repos;     // StreamingLLM position re-encoding at read
  int v_q4_0;         // V in the symmetric q4_0 form (scale d, zero -8 d)
  int k_pre_rope;     // keys stored before RoPE, rotated when read
  int act_bf16;
  int64_t max_tokens;
  int n_slots;        // group chunks per (layer, b, h)
  int tail_cap;       // rows per (layer, b, h) in the tail ring (power of 2)
  int n_sink_slots;   // rows per (layer, b, h) in the sink buffer
  int max_splits;
  Chunk chunk;
  int64_t rope_max_pos;
  // byte offsets inside the arena
  size_t off_err, off_rope, off_signs, off_cbk, off_cbv, off_part_o, off_part_ml;
  size_t off_norms, off_cand_m, off_cand_p, n_cand_chunks;
  size_t off_layers, layer_bytes;
  size_t l_chunks, l_tail_k, l_tail_v, l_sink_k, l_sink_v, l_sink_pos, l_sink_m, l_sink_mask;
  size_t total;
};

}  // namespace kvq
