// Pieces shared by the decode kernels (internal): PTX wrappers for bulk
// copies, mbarriers, tensor-core MMA and movmatrix; the query prologue; the
// exact-pool partition (sinks and tail) and the per-CTA partial write.
#pragma once

#include "kvq_device.cuh"

namespace kvq {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Test for completion of phase `parity`; a thread whose phase is not complete
// may be suspended for up to about a microsecond before the call returns
// false, so waiting loops spin slowly.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000u)
      : "memory");
  return ok != 0;
}

// Non-blocking test for completion of phase `parity`.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` for at most `budget` SM clock cycles
// (about one second by default).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long budget = kWaitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > budget) return false;
  }
  return true;
}

// 1-D bulk copy global -> shared (both 16-byte aligned, size a multiple of 16)
// completing on `bar` with a transaction count.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// bulk_g2s with its transaction count armed on `bar`, both done only where
// `pred` holds: predicated instructions, so a warp whose lane 0 issues for
// it does not diverge.
__device__ __forceinline__ void bulk_g2s_if(bool pred, void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%3], %2;\n\t"
      "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "r"(static_cast<int>(pred))
      : "memory");
}

// The transaction count of a coming copy armed on `bar` (with this thread's
// arrival), and a 1-D bulk copy completing on `bar`: each done only where
// `pred` holds (predicated instructions, no divergence).
__device__ __forceinline__ void expect_tx_if(bool pred, uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %2, 0;\n\t"
      "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes), "r"(static_cast<int>(pred))
      : "memory");
}
__device__ __forceinline__ void copy_g2s_if(bool pred, void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "r"(static_cast<int>(pred))
      : "memory");
}

// D += A B with A 16x16 f16 (row), B 16x8 f16 (col), D 16x8 f32.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four 8x8 b16 matrices from shared memory into the MMA A-fragment layout;
// lane L gives the address of row L % 8 of matrix L / 8.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* row_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(row_addr)));
}

// 2^x by the hardware approximation (relative error about 2^-22; -inf -> 0),
// enough for softmax weights.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch: a split kernel lets the merge kernel that
// follows it on the stream be scheduled early (its exact pools do not read
// the partials), and the merge kernel waits for the split kernel's completion
// and memory before it reads them. Without the launch attribute the wait is
// a no-op.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Barrier `id` (1..15) over the first `threads` threads of the CTA.
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// A value the compiler must keep in a register (it cannot re-derive it).
__device__ __forceinline__ uint32_t pin(uint32_t x) {
  uint32_t y;
  asm volatile("mov.b32 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Transpose of an 8x8 b16 matrix held one b32 per lane in the MMA layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t x) {
  return __half22float2(*reinterpret_cast<__half2*>(&x));
}

// f16x2 of two fp32 values split as hi + lo: lanes that own a "lo" column of
// the MMA get the residual x - f32(f16(x)), the others get f16(x).
__device__ __forceinline__ uint32_t split_h2(float x0, float x1, bool lo) {
  const uint32_t h = f2_to_h2(x0, x1);
  if (!lo) return h;
  const float2 hf = h2_to_f2(h);
  return f2_to_h2(__fsub_rn(x0, hf.x), __fsub_rn(x1, hf.y));
}

// The query of one GQA row at full precision: RoPE at position qpos (L - 1
// unless keys are re-positioned) when the cache applies it (float32, not
// rounded), then times log2(e) / sqrt(D).
__device__ __forceinline__ float query_value(const DecodeArgs& a, int b, int hq, int c, int64_t qpos = -1) {
  const Geometry& G = a.geo;
  const int D = G.D, half = D / 2;
  const uint16_t* qrow = a.q + (static_cast<size_t>(b) * G.Hq + hq) * D;
  float x = act_to_float(qrow[c], G.act_bf16);
  if (a.tab.rope) {
    const int i = c < half ? c : c - half;
    const float y = act_to_float(qrow[c < half ? c + half : c - half], G.act_bf16);
    const float* tr = a.tab.rope + static_cast<size_t>(qpos >= 0 ? qpos : a.L - 1) * D;
    float ra, rb;
    if (c < half) rope_pair(x, y, tr[2 * i], tr[2 * i + 1], &ra, &rb), x = ra;
    else rope_pair(y, x, tr[2 * i], tr[2 * i + 1], &ra, &rb), x = rb;
  }
  return x * a.qscale;
}

// The channel pair (c0, c0 + 1), c0 even, of a query row times `scale`,
// RoPE'd at position qpos (query_value's arithmetic element by element when
// scale is a.qscale and qpos is L - 1): one 32-bit load of the pair (q must
// be 4-byte aligned) and, with RoPE, of its rotation partner and one 16-byte
// load of the two table entries.
__device__ __forceinline__ float2 query_pair(const DecodeArgs& a, int b, int hq, int c0, float scale,
                                             int64_t qpos) {
  const Geometry& G = a.geo;
  const int D = G.D, half = D / 2;
  const uint16_t* qrow = a.q + (static_cast<size_t>(b) * G.Hq + hq) * D;
  const uint32_t xw = *reinterpret_cast<const uint32_t*>(qrow + c0);
  float x0 = act_to_float(static_cast<uint16_t>(xw & 0xffffu), G.act_bf16);
  float x1 = act_to_float(static_cast<uint16_t>(xw >> 16), G.act_bf16);
  if (a.tab.rope) {
    const bool lo = c0 < half;
    const int i = lo ? c0 : c0 - half;
    const uint32_t yw = *reinterpret_cast<const uint32_t*>(qrow + (lo ? c0 + half : c0 - half));
    const float y0 = act_to_float(static_cast<uint16_t>(yw & 0xffffu), G.act_bf16);
    const float y1 = act_to_float(static_cast<uint16_t>(yw >> 16), G.act_bf16);
    const float4 tr = *reinterpret_cast<const float4*>(a.tab.rope + static_cast<size_t>(qpos) * D + 2 * i);
    float ra, rb;
    if (lo) {
      rope_pair(x0, y0, tr.x, tr.y, &ra, &rb), x0 = ra;
      rope_pair(x1, y1, tr.z, tr.w, &ra, &rb), x1 = ra;
    } else {
      rope_pair(y0, x0, tr.x, tr.y, &ra, &rb), x0 = rb;
      rope_pair(y1, x1, tr.z, tr.w, &ra, &rb), x1 = rb;
    }
  }
  return make_float2(x0 * scale, x1 * scale);
}

// Per-warp online-softmax states of one CTA merged through shared memory and
// written as partial `slot` of each of the G query heads: m (log2 units), l,
// and the unnormalised output o[D]. NW warps do the writing; `red` holds
// nrows * kMaxGqa * (D + 2) floats: [w][j][0..D-1] = o, [w][j][D] = m,
// [w][j][D+1] = l.
template <int D, int NW>
__device__ __forceinline__ void write_partial(const DecodeArgs& a, const float* red, int b, int h,
                                              int slot, int nrows = NW) {
  const Geometry& G = a.geo;
  const int ns = a.ns;
  for (int idx = threadIdx.x; idx < G.gqa * D; idx += NW * 32) {
    const int j = idx / D, c = idx % D;
    float M = -INFINITY;
    for (int w = 0; w < nrows; ++w) M = fmaxf(M, red[(w * kMaxGqa + j) * (D + 2) + D]);
    float o = 0.0f, l = 0.0f;
    if (M != -INFINITY) {
      for (int w = 0; w < nrows; ++w) {
        const float* r = red + (w * kMaxGqa + j) * (D + 2);
        const float sc = (r[D] == -INFINITY) ? 0.0f : exp2f(r[D] - M);
        o += r[c] * sc;
        l += r[D + 1] * sc;
      }
    }
    const size_t row = (static_cast<size_t>(b) * G.Hq + h * G.gqa + j) * ns + slot;
    a.part_o[row * D + c] = o;
    if (c == 0) {
      a.part_ml[row * 2 + 0] = M;
      a.part_ml[row * 2 + 1] = l;
    }
  }
}

// Walsh-Hadamard butterflies (stage length 1, 2, ..., D/2) over a vector held
// as lane l -> elements i*32 + l.
template <int D>
__device__ __forceinline__ void warp_fwht(float (&y)[D / 32]) {
  constexpr int NS = D / 32;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int len = 1; len < 32; len <<= 1) {
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, y[i], len);
      y[i] = (lane & len) ? o - y[i] : y[i] + o;
    }
  }
#pragma unroll
  for (int sl = 1; sl < NS; sl <<= 1) {
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      if ((i & sl) == 0) {
        const float u = y[i], v = y[i + sl];
        y[i] = u + v;
        y[i + sl] = u - v;
      }
    }
  }
}

// Bounded wait (`budget` SM clock cycles, about one second by default) that
// also gives up when another warp of the CTA has given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              long long budget = kWaitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// D += A B with A 16x16, B 16x8 of the activation type (bf16 or f16, the same
// for both operands), D 16x8 f32.
template <bool BF>
__device__ __forceinline__ void mma_act(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  if (BF)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    mma_f16(d, a0, a1, a2, a3, b0, b1);
}

// Four 8x8 b16 matrices, each stored as 8 rows of 16 bytes, transposed into
// the MMA A-fragment layout; lane L gives the address of row L % 8 of matrix
// L / 8.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void* row_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(row_addr)));
}

// Two floats as a pair of the activation type (x0 in the low half), rounded
// to nearest, and back.
template <bool BF>
__device__ __forceinline__ uint32_t pack_act2(float x0, float x1) {
  if (BF) {
    __nv_bfloat162 v = __floats2bfloat162_rn(x0, x1);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  return f2_to_h2(x0, x1);
}
template <bool BF>
__device__ __forceinline__ float2 unpack_act2(uint32_t x) {
  if (BF) return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&x));
  return h2_to_f2(x);
}

// A pair of the activation type holding x split as hi + lo: lanes that own a
// "lo" MMA column get the residual x - hi, the others hi.
template <bool BF>
__device__ __forceinline__ uint32_t split_act2(float x0, float x1, bool lo) {
  const uint32_t h = pack_act2<BF>(x0, x1);
  if (!lo) return h;
  const float2 hf = unpack_act2<BF>(h);
  return pack_act2<BF>(__fsub_rn(x0, hf.x), __fsub_rn(x1, hf.y));
}

// The exact pools of one (b, h) when keys are stored before RoPE: every
// row's key is rotated at its position (its cache slot: p below n_sink, else
// p - key_shift) in fp32 with the table and scored against the query (RoPE
// at q_pos, scale in) by warp dot products, values as stored. Warp w takes
// rows w, w + NW, ...; lane l holds channels l + 32 k, so the RoPE partners
// c and c + D/2 are in one lane. `qs` is shared memory for kMaxGqa * D
// floats. Leaves the warps' states in `red` like exact_states_tc.
template <int D, int NW>
__device__ void exact_states_prerope(const DecodeArgs& a, int b, int h, float* red, float* qs) {
  constexpr int NS = D / 32, HS = NS / 2;
  const unsigned full = 0xffffffffu;
  const Geometry& G = a.geo;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = G.gqa, bh = b * G.H + h;
  for (int idx = threadIdx.x; idx < gq * D; idx += NW * 32)
    qs[idx] = query_value(a, b, h * gq + idx / D, idx % D, a.q_pos);
  __syncthreads();
  const int n_sink_items = a.n_sink_read;
  const int n_items = n_sink_items + static_cast<int>(a.L - a.F);
  float m_run[kMaxGqa], l_run[kMaxGqa], o[kMaxGqa][NS];
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j) {
    m_run[j] = -INFINITY, l_run[j] = 0.0f;
#pragma unroll
    for (int k = 0; k < NS; ++k) o[j][k] = 0.0f;
  }
  for (int it = warp; it < n_items; it += NW) {
    int64_t pos;
    const uint16_t *krow, *vrow;
    if (it < n_sink_items) {
      pos = it;
      krow = a.lay.sink_k + (static_cast<size_t>(bh) * G.n_sink_slots + it) * D;
      vrow = a.lay.sink_v + (static_cast<size_t>(bh) * G.n_sink_slots + it) * D;
    } else {
      pos = a.F + (it - n_sink_items);
      const size_t off = (static_cast<size_t>(bh) * G.tail_cap + (pos & (G.tail_cap - 1))) * D;
      krow = a.lay.tail_k + off;
      vrow = a.lay.tail_v + off;
    }
    const int64_t kpos = pos < G.n_sink ? pos : pos - a.key_shift;
    const float* tr = a.tab.rope + static_cast<size_t>(kpos) * D;
    float k[NS], v[NS];
#pragma unroll
    for (int kk = 0; kk < NS; ++kk) {
      k[kk] = act_to_float(krow[kk * 32 + lane], G.act_bf16);
      v[kk] = act_to_float(vrow[kk * 32 + lane], G.act_bf16);
    }
#pragma unroll
    for (int kk = 0; kk < HS; ++kk) {  // channel i = lane + 32 kk and its partner i + D/2
      const float2 cs = *reinterpret_cast<const float2*>(tr + 2 * (lane + 32 * kk));
      float ra, rb;
      rope_pair(k[kk], k[kk + HS], cs.x, cs.y, &ra, &rb);
      k[kk] = ra, k[kk + HS] = rb;
    }
#pragma unroll
    for (int j = 0; j < kMaxGqa; ++j) {
      if (j >= gq) break;
      float d = 0.0f;
#pragma unroll
      for (int kk = 0; kk < NS; ++kk) d = fmaf(k[kk], qs[j * D + kk * 32 + lane], d);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) d += __shfl_xor_sync(full, d, off);
      const float mn = fmaxf(m_run[j], d);
      const float al = fast_exp2(m_run[j] - mn);  // 0 while nothing was seen
      const float p = fast_exp2(d - mn);
      m_run[j] = mn;
      l_run[j] = fmaf(l_run[j], al, p);
#pragma unroll
      for (int kk = 0; kk < NS; ++kk) o[j][kk] = fmaf(o[j][kk], al, p * v[kk]);
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j) {
    if (j >= gq) break;
    float* rj = red + (warp * kMaxGqa + j) * (D + 2);
#pragma unroll
    for (int kk = 0; kk < NS; ++kk) rj[kk * 32 + lane] = o[j][kk];
    if (lane == 0) {
      rj[D] = m_run[j];
      rj[D + 1] = l_run[j];
    }
  }
  __syncthreads();
}

// Rows per tile of the exact pools and the row capacity a stage of
// `stage_bytes` gives (whole tiles).
constexpr int kExactTile = 32;

// Warp-wide bounded wait for phase `parity` of `bar`: every decision is taken
// by warp votes, so the warp stays converged and the common case (the phase
// is already complete) costs one test and one vote. Gives up, raising the
// CTA's abort flag, after `budget` SM clock cycles (about one second by
// default) or as soon as another warp has raised it.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          long long budget = kWaitCycles) {
  const unsigned full = 0xffffffffu;
  if (__all_sync(full, mbar_test(bar, parity))) return true;
  const long long t0 = clock64();
  while (true) {
    if (__all_sync(full, mbar_try_wait(bar, parity))) return true;
    if (__any_sync(full, *abort_flag != 0)) return false;
    if (__any_sync(full, clock64() - t0 > budget)) {
      *abort_flag = 1;
      return false;
    }
  }
}

// The exact pools of one (b, h): the sinks read from the sink buffer and the
// tail [F, L) read from the ring, with the query at full precision (RoPE at
// L - 1 when the cache applies it). The rows are staged in shared memory:
// batches of sink and tail rows (K and V) are fetched by 1-D bulk copies
// (the tail ring in at most two contiguous runs) into `stage` (stage_bytes,
// 128-byte aligned, a whole number of 32-row tiles of K and V), the first
// batch requested before the query prologue. Each warp takes 32-row tiles in
// turn and runs them on the tensor cores in the activation type, straight
// from shared memory: scores^T = K_tile q^T with q split as hi + lo in the
// two columns of each query head (about 16 bits for bf16, 22 for f16), then
// an online softmax, then out^T += V_tile^T p^T with p split the same way.
// Each warp leaves its state in `red` (NW * kMaxGqa * (D + 2) floats:
// [w][j][0..D-1] = o, [w][j][D] = m in log2 units, [w][j][D+1] = l). `bar`
// is an mbarrier this function initialises; `abort_flag` is the CTA's shared
// give-up flag. Returns false (for every thread) when a wait gave up.
// REPOS: the cache re-positions RoPE (the sink rows are scored against the
// query rotated at sink_qpos); a separate instance so that the common one
// carries none of its registers.
template <int D, int NW, bool BF, bool REPOS>
__device__ bool exact_states_tc(const DecodeArgs& a, int b, int h, float* red, uint8_t* stage, int stage_bytes,
                                uint64_t* bar, volatile int* abort_flag) {
  constexpr int S = D / 16, MV = D / 16;
  constexpr int ROW = D * 2;  // bytes of one act-dtype row
  const unsigned full = 0xffffffffu;
  const Geometry& G = a.geo;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int gq = G.gqa;
  const int bh = b * G.H + h;
  const int n_sink_items = G.n_dyn ? a.n_dyn_sel : a.n_sink_read;
  const int n_items = n_sink_items + static_cast<int>(a.L - a.F);
  const int cap = stage_bytes / (2 * ROW);  // rows per batch, a multiple of kExactTile
  uint16_t* sk = reinterpret_cast<uint16_t*>(stage);
  uint16_t* sv = sk + static_cast<size_t>(cap) * D;
  // rows [i0, i1) of the item list (sinks, then the tail in position order)
  auto issue = [&](int i0, int i1) {
    mbar_expect_tx(bar, static_cast<uint32_t>((i1 - i0) * 2 * ROW));
    int r = i0;
    if (r < n_sink_items) {
      const int e = i1 < n_sink_items ? i1 : n_sink_items;
      const size_t off = (static_cast<size_t>(bh) * G.n_sink_slots + r) * D;
      bulk_g2s(sk + (r - i0) * D, a.lay.sink_k + off, (e - r) * ROW, bar);
      bulk_g2s(sv + (r - i0) * D, a.lay.sink_v + off, (e - r) * ROW, bar);
      r = e;
    }
    while (r < i1) {  // tail rows in ring order
      const int slot = static_cast<int>((a.F + (r - n_sink_items)) & (G.tail_cap - 1));
      const int n = (i1 - r) < (G.tail_cap - slot) ? (i1 - r) : (G.tail_cap - slot);
      const size_t off = (static_cast<size_t>(bh) * G.tail_cap + slot) * D;
      bulk_g2s(sk + (r - i0) * D, a.lay.tail_k + off, n * ROW, bar);
      bulk_g2s(sv + (r - i0) * D, a.lay.tail_v + off, n * ROW, bar);
      r += n;
    }
  };
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar, 1);
    mbar_fence_init();
    if (n_items > 0) issue(0, n_items < cap ? n_items : cap);
  }
  __syncthreads();
  // B operand of the scores: column g = query head g / 2, value (g even) or
  // residual (g odd); rows 2t, 2t + 1 and 2t + 8, 2t + 9 of k-step s are
  // channels 16 s + 2t (+1) and 16 s + 2t + 8 (+1).
  const int jc = g >> 1;
  const bool col_lo = g & 1;
  uint32_t qb[S][2];
#pragma unroll
  for (int s = 0; s < S; ++s)
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int c0 = 16 * s + 2 * t + 8 * p;
      const float2 x = jc < gq ? query_pair(a, b, h * gq + jc, c0, a.qscale, a.L - 1) : make_float2(0.0f, 0.0f);
      qb[s][p] = split_act2<BF>(x.x, x.y, col_lo);
    }
  float m_run = -INFINITY, l_run = 0.0f;  // of query head t (this lane's C columns)
  float oacc[MV][4];
#pragma unroll
  for (int m = 0; m < MV; ++m) oacc[m][0] = oacc[m][1] = oacc[m][2] = oacc[m][3] = 0.0f;
  uint32_t phase = 0;
  bool ok = true;
  for (int i0 = 0; i0 < n_items; i0 += cap) {
    const int i1 = i0 + cap < n_items ? i0 + cap : n_items;
    const int nb = i1 - i0;
    ok = ok && wait_or_abort(bar, phase, abort_flag);
    phase ^= 1;
    if (ok) {
      for (int tile = warp; tile * kExactTile < nb; tile += NW) {
        const int rb = tile * kExactTile;
        if (rb + kExactTile > nb) {
          // rows past the batch hold stale bytes: zero their V so that a zero
          // weight times them is zero
          for (int i = (nb - rb) * (ROW / 16) + lane; i < kExactTile * (ROW / 16); i += 32)
            reinterpret_cast<uint4*>(sv + static_cast<size_t>(rb) * D)[i] = make_uint4(0u, 0u, 0u, 0u);
          __syncwarp();
        }
        float sc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int s = 0; s < S; ++s) {
            uint32_t A[4];
            ldmatrix_x4(A, sk + static_cast<size_t>(rb + 16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1)) * D +
                               16 * s + 8 * (lane >> 4));
            mma_act<BF>(sc[mt], A[0], A[1], A[2], A[3], qb[s][0], qb[s][1]);
          }
        if (REPOS && i0 + rb < n_sink_items && a.sink_qpos != a.L - 1) {
          // re-positioning: the sink rows of this tile meet the query
          // rotated at sink_qpos; their scores again with that operand
          float ss[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll 1  // one tile per decode: kept rolled, it costs the instance no registers
          for (int s = 0; s < S; ++s) {
            uint32_t qs[2];
#pragma unroll
            for (int p = 0; p < 2; ++p) {
              const int c0 = 16 * s + 2 * t + 8 * p;
              const float2 x = jc < gq ? query_pair(a, b, h * gq + jc, c0, a.qscale, a.sink_qpos)
                                       : make_float2(0.0f, 0.0f);
              qs[p] = split_act2<BF>(x.x, x.y, col_lo);
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              uint32_t A[4];
              ldmatrix_x4(A, sk + static_cast<size_t>(rb + 16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1)) * D +
                                 16 * s + 8 * (lane >> 4));
              mma_act<BF>(ss[mt], A[0], A[1], A[2], A[3], qs[0], qs[1]);
            }
          }
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (i0 + rb + 16 * mt + g + 8 * (e >> 1) < n_sink_items) sc[mt][e] = ss[mt][e];
        }
        float pr[2][2];
        float mx = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int it = i0 + rb + 16 * mt + g + 8 * r;
            bool valid = (it < i1) && (t < gq);
            if (valid && it < n_sink_items && G.n_dyn && a.lay.sink_pos[b * kMaxSinks + it] >= a.F)
              valid = false;  // a KVSink sink still in the tail is read there
            pr[mt][r] = valid ? sc[mt][2 * r] + sc[mt][2 * r + 1] : -INFINITY;
            mx = fmaxf(mx, pr[mt][r]);
          }
        mx = fmaxf(mx, __shfl_xor_sync(full, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(full, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(full, mx, 16));
        const float mn = fmaxf(m_run, mx);
        const float mref = (mn == -INFINITY) ? 0.0f : mn;
        const float al = fast_exp2(m_run - mref);  // 0 while nothing was valid
        m_run = mn;
        l_run *= al;
#pragma unroll
        for (int m = 0; m < MV; ++m) {
          oacc[m][0] *= al;
          oacc[m][1] *= al;
          oacc[m][2] *= al;
          oacc[m][3] *= al;
        }
        uint32_t R[4];  // weights of rows g (+8) of m-tile mt as (value, residual) in the C layout
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float p = fast_exp2(pr[mt][r] - mref);
            l_run += p;
            const uint32_t hv = pack_act2<BF>(p, 0.0f);
            const float ph = unpack_act2<BF>(hv).x;
            R[mt * 2 + r] = pack_act2<BF>(ph, __fsub_rn(p, ph));
          }
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint32_t b0 = movmatrix_t(R[2 * kb]);
          const uint32_t b1 = movmatrix_t(R[2 * kb + 1]);
#pragma unroll
          for (int m = 0; m < MV; ++m) {
            uint32_t A[4];
            ldmatrix_x4_trans(A, sv + static_cast<size_t>(rb + 16 * kb + 8 * (lane >> 4) + (lane & 7)) * D +
                                     16 * m + 8 * ((lane >> 3) & 1));
            mma_act<BF>(oacc[m], A[0], A[1], A[2], A[3], b0, b1);
          }
        }
      }
    }
    ok = __syncthreads_and(ok);  // the batch is consumed (and the verdict shared) before the next copy
    if (!ok) break;
    if (threadIdx.x == 0 && i1 < n_items) issue(i1, i1 + cap < n_items ? i1 + cap : n_items);
  }
  if (!ok) {
    // copies of the failed batch may still be in flight: let them land
    if (threadIdx.x == 0) (void)mbar_wait_bounded(bar, phase ^ 1);
    __syncthreads();
  }
  l_run += __shfl_xor_sync(full, l_run, 4);
  l_run += __shfl_xor_sync(full, l_run, 8);
  l_run += __shfl_xor_sync(full, l_run, 16);
  if (t < gq) {
    float* rj = red + (warp * kMaxGqa + t) * (D + 2);
#pragma unroll
    for (int m = 0; m < MV; ++m) {
      rj[16 * m + g] = oacc[m][0] + oacc[m][1];
      rj[16 * m + g + 8] = oacc[m][2] + oacc[m][3];
    }
    if (g == 0) {
      rj[D] = m_run;
      rj[D + 1] = l_run;
    }
  }
  __syncthreads();
  return ok;
}

}  // namespace kvq
