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

// Wait for phase `parity` of `bar` for at most about one second of SM clock.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) return false;
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

// The query of one GQA row at full precision: RoPE at position L - 1 when the
// cache applies it (float32, not rounded), then times log2(e) / sqrt(D).
__device__ __forceinline__ float query_value(const DecodeArgs& a, int b, int hq, int c) {
  const Geometry& G = a.geo;
  const int D = G.D, half = D / 2;
  const uint16_t* qrow = a.q + (static_cast<size_t>(b) * G.Hq + hq) * D;
  float x = act_to_float(qrow[c], G.act_bf16);
  if (a.tab.rope) {
    const int i = c < half ? c : c - half;
    const float y = act_to_float(qrow[c < half ? c + half : c - half], G.act_bf16);
    const float* tr = a.tab.rope + static_cast<size_t>(a.L - 1) * D;
    float ra, rb;
    if (c < half) rope_pair(x, y, tr[2 * i], tr[2 * i + 1], &ra, &rb), x = ra;
    else rope_pair(y, x, tr[2 * i], tr[2 * i + 1], &ra, &rb), x = rb;
  }
  return x * a.qscale;
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

// The exact pools of one (b, h): the sinks read from the sink buffer and the
// tail [F, L) read from the ring, at fp32 with the query at full precision.
// NW warps take the tokens in turn; lane l holds channels i*32 + l. `red`
// must hold NW * kMaxGqa * (D + 2) floats.
template <int D, int NW>
__device__ void exact_partition(const DecodeArgs& a, int b, int h, float* red) {
  constexpr int NS = D / 32;
  const Geometry& G = a.geo;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = G.gqa;
  float qv[kMaxGqa][NS];
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j)
#pragma unroll
    for (int i = 0; i < NS; ++i) qv[j][i] = (j < gq) ? query_value(a, b, h * gq + j, i * 32 + lane) : 0.0f;
  float m[kMaxGqa], l[kMaxGqa], o[kMaxGqa][NS];
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.0f;
#pragma unroll
    for (int i = 0; i < NS; ++i) o[j][i] = 0.0f;
  }
  const int bh = b * G.H + h;
  const int n_sink_items = G.n_dyn ? a.n_dyn_sel : a.n_sink_read;
  const int64_t n_tail = a.L - a.F;
  const int64_t n_items = n_sink_items + n_tail;
  for (int64_t it = warp; it < n_items; it += NW) {
    const uint16_t* kr;
    const uint16_t* vr;
    if (it < n_sink_items) {
      if (G.n_dyn && a.lay.sink_pos[b * kMaxSinks + it] >= a.F) continue;  // read from the tail
      const size_t t = (static_cast<size_t>(bh) * G.n_sink_slots + it) * D;
      kr = a.lay.sink_k + t;
      vr = a.lay.sink_v + t;
    } else {
      const int64_t pos = a.F + (it - n_sink_items);
      const size_t t = (static_cast<size_t>(bh) * G.tail_cap + (pos & (G.tail_cap - 1))) * D;
      kr = a.lay.tail_k + t;
      vr = a.lay.tail_v + t;
    }
    float kx[NS], vx[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      kx[i] = act_to_float(kr[i * 32 + lane], G.act_bf16);
      vx[i] = act_to_float(vr[i * 32 + lane], G.act_bf16);
    }
#pragma unroll
    for (int j = 0; j < kMaxGqa; ++j) {
      if (j >= gq) break;
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < NS; ++i) s = fmaf(qv[j][i], kx[i], s);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      const float mn = fmaxf(m[j], s);
      const float al = exp2f(m[j] - mn);
      const float p = exp2f(s - mn);
      l[j] = l[j] * al + p;
#pragma unroll
      for (int i = 0; i < NS; ++i) o[j][i] = fmaf(o[j][i], al, p * vx[i]);
      m[j] = mn;
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxGqa; ++j) {
    if (j >= gq) break;
    float* r = red + (warp * kMaxGqa + j) * (D + 2);
#pragma unroll
    for (int i = 0; i < NS; ++i) r[i * 32 + lane] = o[j][i];
    if (lane == 0) {
      r[D] = m[j];
      r[D + 1] = l[j];
    }
  }
  __syncthreads();
  write_partial<D, NW>(a, red, b, h, 0);
}

}  // namespace kvq
