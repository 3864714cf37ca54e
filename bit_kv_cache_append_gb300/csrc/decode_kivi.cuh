// Split-KV decode attention over the KIVI cache (internal template; the
// instantiations live in decode_d64.cu and decode_d128.cu).
//
// Work decomposition (stream-K): the quantised segment of every (sequence,
// KV head) unit is a run of 32-token groups; all units' groups form one flat
// list that is cut into n_ctas equal contiguous ranges, one per persistent
// CTA (n_ctas a multiple of the SM count). A CTA walks its range unit by
// unit; for each unit it touches, its 4 warps take the unit's groups in turn
// (w, w+4, ...) with private online-softmax states that the CTA merges into
// one partial (max, sum, unnormalised output) per query head. The first
// B*Hkv CTAs instead handle the exact pools of one unit each (sinks and
// tail, exact_partition). The LSE merge kernel combines every partial of a
// (sequence, query head).
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
// The codes enter the MMA exactly (small integers in f16). The 8 MMA columns
// hold, for query head j, column 2j = the f16 value of the folded operand
// and column 2j+1 its f16 residual, so each product is carried at about 22
// bits and thread (g, t) of the C fragment owns query head t. The residual
// of q * sK is formed exactly in f16 (an FMA returns q_hi * s - f16(q_hi * s)
// without rounding), so building the operand costs four f16x2 instructions
// per register.
//
// The group chunks (codes stored in fragment order, see kvq_layout.h) are
// staged into shared memory by 1-D bulk copies (cp.async.bulk) on an
// mbarrier, several stages deep per warp, prefetching across unit
// boundaries; every wait is bounded.
#pragma once

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

// Pair j of a packed word (elements at bits BITS*j and BITS*j + 16) as an
// exact f16x2 of the two codes. The code bits are OR-ed into the mantissa of
// 1024.0 (0x6400), giving 1024 + c * 2^k exactly, and one f16x2 FMA by
// 2^-k and -1024 * 2^-k leaves c exactly.
template <int BITS>
__device__ __forceinline__ uint32_t code_pair(uint32_t w, int j) {
  if (BITS == 2) {
    const int jj = j < 5 ? j : j - 5;
    const uint32_t x = j < 5 ? w : (w >> 10);
    const uint32_t hv = (x & (0x00030003u << (2 * jj))) | 0x64006400u;
    return hfma2_bits(hv, h2pow2(-2 * jj), h2negpow2(10 - 2 * jj));
  } else if (BITS == 4) {
    const int jj = j < 2 ? j : j - 2;
    const uint32_t x = j < 2 ? w : (w >> 8);
    const uint32_t hv = (x & (0x000F000Fu << (4 * jj))) | 0x64006400u;
    return hfma2_bits(hv, h2pow2(-4 * jj), h2negpow2(10 - 4 * jj));
  } else {
    const uint32_t hv = __byte_perm(w, 0x6464u, static_cast<uint32_t>(j | 0x40 | ((j + 2) << 8) | 0x4000));
    return hfma2_bits(hv, h2pow2(0), h2negpow2(10));
  }
}

template <int D, int KB, int VB>
struct KiviTile {
  static constexpr int KC = 32 * D * KB / 8;
  static constexpr int KMETA = KC;
  static constexpr int VC = KMETA + 4 * D;
  static constexpr int VMETA = VC + 32 * D * VB / 8;
  static constexpr int CHUNK = VMETA + 4 * D;
  static constexpr int NST = CHUNK <= 6144 ? 3 : 2;  // bulk-copy stages per warp
  static constexpr int NW = 4;
  static constexpr int RED_FLOATS = NW * kMaxGqa * (D + 2);
  static constexpr size_t smem_bytes() {
    return static_cast<size_t>(NW) * NST * CHUNK + NW * NST * 8 + RED_FLOATS * 4;
  }
};

// CTA that owns flattened item i under the equal split of `work` items into
// `n` ranges [floor(c work / n), floor((c+1) work / n)).
__device__ __forceinline__ int owner_cta(int64_t i, int64_t work, int n) {
  return static_cast<int>(((i + 1) * n - 1) / work);
}

// Walks the items of warp w inside its CTA's range [i0, i1): per unit (run of
// ng items), the unit's items s + w, s + w + 4, ... where s is the first item
// of the unit inside the range. The group index and its ring slot advance by
// additions; divisions happen only when the walk enters a new unit.
struct ItemCursor {
  int64_t item;      // current item (-1: exhausted)
  int64_t seg_end;   // end of the current unit inside the range
  int64_t unit;
  int64_t grp;       // absolute group index of `item`
  int slot;          // grp mod n_slots

  __device__ __forceinline__ void enter(int64_t s, int64_t i1, int64_t ng, int w, int64_t g_begin, int n_slots) {
    while (s < i1) {
      const int64_t u = s / ng;
      const int64_t e = (u + 1) * ng < i1 ? (u + 1) * ng : i1;
      if (s + w < e) {
        item = s + w;
        seg_end = e;
        unit = u;
        grp = g_begin + (item - u * ng);
        slot = static_cast<int>(grp % n_slots);
        return;
      }
      s = e;
    }
    item = -1;
  }
  __device__ __forceinline__ void advance(int64_t i1, int64_t ng, int w, int64_t g_begin, int n_slots) {
    if (item + 4 < seg_end) {
      item += 4;
      grp += 4;
      slot += 4;
      while (slot >= n_slots) slot -= n_slots;
    } else {
      enter(seg_end, i1, ng, w, g_begin, n_slots);
    }
  }
};

template <int D, int KB, int VB>
__global__ void __launch_bounds__(128, 3) decode_kivi_kernel(DecodeArgs a) {
  using T = KiviTile<D, KB, VB>;
  constexpr int NW = T::NW, NST = T::NST, CHUNK = T::CHUNK;
  constexpr int S = D / 16, MV = D / 16, NVG = D / 32;
  constexpr int KW = D * KB / 32, VW = D * VB / 32;
  constexpr int KPPW = 16 / KB, VPPW = 16 / VB;  // code pairs per 32-bit word
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * NST * CHUNK);
  float* red = reinterpret_cast<float*>(smem + NW * NST * CHUNK + NW * NST * 8);

  const Geometry& G = a.geo;
  const int n_exact = G.B * G.H;
  if (static_cast<int>(blockIdx.x) < n_exact) {
    exact_partition<D>(a, blockIdx.x / G.H, blockIdx.x % G.H, red);
    return;
  }
  const unsigned full = 0xffffffffu;
  const int cta = blockIdx.x - n_exact;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int gq = G.gqa;
  const int jc = g >> 1;          // query head of this lane's B column
  const bool col_lo = g & 1;      // B column holds the residual part
  const int64_t ng = a.n_groups, work = a.work;
  const int64_t i0 = cta * work / a.n_ctas, i1 = (cta + 1) * work / a.n_ctas;

  uint8_t* stages = smem + warp * NST * CHUNK;
  uint64_t* wb = bars + warp * NST;
  const int n_slots = G.n_slots;
  auto chunk_src = [&](const ItemCursor& c) {
    return a.lay.chunks + (static_cast<size_t>(c.unit) * n_slots + c.slot) * CHUNK;
  };
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < NST; ++st) mbar_init(&wb[st], 1);
    mbar_fence_init();
  }
  __syncwarp();
  ItemCursor pc;  // producer: the next item whose chunk is to be fetched
  pc.enter(i0, i1, ng, warp, a.g_begin, n_slots);
  int issued = 0, consumed = 0;
  if (lane == 0) {
    for (int i = 0; i < NST && pc.item >= 0; ++i) {
      mbar_expect_tx(&wb[i], CHUNK);
      bulk_g2s(stages + i * CHUNK, chunk_src(pc), CHUNK, &wb[i]);
      pc.advance(i1, ng, warp, a.g_begin, n_slots);
      ++issued;
    }
  }
  bool failed = false;

  int64_t seg = i0;
  while (seg < i1) {
    const int64_t unit = seg / ng;
    const int64_t seg_e = (unit + 1) * ng < i1 ? (unit + 1) * ng : i1;
    const int b = static_cast<int>(unit / G.H), h = static_cast<int>(unit % G.H);
    int64_t grp = a.g_begin + (seg - unit * ng) + warp;   // group of this warp's first item
    int slot = static_cast<int>(grp % n_slots);

    // query of this lane's B column at full precision, split as f16 hi + lo,
    // for the lane's quarter of the channels (pairs of adjacent channels)
    uint32_t qh[S][2], qa[S][2];
#pragma unroll
    for (int s = 0; s < S; ++s)
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int c0 = t * (D / 4) + 4 * s + 2 * p;
        float x0 = 0.0f, x1 = 0.0f;
        if (jc < gq) {
          x0 = query_value(a, b, h * gq + jc, c0);
          x1 = query_value(a, b, h * gq + jc, c0 + 1);
        }
        const uint32_t hi = f2_to_h2(x0, x1);
        const float2 hf = h2_to_f2(hi);
        const uint32_t lo = f2_to_h2(x0 - hf.x, x1 - hf.y);
        qh[s][p] = hi;
        qa[s][p] = col_lo ? lo : hi;
      }

    float m_run = -INFINITY, l_run = 0.0f;
    float oacc[MV][4];
    float zacc[NVG];
#pragma unroll
    for (int m = 0; m < MV; ++m) oacc[m][0] = oacc[m][1] = oacc[m][2] = oacc[m][3] = 0.0f;
#pragma unroll
    for (int v = 0; v < NVG; ++v) zacc[v] = 0.0f;

    for (int64_t item = seg + warp; item < seg_e && !failed; item += 4) {
      const int st = consumed % NST;
      const bool ok = mbar_wait_bounded(&wb[st], static_cast<uint32_t>((consumed / NST) & 1));
      if (__any_sync(full, !ok)) {
        failed = true;
        break;
      }
      const uint8_t* tile = stages + st * CHUNK;

      uint32_t kr[KW], vr[VW];
#pragma unroll
      for (int i = 0; i < KW / 4; ++i)
        *reinterpret_cast<uint4*>(&kr[4 * i]) = reinterpret_cast<const uint4*>(tile)[i * 32 + lane];
#pragma unroll
      for (int i = 0; i < VW / 4; ++i)
        *reinterpret_cast<uint4*>(&vr[4 * i]) = reinterpret_cast<const uint4*>(tile + T::VC)[i * 32 + lane];

      // scores^T: zero-point row first, then codes_K . qt
      float sc[2][4];
      {
        const uint4* ks = reinterpret_cast<const uint4*>(tile + T::KMETA);
        const uint4* kz = reinterpret_cast<const uint4*>(tile + T::KMETA + 2 * D);
        uint32_t bq[S][2];
        float zb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int u = 0; u < S / 2; ++u) {
          const uint4 s4 = ks[u * 4 + t];
          const uint4 z4 = kz[u * 4 + t];
          const uint32_t sp[4] = {s4.x, s4.y, s4.z, s4.w};
          const uint32_t zp[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
          for (int hlf = 0; hlf < 2; ++hlf) {
            const int s = 2 * u + hlf;
#pragma unroll
            for (int p = 0; p < 2; ++p) {
              const __half2 sv = as_h2(sp[2 * hlf + p]);
              const __half2 x = __hmul2(as_h2(qh[s][p]), sv);
              const __half2 y = __hfma2(as_h2(qh[s][p]), sv, __hneg2(x));
              const __half2 z = __hfma2(as_h2(qa[s][p]), sv, y);
              bq[s][p] = col_lo ? as_u32(z) : as_u32(x);
            }
            mma_f16(zb, zp[2 * hlf], zp[2 * hlf], zp[2 * hlf + 1], zp[2 * hlf + 1], qa[s][0], qa[s][1]);
          }
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[mt][e] = zb[e];
#pragma unroll
          for (int s = 0; s < S; ++s) {
            const int pb = (mt * S + s) * 4;
            const uint32_t a0 = code_pair<KB>(kr[(pb + 0) / KPPW], (pb + 0) % KPPW);
            const uint32_t a1 = code_pair<KB>(kr[(pb + 1) / KPPW], (pb + 1) % KPPW);
            const uint32_t a2 = code_pair<KB>(kr[(pb + 2) / KPPW], (pb + 2) % KPPW);
            const uint32_t a3 = code_pair<KB>(kr[(pb + 3) / KPPW], (pb + 3) % KPPW);
            mma_f16(sc[mt], a0, a1, a2, a3, bq[s][0], bq[s][1]);
          }
        }
      }

      // valid tokens: inside [qlo, F) and not a KVSink sink of this group
      const int64_t p0 = grp * kGroup;
      uint32_t vbits = 0xffffffffu;
      if (p0 < a.qlo) vbits &= 0xffffffffu << static_cast<int>(a.qlo - p0);
      if (p0 + kGroup > a.F) vbits &= (1u << static_cast<int>(a.F - p0)) - 1u;
      if (G.n_dyn) vbits &= ~a.lay.sink_mask[b * G.n_slots + slot];
      const bool qvalid = t < gq;

      float pr[2][2];  // [mt][row half]: scores, then probabilities
      float mx = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int tok = 16 * mt + g + 8 * r;
          const float v = sc[mt][2 * r] + sc[mt][2 * r + 1];
          pr[mt][r] = (qvalid && ((vbits >> tok) & 1u)) ? v : -INFINITY;
          mx = fmaxf(mx, pr[mt][r]);
        }
      mx = fmaxf(mx, __shfl_xor_sync(full, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(full, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(full, mx, 16));
      // lazy rescaling: keep the running max unless the tile exceeds it by
      // more than 2^8, so probabilities stay below 256 (exact either way)
      const bool grow = mx > m_run + 8.0f;
      if (__any_sync(full, grow)) {
        const float mn = grow ? mx : m_run;
        const float al = (m_run == -INFINITY) ? 0.0f : exp2f(m_run - mn);
        l_run *= al;
#pragma unroll
        for (int m = 0; m < MV; ++m) {
          oacc[m][0] *= al;
          oacc[m][1] *= al;
          oacc[m][2] *= al;
          oacc[m][3] *= al;
        }
#pragma unroll
        for (int v = 0; v < NVG; ++v) zacc[v] *= al;
        m_run = mn;
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float p = (pr[mt][r] == -INFINITY) ? 0.0f : exp2f(pr[mt][r] - m_run);
          pr[mt][r] = p;
          l_run += p;
        }

      // out^T += codes_V^T . pt, one folded pt per V channel group
      // V scales and zeros of this thread's four tokens (NVG/2 f16x2 words of
      // scales, then NVG/2 of zeros, per token)
      __half2 vsp[2][2][NVG / 2], vzp[2][2][NVG / 2];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const __half2* row = reinterpret_cast<const __half2*>(tile + T::VMETA) + (16 * mt + g + 8 * r) * NVG;
#pragma unroll
          for (int i = 0; i < NVG / 2; ++i) {
            vsp[mt][r][i] = row[i];
            vzp[mt][r][i] = row[NVG / 2 + i];
          }
        }
#pragma unroll
      for (int v = 0; v < NVG; ++v) {
        uint32_t R[2][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const __half2 sp = vsp[mt][r][v >> 1], zp = vzp[mt][r][v >> 1];
            const float sv = (v & 1) ? __high2float(sp) : __low2float(sp);
            const float zv = (v & 1) ? __high2float(zp) : __low2float(zp);
            const float x = pr[mt][r] * sv;
            const __half hx = __float2half_rn(x);
            R[mt][r] = f2_to_h2(__half2float(hx), x - __half2float(hx));
            zacc[v] = fmaf(pr[mt][r], zv, zacc[v]);
          }
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint32_t b0 = movmatrix_t(R[kb][0]);
          const uint32_t b1 = movmatrix_t(R[kb][1]);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int m = 2 * v + hh;
            const int pb = (m * 2 + kb) * 4;
            const uint32_t a0 = code_pair<VB>(vr[(pb + 0) / VPPW], (pb + 0) % VPPW);
            const uint32_t a1 = code_pair<VB>(vr[(pb + 1) / VPPW], (pb + 1) % VPPW);
            const uint32_t a2 = code_pair<VB>(vr[(pb + 2) / VPPW], (pb + 2) % VPPW);
            const uint32_t a3 = code_pair<VB>(vr[(pb + 3) / VPPW], (pb + 3) % VPPW);
            mma_f16(oacc[m], a0, a1, a2, a3, b0, b1);
          }
        }
      }

      __syncwarp();
      ++consumed;
      if (lane == 0 && pc.item >= 0) {
        mbar_expect_tx(&wb[st], CHUNK);
        bulk_g2s(stages + st * CHUNK, chunk_src(pc), CHUNK, &wb[st]);
        pc.advance(i1, ng, warp, a.g_begin, n_slots);
        ++issued;
      }
      grp += 4;
      slot += 4;
      while (slot >= n_slots) slot -= n_slots;
    }
    issued = __shfl_sync(full, issued, 0);

    // warp state -> shared memory (thread (g, t) owns query t, rows g, g+8)
    l_run += __shfl_xor_sync(full, l_run, 4);
    l_run += __shfl_xor_sync(full, l_run, 8);
    l_run += __shfl_xor_sync(full, l_run, 16);
#pragma unroll
    for (int v = 0; v < NVG; ++v) {
      zacc[v] += __shfl_xor_sync(full, zacc[v], 4);
      zacc[v] += __shfl_xor_sync(full, zacc[v], 8);
      zacc[v] += __shfl_xor_sync(full, zacc[v], 16);
    }
    if (t < gq) {
      float* rj = red + (warp * kMaxGqa + t) * (D + 2);
#pragma unroll
      for (int m = 0; m < MV; ++m) {
        rj[16 * m + g] = oacc[m][0] + oacc[m][1] + zacc[m / 2];
        rj[16 * m + g + 8] = oacc[m][2] + oacc[m][3] + zacc[m / 2];
      }
      if (g == 0) {
        rj[D] = m_run;
        rj[D + 1] = l_run;
      }
    }
    __syncthreads();
    write_partial<D, NW>(a, red, b, h, 1 + cta - owner_cta(unit * ng, work, a.n_ctas));
    __syncthreads();
    seg = seg_e;
  }
  if (failed) {
    if (lane == 0) set_error(a.tab.err_flag, kErrTimeout);
    // let the copies still in flight land before the CTA exits
    for (int i = consumed; i < issued; ++i)
      (void)mbar_wait_bounded(&wb[i % NST], static_cast<uint32_t>((i / NST) & 1));
  }
}

template <int D, int KB, int VB>
cudaError_t launch_kivi_instance(DecodeArgs& a, cudaStream_t s, int sm_count) {
  using T = KiviTile<D, KB, VB>;
  const size_t smem = T::smem_bytes();
  static int occupancy = 0;
  if (!occupancy) {
    cudaError_t e = cudaFuncSetAttribute(decode_kivi_kernel<D, KB, VB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occupancy, decode_kivi_kernel<D, KB, VB>, 128, smem);
    if (e != cudaSuccess) return e;
    if (occupancy < 1) occupancy = 1;
  }
  // stream-K CTAs: fill the machine, never more than one per group, and at
  // most max_splits - 1 per unit (partial slots per query head)
  int64_t n = a.n_ctas_hint > 0 ? a.n_ctas_hint : static_cast<int64_t>(sm_count) * occupancy;
  const int64_t units = static_cast<int64_t>(a.geo.B) * a.geo.H;
  if (n > a.work) n = a.work;
  if (n > units * (a.geo.max_splits - 2)) n = units * (a.geo.max_splits - 2);
  if (n < 1) n = 1;
  a.n_ctas = static_cast<int>(n);
  const int n_exact = a.geo.B * a.geo.H;
  decode_kivi_kernel<D, KB, VB><<<n_exact + (a.work > 0 ? a.n_ctas : 0), 128, smem, s>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_kivi_d(DecodeArgs& a, cudaStream_t s, int sm_count) {
  const int kb = a.geo.kb, vb = a.geo.vb;
#define KVQ_CASE(K, V) \
  if (kb == K && vb == V) return launch_kivi_instance<D, K, V>(a, s, sm_count);
  KVQ_CASE(2, 2) KVQ_CASE(2, 4) KVQ_CASE(2, 8)
  KVQ_CASE(4, 2) KVQ_CASE(4, 4) KVQ_CASE(4, 8)
  KVQ_CASE(8, 2) KVQ_CASE(8, 4) KVQ_CASE(8, 8)
#undef KVQ_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kvq
