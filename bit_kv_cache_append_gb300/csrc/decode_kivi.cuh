// Split-KV decode attention over the KIVI cache (internal template; the
// instantiations live in decode_d64.cu and decode_d128.cu).
//
// One CTA per (partition, kv head, sequence); 4 warps; every warp walks its
// own 32-token groups of the partition (group w, w+4, ...) with a private
// online-softmax state, and the CTA merges its warps into one partial
// (max, sum, unnormalised output) per query head. Partition n_splits is the
// exact pool (sinks and tail, exact_partition); the LSE merge kernel combines
// all partials.
//
// Per group, on the tensor cores (mma.sync m16n8k16, f16 in, f32 out):
//   scores^T [32 tokens x 8 cols] = codes_K [32 x D] . qt [D x 8]
//   out^T    [D x 8]             += codes_V^T [D x 32] . pt [32 x 8]
// with the KIVI scales folded into the small operand:
//   qt[c][j]  = q_j[c] * sK[c]            (K scale per channel of the group)
//   pt[t][j]  = p_j[t] * sV[t][c / 32]    (V scale per token and 32 channels;
//                                          one pt per V channel group)
// and the zero points added outside the MMA in fp32:
//   score_j[t] += sum_c q_j[c] zK[c];   out_j[c] += sum_t p_j[t] zV[t][c/32].
// The codes enter the MMA exactly (small integers in f16). The 8 MMA columns
// carry the up-to-4 GQA query heads twice: columns 0-3 the f16 value of the
// folded operand, columns 4-7 its f16 residual, so each product is formed at
// about 22 bits and the two halves are summed in fp32 afterwards.
//
// The group chunks (codes stored in fragment order, see kvq_layout.h) are
// staged into shared memory by 1-D bulk copies (cp.async.bulk) on an
// mbarrier, several stages deep per warp; every wait is bounded.
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
  static constexpr size_t smem_bytes() { return static_cast<size_t>(NW) * NST * CHUNK + NW * NST * 8; }
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
  float* red = reinterpret_cast<float*>(smem);

  const Geometry& G = a.geo;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (split == a.n_splits) {
    exact_partition<D>(a, b, h, red);
    return;
  }
  const unsigned full = 0xffffffffu;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int gq = G.gqa;
  const int jq = g & 3;               // query head of this lane's B column
  const bool col_lo = g >= 4;         // B column holds the residual part
  const bool row_lo = t >= 2;         // C columns 2t, 2t+1 hold residual parts
  const int j0 = 2 * (t & 1);         // query heads of the C columns: j0, j0 + 1

  float qv[D / 4];
#pragma unroll
  for (int c4 = 0; c4 < D / 4; ++c4)
    qv[c4] = (jq < gq) ? query_value(a, b, h * gq + jq, t * (D / 4) + c4) : 0.0f;

  const int64_t gs0 = a.g_begin + static_cast<int64_t>(split) * a.groups_per_split;
  const int64_t gend = a.g_begin + a.n_groups;
  const int64_t gs1 = gs0 + a.groups_per_split < gend ? gs0 + a.groups_per_split : gend;
  const int64_t my0 = gs0 + warp;
  const int cnt = (my0 < gs1) ? static_cast<int>((gs1 - my0 + NW - 1) / NW) : 0;
  uint8_t* stages = smem + warp * NST * CHUNK;
  uint64_t* wb = bars + warp * NST;
  const int bh = b * G.H + h;
  const uint8_t* chunk_base = a.lay.chunks + static_cast<size_t>(bh) * G.n_slots * CHUNK;

  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < NST; ++st) mbar_init(&wb[st], 1);
    mbar_fence_init();
  }
  __syncwarp();
  if (lane == 0) {
    for (int i = 0; i < NST && i < cnt; ++i) {
      const int64_t gg = my0 + static_cast<int64_t>(i) * NW;
      mbar_expect_tx(&wb[i], CHUNK);
      bulk_g2s(stages + i * CHUNK, chunk_base + static_cast<size_t>(gg % G.n_slots) * CHUNK, CHUNK, &wb[i]);
    }
  }

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
  float oacc[MV][4];
  float zacc[2][NVG];
#pragma unroll
  for (int m = 0; m < MV; ++m) oacc[m][0] = oacc[m][1] = oacc[m][2] = oacc[m][3] = 0.0f;
#pragma unroll
  for (int v = 0; v < NVG; ++v) zacc[0][v] = zacc[1][v] = 0.0f;

  int it = 0;
  bool failed = false;
  for (; it < cnt; ++it) {
    const int st = it % NST;
    const bool ok = mbar_wait_bounded(&wb[st], static_cast<uint32_t>((it / NST) & 1));
    if (__any_sync(full, !ok)) { failed = true; break; }
    const uint8_t* tile = stages + st * CHUNK;
    const int64_t gg = my0 + static_cast<int64_t>(it) * NW;
    const int slot = static_cast<int>(gg % G.n_slots);

    uint32_t kr[KW], vr[VW];
#pragma unroll
    for (int i = 0; i < KW / 4; ++i)
      *reinterpret_cast<uint4*>(&kr[4 * i]) = reinterpret_cast<const uint4*>(tile)[lane * (KW / 4) + i];
#pragma unroll
    for (int i = 0; i < VW / 4; ++i)
      *reinterpret_cast<uint4*>(&vr[4 * i]) = reinterpret_cast<const uint4*>(tile + T::VC)[lane * (VW / 4) + i];

    // Folded K operand (q times the channel's K scale) and the zero-point term.
    uint32_t bq[S][2];
    float bias = 0.0f;
    const uint4* kmeta = reinterpret_cast<const uint4*>(tile + T::KMETA) + t * (D / 16);
#pragma unroll
    for (int s = 0; s < S; ++s) {
      const uint4 m4 = kmeta[s];
      const float2 sz0 = h2_to_f2(m4.x), sz1 = h2_to_f2(m4.y), sz2 = h2_to_f2(m4.z), sz3 = h2_to_f2(m4.w);
      bias = fmaf(qv[4 * s + 0], sz0.y, bias);
      bias = fmaf(qv[4 * s + 1], sz1.y, bias);
      bias = fmaf(qv[4 * s + 2], sz2.y, bias);
      bias = fmaf(qv[4 * s + 3], sz3.y, bias);
      bq[s][0] = split_h2(qv[4 * s + 0] * sz0.x, qv[4 * s + 1] * sz1.x, col_lo);
      bq[s][1] = split_h2(qv[4 * s + 2] * sz2.x, qv[4 * s + 3] * sz3.x, col_lo);
    }
    bias += __shfl_xor_sync(full, bias, 1);
    bias += __shfl_xor_sync(full, bias, 2);
    const float bias0 = __shfl_sync(full, bias, 4 * j0);
    const float bias1 = __shfl_sync(full, bias, 4 * (j0 + 1));

    // scores^T = codes_K . qt, per 16-token half of the group
    float sc[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.0f;
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

    // Valid tokens: inside [qlo, F) and not a KVSink sink of this group.
    const int64_t p0 = gg * kGroup;
    uint32_t vbits = 0xffffffffu;
    if (p0 < a.qlo) vbits &= 0xffffffffu << static_cast<int>(a.qlo - p0);
    if (p0 + kGroup > a.F) vbits &= (1u << static_cast<int>(a.F - p0)) - 1u;
    if (G.n_dyn) vbits &= ~a.lay.sink_mask[b * G.n_slots + slot];

    float pr[2][2][2];  // [mt][row half][query]: scores, then probabilities
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float v = sc[mt][2 * r + q];
          v += __shfl_xor_sync(full, v, 2);  // value + residual columns
          const int tok = 16 * mt + g + 8 * r;
          const bool valid = ((vbits >> tok) & 1u) && (j0 + q < gq);
          pr[mt][r][q] = valid ? v + (q ? bias1 : bias0) : -INFINITY;
        }

#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float mx = fmaxf(fmaxf(pr[0][0][q], pr[0][1][q]), fmaxf(pr[1][0][q], pr[1][1][q]));
      mx = fmaxf(mx, __shfl_xor_sync(full, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(full, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(full, mx, 16));
      const float mn = fmaxf(m_run[q], mx);
      const float al = (mn == -INFINITY) ? 1.0f : exp2f(m_run[q] - mn);
      float ps = 0.0f;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float p = (mn == -INFINITY) ? 0.0f : exp2f(pr[mt][r][q] - mn);
          pr[mt][r][q] = p;
          ps += p;
        }
      l_run[q] = l_run[q] * al + ps;
      m_run[q] = mn;
#pragma unroll
      for (int m = 0; m < MV; ++m) {
        oacc[m][q] *= al;
        oacc[m][2 + q] *= al;
      }
#pragma unroll
      for (int v = 0; v < NVG; ++v) zacc[q][v] *= al;
    }

    // out^T += codes_V^T . pt, one folded pt per V channel group
    float2 vsz[2][2][NVG];
    const uint32_t* vmeta = reinterpret_cast<const uint32_t*>(tile + T::VMETA);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int tok = 16 * mt + g + 8 * r;
#pragma unroll
        for (int v = 0; v < NVG; ++v) vsz[mt][r][v] = h2_to_f2(vmeta[tok * NVG + v]);
      }
#pragma unroll
    for (int v = 0; v < NVG; ++v) {
      uint32_t R[2][2];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float2 sz = vsz[mt][r][v];
          R[mt][r] = split_h2(pr[mt][r][0] * sz.x, pr[mt][r][1] * sz.x, row_lo);
          zacc[0][v] = fmaf(pr[mt][r][0], sz.y, zacc[0][v]);
          zacc[1][v] = fmaf(pr[mt][r][1], sz.y, zacc[1][v]);
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
    if (lane == 0 && it + NST < cnt) {
      const int64_t gn = my0 + static_cast<int64_t>(it + NST) * NW;
      mbar_expect_tx(&wb[st], CHUNK);
      bulk_g2s(stages + st * CHUNK, chunk_base + static_cast<size_t>(gn % G.n_slots) * CHUNK, CHUNK, &wb[st]);
    }
  }
  if (failed) {
    if (lane == 0) set_error(a.tab.err_flag, kErrTimeout);
    // let the copies still in flight land before the shared memory is reused
    for (int i = it; i < cnt && i < it + NST; ++i) (void)mbar_wait_bounded(&wb[i % NST], static_cast<uint32_t>((i / NST) & 1));
  }

#pragma unroll
  for (int q = 0; q < 2; ++q) {
    l_run[q] += __shfl_xor_sync(full, l_run[q], 4);
    l_run[q] += __shfl_xor_sync(full, l_run[q], 8);
    l_run[q] += __shfl_xor_sync(full, l_run[q], 16);
#pragma unroll
    for (int v = 0; v < NVG; ++v) {
      zacc[q][v] += __shfl_xor_sync(full, zacc[q][v], 4);
      zacc[q][v] += __shfl_xor_sync(full, zacc[q][v], 8);
      zacc[q][v] += __shfl_xor_sync(full, zacc[q][v], 16);
    }
  }
#pragma unroll
  for (int m = 0; m < MV; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[m][e] += __shfl_xor_sync(full, oacc[m][e], 2);

  __syncthreads();  // every warp is done with its stages: reuse them as `red`
  float* rw = red + warp * kMaxGqa * (D + 2);
  if (t < 2) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int j = j0 + q;
      if (j < gq) {
        float* rj = rw + j * (D + 2);
#pragma unroll
        for (int m = 0; m < MV; ++m) {
          rj[16 * m + g] = oacc[m][q] + zacc[q][m / 2];
          rj[16 * m + g + 8] = oacc[m][2 + q] + zacc[q][m / 2];
        }
        if (g == 0) {
          rj[D] = m_run[q];
          rj[D + 1] = l_run[q];
        }
      }
    }
  }
  __syncthreads();
  write_partial<D, NW>(a, red, b, h, split);
}

template <int D, int KB, int VB>
cudaError_t launch_kivi_instance(const DecodeArgs& a, cudaStream_t s) {
  using T = KiviTile<D, KB, VB>;
  const size_t smem = T::smem_bytes();
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(decode_kivi_kernel<D, KB, VB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  dim3 grid(a.n_splits + 1, a.geo.H, a.geo.B);
  decode_kivi_kernel<D, KB, VB><<<grid, 128, smem, s>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_kivi_d(const DecodeArgs& a, cudaStream_t s) {
  const int kb = a.geo.kb, vb = a.geo.vb;
#define KVQ_CASE(K, V) \
  if (kb == K && vb == V) return launch_kivi_instance<D, K, V>(a, s);
  KVQ_CASE(2, 2) KVQ_CASE(2, 4) KVQ_CASE(2, 8)
  KVQ_CASE(4, 2) KVQ_CASE(4, 4) KVQ_CASE(4, 8)
  KVQ_CASE(8, 2) KVQ_CASE(8, 4) KVQ_CASE(8, 8)
#undef KVQ_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kvq
