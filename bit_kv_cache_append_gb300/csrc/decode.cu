// The merge kernel (exact pools of each unit and the log-sum-exp merge of
// the partials) and the decode dispatch; the split kernels (KIVI and
// TurboQuant) are in decode_kivi.cuh.
#include "decode_common.cuh"

namespace kvq {

// The split kernels' launchers, instantiated in decode_d{64,128}_{k2,k3,k4,k8,tq}.cu.
template <int D, int K>
cudaError_t launch_kivi_k(DecodeArgs& a, cudaStream_t s, int sm_count);
template <int D>
cudaError_t launch_tq_d(DecodeArgs& a, cudaStream_t s, int sm_count);

template <int D>
cudaError_t launch_split(DecodeArgs& a, cudaStream_t s, int sm_count) {
  if (a.geo.mode_tq) return launch_tq_d<D>(a, s, sm_count);
  switch (a.geo.kb) {
    case 2: return launch_kivi_k<D, 2>(a, s, sm_count);
    case 3: return launch_kivi_k<D, 3>(a, s, sm_count);
    case 4: return launch_kivi_k<D, 4>(a, s, sm_count);
    case 8: return launch_kivi_k<D, 8>(a, s, sm_count);
    default: return cudaErrorInvalidValue;
  }
}

namespace {

// Number of partial slots of unit u: the stream-K CTAs whose item ranges
// meet the unit's items.
__device__ __forceinline__ int slots_of_unit(const DecodeArgs& a, int64_t u) {
  if (a.work <= 0 || a.n_groups <= 0) return 0;
  const int64_t first = u * a.n_groups, last = first + a.n_groups - 1;
  const int c0 = static_cast<int>(((first + 1) * a.n_ctas - 1) / a.work);
  const int c1 = static_cast<int>(((last + 1) * a.n_ctas - 1) / a.work);
  return c1 - c0 + 1;
}

constexpr int kMergeWarps = 8;

// Shared memory of the merge kernel: the row stage, the warps' exact states,
// an mbarrier and the abort flag.
template <int D>
size_t merge_smem_bytes(int stage_bytes) {
  return static_cast<size_t>(stage_bytes) + kMergeWarps * kMaxGqa * (D + 2) * 4 + 32;
}

// One CTA per (sequence, KV head) unit. First the unit's exact pools (sinks
// and tail), staged through shared memory and run on the tensor cores
// (exact_states_tc);
// then warp j < gqa combines, for query head j, the exact states with the
// split partials by log-sum-exp (M = max m, o = sum 2^(m - M) o / sum
// 2^(m - M) l) and writes the output and lse. In TurboQuant mode the split
// partials are in the rotated domain: their sum is rotated back
// (x = D FWHT(y) / sqrt(d)) before the exact part, which is in the original
// domain, is added (Foundry "TurboQuant KV Cache Compression - Spec",
// "Optimization: Fused dequant-dot": rotate the accumulated output once).
// XM: 0 the exact rows as stored, 1 re-positioning (sinks re-scored against
// the query at sink_qpos), 2 keys stored before RoPE (rotated on read).
template <int D, int XM>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(DecodeArgs a, int stage_bytes) {
  constexpr int NS = D / 32, NW = kMergeWarps;
  extern __shared__ __align__(128) uint8_t smem[];
  float* red = reinterpret_cast<float*>(smem + stage_bytes);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + stage_bytes + NW * kMaxGqa * (D + 2) * 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 1);
  const Geometry& G = a.geo;
  const int u = blockIdx.x, b = u / G.H, h = u % G.H;
  bool ok = true;
  if constexpr (XM == 2)
    exact_states_prerope<D, NW>(a, b, h, red, reinterpret_cast<float*>(smem));
  else
    ok = G.act_bf16 ? exact_states_tc<D, NW, true, XM == 1>(a, b, h, red, smem, stage_bytes, bar, abort_flag)
                    : exact_states_tc<D, NW, false, XM == 1>(a, b, h, red, smem, stage_bytes, bar, abort_flag);
  if (!ok && threadIdx.x == 0) set_error(a.tab.err_flag, kErrTimeout);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= G.gqa) return;
  // what does not read the partials comes before the wait: the unit's slot
  // count (two 64-bit divisions) and the exact states' max (shared memory)
  const int j = warp;
  const int row = b * G.Hq + h * G.gqa + j;
  const int ns = slots_of_unit(a, u);
  const float* ml = a.part_ml + static_cast<size_t>(row) * a.ns * 2;
  const float* rj = red + j * (D + 2);  // warp w's state at rj + w * kMaxGqa * (D + 2)
  float M = lane < NW ? rj[lane * kMaxGqa * (D + 2) + D] : -INFINITY;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  pdl_wait_primary();  // the split partials are complete and visible from here on
  // the split partials in chunks of four slots whose loads are all issued
  // before any is used: the running max only grows, the sums so far are
  // rescaled when it does
  float L = 0.0f, oq[NS], oe[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) oq[i] = oe[i] = 0.0f;
  for (int s0 = 0; s0 < ns; s0 += 4) {  // a slot with m = -inf has o = 0 and l = 0
    float ms[4], ls[4], po[4][NS];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int s = s0 + c;
      const bool in = s < ns;
      ms[c] = in ? ml[2 * s] : -INFINITY;
      ls[c] = in ? ml[2 * s + 1] : 0.0f;
      const float* p = a.part_o + (static_cast<size_t>(row) * a.ns + (in ? s : 0)) * D;
#pragma unroll
      for (int i = 0; i < NS; ++i) po[c][i] = in ? p[i * 32 + lane] : 0.0f;
    }
    const float Mn = fmaxf(fmaxf(M, fmaxf(ms[0], ms[1])), fmaxf(ms[2], ms[3]));
    if (Mn > M) {  // warp-uniform (every lane holds the same values)
      const float r = M == -INFINITY ? 0.0f : exp2f(M - Mn);
      L *= r;
#pragma unroll
      for (int i = 0; i < NS; ++i) oq[i] *= r;
      M = Mn;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float w = ms[c] == -INFINITY ? 0.0f : exp2f(ms[c] - M);
      L = fmaf(ls[c], w, L);
#pragma unroll
      for (int i = 0; i < NS; ++i) oq[i] = fmaf(po[c][i], w, oq[i]);
    }
  }
  for (int w = 0; w < NW; ++w) {
    const float* r = rj + w * kMaxGqa * (D + 2);
    if (r[D] == -INFINITY) continue;
    const float sc = exp2f(r[D] - M);
    L += r[D + 1] * sc;
#pragma unroll
    for (int i = 0; i < NS; ++i) oe[i] = fmaf(r[i * 32 + lane], sc, oe[i]);
  }
  if (G.mode_tq) {
    warp_fwht<D>(oq);
    const float rsq = static_cast<float>(1.0 / sqrt(static_cast<double>(D)));
#pragma unroll
    for (int i = 0; i < NS; ++i) oq[i] = oq[i] * rsq * a.tab.signs[i * 32 + lane];
  }
  const float inv = 1.0f / L;
#pragma unroll
  for (int i = 0; i < NS; ++i) a.out[static_cast<size_t>(row) * D + i * 32 + lane] = (oq[i] + oe[i]) * inv;
  if (a.lse && lane == 0) a.lse[row] = (M + log2f(L)) * 0.69314718055994530942f;
}

// Rows (K and V) one merge CTA stages at once, in whole 32-row tiles: every
// sink and tail row when they fit in 80 KB, else batches of that size.
int merge_stage_bytes(const Geometry& G) {
  const int row_pair = 4 * G.D;  // K and V rows of the activation dtype
  int rows = G.n_sink_slots + G.tail_cap;
  const int cap = (80 << 10) / row_pair;
  if (rows > cap) rows = cap;
  rows = (rows + kExactTile - 1) / kExactTile * kExactTile;
  return rows * row_pair;
}

// `after_split`: the merge follows a split kernel on the stream and may be
// scheduled before it ends (programmatic dependent launch); otherwise it is
// an ordinary launch, since its exact pools read rows the appends before it
// wrote.
template <int D, int XM>
cudaError_t launch_merge_instance(DecodeArgs& a, cudaStream_t s, bool after_split) {
  const int stage = merge_stage_bytes(a.geo);
  const size_t smem = merge_smem_bytes<D>(stage);
  static size_t configured[kMaxDevices] = {};  // per device and instance: the attribute is per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (smem > configured[dev]) {
    e = cudaFuncSetAttribute(merge_kernel<D, XM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.geo.B * a.geo.H);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_split ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, merge_kernel<D, XM>, a, stage);
}

template <int D>
cudaError_t launch_merge(DecodeArgs& a, cudaStream_t s, bool after_split) {
  if (a.geo.k_pre_rope) return launch_merge_instance<D, 2>(a, s, after_split);
  return a.sink_qpos != a.L - 1 ? launch_merge_instance<D, 1>(a, s, after_split)
                                : launch_merge_instance<D, 0>(a, s, after_split);
}

}  // namespace

cudaError_t launch_decode(DecodeArgs& a, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1, int sm_count,
                          int64_t* launches) {
  const Geometry& G = a.geo;
  cudaError_t e;
  if (ev0) cudaEventRecord(ev0, s);
  e = (G.D == 128) ? launch_split<128>(a, s, sm_count) : launch_split<64>(a, s, sm_count);
  if (e != cudaSuccess) return e;
  const bool split_ran = a.work > 0;
  if (split_ran) ++*launches;
  e = (G.D == 128) ? launch_merge<128>(a, s, split_ran) : launch_merge<64>(a, s, split_ran);
  if (e != cudaSuccess) return e;
  ++*launches;
  if (ev1) cudaEventRecord(ev1, s);
  return cudaSuccess;
}

// 16-byte vectorised grid-stride copy: the in-process bandwidth reference.
namespace {
__global__ void __launch_bounds__(256) copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                   size_t n) {
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (; i + 3 * step < n; i += 4 * step) {
    const uint4 a0 = src[i], a1 = src[i + step], a2 = src[i + 2 * step], a3 = src[i + 3 * step];
    dst[i] = a0;
    dst[i + step] = a1;
    dst[i + 2 * step] = a2;
    dst[i + 3 * step] = a3;
  }
  for (; i < n; i += step) dst[i] = src[i];
}
}  // namespace

// The bounded waits of the decode kernels made to run out, on purpose and
// safely: two mbarriers that no thread arrives at and no copy completes on.
// Warp 0 waits on the first with a short budget (warp_wait) and, giving up,
// raises the CTA's abort flag; warp 1 waits on the second with the default
// budget of about one second and must give up through that flag long before
// its own budget; then thread 0 times out once more through wait_or_abort
// (abort flag cleared first) and mbar_wait_bounded. res[0..3]: 1 where each
// of the four waits returned "completed" (all must be 0), res[4]: SM clock
// cycles warp 1 waited. Every give-up sets the error flag.
namespace {
__global__ void __launch_bounds__(64) wait_probe_kernel(int* err_flag, long long* res, long long budget) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_fence_init();
  }
  __syncthreads();
  volatile int* ab = &abort_flag;
  bool ok = false;
  long long waited = 0;
  if (warp == 0) {
    ok = warp_wait(&bars[0], 0, ab, budget);
  } else {
    const long long t0 = clock64();
    ok = warp_wait(&bars[1], 0, ab);
    waited = clock64() - t0;
  }
  __syncthreads();
  if (lane == 0) res[warp] = ok ? 1 : 0;
  if (warp == 1 && lane == 0) res[4] = waited;
  bool ok2 = false, ok3 = false;
  if (threadIdx.x == 0) {
    *ab = 0;
    ok2 = wait_or_abort(&bars[0], 0, ab, budget);
    ok3 = mbar_wait_bounded(&bars[0], 0, budget);
    res[2] = ok2 ? 1 : 0;
    res[3] = ok3 ? 1 : 0;
  }
  if (lane == 0 && (!ok || (threadIdx.x == 0 && (!ok2 || !ok3)))) set_error(err_flag, kErrTimeout);
}
}  // namespace

cudaError_t launch_wait_probe(int* err_flag, long long* res, long long budget, cudaStream_t s,
                              int64_t* launches) {
  wait_probe_kernel<<<1, 64, 0, s>>>(err_flag, res, budget);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_copy(const void* src, void* dst, size_t bytes, cudaStream_t s, int64_t* launches) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t n = bytes / 16;
  copy_kernel<<<sms * 8, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace kvq
