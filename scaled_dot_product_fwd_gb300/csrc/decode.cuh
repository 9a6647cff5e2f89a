// decode.cuh — single-query (Lq = 1) attention: split-KV vector pass.
//
// MLX PR #4459 ("Add D512 support to Metal vector attention") serves
// single-token decode with a single-pass and a two-pass vector kernel: the
// first pass reduces chunks of the key range to partial results, the second
// merges them.  This file is the first pass for sm_103a, written for this
// GPU: one CTA per (key-range split, kv head and query-head group, batch).
//
//  - Warp 8 (producer) streams the split's K and V rows, which are contiguous
//    in [B, Hkv, Lk, D], into a ring of shared-memory stages with 1-D bulk
//    copies (cp.async.bulk, completion counted on an mbarrier).
//  - Warps 0-7 (consumers) each take KB keys of every stage.  A lane owns
//    D/32 elements of a row (16-byte pieces where the row is long enough, so
//    a warp reads one row with conflict-free, coalesced shared-memory loads),
//    keeps the HG query rows of its head group in registers, and forms
//    HG x KB partial dot products.  One butterfly reduce-scatter over the 32
//    lanes turns them into complete scores (one per lane, or replicated), a
//    group xor-shuffle gives the per-head tile max, and the probabilities
//    and rescale factors are broadcast through a small per-warp buffer.
//  - At the end the 8 warps' (m, l, acc) states are merged in shared memory
//    and the split writes its normalised partial output and its log2-domain
//    log-sum-exp to the workspace.  The combine kernel merges the splits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace dec {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr float kLog2e = 1.4426950408889634f;

struct SplitArgs {
  const void* q;
  const void* k;
  const void* v;
  int Hq, Hkv, G, Lk;
  int num_groups;   // query-head groups per kv head
  int num_splits;
  int split_keys;
  int stages;
  float sl2;  // scale * log2(e)
  const void* mask;
  long long ms0, ms1;  // batch and head strides of the mask (row 0, key stride 1)
  float* ws_o;    // [B, Hq, num_splits, D], normalised partial outputs
  float* ws_lse;  // [B, Hq, num_splits], log2-domain log-sum-exp
  int* status;
  unsigned long long wait_ns;
  // Failure-detection test hook: when set, the producer does not issue the
  // copies of the last tile, so the consumers' bounded wait on it expires.
  int debug_drop_last;
};

template <typename T>
struct Ld;
template <>
struct Ld<float> {
  static __device__ __forceinline__ float f(float x) { return x; }
};
template <>
struct Ld<__half> {
  static __device__ __forceinline__ float f(__half x) { return __half2float(x); }
};
template <>
struct Ld<__nv_bfloat16> {
  static __device__ __forceinline__ float f(__nv_bfloat16 x) { return __bfloat162float(x); }
};

// Load PIECE consecutive elements (4, 8 or 16 bytes) and widen to fp32.
template <typename T, int PIECE>
__device__ __forceinline__ void load_piece(const T* p, float* out) {
  constexpr int BYTES = PIECE * static_cast<int>(sizeof(T));
  static_assert(BYTES == 4 || BYTES == 8 || BYTES == 16, "piece size");
  T tmp[PIECE];
  if constexpr (BYTES == 16) {
    *reinterpret_cast<uint4*>(tmp) = *reinterpret_cast<const uint4*>(p);
  } else if constexpr (BYTES == 8) {
    *reinterpret_cast<uint2*>(tmp) = *reinterpret_cast<const uint2*>(p);
  } else {
    *reinterpret_cast<uint32_t*>(tmp) = *reinterpret_cast<const uint32_t*>(p);
  }
#pragma unroll
  for (int i = 0; i < PIECE; ++i) out[i] = Ld<T>::f(tmp[i]);
}

// Butterfly reduce-scatter of NV (power of two <= 32) values over the warp:
// afterwards lane l holds the full sum of value index l >> (5 - log2 NV).
template <int NV>
__device__ __forceinline__ float reduce_scatter(float (&v)[NV], int lane) {
  constexpr int LOG = (NV >= 32) ? 5 : (NV >= 16) ? 4 : (NV >= 8) ? 3 : (NV >= 4) ? 2 : (NV >= 2) ? 1 : 0;
  static_assert((1 << LOG) == NV, "NV must be a power of two <= 32");
#pragma unroll
  for (int lev = 0; lev < LOG; ++lev) {
    const int n = NV >> lev;
    const int msk = 16 >> lev;
    const bool upper = (lane & msk) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, msk);
    }
  }
#pragma unroll
  for (int msk = 16 >> LOG; msk >= 1; msk >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], msk);
  return v[0];
}

template <typename T, int D, int HG, int KB>
struct SplitCfg {
  static constexpr int EPL = D / 32;                          // elements per lane
  static constexpr int CE = 16 / static_cast<int>(sizeof(T));  // elements per 16 bytes
  static constexpr int PIECE = EPL < CE ? EPL : CE;
  static constexpr int NPIECE = EPL / PIECE;
  static constexpr int NV = HG * KB;
  static constexpr int TK = kConsumerWarps * KB;               // keys per stage
  static constexpr int TILE_BYTES = TK * D * static_cast<int>(sizeof(T));
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int LOG_NV = (NV >= 32) ? 5 : (NV >= 16) ? 4 : (NV >= 8) ? 3 : (NV >= 4) ? 2 : (NV >= 2) ? 1 : 0;
  static constexpr int HLANES = 32 / HG;                       // lanes per head after the scatter
  static constexpr int VLANES = 32 / NV;                       // lanes per value
  // per-warp broadcast buffer: NV probabilities + HG rescale factors
  static constexpr int PB_FLOATS = NV + HG;
  static constexpr int COMBINE_BYTES = kConsumerWarps * HG * (D + 2) * 4;
  static_assert(NV <= 32, "too many partial sums per lane");
  static_assert((TILE_BYTES % 16) == 0, "bulk copy granularity");
  static size_t smem_bytes(int stages) {
    size_t ring = static_cast<size_t>(stages) * STAGE_BYTES;
    if (ring < static_cast<size_t>(COMBINE_BYTES)) ring = COMBINE_BYTES;
    return 128 /*align*/ + ring + kConsumerWarps * PB_FLOATS * 4 + 2 * 8 * 8 /*bars*/ + 16;
  }
};

template <typename T, int D, int HG, int KB>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const SplitArgs a) {
  using C = SplitCfg<T, D, HG, KB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((128u - (raw_addr & 127u)) & 127u);
  const int NS = a.stages;
  uint8_t* ring = smem;
  size_t ring_bytes = static_cast<size_t>(NS) * C::STAGE_BYTES;
  if (ring_bytes < static_cast<size_t>(C::COMBINE_BYTES)) ring_bytes = C::COMBINE_BYTES;
  float* pbuf = reinterpret_cast<float*>(smem + ring_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(pbuf + kConsumerWarps * C::PB_FLOATS);
  uint64_t* empty = full + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / a.num_groups;
  const int grp = blockIdx.y % a.num_groups;
  const int b = blockIdx.z;
  const int key_begin = split * a.split_keys;
  const int key_end = min(a.Lk, key_begin + a.split_keys);
  const int nkeys = max(0, key_end - key_begin);
  const int ntiles = (nkeys + C::TK - 1) / C::TK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{a.wait_ns, abort_flag, a.status};

  const size_t kv_row0 = (static_cast<size_t>(b) * a.Hkv + kvh) * a.Lk;
  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    int last_use[8];  // last fill of each stage (-1: none)
#pragma unroll
    for (int s = 0; s < 8; ++s) last_use[s] = -1;
    if (lane == 0) {
      const T* kg = static_cast<const T*>(a.k) + (kv_row0 + key_begin) * D;
      const T* vg = static_cast<const T*>(a.v) + (kv_row0 + key_begin) * D;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % NS;
        const int use = t / NS;
        if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, wc)) break;
        if (a.debug_drop_last && t == ntiles - 1) break;
        const int rows = min(C::TK, nkeys - t * C::TK);
        const uint32_t bytes = static_cast<uint32_t>(rows * D * sizeof(T));
        mbar_arrive_expect_tx(&full[s], 2 * bytes);
        uint8_t* st = ring + static_cast<size_t>(s) * C::STAGE_BYTES;
        bulk_load(st, kg + static_cast<size_t>(t) * C::TK * D, bytes, &full[s]);
        bulk_load(st + C::TILE_BYTES, vg + static_cast<size_t>(t) * C::TK * D, bytes, &full[s]);
        last_use[s] = use;
      }
    }
    __syncwarp();
    named_bar_sync(1, kThreads);  // joins the consumers' combine barrier
    if (lane == 0 && *abort_flag) {
      // a wait gave up: every copy issued here lands before the CTA exits
      for (int s = 0; s < NS; ++s) {
        if (last_use[s] < 0) continue;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[s], last_use[s] & 1))
          if (globaltimer_ns() - t0 > kDrainNs) break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int vidx = lane >> (5 - C::LOG_NV);  // value index held after the scatter
  const int hl = vidx / KB;                  // its head inside the group
  const int kl = vidx % KB;                  // its key inside the warp's batch
  float qv[HG][C::EPL];
  bool head_ok[HG];
#pragma unroll
  for (int hh = 0; hh < HG; ++hh) {
    const int gh = grp * HG + hh;
    head_ok[hh] = gh < a.G;
    const int hq = kvh * a.G + gh;
    const T* qrow = static_cast<const T*>(a.q) + (static_cast<size_t>(b) * a.Hq + hq) * D;
#pragma unroll
    for (int pi = 0; pi < C::NPIECE; ++pi) {
      float tmp[C::PIECE];
      if (head_ok[hh]) {
        load_piece<T, C::PIECE>(qrow + (pi * 32 + lane) * C::PIECE, tmp);
      } else {
#pragma unroll
        for (int i = 0; i < C::PIECE; ++i) tmp[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < C::PIECE; ++i) qv[hh][pi * C::PIECE + i] = tmp[i];
    }
  }
  const int my_hq = kvh * a.G + grp * HG + hl;
  const bool my_head_ok = grp * HG + hl < a.G;
  const T* mrow = nullptr;
  if (a.mask && my_head_ok) mrow = static_cast<const T*>(a.mask) + b * a.ms0 + my_hq * a.ms1;

  float acc[HG][C::EPL];
  float lsum[HG];
#pragma unroll
  for (int hh = 0; hh < HG; ++hh) {
    lsum[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < C::EPL; ++e) acc[hh][e] = 0.f;
  }
  float m_own = -INFINITY;  // running max of head hl (log2 units)
  float* pb = pbuf + warp * C::PB_FLOATS;
  bool ok = true;

  for (int t = 0; t < ntiles; ++t) {
    const int s = t % NS;
    ok = mbar_wait(&full[s], (t / NS) & 1, wc);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    const uint8_t* st = ring + static_cast<size_t>(s) * C::STAGE_BYTES;
    const T* Ks = reinterpret_cast<const T*>(st) + warp * KB * D;
    const T* Vs = reinterpret_cast<const T*>(st + C::TILE_BYTES) + warp * KB * D;
    const int key0 = key_begin + t * C::TK + warp * KB;  // key of kk = 0

    float part[C::NV];
#pragma unroll
    for (int kk = 0; kk < KB; ++kk) {
      float kf[C::EPL];
      if (key0 + kk < key_end) {
#pragma unroll
        for (int pi = 0; pi < C::NPIECE; ++pi)
          load_piece<T, C::PIECE>(Ks + kk * D + (pi * 32 + lane) * C::PIECE, kf + pi * C::PIECE);
      } else {
#pragma unroll
        for (int e = 0; e < C::EPL; ++e) kf[e] = 0.f;
      }
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) {
        float d0 = 0.f;
#pragma unroll
        for (int e = 0; e < C::EPL; ++e) d0 = fmaf(qv[hh][e], kf[e], d0);
        part[hh * KB + kk] = d0;
      }
    }
    const float sc = reduce_scatter<C::NV>(part, lane);
    const int key = key0 + kl;
    float x = sc * a.sl2;
    if (key >= key_end) {
      x = -INFINITY;
    } else if (mrow) {
      x += Ld<T>::f(mrow[key]) * kLog2e;
    }
    float tmax = x;
#pragma unroll
    for (int off = 1; off < C::HLANES; off <<= 1)
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float m_new = fmaxf(m_own, tmax);
    const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m_own - m_new);
    const float p = (x == -INFINITY) ? 0.f : ex2(x - m_new);
    m_own = m_new;
    if ((lane & (C::VLANES - 1)) == 0) pb[vidx] = p;
    if ((lane & (C::HLANES - 1)) == 0) pb[C::NV + hl] = alpha;
    __syncwarp();
    float pv[C::NV], al[HG];
#pragma unroll
    for (int i = 0; i < C::NV; ++i) pv[i] = pb[i];
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) al[hh] = pb[C::NV + hh];
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
      float ssum = 0.f;
#pragma unroll
      for (int kk = 0; kk < KB; ++kk) ssum += pv[hh * KB + kk];
      lsum[hh] = lsum[hh] * al[hh] + ssum;
#pragma unroll
      for (int e = 0; e < C::EPL; ++e) acc[hh][e] *= al[hh];
    }
#pragma unroll
    for (int kk = 0; kk < KB; ++kk) {
      if (key0 + kk >= key_end) continue;  // rows past the split were not loaded
      float vf[C::EPL];
#pragma unroll
      for (int pi = 0; pi < C::NPIECE; ++pi)
        load_piece<T, C::PIECE>(Vs + kk * D + (pi * 32 + lane) * C::PIECE, vf + pi * C::PIECE);
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) {
        const float w = pv[hh * KB + kk];
#pragma unroll
        for (int e = 0; e < C::EPL; ++e) acc[hh][e] = fmaf(w, vf[e], acc[hh][e]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- merge the warps' states (the ring is idle: every copy was consumed)
  named_bar_sync(1, kThreads);
  float* wm = reinterpret_cast<float*>(ring);       // [warps][HG]
  float* wl = wm + kConsumerWarps * HG;             // [warps][HG]
  float* wacc = wl + kConsumerWarps * HG;           // [warps][HG][D]
  if (ok) {
    if ((lane & (C::HLANES - 1)) == 0) wm[warp * HG + hl] = m_own;
    if (lane == 0)
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) wl[warp * HG + hh] = lsum[hh];
#pragma unroll
    for (int hh = 0; hh < HG; ++hh)
#pragma unroll
      for (int pi = 0; pi < C::NPIECE; ++pi)
#pragma unroll
        for (int i = 0; i < C::PIECE; ++i)
          wacc[(warp * HG + hh) * D + (pi * 32 + lane) * C::PIECE + i] = acc[hh][pi * C::PIECE + i];
  }
  named_bar_sync(2, kConsumerWarps * 32);
  if (*abort_flag) return;
  for (int e = threadIdx.x; e < HG * D; e += kConsumerWarps * 32) {
    const int hh = e / D, d = e % D;
    if (grp * HG + hh >= a.G) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wm[w * HG + hh]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float f = ex2(wm[w * HG + hh] - M);
        L = fmaf(wl[w * HG + hh], f, L);
        O = fmaf(wacc[(w * HG + hh) * D + d], f, O);
      }
    }
    const int hq = kvh * a.G + grp * HG + hh;
    const size_t row = (static_cast<size_t>(b) * a.Hq + hq) * a.num_splits + split;
    a.ws_o[row * D + d] = (L > 0.f) ? O / L : 0.f;
    if (d == 0) a.ws_lse[row] = (L > 0.f) ? M + __log2f(L) : -INFINITY;
  }
}

// Host-side launch of one instantiation.
template <typename T, int D, int HG, int KB>
sdpa_status_t launch_split(const SplitArgs& a, int batch, cudaStream_t stream) {
  using C = SplitCfg<T, D, HG, KB>;
  auto kern = decode_split_kernel<T, D, HG, KB>;
  const size_t smem = C::smem_bytes(a.stages);
  cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return SDPA_ERR_CUDA;
  dim3 grid(a.num_splits, a.Hkv * a.num_groups, batch);
  kern<<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

// Keys per warp batch for a (dtype, D, head group): at most 32 partial sums
// per lane, about 4 KiB of K per warp batch.
__host__ __device__ constexpr int keys_per_warp(int elem_bytes, int D, int HG) {
  int kb = 4096 / (D * elem_bytes);
  if (kb > 8) kb = 8;
  if (kb > 32 / HG) kb = 32 / HG;
  if (kb < 1) kb = 1;
  return kb;
}

template <typename T, int D, int HG>
sdpa_status_t launch_split_hg(const SplitArgs& a, int batch, cudaStream_t stream) {
  constexpr int KB = keys_per_warp(static_cast<int>(sizeof(T)), D, HG);
  return launch_split<T, D, HG, KB>(a, batch, stream);
}

template <typename T, int D>
sdpa_status_t launch_split_d(const SplitArgs& a, int hg, int batch, cudaStream_t stream) {
  switch (hg) {
    case 1: return launch_split_hg<T, D, 1>(a, batch, stream);
    case 2: return launch_split_hg<T, D, 2>(a, batch, stream);
    case 4: return launch_split_hg<T, D, 4>(a, batch, stream);
    case 8:
      if constexpr (D <= 128) return launch_split_hg<T, D, 8>(a, batch, stream);
      return SDPA_ERR_UNSUPPORTED;
    default: return SDPA_ERR_UNSUPPORTED;
  }
}

template <typename T>
sdpa_status_t launch_split_t(const SplitArgs& a, int D, int hg, int batch, cudaStream_t stream) {
  switch (D) {
    case 64: return launch_split_d<T, 64>(a, hg, batch, stream);
    case 128: return launch_split_d<T, 128>(a, hg, batch, stream);
    case 512: return launch_split_d<T, 512>(a, hg, batch, stream);
    default: return SDPA_ERR_UNSUPPORTED;
  }
}

// Per-dtype entry points (one translation unit each).
sdpa_status_t launch_split_f32(const SplitArgs& a, int D, int hg, int batch, cudaStream_t s);
sdpa_status_t launch_split_f16(const SplitArgs& a, int D, int hg, int batch, cudaStream_t s);
sdpa_status_t launch_split_bf16(const SplitArgs& a, int D, int hg, int batch, cudaStream_t s);

}  // namespace dec
}  // namespace gb300
