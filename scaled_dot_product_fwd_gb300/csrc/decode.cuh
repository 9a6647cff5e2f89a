// decode.cuh — single-query (Lq = 1) and few-query (Lq <= 8) attention:
// split-KV vector pass.  The G x Lq query rows of a kv head form its head
// groups, so they all share one K/V stream.
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
//  - Warps 0-7 (consumers) each take KB keys of every stage.  A lane owns a
//    16-byte piece (or more) of a key row, so a D=128 bf16 row spans 16
//    lanes and one warp-wide load covers two keys; shared-memory reads are
//    coalesced and conflict-free.  The HG query rows of the head group stay
//    in registers as fp32 pairs; dot products and the V accumulation use the
//    packed f32x2 FMA.  A butterfly reduce-scatter over the lanes of a row
//    turns the HG x (KB / rows-per-load) partial sums into complete scores,
//    a shuffle max gives the per-head tile max, and probabilities and rescale
//    factors are broadcast through a small per-warp buffer.
//  - At the end the 8 warps' (m, l, acc) states are merged in shared memory
//    and the split writes its normalised partial output and its log2-domain
//    log-sum-exp to the workspace; the combine kernel merges the splits.
//  - When the splits of a head group fit one thread-block cluster (2, 4, 8
//    or 16 CTAs that divide D), the launcher makes them one, and the merge
//    happens inside it instead: each CTA keeps its partial in shared memory,
//    and after a cluster barrier CTA r reads every partial's lse and its
//    slice of D columns through distributed shared memory, applies the same
//    weights as the combine kernel, and writes that slice of O (CTA 0 also
//    writes the LSE).  No workspace traffic and no second launch.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "tensor_map.h"

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
  int Lq;           // query rows per head (1 for decode, up to 8 for multi-query)
  int causal;       // bottom-right: key j visible to row i iff j <= i + Lk - Lq
  // element strides (batch, head, row) of q, k, v and o; D is contiguous
  long long qs0, qs1, qs2, ks0, ks1, ks2, vs0, vs1, vs2, os0, os1, os2;
  int mask_bool;    // mask holds bytes, nonzero = visible
  const int* seq_lens_q;   // nullptr or per-batch valid query rows
  const int* seq_lens_kv;  // nullptr or per-batch valid keys
  int num_groups;   // groups of HG query rows per kv head (rows: G heads x Lq)
  int num_splits;
  int split_keys;
  int stages;
  float sl2;  // scale * log2(e)
  const void* mask;
  long long ms0, ms1, ms2;  // batch, head and row strides of the mask (key stride 1)
  float* ws_o;    // [B, Hq, num_splits, D], normalised partial outputs
  // [B, Hq, num_splits][2]: each split's running max m (log2 units) and sum
  // l relative to it.  Carried apart rather than as m + log2 l: a row whose
  // keys all carry a huge mask value has m at the huge-mask value, beside
  // which log2 l vanishes in fp32, yet l still weighs the split.
  float* ws_ml;
  // in-cluster merge (set by the launcher): output, LSE and sinks
  void* o;
  float* lse;
  const float* sinks;
  int cluster;      // 1: the num_splits CTAs of a head group form one cluster
  int cluster_ok;   // 0: the caller asks for the two-pass form
  int* status;
  unsigned long long wait_ns;
  // Failure-detection test hook: when set, the producer does not issue the
  // copies of the last tile, so the consumers' bounded wait on it expires.
  int debug_drop_last;
  // K and V rows that are not contiguous (e.g. [B, L, Hkv, D] storage): one
  // tiled tensor copy per tile (box D x TK rows, no swizzle, rows past Lk
  // read as zero) instead of one bulk copy per row; set by the launcher when
  // the driver accepts both maps.
  int use_tma;
  CUtensorMap tmK, tmV;
  // Ragged plan (per-batch key lengths on the device): the grid is one
  // linear range of work items and every CTA derives the split size from
  // seq_lens_kv itself (ragged_tiles_per_split), so that the items of the
  // call's real keys fill whole waves of the GPU.  num_splits is then the
  // workspace's split capacity per row.
  int ragged;
  int batch;        // B
  int slots;        // CTAs resident at once
  int tiles_base;   // tiles per split of the plan for rows of Lk keys
};

// Ragged plan: tiles per split for the batches' real key counts.  W = the
// real tiles of all (batch, unit) pairs; the splits of the plan for full
// rows (tiles_base tiles) would fill `waves` waves of `slots` CTAs; the split
// size is the smallest that keeps the items (every pair's real tiles cut
// into splits) within those waves, and at least the size that keeps each
// row within `max_splits` splits.
__host__ __device__ inline int ragged_tiles_per_split(const int* lens, int B, int Lk, int tk,
                                                      int units, int slots, int tiles_base,
                                                      int max_splits) {
  long long W = 0;
  for (int b = 0; b < B; ++b) {
    const int L = lens[b] < 0 ? 0 : (lens[b] > Lk ? Lk : lens[b]);
    W += (L + tk - 1) / tk;
  }
  W *= units;
  const int tiles_cap = (Lk + tk - 1) / tk;
  int tp_min = (tiles_cap + max_splits - 1) / max_splits;
  if (tp_min < 1) tp_min = 1;
  if (W == 0) return tp_min;
  const long long per_wave = static_cast<long long>(slots) * (tiles_base > 0 ? tiles_base : 1);
  long long waves = (W + per_wave / 2) / per_wave;  // nearest whole number of waves
  if (waves < 1) waves = 1;
  const long long cap = waves * slots;
  int tp = static_cast<int>((W + cap - 1) / cap);
  if (tp < tp_min) tp = tp_min;
  for (int it = 0; it < 64; ++it, ++tp) {  // per-pair rounding adds items
    long long items = 0;
    for (int b = 0; b < B; ++b) {
      const int L = lens[b] < 0 ? 0 : (lens[b] > Lk ? Lk : lens[b]);
      items += (((L + tk - 1) / tk) + tp - 1) / tp;
    }
    if (items * units <= cap) break;
  }
  return tp;
}

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

// fp32 -> storage type, round to nearest even.
template <typename T>
struct StoreAs;
template <>
struct StoreAs<float> {
  static __device__ __forceinline__ float c(float x) { return x; }
};
template <>
struct StoreAs<__half> {
  static __device__ __forceinline__ __half c(float x) { return __float2half_rn(x); }
};
template <>
struct StoreAs<__nv_bfloat16> {
  static __device__ __forceinline__ __nv_bfloat16 c(float x) { return __float2bfloat16_rn(x); }
};

constexpr int kMaxClusterSplits = 16;

// Pairs of fp32 values in one 64-bit register for the packed f32x2 ops.
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float f2_sum(uint64_t r) {
  float a, b;
  f2_split(r, a, b);
  return a + b;
}

// 16 bytes of T widened exactly to fp32 pairs (element 2i in the low half).
template <typename T>
struct Widen;
template <>
struct Widen<__nv_bfloat16> {
  static constexpr int CE = 8;
  static __device__ __forceinline__ void pairs(uint4 w, uint64_t* p) {
    p[0] = f2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
    p[1] = f2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    p[2] = f2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u));
    p[3] = f2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
  }
};
template <>
struct Widen<__half> {
  static constexpr int CE = 8;
  static __device__ __forceinline__ uint64_t one(uint32_t x) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&x));
    return f2(f.x, f.y);
  }
  static __device__ __forceinline__ void pairs(uint4 w, uint64_t* p) {
    p[0] = one(w.x);
    p[1] = one(w.y);
    p[2] = one(w.z);
    p[3] = one(w.w);
  }
};
template <>
struct Widen<float> {
  static constexpr int CE = 4;
  static __device__ __forceinline__ void pairs(uint4 w, uint64_t* p) {
    p[0] = f2(__uint_as_float(w.x), __uint_as_float(w.y));
    p[1] = f2(__uint_as_float(w.z), __uint_as_float(w.w));
  }
};

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// Butterfly reduce-scatter of NV (power of two) values over the LR lanes of
// a row group (lanes differing in their low log2(LR) bits): afterwards lane
// position c holds the full sum of value index c >> (log2 LR - log2 NV).
template <int NV, int LR>
__device__ __forceinline__ float reduce_scatter(float (&v)[NV], int c) {
  constexpr int LOG = ilog2(NV);
  static_assert((1 << LOG) == NV && NV <= LR, "NV must be a power of two <= LR");
#pragma unroll
  for (int lev = 0; lev < LOG; ++lev) {
    const int n = NV >> lev;
    const int msk = (LR / 2) >> lev;
    const bool upper = (c & msk) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, msk);
    }
  }
#pragma unroll
  for (int msk = (LR / 2) >> LOG; msk >= 1; msk >>= 1)
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], msk);
  return v[0];
}

template <typename T, int D, int HG, int KB>
struct SplitCfg {
  static constexpr int CE = Widen<T>::CE;                     // elements per 16 bytes
  static constexpr int EPL = (D / 32 > CE) ? D / 32 : CE;    // elements per lane and row
  static constexpr int LR = D / EPL;                          // lanes per key row
  static constexpr int RPW = 32 / LR;                         // key rows per warp-wide load
  static constexpr int NPIECE = EPL / CE;                     // 16-byte pieces per lane and row
  static constexpr int NP2 = EPL / 2;                         // fp32 pairs per lane and row
  static constexpr int LPB = KB / RPW;                        // loads per lane per batch
  static constexpr int NVL = HG * LPB;                        // partial sums per lane
  static constexpr int LOG_LR = ilog2(LR);
  static constexpr int VSHIFT = LOG_LR - ilog2(NVL);          // value index = c >> VSHIFT
  static constexpr int HBIT = VSHIFT + ilog2(LPB);            // head index = c >> HBIT
  static constexpr int TK = kConsumerWarps * KB;              // keys per stage
  static constexpr int TILE_BYTES = TK * D * static_cast<int>(sizeof(T));
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  // per-warp broadcast buffer: (p, p) pairs per (head, key), then HG factors
  static constexpr int PB_WORDS = 2 * HG * KB + ((HG + 1) & ~1);
  static constexpr int COMBINE_BYTES = kConsumerWarps * HG * (D + 2) * 4;
  // in-cluster merge, after the warps' states: partial O [HG][D], m and l
  // [HG][2], split weights [HG][16], 1/L [HG]
  static constexpr int MERGE_BYTES =
      COMBINE_BYTES + (HG * D + 2 * HG + HG * kMaxClusterSplits + HG) * 4;
  static_assert(LR * EPL == D && RPW * LR == 32, "lane layout");
  static_assert(KB % RPW == 0 && NVL <= LR, "batch layout");
  static_assert((TILE_BYTES % 16) == 0, "bulk copy granularity");
  static size_t smem_bytes(int stages) {
    size_t ring = static_cast<size_t>(stages) * STAGE_BYTES;
    if (ring < static_cast<size_t>(MERGE_BYTES)) ring = MERGE_BYTES;
    return 128 /*align*/ + ring + kConsumerWarps * PB_WORDS * 4 + 2 * 8 * 8 /*bars*/ + 16;
  }
};

template <typename T, int D, int HG, int KB>
__global__ void __launch_bounds__(kThreads, (D <= 128 && HG <= 4) ? 2 : 1)
    decode_split_kernel(const __grid_constant__ SplitArgs a) {
  using C = SplitCfg<T, D, HG, KB>;
  using Wd = Widen<T>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((128u - (raw_addr & 127u)) & 127u);
  const int NS = a.stages;
  uint8_t* ring = smem;
  size_t ring_bytes = static_cast<size_t>(NS) * C::STAGE_BYTES;
  if (ring_bytes < static_cast<size_t>(C::MERGE_BYTES)) ring_bytes = C::MERGE_BYTES;
  float* pbuf = reinterpret_cast<float*>(smem + ring_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(pbuf + kConsumerWarps * C::PB_WORDS);
  uint64_t* empty = full + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int split = blockIdx.x;
  int kvh = blockIdx.y / a.num_groups;
  int grp = blockIdx.y % a.num_groups;
  int b = blockIdx.z;
  int split_keys = a.split_keys;
  if (a.ragged) {
    // item blockIdx.x of the ragged plan: (batch, unit, split) in that order
    const int units = a.Hkv * a.num_groups;
    split_keys = C::TK * ragged_tiles_per_split(a.seq_lens_kv, a.batch, a.Lk, C::TK, units,
                                                a.slots, a.tiles_base, a.num_splits);
    int item = blockIdx.x;
    b = -1;
    for (int bb = 0; bb < a.batch; ++bb) {
      const int L = min(max(a.seq_lens_kv[bb], 0), a.Lk);
      const int sb = (L + split_keys - 1) / split_keys;
      if (item < units * sb) {
        b = bb;
        split = item % sb;
        kvh = (item / sb) / a.num_groups;
        grp = (item / sb) % a.num_groups;
        break;
      }
      item -= units * sb;
    }
    if (b < 0) return;  // past the call's last item (the whole CTA)
  }
  // this batch's lengths (padding masks), clamped to the call's maxima
  const int Lkb = a.seq_lens_kv ? min(max(a.seq_lens_kv[b], 0), a.Lk) : a.Lk;
  const int Lqb = a.seq_lens_q ? min(max(a.seq_lens_q[b], 0), a.Lq) : a.Lq;
  const int key_begin = split * split_keys;
  const int key_end = min(Lkb, key_begin + split_keys);
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

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    int last_use[8];  // last fill of each stage (-1: none)
#pragma unroll
    for (int s = 0; s < 8; ++s) last_use[s] = -1;
    if (lane == 0) {
      const T* kg = static_cast<const T*>(a.k) + b * a.ks0 + kvh * a.ks1 + key_begin * a.ks2;
      const T* vg = static_cast<const T*>(a.v) + b * a.vs0 + kvh * a.vs1 + key_begin * a.vs2;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % NS;
        const int use = t / NS;
        if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, wc)) break;
        if (a.debug_drop_last && t == ntiles - 1) break;
        const int rows = min(C::TK, nkeys - t * C::TK);
        const uint32_t bytes = static_cast<uint32_t>(rows * D * sizeof(T));
        uint8_t* st = ring + static_cast<size_t>(s) * C::STAGE_BYTES;
        const long long r0 = static_cast<long long>(t) * C::TK;
        if (a.use_tma) {
          // whole TK-row boxes: rows past the split hold keys the consumers
          // skip, rows past Lk read as zero
          const int key = key_begin + static_cast<int>(r0);
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(2 * C::TILE_BYTES));
          tma_load_4d(st, &a.tmK, &full[s], 0, key, kvh, b);
          tma_load_4d(st + C::TILE_BYTES, &a.tmV, &full[s], 0, key, kvh, b);
          last_use[s] = use;
          continue;
        }
        mbar_arrive_expect_tx(&full[s], 2 * bytes);
        // a tile's rows are one copy when they are contiguous, else one per row
        if (a.ks2 == D) {
          bulk_load(st, kg + r0 * D, bytes, &full[s]);
        } else {
          for (int r = 0; r < rows; ++r)
            bulk_load(st + r * D * sizeof(T), kg + (r0 + r) * a.ks2, D * sizeof(T), &full[s]);
        }
        if (a.vs2 == D) {
          bulk_load(st + C::TILE_BYTES, vg + r0 * D, bytes, &full[s]);
        } else {
          for (int r = 0; r < rows; ++r)
            bulk_load(st + C::TILE_BYTES + r * D * sizeof(T), vg + (r0 + r) * a.vs2,
                      D * sizeof(T), &full[s]);
        }
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
  const int r = lane / C::LR;          // key row inside a warp-wide load
  const int c = lane % C::LR;          // lane position inside the row
  const int vi = c >> C::VSHIFT;       // value held after the reduce-scatter
  const int hl = vi / C::LPB;          // its head inside the group
  const int kl = (vi % C::LPB) * C::RPW + r;  // its key inside the warp batch
  // The group's HG rows are (query head, query row) pairs of this kv head:
  // row rr of the kv head is head kvh * G + rr / Lq, query row rr % Lq.
  const int R = a.G * a.Lq;  // rows per kv head
  auto row_index = [&](int rr) {  // global query row [b, hq, qi] (lse, workspace)
    const int hq = kvh * a.G + rr / a.Lq;
    return (static_cast<size_t>(b) * a.Hq + hq) * a.Lq + rr % a.Lq;
  };
  auto q_off = [&](int rr) {  // element offset of a query row in q
    return b * a.qs0 + (kvh * a.G + rr / a.Lq) * a.qs1 + (rr % a.Lq) * a.qs2;
  };
  uint64_t q2[HG][C::NP2];
#pragma unroll
  for (int hh = 0; hh < HG; ++hh) {
    const int rr = grp * HG + hh;
    const T* qrow = static_cast<const T*>(a.q) + q_off(rr < R ? rr : 0);
#pragma unroll
    for (int pi = 0; pi < C::NPIECE; ++pi) {
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (rr < R) w = *reinterpret_cast<const uint4*>(qrow + (pi * C::LR + c) * C::CE);
      Wd::pairs(w, &q2[hh][pi * (C::CE / 2)]);
    }
  }
  const int my_rr = grp * HG + hl;
  const bool my_head_ok = my_rr < R;
  const int my_hq = kvh * a.G + (my_head_ok ? my_rr / a.Lq : 0);
  const int my_qi = my_head_ok ? my_rr % a.Lq : 0;
  // last key this lane's row sees (bounds, and the causal rule)
  int my_limit = Lkb - 1;
  if (a.causal) my_limit = min(my_limit, my_qi + (Lkb - Lqb));
  if (my_qi >= Lqb) my_limit = -1;  // a padding row sees no key
  // additive mask row (mrow) or boolean mask row (mrowb)
  const T* mrow = nullptr;
  const uint8_t* mrowb = nullptr;
  if (a.mask && my_head_ok) {
    const long long moff = b * a.ms0 + my_hq * a.ms1 + my_qi * a.ms2;
    if (a.mask_bool)
      mrowb = static_cast<const uint8_t*>(a.mask) + moff;
    else
      mrow = static_cast<const T*>(a.mask) + moff;
  }

  uint64_t acc2[HG][C::NP2];
  float lsum[HG];
#pragma unroll
  for (int hh = 0; hh < HG; ++hh) {
    lsum[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < C::NP2; ++e) acc2[hh][e] = 0ull;
  }
  float m_own = -INFINITY;  // running max of head hl (log2 units)
  float* pb = pbuf + warp * C::PB_WORDS;
  uint64_t* pb2 = reinterpret_cast<uint64_t*>(pb);  // (p, p) per (head, key)
  float* pba = pb + 2 * HG * KB;                    // rescale factor per head
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

    float part[C::NVL];
#pragma unroll
    for (int i = 0; i < C::LPB; ++i) {
      const int kk = i * C::RPW + r;
      uint64_t k2[C::NP2];
#pragma unroll
      for (int pi = 0; pi < C::NPIECE; ++pi) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (key0 + kk < key_end)  // rows past the split were not loaded
          w = *reinterpret_cast<const uint4*>(Ks + kk * D + (pi * C::LR + c) * C::CE);
        Wd::pairs(w, &k2[pi * (C::CE / 2)]);
      }
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) {
        uint64_t d2 = 0ull;
#pragma unroll
        for (int e = 0; e < C::NP2; ++e) d2 = f2_fma(q2[hh][e], k2[e], d2);
        part[hh * C::LPB + i] = f2_sum(d2);
      }
    }
    const float sc = reduce_scatter<C::NVL, C::LR>(part, c);
    const int key = key0 + kl;
    float x = sc * a.sl2;
    if (key >= key_end || key > my_limit) {
      x = -INFINITY;
    } else if (mrow) {
      x += mask_log2(Ld<T>::f(mrow[key]), mask_huge_log2(a.sl2));
    } else if (mrowb && !mrowb[key]) {
      x = -INFINITY;
    }
    // tile max of head hl: lanes differing below HBIT or in the row bits
    float tmax = x;
#pragma unroll
    for (int bit = 0; bit < 5; ++bit)
      if (bit < C::HBIT || bit >= C::LOG_LR)
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1 << bit));
    const float m_new = fmaxf(m_own, tmax);
    const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m_own - m_new);
    const float p = (x == -INFINITY) ? 0.f : ex2(x - m_new);
    m_own = m_new;
    if ((c & ((1 << C::VSHIFT) - 1)) == 0) pb2[hl * KB + kl] = f2(p, p);
    if (r == 0 && (c & ((1 << C::HBIT) - 1)) == 0) pba[hl] = alpha;
    __syncwarp();
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
      const float al = pba[hh];
      lsum[hh] *= al;
      const uint64_t al2 = f2(al, al);
#pragma unroll
      for (int e = 0; e < C::NP2; ++e) acc2[hh][e] = f2_mul(acc2[hh][e], al2);
    }
#pragma unroll
    for (int i = 0; i < C::LPB; ++i) {
      const int kk = i * C::RPW + r;
      if (key0 + kk >= key_end) continue;  // rows past the split were not loaded (p = 0)
      uint64_t v2[C::NP2];
#pragma unroll
      for (int pi = 0; pi < C::NPIECE; ++pi)
        Wd::pairs(*reinterpret_cast<const uint4*>(Vs + kk * D + (pi * C::LR + c) * C::CE),
                  &v2[pi * (C::CE / 2)]);
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) {
        const uint64_t pp = pb2[hh * KB + kk];
        float p0, p1;
        f2_split(pp, p0, p1);
        lsum[hh] += p0;
#pragma unroll
        for (int e = 0; e < C::NP2; ++e) acc2[hh][e] = f2_fma(pp, v2[e], acc2[hh][e]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- fold the row groups of the warp together (same heads, other keys)
#pragma unroll
  for (int bit = C::LOG_LR; bit < 5; ++bit) {
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
      lsum[hh] += __shfl_xor_sync(0xffffffffu, lsum[hh], 1 << bit);
#pragma unroll
      for (int e = 0; e < C::NP2; ++e) {
        float a0, a1;
        f2_split(acc2[hh][e], a0, a1);
        a0 += __shfl_xor_sync(0xffffffffu, a0, 1 << bit);
        a1 += __shfl_xor_sync(0xffffffffu, a1, 1 << bit);
        acc2[hh][e] = f2(a0, a1);
      }
    }
  }

  // ---- merge the warps' states (the ring is idle: every copy was consumed)
  named_bar_sync(1, kThreads);
  float* wm = reinterpret_cast<float*>(ring);       // [warps][HG]
  float* wl = wm + kConsumerWarps * HG;             // [warps][HG]
  float* wacc = wl + kConsumerWarps * HG;           // [warps][HG][D]
  if (ok) {
    if (r == 0 && (c & ((1 << C::HBIT) - 1)) == 0) wm[warp * HG + hl] = m_own;
    if (lane == 0)
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) wl[warp * HG + hh] = lsum[hh];
    if (r == 0) {
#pragma unroll
      for (int hh = 0; hh < HG; ++hh)
#pragma unroll
        for (int pi = 0; pi < C::NPIECE; ++pi)
#pragma unroll
          for (int j = 0; j < C::CE / 2; ++j) {
            float a0, a1;
            f2_split(acc2[hh][pi * (C::CE / 2) + j], a0, a1);
            float* dst = wacc + (warp * HG + hh) * D + (pi * C::LR + c) * C::CE + 2 * j;
            dst[0] = a0;
            dst[1] = a1;
          }
    }
  }
  named_bar_sync(2, kConsumerWarps * 32);
  const bool aborted = *abort_flag != 0;
  // this split's state of head hh: normalised partial output at column d,
  // running max m (log2 units) and the sum l relative to it
  auto split_state = [&](int hh, int d, float& o_out, float& m_out, float& l_out) {
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
    o_out = (L > 0.f) ? O / L : 0.f;
    m_out = (L > 0.f) ? M : -INFINITY;
    l_out = L;
  };
  if (!a.cluster) {
    if (aborted) return;
    for (int e = threadIdx.x; e < HG * D; e += kConsumerWarps * 32) {
      const int hh = e / D, d = e % D;
      if (grp * HG + hh >= R) continue;
      float ov, mv, lv;
      split_state(hh, d, ov, mv, lv);
      const size_t row = row_index(grp * HG + hh) * a.num_splits + split;
      a.ws_o[row * D + d] = ov;
      if (d == 0) {
        a.ws_ml[2 * row] = mv;
        a.ws_ml[2 * row + 1] = lv;
      }
    }
    return;
  }

  // ---- splits merged inside the cluster.  Every consumer thread meets both
  // cluster barriers, also after a failed wait (the results are then not
  // used: the status word reports the timeout), so that no CTA leaves while
  // another still reads its shared memory.
  float* cpo = wacc + kConsumerWarps * HG * D;  // [HG][D] partial output
  float* cpl = cpo + HG * D;                    // [HG][2] m (log2), l
  float* wts = cpl + 2 * HG;                    // [HG][kMaxClusterSplits]
  float* hinv = wts + HG * kMaxClusterSplits;   // [HG] 1 / L
  for (int e = threadIdx.x; e < HG * D; e += kConsumerWarps * 32) {
    const int hh = e / D, d = e % D;
    float ov = 0.f, mv = -INFINITY, lv = 0.f;
    if (!aborted && grp * HG + hh < R) split_state(hh, d, ov, mv, lv);
    cpo[e] = ov;
    if (d == 0) {
      cpl[2 * hh] = mv;
      cpl[2 * hh + 1] = lv;
    }
  }
  cluster_sync_all();
  const int S = a.num_splits;
  const uint32_t rank = cluster_rank();
  if (threadIdx.x < HG) {
    // weights l_s 2^(m_s - M) of the splits, and the sink in the denominator
    const int hh = threadIdx.x;
    const int rr = grp * HG + hh;
    const bool valid = rr < R;
    const int hq = kvh * a.G + (valid ? rr / a.Lq : 0);
    // all remote loads in flight before any is used
    float mq[kMaxClusterSplits], lq[kMaxClusterSplits];
#pragma unroll
    for (int q = 0; q < kMaxClusterSplits; ++q)
      if (q < S) {
        mq[q] = ld_cluster(cpl + 2 * hh, static_cast<uint32_t>(q));
        lq[q] = ld_cluster(cpl + 2 * hh + 1, static_cast<uint32_t>(q));
      }
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < kMaxClusterSplits; ++q)
      if (q < S) M = fmaxf(M, mq[q]);
    float sk = -INFINITY;
    if (a.sinks && valid) {
      sk = a.sinks[hq] * kLog2e;
      M = fmaxf(M, sk);
    }
    float L = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxClusterSplits; ++q)
      if (q < S) {
        const float w = (lq[q] > 0.f) ? lq[q] * ex2(mq[q] - M) : 0.f;
        wts[hh * kMaxClusterSplits + q] = w;
        L += w;
      }
    if (a.sinks && M != -INFINITY) L += ex2(sk - M);
    hinv[hh] = (L > 0.f) ? 1.f / L : 0.f;
    if (rank == 0 && a.lse && valid && !aborted)
      a.lse[row_index(rr)] =
          (L > 0.f) ? (M + __log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
  named_bar_sync(3, kConsumerWarps * 32);
  const int dpr = D / S;  // output columns of this CTA
  for (int e = threadIdx.x; e < HG * dpr; e += kConsumerWarps * 32) {
    const int hh = e / dpr;
    const int d = static_cast<int>(rank) * dpr + e % dpr;
    const int rr = grp * HG + hh;
    if (rr >= R || aborted) continue;
    float pv[kMaxClusterSplits];  // all remote loads in flight first
#pragma unroll
    for (int q = 0; q < kMaxClusterSplits; ++q)
      if (q < S) pv[q] = ld_cluster(cpo + hh * D + d, static_cast<uint32_t>(q));
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxClusterSplits; ++q)
      if (q < S) acc = fmaf(wts[hh * kMaxClusterSplits + q], pv[q], acc);
    static_cast<T*>(a.o)[b * a.os0 + (kvh * a.G + rr / a.Lq) * a.os1 + (rr % a.Lq) * a.os2 + d] =
        StoreAs<T>::c(acc * hinv[hh]);
  }
  cluster_sync_all();
}

// Host-side launch of one instantiation.  *merged tells the caller whether
// the splits were merged inside a cluster (no combine pass needed).
template <typename T, int D, int HG, int KB>
sdpa_status_t launch_split(SplitArgs a, int batch, cudaStream_t stream, bool* merged) {
  using C = SplitCfg<T, D, HG, KB>;
  auto kern = decode_split_kernel<T, D, HG, KB>;
  const size_t smem = C::smem_bytes(a.stages);
  // rows that are not contiguous: tiled tensor copies when the driver takes
  // the maps (box D x TK, at most 256 elements per side)
  a.use_tma = 0;
  if ((a.ks2 != D || a.vs2 != D) && D <= 256 && C::TK <= 256) {
    const CUtensorMapDataType dt = sizeof(T) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : std::is_same<T, __half>::value
                                       ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t es = static_cast<uint32_t>(sizeof(T));
    const bool okk = encode_tiled_4d(&a.tmK, dt, a.k, D, a.Lk, a.Hkv, batch, es, D, C::TK,
                                     a.ks2, a.ks1, a.ks0, CU_TENSOR_MAP_SWIZZLE_NONE);
    const bool okv = okk && encode_tiled_4d(&a.tmV, dt, a.v, D, a.Lk, a.Hkv, batch, es, D,
                                            C::TK, a.vs2, a.vs1, a.vs0,
                                            CU_TENSOR_MAP_SWIZZLE_NONE);
    a.use_tma = okv ? 1 : 0;
  }
  cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return SDPA_ERR_CUDA;
  dim3 grid(a.num_splits, a.Hkv * a.num_groups, batch);
  if (a.ragged) {
    // at most the plan's waves plus one partial split per (batch, unit) pair
    const long long units = static_cast<long long>(a.Hkv) * a.num_groups;
    long long items = static_cast<long long>(a.num_splits) * units * batch;
    const long long bound = static_cast<long long>(a.slots) *
                                ((units * batch * ((a.Lk + C::TK - 1) / C::TK) +
                                  static_cast<long long>(a.slots) * a.tiles_base - 1) /
                                 (static_cast<long long>(a.slots) * a.tiles_base) + 1) +
                            units * batch;
    if (bound < items) items = bound;
    grid = dim3(static_cast<unsigned>(items), 1, 1);
    a.cluster_ok = 0;
  }
  *merged = false;
  const int S = a.num_splits;
  if (a.cluster_ok && S >= 2 && S <= kMaxClusterSplits && (S & (S - 1)) == 0 && D % S == 0) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // whether such a cluster can be resident at all (once per cluster size)
    static int fits[5] = {0, 0, 0, 0, 0};  // 0 unknown, 1 yes, -1 no
    int li = 0;
    while ((1 << li) < S) ++li;
    if (fits[li] == 0) {
      if (S > 8) cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      int n = 0;
      fits[li] = (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) ? 1 : -1;
      cudaGetLastError();
    }
    if (fits[li] > 0) {
      a.cluster = 1;
      if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return SDPA_ERR_CUDA;
      *merged = true;
      return SDPA_OK;
    }
  }
  a.cluster = 0;
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
sdpa_status_t launch_split_hg(const SplitArgs& a, int batch, cudaStream_t stream, bool* merged) {
  constexpr int KB = keys_per_warp(static_cast<int>(sizeof(T)), D, HG);
  return launch_split<T, D, HG, KB>(a, batch, stream, merged);
}

template <typename T, int D>
sdpa_status_t launch_split_d(const SplitArgs& a, int hg, int batch, cudaStream_t stream,
                             bool* merged) {
  switch (hg) {
    case 1: return launch_split_hg<T, D, 1>(a, batch, stream, merged);
    case 2: return launch_split_hg<T, D, 2>(a, batch, stream, merged);
    case 4: return launch_split_hg<T, D, 4>(a, batch, stream, merged);
    case 8:
      if constexpr (D <= 128) return launch_split_hg<T, D, 8>(a, batch, stream, merged);
      return SDPA_ERR_UNSUPPORTED;
    default: return SDPA_ERR_UNSUPPORTED;
  }
}

template <typename T>
sdpa_status_t launch_split_t(const SplitArgs& a, int D, int hg, int batch, cudaStream_t stream,
                             bool* merged) {
  switch (D) {
    case 64: return launch_split_d<T, 64>(a, hg, batch, stream, merged);
    case 128: return launch_split_d<T, 128>(a, hg, batch, stream, merged);
    case 512: return launch_split_d<T, 512>(a, hg, batch, stream, merged);
    default: return SDPA_ERR_UNSUPPORTED;
  }
}

// Per-dtype entry points (one translation unit each).
sdpa_status_t launch_split_f32(const SplitArgs& a, int D, int hg, int batch, cudaStream_t s,
                              bool* merged);
sdpa_status_t launch_split_f16(const SplitArgs& a, int D, int hg, int batch, cudaStream_t s,
                              bool* merged);
sdpa_status_t launch_split_bf16(const SplitArgs& a, int D, int hg, int batch, cudaStream_t s,
                              bool* merged);

}  // namespace dec
}  // namespace gb300
