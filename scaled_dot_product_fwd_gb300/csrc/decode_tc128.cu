// decode_tc128.cu — single- and few-query attention at head_dim 128 (and
// 64) for fp16/bf16 on the 5th-generation tensor cores: the split-KV first
// pass of long key ranges (KV-cache decode), with the query rows of one kv
// head (its G heads x Lq rows, up to 16) on the narrow side of both products.
//
// The method is the two-pass split-KV attention of MLX PR #4459 ("Add D512
// support to Metal vector attention"): a first pass over chunks of the key
// range, each leaving its normalised partial output and log-sum-exp, and a
// second pass that merges the chunks by their log-sum-exp (the combine
// kernel).  With G query heads per kv head, a split's per-key dot products
// and its value accumulation are two skinny matrix products,
//     S^T  = K Q^T     M = 128 keys,       N = 16 rows, K = D
//     O^T += V^T P^T   M = 128 head dims,  N = 16 rows, K = 128 keys
// (at D = 64 the second 64 rows of V^T are the slot's unused half: those
// rows of O^T are never read)
// which leave the CUDA cores nothing per key but the exponential: a vector
// kernel spends about 250 FMAs of dot products and accumulation per (key,
// head) and cannot stream K and V faster than its arithmetic, while here the
// pass is bound by the copies.
//
// One CTA per (split of at most kMaxTiles tiles of 128 keys, kv head,
// batch), two CTAs per SM (256 TMEM columns and 110 KB of shared memory
// each).  Warp 4 loads Q (one box per 64 columns), then the split's K tiles,
// then its V tiles, through a 3-slot ring of 32 KB (a tile: D / 64 chunks of
// 64 columns and 128 rows, 128-byte swizzle); warp 5 (one thread) issues the
// MMAs.  Every score tile of the split stays in TMEM (16 columns each), so
// warps 0-3 (thread = TMEM lane: a key of the tile, later a head dimension of
// O^T) take the exact row max over the whole split before any probability is
// formed, and O is never rescaled; they then write P = 2^(x - m) tile by
// tile (two buffers) as the B operand of the value product, and finally read
// O^T.  A split past a batch's key count (per-batch lengths) leaves an empty
// partial result (m = -inf, l = 0), which the combine weighs as zero.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "tensor_map.h"

namespace gb300 {
namespace dtc128 {

constexpr int kTK = 128;                 // keys per tile (rows of S^T)
constexpr int kN = 16;                   // query rows of a kv head, padded
constexpr int kMaxTiles = 14;            // key tiles per split (score tiles in TMEM)
constexpr int kChunkBytes = 128 * 128;   // 128 rows x 64 columns of 2 bytes
constexpr int kSlotBytes = 2 * kChunkBytes;  // a K or V tile (two chunks at D = 128)
constexpr int kRing = 3;
constexpr int kQChunkBytes = kN * 128;   // Q: D / 64 chunks of kN rows x 64 columns
constexpr int kQBytes = 2 * kQChunkBytes;
constexpr int kPChunkBytes = kN * 128;   // P^T of a tile: 2 chunks of kN rows x 64 keys
constexpr int kPBytes = 2 * kPChunkBytes;
constexpr int kPBufs = 2;
constexpr int kThreads = 192;
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kOCol = kMaxTiles * kN;  // O^T after the score tiles
constexpr int kQOff = 0;
constexpr int kPOff = kQOff + kQBytes;
constexpr int kRingOff = kPOff + kPBufs * kPBytes;
constexpr int kBarOff = kRingOff + kRing * kSlotBytes;
// q_full, full[kRing], empty[kRing], s_full[kMaxTiles], p_ready[kPBufs],
// p_free[kPBufs], o_done, drain
constexpr int kNBars = 1 + 2 * kRing + kMaxTiles + 2 * kPBufs + 2;
constexpr int kMiscOff = kBarOff + kNBars * 8;
constexpr int kRedOff = kMiscOff + 16;  // two [4 warps][kN] reduction buffers
constexpr int kSmem = kRedOff + 2 * 4 * kN * 4 + 1024;  // + alignment slack
static_assert(2 * (kSmem + 1024) <= 233472, "two CTAs per SM");
static_assert(kOCol + kN <= kTmemCols && 2 * kTmemCols <= 512, "TMEM budget");
static_assert((kPOff % 1024) == 0 && (kRingOff % 1024) == 0, "swizzle atoms 1024-aligned");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Args {
  int Hq, Hkv, G, Lq, Lk;
  int R;                     // rows per kv head (G x Lq <= kN)
  // row c of a kv head: head kvh * G + row_h[c], query row row_q[c]; its
  // mask row at element offset row_moff[c] from the (batch, kv head) base
  int row_h[kN];
  int row_q[kN];
  long long row_moff[kN];
  int causal;                // bottom-right: key j visible to row i iff j <= i + Lk - Lq
  long long os0, os1, os2;   // element strides of o (batch, head, row)
  const void* mask;
  long long ms0, ms1, ms2;   // mask element strides (key stride 1)
  int mask_bool;             // mask holds bytes, nonzero = visible
  const int* seq_lens_q;
  const int* seq_lens_kv;
  const float* sinks;
  float sl2;                 // scale * log2(e)
  int num_splits;
  int split_keys;            // multiple of kTK, at most kMaxTiles * kTK
  int single;                // one split: O and LSE directly
  void* o;
  float* lse;
  float* ws_o;   // two-pass: [B, Hq, Lq][splits][D] normalised partial outputs
  float* ws_ml;  // two-pass: [B, Hq, Lq][splits][2] (m in log2 units, l)
  int* status;
  unsigned long long wait_ns;
  int debug_drop_last;  // test hook: the producer skips the last V tile
};

template <bool BF16>
struct Elem;
template <>
struct Elem<true> {
  using T = __nv_bfloat16;
  static __device__ __forceinline__ float f(T x) { return __bfloat162float(x); }
  static __device__ __forceinline__ T c(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct Elem<false> {
  using T = __half;
  static __device__ __forceinline__ float f(T x) { return __half2float(x); }
  static __device__ __forceinline__ T c(float x) { return __float2half_rn(x); }
};

// TMEM load of 16 columns: thread t of the warp receives row (lane quarter
// base + t), columns [col, col + 16).  Load and wait form one statement.
__device__ __forceinline__ void ld16(uint32_t t0, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(t0)
      : "memory");
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) break;
  }
}

// Butterfly reduce-scatter of NV values over the 32 lanes of a warp (max or
// sum): afterwards lane l holds the reduction of value l >> (5 - log2 NV)
// over the warp.
template <int NV, bool kMax>
__device__ __forceinline__ float reduce_lanes(float (&v)[NV], int lane) {
  constexpr int LOG = NV == 16 ? 4 : NV == 8 ? 3 : NV == 4 ? 2 : NV == 2 ? 1 : 0;
  static_assert((1 << LOG) == NV, "power of two");
#pragma unroll
  for (int lev = 0; lev < LOG; ++lev) {
    const int n = NV >> lev;   // values still held
    const int msk = 16 >> lev;
    const bool upper = (lane & msk) != 0;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float send = upper ? v[k] : v[k + n / 2];
      const float keep = upper ? v[k + n / 2] : v[k];
      const float got = __shfl_xor_sync(0xffffffffu, send, msk);
      v[k] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int msk = 16 >> LOG; msk >= 1; msk >>= 1) {
    const float got = __shfl_xor_sync(0xffffffffu, v[0], msk);
    v[0] = kMax ? fmaxf(v[0], got) : v[0] + got;
  }
  return v[0];
}

// 1 / x to within an ulp (one MUFU operation)
__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// D: head_dim (64 or 128).  NR: rows of a kv head the softmax handles (8 or
// 16; R <= NR); the products always carry kN = 16 columns.
template <int D, bool BF16, int NR>
__global__ void __launch_bounds__(kThreads, 2)
    decode_tc128_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const Args a) {
  using E = Elem<BF16>;
  using T = typename E::T;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sQ = smem + kQOff;
  uint8_t* sP = smem + kPOff;
  uint8_t* sRing = smem + kRingOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* q_full = bars;
  uint64_t* full = bars + 1;
  uint64_t* empty = full + kRing;
  uint64_t* s_full = empty + kRing;
  uint64_t* p_ready = s_full + kMaxTiles;
  uint64_t* p_free = p_ready + kPBufs;
  uint64_t* o_done = p_free + kPBufs;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
  float* red_m = reinterpret_cast<float*>(smem + kRedOff);  // [4][kN]
  float* red_l = red_m + 4 * kN;                            // [4][kN]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < kMaxTiles; ++t) mbar_init(&s_full[t], 1);
    for (int j = 0; j < kPBufs; ++j) {
      mbar_init(&p_ready[j], 128);
      mbar_init(&p_free[j], 1);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProdWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched with programmatic stream serialization: the next grid in the
  // stream may start its set-up on idle SMs now; global memory is touched
  // only after the previous grid has completed.
  griddep_launch_dependents();
  griddep_wait();
  const int Lkb = a.seq_lens_kv ? min(max(a.seq_lens_kv[b], 0), a.Lk) : a.Lk;
  const int Lqb = a.seq_lens_q ? min(max(a.seq_lens_q[b], 0), a.Lq) : a.Lq;
  const int key_begin = split * a.split_keys;
  const int key_end = min(Lkb, key_begin + a.split_keys);
  const int nkeys = max(0, key_end - key_begin);
  const int ntile = (nkeys + kTK - 1) / kTK;
  const WaitCtl wc{a.wait_ns, abort_flag, a.status};
  int last_use[kRing];  // producer: last fill of each slot (-1: none)
#pragma unroll
  for (int s = 0; s < kRing; ++s) last_use[s] = -1;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && ntile > 0) {
      // Q: per 64 columns one box of the kv head's G heads x Lq rows, which
      // lands as rows (head, query row) = c of the chunk (rows past R are
      // not written: they only reach score columns that are never read)
      mbar_arrive_expect_tx(q_full, static_cast<uint32_t>((D / 64) * a.R * 128));
      for (int c = 0; c < D / 64; ++c)
        tma_load_4d(sQ + c * kQChunkBytes, &tmQ, q_full, 64 * c, 0, kvh * a.G, b);
      // the split's K tiles, then its V tiles; keys past Lk read as zero
      int seq = 0;
      bool pok = true;
      for (int ph = 0; ph < 2 && pok; ++ph) {
        const CUtensorMap* map = ph == 0 ? &tmK : &tmV;
        for (int t = 0; t < ntile; ++t, ++seq) {
          if (a.debug_drop_last && ph == 1 && t == ntile - 1) {
            pok = false;
            break;
          }
          const int s = seq % kRing;
          const int use = seq / kRing;
          if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, wc)) {
            pok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>((D / 64) * kChunkBytes));
          uint8_t* dst = sRing + s * kSlotBytes;
          const int key = key_begin + t * kTK;
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(dst + c * kChunkBytes, map, &full[s], 64 * c, key, kvh, b);
          last_use[s] = use;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_f16(BF16, 128, kN, false, false);
      constexpr uint32_t idO = idesc_f16(BF16, 128, kN, true, false);
      // K (A, K-major: 128 key rows of 128 bytes) and Q (B, K-major: kN
      // rows); a K step of 16 elements is 32 bytes inside the swizzled rows
      const uint64_t k_desc = sdesc(smem_addr(sRing), 16, 1024, kSwizzle128B);
      const uint64_t q_desc = sdesc(smem_addr(sQ), 16, 1024, kSwizzle128B);
      // V^T (A, MN-major: the two 64-column atoms 16 KB apart, 8-key groups
      // 1024 bytes apart; a K step of 16 keys is 2048 bytes; at D = 64 the
      // second atom is the slot's unused half) and P^T (B, K-major)
      const uint64_t v_desc = sdesc(smem_addr(sRing), kChunkBytes, 1024, kSwizzle128B);
      const uint64_t p_desc = sdesc(smem_addr(sP), 16, 1024, kSwizzle128B);
      bool mok = ntile == 0 || mbar_wait(q_full, 0, wc);
      int seq = 0;
      for (int t = 0; t < ntile; ++t, ++seq) {
        // S^T_t = K_t Q^T over the D / 16 column steps
        const int s = seq % kRing;
        mok = mok && mbar_wait(&full[s], static_cast<uint32_t>((seq / kRing) & 1), wc);
        if (mok) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = s * kSlotBytes + (kk >> 2) * kChunkBytes + (kk & 3) * 32;
            const uint32_t qo = (kk >> 2) * kQChunkBytes + (kk & 3) * 32;
            mma_f16_ss(tmem + t * kN, k_desc + (ko >> 4), q_desc + (qo >> 4), idS,
                       kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(&empty[s]);
        mma_commit(&s_full[t]);
      }
      for (int t = 0; t < ntile; ++t, ++seq) {
        // O^T += V_t^T P_t^T.  Both waits come before the tile's products.
        const int s = seq % kRing;
        const int pb = t & 1;
        mok = mok && mbar_wait(&p_ready[pb], static_cast<uint32_t>((t >> 1) & 1), wc);
        mok = mok && mbar_wait(&full[s], static_cast<uint32_t>((seq / kRing) & 1), wc);
        if (mok) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t vo = s * kSlotBytes + kk * 2048;
            const uint32_t po = pb * kPBytes + (kk >> 2) * kPChunkBytes + (kk & 3) * 32;
            mma_f16_ss(tmem + kOCol, v_desc + (vo >> 4), p_desc + (po >> 4), idO,
                       (t > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&empty[s]);
        mma_commit(&p_free[pb]);
      }
      mma_commit(o_done);
      // every product completes before TMEM is freed
      mma_commit(drain);
      drain_wait(drain, 0, kDrainNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax and epilogue
    const int i = threadIdx.x;  // key of a tile; head dimension of O^T
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    // row c of the kv head: head kvh * G + c / Lq, query row c % Lq.  Last
    // key each row sees (split end, bounds, the causal rule, padding rows;
    // -1 for the padding columns past R).
    int lim[NR];
#pragma unroll
    for (int c = 0; c < NR; ++c) {
      const int qi = a.row_q[c];
      int l = key_end - 1;
      if (a.causal) l = min(l, qi + (Lkb - Lqb));
      if (qi >= Lqb) l = -1;
      lim[c] = (c < a.R) ? l : -1;
    }
    const long long mbase = b * a.ms0 + static_cast<long long>(kvh) * a.G * a.ms1;
    const float mhuge = mask_huge_log2(a.sl2);
    // log2-domain scores of the NR rows at this thread's key of tile t (-inf
    // where not visible).  The mask test is hoisted out of the column loops:
    // a lane-dependent branch per column costs far more than the column.
    auto scores = [&](int t, float (&x)[NR]) {
      uint32_t sv[16];
      ld16(tmem + lane_off + t * kN, sv);
      const int key = key_begin + t * kTK + i;
      if (a.mask == nullptr) {
#pragma unroll
        for (int c = 0; c < NR; ++c)
          x[c] = key <= lim[c] ? __uint_as_float(sv[c]) * a.sl2 : -INFINITY;
      } else if (a.mask_bool) {
        const uint8_t* mb = static_cast<const uint8_t*>(a.mask) + mbase + key;
#pragma unroll
        for (int c = 0; c < NR; ++c) {
          const bool vis = key <= lim[c];
          const uint8_t m = vis ? mb[a.row_moff[c]] : 0;
          x[c] = m ? __uint_as_float(sv[c]) * a.sl2 : -INFINITY;
        }
      } else {
        const T* mt = static_cast<const T*>(a.mask) + mbase + key;
#pragma unroll
        for (int c = 0; c < NR; ++c) {
          const bool vis = key <= lim[c];
          const float mv = vis ? mask_log2(E::f(mt[a.row_moff[c]]), mhuge) : 0.f;
          x[c] = vis ? fmaf(__uint_as_float(sv[c]), a.sl2, mv) : -INFINITY;
        }
      }
    };

    bool ok = true;
    // pass 1: the exact max of every row over the split
    float mt[NR];
#pragma unroll
    for (int c = 0; c < NR; ++c) mt[c] = -INFINITY;
#pragma unroll 1
    for (int t = 0; t < ntile; ++t) {
      ok = __all_sync(0xffffffffu, ok && mbar_wait(&s_full[t], 0, wc));
      if (!ok) break;
      tc_fence_after();
      __syncwarp();
      float x[NR];
      scores(t, x);
#pragma unroll
      for (int c = 0; c < NR; ++c) mt[c] = fmaxf(mt[c], x[c]);
    }
    float Mr[NR], Lr[NR];
    {
      const float v = reduce_lanes<NR, true>(mt, lane);
      if ((lane & (32 / NR - 1)) == 0) red_m[warp * NR + lane / (32 / NR)] = v;
    }
    named_bar_sync(1, 128);
#pragma unroll
    for (int c = 0; c < NR; ++c)
      Mr[c] = fmaxf(fmaxf(red_m[c], red_m[NR + c]), fmaxf(red_m[2 * NR + c], red_m[3 * NR + c]));

    // pass 2: P^T of each tile into buffer t & 1 (B operand: row c, key i at
    // chunk i / 64, row c * 128 bytes, 16-byte unit ((i % 64) / 8) ^ (c % 8)),
    // and the sums.  Rows of P^T past NR are not written: they reach only
    // columns of O^T that are never read.
    float lp[NR];
#pragma unroll
    for (int c = 0; c < NR; ++c) lp[c] = 0.f;
#pragma unroll 1
    for (int t = 0; t < ntile; ++t) {
      const int pb = t & 1;
      // the buffer's previous tile (t - 2) has been read by its products
      if (t >= 2)
        ok = __all_sync(0xffffffffu,
                        ok && mbar_wait(&p_free[pb], static_cast<uint32_t>(((t >> 1) - 1) & 1), wc));
      if (ok) {
        tc_fence_after();
        __syncwarp();
        float x[NR];
        scores(t, x);
        uint8_t* pcol = sP + pb * kPBytes + (i >> 6) * kPChunkBytes + (i & 7) * 2;
        const int unit = (i & 63) >> 3;
#pragma unroll
        for (int c = 0; c < NR; ++c) {
          const float p = (x[c] == -INFINITY) ? 0.f : ex2(x[c] - Mr[c]);
          lp[c] += p;
          *reinterpret_cast<T*>(pcol + c * 128 + ((unit ^ (c & 7)) << 4)) = E::c(p);
        }
        fence_proxy_async_shared();
      }
      // every thread arrives every tile, also after a failed wait
      mbar_arrive(&p_ready[pb]);
    }
    {
      const float v = reduce_lanes<NR, false>(lp, lane);
      if ((lane & (32 / NR - 1)) == 0) red_l[warp * NR + lane / (32 / NR)] = v;
    }
    named_bar_sync(1, 128);
#pragma unroll
    for (int c = 0; c < NR; ++c)
      Lr[c] = (red_l[c] + red_l[NR + c]) + (red_l[2 * NR + c] + red_l[3 * NR + c]);

    // O^T: thread i holds head dimension i of the NR rows (i < D)
    ok = __all_sync(0xffffffffu, ok && (ntile == 0 || mbar_wait(o_done, 0, wc)));
    float ov[NR];
#pragma unroll
    for (int c = 0; c < NR; ++c) ov[c] = 0.f;
    if (ok && ntile > 0) {
      tc_fence_after();
      __syncwarp();
      uint32_t r[16];
      ld16(tmem + lane_off + kOCol, r);
#pragma unroll
      for (int c = 0; c < NR; ++c) ov[c] = __uint_as_float(r[c]);
    }
    // normalised partial output (0 where the row saw no key)
#pragma unroll
    for (int c = 0; c < NR; ++c) {
      const bool any = Lr[c] > 0.f;
      ov[c] = any ? ov[c] * rcp(Lr[c]) : 0.f;
    }

    if (ok && a.single) {
      // one split: the sink logit joins the denominator, then O and LSE
#pragma unroll
      for (int c = 0; c < NR; ++c) {
        if (c < a.R) {
          const int hq = kvh * a.G + a.row_h[c];
          float M = Lr[c] > 0.f ? Mr[c] : -INFINITY;
          float L = Lr[c];
          float f = 1.f;
          if (a.sinks) {
            const float sk = a.sinks[hq] * kLog2e;
            const float mn = fmaxf(M, sk);
            f = (M == -INFINITY) ? 0.f : ex2(M - mn);
            L = L * f + ex2(sk - mn);
            M = mn;
          }
          const float w = (L > 0.f && Lr[c] > 0.f) ? Lr[c] * f * rcp(L) : 0.f;
          T* orow = static_cast<T*>(a.o) + b * a.os0 + hq * a.os1 + a.row_q[c] * a.os2 + i;
          if (i < D) orow[0] = E::c(ov[c] * w);
          if (i == c && a.lse) {
            const size_t row = (static_cast<size_t>(b) * a.Hq + hq) * a.Lq + a.row_q[c];
            a.lse[row] = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
          }
        }
      }
    } else if (ok) {
#pragma unroll
      for (int c = 0; c < NR; ++c) {
        if (c < a.R) {
          const int hq = kvh * a.G + a.row_h[c];
          const size_t row = (static_cast<size_t>(b) * a.Hq + hq) * a.Lq + a.row_q[c];
          const size_t slot = row * a.num_splits + split;
          if (i < D) a.ws_o[slot * D + i] = ov[c];
          if (i == c) {
            a.ws_ml[2 * slot] = Lr[c] > 0.f ? Mr[c] : -INFINITY;
            a.ws_ml[2 * slot + 1] = Lr[c];
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ common tail
  __syncwarp();
  tc_fence_before();
  __syncthreads();  // every TMEM read and every product is done
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (warp == kProdWarp && lane == 0 && *abort_flag) {
    // a role gave up: every copy the producer issued lands before the CTA
    // exits
    if (ntile > 0) drain_wait(q_full, 0, kDrainNs);
    for (int s = 0; s < kRing; ++s)
      if (last_use[s] >= 0) drain_wait(&full[s], last_use[s] & 1, kDrainNs);
  }
}

}  // namespace dtc128

// Whether the tensor-core pass takes a decode problem: head_dim 64 or 128,
// fp16 or bf16, up to 16 rows per kv head, and q, k, v strides that a tensor map
// takes (positive multiples of 16 bytes, the dense layout when the caller
// gave none).
static bool tc128_fits(const sdpa_params_t& p) {
  if ((p.head_dim != 64 && p.head_dim != 128) || p.dtype == SDPA_F32) return false;
  const int R = p.num_q_heads / p.num_kv_heads * p.seq_len_q;
  if (R > dtc128::kN || p.num_kv_heads > 65535 || p.batch > 65535) return false;
  if (debug_option(SDPA_DEBUG_DECODE_VECTOR) == 1) return false;  // test hook
  const sdpa_params_t n = normalized_params(p);
  const int64_t* st[3] = {n.q_stride, n.k_stride, n.v_stride};
  for (const int64_t* s : st)
    for (int i = 0; i < 3; ++i)
      if (s[i] <= 0 || (s[i] % 8) != 0 || s[i] >= (int64_t(1) << 38)) return false;
  return true;
}

// Plan of the tensor-core decode at head_dim 64/128: as many splits per (kv head,
// batch) as one wave of two CTAs per SM holds, each at most kMaxTiles tiles
// (more splits, in further waves, where that bound requires), the tiles
// spread evenly over the splits.  Returns false when the problem is not one
// for this kernel.
bool decode_tc128_plan(const sdpa_params_t& p, int num_sms, DecodePlan* out) {
  if (!tc128_fits(p)) return false;
  const int R = p.num_q_heads / p.num_kv_heads * p.seq_len_q;
  const int ntiles = (p.seq_len_kv + dtc128::kTK - 1) / dtc128::kTK;
  const long long units = static_cast<long long>(p.batch) * p.num_kv_heads;
  const long long slots = 2LL * (num_sms > 0 ? num_sms : 152);
  const long long fill = slots / (units > 0 ? units : 1);
  int S = static_cast<int>(fill < ntiles ? fill : ntiles);
  const int forced = debug_option(SDPA_DEBUG_DECODE_SPLITS);  // test hook
  if (forced >= 1) S = forced < ntiles ? forced : ntiles;
  if (S < 1) S = 1;
  int tiles_per = (ntiles + S - 1) / S;
  if (tiles_per > dtc128::kMaxTiles) tiles_per = dtc128::kMaxTiles;
  if (tiles_per < 1) tiles_per = 1;
  S = (ntiles + tiles_per - 1) / tiles_per;
  if (S < 1) S = 1;
  tiles_per = (ntiles + S - 1) / S;  // the same count of splits, evenly filled
  if (tiles_per < 1) tiles_per = 1;
  out->head_group = R;
  out->num_groups = 1;
  out->tile_keys = dtc128::kTK;
  out->num_splits = S;
  out->split_keys = tiles_per * dtc128::kTK;
  out->stages = dtc128::kRing;
  out->cluster = false;
  out->ragged = false;
  out->tc = false;
  out->tc128 = true;
  out->workspace = 0;
  if (S > 1) {
    const size_t rows = static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q * S;
    out->workspace = ((rows * p.head_dim * sizeof(float) + 255) & ~static_cast<size_t>(255)) +
                     ((rows * 2 * sizeof(float) + 255) & ~static_cast<size_t>(255));
  }
  return true;
}

template <int D, bool BF16>
static sdpa_status_t launch_tc128(const sdpa_params_t& p, const DecodePlan& plan, const void* q,
                                  const void* k, const void* v, void* o, float* lse,
                                  float* ws_o, float* ws_ml, const LaunchEnv& env,
                                  bool* merged) {
  using namespace dtc128;
  const CUtensorMapDataType dt =
      BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int G = p.num_q_heads / p.num_kv_heads;
  CUtensorMap tq, tk, tv;
  // q as [B, Hq, Lq, D], box 64 x Lq rows x G heads; k, v as
  // [B, Hkv, Lk, D], box 64 x 128 rows (rows past Lk read as zero); all
  // with the given strides, innermost first, 128-byte swizzle
  if (!encode_tiled_4d_box(&tq, dt, q, D, p.seq_len_q, p.num_q_heads, p.batch, 2, 64,
                           static_cast<uint32_t>(p.seq_len_q), static_cast<uint32_t>(G),
                           p.q_stride[2], p.q_stride[1], p.q_stride[0]) ||
      !encode_tiled_4d(&tk, dt, k, D, p.seq_len_kv, p.num_kv_heads, p.batch, 2, 64, kTK,
                       p.k_stride[2], p.k_stride[1], p.k_stride[0]) ||
      !encode_tiled_4d(&tv, dt, v, D, p.seq_len_kv, p.num_kv_heads, p.batch, 2, 64, kTK,
                       p.v_stride[2], p.v_stride[1], p.v_stride[0]))
    return SDPA_ERR_CUDA;
  Args a;
  a.Hq = p.num_q_heads;
  a.Hkv = p.num_kv_heads;
  a.G = G;
  a.Lq = p.seq_len_q;
  a.Lk = p.seq_len_kv;
  a.R = G * p.seq_len_q;
  for (int c = 0; c < kN; ++c) {
    const int h = c < a.R ? c / p.seq_len_q : 0, qi = c < a.R ? c % p.seq_len_q : 0;
    a.row_h[c] = h;
    a.row_q[c] = qi;
    a.row_moff[c] = h * p.mask_stride[1] + qi * p.mask_stride[2];
  }
  a.causal = p.causal ? 1 : 0;
  a.os0 = p.o_stride[0];
  a.os1 = p.o_stride[1];
  a.os2 = p.o_stride[2];
  a.mask = p.mask;
  a.ms0 = p.mask_stride[0];
  a.ms1 = p.mask_stride[1];
  a.ms2 = p.mask_stride[2];
  a.mask_bool = (p.flags & SDPA_FLAG_BOOL_MASK) ? 1 : 0;
  a.seq_lens_q = p.seq_lens_q;
  a.seq_lens_kv = p.seq_lens_kv;
  a.sinks = p.sinks;
  a.sl2 = p.scale * kLog2e;
  a.num_splits = plan.num_splits;
  a.split_keys = plan.split_keys;
  a.single = plan.num_splits == 1 ? 1 : 0;
  a.o = o;
  a.lse = lse;
  a.ws_o = ws_o;
  a.ws_ml = ws_ml;
  a.status = env.status;
  a.wait_ns = env.wait_limit_ns;
  a.debug_drop_last = debug_option(SDPA_DEBUG_DECODE_DROP_LAST) == 1 ? 1 : 0;
  auto kern = a.R <= 8 ? decode_tc128_kernel<D, BF16, 8> : decode_tc128_kernel<D, BF16, 16>;
  static bool attr_set[2] = {false, false};
  if (!attr_set[a.R <= 8]) {
    cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
        cudaSuccess)
      return SDPA_ERR_CUDA;
    attr_set[a.R <= 8] = true;
  }
  // programmatic stream serialization (the kernel waits for the previous
  // grid before it touches global memory)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan.num_splits),
                     static_cast<unsigned>(p.num_kv_heads), static_cast<unsigned>(p.batch));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = env.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  *merged = plan.num_splits == 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, a) == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

sdpa_status_t launch_decode_tc128(const sdpa_params_t& p, const DecodePlan& plan, const void* q,
                                  const void* k, const void* v, void* o, float* lse,
                                  float* ws_o, float* ws_ml, const LaunchEnv& env,
                                  bool* merged) {
  const bool bf16 = p.dtype == SDPA_BF16;
  if (p.dtype != SDPA_BF16 && p.dtype != SDPA_F16) return SDPA_ERR_UNSUPPORTED;
  if (p.head_dim == 128)
    return bf16 ? launch_tc128<128, true>(p, plan, q, k, v, o, lse, ws_o, ws_ml, env, merged)
                : launch_tc128<128, false>(p, plan, q, k, v, o, lse, ws_o, ws_ml, env, merged);
  if (p.head_dim == 64)
    return bf16 ? launch_tc128<64, true>(p, plan, q, k, v, o, lse, ws_o, ws_ml, env, merged)
                : launch_tc128<64, false>(p, plan, q, k, v, o, lse, ws_o, ws_ml, env, merged);
  return SDPA_ERR_UNSUPPORTED;
}

}  // namespace gb300
