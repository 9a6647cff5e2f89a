// decode_tc.cu — single- and few-query attention at head_dim 512 for
// fp16/bf16 on the 5th-generation tensor cores: the split-KV first pass, with
// the query rows of one kv head (its G heads x Lq rows, up to 16) on the
// narrow side of both products.
//
// MLX PR #4459 ("Add D512 support to Metal vector attention") serves
// head_dim-512 single-token decode with vector kernels: one pass, or a first
// pass over chunks of the key range and a second that merges the chunks'
// partial results by their log-sum-exp.  The same two steps run here, but a
// head group's per-key dot products and its value accumulation are two
// skinny matrix products, which on sm_103a belong on tcgen05 with the long
// dimensions on the 128-row side:
//     S^T  = K Q^T     M = 128 keys,             N = 16 rows, K = 512
//     O^T += V^T P^T   M = 128 head dims (x 4),  N = 16 rows, K = 128 keys
// so neither a 128-row O accumulator (512 fp32 columns, all of TMEM) nor Q
// padded to 128 rows is needed: TMEM holds the split's score tiles (16
// columns each) and O^T (64 columns).
//
// One CTA per (split of the key range, half of the head dimensions, kv head,
// batch); a split is at most kMaxTiles tiles of 128 keys.  Both halves of a
// split compute the same scores and probabilities (the S^T products are
// small) and each accumulates its own 256 columns of O, so one CTA holds all
// of a tile's K (128 KB) and half of its V (64 KB) at once: for a split of
// one tile every copy of the CTA is in flight from the start.  Warp 4 loads
// Q (one box per 64 columns: the G heads x Lq rows of the kv head), then the
// split's K tiles, then its V tiles, as 32 KB slots (two 64-column chunks of
// 128 rows, 128-byte swizzle) through a 6-slot ring; warp 5 (one thread)
// issues the MMAs.  Warps 0-3 (thread = TMEM lane: a key of the tile, later
// a head dimension of each 128-block) take the exact row max over the whole
// split from the score tiles left in TMEM, then write P = 2^(x - m) tile by
// tile as the B operand of the value product, and finally read O^T; since
// the max is known before any probability is formed, O is never rescaled.
// The splits' normalised partial outputs and (m, l) of one (half, kv head,
// batch) merge inside a thread-block cluster of the S splits when it can be
// resident: split r sends column slice q of its partial (with the rows'
// (m, l)) by bulk copy into CTA q's inbox, and CTA q merges slice q of every
// row, so the exchange is spread over all S SMs; else they merge through the
// workspace and the combine kernel.  A call with one split writes O
// directly.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "tensor_map.h"

namespace gb300 {
namespace dtc {

constexpr int kD = 512;
constexpr int kDH = 256;                 // head dimensions of O per CTA
constexpr int kTK = 128;                 // keys per tile (rows of S^T)
constexpr int kN = 16;                   // query rows of a kv head, padded
constexpr int kMaxTiles = 4;             // key tiles per split (score tiles in TMEM)
constexpr int kChunkBytes = 128 * 128;   // 128 rows x 64 columns of 2 bytes
constexpr int kSlotBytes = 2 * kChunkBytes;
constexpr int kRing = 5;                 // a tile's 4 K slots and its first V slot
constexpr int kQChunkBytes = kN * 128;   // Q: 8 chunks of kN rows x 64 columns
constexpr int kQBytes = 8 * kQChunkBytes;
constexpr int kPChunkBytes = kN * 128;   // P^T of a tile: 2 chunks of kN rows x 64 keys
constexpr int kPBytes = 2 * kPChunkBytes;
constexpr int kThreads = 192;
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kOCol = kMaxTiles * kN;  // O^T blocks after the score tiles
constexpr int kQOff = 0;
constexpr int kPOff = kQOff + kQBytes;
constexpr int kRingOff = kPOff + kMaxTiles * kPBytes;
constexpr int kInboxOff = kRingOff + kRing * kSlotBytes;
constexpr int kInboxBytes = 32 * 1024;   // the cluster merge's incoming slices
constexpr int kBarOff = kInboxOff + kInboxBytes;
// q_full, full[kRing], empty[kRing], s_full[kMaxTiles], p_ready[kMaxTiles], o_done,
// drain, inbox
constexpr int kNBars = 1 + 2 * kRing + 2 * kMaxTiles + 3;
constexpr int kMiscOff = kBarOff + kNBars * 8;
constexpr int kRedOff = kMiscOff + 16;  // two [4 warps][kN] reduction buffers
constexpr int kSmem = kRedOff + 2 * 4 * kN * 4 + 1024;  // + alignment slack
static_assert(kSmem <= 232448, "shared memory budget");
static_assert(kOCol + 2 * kN <= kTmemCols, "TMEM budget");
static_assert((kPOff % 1024) == 0 && (kRingOff % 1024) == 0, "swizzle atoms 1024-aligned");
constexpr int kMaxCluster = 16;  // splits merged in a cluster (a power of two)
// a slice record: R rows x kDH / S columns of a split's partial output, then
// (m, l) of the kN rows; S records leave and S arrive per CTA
__host__ __device__ constexpr int slice_bytes(int R, int S) { return R * (kDH / S) * 4 + 2 * kN * 4; }
static_assert(2 * slice_bytes(kN, 2) <= kInboxBytes && 16 * slice_bytes(kN, 16) <= kInboxBytes,
              "inbox");
static_assert(2 * slice_bytes(kN, 2) <= kRing * kSlotBytes, "staging");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum Mode { kSingle = 0, kCluster = 1, kTwoPass = 2 };

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
  int mode;
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
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};
template <>
struct Elem<false> {
  using T = __half;
  static __device__ __forceinline__ float f(T x) { return __half2float(x); }
  static __device__ __forceinline__ T c(float x) { return __float2half_rn(x); }
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
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

__device__ __forceinline__ void ld2x16(uint32_t t0, uint32_t t1, uint32_t (&r0)[16],
                                       uint32_t (&r1)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, "
      "%25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r0[0]), "=r"(r0[1]), "=r"(r0[2]), "=r"(r0[3]), "=r"(r0[4]), "=r"(r0[5]),
        "=r"(r0[6]), "=r"(r0[7]), "=r"(r0[8]), "=r"(r0[9]), "=r"(r0[10]), "=r"(r0[11]),
        "=r"(r0[12]), "=r"(r0[13]), "=r"(r0[14]), "=r"(r0[15]), "=r"(r1[0]), "=r"(r1[1]),
        "=r"(r1[2]), "=r"(r1[3]), "=r"(r1[4]), "=r"(r1[5]), "=r"(r1[6]), "=r"(r1[7]),
        "=r"(r1[8]), "=r"(r1[9]), "=r"(r1[10]), "=r"(r1[11]), "=r"(r1[12]), "=r"(r1[13]),
        "=r"(r1[14]), "=r"(r1[15])
      : "r"(t0), "r"(t1)
      : "memory");
}

// Loads from the shared memory of CTA `rank` of the cluster, at the offset of
// `local` in this CTA's.
__device__ __forceinline__ float2 ld_cluster2(const float* local, uint32_t rank) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
               : "=f"(v.x), "=f"(v.y)
               : "r"(cluster_map(local, rank))
               : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster4(const float* local, uint32_t rank) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_map(local, rank))
               : "memory");
  return v;
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

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
// 1 / x to within an ulp (one MUFU operation)
__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <bool BF16, int NR, int S>
__device__ __forceinline__ void cluster_merge(const Args& a, uint8_t* smem, int split, int kvh,
                                              int half, int b, bool ok, const float (&Mr)[NR],
                                              const float (&Lr)[NR], const float (&ov)[2][NR]);

// NR: rows of a kv head the softmax handles (8 or 16; R <= NR); the products
// always carry kN = 16 columns.
template <bool BF16, int NR>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
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
  uint64_t* o_done = p_ready + kMaxTiles;
  uint64_t* drain = o_done + 1;
  uint64_t* inbox_full = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
  float* red_m = reinterpret_cast<float*>(smem + kRedOff);  // [4][kN]
  float* red_l = red_m + 4 * kN;                            // [4][kN]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y >> 1;
  const int half = blockIdx.y & 1;
  const int b = blockIdx.z;
  const bool clustered = a.mode == kCluster;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < kMaxTiles; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_ready[t], 128);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(inbox_full, 1);
    if (clustered)  // every split of the cluster sends this CTA one slice
      mbar_arrive_expect_tx(inbox_full, static_cast<uint32_t>(
                                            a.num_splits * slice_bytes(a.R, a.num_splits)));
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
  // (the inbox barrier's set-up is ordered by the mbarrier-init fence; the
  // matching wait comes before the first copy into a peer)
  if (clustered) cluster_arrive_relaxed();
  // Launched with programmatic stream serialization: the next call's CTAs
  // may start their set-up on idle SMs now; global memory is touched only
  // after the previous grid in the stream has completed.
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

  // softmax-side results, kept for the merge in the common tail
  float Mr[NR], Lr[NR];
  float ov[2][NR];
  bool ok = true;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && ntile > 0) {
      // K tiles (all 512 columns), then V tiles (this half's 256); a slot
      // holds 128 columns of 128 keys as two 64-column chunks.  Keys past Lk
      // read as zero.
      int seq = 0;
      bool pok = true;
      for (int ph = 0; ph < 2 && pok; ++ph) {
        const CUtensorMap* map = ph == 0 ? &tmK : &tmV;
        const int nslot = ph == 0 ? 4 : 2;
        const int col0 = ph == 0 ? 0 : half * kDH;
        for (int t = 0; t < ntile && pok; ++t) {
          if (a.debug_drop_last && ph == 1 && t == ntile - 1) {
            pok = false;
            break;
          }
          const int key = key_begin + t * kTK;
          for (int c = 0; c < nslot; ++c, ++seq) {
            const int s = seq % kRing;
            const int use = seq / kRing;
            if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, wc)) {
              pok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[s], kSlotBytes);
            uint8_t* dst = sRing + s * kSlotBytes;
            tma_load_4d(dst, map, &full[s], col0 + 128 * c, key, kvh, b);
            tma_load_4d(dst + kChunkBytes, map, &full[s], col0 + 128 * c + 64, key, kvh, b);
            last_use[s] = use;
          }
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
      // V^T (A, MN-major: 64-column atoms 16 KB apart, 8-key groups 1024
      // bytes apart; a K step of 16 keys is 2048 bytes) and P^T (B, K-major)
      const uint64_t v_desc = sdesc(smem_addr(sRing), kChunkBytes, 1024, kSwizzle128B);
      const uint64_t p_desc = sdesc(smem_addr(sP), 16, 1024, kSwizzle128B);
      if (ntile > 0) {
        // Q (issued here, beside the producer's K stream): per 64 columns one
        // box of the kv head's G heads x Lq rows, which lands as rows (head,
        // query row) = c of the chunk (rows past R are not written: they only
        // reach score columns that are never read)
        mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(8 * a.R * 128));
        for (int c = 0; c < 8; ++c)
          tma_load_4d(sQ + c * kQChunkBytes, &tmQ, q_full, 64 * c, 0, kvh * a.G, b);
      }
      bool mok = ntile == 0 || mbar_wait(q_full, 0, wc);
      int seq = 0;
      for (int t = 0; t < ntile; ++t) {
        // S^T_t = sum over the 32 column steps of K_t Q^T
        for (int c = 0; c < 4; ++c, ++seq) {
          const int s = seq % kRing;
          mok = mok && mbar_wait(&full[s], static_cast<uint32_t>((seq / kRing) & 1), wc);
          if (mok) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t ko = s * kSlotBytes + (kk >> 2) * kChunkBytes + (kk & 3) * 32;
              const uint32_t qo = (2 * c + (kk >> 2)) * kQChunkBytes + (kk & 3) * 32;
              mma_f16_ss(tmem + t * kN, k_desc + (ko >> 4), q_desc + (qo >> 4), idS,
                         (c > 0 || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit(&empty[s]);
        }
        mma_commit(&s_full[t]);
      }
      for (int t = 0; t < ntile; ++t) {
        // O^T block j += V_t[:, 256 half + 128 j + (0..127)]^T P_t^T.  The
        // tile's waits all come before its products: a wait of this thread
        // between products holds up the issue far longer than it waits.
        const int s0 = seq % kRing, s1 = (seq + 1) % kRing;
        mok = mok && mbar_wait(&p_ready[t], 0, wc);
        mok = mok && mbar_wait(&full[s0], static_cast<uint32_t>((seq / kRing) & 1), wc);
        mok = mok && mbar_wait(&full[s1], static_cast<uint32_t>(((seq + 1) / kRing) & 1), wc);
        if (mok) {
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int s = j == 0 ? s0 : s1;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t vo = s * kSlotBytes + kk * 2048;
              const uint32_t po = t * kPBytes + (kk >> 2) * kPChunkBytes + (kk & 3) * 32;
              mma_f16_ss(tmem + kOCol + j * kN, v_desc + (vo >> 4), p_desc + (po >> 4), idO,
                         (t > 0 || kk > 0) ? 1u : 0u);
            }
          }
        }
        mma_commit(&empty[s0]);
        mma_commit(&empty[s1]);
        seq += 2;
      }
      mma_commit(o_done);
      // every product completes before TMEM is freed
      mma_commit(drain);
      drain_wait(drain, 0, kDrainNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax and epilogue
    const int i = threadIdx.x;  // key of a tile; head dimension of an O^T block
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
    {
      const float v = reduce_lanes<NR, true>(mt, lane);
      if ((lane & (32 / NR - 1)) == 0) red_m[warp * NR + lane / (32 / NR)] = v;
    }
    named_bar_sync(1, 128);
#pragma unroll
    for (int c = 0; c < NR; ++c)
      Mr[c] = fmaxf(fmaxf(red_m[c], red_m[NR + c]), fmaxf(red_m[2 * NR + c], red_m[3 * NR + c]));

    // pass 2: P^T of each tile (B operand: row c, key i at chunk i / 64, row
    // c * 128 bytes, 16-byte unit ((i % 64) / 8) ^ (c % 8)), and the sums.
    // Rows of P^T past NR are not written: they reach only columns of O^T
    // that are never read.
    float lp[NR];
#pragma unroll
    for (int c = 0; c < NR; ++c) lp[c] = 0.f;
#pragma unroll 1
    for (int t = 0; t < ntile; ++t) {
      if (ok) {
        __syncwarp();
        float x[NR];
        scores(t, x);
        uint8_t* pcol = sP + t * kPBytes + (i >> 6) * kPChunkBytes + (i & 7) * 2;
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
      mbar_arrive(&p_ready[t]);
    }
    {
      const float v = reduce_lanes<NR, false>(lp, lane);
      if ((lane & (32 / NR - 1)) == 0) red_l[warp * NR + lane / (32 / NR)] = v;
    }
    named_bar_sync(1, 128);
#pragma unroll
    for (int c = 0; c < NR; ++c)
      Lr[c] = (red_l[c] + red_l[NR + c]) + (red_l[2 * NR + c] + red_l[3 * NR + c]);

    // O^T: thread i holds head dimensions 256 half + i and 256 half + 128 + i
    ok = __all_sync(0xffffffffu, ok && (ntile == 0 || mbar_wait(o_done, 0, wc)));
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int c = 0; c < NR; ++c) ov[j][c] = 0.f;
    if (ok && ntile > 0) {
      tc_fence_after();
      __syncwarp();
      uint32_t r[2][16];
      ld2x16(tmem + lane_off + kOCol, tmem + lane_off + kOCol + kN, r[0], r[1]);
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < NR; ++c) ov[j][c] = __uint_as_float(r[j][c]);
    }
    // normalised partial output (0 where the row saw no key)
#pragma unroll
    for (int c = 0; c < NR; ++c) {
      const bool any = Lr[c] > 0.f;
      const float inv = any ? rcp(Lr[c]) : 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j) ov[j][c] = any ? ov[j][c] * inv : 0.f;
    }

    if (ok && a.mode == kSingle) {
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
          T* orow = static_cast<T*>(a.o) + b * a.os0 + hq * a.os1 + a.row_q[c] * a.os2 +
                    half * kDH + i;
          orow[0] = E::c(ov[0][c] * w);
          orow[128] = E::c(ov[1][c] * w);
          if (half == 0 && i == c && a.lse) {
            const size_t row = (static_cast<size_t>(b) * a.Hq + hq) * a.Lq + a.row_q[c];
            a.lse[row] = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
          }
        }
      }
    } else if (ok && a.mode == kTwoPass) {
#pragma unroll
      for (int c = 0; c < NR; ++c) {
        if (c < a.R) {
          const int hq = kvh * a.G + a.row_h[c];
          const size_t row = (static_cast<size_t>(b) * a.Hq + hq) * a.Lq + a.row_q[c];
          const size_t slot = row * a.num_splits + split;
          float* dst = a.ws_o + slot * kD + half * kDH + i;
          dst[0] = ov[0][c];
          dst[128] = ov[1][c];
          if (half == 0 && i == c) {
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
    // a role gave up: every copy the producer issued lands before the ring
    // is reused and before the CTA exits
    if (ntile > 0) drain_wait(q_full, 0, kDrainNs);
    for (int s = 0; s < kRing; ++s)
      if (last_use[s] >= 0) drain_wait(&full[s], last_use[s] & 1, kDrainNs);
  }
  if (a.mode != kCluster) return;

  __syncthreads();  // the producer's drain precedes the staging below
  switch (a.num_splits) {
    case 2: cluster_merge<BF16, NR, 2>(a, smem, split, kvh, half, b, ok, Mr, Lr, ov); break;
    case 4: cluster_merge<BF16, NR, 4>(a, smem, split, kvh, half, b, ok, Mr, Lr, ov); break;
    case 8: cluster_merge<BF16, NR, 8>(a, smem, split, kvh, half, b, ok, Mr, Lr, ov); break;
    default: cluster_merge<BF16, NR, 16>(a, smem, split, kvh, half, b, ok, Mr, Lr, ov); break;
  }
}

// Splits merged inside the cluster (CTA rank = split r of S).  Each CTA
// stages its normalised partial output as S slice records (R rows x 256/S
// columns, then (m, l) of the rows) in its idle ring, sends record q to CTA
// q's inbox slot r, waits for its own S incoming records and merges column
// slice r of the half for every row: M = max of the m's (and the sink
// logit), weights l_s 2^(m_s - M), O = sum of weight x partial / (sum of
// weights + the sink's), LSE = (M + log2 L) ln 2.  The second cluster
// barrier keeps every CTA alive until all copies have landed (their sources
// are read until then).  Every thread meets both cluster barriers, also
// after a failed wait.
template <bool BF16, int NR, int S>
__device__ __forceinline__ void cluster_merge(const Args& a, uint8_t* smem, int split, int kvh,
                                              int half, int b, bool ok, const float (&Mr)[NR],
                                              const float (&Lr)[NR], const float (&ov)[2][NR]) {
  using E = Elem<BF16>;
  using T = typename E::T;
  constexpr int W = kDH / S;  // columns of a slice
  const int RB = slice_bytes(a.R, S);
  uint8_t* stage = smem + kRingOff;
  uint8_t* inbox = smem + kInboxOff;
  uint64_t* inbox_full = reinterpret_cast<uint64_t*>(smem + kBarOff) + 1 + 2 * kRing +
                         2 * kMaxTiles + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
  const int warp = threadIdx.x >> 5;
  if (warp < 4) {
    const int i = threadIdx.x;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int d = 128 * j + i;  // column of the half
      float* rec = reinterpret_cast<float*>(stage + (d / W) * RB) + (d % W);
#pragma unroll
      for (int c = 0; c < NR; ++c)
        if (c < a.R) rec[c * W] = ok ? ov[j][c] : 0.f;
    }
    if (i < kN) {
      float m = -INFINITY, l = 0.f;
#pragma unroll
      for (int c = 0; c < NR; ++c)
        if (i == c) {
          m = (ok && Lr[c] > 0.f) ? Mr[c] : -INFINITY;
          l = ok ? Lr[c] : 0.f;
        }
#pragma unroll
      for (int q = 0; q < S; ++q) {
        float* ml = reinterpret_cast<float*>(stage + q * RB + a.R * W * 4);
        ml[2 * i] = m;
        ml[2 * i + 1] = l;
      }
    }
    fence_proxy_async_shared();
  }
  __syncthreads();
  cluster_wait();  // every inbox barrier of the cluster is set up
  if (threadIdx.x < S) {
    const uint32_t q = threadIdx.x;
    bulk_copy_to_cluster(cluster_map(inbox + split * RB, q), smem_addr(stage + q * RB),
                         static_cast<uint32_t>(RB), cluster_map(inbox_full, q));
  }
  const WaitCtl wc{a.wait_ns, abort_flag, a.status};
  // bounded by the limit only: copies into this CTA must land before it leaves
  const bool got = __syncthreads_and(mbar_wait_cluster(inbox_full, 0, wc));
  // every copy into this CTA has landed (the peers only learn that their
  // sources are no longer read: no data of this CTA's to publish)
  cluster_arrive_relaxed();
  const bool aborted = *abort_flag != 0;
  if (got && !aborted) {
    constexpr int kQ4 = W / 4;
    for (int task = threadIdx.x; task < a.R * kQ4; task += kThreads) {
      const int c = task / kQ4;
      const int w = 4 * (task % kQ4);
      const int hq = kvh * a.G + a.row_h[c];
      float mq[S], lq[S];
      float M = -INFINITY;
#pragma unroll
      for (int q = 0; q < S; ++q) {
        const float2 ml =
            reinterpret_cast<const float2*>(inbox + q * RB + a.R * W * 4)[c];
        mq[q] = ml.x;
        lq[q] = ml.y;
        M = fmaxf(M, mq[q]);
      }
      float sk = -INFINITY;
      if (a.sinks) {
        sk = a.sinks[hq] * kLog2e;
        M = fmaxf(M, sk);
      }
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < S; ++q) {
        const float wq = (lq[q] > 0.f) ? lq[q] * ex2(mq[q] - M) : 0.f;
        const float4 v = *reinterpret_cast<const float4*>(inbox + q * RB + (c * W + w) * 4);
        L += wq;
        acc.x = fmaf(wq, v.x, acc.x);
        acc.y = fmaf(wq, v.y, acc.y);
        acc.z = fmaf(wq, v.z, acc.z);
        acc.w = fmaf(wq, v.w, acc.w);
      }
      if (a.sinks && M != -INFINITY) L += ex2(sk - M);
      const float inv = (L > 0.f) ? rcp(L) : 0.f;
      T* orow = static_cast<T*>(a.o) + b * a.os0 + hq * a.os1 + a.row_q[c] * a.os2 +
                half * kDH + split * W + w;
      *reinterpret_cast<uint2*>(orow) =
          make_uint2(E::pack(acc.x * inv, acc.y * inv), E::pack(acc.z * inv, acc.w * inv));
      if (split == 0 && half == 0 && w == 0 && a.lse) {
        const size_t row = (static_cast<size_t>(b) * a.Hq + hq) * a.Lq + a.row_q[c];
        a.lse[row] = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
      }
    }
  }
  cluster_wait();
}

}  // namespace dtc

namespace {
// Clusters of `size` CTAs of the kernel that can be resident at once (cached
// per size; a large number when it cannot be asked, e.g. without a device).
int max_active_clusters(int size) {
  static int cache[dtc::kMaxCluster + 1] = {};
  if (size < 2 || size > dtc::kMaxCluster) return 0;
  if (cache[size] != 0) return cache[size];
  auto kern = dtc::decode_tc_kernel<true, 8>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dtc::kSmem);
  cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(size);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(size));
  cfg.blockDim = dim3(dtc::kThreads);
  cfg.dynamicSmemBytes = dtc::kSmem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 1 << 30;  // not cached: asked again once a device is there
  }
  cache[size] = n > 0 ? n : -1;
  return cache[size];
}
}  // namespace

// Plan of the head_dim-512 tensor-core decode: split count and form of the
// merge.  Returns false when the problem is not one for this kernel.
bool decode_tc_plan(const sdpa_params_t& p, int num_sms, DecodePlan* out) {
  const int R = p.num_q_heads / p.num_kv_heads * p.seq_len_q;
  if (p.head_dim != dtc::kD || p.dtype == SDPA_F32 || R > dtc::kN) return false;
  if (2LL * p.num_kv_heads > 65535 || p.batch > 65535) return false;
  const int ntiles = (p.seq_len_kv + dtc::kTK - 1) / dtc::kTK;
  // CTAs of one split: (half, kv head, batch)
  const long long units = 2LL * p.batch * p.num_kv_heads;
  const long long nsm = num_sms > 0 ? num_sms : 152;
  // one CTA per SM: as many splits as fill the GPU, each at most kMaxTiles tiles
  long long want = nsm / (units > 0 ? units : 1);
  if (want < 1) want = 1;
  int S = static_cast<int>(want < ntiles ? want : ntiles);
  const int forced = debug_option(SDPA_DEBUG_DECODE_SPLITS);  // test hook
  if (forced >= 1) S = forced < ntiles ? forced : ntiles;
  if (S < 1) S = 1;
  int tiles_per = (ntiles + S - 1) / S;
  if (tiles_per > dtc::kMaxTiles) tiles_per = dtc::kMaxTiles;
  S = (ntiles + tiles_per - 1) / tiles_per;
  if (S < 1) S = 1;
  // The splits of one (half, kv head, batch) form a cluster (2, 4, 8 or 16
  // CTAs; empty splits past the keys) when all the plan's clusters can be
  // resident at once: the smallest power of two >= S if that fits, else the
  // largest smaller one whose splits stay within kMaxTiles tiles (not for a
  // forced count).
  bool cluster = false;
  if (S > 1 && S <= dtc::kMaxCluster) {
    int c = 2;
    while (c < S) c <<= 1;
    for (; c >= 2; c >>= 1) {
      const int tp = (ntiles + c - 1) / c;
      if (tp <= dtc::kMaxTiles && units <= max_active_clusters(c)) {
        cluster = true;
        S = c;
        tiles_per = tp;
        break;
      }
      if (forced >= 1) break;
    }
  }
  out->head_group = R;
  out->num_groups = 1;
  out->tile_keys = dtc::kTK;
  out->num_splits = S;
  out->split_keys = tiles_per * dtc::kTK;
  out->stages = dtc::kRing;
  out->cluster = cluster;
  out->tc = true;
  out->workspace = 0;
  if (S > 1) {
    const size_t rows = static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q * S;
    out->workspace = ((rows * dtc::kD * sizeof(float) + 255) & ~static_cast<size_t>(255)) +
                     ((rows * 2 * sizeof(float) + 255) & ~static_cast<size_t>(255));
  }
  return true;
}

template <bool BF16>
static sdpa_status_t launch_tc(const sdpa_params_t& p, const DecodePlan& plan, const void* q,
                               const void* k, const void* v, void* o, float* lse, float* ws_o,
                               float* ws_ml, const LaunchEnv& env, bool* merged) {
  using namespace dtc;
  const CUtensorMapDataType dt =
      BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int G = p.num_q_heads / p.num_kv_heads;
  CUtensorMap tq, tk, tv;
  // q as [B, Hq, Lq, 512], box 64 x Lq rows x G heads; k, v as
  // [B, Hkv, Lk, 512], box 64 x 128 rows (rows past Lk read as zero); all
  // with the given strides, innermost first, 128-byte swizzle
  if (!encode_tiled_4d_box(&tq, dt, q, kD, p.seq_len_q, p.num_q_heads, p.batch, 2, 64,
                           static_cast<uint32_t>(p.seq_len_q), static_cast<uint32_t>(G),
                           p.q_stride[2], p.q_stride[1], p.q_stride[0]) ||
      !encode_tiled_4d(&tk, dt, k, kD, p.seq_len_kv, p.num_kv_heads, p.batch, 2, 64, kTK,
                       p.k_stride[2], p.k_stride[1], p.k_stride[0]) ||
      !encode_tiled_4d(&tv, dt, v, kD, p.seq_len_kv, p.num_kv_heads, p.batch, 2, 64, kTK,
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
  a.o = o;
  a.lse = lse;
  a.ws_o = ws_o;
  a.ws_ml = ws_ml;
  a.status = env.status;
  a.wait_ns = env.wait_limit_ns;
  a.debug_drop_last = debug_option(SDPA_DEBUG_DECODE_DROP_LAST) == 1 ? 1 : 0;
  auto kern = a.R <= 8 ? decode_tc_kernel<BF16, 8> : decode_tc_kernel<BF16, 16>;
  static bool attr_set[2] = {false, false};
  if (!attr_set[a.R <= 8]) {
    cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
        cudaSuccess)
      return SDPA_ERR_CUDA;
    cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    attr_set[a.R <= 8] = true;
  }
  const int S = plan.num_splits;
  // cluster merge (test hook: 0 = two passes) when the plan's clusters of S
  // splits and a merging CTA are all resident at once
  const long long nclusters = 2LL * p.num_kv_heads * p.batch;
  const bool clustered = S > 1 && plan.cluster && debug_option(SDPA_DEBUG_DECODE_CLUSTER) != 0 &&
                         S <= kMaxCluster && (S & (S - 1)) == 0 &&
                         nclusters <= max_active_clusters(S);
  const dim3 grid(static_cast<unsigned>(S),
                  static_cast<unsigned>(2 * p.num_kv_heads), static_cast<unsigned>(p.batch));
  // programmatic stream serialization (the kernel waits for the previous
  // grid before it touches global memory), plus the cluster when merging
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(S);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = env.stream;
  cfg.attrs = attr;
  cfg.numAttrs = clustered ? 2 : 1;
  a.mode = S == 1 ? kSingle : clustered ? kCluster : kTwoPass;
  *merged = a.mode != kTwoPass;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, a) == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

sdpa_status_t launch_decode_tc(const sdpa_params_t& p, const DecodePlan& plan, const void* q,
                               const void* k, const void* v, void* o, float* lse, float* ws_o,
                               float* ws_ml, const LaunchEnv& env, bool* merged) {
  if (p.dtype == SDPA_BF16)
    return launch_tc<true>(p, plan, q, k, v, o, lse, ws_o, ws_ml, env, merged);
  if (p.dtype == SDPA_F16)
    return launch_tc<false>(p, plan, q, k, v, o, lse, ws_o, ws_ml, env, merged);
  return SDPA_ERR_UNSUPPORTED;
}

}  // namespace gb300
