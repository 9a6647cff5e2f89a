// prefill_d512.cu — fused attention forward at head_dim 512 for fp16/bf16
// and more query rows than the vector path takes, on the 5th-generation
// tensor cores of sm_103a.
//
// MLX PR #4459 ("Add D512 support to Metal vector attention") brings
// head_dim 512 to the vector kernels for single-token decode and leaves
// longer query blocks to the fused path; this kernel is that fused path.
// It computes the tiled online softmax of the rustytorch
// flash_attention.metal forward kernel (per key tile: row max, running max
// m and sum l, accumulator rescale by 2^(m_old - m_new), final O / l and
// LSE = m + log l) with causal block skipping, bounds masking, additive and
// boolean masks, per-head sinks and grouped-query heads.
//
// GB300 design: a 128 x 512 fp32 output tile alone would fill the 512 TMEM
// columns, so each CTA owns one D-half: (query tile of 128 rows, half, head,
// batch).  TMEM holds two S buffers (128 columns each) and the CTA's half
// of O (256 columns); both halves of a query tile compute the same S and
// softmax (the price of the split is S computed twice: 1.5x the MMA work of
// the definition).
// Q (128 rows x 512, 128 KB) stays in shared memory as eight 128-byte
// swizzled chunks of 64 columns; the producer streams K_j (eight chunks)
// before V_{j-1} (the half's four chunks) through a ring of three 32 KB
// slots, two chunks a slot.  Warps: 0-3 softmax (one query row per thread =
// TMEM lane), 4 TMA producer, 5 MMA issuer (one thread): S_j = sum_c Q_c K_c^T
// (M128 N128 K16) into TMEM buffer j % 2, then O_half += P_{j-1} V_{j-1}
// (P from TMEM, four N64 column blocks), so that S_j runs while the softmax
// warps work on S_{j-1}.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "tensor_map.h"

namespace gb300 {
namespace {

constexpr int kD = 512;
constexpr int kBM = 128;                 // query rows per tile (TMEM lanes)
constexpr int kBN = 128;                 // keys per tile
constexpr int kDH = 256;                 // output columns per CTA
constexpr int kChunkCols = 64;           // columns of one 128-byte swizzled chunk
constexpr int kChunkBytes = 128 * 128;   // 128 rows x 128 bytes
constexpr int kQChunks = kD / kChunkCols;    // 8
constexpr int kVChunks = kDH / kChunkCols;   // 4
// The ring moves chunks in pairs (a slot holds two chunks of one operand):
// the issuing thread's wait on a slot costs it hundreds of clk of issue while
// products are in flight, so fewer, larger slots (same 96 KB) halve those
// waits.
constexpr int kSlotBytes = 2 * kChunkBytes;
constexpr int kKSlots = kQChunks / 2;                 // 4
constexpr int kVSlots = kVChunks / 2;                 // 2
constexpr int kStepSlots = kKSlots + kVSlots;         // per key tile: K slots, then V slots
constexpr int kRing = 3;
constexpr int kThreads = 192;
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;      // allocation (power of two)
constexpr uint32_t kSCol = 0;            // S of tile j in buffer j % 2 (columns
                                         // 128 (j % 2) ...), P over its first 64
constexpr uint32_t kOCol = 2 * kBN;      // the half of O
constexpr int kQOff = 0;
constexpr int kRingOff = kQChunks * kChunkBytes;
constexpr int kBarOff = kRingOff + kRing * kSlotBytes;
// q_full, full[kRing], empty[kRing], s_full[2], p_ready[2], o_done, drain, pv_done
constexpr int kNBars = 1 + 2 * kRing + 7;
constexpr int kMiscOff = kBarOff + kNBars * 8;
constexpr int kSmem = kMiscOff + 16 + 1024;  // + alignment slack
static_assert(kSmem <= 232448, "shared memory budget");
static_assert(kOCol + kDH <= kTmemCols, "TMEM budget");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct D512Args {
  int B, Hq, Hkv, G, Lq, Lk, num_qtiles;
  float sl2;  // scale * log2(e)
  int causal;
  const void* mask;
  long long ms0, ms1, ms2;  // mask element strides (key stride 1)
  int mask_bool;            // mask holds bytes, nonzero = visible
  const float* sinks;
  void* o;
  long long os0, os1, os2;  // element strides of o (batch, head, row)
  float* lse;
  int* status;
  unsigned long long wait_ns;
  const int* seq_lens_q;
  const int* seq_lens_kv;
};

template <bool BF16>
struct Half2;
template <>
struct Half2<true> {
  using T = __nv_bfloat16;
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  static __device__ __forceinline__ float to_f(T x) { return __bfloat162float(x); }
};
template <>
struct Half2<false> {
  using T = __half;
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  static __device__ __forceinline__ float to_f(T x) { return __half2float(x); }
};

__device__ __forceinline__ void drain_wait512(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) break;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_d512_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const D512Args a) {
  using H = Half2<BF16>;
  using T = typename H::T;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sQ = smem + kQOff;
  uint8_t* sRing = smem + kRingOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* q_full = bars;
  uint64_t* full = bars + 1;
  uint64_t* empty = full + kRing;
  uint64_t* s_full = empty + kRing;  // [2]: S of a buffer complete
  uint64_t* p_ready = s_full + 2;    // [2]: P of a buffer written
  uint64_t* o_done = p_ready + 2;
  uint64_t* drain = o_done + 1;
  uint64_t* pv_done = drain + 1;     // one phase per tile: its PV products complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // (query tile, D-half) pairs along x; causal grids heaviest tiles first
  const int half = static_cast<int>(blockIdx.x & 1u);
  int qt = static_cast<int>(blockIdx.x >> 1);
  if (a.causal) qt = a.num_qtiles - 1 - qt;
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / a.G;
  const int m0 = qt * kBM;
  const int Lkb = a.seq_lens_kv ? min(max(a.seq_lens_kv[b], 0), a.Lk) : a.Lk;
  const int Lqb = a.seq_lens_q ? min(max(a.seq_lens_q[b], 0), a.Lq) : a.Lq;
  // key tiles this query tile reads (up to its last row's last visible key)
  int nkv = 0;
  {
    const int last_row = min(m0 + kBM - 1, Lqb - 1);
    if (last_row >= m0) {
      const int all = (Lkb + kBN - 1) / kBN;
      if (a.causal) {
        const int lim = last_row + (Lkb - Lqb);
        nkv = lim < 0 ? 0 : min(all, lim / kBN + 1);
      } else {
        nkv = all;
      }
    }
  }

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_ready[i], kBM);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(pv_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{a.wait_ns, abort_flag, a.status};
  int last_use[kRing];  // producer: last fill of each slot (-1: none)
#pragma unroll
  for (int s = 0; s < kRing; ++s) last_use[s] = -1;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(q_full, kQChunks * kChunkBytes);
      for (int c = 0; c < kQChunks; ++c)
        tma_load_4d(sQ + c * kChunkBytes, &tmQ, q_full, c * kChunkCols, m0, h, b);
      // the MMA issuer's order: K_0, then per step j >= 1 K_j and V_{j-1}
      // (S_j is computed while the softmax warps work on S_{j-1}), then the
      // last V
      int seq = 0;
      bool pok = true;
      for (int j = 0; j <= nkv && pok; ++j) {
        for (int i = 0; i < kStepSlots; ++i) {
          const bool is_k = i < kKSlots;
          const int tile = is_k ? j : j - 1;
          if (tile < 0 || tile >= nkv) continue;
          const int s = seq % kRing;
          const int use = seq / kRing;
          if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, wc)) {
            pok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], kSlotBytes);
          uint8_t* dst = sRing + s * kSlotBytes;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if (is_k)
              tma_load_4d(dst + hh * kChunkBytes, &tmK, &full[s], (2 * i + hh) * kChunkCols,
                          tile * kBN, kvh, b);
            else
              tma_load_4d(dst + hh * kChunkBytes, &tmV, &full[s],
                          half * kDH + (2 * (i - kKSlots) + hh) * kChunkCols, tile * kBN, kvh, b);
          }
          last_use[s] = use;
          ++seq;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // One thread issues, per step j: S_j = sum over the eight K chunks into
    // S buffer j % 2 and a commit that hands it to the softmax warps; then,
    // once they have written P_{j-1}, the half's four V chunks' products
    // O += P_{j-1} V_{j-1} and a commit (pv_done) for a rescale of O.  S_j
    // thus runs while the softmax warps work on S_{j-1}; S_{j+2} overwrites
    // buffer j % 2 only after PV_j, issued before it, has read P_j (the MMAs
    // run in issue order).  Each chunk's slot is released by a commit once
    // its products complete.
    if (lane == 0) {
      constexpr uint32_t idS = idesc_f16(BF16, kBM, kBN, false, false);
      constexpr uint32_t idO = idesc_f16(BF16, kBM, kChunkCols, false, true);
      const uint64_t q_desc = sdesc(smem_addr(sQ), 16, 1024, kSwizzle128B);
      const uint64_t k_desc = sdesc(smem_addr(sRing), 16, 1024, kSwizzle128B);
      const uint64_t v_desc = sdesc(smem_addr(sRing), kBN * 128, 1024, kSwizzle128B);
      bool ok = mbar_wait(q_full, 0, wc);
      int seq = 0;
      for (int j = 0; j <= nkv; ++j) {
        if (j < nkv) {
          // S_j = sum over the eight column chunks c of Q_c K_c^T; a K step
          // of 16 elements is 32 bytes inside the 128-byte swizzled rows
          const uint32_t dS = tmem + kSCol + (j & 1) * kBN;
          for (int i = 0; i < kKSlots; ++i, ++seq) {
            const int s = seq % kRing;
            ok = ok && mbar_wait(&full[s], static_cast<uint32_t>((seq / kRing) & 1), wc);
            if (ok) {
              tc_fence_after();
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int c = 2 * i + hh;
#pragma unroll
                for (int kk = 0; kk < kChunkCols / 16; ++kk) {
                  const uint64_t qd =
                      q_desc + static_cast<uint64_t>((c * kChunkBytes + kk * 32) >> 4);
                  const uint64_t kd = k_desc + static_cast<uint64_t>(
                                                   (s * kSlotBytes + hh * kChunkBytes + kk * 32) >> 4);
                  mma_f16_ss(dS, qd, kd, idS, (c > 0 || kk > 0) ? 1u : 0u);
                }
              }
            }
            mma_commit(&empty[s]);
          }
          mma_commit(&s_full[j & 1]);
        }
        if (j == 0) continue;
        // O_half += P_{j-1} V_{j-1}: P (128 x 128, K-major) from TMEM, 2
        // elements per column; V chunk c (64 columns of the half) MN-major,
        // 16 keys per K step (2048 bytes)
        const int pj = j - 1;
        ok = ok && mbar_wait(&p_ready[pj & 1], static_cast<uint32_t>((pj >> 1) & 1), wc);
        if (ok) tc_fence_after();
        const uint32_t aP = tmem + kSCol + (pj & 1) * kBN;
        for (int i = 0; i < kVSlots; ++i, ++seq) {
          const int s = seq % kRing;
          ok = ok && mbar_wait(&full[s], static_cast<uint32_t>((seq / kRing) & 1), wc);
          if (ok) {
            tc_fence_after();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int c = 2 * i + hh;
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk) {
                const uint64_t vd = v_desc + static_cast<uint64_t>(
                                                 (s * kSlotBytes + hh * kChunkBytes + kk * 16 * 128) >> 4);
                mma_f16_ts(tmem + kOCol + c * kChunkCols, aP + kk * 8, vd, idO,
                           (pj > 0 || kk > 0) ? 1u : 0u);
              }
            }
          }
          mma_commit(&empty[s]);
        }
        mma_commit(pv_done);
      }
      mma_commit(o_done);
      // every product completes before TMEM is freed
      mma_commit(drain);
      drain_wait512(drain, 0, kDrainNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int r = warp * 32 + lane;  // row of the tile = TMEM lane
    const int qi = m0 + r;
    const bool row_ok = qi < a.Lq;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem + lane_off + kOCol;
    int limit = Lkb - 1;  // last key visible to this row
    if (a.causal) limit = min(limit, qi + (Lkb - Lqb));
    if (qi >= Lqb) limit = -1;  // a padding row sees no key
    const T* mrow = nullptr;
    const uint8_t* mrowb = nullptr;
    if (a.mask && row_ok) {
      const long long moff = b * a.ms0 + h * a.ms1 + qi * a.ms2;
      if (a.mask_bool)
        mrowb = static_cast<const uint8_t*>(a.mask) + moff;
      else
        mrow = static_cast<const T*>(a.mask) + moff;
    }
    const float mhuge = mask_huge_log2(a.sl2);
    float m = -INFINITY;  // reference max (log2 units)
    float l = 0.f;        // running sum relative to m
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const uint32_t tS = tmem + lane_off + kSCol + (j & 1) * kBN;  // S_j, then P_j
      ok = __all_sync(0xffffffffu,
                      ok && mbar_wait(&s_full[j & 1], static_cast<uint32_t>((j >> 1) & 1), wc));
      if (ok) {
        tc_fence_after();
        uint32_t s[kBN];
        __syncwarp();
        tmem_ld4x32_sync(tS, tS + 32, tS + 64, tS + 96,
                         *reinterpret_cast<uint32_t(*)[32]>(&s[0]),
                         *reinterpret_cast<uint32_t(*)[32]>(&s[32]),
                         *reinterpret_cast<uint32_t(*)[32]>(&s[64]),
                         *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
        const int kv0 = j * kBN;
        // log2-domain scores; the mask tests are hoisted out of the element
        // loops (a lane-dependent branch per element cost several times the
        // element's work: the softmax took 9811 of a tile's 17388 clk)
        float x[kBN];
        if (mrow) {
#pragma unroll
          for (int i = 0; i < kBN; ++i) {
            const bool vis = kv0 + i <= limit;
            const float mv = vis ? mask_log2(H::to_f(mrow[kv0 + i]), mhuge) : 0.f;
            x[i] = vis ? fmaf(__uint_as_float(s[i]), a.sl2, mv) : -INFINITY;
          }
        } else if (mrowb) {
#pragma unroll
          for (int i = 0; i < kBN; ++i) {
            const bool vis = kv0 + i <= limit;
            const uint8_t mb = vis ? mrowb[kv0 + i] : 0;
            x[i] = mb ? __uint_as_float(s[i]) * a.sl2 : -INFINITY;
          }
        } else if (kv0 + kBN - 1 <= limit) {
#pragma unroll
          for (int i = 0; i < kBN; ++i) x[i] = __uint_as_float(s[i]) * a.sl2;
        } else {
#pragma unroll
          for (int i = 0; i < kBN; ++i)
            x[i] = kv0 + i <= limit ? __uint_as_float(s[i]) * a.sl2 : -INFINITY;
        }
        float mr[8];  // eight running maxima, every column read once
#pragma unroll
        for (int c = 0; c < 8; ++c) mr[c] = x[c];
#pragma unroll
        for (int i = 8; i < kBN; i += 8)
#pragma unroll
          for (int c = 0; c < 8; ++c) mr[c] = fmaxf(mr[c], x[i + c]);
        const float mx = fmaxf(fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3])),
                               fmaxf(fmaxf(mr[4], mr[5]), fmaxf(mr[6], mr[7])));
        float alpha = 1.f;
        const bool resc = mx > m + kRescaleThreshold;  // true on the first visible tile
        if (resc) {
          alpha = ex2(m - mx);  // 0 when m = -inf
          m = mx;
        }
        const float mu = (m == -INFINITY) ? 0.f : m;
        float rp[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[kBN / 2];
#pragma unroll
        for (int i = 0; i < kBN / 2; ++i) {
          const float p0 = ex2(x[2 * i] - mu);
          const float p1 = ex2(x[2 * i + 1] - mu);
          rp[i & 3] += p0 + p1;
          pk[i] = H::pack(p0, p1);
        }
        l = l * alpha + ((rp[0] + rp[1]) + (rp[2] + rp[3]));
        // Rescale rows whose max moved, once O holds the sum through
        // P_{j-1} V_{j-1}: PV_{j-1} runs beside this step (issued after
        // S_j), PV_{j-2} has completed (issued before S_j, whose commit this
        // step waited for), so phase j-1 of pv_done is the next to complete
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          ok = __all_sync(0xffffffffu,
                          ok && mbar_wait(pv_done, static_cast<uint32_t>((j - 1) & 1), wc));
          tc_fence_after();
          __syncwarp();
#pragma unroll 1
          for (int c = 0; c < kDH / 32; ++c) {
            uint32_t ob[32];
            tmem_ld32_sync(tO + c * 32, ob);
#pragma unroll
            for (int i = 0; i < 32; ++i) ob[i] = __float_as_uint(__uint_as_float(ob[i]) * alpha);
            tmem_st32(tO + c * 32, ob);
          }
        }
        __syncwarp();
        tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        tmem_wait_st();
        tc_fence_before();
      }
      // P_j is in TMEM: every thread arrives every step, also after a failed wait
      mbar_arrive(&p_ready[j & 1]);
    }
    ok = __all_sync(0xffffffffu, ok && mbar_wait(o_done, 0, wc));
    if (ok) {
      tc_fence_after();
      float oscale = 1.f;
      if (a.sinks) {  // the sink logit joins the denominator only (value row 0)
        const float sk = a.sinks[h] * kLog2e;
        const float mn = fmaxf(m, sk);
        oscale = ex2(m - mn);
        l = l * oscale + ex2(sk - mn);
        m = mn;
      }
      const float inv = (l > 0.f) ? oscale / l : 0.f;
      T* orow = static_cast<T*>(a.o) + (b * a.os0 + h * a.os1 + qi * a.os2) + half * kDH;
      __syncwarp();
#pragma unroll 1
      for (int c = 0; c < kDH / 32; ++c) {
        uint32_t ob[32];
        tmem_ld32_sync(tO + c * 32, ob);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float v0 = (inv == 0.f || nkv == 0) ? 0.f : __uint_as_float(ob[2 * i]) * inv;
          const float v1 = (inv == 0.f || nkv == 0) ? 0.f : __uint_as_float(ob[2 * i + 1]) * inv;
          w[i] = H::pack(v0, v1);
        }
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (row_ok && half == 0 && a.lse)
        a.lse[(static_cast<size_t>(b) * a.Hq + h) * a.Lq + qi] =
            (l > 0.f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (warp == kProdWarp && lane == 0 && *abort_flag) {
    // a role gave up: every copy the producer issued lands before the CTA exits
    drain_wait512(q_full, 0, kDrainNs);
    for (int s = 0; s < kRing; ++s)
      if (last_use[s] >= 0) drain_wait512(&full[s], last_use[s] & 1, kDrainNs);
  }
}

template <bool BF16>
sdpa_status_t launch_d512(const sdpa_params_t& p, const void* q, const void* k, const void* v,
                          void* o, float* lse, const LaunchEnv& env) {
  const CUtensorMapDataType dt =
      BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t B = p.batch, Hq = p.num_q_heads, Hkv = p.num_kv_heads;
  const uint64_t Lq = p.seq_len_q, Lk = p.seq_len_kv;
  // [B, H, L, 512] with the given strides, viewed innermost-first; box
  // 64 x 128 rows, 128-byte swizzle; rows past L read as zero
  CUtensorMap tq, tk, tv;
  if (!encode_tiled_4d(&tq, dt, q, kD, Lq, Hq, B, 2, kChunkCols, kBM, p.q_stride[2],
                       p.q_stride[1], p.q_stride[0]) ||
      !encode_tiled_4d(&tk, dt, k, kD, Lk, Hkv, B, 2, kChunkCols, kBN, p.k_stride[2],
                       p.k_stride[1], p.k_stride[0]) ||
      !encode_tiled_4d(&tv, dt, v, kD, Lk, Hkv, B, 2, kChunkCols, kBN, p.v_stride[2],
                       p.v_stride[1], p.v_stride[0]))
    return SDPA_ERR_CUDA;
  D512Args a;
  a.B = p.batch;
  a.Hq = p.num_q_heads;
  a.Hkv = p.num_kv_heads;
  a.G = p.num_q_heads / p.num_kv_heads;
  a.Lq = p.seq_len_q;
  a.Lk = p.seq_len_kv;
  a.num_qtiles = (p.seq_len_q + kBM - 1) / kBM;
  a.sl2 = p.scale * kLog2e;
  a.causal = p.causal ? 1 : 0;
  a.mask = p.mask;
  a.ms0 = p.mask_stride[0];
  a.ms1 = p.mask_stride[1];
  a.ms2 = p.mask_stride[2];
  a.mask_bool = (p.flags & SDPA_FLAG_BOOL_MASK) ? 1 : 0;
  a.sinks = p.sinks;
  a.o = o;
  a.os0 = p.o_stride[0];
  a.os1 = p.o_stride[1];
  a.os2 = p.o_stride[2];
  a.lse = lse;
  a.status = env.status;
  a.wait_ns = env.wait_limit_ns;
  a.seq_lens_q = p.seq_lens_q;
  a.seq_lens_kv = p.seq_lens_kv;
  auto kern = prefill_d512_kernel<BF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
      cudaSuccess)
    return SDPA_ERR_CUDA;
  const long long gx = 2LL * a.num_qtiles;
  if (gx > 0x7fffffffLL || Hq > 65535 || B > 65535) return SDPA_ERR_UNSUPPORTED;
  kern<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(Hq), static_cast<unsigned>(B)),
         kThreads, kSmem, env.stream>>>(tq, tk, tv, a);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // namespace

sdpa_status_t launch_prefill_tc_d512(const sdpa_params_t& p, const void* q, const void* k,
                                     const void* v, void* o, float* lse, const LaunchEnv& env,
                                     int* grids) {
  *grids = 0;
  const sdpa_status_t st = p.dtype == SDPA_BF16 ? launch_d512<true>(p, q, k, v, o, lse, env)
                                                : launch_d512<false>(p, q, k, v, o, lse, env);
  if (st == SDPA_OK) *grids = 1;
  return st;
}

}  // namespace gb300
