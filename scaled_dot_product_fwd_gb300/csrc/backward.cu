// backward.cu — gradients dQ, dK, dV of the attention forward (fp16/bf16,
// head_dim 64/128) on the 5th-generation tensor cores of sm_103a.
//
// The computation is the backward pass of the rustytorch flash_attention.metal
// page (backward kernels for dQ and for dK, dV): P recomputed from the
// forward's log-sum-exp, P = exp(S - LSE); D_i = dO_i . O_i; dS = P (dP - D)
// with dP = dO V^T; dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO; with the
// options of the mlx cuDNN backward graph (attention scale, bottom-right
// causal mask, additive bias, sink token: the sink enters through LSE).
//
// GB300 design (not the page's): one CTA per (key tile of 128 keys, kv head,
// batch) owns dK and dV of its keys in TMEM for the whole pass (no atomics)
// and walks the query tiles of every query head of the group.  Per query
// tile the MMA warp computes S^T = K Q^T and dP^T = V dO^T with the keys as
// TMEM lanes, so the compute warps (one thread per key) turn a row of S^T
// into P^T and dS^T and write them back to TMEM as the A operands of
// dV += P^T dO and dK += dS^T Q; dS^T also goes to shared memory (128-byte
// swizzled rows of keys), the MN-major A operand of dQ = dS K, whose tile the
// compute warps then add into an fp32 workspace with vector reductions.
// Before the pass a small kernel computes D_i and LSE in log2 units per query
// row and clears the dQ workspace; after it, another scales dQ and stores it
// in the input dtype.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"
#include "tensor_map.h"

namespace gb300 {
namespace {

constexpr int kBT = 128;            // keys per CTA tile = query rows per step
// 8 compute warps: warp w reads TMEM lanes 32 (w % 4) .. +31 (keys; query rows
// for dQ) and takes half w / 4 of the columns.  Warps 8-11 form the control
// warpgroup (producer, MMA issuer, two idle warps) and give registers to the
// compute warpgroups with setmaxnreg (launch: 384 x 168 = 256 x 224 + 128 x 56).
constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kBwdThreads = 32 * 12;
constexpr uint32_t kComputeRegs = 224;
constexpr uint32_t kControlRegs = 56;
constexpr float kLog2eB = 1.4426950408889634f;
// named barriers: kBarLse (the compute warps), kBarPair + q (the two warps
// that share TMEM lane quarter q)
constexpr uint32_t kBarLse = 1;
constexpr uint32_t kBarPair = 2;

template <int D>
struct BwdCfg {
  static constexpr int CB = D / 64;             // 128-byte column blocks per row
  static constexpr int TILE = kBT * D * 2;      // one 128-row fp16/bf16 tile
  // stages of the Q, dO ring (the next step's tiles load during this one;
  // one stage at D = 128, where shared memory holds no second)
  static constexpr int NST = D == 64 ? 2 : 1;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILE;
  static constexpr int Q_OFF = V_OFF + TILE;          // NST tiles
  static constexpr int DO_OFF = Q_OFF + NST * TILE;   // NST tiles
  static constexpr int DS_OFF = DO_OFF + NST * TILE;  // dS^T: 128 keys x 128 query rows
  static constexpr int DS_BYTES = kBT * kBT * 2;
  // D = 64: the MMAs of step s+1's S^T and dP^T are issued before step s's
  // dQ MMA, which then runs while the compute warps work on step s+1: dS^T
  // has two buffers (step parity)
  static constexpr int NDS = D == 64 ? 2 : 1;
  // -LSE and -D of a step's 128 query rows, two buffers each (step parity)
  static constexpr int LSE_OFF = DS_OFF + NDS * DS_BYTES;  // 2 x 128 floats
  static constexpr int DV_OFF = LSE_OFF + 2 * kBT * 4;
  static constexpr int BAR_OFF = DV_OFF + 2 * kBT * 4;
  // kv_full, q_full[2], q_empty[2], s_full, p_ready, mma_done, dq_read, drain
  static constexpr int NBARS = 10;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
  // + alignment slack; at least 116 KB so that one CTA holds an SM (each
  // allocates all 512 TMEM columns)
  static constexpr int SMEM = (MISC_OFF + 16 + 1024) > 116 * 1024 ? (MISC_OFF + 16 + 1024)
                                                                   : 116 * 1024;
  // TMEM: S^T (P^T packed over its first 64 columns) | dP^T (dS^T packed) |
  // dV | dK | dQ x 2 (D = 64; at D = 128 dQ reuses the S^T columns once the
  // dV MMA, issued before it, has read P^T)
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_DP = 128;
  static constexpr uint32_t COL_DV = 256;
  static constexpr uint32_t COL_DK = 256 + D;
  // dQ: at D = 64 two buffers (step s in buffer s % 2, read while the next
  // step's MMAs run); at D = 128 one, over the S^T columns
  static constexpr bool PIPE_DQ = D == 64;
  static_assert(!PIPE_DQ || NDS == 2, "the pipelined dQ reads one dS^T buffer while the next is written");
  static constexpr int ds_off(int s) { return DS_OFF + (NDS == 2 ? (s & 1) * DS_BYTES : 0); }
  static constexpr uint32_t COL_DQ = D == 64 ? 384 : 0;
  static constexpr uint32_t dq_col(int s) { return PIPE_DQ ? COL_DQ + (s & 1) * 64 : COL_DQ; }
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(COL_DK + D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct BwdArgs {
  int B, Hq, Hkv, G, Lq, Lk;
  float sl2;    // scale * log2(e)
  float scale;
  int causal;
  const void* mask;
  long long ms0, ms1, ms2;
  int mask_bool;
  const float* lse2;  // [B, Hq, Lq]: LSE in log2 units (+inf: the row sees nothing)
  const float* dvec;  // [B, Hq, Lq]: D_i = dO_i . O_i
  const int* seq_lens_q;   // NULL or [B]: query rows [0, len) of batch b take part
  const int* seq_lens_kv;  // NULL or [B]: keys [0, len) of batch b are visible
  float* dq_acc;      // [B, Hq, Lq, D] fp32, cleared before the pass
  void* dk;
  void* dv;
  long long dks0, dks1, dks2, dvs0, dvs1, dvs2;  // element strides of dk, dv
  int* status;
  unsigned long long wait_ns;
};

template <bool BF16>
struct BwdElem;
template <>
struct BwdElem<true> {
  using T = __nv_bfloat16;
  static __device__ __forceinline__ float to_f(T x) { return __bfloat162float(x); }
  static __device__ __forceinline__ T from_f(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};
template <>
struct BwdElem<false> {
  using T = __half;
  static __device__ __forceinline__ float to_f(T x) { return __half2float(x); }
  static __device__ __forceinline__ T from_f(float x) { return __float2half_rn(x); }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};

// Pairs of fp32 values in one 64-bit register for the packed f32x2 ops.
__device__ __forceinline__ uint64_t bf2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void bf2_unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t bf2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t bf2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t bf2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// 16-byte shared-memory load (32-bit shared address)
__device__ __forceinline__ float4 bld4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// ---------------------------------------------------------------- pre / post
// Per query row (b, h, i): D_i = dO_i . O_i, LSE in log2 units (+inf for a
// row that saw nothing, or lies past its batch's query length, so that every
// P of it is 0), and a cleared dQ row.  One warp per row.
struct PreArgs {
  const void* o;
  const void* d_o;
  const float* lse;
  float* lse2;
  float* dvec;
  float* dq_acc;
  const int* seq_lens_q;  // NULL or [B]: rows at or past a batch's length take no part
  int Hq, Lq, D;
  long long os0, os1, os2;  // strides of o and dO (dO has o's layout)
  long long rows;
};

template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f(const __half* p) { return __half2float(*p); }
template <>
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
template <>
__device__ __forceinline__ float ld_f(const float* p) { return *p; }

template <typename T>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const PreArgs a) {
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= a.rows) return;
  const long long i = row % a.Lq;
  const long long bh = row / a.Lq;
  const long long h = bh % a.Hq, b = bh / a.Hq;
  const long long off = b * a.os0 + h * a.os1 + i * a.os2;
  const T* o = static_cast<const T*>(a.o) + off;
  const T* g = static_cast<const T*>(a.d_o) + off;
  float s = 0.f;
  for (int d = lane; d < a.D; d += 32) s = fmaf(ld_f(o + d), ld_f(g + d), s);
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) s += __shfl_xor_sync(0xffffffffu, s, w);
  if (a.dq_acc) {
    float* dq = a.dq_acc + row * a.D;
    for (int d = lane; d < a.D; d += 32) dq[d] = 0.f;
  }
  if (lane == 0) {
    a.dvec[row] = s;
    const bool live = !a.seq_lens_q || i < min(max(a.seq_lens_q[b], 0), a.Lq);
    const float l = live ? a.lse[row] : -INFINITY;
    // A row that saw no key, or only keys whose mask values were huge (LSE
    // -2^100 * scale, beside which its scores vanish), takes no part: P = 0
    // there.  For the latter that is exact for dQ and dK (the scores do not
    // reach the output) and leaves out its share dO / n of those keys' dV.
    a.lse2[row] = (l == -INFINITY || l <= -kMaskBig) ? INFINITY : l * kLog2eB;
  }
}

template <typename T>
__device__ __forceinline__ T cvt(float x);
template <>
__device__ __forceinline__ __half cvt<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// dQ = scale * dq_acc in the input dtype, q's layout.  One warp per row.
struct PostArgs {
  const float* dq_acc;
  void* dq;
  int Hq, Lq, D;
  float scale;
  long long qs0, qs1, qs2;
  long long rows;
};

template <typename T>
__global__ void __launch_bounds__(256) bwd_post_kernel(const PostArgs a) {
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= a.rows) return;
  const long long i = row % a.Lq;
  const long long bh = row / a.Lq;
  const long long h = bh % a.Hq, b = bh / a.Hq;
  T* dq = static_cast<T*>(a.dq) + b * a.qs0 + h * a.qs1 + i * a.qs2;
  const float* src = a.dq_acc + row * a.D;
  for (int d = lane; d < a.D; d += 32) dq[d] = cvt<T>(src[d] * a.scale);
}

// Wait for a phase ignoring the abort flag (drains in-flight asynchronous
// work before the CTA exits); bounded by limit_ns.
__device__ __forceinline__ void bwd_drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) break;
  }
}

// ---------------------------------------------------------------- main pass
// LENS: the call has per-batch length arrays (without them the lengths stay
// the call's own, read from the kernel parameters where they are used).
template <int D, bool BF16, bool LENS>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
               const BwdArgs a) {
  using C = BwdCfg<D>;
  using E = BwdElem<BF16>;
  using T = typename E::T;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sK = smem + C::K_OFF;
  uint8_t* sV = smem + C::V_OFF;
  uint8_t* sQ = smem + C::Q_OFF;
  uint8_t* sDO = smem + C::DO_OFF;
  // per step: -LSE (log2 units) and -D of the 128 query rows
  float* sLse = reinterpret_cast<float*>(smem + C::LSE_OFF);
  float* sDv = reinterpret_cast<float*>(smem + C::DV_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;   // [2]: stage filled
  uint64_t* q_empty = bars + 3;  // [2]: stage read by its step's MMAs
  uint64_t* s_full = bars + 5;
  uint64_t* p_ready = bars + 6;
  uint64_t* mma_done = bars + 7;
  uint64_t* dq_read = bars + 8;
  uint64_t* drain = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int j0 = blockIdx.x * kBT;  // first key of the tile
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  // this batch's lengths (padding masks), clamped to the call's
  const int Lkb = (LENS && a.seq_lens_kv) ? min(max(a.seq_lens_kv[b], 0), a.Lk) : a.Lk;
  const int Lqb = (LENS && a.seq_lens_q) ? min(max(a.seq_lens_q[b], 0), a.Lq) : a.Lq;
  const int off = Lkb - Lqb;  // bottom-right causal: key j visible to row i iff j <= i + off
  // query tiles of each head that hold a row seeing a key of this tile (none
  // when the tile lies past the batch's keys)
  const int nqt = (Lqb + kBT - 1) / kBT;
  int qt0 = 0;
  if (a.causal && j0 - off > 0) qt0 = (j0 - off) / kBT;
  const int per_head = (nqt > qt0 && j0 < Lkb) ? nqt - qt0 : 0;
  const int nsteps = a.G * per_head;  // (query head of the group, query tile) pairs

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int st = 0; st < 2; ++st) {
      mbar_init(&q_full[st], 1);
      mbar_init(&q_empty[st], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_ready, kComputeThreads);
    mbar_init(mma_done, 1);
    mbar_init(dq_read, kComputeThreads);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{a.wait_ns, abort_flag, a.status};
  int q_last[2] = {-1, -1};  // producer: last use of each Q, dO stage (-1: none)

  if (warp >= kComputeWarps) {
    setmaxnreg_dec<kControlRegs>();
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(kv_full, 2 * C::TILE);
      for (int cb = 0; cb < C::CB; ++cb) {
        tma_load_4d(sK + cb * kBT * 128, &tmK, kv_full, cb * 64, j0, kvh, b);
        tma_load_4d(sV + cb * kBT * 128, &tmV, kv_full, cb * 64, j0, kvh, b);
      }
      for (int s = 0; s < nsteps; ++s) {
        const int st = s % C::NST;
        const int use = s / C::NST;
        // the stage's previous step's MMAs have read its Q and dO
        if (use > 0 && !mbar_wait(&q_empty[st], (use - 1) & 1, wc)) break;
        const int hq = kvh * a.G + s / per_head;
        const int q0 = (qt0 + s % per_head) * kBT;
        mbar_arrive_expect_tx(&q_full[st], 2 * C::TILE);
        for (int cb = 0; cb < C::CB; ++cb) {
          tma_load_4d(sQ + st * C::TILE + cb * kBT * 128, &tmQ, &q_full[st], cb * 64, q0, hq, b);
          tma_load_4d(sDO + st * C::TILE + cb * kBT * 128, &tmDO, &q_full[st], cb * 64, q0, hq,
                      b);
        }
        q_last[st] = use;
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // K-major operands (S^T = K Q^T, dP^T = V dO^T): a K step of 16
      // elements is 32 bytes inside a 128-byte row, 4 steps per column block
      auto kmaj = [&](const uint8_t* base, int kk) {
        return sdesc(smem_addr(base) + (kk >> 2) * (kBT * 128) + (kk & 3) * 32, 16, 1024,
                     kSwizzle128B);
      };
      // MN-major operands (rows along K, 64-wide column blocks kBT*128 bytes
      // apart, 8-row groups 1024 bytes apart); a K step is 16 rows
      auto mnmaj = [&](const uint8_t* base, int kk) {
        return sdesc(smem_addr(base) + kk * 16 * 128, kBT * 128, 1024, kSwizzle128B);
      };
      constexpr uint32_t idS = idesc_f16(BF16, kBT, kBT, false, false);
      constexpr uint32_t idKV = idesc_f16(BF16, kBT, D, false, true);
      constexpr uint32_t idQ = idesc_f16(BF16, kBT, D, true, true);
      bool ok = mbar_wait(kv_full, 0, wc);
      // S^T = K Q^T and dP^T = V dO^T of step s (Q, dO stage s % NST)
      auto issue_sdp = [&](int s) {
        const int st = s % C::NST;
        const uint8_t* q_st = sQ + st * C::TILE;
        const uint8_t* do_st = sDO + st * C::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          mma_f16_ss(tmem + C::COL_S, kmaj(sK, kk), kmaj(q_st, kk), idS, kk > 0 ? 1u : 0u);
          mma_f16_ss(tmem + C::COL_DP, kmaj(sV, kk), kmaj(do_st, kk), idS, kk > 0 ? 1u : 0u);
        }
      };
      // dV += P^T dO and dK += dS^T Q (A from TMEM: 128 query rows, two
      // elements per column)
      auto issue_dkv = [&](int s) {
        const int st = s % C::NST;
        const uint8_t* q_st = sQ + st * C::TILE;
        const uint8_t* do_st = sDO + st * C::TILE;
#pragma unroll
        for (int kk = 0; kk < kBT / 16; ++kk) {
          const uint32_t acc = (s > 0 || kk > 0) ? 1u : 0u;
          mma_f16_ts(tmem + C::COL_DV, tmem + C::COL_S + kk * 8, mnmaj(do_st, kk), idKV, acc);
          mma_f16_ts(tmem + C::COL_DK, tmem + C::COL_DP + kk * 8, mnmaj(q_st, kk), idKV, acc);
        }
      };
      // dQ = dS K (A: dS^T rows in shared memory)
      auto issue_dq = [&](int s) {
        const uint8_t* ds = smem + C::ds_off(s);
#pragma unroll
        for (int kk = 0; kk < kBT / 16; ++kk)
          mma_f16_ss(tmem + C::dq_col(s), mnmaj(ds, kk), mnmaj(sK, kk), idQ, kk > 0 ? 1u : 0u);
      };
      if constexpr (C::PIPE_DQ) {
        // Order per step: dV_s, dK_s, then S^T and dP^T of step s+1 (they
        // overwrite the columns dV_s and dK_s read: the MMAs run in issue
        // order), then dQ_s, which runs while the compute warps start on
        // step s+1 (dS^T and dQ have two buffers each).
        if (ok && nsteps > 0) {
          ok = mbar_wait(&q_full[0], 0, wc);
          if (ok) {
            tc_fence_after();
            issue_sdp(0);
            mma_commit(s_full);
          }
        }
        for (int s = 0; s < nsteps && ok; ++s) {
          if (!mbar_wait(p_ready, s & 1, wc)) break;
          tc_fence_after();
          issue_dkv(s);
          mma_commit(&q_empty[s % C::NST]);
          if (s + 1 < nsteps) {
            const int st1 = (s + 1) % C::NST;
            if (!mbar_wait(&q_full[st1], ((s + 1) / C::NST) & 1, wc)) break;
            tc_fence_after();
            issue_sdp(s + 1);
            mma_commit(s_full);
          }
          issue_dq(s);
          mma_commit(mma_done);
        }
      } else {
        for (int s = 0; s < nsteps && ok; ++s) {
          const int st = s % C::NST;
          ok = mbar_wait(&q_full[st], (s / C::NST) & 1, wc);
          // At D = 128 the dQ tile shares the S^T columns: the compute warps
          // have read the previous one.
          if (ok && s > 0) ok = mbar_wait(dq_read, (s - 1) & 1, wc);
          if (!ok) break;
          tc_fence_after();
          issue_sdp(s);
          mma_commit(s_full);
          if (!mbar_wait(p_ready, s & 1, wc)) break;
          tc_fence_after();
          issue_dkv(s);
          issue_dq(s);
          mma_commit(&q_empty[st]);
          mma_commit(mma_done);
        }
      }
      // every MMA issued here completes before TMEM is freed
      mma_commit(drain);
      bwd_drain_wait(drain, 0, kDrainNs);
    }
  }
  // warps 10 and 11: idle
  } else {
    setmaxnreg_inc<kComputeRegs>();
    // ------------------------------------------------------- compute warps
    // Thread (warp w, lane) owns key j0 + 32 (w % 4) + lane (TMEM lane) for
    // P^T and dS^T on query columns [64 h, 64 h + 64) with h = w / 4, and
    // query row q0 + 32 (w % 4) + lane of the dQ tile on D/2 of its columns.
    // Every step meets the same barriers, also after a failed wait (no path
    // can hang).
    const int quarter = warp & 3;
    const int hf = warp >> 2;
    const int r = quarter * 32 + lane;  // TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int jr = j0 + r;
    bool ok = true;
    // -LSE (log2 units; threads 0-127) or -D (threads 128-255) of one query
    // row of a step, loaded a step ahead (-inf: P = 0)
    auto row_stat = [&](int s) {
      const int hq = kvh * a.G + s / per_head;
      const int i = (qt0 + s % per_head) * kBT + (threadIdx.x & (kBT - 1));
      const size_t row = (static_cast<size_t>(b) * a.Hq + hq) * a.Lq + i;
      if (threadIdx.x < kBT) return i < Lqb ? -a.lse2[row] : -INFINITY;
      return i < Lqb ? -a.dvec[row] : 0.f;
    };
    float stat = nsteps > 0 ? row_stat(0) : 0.f;
    // dQ tile of step s (TMEM lane r = query row q0 + r) added into the fp32
    // accumulator, D/2 columns per warp
    auto read_dq = [&](int s) {
      if (!ok) return;
      tc_fence_after();
      const int hq = kvh * a.G + s / per_head;
      const int i = (qt0 + s % per_head) * kBT + r;
      float* dst = a.dq_acc + ((static_cast<size_t>(b) * a.Hq + hq) * a.Lq + i) * D + hf * (D / 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
        __syncwarp();  // .aligned TMEM access after per-lane stores
        tmem_ld32_sync(tmem + lane_off + C::dq_col(s) + hf * (D / 2) + c * 32, v);
        if (i < Lqb) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            red_add_v4(dst + c * 32 + 4 * e, __uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                       __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
        }
      }
    };
    for (int s = 0; s < nsteps; ++s) {
      const int hq = kvh * a.G + s / per_head;
      const int q0 = (qt0 + s % per_head) * kBT;
      // buffer s % 2: a thread reaches this step's barrier only after every
      // thread has passed the previous one, so the buffer of step s - 2 is free
      float* const sl = sLse + (s & 1) * kBT;
      float* const sd = sDv + (s & 1) * kBT;
      if (threadIdx.x < kBT)
        sl[threadIdx.x] = stat;
      else
        sd[threadIdx.x - kBT] = stat;
      named_bar_sync(kBarLse, kComputeThreads);
      if (s + 1 < nsteps) stat = row_stat(s + 1);
      ok = __all_sync(0xffffffffu, ok && mbar_wait(s_full, s & 1, wc));
      uint32_t sv[64], dp[64];
      if (ok) {
        tc_fence_after();
        const uint32_t ts = tmem + lane_off + C::COL_S + hf * 64;
        const uint32_t td = tmem + lane_off + C::COL_DP + hf * 64;
        // tcgen05.ld/st are .aligned: the warp reconverges before each one
        // (the code around them branches per lane)
        __syncwarp();
        tmem_ld4x32_sync(ts, ts + 32, td, td + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]),
                         *reinterpret_cast<uint32_t(*)[32]>(&sv[32]),
                         *reinterpret_cast<uint32_t(*)[32]>(&dp[0]),
                         *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      }
      // P^T and dS^T are written packed over the first 64 columns of S^T and
      // dP^T, which the other warp of this quarter reads: both have read first
      named_bar_sync(kBarPair + quarter, 64);
      if (ok) {
        // visible query columns of this key: [clo, chi) of the tile
        int clo = 0, chi = min(kBT, Lqb - q0);
        if (jr >= Lkb) chi = 0;
        if (a.causal) clo = min(max(jr - off - q0, 0), kBT);
        // mask entries of this key for the tile's rows (ms2 apart): additive
        // (mrow) or boolean (mrowb)
        const T* mrow = nullptr;
        const uint8_t* mrowb = nullptr;
        if (a.mask && jr < Lkb) {
          const long long moff = b * a.ms0 + hq * a.ms1 + q0 * a.ms2 + jr;
          if (a.mask_bool)
            mrowb = static_cast<const uint8_t*>(a.mask) + moff;
          else
            mrow = static_cast<const T*>(a.mask) + moff;
        }
        uint32_t pk[32], dk[32];
        const bool plain = clo <= hf * 64 && chi >= hf * 64 + 64 && !mrow && !mrowb;
        if (__all_sync(0xffffffffu, plain)) {
          // every column of this half visible, no mask: p = 2^(s sl2 - LSE),
          // dS = p (dP - D) in packed pairs, -LSE and -D read 8 columns at a time
          const uint64_t SL = bf2_pack(a.sl2, a.sl2);
          const uint32_t la = smem_addr(sl + hf * 64), da = smem_addr(sd + hf * 64);
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const float4 l0 = bld4(la + c8 * 32), l1 = bld4(la + c8 * 32 + 16);
            const float4 d0 = bld4(da + c8 * 32), d1 = bld4(da + c8 * 32 + 16);
            const float nl[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
            const float nd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
              const int c2 = c8 * 4 + pp;
              const uint64_t X = bf2_fma(bf2_pack(__uint_as_float(sv[2 * c2]),
                                                  __uint_as_float(sv[2 * c2 + 1])),
                                         SL, bf2_pack(nl[2 * pp], nl[2 * pp + 1]));
              float x0, x1;
              bf2_unpack(X, x0, x1);
              const float p0 = ex2(x0), p1 = ex2(x1);
              const uint64_t DS = bf2_mul(
                  bf2_pack(p0, p1),
                  bf2_add(bf2_pack(__uint_as_float(dp[2 * c2]), __uint_as_float(dp[2 * c2 + 1])),
                          bf2_pack(nd[2 * pp], nd[2 * pp + 1])));
              float s0, s1;
              bf2_unpack(DS, s0, s1);
              pk[c2] = E::pack(p0, p1);
              dk[c2] = E::pack(s0, s1);
            }
          }
        } else {
#pragma unroll
        for (int c2 = 0; c2 < 32; ++c2) {
          float pv[2], dv2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = hf * 64 + 2 * c2 + e;  // query row within the tile
            bool vis = c >= clo && c < chi;
            float x = __uint_as_float(sv[2 * c2 + e]) * a.sl2;
            if (mrow || mrowb) {
              if (vis && mrowb) vis = mrowb[static_cast<long long>(c) * a.ms2] != 0;
              if (vis && mrow)
                x += mask_log2(E::to_f(mrow[static_cast<long long>(c) * a.ms2]), mask_huge_log2(a.sl2));
            }
            const float p = vis ? ex2(x + sl[c]) : 0.f;
            pv[e] = p;
            dv2[e] = p * (__uint_as_float(dp[2 * c2 + e]) + sd[c]);
          }
          pk[c2] = E::pack(pv[0], pv[1]);
          dk[c2] = E::pack(dv2[0], dv2[1]);
        }
        }
        __syncwarp();
        tmem_st32(tmem + lane_off + C::COL_S + hf * 32, pk);
        tmem_st32(tmem + lane_off + C::COL_DP + hf * 32, dk);
        // dS^T row r, query rows 64h..64h+63: column block h, 16-byte chunks
        // swizzled by the row (128-byte swizzle)
        uint8_t* drow = smem + C::ds_off(s) + hf * (kBT * 128) + r * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          *reinterpret_cast<uint4*>(drow + ((ch ^ (r & 7)) << 4)) =
              make_uint4(dk[4 * ch], dk[4 * ch + 1], dk[4 * ch + 2], dk[4 * ch + 3]);
        tmem_wait_st();
        fence_proxy_async_shared();  // dS^T is read by the dQ MMA
        tc_fence_before();
      }
      if constexpr (C::PIPE_DQ) {
        // Step s-1's MMAs are complete (waited before this thread's p_ready
        // arrival, so the phase cannot be confused with step s's); its dQ tile
        // is read while step s's MMAs write the other buffer.
        if (s > 0) ok = __all_sync(0xffffffffu, ok && mbar_wait(mma_done, (s - 1) & 1, wc));
        mbar_arrive(p_ready);
        if (s > 0) read_dq(s - 1);
      } else {
        mbar_arrive(p_ready);
        ok = __all_sync(0xffffffffu, ok && mbar_wait(mma_done, s & 1, wc));
        read_dq(s);
        tc_fence_before();
        mbar_arrive(dq_read);
      }
    }
    if constexpr (C::PIPE_DQ) {  // the last step's dQ tile
      if (nsteps > 0) {
        ok = __all_sync(0xffffffffu, ok && mbar_wait(mma_done, (nsteps - 1) & 1, wc));
        read_dq(nsteps - 1);
      }
    }
    // dK (scaled) and dV of key jr, D/2 columns per warp: complete after the
    // last step's MMAs.  The TMEM loads are warp-collective: every lane takes
    // them (ok is warp-uniform) and only keys inside Lk are stored.
    if (ok) {
      tc_fence_after();
      const bool key_ok = jr < a.Lk;
      T* dkrow = static_cast<T*>(a.dk) + b * a.dks0 + kvh * a.dks1 + jr * a.dks2 + hf * (D / 2);
      T* dvrow = static_cast<T*>(a.dv) + b * a.dvs0 + kvh * a.dvs1 + jr * a.dvs2 + hf * (D / 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t kv[32], vv[32];
        if (nsteps > 0) {
          __syncwarp();
          tmem_ld2x32_sync(tmem + lane_off + C::COL_DK + hf * (D / 2) + c * 32,
                           tmem + lane_off + C::COL_DV + hf * (D / 2) + c * 32, kv, vv);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) kv[e] = vv[e] = 0u;
        }
        uint32_t wk[16], wv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          wk[e] = E::pack(__uint_as_float(kv[2 * e]) * a.scale,
                          __uint_as_float(kv[2 * e + 1]) * a.scale);
          wv[e] = E::pack(__uint_as_float(vv[2 * e]), __uint_as_float(vv[2 * e + 1]));
        }
        if (key_ok) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            reinterpret_cast<uint4*>(dkrow + c * 32)[e] =
                make_uint4(wk[4 * e], wk[4 * e + 1], wk[4 * e + 2], wk[4 * e + 3]);
            reinterpret_cast<uint4*>(dvrow + c * 32)[e] =
                make_uint4(wv[4 * e], wv[4 * e + 1], wv[4 * e + 2], wv[4 * e + 3]);
          }
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (warp == kProducerWarp && lane == 0 && *abort_flag) {
    // a role gave up: every copy the producer issued lands before the CTA exits
    bwd_drain_wait(kv_full, 0, kDrainNs);
    for (int st = 0; st < 2; ++st)
      if (q_last[st] >= 0) bwd_drain_wait(&q_full[st], q_last[st] & 1, kDrainNs);
  }
}

size_t align256b(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t backward_workspace(const sdpa_params_t& p) {
  const size_t rows = static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q;
  return align256b(rows * p.head_dim * 4) + 2 * align256b(rows * 4);
}

void backward_stats_slots(const sdpa_params_t& p, void* workspace, float** lse2, float** dvec) {
  const size_t rows = static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  *lse2 = reinterpret_cast<float*>(w + align256b(rows * p.head_dim * 4));
  *dvec = reinterpret_cast<float*>(w + align256b(rows * p.head_dim * 4) + align256b(rows * 4));
}

sdpa_status_t launch_backward_pre(const sdpa_params_t& p, const void* o, const void* d_o,
                                  const float* lse, float* lse2, float* dvec, float* dq_acc,
                                  cudaStream_t stream) {
  PreArgs pa;
  pa.o = o;
  pa.d_o = d_o;
  pa.lse = lse;
  pa.lse2 = lse2;
  pa.dvec = dvec;
  pa.dq_acc = dq_acc;
  pa.seq_lens_q = p.seq_lens_q;
  pa.Hq = p.num_q_heads;
  pa.Lq = p.seq_len_q;
  pa.D = p.head_dim;
  pa.os0 = p.o_stride[0];
  pa.os1 = p.o_stride[1];
  pa.os2 = p.o_stride[2];
  pa.rows = static_cast<long long>(p.batch) * p.num_q_heads * p.seq_len_q;
  if (pa.rows <= 0) return SDPA_OK;
  const unsigned blocks = static_cast<unsigned>((pa.rows * 32 + 255) / 256);
  switch (p.dtype) {
    case SDPA_F32: bwd_pre_kernel<float><<<blocks, 256, 0, stream>>>(pa); break;
    case SDPA_F16: bwd_pre_kernel<__half><<<blocks, 256, 0, stream>>>(pa); break;
    default: bwd_pre_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(pa); break;
  }
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

namespace {

template <int D, bool BF16>
sdpa_status_t launch_bwd_impl(const sdpa_params_t& p, const void* q, const void* k,
                              const void* v, const void* o, const void* d_o, const float* lse,
                              void* dq, void* dk, void* dv, void* workspace,
                              const LaunchEnv& env) {
  using C = BwdCfg<D>;
  using T = typename BwdElem<BF16>::T;
  const long long rows = static_cast<long long>(p.batch) * p.num_q_heads * p.seq_len_q;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  float* dq_acc = reinterpret_cast<float*>(w);
  float* lse2 = reinterpret_cast<float*>(w + align256b(rows * D * 4));
  float* dvec = reinterpret_cast<float*>(w + align256b(rows * D * 4) + align256b(rows * 4));
  // D_i, LSE in log2 units, cleared dQ accumulator
  int launched = 0;
  if (rows > 0) {
    const sdpa_status_t st = launch_backward_pre(p, o, d_o, lse, lse2, dvec, dq_acc, env.stream);
    if (st != SDPA_OK) return st;
    ++launched;
  }
  if (p.seq_len_kv > 0) {
    const CUtensorMapDataType dt =
        BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint64_t B = p.batch, Hq = p.num_q_heads, Hkv = p.num_kv_heads;
    const uint64_t Lq = p.seq_len_q, Lk = p.seq_len_kv;
    CUtensorMap tq, tk, tv, tdo;
    auto enc = [&](CUtensorMap* m, const void* base, uint64_t L, uint64_t H,
                   const int64_t (&sd)[3]) {
      return encode_tiled_4d(m, dt, base, D, L, H, B, 2, 64, kBT, sd[2], sd[1], sd[0]);
    };
    // dO has o's layout; with no query row the Q and dO maps are never
    // read (they describe k's first row so that the driver accepts them)
    const bool noq = Lq == 0 || Hq == 0;
    if (!enc(&tq, noq ? k : q, noq ? 1 : Lq, noq ? 1 : Hq, noq ? p.k_stride : p.q_stride) ||
        !enc(&tk, k, Lk, Hkv, p.k_stride) || !enc(&tv, v, Lk, Hkv, p.v_stride) ||
        !enc(&tdo, noq ? k : d_o, noq ? 1 : Lq, noq ? 1 : Hq, noq ? p.k_stride : p.o_stride))
      return SDPA_ERR_CUDA;
    BwdArgs a;
    a.B = p.batch;
    a.Hq = p.num_q_heads;
    a.Hkv = p.num_kv_heads;
    a.G = p.num_q_heads / p.num_kv_heads;
    a.Lq = p.seq_len_q;
    a.Lk = p.seq_len_kv;
    a.sl2 = p.scale * kLog2eB;
    a.scale = p.scale;
    a.causal = p.causal ? 1 : 0;
    a.mask = p.mask;
    a.ms0 = p.mask_stride[0];
    a.ms1 = p.mask_stride[1];
    a.ms2 = p.mask_stride[2];
    a.mask_bool = (p.flags & SDPA_FLAG_BOOL_MASK) ? 1 : 0;
    a.lse2 = lse2;
    a.dvec = dvec;
    a.seq_lens_q = p.seq_lens_q;
    a.seq_lens_kv = p.seq_lens_kv;
    a.dq_acc = dq_acc;
    a.dk = dk;
    a.dv = dv;
    a.dks0 = p.k_stride[0];  // dK has k's layout, dV v's
    a.dks1 = p.k_stride[1];
    a.dks2 = p.k_stride[2];
    a.dvs0 = p.v_stride[0];
    a.dvs1 = p.v_stride[1];
    a.dvs2 = p.v_stride[2];
    a.status = env.status;
    a.wait_ns = env.wait_limit_ns;
    const bool lens = p.seq_lens_q || p.seq_lens_kv;
    auto kern = lens ? bwd_kernel<D, BF16, true> : bwd_kernel<D, BF16, false>;
    // The setmaxnreg split must fit the registers the kernel is launched with
    // (an increase beyond them would wait forever): check once per kernel.
    static int regs_ok[2] = {0, 0};  // 0 unknown, 1 fits, -1 does not
    if (regs_ok[lens] == 0) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return SDPA_ERR_CUDA;
      const long alloc = static_cast<long>((fa.numRegs + 7) & ~7) * kBwdThreads;
      const long need = static_cast<long>(kComputeThreads) * kComputeRegs +
                        static_cast<long>(kBwdThreads - kComputeThreads) * kControlRegs;
      regs_ok[lens] = alloc >= need ? 1 : -1;
    }
    if (regs_ok[lens] < 0) return SDPA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
      return SDPA_ERR_CUDA;
    const dim3 grid((p.seq_len_kv + kBT - 1) / kBT, p.num_kv_heads, p.batch);
    kern<<<grid, kBwdThreads, C::SMEM, env.stream>>>(tq, tk, tv, tdo, a);
    if (cudaGetLastError() != cudaSuccess) return SDPA_ERR_CUDA;
    ++launched;
  }
  PostArgs qa;
  qa.dq_acc = dq_acc;
  qa.dq = dq;
  qa.Hq = p.num_q_heads;
  qa.Lq = p.seq_len_q;
  qa.D = D;
  qa.scale = p.scale;
  qa.qs0 = p.q_stride[0];  // dQ has q's layout
  qa.qs1 = p.q_stride[1];
  qa.qs2 = p.q_stride[2];
  qa.rows = rows;
  if (rows > 0) {
    const unsigned row_blocks = static_cast<unsigned>((rows * 32 + 255) / 256);
    bwd_post_kernel<T><<<row_blocks, 256, 0, env.stream>>>(qa);
    if (cudaGetLastError() != cudaSuccess) return SDPA_ERR_CUDA;
    ++launched;
  }
  set_last_launches(launched);
  return SDPA_OK;
}

}  // namespace

sdpa_status_t launch_backward(const sdpa_params_t& p, const void* q, const void* k,
                              const void* v, const void* o, const void* d_o, const float* lse,
                              void* dq, void* dk, void* dv, void* workspace,
                              const LaunchEnv& env) {
  if (p.dtype == SDPA_F32)
    return launch_backward_f32(p, q, k, v, o, d_o, lse, dq, dk, dv, workspace, env);
  const bool bf16 = p.dtype == SDPA_BF16;
  if (p.head_dim == 64)
    return bf16 ? launch_bwd_impl<64, true>(p, q, k, v, o, d_o, lse, dq, dk, dv, workspace, env)
                : launch_bwd_impl<64, false>(p, q, k, v, o, d_o, lse, dq, dk, dv, workspace, env);
  if (p.head_dim == 128)
    return bf16 ? launch_bwd_impl<128, true>(p, q, k, v, o, d_o, lse, dq, dk, dv, workspace, env)
                : launch_bwd_impl<128, false>(p, q, k, v, o, d_o, lse, dq, dk, dv, workspace, env);
  return SDPA_ERR_UNSUPPORTED;
}

}  // namespace gb300
