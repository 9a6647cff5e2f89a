// prefill_tc.cuh — fused attention forward for fp16/bf16, head_dim 64/128,
// on the 5th-generation tensor cores of sm_103a: the kernel and its launch.
// Instantiated per head size in prefill_tc_d64.cu and prefill_tc_d128.cu,
// and for fp32 inputs (bf16 hi/lo parts, head_dim 64) in prefill_tc.cu.
//
// The computation is the tiled online-softmax forward of the rustytorch
// flash_attention.metal page (forward kernel: per key tile, row max, running
// max m and sum l, accumulator rescale by exp(m_old - m_new), final O / l
// and LSE = m + log l), with the options of the MLX pages (causal block
// skipping, bounds masking of the ragged key tail, additive mask, per-head
// sinks in the denominator, grouped-query head mapping).
//
// GB300 design (not the page's): one CTA owns NQ = 2 query tiles of 128 rows
// that share every K/V tile.  Warp roles:
//   warps 0-7  softmax: warpgroup t owns query tile t, one thread per row
//              (TMEM lane); it also rescales O in TMEM and writes the output;
//   warp 8     TMA producer: Q tiles once, then K_j, V_j into a ring of
//              shared-memory buffers (128-byte swizzle), and with a shared
//              key-mask row each stage's key bias column (kbias);
//   warp 9     MMA issuer: one elected lane issues tcgen05.mma,
//              S_t = Q_t K_j^T (A, B from shared memory, fp32 in TMEM) and
//              O_t += P_t V_j (P from TMEM, written there by the softmax
//              warps; V from shared memory), while the whole warp runs the
//              loop in step and meets the other roles only at named
//              barriers (no shared-memory access between MMAs);
//   warp 10    stage helper: waits for each K/V stage to land and passes
//              it to the MMA issuer;
//   warp 11    idle (completes the control warpgroup).
// Each ring stage holds K_j and V_j (one full and one empty barrier per
// step).  TMEM (512 columns): S_0 | S_1 | O_0 | O_1, with P written over
// the columns of S_t.  The issue order S_0,j+1 right after PV_0,j lets
// softmax of one tile overlap the MMAs of the other.  The O rescale is
// lazy: a row's reference max moves only when the new max exceeds it (by
// more than 8 in log2 units on masked tiles, or so far that a row sum passes
// 2^15 on interior tiles), so P stays <= 2^15.
//
// Scheduling: one CTA per SM, units (query-tile pair, head, batch) in a 1-D
// grid; causal grids take the heaviest query blocks of every head first.
// When the unit count leaves a partial last wave, its units go to a second
// grid (programmatic dependent launch, so it fills SMs as the first drains)
// that shares each unit's key tiles among the 2 or 4 CTAs of a cluster; the
// partial results (O, m, l) meet in the finalising CTA's shared memory
// through bulk copies and merge by the log-sum-exp rule of split-KV decode.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "tensor_map.h"

namespace gb300 {
namespace {

constexpr int BM = 128;  // query rows per tile (= TMEM lanes)
constexpr int BN = 128;  // keys per K/V tile
constexpr int NQ = 2;    // query tiles per CTA
constexpr int kSoftmaxWarps = 4 * NQ;
constexpr int kLoadWarp = kSoftmaxWarps;
constexpr int kMmaWarp = kSoftmaxWarps + 1;
// warps 8-11 form the control warpgroup (producer, MMA issuer, stage
// helper, one idle warp); it gives registers to the softmax warpgroups with
// setmaxnreg (launch: 384 x 168 = 256 x 224 + 128 x 56).
constexpr int kThreads = 32 * (kSoftmaxWarps + 4);
constexpr uint32_t kSoftmaxRegs = 224;
constexpr uint32_t kControlRegs = 56;
// named barriers: kBarP + t (softmax warps of tile t with the MMA warp),
// kBarK (stage helper with the MMA warp), kBarX + t (below)
constexpr uint32_t kBarP = 1;
constexpr uint32_t kBarK = kBarP + NQ;
constexpr uint32_t kBarX = kBarK + 1;  // + t: the 4 warps of tile t (split units)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units (masked path)
constexpr float kFusedSumLimit = 32768.0f;  // 2^15: bound on p (fused path)
constexpr int kMaxSplit = 4;  // CTAs that share the key tiles of one unit

// X3: fp32 inputs given as bf16 hi + lo splits (x = hi + lo + O(2^-16 x));
// S = Q_hi K_hi^T + Q_hi K_lo^T + Q_lo K_hi^T and O += P_hi V_hi + P_hi V_lo
// + P_lo V_hi, each product on the bf16 tensor path with fp32 accumulation.
template <int D, bool X3 = false>
struct Cfg {
  static constexpr int CB = D / 64;           // 128-byte column blocks per row
  static constexpr int TILE = BM * D * 2;     // bytes of one 128-row fp16/bf16 tile
  static constexpr int QT = X3 ? 2 : 1;       // tiles per query tile (hi, lo)
  static constexpr int KVT = X3 ? 4 : 2;      // tiles per stage: K (hi, lo), V (hi, lo)
  static constexpr int NS = X3 ? 2 : ((D == 64) ? 4 : 2);  // ring stages
  static constexpr int STAGE = KVT * TILE;
  static constexpr int K_LO = TILE;                  // offsets inside a stage
  static constexpr int V_OFF = (X3 ? 2 : 1) * TILE;
  static constexpr int V_LO = 3 * TILE;
  static constexpr int Q_OFF = 0;
  static constexpr int RING_OFF = NQ * QT * TILE;
  static constexpr int BAR_OFF = RING_OFF + NS * STAGE;
  // q_full, full[NS], empty[NS], s_full[NQ], o_done[NQ], drain, xbar,
  // q_empty; xbar: partial results of a split unit received; q_empty: the
  // unit's last S products have read the Q tiles
  static constexpr int NBARS = 1 + 2 * NS + 2 * NQ + 1 + 1 + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
  static constexpr int SMEM = MISC_OFF + 16 + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t s_col(int t) { return static_cast<uint32_t>(t * BN); }
  static constexpr uint32_t o_col(int t) { return static_cast<uint32_t>(NQ * BN + t * D); }
  static_assert(o_col(NQ - 1) + D <= TMEM_COLS, "TMEM budget");
  // split units: partial results of a tile, fp32 O rows (SLOT_O bytes) in the
  // ring and m, l (SLOT_ML bytes) over the Q tiles; a CTA holds up to
  // MAX_SPLIT slots (received ones and the ones it stages to send)
  static constexpr int SLOT_O = BM * D * 4;
  static constexpr int SLOT_ML = 2 * BM * 4;
  static constexpr int MAX_SPLIT = kMaxSplit * SLOT_O <= NS * STAGE ? kMaxSplit : 2;
  static_assert(MAX_SPLIT * SLOT_O <= NS * STAGE, "partial O slots fit the ring");
  static_assert(kMaxSplit * SLOT_ML <= NQ * QT * TILE, "partial m, l fit the Q tiles");
  static_assert(SMEM <= 232448, "shared memory budget");
  // Boolean key-mask bias (extended inputs, fp16/bf16): per ring stage a
  // chunk of BN keys x 16 columns whose column 0 holds 0 (visible) or -inf
  // per key, and per query tile a chunk of BM rows whose column 0 holds 1;
  // one more K step of S = Q K^T then adds the bias.  No-swizzle K-major
  // layout: core matrices of 8 rows x 16 bytes, the two of a row group
  // (columns 0-7, 8-15) 128 bytes apart (LBO), row groups 256 bytes apart
  // (SBO).
  static constexpr int BIAS_CHUNK = BN * 32;
  static constexpr int BIAS_LBO = 128;
  static constexpr int BIAS_SBO = 256;
  static constexpr int KB_OFF = (MISC_OFF + 16 + 127) / 128 * 128;
  static constexpr int QB_OFF = KB_OFF + NS * BIAS_CHUNK;
  static constexpr int SMEM_EXT = X3 ? SMEM : QB_OFF + NQ * BIAS_CHUNK + 1024;
  static_assert(BM == BN, "one bias chunk shape for keys and query rows");
  static_assert(SMEM_EXT <= 232448, "shared memory budget (extended inputs)");
  // byte offset of (row, column 0) inside a bias chunk
  static constexpr uint32_t bias_at(int r) {
    return static_cast<uint32_t>((r >> 3) * BIAS_SBO + (r & 7) * 16);
  }
};

struct PrefillArgs {
  int B, Hq, Hkv, G, Lq, Lk;
  int num_qblocks;
  // Work units (query block, head, batch) follow the linear block index
  // from unit0 on; a split grid gives each unit to the ksplit CTAs of a
  // thread-block cluster, which share its key tiles.
  int unit0;
  int ksplit;
  // units of the grid (whole units: CTA x takes unit0 + x, unit0 + x +
  // gridDim.x, ... below unit0 + nunits)
  int nunits;
  float sl2;  // scale * log2(e)
  int causal;
  const void* mask;
  long long ms0, ms1, ms2;  // mask element strides (last stride is 1)
  const float* sinks;
  void* o;
  float* lse;
  int* status;
  unsigned long long wait_ns;
  const int* seq_lens_q;   // nullptr or per-batch valid query rows
  const int* seq_lens_kv;  // nullptr or per-batch valid keys
  int mask_bool;           // mask holds bytes, nonzero = visible (EXT only)
  long long os0, os1, os2; // element strides of o (batch, head, row)
  // key-mask bias step (EXT, fp16/bf16): the mask row is shared by every
  // query row (row stride 0) and the scale is positive.  qbias holds the
  // query chunk's columns 0 and 1 (two fp16/bf16 values): 1 and 0 for a
  // boolean mask, 1/scale as hi + lo for an additive one.
  int kbias;
  uint32_t qbias;
  // EXT: a mask with a row per query copied into score tiles (mask_tiles.cu),
  // or nullptr.  Tile (plane, query tile, key tile) of 128 x 128 holds
  // [key group][128 rows][16 bytes]; plane = b * tm_bmul + h * tm_hmul.
  const uint8_t* tmask;
  int tm_nqt, tm_nkt, tm_bmul, tm_hmul;
};

template <bool BF16>
struct Elem;
template <>
struct Elem<true> {
  using T = __nv_bfloat16;
  static __device__ __forceinline__ float to_f(T x) { return __bfloat162float(x); }
  static __device__ __forceinline__ float bits_to_f(uint32_t h) { return __uint_as_float(h << 16); }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};
template <>
struct Elem<false> {
  using T = __half;
  static __device__ __forceinline__ float to_f(T x) { return __half2float(x); }
  static __device__ __forceinline__ float bits_to_f(uint32_t h) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
};

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

// ---------------------------------------------------------------- softmax math
// Pairs of fp32 values in one 64-bit register for the packed f32x2 FMA/add.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// p_i = 2^(s_i * sl2 - m) for one row of raw scores, packed to fp16/bf16
// pairs; rs receives the fp32 sum of the p_i.
// With X3, pk2 receives the bf16 residuals p - bf16(p) (P_lo).
template <bool BF16, int N, bool X3 = false>
__device__ __forceinline__ void softmax_pairs(const uint32_t (&s)[N], float sl2, float m,
                                              uint32_t (&pk)[N / 2], float& rs,
                                              uint32_t* pk2 = nullptr) {
  const uint64_t SL = f2_pack(sl2, sl2);
  const uint64_t NM = f2_pack(-m, -m);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const uint64_t X = f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])),
                              SL, NM);
    float x0, x1;
    f2_unpack(X, x0, x1);
    const float p0 = ex2(x0);
    const float p1 = ex2(x1);
    acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
    pk[i] = Elem<BF16>::pack(p0, p1);
    if constexpr (X3) {
      const float h0 = __uint_as_float(pk[i] << 16);
      const float h1 = __uint_as_float(pk[i] & 0xffff0000u);
      pk2[i] = Elem<true>::pack(p0 - h0, p1 - h1);
    }
  }
  const uint64_t t = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
  float t0, t1;
  f2_unpack(t, t0, t1);
  rs = t0 + t1;
}

// Max of the N values of one row (N a multiple of 16): eight running maxima
// (every column read exactly once), then combined.
template <int N>
__device__ __forceinline__ float row_max16(const float (&x)[N]) {
  static_assert(N % 16 == 0, "row length");
  float mr[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) mr[c] = x[c];
  // columns 8 .. N - 9 in pairs, then the last 8 singly
#pragma unroll
  for (int i = 8; i + 16 <= N - 8; i += 16)
#pragma unroll
    for (int c = 0; c < 8; ++c) mr[c] = fmax3(mr[c], x[i + 2 * c], x[i + 2 * c + 1]);
#pragma unroll
  for (int c = 0; c < 8; ++c) mr[c] = fmaxf(mr[c], x[N - 8 + c]);
  return fmaxf(fmax3(mr[0], mr[1], mr[2]), fmaxf(fmax3(mr[3], mr[4], mr[5]), fmaxf(mr[6], mr[7])));
}
// Max of the raw scores (fp32 bit patterns) of one row.
template <int N>
__device__ __forceinline__ float row_max_raw(const uint32_t (&s)[N]) {
  return row_max16(*reinterpret_cast<const float(*)[N]>(&s[0]));
}


// Bring the cache line holding global address p into L1 (a hint; p must
// point into a live allocation).
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

// Wait for a phase ignoring the abort flag (used only to drain in-flight
// asynchronous work before the CTA exits); bounded by limit_ns.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) break;
  }
}

// Work unit of a linear block index: (query block, head, batch) and, in a
// split grid, the CTA's part of the unit's key tiles (= its cluster rank).
// Causal grids take the heaviest query blocks of every head first.
struct Unit {
  int qb, h, b, part;
};
template <bool SPLIT>
__device__ __forceinline__ Unit unit_of(const PrefillArgs& a, uint32_t bx) {
  Unit w;
  const int u = a.unit0 + static_cast<int>(SPLIT ? bx / a.ksplit : bx);
  w.part = SPLIT ? static_cast<int>(bx % a.ksplit) : 0;
  if (a.causal) {
    const int hb = a.Hq * a.B;
    w.qb = a.num_qblocks - 1 - u / hb;
    w.h = (u % hb) % a.Hq;
    w.b = (u % hb) / a.Hq;
  } else {
    w.qb = u % a.num_qblocks;
    w.h = (u / a.num_qblocks) % a.Hq;
    w.b = u / (a.num_qblocks * a.Hq);
  }
  return w;
}

// Geometry of one work unit for one CTA: query block, head, batch, the
// CTA's part of a split unit, first query row, active query tiles, kv head,
// the batch's lengths (padding masks, clamped to the call's maxima: rows at
// or past Lqb see no key), the CTA's first key tile and the key tiles of each
// query tile (all of the CTA's part; causal: up to the tile's last visible
// key; splits are never causal).
struct Geo {
  int qb, h, b, part, m0, nt, kvh, Lkb, Lqb, jb, nmax;
  int nkv[NQ];
};
template <bool EXT, bool SPLIT>
__device__ __forceinline__ Geo unit_geo(const PrefillArgs& a, uint32_t bx) {
  Geo g;
  const Unit w = unit_of<SPLIT>(a, bx);
  g.qb = w.qb;
  g.h = w.h;
  g.b = w.b;
  g.part = w.part;
  g.m0 = w.qb * (BM * NQ);
  g.nt = min(NQ, (a.Lq - g.m0 + BM - 1) / BM);  // >= 1
  g.kvh = w.h / a.G;
  g.Lkb = (EXT && a.seq_lens_kv) ? min(max(a.seq_lens_kv[w.b], 0), a.Lk) : a.Lk;
  g.Lqb = (EXT && a.seq_lens_q) ? min(max(a.seq_lens_q[w.b], 0), a.Lq) : a.Lq;
  const int nkv_all = (g.Lkb + BN - 1) / BN;
  const int nparts = SPLIT ? a.ksplit : 1;
  g.jb = w.part * nkv_all / nparts;
  const int je = (w.part + 1) * nkv_all / nparts;
  g.nmax = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    int n = 0;
    const int last_row = min(g.m0 + t * BM + BM - 1, g.Lqb - 1);  // last row that sees keys
    if (t < g.nt && last_row >= g.m0 + t * BM) {
      if (a.causal) {
        const int lim = last_row + (g.Lkb - g.Lqb);  // last key visible to the tile
        n = lim < 0 ? 0 : min(nkv_all, lim / BN + 1);
      } else {
        n = je - g.jb;
      }
    }
    g.nkv[t] = n;
    g.nmax = max(g.nmax, n);
  }
  return g;
}

// Key columns whose exponentials are computed for key tile j of a unit
// (counted from the CTA's first): BN, except that on the last, ragged tile
// of a plain call at head_dim 64 without causal masking only its keys,
// rounded up to 32, are (the columns past them are masked: P = 0 there).
template <int D, bool X3, bool EXT>
__device__ __forceinline__ int tile_cols(const PrefillArgs& a, const Geo& u, int j) {
  if constexpr (D != 64 || X3 || EXT) {
    return BN;
  } else {
    if (a.causal) return BN;
    const int keys = u.Lkb - (u.jb + j) * BN;
    return keys >= BN ? BN : ((keys + 31) >> 5) << 5;
  }
}

// EXT: extended inputs (per-batch length arrays, a boolean mask, a mask row
// shared by every query row, or additive rows that are all 16-byte aligned);
// without them the lengths are the kernel arguments and the code is that of
// plain inputs (any strides of q, k, v and o; other additive masks on the
// general softmax path).
// SPLIT: every unit is shared by the CTAs of a cluster (the units of a last,
// partial wave); its own instantiation, so that whole units run code without
// the merge.
template <int D, bool BF16, bool X3, bool EXT, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmQ2,
                      const __grid_constant__ CUtensorMap tmK2,
                      const __grid_constant__ CUtensorMap tmV2, const PrefillArgs a) {
  using C = Cfg<D, X3>;
  using E = Elem<BF16>;
  // element type of the output and of the mask: the caller's dtype (fp32 in X3)
  using T = std::conditional_t<X3, float, typename E::T>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment of the shared-memory window (128-byte swizzle atoms).
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sQ = smem + C::Q_OFF;
  uint8_t* sRing = smem + C::RING_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* full = bars + 1;
  uint64_t* empty = full + C::NS;
  uint64_t* s_full = empty + C::NS;
  uint64_t* o_done = s_full + NQ;
  uint64_t* drain = o_done + NQ;
  uint64_t* xbar = drain + 1;
  uint64_t* q_empty = xbar + 1;
  uint8_t* sKB = smem + C::KB_OFF;  // key-mask bias chunks (extended inputs)
  uint8_t* sQB = smem + C::QB_OFF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // a split grid that follows the grid of whole units may start as soon as
  // every CTA of that grid is running
  if constexpr (!SPLIT) griddep_launch_dependents();
  // Units of this CTA.  A split grid gives one unit to the ksplit CTAs of a
  // cluster.  The grid of whole units may be persistent: in round k CTA x
  // takes unit k G + x (k even) or k G + G - 1 - x (k odd), G = gridDim.x,
  // below nunits (the snake order evens out causal units, which come
  // heaviest first), and every role runs on from one unit into the next (the producer loads the next unit's Q once the last S
  // products of the current one have read the Q tiles, and its K/V through
  // the same ring; the MMA warp issues its first S products right behind the
  // current unit's last P V), so that the start of a unit overlaps the end
  // of the previous one.
  const int bxi = static_cast<int>(blockIdx.x);
  const int gdx = static_cast<int>(gridDim.x);
  const int rounds = a.nunits / gdx;
  const int rem = a.nunits - rounds * gdx;
  const int n_my =
      SPLIT ? 1 : rounds + ((rem > 0 && ((rounds & 1) ? bxi >= gdx - rem : bxi < rem)) ? 1 : 0);
  auto geo = [&](int it) {
    const int x = (it & 1) ? gdx - 1 - bxi : bxi;
    return unit_geo<EXT, SPLIT>(a, static_cast<uint32_t>(SPLIT ? bxi : it * gdx + x));
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < NQ; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&o_done[t], 1);
    }
    mbar_init(drain, 1);
    mbar_init(xbar, 1);
    mbar_init(q_empty, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  // A mask row that every query row shares (row stride 0, e.g. a key padding
  // mask) enters S through the tensor cores on the fused path: the producer
  // writes each stage's key bias (boolean: 0 / -inf in column 0; additive:
  // the mask value in columns 0 and 1), the query chunks hold qbias, and the
  // MMA warp adds one K step: S + bias / scale, so x = S * scale*log2e gains
  // mask * log2e.  Written here through
  // the generic proxy, read by the tensor cores: zero the key chunks, write
  // the query chunks, then a proxy fence before the CTA barrier.
  const bool kbias = EXT && !X3 && a.kbias;
  if (kbias) {
    uint4* z = reinterpret_cast<uint4*>(sKB);
    constexpr int n16 = (C::NS + NQ) * C::BIAS_CHUNK / 16;
    constexpr int q16 = C::NS * C::BIAS_CHUNK / 16;  // first word of the query chunks
    for (int i = threadIdx.x; i < n16; i += kThreads) {
      // a query-chunk word of columns 0-7 starts a 256-byte row group's first half
      const bool col0 = i >= q16 && ((i * 16) % C::BIAS_SBO) < C::BIAS_LBO;
      // column 2 of the query chunks holds 1 (huge key-mask values)
      z[i] = make_uint4(col0 ? a.qbias : 0u, col0 ? (BF16 ? 0x3f80u : 0x3c00u) : 0u, 0u, 0u);
    }
    fence_proxy_async_shared();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{a.wait_ns, abort_flag, a.status};
  int last_use[C::NS];  // producer: last fill of each ring buffer (-1: none)
  int last_q = -1;      // producer: last unit whose Q tiles it loaded
#pragma unroll
  for (int s = 0; s < C::NS; ++s) last_use[s] = -1;

  // launch: 384 threads x 168 registers; the control warpgroup drops to 56
  // and the softmax warpgroups rise to 224 (256*224 + 128*56 = 384*168).
  if (warp >= kSoftmaxWarps) {
    setmaxnreg_dec<kControlRegs>();
  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    // Per unit: its Q tiles (after the previous unit's last S products have
    // read them), then K_j, V_j into the ring, which runs on across units.
    // With the key-mask bias step the whole warp fills each stage's bias
    // chunk before lane 0 arms the stage; otherwise lane 0 alone works.
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    if (kbias || lane == 0) {
      const uint32_t ninf = BF16 ? 0xff80u : 0xfc00u;
      int g = 0;  // ring stages filled so far
      bool pok = true;
      for (int it = 0; it < n_my && pok; ++it) {
        const Geo u = geo(it);
        if (lane == 0) {
          if (it > 0) pok = mbar_wait(q_empty, (it - 1) & 1, wc);
          if (pok) {
            last_q = it;
            mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(u.nt * C::QT * C::TILE));
            for (int t = 0; t < u.nt; ++t)
              for (int cb = 0; cb < C::CB; ++cb) {
                tma_load_4d(sQ + t * C::QT * C::TILE + cb * BM * 128, &tmQ, q_full, cb * 64,
                            u.m0 + t * BM, u.h, u.b);
                if constexpr (X3)
                  tma_load_4d(sQ + (t * C::QT + 1) * C::TILE + cb * BM * 128, &tmQ2, q_full,
                              cb * 64, u.m0 + t * BM, u.h, u.b);
              }
          }
        }
        if (kbias) pok = __shfl_sync(0xffffffffu, pok ? 1 : 0, 0) != 0;
        if (!pok) break;
        const long long moff = kbias ? u.b * a.ms0 + u.h * a.ms1 : 0;
        const uint8_t* mk = static_cast<const uint8_t*>(a.mask) + moff;    // boolean
        const uint16_t* mv = static_cast<const uint16_t*>(a.mask) + moff;  // additive
        for (int j = 0; j < u.nmax; ++j, ++g) {
          const int s = g % C::NS;
          const int use = g / C::NS;
          const int key0 = (u.jb + j) * BN;
          if (kbias) {
            // each lane writes the bias of keys 32c + lane of the tile
            const bool w = use == 0 || mbar_wait(&empty[s], (use - 1) & 1, wc);
            if (!__all_sync(0xffffffffu, w)) {
              pok = false;
              break;
            }
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
              const int r = 32 * c + lane;
              const int key = key0 + r;
              uint32_t v = ninf;  // keys past this batch's length: -inf
              uint32_t v2 = 0u;   // columns 2, 3
              if (key < u.Lkb) {
                if (a.mask_bool) {
                  v = mk[key] != 0 ? 0u : ninf;
                } else {
                  // columns 0 and 1 (1/scale = hi + lo); with lo = 0 column 1
                  // stays 0, so that a -inf mask value never meets a zero.  A
                  // finite value of magnitude 2^64 or more goes to column 2
                  // (query side 1) as -+2^100, so that S is exactly that.
                  const uint32_t m16 = mv[key];
                  const uint32_t mag = m16 & 0x7fffu;
                  if (BF16 && mag >= 0x5f80u && mag < 0x7f80u) {
                    v = 0u;
                    v2 = (m16 & 0x8000u) | 0x7180u;  // 2^100
                  } else {
                    v = m16 | ((a.qbias >> 16) != 0u ? (m16 << 16) : 0u);
                  }
                }
              }
              if constexpr (BF16) {  // columns 0-3 (fp16 holds no huge value: column 2 stays 0)
                *reinterpret_cast<uint2*>(sKB + s * C::BIAS_CHUNK + C::bias_at(r)) = make_uint2(v, v2);
              } else {
                *reinterpret_cast<uint32_t*>(sKB + s * C::BIAS_CHUNK + C::bias_at(r)) = v;
              }
            }
            fence_proxy_async_shared();
            __syncwarp();
          } else if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, wc)) {
            pok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&full[s], C::STAGE);
            uint8_t* st = sRing + s * C::STAGE;
            for (int cb = 0; cb < C::CB; ++cb) {
              tma_load_4d(st + cb * BN * 128, &tmK, &full[s], cb * 64, key0, u.kvh, u.b);
              tma_load_4d(st + C::V_OFF + cb * BN * 128, &tmV, &full[s], cb * 64, key0, u.kvh,
                          u.b);
              if constexpr (X3) {
                tma_load_4d(st + C::K_LO + cb * BN * 128, &tmK2, &full[s], cb * 64, key0, u.kvh,
                            u.b);
                tma_load_4d(st + C::V_LO + cb * BN * 128, &tmV2, &full[s], cb * 64, key0, u.kvh,
                            u.b);
              }
            }
          }
          last_use[s] = use;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs the issue loop in step; one lane, picked by
    // elect.sync inside each instruction, issues, so the warp never branches
    // around it.  The loop touches no shared memory: the softmax warps of
    // tile t hand P_t over through named barrier kBarP + t and the stage
    // helper reports each K/V stage that has landed through kBarK (an
    // mbarrier poll, a local-memory spill or a warp reconvergence here holds
    // the issuing thread until the MMAs in flight drain), also at the start
    // of each unit (Q and the first K/V stage landed).  Fixed order:
    // PV_0,j S_0,j+1 PV_1,j S_1,j+1, so each tile's next scores are ready as
    // early as possible; the next unit's S_t,0 follow its last P V products.
    const uint32_t lead = lane == 0 ? 1u : 0u;
    constexpr uint32_t idS = idesc_f16(BF16, BM, BN, false, false);
    constexpr uint32_t idO = idesc_f16(BF16, BM, D, false, true);
    // Descriptors of Q_0 and ring buffer 0.  Other tiles, buffers and K
    // steps differ only in the start-address field (bits 0-13, 16-byte
    // units) of the low word, so the loop adds 32-bit offsets to the low
    // words and pairs them with the fixed high words.
    const uint64_t q_desc = sdesc(smem_addr(sQ), 16, 1024, kSwizzle128B);
    const uint64_t k_desc = sdesc(smem_addr(sRing), 16, 1024, kSwizzle128B);
    const uint64_t v_desc = sdesc(smem_addr(sRing), BN * 128, 1024, kSwizzle128B);
    const uint32_t qk_hi = static_cast<uint32_t>(q_desc >> 32);
    const uint32_t v_hi = static_cast<uint32_t>(v_desc >> 32);
    const uint32_t q_lo = static_cast<uint32_t>(q_desc);
    const uint32_t k_lo = static_cast<uint32_t>(k_desc);
    const uint32_t v_lo = static_cast<uint32_t>(v_desc);
    auto qk = [&](uint32_t lo) { return (static_cast<uint64_t>(qk_hi) << 32) | lo; };
    // key-mask bias chunks (no swizzle): query chunk t, key chunk of a stage
    const uint64_t qb_desc = sdesc(smem_addr(sQB), C::BIAS_LBO, C::BIAS_SBO, 0);
    const uint64_t kb_desc = sdesc(smem_addr(sKB), C::BIAS_LBO, C::BIAS_SBO, 0);
    auto vv = [&](uint32_t lo) { return (static_cast<uint64_t>(v_hi) << 32) | lo; };
    // ring stage of the g-th K/V tile loaded by this CTA
    auto stage = [](int g) { return g % C::NS; };
    // The issuer never waits on an mbarrier itself, so it does not learn of
    // a wait that gave up elsewhere; it keeps issuing (the products may then
    // read stale tiles: the call reports the timeout and its results are
    // not used) and meets every named barrier, so that no role can hang.
    const uint32_t go = 1u;
    // S_t = Q_t K_j^T: both operands K-major, 128-byte swizzle; a K step of
    // 16 elements is 32 bytes inside a 128-byte row, 4 steps per column block.
    auto issue_s = [&](int t, int g) {
      const uint32_t qd = q_lo + static_cast<uint32_t>((t * C::QT * C::TILE) >> 4);
      const uint32_t kd = k_lo + static_cast<uint32_t>((stage(g) * C::STAGE) >> 4);
      const uint32_t dS = tmem + C::s_col(t);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4;
        mma_f16_ss_elect(dS, qk(qd + off), qk(kd + off), idS, kk > 0 ? 1u : 0u, go);
        if constexpr (X3) {  // Q_hi K_lo^T + Q_lo K_hi^T
          mma_f16_ss_elect(dS, qk(qd + off), qk(kd + (C::K_LO >> 4) + off), idS, 1u, go);
          mma_f16_ss_elect(dS, qk(qd + (C::TILE >> 4) + off), qk(kd + off), idS, 1u, go);
        }
      }
      if constexpr (EXT && !X3) {  // + 1 * bias_j: the key mask
        if (kbias)
          mma_f16_ss_elect(dS, qb_desc + static_cast<uint32_t>((t * C::BIAS_CHUNK) >> 4),
                           kb_desc + static_cast<uint32_t>((stage(g) * C::BIAS_CHUNK) >> 4),
                           idS, 1u, go);
      }
    };
    // O_t += P_t V_j: P (128 x 128, K-major) from TMEM columns of S_t,
    // 2 elements per column; V MN-major: 64-wide column blocks BN*128 bytes
    // apart (LBO), 8-key groups 1024 bytes apart (SBO).  In X3, P_hi sits in
    // the first 64 columns of S_t and P_lo in the next 64.
    auto issue_pv = [&](int t, int g, bool first) {
      const uint32_t vd = v_lo + static_cast<uint32_t>((stage(g) * C::STAGE + C::V_OFF) >> 4);
      const uint32_t dO = tmem + C::o_col(t);
      const uint32_t aP = tmem + C::s_col(t);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const uint32_t voff = (kk * 16 * 128) >> 4;
        mma_f16_ts_elect(dO, aP + kk * 8, vv(vd + voff), idO, (!first || kk > 0) ? 1u : 0u, go);
        if constexpr (X3) {  // P_hi V_lo + P_lo V_hi
          mma_f16_ts_elect(dO, aP + kk * 8, vv(vd + ((C::V_LO - C::V_OFF) >> 4) + voff), idO, 1u,
                           go);
          mma_f16_ts_elect(dO, aP + BN / 2 + kk * 8, vv(vd + voff), idO, 1u, go);
        }
      }
    };
    int g0 = 0;  // K/V tiles of earlier units (ring position of this unit's first)
    for (int it = 0; it < n_my; ++it) {
      const Geo u = geo(it);
      // this unit's Q tiles and first K/V stage have landed (stage helper)
      named_bar_sync(kBarK, 64);
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < NQ; ++t) {
        if (t >= u.nt) continue;
        if (u.nkv[t] == 0) {
          mma_commit_elect(&o_done[t], go);
        } else {
          issue_s(t, g0);
          mma_commit_elect(&s_full[t], go);
        }
      }
      // the Q tiles are free for the next unit once the last S products of
      // this one have completed
      if (u.nmax <= 1) mma_commit_elect(q_empty, go);
      for (int j = 0; j < u.nmax; ++j) {
        bool kwaited = false;
        // stage j+1 has landed (the helper saw it); once per step
        auto wait_stage = [&]() {
          if (!kwaited) {
            named_bar_sync(kBarK, 64);
            kwaited = true;
          }
        };
#pragma unroll
        for (int t = 0; t < NQ; ++t) {
          if (t >= u.nt || j >= u.nkv[t]) continue;
          // P_t,j is in TMEM (4 softmax warps and this one meet)
          named_bar_sync(kBarP + t, 32 * 5);
          tc_fence_after();
          issue_pv(t, g0 + j, j == 0);
          if (j + 1 < u.nkv[t]) {
            wait_stage();
            issue_s(t, g0 + j + 1);
            mma_commit_elect(&s_full[t], go);
          } else {
            mma_commit_elect(&o_done[t], go);
          }
        }
        if (j == u.nmax - 2) mma_commit_elect(q_empty, go);
        // stage j (K_j read by S_t,j, V_j by PV_t,j) is free once these land
        mma_commit_elect(&empty[stage(g0 + j)], go);
      }
      g0 += u.nmax;
    }
    // every MMA issued by this warp completes before TMEM is freed
    mma_commit_elect(drain, go);
    if (lead) drain_wait(drain, 0, kDrainNs);
    __syncwarp();
  } else if (warp == kMmaWarp + 1) {
    // -------------------------------------------------------- stage helper
    // Per unit: waits for its Q tiles and first K/V stage, then for stage
    // j+1 of every step that reads one, and hands each to the MMA issuer
    // through kBarK (same count of meetings on both sides, also after a
    // failed wait).
    bool ok = true;
    int g0 = 0;
    for (int it = 0; it < n_my; ++it) {
      const Geo u = geo(it);
      ok = ok && mbar_wait(q_full, static_cast<uint32_t>(it & 1), wc);
      if (u.nmax > 0)
        ok = ok && mbar_wait(&full[g0 % C::NS], static_cast<uint32_t>((g0 / C::NS) & 1), wc);
      named_bar_sync(kBarK, 64);
      for (int j = 0; j + 1 < u.nmax; ++j) {
        const int g = g0 + j + 1;
        ok = ok && mbar_wait(&full[g % C::NS], static_cast<uint32_t>((g / C::NS) & 1), wc);
        named_bar_sync(kBarK, 64);
      }
      g0 += u.nmax;
    }
  }
  // a split unit's CTAs meet twice at the end (partial results written, then
  // read); every thread of the cluster takes part
  if constexpr (SPLIT) {
    __syncwarp();
    cluster_sync_all();
    cluster_sync_all();
  }
  } else {
    setmaxnreg_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------- softmax
    const int t = warp >> 2;
    const int r = (warp & 3) * 32 + lane;  // row inside the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::s_col(t);
    const uint32_t tO = tmem + lane_off + C::o_col(t);
    bool ok = true;
    int sph = 0;  // phases of s_full[t] consumed (earlier units)
    int oph = 0;  // phases of o_done[t] consumed (earlier units)
    for (int it = 0; it < n_my; ++it) {
    const Geo u = geo(it);
    const int qb = u.qb, h = u.h, b = u.b, part = u.part, m0 = u.m0, nt = u.nt;
    const int Lkb = u.Lkb, Lqb = u.Lqb, jb = u.jb;
    const int nkv_t = t == 0 ? u.nkv[0] : u.nkv[1];
    (void)qb;
    const int qi = m0 + t * BM + r;        // query row
    const bool row_ok = qi < a.Lq;
    // last key visible to this row (bounds and causal)
    int limit = Lkb - 1;
    if (a.causal) limit = min(limit, qi + (Lkb - Lqb));
    if (EXT && qi >= Lqb) limit = -1;  // a padding row sees no key
    // additive mask row (mrow) or, with EXT, boolean mask row (mrowb)
    const T* mrow = nullptr;
    const uint8_t* mrowb = nullptr;
    if (a.mask && row_ok) {
      const long long moff = b * a.ms0 + h * a.ms1 + qi * a.ms2 + jb * BN;
      if (EXT && a.mask_bool)
        mrowb = static_cast<const uint8_t*>(a.mask) + moff;
      else
        mrow = static_cast<const T*>(a.mask) + moff;
    }
    // A mask row shared by every query row (boolean or additive) reaches the
    // fused path through S itself (kbias); a mask with a row per query takes
    // 16-byte loads where the row is 16-byte aligned.
    // With the mask's score-tile copy, this row's 16 bytes of key group 0 of
    // key tile jb; group g of tile jb + j is g * 2048 (additive) or g * 2048
    // (boolean: 16 keys a group) further, tile j at j tile-bytes.
    const uint8_t* mt = nullptr;
    if (EXT && a.tmask && row_ok) {
      const long long plane = static_cast<long long>(b) * a.tm_bmul + h * a.tm_hmul;
      mt = a.tmask +
           ((plane * a.tm_nqt + qi / BM) * a.tm_nkt + jb) * (a.mask_bool ? 16384 : 32768) +
           (qi % BM) * 16;
    }
    const bool mrow16 =
        EXT && mrowb && !kbias && (mt || (reinterpret_cast<uintptr_t>(mrowb) & 15u) == 0);
    const bool mrowa16 =
        EXT && mrow && !kbias && (mt || (reinterpret_cast<uintptr_t>(mrow) & 15u) == 0);
    // keys are counted from this CTA's first key tile from here on
    limit -= jb * BN;
    float m = -INFINITY;  // reference max (log2 units)
    float l = 0.f;        // running sum relative to m
    // interior tiles take the fused path when the scores need no mask and
    // the scale is positive (max of raw scores = max of scaled scores)
    const bool fast_ok = (a.sl2 > 0.f) && (a.mask == nullptr);
    // tiles that may hold invisible keys take the fused path too at D = 128,
    // and with extended inputs (masks, per-batch lengths) at any D
    constexpr bool kFusedPartial = (D == 128) || EXT;
    // With extended inputs a mask takes the fused path too: a shared row is
    // in S already (kbias); a boolean row sets -inf (16-byte loads where
    // aligned, else byte loads); an additive row adds mask / scale to the
    // raw scores (x = S * scale*log2e then gains mask * log2e) when every
    // lane's row is 16-byte aligned (a warp-wide choice: the host routes
    // calls whose additive rows are not all aligned to the plain
    // instantiation, and a warp never runs both paths), on tiles inside the
    // row's visible keys.  Other warps and tiles take the general path.
    const bool mvec = __all_sync(0xffffffffu, mrowb ? mrow16 : (mrow ? mrowa16 : true));
    const bool fused_ok =
        (a.sl2 > 0.f) && (a.mask == nullptr || (EXT && (kbias || a.mask_bool || mvec)));
    const float rscale = kLog2e / a.sl2;  // 1 / scale
    // Huge mask values (magnitude 2^64 or more) exist only in bfloat16 and
    // float masks.  Key masks (one row shared by the query rows) give them
    // their exact form: on the key-mask MMA step (bfloat16) and, in the fp32
    // hi/lo kernel, on the extended instantiation's general path; so do the
    // fused path's bfloat16 rows (masks with a row per query, read from the
    // score-tile copy or aligned rows).  The general path keeps the plain
    // product, whose unrolled code is a third of the size (carried by the
    // boundary tiles' general path, its size alone measured 3.5 % of the
    // unmasked DiT loop): there a finite value whose scaled product overflows
    // fp32 acts as -inf.
    constexpr bool kHugeMask = EXT && X3;
    const float mhuge = mask_huge_log2(a.sl2);  // a huge mask value in log2 units
    auto mlog2 = [&](float mv) { return kHugeMask ? mask_log2(mv, mhuge) : mv * kLog2e; };
    // Output of the tile (whole units: right after its loop; split units:
    // after the CTAs of the cluster have exchanged partial results).
    auto epilogue = [&]() {
      const int qi = m0 + t * BM + r;
      const bool row_ok = qi < a.Lq;
      // A split unit: CTA `part` finalises query tile `part` (part < NQ); each
      // other CTA sends it its partial result of that tile (O relative to
      // 2^m, m, l): staged in its own shared memory, then one bulk copy into
      // a slot of the finaliser's, counted on the finaliser's xbar.  Slot of
      // CTA q at finaliser t: q - (q > t); the first ksplit - 1 slots receive,
      // the next ones stage (a CTA that finalises nothing stages in slot t).
      // The cluster meets once every CTA's MMAs have completed (its buffers
      // are free) and its expectation is set, and again at the end, so that
      // no CTA leaves while its copies may still read its shared memory.
      uint8_t* const slotO = sRing;
      uint8_t* const slotML = sQ;
      if constexpr (SPLIT) {
        for (int t2 = 0; t2 < nt; ++t2)
          if (ok) ok = mbar_wait(&o_done[t2], 0, wc);
        ok = __all_sync(0xffffffffu, ok);
        const int nin = a.ksplit - 1;
        if (t < nt && t == part && r == 0)
          mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(nin * (C::SLOT_O + C::SLOT_ML)));
        const int st = part < NQ ? nin : t;  // staging slot
        const bool send = t < nt && t != part && ok;
        if (send) {
          tc_fence_after();
          __syncwarp();
          float4* prow = reinterpret_cast<float4*>(slotO + st * C::SLOT_O + r * D * 4);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ob[32];
            tmem_ld32_sync(tO + c * 32, ob);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
              if (l > 0.f)  // a tile that saw no key holds no O
                v = make_float4(__uint_as_float(ob[4 * i]), __uint_as_float(ob[4 * i + 1]),
                                __uint_as_float(ob[4 * i + 2]), __uint_as_float(ob[4 * i + 3]));
              prow[(c * 8 + i) ^ (r & 7)] = v;
            }
          }
          float* ml = reinterpret_cast<float*>(slotML + st * C::SLOT_ML);
          ml[r] = m;
          ml[BM + r] = l;
          fence_proxy_async_shared();
        }
        named_bar_sync(kBarX + t, 128);  // the tile's rows are staged
        __syncwarp();
        cluster_sync_all();
        if (send && r == 0) {
          const uint32_t dst = static_cast<uint32_t>(t);
          const int slot = part - (part > t ? 1 : 0);
          const uint32_t bar = cluster_map(xbar, dst);
          bulk_copy_to_cluster(cluster_map(slotO + slot * C::SLOT_O, dst),
                               smem_addr(slotO + st * C::SLOT_O), C::SLOT_O, bar);
          bulk_copy_to_cluster(cluster_map(slotML + slot * C::SLOT_ML, dst),
                               smem_addr(slotML + st * C::SLOT_ML), C::SLOT_ML, bar);
        }
        // the finaliser waits for its slots whatever happened before: no CTA
        // may leave while copies into or out of it are in flight
        if (t < nt && t == part) {
          const bool got = mbar_wait_cluster(xbar, 0, wc);
          ok = __all_sync(0xffffffffu, ok && got);
        }
      }
      if (t < nt && ok && (!SPLIT || t == part)) {
        tc_fence_after();
        // split unit: merge the other CTAs' partial results of this tile,
        // M = max of the m's, weights 2^(m - M), l = sum of l * weight
        float w_own = 1.f;
        float wq[kMaxSplit - 1];
        if constexpr (SPLIT) {
          float M = m;
          float mq[kMaxSplit - 1], lq[kMaxSplit - 1];
#pragma unroll
          for (int q = 0; q < kMaxSplit - 1; ++q) {
            mq[q] = -INFINITY;
            lq[q] = 0.f;
            if (q < a.ksplit - 1) {
              const float* ml = reinterpret_cast<const float*>(slotML + q * C::SLOT_ML);
              mq[q] = ml[r];
              lq[q] = ml[BM + r];
            }
            M = fmaxf(M, mq[q]);
          }
          w_own = (l > 0.f) ? ex2(m - M) : 0.f;
          float L = (l > 0.f) ? l * w_own : 0.f;
#pragma unroll
          for (int q = 0; q < kMaxSplit - 1; ++q) {
            wq[q] = (lq[q] > 0.f) ? ex2(mq[q] - M) : 0.f;
            L += lq[q] * wq[q];
          }
          m = M;
          l = L;
        }
        // sink logit joins the denominator only (value row 0)
        float oscale = 1.f;
        if (a.sinks) {
          const float sk = a.sinks[h] * kLog2e;
          const float mn = fmaxf(m, sk);
          oscale = ex2(m - mn);
          l = l * oscale + ex2(sk - mn);
          m = mn;
        }
        const float inv = (l > 0.f) ? oscale / l : 0.f;
        T* orow = static_cast<T*>(a.o) + (b * a.os0 + h * a.os1 + qi * a.os2);
        __syncwarp();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ob[32];
          tmem_ld32_sync(tO + c * 32, ob);
          if constexpr (SPLIT) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              ob[i] = __float_as_uint((w_own > 0.f) ? __uint_as_float(ob[i]) * w_own : 0.f);
#pragma unroll
            for (int q = 0; q < kMaxSplit - 1; ++q) {
              if (q < a.ksplit - 1) {
                const float4* srow =
                    reinterpret_cast<const float4*>(slotO + q * C::SLOT_O + r * D * 4);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 v = srow[(c * 8 + i) ^ (r & 7)];
                  ob[4 * i] = __float_as_uint(fmaf(v.x, wq[q], __uint_as_float(ob[4 * i])));
                  ob[4 * i + 1] =
                      __float_as_uint(fmaf(v.y, wq[q], __uint_as_float(ob[4 * i + 1])));
                  ob[4 * i + 2] =
                      __float_as_uint(fmaf(v.z, wq[q], __uint_as_float(ob[4 * i + 2])));
                  ob[4 * i + 3] =
                      __float_as_uint(fmaf(v.w, wq[q], __uint_as_float(ob[4 * i + 3])));
                }
              }
            }
          }
          if constexpr (X3) {  // fp32 output
#pragma unroll
            for (int i = 0; i < 32; ++i)
              ob[i] = __float_as_uint((inv == 0.f) ? 0.f : __uint_as_float(ob[i]) * inv);
            if (row_ok) {
              uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[i] = make_uint4(ob[4 * i], ob[4 * i + 1], ob[4 * i + 2], ob[4 * i + 3]);
            }
          } else {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float v0 = (inv == 0.f) ? 0.f : __uint_as_float(ob[2 * i]) * inv;
              const float v1 = (inv == 0.f) ? 0.f : __uint_as_float(ob[2 * i + 1]) * inv;
              w[i] = E::pack(v0, v1);
            }
            if (row_ok) {
              uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            }
          }
        }
        if (row_ok && a.lse) {
          a.lse[(static_cast<size_t>(b) * a.Hq + h) * a.Lq + qi] =
              (l > 0.f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
        }
      }
      if constexpr (SPLIT) {  // every copy has landed before any CTA of the cluster leaves
        __syncwarp();
        cluster_sync_all();
      }
    };
    if (t < nt) {
      for (int j = 0; j < nkv_t; ++j) {
        // a 16-byte aligned per-query mask row is brought into L1 before the
        // scores are waited for, and loaded after with 16-byte loads
        // (measured: prefetching unaligned rows, read byte by byte, slowed
        // the loop)
        if constexpr (EXT) {
          const int kv0 = j * BN;
          if (mt) {
            // the warp's 32 rows of a key group are 512 contiguous bytes (4
            // lines): lanes l, l + 8, l + 16, l + 24 cover a group's lines
            const int g = r & 7;
            if (a.mask_bool) {
              prefetch_l1(mt + j * 16384 + g * 2048);
            } else {
              prefetch_l1(mt + j * 32768 + (2 * g) * 2048);
              prefetch_l1(mt + j * 32768 + (2 * g + 1) * 2048);
            }
          } else if (kv0 + BN - 1 <= limit) {
            if (mrow16) {
              prefetch_l1(mrowb + kv0);
              prefetch_l1(mrowb + kv0 + BN - 1);
            } else if (mrowa16) {
              prefetch_l1(mrow + kv0);
              prefetch_l1(mrow + kv0 + BN - 1);
            }
          }
        }
        ok = __all_sync(0xffffffffu, ok && mbar_wait(&s_full[t], (sph + j) & 1, wc));
        if (ok) {
          tc_fence_after();
          uint32_t s[BN];
          static_assert(BN == 128, "score tile of 4 x 32 TMEM columns");
          // tcgen05.ld/st are .aligned: the whole warp executes each one
          // together.  Code before them may branch per lane (mask and bounds
          // tests, spin waits); without an explicit reconvergence point the
          // compiler may leave the warp split here (measured: a build did, and
          // the loaded scores were wrong).
          __syncwarp();
          tmem_ld4x32_sync(tS, tS + 32, tS + 64, tS + 96,
                           *reinterpret_cast<uint32_t(*)[32]>(&s[0]),
                           *reinterpret_cast<uint32_t(*)[32]>(&s[32]),
                           *reinterpret_cast<uint32_t(*)[32]>(&s[64]),
                           *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
          const int kv0 = j * BN;
          float alpha = 1.f;
          bool resc;
          float rs;
          uint32_t pk[BN / 2];
          uint32_t pk2[X3 ? BN / 2 : 1];  // P_lo (X3)
          const bool fast = fast_ok && kv0 + BN - 1 <= limit;
          if constexpr (X3) {
            // bf16 hi/lo P: computed half a row at a time and stored to TMEM
            // as soon as each half exists, so that the 128 scores plus one
            // half of P_hi and P_lo are the most that is live at once.  The
            // scores are used raw with p = 2^(s * scale*log2e - m) on the
            // fused path, and as scaled, masked x = s * scale*log2e + bias
            // (rewritten in place) with p = 2^(x - m) elsewhere.
            float mul = a.sl2;
            if (!fast) {
#pragma unroll
              for (int i = 0; i < BN; ++i) {
                float x = __uint_as_float(s[i]) * a.sl2;
                if (mrow && kv0 + i <= limit) x += mlog2(to_float(mrow[kv0 + i]));
                if (EXT && mrowb && kv0 + i <= limit && !mrowb[kv0 + i]) x = -INFINITY;
                if (kv0 + i > limit) x = -INFINITY;
                s[i] = __float_as_uint(x);
              }
              mul = 1.f;
            }
            // fused rows with a reference max skip the tile max, others take it
            bool need_max = !fast || !(m > -INFINITY);
            resc = false;
            for (int pass = 0; pass < 2; ++pass) {
              if (need_max) {
                const float mx = row_max_raw(s) * mul;
                // the fused path always moves to the tile max; the general
                // path only when it grew by more than the threshold
                if (fast || mx > m + kRescaleThreshold) {
                  alpha = ex2(m - mx);  // 0 when m = -inf
                  m = mx;
                  resc = true;
                }
              }
              const float mu = (m == -INFINITY) ? 0.f : m;
              if (pass > 0) tmem_wait_st();  // the first pass's P is overwritten
              __syncwarp();
              float rs0, rs1;
              softmax_pairs<BF16, BN / 2, true>(
                  *reinterpret_cast<const uint32_t(*)[BN / 2]>(&s[0]), mul, mu,
                  *reinterpret_cast<uint32_t(*)[BN / 4]>(&pk[0]), rs0, &pk2[0]);
              tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
              tmem_st32(tS + BN / 2, *reinterpret_cast<uint32_t(*)[32]>(&pk2[0]));
              softmax_pairs<BF16, BN / 2, true>(
                  *reinterpret_cast<const uint32_t(*)[BN / 2]>(&s[BN / 2]), mul, mu,
                  *reinterpret_cast<uint32_t(*)[BN / 4]>(&pk[BN / 4]), rs1, &pk2[BN / 4]);
              tmem_st32(tS + BN / 4, *reinterpret_cast<uint32_t(*)[32]>(&pk[BN / 4]));
              tmem_st32(tS + BN / 2 + BN / 4, *reinterpret_cast<uint32_t(*)[32]>(&pk2[BN / 4]));
              rs = rs0 + rs1;
              // a fused row whose sum exceeds 2^15 (its max grew) takes the
              // tile max and the warp computes the tile again; the second
              // pass cannot fail (every p <= 1)
              const bool redo = fast && !need_max && !(rs <= kFusedSumLimit);
              if (!__any_sync(0xffffffffu, redo)) break;
              need_max = redo;
            }
          } else if (kFusedPartial
                         ? fused_ok && !(mrow && !kbias && !(EXT && mt) && kv0 + BN - 1 > limit)
                         : fast) {
            // Positive scale, no additive mask: p = 2^(s * scale*log2e - m)
            // with the scale folded into one packed FMA per pair, taken
            // against the current reference max m without looking for the
            // tile max.  Every p is at most the row sum, so a sum <= 2^15
            // proves all p <= 2^15 (exact range in fp16 and bf16); only a row
            // whose sum exceeds it (its max grew) or that has no max yet finds
            // the tile max of the raw scores and repeats.  At D = 128, and
            // with extended inputs at any D, the tiles that cross the row's
            // last visible key (bounds, causal diagonal) or carry a boolean
            // mask take this path too, with their invisible keys scored -inf;
            // at D = 64 on plain inputs, where the softmax warps set the pace,
            // the few boundary tiles stay on the general path below
            // (measured: routing them here slowed the loop).
            if (!fast) {
              if (kv0 + BN - 1 > limit) {
                const int nvis = limit - kv0 + 1;  // visible keys of the row here
#pragma unroll
                for (int i = 0; i < BN; ++i)
                  if (i >= nvis) s[i] = 0xff800000u;  // -inf
              }
              // the mask row of this query row (a shared one is already in S:
              // kbias)
              if constexpr (EXT) {
                if (kbias) {
                  // nothing to apply
                } else if (mrow16 && (mt || kv0 + BN - 1 <= limit)) {
                  // 16 keys a load: the row's own bytes, or its group rows of
                  // the score-tile copy (keys past the row's limit are -inf
                  // already; the copy is in bounds for every key of the tile)
                  const uint4* src = mt ? reinterpret_cast<const uint4*>(mt + j * 16384)
                                        : reinterpret_cast<const uint4*>(mrowb + kv0);
                  const int cstep = mt ? 128 : 1;
#pragma unroll
                  for (int c = 0; c < BN / 16; ++c) {
                    const uint4 q4 = src[c * cstep];
                    const uint32_t wd[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                      if (((wd[e >> 2] >> (8 * (e & 3))) & 0xffu) == 0u)
                        s[16 * c + e] = 0xff800000u;
                  }
                } else if (mrowb) {
#pragma unroll
                  for (int i = 0; i < BN; ++i)
                    if (kv0 + i <= limit && !mrowb[kv0 + i]) s[i] = 0xff800000u;
                } else if (mrow && mrowa16 && (mt || kv0 + BN - 1 <= limit)) {
                  // additive row, 8 values a load: the row where it is 16-byte
                  // aligned, else its group rows of the score-tile copy
                  const uint4* src = mt ? reinterpret_cast<const uint4*>(mt + j * 32768)
                                        : reinterpret_cast<const uint4*>(mrow + kv0);
                  const int cstep = mt ? 128 : 1;
#pragma unroll
                  for (int c = 0; c < BN / 8; ++c) {
                    const uint4 q4 = src[c * cstep];
                    const uint32_t wd[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                      const float mv = E::bits_to_f((wd[e >> 1] >> (16 * (e & 1))) & 0xffffu);
                      // a bfloat16 value of magnitude 2^64 or more enters as
                      // +-2^100 raw-score units (exact; fp16 has none)
                      const bool huge = BF16 && fabsf(mv) >= kMaskBig;
                      s[8 * c + e] = __float_as_uint(fmaf(huge ? copysignf(kMaskHugeRaw, mv) : mv,
                                                          huge ? 1.f : rscale,
                                                          __uint_as_float(s[8 * c + e])));
                    }
                  }
                }
              }
            }
            resc = !(m > -INFINITY);
            if (!resc) {
              softmax_pairs<BF16, BN>(s, a.sl2, m, pk, rs);
              resc = !(rs <= kFusedSumLimit);  // also true for inf or nan
            }
            if (resc) {
              const float mx = row_max_raw(s) * a.sl2;  // -inf: no visible key
              // (a row may see no key of a partial tile: m stays)
              if (!kFusedPartial || mx > -INFINITY) {
                alpha = ex2(m - mx);  // 0 when m = -inf
                m = mx;
              }
              softmax_pairs<BF16, BN>(s, a.sl2, (kFusedPartial && m == -INFINITY) ? 0.f : m,
                                      pk, rs);
            }
          } else {
            float x[BN];
#pragma unroll
            for (int i = 0; i < BN; ++i) x[i] = __uint_as_float(s[i]) * a.sl2;
            if (mrow) {
#pragma unroll
              for (int i = 0; i < BN; ++i)
                if (kv0 + i <= limit) x[i] += mlog2(to_float(mrow[kv0 + i]));
            }
            if constexpr (EXT) {
              if (mrowb) {
#pragma unroll
                for (int i = 0; i < BN; ++i)
                  if (kv0 + i <= limit && !mrowb[kv0 + i]) x[i] = -INFINITY;
              }
            }
            if (kv0 + BN - 1 > limit) {
#pragma unroll
              for (int i = 0; i < BN; ++i)
                if (kv0 + i > limit) x[i] = -INFINITY;
            }
            const float mx = row_max16(x);
            resc = mx > m + kRescaleThreshold;  // true on the first visible tile
            if (resc) {
              alpha = ex2(m - mx);  // 0 when m = -inf
              m = mx;
            }
            const float mu = (m == -INFINITY) ? 0.f : m;
            float rp[4] = {0.f, 0.f, 0.f, 0.f};
            // columns past a narrowed tile's nw are not computed (P = 0)
            const int nw = tile_cols<D, X3, EXT>(a, u, j);
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
              if (c * 32 < nw) {
#pragma unroll
                for (int i = 16 * c; i < 16 * c + 16; ++i) {
                  const float p0 = ex2(x[2 * i] - mu);
                  const float p1 = ex2(x[2 * i + 1] - mu);
                  rp[i & 3] += p0 + p1;
                  pk[i] = E::pack(p0, p1);
                }
              } else {
#pragma unroll
                for (int i = 16 * c; i < 16 * c + 16; ++i) pk[i] = 0u;
              }
            }
            rs = (rp[0] + rp[1]) + (rp[2] + rp[3]);
          }
          __syncwarp();
          l = l * alpha + rs;
          // O_t holds the sum through PV_{t,j-1} (complete: the commit behind
          // s_full tracks every earlier MMA); rescale rows whose max moved.
          if (j > 0 && __any_sync(0xffffffffu, resc)) {
            __syncwarp();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t ob[32];
              tmem_ld32_sync(tO + c * 32, ob);
#pragma unroll
              for (int i = 0; i < 32; ++i) ob[i] = __float_as_uint(__uint_as_float(ob[i]) * alpha);
              tmem_st32(tO + c * 32, ob);
            }
          }
          if constexpr (!X3) {
            tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
          }
          tmem_wait_st();
          tc_fence_before();
        }
        // hand P_t,j to the MMA warp; met every step, also after a failed wait
        named_bar_sync(kBarP + t, 32 * 5);
      }
      if (ok) ok = mbar_wait(&o_done[t], static_cast<uint32_t>(oph & 1), wc);
      ok = __all_sync(0xffffffffu, ok);
      if constexpr (!SPLIT) epilogue();
      sph += nkv_t;
      ++oph;
    }
    if constexpr (SPLIT) epilogue();
    }  // units
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (warp == kLoadWarp && lane == 0 && *abort_flag) {
    // a role gave up: every copy the producer issued lands before the CTA exits
    if (last_q >= 0) drain_wait(q_full, static_cast<uint32_t>(last_q & 1), kDrainNs);
    for (int s = 0; s < C::NS; ++s)
      if (last_use[s] >= 0) drain_wait(&full[s], last_use[s] & 1, kDrainNs);
  }
  // a split grid ends after the grid of whole units that it overlaps
  if constexpr (SPLIT) griddep_wait();
}

// Element strides (batch, head, row) of q, k and v as passed to launch_impl
// (in X3, of the hi/lo copies; q2, k2, v2 share them).
struct QkvStrides {
  int64_t q[3], k[3], v[3];
};

template <int D, bool BF16, bool X3, bool EXT>
sdpa_status_t launch_impl(const sdpa_params_t& p, const void* q, const void* k, const void* v,
                          const void* q2, const void* k2, const void* v2, void* o, float* lse,
                          const QkvStrides& st, const LaunchEnv& env, int* grids) {
  using C = Cfg<D, X3>;
  // extended inputs carry the key-mask bias chunks
  constexpr int kSmem = EXT ? C::SMEM_EXT : C::SMEM;
  const CUtensorMapDataType dt =
      BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t B = p.batch, Hq = p.num_q_heads, Hkv = p.num_kv_heads;
  const uint64_t Lq = p.seq_len_q, Lk = p.seq_len_kv;
  // [B, H, L, D] with the given strides, viewed innermost-first; box 64 x 128
  // rows, 128-byte swizzle.  The maps stop at Lq and Lk: rows past them (a KV
  // cache keeps more) read as zero and are never loaded.
  CUtensorMap tq, tk, tv, tq2, tk2, tv2;
  auto enc = [&](CUtensorMap* m, const void* base, uint64_t L, uint64_t H, uint32_t box_rows,
                 const int64_t (&sd)[3]) {
    return encode_tiled_4d(m, dt, base, D, L, H, B, 2, 64, box_rows, sd[2], sd[1], sd[0]);
  };
  if (!enc(&tq, q, Lq, Hq, BM, st.q) || !enc(&tk, k, Lk, Hkv, BN, st.k) ||
      !enc(&tv, v, Lk, Hkv, BN, st.v))
    return SDPA_ERR_CUDA;
  if (X3) {
    if (!enc(&tq2, q2, Lq, Hq, BM, st.q) || !enc(&tk2, k2, Lk, Hkv, BN, st.k) ||
        !enc(&tv2, v2, Lk, Hkv, BN, st.v))
      return SDPA_ERR_CUDA;
  } else {
    tq2 = tq;
    tk2 = tk;
    tv2 = tv;
  }
  PrefillArgs a;
  a.B = p.batch;
  a.Hq = p.num_q_heads;
  a.Hkv = p.num_kv_heads;
  a.G = p.num_q_heads / p.num_kv_heads;
  a.Lq = p.seq_len_q;
  a.Lk = p.seq_len_kv;
  a.num_qblocks = (p.seq_len_q + BM * NQ - 1) / (BM * NQ);
  a.sl2 = p.scale * kLog2e;
  a.causal = p.causal ? 1 : 0;
  a.mask = p.mask;
  a.ms0 = p.mask_stride[0];
  a.ms1 = p.mask_stride[1];
  a.ms2 = p.mask_stride[2];
  a.sinks = p.sinks;
  a.o = o;
  a.lse = lse;
  a.status = env.status;
  a.wait_ns = env.wait_limit_ns;
  a.seq_lens_q = p.seq_lens_q;
  a.seq_lens_kv = p.seq_lens_kv;
  a.mask_bool = (p.flags & SDPA_FLAG_BOOL_MASK) ? 1 : 0;
  a.tmask = EXT ? static_cast<const uint8_t*>(env.mask_tiles) : nullptr;
  a.tm_nqt = (p.seq_len_q + 127) / 128;
  a.tm_nkt = (p.seq_len_kv + 127) / 128;
  a.tm_bmul = p.mask_stride[0] ? (p.mask_stride[1] ? p.num_q_heads : 1) : 0;
  a.tm_hmul = p.mask_stride[1] ? 1 : 0;
  a.os0 = p.o_stride[0];
  a.os1 = p.o_stride[1];
  a.os2 = p.o_stride[2];
  a.kbias = 0;
  a.qbias = 0;

  if (EXT && !X3 && p.mask && p.mask_stride[2] == 0 && p.scale > 0.f) {
    if (p.flags & SDPA_FLAG_BOOL_MASK) {
      a.kbias = 1;
      a.qbias = BF16 ? 0x3f80u : 0x3c00u;  // 1, 0
    } else {
      // 1/scale = hi + lo: hi rounded toward zero so that lo >= 0 (a -inf
      // mask value then gives -inf in both products)
      const float inv = 1.f / p.scale;
      uint32_t hi, lo;
      bool fits = true;
      if (BF16) {
        const __nv_bfloat16_raw h = __float2bfloat16_rz(inv);
        const __nv_bfloat16_raw l = __float2bfloat16_rn(inv - __bfloat162float(h));
        hi = h.x;
        lo = l.x;
      } else {
        fits = inv <= 65504.f;
        const __half_raw h = __float2half_rz(inv);
        const __half_raw l = __float2half_rn(inv - __half2float(h));
        hi = h.x;
        lo = l.x;
      }
      if (fits) {
        a.kbias = 1;
        a.qbias = hi | (lo << 16);

      }
    }
  }
  auto kern = prefill_tc_kernel<D, BF16, X3, EXT, false>;
  auto kern_split = prefill_tc_kernel<D, BF16, X3, EXT, true>;
  // The setmaxnreg split must fit the registers the kernel is launched with
  // (an increase beyond them would wait forever): check the compiled count
  // once per instantiation.
  static int regs_ok[2] = {0, 0};  // 0 unknown, 1 fits, -1 does not
  for (int v2 = 0; v2 < 2; ++v2) {
    if (regs_ok[v2] == 0) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, v2 ? kern_split : kern) != cudaSuccess) return SDPA_ERR_CUDA;
      const long alloc = static_cast<long>((fa.numRegs + 7) & ~7) * kThreads;
      const long need =
          32L * (kSoftmaxWarps * static_cast<long>(kSoftmaxRegs) + 4L * kControlRegs);
      regs_ok[v2] = alloc >= need ? 1 : -1;
    }
    if (regs_ok[v2] < 0) return SDPA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(v2 ? kern_split : kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmem) != cudaSuccess)
      return SDPA_ERR_CUDA;
  }
  // One CTA per SM: the last wave of units is partial when the unit count is
  // not a multiple of the SM count.  Those units go to a second grid that
  // splits each over its key tiles among the CTAs of a cluster (2 or 4,
  // whichever fits the free SMs), so that the last wave lasts a split, not a
  // whole unit; it starts while the first grid drains (programmatic
  // dependent launch).  Causal units differ in length and are ordered
  // heaviest first instead.
  const long long units = static_cast<long long>(a.num_qblocks) * p.num_q_heads * p.batch;
  if (units > 0x7fffffffLL) return SDPA_ERR_UNSUPPORTED;
  const int U = static_cast<int>(units);
  const int nkv = (p.seq_len_kv + BN - 1) / BN;
  int ksplit = 1, tail = 0;
  // test hook: -1 the plan's; 0 never; 2, 4 every unit
  const int forced = debug_option(SDPA_DEBUG_PREFILL_SPLIT);
  // (not for a call that shares the GPU: its last wave is not idle SMs)
  if (!p.causal && forced != 0 && (forced > 0 || !(p.flags & SDPA_FLAG_SHARED_GPU))) {
    static int active[2] = {0, 0};  // clusters of 2, 4 that can be resident (-1: none)
    const int r = U % env.num_sms;
    // (a split count above C::MAX_SPLIT would overflow the finaliser's slots)
    const int fk = forced > C::MAX_SPLIT ? C::MAX_SPLIT : forced;
    for (int k = C::MAX_SPLIT; k >= 2; k /= 2) {
      const bool want =
          (fk == k) || (fk < 0 && r > 0 && k * r <= env.num_sms && nkv >= 4 * k);
      if (!want) continue;
      int& act = active[k == 2 ? 0 : 1];
      if (act == 0) {
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = static_cast<unsigned>(k);
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t oc = {};
        oc.gridDim = dim3(static_cast<unsigned>(k * env.num_sms));
        oc.blockDim = dim3(kThreads);
        oc.dynamicSmemBytes = kSmem;
        oc.attrs = at;
        oc.numAttrs = 1;
        int n = 0;
        act = (cudaOccupancyMaxActiveClusters(&n, kern_split, &oc) == cudaSuccess && n > 0) ? n
                                                                                          : -1;
        cudaGetLastError();
      }
      if (fk == k && act > 0) {
        ksplit = k;
        tail = U;
        break;
      }
      if (act >= r) {  // every split unit of the last wave runs at once
        ksplit = k;
        tail = r;
        break;
      }
    }
  }
  const int n_whole = U - tail;
  *grids = 0;
  if (n_whole > 0) {
    a.unit0 = 0;
    a.ksplit = 1;
    a.nunits = n_whole;
    // Persistent grid (one CTA per SM looping over units); a call that
    // shares the GPU keeps one CTA per unit.
    const bool persist = !(p.flags & SDPA_FLAG_SHARED_GPU);
    const int grid = persist ? std::min(n_whole, env.num_sms) : n_whole;
    kern<<<dim3(static_cast<unsigned>(grid)), kThreads, kSmem, env.stream>>>(tq, tk, tv, tq2, tk2,
                                                                             tv2, a);
    if (cudaGetLastError() != cudaSuccess) return SDPA_ERR_CUDA;
    *grids = 1;
  }
  if (tail == 0) return SDPA_OK;
  a.unit0 = n_whole;
  a.ksplit = ksplit;
  a.nunits = tail;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(ksplit);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ksplit * tail));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = env.stream;
  cfg.attrs = attr;
  cfg.numAttrs = n_whole > 0 ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, kern_split, tq, tk, tv, tq2, tk2, tv2, a) != cudaSuccess)
    return SDPA_ERR_CUDA;
  *grids += 1;
  return SDPA_OK;
}

}  // namespace

// Whether a call takes the EXT instantiation: per-batch lengths, a boolean
// mask, a mask row shared by every query row (the key-mask bias step), or an
// additive mask whose rows are all 16-byte aligned.  Other additive masks
// stay on the plain instantiation's general path (measured faster there for
// unaligned rows than any EXT path).
inline bool prefill_needs_ext(const sdpa_params_t& p) {
  if (p.seq_lens_q || p.seq_lens_kv) return true;
  if (!p.mask) return false;
  if ((p.flags & SDPA_FLAG_BOOL_MASK) || p.mask_stride[2] == 0) return true;
  // an additive mask with a row per query: the fused path with 16-byte
  // loads when every row is 16-byte aligned (fp16/bf16)
  if (p.dtype == SDPA_F32) return false;
  const int64_t es = 2;
  bool aligned = (reinterpret_cast<uintptr_t>(p.mask) & 15u) == 0;
  for (int d = 0; d < 3; ++d) aligned = aligned && (p.mask_stride[d] * es) % 16 == 0;
  return aligned;
}

// Head-size entry points (one translation unit each), p normalised;
// `grids` receives the number of grids launched (1, or 2 when the last
// wave is split).
sdpa_status_t launch_prefill_tc_d64(const sdpa_params_t& p, const void* q, const void* k,
                                    const void* v, void* o, float* lse, const LaunchEnv& env,
                                    int* grids);
sdpa_status_t launch_prefill_tc_d128(const sdpa_params_t& p, const void* q, const void* k,
                                     const void* v, void* o, float* lse, const LaunchEnv& env,
                                     int* grids);
// head_dim 512, fp16/bf16 (prefill_d512.cu)
sdpa_status_t launch_prefill_tc_d512(const sdpa_params_t& p, const void* q, const void* k,
                                     const void* v, void* o, float* lse, const LaunchEnv& env,
                                     int* grids);

}  // namespace gb300
