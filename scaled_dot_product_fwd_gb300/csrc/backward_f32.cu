// backward_f32.cu — gradients dQ, dK, dV of the attention forward for fp32
// inputs (head_dim 64/128), on the CUDA cores in fp32 throughout.
//
// The computation is the backward pass of the rustytorch flash_attention.metal
// page (its backward kernels for dQ and for dK, dV), as in backward.cu:
// P = exp(S - LSE) recomputed from the forward's log-sum-exp, D_i = dO_i . O_i,
// dS = P (dP - D) with dP = dO V^T, dQ = scale dS K, dK = scale dS^T Q,
// dV = P^T dO; the options of the mlx cuDNN backward graph (scale,
// bottom-right causal mask, additive or boolean mask, sink token through
// LSE) and per-batch lengths.
//
// Two kernels and no atomics, as the page splits the work: kernel A holds a
// tile of 64 keys of one (kv head, batch) and walks the query tiles of every
// query head of the group, keeping dK and dV of its keys in registers;
// kernel B holds a tile of 64 query rows and walks the key tiles, keeping dQ.
// Each recomputes S and dP per (query tile, key tile) pair.  A thread owns a
// 4 x 4 block of a pair's 64 x 64 scores: K^T and V^T sit transposed in
// shared memory (4 keys per 16-byte load), Q and dO row-major (each load a
// broadcast of two addresses per warp).  The pre pass of backward.cu gives
// LSE in log2 units (+inf where a row takes no part) and D_i.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int kT = 64;         // query rows and keys of a tile
constexpr int kThreads = 256;  // 16 x 16 threads, 4 x 4 elements each
constexpr int kPadT = kT + 4;  // pitch of the [D][64] and [64][64] tiles (floats)

template <int D>
struct F32Cfg {
  static constexpr int PQ = D + 4;  // pitch of the row-major [64][D] tiles
  static constexpr int NDV = D / 16;  // head dimensions per thread in dK, dV, dQ
  // kernel A: K^T, V^T [D][kPadT]; Q, dO [64][PQ]; P, dS [64][kPadT]; -LSE, -D
  static constexpr int A_KT = 0;
  static constexpr int A_VT = A_KT + D * kPadT;
  static constexpr int A_Q = A_VT + D * kPadT;
  static constexpr int A_DO = A_Q + kT * PQ;
  static constexpr int A_P = A_DO + kT * PQ;
  static constexpr int A_DS = A_P + kT * kPadT;
  static constexpr int A_ST = A_DS + kT * kPadT;
  static constexpr int A_BYTES = (A_ST + 2 * kT) * 4;
  // kernel B: Q, dO [64][PQ]; K^T, V^T [D][kPadT]; K [64][PQ]; dS [64][kPadT]; -LSE, -D
  static constexpr int B_Q = 0;
  static constexpr int B_DO = B_Q + kT * PQ;
  static constexpr int B_KT = B_DO + kT * PQ;
  static constexpr int B_VT = B_KT + D * kPadT;
  static constexpr int B_K = B_VT + D * kPadT;
  static constexpr int B_DS = B_K + kT * PQ;
  static constexpr int B_ST = B_DS + kT * kPadT;
  static constexpr int B_BYTES = (B_ST + 2 * kT) * 4;
  static_assert(A_BYTES <= 232448 && B_BYTES <= 232448, "shared memory budget");
};

struct F32Args {
  const float* q;
  const float* k;
  const float* v;
  const float* d_o;
  const float* lse2;  // [B, Hq, Lq]: LSE in log2 units (+inf: the row takes no part)
  const float* dvec;  // [B, Hq, Lq]: D_i = dO_i . O_i
  float* dq;
  float* dk;
  float* dv;
  long long qs0, qs1, qs2;  // q and dq
  long long ks0, ks1, ks2;  // k and dk
  long long vs0, vs1, vs2;  // v and dv
  long long os0, os1, os2;  // dO (o's layout)
  const void* mask;
  long long ms0, ms1, ms2;
  int mask_bool;
  const int* seq_lens_q;
  const int* seq_lens_kv;
  int Hq, Hkv, G, Lq, Lk, causal;
  float sl2;    // scale * log2(e)
  float scale;
};

// Rows [r0, r0 + 64) of a slab (row stride rs elements, D contiguous) into a
// row-major [64][D + 4] tile; rows at or past n read as zero.
template <int D>
__device__ __forceinline__ void load_rows(float* dst, const float* src, long long rs, int r0,
                                          int n) {
  for (int e = threadIdx.x; e < kT * D; e += kThreads) {
    const int r = e / D, c = e % D;
    dst[r * (D + 4) + c] = (r0 + r < n) ? src[static_cast<long long>(r0 + r) * rs + c] : 0.f;
  }
}
// The same rows transposed into [D][kPadT].
template <int D>
__device__ __forceinline__ void load_rows_t(float* dst, const float* src, long long rs, int r0,
                                            int n) {
  for (int e = threadIdx.x; e < kT * D; e += kThreads) {
    const int r = e / D, c = e % D;
    dst[c * kPadT + r] = (r0 + r < n) ? src[static_cast<long long>(r0 + r) * rs + c] : 0.f;
  }
}

// acc[a][c] = sum over d of A[4 tr + a][d] * Bt[d][4 tk + c] (A row-major
// [64][D + 4], Bt transposed [D][kPadT]).
template <int D>
__device__ __forceinline__ void tile_dot(const float* A, const float* Bt, int tr, int tk,
                                         float (&acc)[4][4]) {
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
#pragma unroll 8
  for (int d = 0; d < D; ++d) {
    const float4 b = *reinterpret_cast<const float4*>(Bt + d * kPadT + 4 * tk);
    float x[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) x[a] = A[(4 * tr + a) * (D + 4) + d];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      acc[a][0] = fmaf(x[a], b.x, acc[a][0]);
      acc[a][1] = fmaf(x[a], b.y, acc[a][1]);
      acc[a][2] = fmaf(x[a], b.z, acc[a][2]);
      acc[a][3] = fmaf(x[a], b.w, acc[a][3]);
    }
  }
}

// P and dS of a thread's 4 x 4 block of one (query tile q0, key tile k0)
// pair: rows q0 + 4 tr + a, keys k0 + 4 tk + c.  s and dp are the raw
// products; nl, nd hold -LSE (log2) and -D of the tile's rows.
struct PairCtx {
  int q0, k0, Lqb, Lkb, off, hq, b;
};
__device__ __forceinline__ void p_ds(const F32Args& a, const PairCtx& x, int tr, int tk,
                                     const float (&s)[4][4], const float (&dp)[4][4],
                                     const float* nl, const float* nd, float (&p)[4][4],
                                     float (&ds)[4][4]) {
  const float mhuge = mask_huge_log2(a.sl2);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int ti = 4 * tr + r;
    const int i = x.q0 + ti;
    const long long mrow = x.b * a.ms0 + x.hq * a.ms1 + static_cast<long long>(i) * a.ms2;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = x.k0 + 4 * tk + c;
      bool vis = i < x.Lqb && j < x.Lkb && (!a.causal || j <= i + x.off);
      float y = s[r][c] * a.sl2;
      if (a.mask) {
        if (a.mask_bool) {
          vis = vis && static_cast<const uint8_t*>(a.mask)[mrow + j] != 0;
        } else {
          const float mv = vis ? static_cast<const float*>(a.mask)[mrow + j] : 0.f;
          y += mask_log2(mv, mhuge);
        }
      }
      const float pv = vis ? ex2(y + nl[ti]) : 0.f;
      p[r][c] = pv;
      ds[r][c] = pv * (dp[r][c] + nd[ti]);
    }
  }
}

// -LSE (log2) and -D of query rows [q0, q0 + 64) of head hq (rows past Lqb:
// -inf and 0, so that their P is 0)
__device__ __forceinline__ void load_stats(const F32Args& a, float* st, int b, int hq, int q0,
                                           int Lqb) {
  if (threadIdx.x < 2 * kT) {
    const int t = threadIdx.x & (kT - 1);
    const int i = q0 + t;
    const size_t row = (static_cast<size_t>(b) * a.Hq + hq) * a.Lq + i;
    if (threadIdx.x < kT)
      st[t] = i < Lqb ? -a.lse2[row] : -INFINITY;
    else
      st[kT + t] = i < Lqb ? -a.dvec[row] : 0.f;
  }
}

// Kernel A: dK and dV of 64 keys (blockIdx.x) of kv head blockIdx.y, batch
// blockIdx.z.
template <int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_f32_dkdv_kernel(const F32Args a) {
  using C = F32Cfg<D>;
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  float* sKt = sm + C::A_KT;
  float* sVt = sm + C::A_VT;
  float* sQ = sm + C::A_Q;
  float* sDO = sm + C::A_DO;
  float* sP = sm + C::A_P;
  float* sDS = sm + C::A_DS;
  float* sSt = sm + C::A_ST;
  const int k0 = blockIdx.x * kT;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int Lkb = a.seq_lens_kv ? min(max(a.seq_lens_kv[b], 0), a.Lk) : a.Lk;
  const int Lqb = a.seq_lens_q ? min(max(a.seq_lens_q[b], 0), a.Lq) : a.Lq;
  const int off = Lkb - Lqb;  // key j visible to row i iff j <= i + off (causal)
  const int tk = threadIdx.x & 15, tr = threadIdx.x >> 4;
  // query tiles that hold a row seeing a key of this tile
  const int nqt = (Lqb + kT - 1) / kT;
  int qt0 = 0;
  if (a.causal && k0 - off > 0) qt0 = (k0 - off) / kT;
  const bool any = k0 < Lkb && qt0 < nqt;
  float accK[4][C::NDV], accV[4][C::NDV];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < C::NDV; ++c) accK[r][c] = accV[r][c] = 0.f;
  if (any) {
    load_rows_t<D>(sKt, a.k + b * a.ks0 + kvh * a.ks1, a.ks2, k0, Lkb);
    load_rows_t<D>(sVt, a.v + b * a.vs0 + kvh * a.vs1, a.vs2, k0, Lkb);
    for (int g = 0; g < a.G; ++g) {
      const int hq = kvh * a.G + g;
      for (int qt = qt0; qt < nqt; ++qt) {
        const int q0 = qt * kT;
        __syncthreads();  // the previous pair's tiles are consumed
        load_rows<D>(sQ, a.q + b * a.qs0 + hq * a.qs1, a.qs2, q0, Lqb);
        load_rows<D>(sDO, a.d_o + b * a.os0 + hq * a.os1, a.os2, q0, Lqb);
        load_stats(a, sSt, b, hq, q0, Lqb);
        __syncthreads();
        float s[4][4], dp[4][4], p[4][4], ds[4][4];
        tile_dot<D>(sQ, sKt, tr, tk, s);
        tile_dot<D>(sDO, sVt, tr, tk, dp);
        const PairCtx x{q0, k0, Lqb, Lkb, off, hq, b};
        p_ds(a, x, tr, tk, s, dp, sSt, sSt + kT, p, ds);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          *reinterpret_cast<float4*>(sP + (4 * tr + r) * kPadT + 4 * tk) =
              make_float4(p[r][0], p[r][1], p[r][2], p[r][3]);
          *reinterpret_cast<float4*>(sDS + (4 * tr + r) * kPadT + 4 * tk) =
              make_float4(ds[r][0], ds[r][1], ds[r][2], ds[r][3]);
        }
        __syncthreads();
        // dV[key][d] += P[row][key] dO[row][d]; dK[key][d] += dS[row][key] Q[row][d]
        // (thread: keys 4 tk + r, head dimensions NDV tr + c)
#pragma unroll 4
        for (int row = 0; row < kT; ++row) {
          const float4 p4 = *reinterpret_cast<const float4*>(sP + row * kPadT + 4 * tk);
          const float4 s4 = *reinterpret_cast<const float4*>(sDS + row * kPadT + 4 * tk);
          const float pr[4] = {p4.x, p4.y, p4.z, p4.w};
          const float sr[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
          for (int c4 = 0; c4 < C::NDV / 4; ++c4) {
            const float4 o4 =
                *reinterpret_cast<const float4*>(sDO + row * C::PQ + C::NDV * tr + 4 * c4);
            const float4 q4 =
                *reinterpret_cast<const float4*>(sQ + row * C::PQ + C::NDV * tr + 4 * c4);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              accV[r][4 * c4 + 0] = fmaf(pr[r], o4.x, accV[r][4 * c4 + 0]);
              accV[r][4 * c4 + 1] = fmaf(pr[r], o4.y, accV[r][4 * c4 + 1]);
              accV[r][4 * c4 + 2] = fmaf(pr[r], o4.z, accV[r][4 * c4 + 2]);
              accV[r][4 * c4 + 3] = fmaf(pr[r], o4.w, accV[r][4 * c4 + 3]);
              accK[r][4 * c4 + 0] = fmaf(sr[r], q4.x, accK[r][4 * c4 + 0]);
              accK[r][4 * c4 + 1] = fmaf(sr[r], q4.y, accK[r][4 * c4 + 1]);
              accK[r][4 * c4 + 2] = fmaf(sr[r], q4.z, accK[r][4 * c4 + 2]);
              accK[r][4 * c4 + 3] = fmaf(sr[r], q4.w, accK[r][4 * c4 + 3]);
            }
          }
        }
      }
    }
  }
  // keys inside Lk (zero past the batch's length)
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int j = k0 + 4 * tk + r;
    if (j >= a.Lk) continue;
    float* dkr = a.dk + b * a.ks0 + kvh * a.ks1 + static_cast<long long>(j) * a.ks2 + C::NDV * tr;
    float* dvr = a.dv + b * a.vs0 + kvh * a.vs1 + static_cast<long long>(j) * a.vs2 + C::NDV * tr;
#pragma unroll
    for (int c = 0; c < C::NDV; ++c) {
      dkr[c] = accK[r][c] * a.scale;
      dvr[c] = accV[r][c];
    }
  }
}

// Kernel B: dQ of 64 query rows (blockIdx.x) of query head blockIdx.y, batch
// blockIdx.z.
template <int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_f32_dq_kernel(const F32Args a) {
  using C = F32Cfg<D>;
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  float* sQ = sm + C::B_Q;
  float* sDO = sm + C::B_DO;
  float* sKt = sm + C::B_KT;
  float* sVt = sm + C::B_VT;
  float* sK = sm + C::B_K;
  float* sDS = sm + C::B_DS;
  float* sSt = sm + C::B_ST;
  const int q0 = blockIdx.x * kT;
  const int hq = blockIdx.y;
  const int b = blockIdx.z;
  const int kvh = hq / a.G;
  const int Lkb = a.seq_lens_kv ? min(max(a.seq_lens_kv[b], 0), a.Lk) : a.Lk;
  const int Lqb = a.seq_lens_q ? min(max(a.seq_lens_q[b], 0), a.Lq) : a.Lq;
  const int off = Lkb - Lqb;
  const int tk = threadIdx.x & 15, tr = threadIdx.x >> 4;
  // key tiles holding a key that a row of this tile sees
  int klast = Lkb - 1;
  if (a.causal) klast = min(klast, q0 + kT - 1 + off);
  const int nkt = (q0 < Lqb && klast >= 0) ? klast / kT + 1 : 0;
  float acc[4][C::NDV];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < C::NDV; ++c) acc[r][c] = 0.f;
  if (nkt > 0) {
    load_rows<D>(sQ, a.q + b * a.qs0 + hq * a.qs1, a.qs2, q0, Lqb);
    load_rows<D>(sDO, a.d_o + b * a.os0 + hq * a.os1, a.os2, q0, Lqb);
    load_stats(a, sSt, b, hq, q0, Lqb);
    for (int kt = 0; kt < nkt; ++kt) {
      const int k0 = kt * kT;
      __syncthreads();  // the previous pair's tiles are consumed
      const float* kb = a.k + b * a.ks0 + kvh * a.ks1;
      load_rows_t<D>(sKt, kb, a.ks2, k0, Lkb);
      load_rows_t<D>(sVt, a.v + b * a.vs0 + kvh * a.vs1, a.vs2, k0, Lkb);
      load_rows<D>(sK, kb, a.ks2, k0, Lkb);
      __syncthreads();
      float s[4][4], dp[4][4], p[4][4], ds[4][4];
      tile_dot<D>(sQ, sKt, tr, tk, s);
      tile_dot<D>(sDO, sVt, tr, tk, dp);
      const PairCtx x{q0, k0, Lqb, Lkb, off, hq, b};
      p_ds(a, x, tr, tk, s, dp, sSt, sSt + kT, p, ds);
#pragma unroll
      for (int r = 0; r < 4; ++r)
        *reinterpret_cast<float4*>(sDS + (4 * tr + r) * kPadT + 4 * tk) =
            make_float4(ds[r][0], ds[r][1], ds[r][2], ds[r][3]);
      __syncthreads();
      // dQ[row][d] += dS[row][key] K[key][d] (thread: rows 4 tr + r, head
      // dimensions NDV tk + c)
#pragma unroll 4
      for (int key = 0; key < kT; ++key) {
        float dsr[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) dsr[r] = sDS[(4 * tr + r) * kPadT + key];
#pragma unroll
        for (int c4 = 0; c4 < C::NDV / 4; ++c4) {
          const float4 k4 =
              *reinterpret_cast<const float4*>(sK + key * C::PQ + C::NDV * tk + 4 * c4);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            acc[r][4 * c4 + 0] = fmaf(dsr[r], k4.x, acc[r][4 * c4 + 0]);
            acc[r][4 * c4 + 1] = fmaf(dsr[r], k4.y, acc[r][4 * c4 + 1]);
            acc[r][4 * c4 + 2] = fmaf(dsr[r], k4.z, acc[r][4 * c4 + 2]);
            acc[r][4 * c4 + 3] = fmaf(dsr[r], k4.w, acc[r][4 * c4 + 3]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = q0 + 4 * tr + r;
    if (i >= a.Lq) continue;
    float* dqr = a.dq + b * a.qs0 + hq * a.qs1 + static_cast<long long>(i) * a.qs2 + C::NDV * tk;
#pragma unroll
    for (int c = 0; c < C::NDV; ++c) dqr[c] = acc[r][c] * a.scale;
  }
}

template <int D>
sdpa_status_t launch_f32_impl(const sdpa_params_t& p, const F32Args& a, cudaStream_t stream,
                              int* launched) {
  using C = F32Cfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(bwd_f32_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::A_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_f32_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::B_BYTES) != cudaSuccess)
      return SDPA_ERR_CUDA;
    attr_set = true;
  }
  if (p.num_q_heads > 65535 || p.batch > 65535) return SDPA_ERR_UNSUPPORTED;
  *launched = 0;
  if (p.seq_len_kv > 0) {  // dK and dV (zero where no query row takes part)
    const dim3 ga((p.seq_len_kv + kT - 1) / kT, p.num_kv_heads, p.batch);
    bwd_f32_dkdv_kernel<D><<<ga, kThreads, C::A_BYTES, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SDPA_ERR_CUDA;
    ++*launched;
  }
  if (p.seq_len_q > 0) {  // dQ (zero where a row sees no key)
    const dim3 gb((p.seq_len_q + kT - 1) / kT, p.num_q_heads, p.batch);
    bwd_f32_dq_kernel<D><<<gb, kThreads, C::B_BYTES, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SDPA_ERR_CUDA;
    ++*launched;
  }
  return SDPA_OK;
}

}  // namespace

// fp32 backward: the pre pass (LSE in log2 units and D_i into the
// workspace), then kernels A and B.  Expects the normalised parameters.
sdpa_status_t launch_backward_f32(const sdpa_params_t& p, const void* q, const void* k,
                                  const void* v, const void* o, const void* d_o,
                                  const float* lse, void* dq, void* dk, void* dv,
                                  void* workspace, const LaunchEnv& env) {
  const long long rows = static_cast<long long>(p.batch) * p.num_q_heads * p.seq_len_q;
  float* lse2 = nullptr;
  float* dvec = nullptr;
  backward_stats_slots(p, workspace, &lse2, &dvec);
  int launched = 0;
  if (rows > 0) {
    const sdpa_status_t st = launch_backward_pre(p, o, d_o, lse, lse2, dvec, nullptr, env.stream);
    if (st != SDPA_OK) return st;
    ++launched;
  }
  F32Args a;
  a.q = static_cast<const float*>(q);
  a.k = static_cast<const float*>(k);
  a.v = static_cast<const float*>(v);
  a.d_o = static_cast<const float*>(d_o);
  a.lse2 = lse2;
  a.dvec = dvec;
  a.dq = static_cast<float*>(dq);
  a.dk = static_cast<float*>(dk);
  a.dv = static_cast<float*>(dv);
  a.qs0 = p.q_stride[0];
  a.qs1 = p.q_stride[1];
  a.qs2 = p.q_stride[2];
  a.ks0 = p.k_stride[0];
  a.ks1 = p.k_stride[1];
  a.ks2 = p.k_stride[2];
  a.vs0 = p.v_stride[0];
  a.vs1 = p.v_stride[1];
  a.vs2 = p.v_stride[2];
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
  a.Hq = p.num_q_heads;
  a.Hkv = p.num_kv_heads;
  a.G = p.num_q_heads / p.num_kv_heads;
  a.Lq = p.seq_len_q;
  a.Lk = p.seq_len_kv;
  a.causal = p.causal ? 1 : 0;
  a.sl2 = p.scale * 1.4426950408889634f;
  a.scale = p.scale;
  int n = 0;
  sdpa_status_t st = SDPA_ERR_UNSUPPORTED;
  if (p.head_dim == 64) st = launch_f32_impl<64>(p, a, env.stream, &n);
  if (p.head_dim == 128) st = launch_f32_impl<128>(p, a, env.stream, &n);
  if (st != SDPA_OK) return st;
  launched += n;
  set_last_launches(launched);
  return SDPA_OK;
}

}  // namespace gb300
