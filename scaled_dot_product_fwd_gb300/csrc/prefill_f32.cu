// prefill_f32.cu — fused attention forward for fp32 inputs, head_dim 64/128,
// on the fp32 FMA pipes (full fp32 products and sums: the MLX D512 page runs
// its checks with TF32 disabled, so the fp32 path may not drop to TF32).
//
// Same computation as the tensor-core kernel: the tiled online softmax of
// the rustytorch flash_attention.metal forward kernel with causal block
// skipping, bounds masking of the ragged key tail, additive mask, sinks in
// the denominator and grouped-query head mapping.
//
// Layout: a CTA of 256 threads owns 64 query rows of one (batch, head) and
// walks 64-key tiles.  Thread (ty = tid / 16, tx = tid % 16) owns query rows
// 4*ty .. 4*ty+3; for S it owns keys tx + 16*c (c < 4), for O the columns
// 4*tx + 64*c.  The 16 threads of a row group share the row statistics
// through xor-shuffles inside their half-warp.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gb300 {
namespace {

constexpr int FBM = 64;
constexpr int FBN = 64;
constexpr int kF32Threads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct F32Args {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  int Hq, Hkv, G, Lq, Lk, num_qblocks;
  float sl2;
  int causal;
  const float* mask;
  long long ms0, ms1, ms2;
  const float* sinks;
  int mask_bool;           // mask holds bytes, nonzero = visible
  // element strides (batch, head, row) of q, k, v and o; D is contiguous
  long long qs0, qs1, qs2, ks0, ks1, ks2, vs0, vs1, vs2, os0, os1, os2;
  const int* seq_lens_q;   // nullptr or per-batch valid query rows
  const int* seq_lens_kv;  // nullptr or per-batch valid keys
};

template <int D>
struct F32Cfg {
  static constexpr int KP = D + 4;    // padded K row (floats)
  static constexpr int PP = FBN + 4;  // padded P row
  static constexpr int SQ = FBM * D;
  static constexpr int SK = FBN * KP;
  static constexpr int SV = FBN * D;
  static constexpr int SP = FBM * PP;
  static constexpr int SMEM = (SQ + SK + SV + SP) * 4;
};

template <int D>
__global__ void __launch_bounds__(kF32Threads) prefill_f32_kernel(const F32Args a) {
  using C = F32Cfg<D>;
  extern __shared__ float4 smem4[];
  float* sQ = reinterpret_cast<float*>(smem4);
  float* sK = sQ + C::SQ;
  float* sV = sK + C::SK;
  float* sP = sV + C::SV;

  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int qb = a.causal ? (a.num_qblocks - 1 - static_cast<int>(blockIdx.x))
                          : static_cast<int>(blockIdx.x);
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / a.G;
  const int q0 = qb * FBM;
  const float* qbase = a.q + b * a.qs0 + h * a.qs1;
  const float* kbase = a.k + b * a.ks0 + kvh * a.ks1;
  const float* vbase = a.v + b * a.vs0 + kvh * a.vs1;
  // this batch's lengths (padding masks), clamped to the call's maxima
  const int Lkb = a.seq_lens_kv ? min(max(a.seq_lens_kv[b], 0), a.Lk) : a.Lk;
  const int Lqb = a.seq_lens_q ? min(max(a.seq_lens_q[b], 0), a.Lq) : a.Lq;

  // Q tile (rows beyond Lq read as zero)
  for (int e = tid; e < FBM * D / 4; e += kF32Threads) {
    const int r = e / (D / 4), c4 = e % (D / 4);
    float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q0 + r < a.Lq) val = reinterpret_cast<const float4*>(qbase + (q0 + r) * a.qs2)[c4];
    reinterpret_cast<float4*>(sQ + r * D)[c4] = val;
  }

  int qrow[4], limit[4];
  const float* mrow[4];     // additive mask rows
  const uint8_t* mrowb[4];  // boolean mask rows
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    qrow[i] = q0 + ty * 4 + i;
    limit[i] = Lkb - 1;
    if (a.causal) limit[i] = min(limit[i], qrow[i] + (Lkb - Lqb));
    if (qrow[i] >= Lqb) limit[i] = -1;  // a padding row sees no key
    const long long moff = b * a.ms0 + h * a.ms1 + qrow[i] * a.ms2;
    const bool has = a.mask && qrow[i] < a.Lq;
    mrow[i] = (has && !a.mask_bool) ? a.mask + moff : nullptr;
    mrowb[i] =
        (has && a.mask_bool) ? reinterpret_cast<const uint8_t*>(a.mask) + moff : nullptr;
  }
  // keys needed by the block: up to the last visible key of its last row
  int kend = q0 < Lqb ? Lkb : 0;
  if (a.causal) kend = min(kend, min(q0 + FBM, Lqb) - 1 + (Lkb - Lqb) + 1);
  const int ntiles = kend > 0 ? (kend + FBN - 1) / FBN : 0;

  constexpr int OC = D / 64;  // float4 column groups per thread in O
  float acc[4][OC][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < OC; ++c)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][c][e] = 0.f;
  float m[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
  }

  for (int jt = 0; jt < ntiles; ++jt) {
    const int k0 = jt * FBN;
    __syncthreads();  // previous tile's K, V, P are no longer read
    for (int e = tid; e < FBN * D / 4; e += kF32Threads) {
      const int r = e / (D / 4), c4 = e % (D / 4);
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
      if (k0 + r < Lkb) {  // keys past the batch's length are never read
        kv = reinterpret_cast<const float4*>(kbase + (k0 + r) * a.ks2)[c4];
        vv = reinterpret_cast<const float4*>(vbase + (k0 + r) * a.vs2)[c4];
      }
      reinterpret_cast<float4*>(sK + r * C::KP)[c4] = kv;
      reinterpret_cast<float4*>(sV + r * D)[c4] = vv;
    }
    __syncthreads();

    // S micro-tile: rows 4*ty+i, keys tx + 16*c
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[i][c] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; d += 4) {
      float4 qv[4], kv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) qv[i] = *reinterpret_cast<const float4*>(sQ + (ty * 4 + i) * D + d);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        kv[c] = *reinterpret_cast<const float4*>(sK + (tx + 16 * c) * C::KP + d);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          s[i][c] = fmaf(qv[i].x, kv[c].x, s[i][c]);
          s[i][c] = fmaf(qv[i].y, kv[c].y, s[i][c]);
          s[i][c] = fmaf(qv[i].z, kv[c].z, s[i][c]);
          s[i][c] = fmaf(qv[i].w, kv[c].w, s[i][c]);
        }
    }

    float alpha[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float x[4];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int kj = k0 + tx + 16 * c;
        float xv = s[i][c] * a.sl2;
        if (mrow[i] && kj <= limit[i]) xv += mask_log2(mrow[i][kj], mask_huge_log2(a.sl2));
        if (mrowb[i] && kj <= limit[i] && !mrowb[i][kj]) xv = -INFINITY;
        if (kj > limit[i]) xv = -INFINITY;
        x[c] = xv;
        mx = fmaxf(mx, xv);
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[i], mx);
      const float mu = (mn == -INFINITY) ? 0.f : mn;
      alpha[i] = ex2(m[i] - mu);  // 0 when m was -inf
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float p = ex2(x[c] - mu);
        rs += p;
        sP[(ty * 4 + i) * C::PP + tx + 16 * c] = p;
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
      l[i] = l[i] * alpha[i] + rs;
      m[i] = mn;
    }
    __syncthreads();

    // O = O * alpha + P V
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < OC; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][c][e] *= alpha[i];
#pragma unroll 4
    for (int kk = 0; kk < FBN; ++kk) {
      float p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = sP[(ty * 4 + i) * C::PP + kk];
#pragma unroll
      for (int c = 0; c < OC; ++c) {
        const float4 vv = *reinterpret_cast<const float4*>(sV + kk * D + 4 * tx + 64 * c);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i][c][0] = fmaf(p[i], vv.x, acc[i][c][0]);
          acc[i][c][1] = fmaf(p[i], vv.y, acc[i][c][1]);
          acc[i][c][2] = fmaf(p[i], vv.z, acc[i][c][2]);
          acc[i][c][3] = fmaf(p[i], vv.w, acc[i][c][3]);
        }
      }
    }
  }

  // epilogue: sinks, normalisation, LSE
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int qi = qrow[i];
    float mi = m[i], li = l[i], oscale = 1.f;
    if (a.sinks) {
      const float sk = a.sinks[h] * kLog2e;
      const float mn = fmaxf(mi, sk);
      oscale = ex2(mi - mn);
      li = li * oscale + ex2(sk - mn);
      mi = mn;
    }
    const float inv = (li > 0.f) ? oscale / li : 0.f;
    if (qi < a.Lq) {
      float* orow = a.o + b * a.os0 + h * a.os1 + qi * a.os2;
#pragma unroll
      for (int c = 0; c < OC; ++c) {
        float4 w;
        w.x = (inv == 0.f) ? 0.f : acc[i][c][0] * inv;
        w.y = (inv == 0.f) ? 0.f : acc[i][c][1] * inv;
        w.z = (inv == 0.f) ? 0.f : acc[i][c][2] * inv;
        w.w = (inv == 0.f) ? 0.f : acc[i][c][3] * inv;
        *reinterpret_cast<float4*>(orow + 4 * tx + 64 * c) = w;
      }
      if (a.lse && tx == 0)
        a.lse[(static_cast<size_t>(b) * a.Hq + h) * a.Lq + qi] =
            (li > 0.f) ? (mi + __log2f(li)) * kLn2 : -INFINITY;
    }
  }
}

template <int D>
sdpa_status_t launch_f32_impl(const sdpa_params_t& p, const void* q, const void* k, const void* v,
                              void* o, float* lse, const LaunchEnv& env) {
  F32Args a;
  a.q = static_cast<const float*>(q);
  a.k = static_cast<const float*>(k);
  a.v = static_cast<const float*>(v);
  a.o = static_cast<float*>(o);
  a.lse = lse;
  a.Hq = p.num_q_heads;
  a.Hkv = p.num_kv_heads;
  a.G = p.num_q_heads / p.num_kv_heads;
  a.Lq = p.seq_len_q;
  a.Lk = p.seq_len_kv;
  a.num_qblocks = (p.seq_len_q + FBM - 1) / FBM;
  a.sl2 = p.scale * kLog2e;
  a.causal = p.causal ? 1 : 0;
  a.mask = static_cast<const float*>(p.mask);
  a.ms0 = p.mask_stride[0];
  a.ms1 = p.mask_stride[1];
  a.ms2 = p.mask_stride[2];
  a.sinks = p.sinks;
  a.mask_bool = (p.flags & SDPA_FLAG_BOOL_MASK) ? 1 : 0;
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
  a.seq_lens_q = p.seq_lens_q;
  a.seq_lens_kv = p.seq_lens_kv;
  auto kern = prefill_f32_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           F32Cfg<D>::SMEM) != cudaSuccess)
    return SDPA_ERR_CUDA;
  dim3 grid(a.num_qblocks, p.num_q_heads, p.batch);
  kern<<<grid, kF32Threads, F32Cfg<D>::SMEM, env.stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // namespace

sdpa_status_t launch_prefill_f32(const sdpa_params_t& p, const void* q, const void* k,
                                 const void* v, void* o, float* lse, const LaunchEnv& env) {
  if (p.head_dim == 64) return launch_f32_impl<64>(p, q, k, v, o, lse, env);
  if (p.head_dim == 128) return launch_f32_impl<128>(p, q, k, v, o, lse, env);
  return SDPA_ERR_UNSUPPORTED;
}

}  // namespace gb300
