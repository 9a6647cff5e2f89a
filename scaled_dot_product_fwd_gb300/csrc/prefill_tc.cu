// prefill_tc.cu — entry of the tensor-core prefill: dispatch by head size,
// and fp32 inputs at head_dim 64 as bf16 hi/lo parts (x = hi + lo +
// O(2^-16 |x|)) with three products per MMA step.
#include "prefill_tc.cuh"

namespace gb300 {
namespace {

// Split of fp32 inputs into bf16 hi and lo parts (x = hi + lo + O(2^-16 |x|)),
// for up to three tensors in one launch.  Tensor s is [B, H[s], L[s], D]
// with element strides sb, sh, sl (D contiguous) in the input; its compact
// output has n4[s] float4 groups, rows of D/4 = 1 << d4_shift groups.
struct SplitJob {
  const float* x[3];
  __nv_bfloat16* hi[3];
  __nv_bfloat16* lo[3];
  size_t n4[3];
  uint32_t H[3], L[3];
  int64_t sb[3], sh[3], sl[3];
  int d4_shift;
};

__global__ void __launch_bounds__(256) split_bf16_kernel(const SplitJob job) {
  const uint32_t d4_mask = (1u << job.d4_shift) - 1u;
  for (int s = 0; s < 3; ++s) {
    const float* x = job.x[s];
    uint2* hi = reinterpret_cast<uint2*>(job.hi[s]);
    uint2* lo = reinterpret_cast<uint2*>(job.lo[s]);
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < job.n4[s];
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
      // compact row (b, h, l) and float4 column; rows fit 32 bits (host check)
      const uint32_t row = static_cast<uint32_t>(i >> job.d4_shift);
      const uint32_t bh = row / job.L[s];
      const uint32_t l = row - bh * job.L[s];
      const uint32_t b = bh / job.H[s];
      const uint32_t h = bh - b * job.H[s];
      const float4 v = *reinterpret_cast<const float4*>(
          x + b * job.sb[s] + h * job.sh[s] + l * job.sl[s] + 4 * (i & d4_mask));
      const uint32_t h01 = Elem<true>::pack(v.x, v.y);
      const uint32_t h23 = Elem<true>::pack(v.z, v.w);
      const uint32_t l01 = Elem<true>::pack(v.x - __uint_as_float(h01 << 16),
                                            v.y - __uint_as_float(h01 & 0xffff0000u));
      const uint32_t l23 = Elem<true>::pack(v.z - __uint_as_float(h23 << 16),
                                            v.w - __uint_as_float(h23 & 0xffff0000u));
      hi[i] = make_uint2(h01, h23);
      lo[i] = make_uint2(l01, l23);
    }
  }
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

sdpa_status_t launch_prefill_tc(const sdpa_params_t& p, const void* q, const void* k,
                                const void* v, void* o, float* lse, const LaunchEnv& env) {
  int g = 0;
  sdpa_status_t st = SDPA_ERR_UNSUPPORTED;
  if (p.head_dim == 64) st = launch_prefill_tc_d64(p, q, k, v, o, lse, env, &g);
  if (p.head_dim == 128) st = launch_prefill_tc_d128(p, q, k, v, o, lse, env, &g);
  if (p.head_dim == 512) st = launch_prefill_tc_d512(p, q, k, v, o, lse, env, &g);
  if (st == SDPA_OK) set_last_launches(g);
  return st;
}

size_t prefill_x3_workspace(const sdpa_params_t& p) {
  const size_t nq = static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q * p.head_dim;
  const size_t nk = static_cast<size_t>(p.batch) * p.num_kv_heads * p.seq_len_kv * p.head_dim;
  return 2 * align256(nq * 2) + 4 * align256(nk * 2);
}

sdpa_status_t launch_prefill_x3(const sdpa_params_t& p, const void* q, const void* k,
                                const void* v, void* o, float* lse, void* workspace,
                                const LaunchEnv& env) {
  if (p.head_dim != 64) return SDPA_ERR_UNSUPPORTED;
  const size_t nq = static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q * p.head_dim;
  // compact hi/lo copies of the used rows [0, seq_len_kv) of k and v
  const size_t nk = static_cast<size_t>(p.batch) * p.num_kv_heads * p.seq_len_kv * p.head_dim;
  // compact rows are counted in 32 bits
  const size_t rows = static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q;
  if (rows > 0xffffffffull || nk / p.head_dim > 0xffffffffull) return SDPA_ERR_UNSUPPORTED;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* qh = reinterpret_cast<__nv_bfloat16*>(w);
  __nv_bfloat16* ql = reinterpret_cast<__nv_bfloat16*>(w + align256(nq * 2));
  __nv_bfloat16* kh = reinterpret_cast<__nv_bfloat16*>(w + 2 * align256(nq * 2));
  __nv_bfloat16* kl = reinterpret_cast<__nv_bfloat16*>(w + 2 * align256(nq * 2) + align256(nk * 2));
  __nv_bfloat16* vh =
      reinterpret_cast<__nv_bfloat16*>(w + 2 * align256(nq * 2) + 2 * align256(nk * 2));
  __nv_bfloat16* vl =
      reinterpret_cast<__nv_bfloat16*>(w + 2 * align256(nq * 2) + 3 * align256(nk * 2));
  SplitJob job;
  job.x[0] = static_cast<const float*>(q);
  job.x[1] = static_cast<const float*>(k);
  job.x[2] = static_cast<const float*>(v);
  job.hi[0] = qh;
  job.lo[0] = ql;
  job.hi[1] = kh;
  job.lo[1] = kl;
  job.hi[2] = vh;
  job.lo[2] = vl;
  job.n4[0] = nq / 4;
  job.n4[1] = nk / 4;
  job.n4[2] = nk / 4;
  job.H[0] = p.num_q_heads;
  job.L[0] = p.seq_len_q;
  job.H[1] = job.H[2] = p.num_kv_heads;
  job.L[1] = job.L[2] = p.seq_len_kv > 0 ? p.seq_len_kv : 1;  // no keys: nothing to split
  const int64_t* xs[3] = {p.q_stride, p.k_stride, p.v_stride};
  for (int t = 0; t < 3; ++t) {
    job.sb[t] = xs[t][0];
    job.sh[t] = xs[t][1];
    job.sl[t] = xs[t][2];
  }
  job.d4_shift = p.head_dim == 64 ? 4 : 5;
  split_bf16_kernel<<<env.num_sms * 8, 256, 0, env.stream>>>(job);
  if (cudaGetLastError() != cudaSuccess) return SDPA_ERR_CUDA;
  // the copies are dense [B, H, L, D]
  QkvStrides st;
  const int64_t D = p.head_dim;
  st.q[2] = st.k[2] = st.v[2] = D;
  st.q[1] = p.seq_len_q * D;
  st.q[0] = p.num_q_heads * st.q[1];
  st.k[1] = st.v[1] = p.seq_len_kv * D;
  st.k[0] = st.v[0] = p.num_kv_heads * st.k[1];
  int g = 0;
  const sdpa_status_t rs =
      prefill_needs_ext(p)
          ? launch_impl<64, true, true, true>(p, qh, kh, vh, ql, kl, vl, o, lse, st, env, &g)
          : launch_impl<64, true, true, false>(p, qh, kh, vh, ql, kl, vl, o, lse, st, env, &g);
  if (rs == SDPA_OK) set_last_launches(1 + g);  // the hi/lo split, then the prefill grids
  return rs;
}

}  // namespace gb300
