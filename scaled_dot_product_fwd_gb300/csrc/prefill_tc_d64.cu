// prefill_tc_d64.cu — head_dim 64 instantiations of the tensor-core prefill
// (fp16, bf16; dense or extended inputs; whole and split units).
#include "prefill_tc.cuh"

namespace gb300 {

sdpa_status_t launch_prefill_tc_d64(const sdpa_params_t& p, const void* q, const void* k,
                                    const void* v, void* o, float* lse, const LaunchEnv& env,
                                    int* grids) {
  const bool bf16 = p.dtype == SDPA_BF16;
  QkvStrides st;
  for (int i = 0; i < 3; ++i) {
    st.q[i] = p.q_stride[i];
    st.k[i] = p.k_stride[i];
    st.v[i] = p.v_stride[i];
  }
  if (prefill_needs_ext(p) || env.mask_tiles)
    return bf16 ? launch_impl<64, true, false, true>(p, q, k, v, q, k, v, o, lse, st, env, grids)
                : launch_impl<64, false, false, true>(p, q, k, v, q, k, v, o, lse, st, env, grids);
  return bf16 ? launch_impl<64, true, false, false>(p, q, k, v, q, k, v, o, lse, st, env, grids)
              : launch_impl<64, false, false, false>(p, q, k, v, q, k, v, o, lse, st, env, grids);
}

}  // namespace gb300
