// prefill_tc_d64.cu — head_dim 64 instantiations of the tensor-core prefill
// (fp16, bf16; dense or per-batch lengths; whole and split units).
#include "prefill_tc.cuh"

namespace gb300 {

sdpa_status_t launch_prefill_tc_d64(const sdpa_params_t& p, const void* q, const void* k,
                                    const void* v, void* o, float* lse, uint64_t kv_plane_rows,
                                    const LaunchEnv& env, int* grids) {
  const bool bf16 = p.dtype == SDPA_BF16;
  const uint64_t cap = kv_plane_rows;
  if (p.seq_lens_q || p.seq_lens_kv)
    return bf16 ? launch_impl<64, true, false, true>(p, q, k, v, q, k, v, o, lse, cap, env, grids)
                : launch_impl<64, false, false, true>(p, q, k, v, q, k, v, o, lse, cap, env, grids);
  return bf16 ? launch_impl<64, true, false, false>(p, q, k, v, q, k, v, o, lse, cap, env, grids)
              : launch_impl<64, false, false, false>(p, q, k, v, q, k, v, o, lse, cap, env, grids);
}

}  // namespace gb300
