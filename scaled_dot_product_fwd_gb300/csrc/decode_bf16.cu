// decode_bf16.cu — instantiations of the split-KV decode pass for __nv_bfloat16 inputs.
#include "decode.cuh"

namespace gb300 {
namespace dec {

sdpa_status_t launch_split_bf16(const SplitArgs& a, int D, int hg, int batch, cudaStream_t s,
                              bool* merged) {
  return launch_split_t<__nv_bfloat16>(a, D, hg, batch, s, merged);
}

}  // namespace dec
}  // namespace gb300
