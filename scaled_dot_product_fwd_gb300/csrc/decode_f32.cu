// decode_f32.cu — instantiations of the split-KV decode pass for float inputs.
#include "decode.cuh"

namespace gb300 {
namespace dec {

sdpa_status_t launch_split_f32(const SplitArgs& a, int D, int hg, int batch, cudaStream_t s,
                              bool* merged) {
  return launch_split_t<float>(a, D, hg, batch, s, merged);
}

}  // namespace dec
}  // namespace gb300
