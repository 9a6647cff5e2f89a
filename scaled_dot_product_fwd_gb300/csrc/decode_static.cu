// decode_static.cu — allocation-free variant of the vector (Lq <= 8)
// split-KV decode: sdpa_forward_decode_noalloc.
//
// Who needs it: callers that cannot call cudaMalloc (or hand the library a
// workspace) at the point where they run attention.  cudaMalloc is not
// allowed while a stream is being captured into a CUDA graph, it can
// synchronise the device, and some hosts (plugins inside another runtime,
// allocator-free serving loops, code that owns every device byte through
// its own pool) have no way to give this library device memory.  This entry
// point needs only the inputs and the outputs.
//
// How: the split-KV partial results (the workspace of sdpa_forward) live in
// one file-scope device array, kStaticScratchBytes long.  Every GPU that
// loads the library holds that array until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on a
// device (with that device current) looks its address up with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture.  All calls on a device share the one array and it keeps the last
// call's contents: calls whose kernels overlap on the GPU (different streams
// without ordering) race on it and must be serialised by the caller.  The
// partial results are fully written by the first kernel before the combine
// kernel reads them, so nothing in the array has to start at zero.
//
// Nothing here allocates: no cudaMalloc, cudaFree or allocating library
// routine is called; a problem whose partial results exceed the array is
// rejected with SDPA_ERR_WORKSPACE_TOO_SMALL before any launch.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "sdpa.h"

namespace {

constexpr size_t kStaticScratchBytes = SDPA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
int g_scratch_sms[kMaxDevices] = {};

// Once per device, with that device current: the device address of the
// scratch array and the SM count.
sdpa_status_t setup_device(void** scratch, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDPA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr)
      return SDPA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SDPA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
    g_scratch_sms[dev] = sms;
  }
  *scratch = g_scratch_ptr[dev];
  *num_sms = g_scratch_sms[dev];
  return SDPA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" sdpa_status_t sdpa_forward_decode_noalloc(const sdpa_params_t* p, const void* q,
                                                     const void* k, const void* v, void* o,
                                                     float* lse, void* stream) {
  gb300::set_last_launches(0);
  sdpa_status_t st = SDPA_OK;
  const sdpa_kernel_t kern = sdpa_select_kernel(p, &st);
  if (st != SDPA_OK) return st;
  if (kern == SDPA_KERNEL_NONE) return SDPA_OK;  // nothing to compute
  if (kern != SDPA_KERNEL_DECODE_SPLITKV) return SDPA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o) return SDPA_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return SDPA_ERR_MISALIGNED;
  if (p->mask && !aligned(p->mask, 16)) return SDPA_ERR_MISALIGNED;
  if (lse && !aligned(lse, 4)) return SDPA_ERR_MISALIGNED;
  if (p->sinks && !aligned(p->sinks, 4)) return SDPA_ERR_MISALIGNED;
  if ((p->seq_lens_q && !aligned(p->seq_lens_q, 4)) ||
      (p->seq_lens_kv && !aligned(p->seq_lens_kv, 4)))
    return SDPA_ERR_MISALIGNED;
  void* scratch = nullptr;
  int num_sms = 0;
  st = setup_device(&scratch, &num_sms);
  if (st != SDPA_OK) return st;
  gb300::DecodePlan plan;
  if (!gb300::decode_plan(*p, num_sms, &plan)) return SDPA_ERR_UNSUPPORTED;
  if (plan.workspace > kStaticScratchBytes) return SDPA_ERR_WORKSPACE_TOO_SMALL;
  gb300::LaunchEnv env;
  env.status = gb300::status_word_current_device();
  if (!env.status) return SDPA_ERR_CUDA;
  env.wait_limit_ns = gb300::current_wait_limit_ns();
  env.num_sms = num_sms;
  env.stream = static_cast<cudaStream_t>(stream);
  return gb300::launch_decode(gb300::normalized_params(*p), plan, q, k, v, o, lse, scratch, env);
}
