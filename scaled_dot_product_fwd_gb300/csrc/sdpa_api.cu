// sdpa_api.cu — the C ABI declared in include/sdpa.h: argument validation,
// kernel selection by shape, workspace sizing, error mapping and the device
// status word.
//
// Selection follows the dispatch role of mlx 0.30.7
// scaled_dot_product_attention.cpp (ScaledDotProductAttention::eval_gpu
// chooses between a fused graph and the sdpa_vector kernel) without any
// fallback: a single query row (Lq = 1), or a few (the rows of a kv head then
// share its K/V stream: up to 2 at D = 64/128, where the tensor-core tiles
// are ahead from 4 rows on, measured on GB300; up to 8 at D = 512), takes the
// split-KV vector path of MLX PR #4459, every other shape takes the fused
// prefill kernel for its dtype (fp32 at D = 512: the vector path with its
// rows grouped, fp32 products and sums), and anything else is reported as
// unsupported (the force_fused admission check of the same PR raises instead
// of falling back).
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "sdpa.h"

namespace {

__device__ int g_status_word;

constexpr int kMaxDevices = 64;
constexpr int kMaxDecodeRows = 8;     // query rows per head of the vector path, D = 512
constexpr int kMaxDecodeRowsTc = 2;   // the same where a tensor-core prefill exists
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
// test hooks (sdpa_debug_set_option), indexed by sdpa_debug_option_t
constexpr int kDebugOptions = 5;
std::atomic<int> g_debug[kDebugOptions] = {{0}, {1}, {0}, {-1}, {0}};
thread_local int g_last_launches = 0;
std::mutex g_dev_mutex;
int* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Host-only checks of the problem description (no CUDA call).
sdpa_status_t validate_problem(const sdpa_params_t* p) {
  if (!p) return SDPA_ERR_INVALID_ARGUMENT;
  if (p->batch < 0 || p->num_q_heads < 0 || p->num_kv_heads < 1 || p->seq_len_q < 0 ||
      p->seq_len_kv < 0 || p->head_dim < 1)
    return SDPA_ERR_INVALID_ARGUMENT;
  if (p->num_q_heads % p->num_kv_heads != 0) return SDPA_ERR_INVALID_ARGUMENT;
  if (p->dtype != SDPA_F32 && p->dtype != SDPA_F16 && p->dtype != SDPA_BF16)
    return SDPA_ERR_INVALID_ARGUMENT;
  if (!isfinite(p->scale)) return SDPA_ERR_INVALID_ARGUMENT;
  if (p->seq_len_q > (1 << 30) || p->seq_len_kv > (1 << 30)) return SDPA_ERR_UNSUPPORTED;
  if (p->mask) {
    for (int i = 0; i < 4; ++i)
      if (p->mask_stride[i] < 0) return SDPA_ERR_INVALID_ARGUMENT;
    if (p->mask_stride[3] != 1) return SDPA_ERR_INVALID_ARGUMENT;
  }
  if ((p->flags & ~(SDPA_FLAG_SHARED_GPU | SDPA_FLAG_BOOL_MASK | SDPA_FLAG_STRIDES)) != 0)
    return SDPA_ERR_INVALID_ARGUMENT;
  if (p->kv_capacity < 0 || (p->kv_capacity > 0 && p->kv_capacity < p->seq_len_kv))
    return SDPA_ERR_INVALID_ARGUMENT;
  if (p->flags & SDPA_FLAG_STRIDES) {
    // explicit layouts replace kv_capacity; rows of every tensor 16-byte aligned
    if (p->kv_capacity != 0) return SDPA_ERR_INVALID_ARGUMENT;
    const int64_t es = p->dtype == SDPA_F32 ? 4 : 2;
    const int64_t* st[4] = {p->q_stride, p->k_stride, p->v_stride, p->o_stride};
    for (const int64_t* s : st)
      for (int i = 0; i < 3; ++i) {
        if (s[i] < 0) return SDPA_ERR_INVALID_ARGUMENT;
        if ((s[i] * es) % 16 != 0) return SDPA_ERR_MISALIGNED;
      }
  }
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 512) return SDPA_ERR_UNSUPPORTED;
  // cuDNN's bottom-right causal mask is undefined for Tq > Tkv (mlx 0.30.7
  // supports_sdpa_cudnn); the same rule holds here.
  if (p->causal && p->seq_len_q > p->seq_len_kv) return SDPA_ERR_UNSUPPORTED;
  // fp32 at head_dim 512 with many rows runs on the vector path, whose grid
  // holds (kv head, group of 4 rows) pairs in its y dimension (<= 65535)
  if (p->dtype == SDPA_F32 && p->head_dim == 512 && p->seq_len_q > kMaxDecodeRows &&
      p->num_kv_heads > 0) {
    const int64_t rows = static_cast<int64_t>(p->num_q_heads / p->num_kv_heads) * p->seq_len_q;
    if (static_cast<int64_t>(p->num_kv_heads) * ((rows + 3) / 4) > 65535)
      return SDPA_ERR_UNSUPPORTED;
  }
  return SDPA_OK;
}

// Bytes of one mask element: 1 for a boolean mask, else the dtype's size.
size_t mask_elem_size(const sdpa_params_t& p) {
  if (p.flags & SDPA_FLAG_BOOL_MASK) return 1;
  return p.dtype == SDPA_F32 ? 4 : 2;
}

// The dense layout (and kv_capacity) written out as strides, so that every
// launcher reads the layout from the stride fields.  Reads the caller's
// stride fields only when it set SDPA_FLAG_STRIDES (a caller built against
// an earlier ABI has no such fields).
sdpa_params_t normalized(const sdpa_params_t* p) {
  sdpa_params_t n;
  if (p->flags & SDPA_FLAG_STRIDES) return *p;
  memset(&n, 0, sizeof(n));
  memcpy(&n, p, offsetof(sdpa_params_t, q_stride));
  const int64_t D = p->head_dim;
  const int64_t cap = p->kv_capacity > 0 ? p->kv_capacity : p->seq_len_kv;
  const int64_t qs[3] = {static_cast<int64_t>(p->num_q_heads) * p->seq_len_q * D,
                         static_cast<int64_t>(p->seq_len_q) * D, D};
  const int64_t ks[3] = {static_cast<int64_t>(p->num_kv_heads) * cap * D, cap * D, D};
  for (int i = 0; i < 3; ++i) {
    n.q_stride[i] = n.o_stride[i] = qs[i];
    n.k_stride[i] = n.v_stride[i] = ks[i];
  }
  n.kv_capacity = 0;
  n.flags |= SDPA_FLAG_STRIDES;
  return n;
}

bool nothing_to_do(const sdpa_params_t* p) {
  return static_cast<int64_t>(p->batch) * p->num_q_heads * p->seq_len_q == 0;
}

sdpa_kernel_t pick(const sdpa_params_t* p) {
  if (nothing_to_do(p)) return SDPA_KERNEL_NONE;
  if (p->seq_len_kv == 0) return SDPA_KERNEL_NO_KEYS;
  if (p->seq_len_q <= (p->head_dim == 512 ? kMaxDecodeRows : kMaxDecodeRowsTc))
    return SDPA_KERNEL_DECODE_SPLITKV;
  // fp32 at head_dim 512: the vector path for any number of rows (fp32
  // products and sums); fp16/bf16: the head-dim-512 tensor-core prefill
  if (p->dtype == SDPA_F32 && p->head_dim == 512) return SDPA_KERNEL_DECODE_SPLITKV;
  if (p->dtype == SDPA_F32)
    return p->head_dim == 64 ? SDPA_KERNEL_PREFILL_TC_F32 : SDPA_KERNEL_PREFILL_F32;
  return SDPA_KERNEL_PREFILL_TC;
}

// Per-device state: address of the status word and the SM count.
bool device_state(int* dev_out, int** status, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_dev_mutex);
  if (!g_status_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return false;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return false;
    g_status_ptr[dev] = static_cast<int*>(ptr);
    g_num_sms[dev] = sms;
  }
  if (dev_out) *dev_out = dev;
  if (status) *status = g_status_ptr[dev];
  if (num_sms) *num_sms = g_num_sms[dev];
  return true;
}

int current_num_sms() {
  int sms = 0;
  if (!device_state(nullptr, nullptr, &sms)) {
    cudaGetLastError();  // no device: plan for a full GB300
    return 152;
  }
  return sms;
}

}  // namespace

namespace gb300 {

int* status_word_current_device() {
  int* status = nullptr;
  return device_state(nullptr, &status, nullptr) ? status : nullptr;
}

uint64_t current_wait_limit_ns() { return g_wait_ns.load(); }
int debug_option(int option) {
  return (option >= 0 && option < kDebugOptions) ? g_debug[option].load() : 0;
}

void set_last_launches(int n) { g_last_launches = n; }

sdpa_params_t normalized_params(const sdpa_params_t& p) { return normalized(&p); }

}  // namespace gb300

extern "C" {

int sdpa_abi_version(void) { return SDPA_ABI_VERSION; }

const char* sdpa_status_string(sdpa_status_t s) {
  switch (s) {
    case SDPA_OK: return "ok";
    case SDPA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case SDPA_ERR_UNSUPPORTED: return "unsupported problem";
    case SDPA_ERR_MISALIGNED: return "misaligned pointer";
    case SDPA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SDPA_ERR_CUDA: return "CUDA error";
    case SDPA_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

sdpa_kernel_t sdpa_select_kernel(const sdpa_params_t* params, sdpa_status_t* status) {
  const sdpa_status_t st = validate_problem(params);
  if (status) *status = st;
  return st == SDPA_OK ? pick(params) : SDPA_KERNEL_NONE;
}

size_t sdpa_workspace_size(const sdpa_params_t* params) {
  if (validate_problem(params) != SDPA_OK) return 0;
  if (pick(params) == SDPA_KERNEL_PREFILL_TC_F32) return gb300::prefill_x3_workspace(*params);
  // a mask with a row per query: room for its score-tile copy (optional:
  // without it the prefill reads the mask where it lies)
  if (pick(params) == SDPA_KERNEL_PREFILL_TC) return gb300::prefill_mask_tiles_bytes(*params);
  if (pick(params) != SDPA_KERNEL_DECODE_SPLITKV) return 0;
  gb300::DecodePlan plan;
  if (!gb300::decode_plan(*params, current_num_sms(), &plan)) return 0;
  return plan.workspace;
}

int sdpa_last_launch_count(void) { return g_last_launches; }

uint64_t sdpa_debug_set_wait_limit_ns(uint64_t ns) {
  return g_wait_ns.exchange(ns == 0 ? kDefaultWaitNs : ns);
}

int sdpa_debug_set_option(int option, int value) {
  if (option < 0 || option >= kDebugOptions) return -1;
  return g_debug[option].exchange(value);
}

sdpa_status_t sdpa_forward(const sdpa_params_t* p, const void* q, const void* k, const void* v,
                           void* o, float* lse, void* workspace, size_t workspace_bytes,
                           void* stream) {
  g_last_launches = 0;
  sdpa_status_t st = validate_problem(p);
  if (st != SDPA_OK) return st;
  if (nothing_to_do(p)) return SDPA_OK;
  // k and v may be empty (NULL) when there are no keys
  if (!q || !o || (p->seq_len_kv > 0 && (!k || !v))) return SDPA_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return SDPA_ERR_MISALIGNED;
  // the mask is read element by element where its rows are not 16-byte
  // aligned (the kernels check each row), so its own element size will do
  if (p->mask && !aligned(p->mask, mask_elem_size(*p))) return SDPA_ERR_MISALIGNED;
  if (lse && !aligned(lse, 4)) return SDPA_ERR_MISALIGNED;
  if (p->sinks && !aligned(p->sinks, 4)) return SDPA_ERR_MISALIGNED;
  if ((p->seq_lens_q && !aligned(p->seq_lens_q, 4)) ||
      (p->seq_lens_kv && !aligned(p->seq_lens_kv, 4)))
    return SDPA_ERR_MISALIGNED;
  const sdpa_kernel_t kern = pick(p);
  // the decode workspace is checked before any launch-side CUDA call
  gb300::DecodePlan plan{};
  if (kern == SDPA_KERNEL_DECODE_SPLITKV) {
    if (!gb300::decode_plan(*p, current_num_sms(), &plan)) return SDPA_ERR_UNSUPPORTED;
    if (plan.workspace > 0) {
      if (!workspace || workspace_bytes < plan.workspace) return SDPA_ERR_WORKSPACE_TOO_SMALL;
      if (!aligned(workspace, 256)) return SDPA_ERR_MISALIGNED;
    }
  }
  if (kern == SDPA_KERNEL_PREFILL_TC_F32) {
    if (!workspace || workspace_bytes < gb300::prefill_x3_workspace(*p))
      return SDPA_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 256)) return SDPA_ERR_MISALIGNED;
  }
  int* status = nullptr;
  int num_sms = 0;
  if (!device_state(nullptr, &status, &num_sms)) return SDPA_ERR_CUDA;
  gb300::LaunchEnv env;
  env.status = status;
  env.wait_limit_ns = g_wait_ns.load();
  env.num_sms = num_sms;
  env.stream = static_cast<cudaStream_t>(stream);
  // every launcher reads the layout from the stride fields
  const sdpa_params_t n = normalized(p);
  switch (kern) {
    case SDPA_KERNEL_PREFILL_TC: {  // sets the count itself (1 or 2 grids)
      const size_t mt = gb300::prefill_mask_tiles_bytes(n);
      if (mt > 0 && workspace && workspace_bytes >= mt && aligned(workspace, 256)) {
        st = gb300::launch_mask_tiles(n, workspace, env.stream);
        if (st != SDPA_OK) return st;
        env.mask_tiles = workspace;
      }
      st = gb300::launch_prefill_tc(n, q, k, v, o, lse, env);
      if (st == SDPA_OK && env.mask_tiles) g_last_launches += 1;
      return st;
    }
    case SDPA_KERNEL_PREFILL_F32:
      st = gb300::launch_prefill_f32(n, q, k, v, o, lse, env);
      if (st == SDPA_OK) g_last_launches = 1;
      return st;
    case SDPA_KERNEL_PREFILL_TC_F32:  // hi/lo split, then the prefill grids (sets the count)
      return gb300::launch_prefill_x3(n, q, k, v, o, lse, workspace, env);
    case SDPA_KERNEL_DECODE_SPLITKV:  // sets the count itself (1 or 2 kernels)
      return gb300::launch_decode(n, plan, q, k, v, o, lse, workspace, env);
    case SDPA_KERNEL_NO_KEYS:
      st = gb300::launch_no_keys(n, o, lse, env);
      if (st == SDPA_OK) g_last_launches = 1;
      return st;
    default:
      return SDPA_ERR_UNSUPPORTED;
  }
}

// ------------------------------------------------------------------ backward
namespace {
sdpa_status_t validate_backward(const sdpa_params_t* p) {
  const sdpa_status_t st = validate_problem(p);
  if (st != SDPA_OK) return st;
  if (p->head_dim != 64 && p->head_dim != 128) return SDPA_ERR_UNSUPPORTED;
  return SDPA_OK;
}
}  // namespace

size_t sdpa_backward_workspace_size(const sdpa_params_t* params) {
  if (validate_backward(params) != SDPA_OK) return 0;
  return gb300::backward_workspace(*params);
}

sdpa_status_t sdpa_backward(const sdpa_params_t* p, const void* q, const void* k,
                            const void* v, const void* o, const void* d_o, const float* lse,
                            void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, void* stream) {
  g_last_launches = 0;
  sdpa_status_t st = validate_backward(p);
  if (st != SDPA_OK) return st;
  const bool has_q = static_cast<int64_t>(p->batch) * p->num_q_heads * p->seq_len_q > 0;
  const bool has_k = static_cast<int64_t>(p->batch) * p->num_kv_heads * p->seq_len_kv > 0;
  if (!has_q && !has_k) return SDPA_OK;
  if (has_q && (!q || !o || !d_o || !lse || !dq)) return SDPA_ERR_INVALID_ARGUMENT;
  if (has_k && (!k || !v || !dk || !dv)) return SDPA_ERR_INVALID_ARGUMENT;
  const void* p16[] = {q, k, v, o, d_o, dq, dk, dv};
  for (const void* ptr : p16)
    if (ptr && !aligned(ptr, 16)) return SDPA_ERR_MISALIGNED;
  if (p->mask && !aligned(p->mask, mask_elem_size(*p))) return SDPA_ERR_MISALIGNED;
  if (lse && !aligned(lse, 4)) return SDPA_ERR_MISALIGNED;
  const size_t need = gb300::backward_workspace(*p);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return SDPA_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 256)) return SDPA_ERR_MISALIGNED;
  }
  int* status = nullptr;
  int num_sms = 0;
  if (!device_state(nullptr, &status, &num_sms)) return SDPA_ERR_CUDA;
  gb300::LaunchEnv env;
  env.status = status;
  env.wait_limit_ns = g_wait_ns.load();
  env.num_sms = num_sms;
  env.stream = static_cast<cudaStream_t>(stream);
  // (no key: dQ = 0 from the cleared accumulator; no query: dK = dV = 0)
  return gb300::launch_backward(normalized(p), q, k, v, o, d_o, lse, dq, dk, dv, workspace, env);
}

sdpa_status_t sdpa_device_status(void* stream) {
  int* status = nullptr;
  if (!device_state(nullptr, &status, nullptr)) return SDPA_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SDPA_ERR_CUDA;
  int val = 0;
  if (cudaMemcpy(&val, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SDPA_ERR_CUDA;
  if (val != 0) {
    const int zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return SDPA_ERR_CUDA;
  }
  return val == 0 ? SDPA_OK : static_cast<sdpa_status_t>(val);
}

}  // extern "C"
