// internal.h — host-side interface between the C ABI (sdpa_api.cu) and the
// kernel launchers (one .cu per kernel family).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "sdpa.h"

namespace gb300 {

// What every launcher needs besides the problem: where kernels report a
// timed-out wait, the wait bound, and the device's SM count.
struct LaunchEnv {
  int* status;          // device status word
  uint64_t wait_limit_ns;
  int num_sms;
  cudaStream_t stream;
  // prefill: the mask re-laid in score tiles (mask_tiles.cu), or nullptr
  const void* mask_tiles = nullptr;
};

// Split-KV decode plan (pure function of the problem and the SM count).
struct DecodePlan {
  int head_group;   // query heads handled by one CTA (power of two)
  int num_groups;   // ceil(G / head_group)
  int tile_keys;    // keys per shared-memory tile
  int num_splits;   // key-range splits per (batch, kv head, head group)
  int split_keys;   // keys per split (multiple of tile_keys)
  int stages;       // shared-memory ring stages
  bool cluster;     // merge the splits inside a thread-block cluster when it
                    // can be resident (else the combine pass does)
  size_t workspace; // bytes of partial results (also reserved for clusters)
  bool ragged = false;  // per-batch lengths: split size derived on the device
  int slots = 0;        // CTAs resident at once (the ragged plan's wave)
  int tiles_base = 0;   // tiles per split for rows of the full length
  bool tc = false;  // head_dim 512, fp16/bf16, up to 16 rows per kv head: the
                    // tensor-core pass (head_group = rows, tile_keys = 128)
  bool tc128 = false;  // head_dim 64/128, fp16/bf16, up to 16 rows per kv
                       // head: the streaming tensor-core pass (two-pass merge)
};

bool decode_plan(const sdpa_params_t& p, int num_sms, DecodePlan* out);
// The tensor-core head_dim-512 part of the plan (false: not such a problem)
// and its launch; *merged is false when the combine pass must follow.
bool decode_tc_plan(const sdpa_params_t& p, int num_sms, DecodePlan* out);
sdpa_status_t launch_decode_tc(const sdpa_params_t& p, const DecodePlan& plan, const void* q,
                               const void* k, const void* v, void* o, float* lse, float* ws_o,
                               float* ws_ml, const LaunchEnv& env, bool* merged);
// The head_dim-64/128 tensor-core pass: its plan (false: not such a problem)
// and its launch; *merged is false when the combine pass must follow.
bool decode_tc128_plan(const sdpa_params_t& p, int num_sms, DecodePlan* out);
sdpa_status_t launch_decode_tc128(const sdpa_params_t& p, const DecodePlan& plan, const void* q,
                                  const void* k, const void* v, void* o, float* lse,
                                  float* ws_o, float* ws_ml, const LaunchEnv& env,
                                  bool* merged);

// Device status word of the current device (nullptr if there is no device)
// and the current bound on device-side waits; both owned by sdpa_api.cu.
int* status_word_current_device();
uint64_t current_wait_limit_ns();
// Current value of a test hook (sdpa_debug_set_option; sdpa_debug_option_t).
int debug_option(int option);
// Kernels enqueued by the calling thread's last call (sdpa_last_launch_count).
void set_last_launches(int n);
// The problem with SDPA_FLAG_STRIDES set and every tensor's strides filled
// in (the dense layout and kv_capacity written out when the caller gave no
// strides).  Launchers take parameters in this form.
sdpa_params_t normalized_params(const sdpa_params_t& p);

sdpa_status_t launch_prefill_tc(const sdpa_params_t& p, const void* q, const void* k,
                                const void* v, void* o, float* lse, const LaunchEnv& env);
// fp32 inputs, D = 64: split into bf16 hi/lo parts in the workspace, then the
// tensor-core kernel with three products per MMA step.
size_t prefill_x3_workspace(const sdpa_params_t& p);
// A mask with a row per query, copied into the prefill's score-tile layout:
// bytes of the copy (0 when the call takes none) and the copy itself.
size_t prefill_mask_tiles_bytes(const sdpa_params_t& p);
sdpa_status_t launch_mask_tiles(const sdpa_params_t& p, void* out, cudaStream_t stream);
sdpa_status_t launch_prefill_x3(const sdpa_params_t& p, const void* q, const void* k,
                                const void* v, void* o, float* lse, void* workspace,
                                const LaunchEnv& env);
sdpa_status_t launch_prefill_f32(const sdpa_params_t& p, const void* q, const void* k,
                                 const void* v, void* o, float* lse, const LaunchEnv& env);
// Lk == 0: o = 0, lse = -inf (or the sink) for every row.
sdpa_status_t launch_no_keys(const sdpa_params_t& p, void* o, float* lse, const LaunchEnv& env);
sdpa_status_t launch_decode(const sdpa_params_t& p, const DecodePlan& plan, const void* q,
                            const void* k, const void* v, void* o, float* lse, void* workspace,
                            const LaunchEnv& env);

// Backward pass (fp16/bf16, D = 64 or 128; p normalised): dQ, dK, dV in the
// layouts of q, k, v; dO in o's layout; lse the forward's.  Workspace:
// backward_workspace(p) bytes (fp32 dQ accumulator, LSE in log2 units, D).
size_t backward_workspace(const sdpa_params_t& p);
// Addresses of the LSE (log2 units) and D arrays inside that workspace.
void backward_stats_slots(const sdpa_params_t& p, void* workspace, float** lse2, float** dvec);
// The backward's pre pass: D_i = dO_i . O_i and LSE in log2 units per query
// row (+inf where the row takes no part), and a cleared dQ accumulator
// (dq_acc may be NULL).
sdpa_status_t launch_backward_pre(const sdpa_params_t& p, const void* o, const void* d_o,
                                  const float* lse, float* lse2, float* dvec, float* dq_acc,
                                  cudaStream_t stream);
// The fp32 backward (CUDA-core kernels; backward_f32.cu).
sdpa_status_t launch_backward_f32(const sdpa_params_t& p, const void* q, const void* k,
                                  const void* v, const void* o, const void* d_o,
                                  const float* lse, void* dq, void* dk, void* dv,
                                  void* workspace, const LaunchEnv& env);
sdpa_status_t launch_backward(const sdpa_params_t& p, const void* q, const void* k,
                              const void* v, const void* o, const void* d_o, const float* lse,
                              void* dq, void* dk, void* dv, void* workspace,
                              const LaunchEnv& env);

}  // namespace gb300
