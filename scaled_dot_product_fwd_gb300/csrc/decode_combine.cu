// decode_combine.cu — split-KV plan, the combine pass and the decode launch.
//
// The combine is the second pass of the two-pass vector attention of MLX PR
// #4459 ("Add D512 support to Metal vector attention"): with split s holding
// the normalised partial output O_s and the log2-domain log-sum-exp
// lse_s of its key range,
//     M   = max(max_s lse_s, sink * log2 e)
//     L   = sum_s 2^(lse_s - M) + [sink] 2^(sink * log2 e - M)
//     O   = sum_s 2^(lse_s - M) O_s / L,    LSE = (M + log2 L) ln 2.
// The sink logit (mlx 0.30.7 scaled_dot_product_attention.cpp,
// set_sink_token) enters only the denominator.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdlib.h>

#include <algorithm>

#include "decode.cuh"
#include "internal.h"

namespace gb300 {
namespace dec {

constexpr int kCombineThreads = 128;
constexpr float kLn2 = 0.6931471805599453f;

struct CombineArgs {
  const float* ws_o;
  const float* ws_ml;  // [rows][splits][2]: m (log2 units), l
  void* o;
  float* lse;
  const float* sinks;
  int Hq, num_splits, D;
  int rows_per_head;  // query rows per (batch, head): 1 for decode
  long long os0, os1, os2;  // element strides of o (batch, head, row)
  // ragged plan: a row of batch b merges only that batch's splits (the
  // split kernel's plan, derived the same way); num_splits is the row stride
  const int* seq_lens_kv;
  int ragged, batch, Lk, tile_keys, units, slots, tiles_base;
};

constexpr int kMaxSplits = 1024;  // upper bound of the split plan

// Block-wide max / sum over the 128 threads (4 warps).
__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  __syncthreads();  // red is reused by consecutive reductions
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int i = 1; i < kCombineThreads / 32; ++i) v = is_max ? fmaxf(v, red[i]) : v + red[i];
  return v;
}

// One block per output row.  Thread t owns float4 column t % (D/4) of the
// splits t / (D/4), t / (D/4) + ng, ... (ng = 128 / (D/4) groups of splits),
// and loads its first kPrefetch partials before the weights are known, so
// that the partial outputs and the (m, l) pairs share one memory round trip;
// the weights 2^(lse_s - M) go to shared memory once, and the groups' sums
// meet in shared memory at the end.
template <typename T>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const CombineArgs a) {
  constexpr int kPrefetch = 8;
  __shared__ float w[kMaxSplits];
  __shared__ float red[kCombineThreads / 32];
  __shared__ float4 part[kCombineThreads];
  // Launched with programmatic stream serialization: the split pass's
  // partial results are complete and visible after this wait.
  griddep_wait();
  griddep_launch_dependents();
  const size_t row = blockIdx.x;  // (b * Hq + hq) * rows_per_head + i
  const int hq = static_cast<int>((row / a.rows_per_head) % a.Hq);
  int S = a.num_splits;
  if (a.ragged) {
    const int b = static_cast<int>(row / (static_cast<size_t>(a.rows_per_head) * a.Hq));
    const int sk = a.tile_keys * ragged_tiles_per_split(a.seq_lens_kv, a.batch, a.Lk, a.tile_keys,
                                                        a.units, a.slots, a.tiles_base,
                                                        a.num_splits);
    const int L = min(max(a.seq_lens_kv[b], 0), a.Lk);
    S = (L + sk - 1) / sk;
  }
  const int D4 = a.D / 4;
  const int ng = D4 >= kCombineThreads ? 1 : kCombineThreads / D4;  // groups of splits
  const int c = static_cast<int>(threadIdx.x) % D4;
  const int g = static_cast<int>(threadIdx.x) / D4;
  const bool col_ok = g < ng;
  const float4* wo = reinterpret_cast<const float4*>(a.ws_o + row * a.num_splits * a.D);
  float4 pre[kPrefetch];
#pragma unroll
  for (int j = 0; j < kPrefetch; ++j) {
    const int s = g + j * ng;
    pre[j] = (col_ok && s < S) ? wo[static_cast<size_t>(s) * D4 + c]
                               : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float* ml = a.ws_ml + row * a.num_splits * 2;
  float M = -INFINITY;
  for (int s = threadIdx.x; s < S; s += kCombineThreads) M = fmaxf(M, ml[2 * s]);
  M = block_reduce(M, true, red);
  float sk = -INFINITY;
  if (a.sinks) {
    sk = a.sinks[hq] * kLog2e;
    M = fmaxf(M, sk);
  }
  float L = 0.f;
  for (int s = threadIdx.x; s < S; s += kCombineThreads) {
    const float l = ml[2 * s + 1];
    const float e = (l > 0.f) ? l * ex2(ml[2 * s] - M) : 0.f;
    w[s] = e;
    L += e;
  }
  L = block_reduce(L, false, red);  // its barriers also publish w[]
  if (a.sinks && M != -INFINITY) L += ex2(sk - M);
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col_ok && L > 0.f) {
#pragma unroll
    for (int j = 0; j < kPrefetch; ++j) {
      const int s = g + j * ng;
      const float ws = s < S ? w[s] : 0.f;
      acc.x = fmaf(ws, pre[j].x, acc.x);
      acc.y = fmaf(ws, pre[j].y, acc.y);
      acc.z = fmaf(ws, pre[j].z, acc.z);
      acc.w = fmaf(ws, pre[j].w, acc.w);
    }
#pragma unroll 4
    for (int s = g + kPrefetch * ng; s < S; s += ng) {
      const float4 v = wo[static_cast<size_t>(s) * D4 + c];
      const float ws = w[s];
      acc.x = fmaf(ws, v.x, acc.x);
      acc.y = fmaf(ws, v.y, acc.y);
      acc.z = fmaf(ws, v.z, acc.z);
      acc.w = fmaf(ws, v.w, acc.w);
    }
  }
  part[threadIdx.x] = acc;
  __syncthreads();
  if (g == 0) {
    float4 t = part[c];
    for (int gg = 1; gg < ng; ++gg) {
      const float4 u = part[gg * D4 + c];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    const size_t bh = row / a.rows_per_head;
    T* orow = static_cast<T*>(a.o) + static_cast<long long>(bh / a.Hq) * a.os0 +
              static_cast<long long>(hq) * a.os1 +
              static_cast<long long>(row - bh * a.rows_per_head) * a.os2;
    orow[4 * c + 0] = StoreAs<T>::c(t.x * inv);
    orow[4 * c + 1] = StoreAs<T>::c(t.y * inv);
    orow[4 * c + 2] = StoreAs<T>::c(t.z * inv);
    orow[4 * c + 3] = StoreAs<T>::c(t.w * inv);
  }
  if (threadIdx.x == 0 && a.lse) a.lse[row] = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
}

}  // namespace dec

static sdpa_status_t launch_combine(int dtype, const dec::CombineArgs& c, unsigned nrows,
                                    cudaStream_t stream);

namespace {
int elem_bytes(int dtype) { return dtype == SDPA_F32 ? 4 : 2; }
size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
}  // namespace

bool decode_plan(const sdpa_params_t& p, int num_sms, DecodePlan* out) {
  if (decode_tc_plan(p, num_sms, out)) return true;
  if (decode_tc128_plan(p, num_sms, out)) return true;
  out->tc = false;
  out->tc128 = false;
  const int es = elem_bytes(p.dtype);
  const int D = p.head_dim;
  // rows per kv head: its G query heads times Lq query rows
  const int G = p.num_q_heads / p.num_kv_heads * p.seq_len_q;
  const int hg_max = (D == 512) ? 4 : 8;
  int hg = 1;
  while (hg < G && hg < hg_max) hg <<= 1;
  const int groups = (G + hg - 1) / hg;
  // the grid's y dimension holds (kv head, head group) pairs, z the batch
  if (static_cast<long long>(p.num_kv_heads) * groups > 65535 || p.batch > 65535) return false;
  const int kb = dec::keys_per_warp(es, D, hg);
  const int tk = dec::kConsumerWarps * kb;
  const int stage_bytes = 2 * tk * D * es;
  int stages = 110000 / stage_bytes;
  if (stages < 2) stages = 2;
  if (stages > 4) stages = 4;
  const size_t smem = static_cast<size_t>(stages) * stage_bytes + 4096;
  int per_sm = static_cast<int>(232448 / (smem + 1024));
  if (per_sm < 1) per_sm = 1;
  if (per_sm > 2) per_sm = 2;
  if (D == 512 || hg == 8) per_sm = 1;  // register-bound (one CTA per SM)
  const long long units = static_cast<long long>(p.batch) * p.num_kv_heads * groups;
  const int ntiles = (p.seq_len_kv + tk - 1) / tk;
  const long long slots = static_cast<long long>(num_sms > 0 ? num_sms : 152) * per_sm;
  int best = 1;
  long long best_cost = -1;
  const int max_s = ntiles < 1024 ? ntiles : 1024;
  for (int s = 1; s <= max_s; ++s) {
    const long long tiles_per = (ntiles + s - 1) / s;
    const long long waves = (units * s + slots - 1) / slots;
    const long long cost = waves * (tiles_per + 2);  // 2 tiles of fixed cost per CTA
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  // The two-pass form pays a second launch and a workspace round trip.  A
  // split count of 2..16 dividing D lets the splits of each head group form
  // one thread-block cluster that merges them itself, when all the plan's
  // clusters are resident at once.  Clusters of C CTAs resident per GPU at
  // one CTA per SM, measured on a 152-SM GB300: 76, 36, 15 and 7 for
  // C = 2, 4, 8, 16 (scaled by the SM count and by CTAs per SM here).
  constexpr long long kCombineCost = 3;  // in tile units
  best_cost += kCombineCost;
  bool cluster = false;
  const long long nsm = num_sms > 0 ? num_sms : 152;
  for (int c = 2; c <= 16 && c <= max_s; c <<= 1) {
    if (D % c != 0) continue;
    const long long per_c = c == 2 ? 76 : c == 4 ? 36 : c == 8 ? 15 : 7;
    if (units > per_c * nsm / 152 * per_sm) continue;
    const long long cost = (ntiles + c - 1) / c + 2;
    if (cost < best_cost) {
      best_cost = cost;
      best = c;
      cluster = true;
    }
  }
  {  // test hook
    const int f = debug_option(SDPA_DEBUG_DECODE_SPLITS);
    if (f >= 1) {
      best = f < max_s ? f : max_s;
      cluster = best >= 2 && best <= 16 && (best & (best - 1)) == 0 && D % best == 0;
    }
  }
  const int tiles_per = (ntiles + best - 1) / best;
  const int split_keys = tiles_per * tk;
  int splits = (p.seq_len_kv + split_keys - 1) / split_keys;
  // Per-batch key lengths on the device: the ragged plan, whose split size
  // the kernels derive from the lengths (room for twice the splits of a
  // full row, so that shorter rows can be cut finer); not with a forced
  // split count (test hook) and not for very large batches (every CTA reads
  // the B lengths).
  out->ragged = false;
  out->slots = static_cast<int>(slots);
  out->tiles_base = tiles_per;
  if (p.seq_lens_kv && p.batch <= 256 && debug_option(SDPA_DEBUG_DECODE_SPLITS) < 1) {
    out->ragged = true;
    cluster = false;
    splits = std::min(std::min(2 * splits, 1024), std::max(ntiles, 1));
  }
  out->head_group = hg;
  out->num_groups = groups;
  out->tile_keys = tk;
  out->num_splits = splits;
  out->split_keys = split_keys;
  out->stages = stages;
  out->cluster = cluster;  // the launcher checks the final split count
  const size_t rows = static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q * splits;
  out->workspace = align256(rows * D * sizeof(float)) + align256(rows * 2 * sizeof(float));
  return true;
}

// The vector split pass (any head_dim, dtype and head group).
static sdpa_status_t launch_vector(const sdpa_params_t& p, const DecodePlan& plan, const void* q,
                                   const void* k, const void* v, void* o, float* lse,
                                   float* ws_o, float* ws_ml, const LaunchEnv& env,
                                   bool* merged) {
  dec::SplitArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.Hq = p.num_q_heads;
  a.Hkv = p.num_kv_heads;
  a.G = p.num_q_heads / p.num_kv_heads;
  a.Lk = p.seq_len_kv;
  a.Lq = p.seq_len_q;
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
  a.mask_bool = (p.flags & SDPA_FLAG_BOOL_MASK) ? 1 : 0;
  a.seq_lens_q = p.seq_lens_q;
  a.seq_lens_kv = p.seq_lens_kv;
  a.causal = p.causal ? 1 : 0;
  a.num_groups = plan.num_groups;
  a.num_splits = plan.num_splits;
  a.split_keys = plan.split_keys;
  a.stages = plan.stages;
  a.sl2 = p.scale * dec::kLog2e;
  a.mask = p.mask;
  a.ms0 = p.mask_stride[0];
  a.ms1 = p.mask_stride[1];
  a.ms2 = p.mask_stride[2];
  a.ws_o = ws_o;
  a.ws_ml = ws_ml;
  a.o = o;
  a.lse = lse;
  a.sinks = p.sinks;
  a.cluster = 0;
  // (test hook: 0 = two passes)
  a.cluster_ok = (plan.cluster && debug_option(SDPA_DEBUG_DECODE_CLUSTER) != 0) ? 1 : 0;
  a.status = env.status;
  a.wait_ns = env.wait_limit_ns;
  a.debug_drop_last = debug_option(SDPA_DEBUG_DECODE_DROP_LAST) == 1 ? 1 : 0;
  a.ragged = plan.ragged ? 1 : 0;
  a.batch = p.batch;
  a.slots = plan.slots;
  a.tiles_base = plan.tiles_base;
  const int D = p.head_dim, hg = plan.head_group;
  switch (p.dtype) {
    case SDPA_F32: return dec::launch_split_f32(a, D, hg, p.batch, env.stream, merged);
    case SDPA_F16: return dec::launch_split_f16(a, D, hg, p.batch, env.stream, merged);
    case SDPA_BF16: return dec::launch_split_bf16(a, D, hg, p.batch, env.stream, merged);
    default: return SDPA_ERR_UNSUPPORTED;
  }
}

sdpa_status_t launch_decode(const sdpa_params_t& p, const DecodePlan& plan, const void* q,
                            const void* k, const void* v, void* o, float* lse, void* workspace,
                            const LaunchEnv& env) {
  const size_t rows =
      static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q * plan.num_splits;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                          align256(rows * p.head_dim * sizeof(float)));
  sdpa_status_t st;
  bool merged = false;
  if (plan.tc) {
    st = launch_decode_tc(p, plan, q, k, v, o, lse, ws_o, ws_ml, env, &merged);
  } else if (plan.tc128) {
    st = launch_decode_tc128(p, plan, q, k, v, o, lse, ws_o, ws_ml, env, &merged);
  } else {
    st = launch_vector(p, plan, q, k, v, o, lse, ws_o, ws_ml, env, &merged);
  }
  if (st != SDPA_OK) return st;
  if (merged) {
    set_last_launches(1);
    return SDPA_OK;
  }
  dec::CombineArgs c;
  c.ws_o = ws_o;
  c.ws_ml = ws_ml;
  c.o = o;
  c.lse = lse;
  c.sinks = p.sinks;
  c.Hq = p.num_q_heads;
  c.num_splits = plan.num_splits;
  c.D = p.head_dim;
  c.rows_per_head = p.seq_len_q;
  c.os0 = p.o_stride[0];
  c.os1 = p.o_stride[1];
  c.os2 = p.o_stride[2];
  c.seq_lens_kv = p.seq_lens_kv;
  c.ragged = plan.ragged ? 1 : 0;
  c.batch = p.batch;
  c.Lk = p.seq_len_kv;
  c.tile_keys = plan.tile_keys;
  c.units = p.num_kv_heads * plan.num_groups;
  c.slots = plan.slots;
  c.tiles_base = plan.tiles_base;
  st = launch_combine(p.dtype, c, static_cast<unsigned>(p.batch) * p.num_q_heads * p.seq_len_q,
                      env.stream);
  if (st == SDPA_OK) set_last_launches(2);
  return st;
}

sdpa_status_t launch_no_keys(const sdpa_params_t& p, void* o, float* lse, const LaunchEnv& env) {
  dec::CombineArgs c;
  c.ws_o = nullptr;
  c.ws_ml = nullptr;
  c.o = o;
  c.lse = lse;
  c.sinks = p.sinks;
  c.Hq = p.num_q_heads;
  c.num_splits = 0;
  c.D = p.head_dim;
  c.rows_per_head = p.seq_len_q;
  c.os0 = p.o_stride[0];
  c.os1 = p.o_stride[1];
  c.os2 = p.o_stride[2];
  c.seq_lens_kv = nullptr;
  c.ragged = 0;
  const size_t rows = static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q;
  if (rows > 0x7fffffffu) return SDPA_ERR_UNSUPPORTED;
  return launch_combine(p.dtype, c, static_cast<unsigned>(rows), env.stream);
}

static sdpa_status_t launch_combine(int dtype, const dec::CombineArgs& c, unsigned nrows,
                                    cudaStream_t stream) {
  const dim3 grid(nrows);
  // Same shared-memory carveout as the split pass and the prefill kernels, so
  // alternating launches do not reconfigure the SM's L1/shared split.
  static bool carveout_set = false;
  if (!carveout_set) {
    cudaFuncSetAttribute(dec::decode_combine_kernel<float>,
                         cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    cudaFuncSetAttribute(dec::decode_combine_kernel<__half>,
                         cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    cudaFuncSetAttribute(dec::decode_combine_kernel<__nv_bfloat16>,
                         cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    carveout_set = true;
  }
  // programmatic stream serialization: the blocks may become resident while
  // the split pass drains; each waits for it before its first global read
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(dec::kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  switch (dtype) {
    case SDPA_F32: e = cudaLaunchKernelEx(&cfg, dec::decode_combine_kernel<float>, c); break;
    case SDPA_F16: e = cudaLaunchKernelEx(&cfg, dec::decode_combine_kernel<__half>, c); break;
    default: e = cudaLaunchKernelEx(&cfg, dec::decode_combine_kernel<__nv_bfloat16>, c); break;
  }
  return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // namespace gb300
