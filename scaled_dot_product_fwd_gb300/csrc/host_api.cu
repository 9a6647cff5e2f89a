// host_api.cu — the forward pass on host buffers: q, k, v come from host
// memory and o, lse go back to it, with the transfers of one piece of the
// problem overlapping the kernels of another.
//
// The mlx page's call (mlx 0.30.7 scaled_dot_product_attention.cpp,
// eval_gpu) takes the framework's arrays and brings them to the device
// before the fused graph runs; this entry point is that whole trip for
// callers whose tensors live on the host.  The (batch, kv-head) pairs are
// cut into pieces within one batch; each piece's q, k, v are copied in on
// two copy streams, its attention runs through sdpa_forward (the library's
// kernels) on one of two compute streams, each with its own workspace, and
// its o and lse are copied out on a fifth stream.  One cudaMemcpyAsync per
// piece and direction of each tensor.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "internal.h"
#include "sdpa.h"

namespace gb300 {
namespace {

constexpr int kHostStreams = 5;  // copy in (q), copy in (k, v), compute x2, copy out
constexpr int kMaxPieces = 256;
constexpr int kMaxDevices = 64;

size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

size_t elem_size(int dtype) { return dtype == SDPA_F32 ? 4 : 2; }

// Streams and events of one device, created on its first call and kept
// until exit (no device memory).
struct HostRes {
  bool ready = false;
  cudaStream_t st[kHostStreams];
  cudaEvent_t fork;
  cudaEvent_t done[kHostStreams];
  cudaEvent_t ev[3 * kMaxPieces];  // per piece: q in, k/v in, computed
};
std::mutex g_host_mu;
HostRes g_host[kMaxDevices];

struct Piece {
  int b, h0, h1;  // batch, kv-head range [h0, h1)
};

// Every batch split into about `pieces` / B contiguous kv-head ranges.
std::vector<Piece> make_pieces(int B, int Hkv, int pieces) {
  const int per_b = std::max(1, std::min(Hkv, (pieces + std::max(B, 1) - 1) / std::max(B, 1)));
  std::vector<Piece> out;
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < per_b; ++i) {
      const int h0 = (Hkv * i) / per_b, h1 = (Hkv * (i + 1)) / per_b;
      if (h1 > h0) out.push_back({b, h0, h1});
    }
  return out;
}

// The problem of one piece: batch 1, the piece's heads, the same lengths;
// mask and sinks moved to the piece's first (batch, head).
sdpa_params_t piece_params(const sdpa_params_t& p, const Piece& c) {
  const int G = p.num_q_heads / p.num_kv_heads;
  sdpa_params_t q = p;
  q.batch = 1;
  q.num_q_heads = (c.h1 - c.h0) * G;
  q.num_kv_heads = c.h1 - c.h0;
  q.flags |= SDPA_FLAG_SHARED_GPU;
  if (p.mask) {
    const size_t es = (p.flags & SDPA_FLAG_BOOL_MASK) ? 1 : elem_size(p.dtype);
    q.mask = static_cast<const uint8_t*>(p.mask) +
             (c.b * p.mask_stride[0] + static_cast<int64_t>(c.h0) * G * p.mask_stride[1]) * es;
  }
  if (p.sinks) q.sinks = p.sinks + c.h0 * G;
  return q;
}

// Checks specific to this entry point: dense layouts only (no strides, no
// KV-cache capacity, no per-batch length arrays).
sdpa_status_t host_checks(const sdpa_params_t* p) {
  if (!p) return SDPA_ERR_INVALID_ARGUMENT;
  if ((p->flags & SDPA_FLAG_STRIDES) || p->seq_lens_q || p->seq_lens_kv ||
      (p->kv_capacity != 0 && p->kv_capacity != p->seq_len_kv))
    return SDPA_ERR_UNSUPPORTED;
  return SDPA_OK;
}

struct Staging {
  size_t q, k, v, o, lse, ws0, ws1, total, ws_bytes;
};

Staging staging_layout(const sdpa_params_t& p, const std::vector<Piece>& pieces) {
  const size_t es = elem_size(p.dtype);
  const size_t qn = static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q * p.head_dim;
  const size_t kn = static_cast<size_t>(p.batch) * p.num_kv_heads * p.seq_len_kv * p.head_dim;
  const size_t ln = static_cast<size_t>(p.batch) * p.num_q_heads * p.seq_len_q;
  size_t ws = 0;
  for (const Piece& c : pieces) {
    const sdpa_params_t pp = piece_params(p, c);
    ws = std::max(ws, sdpa_workspace_size(&pp));
  }
  Staging s;
  s.q = 0;
  s.k = s.q + align256(qn * es);
  s.v = s.k + align256(kn * es);
  s.o = s.v + align256(kn * es);
  s.lse = s.o + align256(qn * es);
  s.ws0 = s.lse + align256(ln * 4);
  s.ws1 = s.ws0 + align256(ws);
  s.total = s.ws1 + align256(ws);
  s.ws_bytes = ws;
  return s;
}

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" {

size_t sdpa_host_staging_size(const sdpa_params_t* params, int pieces) {
  if (host_checks(params) != SDPA_OK) return 0;
  sdpa_status_t st;
  if (sdpa_select_kernel(params, &st) == SDPA_KERNEL_NONE && st != SDPA_OK) return 0;
  if (pieces < 1) pieces = 1;
  const std::vector<Piece> pc =
      make_pieces(params->batch, params->num_kv_heads, std::min(pieces, kMaxPieces));
  return staging_layout(*params, pc).total;
}

sdpa_status_t sdpa_forward_host(const sdpa_params_t* params, const void* q_host,
                                const void* k_host, const void* v_host, void* o_host,
                                float* lse_host, void* staging, size_t staging_bytes, int pieces,
                                void* stream) {
  set_last_launches(0);
  sdpa_status_t st = host_checks(params);
  if (st != SDPA_OK) return st;
  sdpa_select_kernel(params, &st);
  if (st != SDPA_OK) return st;
  const sdpa_params_t& p = *params;
  if (static_cast<int64_t>(p.batch) * p.num_q_heads * p.seq_len_q == 0) return SDPA_OK;
  if (!q_host || !o_host || (p.seq_len_kv > 0 && (!k_host || !v_host)))
    return SDPA_ERR_INVALID_ARGUMENT;
  if (pieces < 1) pieces = 1;
  const std::vector<Piece> pc = make_pieces(p.batch, p.num_kv_heads, std::min(pieces, kMaxPieces));
  const Staging sl = staging_layout(p, pc);
  if (!staging || staging_bytes < sl.total) return SDPA_ERR_WORKSPACE_TOO_SMALL;
  if ((reinterpret_cast<uintptr_t>(staging) & 255u) != 0) return SDPA_ERR_MISALIGNED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDPA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_host_mu);
  HostRes& r = g_host[dev];
  if (!r.ready) {
    for (int i = 0; i < kHostStreams; ++i)
      if (cudaStreamCreateWithFlags(&r.st[i], cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&r.done[i], cudaEventDisableTiming) != cudaSuccess)
        return SDPA_ERR_CUDA;
    if (cudaEventCreateWithFlags(&r.fork, cudaEventDisableTiming) != cudaSuccess)
      return SDPA_ERR_CUDA;
    for (int i = 0; i < 3 * kMaxPieces; ++i)
      if (cudaEventCreateWithFlags(&r.ev[i], cudaEventDisableTiming) != cudaSuccess)
        return SDPA_ERR_CUDA;
    r.ready = true;
  }
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  cudaStream_t s_in0 = r.st[0], s_in1 = r.st[1], s_out = r.st[4];
  // every stream starts after the work already on the caller's stream
  bool ok = cudaEventRecord(r.fork, caller) == cudaSuccess;
  for (int i = 0; i < kHostStreams && ok; ++i) ok = cudaStreamWaitEvent(r.st[i], r.fork, 0) == cudaSuccess;

  uint8_t* base = static_cast<uint8_t*>(staging);
  const size_t es = elem_size(p.dtype);
  const int G = p.num_q_heads / p.num_kv_heads;
  const size_t qrow = static_cast<size_t>(p.seq_len_q) * p.head_dim * es;  // one query head
  const size_t krow = static_cast<size_t>(p.seq_len_kv) * p.head_dim * es;  // one kv head
  const size_t lrow = static_cast<size_t>(p.seq_len_q) * 4;
  int launches = 0;
  for (size_t i = 0; i < pc.size() && ok; ++i) {
    const Piece& c = pc[i];
    const size_t hq0 = static_cast<size_t>(c.b) * p.num_q_heads + static_cast<size_t>(c.h0) * G;
    const size_t nq = static_cast<size_t>(c.h1 - c.h0) * G;
    const size_t hk0 = static_cast<size_t>(c.b) * p.num_kv_heads + c.h0;
    const size_t nk = static_cast<size_t>(c.h1 - c.h0);
    cudaEvent_t e_q = r.ev[3 * i], e_kv = r.ev[3 * i + 1], e_c = r.ev[3 * i + 2];
    ok = cudaMemcpyAsync(base + sl.q + hq0 * qrow, static_cast<const uint8_t*>(q_host) + hq0 * qrow,
                         nq * qrow, cudaMemcpyHostToDevice, s_in0) == cudaSuccess &&
         cudaEventRecord(e_q, s_in0) == cudaSuccess;
    if (ok && krow > 0)
      ok = cudaMemcpyAsync(base + sl.k + hk0 * krow, static_cast<const uint8_t*>(k_host) + hk0 * krow,
                           nk * krow, cudaMemcpyHostToDevice, s_in1) == cudaSuccess &&
           cudaMemcpyAsync(base + sl.v + hk0 * krow, static_cast<const uint8_t*>(v_host) + hk0 * krow,
                           nk * krow, cudaMemcpyHostToDevice, s_in1) == cudaSuccess;
    ok = ok && cudaEventRecord(e_kv, s_in1) == cudaSuccess;
    cudaStream_t s_c = r.st[2 + (i & 1)];
    ok = ok && cudaStreamWaitEvent(s_c, e_q, 0) == cudaSuccess &&
         cudaStreamWaitEvent(s_c, e_kv, 0) == cudaSuccess;
    if (!ok) break;
    const sdpa_params_t pp = piece_params(p, c);
    st = sdpa_forward(&pp, base + sl.q + hq0 * qrow, base + sl.k + hk0 * krow,
                      base + sl.v + hk0 * krow, base + sl.o + hq0 * qrow,
                      reinterpret_cast<float*>(base + sl.lse + hq0 * lrow),
                      sl.ws_bytes ? base + ((i & 1) ? sl.ws1 : sl.ws0) : nullptr, sl.ws_bytes, s_c);
    if (st != SDPA_OK) break;
    launches += sdpa_last_launch_count();
    ok = cudaEventRecord(e_c, s_c) == cudaSuccess &&
         cudaStreamWaitEvent(s_out, e_c, 0) == cudaSuccess &&
         cudaMemcpyAsync(static_cast<uint8_t*>(o_host) + hq0 * qrow, base + sl.o + hq0 * qrow,
                         nq * qrow, cudaMemcpyDeviceToHost, s_out) == cudaSuccess;
    if (ok && lse_host)
      ok = cudaMemcpyAsync(reinterpret_cast<uint8_t*>(lse_host) + hq0 * lrow,
                           base + sl.lse + hq0 * lrow, nq * lrow, cudaMemcpyDeviceToHost,
                           s_out) == cudaSuccess;
  }
  // the caller's stream continues once every stream has finished (also
  // after an error, so that no work is left unordered with the caller's)
  bool joined = true;
  for (int i = 0; i < kHostStreams; ++i)
    joined = joined && cudaEventRecord(r.done[i], r.st[i]) == cudaSuccess &&
             cudaStreamWaitEvent(caller, r.done[i], 0) == cudaSuccess;
  set_last_launches(launches);
  if (st != SDPA_OK) return st;
  return (ok && joined) ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // extern "C"
