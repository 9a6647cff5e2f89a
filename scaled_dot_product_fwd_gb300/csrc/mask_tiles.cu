// mask_tiles.cu — a mask with its own row per query, re-laid for the
// tensor-core prefill's softmax warps.
//
// The pages add the mask to each score (rustytorch flash_attention.metal: the
// mask element of (query, key) joins the score before the row max; mlx
// 0.30.7 scaled_dot_product_attention.cpp: an additive bias with its own
// strides).  In the prefill kernel each softmax thread owns one query row,
// so reading the mask where it lies makes every warp-wide load touch 32 rows
// (and, where rows are not 16-byte aligned, one element at a time).  This
// pass copies the mask once per call into tiles that match the kernel's
// 128 x 128 score tiles: tile (plane, query tile, key tile) holds
// [key group][128 rows][16 bytes] (groups of 8 fp16/bf16 keys or 16 boolean
// bytes), so a warp's 16-byte loads read 512 contiguous bytes.  Rows past Lq
// and keys past Lk are zero.  A plane is one distinct (batch, head) of the
// mask's broadcast (stride 0 = one plane for every batch or head).
#include <cuda_runtime.h>

#include "internal.h"

namespace gb300 {
namespace {

constexpr int kTile = 128;     // rows and keys of a tile
constexpr int kThreads = 256;
constexpr int kPitch = 272;    // bytes per staged row: 256 + 16 (conflict-free 16-byte reads)

struct TileArgs {
  const uint8_t* mask;
  uint8_t* out;
  long long ms0, ms1, ms2;  // element strides of the mask (batch, head, row)
  int es;                   // bytes per element (2, or 1 for a boolean mask)
  int Lq, Lk, nqt, nkt, nh; // nh: head planes (1 when broadcast over heads)
};

__global__ void __launch_bounds__(kThreads) mask_tiles_kernel(const TileArgs a) {
  __shared__ __align__(16) uint8_t st[kTile * kPitch];
  const int kt = blockIdx.x, qt = blockIdx.y, plane = blockIdx.z;
  const int pb = plane / a.nh, ph = plane % a.nh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_bytes = kTile * a.es;  // 256 (fp16/bf16) or 128 (bool)
  // rows in: lanes along the row, one element per lane and step (any alignment)
  for (int r = warp; r < kTile; r += kThreads / 32) {
    const int qi = qt * kTile + r;
    const uint8_t* src = a.mask + (pb * a.ms0 + ph * a.ms1 + static_cast<long long>(qi) * a.ms2 +
                                   static_cast<long long>(kt) * kTile) * a.es;
    uint8_t* dst = st + r * kPitch;
    for (int k = lane; k < kTile; k += 32) {
      const bool in = qi < a.Lq && kt * kTile + k < a.Lk;
      if (a.es == 2) {
        const uint16_t v = in ? reinterpret_cast<const uint16_t*>(src)[k] : 0;
        reinterpret_cast<uint16_t*>(dst)[k] = v;
      } else {
        dst[k] = in ? src[k] : 0;
      }
    }
  }
  __syncthreads();
  // tile out: chunk c = (group g, row r) is 16 bytes at c * 16
  uint8_t* out = a.out + ((static_cast<size_t>(plane) * a.nqt + qt) * a.nkt + kt) *
                             static_cast<size_t>(kTile) * row_bytes;
  const int groups = row_bytes / 16;
  for (int c = threadIdx.x; c < groups * kTile; c += kThreads) {
    const int g = c / kTile, r = c % kTile;
    reinterpret_cast<uint4*>(out)[c] = *reinterpret_cast<const uint4*>(st + r * kPitch + g * 16);
  }
}

}  // namespace

// Bytes of the tiled copy (0: the call does not use one).  fp16/bf16 data
// with a mask that has a row per query (additive, or boolean).
size_t prefill_mask_tiles_bytes(const sdpa_params_t& p) {
  if (!p.mask || p.mask_stride[2] == 0 || p.dtype == SDPA_F32 || p.head_dim == 512) return 0;
  if (p.seq_len_q <= 0 || p.seq_len_kv <= 0) return 0;
  const size_t es = (p.flags & SDPA_FLAG_BOOL_MASK) ? 1 : 2;
  const size_t nb = p.mask_stride[0] ? static_cast<size_t>(p.batch) : 1;
  const size_t nh = p.mask_stride[1] ? static_cast<size_t>(p.num_q_heads) : 1;
  const size_t nqt = (p.seq_len_q + kTile - 1) / kTile, nkt = (p.seq_len_kv + kTile - 1) / kTile;
  return (nb * nh * nqt * nkt * kTile * kTile * es + 255) & ~static_cast<size_t>(255);
}

sdpa_status_t launch_mask_tiles(const sdpa_params_t& p, void* out, cudaStream_t stream) {
  TileArgs a;
  a.mask = static_cast<const uint8_t*>(p.mask);
  a.out = static_cast<uint8_t*>(out);
  a.ms0 = p.mask_stride[0];
  a.ms1 = p.mask_stride[1];
  a.ms2 = p.mask_stride[2];
  a.es = (p.flags & SDPA_FLAG_BOOL_MASK) ? 1 : 2;
  a.Lq = p.seq_len_q;
  a.Lk = p.seq_len_kv;
  a.nqt = (p.seq_len_q + kTile - 1) / kTile;
  a.nkt = (p.seq_len_kv + kTile - 1) / kTile;
  a.nh = p.mask_stride[1] ? p.num_q_heads : 1;
  const int nb = p.mask_stride[0] ? p.batch : 1;
  if (a.nqt > 65535 || static_cast<long long>(nb) * a.nh > 65535) return SDPA_ERR_UNSUPPORTED;
  const dim3 grid(static_cast<unsigned>(a.nkt), static_cast<unsigned>(a.nqt),
                  static_cast<unsigned>(nb * a.nh));
  mask_tiles_kernel<<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

}  // namespace gb300
