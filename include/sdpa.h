/*
 * sdpa.h — C ABI of a fused, memory-efficient scaled-dot-product attention
 * forward pass for NVIDIA GB300 (sm_103a).
 *
 *   O   = softmax(scale * Q K^T + mask [+ sink column]) V
 *   LSE = ln( sum_j exp(scale * q.k_j + mask_j) [+ exp(sink)] )
 *
 * The operation is the one named by the problem statement of MLX PR #964
 * ("Metal shaders for memory efficient self attention on large sequences",
 * the call mx.fast.scaled_dot_product_attention(queries, keys, values,
 * scale=scale, mask=None)) widened by MLX PR #4459 ("Add D512 support to
 * Metal vector attention": grouped-query heads, head_dim 512, per-head
 * sinks, single-query decode through single-pass and two-pass vector
 * kernels) and by the option set of the cuDNN graph built in mlx 0.30.7
 * mlx/backend/cuda/scaled_dot_product_attention.cpp (build_sdpa_graph:
 * attention scale, log-sum-exp statistics output, bottom-right causal mask,
 * additive bias, sink token).  The score matrix is computed tile by tile with
 * an online softmax (running max m and running sum l, rustytorch
 * flash_attention.metal, forward kernel) and never written to device memory.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layout: q is [B, Hq, Lq, D], k and v are [B, Hkv, Lk, D], o is
 *    [B, Hq, Lq, D], element type params->dtype, dense row-major
 *    ("contiguous") unless SDPA_FLAG_STRIDES gives their strides (the D
 *    dimension stays contiguous).  lse is [B, Hq, Lq] float32, dense.  The query head h
 *    reads key/value head floor(h / (Hq / Hkv)) (contiguous head groups).
 *  - Pointers q, k, v, o, lse, mask, sinks and workspace are DEVICE pointers
 *    owned by the caller; the library never allocates, frees or retains them.
 *    Base pointers of q, k, v and o must be 16-byte aligned; mask aligned to
 *    its element size; lse, sinks 4-byte aligned; workspace 256-byte
 *    aligned.
 *  - sdpa_forward is asynchronous on `stream` (a cudaStream_t, passed as
 *    void* so that this header needs no CUDA include; NULL = legacy default
 *    stream).  It never synchronises the host.
 *  - Argument and layout errors are detected on the host before any launch,
 *    and nothing is written.  Launch failures are reported as SDPA_ERR_CUDA.
 *    No C++ exception crosses this ABI.  Kernels never trap: a device-side
 *    wait that gives up sets a device status word, read and cleared by
 *    sdpa_device_status().
 */
#ifndef GB300_SDPA_H_
#define GB300_SDPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SDPA_ABI_VERSION 5

#if defined(__GNUC__)
#define SDPA_API __attribute__((visibility("default")))
#else
#define SDPA_API
#endif

typedef enum {
  SDPA_F32 = 0,
  SDPA_F16 = 1,
  SDPA_BF16 = 2
} sdpa_dtype_t;

typedef enum {
  SDPA_OK = 0,
  SDPA_ERR_INVALID_ARGUMENT = 1, /* null pointer, non-positive size, bad stride */
  SDPA_ERR_UNSUPPORTED = 2,      /* valid problem outside the supported space */
  SDPA_ERR_MISALIGNED = 3,       /* a base pointer breaks the alignment rule */
  SDPA_ERR_WORKSPACE_TOO_SMALL = 4,
  SDPA_ERR_CUDA = 5,             /* a CUDA runtime call or launch failed */
  SDPA_ERR_TIMEOUT = 6           /* a device-side wait gave up (status word) */
} sdpa_status_t;

/* Kernel paths.  The launcher picks one from the shape alone: one query row
 * per head (decode), or a few (up to 2 at D = 64/128, up to 8 at D = 512),
 * take the split-KV vector path, where the rows of a kv head share its K/V
 * stream; longer query sequences take the prefill kernels. */
typedef enum {
  SDPA_KERNEL_NONE = 0,
  SDPA_KERNEL_PREFILL_TC = 1,   /* fp16/bf16, Lq > 2: TMA + tcgen05 + TMEM */
  SDPA_KERNEL_PREFILL_F32 = 2,  /* fp32, D = 128, Lq > 2: fp32 FMA tiles */
  SDPA_KERNEL_DECODE_SPLITKV = 3, /* small Lq: split-KV vector pass + merge */
  SDPA_KERNEL_NO_KEYS = 4,       /* Lk == 0: writes o = 0 and the empty lse */
  SDPA_KERNEL_PREFILL_TC_F32 = 5 /* fp32, D = 64, Lq > 2: bf16 hi/lo splits on
                                    tcgen05 (three products per step) */
} sdpa_kernel_t;

/*
 * Problem description.
 *  batch, num_q_heads, num_kv_heads, seq_len_q, seq_len_kv, head_dim:
 *      B, Hq, Hkv, Lq, Lk, D.  Hkv >= 1, the others >= 0, Hq % Hkv == 0,
 *      D in {64, 128, 512} (512: Lq <= 8 only), Lq and Lk at most 2^30.  When B * Hq * Lq == 0
 *      there is nothing to compute and the call returns SDPA_OK at once.
 *      When Lk == 0 every row sees no key: o = 0 and lse = -inf (the sink
 *      logit itself with sinks).
 *  dtype: element type of q, k, v, o and mask.
 *  scale: multiplies q.k before the mask is added; the caller passes it
 *      explicitly (1/sqrt(D) for the usual choice).  Must be finite.
 *  causal: nonzero = bottom-right aligned causal mask, key j is visible to
 *      query i iff j <= i + (Lk - Lq) (the alignment of the cuDNN graph's
 *      causal_mask_bottom_right; identical to "j <= i" when Lq == Lk).
 *      Requires Lq <= Lk.
 *  mask: NULL or an additive bias added to the scaled scores, element type
 *      dtype, addressed as mask[b*s0 + h*s1 + i*s2 + j*s3] with
 *      mask_stride = {s0, s1, s2, s3} in ELEMENTS; a stride of 0 broadcasts
 *      that dimension; s3 must be 1.  -inf entries remove a key.  With
 *      SDPA_FLAG_BOOL_MASK it is a boolean mask instead: one byte per
 *      element (same addressing, strides in bytes), nonzero = the key is
 *      visible to the query, zero = removed.  When both mask and causal are
 *      given, both apply.
 *  sinks: NULL or float32 [Hq]: one extra logit per query head that enters
 *      the softmax denominator only (a key with a zero value row).  It is
 *      not multiplied by scale and not masked.
 *  kv_capacity: 0, or the number of rows per (batch, kv head) that k and v
 *      hold (>= seq_len_kv): k and v are then [B, Hkv, kv_capacity, D], a
 *      fixed-capacity KV cache of which rows [0, seq_len_kv) are used (the
 *      rest is never read into a result).  0 means kv_capacity = seq_len_kv.
 *  seq_lens_q, seq_lens_kv: NULL, or DEVICE int32 [B] arrays of per-batch
 *      lengths (padding masks): batch b uses query rows [0, seq_lens_q[b])
 *      and keys [0, seq_lens_kv[b]) (values are clamped to [0, seq_len_q]
 *      and [0, seq_len_kv]); query rows at or past its length see no key
 *      (o = 0, lse = -inf or the sink), and the bottom-right causal rule
 *      uses the batch's own lengths: key j visible to query i iff
 *      j <= i + (seq_lens_kv[b] - seq_lens_q[b]).  Both arrays must stay
 *      valid until the call's kernels have run.  The prefill kernels and
 *      the fp16/bf16 decode passes load whole key
 *      tiles, so v rows [seq_lens_kv[b], seq_len_kv) meet zero weights there
 *      and must hold finite values (rows past seq_len_kv are never read).
 *  flags: an OR of the SDPA_FLAG_* bits below (other bits must be 0, else
 *      SDPA_ERR_INVALID_ARGUMENT).
 *  q_stride, k_stride, v_stride, o_stride (ABI 4): read only with
 *      SDPA_FLAG_STRIDES (a caller built against ABI 3 leaves the flag clear
 *      and need not provide them).  Element strides of dimensions B, H and L
 *      of each tensor (D is contiguous), each >= 0 and, times the element
 *      size, a multiple of 16 bytes; o must not overlap q, k or v.  They
 *      replace the dense layout and kv_capacity (which must then be 0).
 *      Example: [B, L, H, D] tensors ("BSHD") have strides {L*H*D, D, H*D}.
 */
/* The call runs beside other work on the GPU (kernels of other streams):
 * launch shapes are not fitted to an idle GPU.  Without it, a prefill whose
 * query-tile units leave a partial last wave on the SMs shares the key tiles
 * of those units among the CTAs of thread-block clusters (a second, shorter
 * grid); with it, every unit runs whole. */
#define SDPA_FLAG_SHARED_GPU 0x1u
/* mask is boolean (bytes, nonzero = visible) instead of an additive bias. */
#define SDPA_FLAG_BOOL_MASK 0x2u
/* q_stride, k_stride, v_stride and o_stride give the tensors' layouts. */
#define SDPA_FLAG_STRIDES 0x4u
typedef struct {
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t seq_len_q;
  int32_t seq_len_kv;
  int32_t head_dim;
  int32_t dtype;   /* sdpa_dtype_t */
  float scale;
  int32_t causal;
  int32_t reserved0;
  const void* mask;
  int64_t mask_stride[4];
  const float* sinks;
  int32_t kv_capacity;          /* ABI 2 */
  uint32_t flags;               /* ABI 3 (was reserved, 0) */
  const int32_t* seq_lens_q;    /* ABI 2 */
  const int32_t* seq_lens_kv;   /* ABI 2 */
  int64_t q_stride[3];          /* ABI 4, with SDPA_FLAG_STRIDES */
  int64_t k_stride[3];
  int64_t v_stride[3];
  int64_t o_stride[3];
} sdpa_params_t;

/*
 * sdpa_workspace_size — bytes of device workspace that sdpa_forward needs for
 * this problem (split-KV partial outputs of the decode path; the bf16 hi/lo
 * copies of q, k and v of the fp32 tensor-core prefill; for an fp16/bf16
 * prefill whose mask has a row per query, room for a copy of the mask laid
 * out in the kernel's 128 x 128 score tiles — optional: with a smaller or
 * NULL workspace that call reads the mask where it lies, slower where a
 * warp's rows are far apart; 0 when the chosen path needs none).  Pure host
 * function; returns 0 for an invalid problem as well (sdpa_forward then
 * reports the error).
 */
SDPA_API size_t sdpa_workspace_size(const sdpa_params_t* params);

/*
 * sdpa_select_kernel — the kernel path sdpa_forward would run for this
 * problem, or SDPA_KERNEL_NONE with *status set when the problem is invalid
 * or unsupported (SDPA_KERNEL_NONE with SDPA_OK: nothing to compute).  Pure
 * host function (no CUDA call).  `status` may be NULL.
 */
SDPA_API sdpa_kernel_t sdpa_select_kernel(const sdpa_params_t* params, sdpa_status_t* status);

/*
 * sdpa_forward — compute o (and lse, when non-NULL) for the problem in
 * `params` on `stream`.
 *  q, k, v: inputs (device, read only).  o: output (device, written).
 *  lse: NULL or float32 [B, Hq, Lq] output in natural-log units; a fully
 *      masked row gives o = 0 and lse = -inf (lse = sink with sinks).
 *  workspace / workspace_bytes: device scratch of at least
 *      sdpa_workspace_size(params) bytes (NULL allowed when that is 0).  Its
 *      contents need no initialisation and are overwritten; two calls that
 *      overlap on the GPU must not share one workspace.
 * Returns SDPA_OK once the work is enqueued.
 */
SDPA_API sdpa_status_t sdpa_forward(const sdpa_params_t* params,
                           const void* q, const void* k, const void* v,
                           void* o, float* lse,
                           void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * sdpa_backward_workspace_size — bytes of device workspace that sdpa_backward
 * needs (an fp32 dQ accumulator [B, Hq, Lq, D] and two fp32 [B, Hq, Lq]
 * arrays); 0 for an invalid or unsupported problem.  Pure host function.
 */
SDPA_API size_t sdpa_backward_workspace_size(const sdpa_params_t* params);

/*
 * sdpa_backward — gradients of the forward pass (the backward kernels of the
 * rustytorch flash_attention.metal page: P = exp(S - LSE), D_i = dO_i . O_i,
 * dS = P (dO V^T - D), dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO; with
 * the options of the mlx cuDNN backward graph: scale, bottom-right causal
 * mask, additive or boolean mask, sink token).  The problem description is
 * the forward's (same params), per-batch length arrays included: rows and
 * keys past a batch's lengths get zero gradients.  Supported: head_dim 64 or
 * 128 (else SDPA_ERR_UNSUPPORTED); fp16/bf16 on the tensor cores, fp32 on
 * fp32 CUDA-core kernels.  Rows of q, k, v and d_o inside seq_len_q /
 * seq_len_kv but past a batch's lengths must hold finite values (whole tiles
 * are read; their weights are zero).
 *  q, k, v, o, lse: the forward's inputs, output and log-sum-exp (lse is
 *      required: the forward must have been asked for it).
 *  d_o: gradient of the loss with respect to o, in o's layout.
 *  dq, dk, dv: outputs in the layouts of q, k and v (their dtype).  With
 *      grouped-query heads dk and dv sum over the query heads of each group.
 *      The sink and the mask receive no gradient.
 *  workspace / workspace_bytes: at least sdpa_backward_workspace_size(params)
 *      bytes, 256-byte aligned; contents need no initialisation.
 * Asynchronous on `stream`; errors as for sdpa_forward.
 */
SDPA_API sdpa_status_t sdpa_backward(const sdpa_params_t* params, const void* q, const void* k,
                                     const void* v, const void* o, const void* d_o,
                                     const float* lse, void* dq, void* dk, void* dv,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * sdpa_host_staging_size — bytes of device staging memory that
 * sdpa_forward_host needs for this problem cut into `pieces` pieces (device
 * copies of q, k, v, o and lse, and two workspaces); 0 for a problem that
 * sdpa_forward_host rejects.  Pure host function.
 */
SDPA_API size_t sdpa_host_staging_size(const sdpa_params_t* params, int pieces);

/*
 * sdpa_forward_host — sdpa_forward for callers whose q, k, v and results
 * live in host memory: the whole trip of the mlx page's call (mlx 0.30.7
 * scaled_dot_product_attention.cpp, eval_gpu: the framework's arrays brought
 * to the device, the fused graph run, the output handed back), with the
 * transfers of one piece overlapping the kernels of another.
 *  q_host, k_host, v_host: inputs in HOST memory, dense [B, H, L, D] in
 *      params->dtype (page-locked memory, cudaMallocHost or
 *      cudaHostRegister, lets the copies overlap; pageable memory works, with
 *      each copy waiting for the host).
 *  o_host, lse_host: outputs in host memory, dense (lse_host may be NULL).
 *  params: as for sdpa_forward; mask and sinks, if any, are DEVICE pointers.
 *      Dense layouts only: SDPA_FLAG_STRIDES, a kv_capacity other than 0 or
 *      seq_len_kv, or per-batch length arrays give SDPA_ERR_UNSUPPORTED.
 *  staging / staging_bytes: caller-owned device memory of at least
 *      sdpa_host_staging_size(params, pieces) bytes, 256-byte aligned; two
 *      calls whose work overlaps must not share it.
 *  pieces: the (batch, kv-head) pairs are cut into about this many pieces,
 *      each within one batch.  Piece i's host-to-device copies run on two
 *      copy streams, its kernels (those of sdpa_forward, with
 *      SDPA_FLAG_SHARED_GPU) on one of two compute streams, its
 *      device-to-host copies on a fifth: one cudaMemcpyAsync per piece and
 *      tensor.
 *  stream: the caller's stream.  The work starts after what is already
 *      enqueued on it, and what the caller enqueues on it afterwards runs
 *      after this call's copies have landed in o_host and lse_host (e.g. a
 *      cudaStreamSynchronize(stream) makes them readable).
 * The five streams and their events belong to the library: created on the
 * first call on a device (with that device current) and kept until exit;
 * calls from several threads are serialised while they enqueue.  Nothing is
 * allocated on the device.  sdpa_last_launch_count counts the kernels of
 * every piece.  Errors as for sdpa_forward; SDPA_ERR_WORKSPACE_TOO_SMALL for
 * too small a staging area.
 */
SDPA_API sdpa_status_t sdpa_forward_host(const sdpa_params_t* params, const void* q_host,
                                         const void* k_host, const void* v_host, void* o_host,
                                         float* lse_host, void* staging, size_t staging_bytes,
                                         int pieces, void* stream);

/* sdpa_status_string — static, NUL-terminated text for a status code. */
SDPA_API const char* sdpa_status_string(sdpa_status_t status);

/*
 * sdpa_device_status — synchronise `stream`, then read and clear the device
 * status word that kernels set when one of their bounded waits gives up.
 * Returns SDPA_OK, SDPA_ERR_TIMEOUT, or SDPA_ERR_CUDA if the synchronisation
 * itself failed.  The status word is per device and shared by all streams.
 */
SDPA_API sdpa_status_t sdpa_device_status(void* stream);

/*
 * sdpa_debug_set_wait_limit_ns — test hook: upper bound in nanoseconds on
 * every device-side barrier wait of later launches (default 2e9).  0
 * restores the default.  Returns the previous value.
 */
SDPA_API uint64_t sdpa_debug_set_wait_limit_ns(uint64_t ns);

/*
 * sdpa_debug_set_option — test hooks that override a launch decision of
 * later calls, process-wide (they exist so that tests reach paths that the
 * planner would not pick for the test's sizes).  Returns the previous value;
 * an unknown option returns -1 and changes nothing.
 *  SDPA_DEBUG_DECODE_SPLITS   split count of the decode passes (0: the plan's)
 *  SDPA_DEBUG_DECODE_CLUSTER  0: never merge the splits inside a cluster
 *                             (two passes); 1: as planned (default)
 *  SDPA_DEBUG_DECODE_DROP_LAST 1: the vector path's producer skips its last
 *                             copy, so that a bounded wait runs out and the
 *                             call reports SDPA_ERR_TIMEOUT (default 0)
 *  SDPA_DEBUG_PREFILL_SPLIT   -1: the plan's (default); 0: never split the
 *                             last wave; 2, 4: every unit shared by that
 *                             many CTAs of a cluster
 *  SDPA_DEBUG_DECODE_VECTOR   1: head_dim-64/128 fp16/bf16 decode on the
 *                             vector path instead of the tensor-core pass
 *                             (default 0)
 */
typedef enum {
  SDPA_DEBUG_DECODE_SPLITS = 0,
  SDPA_DEBUG_DECODE_CLUSTER = 1,
  SDPA_DEBUG_DECODE_DROP_LAST = 2,
  SDPA_DEBUG_PREFILL_SPLIT = 3,
  SDPA_DEBUG_DECODE_VECTOR = 4
} sdpa_debug_option_t;
SDPA_API int sdpa_debug_set_option(int option, int value);

/* sdpa_abi_version — SDPA_ABI_VERSION of the built library. */
SDPA_API int sdpa_abi_version(void);

/*
 * sdpa_last_launch_count — number of kernels that the calling thread's last
 * sdpa_forward or sdpa_forward_decode_noalloc call enqueued (0 if it
 * returned an error or had nothing to compute): 1 for the prefill kernels
 * and for a decode whose splits merge inside a thread-block cluster, 2 for
 * the fp32 hi/lo prefill (split, then prefill) and the two-pass decode.
 * Host function, no CUDA call.
 */
SDPA_API int sdpa_last_launch_count(void);

/*
 * sdpa_forward_decode_noalloc — the vector path (decode) without a
 * caller workspace.  The pages have no counterpart: this entry point exists
 * for callers that cannot call cudaMalloc or pass device scratch where they
 * run attention (a stream being captured into a CUDA graph may not
 * allocate, cudaMalloc can synchronise the device, and some hosts own every
 * device byte through their own pool and have none to spare for a library).
 *
 * Same problem description, inputs, outputs, stream and errors as
 * sdpa_forward, restricted to problems that sdpa_select_kernel maps to
 * SDPA_KERNEL_DECODE_SPLITKV (others: SDPA_ERR_UNSUPPORTED; nothing to
 * compute: SDPA_OK).  The split-KV partial results go to one static device
 * array of SDPA_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU loading the
 * library holds until exit; a problem whose partial results do not fit
 * (about B * Hq * Lq * splits * (D + 1) * 4 bytes) returns
 * SDPA_ERR_WORKSPACE_TOO_SMALL before any launch.  Nothing is allocated.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address (cudaGetSymbolAddress) and caches it: make that
 *    first call before any stream capture.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents; calls whose kernels overlap on the GPU race on it, so the
 *    caller must order them (one stream, or events).  Nothing in it needs to
 *    start at zero: each call writes every partial result before reading it.
 */
#define SDPA_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
SDPA_API sdpa_status_t sdpa_forward_decode_noalloc(const sdpa_params_t* params,
                                                   const void* q, const void* k,
                                                   const void* v, void* o, float* lse,
                                                   void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_SDPA_H_ */
