"""ctypes binding of the C ABI in include/sdpa.h (argument marshalling only).

Every step of the computation runs in the CUDA kernels of libsdpa_gb300.so;
this module only checks tensor properties, fills ``sdpa_params_t``, hands
device pointers and the current CUDA stream to the library, and turns status
codes into exceptions.  There is no CPU path: if the library cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libsdpa_gb300.so")

SDPA_F32, SDPA_F16, SDPA_BF16 = 0, 1, 2
SDPA_FLAG_SHARED_GPU = 0x1
SDPA_FLAG_BOOL_MASK = 0x2
SDPA_FLAG_STRIDES = 0x4
STATUS = {0: "SDPA_OK", 1: "SDPA_ERR_INVALID_ARGUMENT", 2: "SDPA_ERR_UNSUPPORTED",
          3: "SDPA_ERR_MISALIGNED", 4: "SDPA_ERR_WORKSPACE_TOO_SMALL", 5: "SDPA_ERR_CUDA",
          6: "SDPA_ERR_TIMEOUT"}
KERNELS = {0: "none", 1: "prefill_tc", 2: "prefill_f32", 3: "decode_splitkv", 4: "no_keys",
           5: "prefill_tc_f32"}

# Every symbol include/sdpa.h declares.
EXPORTS = ("sdpa_workspace_size", "sdpa_select_kernel", "sdpa_forward", "sdpa_status_string",
           "sdpa_device_status", "sdpa_debug_set_wait_limit_ns", "sdpa_abi_version",
           "sdpa_forward_decode_noalloc", "sdpa_last_launch_count",
           "sdpa_backward_workspace_size", "sdpa_backward", "sdpa_debug_set_option",
           "sdpa_host_staging_size", "sdpa_forward_host")

# sdpa_debug_option_t
DEBUG_OPTIONS = {"decode_splits": 0, "decode_cluster": 1, "decode_drop_last": 2,
                 "prefill_split": 3, "decode_vector": 4}


class SdpaParams(ctypes.Structure):
    """Mirror of sdpa_params_t."""
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("seq_len_q", ctypes.c_int32),
                ("seq_len_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("causal", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("mask", ctypes.c_void_p), ("mask_stride", ctypes.c_int64 * 4),
                ("sinks", ctypes.c_void_p), ("kv_capacity", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("seq_lens_q", ctypes.c_void_p),
                ("seq_lens_kv", ctypes.c_void_p), ("q_stride", ctypes.c_int64 * 3),
                ("k_stride", ctypes.c_int64 * 3), ("v_stride", ctypes.c_int64 * 3),
                ("o_stride", ctypes.c_int64 * 3)]


class SdpaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__("%s%s" % (STATUS.get(status, str(status)), (": " + what) if what else ""))


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load (once) and return the ctypes handle of libsdpa_gb300.so."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError("libsdpa_gb300.so is not built (run __graft_entry__.build())")
            lib = ctypes.CDLL(path)
            P = ctypes.POINTER(SdpaParams)
            lib.sdpa_workspace_size.argtypes = [P]
            lib.sdpa_workspace_size.restype = ctypes.c_size_t
            lib.sdpa_select_kernel.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
            lib.sdpa_select_kernel.restype = ctypes.c_int
            lib.sdpa_forward.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_size_t, ctypes.c_void_p]
            lib.sdpa_forward.restype = ctypes.c_int
            lib.sdpa_status_string.argtypes = [ctypes.c_int]
            lib.sdpa_status_string.restype = ctypes.c_char_p
            lib.sdpa_device_status.argtypes = [ctypes.c_void_p]
            lib.sdpa_device_status.restype = ctypes.c_int
            lib.sdpa_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            lib.sdpa_debug_set_wait_limit_ns.restype = ctypes.c_uint64
            lib.sdpa_abi_version.restype = ctypes.c_int
            lib.sdpa_debug_set_option.argtypes = [ctypes.c_int, ctypes.c_int]
            lib.sdpa_debug_set_option.restype = ctypes.c_int
            lib.sdpa_last_launch_count.restype = ctypes.c_int
            lib.sdpa_host_staging_size.argtypes = [P, ctypes.c_int]
            lib.sdpa_host_staging_size.restype = ctypes.c_size_t
            lib.sdpa_forward_host.argtypes = [P] + [ctypes.c_void_p] * 6 + [
                ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
            lib.sdpa_forward_host.restype = ctypes.c_int
            lib.sdpa_forward_decode_noalloc.argtypes = [P] + [ctypes.c_void_p] * 6
            lib.sdpa_forward_decode_noalloc.restype = ctypes.c_int
            lib.sdpa_backward_workspace_size.argtypes = [P]
            lib.sdpa_backward_workspace_size.restype = ctypes.c_size_t
            lib.sdpa_backward.argtypes = [P] + [ctypes.c_void_p] * 10 + [ctypes.c_size_t,
                                                                         ctypes.c_void_p]
            lib.sdpa_backward.restype = ctypes.c_int
            _lib = lib
    return _lib


def make_params(B, Hq, Hkv, Lq, Lk, D, dtype, scale, causal=False, mask_ptr=None,
                mask_stride=(0, 0, 0, 1), sinks_ptr=None, kv_capacity=0, seq_lens_q_ptr=None,
                seq_lens_kv_ptr=None, flags=0, strides=None) -> SdpaParams:
    """strides: None, or element strides (batch, head, row) of q, k, v and o
    as four 3-tuples; sets SDPA_FLAG_STRIDES."""
    p = SdpaParams()
    p.batch, p.num_q_heads, p.num_kv_heads = int(B), int(Hq), int(Hkv)
    p.seq_len_q, p.seq_len_kv, p.head_dim = int(Lq), int(Lk), int(D)
    p.dtype = int(dtype)
    p.scale = float(scale)
    p.causal = 1 if causal else 0
    p.reserved0 = 0
    p.mask = mask_ptr
    for i in range(4):
        p.mask_stride[i] = int(mask_stride[i])
    p.sinks = sinks_ptr
    p.kv_capacity = int(kv_capacity)
    p.flags = int(flags)
    if strides is not None:
        p.flags |= SDPA_FLAG_STRIDES
        for field, st in zip(("q_stride", "k_stride", "v_stride", "o_stride"), strides):
            arr = getattr(p, field)
            for i in range(3):
                arr[i] = int(st[i])
    p.seq_lens_q = seq_lens_q_ptr
    p.seq_lens_kv = seq_lens_kv_ptr
    return p


def sdpa_status_string(status: int) -> str:
    return load_library().sdpa_status_string(int(status)).decode()


def sdpa_select_kernel(params: SdpaParams):
    """Returns (kernel name, status code) for a params struct."""
    st = ctypes.c_int(0)
    k = load_library().sdpa_select_kernel(ctypes.byref(params), ctypes.byref(st))
    return KERNELS.get(k, str(k)), st.value


def sdpa_workspace_size(params: SdpaParams) -> int:
    return int(load_library().sdpa_workspace_size(ctypes.byref(params)))


def sdpa_forward_raw(params: SdpaParams, q, k, v, o, lse, workspace, workspace_bytes, stream) -> int:
    """Direct call of the C entry point with integer device addresses."""
    pp = ctypes.byref(params) if params is not None else None
    return int(load_library().sdpa_forward(pp, q, k, v, o, lse, workspace,
                                           int(workspace_bytes), stream))


def sdpa_forward_decode_noalloc_raw(params: SdpaParams, q, k, v, o, lse, stream) -> int:
    """Direct call of the allocation-free decode entry point (integer device
    addresses; partial results in the library's static device scratch)."""
    pp = ctypes.byref(params) if params is not None else None
    return int(load_library().sdpa_forward_decode_noalloc(pp, q, k, v, o, lse, stream))


def sdpa_backward_raw(params: SdpaParams, q, k, v, o, d_o, lse, dq, dk, dv, workspace,
                      workspace_bytes, stream) -> int:
    """Direct call of the backward entry point with integer device addresses."""
    pp = ctypes.byref(params) if params is not None else None
    return int(load_library().sdpa_backward(pp, q, k, v, o, d_o, lse, dq, dk, dv, workspace,
                                            int(workspace_bytes), stream))


def sdpa_backward_workspace_size(params: SdpaParams) -> int:
    return int(load_library().sdpa_backward_workspace_size(ctypes.byref(params)))


def sdpa_backward(q, k, v, o, lse, d_o, scale=None, causal=False, mask=None, sinks=None,
                  dq=None, dk=None, dv=None, workspace=None, stream=None, seq_lens_q=None,
                  seq_lens_kv=None):
    """dQ, dK, dV of sdpa_forward on the GPU (fp32/fp16/bf16, head_dim 64 or
    128).

    q, k, v, mask, sinks, scale, causal and the per-batch lengths
    (seq_lens_q, seq_lens_kv: int32 CUDA tensors of B elements) as given to
    sdpa_forward; o and lse its outputs; d_o the gradient of the loss with
    respect to o (o's shape and dtype).  Tensors need a contiguous last
    dimension; dq, dk, dv default to the layouts of q, k, v.  dk and dv sum
    over the query heads of each kv head; rows past a batch's lengths get
    zero gradients.  Returns (dq, dk, dv).
    """
    torch = _torch()
    for t in (q, k, v, o, d_o):
        if t.dim() != 4 or not t.is_cuda or t.stride(-1) != 1:
            raise ValueError("q, k, v, o, d_o must be 4-D CUDA tensors with a contiguous last "
                             "dimension")
    if not (q.dtype == k.dtype == v.dtype == o.dtype == d_o.dtype):
        raise TypeError("q, k, v, o, d_o must share a dtype")
    B, Hq, Lq, D = q.shape
    _, Hkv, Lk, _ = k.shape
    if v.shape != k.shape or o.shape != q.shape or d_o.shape != q.shape:
        raise ValueError("shape mismatch")
    if lse is None or lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Lq) \
            or not lse.is_contiguous():
        raise ValueError("lse must be the forward's contiguous float32 [B, Hq, Lq] output")
    if d_o.stride() != o.stride():
        raise ValueError("d_o must have o's layout (strides)")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    flags = 0
    mask_ptr, mstride = None, (0, 0, 0, 1)
    if mask is not None:
        if (mask.dtype != q.dtype and mask.dtype != torch.bool) or mask.device != q.device:
            raise TypeError("mask must have q's dtype (or bool) and q's device")
        if mask.dtype == torch.bool:
            flags |= SDPA_FLAG_BOOL_MASK
        mexp = mask.expand(B, Hq, Lq, Lk)
        mstride = tuple(int(s) for s in mexp.stride())
        if Lk == 1:
            mstride = mstride[:3] + (1,)
        mask_ptr = mexp.data_ptr()
    sinks_ptr = None
    if sinks is not None:
        if sinks.dtype != torch.float32 or not sinks.is_cuda or sinks.numel() != Hq:
            raise TypeError("sinks must be a float32 CUDA tensor with Hq elements")
        sinks = sinks.contiguous()
        sinks_ptr = sinks.data_ptr()
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for g, t in ((dq, q), (dk, k), (dv, v)):
        if g.shape != t.shape or g.dtype != t.dtype or g.stride() != t.stride():
            raise ValueError("dq, dk, dv must have the shapes, dtype and layouts of q, k, v")
    lens = []
    for t in (seq_lens_q, seq_lens_kv):
        if t is not None:
            if t.dtype != torch.int32 or not t.is_cuda or t.numel() != B:
                raise TypeError("seq_lens_q / seq_lens_kv must be int32 CUDA tensors of B elements")
            t = t.contiguous()
        lens.append(t)
    strides = tuple(tuple(int(s) for s in t.stride()[:3]) for t in (q, k, v, o))
    params = make_params(B, Hq, Hkv, Lq, Lk, D, dtype_code(q.dtype), scale, causal, mask_ptr,
                         mstride, sinks_ptr, flags=flags, strides=strides,
                         seq_lens_q_ptr=None if lens[0] is None else lens[0].data_ptr(),
                         seq_lens_kv_ptr=None if lens[1] is None else lens[1].data_ptr())
    nbytes = sdpa_backward_workspace_size(params)
    if workspace is None and nbytes > 0:
        workspace = _workspace(nbytes, q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    st = sdpa_backward_raw(params, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           d_o.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                           dv.data_ptr(), ws_ptr, ws_bytes, stream)
    if st != 0:
        raise SdpaError(st, sdpa_status_string(st))
    return dq, dk, dv


def sdpa_device_status(stream=None) -> int:
    return int(load_library().sdpa_device_status(stream))


def sdpa_debug_set_wait_limit_ns(ns: int) -> int:
    return int(load_library().sdpa_debug_set_wait_limit_ns(int(ns)))


def sdpa_debug_set_option(option, value: int) -> int:
    """Set a test hook of the library (a DEBUG_OPTIONS name or its number);
    returns the previous value."""
    code = DEBUG_OPTIONS[option] if isinstance(option, str) else int(option)
    prev = int(load_library().sdpa_debug_set_option(code, int(value)))
    if prev == -1 and not 0 <= code < len(DEBUG_OPTIONS):
        raise ValueError("unknown debug option %r" % (option,))
    return prev


def sdpa_abi_version() -> int:
    return int(load_library().sdpa_abi_version())


def sdpa_last_launch_count() -> int:
    """Kernels enqueued by this thread's last sdpa_forward call (C ABI)."""
    return int(load_library().sdpa_last_launch_count())


# ----------------------------------------------------------------- torch layer
_ws_cache = {}


def _torch():
    import torch
    return torch


def dtype_code(t) -> int:
    torch = _torch()
    m = {torch.float32: SDPA_F32, torch.float16: SDPA_F16, torch.bfloat16: SDPA_BF16}
    if t not in m:
        raise TypeError("unsupported dtype %s" % t)
    return m[t]


def _workspace(nbytes: int, device):
    torch = _torch()
    key = (device.index, threading.get_ident())
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def sdpa_forward(q, k, v, scale=None, causal=False, mask=None, sinks=None, out=None,
                 lse=None, return_lse=True, workspace=None, stream=None, kv_len=None,
                 seq_lens_q=None, seq_lens_kv=None, shared_gpu=False):
    """O (and LSE) of softmax(scale * q k^T + mask [+ sinks]) v on the GPU.

    q [B, Hq, Lq, D], k/v [B, Hkv, C, D]: CUDA tensors of one dtype (float32,
    float16 or bfloat16) whose last dimension is contiguous; any strides of
    the other dimensions (multiples of 16 bytes), e.g. a [B, L, H, D] tensor
    seen through .transpose(1, 2).  The keys are rows [0, Lk) of k and v, Lk
    = kv_len (default C: with kv_len < C, k and v are a fixed-capacity KV
    cache).  out defaults to q's layout.  mask: None, a tensor of q's dtype
    broadcastable to [B, Hq, Lq, Lk] (additive), or a bool tensor of that
    shape (True = the key is visible).  sinks: None or float32 [Hq].  seq_lens_q,
    seq_lens_kv: None or int32 CUDA tensors [B] of per-batch lengths (padding
    masks; rows past a batch's query length see no key).  scale defaults to
    1/sqrt(D).  shared_gpu: the call runs beside other kernels (sets
    SDPA_FLAG_SHARED_GPU: launch shapes not fitted to an idle GPU).  Returns
    (o, lse) or o.
    """
    torch = _torch()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, L, D]")
    for t in (q, k, v):
        if not t.is_cuda:
            raise ValueError("q, k, v must be CUDA tensors")
        if t.stride(-1) != 1:
            raise ValueError("the last dimension of q, k, v must be contiguous")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share a dtype")
    B, Hq, Lq, D = q.shape
    _, Hkv, cap, _ = k.shape
    if v.shape != k.shape:
        raise ValueError("k and v must have one shape")
    Lk = cap if kv_len is None else int(kv_len)
    if Lk < 0 or Lk > cap:
        raise ValueError("kv_len must be within [0, k.shape[2]]")
    lens = []
    for t in (seq_lens_q, seq_lens_kv):
        if t is not None:
            if t.dtype != torch.int32 or not t.is_cuda or t.numel() != B or not t.is_contiguous():
                raise TypeError("seq_lens_q / seq_lens_kv must be contiguous int32 CUDA "
                                "tensors with B elements")
            lens.append(t.data_ptr())
        else:
            lens.append(None)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dt = dtype_code(q.dtype)
    mask_ptr, mstride = None, (0, 0, 0, 1)
    flags = SDPA_FLAG_SHARED_GPU if shared_gpu else 0
    if mask is not None:
        if (mask.dtype != q.dtype and mask.dtype != torch.bool) or mask.device != q.device:
            raise TypeError("mask must have q's dtype (or bool) and q's device")
        if mask.dtype == torch.bool:
            flags |= SDPA_FLAG_BOOL_MASK
        mexp = mask.expand(B, Hq, Lq, Lk)
        mstride = tuple(int(s) for s in mexp.stride())
        if Lk == 1:
            mstride = mstride[:3] + (1,)
        mask_ptr = mexp.data_ptr()
    sinks_ptr = None
    if sinks is not None:
        if sinks.dtype != torch.float32 or not sinks.is_cuda or sinks.numel() != Hq:
            raise TypeError("sinks must be a float32 CUDA tensor with Hq elements")
        sinks = sinks.contiguous()
        sinks_ptr = sinks.data_ptr()
    if out is None:
        out = torch.empty_like(q)  # q's layout (a dense permutation stays one)
    elif (tuple(out.shape) != (B, Hq, Lq, D) or out.dtype != q.dtype or not out.is_cuda
          or out.stride(-1) != 1):
        raise ValueError("out must be a CUDA tensor like q with a contiguous last dimension")
    dense = all(t.is_contiguous() for t in (q, k, v, out))
    strides = None if dense else tuple(tuple(int(s) for s in t.stride()[:3])
                                       for t in (q, k, v, out))
    params = make_params(B, Hq, Hkv, Lq, Lk, D, dt, scale, causal, mask_ptr, mstride, sinks_ptr,
                         kv_capacity=cap if (dense and cap != Lk) else 0, seq_lens_q_ptr=lens[0],
                         seq_lens_kv_ptr=lens[1], flags=flags, strides=strides)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    nbytes = sdpa_workspace_size(params)
    if workspace is None and nbytes > 0:
        workspace = _workspace(nbytes, q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    st = sdpa_forward_raw(params, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr() if lse is not None else None, ws_ptr, ws_bytes, stream)
    if st != 0:
        raise SdpaError(st, sdpa_status_string(st))
    return (out, lse) if return_lse else out


# --------------------------------------------------- host-buffer entry point
_host_cache = {}


def sdpa_host_staging_size(params, pieces: int) -> int:
    return int(load_library().sdpa_host_staging_size(ctypes.byref(params), int(pieces)))


def sdpa_forward_host(q, k, v, scale=None, causal=False, mask=None, sinks=None, out=None,
                      lse=None, chunks=8, device=None):
    """sdpa_forward on host tensors through the C call sdpa_forward_host.

    q [B, Hq, Lq, D] and k/v [B, Hkv, Lk, D] are contiguous CPU tensors of one
    dtype (pinned, so that the copies overlap the kernels); mask and sinks,
    if given, are CUDA tensors as for sdpa_forward.  The library cuts the
    (batch, kv-head) pairs into about `chunks` pieces and overlaps each
    piece's copies with the others' kernels on its own streams, forked from
    and joined back to the current stream of `device`; the results (`out`,
    `lse` or new pinned tensors, returned) are complete once that stream
    reaches the end of the call, e.g. after torch.cuda.synchronize().  This
    function only allocates the device staging area (cached per device,
    size and stream: calls on different streams never share one).
    """
    torch = _torch()
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous host tensors")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share a dtype")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, L, D]")
    if device is None:
        device = torch.device("cuda", torch.cuda.current_device())
    B, Hq, Lq, D = q.shape
    _, Hkv, Lk, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, pin_memory=True)
    for t in (out, lse):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("out and lse must be contiguous host tensors")
    mask_ptr, mstride, flags = None, (0, 0, 0, 1), 0
    if mask is not None:
        if (mask.dtype != q.dtype and mask.dtype != torch.bool) or not mask.is_cuda:
            raise TypeError("mask must have q's dtype (or bool) and live on the GPU")
        if mask.dtype == torch.bool:
            flags |= SDPA_FLAG_BOOL_MASK
        mexp = mask.expand(B, Hq, Lq, Lk)
        if mexp.stride(3) != 1:
            raise ValueError("mask must be contiguous along the key dimension")
        mask_ptr, mstride = mexp.data_ptr(), tuple(mexp.stride())
    sinks_ptr = None
    if sinks is not None:
        if sinks.dtype != torch.float32 or not sinks.is_cuda or sinks.numel() != Hq:
            raise TypeError("sinks must be a float32 CUDA tensor of Hq values")
        sinks_ptr = sinks.data_ptr()
    params = make_params(B, Hq, Hkv, Lq, Lk, D, dtype_code(q.dtype), scale, causal, mask_ptr,
                         mstride, sinks_ptr)
    params.flags |= flags
    pieces = max(1, int(chunks))
    nbytes = sdpa_host_staging_size(params, pieces)
    if nbytes == 0:
        raise SdpaError(2, "problem not supported by sdpa_forward_host")
    stream = torch.cuda.current_stream(device)
    key = (device.index, nbytes, stream.cuda_stream)
    buf = _host_cache.get(key)
    if buf is None:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _host_cache[key] = buf
    st = load_library().sdpa_forward_host(ctypes.byref(params), q.data_ptr(), k.data_ptr(),
                                          v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                          buf.data_ptr(), nbytes, pieces, stream.cuda_stream)
    if st != 0:
        raise SdpaError(st, sdpa_status_string(st))
    return out, lse
