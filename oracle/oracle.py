"""Python access to the float64 CPU oracle (oracle/sdpa_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The library
(``scaled_dot_product_fwd_gb300``) never imports it, and the oracle shares no
code with the CUDA path.

Every array handed to the oracle is float64.  Inputs stored as fp16/bf16/fp32
are widened exactly (every such value is a double) before the call, so the
oracle sees the same values the GPU reads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_d = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64
_pi64 = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/liboracle.so (gcc, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    args = [_i64] * 6 + [ctypes.c_double, ctypes.c_int, _d, _d, _d, _d,
                         _pi64, _d, _pi64, _i64, _d, _d]
    lib.oracle_sdpa.argtypes = args + [_d]
    lib.oracle_sdpa.restype = ctypes.c_int
    lib.oracle_sdpa_online.argtypes = args + [_i64]
    lib.oracle_sdpa_online.restype = ctypes.c_int
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def compile_variant(src_text: str, out_path: str) -> "OracleLib":
    """Compile C source text (a variant of the oracle) and bind it.  Used by
    the tests that plant mistakes in a copy of the oracle to show the pins
    catch them."""
    src = out_path[:-3] + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-fno-fast-math", "-ffp-contract=off", src, "-o", out_path, "-lm"],
                   check=True)
    return OracleLib(_bind(ctypes.CDLL(out_path)))


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_d)


def _prepare(q, k, v, mask, sinks, rows):
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, L, D]")
    B, Hq, Lq, D = q.shape
    _, Hkv, Lk, _ = k.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("shape mismatch")
    mstride = None
    if mask is not None:
        mask = np.asarray(mask)
        if mask.dtype == np.bool_:
            # A boolean mask keeps the keys it marks True and removes the
            # others (mlx 0.30.7 scaled_dot_product_attention.cpp: the CUDA
            # backend declares no boolean-mask support, so a boolean mask
            # reaches it as the additive mask 0 / -inf).
            mask = np.where(mask, 0.0, -np.inf)
        mask = np.ascontiguousarray(mask, dtype=np.float64)
        view = np.broadcast_to(mask, (B, Hq, Lq, Lk))
        mstride = np.array([s // 8 for s in view.strides], dtype=np.int64)
        # the view shares mask's buffer; strides are 0 on broadcast dims
    if sinks is not None:
        sinks = np.ascontiguousarray(sinks, dtype=np.float64).reshape(Hq)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
    return q, k, v, mask, mstride, sinks, rows, (B, Hq, Hkv, Lq, Lk, D)


class OracleLib:
    """One loaded build of the oracle."""

    def __init__(self, lib):
        self.lib = lib

    def sdpa(self, q, k, v, scale, causal=False, mask=None, sinks=None, rows=None,
             want_probs=False):
        """Plain-definition oracle.

        Returns (o, lse) or (o, lse, probs).  With ``rows`` (flat ids
        ``(b*Hq + h)*Lq + i``) o is [len(rows), D], lse [len(rows)] and probs
        [len(rows), Lk]; without, o is [B, Hq, Lq, D], lse [B, Hq, Lq] and probs
        [B, Hq, Lq, Lk].
        """
        q, k, v, mask, mstride, sinks, rows, dims = _prepare(q, k, v, mask, sinks, rows)
        B, Hq, Hkv, Lq, Lk, D = dims
        n = B * Hq * Lq if rows is None else rows.size
        o = np.empty((n, D), np.float64)
        lse = np.empty((n,), np.float64)
        probs = np.empty((n, Lk), np.float64) if want_probs else None
        rc = self.lib.oracle_sdpa(B, Hq, Hkv, Lq, Lk, D, float(scale), int(bool(causal)),
                                 _ptr(q), _ptr(k), _ptr(v), _ptr(mask),
                                 None if mstride is None else mstride.ctypes.data_as(_pi64),
                                 _ptr(sinks),
                                 None if rows is None else rows.ctypes.data_as(_pi64),
                                 n, _ptr(o), _ptr(lse), _ptr(probs))
        if rc != 0:
            raise ValueError("oracle_sdpa rejected its arguments")
        if rows is None:
            o = o.reshape(B, Hq, Lq, D)
            lse = lse.reshape(B, Hq, Lq)
            if probs is not None:
                probs = probs.reshape(B, Hq, Lq, Lk)
        return (o, lse, probs) if want_probs else (o, lse)


    def sdpa_online(self, q, k, v, scale, tile, causal=False, mask=None, sinks=None, rows=None):
        """Tiled online-softmax recurrence with key tiles of width ``tile``."""
        q, k, v, mask, mstride, sinks, rows, dims = _prepare(q, k, v, mask, sinks, rows)
        B, Hq, Hkv, Lq, Lk, D = dims
        n = B * Hq * Lq if rows is None else rows.size
        o = np.empty((n, D), np.float64)
        lse = np.empty((n,), np.float64)
        rc = self.lib.oracle_sdpa_online(B, Hq, Hkv, Lq, Lk, D, float(scale), int(bool(causal)),
                                        _ptr(q), _ptr(k), _ptr(v), _ptr(mask),
                                        None if mstride is None else mstride.ctypes.data_as(_pi64),
                                        _ptr(sinks),
                                        None if rows is None else rows.ctypes.data_as(_pi64),
                                        n, _ptr(o), _ptr(lse), int(tile))
        if rc != 0:
            raise ValueError("oracle_sdpa_online rejected its arguments")
        if rows is None:
            o = o.reshape(B, Hq, Lq, D)
            lse = lse.reshape(B, Hq, Lq)
        return o, lse


def default() -> OracleLib:
    return OracleLib(_load())


def sdpa(*args, **kw):
    """Plain-definition oracle; see OracleLib.sdpa."""
    return default().sdpa(*args, **kw)


def sdpa_online(*args, **kw):
    """Tiled online-softmax recurrence; see OracleLib.sdpa_online."""
    return default().sdpa_online(*args, **kw)


def sdpa_backward(q, k, v, d_o, scale, causal=False, mask=None, sinks=None):
    """Gradients dQ, dK, dV of the attention forward, written out from the
    plain definition in float64 (the backward kernels of the rustytorch
    flash_attention.metal page: P recomputed as exp(S - LSE), D_i = dO_i . O_i,
    dS = P * (dO V^T - D), dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO;
    the options are those of the mlx 0.30.7 cuDNN backward graph: attention
    scale, bottom-right causal mask, additive bias, sink token).

    q [B, Hq, Lq, D], k, v [B, Hkv, Lk, D], d_o [B, Hq, Lq, D]; mask as for
    sdpa (additive, broadcastable, or boolean); sinks [Hq] or None.  The sink
    is a logit with a zero value row: it enters the denominator, so P and the
    gradients of q, k, v account for it; no gradient is returned for it, nor
    for the mask.  Query heads h read kv head h // (Hq / Hkv); dK and dV sum
    over the heads of a group.  Rows that see no key (and no sink) have
    P = 0.  Returns (dq, dk, dv) as float64 arrays.
    """
    q, k, v, mask, _, sinks, _, (B, Hq, Hkv, Lq, Lk, D) = _prepare(q, k, v, mask, sinks, None)
    d_o = np.ascontiguousarray(d_o, dtype=np.float64)
    G = Hq // Hkv
    kk = np.repeat(k, G, axis=1)  # [B, Hq, Lk, D]: the kv head of every query head
    vv = np.repeat(v, G, axis=1)
    s = scale * np.matmul(q, np.swapaxes(kk, -1, -2))  # [B, Hq, Lq, Lk]
    if mask is not None:
        s = s + np.broadcast_to(mask, s.shape)
    if causal:
        vis = np.tril(np.ones((Lq, Lk), bool), k=Lk - Lq)  # key j visible iff j <= i + Lk - Lq
        s = np.where(vis, s, -np.inf)
    # log-sum-exp over the keys and the sink logit
    parts = [s]
    if sinks is not None:
        parts.append(np.broadcast_to(sinks.reshape(1, Hq, 1, 1), (B, Hq, Lq, 1)))
    full = np.concatenate(parts, axis=-1)
    mx = np.max(full, axis=-1, keepdims=True)
    seen = np.isfinite(mx)
    mx_safe = np.where(seen, mx, 0.0)
    with np.errstate(divide="ignore"):  # rows that see nothing: log 0, unused below
        lse = mx_safe + np.log(np.sum(np.exp(full - mx_safe), axis=-1, keepdims=True))
    p = np.where(seen, np.exp(s - np.where(seen, lse, 0.0)), 0.0)  # [B, Hq, Lq, Lk]
    o = np.matmul(p, vv)
    dv_h = np.matmul(np.swapaxes(p, -1, -2), d_o)  # per query head
    dp = np.matmul(d_o, np.swapaxes(vv, -1, -2))
    dvec = np.sum(d_o * o, axis=-1, keepdims=True)
    ds = p * (dp - dvec)
    dq = scale * np.matmul(ds, kk)
    dk_h = scale * np.matmul(np.swapaxes(ds, -1, -2), q)
    dk = dk_h.reshape(B, Hkv, G, Lk, D).sum(axis=2)
    dv = dv_h.reshape(B, Hkv, G, Lk, D).sum(axis=2)
    return dq, dk, dv
