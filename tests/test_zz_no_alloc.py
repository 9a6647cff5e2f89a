"""The allocation-free decode entry point, sdpa_forward_decode_noalloc.

It serves callers that cannot call cudaMalloc or pass device scratch where
they run attention (a stream under CUDA-graph capture, hosts whose device
memory is all owned by their own pool).  Its partial results live in a
static device array inside the library instead of a caller workspace.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It must pass both alone in
a fresh process and after the other tests (the static array keeps the last
call's contents, which must not matter).
"""
import ctypes

import numpy as np
import pytest

from scaled_dot_product_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"float32": 1e-4, "float16": 2e-2, "bfloat16": 2e-2}
LSE_TOL = 1e-3
SCRATCH_BYTES = 8 * 1024 * 1024


def _lib():
    import scaled_dot_product_fwd_gb300 as S
    lib = S.load_library()
    return S, lib


def _params(S, w, sinks_ptr):
    import torch
    dt = {"float32": S.SDPA_F32, "float16": S.SDPA_F16, "bfloat16": S.SDPA_BF16}[w.dtype]
    return S.make_params(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D, dt, w.scale, w.causal,
                         None, (0, 0, 0, 1), sinks_ptr)


CASES = [W.DECODE_D512[(2, "bfloat16", True)], W.DECODE_D512[(1, "float32", False)],
         W.Workload("noalloc_d128_g4", 4, 16, 4, 1, 5000, 128, "float16", sinks=True)]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_sdpa_forward_twice(cuda, w):
    torch = cuda
    S, lib = _lib()
    inp = W.make_inputs(w)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    sinks = inp["sinks"].cuda() if inp["sinks"] is not None else None
    p = _params(S, w, sinks.data_ptr() if sinks is not None else None)
    assert S.sdpa_workspace_size(p) <= SCRATCH_BYTES
    # the existing entry point, with a caller workspace
    o_ref, lse_ref = S.sdpa_forward(q, k, v, scale=w.scale, sinks=sinks)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # two calls in a row share the static scratch
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        st = lib.sdpa_forward_decode_noalloc(ctypes.byref(p), q.data_ptr(), k.data_ptr(),
                                             v.data_ptr(), o.data_ptr(), lse.data_ptr(), stream)
        assert st == 0, S.sdpa_status_string(st)
        torch.cuda.synchronize()
        assert S.sdpa_device_status() == 0
        d_o = (o.double() - o_ref.double()).abs().max().item()
        d_l = (lse.double() - lse_ref.double()).abs().max().item()
        assert np.isfinite(d_o) and d_o <= TOL[w.dtype], (call, d_o)
        assert np.isfinite(d_l) and d_l <= LSE_TOL, (call, d_l)


def test_noalloc_rejects_problems_beyond_scratch(cuda):
    torch = cuda
    S, lib = _lib()
    # partial results of B * Hq * splits * (D + 1) floats exceed 8 MiB
    p = S.make_params(64, 64, 8, 1, 65536, 512, S.SDPA_BF16, 0.0441941738)
    assert S.sdpa_workspace_size(p) > SCRATCH_BYTES
    st = lib.sdpa_forward_decode_noalloc(ctypes.byref(p), 256, 256, 256, 256, None,
                                         torch.cuda.current_stream().cuda_stream)
    assert st == 4  # SDPA_ERR_WORKSPACE_TOO_SMALL, before any launch
    # shapes outside the decode path are refused, not served another way
    p2 = S.make_params(1, 4, 4, 16, 64, 128, S.SDPA_BF16, 0.088)
    st = lib.sdpa_forward_decode_noalloc(ctypes.byref(p2), 256, 256, 256, 256, None, None)
    assert st == 2  # SDPA_ERR_UNSUPPORTED
