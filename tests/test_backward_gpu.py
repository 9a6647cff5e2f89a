"""Parity of the backward pass (sdpa_backward, the tensor-core kernel behind
the C ABI) with the float64 backward oracle on the same rounded inputs.

The GPU path takes the forward's own o and lse (computed on the GPU), as a
training step does; the oracle recomputes everything from q, k, v and dO in
float64.  Gradients are compared relative to their largest magnitude:
max |d - d_ref| <= 2e-2 * max |d_ref| and mean |d - d_ref| <= 2e-3 * max |d_ref|
(fp16/bf16 P and dS enter the products rounded to 8-11 significant bits).
"""
import numpy as np
import pytest

from oracle import oracle as O
from scaled_dot_product_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

REL_MAX, REL_MEAN = 2e-2, 2e-3


def wl(B, Hq, Hkv, Lq, Lk, D, dtype, **kw):
    name = "bwd_%d_%d_%d_%d_%d_%d_%s" % (B, Hq, Hkv, Lq, Lk, D, dtype)
    return W.Workload(name, B, Hq, Hkv, Lq, Lk, D, dtype, **kw)


def run_case(w, layout="dense"):
    import torch
    import scaled_dot_product_fwd_gb300 as S
    inp = W.make_inputs(w)
    rng = np.random.default_rng(99)
    d_o = torch.from_numpy(rng.standard_normal((w.B, w.Hq, w.Lq, w.D), dtype=np.float32)).to(
        inp["q"].dtype)
    q, k, v, g = (t.cuda() for t in (inp["q"], inp["k"], inp["v"], d_o))
    if layout == "bshd":
        q, k, v, g = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (q, k, v, g))
    mask = None if inp["mask"] is None else inp["mask"].cuda()
    sinks = None if inp["sinks"] is None else inp["sinks"].cuda()
    o, lse = S.sdpa_forward(q, k, v, scale=w.scale, causal=w.causal, mask=mask, sinks=sinks)
    if layout == "bshd":
        assert g.stride() == o.stride()
    dq, dk, dv = S.sdpa_backward(q, k, v, o, lse, g, scale=w.scale, causal=w.causal, mask=mask,
                                 sinks=sinks)
    torch.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    f = W.as_float64
    m = inp["mask"]
    if m is not None:
        m = m.numpy() if m.dtype == torch.bool else f(m)
    ref = O.sdpa_backward(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(d_o), w.scale, w.causal, m,
                          None if inp["sinks"] is None else f(inp["sinks"]))
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        got = f(got.contiguous().cpu())
        assert np.all(np.isfinite(got)), name + " not finite"
        scale = max(np.max(np.abs(want)), 1e-6)
        err = np.abs(got - want)
        assert err.max() <= REL_MAX * scale, "%s max err %.3g vs %.3g" % (name, err.max(), scale)
        assert err.mean() <= REL_MEAN * scale, "%s mean err %.3g vs %.3g" % (name, err.mean(), scale)


CASES = {
    "f16_d64": wl(1, 2, 2, 300, 333, 64, "float16"),
    "bf16_d128_causal_gqa": wl(2, 4, 2, 260, 300, 128, "bfloat16", causal=True),
    "bf16_d64_sinks_mask": wl(1, 4, 1, 129, 200, 64, "bfloat16", sinks=True, mask="full"),
    "f16_d128_bool_mask": wl(1, 2, 2, 140, 100, 128, "float16", mask="bool_full"),
    "f16_d64_causal_short_q": wl(1, 2, 1, 64, 1000, 64, "float16", causal=True),
    "bf16_d128_one_query": wl(1, 2, 2, 1, 500, 128, "bfloat16"),
    "f16_d64_key_mask_gqa8": wl(2, 8, 1, 200, 256, 64, "float16", mask="bool_key"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_matches_oracle(cuda, case):
    run_case(CASES[case])


@pytest.mark.parametrize("case", ["f16_d64", "bf16_d128_causal_gqa"])
def test_backward_strided_layouts(cuda, case):
    run_case(CASES[case], layout="bshd")


def test_backward_empty_sides(cuda):
    """No key: dQ = 0.  No query row: dK = dV = 0."""
    import torch
    import scaled_dot_product_fwd_gb300 as S
    q = torch.randn(1, 2, 5, 64, device="cuda", dtype=torch.float16)
    kk = torch.zeros(1, 2, 0, 64, device="cuda", dtype=torch.float16)
    o, lse = S.sdpa_forward(q, kk, kk)
    dq, dk, dv = S.sdpa_backward(q, kk, kk, o, lse, torch.randn_like(q))
    torch.cuda.synchronize()
    assert torch.all(dq == 0)
    k = torch.randn(1, 2, 70, 64, device="cuda", dtype=torch.float16)
    q0 = torch.zeros(1, 2, 0, 64, device="cuda", dtype=torch.float16)
    lse0 = torch.zeros(1, 2, 0, device="cuda")
    dk = torch.full_like(k, 5.0)
    dv = torch.full_like(k, 5.0)
    S.sdpa_backward(q0, k, k, q0, lse0, q0, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)
