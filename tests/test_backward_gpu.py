"""Parity of the backward pass (sdpa_backward, the tensor-core kernel behind
the C ABI) with the float64 backward oracle on the same rounded inputs.

The GPU path takes the forward's own o and lse (computed on the GPU), as a
training step does; the oracle recomputes everything from q, k, v and dO in
float64.  Gradients are compared relative to their largest magnitude:
max |d - d_ref| <= 2e-2 * max |d_ref| and mean |d - d_ref| <= 2e-3 * max |d_ref|
(fp16/bf16 P and dS enter the products rounded to 8-11 significant bits); for
fp32 inputs (fp32 products and sums; the forward's O within about 4e-6 of the
definition enters through D_i) 2e-4 and 2e-5.
"""
import numpy as np
import pytest

from oracle import oracle as O
from scaled_dot_product_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

REL_MAX, REL_MEAN = 2e-2, 2e-3
REL_MAX_F32, REL_MEAN_F32 = 2e-4, 2e-5


def wl(B, Hq, Hkv, Lq, Lk, D, dtype, **kw):
    name = "bwd_%d_%d_%d_%d_%d_%d_%s" % (B, Hq, Hkv, Lq, Lk, D, dtype)
    return W.Workload(name, B, Hq, Hkv, Lq, Lk, D, dtype, **kw)


def _compare(w, grads, ref):
    f = W.as_float64
    rmax, rmean = (REL_MAX_F32, REL_MEAN_F32) if w.dtype == "float32" else (REL_MAX, REL_MEAN)
    for name, got, want in zip(("dq", "dk", "dv"), grads, ref):
        got = f(got.contiguous().cpu())
        assert np.all(np.isfinite(got)), name + " not finite"
        scale = max(np.max(np.abs(want)), 1e-6)
        err = np.abs(got - want)
        assert err.max() <= rmax * scale, "%s max err %.3g vs %.3g" % (name, err.max(), scale)
        assert err.mean() <= rmean * scale, "%s mean err %.3g vs %.3g" % (name, err.mean(), scale)


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
    _compare(w, (dq, dk, dv), ref)


CASES = {
    "f16_d64": wl(1, 2, 2, 300, 333, 64, "float16"),
    "bf16_d128_causal_gqa": wl(2, 4, 2, 260, 300, 128, "bfloat16", causal=True),
    "bf16_d64_sinks_mask": wl(1, 4, 1, 129, 200, 64, "bfloat16", sinks=True, mask="full"),
    "f16_d128_bool_mask": wl(1, 2, 2, 140, 100, 128, "float16", mask="bool_full"),
    "f16_d64_causal_short_q": wl(1, 2, 1, 64, 1000, 64, "float16", causal=True),
    "bf16_d128_one_query": wl(1, 2, 2, 1, 500, 128, "bfloat16"),
    "f16_d64_key_mask_gqa8": wl(2, 8, 1, 200, 256, 64, "float16", mask="bool_key"),
    # fp32: the CUDA-core kernels (dK/dV per key tile, dQ per query tile)
    "f32_d64_causal_gqa_sinks": wl(2, 4, 2, 150, 200, 64, "float32", causal=True, sinks=True),
    "f32_d128_mask": wl(1, 2, 1, 100, 130, 128, "float32", mask="full"),
    "f32_d64_bool_key_mask": wl(1, 4, 4, 70, 65, 64, "float32", mask="bool_key"),
    "f32_d128_one_query": wl(1, 2, 2, 1, 500, 128, "float32"),
}


def run_lens_case(w, lens_q, lens_kv):
    """Forward and backward with per-batch lengths on the device; the oracle
    sees them as an explicit -inf mask (padding rows and keys, and the
    bottom-right causal rule with each batch's own lengths)."""
    import torch
    import scaled_dot_product_fwd_gb300 as S
    inp = W.make_inputs(w)
    rng = np.random.default_rng(7)
    d_o = torch.from_numpy(rng.standard_normal((w.B, w.Hq, w.Lq, w.D), dtype=np.float32)).to(
        inp["q"].dtype)
    q, k, v, g = (t.cuda() for t in (inp["q"], inp["k"], inp["v"], d_o))
    sinks = None if inp["sinks"] is None else inp["sinks"].cuda()
    tq = torch.tensor(lens_q, dtype=torch.int32, device="cuda")
    tk = torch.tensor(lens_kv, dtype=torch.int32, device="cuda")
    o, lse = S.sdpa_forward(q, k, v, scale=w.scale, causal=w.causal, sinks=sinks, seq_lens_q=tq,
                            seq_lens_kv=tk)
    dq, dk, dv = S.sdpa_backward(q, k, v, o, lse, g, scale=w.scale, causal=w.causal, sinks=sinks,
                                 seq_lens_q=tq, seq_lens_kv=tk)
    torch.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    mask = np.zeros((w.B, w.Hq, w.Lq, w.Lk))
    for b in range(w.B):
        i = np.arange(w.Lq)[:, None]
        j = np.arange(w.Lk)[None, :]
        hide = (i >= lens_q[b]) | (j >= lens_kv[b])
        if w.causal:
            hide |= j > i + (lens_kv[b] - lens_q[b])
        mask[b, :, hide] = -np.inf
    f = W.as_float64
    ref = O.sdpa_backward(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(d_o), w.scale, False, mask,
                          None if inp["sinks"] is None else f(inp["sinks"]))
    _compare(w, (dq, dk, dv), ref)


LEN_CASES = {
    # a batch with no query row, one with few keys; sinks make the LSE of
    # padding rows finite (their P must still be 0)
    "f16_d64_causal_sinks": (wl(3, 4, 2, 200, 300, 64, "float16", causal=True, sinks=True),
                             [200, 77, 0], [300, 129, 5]),
    # one query row seeing no key, one batch at full length
    "bf16_d128": (wl(2, 4, 4, 130, 257, 128, "bfloat16"), [1, 130], [0, 257]),
    "f32_d64_causal_gqa": (wl(2, 4, 2, 90, 140, 64, "float32", causal=True), [90, 33],
                           [140, 64]),
}


@pytest.mark.parametrize("case", sorted(LEN_CASES))
def test_backward_per_batch_lengths(cuda, case):
    w, lens_q, lens_kv = LEN_CASES[case]
    run_lens_case(w, lens_q, lens_kv)


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_matches_oracle(cuda, case):
    run_case(CASES[case])


@pytest.mark.parametrize("case", ["f16_d64", "bf16_d128_causal_gqa", "f32_d64_causal_gqa_sinks"])
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
