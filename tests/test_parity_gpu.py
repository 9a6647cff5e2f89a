"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs.

Bars (from the method's statement of accuracy): max |dO| <= 1e-4 for fp32 and
<= 2e-2 for fp16/bf16, mean |dO| <= 2e-3, |dLSE| <= 1e-3 on finite entries;
non-finite LSE entries (fully masked rows) must match exactly and O must be
exactly 0 there.  Small cases compare every element; the full-size workloads
compare sampled rows (every row of a few (b, h) pairs' ragged tails plus
seeded random rows) that the oracle evaluates one by one.
"""
import os

import numpy as np
import pytest

from oracle import oracle as O
from scaled_dot_product_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"float32": 1e-4, "float16": 2e-2, "bfloat16": 2e-2}
MEAN_TOL = 2e-3
LSE_TOL = 1e-3


def to_dev(t, torch):
    return None if t is None else t.to("cuda")


def run_gpu(torch, w, inp):
    import scaled_dot_product_fwd_gb300 as S
    q, k, v = (to_dev(inp[x], torch) for x in ("q", "k", "v"))
    o, lse = S.sdpa_forward(q, k, v, scale=w.scale, causal=w.causal,
                            mask=to_dev(inp["mask"], torch), sinks=to_dev(inp["sinks"], torch))
    torch.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    return o.cpu(), lse.cpu()


def oracle_rows(w, inp, rows):
    f = W.as_float64
    mask = inp["mask"]
    if mask is not None:  # boolean masks go to the oracle as booleans
        mask = mask.numpy() if mask.dtype == __import__("torch").bool else f(mask)
    sinks = None if inp["sinks"] is None else f(inp["sinks"])
    return O.sdpa(f(inp["q"]), f(inp["k"]), f(inp["v"]), w.scale, w.causal, mask, sinks,
                  rows=rows)


def compare(w, o_gpu, lse_gpu, o_ref, lse_ref, rows):
    D = w.D
    og = W.as_float64(o_gpu).reshape(-1, D)
    lg = lse_gpu.double().numpy().reshape(-1)
    if rows is not None:
        og, lg = og[rows], lg[rows]
    o_ref = o_ref.reshape(-1, D)
    lse_ref = lse_ref.reshape(-1)
    assert np.all(np.isfinite(og)), "non-finite output"
    err = np.abs(og - o_ref)
    tol = TOL[w.dtype]
    assert err.max() <= tol, "max |dO| %.3g > %.3g" % (err.max(), tol)
    assert err.mean() <= MEAN_TOL, "mean |dO| %.3g" % err.mean()
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin), "LSE finiteness differs"
    assert np.array_equal(lg[~fin], lse_ref[~fin])
    assert np.all(og[~fin] == 0)
    if fin.any():
        lerr = np.abs(lg[fin] - lse_ref[fin]).max()
        assert lerr <= LSE_TOL, "max |dLSE| %.3g" % lerr
    return err.max()


def check(torch, w, rows=None):
    inp = W.make_inputs(w)
    o_gpu, lse_gpu = run_gpu(torch, w, inp)
    o_ref, lse_ref = oracle_rows(w, inp, rows)
    return compare(w, o_gpu, lse_gpu, o_ref, lse_ref, rows)


def sample_rows(w, n_random=400, tail=160, seed=7):
    """Rows of a few (b, h) pairs' first and last query rows plus random rows."""
    rng = np.random.default_rng(seed)
    total = w.B * w.Hq * w.Lq
    picks = []
    for (b, h) in {(0, 0), (w.B - 1, w.Hq - 1), (0, w.Hq // 2)}:
        base = (b * w.Hq + h) * w.Lq
        picks += [base + i for i in range(min(w.Lq, 8))]
        picks += [base + i for i in range(max(0, w.Lq - tail), w.Lq)]
    picks += list(rng.integers(0, total, size=n_random))
    return np.unique(np.array(picks, dtype=np.int64))


@pytest.fixture
def hooks():
    """Set library test hooks (sdpa_debug_set_option by name); each hook the
    test touches gets its previous value back afterwards."""
    import scaled_dot_product_fwd_gb300 as S
    saved = {}

    def set_hook(name, value):
        prev = S.sdpa_debug_set_option(name, int(value))
        saved.setdefault(name, prev)

    yield set_hook
    for name, prev in saved.items():
        S.sdpa_debug_set_option(name, prev)


def wl(B, Hq, Hkv, Lq, Lk, D, dtype, **kw):
    name = "case_%d_%d_%d_%d_%d_%d_%s" % (B, Hq, Hkv, Lq, Lk, D, dtype)
    return W.Workload(name, B, Hq, Hkv, Lq, Lk, D, dtype, **kw)


# ------------------------------------------------------------ named workloads
def test_tiny_full(cuda):
    check(cuda, W.TINY)


@pytest.mark.parametrize("w", [W.DIT_F16, W.DIT_F32], ids=lambda w: w.name)
def test_dit_sampled(cuda, w):
    check(cuda, w, sample_rows(w))


def test_dit_f32_accuracy_margin(cuda, capsys):
    """fp32 DiT through the tensor cores (bf16 hi/lo parts, three products per
    score, P split the same way against V's parts): the largest |dO| against
    the fp64 oracle on the sampled rows, printed so that the margin to the fp32
    tolerance is on record, and held to a quarter of that tolerance."""
    w = W.DIT_F32
    err = check(cuda, w, sample_rows(w))
    with capsys.disabled():
        print("\n%s: max |dO| %.3g (tolerance %.3g)" % (w.name, err, TOL[w.dtype]))
    assert err <= TOL[w.dtype] / 4


def test_causal_gqa_sampled(cuda):
    check(cuda, W.CAUSAL_GQA, sample_rows(W.CAUSAL_GQA, n_random=300, tail=130))


@pytest.mark.parametrize("key", sorted(W.DECODE_D512), ids=lambda k: W.DECODE_D512[k].name)
def test_decode_d512_full(cuda, key):
    check(cuda, W.DECODE_D512[key])


def test_decode_long_full(cuda):
    check(cuda, W.DECODE_LONG)


# ---------------------------------------------------- small shapes, all rows
PREFILL_SHAPES = [(2, 4, 2, 300, 333), (1, 2, 1, 129, 129), (1, 3, 3, 7, 200), (1, 1, 1, 2, 1),
                  (1, 2, 2, 256, 256), (2, 8, 1, 97, 1000), (1, 2, 1, 513, 520),
                  # key tails of exactly one 32-key chunk, of three chunks with a
                  # short first tile, and of 26 keys under a causal offset
                  (1, 2, 1, 160, 160), (1, 4, 2, 64, 224), (1, 2, 2, 200, 4250),
                  # a last key tile of exactly 64 keys
                  (1, 2, 2, 130, 192)]


@pytest.mark.parametrize("dtype", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", PREFILL_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_prefill_small(cuda, dtype, D, causal, shape):
    B, Hq, Hkv, Lq, Lk = shape
    if causal and Lq > Lk:
        pytest.skip("causal needs Lq <= Lk")
    check(cuda, wl(B, Hq, Hkv, Lq, Lk, D, dtype, causal=causal))


@pytest.mark.parametrize("dtype", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("mask", ["full", "row", "key"])
@pytest.mark.parametrize("sinks", [False, True])
@pytest.mark.parametrize("Lq", [1, 150])
@pytest.mark.parametrize("D", [64, 128])
def test_mask_and_sinks(cuda, dtype, mask, sinks, Lq, D):
    check(cuda, wl(2, 4, 2, Lq, 300, D, dtype, mask=mask, sinks=sinks, causal=(Lq > 1)))


@pytest.mark.parametrize("dtype,D", [("float16", 64), ("bfloat16", 64), ("float16", 128),
                                     ("bfloat16", 128)])
@pytest.mark.parametrize("scale_mul", [1.0, 0.37, 3.0])
def test_additive_key_mask_scales(cuda, dtype, D, scale_mul):
    # an additive mask row shared by the query rows enters S as one more
    # tensor-core step with 1/scale split into two 16-bit values; scales
    # whose inverse is exact (lo = 0) and inexact, several tiles, GQA
    import scaled_dot_product_fwd_gb300 as S
    w = wl(2, 8, 2, 300, 700, D, dtype, mask="key")
    inp = W.make_inputs(w)
    scale = w.scale * scale_mul
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o, lse = S.sdpa_forward(q, k, v, scale=scale, mask=inp["mask"].cuda())
    cuda.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    f = W.as_float64
    o_ref, lse_ref = O.sdpa(f(inp["q"]), f(inp["k"]), f(inp["v"]), scale, False, f(inp["mask"]))
    compare(w, o.cpu(), lse.cpu(), o_ref, lse_ref, None)


@pytest.mark.parametrize("dtype", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("Lq", [1, 140])
def test_large_sinks(cuda, dtype, Lq):
    check(cuda, wl(1, 8, 2, Lq, 257, 64, dtype, sinks=True, sink_scale=10.0))


@pytest.mark.parametrize("dtype", ["float16", "float32"])
@pytest.mark.parametrize("Lq", [1, 70])
@pytest.mark.parametrize("sinks", [False, True])
def test_fully_masked_rows(cuda, dtype, Lq, sinks):
    import torch
    import scaled_dot_product_fwd_gb300 as S
    w = wl(1, 2, 1, Lq, 90, 64, dtype, sinks=sinks)
    inp = W.make_inputs(w)
    m = torch.zeros((1, 2, Lq, 90), dtype=inp["q"].dtype)
    m[:, :, ::3, :] = float("-inf")  # every third row sees nothing
    inp["mask"] = m
    o_gpu, lse_gpu = run_gpu(torch, w, inp)
    o_ref, lse_ref = oracle_rows(w, inp, None)
    compare(w, o_gpu, lse_gpu, o_ref, lse_ref, None)
    assert S.sdpa_device_status() == 0


# ----------------------------------------------------------------- decode sweep
@pytest.mark.parametrize("dtype", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("D", [64, 128, 512])
@pytest.mark.parametrize("G", [1, 3, 4, 8, 16])
@pytest.mark.parametrize("Lk", [1, 7, 1000, 4097])
def test_decode_sweep(cuda, dtype, D, G, Lk):
    Hkv = 2
    check(cuda, wl(2, Hkv * G, Hkv, 1, Lk, D, dtype, sinks=(Lk % 2 == 1)))


@pytest.mark.parametrize("path", ["tc", "vector"])
@pytest.mark.parametrize("cluster", [1, 0])
@pytest.mark.parametrize("splits", [1, 2, 4, 5, 8, 16, 64])
def test_decode_forced_splits(cuda, splits, cluster, path, hooks):
    """Split counts on both head_dim-128 decode passes.  The vector pass
    merges 2, 4, 8 or 16 splits inside a thread-block cluster (cluster "0"
    forces its two-pass form); the tensor-core pass always merges through the
    combine kernel, and holds at most 14 tiles of 128 keys per split (1 forced
    split of 3001 keys runs as 2 splits of 12 tiles)."""
    if path == "tc" and cluster == 0:
        pytest.skip("the tensor-core pass has no cluster merge")
    hooks("decode_vector", 1 if path == "vector" else 0)
    hooks("decode_splits", splits)
    hooks("decode_cluster", cluster)
    check(cuda, wl(1, 8, 1, 1, 3001, 128, "bfloat16", sinks=True))


@pytest.mark.parametrize("dtype", ["bfloat16", "float32"])
@pytest.mark.parametrize("splits", [2, 16])
def test_decode_d512_cluster_merge_matches_two_pass(cuda, dtype, splits, hooks):
    """The in-cluster merge and the combine kernel give the same result on the
    head_dim 512 GQA-8 shape with sinks (both against the oracle too)."""
    import torch
    hooks("decode_splits", splits)
    w = wl(2, 32, 4, 1, 1024, 512, dtype, sinks=True)
    inp = W.make_inputs(w)
    outs = []
    for cl in (1, 0):
        hooks("decode_cluster", cl)
        outs.append(run_gpu(torch, w, inp))
    o_ref, lse_ref = oracle_rows(w, inp, None)
    for o_gpu, lse_gpu in outs:
        compare(w, o_gpu, lse_gpu, o_ref, lse_ref, None)
    tol = 1e-6 if dtype == "float32" else 1e-2
    assert float((outs[0][0].float() - outs[1][0].float()).abs().max()) <= tol
    assert float((outs[0][1] - outs[1][1]).abs().max()) <= 1e-5


# ----------------------------------------------------------------- edge cases
@pytest.mark.parametrize("Lq", [1, 5])
@pytest.mark.parametrize("sinks", [False, True])
def test_no_keys(cuda, Lq, sinks):
    import torch
    import scaled_dot_product_fwd_gb300 as S
    q = torch.randn(2, 4, Lq, 64, device="cuda", dtype=torch.float16)
    k = torch.empty(2, 2, 0, 64, device="cuda", dtype=torch.float16)
    s = torch.tensor([0.5, -1.0, 2.0, 0.0], device="cuda") if sinks else None
    o, lse = S.sdpa_forward(q, k, k, sinks=s)
    torch.cuda.synchronize()
    assert torch.all(o == 0)
    if sinks:
        assert torch.equal(lse, s.view(1, 4, 1).expand(2, 4, Lq).contiguous())
    else:
        assert torch.all(torch.isneginf(lse))


def test_empty_batch_is_noop(cuda):
    import torch
    import scaled_dot_product_fwd_gb300 as S
    q = torch.empty(0, 4, 10, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.empty(0, 2, 10, 64, device="cuda", dtype=torch.bfloat16)
    o, lse = S.sdpa_forward(q, k, k)
    assert o.shape == (0, 4, 10, 64)


def test_long_causal_prefill_sampled(cuda):
    w = wl(1, 2, 1, 32768, 32768, 128, "bfloat16", causal=True)
    check(cuda, w, sample_rows(w, n_random=120, tail=40))


def test_long_decode_sampled(cuda):
    w = wl(1, 8, 1, 1, 1 << 20, 128, "float16")
    check(cuda, w)


def test_bottom_right_causal_lq_lt_lk(cuda):
    check(cuda, wl(1, 4, 2, 200, 1000, 128, "bfloat16", causal=True))


@pytest.mark.parametrize("path", ["tc", "vector"])
def test_wait_timeout_reports_status(cuda, path, hooks):
    """A device wait that runs out sets the status word; the context stays
    usable.  The failure is made on the host: the decode producer is told to
    drop its last copy, so the consumers' bounded wait on it expires (on the
    tensor-core pass, the MMA thread's wait on the last V tile)."""
    import torch
    import scaled_dot_product_fwd_gb300 as S
    w = wl(1, 4, 1, 1, 640, 128, "bfloat16")
    inp = W.make_inputs(w)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    hooks("decode_vector", 1 if path == "vector" else 0)
    hooks("decode_splits", 1)
    hooks("decode_drop_last", 1)
    old = S.sdpa_debug_set_wait_limit_ns(50_000_000)
    try:
        S.sdpa_forward(q, k, v)
        assert S.sdpa_device_status() == 6  # SDPA_ERR_TIMEOUT
    finally:
        S.sdpa_debug_set_wait_limit_ns(old)
        hooks("decode_drop_last", 0)
    assert S.sdpa_device_status() == 0  # cleared by the read
    check(torch, w)  # the context still works


# ------------------------------------------------------ host-buffer entry point
@pytest.mark.parametrize("case", ["f16_mha", "bf16_gqa_causal_sinks", "f32_hilo"])
def test_host_entry_matches_device_entry(cuda, case):
    """sdpa_forward_host (the C call: pinned host buffers, pieces on the
    library's streams) gives the same bytes as sdpa_forward on device
    buffers: every (b, h) is computed by the same kernel either way (the fp32
    case also checks that the two compute streams do not share a
    workspace)."""
    import torch
    import scaled_dot_product_fwd_gb300 as S
    w = {"f16_mha": wl(2, 6, 6, 300, 300, 64, "float16"),
         "bf16_gqa_causal_sinks": wl(2, 8, 2, 200, 333, 128, "bfloat16", causal=True, sinks=True),
         "f32_hilo": wl(1, 6, 6, 257, 257, 64, "float32")}[case]
    inp = W.make_inputs(w)
    q, k, v = (inp[x].pin_memory() for x in ("q", "k", "v"))
    s = None if inp["sinks"] is None else inp["sinks"].cuda()
    o_d, l_d = S.sdpa_forward(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, causal=w.causal, sinks=s)
    torch.cuda.synchronize()
    o_h = torch.empty_like(q).pin_memory()
    l_h = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
    # the C call sdpa_forward_host (through ctypes), twice on the same buffers
    for _ in range(2):
        o_h.zero_()
        l_h.zero_()
        S.sdpa_forward_host(q, k, v, scale=w.scale, causal=w.causal, sinks=s, out=o_h, lse=l_h,
                            chunks=5)
        torch.cuda.synchronize()
        assert S.sdpa_device_status() == 0
        assert torch.equal(o_h, o_d.cpu())
        assert torch.equal(l_h, l_d.cpu())


def test_host_entry_decode_against_oracle(cuda):
    import torch
    import scaled_dot_product_fwd_gb300 as S
    w = wl(2, 32, 4, 1, 1024, 512, "bfloat16", sinks=True)
    inp = W.make_inputs(w)
    q, k, v = (inp[x].pin_memory() for x in ("q", "k", "v"))
    o_h, l_h = S.sdpa_forward_host(q, k, v, scale=w.scale, sinks=inp["sinks"].cuda(), chunks=4)
    torch.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    o_ref, lse_ref = oracle_rows(w, inp, None)
    compare(w, o_h, l_h, o_ref, lse_ref, None)


@pytest.mark.parametrize("mask", ["key", "full", "bool_key"])
def test_host_entry_masks_against_oracle(cuda, mask):
    """The C host-buffer call with masks: each piece reads the mask from its
    own (batch, head) offset (element-aligned, not 16-byte aligned for 333
    keys)."""
    import torch
    import scaled_dot_product_fwd_gb300 as S
    w = wl(2, 8, 4, 150, 333, 64, "float16", mask=mask, causal=True)
    inp = W.make_inputs(w)
    q, k, v = (inp[x].pin_memory() for x in ("q", "k", "v"))
    o_h, l_h = S.sdpa_forward_host(q, k, v, scale=w.scale, causal=True, mask=inp["mask"].cuda(),
                                   chunks=6)
    torch.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    o_ref, lse_ref = oracle_rows(w, inp, None)
    compare(w, o_h, l_h, o_ref, lse_ref, None)


# ------------------------------------------------ few-query rows (Lq 2..8)
@pytest.mark.parametrize("dtype", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("D", [64, 128, 512])
@pytest.mark.parametrize("G,Lq", [(1, 2), (4, 2), (4, 3), (8, 8), (16, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_multi_query_vector_path(cuda, dtype, D, G, Lq, causal):
    """A few query rows per head: the vector path (2 rows at D = 64/128, up to
    8 at D = 512; the G x Lq rows of a kv head share its K/V stream) or the
    prefill tiles for the rest; bottom-right causal rule per row."""
    Hkv = 2
    check(cuda, wl(2, Hkv * G, Hkv, Lq, 777, D, dtype, causal=causal, sinks=(G % 2 == 0)))


@pytest.mark.parametrize("dtype", ["float16", "float32"])
@pytest.mark.parametrize("mask", ["full", "row", "key"])
def test_multi_query_mask(cuda, dtype, mask):
    check(cuda, wl(2, 8, 2, 2, 300, 128, dtype, mask=mask, sinks=True, causal=True))
    check(cuda, wl(2, 8, 2, 5, 300, 512, dtype, mask=mask, sinks=True, causal=True))


def test_multi_query_fully_masked_rows(cuda):
    import torch
    w = wl(1, 4, 2, 6, 90, 512, "bfloat16", sinks=True)
    inp = W.make_inputs(w)
    m = torch.zeros((1, 4, 6, 90), dtype=inp["q"].dtype)
    m[:, :, ::3, :] = float("-inf")  # every third row sees nothing
    inp["mask"] = m
    o_gpu, lse_gpu = run_gpu(torch, w, inp)
    o_ref, lse_ref = oracle_rows(w, inp, None)
    compare(w, o_gpu, lse_gpu, o_ref, lse_ref, None)


@pytest.mark.parametrize("splits", [2, 16])
def test_multi_query_forced_splits(cuda, splits, hooks):
    hooks("decode_splits", splits)
    check(cuda, wl(1, 16, 2, 2, 3001, 128, "bfloat16", causal=True, sinks=True))
    check(cuda, wl(1, 8, 1, 6, 3001, 512, "bfloat16", causal=True, sinks=True))


def test_launch_count_reports_kernels_per_call(cuda, hooks):
    """sdpa_last_launch_count: 1 for prefill, 2 for the fp32 hi/lo prefill
    (split + prefill), 1 or 2 for decode (in-cluster merge or combine pass),
    1 for no keys, 0 after an error or an empty problem."""
    import torch
    import scaled_dot_product_fwd_gb300 as S

    def run(w, **kw):
        inp = W.make_inputs(w)
        q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
        S.sdpa_forward(q, k, v, scale=w.scale, causal=w.causal, **kw)
        torch.cuda.synchronize()
        return S.sdpa_last_launch_count()

    assert run(wl(1, 2, 2, 300, 300, 64, "float16")) == 1
    assert run(wl(1, 2, 2, 300, 300, 64, "float32")) == 2
    hooks("decode_splits", 4)
    assert run(wl(1, 8, 1, 1, 4096, 128, "bfloat16")) == 2  # tensor-core pass + combine
    hooks("decode_splits", 1)
    assert run(wl(1, 8, 1, 1, 1000, 128, "bfloat16")) == 1  # one split writes O
    hooks("decode_splits", 4)
    hooks("decode_vector", 1)
    assert run(wl(1, 8, 1, 1, 4096, 128, "bfloat16")) == 1  # 4 CTAs per cluster
    hooks("decode_cluster", 0)
    assert run(wl(1, 8, 1, 1, 4096, 128, "bfloat16")) == 2
    hooks("decode_vector", 0)
    hooks("decode_cluster", 1)
    hooks("decode_splits", 0)
    q = torch.zeros(1, 2, 4, 64, device="cuda", dtype=torch.float16)
    kk = torch.zeros(1, 2, 0, 64, device="cuda", dtype=torch.float16)
    S.sdpa_forward(q, kk, kk)
    assert S.sdpa_last_launch_count() == 1
    S.sdpa_forward(q[:0], q[:0], q[:0])
    assert S.sdpa_last_launch_count() == 0


# ------------------------------------------- KV-cache views, per-batch lengths
def _kv_view_check(B, Hq, Hkv, Lq, Lk, cap, D, dtype, causal, sinks, lens_q, lens_kv,
                   noalloc=False):
    """k, v as rows [0, Lk) of a [B, Hkv, cap, D] cache, per-batch lengths.
    Rows [Lk, cap) hold NaN (never read); rows [len_kv_b, Lk) hold large
    finite junk (weighted by zero).  Expected: the oracle on the used rows
    with an explicit -inf mask for padding and the per-batch causal rule."""
    import torch
    import scaled_dot_product_fwd_gb300 as S
    w = wl(B, Hq, Hkv, Lq, Lk, D, dtype, causal=causal, sinks=sinks)
    inp = W.make_inputs(w)
    kc = torch.full((B, Hkv, cap, D), float("nan"), dtype=inp["k"].dtype)
    vc = kc.clone()
    kc[:, :, :Lk] = inp["k"]
    vc[:, :, :Lk] = inp["v"]
    for b in range(B):
        kc[b, :, lens_kv[b]:Lk] = 300.0
        vc[b, :, lens_kv[b]:Lk] = -300.0
    mask = np.zeros((B, Hq, Lq, Lk))
    for b in range(B):
        i = np.arange(Lq)[:, None]
        j = np.arange(Lk)[None, :]
        hide = (i >= lens_q[b]) | (j >= lens_kv[b])
        if causal:
            hide |= j > i + (lens_kv[b] - lens_q[b])
        mask[b, :, hide] = -np.inf
    f = W.as_float64
    o_ref, l_ref = O.sdpa(f(inp["q"]), f(kc[:, :, :Lk]), f(vc[:, :, :Lk]), w.scale, False, mask,
                          None if inp["sinks"] is None else f(inp["sinks"]))
    q = inp["q"].cuda()
    s = None if inp["sinks"] is None else inp["sinks"].cuda()
    tq = torch.tensor(lens_q, dtype=torch.int32, device="cuda")
    tk = torch.tensor(lens_kv, dtype=torch.int32, device="cuda")
    if noalloc:
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
        p = S.make_params(B, Hq, Hkv, Lq, Lk, D, S.dtype_code(q.dtype), w.scale, causal, None,
                          (0, 0, 0, 1), None if s is None else s.data_ptr(), kv_capacity=cap,
                          seq_lens_q_ptr=tq.data_ptr(), seq_lens_kv_ptr=tk.data_ptr())
        kcd, vcd = kc.cuda(), vc.cuda()
        st = S._binding.sdpa_forward_decode_noalloc_raw(
            p, q.data_ptr(), kcd.data_ptr(), vcd.data_ptr(), o.data_ptr(), lse.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
        assert st == 0
    else:
        o, lse = S.sdpa_forward(q, kc.cuda(), vc.cuda(), scale=w.scale, causal=causal, sinks=s,
                                kv_len=Lk, seq_lens_q=tq, seq_lens_kv=tk)
    torch.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    compare(w, o.cpu(), lse.cpu(), o_ref, l_ref, None)


@pytest.mark.parametrize("dtype,D", [("float16", 64), ("bfloat16", 128), ("float32", 64),
                                     ("float32", 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_kv_view_prefill(cuda, dtype, D, causal):
    # batch 1 has more query rows than keys: under the causal rule its first
    # 50 rows see no key
    _kv_view_check(3, 4, 2, 260, 300, 384, D, dtype, causal, sinks=True,
                   lens_q=[260, 150, 0], lens_kv=[300, 100, 50])


@pytest.mark.parametrize("dtype,D", [("bfloat16", 512), ("float16", 128), ("float32", 64)])
def test_kv_view_decode(cuda, dtype, D):
    _kv_view_check(4, 32, 4, 1, 1024, 1100, D, dtype, False, sinks=True,
                   lens_q=[1, 1, 1, 0], lens_kv=[1024, 1, 700, 0])


def test_kv_view_long_decode_and_few_queries(cuda):
    _kv_view_check(3, 16, 2, 1, 5000, 6000, 128, "bfloat16", False, sinks=False,
                   lens_q=[1, 1, 1], lens_kv=[5000, 4097, 1])
    _kv_view_check(2, 8, 2, 2, 777, 800, 64, "float16", True, sinks=True,
                   lens_q=[2, 1], lens_kv=[777, 300])


@pytest.mark.parametrize("path", ["tc", "vector"])
@pytest.mark.parametrize("lens_kv", [[4096, 3584, 3072, 2560, 2048, 1536, 1024, 512],
                                     [4095, 1, 0, 2049, 17, 4096, 1000, 3]],
                         ids=["descending", "odd_and_empty"])
def test_kv_view_ragged_plan(cuda, lens_kv, path, hooks):
    """Decode over a KV cache with ragged per-batch lengths at the long
    decode's head shape.  Vector pass: the split size comes from the device
    lengths (every CTA derives it, and the combine derives each row's split
    count), so the items of the real keys fill whole waves.  Tensor-core
    pass: splits past a batch's length leave empty partial results."""
    hooks("decode_vector", 1 if path == "vector" else 0)
    _kv_view_check(8, 32, 8, 1, 4096, 4096, 128, "bfloat16", False, sinks=True,
                   lens_q=[1] * 8, lens_kv=lens_kv)


@pytest.mark.parametrize("dtype", ["float16", "bfloat16"])
def test_kv_view_tc128_multi_tile_splits(cuda, dtype):
    """The head_dim-128 tensor-core pass with splits of 14 tiles of 128 keys
    (all score tiles of a split in TMEM, the K/V ring wrapping many times):
    two query rows per batch (16 rows per kv head with G = 8), the causal rule,
    sinks, ragged query and key lengths including empty and one-key rows."""
    _kv_view_check(8, 64, 8, 2, 9000, 9100, 128, dtype, True, sinks=True,
                   lens_q=[2, 1, 2, 0, 2, 2, 1, 2],
                   lens_kv=[9000, 1, 4000, 0, 8999, 1793, 128, 129])


def test_kv_view_noalloc(cuda):
    _kv_view_check(2, 32, 4, 1, 1024, 1100, 512, "bfloat16", False, sinks=True,
                   lens_q=[1, 1], lens_kv=[1000, 3], noalloc=True)


# --------------------------------------- prefill units split over a cluster
SPLIT_CASES = {
    "f16_d64_gqa": wl(2, 4, 2, 300, 1000, 64, "float16"),
    "bf16_d128_sinks": wl(1, 3, 1, 260, 333, 128, "bfloat16", sinks=True),
    # fp32 at D = 64 (bf16 hi/lo products); two key tiles: with four CTAs two
    # of them have no key tile
    "f32_d64_two_tiles": wl(1, 2, 2, 129, 200, 64, "float32"),
    # one key tile: every CTA but one has none; additive mask
    "f16_d128_mask_one_tile": wl(1, 2, 1, 140, 100, 128, "float16", mask="full"),
}


@pytest.mark.parametrize("ksplit", [2, 4])
@pytest.mark.parametrize("case", sorted(SPLIT_CASES))
def test_prefill_forced_split(cuda, ksplit, case, hooks):
    """Every query-block unit split over its key tiles among the 2 or 4 CTAs
    of a cluster, the partial results merged through distributed shared
    memory (the form the last partial wave of units takes)."""
    hooks("prefill_split", ksplit)
    check(cuda, SPLIT_CASES[case])


@pytest.mark.parametrize("ksplit", [2, 4])
def test_prefill_forced_split_kv_view(cuda, ksplit, hooks):
    """Split units with per-batch key lengths (some batches shorter than the
    split count in key tiles, one with no key at all)."""
    hooks("prefill_split", ksplit)
    _kv_view_check(3, 4, 2, 260, 600, 700, 64, "float16", False, sinks=True,
                   lens_q=[260, 150, 0], lens_kv=[600, 100, 0])


def test_prefill_tail_split_and_shared_gpu(cuda):
    """The DiT shape (1292 units: a half-empty last wave on 152 SMs): by
    default its last wave goes to a second, split grid; with shared_gpu
    (SDPA_FLAG_SHARED_GPU) every unit runs whole in one grid.  Both against
    the oracle."""
    import torch
    import scaled_dot_product_fwd_gb300 as S
    w = W.DIT_F16
    rows = sample_rows(w, n_random=200, tail=40)
    inp = W.make_inputs(w)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o_ref, lse_ref = oracle_rows(w, inp, rows)
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    units = w.B * w.Hq * (-(-w.Lq // 256))
    r = units % nsm
    for shared in (False, True):
        o, lse = S.sdpa_forward(q, k, v, scale=w.scale, shared_gpu=shared)
        torch.cuda.synchronize()
        grids = S.sdpa_last_launch_count()
        assert grids == (1 if shared or r == 0 or 2 * r > nsm else 2)
        compare(w, o.cpu(), lse.cpu(), o_ref, lse_ref, rows)


# ------------------------------------------- boolean masks (True = visible)
BOOL_CASES = {
    "prefill_f16_d64": wl(2, 4, 2, 300, 333, 64, "float16", mask="bool_full"),
    "prefill_bf16_d128_causal_sinks": wl(1, 4, 1, 260, 300, 128, "bfloat16", causal=True,
                                         sinks=True, mask="bool_key"),
    "prefill_f32_d64_hilo": wl(1, 2, 2, 129, 200, 64, "float32", mask="bool_full"),
    "prefill_f32_d128_fma": wl(1, 2, 1, 100, 150, 128, "float32", mask="bool_full", sinks=True),
    "decode_bf16_d128_sinks": wl(2, 8, 2, 1, 1000, 128, "bfloat16", mask="bool_full",
                                 sinks=True),
    "decode_f16_d512": wl(1, 32, 4, 1, 1024, 512, "float16", mask="bool_key"),
    "few_queries_f16_causal": wl(1, 8, 2, 2, 777, 64, "float16", causal=True, mask="bool_full"),
    # rows of 512 and 384 keys: every mask row 16-byte aligned (vector loads)
    "prefill_f16_d64_rows16": wl(2, 4, 2, 300, 512, 64, "float16", mask="bool_full"),
    "prefill_bf16_d128_rows16_sinks": wl(1, 4, 2, 200, 384, 128, "bfloat16", mask="bool_full",
                                         sinks=True),
    # a key mask shared by the query rows under the causal rule, ragged tail
    "prefill_bf16_d64_key_causal": wl(2, 4, 2, 300, 333, 64, "bfloat16", causal=True,
                                      mask="bool_key"),
    "prefill_f16_d64_key_gqa": wl(1, 8, 1, 257, 1000, 64, "float16", mask="bool_key"),
}


@pytest.mark.parametrize("case", sorted(BOOL_CASES))
def test_bool_mask(cuda, case):
    check(cuda, BOOL_CASES[case])


@pytest.mark.parametrize("D,dtype,kind", [(64, "float16", "bool_key"),
                                          (64, "bfloat16", "bool_full"),
                                          (128, "float16", "bool_key"),
                                          (64, "float16", "full"),
                                          (128, "bfloat16", "key")])
def test_mask_negative_scale(cuda, D, dtype, kind):
    # a negative scale turns the row max of the raw scores into the row min:
    # the kernels take their general (unfused) softmax
    import scaled_dot_product_fwd_gb300 as S
    w = wl(2, 4, 2, 200, 333, D, dtype, mask=kind)
    inp = W.make_inputs(w)
    q, k, v = (to_dev(inp[x], cuda) for x in ("q", "k", "v"))
    o, lse = S.sdpa_forward(q, k, v, scale=-w.scale, mask=inp["mask"].cuda())
    cuda.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    f = W.as_float64
    m = inp["mask"]
    m = m.numpy() if m.dtype == cuda.bool else f(m)
    o_ref, lse_ref = O.sdpa(f(inp["q"]), f(inp["k"]), f(inp["v"]), -w.scale, False, m)
    compare(w, o.cpu(), lse.cpu(), o_ref, lse_ref, None)


@pytest.mark.parametrize("D,dtype", [(64, "float16"), (128, "bfloat16")])
@pytest.mark.parametrize("boolean", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_key_mask_edges(cuda, D, dtype, boolean, causal):
    # key masks on the tensor-core bias step: one row per (batch, head)
    # ([B, Hq, 1, Lk], head offsets in the mask), batch 1 hides every key
    # (its rows see nothing: O = 0, LSE = -inf), large finite biases
    import torch
    import scaled_dot_product_fwd_gb300 as S
    B, Hq, Hkv, Lq, Lk = 2, 4, 2, 260, 333
    w = wl(B, Hq, Hkv, Lq, Lk, D, dtype, causal=causal)
    inp = W.make_inputs(w)
    rng = np.random.default_rng(11)
    if boolean:
        keep = rng.random((B, Hq, 1, Lk)) >= 0.3
        keep[1] = False
        m_host = torch.from_numpy(keep)
        m_ref = keep
    else:
        vals = rng.standard_normal((B, Hq, 1, Lk)) * 4.0
        vals[rng.random((B, Hq, 1, Lk)) < 0.2] = -np.inf
        vals[0, 0, 0, :5] = -60000.0  # large finite
        vals[1] = -np.inf
        m_host = torch.from_numpy(vals.astype(np.float32)).to(inp["q"].dtype)
        m_ref = W.as_float64(m_host)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o, lse = S.sdpa_forward(q, k, v, scale=w.scale, causal=causal, mask=m_host.cuda())
    cuda.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    f = W.as_float64
    o_ref, lse_ref = O.sdpa(f(inp["q"]), f(inp["k"]), f(inp["v"]), w.scale, causal, m_ref)
    assert np.all(np.isneginf(lse_ref[1]))
    compare(w, o.cpu(), lse.cpu(), o_ref, lse_ref, None)


# additive masks with a row per query: rows of 512 keys are 16-byte aligned
# (vector loads), rows of 333 keys mostly not; GQA, causal, several tiles
@pytest.mark.parametrize("dtype", ["float16", "bfloat16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Lk", [512, 333])
@pytest.mark.parametrize("causal", [False, True])
def test_additive_row_mask(cuda, dtype, D, Lk, causal):
    check(cuda, wl(2, 8, 2, 300, Lk, D, dtype, mask="full", causal=causal, sinks=causal))


@pytest.mark.parametrize("kind", ["full", "bool_full"])
@pytest.mark.parametrize("Lk", [512, 333])
@pytest.mark.parametrize("workspace", [False, True])
def test_row_mask_workspace_forms(cuda, kind, Lk, workspace):
    """A mask with a row per query through the C call: with the workspace
    that sdpa_workspace_size reports the call first copies the mask into
    score tiles; with none it reads the mask where it lies (16-byte loads
    where rows are aligned, else per element).  Both against the oracle,
    causal with a ragged tail, GQA."""
    import torch
    import scaled_dot_product_fwd_gb300 as S
    w = wl(2, 8, 2, 300, Lk, 64, "float16", mask=kind, causal=True, sinks=True)
    inp = W.make_inputs(w)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    m, sk = inp["mask"].cuda(), inp["sinks"].cuda()
    mexp = m.expand(w.B, w.Hq, w.Lq, w.Lk)
    flags = S._binding.SDPA_FLAG_BOOL_MASK if m.dtype == torch.bool else 0
    p = S.make_params(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D, S.dtype_code(q.dtype), w.scale, True,
                      mexp.data_ptr(), tuple(int(x) for x in mexp.stride()), sk.data_ptr(),
                      flags=flags)
    need = S._binding.sdpa_workspace_size(p)
    assert need > 0  # the tiled copy is offered for a row-per-query mask
    ws = torch.empty(need, dtype=torch.uint8, device="cuda") if workspace else None
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    st = S._binding.sdpa_forward_raw(p, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), None if ws is None else ws.data_ptr(),
                                     0 if ws is None else need,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == 0
    assert S.sdpa_last_launch_count() == (2 if workspace else 1)
    torch.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    o_ref, lse_ref = oracle_rows(w, inp, None)
    compare(w, o.cpu(), lse.cpu(), o_ref, lse_ref, None)


@pytest.mark.parametrize("D,dtype,kind,causal", [(64, "float16", "bool_key", False),
                                                 (64, "bfloat16", "bool_full", True),
                                                 (128, "bfloat16", "bool_key", True)])
def test_bool_mask_with_lengths(cuda, D, dtype, kind, causal):
    # per-batch query and key lengths together with a boolean mask; the
    # expected values take both as one additive 0 / -inf mask
    import scaled_dot_product_fwd_gb300 as S
    B, Hq, Hkv, Lq, Lk = 3, 4, 2, 300, 400
    lens_q, lens_kv = [300, 129, 0], [400, 250, 77]
    w = wl(B, Hq, Hkv, Lq, Lk, D, dtype, causal=False, mask=kind)
    inp = W.make_inputs(w)
    keep = np.broadcast_to(inp["mask"].numpy(), (B, Hq, Lq, Lk))
    add = np.where(keep, 0.0, -np.inf)
    for b in range(B):
        i = np.arange(Lq)[:, None]
        j = np.arange(Lk)[None, :]
        hide = (i >= lens_q[b]) | (j >= lens_kv[b])
        if causal:
            hide |= j > i + (lens_kv[b] - lens_q[b])
        add[b, :, hide] = -np.inf
    f = W.as_float64
    o_ref, lse_ref = O.sdpa(f(inp["q"]), f(inp["k"]), f(inp["v"]), w.scale, False, add)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    tq = cuda.tensor(lens_q, dtype=cuda.int32, device="cuda")
    tk = cuda.tensor(lens_kv, dtype=cuda.int32, device="cuda")
    o, lse = S.sdpa_forward(q, k, v, scale=w.scale, causal=causal, mask=inp["mask"].cuda(),
                            seq_lens_q=tq, seq_lens_kv=tk)
    cuda.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    compare(w, o.cpu(), lse.cpu(), o_ref, lse_ref, None)


# ------------------------------------ non-contiguous q, k, v, o (D contiguous)
def _bshd(t):
    """[B, H, L, D] values stored as a dense [B, L, H, D] tensor, seen as
    [B, H, L, D] (strides L*H*D, D, H*D)."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


def _strided_check(w, layout, hooks=None, split=None):
    import torch
    import scaled_dot_product_fwd_gb300 as S
    if split is not None:
        hooks("prefill_split", split)
    inp = W.make_inputs(w)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    mask = None if inp["mask"] is None else inp["mask"].cuda()
    sinks = None if inp["sinks"] is None else inp["sinks"].cuda()
    out, kv_len = None, None
    if layout == "bshd":  # inputs [B, L, H, D]; out takes q's layout
        q, k, v = _bshd(q), _bshd(k), _bshd(v)
    elif layout == "kv_cache_bshd":  # k, v: rows [0, Lk) of a [B, C, Hkv, D] cache
        C = w.Lk + 37
        kc = torch.full((w.B, C, w.Hkv, w.D), float("nan"), dtype=k.dtype, device="cuda")
        vc = kc.clone()
        kc[:, :w.Lk] = k.transpose(1, 2)
        vc[:, :w.Lk] = v.transpose(1, 2)
        k, v, kv_len = kc.transpose(1, 2), vc.transpose(1, 2), w.Lk
        out = _bshd(torch.empty_like(q))
    elif layout == "padded_rows":  # rows of q, k, v and o padded to 2 D elements
        def pad(t):
            big = torch.zeros(t.shape[:3] + (2 * w.D,), dtype=t.dtype, device="cuda")
            big[..., :w.D] = t
            return big[..., :w.D]
        q, k, v = pad(q), pad(k), pad(v)
        out = pad(torch.zeros_like(q))
    # (with one kv head the cache view is contiguous: the kv_capacity form)
    o, lse = S.sdpa_forward(q, k, v, scale=w.scale, causal=w.causal, mask=mask, sinks=sinks,
                            out=out, kv_len=kv_len)
    torch.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    if layout == "bshd":
        assert o.stride() == q.stride()  # the output keeps q's layout
    o_ref, lse_ref = oracle_rows(w, inp, None)
    compare(w, o.contiguous().cpu(), lse.cpu(), o_ref, lse_ref, None)


STRIDE_CASES = {
    "prefill_f16_d64": wl(2, 4, 2, 300, 333, 64, "float16", sinks=True),
    "prefill_bf16_d128_causal": wl(1, 4, 1, 260, 300, 128, "bfloat16", causal=True,
                                   mask="bool_key"),
    "prefill_f32_d64_hilo": wl(1, 2, 2, 129, 200, 64, "float32", mask="full"),
    "prefill_f32_d128_fma": wl(1, 2, 1, 100, 150, 128, "float32"),
    "decode_bf16_d128": wl(2, 8, 2, 1, 1000, 128, "bfloat16", sinks=True),
    "decode_f32_d512": wl(1, 32, 4, 1, 1024, 512, "float32"),
    "few_queries_f16_d64": wl(1, 8, 2, 2, 777, 64, "float16", causal=True),
}


@pytest.mark.parametrize("layout", ["bshd", "kv_cache_bshd", "padded_rows"])
@pytest.mark.parametrize("case", sorted(STRIDE_CASES))
def test_strided_layouts(cuda, case, layout):
    _strided_check(STRIDE_CASES[case], layout)


@pytest.mark.parametrize("split", [2, 4])
def test_strided_output_split_units(cuda, split, hooks):
    """Split units (partial results merged in the cluster) writing a strided
    output."""
    _strided_check(wl(1, 4, 2, 300, 1000, 64, "float16"), "kv_cache_bshd", hooks, split)


def test_strided_no_keys(cuda):
    import torch
    import scaled_dot_product_fwd_gb300 as S
    q = _bshd(torch.randn(2, 4, 5, 64, device="cuda", dtype=torch.float16))
    kk = torch.zeros(2, 4, 0, 64, device="cuda", dtype=torch.float16)
    out = _bshd(torch.full_like(q, 7.0))
    o, lse = S.sdpa_forward(q, kk, kk, out=out)
    torch.cuda.synchronize()
    assert o.data_ptr() == out.data_ptr()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


# ------------------------------------- masks holding the dtype's lowest finite value
LOWEST_CASES = [("key", 150, 300), ("row", 150, 304), ("row", 150, 300), ("full", 150, 300),
                ("key", 1, 300), ("full", 4, 1000)]


@pytest.mark.parametrize("dtype", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind,Lq,Lk", LOWEST_CASES, ids=lambda c: str(c))
def test_lowest_finite_mask(cuda, dtype, D, kind, Lq, Lk):
    """Additive masks that use the dtype's most negative finite value as padding.

    The float64 definition gives softmax(s + low) on a row masked by it
    throughout, which for bfloat16/float32's lowest value (about -3.4e38) is
    the uniform average of V: the scores vanish beside the mask.  Keys masked
    by it in other rows weigh nothing.  Key masks (one row shared by the
    query rows), the single-query path and the fp32 head-dim-128 kernel give
    such rows that result, with LSE -2^100 * scale (a mask value of magnitude
    2^64 or more enters as 2^100 in raw-score units), and so do bfloat16
    masks with a row per query on the tensor-core prefill (read from their
    score-tile copy); fp16's lowest value (-65504) is an ordinary value
    everywhere (LSE within 1e-6 relative).  On the fp32 tensor-core path
    (head_dim 64) for masks with a row per query, a value whose scaled
    product overflows fp32 acts as -inf: a row masked by it throughout sees
    no key (O = 0, LSE = -inf).  Every other row matches the oracle at the
    usual bars.
    """
    torch = cuda
    w = wl(2, 4, 2, Lq, Lk, D, dtype, mask=kind, causal=False)
    inp = W.make_inputs(w)
    m = inp["mask"].clone()
    low = torch.finfo(m.dtype).min
    if kind == "row":       # [1, 1, Lq, Lk]: the first rows entirely, every third key of the rest
        m[:, :, : min(Lq, 10), :] = low
        m[:, :, 10:, ::3] = low
    else:                   # batch 0 entirely, every third key of batch 1
        m[0] = low
        m[1, ..., ::3] = low
    inp["mask"] = m
    o_gpu, lse_gpu = run_gpu(torch, w, inp)
    o_ref, lse_ref = oracle_rows(w, inp, None)
    og = W.as_float64(o_gpu).reshape(-1, D)
    lg = lse_gpu.double().numpy().reshape(-1)
    o_ref, lse_ref = o_ref.reshape(-1, D), lse_ref.reshape(-1)
    assert np.all(np.isfinite(og))
    per_query_tc = kind != "key" and Lq > 2 and dtype == "float32" and D == 64
    gone = (lse_ref < -1e30) if per_query_tc else np.zeros_like(lse_ref, dtype=bool)
    if gone.any():          # rows that see no key on the per-query tensor-core paths
        assert np.all(np.isneginf(lg[gone])) and np.all(og[gone] == 0)
    keep = ~gone
    err = np.abs(og[keep] - o_ref[keep])
    assert err.max() <= TOL[dtype], "max |dO| %.3g" % err.max()
    assert err.mean() <= MEAN_TOL
    big = (lse_ref < -1e4) & keep
    norm = keep & ~big
    assert np.all(np.isfinite(lg[keep]))
    lerr = np.abs(lg[norm] - lse_ref[norm]).max()
    assert lerr <= LSE_TOL, "max |dLSE| %.3g" % lerr
    mid = big & (lse_ref > -1e30)
    assert np.all(np.abs(lg[mid] - lse_ref[mid]) <= 1e-6 * np.abs(lse_ref[mid]))
    hug = big & ~mid
    assert np.allclose(lg[hug], -(2.0 ** 100) * w.scale, rtol=1e-5, atol=0)


# ------------------------------------------------ head_dim 512 with many query rows
D512_CASES = [(9, 300), (129, 333), (1024, 1024)]


@pytest.mark.parametrize("dtype", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("Lq,Lk", D512_CASES, ids=lambda c: str(c))
@pytest.mark.parametrize("causal", [False, True])
def test_d512_prefill(cuda, dtype, Lq, Lk, causal):
    """head_dim 512 beyond the vector path's 8 rows: the tensor-core kernel
    (fp16/bf16; two CTAs per query tile, one per half of O) or the vector
    path with grouped rows (fp32); GQA-8 with sinks, every row compared."""
    w = wl(1, 8, 1, Lq, Lk, 512, dtype, causal=causal, sinks=True)
    check(cuda, w)


@pytest.mark.parametrize("dtype", ["float16", "bfloat16"])
@pytest.mark.parametrize("mask", ["key", "full", "bool_key", "bool_full"])
def test_d512_prefill_masks(cuda, dtype, mask):
    check(cuda, wl(2, 4, 2, 150, 333, 512, dtype, mask=mask, causal=True))


def test_d512_prefill_strided_and_lengths(cuda):
    """[B, L, H, D] q, k, v (strides) and per-batch lengths at head_dim 512."""
    import torch
    import scaled_dot_product_fwd_gb300 as S
    B, Hq, Hkv, Lq, Lk, D = 2, 4, 2, 200, 300, 512
    w = wl(B, Hq, Hkv, Lq, Lk, D, "bfloat16", causal=True)
    inp = W.make_inputs(w)
    q, k, v = (_bshd(inp[x].cuda()) for x in ("q", "k", "v"))
    lq = torch.tensor([200, 131], dtype=torch.int32, device="cuda")
    lk = torch.tensor([300, 190], dtype=torch.int32, device="cuda")
    o, lse = S.sdpa_forward(q, k, v, scale=w.scale, causal=True, seq_lens_q=lq, seq_lens_kv=lk)
    torch.cuda.synchronize()
    assert S.sdpa_device_status() == 0
    f = W.as_float64
    for b in range(B):
        nq, nk = int(lq[b]), int(lk[b])
        o_ref, lse_ref = O.sdpa(f(inp["q"][b:b + 1, :, :nq]), f(inp["k"][b:b + 1, :, :nk]),
                                f(inp["v"][b:b + 1, :, :nk]), w.scale, True, None, None)
        og = f(o[b:b + 1, :, :nq].cpu())
        assert np.abs(og - o_ref).max() <= TOL["bfloat16"]
        assert np.abs(lse[b:b + 1, :, :nq].cpu().double().numpy() - lse_ref).max() <= LSE_TOL
        # rows past the batch's query length see no key
        assert torch.all(o[b, :, nq:] == 0) and torch.all(torch.isneginf(lse[b, :, nq:]))
