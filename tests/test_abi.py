"""Host-side checks of the C ABI: the library loads without a GPU, exports
every symbol include/sdpa.h declares, and rejects bad problems before any
CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

import scaled_dot_product_fwd_gb300 as S
from scaled_dot_product_fwd_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdpa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    assert declared_functions() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(sdpa_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", S.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    syms = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    for name in declared_functions():
        assert name in syms, name
        assert getattr(sdpa_lib, name) is not None
    # nothing else leaks out of the library
    assert not [s for s in syms if s.startswith("_ZN5gb300")]


def test_params_struct_layout():
    assert ctypes.sizeof(B.SdpaParams) == 208
    assert B.SdpaParams.mask.offset == 40
    assert B.SdpaParams.mask_stride.offset == 48
    assert B.SdpaParams.sinks.offset == 80
    assert B.SdpaParams.kv_capacity.offset == 88
    assert B.SdpaParams.seq_lens_q.offset == 96
    assert B.SdpaParams.seq_lens_kv.offset == 104
    assert B.SdpaParams.q_stride.offset == 112
    assert B.SdpaParams.k_stride.offset == 136
    assert B.SdpaParams.v_stride.offset == 160
    assert B.SdpaParams.o_stride.offset == 184


def test_launch_count_is_zero_after_a_rejected_call(sdpa_lib):
    assert S.sdpa_forward_raw(P(D=96), 256, 256, 256, 256, None, None, 0, None) == 2
    assert S.sdpa_last_launch_count() == 0


def test_abi_version_and_status_strings(sdpa_lib):
    assert S.sdpa_abi_version() == 5
    assert S.sdpa_status_string(0) == "ok"
    assert S.sdpa_status_string(2) == "unsupported problem"
    assert S.sdpa_status_string(99) == "unknown status"


def P(**kw):
    d = dict(B=1, Hq=4, Hkv=2, Lq=16, Lk=32, D=64, dtype=S.SDPA_BF16, scale=0.125)
    d.update(kw)
    causal = d.pop("causal", False)
    return S.make_params(d["B"], d["Hq"], d["Hkv"], d["Lq"], d["Lk"], d["D"], d["dtype"],
                         d["scale"], causal, d.get("mask"), d.get("ms", (0, 0, 0, 1)),
                         d.get("sinks"))


@pytest.mark.parametrize("kw,kernel", [
    (dict(), "prefill_tc"),
    (dict(dtype=S.SDPA_F16, D=128), "prefill_tc"),
    (dict(dtype=S.SDPA_F32), "prefill_tc_f32"),
    (dict(dtype=S.SDPA_F32, D=128), "prefill_f32"),
    (dict(Lq=1), "decode_splitkv"),
    (dict(Lq=1, D=512, dtype=S.SDPA_F32), "decode_splitkv"),
    (dict(Lq=2), "decode_splitkv"),
    (dict(Lq=3), "prefill_tc"),
    (dict(Lq=8, D=512, causal=True), "decode_splitkv"),
    (dict(Lq=9, D=512), "prefill_tc"),
    (dict(Lq=4096, Lk=4096, D=512, dtype=S.SDPA_BF16, causal=True), "prefill_tc"),
    (dict(Lq=9, D=512, dtype=S.SDPA_F32), "decode_splitkv"),
    (dict(Lq=3, dtype=S.SDPA_F32), "prefill_tc_f32"),
    (dict(Lk=0), "no_keys"),
    (dict(Lq=1, Lk=0, D=512), "no_keys"),
    (dict(B=0), "none"),
    (dict(Lq=0), "none"),
    (dict(Hq=0), "none"),
])
def test_select_kernel(sdpa_lib, kw, kernel):
    name, st = S.sdpa_select_kernel(P(**kw))
    assert (name, st) == (kernel, 0)


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=3, Hkv=2), 1),
    (dict(Hkv=0), 1),
    (dict(B=-1), 1),
    (dict(Lk=-2), 1),
    (dict(dtype=7), 1),
    (dict(scale=float("nan")), 1),
    (dict(scale=float("inf")), 1),
    (dict(D=96), 2),
    (dict(D=256), 2),
    # fp32 at head_dim 512 on the vector path: (kv head, row group) pairs
    # past the grid's 65535
    (dict(D=512, Lq=1 << 17, Lk=1 << 17, Hq=4, Hkv=2, dtype=S.SDPA_F32), 2),
    (dict(Lq=64, Lk=32, causal=True), 2),
    (dict(Lq=(1 << 30) + 1), 2),
    (dict(mask=16, ms=(0, 0, 32, 2)), 1),
    (dict(mask=16, ms=(-1, 0, 32, 1)), 1),
])
def test_invalid_problems_rejected(sdpa_lib, kw, status):
    p = P(**kw)
    name, st = S.sdpa_select_kernel(p)
    assert (name, st) == ("none", status)
    assert S.sdpa_workspace_size(p) == 0
    # sdpa_forward returns the same status before touching CUDA
    assert S.sdpa_forward_raw(p, 256, 256, 256, 256, None, None, 0, None) == status


def test_null_and_misaligned_pointers_rejected(sdpa_lib):
    p = P()
    assert S.sdpa_forward_raw(p, None, 256, 256, 256, None, None, 0, None) == 1
    assert S.sdpa_forward_raw(p, 256, None, 256, 256, None, None, 0, None) == 1
    assert S.sdpa_forward_raw(p, 256, 256, 256, None, None, None, 0, None) == 1
    assert S.sdpa_forward_raw(None, 256, 256, 256, 256, None, None, 0, None) == 1
    assert S.sdpa_forward_raw(p, 264, 256, 256, 256, None, None, 0, None) == 3
    assert S.sdpa_forward_raw(p, 256, 256, 256, 258, None, None, 0, None) == 3
    assert S.sdpa_forward_raw(p, 256, 256, 256, 256, 258, None, 0, None) == 3
    pm = P(mask=9)  # a mask must be aligned to its element size (2 bytes here)
    assert S.sdpa_forward_raw(pm, 256, 256, 256, 256, None, None, 0, None) == 3
    ps = P(sinks=2)
    assert S.sdpa_forward_raw(ps, 256, 256, 256, 256, None, None, 0, None) == 3


def test_nothing_to_compute_is_ok_without_pointers(sdpa_lib):
    for kw in (dict(B=0), dict(Lq=0), dict(Hq=0)):
        assert S.sdpa_forward_raw(P(**kw), None, None, None, None, None, None, 0, None) == 0


def test_decode_workspace_size_and_check(sdpa_lib):
    p = P(Lq=1, Lk=32768, B=8, Hq=32, Hkv=8, D=128)
    ws = S.sdpa_workspace_size(p)
    assert ws > 0 and ws % 256 == 0
    # bounded by B*Hq*splits*(D+1) floats with at most 1024 splits
    assert ws <= 8 * 32 * 1024 * 129 * 4 + 512
    # too small a workspace is refused before any launch
    assert S.sdpa_forward_raw(p, 256, 256, 256, 256, None, 256, ws - 1, None) == 4
    assert S.sdpa_forward_raw(p, 256, 256, 256, 256, None, None, 0, None) == 4
    # the fp16/bf16 prefill needs none
    assert S.sdpa_workspace_size(P()) == 0
    # the fp32 tensor-core prefill keeps bf16 hi/lo copies of q, k and v
    pf = P(dtype=S.SDPA_F32, B=1, Hq=4, Hkv=2, Lq=16, Lk=32, D=64)
    assert S.sdpa_workspace_size(pf) == 2 * 2 * 4 * 16 * 64 // 256 * 256 + 4 * 2 * 2 * 32 * 64
    assert S.sdpa_forward_raw(pf, 256, 256, 256, 256, None, None, 0, None) == 4


def _ws(rows, splits, D):
    """Workspace of a two-pass decode plan: rows x splits partial outputs of D
    floats, then rows x splits (m, l) pairs, each part 256-byte aligned."""
    a = lambda x: (x + 255) // 256 * 256
    return a(rows * splits * D * 4) + a(rows * splits * 2 * 4)


def test_tc128_decode_plan(sdpa_lib):
    """The head_dim-128 tensor-core decode plan, through the workspace it
    asks for (pure host logic; 152 SMs when no device is visible): splits of
    at most 14 tiles of 128 keys, as many per (kv head, batch) as one wave of
    two CTAs per SM holds, the tiles spread evenly over them."""
    # long decode: 64 (kv head, batch) units, 256 tiles: 4 splits a unit
    # would exceed 14 tiles, so 19 splits of 14 (the last one 4)
    p = P(Lq=1, Lk=32768, B=8, Hq=32, Hkv=8, D=128)
    assert S.sdpa_workspace_size(p) == _ws(8 * 32, 19, 128)
    # one tile: one split, O written directly, no workspace
    assert S.sdpa_workspace_size(P(Lq=1, Lk=128, B=1, Hq=8, Hkv=1, D=128)) == 0
    # a single kv head of 3001 keys (24 tiles): 24 one-tile splits fill the wave
    p1 = P(Lq=1, Lk=3001, B=1, Hq=8, Hkv=1, D=128, dtype=S.SDPA_F16)
    assert S.sdpa_workspace_size(p1) == _ws(8, 24, 128)
    prev = S.sdpa_debug_set_option("decode_splits", 1)
    try:
        # one forced split exceeds 14 tiles: two splits of 12
        assert S.sdpa_workspace_size(p1) == _ws(8, 2, 128)
    finally:
        S.sdpa_debug_set_option("decode_splits", prev)
    # one kv head of 131072 keys (1024 tiles): 304 splits would hold 3.4
    # tiles, so 256 splits of 4
    assert S.sdpa_workspace_size(P(Lq=1, Lk=131072, B=1, Hq=16, Hkv=1, D=128)) == \
        _ws(16, 256, 128)
    prev = S.sdpa_debug_set_option("decode_vector", 1)
    try:
        # the vector path's own plan (a different split count)
        ws_vec = S.sdpa_workspace_size(p1)
        assert ws_vec > 0 and ws_vec != _ws(8, 24, 128)
    finally:
        S.sdpa_debug_set_option("decode_vector", prev)
    # fp32 and more than 16 rows per kv head stay on the vector path
    assert S.sdpa_workspace_size(P(Lq=1, Lk=32768, B=8, Hq=32, Hkv=8, D=128,
                                   dtype=S.SDPA_F32)) != _ws(8 * 32, 19, 128)


def test_backward_workspace_size(sdpa_lib):
    """sdpa_backward_workspace_size (pure host): an fp32 dQ accumulator
    [B, Hq, Lq, D] and two fp32 [B, Hq, Lq] arrays, each 256-byte aligned, for
    fp32, fp16 and bf16 at head_dim 64 and 128, with or without per-batch
    length arrays; 0 for head_dim 512."""
    a = lambda x: (x + 255) // 256 * 256
    for dtype in (S.SDPA_F32, S.SDPA_F16, S.SDPA_BF16):
        for D in (64, 128):
            p = P(dtype=dtype, D=D, B=2, Hq=4, Hkv=2, Lq=33, Lk=70)
            rows = 2 * 4 * 33
            assert S.sdpa_backward_workspace_size(p) == a(rows * D * 4) + 2 * a(rows * 4)
    # per-batch lengths are accepted (only the pointers are looked at here)
    pl = S.make_params(2, 4, 2, 33, 70, 64, S.SDPA_BF16, 0.125, True, None, (0, 0, 0, 1), None,
                       seq_lens_q_ptr=256, seq_lens_kv_ptr=512)
    assert S.sdpa_backward_workspace_size(pl) == a(264 * 64 * 4) + 2 * a(264 * 4)
    assert S.sdpa_backward_workspace_size(P(D=512, Lq=4, Lk=9)) == 0


def test_python_binding_rejects_cpu_tensors(sdpa_lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        S.sdpa_forward(q, q, q)


def test_host_entry_rejects_bad_tensors(sdpa_lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 2, 4, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        S.sdpa_forward_host(q[0], q[0], q[0])  # not 4-D
    with pytest.raises(ValueError):
        S.sdpa_forward_host(q.transpose(1, 2), q, q)  # not contiguous


def _align(n):
    return (n + 255) // 256 * 256


@pytest.mark.parametrize("pieces", [1, 3, 8, 64])
def test_host_staging_size(sdpa_lib, pieces):
    # prefill (no workspace): device copies of q, k, v, o and lse, each
    # 256-byte aligned, whatever the number of pieces
    B_, Hq, Hkv, Lq, Lk, D = 2, 6, 3, 300, 333, 64
    p = S.make_params(B_, Hq, Hkv, Lq, Lk, D, S.SDPA_F16, 0.125)
    q = B_ * Hq * Lq * D * 2
    kv = B_ * Hkv * Lk * D * 2
    want = 2 * _align(q) + 2 * _align(kv) + _align(B_ * Hq * Lq * 4)
    assert S.sdpa_host_staging_size(p, pieces) == want
    # decode: plus two workspaces of the widest piece, which shrink as the
    # pieces get narrower
    d1 = S.sdpa_host_staging_size(S.make_params(2, 32, 8, 1, 32768, 128, S.SDPA_BF16, 0.088), 1)
    d8 = S.sdpa_host_staging_size(S.make_params(2, 32, 8, 1, 32768, 128, S.SDPA_BF16, 0.088), 8)
    assert d1 > d8 > 0


def test_host_entry_rejects_strided_problems(sdpa_lib):
    p = S.make_params(1, 4, 2, 300, 300, 64, S.SDPA_F16, 0.125, kv_capacity=512)
    assert S.sdpa_host_staging_size(p, 4) == 0
    lib = sdpa_lib
    assert lib.sdpa_forward_host(ctypes.byref(p), 256, 256, 256, 256, None, 256, 1 << 30, 4,
                                 None) == 2  # SDPA_ERR_UNSUPPORTED, before any CUDA call


def test_flags_are_checked(sdpa_lib):
    p = S.make_params(1, 4, 2, 300, 300, 64, S.SDPA_F16, 0.125, flags=S.SDPA_FLAG_SHARED_GPU)
    assert S.sdpa_select_kernel(p) == ("prefill_tc", 0)
    for ok in (S.SDPA_FLAG_BOOL_MASK, S.SDPA_FLAG_SHARED_GPU | S.SDPA_FLAG_BOOL_MASK):
        p = S.make_params(1, 4, 2, 300, 300, 64, S.SDPA_F16, 0.125, flags=ok)
        assert S.sdpa_select_kernel(p) == ("prefill_tc", 0)
    for bad in (8, 0x80000000):
        p = S.make_params(1, 4, 2, 300, 300, 64, S.SDPA_F16, 0.125, flags=bad)
        assert S.sdpa_select_kernel(p) == ("none", 1)
        assert S.sdpa_forward_raw(p, 256, 256, 256, 256, None, None, 0, None) == 1


def test_strides_are_checked(sdpa_lib):
    B, H, L, D = 1, 4, 300, 64
    dense = (H * L * D, L * D, D)
    bshd = (L * H * D, D, H * D)  # [B, L, H, D] seen as [B, H, L, D]
    p = S.make_params(B, H, H, L, L, D, S.SDPA_F16, 0.125, strides=(bshd, bshd, bshd, dense))
    assert p.flags & S.SDPA_FLAG_STRIDES
    assert S.sdpa_select_kernel(p) == ("prefill_tc", 0)
    # a negative stride is invalid; a row stride of 3 fp16 elements (6 bytes)
    # breaks the 16-byte rule; strides replace kv_capacity
    p = S.make_params(B, H, H, L, L, D, S.SDPA_F16, 0.125, strides=(dense, (-1, L * D, D), dense, dense))
    assert S.sdpa_select_kernel(p) == ("none", 1)
    p = S.make_params(B, H, H, L, L, D, S.SDPA_F16, 0.125, strides=(dense, dense, (H * L * D, L * D, 3), dense))
    assert S.sdpa_select_kernel(p) == ("none", 3)
    p = S.make_params(B, H, H, L, L, D, S.SDPA_F16, 0.125, kv_capacity=400,
                      strides=(dense, dense, dense, dense))
    assert S.sdpa_select_kernel(p) == ("none", 1)
    # fp32 rows: 4 elements are 16 bytes
    p = S.make_params(B, H, H, L, L, D, S.SDPA_F32, 0.125, strides=(dense, dense, (H * L * D, L * D, 68), dense))
    assert S.sdpa_select_kernel(p) == ("prefill_tc_f32", 0)


def test_kv_capacity_and_length_arrays_are_checked(sdpa_lib):
    # a KV cache must hold at least the keys used
    p = S.make_params(1, 4, 2, 16, 32, 64, S.SDPA_BF16, 0.125, kv_capacity=31)
    assert S.sdpa_select_kernel(p) == ("none", 1)
    assert S.sdpa_forward_raw(p, 256, 256, 256, 256, None, None, 0, None) == 1
    p = S.make_params(1, 4, 2, 16, 32, 64, S.SDPA_BF16, 0.125, kv_capacity=-1)
    assert S.sdpa_select_kernel(p) == ("none", 1)
    p = S.make_params(1, 4, 2, 16, 32, 64, S.SDPA_BF16, 0.125, kv_capacity=64)
    assert S.sdpa_select_kernel(p) == ("prefill_tc", 0)
    # per-batch length arrays are int32: 4-byte aligned
    p = S.make_params(1, 4, 2, 16, 32, 64, S.SDPA_BF16, 0.125, seq_lens_q_ptr=258)
    assert S.sdpa_forward_raw(p, 256, 256, 256, 256, None, None, 0, None) == 3
    p = S.make_params(1, 4, 2, 16, 32, 64, S.SDPA_BF16, 0.125, seq_lens_kv_ptr=258)
    assert S.sdpa_forward_raw(p, 256, 256, 256, 256, None, None, 0, None) == 3
