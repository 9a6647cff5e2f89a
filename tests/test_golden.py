"""Figures the pages print, checked against the workloads and closed forms."""
import os

from scaled_dot_product_fwd_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_d512_cases_match_decode_workloads():
    cases = {r[0]: r for r in rows("d512_cases.txt")}
    for name in ("b1_fp16", "b2_fp16", "sinks_fp16", "b1_bf16", "b1_fp32"):
        _, B, Hq, Hkv, qL, kL, D, dt, sinks, _ = cases[name]
        w = W.DECODE_D512[(int(B), dt, bool(int(sinks)))]
        assert (w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D, w.dtype, w.sinks) == (
            int(B), int(Hq), int(Hkv), int(qL), int(kL), int(D), dt, bool(int(sinks)))
        assert abs(w.scale - 512 ** -0.5) < 1e-15  # the reproducer's scale=d**-0.5
    # the five reported cases are all GQA factor 8 single-token decode
    for name in ("b1_fp16", "b2_fp16", "sinks_fp16", "b1_bf16", "b1_fp32"):
        assert int(cases[name][2]) // int(cases[name][3]) == 8 and cases[name][4] == "1"


def test_dit_memory_savings_closed_form():
    for B, H, L, es, bound in rows("dit_memory.txt"):
        saved = int(B) * int(H) * int(L) ** 2 * int(es)
        assert saved > float(bound)
    # the named DiT workload is the 4250-token case of the page
    w = W.DIT_F32
    assert (w.B, w.Hq, w.Lq, w.Lk, w.D) == (2, 38, 4250, 4250, 64)
    assert w.B * w.Hq * w.Lq * w.Lk * 4 == 5_491_000_000


def test_flop_and_byte_counts():
    # 4*D FLOPs per visible (query, key) pair
    assert W.DIT_F16.flops() == 4 * 64 * 2 * 38 * 4250 * 4250
    assert W.CAUSAL_GQA.visible_pairs() == 8192 * 8193 // 2
    assert W.CAUSAL_GQA.flops() == 4 * 128 * 32 * 8192 * 8193 // 2
    # K and V read once
    assert W.DECODE_LONG.kv_bytes() == 2 * 8 * 8 * 32768 * 128 * 2 == 1 << 30
