"""Seeded synthetic inputs and the named workloads.

This module holds no arithmetic of the attention method: it only draws
random numbers and rounds them to the storage dtype.  The same tensors feed
the CUDA path and the CPU oracle.

Recipe: numpy ``default_rng(seed)`` (PCG64), ``standard_normal`` in float32,
drawn in the order Q, K, V, then sinks (times ``sink_scale``), then the mask;
each rounded to the storage dtype with round-to-nearest-even.  Seed 0 for
every named workload.  The shapes are those of the workloads on the pages:
the SD3-8B diffusion-transformer self-attention of MLX PR #964 (B=2, H=38,
L up to 4250, D=64) and the Gemma-4 global-attention decode of MLX PR #4459
(D=512, 32 query heads over 4 KV heads, 1024 keys); their weights are not
needed and N(0,1) values stand in for activations.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lk: int
    D: int
    dtype: str  # "float32" | "float16" | "bfloat16"
    causal: bool = False
    sinks: bool = False
    sink_scale: float = 1.0
    # None | "full" | "row" (broadcast over heads/batch) | "key": additive;
    # "bool_full" | "bool_key": boolean (True = visible)
    mask: str | None = None
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))

    def visible_pairs(self) -> int:
        """(query, key) pairs the causal rule leaves visible, per (b, h)."""
        if not self.causal:
            return self.Lq * self.Lk
        off = self.Lk - self.Lq
        return sum(min(self.Lk, max(0, i + off + 1)) for i in range(self.Lq))

    def flops(self) -> int:
        """Algorithmic FLOPs: 4 D per visible (query, key) pair (QK^T and PV)."""
        return 4 * self.D * self.B * self.Hq * self.visible_pairs()

    def kv_bytes(self) -> int:
        """Bytes of K and V that must be read once."""
        es = 4 if self.dtype == "float32" else 2
        return 2 * self.B * self.Hkv * self.Lk * self.D * es


# Named workloads (the configurations the pages' workloads fix).
TINY = Workload("tiny_mha_f32", 1, 2, 2, 128, 128, 64, "float32")
DIT_F16 = Workload("dit_b2_h38_l4250_d64_f16", 2, 38, 38, 4250, 4250, 64, "float16")
DIT_F32 = Workload("dit_b2_h38_l4250_d64_f32", 2, 38, 38, 4250, 4250, 64, "float32")
CAUSAL_GQA = Workload("causal_gqa_l8192_d128_bf16", 1, 32, 8, 8192, 8192, 128, "bfloat16",
                      causal=True)
DECODE_D512 = {
    (b, dt, s): Workload("decode_d512_b%d_%s%s" % (b, dt, "_sinks" if s else ""), b, 32, 4, 1,
                         1024, 512, dt, sinks=s)
    for b in (1, 2) for dt in ("bfloat16", "float16", "float32") for s in (False, True)
}
DECODE_LONG = Workload("decode_long_b8_kl32768_d128_bf16", 8, 32, 8, 1, 32768, 128, "bfloat16")
# The D512 decode workload's heads (32 query heads over 4 KV heads, head_dim
# 512) over a 4096-token prompt: the prefill that precedes that decode.
PREFILL_D512 = Workload("prefill_d512_b1_h32_kv4_l4096_bf16_causal", 1, 32, 4, 4096, 4096, 512,
                        "bfloat16", causal=True)

NAMED = {w.name: w for w in [TINY, DIT_F16, DIT_F32, CAUSAL_GQA, DECODE_LONG, PREFILL_D512,
                             *DECODE_D512.values()]}


def _torch_dtype(name):
    import torch
    return {"float32": torch.float32, "float16": torch.float16, "bfloat16": torch.bfloat16}[name]


def make_inputs(w: Workload):
    """Host tensors (torch, CPU) of the workload in its storage dtype.

    Returns dict(q, k, v, sinks (float32 or None), mask (storage dtype or None)).
    """
    import torch
    rng = np.random.default_rng(w.seed)
    tdt = _torch_dtype(w.dtype)

    def draw(shape):
        a = rng.standard_normal(size=shape, dtype=np.float32)
        return torch.from_numpy(a).to(tdt)

    q = draw((w.B, w.Hq, w.Lq, w.D))
    k = draw((w.B, w.Hkv, w.Lk, w.D))
    v = draw((w.B, w.Hkv, w.Lk, w.D))
    sinks = None
    if w.sinks:
        sinks = torch.from_numpy(
            (rng.standard_normal(size=(w.Hq,), dtype=np.float32) * np.float32(w.sink_scale)))
    mask = None
    if w.mask in ("bool_full", "bool_key"):
        shape = (w.B, w.Hq, w.Lq, w.Lk) if w.mask == "bool_full" else (w.B, 1, 1, w.Lk)
        keep = rng.random(size=shape) >= 0.3  # about 30% of the keys removed
        if w.mask == "bool_full":
            keep[0, 0, 0, :] = False  # one row sees no key
        mask = torch.from_numpy(keep)
    elif w.mask is not None:
        shape = {"full": (w.B, w.Hq, w.Lq, w.Lk), "row": (1, 1, w.Lq, w.Lk),
                 "key": (w.B, 1, 1, w.Lk)}[w.mask]
        m = rng.standard_normal(size=shape, dtype=np.float32)
        hide = rng.random(size=shape) < 0.1  # about 10% of the keys removed
        m[hide] = -np.inf
        mask = torch.from_numpy(m).to(tdt)
    return dict(q=q, k=k, v=v, sinks=sinks, mask=mask)


def as_float64(t):
    """Exact widening of a stored tensor to a float64 numpy array."""
    import torch
    return t.to(torch.float64).numpy()
