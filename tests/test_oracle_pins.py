"""Pins of the float64 oracle against facts the pages and the mathematics fix.

No page prints a worked example with output values, so the oracle is pinned
by closed forms, special cases that reduce to a textbook routine, invariants
of the definition, and a brute-force check of the online recurrence.  Each
pin is chosen so that a plausible mistake in the oracle (a dropped scale, a
wrong head index, a flipped causal test, a sink left out of the denominator,
an LSE without its max, a transposed mask) fails at least one of them;
test_planted_mistakes_are_caught shows that on mutated copies of the oracle.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import oracle as O

RNG = np.random.default_rng(1234)


def rand(*shape):
    return RNG.standard_normal(shape)


def textbook(q, k, v, scale, causal=False, mask=None, sinks=None):
    """Independent route: repeat K/V heads, masked score matrix, scipy softmax.

    Rows with nothing visible give O = 0, LSE = -inf (or the sink).
    """
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    kk = np.repeat(k, Hq // Hkv, axis=1)
    vv = np.repeat(v, Hq // Hkv, axis=1)
    s = scale * np.einsum("bhid,bhjd->bhij", q, kk)
    if mask is not None:
        s = s + np.broadcast_to(mask, s.shape)
    if causal:
        vis = np.tril(np.ones((Lq, Lk), bool), k=Lk - Lq)
        s = np.where(vis, s, -np.inf)
    if sinks is not None:
        col = np.broadcast_to(np.asarray(sinks).reshape(1, Hq, 1, 1), (B, Hq, Lq, 1))
        s = np.concatenate([s, col], axis=-1)
    o = np.zeros((B, Hq, Lq, D))
    lse = np.full((B, Hq, Lq), -np.inf)
    for b in range(B):
        for h in range(Hq):
            for i in range(Lq):
                row = s[b, h, i]
                if np.all(np.isneginf(row)):
                    continue
                p = softmax(row)
                lse[b, h, i] = logsumexp(row)
                o[b, h, i] = p[:Lk] @ vv[b, h]
    return o, lse


def close(a, b, tol=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    if a.shape != b.shape:
        return False
    fin = np.isfinite(b)
    if not np.array_equal(np.isfinite(a), fin):
        return False
    if not np.array_equal(a[~fin], b[~fin]):
        return False
    return bool(np.all(np.abs(a[fin] - b[fin]) <= tol * (1 + np.abs(b[fin]))))


# ------------------------------------------------------------------ pin suite
# Each pin takes an oracle build and returns True when it holds.

def pin_textbook(orc):
    ok = True
    for causal in (False, True):
        for use_mask in (False, True):
            for use_sinks in (False, True):
                B, Hq, Hkv, Lq, Lk, D = 2, 6, 3, 5, 9, 4
                q, k, v = rand(B, Hq, Lq, D), rand(B, Hkv, Lk, D), rand(B, Hkv, Lk, D)
                mask = rand(B, 1, Lq, Lk) if use_mask else None
                sinks = 2 * rand(Hq) if use_sinks else None
                o1, l1 = orc.sdpa(q, k, v, 0.37, causal, mask, sinks)
                o2, l2 = textbook(q, k, v, 0.37, causal, mask, sinks)
                ok &= close(o1, o2, 1e-11) and close(l1, l2, 1e-11)
    return ok


def pin_probs_sum_to_one(orc):
    B, Hq, Hkv, Lq, Lk, D = 1, 4, 2, 6, 11, 3
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hkv, Lk, D), rand(B, Hkv, Lk, D)
    _, lse, p = orc.sdpa(q, k, v, 0.8, True, rand(1, 1, Lq, Lk), None, want_probs=True)
    ok = np.all(np.abs(p.sum(-1) - 1) < 1e-12) and np.all(p >= 0)
    sinks = rand(Hq)
    _, lse_s, ps = orc.sdpa(q, k, v, 0.8, False, None, sinks, want_probs=True)
    sink_w = np.exp(sinks.reshape(1, Hq, 1) - lse_s)
    ok &= np.all(np.abs(ps.sum(-1) + sink_w - 1) < 1e-12)
    return bool(ok)


def pin_constant_v(orc):
    B, Hq, Hkv, Lq, Lk, D = 2, 4, 2, 7, 10, 5
    q, k = 3 * rand(B, Hq, Lq, D), rand(B, Hkv, Lk, D)
    c = rand(B, Hkv, 1, D)
    v = np.broadcast_to(c, (B, Hkv, Lk, D)).copy()
    o, _ = orc.sdpa(q, k, v, 0.5, True, rand(B, Hq, Lq, Lk), None)
    expect = np.repeat(c, Hq // Hkv, axis=1)
    return close(o, np.broadcast_to(expect, o.shape), 1e-12)


def pin_single_key(orc):
    B, Hq, Hkv, Lq, D = 1, 3, 1, 4, 6
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hkv, 1, D), rand(B, Hkv, 1, D)
    o, lse = orc.sdpa(q, k, v, 0.25, False, None, None)
    ok = close(o, np.broadcast_to(v, o.shape), 1e-14)
    expect_lse = 0.25 * (q @ k[0, 0, 0])  # the only score
    return ok and close(lse, expect_lse, 1e-13)


def pin_causal_row0(orc):
    B, Hq, L, D = 2, 2, 8, 4
    q, k, v = rand(B, Hq, L, D), rand(B, Hq, L, D), rand(B, Hq, L, D)
    o, lse = orc.sdpa(q, k, v, 0.6, True, None, None)
    ok = close(o[:, :, 0], v[:, :, 0], 1e-14)
    s00 = 0.6 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    return ok and close(lse[:, :, 0], s00, 1e-13)


def pin_uniform(orc):
    # scale 0: every visible key has weight 1/n; bottom-right causal with
    # Lq=3, Lk=7 leaves 5, 6, 7 keys visible to rows 0, 1, 2.
    B, Hq, Lq, Lk, D = 1, 2, 3, 7, 4
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hq, Lk, D), rand(B, Hq, Lk, D)
    o, lse = orc.sdpa(q, k, v, 0.0, True, None, None)
    ok = True
    for i, n in enumerate((5, 6, 7)):
        ok &= close(o[:, :, i], v[:, :, :n].mean(axis=2), 1e-13)
        ok &= close(lse[:, :, i], np.full((B, Hq), math.log(n)), 1e-13)
    return bool(ok)


def pin_sinks_shrink(orc):
    B, Hq, Hkv, Lq, Lk, D = 1, 4, 2, 5, 8, 3
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hkv, Lk, D), rand(B, Hkv, Lk, D)
    sinks = 3 * rand(Hq)
    o0, l0 = orc.sdpa(q, k, v, 0.5, False, None, None)
    o1, l1 = orc.sdpa(q, k, v, 0.5, False, None, sinks)
    s = sinks.reshape(1, Hq, 1)
    ok = close(l1, np.logaddexp(l0, s), 1e-12)
    ok &= close(o1, o0 * np.exp(l0 - l1)[..., None], 1e-12)
    ok &= bool(np.all(np.abs(o1) <= np.abs(o0) + 1e-15))
    return bool(ok)


def pin_mask_shift(orc):
    B, Hq, Lq, Lk, D = 1, 2, 4, 6, 3
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hq, Lk, D), rand(B, Hq, Lk, D)
    m = rand(B, Hq, Lq, Lk)
    o0, l0 = orc.sdpa(q, k, v, 0.7, False, m, None)
    o1, l1 = orc.sdpa(q, k, v, 0.7, False, m + 2.5, None)
    return close(o1, o0, 1e-12) and close(l1, l0 + 2.5, 1e-12)


def pin_mask_orientation(orc):
    # a mask that removes all but key j from row i picks V[j]
    B, Hq, Lq, Lk, D = 1, 1, 3, 5, 2
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hq, Lk, D), rand(B, Hq, Lk, D)
    m = np.full((B, Hq, Lq, Lk), -np.inf)
    pick = [4, 0, 2]
    for i, j in enumerate(pick):
        m[0, 0, i, j] = 0.0
    o, _ = orc.sdpa(q, k, v, 1.0, False, m, None)
    return close(o[0, 0], v[0, 0, pick], 1e-14)


def pin_permutation(orc):
    B, Hq, Lq, Lk, D = 1, 2, 4, 9, 3
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hq, Lk, D), rand(B, Hq, Lk, D)
    m = rand(B, Hq, Lq, Lk)
    perm = RNG.permutation(Lk)
    o0, l0 = orc.sdpa(q, k, v, 0.9, False, m, None)
    o1, l1 = orc.sdpa(q, k[:, :, perm], v[:, :, perm], 0.9, False, m[..., perm], None)
    return close(o1, o0, 1e-12) and close(l1, l0, 1e-12)


def pin_gqa(orc):
    B, Hq, Hkv, Lq, Lk, D = 2, 8, 2, 3, 5, 4
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hkv, Lk, D), rand(B, Hkv, Lk, D)
    o0, l0 = orc.sdpa(q, k, v, 0.5, False, None, None)
    o1, l1 = orc.sdpa(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), 0.5, False, None, None)
    return close(o0, o1, 1e-14) and close(l0, l1, 1e-14)


def pin_split_combine(orc):
    # the keys split in two, each part's (O, LSE) merged by LSE weights
    B, Hq, Lq, Lk, D = 1, 2, 3, 10, 4
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hq, Lk, D), rand(B, Hq, Lk, D)
    o, l = orc.sdpa(q, k, v, 0.5, False, None, None)
    oa, la = orc.sdpa(q, k[:, :, :4], v[:, :, :4], 0.5, False, None, None)
    ob, lb = orc.sdpa(q, k[:, :, 4:], v[:, :, 4:], 0.5, False, None, None)
    lm = np.logaddexp(la, lb)
    om = oa * np.exp(la - lm)[..., None] + ob * np.exp(lb - lm)[..., None]
    return close(om, o, 1e-12) and close(lm, l, 1e-12)


def pin_two_keys(orc):
    # two keys: weights are the logistic function of the score difference
    B, Hq, Lq, D = 1, 1, 4, 3
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hq, 2, D), rand(B, Hq, 2, D)
    o, lse = orc.sdpa(q, k, v, 1.3, False, None, None)
    s = 1.3 * q[0, 0] @ k[0, 0].T
    w0 = 1.0 / (1.0 + np.exp(s[:, 1] - s[:, 0]))
    expect = w0[:, None] * v[0, 0, 0] + (1 - w0)[:, None] * v[0, 0, 1]
    return close(o[0, 0], expect, 1e-13) and close(lse[0, 0], np.logaddexp(s[:, 0], s[:, 1]), 1e-13)


def pin_fully_masked(orc):
    B, Hq, Lq, Lk, D = 1, 2, 3, 4, 2
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hq, Lk, D), rand(B, Hq, Lk, D)
    m = np.zeros((B, Hq, Lq, Lk))
    m[0, :, 1, :] = -np.inf
    o, l = orc.sdpa(q, k, v, 1.0, False, m, None)
    ok = np.all(o[0, :, 1] == 0) and np.all(np.isneginf(l[0, :, 1]))
    sinks = np.array([0.5, -1.5])
    o, l = orc.sdpa(q, k, v, 1.0, False, m, sinks)
    ok &= np.all(o[0, :, 1] == 0) and np.allclose(l[0, :, 1], sinks, rtol=0, atol=0)
    return bool(ok)


def pin_online_bruteforce(orc):
    ok = True
    for Lq in (1, 2, 5):
        for Lk in range(max(1, Lq), 10):
            for D in (1, 2, 4):
                q, k, v = rand(1, 2, Lq, D), rand(1, 1, Lk, D), rand(1, 1, Lk, D)
                m = rand(1, 2, Lq, Lk)
                m[RNG.random(m.shape) < 0.2] = -np.inf
                sinks = rand(2)
                for causal, mask, sk in ((False, None, None), (True, None, None),
                                         (False, m, None), (True, m, sinks)):
                    o0, l0 = orc.sdpa(q, k, v, 0.9, causal, mask, sk)
                    for tile in range(1, Lk + 1):
                        o1, l1 = orc.sdpa_online(q, k, v, 0.9, tile, causal, mask, sk)
                        ok &= close(o1, o0, 1e-12) and close(l1, l0, 1e-12)
    return bool(ok)


def pin_bool_mask_selects_keys(orc):
    """A boolean mask keeps exactly the keys it marks True: each row equals
    plain attention over the selected keys alone (K and V rows dropped, no
    -inf arithmetic), with sinks and the causal rule; a row with no key
    selected gives O = 0 and LSE = -inf (the sink with sinks)."""
    ok = True
    for causal in (False, True):
        for with_sinks in (False, True):
            B, Hq, Hkv, Lq, Lk, D = 2, 4, 2, 5, 7, 3
            q, k, v = rand(B, Hq, Lq, D), rand(B, Hkv, Lk, D), rand(B, Hkv, Lk, D)
            sel = RNG.random((B, Hq, Lq, Lk)) < 0.6
            sel[0, 1, 2, :] = False  # one row keeps nothing
            sinks = rand(Hq) if with_sinks else None
            o, lse = orc.sdpa(q, k, v, 0.7, causal, sel, sinks)
            for b in range(B):
                for h in range(Hq):
                    g = h // (Hq // Hkv)
                    for i in range(Lq):
                        keep = [j for j in range(Lk) if sel[b, h, i, j]
                                and (not causal or j <= i + Lk - Lq)]
                        logits = [0.7 * float(q[b, h, i] @ k[b, g, j]) for j in keep]
                        if with_sinks:
                            logits.append(float(sinks[h]))
                        if not logits:
                            ok &= np.all(o[b, h, i] == 0) and np.isneginf(lse[b, h, i])
                            continue
                        mx = max(logits)
                        w = [math.exp(x - mx) for x in logits]
                        den = sum(w)
                        ref = sum(w[n] * v[b, g, j] for n, j in enumerate(keep)) / den \
                            if keep else np.zeros(D)
                        ok &= close(o[b, h, i], ref) and close(lse[b, h, i], mx + math.log(den))
    return bool(ok)


PINS = [pin_textbook, pin_probs_sum_to_one, pin_constant_v, pin_single_key, pin_causal_row0,
        pin_uniform, pin_sinks_shrink, pin_mask_shift, pin_mask_orientation, pin_permutation,
        pin_gqa, pin_split_combine, pin_two_keys, pin_fully_masked, pin_online_bruteforce,
        pin_bool_mask_selects_keys]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    assert pin(O.default())


def test_rows_subset_matches_full():
    B, Hq, Hkv, Lq, Lk, D = 2, 4, 2, 6, 9, 8
    q, k, v = rand(B, Hq, Lq, D), rand(B, Hkv, Lk, D), rand(B, Hkv, Lk, D)
    sinks = rand(Hq)
    rows = np.array([0, 5, 17, B * Hq * Lq - 1])
    o2, l2 = O.sdpa(q, k, v, 0.3, True, None, sinks, rows=rows)
    o3, l3 = O.sdpa(q, k, v, 0.3, True, None, sinks)
    assert close(o2, o3.reshape(-1, D)[rows], 0) and close(l2, l3.reshape(-1)[rows], 0)


# ------------------------------------------------------------- planted mistakes
SRC = os.path.join(os.path.dirname(O.__file__), "sdpa_oracle.c")
MUTATIONS = {
    "scale_dropped": ("double sj = scale * dot;", "double sj = dot;"),
    "gqa_index_modulo": ("const int64_t g = h / G; /* key/value head of query head h */",
                         "const int64_t g = h % Hkv;"),
    "causal_top_left": ("return j <= i + (Lk - Lq);", "return j <= i;"),
    "causal_flipped": ("return j <= i + (Lk - Lq);", "return j >= i + (Lk - Lq);"),
    "sink_not_in_denominator": ("if (sinks) den += exp(sinks[h] - m);", ""),
    "lse_without_max": ("if (lse) lse[n] = m + log(den);", "if (lse) lse[n] = log(den);"),
    "mask_transposed": ("if (mask) sj += mask_at(mask, mask_stride, b, h, i, j);",
                        "if (mask) sj += mask_at(mask, mask_stride, b, h, j % Lq, i % Lk);"),
    "value_row_of_query_head": ("const double* vj = v + ((b * Hkv + g) * Lk + j) * D;\n        for (int64_t d = 0; d < D; ++d) oi[d] += w * vj[d];",
                                "const double* vj = v + ((b * Hkv + (h % Hkv)) * Lk + j) * D;\n        for (int64_t d = 0; d < D; ++d) oi[d] += w * vj[d];"),
    "online_rescale_inverted": ("const double corr = exp(m - m_new); /* 0 when m was -inf */",
                                "const double corr = (m == -INFINITY) ? 0.0 : exp(m_new - m);"),
    "online_sum_not_rescaled": ("      l *= corr;\n", "\n"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert old in text, "mutation site not found: %s" % name
    mutant = O.compile_variant(text.replace(old, new, 1), str(tmp_path / ("m_%s.so" % name)))
    failed = [p.__name__ for p in PINS if not p(mutant)]
    assert failed, "planted mistake %s passed every pin" % name


# ------------------------------------------------------------ backward oracle
def _fd_grads(q, k, v, d_o, scale, causal, mask, sinks, h=1e-6):
    """Central differences of L = sum(O * dO) through the forward oracle."""
    def loss(q_, k_, v_):
        o, _ = O.sdpa(q_, k_, v_, scale, causal, mask, sinks)
        return float(np.sum(o * d_o))
    out = []
    for which in range(3):
        base = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(base[which])
        it = np.nditer(g, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [a.copy() for a in base]
            minus = [a.copy() for a in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            g[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        out.append(g)
    return out


@pytest.mark.parametrize("variant", ["plain", "causal", "mask", "bool_mask", "sinks_gqa",
                                     "causal_mask_sinks"])
def test_backward_oracle_matches_finite_differences(variant):
    """dQ, dK, dV of the backward oracle equal the central differences of the
    pinned forward oracle (loss = sum O * dO) on small problems."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, Lq, Lk, D = 1, 2, 2, 3, 4, 3
    if variant in ("sinks_gqa", "causal_mask_sinks"):
        Hq, Hkv = 4, 2
    q, k, v = (rng.standard_normal(s) for s in ((B, Hq, Lq, D), (B, Hkv, Lk, D), (B, Hkv, Lk, D)))
    d_o = rng.standard_normal((B, Hq, Lq, D))
    causal = variant in ("causal", "causal_mask_sinks")
    mask = sinks = None
    if variant in ("mask", "causal_mask_sinks"):
        mask = rng.standard_normal((B, Hq, Lq, Lk))
        mask[0, 0, 1, 2] = -np.inf
    if variant == "bool_mask":
        mask = rng.random((B, Hq, Lq, Lk)) < 0.7
        mask[0, 1, 0, :] = False  # a row that sees nothing: zero gradients
    if variant in ("sinks_gqa", "causal_mask_sinks"):
        sinks = rng.standard_normal(Hq)
    got = O.sdpa_backward(q, k, v, d_o, 0.8, causal, mask, sinks)
    want = _fd_grads(q, k, v, d_o, 0.8, causal, mask, sinks)
    for g, w in zip(got, want):
        assert np.max(np.abs(g - w)) < 1e-6 * max(1.0, np.max(np.abs(w)))


def test_backward_oracle_closed_forms():
    """q = 0 gives uniform attention: dV_j = (1/Lk) sum_i dO_i over the group's
    heads and dK = 0 (no score depends on k).  Without sinks the scores of a
    row are invariant to adding one vector to every key, so sum_j dK_j = 0."""
    rng = np.random.default_rng(8)
    B, Hq, Hkv, Lq, Lk, D = 2, 4, 2, 5, 6, 3
    k, v = rng.standard_normal((B, Hkv, Lk, D)), rng.standard_normal((B, Hkv, Lk, D))
    d_o = rng.standard_normal((B, Hq, Lq, D))
    dq, dk, dv = O.sdpa_backward(np.zeros((B, Hq, Lq, D)), k, v, d_o, 0.7)
    want = d_o.reshape(B, Hkv, 2, Lq, D).sum(axis=(2, 3))[:, :, None, :] / Lk
    assert close(dv, np.broadcast_to(want, dv.shape)) and close(dk, np.zeros_like(dk))
    q = rng.standard_normal((B, Hq, Lq, D))
    dq, dk, dv = O.sdpa_backward(q, k, v, d_o, 0.7, causal=True)
    assert close(dk.sum(axis=2), np.zeros((B, Hkv, D)))
