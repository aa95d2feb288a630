"""Pins of the fp64 CPU oracle against things other than itself: hand-derived
closed forms (tests/golden), pure-Python brute force on tiny inputs, the
torch float64 scaled_dot_product_attention library routine, and invariants of
the attention definition. Each planted mistake at the end must fail a pin."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.mha as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- closed forms

def _closed_form_cases():
    with open(os.path.join(GOLDEN, "closed_form_cases.json")) as f:
        return json.load(f)["cases"]


def check_closed_forms():
    for c in _closed_form_cases():
        kw = dict(causal=c["causal"], scale=c["scale"])
        if "q_heads" in c:
            q = np.array(c["q_heads"], dtype=np.float64).transpose(1, 0, 2)[None]  # [1,S,H,D]
            k = np.array(c["k"])[None, :, None, :]
            v = np.array(c["v"])[None, :, None, :]
            o, lse = oracle.attention(q, k, v, **kw)
            np.testing.assert_allclose(o[0].transpose(1, 0, 2), np.array(c["o_heads"]), atol=1e-12)
            np.testing.assert_allclose(lse[0], np.array(c["lse_heads"]), atol=1e-12)
            continue
        q = np.array(c["q"])[None, :, None, :]
        k = np.array(c["k"])[None, :, None, :]
        v = np.array(c["v"])[None, :, None, :]
        if "q_rope" in c:
            kw["q_rope"] = np.array(c["q_rope"])[None, :, None, :]
            kw["k_rope"] = np.array(c["k_rope"])[None]
        if "q_scale" in c:
            kw["q_scale"] = np.array(c["q_scale"])[None, None, :]
            kw["k_scale"] = np.array(c["k_scale"])[None, None, :]
        o, lse = oracle.attention(q, k, v, **kw)
        np.testing.assert_allclose(o[0, :, 0], np.array(c["o"]), atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(lse[0, 0], np.array(c["lse"]), atol=1e-12, err_msg=c["name"])


def test_closed_forms():
    check_closed_forms()


# ---------------------------------------------------------------- brute force

def brute_force(q, k, v, causal, scale, q_rope=None, k_rope=None, q_scale=None, k_scale=None, cu=None):
    """Pure-Python enumeration: every score by an explicit loop over depth,
    softmax by explicit sums. Fixed layout [B,S,H,D] or packed [T,H,D]."""
    if cu is None:
        B, S, Hq, _ = q.shape
        seqs = [(b, 0, S) for b in range(B)]
    else:
        Hq = q.shape[1]
        seqs = [(b, int(cu[b]), int(cu[b + 1])) for b in range(len(cu) - 1)]
    Hkv = k.shape[-2]
    g = Hq // Hkv
    dv = v.shape[-1]
    o = np.zeros(q.shape[:-1] + (dv,))
    lse = np.zeros((len(seqs), Hq, q.shape[1]) if cu is None else (Hq, q.shape[0]))
    for b, t0, t1 in seqs:
        n = t1 - t0
        for h in range(Hq):
            hk = h // g
            for i in range(n):
                def qv(d):
                    return q[b, i, h, d] if cu is None else q[t0 + i, h, d]
                s = []
                for j in range(n):
                    if causal and j > i:
                        continue
                    kk = (lambda d: k[b, j, hk, d]) if cu is None else (lambda d: k[t0 + j, hk, d])
                    dot = sum(qv(d) * kk(d) for d in range(q.shape[-1]))
                    if q_rope is not None:
                        qr = q_rope[b, i, h] if cu is None else q_rope[t0 + i, h]
                        kr = k_rope[b, j] if cu is None else k_rope[t0 + j]
                        dot += sum(qr[r] * kr[r] for r in range(len(qr)))
                    val = scale * dot
                    if q_scale is not None:
                        qs = q_scale[b, h, i] if cu is None else q_scale[h, t0 + i]
                        ks = k_scale[b, hk, j] if cu is None else k_scale[hk, t0 + j]
                        val *= qs * ks
                    s.append((j, val))
                mx = max(val for _, val in s)
                tot = sum(math.exp(val - mx) for _, val in s)
                l = mx + math.log(tot)
                acc = [0.0] * dv
                for j, val in s:
                    w = math.exp(val - l)
                    vj = v[b, j, hk] if cu is None else v[t0 + j, hk]
                    for d in range(dv):
                        acc[d] += w * vj[d]
                if cu is None:
                    o[b, i, h] = acc
                    lse[b, h, i] = l
                else:
                    o[t0 + i, h] = acc
                    lse[h, t0 + i] = l
    return o, lse


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


BRUTE_CASES = [
    # (B, S, Hq, Hkv, D, Dv, R, causal, fp8scales)
    (2, 5, 2, 2, 4, 3, 0, True, False),
    (1, 6, 4, 2, 3, 5, 0, False, False),
    (2, 4, 2, 1, 4, 4, 2, True, False),
    (1, 7, 2, 2, 8, 2, 0, True, True),
    (1, 3, 6, 3, 2, 2, 0, False, True),
]


def check_brute_force():
    for n, (B, S, Hq, Hkv, D, Dv, R, causal, sc) in enumerate(BRUTE_CASES):
        q = _rand((B, S, Hq, D), 10 * n)
        k = _rand((B, S, Hkv, D), 10 * n + 1)
        v = _rand((B, S, Hkv, Dv), 10 * n + 2)
        kw = dict(causal=causal, scale=0.7)
        if R:
            kw["q_rope"] = _rand((B, S, Hq, R), 10 * n + 3)
            kw["k_rope"] = _rand((B, S, R), 10 * n + 4)
        if sc:
            kw["q_scale"] = np.abs(_rand((B, Hq, S), 10 * n + 5)) + 0.1
            kw["k_scale"] = np.abs(_rand((B, Hkv, S), 10 * n + 6)) + 0.1
        o, lse = oracle.attention(q, k, v, **kw)
        ob, lb = brute_force(q, k, v, **kw)
        np.testing.assert_allclose(o, ob, atol=1e-12, rtol=0)
        np.testing.assert_allclose(lse, lb, atol=1e-12, rtol=0)
    # packed layout, including a length-1 sequence
    lens = [3, 1, 4]
    cu = np.cumsum([0] + lens)
    T = int(cu[-1])
    q, k, v = _rand((T, 4, 3), 91), _rand((T, 2, 3), 92), _rand((T, 2, 2), 93)
    for causal in (True, False):
        o, lse = oracle.attention(q, k, v, causal=causal, scale=0.9, cu_seqlens_q=cu, cu_seqlens_k=cu)
        ob, lb = brute_force(q, k, v, causal, 0.9, cu=cu)
        np.testing.assert_allclose(o, ob, atol=1e-12, rtol=0)
        np.testing.assert_allclose(lse, lb, atol=1e-12, rtol=0)


def test_brute_force_tiny():
    check_brute_force()


# ---------------------------------------------------------------- library routine

def check_sdpa():
    """torch float64 scaled_dot_product_attention (its causal mask is the
    top-left lower triangle) and torch.logsumexp of the library matmul."""
    for causal, (B, Sq, Sk, H, D, Dv) in itertools.product(
            (True, False), [(2, 33, 33, 3, 16, 8), (1, 70, 70, 2, 64, 64), (1, 17, 40, 2, 8, 8)]):
        if causal and Sq != Sk:
            continue
        q = torch.from_numpy(_rand((B, Sq, H, D), Sq + D))
        k = torch.from_numpy(_rand((B, Sk, H, D), Sk + D + 1))
        v = torch.from_numpy(_rand((B, Sk, H, Dv), Sk + Dv + 2))
        scale = 1.0 / math.sqrt(D)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2), is_causal=causal, scale=scale)
        s = torch.matmul(q.transpose(1, 2), k.transpose(1, 2).transpose(-1, -2)) * scale
        if causal:
            s = s.masked_fill(torch.ones(Sq, Sk, dtype=torch.bool).triu(1), float("-inf"))
        lse_ref = torch.logsumexp(s, dim=-1)
        o, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), causal=causal, scale=scale)
        np.testing.assert_allclose(o, ref.transpose(1, 2).numpy(), atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref.numpy(), atol=1e-12)


def test_sdpa_library():
    check_sdpa()


# ---------------------------------------------------------------- invariants

def check_constant_v():
    q, k = _rand((1, 9, 2, 4), 1), _rand((1, 9, 2, 4), 2)
    v = np.full((1, 9, 2, 3), 2.5)
    for causal in (True, False):
        o, _ = oracle.attention(q, k, v, causal=causal, scale=1.3)
        np.testing.assert_allclose(o, 2.5, atol=1e-13)


def check_causal_row0_and_single_key():
    q, k, v = _rand((2, 6, 2, 5), 3), _rand((2, 6, 2, 5), 4), _rand((2, 6, 2, 3), 5)
    o, lse = oracle.attention(q, k, v, causal=True, scale=0.4)
    np.testing.assert_allclose(o[:, 0], v[:, 0], atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], 0.4 * np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0]), atol=1e-13)
    o1, l1 = oracle.attention(q, k[:, :1], v[:, :1], causal=False, scale=0.4)
    np.testing.assert_allclose(o1, np.broadcast_to(v[:, :1], o1.shape), atol=1e-14)
    np.testing.assert_allclose(l1, 0.4 * np.einsum("bshd,bhd->bhs", q, k[:, 0]), atol=1e-13)


def check_permutation():
    q, k, v = _rand((1, 7, 2, 4), 6), _rand((1, 11, 2, 4), 7), _rand((1, 11, 2, 3), 8)
    perm = np.random.default_rng(9).permutation(11)
    o, lse = oracle.attention(q, k, v, causal=False, scale=0.8)
    op, lp = oracle.attention(q, k[:, perm], v[:, perm], causal=False, scale=0.8)
    np.testing.assert_allclose(o, op, atol=1e-13)
    np.testing.assert_allclose(lse, lp, atol=1e-13)


def check_zero_q():
    k, v = _rand((1, 10, 1, 4), 10), _rand((1, 10, 1, 3), 11)
    q = np.zeros((1, 10, 1, 4))
    o, lse = oracle.attention(q, k, v, causal=True, scale=1.0)
    for i in range(10):
        np.testing.assert_allclose(o[0, i, 0], v[0, :i + 1, 0].mean(axis=0), atol=1e-13)
        assert abs(lse[0, 0, i] - math.log(i + 1)) < 1e-13


def check_gqa_equals_repeated_mha():
    q = _rand((2, 8, 6, 4), 12)
    k, v = _rand((2, 8, 2, 4), 13), _rand((2, 8, 2, 3), 14)
    o, lse = oracle.attention(q, k, v, causal=True, scale=0.5)
    kr = np.repeat(k, 3, axis=2)   # query heads 0,1,2 -> kv head 0; 3,4,5 -> 1
    vr = np.repeat(v, 3, axis=2)
    o2, l2 = oracle.attention(q, kr, vr, causal=True, scale=0.5)
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(lse, l2, atol=1e-14)


def check_varlen_equals_independent():
    lens = [5, 1, 9, 3]
    cu = np.cumsum([0] + lens)
    T = int(cu[-1])
    q, k, v = _rand((T, 4, 3), 15), _rand((T, 2, 3), 16), _rand((T, 2, 4), 17)
    qr, kr = _rand((T, 4, 2), 18), _rand((T, 2), 19)
    o, lse = oracle.attention(q, k, v, causal=True, scale=0.6, q_rope=qr, k_rope=kr,
                              cu_seqlens_q=cu, cu_seqlens_k=cu)
    for b in range(len(lens)):
        a, e = cu[b], cu[b + 1]
        ob, lb = oracle.attention(q[None, a:e], k[None, a:e], v[None, a:e], causal=True, scale=0.6,
                                  q_rope=qr[None, a:e], k_rope=kr[None, a:e])
        np.testing.assert_allclose(o[a:e], ob[0], atol=1e-14)
        np.testing.assert_allclose(lse[:, a:e], lb[0], atol=1e-14)


def check_rope_equals_concat():
    B, S, H, D, R = 2, 9, 3, 4, 2
    q, k, v = _rand((B, S, H, D), 20), _rand((B, S, H, D), 21), _rand((B, S, H, 3), 22)
    qr, kr = _rand((B, S, H, R), 23), _rand((B, S, R), 24)
    o, lse = oracle.attention(q, k, v, causal=True, scale=0.3, q_rope=qr, k_rope=kr)
    qc = np.concatenate([q, qr], axis=-1)
    kc = np.concatenate([k, np.repeat(kr[:, :, None, :], H, axis=2)], axis=-1)
    o2, l2 = oracle.attention(qc, kc, v, causal=True, scale=0.3)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(lse, l2, atol=1e-13)


def check_scales():
    B, S, H, D = 1, 8, 2, 4
    q, k, v = _rand((B, S, H, D), 25), _rand((B, S, H, D), 26), _rand((B, S, H, 3), 27)
    qs = np.abs(_rand((B, H, S), 28)) + 0.2
    ks = np.abs(_rand((B, H, S), 29)) + 0.2
    o, lse = oracle.attention(q, k, v, causal=True, scale=0.5, q_scale=qs, k_scale=ks)
    # the dequantised values Q8*q_scale, K8*k_scale in plain attention
    qd = q * qs.transpose(0, 2, 1)[..., None]
    kd = k * ks.transpose(0, 2, 1)[..., None]
    o2, l2 = oracle.attention(qd, kd, v, causal=True, scale=0.5)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(lse, l2, atol=1e-13)
    ones = np.ones((B, H, S))
    o3, l3 = oracle.attention(q, k, v, causal=True, scale=0.5, q_scale=ones, k_scale=ones)
    o4, l4 = oracle.attention(q, k, v, causal=True, scale=0.5)
    np.testing.assert_array_equal(o3, o4)
    np.testing.assert_array_equal(l3, l4)


def check_score_shift():
    """A constant c added to every score of a row (here through a constant
    rope part) leaves O unchanged and moves LSE by exactly c."""
    B, S, H, D = 1, 6, 2, 4
    q, k, v = _rand((B, S, H, D), 30), _rand((B, S, H, D), 31), _rand((B, S, H, 3), 32)
    qr = np.full((B, S, H, 1), 2.0)
    kr = np.full((B, S, 1), 1.5)
    o, lse = oracle.attention(q, k, v, causal=True, scale=0.5, q_rope=qr, k_rope=kr)
    o2, l2 = oracle.attention(q, k, v, causal=True, scale=0.5)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(lse, l2 + 0.5 * 3.0, atol=1e-13)


def check_causality():
    """Causal rows do not depend on keys or values after them."""
    q, k, v = _rand((1, 8, 2, 4), 33), _rand((1, 8, 2, 4), 34), _rand((1, 8, 2, 3), 35)
    o, lse = oracle.attention(q, k, v, causal=True, scale=1.0)
    k2, v2 = k.copy(), v.copy()
    k2[:, 5:] = 100.0
    v2[:, 5:] = -7.0
    o2, l2 = oracle.attention(q, k2, v2, causal=True, scale=1.0)
    np.testing.assert_array_equal(o[:, :5], o2[:, :5])
    np.testing.assert_array_equal(lse[:, :, :5], l2[:, :, :5])
    assert not np.allclose(o[:, 5:], o2[:, 5:])


def check_empty_rows():
    cu = np.array([0, 3, 3])
    q, k, v = _rand((3, 1, 2), 36), _rand((3, 1, 2), 37), _rand((3, 1, 2), 38)
    cuk = np.array([0, 0, 3])   # sequence 0 has 3 queries and no key
    o, lse = oracle.attention(q, k, v, causal=False, scale=1.0, cu_seqlens_q=cu, cu_seqlens_k=cuk)
    np.testing.assert_array_equal(o[:3], 0.0)
    assert np.all(np.isneginf(lse[:, :3]))


def check_rows_api():
    q, k, v = _rand((2, 12, 4, 4), 39), _rand((2, 12, 2, 4), 40), _rand((2, 12, 2, 3), 41)
    o, lse = oracle.attention(q, k, v, causal=True, scale=0.5)
    rows = [(0, 0, 0), (1, 3, 11), (0, 2, 7), (1, 1, 4)]
    ro, rl = oracle.attention_rows(q, k, v, rows, causal=True, scale=0.5)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(ro[n], o[b, i, h], atol=1e-14, rtol=0)
        assert abs(rl[n] - lse[b, h, i]) < 1e-14


INVARIANTS = [check_constant_v, check_causal_row0_and_single_key, check_permutation, check_zero_q,
              check_gqa_equals_repeated_mha, check_varlen_equals_independent, check_rope_equals_concat,
              check_scales, check_score_shift, check_causality, check_empty_rows, check_rows_api]


@pytest.mark.parametrize("check", INVARIANTS, ids=lambda f: f.__name__)
def test_invariant(check):
    check()


ALL_PINS = [check_closed_forms, check_brute_force, check_sdpa] + INVARIANTS


def _pins_fail():
    failed = []
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    return failed


# ---------------------------------------------------------------- planted mistakes

def _scores_dropped_rope(qh, kh, scale, qr=None, kr=None, qs=None, ks=None):
    return _orig_scores(qh, kh, scale, None, None, qs, ks)


def _scores_transposed(qh, kh, scale, qr=None, kr=None, qs=None, ks=None):
    s = _orig_scores(qh, kh, scale, qr, kr, qs, ks)
    return s.T if s.shape[0] == s.shape[1] else s


def _scores_k_scale_by_row(qh, kh, scale, qr=None, kr=None, qs=None, ks=None):
    s = _orig_scores(qh, kh, scale, qr, kr, None, None)
    if qs is not None:
        s = s * qs[:, None] * ks[: s.shape[0], None]
    return s


def _mask_strict(sq, sk, causal, rows=None):
    rows = np.arange(sq) if rows is None else np.asarray(rows)
    m = _orig_mask(sq, sk, causal, rows)
    if causal:
        m = np.arange(sk)[None, :] < rows[:, None]
    return m


def _softmax_log2(s, visible):
    w, lse = _orig_softmax(s, visible)
    return w, lse / math.log(2.0)


def _softmax_no_max(s, visible):
    w, lse = _orig_softmax(s, visible)
    return w, lse - np.where(visible, s, -np.inf).max(axis=1)


_orig_scores = oa.scores
_orig_mask = oa.visible_mask
_orig_softmax = oa.softmax_lse

MUTANTS = {
    "dropped_rope_term": ("scores", _scores_dropped_rope),
    "transposed_scores": ("scores", _scores_transposed),
    "k_scale_indexed_by_query": ("scores", _scores_k_scale_by_row),
    "causal_mask_excludes_diagonal": ("visible_mask", _mask_strict),
    "lse_in_log2": ("softmax_lse", _softmax_log2),
    "lse_drops_max": ("softmax_lse", _softmax_no_max),
    "gqa_head_interleaved": ("kv_head_of", lambda h, hq, hkv: h % hkv),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(oa, attr, fn)
    failed = _pins_fail()
    assert failed, f"planted mistake {name} passed every pin"
