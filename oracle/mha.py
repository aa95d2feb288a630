"""Plain CPU float64 oracle of the fused attention forward.

TEST INFRASTRUCTURE. Only the tests, the smoke check of ``__graft_entry__``
and the CPU-baseline leg of ``bench.py`` may import this module. The product
path (the C-ABI library and its Python binding) never imports or calls it, and
this module imports nothing from the product.

What is computed: the forward pass of the flash-attention kernel whose
shared-memory layout the "SM100AttentionSMem" page documents (description),
including the two optional parts listed in that page's Parameters section, a
rope sub-depth of Q and K and a per-token scale of Q and K:

  for every sequence b, query head h and query row i:
    g     = Hq / Hkv,  hk = h // g               (consecutive query heads share a KV head)
    J_i   = { j < Sk_b : not causal or j <= i }   (causal: query i sees keys 0..i)
    s_ij  = scale * ( q_i . k_j  +  q_rope_i . k_rope_j )          (rope part optional)
    s_ij  = scale * q_scale_i * k_scale_j * ( Q8_i . K8_j )        (per-token scaled FP8)
    LSE_i = m + ln sum_{j in J_i} exp(s_ij - m),  m = max_{j in J_i} s_ij
    O_i   = sum_{j in J_i} exp(s_ij - LSE_i) v_j
  A row with empty J_i gets O_i = 0 and LSE_i = -inf.

It materialises the whole score matrix of one (sequence, head) and uses a
library matmul, exp and log as its only primitives; there is no tiling, no
online softmax and no reordering beyond the definition above.

Array conventions (numpy float64; the exact values of the GPU inputs):
  fixed length: q [B,Sq,Hq,D], k [B,Sk,Hkv,D], v [B,Sk,Hkv,Dv],
                q_rope [B,Sq,Hq,R], k_rope [B,Sk,R],
                q_scale [B,Hq,Sq], k_scale [B,Hkv,Sk];
                returns O [B,Sq,Hq,Dv], LSE [B,Hq,Sq].
  packed:       q [Tq,Hq,D], k [Tk,Hkv,D], v [Tk,Hkv,Dv], q_rope [Tq,Hq,R],
                k_rope [Tk,R], q_scale [Hq,Tq], k_scale [Hkv,Tk],
                cu_seqlens_q / cu_seqlens_k int arrays of length B+1;
                returns O [Tq,Hq,Dv], LSE [Hq,Tq].
"""
from __future__ import annotations

import numpy as np


def scores(qh, kh, scale, qr=None, kr=None, qs=None, ks=None):
    """Scaled scores of one (sequence, head): s_ij as defined in the header.

    qh [Sq,D], kh [Sk,D]; optional rope parts qr [Sq,R], kr [Sk,R]
    (rope parameter of the SM100AttentionSMem page) and per-token scales
    qs [Sq], ks [Sk] (its scale parameter: per-token scale for Q and K).
    """
    s = qh @ kh.T
    if qr is not None:
        s = s + qr @ kr.T
    s = scale * s
    if qs is not None:
        s = s * qs[:, None] * ks[None, :]
    return s


def visible_mask(sq, sk, causal, rows=None):
    """Boolean [len(rows), Sk]: key j visible to query i (j <= i when causal)."""
    rows = np.arange(sq) if rows is None else np.asarray(rows)
    cols = np.arange(sk)
    if causal:
        return cols[None, :] <= rows[:, None]
    return np.ones((len(rows), sk), dtype=bool)


def softmax_lse(s, visible):
    """Row-wise LSE over the visible entries and the normalised weights.

    LSE = m + ln sum exp(s - m) with m the row max over visible entries;
    weights = exp(s - LSE) on visible entries, 0 elsewhere. Rows without a
    visible entry get LSE = -inf and all-zero weights.
    """
    s = np.where(visible, s, -np.inf)
    any_vis = visible.any(axis=1)
    m = np.where(any_vis, s.max(axis=1, initial=-np.inf), 0.0)
    e = np.exp(s - m[:, None])                     # exp(-inf) = 0 on masked entries
    total = e.sum(axis=1)
    with np.errstate(divide="ignore"):
        lse = np.where(any_vis, m + np.log(np.where(any_vis, total, 1.0)), -np.inf)
    w = np.where(visible, np.exp(s - np.where(any_vis, lse, 0.0)[:, None]), 0.0)
    return w, lse


def attention_head(qh, kh, vh, scale, causal, qr=None, kr=None, qs=None, ks=None, rows=None):
    """O [n, Dv] and LSE [n] of one (sequence, head), for all query rows or
    the given row indices."""
    sq, sk = qh.shape[0], kh.shape[0]
    idx = np.arange(sq) if rows is None else np.asarray(rows, dtype=np.int64)
    s = scores(qh[idx], kh, scale,
               None if qr is None else qr[idx], kr,
               None if qs is None else qs[idx], ks)
    w, lse = softmax_lse(s, visible_mask(sq, sk, causal, idx))
    return w @ vh, lse


def _seq_bounds(cu, b):
    return int(cu[b]), int(cu[b + 1])


def _head_slices(q, k, v, q_rope, k_rope, q_scale, k_scale, b, h, hk, varlen, cu_q, cu_k):
    if varlen:
        q0, q1 = _seq_bounds(cu_q, b)
        k0, k1 = _seq_bounds(cu_k, b)
        qh, kh, vh = q[q0:q1, h], k[k0:k1, hk], v[k0:k1, hk]
        qr = None if q_rope is None else q_rope[q0:q1, h]
        kr = None if k_rope is None else k_rope[k0:k1]
        qs = None if q_scale is None else q_scale[h, q0:q1]
        ks = None if k_scale is None else k_scale[hk, k0:k1]
        return qh, kh, vh, qr, kr, qs, ks, q0
    qh, kh, vh = q[b, :, h], k[b, :, hk], v[b, :, hk]
    qr = None if q_rope is None else q_rope[b, :, h]
    kr = None if k_rope is None else k_rope[b]
    qs = None if q_scale is None else q_scale[b, h]
    ks = None if k_scale is None else k_scale[b, hk]
    return qh, kh, vh, qr, kr, qs, ks, 0


def _check_heads(hq, hkv):
    if hkv <= 0 or hq % hkv != 0:
        raise ValueError(f"query heads {hq} not a multiple of kv heads {hkv}")
    return hq // hkv


def kv_head_of(h, heads_q, heads_kv):
    """KV head read by query head h when heads_q / heads_kv query heads share
    one KV head: heads [hk*g, (hk+1)*g) map to hk (consecutive grouping)."""
    return h // (heads_q // heads_kv)


def attention(q, k, v, *, causal, scale, q_rope=None, k_rope=None,
              q_scale=None, k_scale=None, cu_seqlens_q=None, cu_seqlens_k=None):
    """Full O and LSE of every (sequence, head, row); layouts in the header."""
    varlen = cu_seqlens_q is not None
    if varlen:
        cu_k = cu_seqlens_k if cu_seqlens_k is not None else cu_seqlens_q
        nb = len(cu_seqlens_q) - 1
        hq, hkv = q.shape[1], k.shape[1]
        o = np.zeros(q.shape[:2] + (v.shape[-1],))
        lse = np.full((hq, q.shape[0]), -np.inf)
    else:
        cu_k = None
        nb, hq, hkv = q.shape[0], q.shape[2], k.shape[2]
        o = np.zeros(q.shape[:3] + (v.shape[-1],))
        lse = np.full((nb, hq, q.shape[1]), -np.inf)
    _check_heads(hq, hkv)
    for b in range(nb):
        for h in range(hq):
            hk = kv_head_of(h, hq, hkv)
            qh, kh, vh, qr, kr, qs, ks, base = _head_slices(
                q, k, v, q_rope, k_rope, q_scale, k_scale, b, h, hk, varlen, cu_seqlens_q, cu_k)
            if qh.shape[0] == 0:
                continue
            oh, lh = attention_head(qh, kh, vh, scale, causal, qr, kr, qs, ks)
            if varlen:
                o[base:base + qh.shape[0], h] = oh
                lse[h, base:base + qh.shape[0]] = lh
            else:
                o[b, :, h] = oh
                lse[b, h] = lh
    return o, lse


def attention_rows(q, k, v, rows, *, causal, scale, q_rope=None, k_rope=None,
                   q_scale=None, k_scale=None, cu_seqlens_q=None, cu_seqlens_k=None):
    """O [n, Dv] and LSE [n] for the listed (sequence, query head, row) triples,
    row index counted within its sequence. Same definition as ``attention``."""
    varlen = cu_seqlens_q is not None
    cu_k = (cu_seqlens_k if cu_seqlens_k is not None else cu_seqlens_q) if varlen else None
    hq = q.shape[1] if varlen else q.shape[2]
    hkv = k.shape[1] if varlen else k.shape[2]
    _check_heads(hq, hkv)
    o = np.zeros((len(rows), v.shape[-1]))
    lse = np.zeros(len(rows))
    for n, (b, h, i) in enumerate(rows):
        qh, kh, vh, qr, kr, qs, ks, _ = _head_slices(
            q, k, v, q_rope, k_rope, q_scale, k_scale, b, h, kv_head_of(h, hq, hkv), varlen, cu_seqlens_q, cu_k)
        oh, lh = attention_head(qh, kh, vh, scale, causal, qr, kr, qs, ks, rows=[i])
        o[n], lse[n] = oh[0], lh[0]
    return o, lse
