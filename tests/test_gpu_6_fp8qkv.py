"""All-FP8 attention (e4m3 Q, K and V; per-token Q/K scales; V depth-major,
no V scale): the kernel rounds the softmax weights to e4m3 before the P.V
product, so it is compared with the exact (fp64) attention over the same
e4m3 inputs through the error bound that rounding implies. Relative to the
row maximum each weight moves by at most 2^-4 of itself (normal e4m3) or
2^-10 (subnormal), so for output column d

  |O_d - O*_d| <= 2^-4 sum_j w_j |v_jd| + 2^-10 exp(max_j s_j - LSE) sum_j |v_jd|

(w the exact normalised weights, sums over visible keys), plus the final
bf16 rounding of O. LSE does not see the rounding (the row sums use the
unrounded weights) and keeps the 1e-3 bar; the relative RMS of O is held to
4e-2 (the RMS of a uniform relative error of at most 2^-4 is 2^-4/sqrt(3))."""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_sm100_gb300 import workloads as W
from helpers import f64, gather_rows, oracle_args, run_lib, v_for_oracle

S = W.AttnSpec
REL_RMS = 4e-2
LSE_TOL = 1e-3


def _fp8qkv(*a, **kw):
    return S(*a, qk_dtype="fp8", v_dtype="fp8", **kw)


CASES = {
    # name: (spec, num_splits)
    "causal_s300": (_fp8qkv(1, 2, 2, 300, 300, 128, 128, True, seed=110), 1),
    "causal_gqa_s1000": (_fp8qkv(2, 8, 2, 1000, 1000, 128, 128, True, seed=111), 1),
    "noncausal_sq200_sk512": (_fp8qkv(2, 4, 4, 200, 512, 128, 128, False, seed=112), 1),
    "noncausal_sk1": (_fp8qkv(1, 2, 2, 130, 16, 128, 128, False, seed=113), 1),
    "noncausal_split3": (_fp8qkv(1, 4, 2, 256, 2048, 128, 128, False, seed=114), 3),
    "causal_sq300_sk160": (_fp8qkv(1, 2, 2, 300, 160, 128, 128, True, seed=115), 1),
    # packed sequences: V's keys per sequence start on 16-key boundaries
    "packed_causal_gqa": (_fp8qkv(4, 8, 2, 640, 640, 128, 128, True, seed=117, lengths_q=(1, 300, 129, 640)), 1),
    "packed_noncausal_qk_differ": (_fp8qkv(3, 4, 4, 400, 400, 128, 128, False, seed=118, lengths_q=(257, 3, 130),
                                           lengths_k=(5, 400, 131)), 1),
    "packed_noncausal_split3": (_fp8qkv(2, 4, 2, 200, 1500, 128, 128, False, seed=119, lengths_q=(200, 77),
                                        lengths_k=(1500, 333)), 3),
}


def _bound_rows(inp, rows):
    """Per-element bound of the e4m3 rounding of the weights for (b, h, i) rows."""
    spec = inp["spec"]
    args = oracle_args(inp)
    q, k, v = f64(inp["q"]), f64(inp["k"]), v_for_oracle(inp)
    g = spec.heads_q // spec.heads_kv
    lq, lk = spec.seq_lengths()
    out = []
    for b, h, i in rows:
        hk = h // g
        if spec.varlen:
            a, c = int(args["cu_seqlens_q"][b]), int(args["cu_seqlens_k"][b])
            qr, kr, vr = q[a + i:a + i + 1, h], k[c:c + lk[b], hk], v[c:c + lk[b], hk]
            qs, ks = args["q_scale"][h, a + i:a + i + 1], args["k_scale"][hk, c:c + lk[b]]
        else:
            qr, kr, vr = q[b, i:i + 1, h], k[b, :, hk], v[b, :, hk]
            qs, ks = args["q_scale"][b, h, i:i + 1], args["k_scale"][b, hk]
        s = oracle.scores(qr, kr, args["scale"], qs=qs, ks=ks)
        vis = oracle.visible_mask(lq[b], lk[b], spec.causal, rows=[i])
        if not vis.any():
            out.append(np.zeros(vr.shape[-1]))
            continue
        w, lse = oracle.softmax_lse(s, vis)
        av = np.abs(vr)
        smax = np.where(vis, s, -np.inf).max()
        out.append(2.0 ** -4 * (w @ av)[0] + 2.0 ** -10 * np.exp(smax - lse[0]) * (vis[0] @ av))
    return np.array(out)


def _check(inp, o, lse, rows):
    spec = inp["spec"]
    o_ref, l_ref = oracle.attention_rows(f64(inp["q"]), f64(inp["k"]), v_for_oracle(inp), rows,
                                         **oracle_args(inp))
    o_gpu, l_gpu = gather_rows(spec, o, lse, rows, inp.get("cu_seqlens_q"))
    bound = _bound_rows(inp, rows) + 2.0 ** -8 * np.abs(o_ref) + 1e-4
    err = np.abs(o_gpu - o_ref)
    worst = float((err / bound).max())
    rel_rms = float(np.linalg.norm(o_gpu - o_ref) / np.linalg.norm(o_ref))
    lse_err = float(np.abs(l_gpu - l_ref).max())
    print(f"err/bound {worst:.3f} rel_rms {rel_rms:.4f} lse {lse_err:.2e}")
    assert worst <= 1.0
    assert rel_rms <= REL_RMS
    assert lse_err <= LSE_TOL


def _all_rows(spec):
    lq, _ = spec.seq_lengths()
    return [(b, h, i) for b in range(spec.batch) for h in range(spec.heads_q) for i in range(lq[b])]


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_fp8qkv_within_rounding_bound(name):
    spec, splits = CASES[name]
    inp = W.make_inputs(spec)
    o, lse = run_lib(inp, num_splits=splits)
    rows = _all_rows(spec)
    if len(rows) > 3000:
        rows = rows[::len(rows) // 3000 + 1] + rows[-3:]
    _check(inp, o, lse, rows)


@pytest.mark.gpu
def test_fp8qkv_padded_key_rows():
    """Depth rows padded past Sk (stride 336 keys for Sk = 333): only the
    first Sk keys of each row are read."""
    spec = _fp8qkv(1, 2, 2, 150, 333, 128, 128, False, seed=116)
    inp = W.make_inputs(spec)
    v = inp["v"]                                   # [B, Hkv, Dv, Sk] contiguous
    padded = torch.full(v.shape[:-1] + (336,), 448.0).to(torch.float8_e4m3fn)
    padded[..., :333] = v
    inp_pad = dict(inp, v=padded[..., :333])
    o, lse = run_lib(inp_pad)
    _check(inp, o, lse, _all_rows(spec))


@pytest.mark.gpu
def test_fp8qkv_full_workload_sampled_rows():
    spec = W.WORKLOADS["fp8qkv_b2_h32_s8192_d128_causal"]
    inp = W.make_inputs(spec)
    o, lse = run_lib(inp)
    rows = W.sample_rows(spec, 128, spec.seed + 200)
    _check(inp, o, lse, rows)


@pytest.mark.gpu
def test_fp8qkv_cross_check_kernel():
    """The fp32 cross-check kernel keeps the weights unrounded: it must sit
    inside the same bound, and both kernels agree on LSE."""
    spec, _ = CASES["causal_gqa_s1000"]
    inp = W.make_inputs(spec)
    o_s, l_s = run_lib(inp, backend="simple")
    o_t, l_t = run_lib(inp)
    assert (l_s - l_t).abs().max().item() < 1e-3
    rows = _all_rows(spec)[::7]
    _check(inp, o_s, l_s, rows)
