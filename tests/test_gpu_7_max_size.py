"""Sizes where 32-bit index arithmetic would overflow: O and Q hold more
than 2^31 elements (one 139264-token sequence, 128 query heads sharing 16 KV
heads, d128, causal), checked on sampled rows against the oracle; and the
split-KV partial buffers at a size where their offsets pass 2^31 too. The
inputs are drawn on the GPU from a seeded generator and copied back for the
oracle, so both sides see the same bits."""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, assert_within, errors, f64


def _draw(shape, gen):
    return torch.randn(shape, generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)


def _rows_check(q, k, v, o, lse, rows, causal, scale, hq, hkv):
    """Oracle rows (b = 0) against the library output. Under the causal mask
    query row i sees keys 0..i, i.e. unmasked attention over those keys."""
    g = hq // hkv
    o_ref, l_ref, o_gpu, l_gpu = [], [], [], []
    qc = {}
    for h, i in rows:
        hk = h // g
        if hk not in qc:
            qc[hk] = (f64(k[0, :, hk].cpu()), f64(v[0, :, hk].cpu()))
        kh, vh = qc[hk]
        n = i + 1 if causal else kh.shape[0]
        oo, ll = oracle.attention_head(f64(q[0, i:i + 1, h].cpu()), kh[:n], vh[:n], scale, False)
        o_ref.append(oo[0]); l_ref.append(ll[0])
        o_gpu.append(f64(o[0, i, h].cpu())); l_gpu.append(float(lse[0, h, i]))
    return errors(np.array(o_gpu), np.array(o_ref), np.array(l_gpu), np.array(l_ref))


@pytest.mark.gpu
def test_output_beyond_2_pow_31_elements():
    import attention_forward_sm100_gb300 as pkg
    S, HQ, HKV, D = 139264, 128, 16, 128
    assert S * HQ * D > 2 ** 31
    gen = torch.Generator(device="cuda").manual_seed(120)
    q = _draw((1, S, HQ, D), gen)
    k = _draw((1, S, HKV, D), gen)
    v = _draw((1, S, HKV, D), gen)
    scale = D ** -0.5
    o, lse = pkg.forward(q, k, v, causal=True, softmax_scale=scale)
    pkg.check()
    rng = np.random.default_rng(120)
    rows = [(HQ - 1, S - 1), (HQ - 1, S - 2), (0, 0), (HQ // 2, S // 2)]
    rows += [(int(rng.integers(HQ)), int(rng.integers(S))) for _ in range(28)]
    err = _rows_check(q, k, v, o, lse, rows, True, scale, HQ, HKV)
    print(err)
    assert_within(err, "bf16")
    del q, k, v, o, lse
    torch.cuda.empty_cache()


@pytest.mark.gpu
def test_split_kv_partials_beyond_2_pow_31_elements():
    import attention_forward_sm100_gb300 as pkg
    Sq, Sk, HQ, HKV, D, N = 16384, 32768, 128, 8, 128, 9
    assert N * Sq * HQ * D > 2 ** 31                   # partial O elements
    gen = torch.Generator(device="cuda").manual_seed(121)
    q = _draw((1, Sq, HQ, D), gen)
    k = _draw((1, Sk, HKV, D), gen)
    v = _draw((1, Sk, HKV, D), gen)
    scale = D ** -0.5
    o, lse = pkg.forward(q, k, v, causal=False, softmax_scale=scale, num_splits=N)
    pkg.check()
    rng = np.random.default_rng(121)
    rows = [(HQ - 1, Sq - 1), (0, 0)] + [(int(rng.integers(HQ)), int(rng.integers(Sq))) for _ in range(14)]
    err = _rows_check(q, k, v, o, lse, rows, False, scale, HQ, HKV)
    print(err)
    assert_within(err, "bf16")
    del q, k, v, o, lse
    torch.cuda.empty_cache()
