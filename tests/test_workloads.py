"""The seeded input recipe: the drawn lengths, the FP8 per-token
quantisation, shapes and the algorithmic FLOP counts of the five workloads."""
import json
import math
import os

import pytest
import torch

from attention_forward_sm100_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_varlen_lengths_reproduce_fixture():
    with open(os.path.join(GOLDEN, "varlen_lengths_seed2.json")) as f:
        fx = json.load(f)
    spec = W.WORKLOADS["varlen_gqa_b8_hq32_hkv8_d128_causal"]
    assert list(spec.lengths_q) == fx["lengths"]
    assert sum(spec.lengths_q) == fx["total_tokens"]
    assert all(512 <= n <= 8192 for n in spec.lengths_q)


def test_fp8_quantisation_properties():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(64, 4, 128, generator=g)
    x8, s = W.quantize_fp8_per_token(x)
    assert x8.dtype == torch.float8_e4m3fn and s.shape == (64, 4)
    deq = x8.float() * s.unsqueeze(-1)
    # e4m3 keeps 3 mantissa bits: relative rounding error at most 2^-4 for
    # normal values; subnormal codes (below 2^-6 of the range) have absolute
    # step 2^-9 * scale.
    err = (deq - x).abs()
    bound = torch.maximum(x.abs() * 2.0 ** -4, s.unsqueeze(-1) * 2.0 ** -10)
    assert bool((err <= bound + 1e-7).all())
    # the per-vector amax maps to exactly 448
    amax_code = x8.float().abs().amax(dim=-1)
    assert bool((amax_code == 448.0).all())


def test_fp8_exact_for_small_integers():
    x = torch.tensor([[[448.0, -448.0, 1.0, 0.5, -3.0, 0.0, 96.0, 2.0]]])
    x8, s = W.quantize_fp8_per_token(x)
    assert s.item() == 1.0
    assert torch.equal(x8.float(), x)
    z8, zs = W.quantize_fp8_per_token(torch.zeros(1, 1, 8))
    assert zs.item() == 1.0 and torch.equal(z8.float(), torch.zeros(1, 1, 8))


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
def test_flops_closed_form(name):
    spec = W.WORKLOADS[name]
    lq, lk = spec.seq_lengths()
    d = spec.d_qk + spec.rope + spec.d_v
    if spec.causal:
        pairs = sum(n * (n + 1) // 2 for n in lq)
    else:
        pairs = sum(a * b for a, b in zip(lq, lk))
    assert spec.flops() == 2 * d * pairs * spec.heads_q


def test_flops_table():
    expect = {
        "mha_b1_h2_s128_d64_noncausal": 8_388_608,
        "mha_b4_h16_s4096_d128_causal": 274_945_015_808,
        "varlen_gqa_b8_hq32_hkv8_d128_causal": 1_060_719_804_416,
        "mla_b2_h128_s4096_d128r64_causal": 1_374_725_079_040,
        "fp8_b2_h32_s8192_d128_causal": 1_099_645_845_504,
        "splitkv_b1_h2_s16384_d128_causal": 137_447_342_080,
    }
    for name, f in expect.items():
        assert W.WORKLOADS[name].flops() == f


def test_small_inputs_shapes_and_determinism():
    spec = W.AttnSpec(batch=2, heads_q=4, heads_kv=2, seqlen_q=9, seqlen_k=9, d_qk=64, d_v=64,
                      causal=True, seed=11)
    a = W.make_inputs(spec)
    b = W.make_inputs(spec)
    assert a["q"].shape == (2, 9, 4, 64) and a["k"].shape == (2, 9, 2, 64)
    assert a["q"].dtype == torch.bfloat16
    assert torch.equal(a["q"].float(), b["q"].float()) and torch.equal(a["v"].float(), b["v"].float())
    assert math.isclose(spec.softmax_scale, 1 / 8)
    vl = W.AttnSpec(batch=3, heads_q=2, heads_kv=1, seqlen_q=7, seqlen_k=7, d_qk=128, d_v=128,
                    causal=True, seed=3, lengths_q=(7, 1, 4))
    c = W.make_inputs(vl)
    assert c["q"].shape == (12, 2, 128) and c["cu_seqlens_q"].tolist() == [0, 7, 8, 12]
    f8 = W.AttnSpec(batch=1, heads_q=2, heads_kv=2, seqlen_q=5, seqlen_k=5, d_qk=128, d_v=128,
                    causal=True, seed=4, qk_dtype="fp8")
    d = W.make_inputs(f8)
    assert d["q"].dtype == torch.float8_e4m3fn and d["q_scale"].shape == (1, 2, 5)
    ml = W.AttnSpec(batch=1, heads_q=2, heads_kv=2, seqlen_q=5, seqlen_k=5, d_qk=128, d_v=128,
                    causal=True, seed=4, rope=64)
    e = W.make_inputs(ml)
    assert e["k_rope"].shape == (1, 5, 64) and e["q_rope"].shape == (1, 5, 2, 64)
    assert math.isclose(ml.softmax_scale, 1 / math.sqrt(192))


def test_sample_rows_in_range():
    spec = W.WORKLOADS["varlen_gqa_b8_hq32_hkv8_d128_causal"]
    rows = W.sample_rows(spec, 256, 102)
    lq, _ = spec.seq_lengths()
    assert len(rows) == 260
    for b, h, i in rows:
        assert 0 <= b < spec.batch and 0 <= h < spec.heads_q and 0 <= i < lq[b]


def test_hbm_bytes_table():
    # Q, K, V (+ rope, scales) read once, O and LSE written once
    expect = {
        "mha_b1_h2_s128_d64_noncausal": 132_096,
        "mha_b4_h16_s4096_d128_causal": 269_484_032,
        "varlen_gqa_b8_hq32_hkv8_d128_causal": 569_893_632,
        "mla_b2_h128_s4096_d128r64_causal": 1_213_202_432,
        "fp8_b2_h32_s8192_d128_causal": 408_944_640,
        # same with V in e4m3: one byte less per V element
        "fp8qkv_b2_h32_s8192_d128_causal": 408_944_640 - 2 * 8192 * 32 * 128,
        "splitkv_b1_h2_s16384_d128_causal": 33_685_504,
    }
    for name, n in expect.items():
        assert W.WORKLOADS[name].hbm_bytes() == n


def test_tile_granular_flops():
    spec = W.WORKLOADS["mha_b4_h16_s4096_d128_causal"]
    # 32 query tiles of 128 rows; tile t touches t + 1 key tiles
    tiles = sum(t + 1 for t in range(32))
    assert spec.flops_tile_granular() == 2 * 256 * 128 * 128 * tiles * 16 * 4
    assert 1.03 < spec.flops_tile_granular() / spec.flops() < 1.032
    nc = W.WORKLOADS["mha_b1_h2_s128_d64_noncausal"]
    assert nc.flops_tile_granular() == nc.flops()


def test_packed_e4m3_v_layout():
    """Packed e4m3 V: [Hkv, Dv, Tv], each sequence's keys at a multiple of 16
    (zeros between sequences), and the gather back to token order returns
    exactly the rounded draws."""
    import torch
    spec = W.AttnSpec(3, 4, 2, 300, 300, 128, 128, True, seed=9, qk_dtype="fp8", v_dtype="fp8",
                      lengths_q=(17, 300, 1))
    inp = W.make_inputs(spec)
    cv = inp["cu_seqlens_v"].tolist()
    assert cv == [0, 32, 336, 352]
    assert all(c % 16 == 0 for c in cv)
    v = inp["v"]
    assert tuple(v.shape) == (2, 128, 352)
    tm = W.v_token_major(v, inp["cu_seqlens_k"], inp["cu_seqlens_v"])
    assert tuple(tm.shape) == (318, 2, 128)
    # zeros between sequences; the gather reads each sequence's own keys
    assert torch.equal(v[:, :, 17:32].float(), torch.zeros(2, 128, 15))
    assert torch.equal(tm[:17].float(), v[:, :, 0:17].permute(2, 0, 1).float())
