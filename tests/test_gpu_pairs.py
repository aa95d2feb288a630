"""CTA pairs (the pair_cta option of the "SM100AttentionSMem" page's barrier
set): two CTAs of a cluster share every M = 256 tcgen05 instruction
(cta_group::2), each holding half of every K and V tile. The pair kernel is
held to the oracle like the one-CTA kernel, on shapes that span several
512-row work tiles, ragged tails, degenerate sizes, packed sequences, GQA,
the shared rope part, split-KV and every schedule; the smallest case (one
cluster, one work tile) runs first."""
import numpy as np
import pytest
import torch

from attention_forward_sm100_gb300 import workloads as W
from helpers import (assert_within, compare_full, errors, f64, gather_rows, run_lib, run_oracle,
                     run_oracle_rows)

S = W.AttnSpec
PAIR = dict(pair_cta="on")


@pytest.mark.gpu
def test_pair_single_cluster_first():
    """One work tile, so one cluster of two CTAs: the protocol's smallest case."""
    spec = S(1, 1, 1, 128, 128, 128, 128, False, seed=300)
    err = compare_full(W.make_inputs(spec), **PAIR)
    assert_within(err, "bf16")


CASES = {
    "causal_s256": S(1, 2, 2, 256, 256, 128, 128, True, seed=301),
    "causal_s1": S(2, 2, 2, 1, 1, 128, 128, True, seed=302),
    "causal_s127": S(2, 2, 1, 127, 127, 128, 128, True, seed=303),
    "causal_s129": S(1, 4, 2, 129, 129, 128, 128, True, seed=304),
    "causal_s513": S(1, 2, 2, 513, 513, 128, 128, True, seed=305),
    "causal_gqa_s1000": S(2, 8, 2, 1000, 1000, 128, 128, True, seed=306),
    "noncausal_s700": S(2, 2, 2, 700, 700, 128, 128, False, seed=307),
    "noncausal_sq200_sk333": S(2, 2, 1, 200, 333, 128, 128, False, seed=308),
    "noncausal_sk1": S(1, 2, 2, 300, 1, 128, 128, False, seed=309),
    "noncausal_sk0": S(2, 2, 2, 130, 0, 128, 128, False, seed=310),
    "causal_sq300_sk170": S(1, 2, 2, 300, 170, 128, 128, True, seed=311),
    "packed_gqa_causal": S(4, 8, 2, 640, 640, 128, 128, True, seed=312, lengths_q=(1, 300, 129, 640)),
    "packed_noncausal_qk_differ": S(3, 4, 4, 400, 400, 128, 128, False, seed=313, lengths_q=(257, 3, 130),
                                    lengths_k=(5, 400, 128)),
    "rope_causal_s700": S(1, 4, 4, 700, 700, 128, 128, True, seed=314, rope=64),
    "rope_packed_causal": S(2, 4, 4, 600, 600, 128, 128, True, seed=315, rope=64, lengths_q=(600, 17)),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_pair_matches_oracle(name):
    spec = CASES[name]
    err = compare_full(W.make_inputs(spec), **PAIR)
    assert_within(err, "bf16")


@pytest.mark.gpu
@pytest.mark.parametrize("schedule", ["static", "grid"])
def test_pair_schedules(schedule):
    spec = S(2, 4, 2, 1100, 1100, 128, 128, True, seed=316)
    inp = W.make_inputs(spec)
    o, lse = run_lib(inp, schedule=schedule, **PAIR)
    o_ref, l_ref = run_oracle(inp)
    assert_within(errors(f64(o), o_ref, lse.double().numpy(), l_ref), "bf16")
    o2, l2 = run_lib(inp, **PAIR)       # dynamic: the same rows in another order, same values
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16)) and torch.equal(lse, l2)


@pytest.mark.gpu
def test_pair_split_kv():
    spec = S(1, 4, 2, 256, 3000, 128, 128, False, seed=317)
    inp = W.make_inputs(spec)
    o, lse = run_lib(inp, num_splits=3, **PAIR)
    o_ref, l_ref = run_oracle(inp)
    assert_within(errors(f64(o), o_ref, lse.double().numpy(), l_ref), "bf16")


@pytest.mark.gpu
def test_pair_causal_row0_is_exact():
    spec = S(2, 4, 2, 1024, 1024, 128, 128, True, seed=318)
    inp = W.make_inputs(spec)
    o, _ = run_lib(inp, **PAIR)
    exp = inp["v"][:, 0].repeat_interleave(2, dim=1)
    assert torch.equal(o[:, 0].view(torch.int16), exp.view(torch.int16))
    # the first row of the second CTA's rows (row 128) and of the second MMA tile (row 256) too
    for r in (128, 256, 384):
        o_ref, _ = run_oracle_rows(inp, [(b, h, r) for b in range(2) for h in range(4)])
        got = np.stack([f64(o[b, r, h]) for b in range(2) for h in range(4)])
        assert np.abs(got - o_ref).max() <= 2e-2


@pytest.mark.gpu
def test_pair_agrees_with_one_cta_kernel():
    """Each row's products and sums are those of the one-CTA kernel."""
    spec = S(2, 8, 2, 1500, 1500, 128, 128, True, seed=319)
    inp = W.make_inputs(spec)
    o1, l1 = run_lib(inp, pair_cta="off")
    o2, l2 = run_lib(inp, **PAIR)
    d = (o1.float() - o2.float()).abs().max().item()
    assert d <= 2e-2 and (l1 - l2).abs().max().item() <= 1e-3
    print("max |pair - one CTA|", d, "identical" if torch.equal(o1.view(torch.int16), o2.view(torch.int16)) else "")


@pytest.mark.gpu
def test_pair_back_to_back_calls():
    spec = W.WORKLOADS["mha_b4_h16_s4096_d128_causal"]
    inp = W.make_inputs(spec)
    o1, l1 = run_lib(inp, **PAIR)
    for _ in range(3):
        o2, l2 = run_lib(inp, **PAIR)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["mha_b4_h16_s4096_d128_causal", "varlen_gqa_b8_hq32_hkv8_d128_causal",
                                  "mla_b2_h128_s4096_d128r64_causal"])
def test_pair_workloads_sampled_rows(name):
    spec = W.WORKLOADS[name]
    inp = W.make_inputs(spec)
    o, lse = run_lib(inp, **PAIR)
    rows = W.sample_rows(spec, 256, spec.seed + 400)
    o_ref, l_ref = run_oracle_rows(inp, rows)
    o_gpu, l_gpu = gather_rows(spec, o, lse, rows, inp.get("cu_seqlens_q"))
    err = errors(o_gpu, o_ref, l_gpu, l_ref)
    print(name, err)
    assert_within(err, "bf16")
