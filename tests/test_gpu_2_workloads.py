"""The five workloads at full size through the tcgen05 kernel: the first
three against the full oracle, the MLA and FP8 workloads on 256 seeded
(sequence, head, row) triples plus the first and last rows of the first and
last heads."""
import pytest

from attention_forward_sm100_gb300 import workloads as W
from helpers import assert_within, compare_full, errors, gather_rows, run_lib, run_oracle_rows

FULL = ["mha_b1_h2_s128_d64_noncausal", "mha_b4_h16_s4096_d128_causal", "varlen_gqa_b8_hq32_hkv8_d128_causal"]
SAMPLED = ["mla_b2_h128_s4096_d128r64_causal", "fp8_b2_h32_s8192_d128_causal"]


@pytest.mark.gpu
@pytest.mark.parametrize("name", FULL)
def test_workload_full(name):
    spec = W.WORKLOADS[name]
    err = compare_full(W.make_inputs(spec))
    print(name, err)
    assert_within(err, spec.qk_dtype)


@pytest.mark.gpu
@pytest.mark.parametrize("name", SAMPLED)
def test_workload_sampled_rows(name):
    spec = W.WORKLOADS[name]
    inp = W.make_inputs(spec)
    o, lse = run_lib(inp)
    rows = W.sample_rows(spec, 256, spec.seed + 100)
    o_ref, l_ref = run_oracle_rows(inp, rows)
    o_gpu, l_gpu = gather_rows(spec, o, lse, rows, inp.get("cu_seqlens_q"))
    err = errors(o_gpu, o_ref, l_gpu, l_ref)
    print(name, err)
    assert_within(err, spec.qk_dtype)
