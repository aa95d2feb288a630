"""The plain CUDA-core cross-check kernel against the oracle (small shapes)."""
import pytest

from attention_forward_sm100_gb300 import workloads as W
from helpers import assert_within, compare_full

CASES = {
    "mha_d64_noncausal": W.AttnSpec(1, 2, 2, 128, 128, 64, 64, False, seed=0),
    "gqa_d128_causal": W.AttnSpec(2, 4, 2, 77, 77, 128, 128, True, seed=21),
    "noncausal_sq_ne_sk": W.AttnSpec(1, 2, 1, 40, 95, 64, 64, False, seed=22),
    "packed_gqa_causal": W.AttnSpec(3, 4, 2, 90, 90, 128, 128, True, seed=23, lengths_q=(1, 90, 33)),
    "rope": W.AttnSpec(1, 3, 3, 65, 65, 128, 128, True, seed=24, rope=64),
    "fp8": W.AttnSpec(1, 2, 2, 70, 70, 128, 128, True, seed=25, qk_dtype="fp8"),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_simple_kernel_matches_oracle(name):
    spec = CASES[name]
    err = compare_full(W.make_inputs(spec), backend="simple")
    assert_within(err, spec.qk_dtype)
