"""Split-KV: the keys of each query tile cut into several ranges, each range
writing a normalised partial O and its LSE, and the LSE-weighted merge. The
merged result is compared with the oracle (which never splits) on shapes that
span several key tiles with ragged ends, for every kernel variant, for
explicit and automatic split counts, unmasked and under the causal mask
(ranges cut from the keys each query tile sees, some of them empty), and at
full size on sampled rows: the short-query / long-key workload, the long
causal workload (one 16k-token sequence, two heads) and one causal sequence
of 8192 tokens with a single head."""
import pytest
import torch

from attention_forward_sm100_gb300 import workloads as W
from helpers import assert_within, errors, f64, gather_rows, run_lib, run_oracle, run_oracle_rows

S = W.AttnSpec
CASES = {
    # name: (spec, num_splits)
    "d128_sk1000_3": (S(1, 4, 2, 200, 1000, 128, 128, False, seed=60), 3),
    "d128_sk1000_auto": (S(1, 4, 2, 200, 1000, 128, 128, False, seed=60), 0),
    "d64_sk777_2": (S(2, 2, 1, 64, 777, 64, 64, False, seed=61), 2),
    "d128_every_tile_own_range": (S(1, 2, 2, 130, 640, 128, 128, False, seed=62), 5),
    "d128_more_splits_than_tiles": (S(1, 2, 2, 33, 300, 128, 128, False, seed=63), 9),
    "d128_gqa_sk2100_16": (S(1, 8, 2, 256, 2100, 128, 128, False, seed=64), 16),
    "rope_sk600_3": (S(1, 2, 2, 100, 600, 128, 128, False, seed=65, rope=64), 3),
    "fp8_sk900_4": (S(1, 2, 2, 130, 900, 128, 128, False, seed=66, qk_dtype="fp8"), 4),
    "d128_sq513_sk1025_7": (S(2, 2, 2, 513, 1025, 128, 128, False, seed=67), 7),
    # packed sequences: each cut by its own key tiles; the 100-key sequence
    # has one key tile, so three of its four ranges are empty
    "packed_gqa_4": (S(3, 8, 2, 700, 1500, 128, 128, False, seed=69, lengths_q=(700, 1, 300),
                       lengths_k=(1500, 100, 640)), 4),
    "packed_d64_auto": (S(2, 4, 4, 256, 3000, 64, 64, False, seed=70, lengths_q=(256, 129),
                          lengths_k=(3000, 2047)), 0),
    "packed_fp8_3": (S(2, 4, 2, 300, 900, 128, 128, False, seed=71, qk_dtype="fp8", lengths_q=(300, 77),
                       lengths_k=(900, 513)), 3),
    "packed_rope_5": (S(2, 2, 2, 200, 800, 128, 128, False, seed=72, rope=64, lengths_q=(200, 130),
                        lengths_k=(800, 129)), 5),
    # causal (top-left mask): each query tile's ranges cut the keys it sees
    "causal_d128_s1000_3": (S(1, 4, 2, 1000, 1000, 128, 128, True, seed=73), 3),
    "causal_d128_gqa_s1300_8": (S(2, 8, 2, 1300, 1300, 128, 128, True, seed=74), 8),
    # nine ranges for at most ten key tiles: the early query tiles' ranges
    # are mostly empty
    "causal_more_splits_than_tiles": (S(1, 2, 2, 600, 600, 128, 128, True, seed=75), 9),
    "causal_sq300_sk1500_4": (S(1, 2, 2, 300, 1500, 128, 128, True, seed=76), 4),
    "causal_sq1500_sk300_3": (S(1, 2, 2, 1500, 300, 128, 128, True, seed=77), 3),
    "causal_d64_s777_5": (S(2, 2, 1, 777, 777, 64, 64, True, seed=78), 5),
    "causal_rope_s700_3": (S(1, 2, 2, 700, 700, 128, 128, True, seed=79, rope=64), 3),
    "causal_fp8_s900_4": (S(1, 2, 2, 900, 900, 128, 128, True, seed=80, qk_dtype="fp8"), 4),
    "causal_fp8qkv_s900_3": (S(1, 2, 2, 900, 900, 128, 128, True, seed=81, qk_dtype="fp8", v_dtype="fp8"), 3),
    "causal_packed_gqa_4": (S(3, 8, 2, 900, 900, 128, 128, True, seed=82, lengths_q=(900, 1, 300),
                              lengths_k=(900, 1, 300)), 4),
    "causal_packed_fp8qkv_3": (S(2, 4, 2, 700, 700, 128, 128, True, seed=83, qk_dtype="fp8", v_dtype="fp8",
                                 lengths_q=(700, 129), lengths_k=(700, 129)), 3),
    "causal_packed_rope_sq_ne_sk_5": (S(2, 2, 2, 600, 900, 128, 128, True, seed=84, rope=64, lengths_q=(600, 200),
                                        lengths_k=(900, 130)), 5),
}


def _assert_case(err, spec):
    if spec.v_dtype == "fp8":
        # P rounded to e4m3: the relative-RMS bar of the all-FP8 tests (the
        # per-element rounding bound is checked in the all-FP8 tests)
        assert err["o_rel_rms"] <= 4e-2 and err["lse_max_abs"] <= 1e-3, err
    else:
        assert_within(err, spec.qk_dtype)


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_split_kv_matches_oracle(name):
    spec, splits = CASES[name]
    inp = W.make_inputs(spec)
    o, lse = run_lib(inp, num_splits=splits)
    o_ref, lse_ref = run_oracle(inp)
    err = errors(f64(o), o_ref, lse.double().numpy(), lse_ref)
    print(name, err)
    _assert_case(err, spec)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_split_kv_agrees_with_unsplit(causal):
    """Splitting changes only the rounding: the split and unsplit results
    differ by at most a few bf16 ulps of O and float ulps of LSE."""
    spec = S(1, 4, 4, 256, 4096, 128, 128, False, seed=68) if not causal else \
        S(1, 4, 4, 2048, 2048, 128, 128, True, seed=85)
    inp = W.make_inputs(spec)
    o1, l1 = run_lib(inp, num_splits=1)
    o8, l8 = run_lib(inp, num_splits=8)
    assert (o1.float() - o8.float()).abs().max().item() < 4e-3
    assert (l1 - l8).abs().max().item() < 1e-4


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["splitkv_b1_hq32_hkv8_sq256_sk32768_d128_noncausal",
                                  "splitkv_b1_h2_s16384_d128_causal"])
def test_split_kv_full_workload_sampled_rows(name):
    spec = W.WORKLOADS[name]
    inp = W.make_inputs(spec)
    import attention_forward_sm100_gb300 as pkg
    o, lse = run_lib(inp)   # automatic split count
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    # the automatic count splits
    assert pkg.workspace_bytes(pkg.make_params(q, k, v, causal=spec.causal)) > 256
    rows = W.sample_rows(spec, 128, spec.seed + 100)
    o_ref, l_ref = run_oracle_rows(inp, rows)
    o_gpu, l_gpu = gather_rows(spec, o, lse, rows)
    err = errors(o_gpu, o_ref, l_gpu, l_ref)
    print(name, err)
    assert_within(err, spec.qk_dtype)


@pytest.mark.gpu
def test_causal_split_kv_long_sequence_sampled_rows():
    """One causal sequence of 8192 tokens and one head: 32 query tiles for
    the whole GPU, so the automatic choice splits the keys; sampled rows
    (the first, the last, and seeded ones between) against the oracle."""
    import attention_forward_sm100_gb300 as pkg
    spec = S(1, 1, 1, 8192, 8192, 128, 128, True, seed=86)
    inp = W.make_inputs(spec)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    assert pkg.workspace_bytes(pkg.make_params(q, k, v, causal=True)) > 256   # the automatic count splits
    o, lse = run_lib(inp)
    rows = W.sample_rows(spec, 96, spec.seed + 100)
    o_ref, l_ref = run_oracle_rows(inp, rows)
    o_gpu, l_gpu = gather_rows(spec, o, lse, rows)
    err = errors(o_gpu, o_ref, l_gpu, l_ref)
    print(err)
    assert_within(err, spec.qk_dtype)
