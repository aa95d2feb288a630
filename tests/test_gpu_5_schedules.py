"""The three work distributions (dynamic atomic counter, static grid
stride, one CTA per work tile) run the same per-tile arithmetic, so their
outputs must agree bit for bit, on fixed-length, packed, split-KV and FP8
problems; and each agrees with the oracle."""
import pytest
import torch

from attention_forward_sm100_gb300 import workloads as W
from helpers import assert_within, errors, f64, run_lib, run_oracle

S = W.AttnSpec
CASES = {
    "causal_gqa_s1500": (S(2, 8, 2, 1500, 1500, 128, 128, True, seed=90), 1),
    "packed_causal": (S(5, 4, 4, 900, 900, 128, 128, True, seed=91, lengths_q=(900, 1, 257, 640, 33)), 1),
    "noncausal_split": (S(1, 4, 2, 300, 2000, 128, 128, False, seed=92), 4),
    "fp8_causal": (S(1, 4, 4, 700, 700, 128, 128, True, seed=93, qk_dtype="fp8"), 1),
    "d64_rope_free": (S(3, 2, 1, 520, 520, 64, 64, False, seed=94), 1),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_schedules_bit_identical(name):
    import attention_forward_sm100_gb300 as pkg
    spec, splits = CASES[name]
    inp = W.make_inputs(spec)
    dev = torch.device("cuda")
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lq, lk = spec.seq_lengths()
    outs = {}
    for mode in ("dynamic", "static", "grid"):
        o, lse = pkg.forward(d["q"], d["k"], d["v"], causal=spec.causal, softmax_scale=spec.softmax_scale,
                             q_scale=d.get("q_scale"), k_scale=d.get("k_scale"),
                             cu_seqlens_q=d.get("cu_seqlens_q"), cu_seqlens_k=d.get("cu_seqlens_k"),
                             max_seqlen_q=max(lq), max_seqlen_k=max(lk), num_splits=splits, schedule=mode)
        pkg.check(device=dev)
        outs[mode] = (o.cpu(), lse.cpu())
    o0, l0 = outs["dynamic"]
    for mode in ("static", "grid"):
        o, lse = outs[mode]
        assert torch.equal(o.view(torch.int16), o0.view(torch.int16)), mode
        assert torch.equal(lse.view(torch.int32), l0.view(torch.int32)), mode
    o_ref, lse_ref = run_oracle(inp)
    assert_within(errors(f64(o0), o_ref, l0.double().numpy(), lse_ref), spec.qk_dtype)
