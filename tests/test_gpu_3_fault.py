"""Failure detection on the GPU without a fault: a V tile that is never
loaded makes a bounded device wait run out; the kernel records the timeout,
aborts cleanly (no hang, no trap) and the host reads ATTN_ERR_DEVICE_TIMEOUT.
The CUDA context stays usable: the next ordinary call is correct."""
import ctypes

import pytest
import torch

from attention_forward_sm100_gb300 import workloads as W
from helpers import assert_within, errors, f64, run_oracle


@pytest.mark.gpu
def test_withheld_tile_times_out_and_context_survives():
    import attention_forward_sm100_gb300 as pkg
    spec = W.AttnSpec(1, 2, 2, 600, 600, 128, 128, True, seed=61)
    inp = W.make_inputs(spec)
    dev = torch.device("cuda")
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    o = torch.empty(q.shape[:-1] + (128,), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1, 2, 600), dtype=torch.float32, device=dev)
    p = pkg.make_params(q, k, v, causal=True, softmax_scale=spec.softmax_scale, out=o, lse=lse, workspace=ws)
    p.fault_injection = 1
    stream = torch.cuda.current_stream(dev)
    assert pkg.lib().attn_fwd(ctypes.byref(p), ctypes.c_void_p(stream.cuda_stream)) == 0
    with pytest.raises(pkg.AttnError) as e:
        pkg.check(workspace=ws, device=dev)
    assert e.value.status == 4
    assert "block 0," in str(e.value)
    # The error record was cleared and the scheduler counters reset: the same
    # workspace serves an ordinary call, whose result is right.
    o2, l2 = pkg.forward(q, k, v, causal=True, softmax_scale=spec.softmax_scale, workspace=ws)
    pkg.check(workspace=ws, device=dev)
    o_ref, l_ref = run_oracle(inp)
    assert_within(errors(f64(o2.cpu()), o_ref, l2.cpu().double().numpy(), l_ref), "bf16")
