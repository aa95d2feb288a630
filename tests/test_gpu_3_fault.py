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


@pytest.mark.gpu
@pytest.mark.parametrize("backend", ["tcgen05", "simple"])
def test_inconsistent_cu_seqlens_are_refused_on_the_device(backend):
    """Packed offsets the host cannot see: a decreasing pair and an end past
    total_q. The kernel checks every sequence's offsets before using them,
    records the error (the tcgen05 kernel; the cross-check kernel skips the
    sequence) and writes nothing outside the tensors: the guard bytes around
    O stay intact. The next ordinary call with the same workspace is right."""
    import attention_forward_sm100_gb300 as pkg
    dev = torch.device("cuda")
    spec = W.AttnSpec(3, 2, 2, 300, 300, 128, 128, False, seed=62, lengths_q=(300, 100, 200))
    inp = W.make_inputs(spec)
    d = W.to_device(inp, dev)
    tq = d["q"].shape[0]                                       # 600
    guard = torch.full((tq + 2048, 2, 128), 3.0, dtype=torch.bfloat16, device=dev)
    o = guard[1024:1024 + tq]
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    for bad in ([0, 300, 250, 600], [0, 300, 400, 700]):       # decreasing / past the end
        cu_q = torch.tensor(bad, dtype=torch.int32, device=dev)
        pkg.forward(d["q"], d["k"], d["v"], causal=False, softmax_scale=spec.softmax_scale, cu_seqlens_q=cu_q,
                    cu_seqlens_k=d["cu_seqlens_k"], max_seqlen_q=400, max_seqlen_k=300, out=o, workspace=ws,
                    backend=backend, num_splits=1)
        if backend == "tcgen05":
            with pytest.raises(pkg.AttnError) as e:
                pkg.check(workspace=ws, device=dev)
            assert e.value.status == 1 and "cu_seqlens" in str(e.value)
        else:
            pkg.check(workspace=ws, device=dev)
        torch.cuda.synchronize()
        assert bool((guard[:1024] == 3.0).all()) and bool((guard[1024 + tq:] == 3.0).all())
    o2, l2 = pkg.forward(d["q"], d["k"], d["v"], causal=False, softmax_scale=spec.softmax_scale,
                         cu_seqlens_q=d["cu_seqlens_q"], cu_seqlens_k=d["cu_seqlens_k"], max_seqlen_q=300,
                         max_seqlen_k=300, workspace=ws, backend=backend, num_splits=1)
    pkg.check(workspace=ws, device=dev)
    o_ref, l_ref = run_oracle(inp)
    assert_within(errors(f64(o2.cpu()), o_ref, l2.cpu().double().numpy(), l_ref), "bf16")
