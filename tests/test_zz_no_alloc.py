"""attn_fwd_noalloc, the entry point for callers that cannot allocate device
memory (for example code that only receives tensors and a stream from a host
framework owning every allocation, or a serving loop that must not allocate
once running): it keeps its scratch in a fixed array inside the library. Its
output must match attn_fwd's, which uses a caller-provided workspace, on two
calls in a row (the second call reuses the array the first one left behind).
This file is collected last on purpose."""
import ctypes

import pytest
import torch

from attention_forward_sm100_gb300 import workloads as W
from helpers import TOL


@pytest.mark.gpu
def test_noalloc_entry_point_matches_attn_fwd():
    import attention_forward_sm100_gb300 as pkg

    spec = W.AttnSpec(2, 4, 2, 700, 700, 128, 128, True, seed=77)
    inp = W.make_inputs(spec)
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    o_ref, l_ref = pkg.forward(q, k, v, causal=True, softmax_scale=spec.softmax_scale)
    pkg.check(device=dev)

    lib = pkg.lib()
    fn = lib.attn_fwd_noalloc
    fn.argtypes = [ctypes.POINTER(pkg.Params), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    stream = torch.cuda.current_stream(dev)
    tol = TOL["bf16"]
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(l_ref, float("nan"))
        p = pkg.make_params(q, k, v, causal=True, softmax_scale=spec.softmax_scale, out=o, lse=lse)
        st = fn(ctypes.byref(p), ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, pkg.last_error()
        torch.cuda.synchronize(dev)
        assert (o.double() - o_ref.double()).abs().max().item() <= tol["o_max_abs"]
        assert (lse.double() - l_ref.double()).abs().max().item() <= tol["lse_max_abs"]


@pytest.mark.gpu
def test_noalloc_never_splits():
    """The fixed array has no room for split-KV partials: the automatic split
    count means "no split" here, and an explicit count is refused on the
    host before anything is enqueued."""
    import attention_forward_sm100_gb300 as pkg

    spec = W.AttnSpec(1, 8, 2, 128, 4096, 128, 128, False, seed=78)
    inp = W.make_inputs(spec)
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    o_ref, l_ref = pkg.forward(q, k, v, causal=False, softmax_scale=spec.softmax_scale)   # splits
    pkg.check(device=dev)
    fn = pkg.lib().attn_fwd_noalloc
    fn.argtypes = [ctypes.POINTER(pkg.Params), ctypes.c_void_p]
    fn.restype = ctypes.c_int
    stream = torch.cuda.current_stream(dev)
    o = torch.full_like(o_ref, float("nan"))
    lse = torch.full_like(l_ref, float("nan"))
    p = pkg.make_params(q, k, v, causal=False, softmax_scale=spec.softmax_scale, out=o, lse=lse)
    assert fn(ctypes.byref(p), ctypes.c_void_p(stream.cuda_stream)) == 0, pkg.last_error()
    torch.cuda.synchronize(dev)
    tol = TOL["bf16"]
    assert (o.double() - o_ref.double()).abs().max().item() <= tol["o_max_abs"]
    assert (lse.double() - l_ref.double()).abs().max().item() <= tol["lse_max_abs"]
    p.num_splits = 2
    assert fn(ctypes.byref(p), ctypes.c_void_p(stream.cuda_stream)) == 2
