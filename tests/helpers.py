"""Shared test helpers: exact fp64 views of workload inputs, and error metrics."""
import numpy as np
import torch


def f64(t):
    """Exact float64 numpy copy of a CPU tensor (bf16 and fp8 upcast exactly)."""
    if t is None:
        return None
    return t.detach().cpu().to(torch.float32).to(torch.float64).numpy()


def oracle_args(inputs):
    """Keyword arguments of ``oracle.attention`` for a workload input dict."""
    spec = inputs["spec"]
    cu_q = inputs.get("cu_seqlens_q")
    cu_k = inputs.get("cu_seqlens_k")
    return dict(
        causal=spec.causal, scale=spec.softmax_scale,
        q_rope=f64(inputs.get("q_rope")), k_rope=f64(inputs.get("k_rope")),
        q_scale=f64(inputs.get("q_scale")), k_scale=f64(inputs.get("k_scale")),
        cu_seqlens_q=None if cu_q is None else cu_q.numpy().astype(np.int64),
        cu_seqlens_k=None if cu_k is None else cu_k.numpy().astype(np.int64),
    )


def v_for_oracle(inputs):
    """V in the oracle's [B, Sk, Hkv, Dv] (or packed [Tk, Hkv, Dv]) layout, exact float64."""
    from attention_forward_sm100_gb300.workloads import v_token_major
    return f64(v_token_major(inputs["v"], inputs.get("cu_seqlens_k"), inputs.get("cu_seqlens_v")))


def run_oracle(inputs):
    import oracle
    return oracle.attention(f64(inputs["q"]), f64(inputs["k"]), v_for_oracle(inputs), **oracle_args(inputs))


def run_oracle_rows(inputs, rows):
    import oracle
    return oracle.attention_rows(f64(inputs["q"]), f64(inputs["k"]), v_for_oracle(inputs), rows,
                                 **oracle_args(inputs))


def errors(o_gpu, o_ref, lse_gpu=None, lse_ref=None):
    """max-abs and relative-RMS of O against the unrounded reference, and
    max-abs of LSE. Inputs are float64 numpy arrays of equal shape."""
    d = o_gpu - o_ref
    out = {
        "o_max_abs": float(np.max(np.abs(d))) if d.size else 0.0,
        "o_rel_rms": float(np.linalg.norm(d) / max(np.linalg.norm(o_ref), 1e-300)) if d.size else 0.0,
    }
    if lse_gpu is not None:
        finite = np.isfinite(lse_ref)
        if not np.array_equal(finite, np.isfinite(lse_gpu)):
            out["lse_max_abs"] = float("inf")
        else:
            dl = np.abs(lse_gpu[finite] - lse_ref[finite])
            out["lse_max_abs"] = float(dl.max()) if dl.size else 0.0
        if d.size:
            out["worst_index"] = tuple(int(x) for x in np.unravel_index(np.argmax(np.abs(d)), d.shape))
    return out


# Tolerances of the parity bar (fixed for the workloads): BF16 O max-abs 2e-2,
# O relative RMS 5e-3, LSE max-abs 1e-3; FP8 O max-abs 4e-2 (relative RMS 1e-2
# and LSE 1e-3 held as our own bar).
TOL = {
    "bf16": {"o_max_abs": 2e-2, "o_rel_rms": 5e-3, "lse_max_abs": 1e-3},
    "fp8": {"o_max_abs": 4e-2, "o_rel_rms": 1e-2, "lse_max_abs": 1e-3},
}


def assert_within(err, dtype):
    tol = TOL[dtype]
    for key, bound in tol.items():
        assert err[key] <= bound, f"{key}={err[key]:.3e} exceeds {bound:.1e} ({err})"


def run_lib(inputs, backend="tcgen05", device="cuda", num_splits=0, **kw):
    """Runs the library on a workload input dict; returns (O, LSE) as CPU tensors."""
    import attention_forward_sm100_gb300 as pkg
    spec = inputs["spec"]
    dev = torch.device(device)
    from attention_forward_sm100_gb300.workloads import to_device
    d = to_device(inputs, dev)
    lq, lk = spec.seq_lengths()
    o, lse = pkg.forward(d["q"], d["k"], d["v"], causal=spec.causal, softmax_scale=spec.softmax_scale,
                         q_rope=d.get("q_rope"), k_rope=d.get("k_rope"), q_scale=d.get("q_scale"),
                         k_scale=d.get("k_scale"), cu_seqlens_q=d.get("cu_seqlens_q"),
                         cu_seqlens_k=d.get("cu_seqlens_k"), cu_seqlens_v=d.get("cu_seqlens_v"), max_seqlen_q=max(lq + [0]),
                         max_seqlen_k=max(lk + [0]), backend=backend, num_splits=num_splits, **kw)
    pkg.check(device=dev)
    return o.cpu(), lse.cpu()


def compare_full(inputs, backend="tcgen05", **kw):
    """Element-wise errors of the library against the full oracle."""
    o, lse = run_lib(inputs, backend, **kw)
    o_ref, lse_ref = run_oracle(inputs)
    return errors(f64(o), o_ref, lse.double().numpy(), lse_ref)


def gather_rows(spec, o, lse, rows, cu_q=None):
    """O rows [n, Dv] and LSE [n] of the library output at (b, h, i) triples."""
    out_o, out_l = [], []
    for b, h, i in rows:
        if spec.varlen:
            t = int(cu_q[b]) + i
            out_o.append(o[t, h])
            out_l.append(lse[h, t])
        else:
            out_o.append(o[b, i, h])
            out_l.append(lse[b, h, i])
    return f64(torch.stack(out_o)), torch.stack(out_l).double().numpy()
