"""ctypes binding of libattn_fwd.so (argument marshalling only).

Every step of the attention forward runs in the library's CUDA kernels; this
module only turns torch tensors into the pointers, sizes and strides of
``attn_fwd_params`` and raises when the library is missing or refuses the
call. There is no CPU path.
"""
from __future__ import annotations

import collections
import ctypes
import os
import threading

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn_fwd.so")

ATTN_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "cuda error", 4: "device timeout"}
BACKENDS = {"tcgen05": 0, "simple": 1}
SCHEDULES = {"dynamic": 0, "static": 1, "grid": 2}
PAIR_CTA = {"auto": 0, "off": 1, "on": 2}
DTYPES = {torch.bfloat16: 0, torch.float8_e4m3fn: 1}
WORKSPACE_BYTES = 256


class AttnError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"attn_fwd: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Params(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("q_rope", ctypes.c_void_p), ("k_rope", ctypes.c_void_p),
        ("q_scale", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("batch", ctypes.c_int32), ("seqlen_q", ctypes.c_int32), ("seqlen_k", ctypes.c_int32),
        ("total_q", ctypes.c_int32), ("total_k", ctypes.c_int32),
        ("num_heads_q", ctypes.c_int32), ("num_heads_kv", ctypes.c_int32),
        ("head_dim_qk", ctypes.c_int32), ("head_dim_v", ctypes.c_int32), ("rope_depth", ctypes.c_int32),
        ("causal", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
        ("qk_dtype", ctypes.c_int32), ("v_dtype", ctypes.c_int32), ("backend", ctypes.c_int32),
        ("q_stride", ctypes.c_int64 * 3), ("k_stride", ctypes.c_int64 * 3), ("v_stride", ctypes.c_int64 * 3),
        ("o_stride", ctypes.c_int64 * 3), ("q_rope_stride", ctypes.c_int64 * 3),
        ("k_rope_stride", ctypes.c_int64 * 2),
        ("fault_injection", ctypes.c_int32),
        ("num_splits", ctypes.c_int32),
        ("schedule", ctypes.c_int32),
        ("pair_cta", ctypes.c_int32),
        ("cu_seqlens_v", ctypes.c_void_p), ("total_v", ctypes.c_int32),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [("backend", ctypes.c_int32), ("rows_per_tile", ctypes.c_int32), ("work_tiles", ctypes.c_int64),
                ("grid", ctypes.c_int32), ("block", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("k_stages", ctypes.c_int32), ("v_stages", ctypes.c_int32), ("tmem_columns", ctypes.c_int32),
                ("num_splits", ctypes.c_int32), ("pair_cta", ctypes.c_int32)]


class WorkTile(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("head", ctypes.c_int32), ("tile", ctypes.c_int32),
                ("split", ctypes.c_int32)]


_lib = None
_lib_lock = threading.Lock()


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built: run attention_forward_sm100_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            L.attn_fwd.argtypes = [ctypes.POINTER(Params), ctypes.c_void_p]
            L.attn_fwd.restype = ctypes.c_int
            L.attn_fwd_check.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
            L.attn_fwd_check.restype = ctypes.c_int
            L.attn_fwd_plan.argtypes = [ctypes.POINTER(Params), ctypes.POINTER(PlanInfo)]
            L.attn_fwd_plan.restype = ctypes.c_int
            L.attn_fwd_schedule.argtypes = [ctypes.POINTER(Params), ctypes.c_void_p, ctypes.POINTER(WorkTile),
                                            ctypes.c_int64]
            L.attn_fwd_schedule.restype = ctypes.c_int64
            L.attn_fwd_key_range.argtypes = [ctypes.POINTER(Params), ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                             ctypes.POINTER(ctypes.c_int32)]
            L.attn_fwd_key_range.restype = ctypes.c_int
            L.attn_fwd_workspace_bytes.argtypes = [ctypes.POINTER(Params)]
            L.attn_fwd_workspace_bytes.restype = ctypes.c_size_t
            L.attn_fwd_params_init.argtypes = [ctypes.POINTER(Params)]
            L.attn_fwd_params_init.restype = None
            L.attn_fwd_params_size.argtypes = []
            L.attn_fwd_params_size.restype = ctypes.c_size_t
            L.attn_status_string.argtypes = [ctypes.c_int]
            L.attn_status_string.restype = ctypes.c_char_p
            L.attn_fwd_last_error.argtypes = []
            L.attn_fwd_last_error.restype = ctypes.c_char_p
            if L.attn_fwd_params_size() != ctypes.sizeof(Params):
                raise RuntimeError("attn_fwd_params layout mismatch between the binding and the library")
            _lib = L
    return _lib


def last_error() -> str:
    return lib().attn_fwd_last_error().decode()


_workspaces = {}
_workspaces_lock = threading.Lock()


def default_workspace(device, nbytes: int = WORKSPACE_BYTES) -> torch.Tensor:
    """A zero-filled workspace per device of at least ``nbytes`` (the library
    keeps its counters zeroed; split-KV partial results need more room, so
    the cached buffer is replaced by a larger one when a call asks for it).
    Calls that use the default workspace must not overlap on the GPU (one
    stream per device, or the caller's own workspaces)."""
    device = torch.device(device)
    key = (device.type, device.index)
    with _workspaces_lock:
        ws = _workspaces.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(max(nbytes, WORKSPACE_BYTES), dtype=torch.uint8, device=device)
            _workspaces[key] = ws
        return ws


# forward(): validated, marshalled parameters of recent calls, keyed by every
# tensor's pointer, shape, strides and dtype and by the options, so that a
# repeated call skips the Python-side checks and struct filling. A key fixes
# the struct up to the output / LSE buffers forward() allocates (fresh,
# contiguous, same shapes) and the workspace, which are set per call.
_PARAMS_CACHE_SIZE = 64
_params_cache = collections.OrderedDict()
_params_cache_lock = threading.Lock()


def _tensor_key(t):
    return None if t is None else (t.data_ptr(), tuple(t.shape), t.stride(), t.dtype)


def workspace_bytes(p: Params) -> int:
    """attn_fwd_workspace_bytes: the workspace size ``p`` needs."""
    return int(lib().attn_fwd_workspace_bytes(ctypes.byref(p)))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _require_cuda(name, t):
    if t is not None and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (this library has no CPU path)")


def head_dim_v(v) -> int:
    """Dv of a V tensor: its last dimension, or the depth dimension of a
    depth-major e4m3 V ([B, Hkv, Dv, Sk])."""
    return v.shape[-2] if v.dtype == torch.float8_e4m3fn else v.shape[-1]


def _check_layout(q, k, v, packed, out=None, lse=None, q_rope=None, k_rope=None, q_scale=None, k_scale=None,
                  cu_seqlens_q=None, cu_seqlens_k=None, cu_seqlens_v=None):
    """Shapes (and, for the tensors passed as bare pointers, contiguity) that
    the library's sizes are derived from; a mismatch would make it read or
    write outside a tensor, so it is refused here."""
    def shape(t):
        return tuple(t.shape)

    def need(cond, msg):
        if not cond:
            raise ValueError(msg)

    v_fp8 = v.dtype == torch.float8_e4m3fn
    if packed:
        need(len(shape(q)) == 3 and len(shape(k)) == 3, "packed q and k must be [T, H, D]")
        tq, hq, d = shape(q)
        tk, hkv, dk = shape(k)
        b = shape(cu_seqlens_q)[0] - 1
        need(shape(cu_seqlens_k) == (b + 1,), "cu_seqlens_k must have the length of cu_seqlens_q")
        dv = shape(v)[1] if v_fp8 else shape(v)[-1]
        if v_fp8:
            # [Hkv, Dv, Tv]: sequence b at keys cu_seqlens_v[b] ... (checked on the device)
            need(len(shape(v)) == 3 and shape(v)[0] == hkv, f"v shape {shape(v)} does not match k")
            need(cu_seqlens_v is not None and shape(cu_seqlens_v) == (b + 1,),
                 "packed e4m3 v needs cu_seqlens_v of the length of cu_seqlens_q")
        else:
            need(shape(v) == (tk, hkv, dv), f"v shape {shape(v)} does not match k")
        o_shape, lse_shape = (tq, hq, dv), (hq, tq)
        qs_shape, ks_shape, kr_lead = (hq, tq), (hkv, tk), (tk,)
    else:
        need(len(shape(q)) == 4 and len(shape(k)) == 4, "q and k must be [B, S, H, D]")
        b, sq, hq, d = shape(q)
        bk, sk, hkv, dk = shape(k)
        need(bk == b, "q and k batch sizes differ")
        dv = shape(v)[2] if v_fp8 else shape(v)[-1]
        need(shape(v) == ((b, hkv, dv, sk) if v_fp8 else (b, sk, hkv, dv)), f"v shape {shape(v)} does not match k")
        o_shape, lse_shape = (b, sq, hq, dv), (b, hq, sq)
        qs_shape, ks_shape, kr_lead = (b, hq, sq), (b, hkv, sk), (b, sk)
    need(dk == d, "q and k depths differ")
    if out is not None:
        need(shape(out) == o_shape, f"out shape {shape(out)} != {o_shape}")
    for name, t, want in (("lse", lse, lse_shape), ("q_scale", q_scale, qs_shape), ("k_scale", k_scale, ks_shape)):
        if t is not None:
            need(shape(t) == want, f"{name} shape {shape(t)} != {want}")
            if isinstance(t, torch.Tensor):
                need(t.is_contiguous(), f"{name} must be contiguous")
    if q_rope is not None:
        r = shape(q_rope)[-1]
        need(shape(q_rope) == shape(q)[:-1] + (r,), "q_rope must match q but for its depth")
        need(k_rope is not None and shape(k_rope) == kr_lead + (r,), f"k_rope must be {kr_lead + (r,)}")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k), ("cu_seqlens_v", cu_seqlens_v)):
        if isinstance(t, torch.Tensor):
            need(t.is_contiguous() and t.dtype == torch.int32, f"{name} must be a contiguous int32 tensor")


def make_params(q, k, v, *, causal, softmax_scale=None, q_rope=None, k_rope=None, q_scale=None, k_scale=None,
                cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None, out=None, lse=None,
                workspace=None, backend="tcgen05", num_splits=0, schedule="dynamic", pair_cta="auto",
                cu_seqlens_v=None) -> Params:
    """attn_fwd_params for torch tensors (shapes are read, nothing is allocated)."""
    packed = cu_seqlens_q is not None
    _check_layout(q, k, v, packed, out=out, lse=lse, q_rope=q_rope, k_rope=k_rope, q_scale=q_scale,
                  k_scale=k_scale, cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k,
                  cu_seqlens_v=cu_seqlens_v if v.dtype == torch.float8_e4m3fn else None)
    p = Params()
    if packed:
        tq, hq, d = q.shape
        tk, hkv, _ = k.shape
        b = cu_seqlens_q.numel() - 1
        p.total_q, p.total_k = tq, tk
        p.seqlen_q = int(max_seqlen_q if max_seqlen_q is not None else tq)
        p.seqlen_k = int(max_seqlen_k if max_seqlen_k is not None else tk)
    else:
        b, sq, hq, d = q.shape
        _, sk, hkv, _ = k.shape
        p.seqlen_q, p.seqlen_k = sq, sk
    rope = 0 if q_rope is None else q_rope.shape[-1]
    v_fp8 = v.dtype == torch.float8_e4m3fn   # depth-major: [B, Hkv, Dv, Sk]
    p.batch, p.num_heads_q, p.num_heads_kv = b, hq, hkv
    p.head_dim_qk, p.head_dim_v, p.rope_depth = d, head_dim_v(v), rope
    p.causal = 1 if causal else 0
    p.softmax_scale = float(softmax_scale if softmax_scale is not None else (d + rope) ** -0.5)
    if q.dtype not in DTYPES:
        raise ValueError(f"unsupported q dtype {q.dtype}")
    p.qk_dtype = DTYPES[q.dtype]
    if v.dtype not in DTYPES:
        raise ValueError(f"unsupported v dtype {v.dtype}")
    p.v_dtype = DTYPES[v.dtype]
    p.backend = BACKENDS[backend]
    p.num_splits = int(num_splits)
    p.schedule = SCHEDULES[schedule]
    p.pair_cta = PAIR_CTA[pair_cta]
    p.q, p.k, p.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    p.q_rope, p.k_rope = _ptr(q_rope), _ptr(k_rope)
    p.q_scale, p.k_scale = _ptr(q_scale), _ptr(k_scale)
    p.cu_seqlens_q, p.cu_seqlens_k = _ptr(cu_seqlens_q), _ptr(cu_seqlens_k)
    if packed and v_fp8:
        p.cu_seqlens_v, p.total_v = _ptr(cu_seqlens_v), v.shape[2]
    p.o = _ptr(out)
    p.lse = _ptr(lse)
    if workspace is not None:
        p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()

    def strides3(t):
        s = t.stride()
        return (0, s[0], s[1]) if packed else (s[0], s[1], s[2])

    p.q_stride[:] = strides3(q)
    p.k_stride[:] = strides3(k)
    if v_fp8:
        s = v.stride()
        p.v_stride[:] = (0, s[1], s[0]) if packed else (s[0], s[2], s[1])   # batch, depth row, head
    else:
        p.v_stride[:] = strides3(v)
    if out is not None:
        p.o_stride[:] = strides3(out)
    if q_rope is not None:
        p.q_rope_stride[:] = strides3(q_rope)
        s = k_rope.stride()
        p.k_rope_stride[:] = (0, s[0]) if packed else (s[0], s[1])
    return p


def forward(q, k, v, *, causal=False, softmax_scale=None, q_rope=None, k_rope=None, q_scale=None, k_scale=None,
            cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None, out=None, lse=None,
            return_lse=True, workspace=None, backend="tcgen05", stream=None, num_splits=0, schedule="dynamic",
            pair_cta="auto", cu_seqlens_v=None):
    """Fused attention forward on the GPU; returns (O, LSE).

    Fixed length: q [B,Sq,Hq,D], k [B,Sk,Hkv,D], v [B,Sk,Hkv,Dv] (e4m3 v:
    depth-major [B,Hkv,Dv,Sk], with e4m3 q/k; P is then rounded to e4m3) -> O
    [B,Sq,Hq,Dv] bf16, LSE [B,Hq,Sq] fp32. Packed: q [Tq,Hq,D] etc. with int32
    cu_seqlens_q / cu_seqlens_k -> O [Tq,Hq,Dv], LSE [Hq,Tq]; packed e4m3 v is
    [Hkv,Dv,Tv] with int32 cu_seqlens_v, each sequence's keys starting at a
    multiple of 16. Optional rope
    parts q_rope [..,Hq,R] and k_rope [..,R] (one per token, shared by heads);
    fp8 e4m3 q/k need per-token fp32 scales q_scale [B,Hq,Sq] / [Hq,Tq] and
    k_scale [B,Hkv,Sk] / [Hkv,Tk]. ``num_splits``: split-KV key ranges per
    query tile (0 = the library's choice, 1 = off; masked or not, fixed
    length or packed; not with causal CTA pairs). ``schedule``: "dynamic" (default), "static" or "grid",
    how work tiles reach CTAs (results are identical). ``pair_cta``: "auto"
    (the library's choice), "off", or "on": two CTAs of a cluster share every
    MMA (bf16, Dqk = Dv = 128, rope 0 or 64). Asynchronous on ``stream``
    (default: the current torch stream). A call with the same tensors
    (pointer, shape, strides, dtype) and options as a recent one reuses its
    validated parameters.
    """
    L = lib()
    packed = cu_seqlens_q is not None
    dev = q.device
    own_out, own_lse = out is None, lse is None and return_lse
    key = None
    if workspace is None:
        key = (dev.type, dev.index, _tensor_key(q), _tensor_key(k), _tensor_key(v), _tensor_key(q_rope),
               _tensor_key(k_rope), _tensor_key(q_scale), _tensor_key(k_scale), _tensor_key(cu_seqlens_q),
               _tensor_key(cu_seqlens_k), _tensor_key(cu_seqlens_v), _tensor_key(out), _tensor_key(lse),
               return_lse, bool(causal), softmax_scale, max_seqlen_q, max_seqlen_k, backend, num_splits, schedule,
               pair_cta)
        with _params_cache_lock:
            hit = _params_cache.get(key)
            if hit is not None:
                _params_cache.move_to_end(key)
    else:
        hit = None
    if hit is None:
        for name, t in (("q", q), ("k", k), ("v", v), ("q_rope", q_rope), ("k_rope", k_rope), ("q_scale", q_scale),
                        ("k_scale", k_scale), ("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k),
                        ("cu_seqlens_v", cu_seqlens_v), ("out", out), ("lse", lse)):
            _require_cuda(name, t)
    if own_out:
        out = torch.empty(q.shape[:-1] + (head_dim_v(v),), dtype=torch.bfloat16, device=dev)
    if own_lse:
        if packed:
            lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=dev)
        else:
            lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=dev)
    if hit is not None:
        p = Params.from_buffer_copy(hit[0])
        need = hit[1]
        if own_out:
            p.o = out.data_ptr()
        if own_lse:
            p.lse = lse.data_ptr()
    else:
        p = make_params(q, k, v, causal=causal, softmax_scale=softmax_scale, q_rope=q_rope, k_rope=k_rope,
                        q_scale=q_scale, k_scale=k_scale, cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k,
                        max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k, out=out, lse=lse,
                        workspace=workspace, backend=backend, num_splits=num_splits, schedule=schedule,
                        pair_cta=pair_cta, cu_seqlens_v=cu_seqlens_v)
        need = 0
        if workspace is None:
            with torch.cuda.device(dev):
                need = workspace_bytes(p)
            with _params_cache_lock:
                _params_cache[key] = (Params.from_buffer_copy(p), need)
                while len(_params_cache) > _PARAMS_CACHE_SIZE:
                    _params_cache.popitem(last=False)
    if workspace is None:
        workspace = default_workspace(dev, need)
        p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel()
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = L.attn_fwd(ctypes.byref(p), ctypes.c_void_p(handle))
    if st != ATTN_OK:
        raise AttnError(st, last_error())
    return out, lse


class PreparedForward:
    """A forward whose tensors, options and workspace stay fixed across calls
    (a serving loop that refills the same buffers): the parameter struct is
    marshalled once, and each ``run`` is one ``attn_fwd`` call (the library
    reuses the tensor maps it encoded for the same tensors). Build it with
    ``prepare`` (same arguments as ``forward``); ``out`` and ``lse`` hold the
    results of the latest run."""

    def __init__(self, q, k, v, **kw):
        for name in ("q", "k", "v"):
            _require_cuda(name, locals()[name])
        stream = kw.pop("stream", None)
        dev = q.device
        packed = kw.get("cu_seqlens_q") is not None
        if kw.get("out") is None:
            kw["out"] = torch.empty(q.shape[:-1] + (head_dim_v(v),), dtype=torch.bfloat16, device=dev)
        if kw.get("lse") is None:
            shape = (q.shape[1], q.shape[0]) if packed else (q.shape[0], q.shape[2], q.shape[1])
            kw["lse"] = torch.empty(shape, dtype=torch.float32, device=dev)
        for name in ("q_rope", "k_rope", "q_scale", "k_scale", "cu_seqlens_q", "cu_seqlens_k", "cu_seqlens_v"):
            _require_cuda(name, kw.get(name))
        self.out, self.lse = kw["out"], kw["lse"]
        self._keep = (q, k, v, kw)   # the tensors must outlive the prepared call
        self._p = make_params(q, k, v, **kw)
        ws = kw.get("workspace")
        if ws is None:
            with torch.cuda.device(dev):
                need = workspace_bytes(self._p)
            ws = default_workspace(dev, need)
            self._p.workspace, self._p.workspace_bytes = ws.data_ptr(), ws.numel()
        self.workspace = ws
        self._ref = ctypes.byref(self._p)
        self._fn = lib().attn_fwd
        self._stream = stream if stream is not None else torch.cuda.current_stream(dev)
        self._handle = ctypes.c_void_p(self._stream.cuda_stream if hasattr(self._stream, "cuda_stream")
                                       else int(self._stream))

    def run(self):
        """Enqueues the forward on the stream given at preparation."""
        st = self._fn(self._ref, self._handle)
        if st != ATTN_OK:
            raise AttnError(st, last_error())
        return self.out, self.lse


def prepare(q, k, v, **kw) -> PreparedForward:
    """A ``PreparedForward`` for fixed tensors and options (see ``forward``)."""
    return PreparedForward(q, k, v, **kw)


def check(workspace=None, device=None, stream=None):
    """Synchronises and raises if a kernel wait ran out of time."""
    L = lib()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    ws = workspace if workspace is not None else default_workspace(dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = L.attn_fwd_check(ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(handle))
    if st != ATTN_OK:
        raise AttnError(st, last_error())


def plan(p: Params) -> PlanInfo:
    info = PlanInfo()
    st = lib().attn_fwd_plan(ctypes.byref(p), ctypes.byref(info))
    if st != ATTN_OK:
        raise AttnError(st, last_error())
    return info


def schedule(p: Params, host_cu_seqlens_q=None, with_split=False):
    """The persistent scheduler's order of work tiles, as (batch, head, tile)
    or, with ``with_split``, (batch, head, tile, split-KV range)."""
    L = lib()
    cu = None
    cu_arr = None
    if host_cu_seqlens_q is not None:
        cu_arr = (ctypes.c_int32 * len(host_cu_seqlens_q))(*[int(x) for x in host_cu_seqlens_q])
        cu = ctypes.cast(cu_arr, ctypes.c_void_p)
    n = L.attn_fwd_schedule(ctypes.byref(p), cu, None, 0)
    if n < 0:
        raise AttnError(1, "bad schedule arguments")
    out = (WorkTile * max(n, 1))()
    L.attn_fwd_schedule(ctypes.byref(p), cu, out, n)
    if with_split:
        return [(w.batch, w.head, w.tile, w.split) for w in out[:n]]
    return [(w.batch, w.head, w.tile) for w in out[:n]]


def key_range(p: Params, tile, split, seqlen_k):
    """Keys (begin, end) of one sequence of ``seqlen_k`` keys that split-KV
    range ``split`` of query tile ``tile`` covers (attn_fwd_key_range)."""
    b, e = ctypes.c_int32(), ctypes.c_int32()
    st = lib().attn_fwd_key_range(ctypes.byref(p), int(tile), int(split), int(seqlen_k), ctypes.byref(b),
                                  ctypes.byref(e))
    if st != ATTN_OK:
        raise AttnError(st, last_error())
    return b.value, e.value
