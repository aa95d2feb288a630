"""The C-ABI library on the CPU: it loads, exports every function the header
declares, validates arguments before touching a GPU, and its host copy of the
persistent schedule visits every work tile exactly once, heaviest first."""
import ctypes
import os
import re

import pytest
import torch

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkg():
    __graft_entry__.build()
    import attention_forward_sm100_gb300 as m
    return m


def _header_functions():
    text = open(os.path.join(ROOT, "include", "attn_fwd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w \*]*?\b(attn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_function(pkg):
    names = _header_functions()
    assert {"attn_fwd", "attn_fwd_check", "attn_fwd_plan", "attn_fwd_schedule"} <= set(names)
    lib = ctypes.CDLL(pkg._binding.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in attn_fwd.h but not exported"


def test_params_layout(pkg):
    assert pkg.lib().attn_fwd_params_size() == ctypes.sizeof(pkg.Params)


def _meta(shape, dtype=torch.bfloat16):
    # Shapes and strides only; plan() never dereferences pointers.
    return torch.empty(shape, dtype=dtype, device="meta")


class _Fake:
    """Tensor stand-in with a chosen data_ptr, for host-side validation."""

    def __init__(self, shape, dtype=torch.bfloat16, ptr=1 << 20, strides=None):
        self.shape = torch.Size(shape)
        self.dtype = dtype
        self._ptr = ptr
        t = torch.empty(shape, device="meta")
        self._strides = strides or t.stride()

    def data_ptr(self):
        return self._ptr

    def stride(self):
        return self._strides

    def numel(self):
        n = 1
        for s in self.shape:
            n *= s
        return n

    def element_size(self):
        return 1


def _params(pkg, B=2, S=512, Hq=8, Hkv=2, D=128, Dv=128, causal=True, **kw):
    q = _Fake((B, S, Hq, D), ptr=kw.pop("qptr", 1 << 20))
    k = _Fake((B, S, Hkv, D), ptr=2 << 20)
    v = _Fake((B, S, Hkv, Dv), ptr=3 << 20)
    o = _Fake((B, S, Hq, Dv), ptr=4 << 20)
    ws = _Fake((256,), dtype=torch.uint8, ptr=5 << 20)
    return pkg.make_params(q, k, v, causal=causal, out=o, lse=None, workspace=ws, **kw)


def test_plan_persistent(pkg):
    info = pkg.plan(_params(pkg))
    assert info.rows_per_tile == 256
    assert info.work_tiles == 2 * 8 * 2
    assert info.block == 512 and info.tmem_columns == 512
    assert 0 < info.smem_bytes <= 232448
    assert info.grid == min(info.work_tiles, 148) or info.grid <= info.work_tiles


@pytest.mark.parametrize("bad", ["heads", "dims", "misaligned", "scale", "noworkspace"])
def test_validation_rejects(pkg, bad):
    if bad == "heads":
        p = _params(pkg, Hq=6, Hkv=4)
        want = 1
    elif bad == "dims":
        p = _params(pkg, D=96, Dv=96)
        want = 2
    elif bad == "misaligned":
        p = _params(pkg, qptr=(1 << 20) + 2)
        want = 1
    elif bad == "scale":
        p = _params(pkg)
        p.softmax_scale = -1.0
        want = 1
    else:
        p = _params(pkg)
        p.workspace = None
        want = 1
    with pytest.raises(pkg.AttnError) as e:
        pkg.plan(p)
    assert e.value.status == want
    assert pkg.last_error()


def test_simple_backend_plan_accepts_odd_dims(pkg):
    p = _params(pkg, D=96, Dv=80, backend="simple")
    info = pkg.plan(p)
    assert info.backend == 1


@pytest.mark.parametrize("B,S,Hq,Hkv", [(1, 1, 1, 1), (2, 700, 8, 2), (3, 256, 4, 4), (1, 4096, 16, 16)])
def test_schedule_fixed_covers_each_tile_once(pkg, B, S, Hq, Hkv):
    p = _params(pkg, B=B, S=S, Hq=Hq, Hkv=Hkv)
    order = pkg.schedule(p)
    T = (S + 255) // 256
    assert len(order) == B * Hq * T
    assert set(order) == {(b, h, t) for b in range(B) for h in range(Hq) for t in range(T)}
    g = Hq // Hkv
    # heaviest first inside each (sequence, KV head)
    for b in range(B):
        for hk in range(Hkv):
            seq = [t for (bb, h, t) in order if bb == b and h // g == hk]
            assert seq == sorted(seq, reverse=True)
    # the query heads of one KV head come back to back for each tile index
    for n in range(0, len(order), g):
        blk = order[n:n + g]
        assert len({(b, h // g, t) for b, h, t in blk}) == 1


def test_schedule_chunks_are_heaviest_first(pkg):
    # 128 KV heads of 2 MB K/V each: several L2-sized chunks per sequence;
    # inside a chunk the tile index never increases.
    p = _params(pkg, B=1, S=4096, Hq=128, Hkv=128)
    order = pkg.schedule(p)
    heads_seen = []
    ts = [t for _, _, t in order]
    chunk_starts = [i for i in range(1, len(order)) if ts[i] > ts[i - 1]]
    assert 1 <= len(chunk_starts) < 16
    bounds = [0] + chunk_starts + [len(order)]
    for a, e in zip(bounds[:-1], bounds[1:]):
        assert ts[a:e] == sorted(ts[a:e], reverse=True)
        heads_seen.append({h for _, h, _ in order[a:e]})
    assert set().union(*heads_seen) == set(range(128))


def test_schedule_packed(pkg):
    lens = [2646, 7628, 1356, 5009, 4477, 3351, 2296, 891]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    p = _params(pkg, B=8, S=8192, Hq=32, Hkv=8)
    order = pkg.schedule(p, host_cu_seqlens_q=cu)
    expect = {(b, h, t) for b, n in enumerate(lens) for h in range(32) for t in range((n + 255) // 256)}
    assert len(order) == len(expect) and set(order) == expect
    # sequences in order
    bs = [b for b, _, _ in order]
    assert bs == sorted(bs)


# ---------------------------------------------------------------- split-KV
def _split_params(pkg, B=1, Sq=256, Sk=32768, Hq=32, Hkv=8, causal=False, splits=0, ws_bytes=1 << 30, packed=False,
                  pair_cta="auto"):
    q = _Fake((B, Sq, Hq, 128), ptr=1 << 20)
    k = _Fake((B, Sk, Hkv, 128), ptr=2 << 20)
    v = _Fake((B, Sk, Hkv, 128), ptr=3 << 20)
    o = _Fake((B, Sq, Hq, 128), ptr=4 << 20)
    ws = _Fake((ws_bytes,), dtype=torch.uint8, ptr=5 << 20)
    kw = {}
    if packed:
        q = _Fake((B * Sq, Hq, 128), ptr=1 << 20)
        k = _Fake((B * Sk, Hkv, 128), ptr=2 << 20)
        v = _Fake((B * Sk, Hkv, 128), ptr=3 << 20)
        o = _Fake((B * Sq, Hq, 128), ptr=4 << 20)
        kw = dict(cu_seqlens_q=_Fake((B + 1,), ptr=6 << 20), cu_seqlens_k=_Fake((B + 1,), ptr=7 << 20),
                  max_seqlen_q=Sq, max_seqlen_k=Sk)
    return pkg.make_params(q, k, v, causal=causal, out=o, lse=None, workspace=ws, num_splits=splits,
                           pair_cta=pair_cta, **kw)


def test_split_kv_explicit_plan_and_workspace(pkg):
    p = _split_params(pkg, B=2, Sq=300, Sk=1000, Hq=4, Hkv=2, splits=3)
    info = pkg.plan(p)
    assert info.num_splits == 3
    assert info.work_tiles == 2 * 4 * 2 * 3          # B * Hq * ceil(300/256) * splits
    lse = 3 * 2 * 4 * 300 * 4
    lse = (lse + 255) // 256 * 256
    assert pkg.workspace_bytes(p) == 256 + lse + 3 * 2 * 300 * 4 * 128 * 4


def test_split_kv_count_capped_at_key_tiles(pkg):
    p = _split_params(pkg, Sq=64, Sk=300, Hq=2, Hkv=2, splits=9)   # 3 key tiles
    assert pkg.plan(p).num_splits == 3


def test_split_kv_automatic_choice(pkg):
    # A short-query / long-key problem with too few query tiles for the GPU splits ...
    auto = pkg.plan(_split_params(pkg)).num_splits
    assert 2 <= auto <= 64
    # ... so does a packed one (from the bound B * ceil(max_len / 256) of its
    # query tiles); one with many query tiles does not, nor a causal one
    # whose 256 query rows see at most 256 keys (top-left mask).
    assert pkg.plan(_split_params(pkg, packed=True)).num_splits == auto
    assert pkg.plan(_split_params(pkg, B=4, Sq=4096, Sk=4096, Hq=16, Hkv=16)).num_splits == 1
    assert pkg.plan(_split_params(pkg, causal=True)).num_splits == 1
    assert pkg.workspace_bytes(_split_params(pkg, causal=True)) == 256
    # a single key tile leaves nothing to split
    assert pkg.plan(_split_params(pkg, Sk=100)).num_splits == 1


def test_causal_split_kv_automatic_choice(pkg):
    # One long causal sequence with few heads: the last query tile sees every
    # key, the first almost none; its 32 x H tiles leave most SMs idle, so
    # the keys split. The causal bench shape (B4 H16 S4096, 1024 tiles) and a
    # long sequence with enough heads (B1 H16 S16384) do not.
    for heads in (1, 2, 4):
        p = _split_params(pkg, B=1, Sq=8192, Sk=8192, Hq=heads, Hkv=heads, causal=True)
        assert pkg.plan(p).num_splits >= 2, heads
        assert pkg.workspace_bytes(p) > 256
    assert pkg.plan(_split_params(pkg, B=4, Sq=4096, Sk=4096, Hq=16, Hkv=16, causal=True)).num_splits == 1
    assert pkg.plan(_split_params(pkg, B=1, Sq=16384, Sk=16384, Hq=16, Hkv=16, causal=True)).num_splits == 1
    # CTA pairs never split a causal problem
    p = _split_params(pkg, B=1, Sq=8192, Sk=8192, Hq=1, Hkv=1, causal=True, pair_cta="on")
    assert pkg.plan(p).num_splits == 1


def test_causal_split_kv_explicit_plan(pkg):
    p = _split_params(pkg, B=2, Sq=1000, Sk=1000, Hq=4, Hkv=2, causal=True, splits=3)
    info = pkg.plan(p)
    assert info.num_splits == 3
    assert info.work_tiles == 2 * 4 * 4 * 3          # B * Hq * ceil(1000/256) * splits


def _ranges(pkg, p, tile, n, sk):
    return [pkg.key_range(p, tile, r, sk) for r in range(n)]


@pytest.mark.parametrize("sq,sk,splits", [(1000, 1000, 3), (8192, 8192, 7), (300, 5000, 4), (5000, 300, 4),
                                          (129, 129, 64), (2048, 2048, 2), (640, 700, 5)])
def test_causal_key_ranges(pkg, sq, sk, splits):
    """Causal ranges: contiguous, in order, on 128-key boundaries, together
    exactly the keys the tile's last row sees (top-left mask), and every range
    that holds keys starts at or before the tile's first row (so its first
    MMA tile visits it and every row sees its first key)."""
    p = _split_params(pkg, B=1, Sq=sq, Sk=sk, Hq=2, Hkv=2, causal=True, splits=splits)
    n = pkg.plan(p).num_splits
    assert n == min(splits, (sk + 127) // 128)
    for t in range((sq + 255) // 256):
        q0 = 256 * t
        rs = _ranges(pkg, p, t, n, sk)
        assert rs[0][0] == 0 and rs[-1][1] == min(sk, q0 + 256), (t, rs)
        for (b0, e0), (b1, e1) in zip(rs, rs[1:]):
            assert e0 == b1
        for b, e in rs:
            assert b <= e and b % 128 == 0
            if e > b:
                assert b <= q0, (t, rs)
        # the pieces are balanced over the first MMA tile's key tiles
        sizes = [(e - b + 127) // 128 for b, e in rs[:-1]]
        if sizes:
            assert max(sizes) - min(sizes) <= 1, rs


@pytest.mark.parametrize("sk,splits", [(1000, 3), (32768, 64), (300, 9)])
def test_unmasked_key_ranges(pkg, sk, splits):
    p = _split_params(pkg, B=1, Sq=256, Sk=sk, Hq=2, Hkv=2, splits=splits)
    n = pkg.plan(p).num_splits
    rs = _ranges(pkg, p, 0, n, sk)
    assert rs[0][0] == 0 and rs[-1][1] == sk
    assert all(e0 == b1 for (_, e0), (b1, _) in zip(rs, rs[1:]))
    assert all(e > b for b, e in rs)                     # n <= key tiles: none empty
    assert _ranges(pkg, p, 5, n, sk) == rs               # the same for every query tile


def test_key_range_without_split_and_rejections(pkg):
    p = _split_params(pkg, B=1, Sq=256, Sk=1000, Hq=2, Hkv=2, splits=1)
    assert pkg.key_range(p, 0, 0, 1000) == (0, 1000)
    for tile, split, sk in ((-1, 0, 10), (0, 1, 10), (0, -1, 10), (0, 0, -1)):
        with pytest.raises(pkg.AttnError) as e:
            pkg.key_range(p, tile, split, sk)
        assert e.value.status == 1


@pytest.mark.parametrize("case,status", [("causal_pairs", 2), ("simple", 2), ("too_many", 1),
                                         ("negative", 1), ("small_workspace", 1)])
def test_split_kv_rejections(pkg, case, status):
    if case == "causal_pairs":
        p = _split_params(pkg, causal=True, splits=2, pair_cta="on")
    elif case == "simple":
        p = _split_params(pkg, splits=2)
        p.backend = 1
    elif case == "too_many":
        p = _split_params(pkg, splits=65)
    elif case == "negative":
        p = _split_params(pkg, splits=-1)
    else:
        p = _split_params(pkg, splits=4, ws_bytes=4096)
    with pytest.raises(pkg.AttnError) as e:
        pkg.plan(p)
    assert e.value.status == status


@pytest.mark.parametrize("B,Sq,Hq,Hkv,Sk,splits,causal", [(1, 256, 32, 8, 32768, 0, False), (2, 700, 4, 2, 1000, 3, False),
                                                           (1, 1, 2, 1, 5000, 64, False), (2, 700, 4, 2, 1000, 3, True),
                                                           (1, 8192, 2, 2, 8192, 0, True)])
def test_schedule_with_splits_covers_each_piece_once(pkg, B, Sq, Hq, Hkv, Sk, splits, causal):
    p = _split_params(pkg, B=B, Sq=Sq, Sk=Sk, Hq=Hq, Hkv=Hkv, splits=splits, causal=causal)
    n = pkg.plan(p).num_splits
    assert n > 1
    order = pkg.schedule(p, with_split=True)
    T = (Sq + 255) // 256
    expect = {(b, h, t, r) for b in range(B) for h in range(Hq) for t in range(T) for r in range(n)}
    assert len(order) == len(expect) and set(order) == expect
    # the ranges of one query tile are handed out next to each other for a
    # KV head's query heads (they share the K/V range in L2)
    g = Hq // Hkv
    for i in range(0, len(order), g):
        blk = order[i:i + g]
        assert len({(b, h // g, t, r) for b, h, t, r in blk}) == 1


# ---------------------------------------------------------------- schedule modes
@pytest.mark.parametrize("mode", ["dynamic", "static", "grid"])
def test_schedule_modes_plan(pkg, mode):
    q = _Fake((2, 4096, 16, 128), ptr=1 << 20)
    k = _Fake((2, 4096, 16, 128), ptr=2 << 20)
    o = _Fake((2, 4096, 16, 128), ptr=4 << 20)
    ws = _Fake((256,), dtype=torch.uint8, ptr=5 << 20)
    p = pkg.make_params(q, k, k, causal=True, out=o, lse=None, workspace=ws, schedule=mode)
    info = pkg.plan(p)
    assert info.work_tiles == 2 * 16 * 16
    if mode == "grid":
        assert info.grid == info.work_tiles            # one CTA per work tile
    else:
        assert info.grid <= 160 and info.grid < info.work_tiles   # one CTA per SM
    # the order of work indices is the same in every mode
    base = pkg.make_params(q, k, k, causal=True, out=o, lse=None, workspace=ws)
    assert pkg.schedule(p) == pkg.schedule(base)


def test_schedule_mode_rejected(pkg):
    p = _params(pkg)
    p.schedule = 3
    with pytest.raises(pkg.AttnError) as e:
        pkg.plan(p)
    assert e.value.status == 1



# ---------------------------------------------------------------- all-FP8
@pytest.mark.parametrize("case,status", [("bf16_qk", 2), ("packed_no_cu_v", 1), ("dv64", 2), ("row_stride", 1)])
def test_fp8_v_rejections(pkg, case, status):
    f8 = torch.float8_e4m3fn
    qdt = torch.bfloat16 if case == "bf16_qk" else f8
    dv = 64 if case == "dv64" else 128
    sk = 333 if case == "row_stride" else 512
    q = _Fake((1, 256, 4, 128), dtype=qdt, ptr=1 << 20)
    k = _Fake((1, sk, 4, 128), dtype=qdt, ptr=2 << 20)
    v = _Fake((1, 4, dv, sk), dtype=f8, ptr=3 << 20)
    o = _Fake((1, 256, 4, dv), ptr=4 << 20)
    qsc = _Fake((1, 4, 256), dtype=torch.float32, ptr=6 << 20)
    ksc = _Fake((1, 4, sk), dtype=torch.float32, ptr=9 << 20)
    ws = _Fake((256,), dtype=torch.uint8, ptr=5 << 20)
    kw = {}
    if case == "packed_no_cu_v":
        q = _Fake((256, 4, 128), dtype=f8, ptr=1 << 20)
        k = _Fake((sk, 4, 128), dtype=f8, ptr=2 << 20)
        v = _Fake((4, dv, sk), dtype=f8, ptr=3 << 20)
        o = _Fake((256, 4, dv), ptr=4 << 20)
        qsc = _Fake((4, 256), dtype=torch.float32, ptr=6 << 20)
        ksc = _Fake((4, sk), dtype=torch.float32, ptr=9 << 20)
        kw = dict(cu_seqlens_q=_Fake((2,), ptr=7 << 20), cu_seqlens_k=_Fake((2,), ptr=8 << 20),
                  cu_seqlens_v=_Fake((2,), ptr=10 << 20))
    p = pkg.make_params(q, k, v, causal=True, out=o, lse=None, workspace=ws, q_scale=qsc, k_scale=ksc, **kw)
    assert p.v_dtype == 1 and p.head_dim_v == dv
    if case == "packed_no_cu_v":
        pkg.plan(p)                       # accepted with the key offsets of V ...
        p.cu_seqlens_v = None             # ... refused without them
        assert p.total_v == sk
    with pytest.raises(pkg.AttnError) as e:
        pkg.plan(p)
    assert e.value.status == status


def test_fp8_v_plan(pkg):
    f8 = torch.float8_e4m3fn
    q = _Fake((2, 8192, 32, 128), dtype=f8, ptr=1 << 20)
    v = _Fake((2, 32, 128, 8192), dtype=f8, ptr=3 << 20)
    o = _Fake((2, 8192, 32, 128), ptr=4 << 20)
    sc = _Fake((2, 32, 8192), dtype=torch.float32, ptr=6 << 20)
    ws = _Fake((256,), dtype=torch.uint8, ptr=5 << 20)
    p = pkg.make_params(q, q, v, causal=True, out=o, lse=None, workspace=ws, q_scale=sc, k_scale=sc)
    assert tuple(p.v_stride) == (32 * 128 * 8192, 8192, 128 * 8192)   # batch, depth row, head
    info = pkg.plan(p)
    assert info.v_stages == 4 and info.k_stages == 4
    assert info.smem_bytes <= 232448


def test_split_kv_packed_workspace_and_schedule(pkg):
    p = _split_params(pkg, B=3, Sq=700, Sk=900, Hq=4, Hkv=2, splits=3, packed=True)
    # packed: rows are the Tq = B * Sq rows of q
    lse = (3 * 2100 * 4 * 4 + 255) // 256 * 256
    assert pkg.workspace_bytes(p) == 256 + lse + 3 * 2100 * 4 * 128 * 4
    lens = [700, 1, 300]
    cu = [0, 700, 701, 1001]
    order = pkg.schedule(p, host_cu_seqlens_q=cu, with_split=True)
    expect = {(b, h, t, r) for b, n in enumerate(lens) for h in range(4) for t in range((n + 255) // 256)
              for r in range(3)}
    assert len(order) == len(expect) and set(order) == expect


def test_output_batch_stride_alignment(pkg):
    """The epilogue stores 16-byte pieces of each O row, so O's batch stride
    must be a multiple of 8 bf16 elements as well (fixed-length layout)."""
    q = _Fake((2, 300, 4, 128), ptr=1 << 20)
    ws = _Fake((256,), dtype=torch.uint8, ptr=5 << 20)
    good = _Fake((2, 300, 4, 128), ptr=4 << 20)
    bad = _Fake((2, 300, 4, 128), ptr=4 << 20, strides=(300 * 4 * 128 + 4, 4 * 128, 128, 1))
    pkg.plan(pkg.make_params(q, q, q, causal=True, out=good, lse=None, workspace=ws))
    with pytest.raises(pkg.AttnError) as e:
        pkg.plan(pkg.make_params(q, q, q, causal=True, out=bad, lse=None, workspace=ws))
    assert e.value.status == 1 and "o must be" in str(e.value)


@pytest.mark.parametrize("case", ["v_len", "v_heads", "out", "lse", "k_scale", "k_rope", "noncontig_lse", "cu_dtype"])
def test_binding_refuses_inconsistent_shapes(pkg, case):
    """The library derives every extent from q and k; the binding refuses
    tensors whose shapes disagree with them before building the call."""
    m = lambda *s, dt=torch.bfloat16: torch.empty(s, dtype=dt, device="meta")  # noqa: E731
    q, k, v = m(2, 64, 4, 128), m(2, 80, 2, 128), m(2, 80, 2, 128)
    kw = {}
    if case == "v_len":
        v = m(2, 79, 2, 128)
    elif case == "v_heads":
        v = m(2, 80, 4, 128)
    elif case == "out":
        kw["out"] = m(2, 64, 4, 64)
    elif case == "lse":
        kw["lse"] = m(2, 64, 4, dt=torch.float32)
    elif case == "k_scale":
        q8, k8 = m(2, 64, 4, 128, dt=torch.float8_e4m3fn), m(2, 80, 2, 128, dt=torch.float8_e4m3fn)
        q, k = q8, k8
        kw.update(q_scale=m(2, 4, 64, dt=torch.float32), k_scale=m(2, 2, 64, dt=torch.float32))
    elif case == "k_rope":
        kw.update(q_rope=m(2, 64, 4, 64), k_rope=m(2, 80, 32))
    elif case == "noncontig_lse":
        kw["lse"] = m(2, 64, 4, dt=torch.float32).permute(0, 2, 1)
    else:
        q, k, v = m(100, 4, 128), m(120, 2, 128), m(120, 2, 128)
        kw.update(cu_seqlens_q=m(3, dt=torch.int64), cu_seqlens_k=m(3, dt=torch.int64))
    with pytest.raises(ValueError):
        pkg.make_params(q, k, v, causal=False, **kw)


# ---------------------------------------------------------------- CTA pairs
def test_pair_plan(pkg):
    p = _params(pkg, B=4, S=4096, Hq=16, Hkv=16, pair_cta="on")
    info = pkg.plan(p)
    assert info.pair_cta == 2 and info.rows_per_tile == 512
    assert info.work_tiles == 4 * 16 * 8
    assert info.grid % 2 == 0 and 2 <= info.grid <= 2 * info.work_tiles
    assert 0 < info.smem_bytes <= 232448
    # more K and V stages than the one-CTA kernel: each holds half a tile
    one = pkg.plan(_params(pkg, B=4, S=4096, Hq=16, Hkv=16, pair_cta="off"))
    assert one.pair_cta == 1 and one.rows_per_tile == 256
    assert info.k_stages > one.k_stages and info.v_stages > one.v_stages
    # the library's own choice keeps one CTA per MMA tile
    assert pkg.plan(_params(pkg, B=4, S=4096, Hq=16, Hkv=16)).pair_cta == 1
    # one cluster per work tile when the grid schedule is asked for
    g = pkg.plan(_params(pkg, B=1, S=1000, Hq=2, Hkv=2, pair_cta="on", schedule="grid"))
    assert g.work_tiles == 2 * 2 and g.grid == 2 * g.work_tiles


def test_pair_plan_rope(pkg):
    q = _Fake((2, 4096, 128, 128), ptr=1 << 20)
    k = _Fake((2, 4096, 128, 128), ptr=2 << 20)
    v = _Fake((2, 4096, 128, 128), ptr=3 << 20)
    o = _Fake((2, 4096, 128, 128), ptr=4 << 20)
    qr = _Fake((2, 4096, 128, 64), ptr=6 << 20)
    kr = _Fake((2, 4096, 64), ptr=7 << 20)
    ws = _Fake((256,), dtype=torch.uint8, ptr=5 << 20)
    p = pkg.make_params(q, k, v, causal=True, out=o, q_rope=qr, k_rope=kr, workspace=ws, pair_cta="on")
    info = pkg.plan(p)
    assert info.pair_cta == 2 and info.rows_per_tile == 512 and info.smem_bytes <= 232448
    assert info.k_stages >= 3 and info.v_stages >= 3


@pytest.mark.parametrize("case,status", [("d64", 2), ("fp8", 2), ("simple", 2), ("fault", 2), ("value", 1)])
def test_pair_rejections(pkg, case, status):
    if case == "d64":
        p = _params(pkg, D=64, Dv=64, pair_cta="on")
    elif case == "fp8":
        q = _Fake((1, 256, 2, 128), dtype=torch.float8_e4m3fn, ptr=1 << 20)
        k = _Fake((1, 256, 2, 128), dtype=torch.float8_e4m3fn, ptr=2 << 20)
        v = _Fake((1, 256, 2, 128), ptr=3 << 20)
        o = _Fake((1, 256, 2, 128), ptr=4 << 20)
        qs = _Fake((1, 2, 256), dtype=torch.float32, ptr=6 << 20)
        ks = _Fake((1, 2, 256), dtype=torch.float32, ptr=7 << 20)
        ws = _Fake((256,), dtype=torch.uint8, ptr=5 << 20)
        p = pkg.make_params(q, k, v, causal=True, out=o, q_scale=qs, k_scale=ks, workspace=ws, pair_cta="on")
    elif case == "simple":
        p = _params(pkg, pair_cta="on", backend="simple")
    elif case == "fault":
        p = _params(pkg, pair_cta="on")
        p.fault_injection = 1
    else:
        p = _params(pkg)
        p.pair_cta = 3
    with pytest.raises(pkg.AttnError) as e:
        pkg.plan(p)
    assert e.value.status == status


@pytest.mark.parametrize("B,S,Hq,Hkv", [(1, 1, 1, 1), (2, 700, 8, 2), (1, 4096, 16, 16)])
def test_pair_schedule_covers_each_tile_once(pkg, B, S, Hq, Hkv):
    p = _params(pkg, B=B, S=S, Hq=Hq, Hkv=Hkv, pair_cta="on")
    order = pkg.schedule(p)
    T = (S + 511) // 512
    assert len(order) == B * Hq * T
    assert set(order) == {(b, h, t) for b in range(B) for h in range(Hq) for t in range(T)}
    g = Hq // Hkv
    for b in range(B):
        for hk in range(Hkv):
            seq = [t for (bb, h, t) in order if bb == b and h // g == hk]
            assert seq == sorted(seq, reverse=True)


def test_pair_schedule_packed(pkg):
    lens = [2646, 7628, 1356, 5009, 4477, 3351, 2296, 891]
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    p = _params(pkg, B=8, S=8192, Hq=32, Hkv=8, pair_cta="on")
    order = pkg.schedule(p, host_cu_seqlens_q=cu)
    expect = {(b, h, t) for b, n in enumerate(lens) for h in range(32) for t in range((n + 511) // 512)}
    assert len(order) == len(expect) and set(order) == expect


def test_causal_ranges_keep_the_kernel_protocol(pkg):
    """The kernel's per-range key-tile counts (tile geometry: MMA tile i of a
    work tile visits ceil(min(range keys, q0 + 128 (i + 1) - range start) /
    128) tiles of the range) must satisfy what its barrier protocol assumes:
    the first MMA tile visits no more tiles than the second, and at least one
    whenever the second visits any; and every row of a visiting MMA tile sees
    the range's first key (a fully masked first tile would leave the running
    max at -inf)."""
    n_checked = 0
    for sq in (1, 128, 129, 256, 257, 600, 1000, 4096):
        for sk in (1, 100, 128, 129, 300, 1000, 4096):
            for splits in (2, 3, 5, 9, 64):
                p = _split_params(pkg, B=1, Sq=sq, Sk=sk, Hq=1, Hkv=1, causal=True, splits=splits)
                n = pkg.plan(p).num_splits
                for t in range((sq + 255) // 256):
                    q0 = 256 * t
                    for r in range(n):
                        b, e = pkg.key_range(p, t, r, sk)
                        counts = []
                        for i in range(2):
                            kv_end = min(e - b, q0 + 128 * (i + 1) - b)
                            counts.append((kv_end + 127) // 128 if kv_end > 0 else 0)
                        assert counts[0] <= counts[1], (sq, sk, splits, t, r, counts)
                        assert counts[1] == 0 or counts[0] >= 1, (sq, sk, splits, t, r, counts)
                        for i in range(2):
                            if counts[i]:
                                assert q0 + 128 * i >= b, (sq, sk, splits, t, r, i)
                        n_checked += 1
    assert n_checked > 1000
