"""Seeded synthetic inputs for the attention forward workloads.

This module only draws and lays out input tensors. It holds none of the
attention arithmetic, so both the CUDA path (through the package) and the CPU
oracle (through the tests) can take their inputs from it and see identical bits.

Recipe (the reading taken for every workload):
  * a torch CPU ``Generator().manual_seed(seed)``;
  * for packed variable-length workloads whose lengths are drawn, the lengths
    are drawn first, ``randint(lo, hi + 1, (batch,))`` (inclusive range);
  * then fp32 ``randn`` tensors in the order Q, K, V (MLA: q_nope, q_rope,
    k_nope, k_rope, v), cast to bf16 with round-to-nearest-even;
  * FP8 workloads draw Q and K in fp32 and quantise each (token, head) vector
    to float8_e4m3fn with an fp32 scale = amax / 448 (amax = 0 -> scale 1);
    the quantised value is clamp(x / scale, -448, 448) rounded to e4m3;
  * all-FP8 workloads also round V (drawn after K, N(0,1)) to e4m3 without a
    scale (clamp to +-448, nearest even) and store it depth-major, each row
    of keys padded with zeros to a multiple of 16; packed: [Hkv, Dv, Tv] with
    every sequence's keys starting at a multiple of 16 (int32 cu_seqlens_v
    gives those starts, zeros between sequences).

Layouts: Q/K/V/O are [B, S, H, D] (fixed length) or [T, H, D] (packed, with
int32 cu_seqlens of length B + 1). The shared K rope part is [B, S, R] or
[T, R]. Per-token scales and LSE are token-contiguous: [B, H, S] or [H, T].
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

FP8_E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class AttnSpec:
    """Shape and type description of one attention forward problem."""

    batch: int
    heads_q: int
    heads_kv: int
    seqlen_q: int            # fixed-length Sq, or max length for packed inputs
    seqlen_k: int
    d_qk: int                # per-head Q/K depth, excluding the rope part
    d_v: int
    causal: bool
    seed: int
    rope: int = 0            # rope depth R (K rope shared by all heads)
    qk_dtype: str = "bf16"   # "bf16" or "fp8"
    v_dtype: str = "bf16"    # "bf16", or "fp8": e4m3 V depth-major [B, Hkv, Dv, Sk] (packed: [Hkv, Dv, Tv])
    lengths_q: Optional[Sequence[int]] = None   # packed layout when set
    lengths_k: Optional[Sequence[int]] = None   # defaults to lengths_q
    scale: Optional[float] = None               # defaults to 1/sqrt(d_qk + rope)

    @property
    def varlen(self) -> bool:
        return self.lengths_q is not None

    @property
    def softmax_scale(self) -> float:
        if self.scale is not None:
            return float(self.scale)
        return 1.0 / math.sqrt(self.d_qk + self.rope)

    def seq_lengths(self):
        """(lengths_q, lengths_k) as python lists, one entry per sequence."""
        if self.varlen:
            lq = [int(x) for x in self.lengths_q]
            lk = [int(x) for x in (self.lengths_k if self.lengths_k is not None else self.lengths_q)]
            return lq, lk
        return [self.seqlen_q] * self.batch, [self.seqlen_k] * self.batch

    def visible_pairs(self) -> int:
        """Number of visible (query, key) pairs per query head, summed over
        sequences (causal: key j visible to query i iff j <= i)."""
        lq, lk = self.seq_lengths()
        total = 0
        for a, b in zip(lq, lk):
            if self.causal:
                # row i sees keys 0..min(i, b-1)
                n = min(a, b)
                total += n * (n + 1) // 2
                if a > b:
                    total += (a - b) * b
            else:
                total += a * b
        return total

    def flops(self) -> int:
        """Algorithmic FLOPs: 2 * (d_qk + rope + d_v) per visible pair per head."""
        return 2 * (self.d_qk + self.rope + self.d_v) * self.visible_pairs() * self.heads_q

    def flops_tile_granular(self, block_m: int = 128, block_n: int = 128) -> int:
        """FLOPs of every block_m x block_n (query, key) tile that holds at
        least one visible pair, counted whole (context for the exact count)."""
        lq, lk = self.seq_lengths()
        tiles = 0
        for a, b in zip(lq, lk):
            for t in range((a + block_m - 1) // block_m):
                last_row = min(a, (t + 1) * block_m) - 1
                keys = min(b, last_row + 1) if self.causal else b
                tiles += (keys + block_n - 1) // block_n
        return 2 * (self.d_qk + self.rope + self.d_v) * block_m * block_n * tiles * self.heads_q

    def hbm_bytes(self) -> int:
        """Algorithmic HBM bytes: Q, K, V (and rope parts, per-token scales)
        read once, O (bf16) and LSE (fp32) written once."""
        lq, lk = self.seq_lengths()
        tq, tk = sum(lq), sum(lk)
        qk_es = 1 if self.qk_dtype == "fp8" else 2
        v_es = 1 if self.v_dtype == "fp8" else 2
        n = tq * self.heads_q * (self.d_qk * qk_es + self.rope * 2)          # Q (+ q rope)
        n += tk * self.heads_kv * self.d_qk * qk_es + tk * self.rope * 2      # K (+ shared k rope)
        n += tk * self.heads_kv * self.d_v * v_es                             # V
        if self.qk_dtype == "fp8":
            n += 4 * (tq * self.heads_q + tk * self.heads_kv)                 # scales
        n += tq * self.heads_q * (2 * self.d_v + 4)                           # O, LSE
        return n


def draw_lengths(batch: int, lo: int, hi: int, seed: int) -> list:
    """Sequence lengths drawn uniformly from the inclusive range [lo, hi]."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (batch,), generator=g).tolist()


# The workloads, named by what they are. The last three are additions: the
# FP8 workload with V rounded to e4m3 as well (same seed, so Q, K and V hold
# the same draws), a short-query, long-key shape (a prefill chunk of 256
# rows against a 32k-token cache, GQA 32/8, no mask) whose few query tiles
# cannot fill the GPU: the shape that split-KV exists for; and its causal
# counterpart, one 16k-token sequence with two heads, whose last query tiles
# see 64 times more keys than the first.
def _workloads():
    return {
        "mha_b1_h2_s128_d64_noncausal": AttnSpec(
            batch=1, heads_q=2, heads_kv=2, seqlen_q=128, seqlen_k=128,
            d_qk=64, d_v=64, causal=False, seed=0),
        "mha_b4_h16_s4096_d128_causal": AttnSpec(
            batch=4, heads_q=16, heads_kv=16, seqlen_q=4096, seqlen_k=4096,
            d_qk=128, d_v=128, causal=True, seed=1),
        "varlen_gqa_b8_hq32_hkv8_d128_causal": AttnSpec(
            batch=8, heads_q=32, heads_kv=8, seqlen_q=8192, seqlen_k=8192,
            d_qk=128, d_v=128, causal=True, seed=2,
            lengths_q=tuple(draw_lengths(8, 512, 8192, 2))),
        "mla_b2_h128_s4096_d128r64_causal": AttnSpec(
            batch=2, heads_q=128, heads_kv=128, seqlen_q=4096, seqlen_k=4096,
            d_qk=128, rope=64, d_v=128, causal=True, seed=3),
        "fp8_b2_h32_s8192_d128_causal": AttnSpec(
            batch=2, heads_q=32, heads_kv=32, seqlen_q=8192, seqlen_k=8192,
            d_qk=128, d_v=128, causal=True, seed=4, qk_dtype="fp8"),
        "fp8qkv_b2_h32_s8192_d128_causal": AttnSpec(
            batch=2, heads_q=32, heads_kv=32, seqlen_q=8192, seqlen_k=8192,
            d_qk=128, d_v=128, causal=True, seed=4, qk_dtype="fp8", v_dtype="fp8"),
        "splitkv_b1_hq32_hkv8_sq256_sk32768_d128_noncausal": AttnSpec(
            batch=1, heads_q=32, heads_kv=8, seqlen_q=256, seqlen_k=32768,
            d_qk=128, d_v=128, causal=False, seed=5),
        "splitkv_b1_h2_s16384_d128_causal": AttnSpec(
            batch=1, heads_q=2, heads_kv=2, seqlen_q=16384, seqlen_k=16384,
            d_qk=128, d_v=128, causal=True, seed=6),
    }


WORKLOADS = _workloads()
WORKLOAD_ORDER = list(WORKLOADS.keys())


def quantize_fp8_per_token(x: torch.Tensor):
    """Quantise [..., H, D] fp32 to float8_e4m3fn per (token, head) vector.

    Returns (x8 with x's shape, scale fp32 of shape x.shape[:-1]).
    """
    x = x.float()
    amax = x.abs().amax(dim=-1)
    scale = amax / FP8_E4M3_MAX
    scale = torch.where(amax == 0, torch.ones_like(scale), scale)
    y = torch.clamp(x / scale.unsqueeze(-1), -FP8_E4M3_MAX, FP8_E4M3_MAX)
    return y.to(torch.float8_e4m3fn), scale


def _scales_token_contiguous(scale: torch.Tensor, varlen: bool) -> torch.Tensor:
    # [B, S, H] -> [B, H, S]; [T, H] -> [H, T]
    if varlen:
        return scale.transpose(0, 1).contiguous()
    return scale.permute(0, 2, 1).contiguous()


def v_token_major(v: torch.Tensor, cu_seqlens_k=None, cu_seqlens_v=None) -> torch.Tensor:
    """V as [B, Sk, Hkv, Dv] (fixed length: a view) or [Tk, Hkv, Dv] (packed):
    depth-major e4m3 V is permuted back, and packed e4m3 V ([Hkv, Dv, Tv],
    sequence b at keys cu_seqlens_v[b] ...) is gathered into token order."""
    if v.dtype != torch.float8_e4m3fn:
        return v
    if v.dim() == 4:
        return v.permute(0, 3, 1, 2)
    parts = []
    for b in range(len(cu_seqlens_k) - 1):
        n = int(cu_seqlens_k[b + 1]) - int(cu_seqlens_k[b])
        s = int(cu_seqlens_v[b])
        parts.append(v[:, :, s:s + n].permute(2, 0, 1))
    return torch.cat(parts, dim=0)


def to_device(inputs: dict, device) -> dict:
    """Copies every tensor of an input dict to ``device`` keeping its strides
    (a padded view such as the depth-major e4m3 V stays padded)."""
    out = {}
    for name, t in inputs.items():
        if isinstance(t, torch.Tensor):
            d = torch.empty_strided(t.size(), t.stride(), dtype=t.dtype, device=device)
            d.copy_(t)
            out[name] = d
        else:
            out[name] = t
    return out


def make_inputs(spec: AttnSpec) -> dict:
    """Draw the inputs of ``spec`` on the CPU.

    Returns a dict with torch CPU tensors: q, k, v, and where applicable
    q_rope, k_rope, q_scale, k_scale, cu_seqlens_q, cu_seqlens_k. FP8 Q/K are
    float8_e4m3fn; everything else bf16 except scales (fp32) and
    cu_seqlens (int32).
    """
    g = torch.Generator().manual_seed(spec.seed)
    if spec.varlen and spec.lengths_q is None:
        raise ValueError("packed spec needs lengths")
    lq, lk = spec.seq_lengths()
    out = {"spec": spec}
    if spec.varlen:
        tq, tk = sum(lq), sum(lk)
        qshape = (tq, spec.heads_q)
        kshape = (tk, spec.heads_kv)
        rshape_k = (tk,)
        cq = [0]
        for n in lq:
            cq.append(cq[-1] + n)
        ck = [0]
        for n in lk:
            ck.append(ck[-1] + n)
        out["cu_seqlens_q"] = torch.tensor(cq, dtype=torch.int32)
        out["cu_seqlens_k"] = torch.tensor(ck, dtype=torch.int32)
    else:
        qshape = (spec.batch, spec.seqlen_q, spec.heads_q)
        kshape = (spec.batch, spec.seqlen_k, spec.heads_kv)
        rshape_k = (spec.batch, spec.seqlen_k)
        out["cu_seqlens_q"] = None
        out["cu_seqlens_k"] = None

    def randn(*shape):
        return torch.randn(*shape, generator=g, dtype=torch.float32)

    if spec.qk_dtype == "fp8":
        if spec.rope:
            raise ValueError("fp8 with a rope part is not a defined workload")
        q32 = randn(*qshape, spec.d_qk)
        k32 = randn(*kshape, spec.d_qk)
        v32 = randn(*kshape, spec.d_v)
        if spec.v_dtype == "fp8" and spec.varlen:
            v8 = torch.clamp(v32, -FP8_E4M3_MAX, FP8_E4M3_MAX).to(torch.float8_e4m3fn)
            # [Tk, Hkv, Dv] -> [Hkv, Dv, Tv]: each sequence's keys start at a
            # multiple of 16 keys (16 bytes, the alignment of a TMA
            # coordinate along the contiguous dimension)
            cv = [0]
            for n in lk:
                cv.append(cv[-1] + (n + 15) // 16 * 16)
            vt = torch.zeros((spec.heads_kv, spec.d_v, max(cv[-1], 16)), dtype=torch.float8_e4m3fn)
            ck = out["cu_seqlens_k"].tolist()
            for b in range(len(lk)):
                vt[:, :, cv[b]:cv[b] + lk[b]] = v8[ck[b]:ck[b + 1]].permute(1, 2, 0)
            v = vt
            out["cu_seqlens_v"] = torch.tensor(cv, dtype=torch.int32)
        elif spec.v_dtype == "fp8":
            v8 = torch.clamp(v32, -FP8_E4M3_MAX, FP8_E4M3_MAX).to(torch.float8_e4m3fn)
            # [B, Sk, Hkv, Dv] -> [B, Hkv, Dv, Sk]; the rows of keys are padded
            # to a multiple of 16 bytes (the alignment a TMA row stride needs)
            # and v is the [..., :Sk] view.
            sk_pad = (spec.seqlen_k + 15) // 16 * 16
            vt = torch.zeros((spec.batch, spec.heads_kv, spec.d_v, sk_pad), dtype=torch.float8_e4m3fn)
            vt[..., :spec.seqlen_k] = v8.permute(0, 2, 3, 1)
            v = vt[..., :spec.seqlen_k]
        else:
            v = v32.to(torch.bfloat16)
        q8, qs = quantize_fp8_per_token(q32)
        k8, ks = quantize_fp8_per_token(k32)
        out.update(q=q8, k=k8, v=v,
                   q_scale=_scales_token_contiguous(qs, spec.varlen),
                   k_scale=_scales_token_contiguous(ks, spec.varlen),
                   q_rope=None, k_rope=None)
        return out
    if spec.qk_dtype != "bf16":
        raise ValueError(f"unknown qk dtype {spec.qk_dtype}")
    if spec.rope:
        q = randn(*qshape, spec.d_qk).to(torch.bfloat16)
        q_rope = randn(*qshape, spec.rope).to(torch.bfloat16)
        k = randn(*kshape, spec.d_qk).to(torch.bfloat16)
        k_rope = randn(*rshape_k, spec.rope).to(torch.bfloat16)
        v = randn(*kshape, spec.d_v).to(torch.bfloat16)
    else:
        q = randn(*qshape, spec.d_qk).to(torch.bfloat16)
        k = randn(*kshape, spec.d_qk).to(torch.bfloat16)
        v = randn(*kshape, spec.d_v).to(torch.bfloat16)
        q_rope = k_rope = None
    out.update(q=q, k=k, v=v, q_rope=q_rope, k_rope=k_rope, q_scale=None, k_scale=None)
    return out


def sample_rows(spec: AttnSpec, n: int, seed: int):
    """Seeded (sequence, query head, query row) triples, uniform over each
    coordinate, plus the first and last row of the first and last head."""
    g = torch.Generator().manual_seed(seed)
    lq, _ = spec.seq_lengths()
    b = torch.randint(0, spec.batch, (n,), generator=g).tolist()
    h = torch.randint(0, spec.heads_q, (n,), generator=g).tolist()
    u = torch.rand((n,), generator=g, dtype=torch.float64).tolist()
    rows = [(bb, hh, min(int(uu * lq[bb]), lq[bb] - 1)) for bb, hh, uu in zip(b, h, u)]
    last_b, last_h = spec.batch - 1, spec.heads_q - 1
    rows += [(0, 0, 0), (0, 0, lq[0] - 1), (last_b, last_h, 0), (last_b, last_h, lq[last_b] - 1)]
    return rows
