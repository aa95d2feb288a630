"""CPU float64 oracle of the fused attention forward.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
never imports it, and it imports nothing from the product.
"""
from .mha import attention, attention_rows, attention_head, scores, softmax_lse, visible_mask

__all__ = ["attention", "attention_rows", "attention_head", "scores", "softmax_lse", "visible_mask"]
