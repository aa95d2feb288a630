"""GB300 (sm_103a) fused attention forward: a C-ABI CUDA library and its
Python binding.

``forward`` computes O = softmax(scale * Q K^T + causal mask) V and the per-row
log-sum-exp with one persistent tcgen05/TMA kernel (and, with split-KV, a
small merge kernel); ``prepare`` fixes the tensors and options of a call so
that repeated calls skip the argument marshalling. Build the library with
``attention_forward_sm100_gb300.build.build()``.
"""
from ._binding import (AttnError, Params, PlanInfo, PreparedForward, check, default_workspace, forward, key_range,
                       last_error, lib, make_params, plan, prepare, schedule, workspace_bytes)

__all__ = ["AttnError", "Params", "PlanInfo", "PreparedForward", "check", "default_workspace", "forward",
           "key_range", "last_error", "lib", "make_params", "plan", "prepare", "schedule", "workspace_bytes"]
