"""Float64 CPU oracle of the KV-cached decoder step (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package. The CUDA library shares no code with it
and never calls it.
"""
from .decoder import (OracleModel, Sequence, argmax_rule, causal_attention, dequant_q8_0, forward_full,
                      gelu_tanh, gelu_tanh_arg, greedy_generate, layer_norm, llama3_scaled_inv_freq, rms_norm, rope,
                      round_bf16, sample_top_k, silu, softmax, teacher_forced, top2_margin)
from .brute import BruteModel

__all__ = ["OracleModel", "Sequence", "argmax_rule", "causal_attention", "dequant_q8_0", "forward_full", "gelu_tanh",
           "gelu_tanh_arg", "greedy_generate", "layer_norm", "llama3_scaled_inv_freq", "rms_norm", "rope", "round_bf16", "sample_top_k", "silu", "softmax",
           "teacher_forced", "top2_margin", "BruteModel"]
