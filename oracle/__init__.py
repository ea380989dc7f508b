"""CPU oracle (test infrastructure only; never imported by the library).

See ``opt_oracle`` for what it computes and which passages it follows.
"""
from .opt_oracle import (OracleModel, generate, greedy, layer_norm, log_softmax_pick,
                         lora_delta, merge_lora, sample_token, sample_uniforms,
                         splitmix64_output, to_f32)

__all__ = ["OracleModel", "generate", "greedy", "layer_norm", "log_softmax_pick",
           "lora_delta", "merge_lora", "sample_token", "sample_uniforms", "splitmix64_output",
           "to_f32"]
