"""CPU oracle (test infrastructure only; never imported by the library).

See ``opt_oracle`` for what it computes and which passages it follows.
"""
from .opt_oracle import (E4M3_MAX, OracleModel, dequantize_rows, e4m3_round, generate, greedy,
                         layer_norm, log_softmax_pick, lora_delta, merge_lora,
                         quantize_rows_e4m3, sample_token, sample_uniforms, splitmix64_output,
                         to_f32)

__all__ = ["E4M3_MAX", "OracleModel", "dequantize_rows", "e4m3_round", "quantize_rows_e4m3",
           "generate", "greedy", "layer_norm", "log_softmax_pick",
           "lora_delta", "merge_lora", "sample_token", "sample_uniforms", "splitmix64_output",
           "to_f32"]
