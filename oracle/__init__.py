"""fp64 CPU oracle for the GPT-2 pre-norm forward (test infrastructure only).

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may import this package; the CUDA product path never does.
"""
from .gpt2_oracle import (EPS, attn, block_forward, block_param_shapes, causal_attention,
                          count, embed, forward, gelu, layer_norm, linear, merge_heads, mlp,
                          model_param_shapes, split_heads)

__all__ = ["EPS", "attn", "block_forward", "block_param_shapes", "causal_attention", "count",
           "embed", "forward", "gelu", "layer_norm", "linear", "merge_heads", "mlp",
           "model_param_shapes", "split_heads"]
