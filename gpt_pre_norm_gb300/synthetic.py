"""Seeded synthetic inputs for the GPT-2 pre-norm forward.

This module draws random numbers and nothing else: it holds none of the
forward's arithmetic, so both the CUDA path and the fp64 oracle can take their
inputs from it without sharing any computation.

Every tensor is drawn from its own PCG64 stream, ``default_rng([seed, sid])``
with a fixed stream id per tensor name, so any one tensor (one layer's
weights, one sequence's KV cache) can be regenerated on its own.  Values are
drawn in float64, scaled, then rounded once to the storage type; the arrays
returned hold values that are exact in that type (bf16 values are kept in
float32 arrays), so the GPU receives them bit-exactly and the oracle receives
the same values widened to float64.

Workloads mirror the GPT-2 shapes of the pages: GPT-2 small (d=768, 12 heads,
n_ctx=1024, V=50257, "Decoder-only", section "GPT-2 small: 124 million"),
GPT-2 medium and XL widths, and the d=64 / 4-head debug block of
"GPT-2 Block - TorchCode", section "Test Your Implementation".  Residual
output projections are scaled by 1/sqrt(2L) as the init rule in
"GPT-2 Decoder Block", section "Overview", item 3 describes (N = 2L residual
layers).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

BLOCK_TENSORS = ("ln1_g", "ln1_b", "attn_w", "attn_b", "proj_w", "proj_b",
                 "ln2_g", "ln2_b", "fc_w", "fc_b", "mlp_proj_w", "mlp_proj_b")


@dataclass(frozen=True)
class Workload:
    """Shape and value distribution of one synthetic workload."""
    name: str
    kind: str            # "block" | "forward" | "forward_loss" | "decode"
    dtype: str           # "bf16" | "fp32"
    d: int
    n_head: int
    B: int
    T: int
    n_layer: int = 1
    n_vocab: int = 50257
    n_ctx: int = 1024
    t_past: int = 0
    w_std: float = 0.02          # Linear weight std
    b_std: float = 0.02          # Linear bias std
    ln_g_std: float = 0.1        # LN gain = 1 + N(0, ln_g_std)
    ln_b_std: float = 0.02       # LN bias std
    resid_scale_layers: int = 0  # residual projections x 1/sqrt(2*this); 0 = unscaled
    wte_std: float = 0.02
    wpe_std: float = 0.01
    past_std: float = 1.0

    @property
    def d_h(self) -> int:
        return self.d // self.n_head

    @property
    def tokens(self) -> int:
        return self.B * self.T

    @property
    def resid_scale(self) -> float:
        if self.resid_scale_layers <= 0:
            return 1.0
        return 1.0 / math.sqrt(2.0 * self.resid_scale_layers)


WORKLOADS = {
    # d=64, 4 heads, B=2, T=8, fp32: the debug block of the TorchCode page.
    "block_fp32_d64": Workload("block_fp32_d64", "block", "fp32", d=64, n_head=4, B=2, T=8,
                               w_std=0.02, b_std=0.02, ln_g_std=0.1, ln_b_std=0.1),
    # GPT-2-small block, bf16 storage, fp32 accumulate.
    "block_bf16_d768": Workload("block_bf16_d768", "block", "bf16", d=768, n_head=12, B=8, T=1024,
                                resid_scale_layers=12),
    # Full GPT-2-small uncached forward.
    "forward_bf16_gpt2_small": Workload("forward_bf16_gpt2_small", "forward", "bf16", d=768,
                                        n_head=12, B=8, T=1024, n_layer=12,
                                        resid_scale_layers=12),
    # The same forward ending in the next-token loss instead of the logits
    # (targets: the next token id, none at the last position).
    "forward_loss_bf16_gpt2_small": Workload("forward_loss_bf16_gpt2_small", "forward_loss",
                                             "bf16", d=768, n_head=12, B=8, T=1024, n_layer=12,
                                             resid_scale_layers=12),
    # The same forward ending in each position's 8 most likely next tokens and
    # the logsumexp instead of the logits.
    "forward_topk_bf16_gpt2_small": Workload("forward_topk_bf16_gpt2_small", "forward_topk",
                                             "bf16", d=768, n_head=12, B=8, T=1024, n_layer=12,
                                             resid_scale_layers=12),
    # GPT-2-XL-shaped block.
    "block_bf16_d1600": Workload("block_bf16_d1600", "block", "bf16", d=1600, n_head=25, B=4,
                                 T=1024, resid_scale_layers=48),
    # Cached single-token decode, GPT-2-medium shape, new token at position 1023.
    "decode_bf16_gpt2_medium": Workload("decode_bf16_gpt2_medium", "decode", "bf16", d=1024,
                                        n_head=16, B=32, T=1, n_layer=24, t_past=1023,
                                        resid_scale_layers=24),
}

# Stream ids: one independent PCG64 stream per tensor.
_SID_X, _SID_IDS, _SID_WTE, _SID_WPE, _SID_LNF_G, _SID_LNF_B = 0, 1, 2, 3, 4, 5


def _sid_block(layer: int, name: str) -> int:
    return 100 + 16 * layer + BLOCK_TENSORS.index(name)


def _sid_past(b: int, layer: int) -> int:
    return 1_000_000 + 4096 * b + layer


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float values to the nearest bf16 (ties to even); float32 result.

    Finite inputs only (the generators draw bounded normals)."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bf16-exact."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def _store(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16(a)
    return np.asarray(a, dtype=np.float32)


def _normal(seed: int, sid: int, shape, std: float, mean: float = 0.0) -> np.ndarray:
    rng = np.random.default_rng([seed, sid])
    return mean + std * rng.standard_normal(shape)


def block_params(w: Workload, seed: int, layer: int = 0) -> dict:
    """Parameters of one block: LN [d]; Linear weights [out, in]; biases [out]."""
    d, s = w.d, w.resid_scale
    shapes = {"ln1_g": (d,), "ln1_b": (d,), "attn_w": (3 * d, d), "attn_b": (3 * d,),
              "proj_w": (d, d), "proj_b": (d,), "ln2_g": (d,), "ln2_b": (d,),
              "fc_w": (4 * d, d), "fc_b": (4 * d,), "mlp_proj_w": (d, 4 * d),
              "mlp_proj_b": (d,)}
    out = {}
    for name in BLOCK_TENSORS:
        sid = _sid_block(layer, name)
        if name in ("ln1_g", "ln2_g"):
            v = _normal(seed, sid, shapes[name], w.ln_g_std, mean=1.0)
        elif name in ("ln1_b", "ln2_b"):
            v = _normal(seed, sid, shapes[name], w.ln_b_std)
        elif name.endswith("_w"):
            std = w.w_std * (s if name in ("proj_w", "mlp_proj_w") else 1.0)
            v = _normal(seed, sid, shapes[name], std)
        else:
            v = _normal(seed, sid, shapes[name], w.b_std)
        out[name] = _store(v, w.dtype)
    return out


def block_input(w: Workload, seed: int, B: int | None = None, T: int | None = None) -> np.ndarray:
    """Block input x ~ N(0, 1), shape [B, T, d]."""
    B = w.B if B is None else B
    T = w.T if T is None else T
    return _store(_normal(seed, _SID_X, (B, T, w.d), 1.0), w.dtype)


def token_ids(w: Workload, seed: int, B: int | None = None, T: int | None = None) -> np.ndarray:
    """Token ids uniform in [0, V), int32 [B, T]."""
    B = w.B if B is None else B
    T = w.T if T is None else T
    rng = np.random.default_rng([seed, _SID_IDS])
    return rng.integers(0, w.n_vocab, size=(B, T), dtype=np.int64).astype(np.int32)


def embeddings(w: Workload, seed: int) -> dict:
    """wte [V, d] ~ N(0, wte_std); wpe [n_ctx, d] ~ N(0, wpe_std); ln_f like the block LNs."""
    d = w.d
    return {
        "wte": _store(_normal(seed, _SID_WTE, (w.n_vocab, d), w.wte_std), w.dtype),
        "wpe": _store(_normal(seed, _SID_WPE, (w.n_ctx, d), w.wpe_std), w.dtype),
        "lnf_g": _store(_normal(seed, _SID_LNF_G, (d,), w.ln_g_std, mean=1.0), w.dtype),
        "lnf_b": _store(_normal(seed, _SID_LNF_B, (d,), w.ln_b_std), w.dtype),
    }


def model_params(w: Workload, seed: int) -> dict:
    """Embeddings, ln_f and the per-layer block parameters (list of dicts)."""
    p = embeddings(w, seed)
    p["blocks"] = [block_params(w, seed, layer) for layer in range(w.n_layer)]
    return p


def past_kv(w: Workload, seed: int, b: int, layer: int, t_past: int | None = None) -> np.ndarray:
    """Cached keys/values of sequence b at one layer: [2, h, T_past, d_h] ~ N(0, past_std).

    Drawn per (sequence, layer) so a sampled subset can be regenerated alone,
    in float32 (the cache of a full decode workload holds ~1.6e9 values)."""
    t_past = w.t_past if t_past is None else t_past
    rng = np.random.default_rng([seed, _sid_past(b, layer)])
    v = rng.standard_normal((2, w.n_head, t_past, w.d_h), dtype=np.float32)
    if w.past_std != 1.0:
        v *= np.float32(w.past_std)
    return _store(v, w.dtype)

