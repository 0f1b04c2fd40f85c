"""fp64 CPU oracle for the GPT-2 pre-norm forward.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the package's
smoke check and the benchmark's CPU-baseline leg may import this module.  It
shares no code with the CUDA path and imports nothing from it.

It is the plain definition of the forward written out in float64 with numpy:
no blocking, fusion or reordering beyond what the definitions state.  A matrix
product (``@``) is the one library primitive it uses as a step.  Inputs are the
exact values the GPU receives (bf16 or fp32 values widened to float64); the
oracle rounds nothing.

Sources (web pages, cited by title and section):
  [DB]  "GPT-2 Decoder Block" (AI Engineer Exhaustive), sections "Overview" and
        "How it works": the two pre-norm residual updates, LN with eps=1e-5,
        n_head heads of width d/n_head, 4d GELU MLP, present returned as cache.
  [DO]  "Decoder-only" (CodeBlanks), sections "The decoder-only architecture"
        and "GPT-2 small: 124 million": embedding sum, pre-LN loop, tied head,
        and the per-layer parameter formula with its printed expected output.
  [TC]  "GPT-2 Block - TorchCode", section "Reference Solution": per-head
        scores q k^T / sqrt(d_k), upper-triangular -inf mask, softmax over keys,
        weights times v, heads merged back to [B, T, d].
  [TB]  "GPT-2 Transformer block" (open-model-atlas), the excerpt of
        openai/gpt-2 src/model.py ``norm``: u = mean(x), s = mean((x-u)^2),
        (x-u) * rsqrt(s+eps) * g + b; the two ``block`` residual lines.
  [FF]  "GPT-2 Full Forward Pass" (AI Engineer Exhaustive), section "How it
        works": H0 = gather(W_e, X) + gather(W_p, pos(X, l_past)); L blocks;
        ln_f; logits = LN_f(H) W_e^T; fused c_attn to 3d split into heads;
        past [B, 2, h, T_past, d_h] concatenated on the sequence axis; present
        stacked as [B, L, 2, h, T, d_h].

Readings where the pages leave a step open (each is also listed in the design
notes): GELU is the GPT-2 tanh form by default, the erf form (nn.GELU of the
TorchCode page) is selectable; masked keys are excluded exactly; a query at
absolute position p sees cached and new keys at positions <= p; present holds
all T_past + T positions; the head has no bias and returns exactly V columns;
Linear weights are stored [out, in] (nn.Linear convention of the TorchCode
page) and the fused c_attn rows are Q | K | V, head j at columns
[j*d_h, (j+1)*d_h) of each.

The post-norm block (the arrangement the pages contrast with GPT-2's) is
the one variant written out besides the pre-norm path.

Pins: every function here is checked against values fixed by the pages or by
mathematics (printed parameter counts, closed forms, invariants, brute force on
tiny inputs, library special cases) in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math

import numpy as np

EPS = 1e-5  # [DB] "How it works"; [TB] norm(..., epsilon=1e-5)

BLOCK_KEYS = ("ln1_g", "ln1_b", "attn_w", "attn_b", "proj_w", "proj_b",
              "ln2_g", "ln2_b", "fc_w", "fc_b", "mlp_proj_w", "mlp_proj_b")


# --------------------------------------------------------------------------
# Parameter shapes and counts  ([DO] "GPT-2 small: 124 million")
# --------------------------------------------------------------------------
def block_param_shapes(d: int) -> dict:
    """Shapes of one block's parameters, as the forward below consumes them.

    Two LayerNorms (g, b of [d] each), c_attn d->3d, attn c_proj d->d,
    c_fc d->4d, mlp c_proj 4d->d, every Linear with a bias ([DO], per-layer
    formula; [DB] "How it works")."""
    return {"ln1_g": (d,), "ln1_b": (d,),
            "attn_w": (3 * d, d), "attn_b": (3 * d,),
            "proj_w": (d, d), "proj_b": (d,),
            "ln2_g": (d,), "ln2_b": (d,),
            "fc_w": (4 * d, d), "fc_b": (4 * d,),
            "mlp_proj_w": (d, 4 * d), "mlp_proj_b": (d,)}


def model_param_shapes(n_vocab: int, n_ctx: int, d: int, n_layer: int) -> dict:
    """Shapes of all model parameters: wte [V, d], wpe [n_ctx, d], L blocks,
    ln_f.  The tied head adds no parameter ([DO] "GPT-2 small: 124 million";
    [FF] "How it works")."""
    shapes = {"wte": (n_vocab, d), "wpe": (n_ctx, d)}
    for layer in range(n_layer):
        for k, s in block_param_shapes(d).items():
            shapes[f"h{layer}.{k}"] = s
    shapes["lnf_g"] = (d,)
    shapes["lnf_b"] = (d,)
    return shapes


def count(shapes: dict, prefix: str | None = None) -> int:
    """Number of scalars in the shapes whose names start with ``prefix``."""
    return sum(math.prod(s) for k, s in shapes.items() if prefix is None or k.startswith(prefix))


def _check_block_shapes(p: dict, d: int) -> None:
    for k, s in block_param_shapes(d).items():
        if tuple(np.shape(p[k])) != s:
            raise ValueError(f"block parameter {k} has shape {np.shape(p[k])}, expected {s}")


# --------------------------------------------------------------------------
# Leaf operations
# --------------------------------------------------------------------------
def layer_norm(x: np.ndarray, g: np.ndarray, b: np.ndarray, eps: float = EPS) -> np.ndarray:
    """[TB] norm: over the last axis, u = mean(x), s = mean((x - u)^2) (biased),
    then (x - u) * rsqrt(s + eps), then the diagonal affine x * g + b."""
    x = np.asarray(x, dtype=np.float64)
    u = np.mean(x, axis=-1, keepdims=True)
    s = np.mean(np.square(x - u), axis=-1, keepdims=True)
    y = (x - u) * (1.0 / np.sqrt(s + eps))
    return y * np.asarray(g, np.float64) + np.asarray(b, np.float64)


def gelu(x: np.ndarray, form: str = "tanh") -> np.ndarray:
    """GELU.  "tanh": the GPT-2 form 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)));
    "erf": the exact form x * Phi(x) that nn.GELU() of the TorchCode page computes."""
    x = np.asarray(x, dtype=np.float64)
    if form == "tanh":
        return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))
    if form == "erf":
        from math import erf
        verf = np.vectorize(erf, otypes=[np.float64])
        return 0.5 * x * (1.0 + verf(x / math.sqrt(2.0)))
    raise ValueError(f"unknown GELU form {form!r}")


def linear(x: np.ndarray, w: np.ndarray, b: np.ndarray | None) -> np.ndarray:
    """y = x W^T + b with W stored [out, in] (nn.Linear of the TorchCode page)."""
    y = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T
    if b is not None:
        y = y + np.asarray(b, np.float64)
    return y


def split_heads(t: np.ndarray, n_head: int) -> np.ndarray:
    """[B, T, d] -> [B, h, T, d_h]; head j takes columns [j*d_h, (j+1)*d_h)
    ([TC] view(B, S, h, d_k).transpose(1, 2))."""
    B, T, d = t.shape
    return t.reshape(B, T, n_head, d // n_head).transpose(0, 2, 1, 3)


def merge_heads(t: np.ndarray) -> np.ndarray:
    """[B, h, T, d_h] -> [B, T, h*d_h] ([TC] transpose(1, 2).view(B, S, -1))."""
    B, h, T, dh = t.shape
    return t.transpose(0, 2, 1, 3).reshape(B, T, h * dh)


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Causal scaled dot-product attention per (b, head).

    q [B, h, T, d_h]; k, v [B, h, T_past + T, d_h] (cached keys first, [FF]).
    Query i sits at absolute position p = T_past + i and sees keys j <= p.
    scores = q k^T / sqrt(d_h); keys j > p are excluded (the -inf entries of
    the [TC] triu mask); softmax over keys; output = weights @ v ([TC])."""
    B, h, T, dh = q.shape
    t_all = k.shape[2]
    t_past = t_all - T
    out = np.empty((B, h, T, dh), dtype=np.float64)
    pos_q = t_past + np.arange(T)[:, None]
    pos_k = np.arange(t_all)[None, :]
    masked = pos_k > pos_q
    for bi in range(B):
        for hi in range(h):
            s = (q[bi, hi] @ k[bi, hi].T) / math.sqrt(dh)
            s = np.where(masked, -np.inf, s)
            m = np.max(s, axis=-1, keepdims=True)
            e = np.exp(s - m)
            w = e / np.sum(e, axis=-1, keepdims=True)
            out[bi, hi] = w @ v[bi, hi]
    return out


# --------------------------------------------------------------------------
# Block and full forward
# --------------------------------------------------------------------------
def attn(x_ln: np.ndarray, p: dict, n_head: int, past: np.ndarray | None = None):
    """Attention sub-layer on normalised input x_ln [B, T, d].

    Fused c_attn to 3d, split into Q | K | V and into heads, concatenate the
    cached keys/values ``past`` [B, 2, h, T_past, d_h] on the sequence axis,
    causal attention, merge heads, c_proj ([FF] "How it works"; [TC]).
    Returns (a [B, T, d], present [B, 2, h, T_past + T, d_h])."""
    d = x_ln.shape[-1]
    qkv = linear(x_ln, p["attn_w"], p["attn_b"])
    q = split_heads(qkv[..., 0:d], n_head)
    k = split_heads(qkv[..., d:2 * d], n_head)
    v = split_heads(qkv[..., 2 * d:3 * d], n_head)
    if past is not None:
        past = np.asarray(past, np.float64)
        k = np.concatenate([past[:, 0], k], axis=2)
        v = np.concatenate([past[:, 1], v], axis=2)
    present = np.stack([k, v], axis=1)
    o = merge_heads(causal_attention(q, k, v))
    return linear(o, p["proj_w"], p["proj_b"]), present


def mlp(x_ln: np.ndarray, p: dict, gelu_form: str = "tanh") -> np.ndarray:
    """c_fc d->4d, GELU, c_proj 4d->d ([DB] "How it works"; [TC] mlp)."""
    return linear(gelu(linear(x_ln, p["fc_w"], p["fc_b"]), gelu_form),
                  p["mlp_proj_w"], p["mlp_proj_b"])


def block_forward(x: np.ndarray, p: dict, n_head: int, past: np.ndarray | None = None,
                  gelu_form: str = "tanh"):
    """One pre-norm block ([DB] "How it works"; [TB] block):
    a = Attn(LN1(x)); x = x + a; m = MLP(LN2(x)); x = x + m.
    x [B, T, d]; past [B, 2, h, T_past, d_h] or None.
    Returns (x_out [B, T, d], present [B, 2, h, T_past + T, d_h])."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    if d % n_head != 0:
        raise ValueError("d must be a multiple of n_head")
    _check_block_shapes(p, d)
    a, present = attn(layer_norm(x, p["ln1_g"], p["ln1_b"]), p, n_head, past)
    x = x + a
    m = mlp(layer_norm(x, p["ln2_g"], p["ln2_b"]), p, gelu_form)
    x = x + m
    return x, present


def block_forward_postnorm(x: np.ndarray, p: dict, n_head: int, gelu_form: str = "tanh"):
    """The post-norm arrangement the pages contrast with GPT-2's ([DB]
    "Overview": the original Transformer applies LayerNorm after the residual
    add): x = LN1(x + Attn(x)); x = LN2(x + MLP(x)), with the same parameters
    as the pre-norm block and no cache.  x [B, T, d] -> [B, T, d]."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    if d % n_head != 0:
        raise ValueError("d must be a multiple of n_head")
    _check_block_shapes(p, d)
    a, _ = attn(x, p, n_head)
    x = layer_norm(x + a, p["ln1_g"], p["ln1_b"])
    m = mlp(x, p, gelu_form)
    return layer_norm(x + m, p["ln2_g"], p["ln2_b"])


def embed(ids: np.ndarray, wte: np.ndarray, wpe: np.ndarray, t_past: int = 0) -> np.ndarray:
    """H0[b, t] = wte[ids[b, t]] + wpe[t_past + t] ([FF] "How it works",
    positions_for with the cache offset; positions must stay below n_ctx)."""
    ids = np.asarray(ids)
    B, T = ids.shape
    if t_past + T > wpe.shape[0]:
        raise ValueError("positions must stay below n_ctx")
    if ids.min(initial=0) < 0 or ids.max(initial=0) >= wte.shape[0]:
        raise ValueError("token id out of range")
    pos = t_past + np.arange(T)
    return np.asarray(wte, np.float64)[ids] + np.asarray(wpe, np.float64)[pos][None, :, :]


def forward(ids: np.ndarray, params: dict, n_head: int, past: np.ndarray | None = None,
            positions: np.ndarray | None = None, gelu_form: str = "tanh"):
    """Full uncached or cached forward ([FF] "How it works"; [DO]).

    ids [B, T] int; params: wte, wpe, lnf_g, lnf_b, blocks (list of block dicts);
    past [B, L, 2, h, T_past, d_h] or None.
    ``positions`` selects which positions' logits to return (default: all);
    the hidden states of every position are computed either way.
    Returns (logits [B, len(positions), V], present [B, L, 2, h, T_past+T, d_h])."""
    t_past = 0 if past is None else past.shape[4]
    h = embed(ids, params["wte"], params["wpe"], t_past)
    presents = []
    for layer, p in enumerate(params["blocks"]):
        layer_past = None if past is None else past[:, layer]
        h, present = block_forward(h, p, n_head, layer_past, gelu_form)
        presents.append(present)
    if positions is not None:
        h = h[:, np.asarray(positions)]
    hf = layer_norm(h, params["lnf_g"], params["lnf_b"])
    logits = linear(hf, params["wte"], None)  # tied head, no bias
    return logits, np.stack(presents, axis=1)


# --------------------------------------------------------------------------
# Next-token cross-entropy and greedy choice on the logits
# --------------------------------------------------------------------------
def next_token_loss(logits: np.ndarray, targets: np.ndarray):
    """Per position: the cross-entropy of the next token, -log softmax(z)[y] =
    logsumexp(z) - z[y], and the greedy choice argmax(z) (the lowest index
    among equal maxima).  ([FF] "Overview": training is next-token language
    modelling of p(s_i | s_<i); "How it works": callers take the logits and a
    next-token cross-entropy themselves.)  A negative target marks a position
    without a loss (0).  logits [..., V], targets [...] int.
    Returns (loss [...], argmax [...])."""
    z = np.asarray(logits, np.float64)
    y = np.asarray(targets)
    m = z.max(axis=-1)
    lse = m + np.log(np.exp(z - m[..., None]).sum(axis=-1))
    safe = np.where(y >= 0, y, 0)
    zy = np.take_along_axis(z, safe[..., None], axis=-1)[..., 0]
    loss = np.where(y >= 0, lse - zy, 0.0)
    return loss, np.argmax(z, axis=-1)


def top_k(logits: np.ndarray, k: int):
    """Per position: the k largest logits in descending order with their ids,
    the lower id first among equal values (the greedy choice argmax is the
    first of them, k = 1), and logsumexp(z), which turns them into
    log-probabilities ([FF] "How it works": the logits give the next token's
    distribution; a sampler draws from its most likely candidates).  NaN and
    -inf logits are never chosen: slots beyond the other entries hold id -1
    and value -inf.  logits [..., V].
    Returns (values [..., k], ids [..., k], lse [...])."""
    z = np.asarray(logits, np.float64)
    V = z.shape[-1]
    flat = z.reshape(-1, V)
    ids = np.full((flat.shape[0], k), -1, np.int64)
    vals = np.full((flat.shape[0], k), -np.inf)
    for r in range(flat.shape[0]):
        ok = np.nonzero(~np.isnan(flat[r]) & (flat[r] > -np.inf))[0]
        order = ok[np.lexsort((ok, -flat[r][ok]))][:k]  # by value descending, then id ascending
        ids[r, :len(order)] = order
        vals[r, :len(order)] = flat[r][order]
    m = z.max(axis=-1)
    lse = m + np.log(np.exp(z - m[..., None]).sum(axis=-1))
    return vals.reshape(z.shape[:-1] + (k,)), ids.reshape(z.shape[:-1] + (k,)), lse
