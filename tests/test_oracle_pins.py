"""Pins for the fp64 oracle: values the pages print, closed forms, invariants,
brute force on tiny inputs and library special cases.

Each check is written so that a plausible mistake in the oracle (a dropped
term, a wrong sign or index, a transposed operand, the other GELU form, an
unbiased variance, a shifted mask) fails at least one of them; the
``test_planted_*`` cases plant such mistakes in the oracle on the CPU and
confirm that a pin catches each one.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import gpt2_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _block_params(d, rng, scale=0.02):
    p = {}
    for k, s in O.block_param_shapes(d).items():
        if k.endswith("_g"):
            p[k] = 1.0 + 0.1 * rng.standard_normal(s)
        else:
            p[k] = scale * rng.standard_normal(s) if k.endswith("_w") else 0.05 * rng.standard_normal(s)
    return p


def _model_params(V, n_ctx, d, L, rng):
    return {"wte": 0.02 * rng.standard_normal((V, d)), "wpe": 0.01 * rng.standard_normal((n_ctx, d)),
            "lnf_g": 1.0 + 0.1 * rng.standard_normal(d), "lnf_b": 0.05 * rng.standard_normal(d),
            "blocks": [_block_params(d, rng, 0.1) for _ in range(L)]}


# ---------------------------------------------------------------- parameters
def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    return rows


def test_param_count_matches_printed_example():
    """Decoder-only page, "Practice GPT-2 parameter count", expected output."""
    (emb, layer), (total,), (untied,) = _read_golden("param_count_gpt2_small.txt")
    s = O.model_param_shapes(50257, 1024, 768, 12)
    assert O.count(s, "wte") + O.count(s, "wpe") == emb
    assert O.count(s, "h0.") == layer
    assert all(O.count(s, f"h{i}.") == layer for i in range(12))
    assert O.count(s) == total
    assert math.prod(s["wte"]) == untied


def test_debug_block_param_count_equals_four_linear_form():
    """The TorchCode block (separate W_q, W_k, W_v, W_o, two LayerNorms, a 4x
    MLP, all with biases) holds exactly as many parameters as the fused form."""
    d, h = 64, 4
    mods = [torch.nn.LayerNorm(d), torch.nn.LayerNorm(d)] + [torch.nn.Linear(d, d) for _ in range(4)]
    mods += [torch.nn.Linear(d, 4 * d), torch.nn.Linear(4 * d, d)]
    n_torch = sum(p.numel() for m in mods for p in m.parameters())
    assert O.count(O.block_param_shapes(d)) == n_torch == 49984
    assert d % h == 0


def test_block_rejects_wrong_parameter_shape():
    rng = _rng()
    p = _block_params(8, rng)
    p["fc_w"] = p["fc_w"].T.copy()
    with pytest.raises(ValueError):
        O.block_forward(rng.standard_normal((1, 3, 8)), p, 2)


# ---------------------------------------------------------------- LayerNorm
@pytest.mark.parametrize("a,c", [(1.0, 0.0), (0.5, 3.0), (2.0, -7.25), (1e-3, 1.0)])
def test_layer_norm_closed_form(a, c):
    """x = c + a*(+1, -1, ...): mean c, biased variance a^2, so with g=1, b=0 the
    output is +-a / sqrt(a^2 + 1e-5) exactly (the norm excerpt, eps = 1e-5)."""
    d = 8
    x = c + a * np.array([1.0 if i % 2 == 0 else -1.0 for i in range(d)])
    y = O.layer_norm(x[None], np.ones(d), np.zeros(d))[0]
    expect = np.array([1.0 if i % 2 == 0 else -1.0 for i in range(d)]) * a / math.sqrt(a * a + 1e-5)
    np.testing.assert_allclose(y, expect, rtol=1e-12, atol=1e-15)


def test_layer_norm_moments_and_affine():
    rng = _rng(1)
    x = 3.0 + 2.0 * rng.standard_normal((5, 37))
    y = O.layer_norm(x, np.ones(37), np.zeros(37))
    for r in range(5):
        row = [float(v) for v in x[r]]
        u = sum(row) / len(row)
        s = sum((v - u) ** 2 for v in row) / len(row)  # biased, brute force
        assert abs(float(np.mean(y[r]))) < 1e-14
        assert abs(float(np.mean(y[r] ** 2)) - s / (s + 1e-5)) < 1e-13
    g, b = rng.standard_normal(37), rng.standard_normal(37)
    np.testing.assert_allclose(O.layer_norm(x, g, b), y * g + b, rtol=1e-13, atol=1e-13)


def test_layer_norm_library_special_case():
    rng = _rng(2)
    x, g, b = rng.standard_normal((4, 6, 24)), rng.standard_normal(24), rng.standard_normal(24)
    ref = F.layer_norm(torch.from_numpy(x), (24,), torch.from_numpy(g), torch.from_numpy(b), eps=1e-5)
    np.testing.assert_allclose(O.layer_norm(x, g, b), ref.numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- GELU
@pytest.mark.parametrize("form", ["tanh", "erf"])
def test_gelu_identities(form):
    x = np.linspace(-6, 6, 241)
    g = O.gelu(x, form)
    np.testing.assert_allclose(g - O.gelu(-x, form), x, rtol=0, atol=1e-14)  # odd part is x/2
    assert O.gelu(np.array([0.0]), form)[0] == 0.0
    assert abs(O.gelu(np.array([30.0]), form)[0] - 30.0) < 1e-12
    assert abs(O.gelu(np.array([-30.0]), form)[0]) < 1e-12


def test_gelu_library_special_case_and_forms_differ():
    x = np.linspace(-8, 8, 801)
    t = torch.from_numpy(x)
    np.testing.assert_allclose(O.gelu(x, "tanh"), F.gelu(t, approximate="tanh").numpy(), atol=1e-14)
    np.testing.assert_allclose(O.gelu(x, "erf"), F.gelu(t).numpy(), atol=1e-14)
    # The two forms differ by ~4.7e-4 near x = -2.7: the choice is observable.
    diff = np.max(np.abs(O.gelu(x, "tanh") - O.gelu(x, "erf")))
    assert 4e-4 < diff < 6e-4


# ---------------------------------------------------------------- Linear
def test_linear_brute_force_non_square():
    rng = _rng(3)
    x, w, b = rng.standard_normal((3, 5)), rng.standard_normal((4, 5)), rng.standard_normal(4)
    y = O.linear(x, w, b)
    assert y.shape == (3, 4)
    for i in range(3):
        for n in range(4):
            ref = b[n] + sum(x[i, k] * w[n, k] for k in range(5))
            assert abs(y[i, n] - ref) < 1e-13


# ---------------------------------------------------------------- attention
def _brute_attention(q, k, v):
    """Per query, per key, scalar loops: query i at position T_past + i,
    keys 0..T_past+i, softmax of q.k / sqrt(d_h), weighted sum of v."""
    B, h, T, dh = q.shape
    tp = k.shape[2] - T
    out = np.zeros_like(q)
    for b in range(B):
        for hh in range(h):
            for i in range(T):
                p = tp + i
                sc = [sum(q[b, hh, i, c] * k[b, hh, j, c] for c in range(dh)) / math.sqrt(dh)
                      for j in range(p + 1)]
                m = max(sc)
                e = [math.exp(s - m) for s in sc]
                z = sum(e)
                for c in range(dh):
                    out[b, hh, i, c] = sum(e[j] * v[b, hh, j, c] for j in range(p + 1)) / z
    return out


@pytest.mark.parametrize("t_past", [0, 3])
def test_attention_brute_force(t_past):
    rng = _rng(4)
    B, h, T, dh = 2, 3, 5, 4
    q = rng.standard_normal((B, h, T, dh))
    k = rng.standard_normal((B, h, t_past + T, dh))
    v = rng.standard_normal((B, h, t_past + T, dh))
    np.testing.assert_allclose(O.causal_attention(q, k, v), _brute_attention(q, k, v),
                               rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    rng = _rng(5)
    B, h, T, dh = 1, 2, 6, 8
    k, v = rng.standard_normal((B, h, T, dh)), rng.standard_normal((B, h, T, dh))
    # T = 1, no cache: the only visible key is the token itself -> output v0.
    q1 = rng.standard_normal((B, h, 1, dh))
    np.testing.assert_allclose(O.causal_attention(q1, k[:, :, :1], v[:, :, :1]), v[:, :, :1], atol=1e-15)
    # q = 0: uniform weights over the visible prefix -> prefix means of v.
    o = O.causal_attention(np.zeros((B, h, T, dh)), k, v)
    prefix_mean = np.cumsum(v, axis=2) / np.arange(1, T + 1)[None, None, :, None]
    np.testing.assert_allclose(o, prefix_mean, rtol=1e-13, atol=1e-14)
    # Adding one vector u to every key shifts every score of a row by q.u:
    # softmax is unchanged.
    q = rng.standard_normal((B, h, T, dh))
    u = rng.standard_normal(dh)
    np.testing.assert_allclose(O.causal_attention(q, k + u, v), O.causal_attention(q, k, v),
                               rtol=1e-11, atol=1e-12)


def test_attention_library_special_case():
    rng = _rng(6)
    q, k, v = (rng.standard_normal((2, 4, 9, 16)) for _ in range(3))
    ref = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                         torch.from_numpy(v), is_causal=True)
    np.testing.assert_allclose(O.causal_attention(q, k, v), ref.numpy(), rtol=1e-12, atol=1e-12)


def test_head_split_and_merge_are_inverse_and_contiguous():
    x = np.arange(2 * 3 * 12, dtype=np.float64).reshape(2, 3, 12)
    s = O.split_heads(x, 4)
    assert s.shape == (2, 4, 3, 3)
    np.testing.assert_array_equal(s[1, 2, 0], x[1, 0, 6:9])  # head j = columns [3j, 3j+3)
    np.testing.assert_array_equal(O.merge_heads(s), x)


# ---------------------------------------------------------------- block
def test_zero_weight_block_is_identity():
    """With all four Linear maps zero (weights and biases), both residual
    branches add zero: the block returns its input exactly."""
    rng = _rng(7)
    d, h = 16, 4
    p = _block_params(d, rng)
    for k in ("attn_w", "attn_b", "proj_w", "proj_b", "fc_w", "fc_b", "mlp_proj_w", "mlp_proj_b"):
        p[k] = np.zeros_like(p[k])
    x = rng.standard_normal((2, 5, d))
    out, present = O.block_forward(x, p, h)
    np.testing.assert_array_equal(out, x)
    assert present.shape == (2, 2, h, 5, d // h)


def test_block_causality():
    rng = _rng(8)
    d, h, T = 16, 4, 7
    p = _block_params(d, rng, 0.3)
    x = rng.standard_normal((2, T, d))
    base, _ = O.block_forward(x, p, h)
    for t in (0, 3, T - 1):
        x2 = x.copy()
        x2[:, t] += rng.standard_normal(d)
        out, _ = O.block_forward(x2, p, h)
        np.testing.assert_array_equal(out[:, :t], base[:, :t])
        assert np.all(np.abs(out[:, t] - base[:, t]).max(axis=-1) > 1e-6)


def _four_linear_attention(x, wq, bq, wk, bk, wv, bv, wo, bo, h):
    """The separate-projection form (TorchCode "Requirements": W_q, W_k, W_v,
    W_o as four Linear maps), written with torch's causal scaled-dot-product
    attention: [B, T, d] -> [B, T, d]."""
    xt = torch.from_numpy(x)
    B, T, d = x.shape

    def heads(t):
        return t.view(B, T, h, d // h).transpose(1, 2)

    q = heads(F.linear(xt, torch.from_numpy(wq), torch.from_numpy(bq)))
    k = heads(F.linear(xt, torch.from_numpy(wk), torch.from_numpy(bk)))
    v = heads(F.linear(xt, torch.from_numpy(wv), torch.from_numpy(bv)))
    o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
    o = o.transpose(1, 2).reshape(B, T, d)
    return F.linear(o, torch.from_numpy(wo), torch.from_numpy(bo)).numpy()


def test_four_linear_form_equals_fused_c_attn():
    """Separate W_q, W_k, W_v concatenated by rows (Q | K | V) are the fused
    c_attn, W_o is c_proj: the oracle's attention reproduces the four-Linear
    form exactly (a wrong concatenation order or head split would not)."""
    rng = _rng(26)
    d, h, B, T = 32, 4, 2, 9
    w = {k: 0.3 * rng.standard_normal((d, d)) for k in ("q", "k", "v", "o")}
    b = {k: 0.1 * rng.standard_normal(d) for k in ("q", "k", "v", "o")}
    x = rng.standard_normal((B, T, d))
    ref = _four_linear_attention(x, w["q"], b["q"], w["k"], b["k"], w["v"], b["v"], w["o"], b["o"], h)
    p = {"attn_w": np.concatenate([w["q"], w["k"], w["v"]], 0),
         "attn_b": np.concatenate([b["q"], b["k"], b["v"]]), "proj_w": w["o"], "proj_b": b["o"]}
    got, _ = O.attn(x, p, h)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-11)


# ------------------------------------------------------- post-norm variant
def test_postnorm_zero_sublayers_is_two_layer_norms():
    """With every Linear map zero, both sublayers add zero, so the post-norm
    block is LN2(LN1(x)); distinct LN1 / LN2 parameters make the order of the
    two normalisations and the residual adds visible (pre-norm would return x,
    a missing residual would return LN of a constant row)."""
    rng = _rng(21)
    d, h = 16, 4
    p = _block_params(d, rng)
    for k in ("attn_w", "attn_b", "proj_w", "proj_b", "fc_w", "fc_b", "mlp_proj_w", "mlp_proj_b"):
        p[k] = np.zeros_like(p[k])
    x = 3.0 * rng.standard_normal((2, 5, d)) + 1.0
    out = O.block_forward_postnorm(x, p, h)
    two = O.layer_norm(O.layer_norm(x, p["ln1_g"], p["ln1_b"]), p["ln2_g"], p["ln2_b"])
    np.testing.assert_allclose(out, two, rtol=0, atol=1e-12)
    assert np.abs(out - x).max() > 0.1


def test_postnorm_output_rows_are_normalised():
    """With LN2's gain 1 and bias 0 every output row has mean 0 and a biased
    variance of s / (s + eps) < 1, whatever the sublayers did."""
    rng = _rng(22)
    d, h = 32, 4
    p = _block_params(d, rng, 0.3)
    p["ln2_g"] = np.ones(d)
    p["ln2_b"] = np.zeros(d)
    x = rng.standard_normal((2, 6, d))
    out = O.block_forward_postnorm(x, p, h)
    np.testing.assert_allclose(out.mean(-1), 0.0, atol=1e-12)
    var = out.var(-1)
    assert np.all(var < 1.0) and np.all(var > 1.0 - 1e-3)


def test_postnorm_mlp_sees_the_normalised_stream():
    """With the attention maps zero, the MLP's input and the second residual
    are LN1(x), which does not change under x -> a x + c (a > 0, c per row)
    except through eps (a relative change of about eps / var(x) ~ 1e-5 here):
    the block output must not change beyond that either (an MLP or a residual
    fed x instead of LN1(x) would change it by O(1))."""
    rng = _rng(23)
    d, h = 16, 4
    p = _block_params(d, rng, 0.5)
    for k in ("attn_w", "attn_b", "proj_w", "proj_b"):
        p[k] = np.zeros_like(p[k])
    x = rng.standard_normal((2, 5, d))
    base = O.block_forward_postnorm(x, p, h)
    moved = O.block_forward_postnorm(2.5 * x + rng.standard_normal((2, 5, 1)), p, h)
    np.testing.assert_allclose(moved, base, rtol=0, atol=1e-4)


@pytest.mark.parametrize("form", ["tanh", "erf"])
def test_postnorm_library_special_case(form):
    """torch's TransformerEncoderLayer with norm_first=False is the post-norm
    arrangement (norm1(x + attention), then norm2(x + feed-forward)) and, with
    the same weights, computes the oracle's post-norm block."""
    rng = _rng(25)
    d, h, B, T = 32, 4, 2, 7
    p = _block_params(d, rng, 0.2)
    x = rng.standard_normal((B, T, d))
    act = (lambda t: F.gelu(t, approximate="tanh")) if form == "tanh" else F.gelu
    layer = torch.nn.TransformerEncoderLayer(d, h, dim_feedforward=4 * d, dropout=0.0, activation=act,
                                             layer_norm_eps=1e-5, batch_first=True, norm_first=False,
                                             dtype=torch.float64)
    sd = {"self_attn.in_proj_weight": p["attn_w"], "self_attn.in_proj_bias": p["attn_b"],
          "self_attn.out_proj.weight": p["proj_w"], "self_attn.out_proj.bias": p["proj_b"],
          "linear1.weight": p["fc_w"], "linear1.bias": p["fc_b"],
          "linear2.weight": p["mlp_proj_w"], "linear2.bias": p["mlp_proj_b"],
          "norm1.weight": p["ln1_g"], "norm1.bias": p["ln1_b"],
          "norm2.weight": p["ln2_g"], "norm2.bias": p["ln2_b"]}
    layer.load_state_dict({k: torch.from_numpy(np.ascontiguousarray(v)) for k, v in sd.items()})
    layer.train(False)
    mask = torch.nn.Transformer.generate_square_subsequent_mask(T, dtype=torch.float64)
    with torch.no_grad():
        ref = layer(torch.from_numpy(x), src_mask=mask, is_causal=True).numpy()
    out = O.block_forward_postnorm(x, p, h, gelu_form=form)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-11)


def test_postnorm_block_causality():
    rng = _rng(24)
    d, h, T = 16, 4, 7
    p = _block_params(d, rng, 0.3)
    x = rng.standard_normal((2, T, d))
    base = O.block_forward_postnorm(x, p, h)
    for t in (0, 3, T - 1):
        x2 = x.copy()
        x2[:, t] += rng.standard_normal(d)
        out = O.block_forward_postnorm(x2, p, h)
        np.testing.assert_array_equal(out[:, :t], base[:, :t])
        assert np.all(np.abs(out[:, t] - base[:, t]).max(axis=-1) > 1e-6)


@pytest.mark.parametrize("form", ["tanh", "erf"])
def test_block_library_special_case(form):
    """torch's pre-norm TransformerEncoderLayer (norm_first, causal mask, 4d MLP,
    eps 1e-5, no dropout) computes the same block from the same weights:
    in_proj = c_attn (Q|K|V rows), out_proj = c_proj, linear1/2 = c_fc / mlp c_proj."""
    rng = _rng(9)
    d, h, B, T = 32, 4, 2, 7
    p = _block_params(d, rng, 0.2)
    x = rng.standard_normal((B, T, d))
    act = (lambda t: F.gelu(t, approximate="tanh")) if form == "tanh" else F.gelu
    layer = torch.nn.TransformerEncoderLayer(d, h, dim_feedforward=4 * d, dropout=0.0, activation=act,
                                             layer_norm_eps=1e-5, batch_first=True, norm_first=True,
                                             dtype=torch.float64)
    sd = {"self_attn.in_proj_weight": p["attn_w"], "self_attn.in_proj_bias": p["attn_b"],
          "self_attn.out_proj.weight": p["proj_w"], "self_attn.out_proj.bias": p["proj_b"],
          "linear1.weight": p["fc_w"], "linear1.bias": p["fc_b"],
          "linear2.weight": p["mlp_proj_w"], "linear2.bias": p["mlp_proj_b"],
          "norm1.weight": p["ln1_g"], "norm1.bias": p["ln1_b"],
          "norm2.weight": p["ln2_g"], "norm2.bias": p["ln2_b"]}
    layer.load_state_dict({k: torch.from_numpy(np.ascontiguousarray(v)) for k, v in sd.items()})
    layer.train(False)
    mask = torch.nn.Transformer.generate_square_subsequent_mask(T, dtype=torch.float64)
    with torch.no_grad():
        ref = layer(torch.from_numpy(x), src_mask=mask, is_causal=True).numpy()
    out, _ = O.block_forward(x, p, h, gelu_form=form)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-11)


def test_present_holds_projected_keys_and_values():
    """present[:, 0] / present[:, 1] are the K / V columns of c_attn(LN1(x)),
    head j at columns [j*d_h, (j+1)*d_h) of the K and V blocks (scalar loops)."""
    rng = _rng(10)
    d, h, B, T = 8, 2, 1, 3
    p = _block_params(d, rng)
    x = rng.standard_normal((B, T, d))
    _, present = O.block_forward(x, p, h)
    ln = O.layer_norm(x, p["ln1_g"], p["ln1_b"])
    dh = d // h
    for which in (0, 1):
        for hh in range(h):
            for t in range(T):
                for c in range(dh):
                    row = (1 + which) * d + hh * dh + c
                    ref = p["attn_b"][row] + sum(ln[0, t, kk] * p["attn_w"][row, kk] for kk in range(d))
                    assert abs(present[0, which, hh, t, c] - ref) < 1e-12


# ---------------------------------------------------------------- full model
def test_zero_block_weights_give_closed_form_logits():
    """All block Linear maps zero: every block is the identity, so the logits are
    LN_f(wte[id] + wpe[pos]) wte^T (closed form, tied head without bias)."""
    rng = _rng(11)
    V, n_ctx, d, L, h = 50, 16, 16, 2, 4
    params = _model_params(V, n_ctx, d, L, rng)
    for p in params["blocks"]:
        for k in ("attn_w", "attn_b", "proj_w", "proj_b", "fc_w", "fc_b", "mlp_proj_w", "mlp_proj_b"):
            p[k] = np.zeros_like(p[k])
    ids = rng.integers(0, V, size=(2, 6))
    logits, present = O.forward(ids, params, h)
    e = torch.from_numpy(params["wte"])[torch.from_numpy(ids)] + torch.from_numpy(params["wpe"][:6])[None]
    ref = F.layer_norm(e, (d,), torch.from_numpy(params["lnf_g"]), torch.from_numpy(params["lnf_b"]),
                       eps=1e-5) @ torch.from_numpy(params["wte"]).T
    np.testing.assert_allclose(logits, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert logits.shape == (2, 6, V)
    assert present.shape == (2, L, 2, h, 6, d // h)


def test_forward_causality():
    rng = _rng(12)
    V, n_ctx, d, L, h = 40, 16, 16, 2, 2
    params = _model_params(V, n_ctx, d, L, rng)
    ids = rng.integers(0, V, size=(2, 8))
    base, _ = O.forward(ids, params, h)
    ids2 = ids.copy()
    ids2[:, 5] = (ids2[:, 5] + 7) % V
    out, _ = O.forward(ids2, params, h)
    np.testing.assert_array_equal(out[:, :5], base[:, :5])
    assert np.abs(out[:, 5] - base[:, 5]).max() > 1e-6


def test_cached_decode_equals_uncached():
    """Feeding the newest token with the previous present reproduces the
    uncached logits and present position by position (Full Forward Pass page,
    end of "How it works")."""
    rng = _rng(13)
    V, n_ctx, d, L, h = 40, 16, 16, 3, 4
    params = _model_params(V, n_ctx, d, L, rng)
    ids = rng.integers(0, V, size=(2, 9))
    full, full_present = O.forward(ids, params, h)
    _, present = O.forward(ids[:, :4], params, h)
    for t in range(4, 9):
        step, present = O.forward(ids[:, t:t + 1], params, h, past=present)
        np.testing.assert_allclose(step[:, 0], full[:, t], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(present, full_present, rtol=1e-11, atol=1e-12)
    # Chunked: a 3-token continuation with a cache equals the uncached positions.
    _, p5 = O.forward(ids[:, :5], params, h)
    chunk, _ = O.forward(ids[:, 5:8], params, h, past=p5)
    np.testing.assert_allclose(chunk, full[:, 5:8], rtol=1e-11, atol=1e-12)


def test_positions_select_rows_and_context_limit():
    rng = _rng(14)
    V, n_ctx, d, L, h = 30, 8, 8, 1, 2
    params = _model_params(V, n_ctx, d, L, rng)
    ids = rng.integers(0, V, size=(1, 8))
    full, _ = O.forward(ids, params, h)
    some, _ = O.forward(ids, params, h, positions=[0, 5, 7])
    np.testing.assert_array_equal(some, full[:, [0, 5, 7]])
    with pytest.raises(ValueError):
        O.embed(rng.integers(0, V, size=(1, 9)), params["wte"], params["wpe"])
    with pytest.raises(ValueError):
        O.embed(np.array([[V]]), params["wte"], params["wpe"])


# ---------------------------------------------------------------- planted mistakes
def _ln_unbiased(x, g, b, eps=1e-5):
    x = np.asarray(x, np.float64)
    u = x.mean(-1, keepdims=True)
    s = ((x - u) ** 2).sum(-1, keepdims=True) / (x.shape[-1] - 1)
    return (x - u) / np.sqrt(s + eps) * g + b


def _ln_eps_outside(x, g, b, eps=1e-5):
    x = np.asarray(x, np.float64)
    u = x.mean(-1, keepdims=True)
    s = ((x - u) ** 2).mean(-1, keepdims=True)
    return (x - u) / (np.sqrt(s) + eps) * g + b


@pytest.mark.parametrize("bad", [_ln_unbiased, _ln_eps_outside])
def test_planted_layer_norm_mistake_is_caught(monkeypatch, bad):
    monkeypatch.setattr(O, "layer_norm", bad)
    with pytest.raises(AssertionError):
        test_layer_norm_closed_form(0.5, 3.0)


def _attn_mask_excludes_self(q, k, v):
    B, h, T, dh = q.shape
    tp = k.shape[2] - T
    out = np.empty_like(q)
    for b in range(B):
        for hh in range(h):
            s = q[b, hh] @ k[b, hh].T / math.sqrt(dh)
            masked = np.arange(k.shape[2])[None] >= (tp + np.arange(T))[:, None]
            masked[:, 0] = False  # keep one key so rows stay finite
            s = np.where(masked, -np.inf, s)
            e = np.exp(s - s.max(-1, keepdims=True))
            out[b, hh] = (e / e.sum(-1, keepdims=True)) @ v[b, hh]
    return out


def _attn_scale_by_dh(q, k, v):
    return _scaled_attention(q, k, v, 1.0 / q.shape[-1])


def _scaled_attention(q, k, v, scale):
    B, h, T, dh = q.shape
    tp = k.shape[2] - T
    out = np.empty_like(q)
    for b in range(B):
        for hh in range(h):
            s = q[b, hh] @ k[b, hh].T * scale
            masked = np.arange(k.shape[2])[None] > (tp + np.arange(T))[:, None]
            s = np.where(masked, -np.inf, s)
            e = np.exp(s - s.max(-1, keepdims=True))
            out[b, hh] = (e / e.sum(-1, keepdims=True)) @ v[b, hh]
    return out


@pytest.mark.parametrize("bad", [_attn_mask_excludes_self, _attn_scale_by_dh])
def test_planted_attention_mistake_is_caught(monkeypatch, bad):
    monkeypatch.setattr(O, "causal_attention", bad)
    with pytest.raises(AssertionError):
        test_attention_brute_force(0)


def test_planted_gelu_form_mistake_is_caught(monkeypatch):
    orig = O.gelu
    monkeypatch.setattr(O, "gelu", lambda x, form="tanh": orig(x, "erf"))
    with pytest.raises(AssertionError):
        test_block_library_special_case("tanh")


def test_planted_transposed_head_split_is_caught(monkeypatch):
    def bad_split(t, n_head):  # heads interleaved instead of contiguous
        B, T, d = t.shape
        return t.reshape(B, T, d // n_head, n_head).transpose(0, 3, 1, 2)
    monkeypatch.setattr(O, "split_heads", bad_split)
    with pytest.raises(AssertionError):
        test_block_library_special_case("tanh")


def test_planted_position_offset_mistake_is_caught(monkeypatch):
    orig = O.embed
    monkeypatch.setattr(O, "embed", lambda ids, wte, wpe, t_past=0: orig(ids, wte, wpe, 0))
    with pytest.raises(AssertionError):
        test_cached_decode_equals_uncached()


# ------------------------------------------------------- next-token loss ----
def test_loss_closed_forms():
    """Equal logits give log V; one logit c above V-1 equal others gives
    log(1 + (V-1) e^-c) for that target and c + log(1 + (V-1) e^-c) for any
    other; a negative target gives 0; the argmax is the lowest maximal index."""
    V = 7
    z = np.zeros((3, V))
    z[1, 4] = 2.5
    z[2, [2, 5]] = 1.0
    loss, am = O.next_token_loss(z, np.array([3, 4, -1]))
    np.testing.assert_allclose(loss[0], math.log(V), rtol=1e-15)
    np.testing.assert_allclose(loss[1], math.log(1 + (V - 1) * math.exp(-2.5)), rtol=1e-14)
    assert loss[2] == 0.0
    loss2, _ = O.next_token_loss(z[1:2], np.array([0]))
    np.testing.assert_allclose(loss2[0], 2.5 + math.log(1 + (V - 1) * math.exp(-2.5)), rtol=1e-14)
    assert list(am) == [0, 4, 2]


def test_loss_shift_invariance_and_library_special_case():
    """Adding a constant to a row of logits changes neither the loss nor the
    argmax; the values equal torch's cross_entropy (reduction none)."""
    rng = _rng(27)
    z = 3.0 * rng.standard_normal((4, 5, 50))
    y = rng.integers(0, 50, size=(4, 5))
    loss, am = O.next_token_loss(z, y)
    loss2, am2 = O.next_token_loss(z + 100.0 * rng.standard_normal((4, 5, 1)), y)
    np.testing.assert_allclose(loss2, loss, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(am2, am)
    ref = F.cross_entropy(torch.from_numpy(z.reshape(-1, 50)), torch.from_numpy(y.reshape(-1)),
                          reduction="none").numpy().reshape(4, 5)
    np.testing.assert_allclose(loss, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(am, torch.from_numpy(z).argmax(-1).numpy())


# ------------------------------------------------------------------- top-k ----
def test_top_k_hand_example_ties_nan_and_short_rows():
    """Worked by hand: values 3 (ids 4 and 1), 5, NaN, 3 again at id 7: the order is
    5 (id 2), then the 3s by id (1, 4, 7); NaN (id 0) is never chosen.  A row
    with only two entries above -inf gives them, then id -1 with -inf."""
    z = np.array([[np.nan, 3.0, 5.0, -1.0, 3.0, 0.5, -2.0, 3.0]])
    vals, ids, _ = O.top_k(z, 4)
    assert ids.tolist() == [[2, 1, 4, 7]]
    assert vals.tolist() == [[5.0, 3.0, 3.0, 3.0]]
    z2 = np.array([[-np.inf, 1.0, -np.inf, np.nan, 2.0]])
    vals2, ids2, _ = O.top_k(z2, 3)
    assert ids2.tolist() == [[4, 1, -1]]
    assert vals2.tolist() == [[2.0, 1.0, -np.inf]]


def test_top_k_first_is_argmax_and_set_is_the_k_largest():
    """k = 1 is numpy's argmax (lowest index among equal maxima); for any k the
    chosen values are the k largest of the row (as a sorted multiset), sorted
    descending, the ids distinct and pointing at those values."""
    rng = _rng(41)
    z = np.round(4.0 * rng.standard_normal((6, 7, 97)), 1)  # rounding makes ties common
    v1, i1, _ = O.top_k(z, 1)
    np.testing.assert_array_equal(i1[..., 0], np.argmax(z, axis=-1))
    for k in (3, 8):
        vals, ids, _ = O.top_k(z, k)
        np.testing.assert_array_equal(vals, -np.sort(-z, axis=-1)[..., :k])
        np.testing.assert_array_equal(np.take_along_axis(z, ids, axis=-1), vals)
        assert all(len(set(r)) == k for r in ids.reshape(-1, k).tolist())
        # among equal values the lower id comes first
        same = vals[..., 1:] == vals[..., :-1]
        assert np.all(ids[..., 1:][same] > ids[..., :-1][same])


def test_top_k_lse_matches_the_loss_and_torch():
    """logsumexp ties the top-k output to the cross-entropy: lse - z[y] is the
    loss of target y; and it equals torch's logsumexp.  Shifting a row by a
    constant shifts its values and lse and keeps its ids."""
    rng = _rng(42)
    z = 3.0 * rng.standard_normal((4, 5, 60))
    y = rng.integers(0, 60, size=(4, 5))
    vals, ids, lse = O.top_k(z, 5)
    loss, _ = O.next_token_loss(z, y)
    np.testing.assert_allclose(lse - np.take_along_axis(z, y[..., None], -1)[..., 0], loss,
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.from_numpy(z), dim=-1).numpy(),
                               rtol=1e-12, atol=1e-12)
    c = 100.0 * rng.standard_normal((4, 5, 1))
    vals2, ids2, lse2 = O.top_k(z + c, 5)
    np.testing.assert_array_equal(ids2, ids)
    np.testing.assert_allclose(vals2, vals + c, rtol=1e-12, atol=1e-9)
    np.testing.assert_allclose(lse2, lse + c[..., 0], rtol=1e-12, atol=1e-9)


def _topk_higher_id_first(logits, k):
    z = np.asarray(logits, np.float64)
    V = z.shape[-1]
    flat = np.where(np.isnan(z), -np.inf, z).reshape(-1, V)
    ids = np.stack([np.lexsort((-np.arange(V), -r))[:k] for r in flat]).reshape(z.shape[:-1] + (k,))
    m = z.max(-1)
    return np.take_along_axis(z, ids, -1), ids, m + np.log(np.exp(z - m[..., None]).sum(-1))


def _topk_nan_as_largest(logits, k):
    z = np.asarray(logits, np.float64)
    V = z.shape[-1]
    flat = np.where(np.isnan(z), np.inf, z).reshape(-1, V)
    ids = np.stack([np.lexsort((np.arange(V), -r))[:k] for r in flat]).reshape(z.shape[:-1] + (k,))
    m = np.nanmax(z, -1)
    return np.take_along_axis(z, ids, -1), ids, m


@pytest.mark.parametrize("bad", [_topk_higher_id_first, _topk_nan_as_largest])
def test_planted_top_k_mistake_is_caught(monkeypatch, bad):
    monkeypatch.setattr(O, "top_k", bad)
    with pytest.raises(AssertionError):
        test_top_k_hand_example_ties_nan_and_short_rows()
