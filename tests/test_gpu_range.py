"""The fp16 operand range of the bf16 mode, on the GPU.

The products of the bf16 mode take fp16 operands: the bf16 weights are
converted to fp16, and the LayerNorm, attention and GELU outputs that feed
products are written as fp16.  fp16 holds magnitudes up to 65504, bf16 up to
about 3e38.  A value past the fp16 range (or a non-finite one) must not pass
silently: the kernel that makes it raises the range bit of the context's
error word and gpt2_sync_status returns GPT2_ERR_RANGE.  Values inside the
range, even large ones, give normal results."""
import numpy as np
import pytest
import torch

from oracle import gpt2_oracle as O
from gpt_pre_norm_gb300 import synthetic as S
from tests.helpers import assert_bf16_close, block_to_device, dev, host

pytestmark = pytest.mark.gpu

BIG = 99840.0  # exact in bf16, past the fp16 maximum 65504


@pytest.fixture(scope="module")
def G():
    from gpt_pre_norm_gb300 import build
    build.build()
    from gpt_pre_norm_gb300 import binding
    return binding


def _block(G, p, B, T, x=None, ctx=None):
    w = S.WORKLOADS["block_bf16_d768"]
    if x is None:
        x = S.block_input(w, seed=2, B=B, T=T)
    if ctx is None:
        ctx = G.Context(50257, 1024, w.d, w.n_head, 1, G.GPT2_BF16, max(B, 8), max(T, 8))
    out = G.gpt2_block_forward(ctx, dev(x), block_to_device(p), B, T, w.d, w.n_head)
    return ctx, out, x


def _params():
    return S.block_params(S.WORKLOADS["block_bf16_d768"], seed=2)


@pytest.mark.parametrize("where", ["fc_w", "attn_w", "proj_w", "mlp_proj_w"])
def test_weight_past_fp16_range_is_reported(G, where):
    p = _params()
    p[where] = p[where].copy()
    p[where][3, 5] = BIG
    ctx, _, _ = _block(G, p, 2, 64)
    assert G.gpt2_sync_status(ctx) == G.GPT2_ERR_RANGE
    # The word is cleared by the read: the same context then runs clean.
    p = _params()
    ctx, out, x = _block(G, p, 2, 64, ctx=ctx)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    assert_bf16_close(host(out), O.block_forward(x, p, 12)[0], what="after the range error")


def test_layer_norm_output_past_fp16_range_is_reported(G):
    p = _params()
    p["ln1_g"] = np.full_like(p["ln1_g"], BIG)  # normalised values near 1 times 1e5
    ctx, _, _ = _block(G, p, 2, 64)
    assert G.gpt2_sync_status(ctx) == G.GPT2_ERR_RANGE


@pytest.mark.parametrize("B,T", [(2, 64), (4, 1)])  # tensor-core and few-row kernels
def test_gelu_output_past_fp16_range_is_reported(G, B, T):
    p = _params()
    p["fc_b"] = p["fc_b"].copy()
    p["fc_b"][7] = BIG  # c_fc output about 1e5 in one feature: GELU(x) = x there
    ctx, _, _ = _block(G, p, B, T)
    assert G.gpt2_sync_status(ctx) == G.GPT2_ERR_RANGE


def test_attention_output_past_fp16_range_is_reported(G):
    p = _params()
    p["attn_b"] = p["attn_b"].copy()
    p["attn_b"][2 * 768 + 3] = BIG  # V feature 3 about 1e5 at every key: so is its output
    ctx, _, _ = _block(G, p, 2, 64)
    assert G.gpt2_sync_status(ctx) == G.GPT2_ERR_RANGE


def test_large_residual_rows_stay_in_range(G):
    # A few features of the residual stream near 1e3 (far from the fp16 limit
    # after LayerNorm, which divides by the row's spread): normal results.
    p = _params()
    w = S.WORKLOADS["block_bf16_d768"]
    x = S.block_input(w, seed=3, B=2, T=96).copy()
    x[:, :, [5, 200, 601]] = S.round_to_bf16(np.array([1000.0, -1500.0, 800.0]))
    ctx, out, _ = _block(G, p, 2, 96, x=x)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    ref = O.block_forward(x.astype(np.float64), p, 12)[0]
    got = host(out)
    assert_bf16_close(got, ref, what="large residual features")
    # The branch (out - x) on the ordinary features; on the three large ones
    # the bf16 rounding of the output (half a unit in the last place, 2 near
    # 1000) is larger than the branch itself, so those are held to that bound.
    big = [5, 200, 601]
    rest = np.setdiff1d(np.arange(768), big)
    assert_bf16_close(got[..., rest] - x[..., rest], ref[..., rest] - x[..., rest], tol=5e-2,
                      what="large residual features, branch")
    assert np.all(np.abs(got[..., big] - ref[..., big]) <= 2.0 ** -8 * np.abs(ref[..., big]) + 0.05)
