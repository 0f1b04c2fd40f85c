"""Kernel-by-kernel parity with the fp64 oracle, through the C ABI.

Sizes span several tiles and a ragged tail (128-row GEMM tiles, 64-column
chunks, 128-query / 64-key attention tiles, split-KV chunks)."""
import numpy as np
import pytest
import torch

from oracle import gpt2_oracle as O
from gpt_pre_norm_gb300 import synthetic as S
from tests.helpers import assert_bf16_close, assert_fp32_close, assert_gemm_f32_close, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    from gpt_pre_norm_gb300 import build
    build.build()
    from gpt_pre_norm_gb300 import binding
    return binding


def _ctx(G, mode, d=768, h=12, B=8, T=1024, V=50257, L=1):
    return G.Context(V, 1024, d, h, L, mode, B, T)


def _rand(rng, shape, std=1.0, bf16=True):
    a = std * rng.standard_normal(shape)
    return S.round_to_bf16(a) if bf16 else a.astype(np.float32)


# ------------------------------------------------------------- LayerNorm ----
@pytest.mark.parametrize("d", [64, 768, 1024, 1600, 100])
@pytest.mark.parametrize("x_fp32", [True, False])
@pytest.mark.parametrize("rows", [1000, 2049])  # one row per warp; two (an odd count)
def test_layer_norm_bf16(G, d, x_fp32, rows):
    rng = np.random.default_rng(d + rows)
    x = (2.0 * rng.standard_normal((rows, d)) + 0.5).astype(np.float32)
    if not x_fp32:
        x = S.round_to_bf16(x)
    g = _rand(rng, (d,), 0.1) + 1.0
    g = S.round_to_bf16(g)
    b = _rand(rng, (d,), 0.1)
    y = G.gpt2_layer_norm(G.GPT2_BF16, dev(x, torch.float32 if x_fp32 else torch.bfloat16),
                          dev(g), dev(b))
    torch.cuda.synchronize()
    ref = O.layer_norm(x.astype(np.float64), g, b)
    got = host(y)
    assert_bf16_close(got, ref, what=f"LN d={d}")
    # bf16 output: each element within a few bf16 ulps of the exact value.
    assert np.max(np.abs(got - ref) / (np.abs(ref) + 1e-2)) < 2 ** -7


@pytest.mark.parametrize("d,rows", [(64, 37), (15, 37), (768, 37), (768, 4095)])
def test_layer_norm_fp32(G, d, rows):
    rng = np.random.default_rng(7 + d)
    x = _rand(rng, (rows, d), 3.0, bf16=False) - 1.0
    g = _rand(rng, (d,), 0.2, bf16=False) + 1.0
    b = _rand(rng, (d,), 0.2, bf16=False)
    y = G.gpt2_layer_norm(G.GPT2_FP32, dev(x, torch.float32), dev(g, torch.float32),
                          dev(b, torch.float32))
    torch.cuda.synchronize()
    assert_fp32_close(host(y), O.layer_norm(x, g, b), what=f"LN fp32 d={d}")


# ----------------------------------------------------------------- GEMMs ----
# K >= 1024 with M > 128 runs on CTA pairs (256-row tiles); (200, 640, 1024) leaves the
# second CTA's rows partly outside M.
GEMM_SHAPES = [(128, 256, 64), (300, 200, 768), (1000, 768, 768), (129, 2304, 768),
               (77, 3072, 200), (1, 64, 64), (32, 1024, 1024), (640, 768, 3072),
               (200, 640, 1024), (1000, 200, 1600)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_linear_bias_resid_bf16(G, M, N, K):
    rng = np.random.default_rng(M * 7 + N + K)
    ctx = _ctx(G, G.GPT2_BF16)
    A = _rand(rng, (M, K))
    W = _rand(rng, (N, K), 0.05)
    bias = _rand(rng, (N,), 0.1)
    resid = rng.standard_normal((M, N)).astype(np.float32)
    Ad, Wd, bd = dev(A), dev(W), dev(bias)
    ref = O.linear(A, W, bias)
    out = G.gpt2_linear(ctx, G.GPT2_EPI_BIAS_RESID, Ad, Wd, bd, dev(resid, torch.float32))
    out_b = G.gpt2_linear(ctx, G.GPT2_EPI_BIAS, Ad, Wd, bd)
    assert G.gpt2_sync_status(ctx) == 0
    # fp32 output: products of bf16 values are exact; only the accumulation differs.
    assert_gemm_f32_close(host(out), ref + resid, A, W, what="linear+resid")
    assert_bf16_close(host(out_b), ref, what="linear+bias")
    assert np.max(np.abs(host(out_b) - ref)) <= 2 ** -7 * np.max(np.abs(ref)) + 1e-3


@pytest.mark.parametrize("M,N,K", [(300, 3072, 768), (128, 256, 1600), (384, 3072, 1024)])
def test_linear_gelu_bf16(G, M, N, K):
    rng = np.random.default_rng(11)
    ctx = _ctx(G, G.GPT2_BF16)
    A = _rand(rng, (M, K))
    W = _rand(rng, (N, K), 0.05)
    bias = _rand(rng, (N,), 0.5)
    out = G.gpt2_linear(ctx, G.GPT2_EPI_BIAS_GELU, dev(A), dev(W), dev(bias))
    assert G.gpt2_sync_status(ctx) == 0
    assert_bf16_close(host(out), O.gelu(O.linear(A, W, bias)), what="linear+gelu")


@pytest.mark.parametrize("M,V,K", [(130, 50257, 768), (1, 50257, 768), (3, 50257, 768),
                                   (256, 1000, 768), (77, 1001, 768), (200, 1002, 768),
                                   (33, 1003, 768), (5, 40, 768), (300, 50257, 1024),
                                   (260, 1001, 1600)])
def test_tied_head_logits(G, M, V, K):
    rng = np.random.default_rng(M + V)
    ctx = _ctx(G, G.GPT2_BF16, V=V)
    A = _rand(rng, (M, K))
    W = _rand(rng, (V, K), 0.02)
    out = G.gpt2_linear(ctx, G.GPT2_EPI_LOGITS, dev(A), dev(W))
    assert G.gpt2_sync_status(ctx) == 0
    assert out.shape == (M, V)
    assert_gemm_f32_close(host(out), O.linear(A, W, None), A, W, what="logits")


def test_linear_fp32(G):
    rng = np.random.default_rng(3)
    ctx = _ctx(G, G.GPT2_FP32, d=64, h=4)
    M, N, K = 70, 130, 66
    A = _rand(rng, (M, K), bf16=False)
    W = _rand(rng, (N, K), 0.1, bf16=False)
    bias = _rand(rng, (N,), 0.1, bf16=False)
    resid = _rand(rng, (M, N), bf16=False)
    f = lambda a: dev(a, torch.float32)  # noqa: E731
    o1 = G.gpt2_linear(ctx, G.GPT2_EPI_BIAS, f(A), f(W), f(bias))
    o2 = G.gpt2_linear(ctx, G.GPT2_EPI_BIAS_GELU, f(A), f(W), f(bias))
    o3 = G.gpt2_linear(ctx, G.GPT2_EPI_BIAS_RESID, f(A), f(W), f(bias), f(resid))
    o4 = G.gpt2_linear(ctx, G.GPT2_EPI_LOGITS, f(A), f(W))
    assert G.gpt2_sync_status(ctx) == 0
    ref = O.linear(A, W, bias)
    assert_fp32_close(host(o1), ref)
    assert_fp32_close(host(o2), O.gelu(ref))
    assert_fp32_close(host(o3), ref + resid)
    assert_fp32_close(host(o4), O.linear(A, W, None))


# ------------------------------------------------------------- attention ----
def _attn_case(rng, B, h, T, t_past, t_cap, dh=64, bf16=True):
    q = _rand(rng, (B, h, T, dh), bf16=bf16)
    kv = np.zeros((B, 2, h, t_cap, dh), np.float32)
    kv[:, :, :, :t_past + T] = _rand(rng, (B, 2, h, t_past + T, dh), bf16=bf16)
    # Poison the unused capacity: the kernels must never read it.
    kv[:, :, :, t_past + T:] = np.nan
    return q, kv


# Query tiles of 128 rows are processed in pairs sharing each 128-key step:
# T = 256 is one full pair, 384 and 513 end in a pair with one (partly)
# filled tile, 257 after 63 cached positions puts every tile across two steps.
@pytest.mark.parametrize("B,h,T,t_past", [(2, 3, 1, 0), (2, 3, 2, 0), (1, 2, 127, 0),
                                          (2, 3, 129, 0), (1, 12, 300, 0), (2, 2, 70, 5),
                                          (1, 2, 200, 130), (1, 1, 1024, 0), (1, 2, 256, 0),
                                          (2, 1, 384, 0), (1, 2, 513, 0), (2, 2, 257, 63)])
def test_attention_prefill_bf16(G, B, h, T, t_past):
    rng = np.random.default_rng(B * 1000 + T + t_past)
    ctx = _ctx(G, G.GPT2_BF16)
    t_cap = t_past + T + 3
    q, kv = _attn_case(rng, B, h, T, t_past, t_cap)
    out = G.gpt2_attention(ctx, dev(q), dev(kv), t_past)
    assert G.gpt2_sync_status(ctx) == 0
    k = kv[:, 0, :, :t_past + T].astype(np.float64)
    v = kv[:, 1, :, :t_past + T].astype(np.float64)
    ref = O.merge_heads(O.causal_attention(q.astype(np.float64), k, v))
    got = host(out)
    assert_bf16_close(got, ref, what="prefill attention")
    assert np.max(np.abs(got - ref)) < 3e-2


def test_attention_prefill_bf16_growing_scores(G):
    # Keys grow with their position, so a row's maximum score keeps rising
    # from step to step by more than the online softmax lets its reference
    # maximum lag: the kernel must rescale the running output and sum.
    rng = np.random.default_rng(77)
    B, h, T = 2, 2, 1024
    ctx = _ctx(G, G.GPT2_BF16)
    q, kv = _attn_case(rng, B, h, T, 0, T)
    q = S.round_to_bf16(2.0 * q)
    grow = (1.0 + np.arange(T) / 128.0)[None, None, :, None]
    kv[:, 0] = S.round_to_bf16(kv[:, 0] * grow)
    out = G.gpt2_attention(ctx, dev(q), dev(kv), 0)
    assert G.gpt2_sync_status(ctx) == 0
    ref = O.merge_heads(O.causal_attention(q.astype(np.float64), kv[:, 0].astype(np.float64),
                                           kv[:, 1].astype(np.float64)))
    got = host(out)
    assert_bf16_close(got, ref, what="prefill attention, growing scores")
    assert np.max(np.abs(got - ref)) < 3e-2


@pytest.mark.parametrize("B,h,t_past", [(32, 16, 1023), (1, 2, 1), (2, 3, 100), (1, 4, 1000),
                                        (3, 1, 5000 // 5)])
def test_attention_decode_bf16(G, B, h, t_past):
    rng = np.random.default_rng(B + h + t_past)
    ctx = _ctx(G, G.GPT2_BF16, d=1024, h=16, B=max(B, 8))
    t_cap = t_past + 1 + 1
    q, kv = _attn_case(rng, B, h, 1, t_past, t_cap)
    out = G.gpt2_attention(ctx, dev(q), dev(kv), t_past)
    assert G.gpt2_sync_status(ctx) == 0
    k = kv[:, 0, :, :t_past + 1].astype(np.float64)
    v = kv[:, 1, :, :t_past + 1].astype(np.float64)
    ref = O.merge_heads(O.causal_attention(q.astype(np.float64), k, v))
    got = host(out)
    assert_bf16_close(got, ref, what="decode attention")
    assert np.max(np.abs(got - ref)) < 3e-2


@pytest.mark.parametrize("dh,T,t_past", [(16, 8, 0), (64, 33, 4), (24, 5, 0), (256, 3, 2)])
def test_attention_fp32(G, dh, T, t_past):
    rng = np.random.default_rng(dh + T)
    h = 3
    ctx = G.Context(100, 1024, dh * h, h, 1, G.GPT2_FP32, 2, 64)
    q, kv = _attn_case(rng, 2, h, T, t_past, t_past + T, dh=dh, bf16=False)
    out = G.gpt2_attention(ctx, dev(q, torch.float32), dev(kv, torch.float32), t_past)
    assert G.gpt2_sync_status(ctx) == 0
    ref = O.merge_heads(O.causal_attention(q.astype(np.float64), kv[:, 0].astype(np.float64),
                                           kv[:, 1].astype(np.float64)))
    assert_fp32_close(host(out), ref, what="fp32 attention")


# ----------------------------------------------------------------- embed ----
@pytest.mark.parametrize("t_past", [0, 17])
def test_embed_bf16(G, t_past):
    w = S.WORKLOADS["forward_bf16_gpt2_small"]
    rng = np.random.default_rng(5)
    emb = S.embeddings(w, seed=1)
    ids = rng.integers(0, w.n_vocab, size=(3, 50)).astype(np.int32)
    ctx = _ctx(G, G.GPT2_BF16)
    H = G.gpt2_embed(ctx, dev(ids, torch.int32), dev(emb["wte"]), dev(emb["wpe"]), t_past)
    assert G.gpt2_sync_status(ctx) == 0
    ref = O.embed(ids, emb["wte"], emb["wpe"], t_past)
    # One fp32 add of two bf16 values: exact or within half an fp32 ulp.
    np.testing.assert_allclose(host(H), ref, rtol=2 ** -24, atol=0)


def test_embed_rejects_bad_token_on_device(G):
    w = S.WORKLOADS["forward_bf16_gpt2_small"]
    emb = S.embeddings(w, seed=1)
    ids = np.array([[0, w.n_vocab, 5]], np.int32)
    ctx = _ctx(G, G.GPT2_BF16)
    G.gpt2_embed(ctx, dev(ids, torch.int32), dev(emb["wte"]), dev(emb["wpe"]))
    assert G.gpt2_sync_status(ctx) == G.GPT2_ERR_INVALID_ARG
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK  # the error word was cleared


# --------------------------------------------------------- failure path ----
def test_bounded_wait_reports_timeout_and_context_survives(G):
    """A wait that nothing completes runs out (2 ms limit), the context reports
    GPT2_ERR_DEVICE_TIMEOUT once, and its next products are still right."""
    ctx = _ctx(G, G.GPT2_BF16)
    G.gpt2_selftest_wait_timeout(ctx, 2000)
    assert G.gpt2_sync_status(ctx) == G.GPT2_ERR_DEVICE_TIMEOUT
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    rng = np.random.default_rng(21)
    A = _rand(rng, (300, 768))
    W = _rand(rng, (512, 768), 0.05)
    bias = _rand(rng, (512,), 0.1)
    out = G.gpt2_linear(ctx, G.GPT2_EPI_BIAS, dev(A), dev(W), dev(bias))
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    assert_bf16_close(host(out), O.linear(A, W, bias), what="linear after a timeout")
