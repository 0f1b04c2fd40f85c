"""Block, full forward and cached decode through the C ABI vs the fp64 oracle
(small, fast cases: several tiles and ragged tails; error paths)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import gpt2_oracle as O
from gpt_pre_norm_gb300 import synthetic as S
from tests.helpers import (ARGMAX_AGREE, argmax_agreement, assert_bf16_close, assert_fp32_close,
                           block_to_device, dev, host, model_to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    from gpt_pre_norm_gb300 import build
    build.build()
    from gpt_pre_norm_gb300 import binding
    return binding


def _kv(G, B, h, t_cap, dh, dtype, L=None):
    shape = (B, 2, h, t_cap, dh) if L is None else (B, L, 2, h, t_cap, dh)
    return G.KV(torch.zeros(shape, dtype=dtype, device="cuda"))


# ------------------------------------------------------------------ block ----
def test_block_fp32_debug_shape(G):
    """The TorchCode debug block: d=64, 4 heads, x [2, 8, 64], fp32."""
    w = S.WORKLOADS["block_fp32_d64"]
    for seed in (0, 1, 2):
        p = S.block_params(w, seed)
        x = S.block_input(w, seed)
        ctx = G.Context(50257, 1024, w.d, w.n_head, 1, G.GPT2_FP32, w.B, w.T)
        present = _kv(G, w.B, w.n_head, 16, w.d_h, torch.float32)
        out = G.gpt2_block_forward(ctx, dev(x, torch.float32), block_to_device(p, torch.float32),
                                   w.B, w.T, w.d, w.n_head, present=present)
        assert G.gpt2_sync_status(ctx) == 0
        assert tuple(out.shape) == (2, 8, 64)
        ref, ref_present = O.block_forward(x, p, w.n_head)
        assert_fp32_close(host(out), ref, what="fp32 block")
        assert present.T_len == w.T
        assert_fp32_close(host(present.data)[:, :, :, :w.T], ref_present, what="fp32 present")


@pytest.mark.parametrize("name,B,T", [("block_bf16_d768", 2, 300), ("block_bf16_d1600", 1, 130),
                                      ("block_bf16_d768", 3, 1), ("block_bf16_d768", 2, 160),
                                      ("block_bf16_d768", 1, 256), ("block_bf16_d1600", 2, 96),
                                      ("block_bf16_d768", 2, 32)])
def test_block_bf16(G, name, B, T):
    w = S.WORKLOADS[name]
    p = S.block_params(w, seed=1)
    x = S.block_input(w, seed=1, B=B, T=T)
    ctx = G.Context(50257, 1024, w.d, w.n_head, 1, G.GPT2_BF16, B, T)
    present = _kv(G, B, w.n_head, T + 5, w.d_h, torch.bfloat16)
    out = G.gpt2_block_forward(ctx, dev(x), block_to_device(p), B, T, w.d, w.n_head,
                               present=present)
    assert G.gpt2_sync_status(ctx) == 0
    ref, ref_present = O.block_forward(x, p, w.n_head)
    assert_bf16_close(host(out), ref, what="block out")
    # The residual branches alone (out - x): loose, the bf16 rounding of out is
    # relative to x; a missing or wrong branch would be off by tens of percent.
    assert_bf16_close(host(out) - x, ref - x, tol=5e-2, what="block branch")
    got_present = host(present.data)[:, :, :, :T]
    assert_bf16_close(got_present[:, 0], ref_present[:, 0], what="present K")
    assert_bf16_close(got_present[:, 1], ref_present[:, 1], what="present V")


def test_block_four_linear_form_by_concatenation(G):
    """A block given as four separate attention Linear maps (W_q, W_k, W_v,
    W_o) runs through the same entry point once W_q | W_k | W_v are stacked by
    rows into c_attn (the oracle pins that identity against the separate
    form)."""
    w = S.WORKLOADS["block_bf16_d768"]
    B, T, d = 2, 200, w.d
    p = S.block_params(w, seed=6)
    rng = np.random.default_rng(6)
    sep = {k: (0.02 * rng.standard_normal((d, d))).astype(np.float32) for k in ("q", "k", "v")}
    sep_b = {k: (0.02 * rng.standard_normal(d)).astype(np.float32) for k in ("q", "k", "v")}
    # bf16-representable values, as the device receives them
    rt = lambda a: torch.from_numpy(np.asarray(a, np.float32)).bfloat16().double().numpy()
    p["attn_w"] = rt(np.concatenate([sep["q"], sep["k"], sep["v"]], 0))
    p["attn_b"] = rt(np.concatenate([sep_b["q"], sep_b["k"], sep_b["v"]]))
    x = S.block_input(w, seed=6, B=B, T=T)
    ctx = G.Context(50257, 1024, d, w.n_head, 1, G.GPT2_BF16, B, T)
    out = G.gpt2_block_forward(ctx, dev(x), block_to_device(p), B, T, d, w.n_head)
    assert G.gpt2_sync_status(ctx) == 0
    ref, _ = O.block_forward(x, p, w.n_head)
    assert_bf16_close(host(out), ref, what="four-Linear block")
    assert_bf16_close(host(out) - x, ref - x, tol=5e-2, what="four-Linear block branch")


def test_block_postnorm_fp32_debug_shape(G):
    """The post-norm arrangement (LayerNorm after each residual add) on the
    TorchCode debug shapes, fp32, against the oracle's post-norm block."""
    w = S.WORKLOADS["block_fp32_d64"]
    for seed in (0, 1):
        p = S.block_params(w, seed)
        x = S.block_input(w, seed)
        ctx = G.Context(50257, 1024, w.d, w.n_head, 1, G.GPT2_FP32, w.B, w.T)
        out = G.gpt2_block_forward_postnorm(ctx, dev(x, torch.float32),
                                            block_to_device(p, torch.float32), w.B, w.T, w.d,
                                            w.n_head)
        assert G.gpt2_sync_status(ctx) == 0
        ref = O.block_forward_postnorm(x, p, w.n_head)
        assert_fp32_close(host(out), ref, what="fp32 post-norm block")


@pytest.mark.parametrize("name,B,T", [("block_bf16_d768", 2, 300), ("block_bf16_d1600", 1, 130),
                                      ("block_bf16_d768", 3, 1), ("block_bf16_d768", 2, 1024)])
def test_block_postnorm_bf16(G, name, B, T):
    w = S.WORKLOADS[name]
    p = S.block_params(w, seed=4)
    x = S.block_input(w, seed=4, B=B, T=T)
    ctx = G.Context(50257, 1024, w.d, w.n_head, 1, G.GPT2_BF16, B, T)
    out = G.gpt2_block_forward_postnorm(ctx, dev(x), block_to_device(p), B, T, w.d, w.n_head)
    assert G.gpt2_sync_status(ctx) == 0
    ref = O.block_forward_postnorm(x, p, w.n_head)
    assert_bf16_close(host(out), ref, what="post-norm block out")
    # The pre-norm block differs from it by O(1): the two are not confused.
    pre, _ = O.block_forward(x, p, w.n_head)
    assert np.abs(host(out) - pre).max() > 0.5


@pytest.mark.parametrize("mode", ["in_place", "copy", "no_present"])
def test_block_with_cache_equals_uncached(G, mode):
    w = S.WORKLOADS["block_bf16_d768"]
    B, T0, T1 = 2, 100, 70
    p = S.block_params(w, seed=2)
    x = S.block_input(w, seed=2, B=B, T=T0 + T1)
    pd = block_to_device(p)
    ctx = G.Context(50257, 1024, w.d, w.n_head, 1, G.GPT2_BF16, B, T0 + T1)
    cache = _kv(G, B, w.n_head, 256, w.d_h, torch.bfloat16)
    G.gpt2_block_forward(ctx, dev(x[:, :T0]), pd, B, T0, w.d, w.n_head, present=cache)
    if mode == "in_place":
        present = cache
    elif mode == "copy":
        present = _kv(G, B, w.n_head, 200, w.d_h, torch.bfloat16)
    else:
        present = None
    out = G.gpt2_block_forward(ctx, dev(x[:, T0:]), pd, B, T1, w.d, w.n_head, past=cache,
                               present=present)
    assert G.gpt2_sync_status(ctx) == 0
    ref, ref_present = O.block_forward(x, p, w.n_head)
    assert_bf16_close(host(out), ref[:, T0:], what="cached block out")
    if present is not None:
        assert present.T_len == T0 + T1
        got = host(present.data)[:, :, :, :T0 + T1]
        assert_bf16_close(got, ref_present, what="present after append")


# ----------------------------------------------------------- full forward ----
def _small_model(n_layer=2, d=768, h=12, V=50257):
    return S.Workload("small", "forward", "bf16", d=d, n_head=h, B=2, T=130, n_layer=n_layer,
                      n_vocab=V, resid_scale_layers=n_layer)


def test_forward_bf16_small(G):
    w = _small_model()
    p = S.model_params(w, seed=3)
    ids = S.token_ids(w, seed=3)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, w.T)
    mp = G.ModelParams(model_to_device(p))
    present = _kv(G, w.B, w.n_head, w.n_ctx, w.d_h, torch.bfloat16, L=w.n_layer)
    logits = G.gpt2_forward(ctx, dev(ids, torch.int32), mp, w.B, w.T, present=present)
    assert G.gpt2_sync_status(ctx) == 0
    ref, ref_present = O.forward(ids, p, w.n_head)
    got = host(logits)
    assert got.shape == (w.B, w.T, w.n_vocab)
    assert_bf16_close(got, ref, what="logits")
    assert argmax_agreement(got, ref) >= ARGMAX_AGREE
    assert_bf16_close(host(present.data)[..., :w.T, :], ref_present, what="present")


def test_forward_bf16_tensor_core_attention(G):
    """T a multiple of 32 with no cached prefix: attention on tcgen05."""
    w = S.Workload("small_tc", "forward", "bf16", d=768, n_head=12, B=2, T=192, n_layer=2,
                   resid_scale_layers=2)
    p = S.model_params(w, seed=6)
    ids = S.token_ids(w, seed=6)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, w.T)
    mp = G.ModelParams(model_to_device(p))
    logits = G.gpt2_forward(ctx, dev(ids, torch.int32), mp, w.B, w.T)
    assert G.gpt2_sync_status(ctx) == 0
    ref, _ = O.forward(ids, p, w.n_head)
    got = host(logits)
    assert_bf16_close(got, ref, what="logits")
    assert argmax_agreement(got, ref) >= ARGMAX_AGREE


def test_forward_fp32_tiny(G):
    w = S.Workload("tiny32", "forward", "fp32", d=64, n_head=4, B=2, T=9, n_layer=2, n_vocab=300,
                   n_ctx=32, w_std=0.1)
    p = S.model_params(w, seed=4)
    ids = S.token_ids(w, seed=4)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_FP32, w.B, w.T)
    mp = G.ModelParams(model_to_device(p, torch.float32))
    logits = G.gpt2_forward(ctx, dev(ids, torch.int32), mp, w.B, w.T)
    assert G.gpt2_sync_status(ctx) == 0
    ref, _ = O.forward(ids, p, w.n_head)
    assert_fp32_close(host(logits), ref, what="fp32 logits")


def test_decode_equals_uncached(G):
    """Prefill 40 tokens with a cache, then 3 one-token steps: the step logits
    match the uncached pass (GPU and oracle) at those positions."""
    w = _small_model(n_layer=3)
    p = S.model_params(w, seed=5)
    ids = S.token_ids(w, seed=5, T=43)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, 43)
    mp = G.ModelParams(model_to_device(p))
    ids_d = dev(ids, torch.int32)
    cache = _kv(G, w.B, w.n_head, 64, w.d_h, torch.bfloat16, L=w.n_layer)
    G.gpt2_forward(ctx, ids_d[:, :40].contiguous(), mp, w.B, 40, present=cache)
    steps = []
    for t in range(40, 43):
        steps.append(host(G.gpt2_forward(ctx, ids_d[:, t:t + 1].contiguous(), mp, w.B, 1,
                                         past=cache, present=cache)))
    full = host(G.gpt2_forward(ctx, ids_d, mp, w.B, 43))
    assert G.gpt2_sync_status(ctx) == 0
    assert cache.T_len == 43
    got = np.concatenate(steps, axis=1)
    ref, _ = O.forward(ids, p, w.n_head, positions=[40, 41, 42])
    assert_bf16_close(got, ref, what="decode vs oracle")
    assert_bf16_close(got, full[:, 40:], what="decode vs gpu uncached")
    assert argmax_agreement(got, ref) >= ARGMAX_AGREE


def test_forward_chunked_prefill(G):
    """Prefill 64 tokens into a cache, then a 66-token chunk after them (T > 1
    with T_past > 0): the chunk's logits match the oracle's uncached pass at
    positions 64..129, and the cache holds all 130 positions."""
    w = _small_model(n_layer=2)
    p = S.model_params(w, seed=8)
    ids = S.token_ids(w, seed=8, T=130)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, 130)
    mp = G.ModelParams(model_to_device(p))
    ids_d = dev(ids, torch.int32)
    cache = _kv(G, w.B, w.n_head, 160, w.d_h, torch.bfloat16, L=w.n_layer)
    G.gpt2_forward(ctx, ids_d[:, :64].contiguous(), mp, w.B, 64, present=cache)
    got = host(G.gpt2_forward(ctx, ids_d[:, 64:].contiguous(), mp, w.B, 66, past=cache,
                              present=cache))
    assert G.gpt2_sync_status(ctx) == 0
    assert cache.T_len == 130
    ref, ref_present = O.forward(ids, p, w.n_head)
    assert_bf16_close(got, ref[:, 64:], what="chunked prefill logits")
    assert argmax_agreement(got, ref[:, 64:]) >= ARGMAX_AGREE
    assert_bf16_close(host(cache.data)[..., :130, :], ref_present, what="cache after the chunk")


def test_generate_greedy(G):
    """Greedy generation on the GPU, checked step by step against the oracle
    fed the GPU's own choices: every chosen token is a maximum of the oracle's
    logits within the bf16 path's error, and nearly all are the exact argmax."""
    w = _small_model(n_layer=2, V=1000)
    p = S.model_params(w, seed=9)
    ids = S.token_ids(w, seed=9, T=24)
    n_new = 8
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, 24)
    mp = G.ModelParams(model_to_device(p))
    cache = _kv(G, w.B, w.n_head, 64, w.d_h, torch.bfloat16, L=w.n_layer)
    out = G.gpt2_generate_greedy(ctx, dev(ids, torch.int32), mp, n_new, cache).cpu().numpy()
    assert G.gpt2_sync_status(ctx) == 0
    assert cache.T_len == 24 + n_new - 1
    assert out.shape == (w.B, n_new) and out.min() >= 0 and out.max() < w.n_vocab
    seq = ids.copy()
    exact = 0
    for i in range(n_new):
        ref, _ = O.forward(seq, p, w.n_head, positions=[seq.shape[1] - 1])
        ref = ref[:, -1]
        for b in range(w.B):
            row = ref[b]
            tol = 5e-3 * np.sqrt(np.mean(row ** 2))
            assert row[out[b, i]] >= row.max() - tol, f"step {i}, sequence {b}"
            exact += int(out[b, i] == np.argmax(row))
        seq = np.concatenate([seq, out[:, i:i + 1]], axis=1)
    assert exact >= 0.9 * w.B * n_new


def test_generate_greedy_graph_captured(G):
    """The generation loop makes no host round trip (each argmax feeds the
    next step on the device), so it captures into one CUDA graph; replaying
    the graph gives the eager run's tokens and (to rounding) its cache."""
    w = _small_model(n_layer=2, V=1000)
    p = S.model_params(w, seed=10)
    ids = dev(S.token_ids(w, seed=10, T=20), torch.int32)
    n_new = 6
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, 20)
    mp = G.ModelParams(model_to_device(p))
    eager_cache = _kv(G, w.B, w.n_head, 64, w.d_h, torch.bfloat16, L=w.n_layer)
    eager = G.gpt2_generate_greedy(ctx, ids, mp, n_new, eager_cache).cpu().numpy()
    assert G.gpt2_sync_status(ctx) == 0
    cache = _kv(G, w.B, w.n_head, 64, w.d_h, torch.bfloat16, L=w.n_layer)
    logits = torch.empty((w.B, 20, w.n_vocab), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = G.gpt2_generate_greedy(ctx, ids, mp, n_new, cache, logits=logits)
    g.replay()
    torch.cuda.synchronize()
    assert G.gpt2_sync_status(ctx) == 0
    np.testing.assert_array_equal(out.cpu().numpy(), eager)
    # The decode steps' fp32 residual adds of the K-chunked products are
    # atomic (their order varies run to run), so the cache agrees to rounding.
    T_all = 20 + n_new - 1
    assert_bf16_close(cache.data[..., :T_all, :].float().cpu().numpy(),
                      eager_cache.data[..., :T_all, :].float().cpu().numpy(), what="graph cache")


@pytest.mark.parametrize("V,L,B,T", [(1000, 2, 2, 130), (50257, 1, 2, 64), (777, 1, 3, 1)])
def test_forward_loss_without_logits(G, V, L, B, T):
    """The fused head + next-token loss: against torch's cross-entropy on this
    library's own logits (same products, so tight) and against the oracle
    (bf16 tolerance); the greedy choices equal the logits' argmax.  V = 50257
    leaves a ragged last block of 81 entries, V = 777 a small one."""
    w = _small_model(n_layer=L, V=V)
    p = S.model_params(w, seed=11)
    rng = np.random.default_rng(11)
    ids = rng.integers(0, V, size=(B, T)).astype(np.int32)
    targets = rng.integers(0, V, size=(B, T)).astype(np.int32)
    targets[0, 0] = -1  # no loss at this position
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, B, T)
    mp = G.ModelParams(model_to_device(p))
    ids_d = dev(ids, torch.int32)
    loss, nxt = G.gpt2_forward_loss(ctx, ids_d, mp, B, T, targets=dev(targets, torch.int32))
    logits = G.gpt2_forward(ctx, ids_d, mp, B, T)
    assert G.gpt2_sync_status(ctx) == 0
    loss, nxt, logits = host(loss), nxt.cpu().numpy(), host(logits)
    assert loss[0, 0] == 0.0
    mine = F.cross_entropy(torch.from_numpy(logits.reshape(-1, V)).double(),
                           torch.from_numpy(np.maximum(targets, 0).reshape(-1)).long(),
                           reduction="none").numpy().reshape(B, T)
    mine[0, 0] = 0.0
    np.testing.assert_allclose(loss, mine, rtol=1e-5, atol=1e-4)
    np.testing.assert_array_equal(nxt, logits.argmax(-1))
    ref_logits, _ = O.forward(ids, p, w.n_head)
    ref_loss, _ = O.next_token_loss(ref_logits, targets)
    np.testing.assert_allclose(loss, ref_loss, rtol=2e-3, atol=5e-3)


def test_forward_loss_bad_target_reported(G):
    """A target outside the vocabulary yields a NaN loss at its position and
    INVALID_ARG from the device error word; other positions are unaffected."""
    w = _small_model(n_layer=1, V=500)
    p = S.model_params(w, seed=13)
    B, T = 2, 40
    rng = np.random.default_rng(13)
    ids = rng.integers(0, 500, size=(B, T)).astype(np.int32)
    targets = rng.integers(0, 500, size=(B, T)).astype(np.int32)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, B, T)
    mp = G.ModelParams(model_to_device(p))
    good, _ = G.gpt2_forward_loss(ctx, dev(ids, torch.int32), mp, B, T,
                                  targets=dev(targets, torch.int32))
    assert G.gpt2_sync_status(ctx) == 0
    bad_t = targets.copy()
    bad_t[1, 7] = 500
    bad, _ = G.gpt2_forward_loss(ctx, dev(ids, torch.int32), mp, B, T,
                                 targets=dev(bad_t, torch.int32))
    assert G.gpt2_sync_status(ctx) == G.GPT2_ERR_INVALID_ARG
    bad, good = host(bad), host(good)
    assert np.isnan(bad[1, 7])
    mask = np.ones_like(bad, dtype=bool)
    mask[1, 7] = False
    np.testing.assert_array_equal(bad[mask], good[mask])


def test_forward_loss_cached_positions(G):
    """With a cache, the loss covers the new positions only and equals the
    uncached pass's loss there; present is filled as by gpt2_forward."""
    w = _small_model(n_layer=2, V=1000)
    p = S.model_params(w, seed=12)
    B, T0, T1 = 2, 50, 30
    rng = np.random.default_rng(12)
    ids = rng.integers(0, 1000, size=(B, T0 + T1)).astype(np.int32)
    targets = rng.integers(0, 1000, size=(B, T0 + T1)).astype(np.int32)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, B, T0 + T1)
    mp = G.ModelParams(model_to_device(p))
    full, _ = G.gpt2_forward_loss(ctx, dev(ids, torch.int32), mp, B, T0 + T1,
                                  targets=dev(targets, torch.int32))
    cache = _kv(G, B, w.n_head, 128, w.d_h, torch.bfloat16, L=w.n_layer)
    G.gpt2_forward_loss(ctx, dev(ids[:, :T0], torch.int32), mp, B, T0,
                        targets=dev(targets[:, :T0], torch.int32), present=cache)
    part, nxt = G.gpt2_forward_loss(ctx, dev(ids[:, T0:], torch.int32), mp, B, T1,
                                    targets=dev(targets[:, T0:], torch.int32), past=cache,
                                    present=cache)
    assert G.gpt2_sync_status(ctx) == 0
    assert cache.T_len == T0 + T1
    np.testing.assert_allclose(host(part), host(full)[:, T0:], rtol=1e-3, atol=5e-3)


# ----------------------------------------------------------- error paths ----
def test_errors_are_reported_before_launch(G):
    w = S.WORKLOADS["block_bf16_d768"]
    p = block_to_device(S.block_params(w, seed=0))
    ctx = G.Context(50257, 1024, w.d, w.n_head, 1, G.GPT2_BF16, 2, 64)
    x = dev(S.block_input(w, 0, B=2, T=64))
    with pytest.raises(G.Gpt2Error) as e:  # B*T beyond the context's sizing
        G.gpt2_block_forward(ctx, dev(S.block_input(w, 0, B=3, T=64)), p, 3, 64, w.d, w.n_head)
    assert e.value.status == G.GPT2_ERR_WORKSPACE
    past = _kv(G, 2, w.n_head, 1024, w.d_h, torch.bfloat16)
    past.T_len = 1000
    with pytest.raises(G.Gpt2Error) as e:  # 1000 + 64 > n_ctx
        G.gpt2_block_forward(ctx, x, p, 2, 64, w.d, w.n_head, past=past, present=past)
    assert e.value.status == G.GPT2_ERR_CTX_OVERFLOW
    small = _kv(G, 2, w.n_head, 32, w.d_h, torch.bfloat16)
    with pytest.raises(G.Gpt2Error) as e:  # present too small
        G.gpt2_block_forward(ctx, x, p, 2, 64, w.d, w.n_head, present=small)
    assert e.value.status == G.GPT2_ERR_CTX_OVERFLOW
    with pytest.raises(G.Gpt2Error) as e:
        G.gpt2_block_forward(ctx, x, p, 2, 64, w.d, 16)  # n_head differs from the context
    assert e.value.status == G.GPT2_ERR_INVALID_ARG
    for B0, T0 in ((0, 64), (2, 0)):  # empty batch or sequence: rejected, nothing launched
        with pytest.raises(G.Gpt2Error) as e:
            G.gpt2_block_forward(ctx, x, p, B0, T0, w.d, w.n_head)
        assert e.value.status == G.GPT2_ERR_INVALID_ARG
    xm = torch.empty(2 * 64 * w.d + 1, dtype=torch.bfloat16, device="cuda")[1:].view(2, 64, w.d)
    with pytest.raises(G.Gpt2Error) as e:
        G.gpt2_block_forward(ctx, xm, p, 2, 64, w.d, w.n_head)
    assert e.value.status == G.GPT2_ERR_ALIGNMENT
    assert G.gpt2_sync_status(ctx) == 0
