"""Calls on cached fp16 weight copies, on the GPU.

With the context's weight cache on, the first call converts the bf16 weights
to fp16 working copies and later calls reuse them.  A call whose copies were
all made by an earlier call starts the few-row products' weight streams before
their wait on the previous kernel (its first launch is a plain one, so the
copies are complete).  These tests run cached decode steps and cached block
calls against the fp64 oracle and against the same calls with the cache off,
with 32 rows at K = 1024, fewer rows, and K below 1024."""
import numpy as np
import pytest
import torch

from oracle import gpt2_oracle as O
from gpt_pre_norm_gb300 import synthetic as S
from tests.helpers import (ARGMAX_AGREE, argmax_agreement, assert_bf16_close, block_to_device,
                           dev, host, model_to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    from gpt_pre_norm_gb300 import build
    build.build()
    from gpt_pre_norm_gb300 import binding
    return binding


def _kv(G, B, h, t_cap, dh, L=None):
    shape = (B, 2, h, t_cap, dh) if L is None else (B, L, 2, h, t_cap, dh)
    return G.KV(torch.zeros(shape, dtype=torch.bfloat16, device="cuda"))


def _model(B, d, h, V=1000, n_layer=2):
    return S.Workload("cached", "forward", "bf16", d=d, n_head=h, B=B, T=24, n_layer=n_layer,
                      n_vocab=V, resid_scale_layers=n_layer)


def _decode(G, w, p, ids, t0, cache_weights):
    """Prefill t0 tokens, then one-token steps to the end of ids; returns the
    step logits [B, steps, V]."""
    B, T = ids.shape
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, B, T)
    G.gpt2_ctx_cache_weights(ctx, cache_weights)
    mp = G.ModelParams(model_to_device(p))
    ids_d = dev(ids, torch.int32)
    cache = _kv(G, B, w.n_head, 64, w.d_h, L=w.n_layer)
    G.gpt2_forward(ctx, ids_d[:, :t0].contiguous(), mp, B, t0, present=cache)
    steps = [host(G.gpt2_forward(ctx, ids_d[:, t:t + 1].contiguous(), mp, B, 1, past=cache,
                                 present=cache)) for t in range(t0, T)]
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    return np.concatenate(steps, axis=1)


@pytest.mark.parametrize("B,d,h", [(32, 1024, 16), (2, 768, 12), (5, 256, 4)])
def test_cached_decode_matches_oracle(G, B, d, h):
    w = _model(B, d, h)
    p = S.model_params(w, seed=21)
    ids = S.token_ids(w, seed=21, T=23)
    got = _decode(G, w, p, ids, 20, cache_weights=True)
    ref, _ = O.forward(ids, p, w.n_head, positions=[20, 21, 22])
    assert_bf16_close(got, ref, what="cached decode vs oracle")
    assert argmax_agreement(got, ref) >= ARGMAX_AGREE


def test_cached_equals_uncached_decode(G):
    """The same arithmetic runs with and without the cache.  Not bit for bit:
    the K chunks of the 4096-wide mlp c_proj add into the fp32 residual with
    atomics, in any order, and an fp16 activation that then rounds the other
    way moves by 2^-11 of itself; measured run to run about 1e-4 of the logits
    (relative L2).  The bound, 1e-3, is ten times below the oracle's."""
    w = _model(8, 1024, 16)
    p = S.model_params(w, seed=22)
    ids = S.token_ids(w, seed=22, T=22)
    cached = _decode(G, w, p, ids, 20, cache_weights=True)
    plain = _decode(G, w, p, ids, 20, cache_weights=False)
    assert_bf16_close(cached, plain, tol=1e-3, what="cached vs uncached decode")


def test_cached_block_decode(G):
    """The standalone block, one new token per sequence after a 40-token
    prefix, weight cache on (the block input is bf16)."""
    w = S.WORKLOADS["block_bf16_d768"]
    B, T0 = 6, 40
    p = S.block_params(w, seed=23)
    x = S.block_input(w, seed=23, B=B, T=T0 + 2)
    pd = block_to_device(p)
    ctx = G.Context(50257, 1024, w.d, w.n_head, 1, G.GPT2_BF16, B, T0)
    G.gpt2_ctx_cache_weights(ctx, True)
    cache = _kv(G, B, w.n_head, 64, w.d_h)
    G.gpt2_block_forward(ctx, dev(x[:, :T0]), pd, B, T0, w.d, w.n_head, present=cache)
    outs = [host(G.gpt2_block_forward(ctx, dev(x[:, t:t + 1]), pd, B, 1, w.d, w.n_head,
                                      past=cache, present=cache)) for t in (T0, T0 + 1)]
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    ref, ref_present = O.block_forward(x, p, w.n_head)
    assert_bf16_close(np.concatenate(outs, axis=1), ref[:, T0:], what="cached block decode")
    assert_bf16_close(host(cache.data)[..., :T0 + 2, :], ref_present, what="present")
