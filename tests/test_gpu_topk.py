"""The tied head reduced to each position's top-k, on the GPU (gpt2_forward_topk).

The same context first writes the logits (gpt2_forward), then the top-k and
logsumexp without them: the k ids must be a top-k of those logits (within the
few fp32 ulps by which the two head layouts' sums may differ), in descending
order, with their values and the logsumexp matching the logits; k = 1 must
equal the greedy choice of gpt2_forward_loss bit for bit (the same head
layout); and the logsumexp must agree with the fp64 oracle, and the top choice
wherever the oracle's top two logits are further apart than the library's
logit error (elsewhere it must be within that error of the maximum).
Vocabularies with a ragged last 256-entry block, one block only, and the
GPT-2 size; a cached decode step; argument errors."""
import numpy as np
import pytest
import torch

from oracle import gpt2_oracle as O
from gpt_pre_norm_gb300 import synthetic as S
from tests.helpers import ARGMAX_AGREE, check_top_choice, dev, host, model_to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    from gpt_pre_norm_gb300 import build
    build.build()
    from gpt_pre_norm_gb300 import binding
    return binding


def _model(V, B=2, T=130, n_layer=1):
    return S.Workload("topk", "forward", "bf16", d=768, n_head=12, B=B, T=T, n_layer=n_layer,
                      n_vocab=V, resid_scale_layers=n_layer)


def _check_against_logits(z, vals, ids, lse, k):
    """ids: a valid top-k of the fp32 logits z (the two head layouts may differ
    by a few ulps, tol), descending; vals match z at ids; lse matches z."""
    V = z.shape[-1]
    zf = z.reshape(-1, V).astype(np.float64)
    vf, idf = vals.reshape(-1, k).astype(np.float64), ids.reshape(-1, k)
    tol = 1e-4 * np.maximum(1.0, np.abs(zf).max(axis=1))
    assert np.all((idf >= 0) & (idf < V))
    assert all(len(set(r)) == k for r in idf.tolist())
    assert np.all(np.abs(np.take_along_axis(zf, idf, 1) - vf) <= tol[:, None])
    assert np.all(vf[:, 1:] <= vf[:, :-1])  # descending
    kth = -np.sort(-zf, axis=1)[:, k - 1]   # the k-th largest logit of each row
    assert np.all(vf[:, -1] >= kth - tol)    # nothing better was left out
    m = zf.max(1)
    ref_lse = m + np.log(np.exp(zf - m[:, None]).sum(1))
    np.testing.assert_allclose(lse.reshape(-1), ref_lse, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("V,k", [(1000, 8), (1000, 1), (200, 5), (50257, 4), (1000, 2), (50257, 7)])
def test_topk_matches_the_logits_and_the_oracle(G, V, k):
    """V = 1000: a ragged last block (232 entries); V = 200: a single block;
    V = 50257: the GPT-2 vocabulary."""
    w = _model(V)
    p = S.model_params(w, seed=31)
    ids = S.token_ids(w, seed=31)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, w.T)
    mp = G.ModelParams(model_to_device(p))
    ids_d = dev(ids, torch.int32)
    z = host(G.gpt2_forward(ctx, ids_d, mp, w.B, w.T))
    vals, tid, lse = G.gpt2_forward_topk(ctx, ids_d, mp, w.B, w.T, k)
    _, nxt = G.gpt2_forward_loss(ctx, ids_d, mp, w.B, w.T, want_next=True)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    vals, tid, lse = host(vals), tid.cpu().numpy(), host(lse)
    assert vals.shape == (w.B, w.T, k) and tid.shape == (w.B, w.T, k)
    _check_against_logits(z, vals, tid, lse, k)
    np.testing.assert_array_equal(tid[..., 0], nxt.cpu().numpy())  # same head layout as the loss
    ref = O.forward(ids, p, w.n_head)[0]
    rv, ri, rlse = O.top_k(ref, max(k, 2))
    check_top_choice(z, ref, tid[..., 0], rv, ri)
    np.testing.assert_allclose(lse, rlse, rtol=2e-3, atol=2e-3)
    np.testing.assert_allclose(vals[..., 0], rv[..., 0], rtol=1e-2, atol=2e-2)


def test_topk_after_a_cached_prefix(G):
    """A one-token step after a 40-token prefix: the step's top-k against the
    uncached oracle at that position."""
    w = _model(1000, B=3, T=41)
    p = S.model_params(w, seed=32)
    ids = S.token_ids(w, seed=32)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, w.T)
    mp = G.ModelParams(model_to_device(p))
    ids_d = dev(ids, torch.int32)
    cache = G.KV(torch.zeros((w.B, w.n_layer, 2, w.n_head, 64, w.d_h), dtype=torch.bfloat16,
                             device="cuda"))
    G.gpt2_forward(ctx, ids_d[:, :40].contiguous(), mp, w.B, 40, present=cache)
    vals, tid, lse = G.gpt2_forward_topk(ctx, ids_d[:, 40:].contiguous(), mp, w.B, 1, 6,
                                         past=cache, present=cache)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    assert cache.T_len == 41
    ref = O.forward(ids, p, w.n_head, positions=[40])[0]
    rv, ri, rlse = O.top_k(ref, 6)
    assert np.mean(tid.cpu().numpy()[..., 0] == ri[..., 0]) >= ARGMAX_AGREE  # 3 positions: all
    np.testing.assert_allclose(host(lse), rlse, rtol=2e-3, atol=2e-3)


def test_topk_argument_errors(G):
    w = _model(300, B=1, T=4)
    p = S.model_params(w, seed=33)
    ids_d = dev(S.token_ids(w, seed=33), torch.int32)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, w.T)
    mp = G.ModelParams(model_to_device(p))
    for k in (0, 9):
        with pytest.raises(RuntimeError, match="invalid argument"):
            G.gpt2_forward_topk(ctx, ids_d, mp, w.B, w.T, k)
    small = _model(5, B=1, T=4)
    ps = S.model_params(small, seed=34)
    c2 = G.Context(5, small.n_ctx, small.d, small.n_head, 1, G.GPT2_BF16, 1, 4)
    with pytest.raises(RuntimeError, match="invalid argument"):
        G.gpt2_forward_topk(c2, dev(np.zeros((1, 4), np.int32), torch.int32),
                            G.ModelParams(model_to_device(ps)), 1, 4, 6)  # k > V
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK


@pytest.mark.parametrize("k", [8, 3])
def test_topk_ties_take_the_lower_ids(G, k):
    """Embedding rows repeating with period 97: each logit value of a row is
    shared by 10 or 11 vocabulary entries spread over every 256-entry block
    (V = 1000, ragged last block), so a position's top k is a run of equal
    values: its ids must be the lowest ids of the largest values, the rule of
    the oracle's top_k applied to the library's own logits."""
    w = _model(1000, B=2, T=40)
    p = S.model_params(w, seed=35)
    p["wte"] = np.ascontiguousarray(p["wte"][np.arange(w.n_vocab) % 97])
    ids = S.token_ids(w, seed=35)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, w.T)
    mp = G.ModelParams(model_to_device(p))
    ids_d = dev(ids, torch.int32)
    z = host(G.gpt2_forward(ctx, ids_d, mp, w.B, w.T))
    vals, tid, lse = G.gpt2_forward_topk(ctx, ids_d, mp, w.B, w.T, k)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    tid = tid.cpu().numpy()
    _, ref_ids, _ = O.top_k(z, k)
    np.testing.assert_array_equal(tid, ref_ids)
    assert np.all(tid[..., 1:] % 97 == tid[..., :1] % 97)  # one run of equal values
