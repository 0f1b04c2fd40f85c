"""Parity at the full workload sizes, in the launch configuration the
benchmark times: the GPU runs the whole batch; the fp64 oracle recomputes
sampled sequences (every position of a sequence depends only on that
sequence, so a sequence is an exact sample)."""
import numpy as np
import pytest
import torch

from oracle import gpt2_oracle as O
from gpt_pre_norm_gb300 import synthetic as S
from tests.helpers import (ARGMAX_AGREE, argmax_agreement, assert_bf16_close, block_to_device,
                           check_top_choice, dev, host, model_to_device)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def G():
    from gpt_pre_norm_gb300 import build
    build.build()
    from gpt_pre_norm_gb300 import binding
    return binding


@pytest.mark.parametrize("name,samples", [("block_bf16_d768", (0, 7)), ("block_bf16_d1600", (0, 3))])
def test_block_full_size(G, name, samples):
    w = S.WORKLOADS[name]
    seed = 0
    p = S.block_params(w, seed)
    x = S.block_input(w, seed)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, 1, G.GPT2_BF16, w.B, w.T)
    present = G.KV(torch.zeros((w.B, 2, w.n_head, w.T, w.d_h), dtype=torch.bfloat16, device="cuda"))
    out = G.gpt2_block_forward(ctx, dev(x), block_to_device(p), w.B, w.T, w.d, w.n_head,
                               present=present)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    got = host(out)
    assert np.all(np.isfinite(got))
    got_present = present.data
    for b in samples:
        ref, ref_present = O.block_forward(x[b:b + 1], p, w.n_head)
        assert_bf16_close(got[b:b + 1], ref, what=f"{name} out, sequence {b}")
        assert_bf16_close(host(got_present[b:b + 1]), ref_present, what=f"{name} present, seq {b}")


def test_forward_full_size(G):
    """Full GPT-2-small forward, B=8, T=1024, V=50257: sequence 5 against the
    oracle at every one of its 1024 positions, plus the cache."""
    w = S.WORKLOADS["forward_bf16_gpt2_small"]
    seed = 0
    p = S.model_params(w, seed)
    ids = S.token_ids(w, seed)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, w.T)
    mp = G.ModelParams(model_to_device(p))
    present = G.KV(torch.zeros((w.B, w.n_layer, 2, w.n_head, w.T, w.d_h), dtype=torch.bfloat16,
                               device="cuda"))
    logits = G.gpt2_forward(ctx, dev(ids, torch.int32), mp, w.B, w.T, present=present)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    b = 5
    got = logits[b].float().cpu().numpy()
    assert np.all(np.isfinite(got))
    ref, ref_present = O.forward(ids[b:b + 1], p, w.n_head)
    assert_bf16_close(got, ref[0], what="full-size logits")
    assert argmax_agreement(got, ref[0]) >= ARGMAX_AGREE
    for layer in (0, w.n_layer - 1):
        assert_bf16_close(host(present.data[b:b + 1, layer]), ref_present[:, layer],
                          what=f"full-size present, layer {layer}")


def test_forward_loss_full_size(G):
    """The fused head + next-token loss at the benchmark's configuration (B=8,
    T=1024, V=50257, targets = the next token, none at the last position):
    every position against torch's cross-entropy on this library's own logits,
    sequence 2 against the oracle's loss, and the greedy choices against the
    logits' argmax."""
    import torch.nn.functional as F
    w = S.WORKLOADS["forward_loss_bf16_gpt2_small"]
    seed = 0
    p = S.model_params(w, seed)
    ids = S.token_ids(w, seed)
    targets = np.concatenate([ids[:, 1:], np.full((w.B, 1), -1, ids.dtype)], axis=1)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, w.T)
    mp = G.ModelParams(model_to_device(p))
    ids_d = dev(ids, torch.int32)
    loss, nxt = G.gpt2_forward_loss(ctx, ids_d, mp, w.B, w.T, targets=dev(targets, torch.int32))
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    loss, nxt = host(loss), nxt.cpu().numpy()
    assert np.all(np.isfinite(loss)) and np.all(loss[:, -1] == 0.0)
    for b in range(w.B):  # one sequence's logits at a time (1.65 GB for all of them)
        lg = G.gpt2_forward(ctx, ids_d, mp, w.B, w.T)[b].double()
        mine = F.cross_entropy(lg[:-1], torch.from_numpy(targets[b, :-1]).long().cuda(),
                               reduction="none").cpu().numpy()
        np.testing.assert_allclose(loss[b, :-1], mine, rtol=1e-5, atol=2e-4)
        np.testing.assert_array_equal(nxt[b], lg.argmax(-1).cpu().numpy())
        del lg
    b = 2
    ref_logits, _ = O.forward(ids[b:b + 1], p, w.n_head)
    ref_loss, _ = O.next_token_loss(ref_logits, targets[b:b + 1])
    np.testing.assert_allclose(loss[b], ref_loss[0], rtol=2e-3, atol=5e-3)


def test_forward_topk_full_size(G):
    """The fused head reduced to each position's top 8 at the benchmark's
    configuration (B=8, T=1024, V=50257): every position against this
    library's own logits (a valid top 8 in descending order, values at their
    ids, logsumexp as torch's), and sequence 3 against the oracle (the top
    choice wherever it is decided at this precision, the logsumexp)."""
    w = S.WORKLOADS["forward_topk_bf16_gpt2_small"]
    k = 8
    seed = 0
    p = S.model_params(w, seed)
    ids = S.token_ids(w, seed)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, w.T)
    mp = G.ModelParams(model_to_device(p))
    ids_d = dev(ids, torch.int32)
    vals, tid, lse = G.gpt2_forward_topk(ctx, ids_d, mp, w.B, w.T, k)
    logits = G.gpt2_forward(ctx, ids_d, mp, w.B, w.T)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    tol = 1e-4 * torch.clamp(logits.abs().amax(-1), min=1.0)           # [B, T]
    ti = tid.long()
    assert bool(((ti >= 0) & (ti < w.n_vocab)).all())
    assert bool((ti.sort(-1).values.diff(dim=-1) != 0).all())          # k distinct ids
    assert bool((logits.gather(-1, ti) - vals).abs().le(tol[..., None]).all())
    assert bool((vals[..., 1:] <= vals[..., :-1]).all())                 # descending
    kth = logits.topk(k, dim=-1).values[..., -1]
    assert bool((vals[..., -1] >= kth - tol).all())                      # nothing better left out
    torch.testing.assert_close(lse, torch.logsumexp(logits.double(), -1).float(), rtol=1e-5,
                               atol=1e-4)
    b = 3
    z = logits[b].cpu().numpy()
    del logits
    ref, _ = O.forward(ids[b:b + 1], p, w.n_head)
    rv, ri, rlse = O.top_k(ref[0], k)
    check_top_choice(z, ref[0], tid[b, :, 0].cpu().numpy(), rv, ri)
    np.testing.assert_allclose(host(lse[b]), rlse, rtol=2e-3, atol=2e-3)


def test_decode_full_size(G):
    """Cached single-token decode, GPT-2-medium shape, B=32, L=24, new token at
    position 1023 over a random past: sequences 0 and 31 against the oracle."""
    w = S.WORKLOADS["decode_bf16_gpt2_medium"]
    seed = 0
    p = S.model_params(w, seed)
    ids = S.token_ids(w, seed)
    shape = (w.B, w.n_layer, 2, w.n_head, w.n_ctx, w.d_h)
    host_cache = torch.zeros(shape, dtype=torch.int16)
    hv = host_cache.numpy()
    pasts = {}
    for bi in range(w.B):
        for layer in range(w.n_layer):
            pk = S.past_kv(w, seed, bi, layer)
            hv[bi, layer, :, :, :w.t_past] = S.bf16_bits(pk).view(np.int16)
            if bi in (0, w.B - 1):
                pasts.setdefault(bi, []).append(pk)
    cache = G.KV(host_cache.cuda().view(torch.bfloat16), w.t_past)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, w.T)
    mp = G.ModelParams(model_to_device(p))
    logits = G.gpt2_forward(ctx, dev(ids, torch.int32), mp, w.B, 1, past=cache, present=cache)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    assert cache.T_len == w.t_past + 1
    got_all = host(logits)
    assert np.all(np.isfinite(got_all))
    for bi in (0, w.B - 1):
        past = np.stack(pasts[bi])[None]  # [1, L, 2, h, T_past, d_h]
        ref, ref_present = O.forward(ids[bi:bi + 1], p, w.n_head, past=past)
        assert_bf16_close(got_all[bi], ref[0], what=f"decode logits, sequence {bi}")
        assert argmax_agreement(got_all[bi], ref[0]) == 1.0
        new_kv = host(cache.data[bi:bi + 1, :, :, :, w.t_past])
        assert_bf16_close(new_kv, ref_present[:, :, :, :, w.t_past], what=f"appended K/V, seq {bi}")
