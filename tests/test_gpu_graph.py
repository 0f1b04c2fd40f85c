"""Steps replayed from CUDA graphs against the same calls made one by one.

The benchmark times the block and full-forward steps both ways.  A captured
call launches the same kernels with the same arguments, and the prefill path
has no atomic accumulation, so a replay must reproduce the eager result bit
for bit, also when replayed more than once."""
import numpy as np
import pytest
import torch

from gpt_pre_norm_gb300 import synthetic as S
from tests.helpers import block_to_device, dev, model_to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    from gpt_pre_norm_gb300 import build
    build.build()
    from gpt_pre_norm_gb300 import binding
    return binding


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()


def _replay(fn):
    """fn() once eagerly, then captured into a graph and replayed twice:
    (eager outputs, replayed outputs)."""
    eager = [t.clone() for t in fn()]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = fn()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    return eager, outs


def test_block_step_replay_is_bit_identical(G):
    w = S.WORKLOADS["block_bf16_d768"]
    p = block_to_device(S.block_params(w, seed=5))
    x = dev(S.block_input(w, seed=5, B=2, T=256))
    ctx = G.Context(50257, 1024, w.d, w.n_head, 1, G.GPT2_BF16, 8, 1024)
    out = torch.empty_like(x)

    def step():
        G.gpt2_block_forward(ctx, x, p, 2, 256, w.d, w.n_head, out=out)
        return [out]

    eager, replayed = _replay(step)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    np.testing.assert_array_equal(_bits(replayed[0]), _bits(eager[0]))


def test_forward_topk_replay_is_bit_identical(G):
    w = S.Workload("graph", "forward", "bf16", d=768, n_head=12, B=2, T=96, n_layer=2,
                   n_vocab=1000, resid_scale_layers=2)
    mp = G.ModelParams(model_to_device(S.model_params(w, seed=6)))
    ids = dev(S.token_ids(w, seed=6), torch.int32)
    ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, G.GPT2_BF16, w.B, w.T)
    vals = torch.empty((w.B, w.T, 5), dtype=torch.float32, device="cuda")
    tid = torch.empty((w.B, w.T, 5), dtype=torch.int32, device="cuda")

    def step():
        v, i, lse = G.gpt2_forward_topk(ctx, ids, mp, w.B, w.T, 5, top_logits=vals, top_ids=tid)
        return [v, i, lse]

    eager, replayed = _replay(step)
    assert G.gpt2_sync_status(ctx) == G.GPT2_OK
    for a, b in zip(replayed, eager):
        np.testing.assert_array_equal(_bits(a), _bits(b))
