"""The C-ABI library: it builds, loads without a GPU, exports every function
include/gpt2.h declares, and rejects bad arguments before touching a device."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gpt2.h")


@pytest.fixture(scope="module")
def G():
    from gpt_pre_norm_gb300 import build
    build.build()
    from gpt_pre_norm_gb300 import binding
    return binding


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|void|const char\s*\*)\s*\**\s*(gpt2_\w+)\s*\(",
                                 src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("gpt2_block_forward", "gpt2_forward", "gpt2_ctx_create", "gpt2_ctx_destroy",
                 "gpt2_sync_status", "gpt2_status_string", "gpt2_workspace_bytes"):
        assert must in names


def test_library_exports_every_declared_symbol(G):
    lib = C.CDLL(G._build.LIB)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(G):
    for s in range(0, 10):
        assert G.status_string(s) and G.status_string(s) != "unknown status"
    assert G.status_string(99) == "unknown status"


def _hp(G, **kw):
    base = dict(n_vocab=50257, n_ctx=1024, n_embd=768, n_head=12, n_layer=12, dtype=G.GPT2_BF16)
    base.update(kw)
    return G.gpt2_hparams(**base)


def test_workspace_sizing_is_host_only_and_monotonic(G):
    sizes = []
    for B, T in ((1, 1), (1, 1024), (8, 1024)):
        n = C.c_size_t()
        assert G.LIB.gpt2_workspace_bytes(C.byref(_hp(G)), B, T, C.byref(n)) == G.GPT2_OK
        sizes.append(n.value)
    assert sizes[0] < sizes[1] < sizes[2]
    n = C.c_size_t()
    # 8 x 1024 tokens of d=768: at least the c_fc activation (8192 x 3072 bf16).
    assert G.LIB.gpt2_workspace_bytes(C.byref(_hp(G)), 8, 1024, C.byref(n)) == 0
    assert n.value >= 8192 * 3072 * 2


@pytest.mark.parametrize("kw,status", [
    (dict(n_embd=768, n_head=16), 2),       # bf16 needs d_h = 64
    (dict(n_embd=100, n_head=3), 2),        # d % n_head != 0
    (dict(dtype=7), 1),                     # bad dtype
    (dict(n_layer=0), 1),
    (dict(n_embd=64, n_head=4, dtype=1), 0),  # fp32 accepts d_h = 16
])
def test_hparams_validation(G, kw, status):
    n = C.c_size_t()
    assert G.LIB.gpt2_workspace_bytes(C.byref(_hp(G, **kw)), 2, 8, C.byref(n)) == status


def test_null_arguments_rejected_without_launch(G):
    assert G.LIB.gpt2_block_forward(None, None, None, 1, 1, 768, 12, None, None, None, None) == 1
    assert G.LIB.gpt2_forward(None, None, 1, 1, None, 12, None, None, None, None) == 1
    assert G.LIB.gpt2_block_forward_postnorm(None, None, None, 1, 1, 768, 12, None, None) == 1
    assert G.LIB.gpt2_forward_loss(None, None, None, 1, 1, None, 12, None, None, None, None,
                                   None) == 1
    assert G.LIB.gpt2_forward_topk(None, None, 1, 1, None, 12, None, None, 4, None, None, None,
                                   None) == 1
    assert G.LIB.gpt2_layer_norm(0, None, 0, None, None, 1, 768, None, None) == 1
    assert G.LIB.gpt2_sync_status(None, None) == 1
    assert G.LIB.gpt2_linear(None, 0, None, None, None, None, None, 1, 1, 1, None) == 1
    assert G.LIB.gpt2_attention(None, None, None, 1, 1, 1, 0, 1, 64, None, None) == 1
    assert G.LIB.gpt2_embed(None, None, None, None, 1, 1, 0, None, None) == 1
    assert G.LIB.gpt2_profile_enable(None, 1) == 1
    G.LIB.gpt2_ctx_destroy(None)


def test_misaligned_pointer_rejected_without_launch(G):
    # Host-side checks run before any CUDA call: fake, never dereferenced addresses.
    a16, bad = 0x10000, 0x10004
    assert G.LIB.gpt2_layer_norm(0, bad, 0, a16, a16, 4, 768, a16, None) == G.GPT2_ERR_ALIGNMENT
    assert G.LIB.gpt2_layer_norm(0, a16, 0, a16, a16, 0, 768, a16, None) == G.GPT2_ERR_INVALID_ARG


def test_ctx_create_rejects_small_or_misaligned_workspace(G):
    h = C.c_void_p()
    n = C.c_size_t()
    G.LIB.gpt2_workspace_bytes(C.byref(_hp(G)), 2, 8, C.byref(n))
    assert G.LIB.gpt2_ctx_create(C.byref(_hp(G)), 2, 8, 0x10010, n.value, C.byref(h)) == G.GPT2_ERR_ALIGNMENT
    assert G.LIB.gpt2_ctx_create(C.byref(_hp(G)), 2, 8, 0x10000, n.value - 1, C.byref(h)) == G.GPT2_ERR_WORKSPACE


def test_noalloc_decode_validates_on_the_host(G):
    # Every check below returns before the device is touched (fake, never
    # dereferenced 16-byte aligned addresses; no GPU needed).
    f = G.LIB.gpt2_attention_decode_noalloc
    a16, bad = 0x10000, 0x10004
    assert f(None, a16, 1, 4, 10, 16, 64, 0, a16, None) == G.GPT2_ERR_INVALID_ARG
    assert f(a16, a16, 0, 4, 10, 16, 64, 0, a16, None) == G.GPT2_ERR_INVALID_ARG    # B = 0
    assert f(a16, a16, 1, 4, 0, 16, 64, 0, a16, None) == G.GPT2_ERR_INVALID_ARG     # no past
    assert f(a16, a16, 1, 4, 10, 16, 64, -1, a16, None) == G.GPT2_ERR_INVALID_ARG   # splits < 0
    assert f(a16, a16, 1, 4, 10, 16, 32, 0, a16, None) == G.GPT2_ERR_UNSUPPORTED    # d_h != 64
    assert f(a16, a16, 1, 4, 16, 16, 64, 0, a16, None) == G.GPT2_ERR_CTX_OVERFLOW   # T_past + 1 > T_cap
    assert f(bad, a16, 1, 4, 10, 16, 64, 0, a16, None) == G.GPT2_ERR_ALIGNMENT
    # One CTA row per (sequence, head): B * h beyond the grid's 65535 rows.
    assert f(a16, a16, 4096, 16, 10, 16, 64, 1, a16, None) == G.GPT2_ERR_UNSUPPORTED
    assert f(a16, a16, 1 << 20, 1 << 12, 10, 16, 64, 0, a16, None) == G.GPT2_ERR_UNSUPPORTED


def test_profiler_kinds_and_null_context(G):
    n = G.LIB.gpt2_profile_kinds()
    assert n >= 8  # embed, LayerNorm, four block products, head, attention, ...
    name = C.c_char_p()
    ll, d1, d2, d3 = C.c_longlong(), C.c_double(), C.c_double(), C.c_double()
    assert G.LIB.gpt2_profile_read(None, 0, C.byref(name), C.byref(ll), C.byref(d1), C.byref(d2),
                                   C.byref(d3)) == G.GPT2_ERR_INVALID_ARG
    assert G.LIB.gpt2_profile_reset(None) == G.GPT2_ERR_INVALID_ARG
    assert G.LIB.gpt2_selftest_wait_timeout(None, 1000, None) == G.GPT2_ERR_INVALID_ARG
    assert G.LIB.gpt2_ctx_set_wait_limit(None, 1000) == G.GPT2_ERR_INVALID_ARG


def test_binding_refuses_to_load_without_the_library():
    # No fallback: with the library missing, importing the binding raises.
    import subprocess
    import sys
    code = ("import gpt_pre_norm_gb300.build as b; b.LIB = '/nonexistent/libgpt2fwd.so'\n"
            "try:\n    import gpt_pre_norm_gb300.binding\nexcept ImportError as e:\n"
            "    print('refused:', 'no fallback' in str(e))\nelse:\n    print('loaded')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == "refused: True"
