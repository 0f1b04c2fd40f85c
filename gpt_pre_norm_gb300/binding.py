"""Thin ctypes binding of libgpt2fwd.so: the C ABI of include/gpt2.h, same names.

Argument marshalling only: torch tensors in, device pointers and sizes out.
Every step of the forward runs in the library's CUDA kernels; there is no
fallback.  Importing this module without the built library raises.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import build as _build

GPT2_OK = 0
GPT2_ERR_INVALID_ARG = 1
GPT2_ERR_UNSUPPORTED = 2
GPT2_ERR_CTX_OVERFLOW = 3
GPT2_ERR_ALIGNMENT = 4
GPT2_ERR_CUDA = 5
GPT2_ERR_DEVICE_TIMEOUT = 6
GPT2_ERR_WORKSPACE = 7
GPT2_ERR_NO_DEVICE = 8
GPT2_ERR_RANGE = 9

GPT2_BF16 = 0
GPT2_FP32 = 1

GPT2_EPI_BIAS = 0
GPT2_EPI_BIAS_GELU = 1
GPT2_EPI_BIAS_RESID = 2
GPT2_EPI_LOGITS = 3

BLOCK_FIELDS = ("ln1_g", "ln1_b", "attn_w", "attn_b", "proj_w", "proj_b",
                "ln2_g", "ln2_b", "fc_w", "fc_b", "mlp_proj_w", "mlp_proj_b")


class gpt2_hparams(C.Structure):
    _fields_ = [("n_vocab", C.c_int), ("n_ctx", C.c_int), ("n_embd", C.c_int),
                ("n_head", C.c_int), ("n_layer", C.c_int), ("dtype", C.c_int)]


class gpt2_block_params(C.Structure):
    _fields_ = [(f, C.c_void_p) for f in BLOCK_FIELDS]


class gpt2_params(C.Structure):
    _fields_ = [("wte", C.c_void_p), ("wpe", C.c_void_p), ("lnf_g", C.c_void_p),
                ("lnf_b", C.c_void_p), ("blocks", C.POINTER(gpt2_block_params))]


class gpt2_kv(C.Structure):
    _fields_ = [("data", C.c_void_p), ("T_cap", C.c_int), ("T_len", C.c_int)]


class Gpt2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def _load() -> C.CDLL:
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(the CUDA library is required; there is no fallback)")
    lib = C.CDLL(path)
    P, I, V, Z, LL, D = C.c_void_p, C.c_int, None, C.c_size_t, C.c_longlong, C.c_double
    sig = {
        "gpt2_workspace_bytes": (I, [C.POINTER(gpt2_hparams), I, I, C.POINTER(Z)]),
        "gpt2_ctx_create": (I, [C.POINTER(gpt2_hparams), I, I, P, Z, C.POINTER(P)]),
        "gpt2_ctx_destroy": (V, [P]),
        "gpt2_sync_status": (I, [P, P]),
        "gpt2_status_string": (C.c_char_p, [I]),
        "gpt2_block_forward": (I, [P, P, C.POINTER(gpt2_block_params), I, I, I, I,
                                   C.POINTER(gpt2_kv), C.POINTER(gpt2_kv), P, P]),
        "gpt2_block_forward_postnorm": (I, [P, P, C.POINTER(gpt2_block_params), I, I, I, I, P,
                                            P]),
        "gpt2_forward": (I, [P, P, I, I, C.POINTER(gpt2_params), I, C.POINTER(gpt2_kv),
                             C.POINTER(gpt2_kv), P, P]),
        "gpt2_forward_loss": (I, [P, P, P, I, I, C.POINTER(gpt2_params), I, C.POINTER(gpt2_kv),
                                  C.POINTER(gpt2_kv), P, P, P]),
        "gpt2_forward_topk": (I, [P, P, I, I, C.POINTER(gpt2_params), I, C.POINTER(gpt2_kv),
                                  C.POINTER(gpt2_kv), I, P, P, P, P]),
        "gpt2_layer_norm": (I, [I, P, I, P, P, I, I, P, P]),
        "gpt2_linear": (I, [P, I, P, P, P, P, P, I, I, I, P]),
        "gpt2_attention": (I, [P, P, P, I, I, I, I, I, I, P, P]),
        "gpt2_embed": (I, [P, P, P, P, I, I, I, P, P]),
        "gpt2_attention_decode_noalloc": (I, [P, P, I, I, I, I, I, I, P, P]),
        "gpt2_attention_decode_noalloc_status": (I, [P]),
        "gpt2_attention_decode_noalloc_set_wait_limit": (I, [LL]),
        "gpt2_ctx_cache_weights": (I, [P, I]),
        "gpt2_selftest_wait_timeout": (I, [P, I, P]),
        "gpt2_ctx_set_wait_limit": (I, [P, LL]),
        "gpt2_generate_greedy": (I, [P, P, I, I, C.POINTER(gpt2_params), I, C.POINTER(gpt2_kv), I,
                                     P, P, P]),
        "gpt2_profile_enable": (I, [P, I]),
        "gpt2_profile_kinds": (I, []),
        "gpt2_profile_read": (I, [P, I, C.POINTER(C.c_char_p), C.POINTER(LL), C.POINTER(D),
                                  C.POINTER(D), C.POINTER(D)]),
        "gpt2_profile_reset": (I, [P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


def status_string(status: int) -> str:
    return LIB.gpt2_status_string(status).decode()


def _check(status: int, where: str) -> None:
    if status != GPT2_OK:
        raise Gpt2Error(status, where)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def dtype_of(mode: int) -> torch.dtype:
    return torch.bfloat16 if mode == GPT2_BF16 else torch.float32


class KV:
    """A KV cache tensor [B, (L,) 2, h, T_cap, d_h] and its valid length."""

    def __init__(self, data: torch.Tensor, T_len: int = 0):
        self.data = data
        self.T_len = T_len

    @property
    def T_cap(self) -> int:
        return self.data.shape[-2]

    def struct(self) -> gpt2_kv:
        return gpt2_kv(_ptr(self.data), self.T_cap, self.T_len)


class Context:
    """A library context and the device workspace it owns (allocated by torch)."""

    def __init__(self, n_vocab: int, n_ctx: int, n_embd: int, n_head: int, n_layer: int,
                 dtype: int, max_B: int, max_T: int):
        self.hp = gpt2_hparams(n_vocab, n_ctx, n_embd, n_head, n_layer, dtype)
        nbytes = C.c_size_t(0)
        _check(LIB.gpt2_workspace_bytes(C.byref(self.hp), max_B, max_T, C.byref(nbytes)),
               "gpt2_workspace_bytes")
        self.workspace = torch.empty(nbytes.value, dtype=torch.uint8, device="cuda")
        h = C.c_void_p()
        _check(LIB.gpt2_ctx_create(C.byref(self.hp), max_B, max_T, self.workspace.data_ptr(),
                                   nbytes.value, C.byref(h)), "gpt2_ctx_create")
        self.handle = h
        self.mode = dtype
        self.max_B, self.max_T = max_B, max_T

    @property
    def dtype(self) -> torch.dtype:
        return dtype_of(self.mode)

    def close(self) -> None:
        if self.handle:
            torch.cuda.synchronize()
            LIB.gpt2_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gpt2_ctx_cache_weights(ctx: Context, enable: bool) -> None:
    _check(LIB.gpt2_ctx_cache_weights(ctx.handle, int(enable)), "gpt2_ctx_cache_weights")


def gpt2_sync_status(ctx: Context, stream=None) -> int:
    return LIB.gpt2_sync_status(ctx.handle, _stream(stream))


def block_params_struct(p: dict) -> gpt2_block_params:
    return gpt2_block_params(*[_ptr(p[f]) for f in BLOCK_FIELDS])


def gpt2_block_forward(ctx: Context, x: torch.Tensor, params: dict, B: int, T: int, d: int,
                       n_head: int, past: KV | None = None, present: KV | None = None,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty_like(x)
    bp = block_params_struct(params)
    ps = past.struct() if past is not None else None
    pr = present.struct() if present is not None else None
    st = LIB.gpt2_block_forward(ctx.handle, _ptr(x), C.byref(bp), B, T, d, n_head,
                                C.byref(ps) if ps is not None else None,
                                C.byref(pr) if pr is not None else None, _ptr(out),
                                _stream(stream))
    _check(st, "gpt2_block_forward")
    if present is not None:
        present.T_len = pr.T_len
    return out


def gpt2_block_forward_postnorm(ctx: Context, x: torch.Tensor, params: dict, B: int, T: int,
                                d: int, n_head: int, out: torch.Tensor | None = None,
                                stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty_like(x)
    bp = block_params_struct(params)
    st = LIB.gpt2_block_forward_postnorm(ctx.handle, _ptr(x), C.byref(bp), B, T, d, n_head,
                                         _ptr(out), _stream(stream))
    _check(st, "gpt2_block_forward_postnorm")
    return out


class ModelParams:
    """Keeps the ctypes records of a model's parameters alive across calls."""

    def __init__(self, p: dict):
        self.tensors = p
        self.blocks = (gpt2_block_params * len(p["blocks"]))(
            *[block_params_struct(b) for b in p["blocks"]])
        self.struct = gpt2_params(_ptr(p["wte"]), _ptr(p["wpe"]), _ptr(p["lnf_g"]),
                                  _ptr(p["lnf_b"]), self.blocks)
        self.n_layer = len(p["blocks"])


def gpt2_forward(ctx: Context, ids: torch.Tensor, params: ModelParams, B: int, T: int,
                 past: KV | None = None, present: KV | None = None,
                 logits: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if logits is None:
        logits = torch.empty((B, T, ctx.hp.n_vocab), dtype=torch.float32, device=ids.device)
    ps = past.struct() if past is not None else None
    pr = present.struct() if present is not None else None
    st = LIB.gpt2_forward(ctx.handle, _ptr(ids), B, T, C.byref(params.struct), params.n_layer,
                          C.byref(ps) if ps is not None else None,
                          C.byref(pr) if pr is not None else None, _ptr(logits), _stream(stream))
    _check(st, "gpt2_forward")
    if present is not None:
        present.T_len = pr.T_len
    return logits


def gpt2_forward_loss(ctx: Context, ids: torch.Tensor, params: ModelParams, B: int, T: int,
                      targets: torch.Tensor | None = None, past: KV | None = None,
                      present: KV | None = None, want_next: bool = True, stream=None,
                      loss: torch.Tensor | None = None):
    """(loss [B, T] fp32 or None, next_ids [B, T] int32 or None) without the
    logits; loss needs targets (written into `loss` when given)."""
    if targets is None:
        loss = None
    elif loss is None:
        loss = torch.empty((B, T), dtype=torch.float32, device=ids.device)
    nxt = torch.empty((B, T), dtype=torch.int32, device=ids.device) if want_next else None
    ps = past.struct() if past is not None else None
    pr = present.struct() if present is not None else None
    _check(LIB.gpt2_forward_loss(ctx.handle, _ptr(ids), _ptr(targets), B, T, C.byref(params.struct),
                                 params.n_layer, C.byref(ps) if ps is not None else None,
                                 C.byref(pr) if pr is not None else None, _ptr(loss), _ptr(nxt),
                                 _stream(stream)), "gpt2_forward_loss")
    if present is not None:
        present.T_len = pr.T_len
    return loss, nxt


def gpt2_forward_topk(ctx: Context, ids: torch.Tensor, params: ModelParams, B: int, T: int,
                      k: int, past: KV | None = None, present: KV | None = None,
                      want_lse: bool = True, stream=None, top_logits: torch.Tensor | None = None,
                      top_ids: torch.Tensor | None = None):
    """(top_logits [B, T, k] fp32, top_ids [B, T, k] int32, lse [B, T] fp32 or
    None) without the logits (written into top_logits / top_ids when given)."""
    tv = top_logits if top_logits is not None else \
        torch.empty((B, T, k), dtype=torch.float32, device=ids.device)
    ti = top_ids if top_ids is not None else \
        torch.empty((B, T, k), dtype=torch.int32, device=ids.device)
    lse = torch.empty((B, T), dtype=torch.float32, device=ids.device) if want_lse else None
    ps = past.struct() if past is not None else None
    pr = present.struct() if present is not None else None
    _check(LIB.gpt2_forward_topk(ctx.handle, _ptr(ids), B, T, C.byref(params.struct),
                                 params.n_layer, C.byref(ps) if ps is not None else None,
                                 C.byref(pr) if pr is not None else None, k, _ptr(tv), _ptr(ti),
                                 _ptr(lse), _stream(stream)), "gpt2_forward_topk")
    if present is not None:
        present.T_len = pr.T_len
    return tv, ti, lse


def gpt2_generate_greedy(ctx: Context, ids: torch.Tensor, params: ModelParams, n_new: int,
                         cache: KV, logits: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """Greedy continuation of the prompt ids [B, T] by n_new tokens (int32
    [B, n_new]); the prompt and the generated tokens go into `cache`."""
    B, T = ids.shape
    if logits is None:
        logits = torch.empty((B, T, ctx.hp.n_vocab), dtype=torch.float32, device=ids.device)
    out = torch.empty((B, n_new), dtype=torch.int32, device=ids.device)
    cs = cache.struct()
    _check(LIB.gpt2_generate_greedy(ctx.handle, _ptr(ids), B, T, C.byref(params.struct),
                                    params.n_layer, C.byref(cs), n_new, _ptr(logits), _ptr(out),
                                    _stream(stream)), "gpt2_generate_greedy")
    cache.T_len = cs.T_len
    return out


def gpt2_layer_norm(mode: int, x: torch.Tensor, g: torch.Tensor, b: torch.Tensor,
                    y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    d = x.shape[-1]
    rows = x.numel() // d
    if y is None:
        y = torch.empty(x.shape, dtype=dtype_of(mode), device=x.device)
    x_dtype = GPT2_FP32 if x.dtype == torch.float32 else GPT2_BF16
    _check(LIB.gpt2_layer_norm(mode, _ptr(x), x_dtype, _ptr(g), _ptr(b), rows, d, _ptr(y),
                               _stream(stream)), "gpt2_layer_norm")
    return y


def gpt2_linear(ctx: Context, epilogue: int, A: torch.Tensor, W: torch.Tensor,
                bias: torch.Tensor | None = None, resid: torch.Tensor | None = None,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    M, K = A.shape
    N = W.shape[0]
    if out is None:
        odt = torch.float32 if epilogue in (GPT2_EPI_BIAS_RESID, GPT2_EPI_LOGITS) else ctx.dtype
        out = torch.empty((M, N), dtype=odt, device=A.device)
    _check(LIB.gpt2_linear(ctx.handle, epilogue, _ptr(A), _ptr(W), _ptr(bias), _ptr(resid),
                           _ptr(out), M, N, K, _stream(stream)), "gpt2_linear")
    return out


def gpt2_attention(ctx: Context, q: torch.Tensor, kv: torch.Tensor, T_past: int,
                   out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    B, h, T, dh = q.shape
    T_cap = kv.shape[-2]
    if out is None:
        out = torch.empty((B, T, h * dh), dtype=q.dtype, device=q.device)
    _check(LIB.gpt2_attention(ctx.handle, _ptr(q), _ptr(kv), B, h, T, T_past, T_cap, dh, _ptr(out),
                              _stream(stream)), "gpt2_attention")
    return out


def gpt2_attention_decode_noalloc(q: torch.Tensor, kv: torch.Tensor, T_past: int, splits: int = 0,
                                  out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Decode attention (T = 1) without a context or workspace: the partial
    results use the library's own fixed device array."""
    B, h, T, dh = q.shape
    if out is None:
        out = torch.empty((B, T, h * dh), dtype=q.dtype, device=q.device)
    _check(LIB.gpt2_attention_decode_noalloc(_ptr(q), _ptr(kv), B, h, T_past, kv.shape[-2], dh,
                                             splits, _ptr(out), _stream(stream)),
           "gpt2_attention_decode_noalloc")
    return out


def gpt2_attention_decode_noalloc_status(stream=None) -> int:
    """The no-allocation decode entry point's device error word: synchronises
    the stream, returns the status (OK or DEVICE_TIMEOUT) and clears it."""
    return LIB.gpt2_attention_decode_noalloc_status(_stream(stream))


def gpt2_attention_decode_noalloc_set_wait_limit(limit_ns: int) -> None:
    """Test support: the no-allocation decode kernel's wait limit (<= 0: default)."""
    _check(LIB.gpt2_attention_decode_noalloc_set_wait_limit(limit_ns),
           "gpt2_attention_decode_noalloc_set_wait_limit")


def gpt2_embed(ctx: Context, ids: torch.Tensor, wte: torch.Tensor, wpe: torch.Tensor,
               T_past: int = 0, H: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    B, T = ids.shape
    if H is None:
        H = torch.empty((B, T, wte.shape[1]), dtype=torch.float32, device=ids.device)
    _check(LIB.gpt2_embed(ctx.handle, _ptr(ids), _ptr(wte), _ptr(wpe), B, T, T_past, _ptr(H),
                          _stream(stream)), "gpt2_embed")
    return H


def gpt2_selftest_wait_timeout(ctx: Context, limit_us: int, stream=None) -> None:
    """Launches a wait that runs out after limit_us (see the header); the next
    gpt2_sync_status reports GPT2_ERR_DEVICE_TIMEOUT."""
    _check(LIB.gpt2_selftest_wait_timeout(ctx.handle, limit_us, _stream(stream)),
           "gpt2_selftest_wait_timeout")


def gpt2_ctx_set_wait_limit(ctx: Context, limit_ns: int) -> None:
    """Limit of the kernels' bounded waits (test support; <= 0 restores 2 s)."""
    _check(LIB.gpt2_ctx_set_wait_limit(ctx.handle, int(limit_ns)), "gpt2_ctx_set_wait_limit")


def gpt2_profile_enable(ctx: Context, enable: bool) -> None:
    _check(LIB.gpt2_profile_enable(ctx.handle, int(enable)), "gpt2_profile_enable")


def gpt2_profile_reset(ctx: Context) -> None:
    _check(LIB.gpt2_profile_reset(ctx.handle), "gpt2_profile_reset")


def gpt2_profile_read(ctx: Context) -> dict:
    """Per kernel kind: launches, total ms, flops, bytes (waits for the events)."""
    out = {}
    for k in range(LIB.gpt2_profile_kinds()):
        name = C.c_char_p()
        n = C.c_longlong()
        ms, fl, by = C.c_double(), C.c_double(), C.c_double()
        _check(LIB.gpt2_profile_read(ctx.handle, k, C.byref(name), C.byref(n), C.byref(ms),
                                     C.byref(fl), C.byref(by)), "gpt2_profile_read")
        if n.value:
            out[name.value.decode()] = {"launches": n.value, "ms": ms.value, "flops": fl.value,
                                        "bytes": by.value}
    return out
