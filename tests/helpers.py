"""Shared helpers of the GPU parity tests: device transfer and the tolerances.

Tolerances (fixed for the whole suite):
  fp32 mode  max |gpu - oracle| <= 1e-4 * max(1, |oracle|), element-wise;
  bf16 mode  relative L2 error ||gpu - oracle|| / ||oracle|| <= 1e-2 per output
             tensor, and for full-model logits the argmax agrees at >= 99% of
             positions.
"""
import numpy as np
import torch

FP32_TOL = 1e-4
BF16_REL_L2 = 1e-2
ARGMAX_AGREE = 0.99


def dev(a: np.ndarray, dtype=torch.bfloat16) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_l2(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def assert_bf16_close(got, ref, tol=BF16_REL_L2, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    e = rel_l2(got, ref)
    assert e <= tol, f"{what}: relative L2 error {e:.3e} > {tol:.1e}"
    return e


def assert_fp32_close(got, ref, tol=FP32_TOL, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    assert float(err.max()) <= tol, f"{what}: max scaled error {float(err.max()):.3e} > {tol:.1e}"
    return float(err.max())


def assert_gemm_f32_close(got, ref, A, W, what=""):
    """fp32-output tensor-core product of bf16 operands: every product is exact
    in fp32 and the error comes from the fp32 accumulation alone.  Bound per
    element: (sqrt(K/16) + 2) * 2^-22 * sum_k |a_k w_k| (K/16 accumulation
    steps of 16 products, each rounding at fp32 precision), plus one fp32 ulp
    of the result."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    K = A.shape[1]
    l1 = np.abs(np.asarray(A, np.float64)) @ np.abs(np.asarray(W, np.float64)).T
    bound = (np.sqrt(K / 16.0) + 2.0) * 2.0 ** -22 * l1 + 2.0 ** -23 * np.abs(ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    excess = np.abs(got - ref) - bound
    assert float(excess.max()) <= 0, f"{what}: error above the fp32 accumulation bound by {float(excess.max()):.3e}"


def argmax_agreement(got_logits, ref_logits) -> float:
    g = np.argmax(np.asarray(got_logits), axis=-1)
    r = np.argmax(np.asarray(ref_logits), axis=-1)
    return float(np.mean(g == r))


def block_to_device(p: dict, dtype=torch.bfloat16) -> dict:
    return {k: dev(v, dtype) for k, v in p.items()}


def model_to_device(p: dict, dtype=torch.bfloat16) -> dict:
    out = {k: dev(p[k], dtype) for k in ("wte", "wpe", "lnf_g", "lnf_b")}
    out["blocks"] = [block_to_device(b, dtype) for b in p["blocks"]]
    return out


def check_top_choice(z, ref, got, rv, ri):
    """The top choice against the fp64 oracle, position by position.  Where
    the oracle's two largest logits are further apart than twice the
    library's logit error on that row (measured on its own logits z, plus the
    few ulps between the two head layouts), the choice is decided at this
    precision and must be the oracle's; elsewhere it must be a logit within
    that error of the oracle's maximum.  Most positions must be decided."""
    zf = z.astype(np.float64)
    err = np.abs(zf - ref).max(axis=-1) + 1e-4 * np.maximum(1.0, np.abs(zf).max(axis=-1))
    decided = rv[..., 0] - rv[..., 1] > 2 * err
    # 0.93-0.99 of the positions on the random-weight models of the GPU tests
    assert np.mean(decided) >= 0.85, f"decided at only {np.mean(decided):.3f} of positions"
    np.testing.assert_array_equal(got[decided], ri[..., 0][decided])
    chosen = np.take_along_axis(ref, got[..., None].astype(np.int64), axis=-1)[..., 0]
    assert np.all(chosen >= rv[..., 0] - 2 * err)
