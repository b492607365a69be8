"""Shared helpers of the GPU parity tests: bf16 bits <-> torch tensors, and the parity bar."""
import numpy as np
import pytest
import torch

COS_MIN = 0.9995        # cosine similarity against the float64 oracle, per output tensor
REL_MAX = 3e-2          # max |gpu - oracle| <= REL_MAX * max |oracle|, per output tensor


def dev():
    return torch.device("cuda:0")


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev())


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def parity_stats(got: np.ndarray, ref: np.ndarray):
    g = np.asarray(got, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    denom = np.sqrt((g * g).sum() * (r * r).sum())
    cos = float((g * r).sum() / denom) if denom > 0 else (1.0 if np.array_equal(g, r) else 0.0)
    mref = float(np.abs(r).max()) if r.size else 0.0
    err = float(np.abs(g - r).max()) if r.size else 0.0
    return cos, err, mref


def assert_parity(got, ref, name=""):
    cos, err, mref = parity_stats(got, ref)
    assert np.isfinite(got).all(), f"{name}: non-finite GPU output"
    assert cos >= COS_MIN, f"{name}: cosine {cos:.6f} < {COS_MIN}"
    assert err <= REL_MAX * mref + 1e-30, f"{name}: max|err| {err:.4g} > {REL_MAX} * max|ref| {mref:.4g}"
    return cos, err / mref if mref > 0 else 0.0


def assert_parity_combination(got, parts, name=""):
    """Parity of a linear combination sum_k c_k ref_k whose parts each carry the per-tensor bar.

    If every part ref_k is reproduced within cosine COS_MIN (relative L2 error at most
    sqrt(2 (1 - COS_MIN))) and max-abs error REL_MAX * max|ref_k|, the combination's error is at most
    the same combination of the parts' bounds: sum_k |c_k| * bound_k (triangle inequality).  Guided
    velocities v = v_neg + g (v_pos - v_neg) = (1 - g) v_neg + g v_pos take this bar."""
    ref = sum(c * r for c, r in parts)
    cos, err, mref = parity_stats(got, ref)
    plain = cos >= COS_MIN and err <= REL_MAX * mref
    print(f"{name}: plain bar {'holds' if plain else 'does not hold'} (cosine {cos:.6f}, "
          f"max|err|/max|ref| {err / mref if mref > 0 else 0.0:.3e})")
    e = np.asarray(got, dtype=np.float64).ravel() - np.asarray(ref, dtype=np.float64).ravel()
    rel_l2 = np.sqrt(2.0 * (1.0 - COS_MIN))
    l2_bound = sum(abs(c) * rel_l2 * np.linalg.norm(r) for c, r in parts)
    max_bound = sum(abs(c) * REL_MAX * np.abs(r).max() for c, r in parts)
    assert np.isfinite(got).all(), f"{name}: non-finite GPU output"
    assert np.linalg.norm(e) <= l2_bound, f"{name}: |err|_2 {np.linalg.norm(e):.4g} > {l2_bound:.4g}"
    assert np.abs(e).max() <= max_bound, f"{name}: max|err| {np.abs(e).max():.4g} > {max_bound:.4g}"


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import diffusion_transformer_denoiser_gb300 as mi
    mi.lib()
    if not mi.device_supported():
        pytest.fail("device is not sm_103: " + mi.lib().mi_last_error().decode())
    return mi
