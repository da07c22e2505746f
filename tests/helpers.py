"""Shared comparison helpers for the parity tests (tolerances from the spec:
bf16 I/O with fp32 accumulation: max-abs <= 2e-2 and relative L2 <= 5e-3;
fp32 I/O: max-abs <= 1e-4)."""
import numpy as np
import torch

BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
F32_MAX_ABS = 1e-4


def to_np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def errors(out, ref):
    out, ref = to_np(out), to_np(ref)
    d = out - ref
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(d) / nref) if nref > 0 else 0.0
    return max_abs, rel


def assert_bf16_close(out, ref, what=""):
    max_abs, rel = errors(out, ref)
    assert np.isfinite(to_np(out)).all(), f"{what}: non-finite output"
    assert max_abs <= BF16_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {BF16_MAX_ABS}"
    assert rel <= BF16_REL_L2, f"{what}: rel-L2 {rel:.3e} > {BF16_REL_L2}"
    return max_abs, rel


def assert_f32_close(out, ref, what=""):
    max_abs, rel = errors(out, ref)
    assert np.isfinite(to_np(out)).all(), f"{what}: non-finite output"
    assert max_abs <= F32_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {F32_MAX_ABS}"
    return max_abs, rel
