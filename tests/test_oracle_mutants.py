"""The pins must catch plausible mistakes in the oracle.

Each case copies the C oracle, plants one mistake (a dropped sink term, an
off-by-one window edge, a wrong GQA head map, a transposed operand, a value
read at the wrong position), builds the copy with gcc and checks that the
independent pins (numpy brute force, torch SDPA, closed forms) reject it.
The mistakes are planted on the CPU, in a temporary copy only.
"""
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle import brute

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "attn_sink_oracle.c")

MUTANTS = {
    "drop_sink_from_denominator": ("double z = zsink;", "double z = 0.0;"),
    "window_one_too_wide": ("i - window + 1 > 0) ? i - window + 1", "i - window > 0) ? i - window"),
    "gqa_map_modulo": ("int g = h / G;", "int g = h % Hkv;"),
    "q_dot_q": ("(double)qv[d] * (double)kv[d]", "(double)qv[d] * (double)qv[d]"),
    "values_reversed": ("vbase + (long)(lo + t) * vstride", "vbase + (long)(hi - t) * vstride"),
    "sink_scaled": ("double m = sigma;", "sigma *= scale; double m = sigma;"),
}


def _build(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", str(path), "-o", str(so), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
    f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
    ci = ctypes.c_int
    lib.oracle_prefill.argtypes = [f32p, f32p, f32p, f32p, f64p, ctypes.c_void_p, ctypes.c_void_p,
                                   ci, ci, ci, ci, ci, ci, ctypes.c_double]
    return lib


def _run(lib, q, k, v, sink, window, scale):
    B, T, Hq, D = q.shape
    o = np.zeros((B, T, Hq, D))
    lib.oracle_prefill(*(np.ascontiguousarray(x.numpy(), np.float32) for x in (q, k, v, sink)),
                       o, None, None, B, T, Hq, k.shape[2], D, int(window or 0), scale)
    return o


def _pins_hold(lib) -> bool:
    """True when the library passes the brute-force and SDPA pins."""
    B, T, Hq, Hkv, D = 1, 24, 4, 2, 8
    q, k, v, sink = synth.prefill_inputs(B, T, Hq, Hkv, D, 31, dtype=torch.float32)
    scale = 1.0 / math.sqrt(D)
    for window in (None, 5):
        ob, _, _ = brute.prefill(q.numpy(), k.numpy(), v.numpy(), sink.numpy(), window, scale)
        if not np.allclose(_run(lib, q, k, v, sink, window, scale), ob, rtol=0, atol=1e-10):
            return False
    nosink = torch.full((Hq,), -math.inf)
    ref = F.scaled_dot_product_attention(*(x.double().transpose(1, 2) for x in (q, k, v)),
                                         is_causal=True, scale=scale, enable_gqa=True).transpose(1, 2)
    return np.allclose(_run(lib, q, k, v, nosink, None, scale), ref.numpy(), rtol=0, atol=1e-10)


def test_unmutated_copy_passes(tmp_path):
    assert _pins_hold(_build(tmp_path, "original", "double z = zsink;", "double z = zsink;"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    assert not _pins_hold(_build(tmp_path, name, old, new)), f"pins missed mutant {name}"
