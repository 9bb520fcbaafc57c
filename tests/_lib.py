"""Helpers shared by the tests: build/load the library, tolerance checks."""

import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpattn.h")


def built_lib():
    from context_causal_attention_load_gb300 import build
    build.build()
    from context_causal_attention_load_gb300 import cpattn
    return cpattn.load()


def header_functions():
    """Names of the functions include/cpattn.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "for")))


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def assert_close_out(got, want, name="out", max_abs=2e-2, rel=5e-3):
    """Forward tolerance: max-abs <= 2e-2 and relative L2 <= 5e-3 (bf16
    inputs, fp32 accumulation, bf16 output)."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    ma = float(np.max(np.abs(got - want))) if got.size else 0.0
    r = rel_l2(got, want)
    assert ma <= max_abs and r <= rel, "%s: max-abs %.3e (<= %.1e), rel-L2 %.3e (<= %.1e)" % (
        name, ma, max_abs, r, rel)


def assert_close_grad(got, want, name, rel=1e-2):
    r = rel_l2(got, want)
    assert r <= rel, "%s: rel-L2 %.3e (<= %.1e)" % (name, r, rel)
