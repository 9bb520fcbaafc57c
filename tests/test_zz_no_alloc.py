"""gqa_decode_noalloc: the decode entry point for callers that cannot let the
library allocate device memory (memory owned by a caching allocator or a
pool sized up front, serving loops that must stay off the driver's
allocation path, processes that keep nearly all of HBM for the KV cache).
It keeps its split partials in a fixed static device array; its results
must equal those of gqa_decode, call after call, even when one call leaves
partials in the array that the next call's shapes do not overwrite.

This file is collected last so that a failure here cannot hide the result of
any other test; it also passes when run alone in a fresh process."""

import ctypes

import pytest
import torch

from context_causal_attention_load_gb300 import synth
from tests._lib import assert_close_out, built_lib

pytestmark = pytest.mark.gpu


def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    lib = built_lib()
    f = lib.gqa_decode_noalloc
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call(lib, q, kc, vc, lens, out):
    B, Hq, D = q.shape
    Hkv, Smax = kc.shape[1], kc.shape[2]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.gqa_decode_noalloc(_p(q), _p(kc), _p(vc), _p(lens), _p(out), B, Hq, Hkv, Smax, D, stream)


def _check(lib, q, kc, vc, lens, what):
    from context_causal_attention_load_gb300 import cpattn
    ref = cpattn.gqa_decode(q, kc, vc, lens)
    out = torch.full_like(q, float("nan"))
    assert _call(lib, q, kc, vc, lens, out) == 0, lib.cp_attn_last_error()
    torch.cuda.synchronize()
    assert_close_out(out.double().cpu().numpy(), ref.double().cpu().numpy(), what)


@pytest.mark.parametrize("shape,seed", [
    ((24, 32, 8, 128, 2048, 1024, 2048), 31),   # the decode workload
    ((3, 12, 4, 64, 700, 1, 700), 32),          # G = 3, D = 64, ragged splits
])
def test_noalloc_matches_gqa_decode_on_two_calls(shape, seed):
    """Two calls in a row with different inputs: the second changes every
    sequence's length (half of them shorter, so they have fewer slices than
    the first call left partials for; half longer) and draws new q/K/V."""
    lib = _lib()
    B, Hq, Hkv, D, Smax, lo, hi = shape
    q, kc, vc, lens = (x.cuda() for x in synth.decode_inputs(B, Hq, Hkv, D, Smax, lo, hi, seed=seed))
    _check(lib, q, kc, vc, lens, "noalloc decode, first call")
    q2, kc2, vc2, _ = (x.cuda() for x in synth.decode_inputs(B, Hq, Hkv, D, Smax, lo, hi, seed=seed + 100))
    short = torch.clamp(lens // 3, min=1)
    long_ = torch.clamp(lens + 300, max=Smax)
    idx = torch.arange(B, device=lens.device)
    lens2 = torch.where(idx % 2 == 0, short, long_).to(torch.int32).contiguous()
    assert bool((lens2 != lens).any())
    _check(lib, q2, kc2, vc2, lens2, "noalloc decode, second call (other lengths)")


def test_noalloc_reads_lens_written_just_before():
    """A device kernel rewrites the lengths immediately before the call (a
    serving loop's lens += 1): the call must use the new lengths."""
    lib = _lib()
    from context_causal_attention_load_gb300 import cpattn
    B, Hq, Hkv, D, Smax = 24, 32, 8, 128, 2048
    q, kc, vc, lens = (x.cuda() for x in synth.decode_inputs(B, Hq, Hkv, D, Smax, 1, 1100, seed=33))
    lens_dev = lens.clone()
    out = torch.full_like(q, float("nan"))
    torch.cuda.synchronize()
    lens_dev.add_(900)  # queued on the stream right before the decode; crosses slice boundaries
    assert _call(lib, q, kc, vc, lens_dev, out) == 0, lib.cp_attn_last_error()
    torch.cuda.synchronize()
    ref = cpattn.gqa_decode(q, kc, vc, (lens + 900).to(torch.int32))
    torch.cuda.synchronize()
    assert_close_out(out.double().cpu().numpy(), ref.double().cpu().numpy(), "noalloc decode, lens just updated")


def test_noalloc_device_flag_is_reported():
    """Lengths past Smax are clamped and flagged in the array's error word;
    cp_attn_check_device reports it once and clears it."""
    lib = _lib()
    from context_causal_attention_load_gb300 import cpattn
    q, kc, vc, lens = (x.cuda() for x in synth.decode_inputs(2, 8, 2, 128, 256, 10, 200, seed=34))
    cpattn.check_device()  # start clean
    bad = lens.clone()
    bad[0] = 10_000
    out = torch.empty_like(q)
    assert _call(lib, q, kc, vc, bad, out) == 0, lib.cp_attn_last_error()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.cp_attn_check_device(stream) == -6
    assert lib.cp_attn_check_device(stream) == 0


def test_noalloc_rejects_shapes_beyond_its_array():
    lib = _lib()
    q = torch.zeros(64, 32, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, dtype=torch.bfloat16, device="cuda")  # never read: rejected before launch
    lens = torch.zeros(64, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.gqa_decode_noalloc(_p(q), _p(kc), _p(kc), _p(lens), _p(out), 64, 32, 8, 32768, 128, stream)
    assert rc == -1
    assert b"scratch" in lib.cp_attn_last_error()
