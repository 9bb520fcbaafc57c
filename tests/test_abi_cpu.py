"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function the header declares, and its host-side helpers and argument
checks behave (no CUDA compute call is made)."""

import ctypes

import numpy as np
import pytest

from oracle import cp_attention as O
from tests._lib import built_lib, header_functions

lib = None


def setup_module(_):
    global lib
    lib = built_lib()


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert {"cp_lb_permute", "cp_lb_unpermute", "cp_attn_fwd", "cp_attn_bwd", "gqa_decode"} <= set(names)
    for n in names:
        assert hasattr(lib, n), "libcpattn.so does not export %s" % n


@pytest.mark.parametrize("S,cp,lb", [(8, 2, 1), (256, 2, 1), (8192, 4, 1), (96, 3, 1), (64, 4, 0), (12, 1, 1)])
def test_positions_match_oracle(S, cp, lb):
    arr = (ctypes.c_int * S)()
    assert lib.cp_lb_positions(S, cp, lb, arr) == 0
    assert np.array_equal(np.array(arr), O.lb_positions(S, cp, bool(lb)))


def _tile_counts(S, cp, lb):
    arr = (ctypes.c_longlong * cp)()
    assert lib.cp_attn_tile_counts(S, cp, lb, arr) == 0
    return list(arr)


@pytest.mark.parametrize("cp,m", [(2, 1), (4, 8), (8, 4), (3, 2)])
def test_tile_counts_closed_form(cp, m):
    """With c = 128m every shard visits (2cp-1)m^2 + m(m+1) (query, key)
    tile pairs; without the reorder shard i visits 4m^2 i + m(2m+1)."""
    S = 2 * cp * 128 * m
    assert _tile_counts(S, cp, 1) == [(2 * cp - 1) * m * m + m * (m + 1)] * cp
    assert _tile_counts(S, cp, 0) == [4 * m * m * i + m * (2 * m + 1) for i in range(cp)]


def test_tile_counts_llama2_workload():
    # 8192 tokens, cp=4: 520 tile pairs per shard balanced; 136..904 unbalanced
    assert _tile_counts(8192, 4, 1) == [520] * 4
    assert _tile_counts(8192, 4, 0) == [136, 392, 648, 904]


def _err():
    return lib.cp_attn_last_error().decode()


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: argument checks fail first


def test_bad_arguments_are_rejected_on_host():
    P = FAKE
    # permute: S not a multiple of 2cp, in place, null
    assert lib.cp_lb_permute(P, ctypes.c_void_p(0x2000000), 1, 10, 16, 2, None) == -1
    assert "2*cp" in _err()
    assert lib.cp_lb_permute(P, P, 1, 16, 16, 2, None) == -1
    assert lib.cp_lb_permute(None, P, 1, 16, 16, 2, None) == -1
    # attention: Hq % Hkv, S % 2cp, head dims, misaligned pointer
    args = [P] * 5
    assert lib.cp_attn_fwd(*args, 1, 6, 4, 256, 128, 128, 2, 1, None) == -1
    assert "multiple of Hkv" in _err()
    assert lib.cp_attn_fwd(*args, 1, 4, 4, 250, 128, 128, 2, 1, None) == -1
    assert lib.cp_attn_fwd(*args, 1, 4, 4, 256, 96, 96, 2, 1, None) == -2
    assert lib.cp_attn_fwd(ctypes.c_void_p(0x1008), *args[1:], 1, 4, 4, 256, 128, 128, 2, 1, None) == -1
    assert "aligned" in _err()
    assert lib.cp_attn_fwd_shard(*args, 1, 4, 4, 256, 128, 128, 2, 1, 2, None) == -1
    assert lib.cp_attn_bwd(*([P] * 9), 1, 4, 4, 256, 64, 128, 2, 1, None) == -2
    # load_balance outside {0, 1, 2}; zero-copy needs whole 128-row tiles per chunk
    assert lib.cp_attn_fwd(*args, 1, 4, 4, 256, 128, 128, 2, 3, None) == -1
    assert lib.cp_attn_fwd(*args, 1, 4, 4, 320, 128, 128, 2, 2, None) == -2
    assert "zero-copy" in _err()
    assert lib.cp_attn_bwd(*([P] * 9), 1, 4, 4, 768, 128, 128, 2, 2, None) == -2
    # per-shard backward: shard out of range
    assert lib.cp_attn_bwd_shard(*([P] * 9), 1, 4, 4, 256, 128, 128, 2, 1, 2, P, P, None) == -1
    # MLA with shared rope keys: null rope keys, S not a multiple of 2cp, misaligned pointer
    assert lib.cp_attn_fwd_mla(P, P, None, P, P, P, 1, 4, 256, 2, 1, None) == -1
    assert lib.cp_attn_fwd_mla(P, P, ctypes.c_void_p(0x1008), P, P, P, 1, 4, 256, 2, 1, None) == -1
    assert "aligned" in _err()
    assert lib.cp_attn_fwd_mla(P, P, P, P, P, P, 1, 4, 250, 2, 1, None) == -1
    assert lib.cp_attn_bwd_mla(*([P] * 11), 1, 4, 250, 2, 1, None) == -1
    assert lib.cp_attn_bwd_mla(P, P, None, *([P] * 8), 1, 4, 256, 2, 1, None) == -1
    assert lib.cp_attn_bwd_mla(P, ctypes.c_void_p(0x1008), *([P] * 9), 1, 4, 256, 2, 1, None) == -1
    assert "aligned" in _err()
    # decode: group too large, bad head dim, null lens
    assert lib.gqa_decode(P, P, P, P, P, 1, 64, 2, 128, 128, None) == -2
    assert lib.gqa_decode(P, P, P, P, P, 1, 8, 2, 128, 96, None) == -2
    assert lib.gqa_decode(P, P, P, None, P, 1, 8, 2, 128, 128, None) == -1
    # int8 decode: head dim, null scales
    assert lib.gqa_decode_int8(P, P, P, P, P, P, P, 1, 8, 2, 128, 64, None) == -2
    assert lib.gqa_decode_int8(P, P, P, None, P, P, P, 1, 8, 2, 128, 128, None) == -1


def _schedule(B, Hq, Hkv, S, cp, lb, n):
    arr = (ctypes.c_longlong * n)()
    assert lib.cp_attn_fwd_schedule(B, Hq, Hkv, S, cp, lb, n, arr) == 0, _err()
    return list(arr)


def test_fwd_schedule_by_hand():
    """S = 256 with one head: the two 128-row query tiles form one unit that
    walks both key tiles, cost (2 steps + 4) x 2 tiles, on the first CTA."""
    assert _schedule(1, 1, 1, 256, 2, 0, 4) == [12, 0, 0, 0]
    assert _schedule(1, 1, 1, 256, 2, 1, 4) == [12, 0, 0, 0]
    # one more query tile (S = 384, natural order): units (tiles 0,1) and (tile 2)
    assert sorted(_schedule(1, 1, 1, 384, 1, 0, 2)) == [7, 12]


@pytest.mark.parametrize("B,Hq,Hkv,S,cp", [(1, 32, 32, 8192, 4), (4, 32, 32, 8192, 4), (1, 64, 8, 16384, 8)])
def test_fwd_schedule_balance(B, Hq, Hkv, S, cp):
    """Every CTA gets work, the total does not depend on how many CTAs share
    it, the plan is deterministic, and with several units per CTA the most
    loaded CTA is within 3% of the mean."""
    c152 = _schedule(B, Hq, Hkv, S, cp, 1, 152)
    assert min(c152) > 0
    total = sum(c152)
    assert sum(_schedule(B, Hq, Hkv, S, cp, 1, 100)) == total
    assert _schedule(B, Hq, Hkv, S, cp, 1, 1) == [total]
    assert _schedule(B, Hq, Hkv, S, cp, 1, 152) == c152
    assert max(c152) <= 1.03 * total / 152


def test_fwd_schedule_by_head_for_many_heads():
    """128 KV heads (the DeepSeek-V3-shaped MLA layer): the units are dealt
    one head after the other; the total is unchanged, the plan deterministic,
    and the most loaded CTA still within 3% of the mean."""
    c152 = _schedule(1, 128, 128, 32768, 4, 1, 152)
    total = sum(c152)
    assert min(c152) > 0
    assert _schedule(1, 128, 128, 32768, 4, 1, 1) == [total]
    assert _schedule(1, 128, 128, 32768, 4, 1, 152) == c152
    assert max(c152) <= 1.03 * total / 152


@pytest.mark.parametrize("B,Hq,Hkv,S,cp", [(1, 128, 128, 32768, 4), (1, 64, 8, 131072, 8)])
def test_fwd_shard_schedules_balance(B, Hq, Hkv, S, cp):
    """Every shard's plan on its own: the shards' totals agree (balanced
    reorder) and each plan's most loaded CTA is within 3% of its mean (one
    shard's units mix a first and a last chunk, so their costs are far
    apart: the small ones must still even out the deal)."""
    totals = []
    for shard in range(cp):
        arr = (ctypes.c_longlong * 152)()
        assert lib.cp_attn_fwd_shard_schedule(B, Hq, Hkv, S, cp, 1, shard, 152, arr) == 0, _err()
        c = list(arr)
        totals.append(sum(c))
        assert max(c) <= 1.03 * sum(c) / 152, "shard %d: %d vs mean %.1f" % (shard, max(c), sum(c) / 152)
    assert max(totals) <= 1.01 * min(totals)
    arr = (ctypes.c_longlong * 152)()
    assert lib.cp_attn_fwd_shard_schedule(B, Hq, Hkv, S, cp, 1, cp, 152, arr) == -1


def test_fwd_schedule_rejects_bad_arguments():
    arr = (ctypes.c_longlong * 4)()
    assert lib.cp_attn_fwd_schedule(1, 1, 1, 256, 2, 1, 0, arr) == -1
    assert lib.cp_attn_fwd_schedule(1, 1, 1, 250, 2, 1, 4, arr) == -1
    assert lib.cp_attn_fwd_schedule(1, 1, 1, 256, 2, 1, 4, None) == -1


def test_binding_checks_tensors_before_the_library():
    """The Python binding refuses host tensors, wrong dtypes and wrong MLA
    shapes itself (no device is needed to see it)."""
    import torch

    from context_causal_attention_load_gb300 import cpattn
    q = torch.zeros(1, 256, 2, 192, dtype=torch.bfloat16)
    kn = torch.zeros(1, 256, 2, 128, dtype=torch.bfloat16)
    kr = torch.zeros(1, 256, 64, dtype=torch.bfloat16)
    v = torch.zeros(1, 256, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        cpattn.attn_fwd_mla(q, kn, kr, v, 2)
    with pytest.raises(ValueError, match="CUDA"):
        cpattn.attn_fwd(q, kn, v, 2)
    with pytest.raises(ValueError):
        cpattn.fwd_schedule(1, 1, 1, 256, 2, 3, 4)  # load_balance must be 0, 1 or 2
    assert cpattn.fwd_schedule(1, 1, 1, 256, 2, True, 2) == [12, 0]


def test_stall_hook_checks_its_limit():
    """The timeout test hook takes a wait limit of 1e5..4e9 cycles; clearing
    it is always accepted (host state only, no device work)."""
    from context_causal_attention_load_gb300 import cpattn
    assert lib.cp_attn_test_stall_forward(0, 10) == -1
    assert lib.cp_attn_test_stall_forward(0, 10 ** 10) == -1
    assert lib.cp_attn_test_stall_forward(-1, 0) == 0
    cpattn.test_stall_forward(-1)
