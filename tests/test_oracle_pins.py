"""Pins of the float64 oracle against things fixed outside the oracle itself:
the pages' worked example, closed forms, invariants, special cases and brute
force on tiny inputs.  CPU only."""

import math
import os

import numpy as np
import pytest

from oracle import cp_attention as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng):
    return rng.standard_normal(shape)


# --------------------------------------------------------------------------
# load-balance reorder
# --------------------------------------------------------------------------

def test_page_example_order():
    """"Add context parallelism", Description: cp=2 splits tokens 0..7 as
    0,1,6,7 | 2,3,4,5."""
    lines = [l for l in open(os.path.join(GOLDEN, "lb_order_page_example.txt"))
             if l.strip() and not l.startswith("#")]
    S, cp = map(int, lines[0].split())
    shards = [list(map(int, l.split())) for l in lines[1:]]
    pos = O.lb_positions(S, cp, True)
    assert [list(pos[s * S // cp:(s + 1) * S // cp]) for s in range(cp)] == shards


def test_tiny_workload_chunk_order():
    """The tiny workload: S=256, cp=2, chunks of 64 tokens, shard 0 holds
    chunks 0 and 3, shard 1 holds chunks 1 and 2."""
    pos = O.lb_positions(256, 2, True)
    chunks = [int(pos[i * 64]) // 64 for i in range(4)]
    assert chunks == [0, 3, 1, 2]
    for i in range(4):
        assert np.array_equal(pos[i * 64:(i + 1) * 64] - pos[i * 64], np.arange(64))


def _closed_form_pos(S, cp):
    # slot j -> chunk slot k = j // c, offset t; shard s = k // 2; chunk is s
    # for the first half of a shard and 2cp-1-s for the second half
    c = S // (2 * cp)
    out = []
    for j in range(S):
        k, t = divmod(j, c)
        s = k // 2
        ch = s if k % 2 == 0 else 2 * cp - 1 - s
        out.append(ch * c + t)
    return np.array(out)


@pytest.mark.parametrize("cp", [1, 2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("mult", [1, 2, 7])
def test_positions_closed_form_and_bijection(cp, mult):
    S = 2 * cp * mult
    pos = O.lb_positions(S, cp, True)
    assert np.array_equal(pos, _closed_form_pos(S, cp))
    assert np.array_equal(np.sort(pos), np.arange(S))
    assert np.array_equal(O.lb_positions(S, cp, False), np.arange(S))


def test_cp1_is_identity():
    assert np.array_equal(O.lb_positions(12, 1, True), np.arange(12))


def test_permute_roundtrip():
    rng = np.random.default_rng(0)
    x = _rand((2, 24, 3, 5), rng)
    pos = O.lb_positions(24, 3, True)
    y = O.permute(x, pos)
    assert np.array_equal(y[:, 0], x[:, pos[0]])
    assert np.array_equal(O.unpermute(y, pos), x)
    assert np.array_equal(O.permute(O.unpermute(x, pos), pos), x)


def test_positions_reject_bad_S():
    with pytest.raises(ValueError):
        O.lb_positions(10, 2, True)


@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8])
def test_shard_work_closed_form(cp):
    """Per-shard visible pairs: shard s holds chunks s and 2cp-1-s; a chunk
    ch sees ch full earlier chunks and one causal triangle, so every shard
    does (2cp-1)c^2 + c(c+1) pairs.  Without the reorder shard i (chunks 2i,
    2i+1) does (4i+1)c^2 + c(c+1)."""
    c = 5
    S = 2 * cp * c
    bal = O.shard_pair_counts(S, cp, True)
    unbal = O.shard_pair_counts(S, cp, False)
    assert bal == [(2 * cp - 1) * c * c + c * (c + 1)] * cp
    assert unbal == [(4 * i + 1) * c * c + c * (c + 1) for i in range(cp)]
    assert sum(bal) == sum(unbal) == S * (S + 1) // 2


def test_tiny_pair_count():
    assert O.shard_pair_counts(256, 2, True) == [16448, 16448]


# --------------------------------------------------------------------------
# forward
# --------------------------------------------------------------------------

def _brute_fwd(q, k, v, qpos, kpos):
    """Literal triple loop over (batch, head, query) with math.exp."""
    B, S, Hq, Dqk = q.shape
    Sk, Hkv, Dv = k.shape[1], k.shape[2], v.shape[3]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(Dqk)
    out = np.zeros((B, S, Hq, Dv))
    lse = np.zeros((B, Hq, S))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i in range(S):
                scores = []
                for j in range(Sk):
                    if kpos[j] <= qpos[i]:
                        dot = 0.0
                        for d in range(Dqk):
                            dot += q[b, i, h, d] * k[b, j, g, d]
                        scores.append((j, scale * dot))
                mx = max(s for _, s in scores)
                wsum = sum(math.exp(s - mx) for _, s in scores)
                for j, s in scores:
                    w = math.exp(s - mx) / wsum
                    for d in range(Dv):
                        out[b, i, h, d] += w * v[b, j, g, d]
                lse[b, h, i] = mx + math.log(wsum)
    return out, lse


@pytest.mark.parametrize("Hq,Hkv,Dqk,Dv", [(2, 2, 4, 4), (4, 2, 3, 5), (2, 1, 6, 4)])
def test_fwd_brute_force(Hq, Hkv, Dqk, Dv):
    rng = np.random.default_rng(1)
    B, S = 2, 9
    q = _rand((B, S, Hq, Dqk), rng)
    k = _rand((B, S, Hkv, Dqk), rng)
    v = _rand((B, S, Hkv, Dv), rng)
    ar = np.arange(S)
    o_ref, l_ref = _brute_fwd(q, k, v, ar, ar)
    o, l = O.causal_attention_fwd(q, k, v)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, rtol=1e-12, atol=1e-12)


def test_cp_fwd_brute_force_reordered_mask():
    """Sharded attention in reordered order against the brute force run with
    the reordered positions (mask on original positions)."""
    rng = np.random.default_rng(2)
    B, S, cp = 1, 12, 3
    q = _rand((B, S, 2, 3), rng)
    k = _rand((B, S, 1, 3), rng)
    v = _rand((B, S, 1, 2), rng)
    pos = O.lb_positions(S, cp, True)
    o, l = O.cp_attention_fwd(q, k, v, cp, True)
    o_ref, l_ref = _brute_fwd(q, k, v, pos, pos)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, rtol=1e-12, atol=1e-12)


def test_probability_rows_sum_to_one():
    """With V = identity (Dv = S) the output rows ARE the attention
    probabilities: non-negative, zero above the diagonal, summing to 1, and
    equal to exp(s_ij - lse_i)."""
    rng = np.random.default_rng(3)
    S, D = 16, 8
    q = _rand((1, S, 1, D), rng)
    k = _rand((1, S, 1, D), rng)
    v = np.eye(S).reshape(1, S, 1, S)
    P, lse = O.causal_attention_fwd(q, k, v)
    P = P[0, :, 0, :]
    assert np.all(P >= 0)
    assert np.allclose(np.triu(P, 1), 0)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-13)
    s = (q[0, :, 0] @ k[0, :, 0].T) / math.sqrt(D)
    Pe = np.tril(np.exp(s - lse[0, 0][:, None]))
    np.testing.assert_allclose(P, Pe, rtol=1e-12, atol=1e-14)


def test_first_row_is_v0():
    rng = np.random.default_rng(4)
    q = _rand((2, 10, 4, 8), rng)
    k = _rand((2, 10, 2, 8), rng)
    v = _rand((2, 10, 2, 6), rng)
    o, _ = O.causal_attention_fwd(q, k, v)
    for h in range(4):
        assert np.allclose(o[:, 0, h], v[:, 0, h // 2], rtol=0, atol=1e-15)


def test_equal_keys_give_prefix_mean():
    rng = np.random.default_rng(5)
    S = 11
    q = _rand((1, S, 1, 4), rng)
    k = np.tile(_rand((1, 1, 1, 4), rng), (1, S, 1, 1))
    v = _rand((1, S, 1, 3), rng)
    o, lse = O.causal_attention_fwd(q, k, v)
    mean = np.cumsum(v[0, :, 0], axis=0) / np.arange(1, S + 1)[:, None]
    np.testing.assert_allclose(o[0, :, 0], mean, rtol=1e-12, atol=1e-13)
    # lse_i = s_i + ln(i+1) when every visible score equals s_i
    s = (q[0, :, 0] @ k[0, 0, 0]) / 2.0
    np.testing.assert_allclose(lse[0, 0], s + np.log(np.arange(1, S + 1)), rtol=1e-12)


def test_constant_v_rows():
    rng = np.random.default_rng(6)
    S = 9
    q = _rand((1, S, 2, 4), rng)
    k = _rand((1, S, 2, 4), rng)
    row = _rand((3,), rng)
    v = np.broadcast_to(row, (1, S, 2, 3)).copy()
    o, _ = O.causal_attention_fwd(q, k, v)
    np.testing.assert_allclose(o, np.broadcast_to(row, o.shape), rtol=1e-13, atol=1e-14)


def test_single_token_lse():
    rng = np.random.default_rng(7)
    q = _rand((1, 1, 1, 16), rng)
    k = _rand((1, 1, 1, 16), rng)
    v = _rand((1, 1, 1, 16), rng)
    o, lse = O.causal_attention_fwd(q, k, v)
    assert np.isclose(lse[0, 0, 0], float(q[0, 0, 0] @ k[0, 0, 0]) / 4.0, rtol=1e-14)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0])


def test_two_token_closed_form():
    """Row 1 of a 2-token sequence: a two-way softmax written out by hand."""
    rng = np.random.default_rng(8)
    D = 4
    q = _rand((1, 2, 1, D), rng)
    k = _rand((1, 2, 1, D), rng)
    v = _rand((1, 2, 1, 3), rng)
    o, lse = O.causal_attention_fwd(q, k, v)
    s0 = float(q[0, 1, 0] @ k[0, 0, 0]) / 2.0
    s1 = float(q[0, 1, 0] @ k[0, 1, 0]) / 2.0
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    np.testing.assert_allclose(o[0, 1, 0], (1 - w1) * v[0, 0, 0] + w1 * v[0, 1, 0], rtol=1e-13)
    assert math.isclose(lse[0, 0, 1], math.log(math.exp(s0) + math.exp(s1)), rel_tol=1e-14)


def test_gqa_equals_repeated_heads():
    """Grouped heads reduce to plain multi-head attention with every K/V head
    repeated Hq/Hkv times (contiguous groups)."""
    rng = np.random.default_rng(9)
    B, S, Hq, Hkv = 1, 10, 6, 2
    q = _rand((B, S, Hq, 4), rng)
    k = _rand((B, S, Hkv, 4), rng)
    v = _rand((B, S, Hkv, 3), rng)
    o, l = O.causal_attention_fwd(q, k, v)
    kr = np.repeat(k, Hq // Hkv, axis=2)
    vr = np.repeat(v, Hq // Hkv, axis=2)
    o2, l2 = O.causal_attention_fwd(q, kr, vr)
    np.testing.assert_allclose(o, o2, rtol=1e-13)
    np.testing.assert_allclose(l, l2, rtol=1e-13)
    # head 3 belongs to group 1: compare with a single-head run on group 1
    o3, _ = O.causal_attention_fwd(q[:, :, 3:4], k[:, :, 1:2], v[:, :, 1:2])
    np.testing.assert_allclose(o[:, :, 3:4], o3, rtol=1e-13)


@pytest.mark.parametrize("cp,lb", [(1, True), (2, True), (2, False), (3, True), (4, True)])
@pytest.mark.parametrize("Hq,Hkv,Dqk,Dv", [(2, 2, 8, 8), (4, 1, 6, 4)])
def test_cp_invariant_fwd(cp, lb, Hq, Hkv, Dqk, Dv):
    """The pages' unit-test criterion: the sharded, reordered computation,
    put back in natural order, equals unsharded causal attention."""
    rng = np.random.default_rng(10)
    B, S = 2, 8 * cp
    q = _rand((B, S, Hq, Dqk), rng)
    k = _rand((B, S, Hkv, Dqk), rng)
    v = _rand((B, S, Hkv, Dv), rng)
    pos = O.lb_positions(S, cp, lb)
    o_lb, l_lb = O.cp_attention_fwd(O.permute(q, pos), O.permute(k, pos),
                                    O.permute(v, pos), cp, lb)
    o, l = O.causal_attention_fwd(q, k, v)
    np.testing.assert_allclose(O.unpermute(o_lb, pos), o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l_lb[:, :, np.argsort(pos)], l, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------

def _loss(q, k, v, dout, qpos, kpos):
    o, _ = O.masked_attention_fwd(q, k, v, qpos, kpos)
    return float(np.sum(o * dout))


def _fd_grad(f, x, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = x[idx]
        x[idx] = old + eps
        fp = f()
        x[idx] = old - eps
        fm = f()
        x[idx] = old
        g[idx] = (fp - fm) / (2 * eps)
    return g


@pytest.mark.parametrize("lb", [False, True])
def test_bwd_finite_differences(lb):
    rng = np.random.default_rng(11)
    B, S, Hq, Hkv, Dqk, Dv, cp = 1, 8, 4, 2, 3, 2, 2
    q = _rand((B, S, Hq, Dqk), rng)
    k = _rand((B, S, Hkv, Dqk), rng)
    v = _rand((B, S, Hkv, Dv), rng)
    dout = _rand((B, S, Hq, Dv), rng)
    pos = O.lb_positions(S, cp, lb)
    o, l = O.cp_attention_fwd(q, k, v, cp, lb)
    dq, dk, dv = O.cp_attention_bwd(q, k, v, o, l, dout, cp, lb)
    f = lambda: _loss(q, k, v, dout, pos, pos)  # noqa: E731
    np.testing.assert_allclose(dq, _fd_grad(f, q), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dk, _fd_grad(f, k), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dv, _fd_grad(f, v), rtol=1e-6, atol=1e-8)



def _mla_brute_key(k_nope, k_rope):
    """Per-head key written out entry by entry: head h of token s is its
    nope columns, then the token's rope key."""
    B, S, H, Dn = k_nope.shape
    Dr = k_rope.shape[-1]
    k = np.zeros((B, S, H, Dn + Dr))
    for b in range(B):
        for s_ in range(S):
            for h in range(H):
                for d in range(Dn):
                    k[b, s_, h, d] = k_nope[b, s_, h, d]
                for d in range(Dr):
                    k[b, s_, h, Dn + d] = k_rope[b, s_, d]
    return k


@pytest.mark.parametrize("lb", [False, True])
def test_mla_shared_rope_key(lb):
    """MLA with one rope key per token shared by the heads: the forward equals
    brute-force attention with that key written out per head, and the
    gradients (above all the rope key's, which collects every head's
    contribution) match finite differences of sum(out * dout)."""
    rng = np.random.default_rng(21)
    B, S, H, Dn, Dr, Dv, cp = 1, 8, 3, 3, 2, 2, 2
    q = _rand((B, S, H, Dn + Dr), rng)
    kn = _rand((B, S, H, Dn), rng)
    kr = _rand((B, S, Dr), rng)
    v = _rand((B, S, H, Dv), rng)
    dout = _rand((B, S, H, Dv), rng)
    pos = O.lb_positions(S, cp, lb)
    o, l = O.cp_attention_mla_fwd(q, kn, kr, v, cp, lb)
    ob, lbr = _brute_fwd(q, _mla_brute_key(kn, kr), v, pos, pos)
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l, lbr, rtol=1e-12, atol=1e-12)
    dq, dkn, dkr, dv = O.cp_attention_mla_bwd(q, kn, kr, v, o, l, dout, cp, lb)
    assert dkr.shape == (B, S, Dr) and dkn.shape == (B, S, H, Dn)
    f = lambda: float(np.sum(_brute_fwd(q, _mla_brute_key(kn, kr), v, pos, pos)[0] * dout))  # noqa: E731
    np.testing.assert_allclose(dkr, _fd_grad(f, kr), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dkn, _fd_grad(f, kn), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dq, _fd_grad(f, q), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dv, _fd_grad(f, v), rtol=1e-6, atol=1e-8)


def test_bwd_shift_invariants():
    """Adding one vector to every key shifts each row of scores by a
    constant, so sum_j dk_j = 0; adding one vector c to every value adds c
    to every output row, so sum_j dv_j = sum_i dout_i (per KV group)."""
    rng = np.random.default_rng(12)
    B, S, Hq, Hkv = 2, 20, 4, 2
    q = _rand((B, S, Hq, 5), rng)
    k = _rand((B, S, Hkv, 5), rng)
    v = _rand((B, S, Hkv, 3), rng)
    dout = _rand((B, S, Hq, 3), rng)
    o, l = O.causal_attention_fwd(q, k, v)
    dq, dk, dv = O.causal_attention_bwd(q, k, v, o, l, dout)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    want = dout.reshape(B, S, Hkv, Hq // Hkv, 3).sum(axis=(1, 3))
    np.testing.assert_allclose(dv.sum(axis=1), want, rtol=1e-12, atol=1e-12)
    # scaling q by a and the softmax scale by 1/a leaves the output fixed:
    # sum(q * dq) is the derivative along that direction's partner, which is
    # sum over scores of s * dS = sum(k * dk) (both equal d/d(scale))
    np.testing.assert_allclose(np.sum(q * dq), np.sum(k * dk), rtol=1e-10)


@pytest.mark.parametrize("cp,lb", [(2, True), (3, True), (2, False)])
def test_cp_invariant_bwd(cp, lb):
    rng = np.random.default_rng(13)
    B, S, Hq, Hkv, Dqk, Dv = 1, 12 * cp, 4, 2, 6, 4
    q = _rand((B, S, Hq, Dqk), rng)
    k = _rand((B, S, Hkv, Dqk), rng)
    v = _rand((B, S, Hkv, Dv), rng)
    dout = _rand((B, S, Hq, Dv), rng)
    pos = O.lb_positions(S, cp, lb)
    P = lambda x: O.permute(x, pos)  # noqa: E731
    o_lb, l_lb = O.cp_attention_fwd(P(q), P(k), P(v), cp, lb)
    g_lb = O.cp_attention_bwd(P(q), P(k), P(v), o_lb, l_lb, P(dout), cp, lb)
    o, l = O.causal_attention_fwd(q, k, v)
    g = O.causal_attention_bwd(q, k, v, o, l, dout)
    for a, b in zip(g_lb, g):
        np.testing.assert_allclose(O.unpermute(a, pos), b, rtol=1e-11, atol=1e-12)


def test_gqa_bwd_equals_repeated_heads():
    rng = np.random.default_rng(14)
    B, S, Hq, Hkv = 1, 9, 4, 2
    q = _rand((B, S, Hq, 4), rng)
    k = _rand((B, S, Hkv, 4), rng)
    v = _rand((B, S, Hkv, 3), rng)
    dout = _rand((B, S, Hq, 3), rng)
    o, l = O.causal_attention_fwd(q, k, v)
    dq, dk, dv = O.causal_attention_bwd(q, k, v, o, l, dout)
    kr = np.repeat(k, 2, axis=2)
    vr = np.repeat(v, 2, axis=2)
    o2, l2 = O.causal_attention_fwd(q, kr, vr)
    dq2, dk2, dv2 = O.causal_attention_bwd(q, kr, vr, o2, l2, dout)
    np.testing.assert_allclose(dq, dq2, rtol=1e-12)
    np.testing.assert_allclose(dk, dk2.reshape(B, S, Hkv, 2, 4).sum(axis=3), rtol=1e-12)
    np.testing.assert_allclose(dv, dv2.reshape(B, S, Hkv, 2, 3).sum(axis=3), rtol=1e-12)


# --------------------------------------------------------------------------
# decode
# --------------------------------------------------------------------------

def test_decode_brute_force():
    rng = np.random.default_rng(15)
    B, Hq, Hkv, D, Smax = 3, 4, 2, 5, 7
    q = _rand((B, Hq, D), rng)
    kc = _rand((B, Hkv, Smax, D), rng)
    vc = _rand((B, Hkv, Smax, D), rng)
    lens = np.array([7, 1, 4])
    out = O.gqa_decode(q, kc, vc, lens)
    for b in range(B):
        for h in range(Hq):
            g = h // 2
            s = [sum(q[b, h, d] * kc[b, g, t, d] for d in range(D)) / math.sqrt(D)
                 for t in range(lens[b])]
            mx = max(s)
            w = [math.exp(x - mx) for x in s]
            ref = [sum(w[t] * vc[b, g, t, d] for t in range(lens[b])) / sum(w)
                   for d in range(D)]
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-12, atol=1e-14)


def test_decode_is_last_row_of_causal():
    """Decoding the token at position n-1 against a cache of n keys equals
    row n-1 of causal attention over those n tokens."""
    rng = np.random.default_rng(16)
    Hq, Hkv, D, n = 4, 2, 8, 13
    q_all = _rand((1, n, Hq, D), rng)
    k = _rand((1, n, Hkv, D), rng)
    v = _rand((1, n, Hkv, D), rng)
    o, _ = O.causal_attention_fwd(q_all, k, v)
    Smax = 16
    kc = np.zeros((1, Hkv, Smax, D))
    vc = np.zeros((1, Hkv, Smax, D))
    kc[0, :, :n] = k[0].transpose(1, 0, 2)
    vc[0, :, :n] = v[0].transpose(1, 0, 2)
    kc[0, :, n:] = 1e3  # garbage past the valid length must be ignored
    out = O.gqa_decode(q_all[:, n - 1], kc, vc, np.array([n]))
    np.testing.assert_allclose(out[0], o[0, n - 1], rtol=1e-12, atol=1e-13)


def test_decode_zero_length_is_zero():
    rng = np.random.default_rng(17)
    out = O.gqa_decode(_rand((2, 2, 4), rng), _rand((2, 1, 3, 4), rng),
                       _rand((2, 1, 3, 4), rng), np.array([0, 3]))
    assert np.all(out[0] == 0)
    assert np.any(out[1] != 0)


# ---------------------------------------------------------------------------
# int8 KV-cache decode
# ---------------------------------------------------------------------------

def _int8_case(seed, B=2, Hq=4, Hkv=2, D=8, Smax=6):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, D))
    kq = rng.integers(-127, 128, (B, Hkv, Smax, D))
    vq = rng.integers(-127, 128, (B, Hkv, Smax, D))
    ks = rng.uniform(0.008, 0.016, (B, Hkv, Smax))
    vs = rng.uniform(0.008, 0.016, (B, Hkv, Smax))
    lens = np.array([Smax, 3][:B])
    return q, kq, vq, ks, vs, lens


def test_decode_int8_brute_force():
    """Element by element: dequantise each cached value, score, softmax, sum."""
    q, kq, vq, ks, vs, lens = _int8_case(31)
    B, Hq, D = q.shape
    Hkv = kq.shape[1]
    G = Hq // Hkv
    got = O.gqa_decode_int8(q, kq, vq, ks, vs, lens)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            sc = []
            for t in range(int(lens[b])):
                acc = 0.0
                for d in range(D):
                    acc += q[b, h, d] * (float(kq[b, g, t, d]) * ks[b, g, t])
                sc.append(acc / math.sqrt(D))
            m = max(sc)
            w = [math.exp(x - m) for x in sc]
            for d in range(D):
                num = sum(w[t] * float(vq[b, g, t, d]) * vs[b, g, t] for t in range(len(w)))
                assert abs(got[b, h, d] - num / sum(w)) < 1e-12


def test_decode_int8_value_scale_is_linear():
    q, kq, vq, ks, vs, lens = _int8_case(32)
    a = O.gqa_decode_int8(q, kq, vq, ks, vs, lens)
    b = O.gqa_decode_int8(q, kq, vq, ks, 3.0 * vs, lens)
    np.testing.assert_allclose(b, 3.0 * a, rtol=1e-12, atol=1e-14)


def test_decode_int8_key_scale_acts_like_query_scale():
    """A common factor on every key scale multiplies the scores, exactly as the
    same factor on the query does."""
    q, kq, vq, ks, vs, lens = _int8_case(33)
    a = O.gqa_decode_int8(q, kq, vq, 2.5 * ks, vs, lens)
    b = O.gqa_decode_int8(2.5 * q, kq, vq, ks, vs, lens)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------
# absorbed-MLA decode
# --------------------------------------------------------------------------

def test_mla_decode_brute_force():
    """Element-by-element loops on a tiny latent cache."""
    rng = np.random.default_rng(41)
    B, H, Dk, Dv, Smax = 2, 3, 8, 6, 5
    q = _rand((B, H, Dk), rng)
    ckv = _rand((B, Smax, Dk), rng)
    lens = [5, 3]
    sc = 0.37
    got = O.mla_decode(q, ckv, lens, dv=Dv, scale=sc)
    for b in range(B):
        for h in range(H):
            sc_t = [sc * sum(q[b, h, i] * ckv[b, t, i] for i in range(Dk)) for t in range(lens[b])]
            mx = max(sc_t)
            w = [math.exp(x - mx) for x in sc_t]
            for d in range(Dv):
                want = sum(w[t] * ckv[b, t, d] for t in range(lens[b])) / sum(w)
                assert abs(got[b, h, d] - want) < 1e-12


def test_mla_decode_equals_unabsorbed_mla():
    """The absorbed form against MLA written out per head: key of head h at
    position t = (its nope key W_uk[h] c_t, the token's rope key r_t), value =
    W_uv[h] c_t, query = (q_nope[h], q_rope[h]).  Decoding that per-head cache
    with the plain GQA decode and projecting the latent output with W_uv
    must agree: q_nope . (W_uk c) = (W_uk^T q_nope) . c by associativity."""
    rng = np.random.default_rng(42)
    B, H, Dc, Dr, Dn, Smax = 2, 4, 16, 4, 6, 9
    lens = np.array([9, 4])
    c = _rand((B, Smax, Dc), rng)
    r = _rand((B, Smax, Dr), rng)
    w_uk = _rand((H, Dn, Dc), rng)
    w_uv = _rand((H, Dn, Dc), rng)
    q_nope = _rand((B, H, Dn), rng)
    q_rope = _rand((B, H, Dr), rng)
    sc = 1.0 / math.sqrt(Dn + Dr)
    # written out per head
    k_full = np.concatenate([np.einsum("hnc,bsc->bhsn", w_uk, c), np.broadcast_to(r[:, None], (B, H, Smax, Dr))],
                            axis=-1)
    v_full = np.einsum("hnc,bsc->bhsn", w_uv, c)
    q_full = np.concatenate([q_nope, q_rope], axis=-1)
    want = O.gqa_decode(q_full, k_full, v_full, lens, scale=sc)
    # absorbed
    q_abs = np.concatenate([np.einsum("hnc,bhn->bhc", w_uk, q_nope), q_rope], axis=-1)
    ckv = np.concatenate([c, r], axis=-1)
    lat = O.mla_decode(q_abs, ckv, lens, dv=Dc, scale=sc)
    got = np.einsum("hnc,bhc->bhn", w_uv, lat)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_mla_decode_special_lengths():
    """lens = 0 gives zeros; lens = 1 gives the first token's value exactly;
    the default scale is 1/sqrt(192)."""
    rng = np.random.default_rng(43)
    q = _rand((2, 3, 10), rng)
    ckv = _rand((2, 4, 10), rng)
    out = O.mla_decode(q, ckv, [0, 1], dv=7)
    assert np.all(out[0] == 0)
    assert np.array_equal(out[1], np.broadcast_to(ckv[1, 0, :7], (3, 7)))
    a = O.mla_decode(q, ckv, [4, 4], dv=7)
    b = O.mla_decode(q, ckv, [4, 4], dv=7, scale=1.0 / math.sqrt(192.0))
    assert np.array_equal(a, b)
