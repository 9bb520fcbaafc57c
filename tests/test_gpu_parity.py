"""Parity of the CUDA path (through the C ABI) with the float64 oracle on the
same seeded bf16 inputs.  Needs a GB300."""

import numpy as np
import pytest
import torch

from context_causal_attention_load_gb300 import synth
from oracle import cp_attention as O
from tests._lib import assert_close_grad, assert_close_out, built_lib

pytestmark = pytest.mark.gpu

cp_ = None


def setup_module(_):
    global cp_
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    built_lib()
    from context_causal_attention_load_gb300 import cpattn
    cp_ = cpattn


def _f64(t):
    return synth.to_f64(t)


def _run_fwd(B, S, Hq, Hkv, Dqk, Dv, cp, lb, seed=0, q_scale=1.0, v_override=None):
    q, k, v, dout = synth.attention_inputs(B, S, Hq, Hkv, Dqk, Dv, seed=seed, q_scale=q_scale)
    if v_override is not None:
        v = v_override
    pos = O.lb_positions(S, cp, lb)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    if lb:
        qd, kd, vd = cp_.lb_permute(qd, cp), cp_.lb_permute(kd, cp), cp_.lb_permute(vd, cp)
    out, lse = cp_.attn_fwd(qd, kd, vd, cp, lb)
    torch.cuda.synchronize()
    cp_.check_device()
    # oracle in slot order on the same bf16 values
    qs, ks, vs = (O.permute(_f64(x), pos) for x in (q, k, v))
    o_ref, l_ref = O.cp_attention_fwd(qs, ks, vs, cp, lb)
    return dict(q=q, k=k, v=v, dout=dout, qd=qd, kd=kd, vd=vd, out=out, lse=lse, o_ref=o_ref,
                l_ref=l_ref, pos=pos)


def _check_fwd(r, name):
    assert_close_out(_f64(r["out"]), r["o_ref"], name + " out")
    lse = r["lse"].cpu().numpy().astype(np.float64)
    err = float(np.max(np.abs(lse - r["l_ref"])))
    assert err <= 1e-2, "%s lse max-abs %.3e" % (name, err)


# ---------------------------------------------------------------------------
# permutation: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,S,cp,row", [(2, 256, 2, 128), (1, 96, 3, 6), (3, 64, 4, 3), (1, 8192, 4, 8192)])
def test_permute_bit_exact(B, S, cp, row):
    g = torch.Generator().manual_seed(B * 1000 + S)
    x = torch.randint(0, 256, (B, S, row), generator=g, dtype=torch.uint8)
    pos = O.lb_positions(S, cp, True)
    y = cp_.lb_permute(x.cuda(), cp)
    assert torch.equal(y.cpu(), torch.from_numpy(O.permute(x.numpy(), pos)))
    z = cp_.lb_unpermute(y, cp)
    assert torch.equal(z.cpu(), x)


def test_permute_bf16_page_example():
    # 8 tokens, cp=2: slots hold tokens 0,1,6,7,2,3,4,5
    x = torch.arange(8, dtype=torch.float32).to(torch.bfloat16).reshape(1, 8, 1).repeat(1, 1, 8).cuda()
    y = cp_.lb_permute(x, 2)
    assert y[0, :, 0].float().cpu().tolist() == [0, 1, 6, 7, 2, 3, 4, 5]


# ---------------------------------------------------------------------------
# forward
# ---------------------------------------------------------------------------

def test_fwd_identity_v_exposes_probabilities():
    """V = identity (128 keys, Dv = 128): out row i is row i of the causal
    attention probability matrix."""
    S = 128
    v = torch.eye(S, dtype=torch.float32).reshape(1, S, 1, S).to(torch.bfloat16)
    r = _run_fwd(1, S, 1, 1, 128, 128, 1, False, seed=3, v_override=v)
    got = _f64(r["out"])[0, :, 0, :]
    want = r["o_ref"][0, :, 0, :]
    err = np.abs(got - want)
    assert float(err.max()) <= 2e-2, "max err %.3e at %s" % (err.max(), np.unravel_index(err.argmax(), err.shape))
    _check_fwd(r, "identity-v")


@pytest.mark.parametrize("cfg", [
    # B, S, Hq, Hkv, Dqk, Dv, cp, lb
    (1, 256, 2, 2, 64, 64, 2, True),      # the tiny workload (chunks of 64)
    (1, 256, 2, 2, 64, 64, 2, False),
    (2, 512, 4, 4, 128, 128, 2, True),
    (1, 1024, 8, 2, 128, 128, 4, True),   # GQA
    (1, 320, 4, 2, 128, 128, 2, True),    # ragged: chunks of 80, last tile partial
    (2, 200, 2, 1, 128, 128, 1, True),    # cp=1, S not a multiple of 128
    (1, 384, 2, 2, 192, 128, 2, True),    # MLA head dims
    (1, 768, 6, 3, 128, 128, 3, True),    # odd cp, group of 2
    (1, 512, 3, 1, 64, 64, 4, True),      # odd group size (3 heads per KV head)
])
def test_fwd_parity(cfg):
    r = _run_fwd(*cfg)
    _check_fwd(r, "fwd%s" % (cfg,))


def test_fwd_cp_invariant():
    """The pages' criterion: permute -> sharded attention -> unpermute equals
    unsharded causal attention computed in natural order."""
    B, S, H, D, cp = 1, 1024, 4, 128, 4
    r = _run_fwd(B, S, H, H, D, D, cp, True, seed=5)
    nat = cp_.lb_unpermute(r["out"], cp)
    o_nat, _ = O.causal_attention_fwd(_f64(r["q"]), _f64(r["k"]), _f64(r["v"]))
    assert_close_out(_f64(nat), o_nat, "unpermuted out")


def test_fwd_shards_partition_the_rows():
    B, S, H, D, cp = 1, 1024, 2, 128, 4
    r = _run_fwd(B, S, H, H, D, D, cp, True, seed=6)
    full = r["out"].clone()
    acc = torch.zeros_like(full)
    for s in range(cp):
        out = torch.full_like(full, float("nan"))
        lse = torch.empty_like(r["lse"])
        cp_.attn_fwd_shard(r["qd"], r["kd"], r["vd"], cp, s, True, out, lse)
        torch.cuda.synchronize()
        rows = slice(s * S // cp, (s + 1) * S // cp)
        assert torch.equal(out[:, rows], full[:, rows])
        acc[:, rows] = out[:, rows]
    assert torch.equal(acc, full)


def test_fwd_deterministic():
    r = _run_fwd(1, 512, 4, 2, 128, 128, 2, True, seed=7)
    out2, lse2 = cp_.attn_fwd(r["qd"], r["kd"], r["vd"], 2, True)
    assert torch.equal(out2, r["out"]) and torch.equal(lse2, r["lse"])


# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg", [
    (1, 256, 2, 2, 64, 64, 2, True),
    (1, 512, 4, 4, 128, 128, 2, True),
    (1, 1024, 8, 2, 128, 128, 4, True),
    (1, 320, 4, 2, 128, 128, 2, True),
    (2, 200, 2, 1, 128, 128, 1, True),
    (1, 384, 2, 2, 192, 128, 2, True),    # MLA head dims: the fused MLA kernel
    (1, 512, 4, 4, 128, 128, 4, False),
    (1, 640, 4, 2, 192, 128, 2, True),    # MLA dims, two query heads per KV head, chunks of 160
    (2, 200, 2, 2, 192, 128, 1, False),   # MLA dims, S not a multiple of 64: the last half-tile partial
])
def test_bwd_parity(cfg):
    B, S, Hq, Hkv, Dqk, Dv, cp, lb = cfg
    r = _run_fwd(*cfg, seed=11)
    doutd = r["dout"].cuda()
    if lb:
        doutd = cp_.lb_permute(doutd, cp)
    dq, dk, dv = cp_.attn_bwd(r["qd"], r["kd"], r["vd"], r["out"], r["lse"], doutd, cp, lb)
    torch.cuda.synchronize()
    cp_.check_device()
    pos = r["pos"]
    qs, ks, vs, ds = (O.permute(_f64(x), pos) for x in (r["q"], r["k"], r["v"], r["dout"]))
    # the oracle's backward runs on its own forward output (no GPU value enters it)
    g_ref = O.cp_attention_bwd(qs, ks, vs, r["o_ref"], r["l_ref"], ds, cp, lb)
    for got, want, name in zip((dq, dk, dv), g_ref, ("dq", "dk", "dv")):
        assert_close_grad(_f64(got), want, "%s %s" % (name, cfg))


@pytest.mark.parametrize("cfg", [
    (1, 512, 4, 2, 128, 128, 4, True),    # shards of 128 rows: every tile inside one shard
    (1, 320, 4, 2, 128, 128, 2, True),    # shards of 160 rows: tiles straddle the boundary
    (2, 256, 2, 2, 64, 64, 2, True),
    (1, 384, 2, 1, 128, 128, 3, False),   # natural order
    (1, 512, 2, 2, 192, 128, 2, True),    # MLA head dims (per shard: the two-kernel backward)
    (1, 480, 2, 2, 192, 128, 3, True),    # MLA, shards of 160 rows: 64-row steps straddle the boundary
])
def test_bwd_shard_partials(cfg):
    """Per-shard backward against the oracle on that shard's rows; the shards'
    dk/dv partials add up to the full backward's dk/dv."""
    B, S, Hq, Hkv, Dqk, Dv, cp, lb = cfg
    r = _run_fwd(*cfg, seed=13)
    doutd = r["dout"].cuda()
    if lb:
        doutd = cp_.lb_permute(doutd, cp)
    pos = r["pos"]
    qs, ks, vs, ds = (O.permute(_f64(x), pos) for x in (r["q"], r["k"], r["v"], r["dout"]))
    _, dk_full, dv_full = cp_.attn_bwd(r["qd"], r["kd"], r["vd"], r["out"], r["lse"], doutd, cp, lb)
    dk_sum = torch.zeros(r["kd"].shape, dtype=torch.float64)
    dv_sum = torch.zeros(r["vd"].shape, dtype=torch.float64)
    for s in range(cp):
        dq, dkp, dvp = cp_.attn_bwd_shard(r["qd"], r["kd"], r["vd"], r["out"], r["lse"], doutd, cp, s, lb)
        torch.cuda.synchronize()
        cp_.check_device()
        rows = slice(s * S // cp, (s + 1) * S // cp)
        dq_s, dk_s, dv_s = O.masked_attention_bwd(qs[:, rows], ks, vs, r["o_ref"][:, rows], r["l_ref"][:, :, rows],
                                                  ds[:, rows], pos[rows], pos)
        dqh = _f64(dq)
        assert_close_grad(dqh[:, rows], dq_s, "dq shard %d %s" % (s, cfg))
        outside = np.ones(S, bool)
        outside[rows] = False
        assert np.all(dqh[:, outside] == 0), "dq outside shard %d" % s
        assert_close_grad(_f64(dkp), dk_s, "dk part %d %s" % (s, cfg))
        assert_close_grad(_f64(dvp), dv_s, "dv part %d %s" % (s, cfg))
        dk_sum += dkp.cpu().double()
        dv_sum += dvp.cpu().double()
    assert_close_grad(dk_sum.numpy(), _f64(dk_full), "sum of dk parts %s" % (cfg,))
    assert_close_grad(dv_sum.numpy(), _f64(dv_full), "sum of dv parts %s" % (cfg,))


@pytest.mark.parametrize("cfg", [
    (1, 512, 4, 2, 128, 128, 4, True),
    (2, 256, 2, 2, 64, 64, 2, True),
])
def test_bwd_shard_bf16_copy_is_the_rounded_partial(cfg):
    """Asked for them, one shard's backward also writes its dk/dv contributions
    rounded to bf16: bit for bit the fp32 partials rounded to nearest even
    (zero for the keys the shard does not touch)."""
    B, S, Hq, Hkv, Dqk, Dv, cp, lb = cfg
    r = _run_fwd(*cfg, seed=14)
    doutd = cp_.lb_permute(r["dout"].cuda(), cp)
    for s in range(cp):
        dk = torch.empty_like(r["kd"])
        dv = torch.empty_like(r["vd"])
        _, dkp, dvp = cp_.attn_bwd_shard(r["qd"], r["kd"], r["vd"], r["out"], r["lse"], doutd, cp, s, lb,
                                         dk=dk, dv=dv)
        torch.cuda.synchronize()
        cp_.check_device()
        assert torch.equal(dk, dkp.to(torch.bfloat16)), "dk bf16 copy, shard %d %s" % (s, cfg)
        assert torch.equal(dv, dvp.to(torch.bfloat16)), "dv bf16 copy, shard %d %s" % (s, cfg)


def test_bwd_shard_rejects_natural_order():
    """The per-shard backward takes tensors in slot order only."""
    B, S, H, cp = 1, 256, 1, 2
    q = torch.zeros(B, S, H, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(B, S, H, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, H, S, dtype=torch.float32, device="cuda")
    with pytest.raises(cp_.CpAttnError) as e:
        cp_.attn_bwd_shard(q, q, q, out, lse, out, cp, 0, 2)
    assert e.value.code == -2


@pytest.mark.parametrize("cfg", [
    # B, S, Hq, Hkv, Dqk, Dv, cp: chunk lengths S/(2cp) of 128, 512 and 256 rows
    (1, 1024, 4, 2, 128, 128, 4),
    (2, 2048, 2, 2, 64, 64, 2),
    (1, 1024, 2, 2, 192, 128, 2),
])
def test_zero_copy_matches_permuted_path(cfg):
    """load_balance=2: natural-order tensors, load-balanced schedule.  out,
    lse, dk and dv are bit-identical to permute -> attend -> unpermute (the
    same tiles in the same order: the backward walks a key tile's query tiles
    by position in both layouts); dq agrees to its reduction order; all of
    them against the oracle on the natural-order inputs."""
    B, S, Hq, Hkv, Dqk, Dv, cp = cfg
    q, k, v, dout = synth.attention_inputs(B, S, Hq, Hkv, Dqk, Dv, seed=17)
    qd, kd, vd, dd = q.cuda(), k.cuda(), v.cuda(), dout.cuda()
    out2, lse2 = cp_.attn_fwd(qd, kd, vd, cp, 2)
    dq2, dk2, dv2 = cp_.attn_bwd(qd, kd, vd, out2, lse2, dd, cp, 2)
    torch.cuda.synchronize()
    cp_.check_device()
    perm = [cp_.lb_permute(x, cp) for x in (qd, kd, vd, dd)]
    out1, lse1 = cp_.attn_fwd(*perm[:3], cp, 1)
    dq1, dk1, dv1 = cp_.attn_bwd(*perm[:3], out1, lse1, perm[3], cp, 1)
    torch.cuda.synchronize()
    pos = torch.from_numpy(O.lb_positions(S, cp, True)).long()
    lse1_nat = torch.empty_like(lse1)
    lse1_nat[:, :, pos.cuda()] = lse1
    assert torch.equal(out2, cp_.lb_unpermute(out1, cp))
    assert torch.equal(lse2, lse1_nat)
    assert torch.equal(dk2, cp_.lb_unpermute(dk1, cp))
    assert torch.equal(dv2, cp_.lb_unpermute(dv1, cp))
    assert_close_grad(_f64(dq2), _f64(cp_.lb_unpermute(dq1, cp)), "dq zero-copy vs permuted")
    o_ref, l_ref = O.causal_attention_fwd(_f64(q), _f64(k), _f64(v))
    assert_close_out(_f64(out2), o_ref, "zero-copy out")
    g_ref = O.causal_attention_bwd(_f64(q), _f64(k), _f64(v), o_ref, l_ref, _f64(dout))
    for got, want, name in zip((dq2, dk2, dv2), g_ref, ("dq", "dk", "dv")):
        assert_close_grad(_f64(got), want, "zero-copy %s %s" % (name, cfg))


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg", [
    # B, Hq, Hkv, D, Smax, lo, hi
    (24, 32, 8, 128, 2048, 1024, 2048),   # the decode workload
    (3, 8, 8, 128, 300, 1, 300),          # G = 1, ragged splits
    (4, 16, 1, 64, 700, 200, 700),        # G = 16, D = 64
    (2, 6, 2, 128, 512, 255, 257),        # G = 3, around a split boundary
    (2, 16, 1, 128, 640, 300, 640),       # G = 16, D = 128 (two-stage ring)
    (1, 2, 1, 128, 128, 128, 128),        # one slice: no merge pass
    (2, 8, 2, 128, 4500, 2100, 4500),     # rows over several CTA ranges
    (1, 4, 1, 128, 65536, 65536, 65536),  # one row cut into every CTA's range
    (1, 2, 1, 128, 64, 5, 5),             # fewer positions than CTAs: one-position ranges
    (3, 32, 8, 128, 1000, 1, 1000),       # lengths from 1 up: rows of one item next to long ones
])
def test_decode_parity(cfg):
    B, Hq, Hkv, D, Smax, lo, hi = cfg
    q, kc, vc, lens = synth.decode_inputs(B, Hq, Hkv, D, Smax, lo, hi, seed=21)
    out = cp_.gqa_decode(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda())
    torch.cuda.synchronize()
    cp_.check_device()
    ref = O.gqa_decode(_f64(q), _f64(kc), _f64(vc), lens.numpy())
    assert_close_out(_f64(out), ref, "decode %s" % (cfg,))
    # a second call reuses the arrival counts (and must give the same bits)
    out2 = cp_.gqa_decode(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda())
    assert torch.equal(out2, out)


def test_decode_edge_lengths():
    B, Hq, Hkv, D, Smax = 5, 8, 2, 128, 1024
    q, kc, vc, _ = synth.decode_inputs(B, Hq, Hkv, D, Smax, 1, 1, seed=22)
    lens = torch.tensor([0, 1, 256, 257, 1024], dtype=torch.int32)
    out = cp_.gqa_decode(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda())
    torch.cuda.synchronize()
    cp_.check_device()
    ref = O.gqa_decode(_f64(q), _f64(kc), _f64(vc), lens.numpy())
    assert torch.all(out[0] == 0)
    assert_close_out(_f64(out), ref, "decode edge lengths")


def test_decode_ignores_rows_past_the_length():
    """Cache rows at or past lens[b] hold NaN: they get zero weight and their
    values are never used (bf16 cache; int8 cache with NaN scales there)."""
    B, Hq, Hkv, D, Smax = 4, 16, 4, 128, 700
    q, kc, vc, _ = synth.decode_inputs(B, Hq, Hkv, D, Smax, 1, 1, seed=24)
    lens = torch.tensor([1, 129, 300, 700], dtype=torch.int32)
    kd, vd = kc.clone(), vc.clone()
    for b in range(B):
        kd[b, :, int(lens[b]):] = float("nan")
        vd[b, :, int(lens[b]):] = float("nan")
    out = cp_.gqa_decode(q.cuda(), kd.cuda(), vd.cuda(), lens.cuda())
    torch.cuda.synchronize()
    cp_.check_device()
    ref = O.gqa_decode(_f64(q), _f64(kc), _f64(vc), lens.numpy())
    assert_close_out(_f64(out), ref, "decode with NaN past the lengths")
    q8, kq, vq, ks, vs, _ = synth.decode_inputs_int8(B, Hq, Hkv, D, Smax, 1, 1, seed=25)
    ksd, vsd = ks.clone(), vs.clone()
    for b in range(B):
        ksd[b, :, int(lens[b]):] = float("nan")
        vsd[b, :, int(lens[b]):] = float("nan")
    out8 = cp_.gqa_decode_int8(q8.cuda(), kq.cuda(), vq.cuda(), ksd.cuda(), vsd.cuda(), lens.cuda())
    torch.cuda.synchronize()
    cp_.check_device()
    ref8 = O.gqa_decode_int8(_f64(q8), kq.numpy(), vq.numpy(), ks.numpy().astype(np.float64),
                             vs.numpy().astype(np.float64), lens.numpy())
    assert_close_out(_f64(out8), ref8, "int8 decode with NaN scales past the lengths")


def test_decode_bad_lengths_are_flagged():
    B, Hq, Hkv, D, Smax = 2, 4, 1, 128, 256
    q, kc, vc, _ = synth.decode_inputs(B, Hq, Hkv, D, Smax, 1, 1, seed=23)
    lens = torch.tensor([300, 10], dtype=torch.int32)  # 300 > Smax: clamped to 256
    out = cp_.gqa_decode(q.cuda(), kc.cuda(), vc.cuda(), lens.cuda())
    with pytest.raises(cp_.CpAttnError) as e:
        cp_.check_device()
    assert e.value.code == -6
    ref = O.gqa_decode(_f64(q), _f64(kc), _f64(vc), np.array([256, 10]))
    assert_close_out(_f64(out), ref, "clamped decode")
    cp_.check_device()  # the flag was cleared


# ---------------------------------------------------------------------------
# int8 KV-cache decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg", [
    # B, Hq, Hkv, D, Smax, lo, hi
    (24, 32, 8, 128, 2048, 1024, 2048),   # the decode workload with an int8 cache
    (3, 8, 8, 128, 300, 1, 300),          # G = 1, cache length not a multiple of 128
    (2, 16, 1, 128, 640, 300, 640),       # G = 16
    (1, 2, 1, 128, 128, 128, 128),        # one slice: no merge pass
])
def test_decode_int8_parity(cfg):
    B, Hq, Hkv, D, Smax, lo, hi = cfg
    q, kq, vq, ks, vs, lens = synth.decode_inputs_int8(B, Hq, Hkv, D, Smax, lo, hi, seed=41)
    out = cp_.gqa_decode_int8(q.cuda(), kq.cuda(), vq.cuda(), ks.cuda(), vs.cuda(), lens.cuda())
    torch.cuda.synchronize()
    cp_.check_device()
    ref = O.gqa_decode_int8(_f64(q), kq.numpy(), vq.numpy(), ks.numpy().astype(np.float64),
                            vs.numpy().astype(np.float64), lens.numpy())
    assert_close_out(_f64(out), ref, "int8 decode %s" % (cfg,))
    out2 = cp_.gqa_decode_int8(q.cuda(), kq.cuda(), vq.cuda(), ks.cuda(), vs.cuda(), lens.cuda())
    assert torch.equal(out2, out)


def test_decode_int8_edge_lengths():
    B, Hq, Hkv, D, Smax = 5, 8, 2, 128, 1024
    q, kq, vq, ks, vs, _ = synth.decode_inputs_int8(B, Hq, Hkv, D, Smax, 1, 1, seed=42)
    lens = torch.tensor([0, 1, 256, 257, 1024], dtype=torch.int32)
    out = cp_.gqa_decode_int8(q.cuda(), kq.cuda(), vq.cuda(), ks.cuda(), vs.cuda(), lens.cuda())
    torch.cuda.synchronize()
    cp_.check_device()
    ref = O.gqa_decode_int8(_f64(q), kq.numpy(), vq.numpy(), ks.numpy().astype(np.float64),
                            vs.numpy().astype(np.float64), lens.numpy())
    assert torch.all(out[0] == 0)
    assert_close_out(_f64(out), ref, "int8 decode edge lengths")


def test_decode_repeatable_over_many_calls():
    """The decode is bitwise repeatable (no atomics; every partial and its
    merge in a fixed order), so repeated calls on the same inputs must agree
    bit for bit.  Many short and partial slices (lengths from 1) stress the
    hand-off between the roles: a wait that confuses one pipeline phase with
    another shows here as an occasional differing call long before it fails
    a tolerance."""
    B, Hq, Hkv, D, Smax = 24, 32, 8, 128, 2048
    q, kc, vc, lens = (x.cuda() for x in synth.decode_inputs(B, Hq, Hkv, D, Smax, 1, Smax, seed=9))
    q8, kq, vq, ks, vs, _ = synth.decode_inputs_int8(B, Hq, Hkv, D, Smax, 1, 1, seed=10)
    q8, kq, vq, ks, vs = (x.cuda() for x in (q8, kq, vq, ks, vs))
    ref = cp_.gqa_decode(q, kc, vc, lens).clone()
    ref8 = cp_.gqa_decode_int8(q8, kq, vq, ks, vs, lens).clone()
    cp_.check_device()
    bad = bad8 = 0
    for _ in range(200):
        bad += not torch.equal(cp_.gqa_decode(q, kc, vc, lens), ref)
        bad8 += not torch.equal(cp_.gqa_decode_int8(q8, kq, vq, ks, vs, lens), ref8)
    cp_.check_device()
    assert bad == 0 and bad8 == 0, (bad, bad8)


# ---------------------------------------------------------------------------
# MLA with the rope key shared by the heads
# ---------------------------------------------------------------------------

def _mla_inputs(B, S, H, seed):
    q, kfull, v, dout = synth.attention_inputs(B, S, H, H, 192, 128, seed=seed)
    kn = kfull[..., :128].contiguous()
    kr = kfull[:, :, 0, 128:].contiguous()  # one 64-column rope key per token
    return q, kn, kr, v, dout


@pytest.mark.parametrize("cfg", [(1, 384, 2, 2, True), (2, 256, 3, 2, True), (1, 512, 4, 4, False)])
def test_mla_shared_rope_parity(cfg):
    B, S, H, cp, lb = cfg
    q, kn, kr, v, dout = _mla_inputs(B, S, H, seed=19)
    dev = [x.cuda() for x in (q, kn, kr, v, dout)]
    if lb:
        dev = [cp_.lb_permute(x, cp) for x in dev]
    qd, knd, krd, vd, dd = dev
    out, lse = cp_.attn_fwd_mla(qd, knd, krd, vd, cp, lb)
    dq, dkn, dkr, dv = cp_.attn_bwd_mla(qd, knd, krd, vd, out, lse, dd, cp, lb)
    torch.cuda.synchronize()
    cp_.check_device()
    pos = O.lb_positions(S, cp, lb)
    qs, kns, krs, vs, ds = (O.permute(_f64(x), pos) for x in (q, kn, kr, v, dout))
    o_ref, l_ref = O.cp_attention_mla_fwd(qs, kns, krs, vs, cp, lb)
    assert_close_out(_f64(out), o_ref, "mla out %s" % (cfg,))
    err = float(np.max(np.abs(lse.cpu().numpy().astype(np.float64) - l_ref)))
    assert err <= 1e-2, "mla lse max-abs %.3e" % err
    g_ref = O.cp_attention_mla_bwd(qs, kns, krs, vs, o_ref, l_ref, ds, cp, lb)
    for got, want, name in zip((dq, dkn, dkr, dv), g_ref, ("dq", "dk_nope", "dk_rope", "dv")):
        assert_close_grad(_f64(got), want, "mla %s %s" % (name, cfg))


def test_mla_shared_rope_matches_materialised_key():
    """The shared rope key gives what the per-head key concat(k_nope, k_rope)
    gives through the plain MLA path: out, lse, dq, dv bit for bit (the same
    tiles), dk_nope equal to that path's nope columns, dk_rope to the sum over
    heads of its rope columns."""
    B, S, H, cp = 1, 512, 4, 2
    q, kn, kr, v, dout = (cp_.lb_permute(x.cuda(), cp) for x in _mla_inputs(B, S, H, seed=23))
    kfull = torch.cat([kn, kr[:, :, None, :].expand(B, S, H, 64)], dim=-1).contiguous()
    out1, lse1 = cp_.attn_fwd_mla(q, kn, kr, v, cp, True)
    out2, lse2 = cp_.attn_fwd(q, kfull, v, cp, True)
    dq1, dkn1, dkr1, dv1 = cp_.attn_bwd_mla(q, kn, kr, v, out1, lse1, dout, cp, True)
    dq2, dk2, dv2 = cp_.attn_bwd(q, kfull, v, out2, lse2, dout, cp, True)
    torch.cuda.synchronize()
    cp_.check_device()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    assert torch.equal(dv1, dv2)
    # dq goes through an fp32 accumulator that several CTAs add into, in an
    # order that varies: equal to rounding
    assert_close_grad(_f64(dq1), _f64(dq2), "dq of the shared and the materialised rope key", rel=1e-3)
    assert torch.equal(dkn1, dk2[..., :128])
    want = dk2[..., 128:].double().sum(dim=2)
    assert_close_grad(_f64(dkr1), want.cpu().numpy(), "dk_rope vs summed rope columns")


def test_mla_shared_rope_zero_copy():
    """load_balance=2 with the shared rope key: natural-order tensors give
    permute -> attend -> unpermute's results (out, lse, dq, dk_nope, dv bit for
    bit; dk_rope to its summation order)."""
    B, S, H, cp = 1, 512, 2, 2
    nat = [x.cuda() for x in _mla_inputs(B, S, H, seed=29)]
    out2, lse2 = cp_.attn_fwd_mla(*nat[:4], cp, 2)
    g2 = cp_.attn_bwd_mla(*nat[:4], out2, lse2, nat[4], cp, 2)
    perm = [cp_.lb_permute(x, cp) for x in nat]
    out1, lse1 = cp_.attn_fwd_mla(*perm[:4], cp, 1)
    g1 = cp_.attn_bwd_mla(*perm[:4], out1, lse1, perm[4], cp, 1)
    torch.cuda.synchronize()
    cp_.check_device()
    pos = torch.from_numpy(O.lb_positions(S, cp, True)).long()
    lse1_nat = torch.empty_like(lse1)
    lse1_nat[:, :, pos.cuda()] = lse1
    assert torch.equal(out2, cp_.lb_unpermute(out1, cp)) and torch.equal(lse2, lse1_nat)
    for a2, a1, name in zip(g2, g1, ("dq", "dk_nope", "dk_rope", "dv")):
        a1n = cp_.lb_unpermute(a1, cp)
        if name in ("dk_rope", "dq"):  # fp32 accumulators added into in a varying order
            assert_close_grad(_f64(a2), _f64(a1n), "zero-copy %s" % name, rel=1e-3)
        else:
            assert torch.equal(a2, a1n), name


# ---------------------------------------------------------------------------
# absorbed-MLA decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg", [
    # B, H, Smax, lo, hi
    (24, 128, 2048, 1024, 2048),   # DeepSeek-V3-shaped: 128 heads, batch and lengths of the decode workload
    (3, 128, 700, 1, 700),         # ragged chunks, lengths from 1
    (2, 16, 512, 256, 257),        # 16 heads, around a chunk boundary
    (1, 128, 256, 256, 256),       # one whole chunk
    (5, 64, 1300, 0, 1300),        # may include an empty cache
    (2, 128, 3000, 2100, 3000),    # more than eight chunks per row: the merge takes them in two groups
    (64, 128, 2048, 1024, 2048),   # about 400 items: two or three per CTA, so items follow one another on an SM
])
def test_mla_decode_parity(cfg):
    B, H, Smax, lo, hi = cfg
    q, ckv, lens = synth.mla_decode_inputs(B, H, Smax, lo, hi, seed=51)
    out = cp_.mla_decode(q.cuda(), ckv.cuda(), lens.cuda())
    torch.cuda.synchronize()
    cp_.check_device()
    ref = O.mla_decode(_f64(q), _f64(ckv), lens.numpy())
    assert_close_out(_f64(out), ref, "mla decode %s" % (cfg,))


def test_mla_decode_repeatable_with_several_items_per_cta():
    """With more items than SMs a CTA's next item loads over the space its last
    one used: 20 calls on a 64-sequence batch give identical bits."""
    q, ckv, lens = synth.mla_decode_inputs(64, 128, 2048, 1, 2048, seed=57)
    q, ckv, lens = q.cuda(), ckv.cuda(), lens.cuda()
    ref = cp_.mla_decode(q, ckv, lens).clone()
    bad = sum(not torch.equal(cp_.mla_decode(q, ckv, lens), ref) for _ in range(20))
    torch.cuda.synchronize()
    cp_.check_device()
    assert bad == 0, "%d of 20 calls differ" % bad


def test_mla_decode_repeatable_over_many_calls():
    """The absorbed-MLA decode writes its partials and merges them in a fixed
    order, so repeated calls agree bit for bit (lengths from 1: whole and
    partial chunks, rows fixed up past the length)."""
    q, ckv, lens = synth.mla_decode_inputs(24, 128, 2048, 1, 2048, seed=53)
    q, ckv, lens = q.cuda(), ckv.cuda(), lens.cuda()
    ref = cp_.mla_decode(q, ckv, lens).clone()
    cp_.check_device()
    bad = sum(not torch.equal(cp_.mla_decode(q, ckv, lens), ref) for _ in range(100))
    cp_.check_device()
    assert bad == 0, bad


def test_mla_decode_ignores_rows_past_the_length():
    """Cache rows at or past lens[b] hold NaN: they get zero weight, and the
    value rows of the last 16-position step that the output product reads
    are cleared first, so nothing leaks (a last chunk of 44, 1, 1 and 32
    positions: partial steps and a whole one)."""
    B, H, Smax = 4, 128, 600
    q, ckv, lens = synth.mla_decode_inputs(B, H, Smax, 1, 600, seed=52)
    lens = torch.tensor([300, 1, 513, 288], dtype=torch.int32)
    dirty = ckv.clone()
    for b in range(B):
        dirty[b, int(lens[b]):] = float("nan")
    out = cp_.mla_decode(q.cuda(), dirty.cuda(), lens.cuda())
    torch.cuda.synchronize()
    cp_.check_device()
    ref = O.mla_decode(_f64(q), _f64(ckv), lens.numpy())
    assert bool(torch.isfinite(out.float()).all())
    assert_close_out(_f64(out), ref, "mla decode with NaN past the lengths")


def test_mla_decode_flags_bad_lengths():
    q, ckv, lens = synth.mla_decode_inputs(2, 8, 300, 10, 300, seed=53)
    bad = torch.tensor([-3, 10_000], dtype=torch.int32)
    out = cp_.mla_decode(q.cuda(), ckv.cuda(), bad.cuda())
    with pytest.raises(cp_.CpAttnError) as e:
        cp_.check_device()
    assert e.value.code == -6
    ref = O.mla_decode(_f64(q), _f64(ckv), np.array([0, 300]))
    assert_close_out(_f64(out), ref, "mla decode, clamped lengths")
