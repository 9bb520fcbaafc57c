"""Parity at the full workload sizes, through the same launches bench.py
times (permute -> forward -> backward on the load-balanced tensors).

Element by element against the float64 oracle:
  * Llama2-shaped layer (S=8192, Hq=Hkv=32): two whole heads -- out, lse,
    dq, dk and dv on every row and every key of heads 0 and 31, so every key
    tile's full accumulation over all 64 query tiles is checked;
  * Llama3.1-70B-shaped GQA (S=131072, 8 query heads per KV head) and the
    DeepSeek-V3-shaped MLA layer (S=32768): dk and dv on the last 1024 key
    positions of one KV head, summed over every query head of its group.
    Only queries at those positions see those keys, so the oracle needs the
    forward of just those 1024 query rows per head (against all keys, for
    their lse and out) and the backward restricted to the tail's key
    columns, which is exact: each column of P, dP and dS depends only on its
    own key and the row's lse and D.  out and lse of those rows, and out,
    lse and dq on sampled rows of sampled heads (each row against every key
    it sees), are checked too.
Extra checks that hold at any size: sum_j dk_j = 0 and sum_j dv_j =
sum_i dout_i per KV head; and the zero-copy mode (natural-order tensors,
load_balance=2) against the permuted run: out, lse, dk, dv bit-identical (the
same steps in the same order), dq to its reduction order."""

import math

import numpy as np
import pytest
import torch

from context_causal_attention_load_gb300 import synth
from oracle import cp_attention as O
from tests._lib import assert_close_grad, assert_close_out, built_lib

pytestmark = pytest.mark.gpu

WORKLOADS = {
    # name: B, S, Hq, Hkv, Dqk, Dv, cp, q_scale
    "llama2_7b_s8192_cp4": (1, 8192, 32, 32, 128, 128, 4, 1.0 / math.sqrt(128)),
    "llama3_70b_s131072_cp8": (1, 131072, 64, 8, 128, 128, 8, 1.0),
    "deepseek_v3_mla_s32768_cp4": (1, 32768, 128, 128, 192, 128, 4, 1.0),
}
TAIL = 1024  # key positions whose dk/dv are checked at the long sequence lengths


def setup_module(_):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    built_lib()


def _f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def _check_lse(got, want, what):
    err = float(np.max(np.abs(got - want)))
    assert err <= 1e-2, "%s: lse max-abs %.3e (<= 1e-2)" % (what, err)


def _whole_heads(name, qp, kp, vp, dp, out, lse, dq, dk, dv, pos, heads):
    """Every row and every key of the given query heads (Hq == Hkv: one
    query head per KV head, so dk/dv of that KV head come from it alone)."""
    for h in heads:
        qq, kk, vv, do = (_f64(x[:, :, h:h + 1]) for x in (qp, kp, vp, dp))
        o_ref, l_ref = O.masked_attention_fwd(qq, kk, vv, pos, pos)
        assert_close_out(_f64(out[:, :, h:h + 1]), o_ref, "%s out head %d" % (name, h))
        _check_lse(_f64(lse[:, h:h + 1]), l_ref, "%s head %d" % (name, h))
        dq_ref, dk_ref, dv_ref = O.masked_attention_bwd(qq, kk, vv, o_ref, l_ref, do, pos, pos)
        assert_close_grad(_f64(dq[:, :, h:h + 1]), dq_ref, "%s dq head %d" % (name, h))
        assert_close_grad(_f64(dk[:, :, h:h + 1]), dk_ref, "%s dk head %d" % (name, h))
        assert_close_grad(_f64(dv[:, :, h:h + 1]), dv_ref, "%s dv head %d" % (name, h))


def _tail_keys(name, qp, kp, vp, dp, out, lse, dk, dv, pos, g, G):
    """dk/dv of the last TAIL key positions of KV head g, summed over the G
    query heads of the group, plus out/lse of the query rows at those
    positions."""
    tail = np.nonzero(pos >= len(pos) - TAIL)[0]  # slots of the last TAIL positions
    kk = _f64(kp[:, :, g:g + 1])
    vv = _f64(vp[:, :, g:g + 1])
    dk_ref = np.zeros((kk.shape[0], len(tail), 1, kk.shape[3]))
    dv_ref = np.zeros((vv.shape[0], len(tail), 1, vv.shape[3]))
    for h in range(g * G, g * G + G):
        qq = _f64(qp[:, tail, h:h + 1])
        o_ref, l_ref = O.masked_attention_fwd(qq, kk, vv, pos[tail], pos)
        assert_close_out(_f64(out[:, tail, h:h + 1]), o_ref, "%s out of the tail rows, head %d" % (name, h))
        _check_lse(_f64(lse[:, h:h + 1, tail]), l_ref, "%s tail rows, head %d" % (name, h))
        _, dk_t, dv_t = O.masked_attention_bwd(qq, kk[:, tail], vv[:, tail], o_ref, l_ref,
                                               _f64(dp[:, tail, h:h + 1]), pos[tail], pos[tail])
        dk_ref += dk_t
        dv_ref += dv_t
    assert_close_grad(_f64(dk[:, tail, g:g + 1]), dk_ref, "%s dk of the last %d keys" % (name, TAIL))
    assert_close_grad(_f64(dv[:, tail, g:g + 1]), dv_ref, "%s dv of the last %d keys" % (name, TAIL))


def _sampled_rows(name, qp, kp, vp, dp, out, lse, dq, pos, G, Hq):
    rng = np.random.default_rng(7)
    heads = sorted(set([0, Hq - 1, int(rng.integers(Hq))]))
    S = len(pos)
    slots = np.unique(np.concatenate([np.sort(rng.choice(S, size=24, replace=False)), [0, S - 1]]))
    for h in heads:
        g = h // G
        kk = _f64(kp[:, :, g:g + 1])
        vv = _f64(vp[:, :, g:g + 1])
        qq = _f64(qp[:, slots, h:h + 1])
        o_ref, l_ref = O.masked_attention_fwd(qq, kk, vv, pos[slots], pos)
        assert_close_out(_f64(out[:, slots, h:h + 1]), o_ref, "%s out head %d" % (name, h))
        _check_lse(_f64(lse[:, h:h + 1, slots]), l_ref, "%s sampled rows, head %d" % (name, h))
        dq_ref, _, _ = O.masked_attention_bwd(qq, kk, vv, o_ref, l_ref, _f64(dp[:, slots, h:h + 1]),
                                              pos[slots], pos)
        assert_close_grad(_f64(dq[:, slots, h:h + 1]), dq_ref, "%s dq head %d" % (name, h))


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_fullsize_parity(name):
    from context_causal_attention_load_gb300 import cpattn
    B, S, Hq, Hkv, Dqk, Dv, cp, qs = WORKLOADS[name]
    G = Hq // Hkv
    q, k, v, dout = synth.attention_inputs_device(B, S, Hq, Hkv, Dqk, Dv, seed=101, q_scale=qs)
    # load-balanced order on the GPU, exactly as the bench step does it
    qp, kp, vp, dp = (cpattn.lb_permute(x, cp) for x in (q, k, v, dout))
    out, lse = cpattn.attn_fwd(qp, kp, vp, cp, True)
    dq, dk, dv = cpattn.attn_bwd(qp, kp, vp, out, lse, dp, cp, True)
    torch.cuda.synchronize()
    cpattn.check_device()
    pos = O.lb_positions(S, cp, True)

    if G == 1 and S <= 8192:
        _whole_heads(name, qp, kp, vp, dp, out, lse, dq, dk, dv, pos, (0, Hq - 1))
    else:
        _sampled_rows(name, qp, kp, vp, dp, out, lse, dq, pos, G, Hq)
        _tail_keys(name, qp, kp, vp, dp, out, lse, dk, dv, pos, Hkv - 1, G)

    # ---- identities over every row (extra checks) --------------------------
    dk32 = dk.float()
    dv32 = dv.float()
    dsum = dp.float().reshape(B, S, Hkv, G, Dv).sum(dim=(1, 3))
    ksum = dk32.sum(dim=1)
    kabs = dk32.abs().sum(dim=1)
    assert float((ksum.abs() / kabs).max()) < 2e-3, "%s: sum_j dk_j is not ~0" % name
    vsum = dv32.sum(dim=1)
    rel = float(((vsum - dsum).norm() / dsum.norm()))
    assert rel < 5e-3, "%s: sum dv != sum dout (rel %.2e)" % (name, rel)

    # ---- zero-copy load balance: the same tiles on natural-order tensors ----
    out_z, lse_z = cpattn.attn_fwd(q, k, v, cp, 2)
    dq_z, dk_z, dv_z = cpattn.attn_bwd(q, k, v, out_z, lse_z, dout, cp, 2)
    torch.cuda.synchronize()
    cpattn.check_device()
    assert torch.equal(out_z, cpattn.lb_unpermute(out, cp)), "%s zero-copy out" % name
    assert torch.equal(lse_z[:, :, torch.from_numpy(pos).long().cuda()], lse), "%s zero-copy lse" % name
    assert torch.equal(dk_z, cpattn.lb_unpermute(dk, cp)), "%s zero-copy dk" % name
    assert torch.equal(dv_z, cpattn.lb_unpermute(dv, cp)), "%s zero-copy dv" % name
    dq_n = cpattn.lb_unpermute(dq, cp).float()
    rel = float((dq_z.float() - dq_n).norm() / dq_n.norm())
    assert rel < 1e-3, "%s zero-copy dq differs beyond its reduction order (rel %.2e)" % (name, rel)
