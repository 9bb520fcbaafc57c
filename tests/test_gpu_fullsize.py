"""Parity at the full workload sizes, through the same launches bench.py
times.  The float64 oracle cannot afford whole tensors at these sizes, so it
checks:
  * out, lse and dq on sampled query rows of sampled heads (each row against
    every key it sees);
  * dk and dv exactly on the last 64 key positions of one KV head (only the
    64 query rows per head at those positions see them);
  * identities that hold at any size: sum_j dk_j = 0 and
    sum_j dv_j = sum_i dout_i per KV head;
  * the zero-copy mode (natural-order tensors, load_balance=2) against the
    permuted run: out, lse, dk, dv bit-identical, dq to its reduction order."""

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


def setup_module(_):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    built_lib()


def _f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


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
    kpos = pos
    rng = np.random.default_rng(7)

    # ---- sampled query rows: out, lse, dq ------------------------------
    heads = sorted(set([0, Hq - 1, int(rng.integers(Hq))]))
    slots = np.sort(rng.choice(S, size=24, replace=False))
    slots = np.unique(np.concatenate([slots, [0, S - 1]]))
    for h in heads:
        g = h // G
        kk = _f64(kp[:, :, g:g + 1])
        vv = _f64(vp[:, :, g:g + 1])
        qq = _f64(qp[:, slots, h:h + 1])
        o_ref, l_ref = O.masked_attention_fwd(qq, kk, vv, pos[slots], kpos)
        assert_close_out(_f64(out[:, slots, h:h + 1]), o_ref, "%s out head %d" % (name, h))
        lse_err = np.max(np.abs(_f64(lse[:, h:h + 1, slots]) - l_ref))
        assert lse_err <= 1e-2, "%s lse head %d: %.3e" % (name, h, lse_err)
        dq_ref, _, _ = O.masked_attention_bwd(qq, kk, vv, o_ref, l_ref, _f64(dp[:, slots, h:h + 1]),
                                              pos[slots], kpos)
        assert_close_grad(_f64(dq[:, slots, h:h + 1]), dq_ref, "%s dq head %d" % (name, h))

    # ---- exact dk/dv on the last 64 key positions of KV head g ----------
    g = Hkv - 1
    tail = np.nonzero(pos >= S - 64)[0]  # slots of the last 64 positions
    kk = _f64(kp[:, :, g:g + 1])
    vv = _f64(vp[:, :, g:g + 1])
    dk_ref = np.zeros((B, len(tail), 1, Dqk))
    dv_ref = np.zeros((B, len(tail), 1, Dv))
    for h in range(g * G, g * G + G):
        qq = _f64(qp[:, tail, h:h + 1])
        o_ref, l_ref = O.masked_attention_fwd(qq, kk, vv, pos[tail], kpos)
        _, dk_all, dv_all = O.masked_attention_bwd(qq, kk, vv, o_ref, l_ref, _f64(dp[:, tail, h:h + 1]),
                                                   pos[tail], kpos)
        dk_ref += dk_all[:, tail]
        dv_ref += dv_all[:, tail]
    assert_close_grad(_f64(dk[:, tail, g:g + 1]), dk_ref, "%s dk tail" % name)
    assert_close_grad(_f64(dv[:, tail, g:g + 1]), dv_ref, "%s dv tail" % name)

    # ---- identities over every row ---------------------------------------
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
