"""The bounded pipeline waits give up and report, instead of hanging.

A test hook makes the next forward launch leave out one ring stage's loads
and shortens every pipeline wait of that launch to about a millisecond.  The
MMA thread's wait on that stage runs out, the CTA's roles leave their loops
(the producer first lets its issued copies land), TMEM is released and the
launch ends; cp_attn_check_device then reports CPATTN_ERR_DEVICE_TIMEOUT.
Nothing faults, traps or hangs: every wait is bounded.  Afterwards the same
process runs the tiny workload again and it matches the oracle, so the GPU
context is healthy."""

import pytest
import torch

from context_causal_attention_load_gb300 import synth
from oracle import cp_attention as O
from tests._lib import assert_close_grad, assert_close_out, built_lib

pytestmark = pytest.mark.gpu

TIMEOUT = -5  # CPATTN_ERR_DEVICE_TIMEOUT


def setup_module(_):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    built_lib()


def _f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def _tiny_parity(cp_):
    B, S, H, D, cp = 1, 256, 2, 64, 2
    q, k, v, dout = synth.attention_inputs(B, S, H, H, D, D, seed=0)
    qd, kd, vd, dd = (cp_.lb_permute(x.cuda(), cp) for x in (q, k, v, dout))
    out, lse = cp_.attn_fwd(qd, kd, vd, cp, True)
    dq, dk, dv = cp_.attn_bwd(qd, kd, vd, out, lse, dd, cp, True)
    torch.cuda.synchronize()
    cp_.check_device()
    pos = O.lb_positions(S, cp, True)
    f = lambda t: O.permute(_f64(t), pos)  # noqa: E731
    o_ref, l_ref = O.cp_attention_fwd(f(q), f(k), f(v), cp, True)
    assert_close_out(_f64(out), o_ref, "tiny out after the timeout")
    g_ref = O.cp_attention_bwd(f(q), f(k), f(v), o_ref, l_ref, f(dout), cp, True)
    for got, want, name in zip((dq, dk, dv), g_ref, ("dq", "dk", "dv")):
        assert_close_grad(_f64(got), want, "tiny %s after the timeout" % name)


@pytest.mark.parametrize("stage", [0, 2])
def test_forward_wait_times_out_and_reports(stage):
    from context_causal_attention_load_gb300 import cpattn as cp_
    _tiny_parity(cp_)  # clean start
    B, S, H, D, cp = 1, 256, 2, 64, 2
    q, k, v, _ = (x.cuda() for x in synth.attention_inputs(B, S, H, H, D, D, seed=1))
    cp_.test_stall_forward(stage, 2_000_000)  # about a millisecond at the SM clock
    out, lse = cp_.attn_fwd(q, k, v, cp, True)
    with pytest.raises(cp_.CpAttnError) as e:
        cp_.check_device()
    assert e.value.code == TIMEOUT, str(e.value)
    cp_.check_device()  # the word was cleared
    # the hook was used up: this forward runs normally
    out2, lse2 = cp_.attn_fwd(q, k, v, cp, True)
    torch.cuda.synchronize()
    cp_.check_device()
    assert bool(torch.isfinite(out2.float()).all())
    _tiny_parity(cp_)

