"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds no attention arithmetic: it only draws numbers.  Each
tensor has its own sub-seed (q=seed, k=seed+1, v=seed+2, dout=seed+3,
lens=seed+4), values are float32 N(0, 1) draws rounded to bfloat16
(round-to-nearest-even), so the CUDA path and the float64 oracle read the
very same bf16 values.
"""

import torch

__all__ = ["attention_inputs", "attention_inputs_device", "decode_inputs", "decode_inputs_int8",
           "mla_decode_inputs", "to_f64"]


def _normal(shape, seed, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(torch.bfloat16)


def attention_inputs(B, S, Hq, Hkv, Dqk, Dv, seed=0, q_scale=1.0):
    """q [B,S,Hq,Dqk], k [B,S,Hkv,Dqk], v [B,S,Hkv,Dv], dout [B,S,Hq,Dv];
    bf16 CPU tensors.  ``q_scale`` multiplies the fp32 draw of q before the
    bf16 rounding (the Llama2-shaped workload draws q with 1/sqrt(128))."""
    q = _normal((B, S, Hq, Dqk), seed, q_scale)
    k = _normal((B, S, Hkv, Dqk), seed + 1)
    v = _normal((B, S, Hkv, Dv), seed + 2)
    dout = _normal((B, S, Hq, Dv), seed + 3)
    return q, k, v, dout


def attention_inputs_device(B, S, Hq, Hkv, Dqk, Dv, seed=0, q_scale=1.0, device="cuda"):
    """Same shapes and distributions as ``attention_inputs`` but drawn by a
    seeded generator on the GPU (for workloads too large to draw on the host;
    the values differ from the host draw of the same seed)."""
    g = torch.Generator(device=device).manual_seed(int(seed))

    def draw(shape, scale=1.0):
        x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        return (x * scale).to(torch.bfloat16) if scale != 1.0 else x.to(torch.bfloat16)

    q = draw((B, S, Hq, Dqk), q_scale)
    k = draw((B, S, Hkv, Dqk))
    v = draw((B, S, Hkv, Dv))
    dout = draw((B, S, Hq, Dv))
    return q, k, v, dout


def decode_inputs(B, Hq, Hkv, D, Smax, len_lo, len_hi, seed=0):
    """q [B,Hq,D], kcache/vcache [B,Hkv,Smax,D] (bf16) and lens [B] (int32)
    drawn uniformly from the closed range [len_lo, len_hi]."""
    q = _normal((B, Hq, D), seed)
    kc = _normal((B, Hkv, Smax, D), seed + 1)
    vc = _normal((B, Hkv, Smax, D), seed + 2)
    g = torch.Generator(device="cpu").manual_seed(int(seed) + 4)
    lens = torch.randint(int(len_lo), int(len_hi) + 1, (B,), generator=g, dtype=torch.int32)
    return q, kc, vc, lens


def decode_inputs_int8(B, Hq, Hkv, D, Smax, len_lo, len_hi, seed=0):
    """q [B,Hq,D] bf16; int8 caches kq/vq [B,Hkv,Smax,D] uniform in
    [-127, 127]; fp32 scales kscale/vscale [B,Hkv,Smax] uniform in
    [0.008, 0.016] (cached values then span about +-2); lens [B] int32
    uniform in [len_lo, len_hi]."""
    q = _normal((B, Hq, D), seed)
    g = torch.Generator(device="cpu").manual_seed(int(seed) + 11)
    kq = torch.randint(-127, 128, (B, Hkv, Smax, D), generator=g, dtype=torch.int32).to(torch.int8)
    vq = torch.randint(-127, 128, (B, Hkv, Smax, D), generator=g, dtype=torch.int32).to(torch.int8)
    ks = 0.008 + 0.008 * torch.rand((B, Hkv, Smax), generator=g, dtype=torch.float32)
    vs = 0.008 + 0.008 * torch.rand((B, Hkv, Smax), generator=g, dtype=torch.float32)
    gl = torch.Generator(device="cpu").manual_seed(int(seed) + 4)
    lens = torch.randint(int(len_lo), int(len_hi) + 1, (B,), generator=gl, dtype=torch.int32)
    return q, kq, vq, ks, vs, lens


def mla_decode_inputs(B, H, Smax, len_lo, len_hi, seed=0, Dk=576):
    """q [B,H,Dk] and latent cache ckv [B,Smax,Dk] (bf16, N(0,1)), lens [B]
    int32 uniform in [len_lo, len_hi]."""
    q = _normal((B, H, Dk), seed)
    ckv = _normal((B, Smax, Dk), seed + 1)
    g = torch.Generator(device="cpu").manual_seed(int(seed) + 4)
    lens = torch.randint(int(len_lo), int(len_hi) + 1, (B,), generator=g, dtype=torch.int32)
    return q, ckv, lens


def to_f64(t):
    """bf16/float torch tensor -> float64 NumPy array (exact upcast)."""
    return t.detach().to("cpu").to(torch.float64).numpy()
