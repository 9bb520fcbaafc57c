"""ctypes binding of libcpattn.so (argument marshalling only).

Every function here takes torch tensors that already live on the GPU, checks
dtype/shape/contiguity, passes raw device pointers and the current CUDA
stream to the C ABI declared in ``include/cpattn.h``, and raises
``CpAttnError`` on a non-zero status.  No computation happens in Python and
there is no fallback: if the library is missing the import of the first
call fails loudly.
"""

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "CpAttnError", "load", "lb_permute", "lb_unpermute", "attn_fwd", "attn_fwd_shard",
    "attn_bwd", "gqa_decode", "lb_positions", "tile_counts", "check_device", "release",
    "profile_start", "profile_stop", "EXPORTED_SYMBOLS",
]

EXPORTED_SYMBOLS = (
    "cp_lb_permute", "cp_lb_unpermute", "cp_attn_fwd", "cp_attn_fwd_shard", "cp_attn_bwd",
    "gqa_decode", "cp_lb_positions", "cp_attn_tile_counts", "cp_attn_check_device",
    "cp_attn_last_error", "cp_attn_release", "cp_attn_profile_start", "cp_attn_profile_stop",
)


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]

_lib = None


class CpAttnError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__("cpattn error %d: %s" % (code, msg))
        self.code = code


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_longlong


def load(path=None):
    """Load libcpattn.so (built in-tree by ``build.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.lib_path()
    if not os.path.exists(path):
        raise RuntimeError("libcpattn.so is not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    sig = {
        "cp_lb_permute": [_P, _P, _I, _I, _L, _I, _P],
        "cp_lb_unpermute": [_P, _P, _I, _I, _L, _I, _P],
        "cp_attn_fwd": [_P, _P, _P, _P, _P] + [_I] * 8 + [_P],
        "cp_attn_fwd_shard": [_P, _P, _P, _P, _P] + [_I] * 9 + [_P],
        "cp_attn_bwd": [_P] * 9 + [_I] * 8 + [_P],
        "cp_attn_bwd_shard": [_P] * 9 + [_I] * 9 + [_P, _P, _P],
        "cp_attn_fwd_mla": [_P] * 6 + [_I] * 5 + [_P],
        "cp_attn_bwd_mla": [_P] * 11 + [_I] * 5 + [_P],
        "gqa_decode": [_P] * 5 + [_I] * 5 + [_P],
        "gqa_decode_int8": [_P] * 7 + [_I] * 5 + [_P],
        "mla_decode": [_P] * 4 + [_I] * 3 + [ctypes.c_float, _P],
        "cp_lb_positions": [_I, _I, _I, ctypes.POINTER(ctypes.c_int)],
        "cp_attn_tile_counts": [_I, _I, _I, ctypes.POINTER(ctypes.c_longlong)],
        "cp_attn_fwd_schedule": [_I] * 7 + [ctypes.POINTER(ctypes.c_longlong)],
        "cp_attn_fwd_shard_schedule": [_I] * 8 + [ctypes.POINTER(ctypes.c_longlong)],
        "cp_attn_check_device": [_P],
        "cp_attn_test_stall_forward": [_I, _L],
        "cp_attn_release": [],
        "cp_attn_profile_start": [],
        "cp_attn_profile_stop": [ctypes.POINTER(KernelStat), ctypes.c_int, ctypes.POINTER(ctypes.c_int)],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.cp_attn_last_error.argtypes = []
    lib.cp_attn_last_error.restype = ctypes.c_char_p
    if path == _build.lib_path():
        _lib = lib
    return lib


def _check(rc):
    if rc != 0:
        msg = load().cp_attn_last_error().decode(errors="replace")
        raise CpAttnError(rc, msg)


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, ndim=None):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims" % (name, ndim))


def lb_permute(x, cp, out=None):
    """Load-balance reorder of axis 1 of a [B, S, ...] CUDA tensor."""
    return _perm(x, cp, out, False)


def lb_unpermute(x, cp, out=None):
    return _perm(x, cp, out, True)


def _perm(x, cp, out, inverse):
    if not x.is_cuda or not x.is_contiguous() or x.dim() < 2:
        raise ValueError("x must be a contiguous CUDA tensor [B, S, ...]")
    out = torch.empty_like(x) if out is None else out
    B, S = x.shape[:2]
    row = x[0, 0].numel() * x.element_size()
    f = load().cp_lb_unpermute if inverse else load().cp_lb_permute
    _check(f(_ptr(x), _ptr(out), B, S, row, cp, _stream(x)))
    return out


def _shape(q, k, v):
    _need(q, torch.bfloat16, "q", 4)
    _need(k, torch.bfloat16, "k", 4)
    _need(v, torch.bfloat16, "v", 4)
    B, S, Hq, Dqk = q.shape
    if k.shape[:2] != (B, S) or v.shape[:3] != k.shape[:3] or k.shape[3] != Dqk:
        raise ValueError("q/k/v shapes do not match")
    return B, S, Hq, k.shape[2], Dqk, v.shape[3]


def attn_fwd(q, k, v, cp, load_balance=True, out=None, lse=None, shard=None):
    """out [B,S,Hq,Dv] bf16 and lse [B,Hq,S] fp32 of causal CP attention;
    q/k/v in load-balanced slot order when load_balance is true."""
    B, S, Hq, Hkv, Dqk, Dv = _shape(q, k, v)
    if out is None:
        out = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    _need(out, torch.bfloat16, "out", 4)
    _need(lse, torch.float32, "lse", 3)
    lib = load()
    if shard is None:
        rc = lib.cp_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, Dqk, Dv,
                             cp, _lb(load_balance), _stream(q))
    else:
        rc = lib.cp_attn_fwd_shard(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, Dqk,
                                   Dv, cp, _lb(load_balance), int(shard), _stream(q))
    _check(rc)
    return out, lse


def attn_fwd_shard(q, k, v, cp, shard, load_balance=True, out=None, lse=None):
    return attn_fwd(q, k, v, cp, load_balance, out, lse, shard)


def attn_bwd(q, k, v, out, lse, dout, cp, load_balance=True, dq=None, dk=None, dv=None):
    """dq, dk, dv (bf16, shapes of q/k/v) of sum(out * dout)."""
    B, S, Hq, Hkv, Dqk, Dv = _shape(q, k, v)
    _need(out, torch.bfloat16, "out", 4)
    _need(dout, torch.bfloat16, "dout", 4)
    _need(lse, torch.float32, "lse", 3)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    rc = load().cp_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                            _ptr(dk), _ptr(dv), B, Hq, Hkv, S, Dqk, Dv, cp, _lb(load_balance),
                            _stream(q))
    _check(rc)
    return dq, dk, dv


def _lb(load_balance):
    """0 natural order, 1 tensors in load-balanced slot order, 2 natural-order
    tensors with the load-balanced schedule (zero-copy); True/False -> 1/0."""
    if load_balance is True or load_balance is False:
        return int(load_balance)
    if load_balance not in (0, 1, 2):
        raise ValueError("load_balance must be 0, 1 or 2")
    return int(load_balance)


def attn_bwd_shard(q, k, v, out, lse, dout, cp, shard, load_balance=True, dq=None, dk_part=None, dv_part=None,
                   dk=None, dv=None):
    """Backward work of one shard: dq (bf16, the shard's rows; zero elsewhere)
    and this shard's fp32 contributions dk_part, dv_part (optionally also
    rounded into bf16 dk, dv)."""
    B, S, Hq, Hkv, Dqk, Dv = _shape(q, k, v)
    _need(out, torch.bfloat16, "out", 4)
    _need(dout, torch.bfloat16, "dout", 4)
    _need(lse, torch.float32, "lse", 3)
    dq = torch.empty_like(q) if dq is None else dq
    dk_part = torch.empty(k.shape, dtype=torch.float32, device=k.device) if dk_part is None else dk_part
    dv_part = torch.empty(v.shape, dtype=torch.float32, device=v.device) if dv_part is None else dv_part
    rc = load().cp_attn_bwd_shard(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                                  _ptr(dk) if dk is not None else None, _ptr(dv) if dv is not None else None,
                                  B, Hq, Hkv, S, Dqk, Dv, cp, _lb(load_balance), int(shard),
                                  _ptr(dk_part), _ptr(dv_part), _stream(q))
    _check(rc)
    return dq, dk_part, dv_part



def _mla_shapes(q, k_nope, k_rope, v):
    _need(q, torch.bfloat16, "q", 4)
    _need(k_nope, torch.bfloat16, "k_nope", 4)
    _need(k_rope, torch.bfloat16, "k_rope", 3)
    _need(v, torch.bfloat16, "v", 4)
    B, S, H, Dqk = q.shape
    if Dqk != 192 or tuple(k_nope.shape) != (B, S, H, 128) or tuple(k_rope.shape) != (B, S, 64) \
            or tuple(v.shape) != (B, S, H, 128):
        raise ValueError("MLA shapes: q [B,S,H,192], k_nope [B,S,H,128], k_rope [B,S,64], v [B,S,H,128]")
    return B, S, H


def attn_fwd_mla(q, k_nope, k_rope, v, cp, load_balance=True, out=None, lse=None):
    """MLA forward with one rope key per token shared by the heads: out
    [B,S,H,128] bf16 and lse [B,H,S] fp32 of attention with the per-head key
    concat(k_nope, k_rope)."""
    B, S, H = _mla_shapes(q, k_nope, k_rope, v)
    out = torch.empty(B, S, H, 128, dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty(B, H, S, dtype=torch.float32, device=q.device) if lse is None else lse
    _check(load().cp_attn_fwd_mla(_ptr(q), _ptr(k_nope), _ptr(k_rope), _ptr(v), _ptr(out), _ptr(lse), B, H, S, cp,
                                  _lb(load_balance), _stream(q)))
    return out, lse


def attn_bwd_mla(q, k_nope, k_rope, v, out, lse, dout, cp, load_balance=True, dq=None, dk_nope=None, dk_rope=None,
                 dv=None):
    """dq, dk_nope, dk_rope (summed over heads), dv of sum(out * dout) for
    ``attn_fwd_mla``."""
    B, S, H = _mla_shapes(q, k_nope, k_rope, v)
    _need(out, torch.bfloat16, "out", 4)
    _need(dout, torch.bfloat16, "dout", 4)
    _need(lse, torch.float32, "lse", 3)
    dq = torch.empty_like(q) if dq is None else dq
    dk_nope = torch.empty_like(k_nope) if dk_nope is None else dk_nope
    dk_rope = torch.empty_like(k_rope) if dk_rope is None else dk_rope
    dv = torch.empty_like(v) if dv is None else dv
    _check(load().cp_attn_bwd_mla(_ptr(q), _ptr(k_nope), _ptr(k_rope), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                  _ptr(dq), _ptr(dk_nope), _ptr(dk_rope), _ptr(dv), B, H, S, cp, _lb(load_balance),
                                  _stream(q)))
    return dq, dk_nope, dk_rope, dv


def gqa_decode(q, kcache, vcache, lens, out=None):
    """q [B,Hq,D], kcache/vcache [B,Hkv,Smax,D] bf16, lens [B] int32 -> out [B,Hq,D]."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kcache, torch.bfloat16, "kcache", 4)
    _need(vcache, torch.bfloat16, "vcache", 4)
    _need(lens, torch.int32, "lens", 1)
    B, Hq, D = q.shape
    Hkv, Smax = kcache.shape[1], kcache.shape[2]
    out = torch.empty_like(q) if out is None else out
    rc = load().gqa_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(lens), _ptr(out), B, Hq, Hkv,
                           Smax, D, _stream(q))
    _check(rc)
    return out


def mla_decode(q, ckv, lens, scale=None, out=None):
    """Absorbed-MLA decode: q [B,H,576] bf16, ckv [B,Smax,576] bf16 (latent
    rows: 512 compressed-KV columns, then 64 rope columns), lens [B] int32 ->
    out [B,H,512] bf16; scale defaults to 1/sqrt(192)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(ckv, torch.bfloat16, "ckv", 3)
    _need(lens, torch.int32, "lens", 1)
    B, H, Dk = q.shape
    if Dk != 576 or ckv.shape[0] != B or ckv.shape[2] != 576 or lens.shape[0] != B:
        raise ValueError("MLA decode shapes: q [B,H,576], ckv [B,Smax,576], lens [B]")
    out = torch.empty(B, H, 512, dtype=torch.bfloat16, device=q.device) if out is None else out
    _need(out, torch.bfloat16, "out", 3)
    sc = (1.0 / 192.0 ** 0.5) if scale is None else float(scale)
    _check(load().mla_decode(_ptr(q), _ptr(ckv), _ptr(lens), _ptr(out), B, H, ckv.shape[1], sc, _stream(q)))
    return out


def lb_positions(S, cp, load_balance=True):
    arr = (ctypes.c_int * S)()
    _check(load().cp_lb_positions(S, cp, _lb(load_balance), arr))
    return list(arr)



def fwd_schedule(B, Hq, Hkv, S, cp, load_balance, num_ctas):
    """Modelled load of each of num_ctas CTAs under the forward's work plan
    (host only: no device work)."""
    arr = (ctypes.c_longlong * num_ctas)()
    _check(load().cp_attn_fwd_schedule(B, Hq, Hkv, S, cp, _lb(load_balance), num_ctas, arr))
    return list(arr)

def fwd_shard_schedule(B, Hq, Hkv, S, cp, load_balance, shard, num_ctas):
    """The same for one shard's forward plan (shard -1: the whole forward)."""
    arr = (ctypes.c_longlong * num_ctas)()
    _check(load().cp_attn_fwd_shard_schedule(B, Hq, Hkv, S, cp, _lb(load_balance), shard, num_ctas, arr))
    return list(arr)


def tile_counts(S, cp, load_balance=True):
    arr = (ctypes.c_longlong * cp)()
    _check(load().cp_attn_tile_counts(S, cp, _lb(load_balance), arr))
    return list(arr)


def check_device(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    _check(load().cp_attn_check_device(ctypes.c_void_p(s)))


def test_stall_forward(stage, wait_limit_cycles=2_000_000):
    """Test hook: the next forward launch leaves out ring stage `stage`'s
    loads and its pipeline waits give up after wait_limit_cycles (the
    bounded-wait timeout path; see include/cpattn.h).  stage < 0 clears it."""
    _check(load().cp_attn_test_stall_forward(int(stage), int(wait_limit_cycles)))


def release():
    _check(load().cp_attn_release())


def profile_start():
    """Start bracketing every library kernel launch with CUDA events."""
    _check(load().cp_attn_profile_start())


def profile_stop():
    """Stop profiling; returns {kernel name: (launches, total device ms)}."""
    arr = (KernelStat * 64)()
    n = ctypes.c_int(0)
    _check(load().cp_attn_profile_stop(arr, 64, ctypes.byref(n)))
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(min(n.value, 64))}


def gqa_decode_int8(q, kq, vq, kscale, vscale, lens, out=None):
    """q [B,Hq,D] bf16, kq/vq [B,Hkv,Smax,D] int8, kscale/vscale [B,Hkv,Smax]
    fp32, lens [B] int32 -> out [B,Hq,D] bf16."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kq, torch.int8, "kcache", 4)
    _need(vq, torch.int8, "vcache", 4)
    _need(kscale, torch.float32, "kscale", 3)
    _need(vscale, torch.float32, "vscale", 3)
    _need(lens, torch.int32, "lens", 1)
    B, Hq, D = q.shape
    Hkv, Smax = kq.shape[1], kq.shape[2]
    out = torch.empty_like(q) if out is None else out
    rc = load().gqa_decode_int8(_ptr(q), _ptr(kq), _ptr(vq), _ptr(kscale), _ptr(vscale), _ptr(lens), _ptr(out),
                                B, Hq, Hkv, Smax, D, _stream(q))
    _check(rc)
    return out
