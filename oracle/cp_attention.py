"""Plain float64 CPU oracle for load-balanced context-parallel causal attention.

TEST INFRASTRUCTURE ONLY.  This module is the checker, not the product: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` may import it.  It shares no code, header, table or helper
with the CUDA library; it takes plain NumPy arrays and returns plain NumPy
arrays, always in float64.

What it computes, and where each step comes from (the source pages are the
MaxText pull requests "Add context parallelism" (#1445), "Add support for EP
to context parallelism in self-attention" (#2023), "rename context to
context_autoregressive" (#1453) and "Add Pallas GPU decode attention in
Maxtext inference" (#1066)):

* ``lb_chunk_order`` / ``lb_positions`` -- the load-balance reorder of
  "Add context parallelism", Description: the sequence is cut into 2*cp
  chunks and device i receives chunks i and 2cp-1-i, so that for cp=2 the
  shards hold tokens (0,1,6,7) and (2,3,4,5).  Built here by listing the
  chunks and concatenating their token ranges (no closed form).
* ``permute`` / ``unpermute`` -- the token gather the page performs with
  ``jnp.take`` ("Add context parallelism", Description) and its inverse.
* ``masked_attention_fwd`` / ``masked_attention_bwd`` -- softmax(scale*QK^T +
  mask) V with the mask "key position <= query position" evaluated on the
  tokens' ORIGINAL positions, which is what "reorder the tokens and the
  attention mask" means ("Add context parallelism", Description).  Backward
  is the textbook gradient of that expression (the pages train with it, and
  give no formula of their own).
* ``cp_attention_fwd`` / ``cp_attention_bwd`` -- the context-parallel
  paradigm of "Add context parallelism", Description: keys and values are
  all-gathered, queries are sharded on the sequence; each shard's queries
  attend to the full gathered K/V under the reordered mask.  Shards are
  evaluated one after the other; the key/value gradient of every shard is
  summed (the transpose of the all-gather).
* ``causal_attention_fwd`` / ``_bwd`` -- plain unsharded causal attention,
  the "dot_product without sharding" that the unit test of "Add support for
  EP to context parallelism", Description ("Verify attention output logit
  against dot product") compares the sharded kernel with.
* ``mla_key`` / ``cp_attention_mla_fwd`` / ``cp_attention_mla_bwd`` -- MLA
  attention under context parallelism ("Add support for EP to context
  parallelism in self-attention", Main code changes) with the key's rope
  part shared by every head: each head's key is its own "nope" columns
  followed by the token's single rope key.  The key is materialised per head
  here and the plain context-parallel attention above is applied; the rope
  key's gradient is the sum over heads of the rope columns of the per-head
  key gradients (the chain rule through the broadcast).
* ``gqa_decode`` -- one query token per sequence against a KV cache,
  grouped-query heads ("Add Pallas GPU decode attention", Description:
  ``pallas_decode_attention.gqa`` replaces dot-product decode attention).
* ``mla_decode`` -- decode against an MLA latent cache in the absorbed form
  (MLA under context parallelism: "Add support for EP to context parallelism
  in self-attention", Main code changes; one query token per sequence:
  "Add Pallas GPU decode attention", Description): every head's key at
  position t is the token's cached latent vector (its compressed KV followed
  by its rope key) and its value is the compressed-KV part of the same
  vector, so all query heads share one cached row per token.  The query of a
  head is its nope query taken into the latent space, followed by its rope
  query.  Per (b, h): softmax over t < lens[b] of scale * q . ckv_t, times
  ckv_t[:Dv].
* ``gqa_decode_int8`` -- the same against an int8-quantised KV cache (the
  inference setup of "rename context to context_autoregressive", Tests, runs
  with ``quantize_kvcache=True``): each cached vector is stored as int8
  values times one float scale per (batch, KV head, position); it is
  dequantised exactly and then decoded as above.

Readings where the pages are silent (each one listed in the design notes):
scale = 1/sqrt(Dqk); query head h uses KV head floor(h / (Hq/Hkv)); lse is the
natural-log logsumexp of the scaled, masked scores; the KV cache layout is
[B, Hkv, Smax, D] with valid keys t < lens[b]; lens[b] == 0 yields zeros.

Layouts: q [B,S,Hq,Dqk], k [B,S,Hkv,Dqk], v [B,S,Hkv,Dv], out [B,S,Hq,Dv],
lse [B,Hq,S].
"""

import math

import numpy as np

__all__ = [
    "lb_chunk_order", "lb_positions", "permute", "unpermute",
    "masked_attention_fwd", "masked_attention_bwd",
    "causal_attention_fwd", "causal_attention_bwd",
    "cp_attention_fwd", "cp_attention_bwd",
    "shard_pair_counts", "gqa_decode", "gqa_decode_int8",
    "mla_key", "cp_attention_mla_fwd", "cp_attention_mla_bwd", "mla_decode",
]

_ROW_BLOCK = 512


def lb_chunk_order(cp, load_balance=True):
    """Order of the 2*cp chunks after the reorder: shard i holds chunk i, then
    its mirror 2cp-1-i ("Add context parallelism", Description: cp=2 gives
    tokens 0,1,6,7 | 2,3,4,5).  Without load balance the order is natural."""
    if cp < 1:
        raise ValueError("cp must be >= 1")
    if not load_balance:
        return list(range(2 * cp))
    order = []
    for i in range(cp):
        order.append(i)
        order.append(2 * cp - 1 - i)
    return order


def lb_positions(S, cp, load_balance=True):
    """pos[j] = original token position held by reordered slot j."""
    if not load_balance:
        return np.arange(S, dtype=np.int64)
    if S % (2 * cp) != 0:
        raise ValueError("S must be a multiple of 2*cp for the load-balance reorder")
    c = S // (2 * cp)
    pieces = [np.arange(ch * c, (ch + 1) * c, dtype=np.int64)
              for ch in lb_chunk_order(cp, True)]
    return np.concatenate(pieces)


def permute(x, pos):
    """Gather along the sequence axis (axis 1): out[:, j] = x[:, pos[j]]."""
    return np.ascontiguousarray(x[:, pos])


def unpermute(x, pos):
    """Inverse of ``permute``: out[:, pos[j]] = x[:, j]."""
    out = np.empty_like(x)
    out[:, pos] = x
    return out


def _check_heads(q, k, v):
    B, S, Hq, Dqk = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if (Bk, Dk) != (B, Dqk) or v.shape[:3] != k.shape[:3]:
        raise ValueError("shape mismatch between q, k and v")
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, S, Sk, Hq, Hkv, Dqk, v.shape[3]


def masked_attention_fwd(q, k, v, qpos, kpos, scale=None):
    """out, lse of softmax(scale * q k^T, masked to kpos[j] <= qpos[i]) v.

    Query head h reads KV head h // (Hq // Hkv).  Rows are processed in
    blocks only to bound memory; every block is the plain formula.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, S, Sk, Hq, Hkv, Dqk, Dv = _check_heads(q, k, v)
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(Dqk)
    qpos = np.asarray(qpos)
    kpos = np.asarray(kpos)
    out = np.zeros((B, S, Hq, Dv))
    lse = np.zeros((B, Hq, S))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            kk = k[b, :, g, :]
            vv = v[b, :, g, :]
            for i0 in range(0, S, _ROW_BLOCK):
                i1 = min(S, i0 + _ROW_BLOCK)
                s = scale * (q[b, i0:i1, h, :] @ kk.T)
                visible = kpos[None, :] <= qpos[i0:i1, None]
                s = np.where(visible, s, -np.inf)
                m = s.max(axis=1)
                m_safe = np.where(np.isfinite(m), m, 0.0)
                p = np.exp(s - m_safe[:, None])
                l = p.sum(axis=1)
                with np.errstate(invalid="ignore", divide="ignore"):
                    o = (p @ vv) / l[:, None]
                    o = np.where(l[:, None] > 0, o, 0.0)
                    lse[b, h, i0:i1] = np.where(l > 0, m_safe + np.log(l), -np.inf)
                out[b, i0:i1, h, :] = o
    return out, lse


def masked_attention_bwd(q, k, v, out, lse, dout, qpos, kpos, scale=None):
    """dq, dk, dv of L = sum(out * dout) for the masked attention above.

    Textbook flash-attention backward: P = exp(s - lse), D_i = sum(dO_i*O_i),
    dV = P^T dO, dP = dO V^T, dS = P*(dP - D), dQ = scale dS K,
    dK = scale dS^T Q; K/V gradients of a group sum over its query heads.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    out = np.asarray(out, np.float64)
    dout = np.asarray(dout, np.float64)
    lse = np.asarray(lse, np.float64)
    B, S, Sk, Hq, Hkv, Dqk, Dv = _check_heads(q, k, v)
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(Dqk)
    qpos = np.asarray(qpos)
    kpos = np.asarray(kpos)
    Dsum = np.sum(dout * out, axis=3)  # [B,S,Hq]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            kk = k[b, :, g, :]
            vv = v[b, :, g, :]
            for i0 in range(0, S, _ROW_BLOCK):
                i1 = min(S, i0 + _ROW_BLOCK)
                qq = q[b, i0:i1, h, :]
                s = scale * (qq @ kk.T)
                visible = kpos[None, :] <= qpos[i0:i1, None]
                p = np.where(visible, np.exp(s - lse[b, h, i0:i1, None]), 0.0)
                do = dout[b, i0:i1, h, :]
                dv[b, :, g, :] += p.T @ do
                dp = do @ vv.T
                ds = p * (dp - Dsum[b, i0:i1, h][:, None])
                dq[b, i0:i1, h, :] = scale * (ds @ kk)
                dk[b, :, g, :] += scale * (ds.T @ qq)
    return dq, dk, dv


def causal_attention_fwd(q, k, v, scale=None):
    """Unsharded causal attention in natural token order (the dot-product
    reference the pages' unit test compares the sharded kernel against)."""
    S = q.shape[1]
    ar = np.arange(S)
    return masked_attention_fwd(q, k, v, ar, ar, scale)


def causal_attention_bwd(q, k, v, out, lse, dout, scale=None):
    S = q.shape[1]
    ar = np.arange(S)
    return masked_attention_bwd(q, k, v, out, lse, dout, ar, ar, scale)


def _shard_slots(S, cp, shard):
    n = S // cp
    return np.arange(shard * n, (shard + 1) * n)


def cp_attention_fwd(q, k, v, cp, load_balance=True, scale=None, shards=None):
    """Context-parallel attention on tensors that are ALREADY in reordered
    token order (slot order).  Each shard s owns query slots
    [s*S/cp, (s+1)*S/cp) and attends to the whole gathered K/V under the
    mask pos(key) <= pos(query).  Returns out [B,S,Hq,Dv] and lse [B,Hq,S]
    in slot order; rows of shards not in ``shards`` stay zero."""
    B, S = q.shape[:2]
    if S % cp != 0:
        raise ValueError("S must be a multiple of cp")
    pos = lb_positions(S, cp, load_balance)
    Dv = v.shape[3]
    Hq = q.shape[2]
    out = np.zeros((B, S, Hq, Dv))
    lse = np.zeros((B, Hq, S))
    for s in (range(cp) if shards is None else shards):
        rows = _shard_slots(S, cp, s)
        o, l = masked_attention_fwd(q[:, rows], k, v, pos[rows], pos, scale)
        out[:, rows] = o
        lse[:, :, rows] = l
    return out, lse


def cp_attention_bwd(q, k, v, out, lse, dout, cp, load_balance=True, scale=None):
    """Backward of ``cp_attention_fwd``: per-shard dq; dk and dv summed over
    every shard (the reduce-scatter that transposes the K/V all-gather)."""
    B, S = q.shape[:2]
    pos = lb_positions(S, cp, load_balance)
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for s in range(cp):
        rows = _shard_slots(S, cp, s)
        dqs, dks, dvs = masked_attention_bwd(
            q[:, rows], k, v, out[:, rows], lse[:, :, rows], dout[:, rows],
            pos[rows], pos, scale)
        dq[:, rows] = dqs
        dk += dks
        dv += dvs
    return dq, dk, dv



def mla_key(k_nope, k_rope):
    """Per-head key of MLA with a shared rope part: k_nope [B,S,H,Dn] (one per
    head) and k_rope [B,S,Dr] (one per token, used by every head) give
    [B,S,H,Dn+Dr], each head's nope columns followed by the rope key."""
    B, S, H, _ = k_nope.shape
    rope = np.broadcast_to(k_rope[:, :, None, :], (B, S, H, k_rope.shape[-1]))
    return np.concatenate([k_nope, rope], axis=-1)


def cp_attention_mla_fwd(q, k_nope, k_rope, v, cp, load_balance=True, scale=None):
    """``cp_attention_fwd`` with the key built by ``mla_key`` (scale defaults
    to 1/sqrt(Dn+Dr), the full key width)."""
    return cp_attention_fwd(q, mla_key(k_nope, k_rope), v, cp, load_balance, scale)


def cp_attention_mla_bwd(q, k_nope, k_rope, v, out, lse, dout, cp, load_balance=True, scale=None):
    """Gradients of ``cp_attention_mla_fwd``: dq, dk_nope [B,S,H,Dn], dk_rope
    [B,S,Dr] (the rope columns of the per-head key gradient summed over the
    heads, since every head reads the same rope key) and dv."""
    dq, dk, dv = cp_attention_bwd(q, mla_key(k_nope, k_rope), v, out, lse, dout, cp, load_balance, scale)
    Dn = k_nope.shape[-1]
    return dq, dk[..., :Dn], dk[..., Dn:].sum(axis=2), dv


def shard_pair_counts(S, cp, load_balance=True):
    """Number of visible (query, key) pairs each shard evaluates, counted by
    brute force over the mask -- the per-shard work the reorder balances."""
    pos = lb_positions(S, cp, load_balance)
    counts = []
    for s in range(cp):
        rows = _shard_slots(S, cp, s)
        counts.append(int(np.sum(pos[None, :] <= pos[rows][:, None])))
    return counts


def gqa_decode(q, kcache, vcache, lens, scale=None):
    """One query token per sequence: out[b,h] = softmax_t<lens[b](scale q.k_t) v_t.

    q [B,Hq,D], kcache/vcache [B,Hkv,Smax,D], lens [B] -> out [B,Hq,D]."""
    q = np.asarray(q, np.float64)
    kc = np.asarray(kcache, np.float64)
    vc = np.asarray(vcache, np.float64)
    B, Hq, D = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, Hq, vc.shape[3]))
    for b in range(B):
        n = int(lens[b])
        if n <= 0:
            continue
        for h in range(Hq):
            g = h // G
            s = scale * (kc[b, g, :n, :] @ q[b, h, :])
            s = s - s.max()
            p = np.exp(s)
            out[b, h] = (p @ vc[b, g, :n, :]) / p.sum()
    return out


def gqa_decode_int8(q, kq, vq, kscale, vscale, lens, scale=None):
    """Decode against an int8 KV cache: kq/vq int8 [B,Hkv,Smax,D] and
    kscale/vscale [B,Hkv,Smax]; the cached key (value) vector at position t is
    kq[b,g,t,:] * kscale[b,g,t].  Dequantised in float64, then ``gqa_decode``."""
    k = np.asarray(kq, np.float64) * np.asarray(kscale, np.float64)[..., None]
    v = np.asarray(vq, np.float64) * np.asarray(vscale, np.float64)[..., None]
    return gqa_decode(q, k, v, lens, scale)


def mla_decode(q, ckv, lens, dv=512, scale=None):
    """Absorbed-MLA decode: q [B,H,Dk] (each head's latent query, then its rope
    query), ckv [B,Smax,Dk] (each token's latent row: compressed KV, then rope
    key), lens [B] -> out [B,H,dv] in the latent space:
        out[b,h] = sum_{t<lens[b]} softmax_t(scale * q[b,h] . ckv[b,t]) ckv[b,t,:dv].
    scale defaults to 1/sqrt(192), the softmax scale of the attention the
    absorption comes from (a 128-column nope plus 64-column rope head)."""
    q = np.asarray(q, np.float64)
    ckv = np.asarray(ckv, np.float64)
    B, H, Dk = q.shape
    if ckv.shape[0] != B or ckv.shape[2] != Dk:
        raise ValueError("q and ckv shapes do not match")
    if scale is None:
        scale = 1.0 / math.sqrt(192.0)
    out = np.zeros((B, H, dv))
    for b in range(B):
        n = int(lens[b])
        if n <= 0:
            continue
        rows = ckv[b, :n, :]
        s = scale * (q[b] @ rows.T)  # [H, n]
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        out[b] = (p @ rows[:, :dv]) / p.sum(axis=1, keepdims=True)
    return out
