"""Oracle primitives: BF16 decode, RMSNorm, RoPE, SDPA, SwiGLU, argmax, accept walk, rollback.

Test infrastructure only (see the package docstring). Every function takes
plain NumPy arrays and a compute dtype `dt` (float32 by default, float64 for the
shadow run). No blocking, fusion or reordering beyond each definition.
"""
from __future__ import annotations

import numpy as np


class OracleError(ValueError):
    pass


# ---------------------------------------------------------------------------
# BF16 weights
# ---------------------------------------------------------------------------

def decode_bf16(bits, dt=np.float32):
    """BF16 bit patterns -> float: the 16 stored bits become the high half of an
    F32 word whose low half is zero.

    tensors.rs (hf2q 0.1.1), `decode_bf16_bytes_to_f32`: `f32_bits = bf16_bits << 16`.
    """
    b = np.asarray(bits, dtype=np.uint16)
    f = (b.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return f.astype(dt, copy=False)


def round_bf16(x, dt=np.float32):
    """Round to the nearest BF16 value, ties to an even last mantissa bit (the value a BF16
    store keeps), returned as floats. Finite inputs: the F32 word's low 16 bits decide
    against the halfway point 0x8000, with the stored half's lowest bit breaking ties."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    low = u & np.uint64(0xFFFF)
    high = u >> np.uint64(16)
    up = (low > np.uint64(0x8000)) | ((low == np.uint64(0x8000)) & ((high & np.uint64(1)) == 1))
    high = high + up.astype(np.uint64)
    return decode_bf16(high.astype(np.uint16), dt)


def decode_bf16_bytes(data: bytes, dt=np.float32):
    """Little-endian BF16 bytes -> floats; an odd byte count is rejected.

    tensors.rs (hf2q 0.1.1), `decode_bf16_bytes_to_f32` and its test
    `decode_bf16_bytes_rejects_odd_length`.
    """
    if len(data) % 2 != 0:
        raise OracleError(f"BF16 byte buffer of length {len(data)} is not even")
    u8 = np.frombuffer(bytes(data), dtype=np.uint8)
    lo = u8[0::2].astype(np.uint16)
    hi = u8[1::2].astype(np.uint16)
    return decode_bf16(lo | (hi << np.uint16(8)), dt)


# ---------------------------------------------------------------------------
# Normalisation, activations
# ---------------------------------------------------------------------------

def rmsnorm(x, w, eps, dt=np.float32):
    """y = x / sqrt(mean(x^2) + eps) * w over the last axis; w multiplies directly.

    mtp.rs (hf2q 0.1.1), `rms_norm_with_weight` (params buffer `[eps, hidden]`);
    tensors.rs, `DFlashLayerTensors` (F32 norm weights passed straight to `rms_norm_f32`).
    """
    x = np.asarray(x, dtype=dt)
    w = np.asarray(w, dtype=dt)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + dt(eps)) * w


def head_rmsnorm(x, w, n_heads, head_dim, eps, dt=np.float32):
    """Per-head RMSNorm: rows of `n_heads*head_dim` are normalised head by head with
    one shared `[head_dim]` weight.

    mtp.rs, `forward_full_attention` (`apply_q_or_k_per_head_rms_norm`);
    tensors.rs, `DFlashLayerTensors::q_norm` / `k_norm` (qwen3-style).
    """
    x = np.asarray(x, dtype=dt)
    lead = x.shape[:-1]
    xh = x.reshape(lead + (n_heads, head_dim))
    return rmsnorm(xh, w, eps, dt).reshape(lead + (n_heads * head_dim,))


def sigmoid(z, dt=np.float32):
    z = np.asarray(z, dtype=dt)
    return dt(1) / (dt(1) + np.exp(-z))


def silu(z, dt=np.float32):
    """silu(z) = z * sigmoid(z) (SwiGLU activation of the gate projection)."""
    z = np.asarray(z, dtype=dt)
    return z * sigmoid(z, dt)


def linear(x, w_bits, dt=np.float32):
    """y = x @ W^T for a row-major BF16 weight W[out, in] and F32 activations x[.., in].

    tensors.rs, `DFlashLayerTensors` (row-major `[out, in]` BF16, consumed by
    BF16-weight x F32-activation matmuls); mtp.rs `apply_linear_projection_f32`.
    """
    W = decode_bf16(w_bits, dt)
    return np.asarray(x, dtype=dt) @ W.T


def swiglu(x, wg_bits, wu_bits, wd_bits, dt=np.float32):
    """down( silu(gate x) * (up x) ).

    tensors.rs, `DFlashLayerTensors::mlp_gate/mlp_up/mlp_down`; mtp.rs,
    `forward_ffn_residual` (dense SwiGLU FFN).
    """
    g = linear(x, wg_bits, dt)
    u = linear(x, wu_bits, dt)
    return linear(silu(g, dt) * u, wd_bits, dt)


# ---------------------------------------------------------------------------
# Rotary position embedding
# ---------------------------------------------------------------------------

def rope_cos_sin(pos, rotary_dim, theta, dt=np.float32):
    """cos/sin of angle pos * theta^(-2j/r), j = 0..r/2-1, computed in float64 and
    rounded to `dt`.

    mtp.rs, `forward_full_attention` (`apply_imrope` with `rotary_dim`, `rope_theta`).
    Text-only positions make all four IMROPE ids equal, which is plain RoPE.
    """
    pos = np.asarray(pos, dtype=np.float64).reshape(-1)
    half = rotary_dim // 2
    j = np.arange(half, dtype=np.float64)
    inv_freq = float(theta) ** (-2.0 * j / rotary_dim)
    ang = pos[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(dt), np.sin(ang).astype(dt)


def rope(x, pos, rotary_dim, theta, dt=np.float32):
    """Rotate-half RoPE on x[T, n_heads, d] at positions pos[T]: pairs (i, i + r/2)
    for i < r/2 are rotated by the pair's angle; dims >= r pass through.
    """
    x = np.asarray(x, dtype=dt)
    T = x.shape[0]
    c, s = rope_cos_sin(pos, rotary_dim, theta, dt)
    c = c.reshape(T, 1, -1)
    s = s.reshape(T, 1, -1)
    half = rotary_dim // 2
    out = x.copy()
    x1 = x[..., :half]
    x2 = x[..., half:rotary_dim]
    out[..., :half] = x1 * c - x2 * s
    out[..., half:rotary_dim] = x2 * c + x1 * s
    return out


def qk_norm_rope(x, w, pos, n_heads, head_dim, eps, rotary_dim, theta, dt=np.float32):
    """Projected q or k rows x[T, n_heads*head_dim] (one row may come unbatched) ->
    [T, n_heads, head_dim], T = len(pos): per-head RMSNorm
    with the shared `[head_dim]` weight first, then RoPE at the rows' positions pos[T].

    mtp.rs, `forward_full_attention`: the per-head q/k RMSNorm is applied to the projections and
    `apply_imrope` rotates the normed heads; tensors.rs, `DFlashLayerTensors::q_norm` / `k_norm`
    (qwen3-style per-head norms of the drafter layer).
    """
    T = np.size(pos)
    x = np.asarray(x, dtype=dt).reshape(T, n_heads * head_dim)
    normed = head_rmsnorm(x, w, n_heads, head_dim, eps, dt)
    return rope(normed.reshape(T, n_heads, head_dim), pos, rotary_dim, theta, dt)


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def sdpa(q, k, v, mask=None, dt=np.float32):
    """softmax(q k^T / sqrt(d)) v with grouped KV heads.

    q[T, n_q, d], k/v[S, n_kv, d]; query head h reads KV head h // (n_q / n_kv).
    `mask[T, S]` (bool, True = may attend) is optional.
    mtp.rs, `forward_full_attention` (`apply_sdpa_with_kv_cache`).
    """
    q = np.asarray(q, dtype=dt)
    k = np.asarray(k, dtype=dt)
    v = np.asarray(v, dtype=dt)
    T, n_q, d = q.shape
    S, n_kv, _ = k.shape
    if n_q % n_kv != 0:
        raise OracleError("n_q must be a multiple of n_kv")
    rep = n_q // n_kv
    scale = dt(1.0 / np.sqrt(d))
    out = np.zeros((T, n_q, d), dtype=dt)
    for h in range(n_q):
        kh = k[:, h // rep, :]
        vh = v[:, h // rep, :]
        s = (q[:, h, :] @ kh.T) * scale                      # [T, S]
        if mask is not None:
            s = np.where(mask, s, -np.inf)
        m = np.max(s, axis=1, keepdims=True)
        p = np.exp(s - m)
        out[:, h, :] = (p @ vh) / np.sum(p, axis=1, keepdims=True)
    return out


# ---------------------------------------------------------------------------
# Argmax over the vocabulary
# ---------------------------------------------------------------------------

def argmax_top2(logits):
    """Per row: index of the largest logit (lowest index among exact ties), the top
    value and the second-largest value (equal to the top when the max is tied).

    qwen35_orchestrator.rs, step 5 (`per_position_argmax_from_normed_hidden`).
    """
    L = np.atleast_2d(np.asarray(logits))
    top1 = np.max(L, axis=1)
    idx = np.array([int(np.flatnonzero(L[r] == top1[r])[0]) for r in range(L.shape[0])],
                   dtype=np.int64)
    if L.shape[1] < 2:
        top2 = np.full_like(top1, -np.inf)
    else:
        top2 = -np.sort(-L, axis=1)[:, 1]
    return idx, top1, top2


def lm_head_logits(x, w_bits, dt=np.float32, v0=0, v1=None):
    """Logits x @ W_lm[v0:v1]^T over a slice of the vocabulary rows."""
    return linear(x, w_bits[v0:v1], dt)


def lm_head_argmax(x, w_bits, dt=np.float32, chunk=16384):
    """argmax_v of x @ W_lm^T per row, without keeping all logits: the vocabulary is
    visited in order in slices, each logit being a full dot product.

    qwen35_orchestrator.rs, step 5; mtp.rs, `forward_shared_head` (lm_head).
    Returns (idx, top1, top2) per row.
    """
    x = np.atleast_2d(np.asarray(x, dtype=dt))
    V = w_bits.shape[0]
    R = x.shape[0]
    best = np.full(R, -np.inf, dtype=np.float64)
    second = np.full(R, -np.inf, dtype=np.float64)
    bidx = np.zeros(R, dtype=np.int64)
    for v0 in range(0, V, chunk):
        L = lm_head_logits(x, w_bits, dt, v0, min(V, v0 + chunk))
        i, t1, t2 = argmax_top2(L)
        for r in range(R):
            if t1[r] > best[r]:
                second[r] = max(best[r], t2[r])
                best[r] = t1[r]
                bidx[r] = v0 + i[r]
            else:
                second[r] = max(second[r], t1[r])
    return bidx, best, second


# ---------------------------------------------------------------------------
# Greedy accept walk and KV rollback
# ---------------------------------------------------------------------------

def accept_walk(drafts, target, eos=()):
    """Greedy accept-prefix walk of one sequence.

    drafts[K] are the drafter's argmaxes for block positions 1..K; target[K+1] are the
    verifier's argmaxes over [last_token, drafts...]. accept_count a = length of the
    longest prefix with drafts[i] == target[i]; the committed tokens are drafts[:a]
    followed by the verifier's free token target[a]; they are cut after the first EOS
    id (hit_eos = 1). rollback = K - a, independent of the EOS cut.

    qwen35_orchestrator.rs, module doc "Greedy accept-walk consistency invariant" and
    the loop's steps 7-9 (`step_round_from_argmaxes`, `rollback = drafts.len() -
    accept_count`, committed tokens never empty).
    Returns (committed list, accept_count, hit_eos, rollback).
    """
    drafts = [int(t) for t in drafts]
    target = [int(t) for t in target]
    K = len(drafts)
    if len(target) != K + 1:
        raise OracleError("target must hold K+1 argmaxes")
    a = 0
    while a < K and drafts[a] == target[a]:
        a += 1
    committed = drafts[:a] + [target[a]]
    eos = set(int(e) for e in eos)
    hit = 0
    for i, t in enumerate(committed):
        if t in eos:
            committed = committed[: i + 1]
            hit = 1
            break
    return committed, a, hit, K - a


def kv_rollback(seq_len, n):
    """Discard the last n positions of a KV cache: seq_len - n, rejected if n > seq_len.

    qwen35_orchestrator.rs, step 8 (`target.rollback_kv(rollback)`) and the
    "KV cache rollback overflow" error.
    """
    seq_len, n = int(seq_len), int(n)
    if n < 0 or n > seq_len:
        raise OracleError(f"rollback of {n} positions exceeds seq_len {seq_len}")
    return seq_len - n
