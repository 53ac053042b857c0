"""Oracle MTP (NextN) single-token draft step, dense or MoE FFN, chained 1..N steps.

Test infrastructure only (see the package docstring).

mtp.rs (hf2q 0.1.1), `MtpWeights::forward_draft_with_hidden`:
    x      = eh_embed . rmsnorm(embed_t, enorm, 1e-6) + eh_hidden . rmsnorm(prev_hidden, hnorm, 1e-6)
                                                         (`project_embedding_and_hidden`)
    xn     = rmsnorm(x, attn_norm)
    q,k,v  = xn Wq^T, xn Wk^T, xn Wv^T;  gate = xn Wgate^T (when present)
    q, k   = rope(headnorm(q), pos), rope(headnorm(k), pos)
    K/V appended at pos; o = softmax(q K[0..pos]^T / sqrt(d)) V[0..pos]
    o      = o * sigmoid(gate)                           (`apply_sigmoid_gate_multiply`)
    h1     = x + o Wo^T                                   (fused residual + post-attn norm)
    hidden = h1 + FFN(rmsnorm(h1, post_attn_norm))        (`forward_ffn_residual`)
    logits = rmsnorm(hidden, shared_head_norm) lm_head^T  (`forward_shared_head`)
Chained steps feed (hidden, embedding of the step's argmax) into the next step at
pos + 1 (`forward_draft_with_hidden` doc: K=N chaining).

MoE FFN (mtp.rs `MtpFfnWeightsGpu::Moe`; routing details are not on the page, read
as): router softmax over all experts, the top-k by probability (lower index first on
ties) renormalised to sum one, weighted sum of the chosen experts' SwiGLU, plus one
shared SwiGLU expert scaled by sigmoid(x . w_shared_gate).
"""
from __future__ import annotations

import numpy as np

from . import stochastic
from .core import (OracleError, decode_bf16, linear, lm_head_argmax, qk_norm_rope, rmsnorm, sdpa,
                   sigmoid, swiglu)


def moe_route(x, router_bits, top_k, dt=np.float32):
    """(expert ids, weights): softmax over router logits, top-k, renormalised."""
    logits = linear(x, router_bits, dt)
    m = np.max(logits)
    p = np.exp(logits - m)
    p = p / np.sum(p)
    order = sorted(range(p.shape[0]), key=lambda e: (-float(p[e]), e))[:top_k]
    sel = np.array(order, dtype=np.int64)
    wsel = p[sel] / np.sum(p[sel])
    return sel, wsel.astype(dt)


def route_margin(x, router_bits, top_k, dt=np.float32):
    """Gap between the top_k-th and (top_k+1)-th largest router logits (inf when every expert
    is chosen): how far the expert choice is from a tie."""
    logits = np.sort(np.asarray(linear(x, router_bits, dt), np.float64))[::-1]
    if top_k >= logits.shape[0]:
        return float("inf")
    return float(logits[top_k - 1] - logits[top_k])


def moe_ffn(x, w, top_k, dt=np.float32):
    sel, ws = moe_route(x, w["router"], top_k, dt)
    out = np.zeros_like(np.asarray(x, dt))
    for e, we in zip(sel, ws):
        out = out + we * swiglu(x, w["exp_g"][e], w["exp_u"][e], w["exp_d"][e], dt)
    sg = sigmoid(linear(x, w["sh_gate"], dt), dt)            # [1]
    out = out + sg[0] * swiglu(x, w["sh_g"], w["sh_u"], w["sh_d"], dt)
    return out, sel, ws


def mtp_step(cfg, w, k_cache, v_cache, pos, prev_hidden, token, dt=np.float32):
    """One MTP draft step for one sequence. k_cache/v_cache [n_kv, cap, d] are updated
    at `pos`. Returns (hidden [H], argmax id, top1, top2, logits-free info dict)."""
    H, nq, nkv, d = cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    eps, theta, rot = cfg.rms_eps, cfg.rope_theta, cfg.rot
    if pos + 1 > k_cache.shape[1]:
        raise OracleError("MTP KV slot capacity exceeded")
    e = decode_bf16(w["embed"][int(token)], dt)
    x = (linear(rmsnorm(e, w["enorm"], 1e-6, dt), w["eh_embed"], dt)
         + linear(rmsnorm(np.asarray(prev_hidden, dt), w["hnorm"], 1e-6, dt), w["eh_hidden"], dt))
    xn = rmsnorm(x, w["attn_norm"], eps, dt)
    q = qk_norm_rope(linear(xn, w["wq"], dt), w["q_norm"], [pos], nq, d, eps, rot, theta, dt)
    k = qk_norm_rope(linear(xn, w["wk"], dt), w["k_norm"], [pos], nkv, d, eps, rot, theta, dt)
    v = linear(xn, w["wv"], dt)
    k_cache[:, pos, :] = k[0]
    v_cache[:, pos, :] = v.reshape(nkv, d)
    keys = np.asarray(k_cache[:, :pos + 1, :], dt).transpose(1, 0, 2)
    vals = np.asarray(v_cache[:, :pos + 1, :], dt).transpose(1, 0, 2)
    o = sdpa(q, keys, vals, None, dt).reshape(nq * d)
    if w.get("w_gate") is not None:
        o = o * sigmoid(linear(xn, w["w_gate"], dt), dt)
    h1 = x + linear(o, w["wo"], dt)
    fin = rmsnorm(h1, w["post_norm"], eps, dt)
    info = {}
    if w.get("router") is not None:
        f, sel, ws = moe_ffn(fin, w, cfg.top_k, dt)
        info["experts"], info["expert_w"] = sel, ws
        info["route_gap"] = route_margin(fin, w["router"], cfg.top_k, dt)
    else:
        f = swiglu(fin, w["wg"], w["wu"], w["wd"], dt)
    hidden = h1 + f
    xh = rmsnorm(hidden, w["shared_head_norm"], eps, dt)
    info["head_in"] = xh
    idx, t1, t2 = lm_head_argmax(xh[None, :], w["lm_head"], dt)
    return hidden, int(idx[0]), float(t1[0]), float(t2[0]), info


def mtp_forward_draft(cfg, w, cache_k, cache_v, seq_len, prev_hidden, tokens, n_steps,
                      dt=np.float32):
    """Chained MTP draft: n_steps steps per sequence. cache_k/cache_v [B, n_kv, cap, d]
    (updated), seq_len [B]. Returns hidden [n_steps, B, H], argmax [n_steps, B],
    top1/top2 [n_steps, B], new seq_len, per-step info."""
    B = len(tokens)
    hid = np.zeros((n_steps, B, cfg.hidden), dtype=dt)
    am = np.zeros((n_steps, B), dtype=np.int64)
    t1s = np.zeros((n_steps, B))
    t2s = np.zeros((n_steps, B))
    seq = np.asarray(seq_len, dtype=np.int64).copy()
    infos = []
    for b in range(B):
        h, tok = np.asarray(prev_hidden[b], dt), int(tokens[b])
        for s in range(n_steps):
            h, tok, t1, t2, info = mtp_step(cfg, w, cache_k[b], cache_v[b], int(seq[b]), h, tok, dt)
            seq[b] += 1
            hid[s, b], am[s, b], t1s[s, b], t2s[s, b] = h, tok, t1, t2
            infos.append(info)
    return hid, am, t1s, t2s, seq, infos


def mtp_forward_draft_sampled(cfg, w, cache_k, cache_v, seq_len, prev_hidden, tokens, n_steps,
                              temperature, u_draft, dt=np.float32):
    """Chained MTP draft at temperature T > 0 (the MTP K=1 path of the non-greedy variant,
    qwen35_orchestrator.rs module doc "Non-greedy (Metropolis-Hastings) is out of scope here"):
    every step's draft is drawn from softmax(logits / T) with u_draft[s, b] and fed to the next
    step in place of the argmax. Returns hidden [n_steps, B, H], drafts [n_steps, B],
    logits [n_steps, B, V] and the new seq_len."""
    B = len(tokens)
    hid = np.zeros((n_steps, B, cfg.hidden), dtype=dt)
    drafts = np.zeros((n_steps, B), dtype=np.int64)
    logits = np.zeros((n_steps, B, cfg.vocab), dtype=dt)
    seq = np.asarray(seq_len, dtype=np.int64).copy()
    for b in range(B):
        h, tok = np.asarray(prev_hidden[b], dt), int(tokens[b])
        for s in range(n_steps):
            h, _, _, _, info = mtp_step(cfg, w, cache_k[b], cache_v[b], int(seq[b]), h, tok, dt)
            seq[b] += 1
            lg = linear(info["head_in"], w["lm_head"], dt)
            tok = stochastic.sample_draft(lg, temperature, u_draft[s][b])
            hid[s, b], drafts[s, b], logits[s, b] = h, tok, lg
    return hid, drafts, logits, seq
