"""Oracle DFlash drafter forward over a K+1 block and the whole draft round.

Test infrastructure only (see the package docstring).

The drafter's layer math lives in a source file the pages name but do not
contain (`dflash/forward.rs`); what follows is the plainest reading of
tensors.rs (`DFlashLayerTensors`, `DFlashModelTensors`: fc + hidden_norm over the
concatenated target hiddens, per layer input/post-attention RMSNorm, q/k/v/o with
per-head q/k RMSNorm, SwiGLU, final norm) and qwen35_orchestrator.rs (the block
`[last_token, mask x K]`, the drafter cache that only tracks committed context rows,
`h_final` already final-normed, argmax of positions 1..K, accept walk, rollback):

    h     = E[block_ids]                                  (embedding rows, F32)
    h_ctx = rmsnorm(X_new @ fc^T, hidden_norm)            (new context rows only)
    per layer:
        xn  = rmsnorm(h, input_norm)
        q   = rope(headnorm(xn Wq^T, q_norm), ctx_len + i)
        k_b = rope(headnorm(xn Wk^T, k_norm), ctx_len + i);  v_b = xn Wv^T
        k_c = rope(headnorm(h_ctx Wk^T, k_norm), absolute);  v_c = h_ctx Wv^T  -> cache
        o   = softmax(q [K_cache; k_b]^T / sqrt(d)) [V_cache; v_b]   (block not causal)
        h  += o Wo^T
        h  += swiglu(rmsnorm(h, post_norm))
    h_final = rmsnorm(h, final_norm)

`cfg` is any object with the attributes hidden, n_q_heads, n_kv_heads, head_dim,
rms_eps, rope_theta, rot (rotary dim), causal_block; weights are dicts of NumPy
arrays (BF16 as uint16 bit patterns, norms as float32).
"""
from __future__ import annotations

import numpy as np

from . import stochastic
from .core import (OracleError, accept_walk, decode_bf16, kv_rollback, linear, lm_head_argmax,
                   qk_norm_rope, rmsnorm, round_bf16, sdpa, swiglu)


def fc_hidden_norm(cfg, w, x_new, dt=np.float32):
    """h_ctx = rmsnorm(concat(target hiddens) @ fc^T) * hidden_norm for new context rows.

    tensors.rs, `DFlashModelTensors::fc` ("projects concatenated target hidden states
    into draft hidden space") and `hidden_norm` ("RMSNorm applied to fc output").
    """
    return rmsnorm(linear(x_new, w["fc"], dt), w["hidden_norm"], cfg.rms_eps, dt)


def dflash_layer(cfg, lw, h, h_ctx, k_cache, v_cache, ctx0, dt=np.float32):
    """One drafter decoder layer for one sequence; `cfg.kv_bf16` (optional, default off)
    selects a BF16 KV cache: every K/V value the attention reads, cached or of the block, is
    rounded to BF16 when it is produced (the verifier of qwen35_orchestrator.rs's "Output
    divergence" note runs its attention in BF16).

    h[blk, H] block residual stream; h_ctx[n_new, H] normed context rows; k_cache,
    v_cache [n_kv, cap, d] of this layer (modified in place: rows ctx0..ctx0+n_new
    receive the context K/V). Returns the new residual stream.
    """
    bf16_kv = bool(getattr(cfg, "kv_bf16", False))
    H, nq, nkv, d = cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    eps, theta, rot = cfg.rms_eps, cfg.rope_theta, cfg.rot
    blk = h.shape[0]
    n_new = h_ctx.shape[0]
    cap = k_cache.shape[1]
    if ctx0 + n_new > cap:
        raise OracleError("KV cache capacity exceeded")
    # Context stream: K/V of the newly committed rows, appended at their positions.
    if n_new:
        pos_c = np.arange(ctx0, ctx0 + n_new)
        kc = qk_norm_rope(linear(h_ctx, lw["wk"], dt), lw["k_norm"], pos_c, nkv, d, eps, rot,
                          theta, dt)
        vc = linear(h_ctx, lw["wv"], dt)
        if bf16_kv:                         # a BF16 KV cache keeps the rounded values
            kc, vc = round_bf16(kc, dt), round_bf16(vc, dt)
        k_cache[:, ctx0:ctx0 + n_new, :] = kc.transpose(1, 0, 2)
        v_cache[:, ctx0:ctx0 + n_new, :] = vc.reshape(n_new, nkv, d).transpose(1, 0, 2)
    ctx_len = ctx0 + n_new
    # Block stream.
    xn = rmsnorm(h, lw["input_norm"], eps, dt)
    pos_b = np.arange(ctx_len, ctx_len + blk)
    q = qk_norm_rope(linear(xn, lw["wq"], dt), lw["q_norm"], pos_b, nq, d, eps, rot, theta, dt)
    kb = qk_norm_rope(linear(xn, lw["wk"], dt), lw["k_norm"], pos_b, nkv, d, eps, rot, theta, dt)
    vb = linear(xn, lw["wv"], dt)
    if bf16_kv:                             # block K/V at the precision of the cache
        kb, vb = round_bf16(kb, dt), round_bf16(vb, dt)
    keys = np.concatenate([np.asarray(k_cache[:, :ctx_len, :], dt).transpose(1, 0, 2), kb], 0)
    vals = np.concatenate([np.asarray(v_cache[:, :ctx_len, :], dt).transpose(1, 0, 2),
                           vb.reshape(blk, nkv, d)], 0)
    mask = None
    if getattr(cfg, "causal_block", 0):
        mask = np.ones((blk, ctx_len + blk), dtype=bool)
        for i in range(blk):
            mask[i, ctx_len + i + 1:] = False
    o = sdpa(q, keys, vals, mask, dt).reshape(blk, nq * d)
    h = h + linear(o, lw["wo"], dt)
    h = h + swiglu(rmsnorm(h, lw["post_norm"], eps, dt), lw["wg"], lw["wu"], lw["wd"], dt)
    return h


def dflash_block_forward(cfg, w, cache_k, cache_v, seq_len, block_ids, target_hidden, n_new,
                         dt=np.float32, embed_scale=1.0):
    """Drafter forward over the block of every sequence.

    cache_k/cache_v: per layer [B, n_kv, cap, d] arrays, updated in place with the
    context rows; seq_len [B] is returned advanced by n_new. Returns
    (h_final [B, blk, H], new seq_len).
    """
    block_ids = np.asarray(block_ids)
    B, blk = block_ids.shape
    seq = np.asarray(seq_len, dtype=np.int64).copy()
    out = np.zeros((B, blk, cfg.hidden), dtype=dt)
    for b in range(B):
        nn = int(n_new[b])
        ctx0 = int(seq[b])
        h = decode_bf16(w["embed"][block_ids[b]], dt) * dt(embed_scale)
        h_ctx = fc_hidden_norm(cfg, w, np.asarray(target_hidden[b, :nn], dt), dt)
        for li, lw in enumerate(w["layers"]):
            h = dflash_layer(cfg, lw, h, h_ctx, cache_k[li][b], cache_v[li][b], ctx0, dt)
        out[b] = rmsnorm(h, w["final_norm"], cfg.rms_eps, dt)
        seq[b] = ctx0 + nn
    return out, seq


def draft_round(cfg, w, cache_k, cache_v, seq_len, block_ids, target_hidden, n_new, target,
                eos, target_seq_len, dt=np.float32):
    """One DFlash draft round: forward, per-position argmax, drafts = argmax[1..K],
    greedy accept walk against the target argmaxes, rollback of the verifier's KV.

    qwen35_orchestrator.rs, the per-round loop (steps 1-9 of the module doc).
    `target_seq_len` is the verifier cache length after its K+1 verify positions.
    """
    h_final, seq = dflash_block_forward(cfg, w, cache_k, cache_v, seq_len, block_ids,
                                        target_hidden, n_new, dt)
    B, blk, H = h_final.shape
    idx, top1, top2 = lm_head_argmax(h_final.reshape(B * blk, H), w["lm_head"], dt)
    idx = idx.reshape(B, blk)
    res = dict(h_final=h_final, seq_len=seq, argmax=idx, top1=top1.reshape(B, blk),
               top2=top2.reshape(B, blk), drafts=idx[:, 1:], committed=[], accept=[], hit_eos=[],
               rollback=[], target_seq_len=[])
    for b in range(B):
        c, a, hit, rb = accept_walk(idx[b, 1:], target[b], eos)
        res["committed"].append(c)
        res["accept"].append(a)
        res["hit_eos"].append(hit)
        res["rollback"].append(rb)
        res["target_seq_len"].append(kv_rollback(target_seq_len[b], rb))
    return res


def draft_round_stochastic(cfg, w, cache_k, cache_v, seq_len, block_ids, target_hidden, n_new,
                           target_logits, temperature, u_draft, u_accept, u_sample, eos,
                           target_seq_len, dt=np.float32):
    """The non-greedy draft round (qwen35_orchestrator.rs, module doc "Non-greedy
    (Metropolis-Hastings) is out of scope here": stochastic acceptance replaces the greedy walk
    at step 11): the drafter forward, the lm_head logits of every block position, each draft
    i = 1..K drawn from softmax(logits_i / T) with u_draft[b, i-1], then the speculative-sampling
    accept step against the verifier's logits target_logits [B, K+1, V] with u_accept [B, K]
    and u_sample [B], and the rollback of the verifier's KV by K - accept_count.
    """
    h_final, seq = dflash_block_forward(cfg, w, cache_k, cache_v, seq_len, block_ids,
                                        target_hidden, n_new, dt)
    B, blk, H = h_final.shape
    K = blk - 1
    logits = np.stack([linear(h_final[b], w["lm_head"], dt) for b in range(B)])   # [B, blk, V]
    res = dict(h_final=h_final, seq_len=seq, logits=logits, drafts=[], committed=[], accept=[],
               hit_eos=[], rollback=[], target_seq_len=[], info=[])
    for b in range(B):
        drafts = [stochastic.sample_draft(logits[b, 1 + i], temperature, u_draft[b][i])
                  for i in range(K)]
        c, a, hit, rb, info = stochastic.accept_stochastic(logits[b, 1:], target_logits[b], drafts,
                                                           temperature, u_accept[b], u_sample[b],
                                                           eos)
        res["drafts"].append(drafts)
        res["committed"].append(c)
        res["accept"].append(a)
        res["hit_eos"].append(hit)
        res["rollback"].append(rb)
        res["target_seq_len"].append(kv_rollback(target_seq_len[b], rb))
        res["info"].append(info)
    return res
