"""Pins of the oracle's DFlash forward, MTP step and MoE routing.

Closed forms from special weights (zero or identity projections), an
incremental-versus-one-shot invariant of the context cache, a float64 shadow, and
planted mistakes that the pins must catch. No expected value here comes from the
CUDA library.
"""
import copy
import inspect
import math

import numpy as np
import pytest

from oracle import core, dflash, mtp
from tests import oracle_fixtures as fx


def _ids(cfg, B, rng):
    ids = np.full((B, cfg.K + 1), cfg.vocab - 1, dtype=np.int64)
    ids[:, 0] = rng.integers(2, cfg.vocab - 1, size=B)
    return ids


def _embed_f64(w, ids):
    return core.decode_bf16(w["embed"][ids], np.float64)


# --------------------------------------------------------------- DFlash forward

def test_zero_output_projections_keep_embedding():
    """wo = wd = 0: the residual stream stays E[ids], so h_final = rmsnorm(E[ids], final_norm);
    the context V rows are h_ctx Wv^T, which is h_ctx's first kv_total columns for Wv = I and
    h_ctx = rmsnorm(X[:, :H], hidden_norm) for fc = [I 0]."""
    cfg = fx.dflash_cfg()
    w = fx.random_dflash_weights(cfg)
    lw = w["layers"][0]
    lw["wo"] = fx.zeros_bits(cfg.hidden, cfg.q_total)
    lw["wd"] = fx.zeros_bits(cfg.hidden, cfg.intermediate)
    lw["wv"] = fx.eye_bits(cfg.kv_total, cfg.hidden)
    w["fc"] = fx.eye_bits(cfg.hidden, cfg.fc_in)
    rng = np.random.default_rng(3)
    B, ctx, nn = 2, 5, 3
    ks, vs = fx.random_cache(1, B, cfg.n_kv_heads, cfg.head_dim, ctx, ctx + nn + 1)
    ids = _ids(cfg, B, rng)
    X = rng.standard_normal((B, nn, cfg.fc_in))
    out, seq = dflash.dflash_block_forward(cfg, w, ks, vs, [ctx, ctx], ids, X, [nn, nn - 1],
                                           np.float64)
    e = _embed_f64(w, ids)
    want = e / np.sqrt(np.mean(e * e, axis=-1, keepdims=True) + 1e-6) * w["final_norm"]
    assert np.allclose(out, want, rtol=1e-12)
    assert list(seq) == [ctx + nn, ctx + nn - 1]
    for b, n_b in enumerate([nn, nn - 1]):
        xc = X[b, :n_b, :cfg.hidden]
        hc = xc / np.sqrt(np.mean(xc * xc, axis=-1, keepdims=True) + 1e-6) * w["hidden_norm"]
        got_v = vs[0][b, 0, ctx:ctx + n_b, :]
        assert np.allclose(got_v, hc[:, :cfg.kv_total], rtol=1e-6)


def test_zero_queries_attend_uniformly():
    """Wq = 0 makes q = 0, so every query averages V over [cache rows incl. the new ones; block].
    With Wo = I (H = q_total), Wv = I and no FFN the output has a closed form."""
    cfg = fx.dflash_cfg(H=16, nq=2, nkv=1, d=8)
    w = fx.random_dflash_weights(cfg, seed=5)
    lw = w["layers"][0]
    lw["wq"] = fx.zeros_bits(cfg.q_total, cfg.hidden)
    lw["wo"] = fx.eye_bits(cfg.hidden, cfg.q_total)
    lw["wv"] = fx.eye_bits(cfg.kv_total, cfg.hidden)
    lw["wd"] = fx.zeros_bits(cfg.hidden, cfg.intermediate)
    w["fc"] = fx.eye_bits(cfg.hidden, cfg.fc_in)
    rng = np.random.default_rng(4)
    B, ctx, nn = 1, 6, 2
    ks, vs = fx.random_cache(1, B, 1, cfg.head_dim, ctx, ctx + nn, dtype=np.float64)
    v_cache_before = vs[0][0, 0, :ctx].copy()
    ids = _ids(cfg, B, rng)
    X = rng.standard_normal((B, nn, cfg.fc_in))
    out, _ = dflash.dflash_block_forward(cfg, w, ks, vs, [ctx], ids, X, [nn], np.float64)
    e = _embed_f64(w, ids)[0]
    xn = e / np.sqrt(np.mean(e * e, axis=-1, keepdims=True) + 1e-6) * lw["input_norm"]
    xc = X[0, :, :cfg.hidden]
    hc = xc / np.sqrt(np.mean(xc * xc, axis=-1, keepdims=True) + 1e-6) * w["hidden_norm"]
    all_v = np.concatenate([v_cache_before, hc[:, :8], xn[:, :8]], 0)   # every key's value row
    mean_v = all_v.mean(0)
    h = e + np.concatenate([mean_v, mean_v])[None, :]                     # both q heads read kv head 0
    want = h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + 1e-6) * w["final_norm"]
    assert np.allclose(out[0], want, rtol=1e-10)


def test_context_rows_incremental_equals_one_shot():
    """Context rows are rotated at their absolute positions and the cache only tracks the
    consumed prefix: feeding rows in two rounds leaves the same cache as one round, and the
    block output after the second round equals the one-shot output."""
    cfg = fx.dflash_cfg(H=16, nq=2, nkv=1, d=8)
    w = fx.random_dflash_weights(cfg, n_layers=2, seed=7)
    rng = np.random.default_rng(8)
    ctx = 4
    ids = _ids(cfg, 1, rng)
    X = rng.standard_normal((1, 5, cfg.fc_in))
    ks1, vs1 = fx.random_cache(2, 1, 1, 8, ctx, 12)
    ks2, vs2 = copy.deepcopy(ks1), copy.deepcopy(vs1)
    out1, seq1 = dflash.dflash_block_forward(cfg, w, ks1, vs1, [ctx], ids, X, [5], np.float64)
    _, s = dflash.dflash_block_forward(cfg, w, ks2, vs2, [ctx], ids, X[:, :2], [2], np.float64)
    out2, seq2 = dflash.dflash_block_forward(cfg, w, ks2, vs2, s, ids, X[:, 2:], [3], np.float64)
    assert seq1[0] == seq2[0] == ctx + 5
    for l in range(2):
        assert np.allclose(ks1[l], ks2[l], rtol=1e-12, atol=1e-12)
        assert np.allclose(vs1[l], vs2[l], rtol=1e-12, atol=1e-12)
    assert np.allclose(out1, out2, rtol=1e-12)


def test_causal_block_flag_only_changes_earlier_rows():
    """With one layer, the last block row sees every key under both mask readings."""
    cfg = fx.dflash_cfg()
    cfgc = fx.dflash_cfg(causal=1)
    w = fx.random_dflash_weights(cfg, seed=9)
    rng = np.random.default_rng(10)
    ids = _ids(cfg, 1, rng)
    X = rng.standard_normal((1, 2, cfg.fc_in))
    ks, vs = fx.random_cache(1, 1, 1, 8, 3, 8)
    a, _ = dflash.dflash_block_forward(cfg, w, copy.deepcopy(ks), copy.deepcopy(vs), [3], ids, X, [2],
                                       np.float64)
    b, _ = dflash.dflash_block_forward(cfgc, w, ks, vs, [3], ids, X, [2], np.float64)
    assert np.allclose(a[0, -1], b[0, -1], rtol=1e-12)
    assert not np.allclose(a[0, 0], b[0, 0])


def test_dflash_f32_vs_f64_shadow():
    cfg = fx.dflash_cfg(H=64, nq=4, nkv=2, d=16, I=96, V=300, K=4)
    w = fx.random_dflash_weights(cfg, n_layers=2, seed=11)
    rng = np.random.default_rng(12)
    ids = _ids(cfg, 2, rng)
    X = rng.standard_normal((2, 3, cfg.fc_in)).astype(np.float32)
    ks, vs = fx.random_cache(2, 2, 2, 16, 20, 30)
    o32, _ = dflash.dflash_block_forward(cfg, w, copy.deepcopy(ks), copy.deepcopy(vs), [20, 20], ids,
                                         X, [3, 1], np.float32)
    o64, _ = dflash.dflash_block_forward(cfg, w, ks, vs, [20, 20], ids, X, [3, 1], np.float64)
    rel = np.max(np.abs(o32 - o64) / np.maximum(np.abs(o64), np.sqrt(np.mean(o64 ** 2))))
    assert rel < 1e-4


def test_draft_round_accept_and_rollback():
    cfg = fx.dflash_cfg(V=64, K=3)
    w = fx.random_dflash_weights(cfg, seed=13)
    rng = np.random.default_rng(14)
    ids = _ids(cfg, 2, rng)
    X = rng.standard_normal((2, 2, cfg.fc_in))
    ks, vs = fx.random_cache(1, 2, 1, 8, 4, 8)
    ref = dflash.dflash_block_forward(cfg, w, copy.deepcopy(ks), copy.deepcopy(vs), [4, 4], ids, X,
                                      [2, 2], np.float64)[0]
    # drafts = argmax of positions 1..K; targets agree on 2 then differ (seq 0), all (seq 1)
    logits = np.einsum("bph,vh->bpv", ref, core.decode_bf16(w["lm_head"], np.float64))
    am = logits.argmax(-1)
    tgt = np.stack([np.r_[am[0, 1:3], (am[0, 3] + 1) % 64, 7], np.r_[am[1, 1:], 9]])
    res = dflash.draft_round(cfg, w, ks, vs, [4, 4], ids, X, [2, 2], tgt, (), [20, 20], np.float64)
    assert list(res["argmax"].reshape(-1)) == list(am.reshape(-1))
    assert res["accept"] == [2, 3]
    assert res["rollback"] == [1, 0]
    assert res["target_seq_len"] == [19, 20]
    assert res["committed"][0] == list(am[0, 1:3]) + [int(tgt[0, 2])]


# --------------------------------------------------------------- MTP

def test_mtp_single_key_closed_form():
    """Empty slot (pos 0): attention over the one new key returns v, gated by sigmoid(gate).
    With eh_* = I, Wo = I, Wv = Wgate = I and no FFN, hidden = x + v * sigmoid(g)."""
    cfg = fx.mtp_cfg(H=16, nq=2, nkv=1, d=8)
    w = fx.random_mtp_weights(cfg, seed=1)
    H = cfg.hidden
    w["eh_embed"] = fx.eye_bits(H, H)
    w["eh_hidden"] = fx.eye_bits(H, H)
    w["wo"] = fx.eye_bits(H, cfg.q_total)
    w["wv"] = fx.eye_bits(cfg.kv_total, H)
    w["w_gate"] = fx.eye_bits(cfg.q_total, H)
    w["wd"] = fx.zeros_bits(H, cfg.intermediate)
    rng = np.random.default_rng(2)
    prev = rng.standard_normal(H)
    kc = np.zeros((1, 4, 8))
    vc = np.zeros((1, 4, 8))
    hidden, idx, t1, t2, _ = mtp.mtp_step(cfg, w, kc, vc, 0, prev, 7, np.float64)
    e = core.decode_bf16(w["embed"][7], np.float64)
    nrm = lambda a, g, eps: a / np.sqrt(np.mean(a * a) + eps) * g
    x = nrm(e, w["enorm"], 1e-6) + nrm(prev, w["hnorm"], 1e-6)
    xn = nrm(x, w["attn_norm"], 1e-6)
    v = xn[:8]
    o = np.concatenate([v, v]) / (1.0 + np.exp(-xn[:16]))
    want = x + o
    assert np.allclose(hidden, want, rtol=1e-10)
    assert np.allclose(vc[0, 0], v, rtol=1e-12)
    logits = core.decode_bf16(w["lm_head"], np.float64) @ nrm(want, w["shared_head_norm"], 1e-6)
    assert idx == int(np.argmax(logits))


def test_mtp_chain_feeds_hidden_and_argmax():
    cfg = fx.mtp_cfg()
    w = fx.random_mtp_weights(cfg, seed=3)
    rng = np.random.default_rng(4)
    kc = np.zeros((1, 1, 12, 8))
    vc = np.zeros((1, 1, 12, 8))
    kc[:, :, :5] = rng.standard_normal((1, 1, 5, 8))
    vc[:, :, :5] = rng.standard_normal((1, 1, 5, 8))
    prev = rng.standard_normal((1, cfg.hidden))
    k2, v2 = kc.copy(), vc.copy()
    hid, am, _, _, seq, _ = mtp.mtp_forward_draft(cfg, w, kc, vc, [5], prev, [3], 3, np.float64)
    assert seq[0] == 8
    h, tok = prev[0], 3
    for s in range(3):
        h, tok, _, _, _ = mtp.mtp_step(cfg, w, k2[0], v2[0], 5 + s, h, tok, np.float64)
        assert np.allclose(hid[s, 0], h) and am[s, 0] == tok


def test_mtp_f32_vs_f64_shadow():
    for cfg in (fx.mtp_cfg(H=64, nq=4, nkv=2, d=16, I=80, V=200),
                fx.mtp_cfg(H=64, nq=4, nkv=2, d=16, V=200, E=8, top_k=2, Ie=24, Is=24)):
        w = fx.random_mtp_weights(cfg, seed=5)
        rng = np.random.default_rng(6)
        k = rng.standard_normal((1, 2, 12, 16)).astype(np.float32)
        v = rng.standard_normal((1, 2, 12, 16)).astype(np.float32)
        prev = rng.standard_normal((1, 64)).astype(np.float32)
        a = mtp.mtp_forward_draft(cfg, w, k.copy(), v.copy(), [9], prev, [5], 2, np.float32)
        b = mtp.mtp_forward_draft(cfg, w, k.copy(), v.copy(), [9], prev, [5], 2, np.float64)
        rel = np.max(np.abs(a[0] - b[0]) / np.maximum(np.abs(b[0]), np.sqrt(np.mean(b[0] ** 2))))
        assert rel < 1e-4


def test_moe_route_hand_example():
    """Router logits [0, ln 2, ln 4, 0] (x = e_0): probs 1/8, 2/8, 4/8, 1/8; top-2 = {2, 1},
    renormalised weights 2/3, 1/3."""
    H = 4
    logits = [0.0, math.log(2), math.log(4), 0.0]
    # BF16 cannot hold ln 2 exactly; build the router from the BF16 values and derive
    # the exact expectation from those.
    router = fx.bf16_bits_rne(np.array([[l, 0, 0, 0] for l in logits], dtype=np.float32))
    lv = core.decode_bf16(router[:, 0], np.float64)
    x = np.array([1.0, 0, 0, 0])
    sel, ws = mtp.moe_route(x, router, 2, np.float64)
    assert list(sel) == [2, 1]
    p = np.exp(lv) / np.sum(np.exp(lv))
    assert np.allclose(ws, [p[2] / (p[2] + p[1]), p[1] / (p[2] + p[1])], rtol=1e-12)
    assert abs(ws[0] - 2.0 / 3.0) < 5e-3
    # a tie in probability goes to the lower expert index
    router2 = fx.bf16_bits_rne(np.array([[1, 0, 0, 0], [2, 0, 0, 0], [2, 0, 0, 0], [0, 0, 0, 0]],
                                        dtype=np.float32))
    sel2, ws2 = mtp.moe_route(x, router2, 1, np.float64)
    assert list(sel2) == [1] and ws2[0] == 1.0


def test_moe_single_expert_reduces_to_dense():
    cfg = fx.mtp_cfg(H=16, E=1, top_k=1, Ie=10, Is=6)
    w = fx.random_mtp_weights(cfg, seed=8)
    rng = np.random.default_rng(9)
    x = rng.standard_normal(16)
    out, sel, ws = mtp.moe_ffn(x, w, 1, np.float64)
    assert list(sel) == [0] and ws[0] == 1.0
    g = 1.0 / (1.0 + np.exp(-(core.decode_bf16(w["sh_gate"], np.float64) @ x)[0]))
    want = (core.swiglu(x, w["exp_g"][0], w["exp_u"][0], w["exp_d"][0], np.float64)
            + g * core.swiglu(x, w["sh_g"], w["sh_u"], w["sh_d"], np.float64))
    assert np.allclose(out, want, rtol=1e-12)


# --------------------------------------------------------------- whole-layer closed forms
#
# Two-dimensional heads (head_dim 2, so RoPE turns the one pair of a head by `position`
# radians), identity projections and norm weights that differ inside a rotation pair: the
# per-head norm weight then does not commute with the rotation, so the order "q/k RMSNorm,
# then RoPE" is fixed by the expected value. Every expected value below is worked out with
# scalar arithmetic on Python floats, following the layer as the pages describe it
# (tensors.rs `DFlashLayerTensors`: q_norm / k_norm per head, post_attention_layernorm between
# the attention residual and the MLP; mtp.rs `forward_full_attention`: per-head norm then
# `apply_imrope`; `forward_ffn_residual`: post-attention norm feeds the FFN, whose output is
# added to the attention residual).

Q_NORM2 = [1.9, 0.4]
K_NORM2 = [0.6, 1.7]


def _nrm(x, w, eps=1e-6):
    """RMSNorm of one row, element by element."""
    ms = sum(v * v for v in x) / len(x)
    r = 1.0 / math.sqrt(ms + eps)
    return [v * r * g for v, g in zip(x, w)]


def _turn(pair, angle):
    """Rotation of the pair (x0, x1) by `angle` radians: the rotate-half RoPE of a 2-dim head
    (inverse frequency theta^0 = 1)."""
    c, s = math.cos(angle), math.sin(angle)
    return [pair[0] * c - pair[1] * s, pair[1] * c + pair[0] * s]


def _silu(z):
    return z / (1.0 + math.exp(-z))


def _attend(q, keys, vals):
    """softmax(q . k / sqrt(2)) weighted sum of the value rows, for one 2-dim query."""
    sc = [(q[0] * k[0] + q[1] * k[1]) / math.sqrt(2.0) for k in keys]
    m = max(sc)
    e = [math.exp(v - m) for v in sc]
    z = sum(e)
    return [sum(e[j] * vals[j][t] for j in range(len(vals))) / z for t in range(2)]


def _reverse_bits(n):
    """BF16 [n, n] reversal permutation (row i selects input n-1-i)."""
    w = fx.zeros_bits(n, n)
    for i in range(n):
        w[i, n - 1 - i] = fx.ONE
    return w


def _dflash_two_dim_case():
    """One drafter layer, H = 4, two q heads sharing one KV head of dim 2, identity q/k/v, gate,
    up and down projections, Wo the reversal permutation J; two cached rows, one new context
    row, a block of two."""
    cfg = fx.dflash_cfg(H=4, nq=2, nkv=1, d=2, I=4, V=10, K=1, n_tl=2)
    w = fx.random_dflash_weights(cfg, seed=21)
    lw = w["layers"][0]
    lw["q_norm"] = np.array(Q_NORM2, np.float32)
    lw["k_norm"] = np.array(K_NORM2, np.float32)
    lw["post_norm"] = np.array([1.5, 0.7, 1.2, 0.9], np.float32)
    for name, (r, c) in dict(wq=(4, 4), wk=(2, 4), wv=(2, 4), wg=(4, 4), wu=(4, 4),
                             wd=(4, 4)).items():
        lw[name] = fx.eye_bits(r, c)
    lw["wo"] = _reverse_bits(4)
    w["fc"] = fx.eye_bits(4, 8)
    rng = np.random.default_rng(22)
    ks, vs = fx.random_cache(1, 1, 1, 2, 2, 6, seed=23, dtype=np.float64)
    X = rng.standard_normal((1, 1, 8))
    ids = np.array([[3, 9]])
    return cfg, w, ks, vs, X, ids


def _dflash_two_dim_expected(w, ks, vs, X, ids):
    lw = w["layers"][0]
    f = lambda a: [float(v) for v in np.asarray(a).reshape(-1)]
    k_cached = [f(ks[0][0, 0, j]) for j in range(2)]
    v_cached = [f(vs[0][0, 0, j]) for j in range(2)]
    # context row (position 2): h_ctx = rmsnorm(X[:4]) * hidden_norm; K = rope(norm(h_ctx[:2]))
    hc = _nrm(f(X[0, 0, :4]), f(w["hidden_norm"]))
    kc = _turn(_nrm(hc[:2], f(lw["k_norm"])), 2.0)
    vc = hc[:2]
    # block rows at positions 3 and 4 (after the one appended context row)
    e = [f(core.decode_bf16(w["embed"][t], np.float64)) for t in ids[0]]
    xn = [_nrm(r, f(lw["input_norm"])) for r in e]
    kb = [_turn(_nrm(xn[i][:2], f(lw["k_norm"])), 3.0 + i) for i in range(2)]
    vb = [xn[i][:2] for i in range(2)]
    keys = k_cached + [kc] + kb
    vals = v_cached + [vc] + vb
    out = []
    for i in range(2):
        o = []
        for hq in range(2):
            q = _turn(_nrm(xn[i][2 * hq:2 * hq + 2], f(lw["q_norm"])), 3.0 + i)
            o += _attend(q, keys, vals)
        h1 = [e[i][t] + o[3 - t] for t in range(4)]            # Wo = J
        x2 = _nrm(h1, f(lw["post_norm"]))
        h2 = [a + _silu(z) * z for a, z in zip(h1, x2)]
        out.append(_nrm(h2, f(w["final_norm"])))
    return np.array(out), kc, vc


def test_dflash_layer_closed_form_two_dim_heads():
    """Whole drafter layer with every projection the identity: context K/V normed then rotated
    at the row's absolute position, block q/k normed then rotated at ctx_len + i, attention over
    cache + context + block (not causal), residual, SwiGLU on the post-attention norm, final
    norm."""
    cfg, w, ks, vs, X, ids = _dflash_two_dim_case()
    want, kc, vc = _dflash_two_dim_expected(w, copy.deepcopy(ks), copy.deepcopy(vs), X, ids)
    out, seq = dflash.dflash_block_forward(cfg, w, ks, vs, [2], ids, X, [1], np.float64)
    assert list(seq) == [3]
    assert np.allclose(ks[0][0, 0, 2], kc, rtol=1e-12, atol=1e-14)
    assert np.allclose(vs[0][0, 0, 2], vc, rtol=1e-12, atol=1e-14)
    assert np.allclose(out[0], want, rtol=1e-10, atol=1e-12)


def test_dflash_swiglu_reads_post_attention_norm():
    """Wo = 0 leaves h = E[ids] after attention; Wg = Wu = Wd = I then give
    h_final = rmsnorm(e + silu(x2) x2, final_norm) with x2 = rmsnorm(e, post_norm)."""
    cfg = fx.dflash_cfg(H=16, I=16)
    w = fx.random_dflash_weights(cfg, seed=31)
    lw = w["layers"][0]
    lw["wo"] = fx.zeros_bits(16, cfg.q_total)
    lw["wg"], lw["wu"], lw["wd"] = fx.eye_bits(16, 16), fx.eye_bits(16, 16), fx.eye_bits(16, 16)
    rng = np.random.default_rng(32)
    ks, vs = fx.random_cache(1, 1, cfg.n_kv_heads, cfg.head_dim, 3, 8)
    ids = _ids(cfg, 1, rng)
    X = rng.standard_normal((1, 1, cfg.fc_in))
    out, _ = dflash.dflash_block_forward(cfg, w, ks, vs, [3], ids, X, [1], np.float64)
    for i, t in enumerate(ids[0]):
        e = [float(v) for v in core.decode_bf16(w["embed"][t], np.float64)]
        x2 = _nrm(e, [float(g) for g in lw["post_norm"]])
        h2 = [a + _silu(z) * z for a, z in zip(e, x2)]
        want = _nrm(h2, [float(g) for g in w["final_norm"]])
        assert np.allclose(out[0, i], want, rtol=1e-10, atol=1e-12)


def _mtp_two_dim_case():
    """MTP step, H = 4, two q heads sharing one KV head of dim 2, eh_embed = I, eh_hidden and Wo
    the reversal permutation J, identity q/k/v/gate and SwiGLU projections, two cached rows."""
    cfg = fx.mtp_cfg(H=4, nq=2, nkv=1, d=2, I=4, V=10)
    w = fx.random_mtp_weights(cfg, seed=41)
    w["q_norm"] = np.array(Q_NORM2, np.float32)
    w["k_norm"] = np.array(K_NORM2, np.float32)
    w["post_norm"] = np.array([1.5, 0.7, 1.2, 0.9], np.float32)
    w["eh_embed"] = fx.eye_bits(4, 4)
    w["eh_hidden"] = _reverse_bits(4)
    for name, (r, c) in dict(wq=(4, 4), wk=(2, 4), wv=(2, 4), w_gate=(4, 4), wg=(4, 4),
                             wu=(4, 4), wd=(4, 4)).items():
        w[name] = fx.eye_bits(r, c)
    w["wo"] = _reverse_bits(4)
    rng = np.random.default_rng(42)
    kc = np.zeros((1, 4, 2))
    vc = np.zeros((1, 4, 2))
    kc[0, :2] = rng.standard_normal((2, 2))
    vc[0, :2] = rng.standard_normal((2, 2))
    prev = rng.standard_normal(4)
    return cfg, w, kc, vc, prev


def test_mtp_step_closed_form_two_dim_heads():
    """Whole MTP step at position 2: x = enorm(e) + J hnorm(h_prev); q/k normed then rotated by
    2 rad; attention over the two cached rows and the new one; output times sigmoid(gate);
    h1 = x + J o; hidden = h1 + SwiGLU(rmsnorm(h1, post_norm)); argmax of the shared head."""
    cfg, w, kc, vc, prev = _mtp_two_dim_case()
    f = lambda a: [float(v) for v in np.asarray(a).reshape(-1)]
    k_cached = [f(kc[0, j]) for j in range(2)]
    v_cached = [f(vc[0, j]) for j in range(2)]
    hidden, idx, _, _, _ = mtp.mtp_step(cfg, w, kc, vc, 2, prev, 7, np.float64)
    e = f(core.decode_bf16(w["embed"][7], np.float64))
    ne = _nrm(e, f(w["enorm"]))
    nh = _nrm(f(prev), f(w["hnorm"]))
    x = [ne[i] + nh[3 - i] for i in range(4)]
    xn = _nrm(x, f(w["attn_norm"]))
    k2 = _turn(_nrm(xn[:2], f(w["k_norm"])), 2.0)
    v2 = xn[:2]
    o = []
    for hq in range(2):
        q = _turn(_nrm(xn[2 * hq:2 * hq + 2], f(w["q_norm"])), 2.0)
        o += _attend(q, k_cached + [k2], v_cached + [v2])
    og = [a / (1.0 + math.exp(-g)) for a, g in zip(o, xn)]
    h1 = [x[i] + og[3 - i] for i in range(4)]                   # Wo = J
    x2 = _nrm(h1, f(w["post_norm"]))
    want = [a + _silu(z) * z for a, z in zip(h1, x2)]
    assert np.allclose(kc[0, 2], k2, rtol=1e-12, atol=1e-14)
    assert np.allclose(vc[0, 2], v2, rtol=1e-12, atol=1e-14)
    assert np.allclose(hidden, want, rtol=1e-10, atol=1e-12)
    xh = _nrm(want, f(w["shared_head_norm"]))
    lm = core.decode_bf16(w["lm_head"], np.float64)
    logits = [sum(float(lm[v, j]) * xh[j] for j in range(4)) for v in range(cfg.vocab)]
    assert idx == max(range(cfg.vocab), key=lambda v: (logits[v], -v))


def test_mtp_dense_ffn_reads_post_attention_norm():
    """Wo = 0 makes h1 = x; with eh_embed = I, eh_hidden = J and Wg = Wu = Wd = I,
    hidden = x + silu(x2) x2 with x = enorm(e) + J hnorm(h_prev), x2 = rmsnorm(x, post_norm)."""
    cfg = fx.mtp_cfg(H=16, I=16)
    w = fx.random_mtp_weights(cfg, seed=51)
    w["wo"] = fx.zeros_bits(16, cfg.q_total)
    w["eh_embed"] = fx.eye_bits(16, 16)
    w["eh_hidden"] = _reverse_bits(16)
    w["wg"], w["wu"], w["wd"] = fx.eye_bits(16, 16), fx.eye_bits(16, 16), fx.eye_bits(16, 16)
    rng = np.random.default_rng(52)
    kc = rng.standard_normal((1, 6, 8))
    vc = rng.standard_normal((1, 6, 8))
    prev = rng.standard_normal(16)
    hidden, _, _, _, _ = mtp.mtp_step(cfg, w, kc, vc, 4, prev, 5, np.float64)
    f = lambda a: [float(v) for v in np.asarray(a).reshape(-1)]
    ne = _nrm(f(core.decode_bf16(w["embed"][5], np.float64)), f(w["enorm"]))
    nh = _nrm(f(prev), f(w["hnorm"]))
    x = [ne[i] + nh[15 - i] for i in range(16)]
    x2 = _nrm(x, f(w["post_norm"]))
    want = [a + _silu(z) * z for a, z in zip(x, x2)]
    assert np.allclose(hidden, want, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------- planted mistakes

def test_planted_mistakes_are_caught(monkeypatch):
    """Each pin above fails when the oracle carries a plausible mistake."""
    # 1. RoPE with the sign of the sine flipped: the hand-worked RoPE value catches it.
    real_rope = core.rope

    def bad_rope(x, pos, r, theta, dt=np.float32):
        return real_rope(x, -np.asarray(pos), r, theta, dt)

    y = bad_rope(np.array([1.0, 0, 0, 0]).reshape(1, 1, 4), [1], 4, 1e4, np.float64)
    assert not np.allclose(y.reshape(-1), [0.5403023058681398, 0.0, 0.8414709848078965, 0.0])

    # 2. A dropped residual in the layer: the zero-output-projection pin catches it.
    orig_layer = dflash.dflash_layer

    def layer_no_residual(cfg, lw, h, h_ctx, kc, vc, ctx0, dt=np.float32):
        return orig_layer(cfg, lw, h, h_ctx, kc, vc, ctx0, dt) - h

    monkeypatch.setattr(dflash, "dflash_layer", layer_no_residual)
    with pytest.raises(AssertionError):
        test_zero_output_projections_keep_embedding()
    monkeypatch.undo()
    test_zero_output_projections_keep_embedding()

    # 3. Wrong GQA head mapping (kv head h % n_kv instead of h // (n_q/n_kv)): the
    #    brute-force SDPA loops catch it.
    from tests.test_oracle_core import _sdpa_loops
    rng = np.random.default_rng(0)
    q = rng.standard_normal((2, 4, 3))
    k = rng.standard_normal((5, 2, 3))
    v = rng.standard_normal((5, 2, 3))
    bad = np.stack([core.sdpa(q[:, h:h + 1], k[:, h % 2:h % 2 + 1], v[:, h % 2:h % 2 + 1], None,
                              np.float64)[:, 0] for h in range(4)], 1)
    assert not np.allclose(bad, _sdpa_loops(q, k, v))
    assert np.allclose(core.sdpa(q, k, v, None, np.float64), _sdpa_loops(q, k, v))

    # 4. An accept walk that forgets the free token breaks the committed-length invariant.
    def walk_no_free(drafts, target, eos=()):
        c, a, hit, rb = core.accept_walk(drafts, target, eos)
        return c[:a], a, hit, rb

    c, a, hit, rb = walk_no_free([1, 2], [4, 0, 5], ())
    assert not (1 <= len(c) <= 3)


def test_bf16_kv_layer_stores_rounded_rows():
    """With a BF16 KV cache the appended context rows are the F32 path's rows rounded to BF16."""
    from oracle import dflash as odf
    from tests.oracle_fixtures import dflash_cfg, random_dflash_weights
    cfg = dflash_cfg(H=16, nq=2, nkv=1, d=8, I=12, V=50, K=3, n_tl=2)
    w = random_dflash_weights(cfg, n_layers=1, seed=3)
    rng = np.random.default_rng(4)
    h = rng.standard_normal((4, 16)).astype(np.float32)
    hc = rng.standard_normal((5, 16)).astype(np.float32)
    k32, v32 = np.zeros((1, 20, 8), np.float32), np.zeros((1, 20, 8), np.float32)
    kb, vb = np.zeros_like(k32), np.zeros_like(v32)
    out32 = odf.dflash_layer(cfg, w["layers"][0], h, hc, k32, v32, 2)
    cfg.kv_bf16 = True
    out16 = odf.dflash_layer(cfg, w["layers"][0], h, hc, kb, vb, 2)
    assert np.array_equal(kb[:, 2:7], core.round_bf16(k32[:, 2:7]))
    assert np.array_equal(vb[:, 2:7], core.round_bf16(v32[:, 2:7]))
    assert not np.array_equal(out16, out32) and np.max(np.abs(out16 - out32)) < 0.05


def _mutant(module, name, edits):
    """`module.name` recompiled from its source with each (old, new) text edit applied once: a
    plausible slip planted in the oracle (on the CPU) to show that some pin fails."""
    src = inspect.getsource(getattr(module, name))
    for old, new in edits:
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    ns = dict(vars(module))
    exec(compile(src, module.__file__, "exec"), ns)
    return ns[name]


def _rope_then_norm(x, w, pos, n_heads, head_dim, eps, rotary_dim, theta, dt=np.float32):
    """The planted slip of the q/k step: RoPE first, per-head RMSNorm after it."""
    T = np.size(pos)
    x = np.asarray(x, dt).reshape(T, n_heads, head_dim)
    turned = core.rope(x, pos, rotary_dim, theta, dt).reshape(T, n_heads * head_dim)
    return core.head_rmsnorm(turned, w, n_heads, head_dim, eps, dt).reshape(T, n_heads, head_dim)


DFLASH_PINS = (test_dflash_layer_closed_form_two_dim_heads,
               test_dflash_swiglu_reads_post_attention_norm)
MTP_PINS = (test_mtp_step_closed_form_two_dim_heads, test_mtp_dense_ffn_reads_post_attention_norm)

LAYER_SLIPS = [
    # the drafter's SwiGLU fed by the input norm instead of the post-attention norm
    ("swiglu_input_norm", dflash, "dflash_layer",
     [('rmsnorm(h, lw["post_norm"]', 'rmsnorm(h, lw["input_norm"]')], DFLASH_PINS),
    # the drafter's context K normed with the q weight
    ("context_k_q_norm", dflash, "dflash_layer",
     [('lw["k_norm"], pos_c', 'lw["q_norm"], pos_c')], DFLASH_PINS[:1]),
    # block rows rotated at positions counted before the context append
    ("block_positions_before_append", dflash, "dflash_layer",
     [("pos_b = np.arange(ctx_len, ctx_len + blk)", "pos_b = np.arange(ctx0, ctx0 + blk)")],
     DFLASH_PINS[:1]),
    # the final norm taken with the hidden (fc) norm weight
    ("final_norm_weight", dflash, "dflash_block_forward",
     [('rmsnorm(h, w["final_norm"]', 'rmsnorm(h, w["hidden_norm"]')], DFLASH_PINS),
    # the MTP FFN fed by the attention-input norm instead of the post-attention norm
    ("mtp_ffn_attn_norm", mtp, "mtp_step",
     [('fin = rmsnorm(h1, w["post_norm"]', 'fin = rmsnorm(h1, w["attn_norm"]')], MTP_PINS),
    # the MTP FFN fed by x (before the attention residual) instead of h1
    ("mtp_ffn_before_attention", mtp, "mtp_step",
     [("fin = rmsnorm(h1,", "fin = rmsnorm(x,")], MTP_PINS[:1]),
    # the two eh_proj halves swapped
    ("mtp_eh_halves_swapped", mtp, "mtp_step",
     [('w["eh_embed"]', 'w["@@"]'), ('w["eh_hidden"]', 'w["eh_embed"]'),
      ('w["@@"]', 'w["eh_hidden"]')], MTP_PINS),
    # the sigmoid gate applied after the output projection instead of before it
    ("mtp_gate_after_wo", mtp, "mtp_step",
     [("o = o * sigmoid(linear(xn, w[\"w_gate\"], dt), dt)", "pass"),
      ('h1 = x + linear(o, w["wo"], dt)',
       'h1 = x + linear(o, w["wo"], dt) * sigmoid(linear(xn, w["w_gate"], dt), dt)')],
     MTP_PINS[:1]),
]


@pytest.mark.parametrize("slip", LAYER_SLIPS, ids=[s[0] for s in LAYER_SLIPS])
def test_planted_layer_composition_mistakes_are_caught(monkeypatch, slip):
    """Each slip in the composition of the drafter layer or the MTP step fails a closed-form
    pin above; the unmodified oracle passes the same pins."""
    _, module, name, edits, pins = slip
    monkeypatch.setattr(module, name, _mutant(module, name, edits))
    for pin in pins:
        with pytest.raises(AssertionError):
            pin()
    monkeypatch.undo()
    for pin in pins:
        pin()


def test_planted_rope_before_norm_is_caught(monkeypatch):
    """RoPE before the per-head q/k norm, in the drafter (block and context rows) and in the
    MTP step: the norm weight does not commute with the rotation, so the two-dim-head closed
    forms fail."""
    monkeypatch.setattr(dflash, "qk_norm_rope", _rope_then_norm)
    with pytest.raises(AssertionError):
        test_dflash_layer_closed_form_two_dim_heads()
    monkeypatch.setattr(mtp, "qk_norm_rope", _rope_then_norm)
    with pytest.raises(AssertionError):
        test_mtp_step_closed_form_two_dim_heads()
    monkeypatch.undo()
    test_dflash_layer_closed_form_two_dim_heads()
    test_mtp_step_closed_form_two_dim_heads()


def test_qk_norm_rope_order_on_one_head():
    """One 2-dim head [1, 0] with norm weight [2, 1] at position pi/2: normed first it is
    [2, 0] (RMS of [1, 0] is 1/sqrt(2), so the normed head is [sqrt(2)*2, 0] up to eps), then
    turned by pi/2 to [0, 2 sqrt(2)]; turned first and normed after it would be [0, sqrt(2)]."""
    y = core.qk_norm_rope(np.array([[1.0, 0.0]]), np.array([2.0, 1.0]), [math.pi / 2], 1, 2, 0.0,
                          2, 1e4, np.float64)
    assert np.allclose(y.reshape(-1), [0.0, 2.0 * math.sqrt(2.0)], atol=1e-12)
