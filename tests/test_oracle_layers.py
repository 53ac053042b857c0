"""Pins of the oracle's DFlash forward, MTP step and MoE routing.

Closed forms from special weights (zero or identity projections), an
incremental-versus-one-shot invariant of the context cache, a float64 shadow, and
planted mistakes that the pins must catch. No expected value here comes from the
CUDA library.
"""
import copy
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
