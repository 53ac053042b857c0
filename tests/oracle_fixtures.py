"""Host-side helpers for the oracle pins: small weight sets built by hand (identity
and zero projections) or drawn with NumPy, as dicts the oracle accepts. Test
infrastructure; holds none of the method's arithmetic."""
from types import SimpleNamespace

import numpy as np

ONE = np.uint16(0x3F80)     # BF16 bit pattern of 1.0


def bf16_bits_rne(a):
    """F32 -> BF16 bit patterns by round-to-nearest-even (finite inputs)."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def eye_bits(rows, cols):
    """BF16 [rows, cols] with ones on the diagonal (row i selects input i)."""
    w = np.zeros((rows, cols), dtype=np.uint16)
    for i in range(min(rows, cols)):
        w[i, i] = ONE
    return w


def zeros_bits(rows, cols):
    return np.zeros((rows, cols), dtype=np.uint16)


def dflash_cfg(H=16, nq=2, nkv=1, d=8, I=12, V=50, K=3, n_tl=2, causal=0, rot=0):
    return SimpleNamespace(hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, intermediate=I,
                           vocab=V, K=K, n_target_layers=n_tl, rms_eps=1e-6, rope_theta=1e4,
                           rot=rot or d, causal_block=causal, fc_in=n_tl * H,
                           q_total=nq * d, kv_total=nkv * d)


def random_dflash_weights(cfg, n_layers=1, seed=0):
    rng = np.random.default_rng(seed)
    H, I = cfg.hidden, cfg.intermediate

    def w(r, c):
        return bf16_bits_rne(rng.standard_normal((r, c)) * 0.3)

    def n(k):
        return (1.0 + 0.1 * rng.standard_normal(k)).astype(np.float32)

    layers = [dict(input_norm=n(H), post_norm=n(H), q_norm=n(cfg.head_dim), k_norm=n(cfg.head_dim),
                   wq=w(cfg.q_total, H), wk=w(cfg.kv_total, H), wv=w(cfg.kv_total, H),
                   wo=w(H, cfg.q_total), wg=w(I, H), wu=w(I, H), wd=w(H, I))
              for _ in range(n_layers)]
    return dict(fc=w(H, cfg.fc_in), hidden_norm=n(H), final_norm=n(H), layers=layers,
                embed=w(cfg.vocab, H), lm_head=w(cfg.vocab, H))


def random_cache(n_layers, B, nkv, d, filled, cap, seed=1, dtype=np.float32):
    rng = np.random.default_rng(seed)
    ks, vs = [], []
    for _ in range(n_layers):
        k = np.zeros((B, nkv, cap, d), dtype=dtype)
        v = np.zeros_like(k)
        k[:, :, :filled] = rng.standard_normal((B, nkv, filled, d))
        v[:, :, :filled] = rng.standard_normal((B, nkv, filled, d))
        ks.append(k)
        vs.append(v)
    return ks, vs


def mtp_cfg(H=16, nq=2, nkv=1, d=8, I=12, V=40, E=0, top_k=0, Ie=6, Is=6):
    return SimpleNamespace(hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, intermediate=I,
                           vocab=V, rms_eps=1e-6, rope_theta=1e4, rot=d, n_experts=E,
                           top_k=top_k, expert_inter=Ie, shared_inter=Is, q_total=nq * d,
                           kv_total=nkv * d)


def random_mtp_weights(cfg, seed=0, gate=True):
    rng = np.random.default_rng(seed)
    H = cfg.hidden

    def w(*shape, s=0.3):
        return bf16_bits_rne(rng.standard_normal(shape) * s)

    def n(k):
        return (1.0 + 0.1 * rng.standard_normal(k)).astype(np.float32)

    mw = dict(enorm=n(H), hnorm=n(H), eh_embed=w(H, H), eh_hidden=w(H, H), attn_norm=n(H),
              post_norm=n(H), q_norm=n(cfg.head_dim), k_norm=n(cfg.head_dim),
              wq=w(cfg.q_total, H), wk=w(cfg.kv_total, H), wv=w(cfg.kv_total, H),
              w_gate=w(cfg.q_total, H) if gate else None, wo=w(H, cfg.q_total),
              shared_head_norm=n(H), embed=w(cfg.vocab, H), lm_head=w(cfg.vocab, H))
    if cfg.n_experts:
        E, Ie, Is = cfg.n_experts, cfg.expert_inter, cfg.shared_inter
        mw.update(router=w(E, H, s=1.0 / np.sqrt(H)), exp_g=w(E, Ie, H), exp_u=w(E, Ie, H),
                  exp_d=w(E, H, Ie), sh_g=w(Is, H), sh_u=w(Is, H), sh_d=w(H, Is), sh_gate=w(1, H))
    else:
        I = cfg.intermediate
        mw.update(wg=w(I, H), wu=w(I, H), wd=w(H, I))
    return mw
