"""Shared test plumbing: host copies of synthetic inputs in the oracle's dict layout, the
relative-error metric, and the near-tie rule for argmax parity. No method arithmetic."""
import numpy as np
import torch

from speculative_decoding_drafter_dflash_gb300 import synth

REL_TOL = 2e-3          # max relative error of hidden states and logits
GAP_MIN = 1e-2          # argmax indices must match where the oracle's top1 - top2 exceeds this


def rel_err(got, ref):
    """max_i |g_i - r_i| / max(|r_i|, rms(r))."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(r * r)) if r.size else 0.0
    den = np.maximum(np.abs(r), rms)
    den[den == 0] = 1.0
    return float(np.max(np.abs(g - r) / den)) if r.size else 0.0


def dflash_weights_host(w: synth.DFlashWeights):
    h = synth.host
    return dict(fc=h(w.fc), hidden_norm=h(w.hidden_norm), final_norm=h(w.final_norm),
                embed=h(w.embed), lm_head=h(w.lm_head),
                layers=[dict(input_norm=h(l.input_norm), post_norm=h(l.post_norm),
                             q_norm=h(l.q_norm), k_norm=h(l.k_norm), wq=h(l.wq), wk=h(l.wk),
                             wv=h(l.wv), wo=h(l.wo), wg=h(l.wg), wu=h(l.wu), wd=h(l.wd))
                        for l in w.layers])


def mtp_weights_host(w: synth.MtpWeights):
    out = {}
    for name in ("enorm", "hnorm", "eh_embed", "eh_hidden", "attn_norm", "post_norm", "q_norm",
                 "k_norm", "wq", "wk", "wv", "w_gate", "wo", "shared_head_norm", "embed",
                 "lm_head", "wg", "wu", "wd", "router", "exp_g", "exp_u", "exp_d", "sh_g", "sh_u",
                 "sh_d", "sh_gate"):
        t = getattr(w, name)
        out[name] = None if t is None else synth.host(t)
    return out


def _as_f32(t):
    """Host F32 copy of a cache tensor (BF16 caches are widened exactly)."""
    return t.detach().float().contiguous().cpu().numpy()


def cache_host(c: synth.KvCache):
    return [_as_f32(k) for k in c.k], [_as_f32(v) for v in c.v], synth.host(c.seq_len).copy()


def assert_argmax_parity(gpu_idx, ref_idx, ref_top1, ref_top2, what=""):
    """Indices agree wherever the oracle's top-1/top-2 gap exceeds GAP_MIN; returns the
    number of gated (near-tie) positions."""
    gi = np.asarray(gpu_idx).reshape(-1)
    ri = np.asarray(ref_idx).reshape(-1)
    gap = (np.asarray(ref_top1) - np.asarray(ref_top2)).reshape(-1)
    clear = gap > GAP_MIN
    bad = np.flatnonzero(clear & (gi != ri))
    assert bad.size == 0, f"{what}: argmax mismatch at {bad[:10]} (gpu {gi[bad[:10]]}, ref {ri[bad[:10]]})"
    return int((~clear).sum())
