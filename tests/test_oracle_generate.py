"""Pins of the multi-round generate-loop oracle: the capture helpers by hand, and the loop's
invariants from the page (output follows the verifier's own decisions, the captured prefix
stays one behind the output, the drafter cache never regresses, committed tokens never empty,
budget truncation, EOS stop, max_new_tokens == 0 returns the prompt and first token)."""
import numpy as np
import pytest

from oracle import generate as og
from tests.oracle_fixtures import dflash_cfg, random_cache, random_dflash_weights


def test_extract_and_append_by_hand():
    cap = np.zeros((3, 6, 2))
    for c in range(3):
        for p in range(6):
            cap[c, p] = [10 * c + p, -(10 * c + p)]
    rows = og.extract_drafter_concat(cap, [2, 0], 1, 3)
    assert rows.tolist() == [[21, -21, 1, -1], [22, -22, 2, -2]]
    prior = np.zeros_like(cap)
    ver = np.ones((3, 4, 2)) * 7
    n = og.append_capture_positions(prior, 2, ver, 3)
    assert n == 5 and np.all(prior[:, 2:5] == 7) and np.all(prior[:, :2] == 0)
    assert og.synthetic_verify([0, 1, 2, 3, 4, 5, 6], [0, 1, 0, 0, 0, 0, 0], 1, [9, 8]) == [9, 3, 4]


def _setup(seed, prompt_len=6, max_len=48, n_comb=3):
    cfg = dflash_cfg(H=16, nq=2, nkv=1, d=8, I=12, V=50, K=3, n_tl=2)
    cfg.mask_id = cfg.vocab - 1
    w = random_dflash_weights(cfg, n_layers=1, seed=seed)
    ks, vs = random_cache(1, 1, cfg.n_kv_heads, cfg.head_dim, 0, max_len + 8, seed=seed + 1)
    rng = np.random.default_rng(seed + 2)
    ref = rng.integers(2, cfg.vocab - 1, max_len).tolist()
    table = rng.standard_normal((n_comb, max_len, cfg.hidden))
    return cfg, w, ks, vs, ref, table, rng


@pytest.mark.parametrize("seed", [0, 1])
def test_output_is_the_reference_when_the_verifier_never_agrees(seed):
    cfg, w, ks, vs, ref, table, rng = _setup(seed)
    prompt_len, max_new = 6, 9
    out0 = ref[:prompt_len + 1]
    agree = [0] * len(ref)
    r = og.generate(cfg, w, ks, vs, 0, out0, prompt_len, ref, agree, table, [0, 2], max_new,
                    cfg.K, eos=(), max_rounds=64)
    assert r["out"] == ref[:prompt_len + max_new]
    assert len(r["accept"]) == r["rounds"] >= 1
    assert r["prior_len"] <= len(r["out"]) - 1


def test_an_agreeing_verifier_accepts_every_draft_and_the_budget_truncates():
    cfg, w, ks, vs, ref, table, rng = _setup(3)
    prompt_len, max_new = 6, 10
    agree = [1] * len(ref)
    r = og.generate(cfg, w, ks, vs, 0, ref[:prompt_len + 1], prompt_len, ref, agree, table,
                    [1, 2], max_new, cfg.K, eos=(), max_rounds=64)
    assert r["accept"] == [cfg.K] * r["rounds"]
    assert len(r["out"]) == prompt_len + max_new          # 1 + 4 + 4 + 4 tokens, truncated
    assert r["rounds"] == 3
    # the drafter consumed the prompt positions, then K+1 per completed round
    assert r["cache_len"] == prompt_len + (cfg.K + 1) * (r["rounds"] - 1)


def test_eos_stops_the_loop_and_max_new_zero_returns_prompt_and_first_token():
    cfg, w, ks, vs, ref, table, rng = _setup(4)
    prompt_len = 6
    ref = list(ref)
    ref[prompt_len + 4] = 1                                # EOS as the 4th generated token
    agree = [0] * len(ref)
    r = og.generate(cfg, w, ks, vs, 0, ref[:prompt_len + 1], prompt_len, ref, agree, table,
                    [0, 1], 20, cfg.K, eos=(1,), max_rounds=64)
    assert r["out"] == ref[:prompt_len + 5] and r["out"][-1] == 1
    r0 = og.generate(cfg, w, ks, vs, 0, ref[:prompt_len + 1], prompt_len, ref, agree, table,
                     [0, 1], 0, cfg.K, eos=(1,), max_rounds=64)
    assert r0["out"] == ref[:prompt_len + 1] and r0["rounds"] == 0


def test_mixed_agreement_follows_the_verifier_decisions():
    cfg, w, ks, vs, ref, table, rng = _setup(5)
    prompt_len, max_new = 6, 14
    agree = (rng.random(len(ref)) < 0.6).astype(int).tolist()
    r = og.generate(cfg, w, ks, vs, 0, ref[:prompt_len + 1], prompt_len, ref, agree, table,
                    [0, 2], max_new, cfg.K, eos=(), max_rounds=64)
    out = r["out"]
    # every generated token after the first is either the reference token or an agreed draft
    for p in range(prompt_len, len(out) - 1):
        assert out[p + 1] == ref[p + 1] or agree[p]
    assert 1 <= r["rounds"] <= max_new and all(0 <= a <= cfg.K for a in r["accept"])
