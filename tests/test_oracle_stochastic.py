"""Pins of the stochastic (non-greedy) accept oracle: hand draws, the speculative-sampling
identity (the committed token is distributed exactly as the target's softmax), a Monte-Carlo
run of the whole walk, the greedy limit at a vanishing temperature, and identical drafter and
target distributions."""
import numpy as np
import pytest

from oracle import core
from oracle import stochastic as st


def test_draw_index_hand_examples():
    w = [1.0, 2.0, 1.0]                      # running sums 1, 3, 4
    assert st.draw_index(w, 0.0) == 0
    assert st.draw_index(w, 0.2499) == 0
    assert st.draw_index(w, 0.25) == 1       # u * 4 = 1 is not above the first sum
    assert st.draw_index(w, 0.7499) == 1
    assert st.draw_index(w, 0.75) == 2
    assert st.draw_index(w, 0.9999) == 2
    assert all(st.draw_index([0, 0, 5, 0], u) == 2 for u in (0.0, 0.3, 0.99))
    assert st.draw_margin(w, 0.5) == pytest.approx(0.25)    # u*4 = 2, between sums 1 and 3


def test_softmax_t_closed_forms():
    p = st.softmax_t([0.0, np.log(3.0)], 1.0)
    assert p == pytest.approx([0.25, 0.75])
    p2 = st.softmax_t([0.0, 2 * np.log(3.0)], 2.0)         # logits / T
    assert p2 == pytest.approx([0.25, 0.75])
    with pytest.raises(core.OracleError):
        st.softmax_t([1.0], 0.0)


@pytest.mark.parametrize("seed", range(6))
def test_first_token_is_distributed_as_the_target(seed):
    rng = np.random.default_rng(seed)
    V = 7
    t0, d0, t1 = rng.normal(0, 1.5, V), rng.normal(0, 1.5, V), rng.normal(0, 1.5, V)
    for T in (0.5, 1.0, 1.7):
        got = st.first_token_distribution(d0, t0, t1, T)
        assert got == pytest.approx(st.softmax_t(t0, T), abs=1e-12)
        # a planted mistake (residual drawn from max(0, q - p)) breaks the identity
        p, q = st.softmax_t(t0, T), st.softmax_t(d0, T)
        acc = np.minimum(1.0, p / q)
        wrong = np.maximum(0.0, q - p)
        bad = q * acc + np.sum(q * (1 - acc)) * wrong / np.sum(wrong)
        assert np.max(np.abs(bad - p)) > 1e-3


def test_walk_monte_carlo_matches_target_distribution():
    rng = np.random.default_rng(7)
    V, K, T, N = 4, 2, 0.8, 40000
    tl = rng.normal(0, 1.2, (K + 1, V))
    dl = tl[:K] + rng.normal(0, 0.8, (K, V))
    q0 = st.softmax_t(dl[0], T)
    q1 = st.softmax_t(dl[1], T)
    counts = np.zeros(V)
    for _ in range(N):
        drafts = [st.draw_index(q0, rng.random()), st.draw_index(q1, rng.random())]
        committed, a, hit, rb, _ = st.accept_stochastic(dl, tl, drafts, T, rng.random(K),
                                                        rng.random())
        assert 1 <= len(committed) <= K + 1 and rb == K - a and hit == 0
        counts[committed[0]] += 1
    emp = counts / N
    assert np.max(np.abs(emp - st.softmax_t(tl[0], T))) < 0.01


def test_greedy_limit_matches_accept_walk():
    rng = np.random.default_rng(3)
    V, K = 12, 5
    for _ in range(200):
        tl = rng.normal(0, 1.0, (K + 1, V)) * 20.0
        dl = rng.normal(0, 1.0, (K, V)) * 20.0
        # drafts agree with the target's argmax on a prefix, then follow the drafter
        n_agree = int(rng.integers(0, K + 1))
        drafts = [int(np.argmax(tl[i])) if i < n_agree else int(np.argmax(dl[i])) for i in range(K)]
        for i in range(n_agree):
            dl[i, drafts[i]] = np.max(dl[i]) + 5.0
        target = [int(np.argmax(tl[i])) for i in range(K + 1)]
        got = st.accept_stochastic(dl, tl, drafts, 1e-3, rng.uniform(0.01, 0.99, K),
                                   rng.uniform(0.01, 0.99), eos=(1,))
        want = core.accept_walk(drafts, target, eos=(1,))
        assert got[:4] == want


def test_identical_distributions_accept_everything():
    rng = np.random.default_rng(5)
    V, K, T = 9, 4, 1.3
    tl = rng.normal(0, 1.0, (K + 1, V))
    drafts = [int(x) for x in rng.integers(0, V, K)]
    u = rng.random(K)
    committed, a, hit, rb, info = st.accept_stochastic(tl[:K], tl, drafts, T, u, 0.37)
    assert a == K and rb == 0
    assert committed == drafts + [st.draw_index(st.softmax_t(tl[K], T), 0.37)]


def test_eos_cut_like_greedy():
    V, K, T = 5, 3, 1.0
    tl = np.zeros((K + 1, V))
    drafts = [3, 1, 4]                       # token 1 is EOS: the list stops after it
    committed, a, hit, rb, _ = st.accept_stochastic(tl[:K], tl, drafts, T, [0.1, 0.2, 0.3], 0.5,
                                                    eos=(1,))
    assert a == K and rb == 0 and hit == 1 and committed == [3, 1]


# --------------------------------------------------------------- sampled drafts (T > 0)

def test_sample_draft_hand_draws():
    """logits [0, ln 3] at T = 1 (or [0, 2 ln 3] at T = 2): q = [1/4, 3/4], so u < 1/4 draws
    token 0 and u >= 1/4 token 1."""
    for logits, T in (([0.0, np.log(3.0)], 1.0), ([0.0, 2.0 * np.log(3.0)], 2.0)):
        assert st.sample_draft(logits, T, 0.0) == 0
        assert st.sample_draft(logits, T, 0.2499) == 0
        assert st.sample_draft(logits, T, 0.2501) == 1
        assert st.sample_draft(logits, T, 0.9999) == 1
    # three tokens, q = [1/6, 2/6, 3/6]: boundaries at 1/6 and 1/2
    lg = np.log([1.0, 2.0, 3.0])
    assert [st.sample_draft(lg, 1.0, u) for u in (0.1, 0.2, 0.49, 0.51, 0.99)] == [0, 1, 1, 2, 2]


def test_sample_draft_frequencies_follow_softmax():
    rng = np.random.default_rng(11)
    V, T, N = 6, 0.7, 60000
    lg = rng.normal(0, 1.0, V)
    counts = np.bincount([st.sample_draft(lg, T, u) for u in rng.random(N)], minlength=V)
    q = st.softmax_t(lg, T)
    # binomial standard deviation sqrt(q (1 - q) / N) <= 0.0021; allow 5 of them
    assert np.max(np.abs(counts / N - q)) < 0.011


def test_sampled_drafts_then_accept_commit_target_distribution():
    """The whole non-greedy path at K = 2: drafts sampled by `sample_draft`, the accept step,
    the first committed token follows p_0 (Monte Carlo)."""
    rng = np.random.default_rng(12)
    V, K, T, N = 5, 2, 0.9, 40000
    tl = rng.normal(0, 1.2, (K + 1, V))
    dl = tl[:K] + rng.normal(0, 0.9, (K, V))
    counts = np.zeros(V)
    for _ in range(N):
        drafts = [st.sample_draft(dl[i], T, rng.random()) for i in range(K)]
        committed, a, hit, rb, _ = st.accept_stochastic(dl, tl, drafts, T, rng.random(K),
                                                        rng.random())
        counts[committed[0]] += 1
    assert np.max(np.abs(counts / N - st.softmax_t(tl[0], T))) < 0.01
    # a planted slip: drafts taken as the drafter's argmax while the test divides by q
    counts_bad = np.zeros(V)
    for _ in range(N // 4):
        drafts = [int(np.argmax(dl[i])) for i in range(K)]
        committed, *_ = st.accept_stochastic(dl, tl, drafts, T, rng.random(K), rng.random())
        counts_bad[committed[0]] += 1
    assert np.max(np.abs(counts_bad / (N // 4) - st.softmax_t(tl[0], T))) > 0.03


def test_stochastic_round_greedy_limit():
    """At a vanishing temperature every softmax is one-hot: the sampled drafts are the drafter's
    argmaxes and the stochastic round commits what the greedy round commits."""
    from oracle import dflash
    from tests import oracle_fixtures as fx
    import copy
    cfg = fx.dflash_cfg(V=40, K=3)
    w = fx.random_dflash_weights(cfg, seed=17)
    rng = np.random.default_rng(18)
    B = 2
    ids = np.full((B, cfg.K + 1), cfg.vocab - 1, dtype=np.int64)
    ids[:, 0] = [5, 9]
    X = rng.standard_normal((B, 2, cfg.fc_in))
    ks, vs = fx.random_cache(1, B, 1, 8, 4, 8)
    greedy = dflash.draft_round(cfg, w, copy.deepcopy(ks), copy.deepcopy(vs), [4, 4], ids, X,
                                [2, 1], np.zeros((B, cfg.K + 1), np.int64), (), [30, 30],
                                np.float64)
    am = greedy["argmax"]
    # verifier logits whose argmax agrees with the drafts on 2 (seq 0) and all (seq 1) positions
    tl = rng.normal(0, 1.0, (B, cfg.K + 1, cfg.vocab))
    target = np.stack([np.r_[am[0, 1:3], (am[0, 3] + 1) % cfg.vocab, 7], np.r_[am[1, 1:], 9]])
    for b in range(B):
        for i in range(cfg.K + 1):
            tl[b, i, target[b, i]] = tl[b, i].max() + 3.0
    greedy = dflash.draft_round(cfg, w, copy.deepcopy(ks), copy.deepcopy(vs), [4, 4], ids, X,
                                [2, 1], target, (), [30, 30], np.float64)
    T = 1e-4
    res = dflash.draft_round_stochastic(cfg, w, ks, vs, [4, 4], ids, X, [2, 1], tl, T,
                                        rng.uniform(0.05, 0.95, (B, cfg.K)),
                                        rng.uniform(0.05, 0.95, (B, cfg.K)),
                                        rng.uniform(0.05, 0.95, B), (), [30, 30], np.float64)
    assert [list(d) for d in res["drafts"]] == [list(r[1:]) for r in am]
    assert res["accept"] == greedy["accept"] == [2, 3]
    assert res["committed"] == greedy["committed"]
    assert res["rollback"] == greedy["rollback"] and res["target_seq_len"] == [29, 30]
    # the logits the draws read are the lm_head of the final-normed block rows
    lm = core.decode_bf16(w["lm_head"], np.float64)
    assert np.allclose(res["logits"], np.einsum("bph,vh->bpv", res["h_final"], lm), rtol=1e-12)


def test_mtp_sampled_chain_greedy_limit_and_feed():
    """At a vanishing temperature the sampled MTP chain is the argmax chain; at T = 1 each
    step's draft is the draw from that step's logits and is the next step's input token."""
    from oracle import mtp
    from tests import oracle_fixtures as fx
    cfg = fx.mtp_cfg(V=30)
    w = fx.random_mtp_weights(cfg, seed=19)
    rng = np.random.default_rng(20)
    kc = np.zeros((1, 1, 12, 8))
    vc = np.zeros((1, 1, 12, 8))
    kc[:, :, :4] = rng.standard_normal((1, 1, 4, 8))
    vc[:, :, :4] = rng.standard_normal((1, 1, 4, 8))
    prev = rng.standard_normal((1, cfg.hidden))
    hid, am, _, _, seq, _ = mtp.mtp_forward_draft(cfg, w, kc.copy(), vc.copy(), [4], prev, [3], 3,
                                                  np.float64)
    u = rng.uniform(0.05, 0.95, (3, 1))
    h2, dr, lg, seq2 = mtp.mtp_forward_draft_sampled(cfg, w, kc.copy(), vc.copy(), [4], prev, [3],
                                                     3, 1e-4, u, np.float64)
    assert np.array_equal(dr, am) and np.allclose(h2, hid) and list(seq2) == list(seq) == [7]
    h3, dr3, lg3, _ = mtp.mtp_forward_draft_sampled(cfg, w, kc.copy(), vc.copy(), [4], prev, [3],
                                                    3, 1.0, u, np.float64)
    for s in range(3):
        assert dr3[s, 0] == st.sample_draft(lg3[s, 0], 1.0, u[s, 0])
    # step 1 read step 0's draft: rerunning step 1 by hand from (h3[0], dr3[0]) reproduces it
    k2, v2 = kc.copy(), vc.copy()
    mtp.mtp_step(cfg, w, k2[0], v2[0], 4, prev[0], 3, np.float64)
    h_1, *_ = mtp.mtp_step(cfg, w, k2[0], v2[0], 5, h3[0, 0], int(dr3[0, 0]), np.float64)
    assert np.allclose(h_1, h3[1, 0], rtol=1e-12)
