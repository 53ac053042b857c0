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
