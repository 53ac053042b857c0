"""Oracle of the non-greedy (stochastic) accept step: test infrastructure only.

qwen35_orchestrator.rs, module doc "Non-greedy (Metropolis-Hastings) is out of scope here":
the stochastic acceptance is wired through the MTP K=1 path and would hook into the DFlash
loop at step 11 (`step_round_from_argmaxes`) in place of the greedy walk. The page does not
spell the rule out; it is read as the standard speculative-sampling acceptance test:

  p_i = softmax(target_logits[i] / T), q_i = softmax(draft_logits[i] / T)
  draft x_i is accepted when u_i * q_i(x_i) < p_i(x_i)   (u_i uniform in [0, 1): probability
                                                          min(1, p_i(x_i) / q_i(x_i)))
  at the first rejection a, the committed token is drawn from max(0, p_a - q_a) (normalised);
  if every draft is accepted (a = K), it is drawn from p_K (the verifier's next position).

Under this rule, with every draft x_i itself drawn from q_i (`sample_draft`), the committed
token at every position is distributed exactly as the target's p (the identity the pins check).
A draw from weights w with a uniform u is the smallest index j whose running sum
w_0 + ... + w_j exceeds u * sum(w). The committed list, its EOS cut and
rollback = K - a follow the greedy walk (core.accept_walk). All arithmetic in float64.
"""
from __future__ import annotations

import numpy as np

from .core import OracleError


def softmax_t(logits, temperature):
    """softmax(logits / T) in float64."""
    if not temperature > 0:
        raise OracleError("temperature must be positive")
    x = np.asarray(logits, dtype=np.float64) / float(temperature)
    e = np.exp(x - np.max(x))
    return e / np.sum(e)


def draw_index(w, u):
    """Smallest j with w[0] + ... + w[j] > u * sum(w), for u in [0, 1) and sum(w) > 0."""
    w = np.asarray(w, dtype=np.float64)
    c = np.cumsum(w)
    if not c[-1] > 0:
        raise OracleError("draw from an all-zero weight vector")
    j = int(np.searchsorted(c, float(u) * c[-1], side="right"))
    return min(j, w.shape[0] - 1)


def draw_margin(w, u):
    """Distance, as a fraction of sum(w), from u * sum(w) to the nearest cumulative boundary of
    the drawn index: how far the draw is from picking a neighbour."""
    w = np.asarray(w, dtype=np.float64)
    c = np.cumsum(w)
    t = float(u) * c[-1]
    j = draw_index(w, u)
    lo = c[j - 1] if j > 0 else 0.0
    return float(min(t - lo, c[j] - t) / c[-1])


def sample_draft(logits, temperature, u):
    """A draft token drawn from q = softmax(logits / T) with the uniform u in [0, 1): the
    drafter's side of the non-greedy path (each drafted position is a sample of the drafter's
    distribution rather than its argmax; the acceptance test below divides by that q)."""
    return draw_index(softmax_t(logits, temperature), u)


def residual(p, q):
    """max(0, p - q): the weights of the draw after a rejection."""
    return np.maximum(0.0, np.asarray(p, np.float64) - np.asarray(q, np.float64))


def accept_stochastic(draft_logits, target_logits, drafts, temperature, u_accept, u_sample,
                      eos=()):
    """One sequence. draft_logits [K, V] (drafter, block positions 1..K), target_logits
    [K+1, V] (verifier at positions 0..K), drafts [K], u_accept [K], u_sample scalar.

    Returns (committed list, accept_count, hit_eos, rollback, info) where info holds the
    decision margins (|u q - p| / max(p, u q) per tested draft, and the draw margin)."""
    drafts = [int(t) for t in drafts]
    K = len(drafts)
    if np.shape(target_logits)[0] != K + 1 or np.shape(draft_logits)[0] != K:
        raise OracleError("need K draft rows and K+1 target rows")
    accept_margins = []
    a = K
    w = None
    for i in range(K):
        p = softmax_t(target_logits[i], temperature)
        q = softmax_t(draft_logits[i], temperature)
        x = drafts[i]
        lhs, rhs = float(u_accept[i]) * q[x], p[x]
        accept_margins.append(abs(lhs - rhs) / max(lhs, rhs, 1e-300))
        if not lhs < rhs:
            a = i
            w = residual(p, q)
            if not np.sum(w) > 0:          # p == q: a rejection cannot happen with u < 1
                w = p
            break
    if w is None:
        w = softmax_t(target_logits[K], temperature)
    token = draw_index(w, u_sample)
    committed = drafts[:a] + [token]
    eos = set(int(e) for e in eos)
    hit = 0
    for i, t in enumerate(committed):
        if t in eos:
            committed = committed[: i + 1]
            hit = 1
            break
    info = {"accept_margins": accept_margins, "draw_margin": draw_margin(w, u_sample),
            "weights": w}
    return committed, a, hit, K - a, info


def first_token_distribution(draft_logits_0, target_logits_0, target_logits_1, temperature):
    """Exact distribution of the first committed token when K = 1 and the draft is drawn from
    q_0: sum over drafts x of q(x) [accept(x) delta_x + (1 - accept(x)) residual], plus the
    all-accepted branch's next-position draw folded in as the token after x (not counted here).
    Used by the pins: it must equal p_0."""
    p = softmax_t(target_logits_0, temperature)
    q = softmax_t(draft_logits_0, temperature)
    acc = np.minimum(1.0, np.divide(p, q, out=np.ones_like(p), where=q > 0))
    r = residual(p, q)
    rs = np.sum(r)
    out = q * acc
    reject_mass = float(np.sum(q * (1.0 - acc)))
    if rs > 0:
        out = out + reject_mass * r / rs
    return out
