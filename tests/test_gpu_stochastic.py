"""GPU parity of the stochastic (speculative-sampling) accept step against the CPU oracle,
through the C ABI. Accept counts, committed tokens, EOS flags and rollbacks are compared
bit-exactly wherever the oracle's decision is farther than 1e-4 (relative) from its threshold;
nearer decisions may legitimately go either way in F32 and are skipped, the rest of the result
still being checked for validity."""
import numpy as np
import pytest
import torch

from oracle import stochastic as ost
from speculative_decoding_drafter_dflash_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"
DECISION_MARGIN = 1e-4    # relative distance of u q(x) from p(x) below which a test is skipped
DRAW_TOL = 1e-9           # of the total weight: float-float weights and running sums


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


def _inputs(Bn, K, V, seed, spread=2.0, noise=0.5, p_random=0.25, same=False, boost=False):
    """Seeded logits and drafts: the drafter's logits are the target's plus noise (or equal);
    drafts are the drafter's top token, or a random token with probability p_random (with
    boost, the drafter's logit of that random token is raised far above the rest, so the
    drafter is confident where the target is not)."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    tl = torch.randn((Bn, K + 1, V), generator=g, device=DEV) * spread
    dl = tl[:, :K].clone() if same else tl[:, :K] + torch.randn((Bn, K, V), generator=g, device=DEV) * noise
    drafts = torch.argmax(dl, dim=-1).to(torch.int32)
    rnd = torch.randint(0, V, (Bn, K), generator=g, device=DEV, dtype=torch.int32)
    pick = torch.rand((Bn, K), generator=g, device=DEV) < p_random
    drafts = torch.where(pick, rnd, drafts).contiguous()
    if boost:
        top = dl.max(dim=-1).values + 8.0
        dl.scatter_(2, drafts.long().unsqueeze(-1), top.unsqueeze(-1))
    ua = torch.rand((Bn, K), generator=g, device=DEV)
    us = torch.rand((Bn,), generator=g, device=DEV)
    return tl.contiguous(), dl.contiguous(), drafts, ua, us


def _run(tl, dl, drafts, ua, us, T, eos=(1,)):
    Bn, K, V = dl.shape
    out = {k: torch.full((Bn,), -7, dtype=torch.int32, device=DEV)
           for k in ("n_committed", "accept", "hit_eos", "rollback")}
    out["committed"] = torch.full((Bn, K + 1), -7, dtype=torch.int32, device=DEV)
    eos_t = torch.tensor(list(eos), dtype=torch.int32, device=DEV) if eos else None
    ws = B.alloc_workspace(B.accept_stochastic_workspace_bytes(Bn, K, V))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.accept_stochastic(dl, tl, drafts, T, ua, us, eos_t, out, ws, st)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}, int(st), ws, out


def _check(tl, dl, drafts, ua, us, T, got, eos=(1,)):
    """Accept counts and rollbacks bit-exact where the accept test is clear of its threshold;
    the drawn token equal to the oracle's wherever u * W lies more than DRAW_TOL * W from a
    cumulative boundary, and otherwise a valid draw (positive weight, u * W within 2 DRAW_TOL * W
    of its interval). Returns how many sequences drew exactly the oracle's token."""
    Bn, K, V = dl.shape
    tlh, dlh = tl.cpu().numpy(), dl.cpu().numpy()
    dh, uah, ush = drafts.cpu().numpy(), ua.cpu().numpy(), us.cpu().numpy()
    exact = 0
    for b in range(Bn):
        committed, a, hit, rb, info = ost.accept_stochastic(dlh[b], tlh[b], dh[b], T, uah[b],
                                                            float(ush[b]), eos)
        tested = info["accept_margins"][:a + 1] if a < K else info["accept_margins"]
        if min(tested, default=1.0) <= DECISION_MARGIN:
            continue                                 # an accept test sits on its threshold
        assert got["accept"][b] == a and got["rollback"][b] == rb, f"sequence {b}"
        n = got["n_committed"][b]
        row = [int(x) for x in got["committed"][b]]
        assert row[n:] == [-1] * (K + 1 - n)
        assert row[:min(a, n)] == committed[:min(a, n)], f"sequence {b}"
        if n <= a:                                   # cut by an EOS among the accepted drafts
            assert got["hit_eos"][b] == 1 and row[:n] == committed
            exact += 1
            continue
        tok = row[a]
        w = info["weights"]
        c = np.cumsum(w)
        t = float(ush[b]) * c[-1]
        lo = c[tok - 1] if tok > 0 else 0.0
        assert w[tok] > 0 and lo - 2 * DRAW_TOL * c[-1] <= t <= c[tok] + 2 * DRAW_TOL * c[-1], \
            f"sequence {b}: token {tok} is not a draw of u={ush[b]}"
        if info["draw_margin"] > DRAW_TOL:
            assert tok == committed[a], f"sequence {b}: drew {tok}, oracle {committed[a]}"
        exact += int(tok == committed[a])
        want_hit = int(tok in set(eos))
        assert got["hit_eos"][b] == want_hit and n == a + 1
    return exact


@pytest.mark.parametrize("Bn,K,V,T,seed", [(4, 4, 4096, 1.0, 0), (8, 3, 4096, 0.6, 1),
                                           (2, 15, 262144, 0.8, 2), (3, 1, 248320, 1.0, 3)])
def test_accept_stochastic_matches_oracle(Bn, K, V, T, seed):
    tl, dl, drafts, ua, us = _inputs(Bn, K, V, seed)
    got, st, _, _ = _run(tl, dl, drafts, ua, us, T)
    assert st == 0
    exact = _check(tl, dl, drafts, ua, us, T, got)
    assert exact >= Bn - 1          # a draw within 1e-9 of a boundary is a rare event


def test_identical_distributions_accept_every_draft():
    tl, dl, drafts, ua, us = _inputs(4, 6, 8192, 11, same=True, p_random=0.5)
    got, st, _, _ = _run(tl, dl, drafts, ua, us, 1.0, eos=())
    assert st == 0 and list(got["accept"]) == [6] * 4 and list(got["rollback"]) == [0] * 4
    _check(tl, dl, drafts, ua, us, 1.0, got, eos=())


def test_random_drafts_reject_early_and_low_temperature():
    tl, dl, drafts, ua, us = _inputs(6, 5, 4096, 12, spread=4.0, noise=3.0, p_random=0.9,
                                     boost=True)
    got, st, _, _ = _run(tl, dl, drafts, ua, us, 0.3)
    assert st == 0
    _check(tl, dl, drafts, ua, us, 0.3, got)
    assert np.mean(got["accept"]) < 2.5


def test_repeatable_and_counters_left_zero():
    tl, dl, drafts, ua, us = _inputs(3, 4, 16384, 13)
    got, st, ws, out = _run(tl, dl, drafts, ua, us, 0.9)
    eos_t = torch.tensor([1], dtype=torch.int32, device=DEV)
    B.accept_stochastic(dl, tl, drafts, 0.9, ua, us, eos_t, out, ws)
    torch.cuda.synchronize()
    for k, v in out.items():
        assert np.array_equal(v.cpu().numpy(), got[k]), k


def test_rejects_zero_temperature():
    tl, dl, drafts, ua, us = _inputs(1, 2, 64, 14)
    with pytest.raises(B.DFlashError) as e:
        _run(tl, dl, drafts, ua, us, 0.0)
    assert e.value.code == B.DF_EINVAL
