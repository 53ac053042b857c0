"""GPU parity of the sampled (T > 0) drafts against the CPU oracle, through the C ABI:
`sample_softmax` alone, the non-greedy DFlash round (`df_draft_round_stochastic`) and the
sampled MTP chain (`mtp_forward_draft_sampled`).

A draw from the same logits must equal the oracle's float64 draw wherever u * total lies more
than DRAW_TOL (a fraction of the total) from a cumulative boundary: the kernels compute the
weights to ~1e-14 relative and sum and scan them as float-float pairs. Where the drafter's own
logits feed a draw, the GPU's logits are compared with the oracle's within the float tolerance and the
draw is checked on the GPU's logits (the integer decision is taken on the kernel's floats); the
drafts must also equal the oracle's own where its draw margin exceeds LOGIT_DRAW_TOL, which
covers the logit differences of the whole forward."""
import copy

import numpy as np
import pytest
import torch

from oracle import dflash as odf
from oracle import mtp as omtp
from oracle import stochastic as ost
from speculative_decoding_drafter_dflash_gb300 import binding as B
from speculative_decoding_drafter_dflash_gb300 import synth
from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15, MTP_TINY, TINY
from tests.harness import REL_TOL, cache_host, dflash_weights_host, mtp_weights_host, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
DRAW_TOL = 1e-9          # same logits: float64 reference vs float-float weights
LOGIT_DRAW_TOL = 1e-3    # drafter logits within ~1e-5 relative of the oracle's


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


def _draws(logits, T, u):
    R, V = logits.shape
    tokens = torch.full((R,), -7, dtype=torch.int32, device=DEV)
    ws = B.alloc_workspace(B.sample_softmax_workspace_bytes(R, V))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.sample_softmax(logits, T, u, tokens, ws, st)
    torch.cuda.synchronize()
    return tokens.cpu().numpy(), int(st), ws, tokens


def _check_draw(logits_row, T, u, tok, tol=DRAW_TOL, what=""):
    """tok must be the oracle's draw unless u * total is within tol of a boundary, where it
    must still be a valid draw of that neighbourhood. Returns 1 if it was checked exactly."""
    q = ost.softmax_t(logits_row, T)
    want = ost.draw_index(q, u)
    if ost.draw_margin(q, u) > tol:
        assert tok == want, f"{what}: drew {tok}, oracle {want} (u={u})"
        return 1
    c = np.cumsum(q)
    t = u * c[-1]
    lo = c[tok - 1] if tok > 0 else 0.0
    assert q[tok] > 0 and lo - 2 * tol <= t <= c[tok] + 2 * tol, f"{what}: {tok} is no draw of u"
    return 0


@pytest.mark.parametrize("R,V,T,spread,seed", [(8, 4096, 1.0, 2.0, 0), (4, 262144, 1.0, 1.0, 1),
                                               (3, 248320, 0.7, 2.0, 2), (16, 262144, 1.3, 3.0, 3),
                                               (5, 1000, 0.5, 1.0, 4), (2, 16, 2.0, 0.5, 5)])
def test_sample_softmax_matches_oracle(R, V, T, spread, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    logits = torch.randn((R, V), generator=g, device=DEV) * spread
    u = torch.rand((R,), generator=g, device=DEV)
    got, st, _, _ = _draws(logits, T, u)
    assert st == 0
    lh, uh = logits.cpu().numpy(), u.cpu().numpy()
    exact = sum(_check_draw(lh[r], T, float(uh[r]), int(got[r]), what=f"row {r}") for r in range(R))
    assert exact >= R - 1            # a draw within 1e-9 of a boundary is a rare event


def test_sample_softmax_closed_forms():
    """Equal logits: the draw is floor(u V). One dominant logit: always that token. A row whose
    first half is -inf never draws from it. The same call twice draws the same tokens."""
    V = 4096
    u = torch.tensor([0.0, 0.3, 0.731, 0.99999], device=DEV)
    flat = torch.zeros((4, V), device=DEV)
    got, st, ws, tokens = _draws(flat, 1.0, u)
    assert st == 0 and list(got) == [int(np.floor(float(x) * V)) for x in u.cpu().numpy()]
    peak = torch.randn((4, V), device=DEV)
    peak[:, 1234] = 200.0
    got, st, _, _ = _draws(peak, 0.9, u)
    assert st == 0 and list(got) == [1234] * 4
    half = torch.randn((4, V), device=DEV)
    half[:, : V // 2] = -float("inf")
    got, st, ws, tokens = _draws(half, 1.0, u)
    assert st == 0 and all(t >= V // 2 for t in got)
    st_t = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.sample_softmax(half, 1.0, u, tokens, ws, st_t)
    torch.cuda.synchronize()
    assert int(st_t) == 0 and np.array_equal(tokens.cpu().numpy(), got)


def test_sample_softmax_all_masked_row_sets_status():
    logits = torch.full((2, 64), -float("inf"), device=DEV)
    logits[1, 7] = 0.0
    got, st, _, _ = _draws(logits, 1.0, torch.tensor([0.5, 0.5], device=DEV))
    assert st == B.DF_EINVAL and got[1] == 7


def test_sample_softmax_rejects_bad_arguments():
    logits = torch.zeros((2, 64), device=DEV)
    u = torch.zeros(2, device=DEV)
    tokens = torch.zeros(2, dtype=torch.int32, device=DEV)
    ws = B.alloc_workspace(B.sample_softmax_workspace_bytes(2, 64))
    with pytest.raises(B.DFlashError) as e:
        B.sample_softmax(logits, 0.0, u, tokens, ws)
    assert e.value.code == B.DF_EINVAL
    with pytest.raises(B.DFlashError) as e:
        B.sample_softmax(torch.zeros((2, 62), device=DEV), 1.0, u, tokens, ws)
    assert e.value.code == B.DF_ESHAPE


# --------------------------------------------------------------- the non-greedy DFlash round

def _stochastic_round(shape, n_new, T, seed=0, spread=2.0):
    w = synth.dflash_weights(shape, seed=seed, device=DEV)
    cache = synth.dflash_cache(shape, seed=seed + 1, device=DEV)
    inp = synth.dflash_round_inputs(shape, n_new, seed=seed + 2, device=DEV)
    model = B.DFlashModel(shape, w, cache)
    hw = dflash_weights_host(w)
    ks, vs, seq0 = cache_host(cache)
    Bn, K, V = shape.batch, shape.K, shape.vocab
    g = torch.Generator(device=DEV).manual_seed(seed + 3)
    tl = torch.randn((Bn, K + 1, V), generator=g, device=DEV) * spread
    ud = torch.rand((Bn, K), generator=g, device=DEV)
    ua = torch.rand((Bn, K), generator=g, device=DEV)
    us = torch.rand((Bn,), generator=g, device=DEV)
    eos = torch.tensor(shape.eos_ids, dtype=torch.int32, device=DEV)
    tsl = torch.full((Bn,), 1000, dtype=torch.int32, device=DEV)
    logits = torch.full((Bn, K + 1, V), float("nan"), device=DEV)
    drafts = torch.full((Bn, K), -7, dtype=torch.int32, device=DEV)
    out = B.RoundOutputs(Bn, K, DEV)
    ws = B.alloc_workspace(B.draft_round_stochastic_workspace_bytes(model, Bn, K, inp.n_new_max))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.df_draft_round_stochastic(model, inp.last_token, inp.target_hidden, inp.n_new,
                                inp.n_new_max, K, tl, T, ud, ua, us, eos, tsl, logits, drafts,
                                out, ws, st)
    torch.cuda.synchronize()
    h = synth.host
    ref = odf.draft_round_stochastic(shape, hw, ks, vs, seq0, h(inp.block_ids),
                                     h(inp.target_hidden), h(inp.n_new), h(tl), T, h(ud), h(ua),
                                     h(us), shape.eos_ids, [1000] * Bn)
    return dict(st=int(st), logits=h(logits), drafts=h(drafts), tl=h(tl), ud=h(ud), ua=h(ua),
                us=h(us), out=out, tsl=h(tsl), ref=ref, cache=cache)


def _check_round(r, T, eos):
    """Logits within the float tolerance; drafts and the accept step exact on the GPU's own
    logits (and equal to the oracle's drafts where its margin covers the logit differences)."""
    ref = r["ref"]
    Bn, K1, V = r["logits"].shape
    K = K1 - 1
    assert rel_err(r["logits"], ref["logits"]) <= REL_TOL
    for b in range(Bn):
        for i in range(K):
            _check_draw(r["logits"][b, 1 + i], T, float(r["ud"][b, i]), int(r["drafts"][b, i]),
                        what=f"seq {b} draft {i}")
            q_ref = ost.softmax_t(ref["logits"][b, 1 + i], T)
            if ost.draw_margin(q_ref, float(r["ud"][b, i])) > LOGIT_DRAW_TOL:
                assert r["drafts"][b, i] == ref["drafts"][b][i], f"seq {b} draft {i}"
        # the accept step on the GPU's drafter logits and drafts
        c, a, hit, rb, info = ost.accept_stochastic(r["logits"][b, 1:], r["tl"][b],
                                                    r["drafts"][b], T, r["ua"][b],
                                                    float(r["us"][b]), eos)
        tested = info["accept_margins"][:a + 1] if a < K else info["accept_margins"]
        if min(tested, default=1.0) <= 1e-4:
            continue
        assert int(r["out"].accept[b]) == a and int(r["out"].rollback[b]) == rb
        assert int(r["tsl"][b]) == 1000 - rb
        n = int(r["out"].n_committed[b])
        row = [int(x) for x in r["out"].committed[b].cpu().numpy()]
        if info["draw_margin"] > DRAW_TOL:
            assert row[:n] == c and int(r["out"].hit_eos[b]) == hit, f"seq {b}"
        else:
            assert row[:min(a, n)] == c[:min(a, n)]


@pytest.mark.parametrize("Bn,n_new,T", [(1, [3], 1.0), (2, [2, 5], 0.7), (3, [1, 0, 4], 1.5)])
def test_tiny_stochastic_round_matches_oracle(Bn, n_new, T):
    shape = TINY.with_(batch=Bn)
    r = _stochastic_round(shape, n_new, T, seed=Bn)
    assert r["st"] == 0
    _check_round(r, T, shape.eos_ids)
    assert list(synth.host(r["cache"].seq_len)) == list(r["ref"]["seq_len"])


def test_tiny_stochastic_round_low_temperature_is_greedy():
    """At T = 1e-3 the drafter's softmax is one-hot: the sampled drafts are its argmaxes."""
    shape = TINY.with_(batch=2)
    r = _stochastic_round(shape, [2, 3], 1e-3, seed=7)
    assert r["st"] == 0
    am = r["logits"].argmax(-1)
    assert np.array_equal(r["drafts"], am[:, 1:])


@pytest.mark.slow
def test_full_size_stochastic_round_k15_ctx4096():
    """The non-greedy round at the DFlash K=15 / ctx 4096 / V = 262144 shape."""
    r = _stochastic_round(DFLASH_K15, [4], 1.0, seed=0, spread=1.0)
    assert r["st"] == 0
    _check_round(r, 1.0, DFLASH_K15.eos_ids)


# --------------------------------------------------------------- the sampled MTP chain

@pytest.mark.parametrize("steps,T", [(1, 1.0), (3, 0.8)])
def test_mtp_sampled_chain_matches_oracle(steps, T):
    shape = MTP_TINY
    w = synth.mtp_weights(shape, seed=4, device=DEV)
    cache = synth.mtp_cache(shape, steps, seed=5, device=DEV)
    prev, tok = synth.mtp_inputs(shape, seed=6, device=DEV)
    hw = mtp_weights_host(w)
    ks, vs, seq0 = cache_host(cache)
    model = B.MtpModel(shape, w, cache)
    Bn, V = shape.batch, shape.vocab
    g = torch.Generator(device=DEV).manual_seed(8)
    u = torch.rand((steps, Bn), generator=g, device=DEV)
    ws = B.alloc_workspace(model.workspace_bytes(Bn))
    hid = torch.empty((steps, Bn, shape.hidden), device=DEV)
    dr = torch.full((steps, Bn), -7, dtype=torch.int32, device=DEV)
    lg = torch.empty((steps, Bn, V), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.mtp_forward_draft_sampled(model, prev, tok, steps, T, u, hid, dr, lg, ws, st)
    torch.cuda.synchronize()
    assert int(st) == 0
    h = synth.host
    uh = h(u)
    ref_hid, ref_dr, ref_lg, ref_seq = omtp.mtp_forward_draft_sampled(
        shape, hw, copy.deepcopy(ks[0]), copy.deepcopy(vs[0]), seq0, h(prev), h(tok), steps, T, uh)
    gh, gd, gl = h(hid), h(dr), h(lg)
    assert list(h(cache.seq_len)) == list(ref_seq)
    # step by step while the chains draw the same tokens (a draw within the logit tolerance of
    # a boundary may legitimately fork them)
    live = np.ones(Bn, dtype=bool)
    for s in range(steps):
        for b in range(Bn):
            if not live[b]:
                continue
            assert rel_err(gh[s, b], ref_hid[s, b]) <= REL_TOL, f"step {s} seq {b}"
            assert rel_err(gl[s, b], ref_lg[s, b]) <= REL_TOL, f"step {s} seq {b}"
            _check_draw(gl[s, b], T, float(uh[s, b]), int(gd[s, b]), what=f"step {s} seq {b}")
            q_ref = ost.softmax_t(ref_lg[s, b], T)
            if ost.draw_margin(q_ref, float(uh[s, b])) > LOGIT_DRAW_TOL:
                assert gd[s, b] == ref_dr[s, b], f"step {s} seq {b}"
            else:
                live[b] = gd[s, b] == ref_dr[s, b]
