"""GPU parity of the device generate loop (df_generate: a CUDA graph whose while node repeats
the draft round) against the CPU oracle's multi-round loop, with a synthetic verifier.

Tokens, rounds, accept histories, drafter cache lengths and captured-prefix lengths are
compared exactly where every drafted position of the oracle run is clear of an argmax near tie
(top-1 - top-2 > 1e-2); with a verifier that never takes a draft the output is the reference
sequence whatever the drafts, and that is checked exactly always."""
import numpy as np
import pytest
import torch

from oracle import generate as og
from speculative_decoding_drafter_dflash_gb300 import binding as B
from speculative_decoding_drafter_dflash_gb300 import synth
from speculative_decoding_drafter_dflash_gb300.workloads import TINY
from tests.harness import GAP_MIN, dflash_weights_host

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


def _case(seed, Bn=3, K=4, prompt=(10, 7, 12), max_len=72, n_comb=3, sel=(0, 2), p_agree=0.5,
          eos_at=None, w_std=None):
    shape = TINY.with_(K=K, batch=Bn) if w_std is None else TINY.with_(K=K, batch=Bn, w_std=w_std)
    w = synth.dflash_weights(shape, seed=seed, device=DEV)
    cache = synth.kv_cache(shape.n_layers, Bn, shape.n_kv_heads, shape.head_dim, 0, max_len + 8,
                           seed + 1, DEV)
    g = torch.Generator(device=DEV).manual_seed(seed + 2)
    ref = torch.randint(2, shape.vocab - 2, (Bn, max_len), generator=g, device=DEV,
                        dtype=torch.int32)
    if eos_at is not None:
        b, p = eos_at
        ref[b, p] = 1
    agree = None
    if p_agree > 0:
        agree = (torch.rand((Bn, max_len), generator=g, device=DEV) < p_agree).to(torch.uint8)
    table = torch.randn((Bn, n_comb, max_len, shape.hidden), generator=g, device=DEV)
    return shape, w, cache, ref, agree, table, list(sel), list(prompt), max_len


def _state(ref, table, prompt, max_len):
    Bn = ref.shape[0]
    out = torch.zeros((Bn, max_len), dtype=torch.int32, device=DEV)
    prior = torch.zeros_like(table)
    for b, pl in enumerate(prompt):
        out[b, :pl + 1] = ref[b, :pl + 1]
        prior[b, :, :pl] = table[b, :, :pl]
    out_len = torch.tensor([p + 1 for p in prompt], dtype=torch.int32, device=DEV)
    prior_len = torch.tensor(prompt, dtype=torch.int32, device=DEV)
    prompt_len = torch.tensor(prompt, dtype=torch.int32, device=DEV)
    return out, out_len, prior, prior_len, prompt_len


def _run_gpu(shape, w, cache, ref, agree, table, sel, prompt, max_len, max_new, max_rounds, ws=None):
    out, out_len, prior, prior_len, prompt_len = _state(ref, table, prompt, max_len)
    Bn, K = ref.shape[0], shape.K
    n_new_max = max(max(prompt), K + 1)
    model = B.DFlashModel(shape, w, cache)
    if ws is None:
        ws = B.alloc_workspace(B.generate_workspace_bytes(model, Bn, K, n_new_max))
    rounds = torch.zeros(Bn, dtype=torch.int32, device=DEV)
    hist = torch.full((max_rounds, Bn), -1, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    eos = torch.tensor([1], dtype=torch.int32, device=DEV)
    B.generate(model, ref, agree, table, sel, prior, prior_len, out, out_len, prompt_len, max_new,
               max_rounds, K, n_new_max, eos, rounds, ws, hist, st)
    torch.cuda.synchronize()
    return dict(out=out.cpu().numpy(), out_len=out_len.cpu().numpy(),
                prior_len=prior_len.cpu().numpy(), rounds=rounds.cpu().numpy(),
                hist=hist.cpu().numpy(), st=int(st), seq=synth.host(cache.seq_len).copy(), ws=ws)


def _run_oracle(shape, w, cache0, ref, agree, table, sel, prompt, max_new, max_rounds):
    hw = dflash_weights_host(w)
    res = []
    for b, pl in enumerate(prompt):
        ks = [synth.host(k)[b:b + 1].copy() for k in cache0.k]
        vs = [synth.host(v)[b:b + 1].copy() for v in cache0.v]
        ag = np.zeros(ref.shape[1], dtype=int) if agree is None else synth.host(agree)[b]
        r = og.generate(shape, hw, ks, vs, int(synth.host(cache0.seq_len)[b]),
                        synth.host(ref)[b, :pl + 1], pl, synth.host(ref)[b], ag,
                        synth.host(table)[b], sel, max_new, shape.K, eos=(1,),
                        max_rounds=max_rounds)
        res.append(r)
    return res


def _compare(g, ref_res, exact_required):
    n_exact = 0
    for b, r in enumerate(ref_res):
        n = int(g["out_len"][b])
        clear = all(gap > GAP_MIN for gap in r["gaps"])
        if not (clear or exact_required):
            continue
        assert list(g["out"][b, :n]) == r["out"], f"sequence {b}"
        if clear:
            assert g["rounds"][b] == r["rounds"], f"sequence {b}"
            assert list(g["hist"][:r["rounds"], b]) == r["accept"], f"sequence {b}"
            assert g["seq"][b] == r["cache_len"] and g["prior_len"][b] == r["prior_len"]
        n_exact += 1
    return n_exact


def test_generate_follows_the_reference_when_the_verifier_never_agrees():
    shape, w, cache, ref, agree, table, sel, prompt, max_len = _case(0, p_agree=0.0)
    cache0 = synth.KvCache([k.clone() for k in cache.k], [v.clone() for v in cache.v],
                           cache.seq_len.clone(), cache.cap)
    g = _run_gpu(shape, w, cache, ref, None, table, sel, prompt, max_len, 11, 40)
    assert g["st"] == 0
    rh = synth.host(ref)
    for b, pl in enumerate(prompt):
        assert g["out_len"][b] == pl + 11
        assert list(g["out"][b, :pl + 11]) == list(rh[b, :pl + 11])
    r = _run_oracle(shape, w, cache0, ref, None, table, sel, prompt, 11, 40)
    assert _compare(g, r, exact_required=True) == len(prompt)


def test_generate_with_agreeing_verifier_and_eos_matches_oracle():
    # larger weights spread the drafter's logits, so fewer rounds hold an argmax near tie
    shape, w, cache, ref, agree, table, sel, prompt, max_len = _case(
        3, Bn=6, prompt=(10, 7, 12, 9, 11, 8), p_agree=0.6, eos_at=(1, 7 + 6), w_std=0.3)
    cache0 = synth.KvCache([k.clone() for k in cache.k], [v.clone() for v in cache.v],
                           cache.seq_len.clone(), cache.cap)
    g = _run_gpu(shape, w, cache, ref, agree, table, sel, prompt, max_len, 16, 40)
    assert g["st"] == 0
    r = _run_oracle(shape, w, cache0, ref, agree, table, sel, prompt, 16, 40)
    assert _compare(g, r, exact_required=False) >= 2
    assert any(a > 0 for rr in r for a in rr["accept"])        # drafts were accepted


def test_generate_round_limit_and_relaunch_of_the_cached_graph():
    shape, w, cache, ref, agree, table, sel, prompt, max_len = _case(5, p_agree=0.3)
    cache0 = synth.KvCache([k.clone() for k in cache.k], [v.clone() for v in cache.v],
                           cache.seq_len.clone(), cache.cap)
    g1 = _run_gpu(shape, w, cache, ref, agree, table, sel, prompt, max_len, 30, 3)
    assert g1["st"] == 0 and list(g1["rounds"]) == [3, 3, 3]
    # same arguments again (the loop graph is relaunched): reset the drafter cache first
    for k, k0 in zip(cache.k, cache0.k):
        k.copy_(k0)
    for v, v0 in zip(cache.v, cache0.v):
        v.copy_(v0)
    cache.seq_len.copy_(cache0.seq_len)
    g2 = _run_gpu(shape, w, cache, ref, agree, table, sel, prompt, max_len, 30, 3, ws=g1["ws"])
    for k in ("out", "out_len", "prior_len", "rounds", "hist", "seq"):
        assert np.array_equal(g1[k], g2[k]), k
    r = _run_oracle(shape, w, cache0, ref, agree, table, sel, prompt, 30, 3)
    _compare(g1, r, exact_required=False)
