"""GPU parity of the DFlash draft round against the CPU oracle, through the C ABI.

Floats: max relative error <= 2e-3 (hidden states, logits). Integers (argmax where the
oracle's top-1/top-2 gap exceeds 1e-2, accept walk, rollback, seq_len): bit-exact.
"""
import copy

import numpy as np
import pytest
import torch

from oracle import core as ocore
from oracle import dflash as odf
from speculative_decoding_drafter_dflash_gb300 import binding as B
from speculative_decoding_drafter_dflash_gb300 import synth
from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15, TINY
from tests.harness import (REL_TOL, assert_argmax_parity, cache_host, dflash_weights_host, rel_err)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


def _setup(shape, n_new, seed=0, extra_cap=0):
    w = synth.dflash_weights(shape, seed=seed, device=DEV)
    cache = synth.dflash_cache(shape, seed=seed + 1, device=DEV, extra=extra_cap)
    inp = synth.dflash_round_inputs(shape, n_new, seed=seed + 2, device=DEV)
    model = B.DFlashModel(shape, w, cache)
    return w, cache, inp, model


def _run_forward(shape, n_new, seed=0, causal=0):
    shape = shape.with_(causal_block=causal)
    w, cache, inp, model = _setup(shape, n_new, seed)
    hw = dflash_weights_host(w)
    ks, vs, seq0 = cache_host(cache)
    nmax = inp.n_new_max
    ws = B.alloc_workspace(model.workspace_bytes(shape.batch, shape.block, nmax))
    h_final = torch.empty((shape.batch, shape.block, shape.hidden), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.dflash_block_forward(model, inp.block_ids, inp.target_hidden, inp.n_new, nmax, h_final, ws, st)
    torch.cuda.synchronize()
    ref, seq_ref = odf.dflash_block_forward(shape, hw, ks, vs, seq0, synth.host(inp.block_ids),
                                            synth.host(inp.target_hidden), synth.host(inp.n_new))
    return dict(shape=shape, w=w, hw=hw, cache=cache, ks=ks, vs=vs, seq0=seq0, seq_ref=seq_ref,
                h_final=h_final, ref=ref, st=int(st.item()), inp=inp, model=model, ws=ws)


@pytest.mark.parametrize("n_new", [[3], [0], [5], [1]])
def test_tiny_forward_matches_oracle(n_new):
    r = _run_forward(TINY, n_new)
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL
    assert np.array_equal(synth.host(r["cache"].seq_len), r["seq_ref"])
    # appended context rows of every layer
    s0, nn = int(r["seq0"][0]), n_new[0]
    for l in range(TINY.n_layers):
        kg = synth.host(r["cache"].k[l])[0, :, s0:s0 + nn]
        vg = synth.host(r["cache"].v[l])[0, :, s0:s0 + nn]
        assert rel_err(kg, r["ks"][l][0, :, s0:s0 + nn]) <= REL_TOL
        assert rel_err(vg, r["vs"][l][0, :, s0:s0 + nn]) <= REL_TOL
        # rows before the append are untouched
        assert np.array_equal(synth.host(r["cache"].k[l])[0, :, :s0], r["ks"][l][0, :, :s0])


def test_tiny_forward_batched_ragged_and_causal():
    shape = TINY.with_(batch=3, n_layers=2)
    r = _run_forward(shape, [4, 1, 0])
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL
    assert list(synth.host(r["cache"].seq_len)) == list(r["seq_ref"])
    rc = _run_forward(shape, [2, 3, 1], causal=1)
    assert rel_err(rc["h_final"].cpu().numpy(), rc["ref"]) <= REL_TOL


def test_forward_shapes_spanning_tiles():
    # several GEMM row tiles, ragged tails in every dimension
    shape = TINY.with_(hidden=384, intermediate=1000, n_q_heads=6, n_kv_heads=3, head_dim=64,
                       vocab=5000, K=7, ctx=150, n_target_layers=3, n_layers=2, batch=2)
    r = _run_forward(shape, [8, 5])
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL


def test_lm_head_argmax_matches_oracle():
    g = torch.Generator(device=DEV).manual_seed(5)
    for rows, H, V in [(5, 256, 4096), (16, 512, 10000), (1, 256, 777), (33, 256, 3000)]:
        W = (torch.randn((V, H), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
        X = torch.randn((rows, H), generator=g, device=DEV)
        # plant an exact tie in row 0 between two vocabulary rows
        W[V // 3] = W[V - 2]
        X[0] = W[V - 2].float() * 50.0
        idx = torch.empty(rows, dtype=torch.int32, device=DEV)
        t1 = torch.empty(rows, device=DEV)
        t2 = torch.empty(rows, device=DEV)
        ws = B.alloc_workspace(B.lm_head_workspace_bytes(rows, H, V))
        B.lm_head_argmax(W, X, idx, t1, t2, ws)
        torch.cuda.synchronize()
        ri, r1, r2 = ocore.lm_head_argmax(synth.host(X), synth.host(W))
        assert_argmax_parity(idx.cpu().numpy(), ri, r1, r2, f"lm_head {rows}x{H}x{V}")
        assert int(idx[0]) == V // 3 and float(t1[0]) == float(t2[0])
        assert rel_err(t1.cpu().numpy(), r1) <= REL_TOL
        assert rel_err(t2.cpu().numpy(), r2) <= REL_TOL


def test_accept_walk_and_rollback_device():
    rng = np.random.default_rng(0)
    Bn, K = 64, 7
    drafts = rng.integers(0, 4, size=(Bn, K + 1)).astype(np.int32)   # column 0 unused
    target = rng.integers(0, 4, size=(Bn, K + 1)).astype(np.int32)
    for b in range(Bn):
        a = rng.integers(0, K + 1)
        target[b, :a] = drafts[b, 1:a + 1]
    eos = torch.tensor([1], dtype=torch.int32, device=DEV)
    d = torch.tensor(drafts, device=DEV)
    t = torch.tensor(target, device=DEV)
    out = B.RoundOutputs(Bn, K, DEV)
    B.accept_prefix_argmax(d[:, 1:].contiguous(), K, t, K, eos, out.committed, out.n_committed,
                           out.accept, out.hit_eos, out.rollback)
    # also through a strided view (drafts = argmax rows 1..K)
    out2 = B.RoundOutputs(Bn, K, DEV)
    B.lib()
    import ctypes
    rc = B.lib().accept_prefix_argmax(ctypes.c_void_p(d.data_ptr() + 4), K + 1,
                                      ctypes.c_void_p(t.data_ptr()), Bn, K,
                                      ctypes.c_void_p(eos.data_ptr()), 1,
                                      ctypes.c_void_p(out2.committed.data_ptr()),
                                      ctypes.c_void_p(out2.n_committed.data_ptr()),
                                      ctypes.c_void_p(out2.accept.data_ptr()),
                                      ctypes.c_void_p(out2.hit_eos.data_ptr()),
                                      ctypes.c_void_p(out2.rollback.data_ptr()), None)
    assert rc == 0
    torch.cuda.synchronize()
    for o in (out, out2):
        for b in range(Bn):
            c, a, hit, rb = ocore.accept_walk(drafts[b, 1:], target[b], [1])
            n = int(o.n_committed[b])
            assert o.committed[b, :n].tolist() == c and n == len(c)
            assert all(x == -1 for x in o.committed[b, n:].tolist())
            assert (int(o.accept[b]), int(o.hit_eos[b]), int(o.rollback[b])) == (a, hit, rb)
    seq = torch.tensor([10, 3, 0, 7], dtype=torch.int32, device=DEV)
    n = torch.tensor([4, 3, 0, 8], dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.kv_rollback(seq, n, st)
    torch.cuda.synchronize()
    assert seq.tolist() == [6, 0, 0, 7] and int(st) == B.DF_ECAPACITY


def test_draft_round_tiny_end_to_end():
    shape = TINY.with_(batch=2)
    w, cache, inp, model = _setup(shape, [2, 4], seed=3)
    hw = dflash_weights_host(w)
    ks, vs, seq0 = cache_host(cache)
    # oracle first: its drafts define the synthetic target argmaxes
    ref_h, _ = odf.dflash_block_forward(shape, hw, copy.deepcopy(ks), copy.deepcopy(vs), seq0,
                                        synth.host(inp.block_ids), synth.host(inp.target_hidden),
                                        synth.host(inp.n_new))
    ri, r1, r2 = ocore.lm_head_argmax(ref_h.reshape(-1, shape.hidden), hw["lm_head"])
    ri = ri.reshape(shape.batch, shape.block)
    acc = np.array([2, 4])
    tgt = synth.targets_from_drafts(ri[:, 1:], acc, shape.vocab, seed=9)
    tsl = torch.tensor([100, 100], dtype=torch.int32, device=DEV)
    out = B.RoundOutputs(shape.batch, shape.K, DEV)
    ws = B.alloc_workspace(model.workspace_bytes(shape.batch, shape.block, inp.n_new_max))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    eos = torch.tensor(shape.eos_ids, dtype=torch.int32, device=DEV)
    B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new, inp.n_new_max, shape.K,
                     torch.tensor(tgt, device=DEV), eos, tsl, out, ws, st)
    torch.cuda.synchronize()
    assert int(st) == 0
    gated = assert_argmax_parity(out.argmax.cpu().numpy(), ri, r1, r2, "round argmax")
    res = odf.draft_round(shape, hw, ks, vs, seq0, synth.host(inp.block_ids),
                          synth.host(inp.target_hidden), synth.host(inp.n_new), tgt,
                          shape.eos_ids, [100, 100])
    if gated == 0:
        assert out.accept.tolist() == res["accept"]
        assert out.rollback.tolist() == res["rollback"]
        assert tsl.tolist() == res["target_seq_len"]
    # the integer tail is exact on the GPU's own drafts
    for b in range(shape.batch):
        c, a, hit, rb = ocore.accept_walk(out.argmax[b, 1:].tolist(), tgt[b], shape.eos_ids)
        assert (int(out.accept[b]), int(out.rollback[b])) == (a, rb)
        assert out.committed[b, :int(out.n_committed[b])].tolist() == c


def test_host_round_entry_matches_device_round_pinned_and_pageable():
    # df_draft_round_host: with page-locked host buffers the call runs as a cached CUDA graph
    # (first call captures it, later calls relaunch it with the buffers' current contents);
    # with pageable buffers it runs on the stream. Both must give df_draft_round's results.
    shape = TINY.with_(batch=2)
    w, cache, inp, model = _setup(shape, [2, 4], seed=3)
    seq0 = cache.seq_len.clone()
    tgt = torch.randint(2, shape.vocab - 1, (shape.batch, shape.block), dtype=torch.int32,
                        generator=torch.Generator().manual_seed(5)).to(DEV)
    eos = torch.tensor(shape.eos_ids, dtype=torch.int32, device=DEV)
    ws = B.alloc_workspace(model.workspace_bytes(shape.batch, shape.block, inp.n_new_max))
    out = B.RoundOutputs(shape.batch, shape.K, DEV)
    tsl = torch.tensor([100, 90], dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new, inp.n_new_max, shape.K,
                     tgt, eos, tsl, out, ws, st)
    torch.cuda.synchronize()
    ref = {k: getattr(out, k).cpu() for k in ("argmax", "committed", "n_committed", "accept",
                                              "hit_eos", "rollback")}
    ref["tsl"] = tsl.cpu()
    ws_h = B.alloc_workspace(B.draft_round_host_workspace_bytes(model, shape.batch, shape.K,
                                                                inp.n_new_max, eos.numel()))
    for pin in (True, True, False):
        cache.seq_len.copy_(seq0)
        mk = (lambda t: t.cpu().pin_memory()) if pin else (lambda t: t.cpu().clone())
        hin = dict(last=mk(inp.last_token), th=mk(inp.target_hidden), nn=mk(inp.n_new),
                   tgt=mk(tgt), eos=mk(eos), tsl=mk(torch.tensor([100, 90], dtype=torch.int32)))
        z = lambda *sh: mk(torch.zeros(sh, dtype=torch.int32))
        hout = {"argmax": z(shape.batch, shape.block), "committed": z(shape.batch, shape.block),
                "n_committed": z(shape.batch), "accept": z(shape.batch), "hit_eos": z(shape.batch),
                "rollback": z(shape.batch), "status": z(1)}
        B.df_draft_round_host(model, hin["last"], hin["th"], hin["nn"], inp.n_new_max, shape.K,
                              hin["tgt"], hin["eos"], hin["tsl"], hout, ws_h)
        assert int(hout["status"][0]) == 0
        for k in ("argmax", "committed", "n_committed", "accept", "hit_eos", "rollback"):
            assert torch.equal(hout[k], ref[k]), (pin, k)
        assert torch.equal(hin["tsl"], ref["tsl"])
        assert torch.equal(cache.seq_len.cpu(), seq0.cpu() + inp.n_new.cpu())
    # the cached graph reads the buffers' contents at each launch: new targets in the same
    # pinned buffers must give the device round's results for those targets
    tgt2 = torch.flip(tgt, dims=[1]).contiguous()
    cache.seq_len.copy_(seq0)
    tsl2 = torch.tensor([100, 90], dtype=torch.int32, device=DEV)
    B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new, inp.n_new_max, shape.K,
                     tgt2, eos, tsl2, out, ws, st)
    torch.cuda.synchronize()
    ref2 = {k: getattr(out, k).cpu() for k in ("argmax", "committed", "n_committed", "accept",
                                               "rollback")}
    cache.seq_len.copy_(seq0)
    pin = lambda t: t.cpu().pin_memory()
    hin = dict(last=pin(inp.last_token), th=pin(inp.target_hidden), nn=pin(inp.n_new),
               tgt=pin(tgt), eos=pin(eos), tsl=pin(torch.tensor([100, 90], dtype=torch.int32)))
    z = lambda *sh: pin(torch.zeros(sh, dtype=torch.int32))
    hout = {"argmax": z(shape.batch, shape.block), "committed": z(shape.batch, shape.block),
            "n_committed": z(shape.batch), "accept": z(shape.batch), "hit_eos": z(shape.batch),
            "rollback": z(shape.batch), "status": z(1)}
    B.df_draft_round_host(model, hin["last"], hin["th"], hin["nn"], inp.n_new_max, shape.K,
                          hin["tgt"], hin["eos"], hin["tsl"], hout, ws_h)
    cache.seq_len.copy_(seq0)
    hin["tgt"].copy_(tgt2.cpu())
    hin["tsl"].copy_(torch.tensor([100, 90], dtype=torch.int32))
    B.df_draft_round_host(model, hin["last"], hin["th"], hin["nn"], inp.n_new_max, shape.K,
                          hin["tgt"], hin["eos"], hin["tsl"], hout, ws_h)
    assert int(hout["status"][0]) == 0
    for k in ("argmax", "committed", "n_committed", "accept", "rollback"):
        assert torch.equal(hout[k], ref2[k]), k
    assert torch.equal(hin["tsl"], tsl2.cpu())


def test_device_status_on_capacity_and_bad_ids():
    shape = TINY
    w, cache, inp, model = _setup(shape, [3], seed=4)
    cache.seq_len.fill_(cache.cap - 1)              # 3 new rows cannot fit
    ws = B.alloc_workspace(model.workspace_bytes(1, shape.block, 3))
    h = torch.empty((1, shape.block, shape.hidden), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.dflash_block_forward(model, inp.block_ids, inp.target_hidden, inp.n_new, 3, h, ws, st)
    torch.cuda.synchronize()
    assert int(st) == B.DF_ECAPACITY
    cache.seq_len.fill_(shape.ctx)
    bad = inp.block_ids.clone()
    bad[0, 0] = shape.vocab + 7
    st.zero_()
    B.dflash_block_forward(model, bad, inp.target_hidden, inp.n_new, 3, h, ws, st)
    torch.cuda.synchronize()
    assert int(st) == B.DF_EINVAL
    cache.seq_len.fill_(shape.ctx)
    nn = torch.tensor([5], dtype=torch.int32, device=DEV)     # above n_new_max = 3
    st.zero_()
    B.dflash_block_forward(model, inp.block_ids, inp.target_hidden, nn, 3, h, ws, st)
    torch.cuda.synchronize()
    assert int(st) == B.DF_ESHAPE


def test_determinism_two_identical_calls():
    shape = TINY.with_(batch=2)
    w, cache, inp, model = _setup(shape, [2, 3], seed=6)
    ws = B.alloc_workspace(model.workspace_bytes(2, shape.block, 3))
    outs = []
    for _ in range(2):
        cache.seq_len.fill_(shape.ctx)
        h = torch.empty((2, shape.block, shape.hidden), device=DEV)
        B.dflash_block_forward(model, inp.block_ids, inp.target_hidden, inp.n_new, 3, h, ws)
        outs.append(h)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.slow
def test_full_size_round_k15_ctx4096():
    """The measured workload at full size: h_final of all 16 rows, every argmax (gap-gated),
    the accept walk and rollback, against the oracle on the host."""
    shape = DFLASH_K15
    acc = 3
    w, cache, inp, model = _setup(shape, [acc + 1], seed=0)
    hw = dflash_weights_host(w)
    ks, vs, seq0 = cache_host(cache)
    ws = B.alloc_workspace(model.workspace_bytes(1, shape.block, inp.n_new_max))
    out = B.RoundOutputs(1, shape.K, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    eos = torch.tensor(shape.eos_ids, dtype=torch.int32, device=DEV)
    ref_h, _ = odf.dflash_block_forward(shape, hw, copy.deepcopy(ks), copy.deepcopy(vs), seq0,
                                        synth.host(inp.block_ids), synth.host(inp.target_hidden),
                                        synth.host(inp.n_new))
    ri, r1, r2 = ocore.lm_head_argmax(ref_h.reshape(-1, shape.hidden), hw["lm_head"])
    tgt = synth.targets_from_drafts(ri[None, 1:], np.array([acc]), shape.vocab, seed=1)
    tsl = torch.tensor([5000], dtype=torch.int32, device=DEV)
    B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new, inp.n_new_max, shape.K,
                     torch.tensor(tgt, device=DEV), eos, tsl, out, ws, st)
    h_final = torch.empty((1, shape.block, shape.hidden), device=DEV)
    cache.seq_len.fill_(shape.ctx)
    B.dflash_block_forward(model, inp.block_ids, inp.target_hidden, inp.n_new, inp.n_new_max,
                           h_final, ws, st)
    torch.cuda.synchronize()
    assert int(st) == 0
    assert rel_err(h_final.cpu().numpy(), ref_h) <= REL_TOL
    gated = assert_argmax_parity(out.argmax.cpu().numpy(), ri, r1, r2, "full-size argmax")
    if gated == 0:
        assert int(out.accept[0]) == acc and int(out.rollback[0]) == shape.K - acc
        assert int(tsl[0]) == 5000 - (shape.K - acc)


@pytest.mark.slow
def test_full_size_forward_ctx32768_streamed_attention():
    """The DFlash shape at a 32K-key context: every layer's attention streams 14-tile chunks (19
    chunks x 8 KV heads, one wave) with the new context rows and the block rows in the last
    chunk; h_final and the appended cache length against the oracle."""
    shape = DFLASH_K15.with_(ctx=32768)
    r = _run_forward(shape, [5], seed=6)
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL
    assert list(synth.host(r["cache"].seq_len)) == list(r["seq_ref"])


@pytest.mark.slow
def test_batched_round_b8_ctx1024():
    """The batched sweep shape: 8 sequences x 16 block rows (128 lm_head rows, 256 projection
    tokens with the context rows), K=15, context 1024, ragged new-row counts."""
    shape = DFLASH_K15.with_(batch=8, ctx=1024)
    n_new = [1, 16, 3, 7, 2, 11, 5, 9]
    r = _run_forward(shape, n_new, seed=5)
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL
    assert list(synth.host(r["cache"].seq_len)) == list(r["seq_ref"])
    # lm_head argmax over all 128 rows
    rows = r["h_final"].reshape(-1, shape.hidden)
    idx = torch.empty(rows.shape[0], dtype=torch.int32, device=DEV)
    ws = B.alloc_workspace(B.lm_head_workspace_bytes(rows.shape[0], shape.hidden, shape.vocab))
    B.lm_head_argmax(r["w"].lm_head, rows, idx, ws=ws)
    torch.cuda.synchronize()
    ri, r1, r2 = ocore.lm_head_argmax(r["ref"].reshape(-1, shape.hidden), r["hw"]["lm_head"])
    assert_argmax_parity(idx.cpu().numpy(), ri, r1, r2, "B=8 argmax")


@pytest.mark.slow
def test_batched_draft_round_b8_ctx1024():
    """df_draft_round itself at 8 sequences (128 lm_head rows whose final norm is the lm_head's
    row scale), K=15, context 1024, ragged new-row counts: every argmax (gap-gated), the accept
    walks, rollbacks and cache lengths against the oracle."""
    shape = DFLASH_K15.with_(batch=8, ctx=1024)
    n_new = [1, 16, 3, 7, 2, 11, 5, 9]
    acc = np.array([0, 1, 2, 3, 4, 5, 15, 7])
    w, cache, inp, model = _setup(shape, n_new, seed=6)
    hw = dflash_weights_host(w)
    ks, vs, seq0 = cache_host(cache)
    ref_h, seq_ref = odf.dflash_block_forward(shape, hw, ks, vs, seq0, synth.host(inp.block_ids),
                                              synth.host(inp.target_hidden), synth.host(inp.n_new))
    ri, r1, r2 = ocore.lm_head_argmax(ref_h.reshape(-1, shape.hidden), hw["lm_head"])
    Bn, blk = shape.batch, shape.block
    tgt = synth.targets_from_drafts(ri.reshape(Bn, blk)[:, 1:], acc, shape.vocab, seed=2)
    ws = B.alloc_workspace(model.workspace_bytes(Bn, blk, inp.n_new_max))
    out = B.RoundOutputs(Bn, shape.K, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    eos = torch.tensor(shape.eos_ids, dtype=torch.int32, device=DEV)
    tsl = torch.full((Bn,), 5000, dtype=torch.int32, device=DEV)
    B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new, inp.n_new_max, shape.K,
                     torch.tensor(tgt, device=DEV), eos, tsl, out, ws, st)
    torch.cuda.synchronize()
    assert int(st) == 0
    am = out.argmax.cpu().numpy()
    assert_argmax_parity(am, ri, r1, r2, "B=8 round argmax")
    assert list(synth.host(cache.seq_len)) == list(seq_ref)
    gap = (r1 - r2).reshape(Bn, blk)
    for b in range(Bn):
        if np.all(gap[b] > 1e-2):
            c, a, hit, rb = ocore.accept_walk(ri.reshape(Bn, blk)[b, 1:], tgt[b], shape.eos_ids)
            assert int(out.accept[b]) == a and int(out.rollback[b]) == rb, f"sequence {b}"
            assert int(synth.host(tsl)[b]) == 5000 - rb
            n = int(out.n_committed[b])
            assert out.committed[b, :n].cpu().numpy().tolist() == c
