"""GPU parity of the MoE FFN (router, top-k, routed + shared experts) against the CPU oracle,
through the C ABI: on its own (df_moe_ffn) and inside chained MTP draft steps."""
import numpy as np
import pytest
import torch

from oracle import core
from oracle import mtp as omtp
from speculative_decoding_drafter_dflash_gb300 import binding as B
from speculative_decoding_drafter_dflash_gb300 import synth
from speculative_decoding_drafter_dflash_gb300.workloads import MTP_MOE, MTP_MOE_TINY
from tests.harness import REL_TOL, assert_argmax_parity, cache_host, mtp_weights_host, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROUTE_GAP_MIN = 1e-3    # the expert choice must match where the k-th / (k+1)-th logit gap exceeds this


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


def _ffn_case(shape, T, seed):
    w = synth.mtp_weights(shape, seed=seed, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(seed + 100)
    x = torch.randn((T, shape.hidden), generator=g, device=DEV)
    model = B.MtpModel(shape, w, synth.mtp_cache(shape, 1, seed=seed + 1, device=DEV))
    ws = B.alloc_workspace(model.moe_workspace_bytes(T))
    out = torch.empty((T, shape.hidden), device=DEV)
    ids = torch.empty((T, shape.top_k), dtype=torch.int32, device=DEV)
    wts = torch.empty((T, shape.top_k + 1), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.moe_ffn(model, x, out, ws, ids, wts, st)
    torch.cuda.synchronize()
    assert int(st) == 0
    return synth.host(x), mtp_weights_host(w), out.cpu().numpy(), ids.cpu().numpy(), \
        wts.cpu().numpy(), model, ws


def _check_ffn(shape, xs, hw, out, ids, wts):
    checked = 0
    for t in range(xs.shape[0]):
        gap = omtp.route_margin(xs[t], hw["router"], shape.top_k)
        ref, sel, wsel = omtp.moe_ffn(xs[t], hw, shape.top_k)
        if gap <= ROUTE_GAP_MIN:
            continue                      # near tie: either choice is correct
        checked += 1
        assert list(ids[t]) == list(sel), f"row {t}: experts {ids[t]} vs {sel}"
        assert rel_err(wts[t, :shape.top_k], wsel) <= REL_TOL
        sg = core.sigmoid(core.linear(xs[t], hw["sh_gate"]))[0]
        assert abs(wts[t, shape.top_k] - sg) <= REL_TOL * max(abs(sg), 1e-3)
        assert rel_err(out[t], ref) <= REL_TOL, f"row {t}"
    return checked


@pytest.mark.parametrize("T", [1, 5, 16])
def test_moe_ffn_tiny_matches_oracle(T):
    xs, hw, out, ids, wts, _, _ = _ffn_case(MTP_MOE_TINY, T, seed=T)
    assert _check_ffn(MTP_MOE_TINY, xs, hw, out, ids, wts) >= max(1, T - 2)


def test_moe_ffn_ragged_widths():
    """Expert and shared intermediates that differ and do not fill a lane batch; top_k = E."""
    shape = MTP_MOE_TINY.with_(hidden=136, n_experts=6, top_k=6, expert_inter=40, shared_inter=88)
    xs, hw, out, ids, wts, _, _ = _ffn_case(shape, 3, seed=9)
    assert _check_ffn(shape, xs, hw, out, ids, wts) == 3


def test_moe_ffn_full_size_experts():
    """The full MoE FFN shape: H=2048, 256 experts, top-8, expert and shared SwiGLU 512."""
    xs, hw, out, ids, wts, _, _ = _ffn_case(MTP_MOE, 4, seed=3)
    assert _check_ffn(MTP_MOE, xs, hw, out, ids, wts) >= 3


def test_moe_ffn_repeatable_and_counter_left_zero():
    """Two calls on one workspace give identical bits (the last-CTA counter is left at zero)."""
    xs, hw, out, ids, wts, model, ws = _ffn_case(MTP_MOE_TINY, 4, seed=12)
    x = torch.from_numpy(xs).to(DEV)
    out2 = torch.empty_like(x)
    ids2 = torch.empty((4, MTP_MOE_TINY.top_k), dtype=torch.int32, device=DEV)
    B.moe_ffn(model, x, out2, ws, ids2)
    torch.cuda.synchronize()
    assert np.array_equal(out2.cpu().numpy(), out)
    assert np.array_equal(ids2.cpu().numpy(), ids)


def test_moe_ffn_rejects_too_many_rows():
    shape = MTP_MOE_TINY
    w = synth.mtp_weights(shape, seed=1, device=DEV)
    model = B.MtpModel(shape, w, synth.mtp_cache(shape, 1, seed=2, device=DEV))
    assert model.moe_workspace_bytes(17) == 0
    x = torch.zeros((17, shape.hidden), device=DEV)
    ws = B.alloc_workspace(model.moe_workspace_bytes(16))
    with pytest.raises(B.DFlashError) as e:
        B.moe_ffn(model, x, torch.empty_like(x), ws)
    assert e.value.code == B.DF_ESHAPE


def _mtp_run(shape, steps, seed):
    w = synth.mtp_weights(shape, seed=seed, device=DEV)
    cache = synth.mtp_cache(shape, steps, seed=seed + 1, device=DEV)
    prev, tok = synth.mtp_inputs(shape, seed=seed + 2, device=DEV)
    hw = mtp_weights_host(w)
    ks, vs, seq0 = cache_host(cache)
    model = B.MtpModel(shape, w, cache)
    Bn = shape.batch
    ws = B.alloc_workspace(model.workspace_bytes(Bn))
    hid = torch.empty((steps, Bn, shape.hidden), device=DEV)
    am = torch.empty((steps, Bn), dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.mtp_forward_draft(model, prev, tok, steps, hid, am, ws, None, st)
    torch.cuda.synchronize()
    ref = omtp.mtp_forward_draft(shape, hw, ks[0], vs[0], seq0, synth.host(prev), synth.host(tok),
                                 steps)
    return hid.cpu().numpy(), am.cpu().numpy(), int(st), ref, synth.host(cache.seq_len)


def _check_mtp(shape, steps, seed):
    hid, am, st, ref, seq = _mtp_run(shape, steps, seed)
    assert st == 0
    hid_ref, am_ref, t1, t2, seq_ref, infos = ref
    Bn = shape.batch
    for b in range(Bn):
        for s in range(steps):
            info = infos[b * steps + s]
            if info["route_gap"] <= ROUTE_GAP_MIN:
                break                      # a near-tie routing may legitimately fork the chain
            assert rel_err(hid[s, b], hid_ref[s, b]) <= REL_TOL, f"seq {b} step {s}"
            if assert_argmax_parity(am[s, b:b + 1], am_ref[s, b:b + 1], t1[s, b:b + 1],
                                    t2[s, b:b + 1], f"seq {b} step {s}"):
                break
    assert list(seq) == list(seq_ref)


@pytest.mark.parametrize("steps", [1, 3])
def test_mtp_moe_tiny_matches_oracle(steps):
    _check_mtp(MTP_MOE_TINY, steps, seed=5)


def test_mtp_moe_batched():
    _check_mtp(MTP_MOE_TINY.with_(batch=4), 2, seed=6)


@pytest.mark.slow
def test_mtp_moe_full_size_two_steps():
    """The MoE MTP shape at full size (H=2048, 16q/2kv x 256, 256 experts top-8, V=248320,
    KV 16384), two chained steps."""
    _check_mtp(MTP_MOE, 2, seed=23)
