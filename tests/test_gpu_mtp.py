"""GPU parity of the MTP (NextN) draft step against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import mtp as omtp
from speculative_decoding_drafter_dflash_gb300 import binding as B
from speculative_decoding_drafter_dflash_gb300 import synth
from speculative_decoding_drafter_dflash_gb300.workloads import MTP_TINY
from tests.harness import REL_TOL, assert_argmax_parity, cache_host, mtp_weights_host, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


def _run(shape, steps, seed=0, logits=False):
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
    lg = torch.empty((Bn, shape.vocab), device=DEV) if logits else None
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.mtp_forward_draft(model, prev, tok, steps, hid, am, ws, lg, st)
    torch.cuda.synchronize()
    ref = omtp.mtp_forward_draft(shape, hw, ks[0], vs[0], seq0, synth.host(prev), synth.host(tok),
                                 steps)
    return dict(hid=hid, am=am, lg=lg, st=int(st), ref=ref, cache=cache, hw=hw, seq0=seq0,
                ks=ks, vs=vs)


@pytest.mark.parametrize("steps", [1, 3])
def test_mtp_dense_tiny_matches_oracle(steps):
    r = _run(MTP_TINY, steps)
    assert r["st"] == 0
    hid_ref, am_ref, t1, t2, seq_ref, _ = r["ref"]
    # Each chained step consumes the previous argmax; compare step by step while the argmax
    # decisions agree (near ties would legitimately fork the chain).
    for s in range(steps):
        assert rel_err(r["hid"][s].cpu().numpy(), hid_ref[s]) <= REL_TOL, f"step {s}"
        gated = assert_argmax_parity(r["am"][s].cpu().numpy(), am_ref[s], t1[s], t2[s], f"step {s}")
        if gated:
            break
    assert list(synth.host(r["cache"].seq_len)) == list(seq_ref)


def test_mtp_batched_with_logits():
    shape = MTP_TINY.with_(batch=3, head_dim=128, n_q_heads=6, n_kv_heads=2)
    r = _run(shape, 2, seed=4, logits=True)
    assert r["st"] == 0
    hid_ref, am_ref, t1, t2, _, _ = r["ref"]
    assert rel_err(r["hid"][0].cpu().numpy(), hid_ref[0]) <= REL_TOL
    g = assert_argmax_parity(r["am"][0].cpu().numpy(), am_ref[0], t1[0], t2[0], "batched")
    if g == 0:
        assert rel_err(r["hid"][1].cpu().numpy(), hid_ref[1]) <= REL_TOL
        # dense logits of the last step agree with the oracle's own logits
        from oracle import core
        sh = r["hw"]
        x = core.rmsnorm(hid_ref[1], sh["shared_head_norm"], shape.rms_eps)
        ref_logits = core.linear(x, sh["lm_head"])
        assert rel_err(r["lg"].cpu().numpy(), ref_logits) <= REL_TOL


def test_mtp_without_output_gate():
    shape = MTP_TINY.with_(gate=False)
    r = _run(shape, 1, seed=7)
    hid_ref = r["ref"][0]
    assert rel_err(r["hid"][0].cpu().numpy(), hid_ref[0]) <= REL_TOL


@pytest.mark.slow
def test_mtp_dense_full_size_two_steps():
    """The dense MTP shape at full size (H=5120, 24q/4kv x 256, I=17408, V=248320, KV 8192),
    two chained steps."""
    from speculative_decoding_drafter_dflash_gb300.workloads import MTP_DENSE
    r = _run(MTP_DENSE, 2, seed=21)
    assert r["st"] == 0
    hid_ref, am_ref, t1, t2, seq_ref, _ = r["ref"]
    assert rel_err(r["hid"][0].cpu().numpy(), hid_ref[0]) <= REL_TOL
    gated = assert_argmax_parity(r["am"][0].cpu().numpy(), am_ref[0], t1[0], t2[0], "step 0")
    if gated == 0:
        assert rel_err(r["hid"][1].cpu().numpy(), hid_ref[1]) <= REL_TOL
        assert_argmax_parity(r["am"][1].cpu().numpy(), am_ref[1], t1[1], t2[1], "step 1")
    assert list(synth.host(r["cache"].seq_len)) == list(seq_ref)
