"""A bounded device wait that runs out, through the C ABI: the failure-detection path of the
tensor-core projection kernel.

With the test hook, every projection CTA's TMA producer withholds the load of its first pipeline
stage, so the MMA warp's wait on that stage runs out after a short limit (1e5 SM cycles). The
call must come back with DF_ETIMEOUT in its status word and leave the context usable: every role
leaves, the loads that were issued land and tensor memory is freed, so an ordinary call right
after it matches the CPU oracle. No GPU fault, trap or unbounded wait is involved."""
import copy

import numpy as np
import pytest
import torch

from oracle import dflash as odf
from speculative_decoding_drafter_dflash_gb300 import binding as B
from speculative_decoding_drafter_dflash_gb300 import synth
from speculative_decoding_drafter_dflash_gb300.workloads import TINY
from tests.harness import REL_TOL, cache_host, dflash_weights_host, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


def _forward(model, inp, ws):
    h_final = torch.full((1, TINY.block, TINY.hidden), float("nan"), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.dflash_block_forward(model, inp.block_ids, inp.target_hidden, inp.n_new, inp.n_new_max,
                           h_final, ws, st)
    torch.cuda.synchronize()
    return h_final, int(st)


def test_projection_wait_runs_out_then_an_ordinary_call_is_exact():
    w = synth.dflash_weights(TINY, seed=0, device=DEV)
    cache = synth.dflash_cache(TINY, seed=1, device=DEV)
    inp = synth.dflash_round_inputs(TINY, [3], seed=2, device=DEV)
    model = B.DFlashModel(TINY, w, cache)
    ws = B.alloc_workspace(model.workspace_bytes(1, TINY.block, inp.n_new_max))
    B.test_wait_hook(100000, True)
    try:
        _, st = _forward(model, inp, ws)
    finally:
        B.test_wait_hook(0, False)
    assert st == B.DF_ETIMEOUT
    # a fresh cache (the aborted call appended meaningless rows), then an ordinary call
    cache = synth.dflash_cache(TINY, seed=1, device=DEV)
    model.set_cache(cache)
    ks, vs, seq0 = cache_host(cache)
    h_final, st = _forward(model, inp, ws)
    assert st == 0
    ref, seq_ref = odf.dflash_block_forward(TINY, dflash_weights_host(w), ks, vs, seq0,
                                            synth.host(inp.block_ids),
                                            synth.host(inp.target_hidden), synth.host(inp.n_new))
    assert rel_err(h_final.cpu().numpy(), ref) <= REL_TOL
    assert np.array_equal(synth.host(cache.seq_len), seq_ref)


def test_hook_rejects_withholding_without_a_limit():
    with pytest.raises(B.DFlashError) as e:
        B.test_wait_hook(0, True)
    assert e.value.code == B.DF_EINVAL
    with pytest.raises(B.DFlashError):
        B.test_wait_hook(-5, False)
    B.test_wait_hook(0, False)
