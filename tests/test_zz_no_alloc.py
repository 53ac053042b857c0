"""lm_head_argmax_noalloc against lm_head_argmax, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device memory (an engine or
plug-in host that owns every allocation, or a loop that cannot take cudaMalloc's implicit
synchronisation): it keeps its scratch in a fixed array inside the library. Two calls in a row
with different inputs must each agree with the workspace-based entry point, which also shows
that nothing left in the shared array by the first call leaks into the second. This file is
named to run last; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_drafter_dflash_gb300 import binding as B
from tests.harness import GAP_MIN, REL_TOL, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


def _reference(W, X):
    rows, H = X.shape
    V = W.shape[0]
    idx = torch.empty(rows, dtype=torch.int32, device=DEV)
    t1 = torch.empty(rows, device=DEV)
    t2 = torch.empty(rows, device=DEV)
    ws = B.alloc_workspace(B.lm_head_workspace_bytes(rows, H, V))
    B.lm_head_argmax(W, X, idx, t1, t2, ws)
    return idx, t1, t2


def _noalloc(W, X):
    rows = X.shape[0]
    idx = torch.empty(rows, dtype=torch.int32, device=DEV)
    t1 = torch.empty(rows, device=DEV)
    t2 = torch.empty(rows, device=DEV)
    B.lm_head_argmax_noalloc(W, X, idx, t1, t2)
    return idx, t1, t2


def _agree(a, b):
    ia, a1, a2 = (t.cpu().numpy() for t in a)
    ib, b1, b2 = (t.cpu().numpy() for t in b)
    clear = (a1 - a2) > GAP_MIN
    assert np.array_equal(ia[clear], ib[clear])
    assert rel_err(b1, a1) <= REL_TOL and rel_err(b2, a2) <= REL_TOL


def test_noalloc_matches_workspace_entry_point_twice():
    g = torch.Generator(device=DEV).manual_seed(11)
    V, H = 70000, 2816
    W = (torch.randn((V, H), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    for rows in (16, 5):                       # two calls in a row, different shapes and inputs
        X = torch.randn((rows, H), generator=g, device=DEV)
        ref = _reference(W, X)
        got = _noalloc(W, X)
        torch.cuda.synchronize()
        _agree(ref, got)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    W = torch.zeros((64, 256), dtype=torch.bfloat16, device=DEV)
    X = torch.zeros((17, 256), device=DEV)
    idx = torch.empty(17, dtype=torch.int32, device=DEV)
    with pytest.raises(B.DFlashError) as e:
        B.lm_head_argmax_noalloc(W, X, idx)
    assert e.value.code == B.DF_ESHAPE
