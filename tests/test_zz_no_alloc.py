"""lm_head_argmax_noalloc against lm_head_argmax, through the C ABI.

The no-allocation entry point serves callers that cannot allocate device memory (an engine or
plug-in host that owns every allocation, or a loop that cannot take cudaMalloc's implicit
synchronisation): it keeps its scratch in a fixed array inside the library. Two calls in a row
with different inputs must each agree with the workspace-based entry point, which also shows
that nothing left in the shared array by the first call leaks into the second; a small case is
also checked straight against the CPU oracle's lm_head argmax. This file is named to run last;
it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from oracle import core as ocore
from speculative_decoding_drafter_dflash_gb300 import binding as B
from tests.harness import GAP_MIN, REL_TOL, assert_argmax_parity, rel_err

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


def test_noalloc_matches_oracle():
    """H = 256, V = 4096, 5 rows: indices equal the oracle's wherever its top-1/top-2 gap
    exceeds GAP_MIN, top values within REL_TOL."""
    g = torch.Generator(device=DEV).manual_seed(12)
    V, H, rows = 4096, 256, 5
    W = (torch.randn((V, H), generator=g, device=DEV) * 0.05).to(torch.bfloat16)
    X = torch.randn((rows, H), generator=g, device=DEV)
    for _ in range(2):
        idx, t1, t2 = _noalloc(W, X)
        torch.cuda.synchronize()
        bits = W.view(torch.int16).cpu().numpy().view(np.uint16)
        ri, r1, r2 = ocore.lm_head_argmax(X.cpu().numpy(), bits)
        assert_argmax_parity(idx.cpu().numpy(), ri, r1, r2, "noalloc")
        assert rel_err(t1.cpu().numpy(), r1) <= REL_TOL and rel_err(t2.cpu().numpy(), r2) <= REL_TOL


@pytest.mark.parametrize("rows,H,V", [(17, 256, 64), (4, 260, 64), (4, 8200, 64), (4, 256, 524289)])
def test_noalloc_rejects_sizes_beyond_its_scratch(rows, H, V):
    """More than 16 rows, H not a multiple of 8 or above 8192, V above 524288: refused on the
    host before any launch (W is only as large as the rows the shape check needs)."""
    W = torch.zeros((min(V, 64), H), dtype=torch.bfloat16, device=DEV)
    X = torch.zeros((rows, H), device=DEV)
    idx = torch.empty(rows, dtype=torch.int32, device=DEV)
    with pytest.raises(B.DFlashError) as e:
        rc = B.lib().lm_head_argmax_noalloc(B._p(W), B._p(X), rows, H, V, B._p(idx), None, None,
                                             B._stream(None))
        B._check(rc)
    assert e.value.code == B.DF_ESHAPE
