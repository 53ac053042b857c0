"""GPU parity of the tensor-core projection (df_linear) against the oracle's plain
definition y = x W^T, over shapes that span several tiles, ragged K / N / token counts,
and more tokens than one MMA holds."""
import numpy as np
import pytest
import torch

from oracle import core as ocore
from speculative_decoding_drafter_dflash_gb300 import binding as B
from speculative_decoding_drafter_dflash_gb300 import synth
from tests.harness import REL_TOL, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"

# The hi/lo split carries ~16 mantissa bits of every activation, so one projection agrees with
# the F32 oracle far inside the round tolerance; a dropped lo half would show up near 2e-3.
LINEAR_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


@pytest.mark.parametrize("T,N,K", [(1, 300, 64), (16, 1000, 520), (33, 128, 2816), (128, 2048, 256),
                                   (200, 256, 128), (16, 2816, 14080), (7, 5000, 8)])
def test_linear_matches_oracle(T, N, K):
    g = torch.Generator(device=DEV).manual_seed(T * 7 + N + K)
    W = (torch.randn((N, K), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    X = torch.randn((T, K), generator=g, device=DEV)
    Y = torch.empty((T, N), device=DEV)
    ws = B.alloc_workspace(B.linear_workspace_bytes(T, N, K))
    B.df_linear(W, X, Y, ws)
    torch.cuda.synchronize()
    ref = ocore.linear(synth.host(X), synth.host(W))
    assert rel_err(Y.cpu().numpy(), ref) <= LINEAR_TOL


def test_linear_repeated_calls_identical():
    g = torch.Generator(device=DEV).manual_seed(1)
    W = (torch.randn((3000, 2816), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    X = torch.randn((16, 2816), generator=g, device=DEV)
    ws = B.alloc_workspace(B.linear_workspace_bytes(16, 3000, 2816))
    Y1 = torch.empty((16, 3000), device=DEV)
    Y2 = torch.empty((16, 3000), device=DEV)
    B.df_linear(W, X, Y1, ws)
    B.df_linear(W, X, Y2, ws)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)
