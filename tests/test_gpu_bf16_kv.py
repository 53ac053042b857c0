"""The BF16 KV cache variant of the drafter (df_dflash_config.kv_bf16) against the oracle's
BF16-KV layer: hidden states within 2e-3, cached rows within one BF16 step of the oracle's
(the two sides round slightly different F32 values), through the forward and the round."""
import numpy as np
import pytest
import torch

from speculative_decoding_drafter_dflash_gb300 import binding as B
from speculative_decoding_drafter_dflash_gb300 import synth
from speculative_decoding_drafter_dflash_gb300.workloads import TINY
from tests.harness import REL_TOL, rel_err
from tests.test_gpu_dflash import _run_forward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


def _within_one_bf16_step(got, ref):
    """|got - ref| <= one BF16 step (2^-7 relative) of max(|ref|, rms(ref)): the values the two
    sides round differ by F32 rounding, most visibly where RoPE nearly cancels."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return bool(np.all(np.abs(got - ref) <= 2.0 ** -7 * np.maximum(np.abs(ref), rms)))


@pytest.mark.parametrize("d,nq,nkv,K,ctx,n_new,causal", [
    (128, 4, 2, 4, 300, [3], 0),
    (256, 4, 2, 15, 130, [5], 0),
    (128, 4, 2, 15, 250, [2], 1),
])
def test_bf16_kv_forward_matches_oracle(d, nq, nkv, K, ctx, n_new, causal):
    shape = TINY.with_(head_dim=d, n_q_heads=nq, n_kv_heads=nkv, K=K, ctx=ctx, kv_bf16=True)
    r = _run_forward(shape, n_new, seed=d + ctx, causal=causal)
    assert r["st"] == 0
    assert r["cache"].k[0].dtype == torch.bfloat16
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL
    s0, nn = int(r["seq0"][0]), n_new[0]
    for l in range(shape.n_layers):
        kg = r["cache"].k[l][0, :, s0:s0 + nn].float().cpu().numpy()
        vg = r["cache"].v[l][0, :, s0:s0 + nn].float().cpu().numpy()
        assert _within_one_bf16_step(kg, r["ks"][l][0, :, s0:s0 + nn])
        assert _within_one_bf16_step(vg, r["vs"][l][0, :, s0:s0 + nn])
        # rows before the append are untouched
        kb = r["cache"].k[l][0, :, :s0].float().cpu().numpy()
        assert np.array_equal(kb, r["ks"][l][0, :, :s0])


def test_bf16_kv_batched_streamed_chunks():
    """Two sequences x 16 KV heads with 12000 cached keys: 4 chunks of 24 tiles per head (128
    CTAs, one wave), streamed tile by tile with BF16 units (four TMEM operand regions)."""
    shape = TINY.with_(head_dim=128, n_q_heads=32, n_kv_heads=16, K=15, ctx=12000, batch=2,
                       kv_bf16=True)
    r = _run_forward(shape, [4, 1], seed=91)
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL


def test_bf16_kv_three_tile_chunks_fill_every_buffer_once():
    """One sequence x 8 KV heads over 6000 cached keys (6032 planned keys: 16 chunks of 3 tiles,
    one wave): a streamed BF16 chunk then has as many units (6) as staging buffers, so every copy
    is requested before the conversions start and the TMA-issuer warp has no refill to make."""
    shape = TINY.with_(head_dim=128, n_q_heads=16, n_kv_heads=8, K=15, ctx=6000, batch=1,
                       kv_bf16=True)
    r = _run_forward(shape, [9], seed=97)
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL


def test_bf16_kv_head_dim_256_streamed_chunks():
    """head_dim 256 with a BF16 cache: 8 sequences x 2 KV heads over ~6000 keys, 6-tile chunks
    streamed tile by tile (both halves of each tile, four TMEM operand regions)."""
    shape = TINY.with_(head_dim=256, n_q_heads=4, n_kv_heads=2, K=15, ctx=6000, batch=8,
                       kv_bf16=True)
    r = _run_forward(shape, [4, 1, 16, 0, 7, 3, 9, 2], seed=93)
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL


def test_bf16_kv_rejects_unsupported_head_dim():
    shape = TINY.with_(kv_bf16=True)                  # head_dim 64
    with pytest.raises(B.DFlashError) as e:
        _run_forward(shape, [1], seed=1)
    assert e.value.code == B.DF_ESHAPE
