"""The tensor-core attention kernel (head_dim 128 / 256, up to 32 query rows per KV head)
against the oracle, through the DFlash forward and the MTP step: ragged context lengths,
tiles that straddle the cache / block boundary, chunks of several tiles, the causal block
variant, and a check that the tensor-core kernel is the one that ran."""
import numpy as np
import pytest
import torch

from speculative_decoding_drafter_dflash_gb300 import binding as B
from speculative_decoding_drafter_dflash_gb300 import synth
from speculative_decoding_drafter_dflash_gb300.workloads import MTP_TINY, TINY
from tests.harness import REL_TOL, rel_err
from tests.test_gpu_dflash import _run_forward
from tests.test_gpu_mtp import _run as _run_mtp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


def _kernels(fn):
    B.profile_enable(True)
    try:
        out = fn()
        torch.cuda.synchronize()
        names = [n for n, _ in B.profile_read()]
    finally:
        B.profile_enable(False)
    return out, names


@pytest.mark.parametrize("d,nq,nkv,K,ctx,n_new", [
    (128, 4, 2, 4, 300, [3]),        # 10 rows per KV head, cache/block boundary inside a tile
    (128, 4, 2, 15, 250, [0]),       # 32 rows per KV head
    (256, 4, 2, 15, 130, [5]),       # head_dim 256: two 128-wide halves
    (256, 8, 8, 7, 64, [1]),         # one query head per KV head, a single partial tile
])
def test_dflash_forward_tensor_core_attention(d, nq, nkv, K, ctx, n_new):
    shape = TINY.with_(head_dim=d, n_q_heads=nq, n_kv_heads=nkv, K=K, ctx=ctx)
    r, names = _kernels(lambda: _run_forward(shape, n_new, seed=d + ctx))
    assert "attn_tc_kernel" in names and "attn_kernel" not in names
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL


def test_dflash_tensor_core_attention_multi_tile_chunks_batched_causal():
    """16 KV heads x 2 sequences leave ~10 chunks per head, so each chunk spans two tiles."""
    shape = TINY.with_(head_dim=128, n_q_heads=16, n_kv_heads=8, K=15, ctx=2000, batch=2)
    r, names = _kernels(lambda: _run_forward(shape, [7, 2], seed=31))
    assert "attn_tc_kernel" in names
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL
    rc = _run_forward(shape, [4, 9], seed=32, causal=1)
    assert rc["st"] == 0
    assert rel_err(rc["h_final"].cpu().numpy(), rc["ref"]) <= REL_TOL


@pytest.mark.parametrize("d,nq,nkv,kv_len,steps", [(256, 4, 2, 300, 2), (128, 6, 1, 700, 1)])
def test_mtp_tensor_core_attention(d, nq, nkv, kv_len, steps):
    shape = MTP_TINY.with_(head_dim=d, n_q_heads=nq, n_kv_heads=nkv, kv_len=kv_len)
    r, names = _kernels(lambda: _run_mtp(shape, steps, seed=d))
    assert "attn_tc_kernel" in names
    assert r["st"] == 0
    hid_ref = r["ref"][0]
    assert rel_err(r["hid"][0].cpu().numpy(), hid_ref[0]) <= REL_TOL
    assert list(synth.host(r["cache"].seq_len)) == list(r["ref"][4])


def _tc_chunk_keys(B, nkv, max_keys, sms=152):
    """Keys per attention chunk as the library plans them: the whole number of 128-key tiles
    that minimises waves x (tiles per chunk + 1), one CTA per SM, the longer chunk on a tie."""
    heads = B * nkv
    tiles = max(1, (max_keys + 127) // 128)
    best, per = None, tiles
    for p in range(tiles, 0, -1):
        waves = (heads * ((tiles + p - 1) // p) + sms - 1) // sms
        if best is None or waves * (p + 1) < best:
            best, per = waves * (p + 1), p
    return per * 128


@pytest.mark.parametrize("ctx,n_new,causal", [
    (3960, [5], 0),    # chunks 0-14: both tiles' K and V converted before the wait; chunk 15:
                       # tile 0 straddles the old context end, nothing early, block rows in both
    (3960, [5], 1),
    (4000, [16], 0),   # chunk 15: tile 0 early, tile 1 new context + block rows
])
def test_dflash_forward_two_tile_chunks_in_place_v(ctx, n_new, causal):
    """Chunks of two 128-key tiles (head_dim 128, F32 cache) take the in-place V^T operand path;
    the three ways a chunk splits into early and late units, against the oracle."""
    shape = TINY.with_(head_dim=128, n_q_heads=16, n_kv_heads=8, K=15, ctx=ctx)
    assert _tc_chunk_keys(1, 8, ctx + 2 * shape.block) == 256
    r, names = _kernels(lambda: _run_forward(shape, n_new, seed=ctx + causal, causal=causal))
    assert "attn_tc_kernel" in names
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL


def test_dflash_forward_streamed_chunks_batched():
    """8 sequences x 8 KV heads over 63 tiles: 7 chunks of 9 tiles streamed tile by tile inside
    the forward (the first K unit of a chunk below the old context end converted before the
    wait; new context rows and block rows in the last chunk), against the oracle."""
    shape = TINY.with_(head_dim=128, n_q_heads=16, n_kv_heads=8, K=15, ctx=8000, batch=8)
    assert _tc_chunk_keys(8, 8, 8000 + 2 * shape.block) == 9 * 128
    n_new = [3, 0, 16, 1, 7, 2, 5, 9]
    r, names = _kernels(lambda: _run_forward(shape, n_new, seed=41))
    assert "attn_tc_kernel" in names
    assert r["st"] == 0
    assert rel_err(r["h_final"].cpu().numpy(), r["ref"]) <= REL_TOL


# ---------------------------------------------------------------- df_attention on its own
ATTN_TOL = 1e-4   # hi/lo BF16 operands carry ~16 mantissa bits; the CUDA-core path is plain F32


def _attention_case(Bn, blk, nq, nkv, d, seq, cap, block_keys, causal, seed):
    from oracle import core
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((Bn, blk, nq, d), generator=g, device="cuda")
    ck = torch.randn((Bn, nkv, cap, d), generator=g, device="cuda")
    cv = torch.randn((Bn, nkv, cap, d), generator=g, device="cuda")
    kb = torch.randn((Bn, nkv, blk, d), generator=g, device="cuda") if block_keys else None
    vb = torch.randn((Bn, nkv, blk, d), generator=g, device="cuda") if block_keys else None
    sl = torch.tensor(seq, dtype=torch.int32, device="cuda")
    out = torch.full((Bn, blk, nq, d), float("nan"), device="cuda")
    ws = B.alloc_workspace(B.attention_workspace_bytes(Bn, blk, nq, nkv, d, cap))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    (_, names) = _kernels(lambda: B.attention(q, ck, cv, sl, out, ws, kb, vb, causal, st))
    assert int(st) == 0
    got = out.cpu().numpy()
    qh, kh, vh = synth.host(q), synth.host(ck), synth.host(cv)
    for b in range(Bn):
        keys = kh[b, :, :seq[b]].transpose(1, 0, 2)
        vals = vh[b, :, :seq[b]].transpose(1, 0, 2)
        mask = None
        if block_keys:
            keys = np.concatenate([keys, synth.host(kb)[b].transpose(1, 0, 2)])
            vals = np.concatenate([vals, synth.host(vb)[b].transpose(1, 0, 2)])
            if causal:
                mask = np.ones((blk, keys.shape[0]), dtype=bool)
                mask[:, seq[b]:] = np.tril(np.ones((blk, blk), dtype=bool))
        if keys.shape[0] == 0:
            assert np.all(got[b] == 0.0)
            continue
        ref = core.sdpa(qh[b], keys, vals, mask, np.float64)
        assert rel_err(got[b], ref) <= ATTN_TOL, f"sequence {b}"
    return names


@pytest.mark.parametrize("Bn,blk,nq,nkv,d,seq,cap,block_keys,causal,kernel", [
    (2, 16, 16, 8, 128, [1000, 333], 1100, True, False, "attn_tc_kernel"),   # DFlash layout
    (2, 16, 16, 8, 128, [257, 0], 400, True, True, "attn_tc_kernel"),        # causal, empty cache
    (1, 1, 24, 4, 256, [2049], 2100, False, False, "attn_tc_kernel"),        # MTP dense GQA
    (1, 1, 16, 2, 256, [3000], 3000, False, False, "attn_tc_kernel"),        # MTP MoE GQA, full cache
    (3, 4, 4, 2, 64, [100, 1, 77], 128, True, False, "attn_kernel"),         # CUDA-core path
    (1, 2, 2, 1, 32, [50], 64, True, True, "attn_kernel"),
])
def test_attention_matches_oracle(Bn, blk, nq, nkv, d, seq, cap, block_keys, causal, kernel):
    names = _attention_case(Bn, blk, nq, nkv, d, seq, cap, block_keys, causal, seed=d + cap)
    assert kernel in names


@pytest.mark.parametrize("seq,causal", [([4000], False), ([3900], False), ([3900], True)])
def test_attention_two_tile_chunks_in_place_v(seq, causal):
    """256-key chunks of 8 KV heads: every chunk converts its units after the (absent) wait; the
    last holds two tiles with block rows in the second (seq 4000) or a single tile (seq 3900)."""
    assert _tc_chunk_keys(1, 8, 4096 + 16) == 256
    names = _attention_case(1, 16, 16, 8, 128, seq, 4096, True, causal, seed=seq[0] + causal)
    assert "attn_tc_kernel" in names


def test_attention_long_chunks_streamed():
    """64 KV heads over 12116 keys: 7 chunks of 14 tiles (three waves), streamed tile by tile at
    32 query rows (two score buffers, the output accumulated in TMEM across the tiles)."""
    assert _tc_chunk_keys(2, 32, 12100 + 16) == 14 * 128
    names = _attention_case(2, 16, 64, 32, 128, [12000, 9000], 12100, True, False, seed=77)
    assert "attn_tc_kernel" in names


@pytest.mark.parametrize("Bn,blk,nq,nkv,seq,cap,causal,chunk_tiles", [
    (1, 16, 16, 8, [5000], 5100, False, 3),            # 32 rows, 3-tile chunks, block rows last
    (1, 16, 16, 8, [4990], 5100, True, 3),             # causal block, ragged last tile
    (8, 2, 16, 8, [3000, 1, 2999, 0, 1500, 2048, 7, 2500], 3000, False, 12),  # 4 rows per head
])
def test_attention_streamed_chunks(Bn, blk, nq, nkv, seq, cap, causal, chunk_tiles):
    """Chunks longer than two tiles of an F32 cache with head_dim 128: every chunk streamed tile
    by tile, ragged sequence ends, empty sequences, block rows in the last chunk."""
    assert _tc_chunk_keys(Bn, nkv, cap + blk) == chunk_tiles * 128
    names = _attention_case(Bn, blk, nq, nkv, 128, seq, cap, True, causal, seed=cap + blk + causal)
    assert "attn_tc_kernel" in names


def test_attention_streamed_rescales_the_accumulator():
    """Keys whose scores grow along the cache (for the first query row each 128-key tile's
    maximum lies ~11 log2 units above the previous one's, beyond the 2^8 the reference may lag
    by), so the streamed form raises its reference maximum and rescales the output accumulator
    and row sums at every tile; 64 KV heads make 5-tile chunks. q and the keys are BF16 values
    (exact in the hi half), so scores up to ~70 stay exact to F32 accumulation and the float64
    softmax bounds the error as tightly as for unit-sized scores."""
    from oracle import core
    Bn, blk, nq, nkv, d, S, cap = 2, 16, 64, 32, 128, 1200, 1200
    assert _tc_chunk_keys(Bn, nkv, cap + blk) == 5 * 128
    g = torch.Generator(device="cuda").manual_seed(5)
    bf = lambda x: x.to(torch.bfloat16).float()
    q = bf(torch.randn((Bn, blk, nq, d), generator=g, device="cuda"))
    direction = q[0, 0, 0] / q[0, 0, 0].norm()
    ramp = torch.arange(cap, device="cuda", dtype=torch.float32) * (0.7 / 128.0) * d ** 0.5
    ck = torch.randn((Bn, nkv, cap, d), generator=g, device="cuda") * 0.1
    ck = bf(ck + ramp[None, None, :, None] * direction)
    cv = torch.randn((Bn, nkv, cap, d), generator=g, device="cuda")
    kb = bf(torch.randn((Bn, nkv, blk, d), generator=g, device="cuda"))
    vb = torch.randn((Bn, nkv, blk, d), generator=g, device="cuda")
    sl = torch.full((Bn,), S, dtype=torch.int32, device="cuda")
    out = torch.full((Bn, blk, nq, d), float("nan"), device="cuda")
    ws = B.alloc_workspace(B.attention_workspace_bytes(Bn, blk, nq, nkv, d, cap))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.attention(q, ck, cv, sl, out, ws, kb, vb, False, st)
    torch.cuda.synchronize()
    assert int(st) == 0
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    qh, kh, vh = synth.host(q), synth.host(ck), synth.host(cv)
    for b in range(Bn):
        keys = np.concatenate([kh[b, :, :S].transpose(1, 0, 2), synth.host(kb)[b].transpose(1, 0, 2)])
        vals = np.concatenate([vh[b, :, :S].transpose(1, 0, 2), synth.host(vb)[b].transpose(1, 0, 2)])
        ref = core.sdpa(qh[b], keys, vals, None, np.float64)
        assert rel_err(got[b], ref) <= ATTN_TOL, f"sequence {b}"


def test_attention_streamed_late_spike_raises_the_reference():
    """Scores of unit size except one key in the middle of a streamed chunk (tile 2 of its
    5-tile chunk), whose score lies ~24 log2 units above the others for the query rows that point
    along it and as far below for those that point away: the reference maximum stands for two
    tiles, then only some rows exceed it by more than the margin, so the vote for gathering the
    row maxima across lane quarters passes after tiles that skipped it, and rows that do not
    raise keep their reference. q and the keys are BF16 values (exact in the hi half)."""
    from oracle import core
    Bn, blk, nq, nkv, d, S, cap = 2, 16, 64, 32, 128, 1200, 1200
    assert _tc_chunk_keys(Bn, nkv, cap + blk) == 5 * 128
    spike = 640 + 2 * 128 + 37           # chunk 1, tile 2
    g = torch.Generator(device="cuda").manual_seed(11)
    bf = lambda x: x.to(torch.bfloat16).float()
    q = bf(torch.randn((Bn, blk, nq, d), generator=g, device="cuda"))
    ck = torch.randn((Bn, nkv, cap, d), generator=g, device="cuda") * 0.5
    # the spike key of every head points along the first query row of the head's first q head
    for h in range(nkv):
        u = q[:, 0, h * (nq // nkv)]
        ck[:, h, spike] = u / u.norm(dim=-1, keepdim=True) * (24.0 / 1.4427 * d ** 0.5 / 11.3)
    ck = bf(ck)
    cv = torch.randn((Bn, nkv, cap, d), generator=g, device="cuda")
    kb = bf(torch.randn((Bn, nkv, blk, d), generator=g, device="cuda"))
    vb = torch.randn((Bn, nkv, blk, d), generator=g, device="cuda")
    sl = torch.full((Bn,), S, dtype=torch.int32, device="cuda")
    out = torch.full((Bn, blk, nq, d), float("nan"), device="cuda")
    ws = B.alloc_workspace(B.attention_workspace_bytes(Bn, blk, nq, nkv, d, cap))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.attention(q, ck, cv, sl, out, ws, kb, vb, False, st)
    torch.cuda.synchronize()
    assert int(st) == 0
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    qh, kh, vh = synth.host(q), synth.host(ck), synth.host(cv)
    for b in range(Bn):
        keys = np.concatenate([kh[b, :, :S].transpose(1, 0, 2), synth.host(kb)[b].transpose(1, 0, 2)])
        vals = np.concatenate([vh[b, :, :S].transpose(1, 0, 2), synth.host(vb)[b].transpose(1, 0, 2)])
        ref = core.sdpa(qh[b], keys, vals, None, np.float64)
        assert rel_err(got[b], ref) <= ATTN_TOL, f"sequence {b}"
        # the case does what it is for: the aimed rows' spike score tops every earlier key of
        # its chunk by more than the 8 log2 units the reference may lag
        for h in range(nkv):
            sc = kh[b, h, 640:spike + 1].astype(np.float64) @ qh[b, 0, h * (nq // nkv)].astype(np.float64)
            sc *= 1.4426950408889634 / np.sqrt(d)
            assert sc[-1] > sc[:-1].max() + 8.0


def test_attention_head_dim_256_long_chunks_streamed():
    """8 sequences x 2 KV heads of head_dim 256 (MTP MoE heads) over 16000 keys: 9 chunks of 14
    tiles per head (144 CTAs), streamed tile by tile with both 128-wide halves of every K and V
    tile, at 16 query rows."""
    assert _tc_chunk_keys(8, 2, 16000) == 14 * 128
    seq = [16000, 15999, 12000, 1, 0, 8191, 14336, 13001]
    names = _attention_case(8, 1, 16, 2, 256, seq, 16000, False, False, seed=256)
    assert "attn_tc_kernel" in names


def test_attention_head_dim_256_32_rows_streamed():
    """head_dim 256 at 32 query rows (16 block rows x 2 query heads per KV head): two staging
    buffers, the output halves and both score buffers fill TMEM; 3-tile chunks streamed, with
    block rows, against the oracle."""
    assert _tc_chunk_keys(8, 2, 3000 + 16) == 3 * 128
    seq = [3000, 2999, 1, 0, 2500, 1777, 3000, 129]
    names = _attention_case(8, 16, 4, 2, 256, seq, 3000, True, False, seed=2560)
    assert "attn_tc_kernel" in names


def test_attention_no_visible_keys_gives_zeros():
    _attention_case(1, 2, 4, 2, 128, [0], 64, False, False, seed=1)
