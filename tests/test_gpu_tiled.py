"""Tiled weights (df_dflash_tile_weights, df_tile_matrix) through the C ABI.

The layout is checked byte for byte against a NumPy re-layout of the same matrix: 128-row x
64-column tiles, tile (m, kb) at (m * kbt + kb) * 16384, row r of a tile at r * 128, its
16-byte piece j at (j ^ (r % 8)) * 16, zeros past the matrix. The kernels that read the tiled
copy must give the same bits as the kernels that read the row-major matrices: both issue the
same MMAs on the same operands in the same order, only the copies that bring the weights into
shared memory differ (and with them the pipeline stage size).
"""
import numpy as np
import pytest
import torch

from speculative_decoding_drafter_dflash_gb300 import binding as B
from speculative_decoding_drafter_dflash_gb300 import synth
from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15, TINY

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_drafter_dflash_gb300 import build
    build.build()
    B.lib()


def _tiled_reference(bits: np.ndarray) -> np.ndarray:
    """NumPy re-layout of a uint16 [N, K] matrix into the tiled byte image."""
    N, K = bits.shape
    nt, kbt = -(-N // 128), -(-K // 64)
    pad = np.zeros((nt * 128, kbt * 64), dtype=np.uint16)
    pad[:N, :K] = bits
    # [m, r, kb, j, 8] -> [m, kb, r, slot, 8] with slot = j ^ (r % 8)
    t = pad.reshape(nt, 128, kbt, 8, 8).transpose(0, 2, 1, 3, 4).copy()
    out = np.empty_like(t)
    for r in range(128):
        for j in range(8):
            out[:, :, r, j ^ (r % 8), :] = t[:, :, r, j, :]
    return out.reshape(-1).view(np.uint8)


@pytest.mark.parametrize("N,K", [(300, 200), (128, 64), (1, 8), (257, 1000)])
def test_tile_matrix_layout(N, K):
    g = torch.Generator(device=DEV).manual_seed(N + K)
    W = torch.randn((N, K), generator=g, device=DEV).to(torch.bfloat16)
    Wt = B.TiledMatrix(W)
    torch.cuda.synchronize()
    got = Wt.bytes_view().cpu().numpy()
    want = _tiled_reference(W.view(torch.int16).cpu().numpy().view(np.uint16))
    assert got.shape == want.shape and np.array_equal(got, want)


def test_tile_matrix_rejects_bad_arguments():
    W = torch.zeros((64, 64), dtype=torch.bfloat16, device=DEV)
    n = int(B.lib().df_tiled_matrix_bytes(64, 64))
    buf, ptr = B._aligned_buffer(n, W.device)
    with pytest.raises(B.DFlashError) as e:            # too small
        B._check(B.lib().df_tile_matrix(B._p(W), 64, 64, ptr, n - 16, B._stream(None)))
    assert e.value.code == B.DF_EWORKSPACE
    with pytest.raises(B.DFlashError) as e:            # misaligned
        B._check(B.lib().df_tile_matrix(B._p(W), 64, 64, ptr + 512, n, B._stream(None)))
    assert e.value.code == B.DF_EINVAL
    with pytest.raises(B.DFlashError) as e:            # K not a multiple of 8
        B._check(B.lib().df_tile_matrix(B._p(W), 64, 60, ptr, n, B._stream(None)))
    assert e.value.code == B.DF_ESHAPE


@pytest.mark.parametrize("rows,H,V", [(16, 512, 5000), (5, 2816, 70000), (33, 256, 3000)])
def test_lm_head_argmax_tiled_bitwise(rows, H, V):
    g = torch.Generator(device=DEV).manual_seed(rows * 7 + V)
    W = (torch.randn((V, H), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    X = torch.randn((rows, H), generator=g, device=DEV)
    W[V // 3] = W[V - 2]                               # an exact tie in row 0
    X[0] = W[V - 2].float() * 50.0
    ws = B.alloc_workspace(B.lm_head_workspace_bytes(rows, H, V))
    outs = []
    for tiled in (False, True):
        idx = torch.empty(rows, dtype=torch.int32, device=DEV)
        t1 = torch.empty(rows, device=DEV)
        t2 = torch.empty(rows, device=DEV)
        if tiled:
            B.lm_head_argmax_tiled(B.TiledMatrix(W), X, idx, t1, t2, ws)
        else:
            B.lm_head_argmax(W, X, idx, t1, t2, ws)
        torch.cuda.synchronize()
        outs.append((idx.cpu(), t1.cpu(), t2.cpu()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    assert int(outs[1][0][0]) == V // 3


@pytest.mark.parametrize("rows,H,V", [(128, 512, 5000), (64, 2816, 70000), (100, 256, 3000)])
def test_lm_head_argmax_tiled_many_rows_matches_oracle(rows, H, V):
    """64 to 128 rows (one K block per stage, activation slices of 16-32 KB): indices equal the
    oracle's wherever its top-1/top-2 gap exceeds GAP_MIN, values within REL_TOL."""
    from oracle import core as ocore
    from tests.harness import REL_TOL, assert_argmax_parity, rel_err
    g = torch.Generator(device=DEV).manual_seed(rows * 7 + V)
    W = (torch.randn((V, H), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    X = torch.randn((rows, H), generator=g, device=DEV)
    W[V // 3] = W[V - 2]
    X[0] = W[V - 2].float() * 50.0
    ws = B.alloc_workspace(B.lm_head_workspace_bytes(rows, H, V))
    idx = torch.empty(rows, dtype=torch.int32, device=DEV)
    t1 = torch.empty(rows, device=DEV)
    t2 = torch.empty(rows, device=DEV)
    B.lm_head_argmax_tiled(B.TiledMatrix(W), X, idx, t1, t2, ws)
    torch.cuda.synchronize()
    ri, r1, r2 = ocore.lm_head_argmax(synth.host(X), synth.host(W))
    assert_argmax_parity(idx.cpu().numpy(), ri, r1, r2, f"tiled lm_head {rows}x{H}x{V}")
    assert rel_err(t1.cpu().numpy(), r1) <= REL_TOL and rel_err(t2.cpu().numpy(), r2) <= REL_TOL


def _forward(shape, tiled, n_new, seed=0):
    w = synth.dflash_weights(shape, seed=seed, device=DEV)
    cache = synth.dflash_cache(shape, seed=seed + 1, device=DEV)
    inp = synth.dflash_round_inputs(shape, n_new, seed=seed + 2, device=DEV)
    model = B.DFlashModel(shape, w, cache, tiled=tiled)
    nmax = inp.n_new_max
    ws = B.alloc_workspace(model.workspace_bytes(shape.batch, shape.block, nmax))
    h = torch.empty((shape.batch, shape.block, shape.hidden), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.dflash_block_forward(model, inp.block_ids, inp.target_hidden, inp.n_new, nmax, h, ws, st)
    torch.cuda.synchronize()
    assert int(st) == 0
    return h.cpu(), [t.cpu() for t in cache.k], cache.seq_len.cpu()


@pytest.mark.parametrize("shape,n_new", [
    (TINY, [3]),
    (TINY.with_(hidden=384, intermediate=1000, n_q_heads=6, n_kv_heads=3, head_dim=64,
                vocab=5000, K=7, ctx=150, n_target_layers=3, n_layers=2, batch=2), [8, 5]),
])
def test_forward_tiled_bitwise(shape, n_new):
    """Gate/up pairs with a ragged last tile (I = 1000), QKV segments of 384 / 192 / 192 rows,
    K blocks with a ragged tail (K = 1000, 1152): h_final and the appended cache rows equal."""
    a = _forward(shape, False, n_new)
    b = _forward(shape, True, n_new)
    assert torch.equal(a[0], b[0])
    assert all(torch.equal(x, y) for x, y in zip(a[1], b[1]))
    assert torch.equal(a[2], b[2])


def test_forward_tiled_batch8():
    """128 block rows (one K block per stage): h_final and the appended cache rows equal the
    row-major run's within 1e-5 relative, the cache lengths exactly."""
    shape = TINY.with_(hidden=384, intermediate=1000, n_q_heads=6, n_kv_heads=3, head_dim=64,
                       vocab=5000, K=15, ctx=150, n_target_layers=3, n_layers=2, batch=8)
    a = _forward(shape, False, [8, 5, 16, 1, 0, 3, 7, 12])
    b = _forward(shape, True, [8, 5, 16, 1, 0, 3, 7, 12])
    scale = float(a[0].abs().max())
    assert float((a[0] - b[0]).abs().max()) <= 1e-5 * scale
    for x, y in zip(a[1], b[1]):
        assert float((x - y).abs().max()) <= 1e-5 * max(1.0, float(x.abs().max()))
    assert torch.equal(a[2], b[2])


def _round(shape, tiled, seed=3):
    w = synth.dflash_weights(shape, seed=seed, device=DEV)
    cache = synth.dflash_cache(shape, seed=seed + 1, device=DEV)
    inp = synth.dflash_round_inputs(shape, [5] * shape.batch, seed=seed + 2, device=DEV)
    model = B.DFlashModel(shape, w, cache, tiled=tiled)
    ws = B.alloc_workspace(model.workspace_bytes(shape.batch, shape.block, inp.n_new_max))
    out = B.RoundOutputs(shape.batch, shape.K, DEV)
    eos = torch.tensor(shape.eos_ids, dtype=torch.int32, device=DEV)
    tsl = torch.full((shape.batch,), 1 << 30, dtype=torch.int32, device=DEV)
    tgt = torch.zeros((shape.batch, shape.block), dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new, inp.n_new_max, shape.K,
                     tgt, eos, tsl, out, ws, st)
    torch.cuda.synchronize()
    assert int(st) == 0
    res = (out.argmax.cpu(), out.committed.cpu(), out.accept.cpu(), cache.seq_len.cpu())
    del model, w, cache
    torch.cuda.empty_cache()
    return res


@pytest.mark.slow
def test_full_size_round_tiled_bitwise():
    """The DFlash K=15, ctx 4096, V = 262144 round: same drafts, walk and cache length."""
    a = _round(DFLASH_K15, False)
    b = _round(DFLASH_K15, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def _mtp(shape, tiled, steps=2, seed=0):
    w = synth.mtp_weights(shape, seed=seed, device=DEV)
    cache = synth.mtp_cache(shape, steps, seed=seed + 1, device=DEV)
    prev, tok = synth.mtp_inputs(shape, seed=seed + 2, device=DEV)
    model = B.MtpModel(shape, w, cache, tiled=tiled)
    ws = B.alloc_workspace(model.workspace_bytes(shape.batch))
    hid = torch.empty((steps, shape.batch, shape.hidden), device=DEV)
    am = torch.empty((steps, shape.batch), dtype=torch.int32, device=DEV)
    lg = torch.empty((shape.batch, shape.vocab), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.mtp_forward_draft(model, prev, tok, steps, hid, am, ws, logits_out=lg, d_status=st)
    torch.cuda.synchronize()
    assert int(st) == 0
    return hid.cpu(), am.cpu(), lg.cpu(), cache.k[0].cpu()


@pytest.mark.parametrize("which", ["dense", "dense_no_gate", "moe"])
def test_mtp_tiled_bitwise(which):
    """eh_proj (one tiled K range over its two halves, activations by one copy per K block),
    QKV with and without the output-gate rows, the dense gate/up and down, the lm_head argmax
    and logits: the tiled MTP step equals the row-major one bit for bit."""
    from speculative_decoding_drafter_dflash_gb300.workloads import MTP_MOE_TINY, MTP_TINY
    shape = {"dense": MTP_TINY.with_(batch=2), "dense_no_gate": MTP_TINY.with_(gate=False),
             "moe": MTP_MOE_TINY}[which]
    a = _mtp(shape, False)
    b = _mtp(shape, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
