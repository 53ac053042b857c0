"""Host checks of the seeded input generators (no GPU)."""
import numpy as np
import torch

from speculative_decoding_drafter_dflash_gb300 import synth
from speculative_decoding_drafter_dflash_gb300.workloads import TINY


def test_accept_lengths_geometric_and_capped():
    a = synth.accept_lengths(200000, 15, 0.6, seed=0)
    assert a.min() >= 0 and a.max() <= 15
    for j in (1, 2, 3, 5):
        assert abs(np.mean(a >= j) - 0.6 ** j) < 0.01
    u = synth.accept_lengths(50000, 4, None, seed=1)
    assert set(np.unique(u)) == {0, 1, 2, 3, 4}


def test_targets_agree_on_prefix_then_differ():
    rng = np.random.default_rng(0)
    drafts = rng.integers(0, 100, size=(64, 7))
    acc = synth.accept_lengths(64, 7, None, seed=2)
    t = synth.targets_from_drafts(drafts, acc, 100, seed=3)
    assert t.shape == (64, 8)
    for b in range(64):
        a = acc[b]
        assert np.array_equal(t[b, :a], drafts[b, :a])
        if a < 7:
            assert t[b, a] != drafts[b, a]


def test_tiny_inputs_shapes_and_seeding():
    w1 = synth.dflash_weights(TINY, seed=0)
    w2 = synth.dflash_weights(TINY, seed=0)
    assert torch.equal(w1.fc.view(torch.int16), w2.fc.view(torch.int16))
    assert w1.fc.dtype == torch.bfloat16 and w1.fc.shape == (256, 512)
    assert w1.layers[0].q_norm.dtype == torch.float32
    c = synth.dflash_cache(TINY)
    assert c.k[0].shape == (1, 2, 64 + 5, 64) and int(c.seq_len[0]) == 64
    r = synth.dflash_round_inputs(TINY, [3])
    assert r.block_ids.shape == (1, 5) and int(r.block_ids[0, 1]) == TINY.vocab - 1
    assert r.target_hidden.shape == (1, 3, 512)
