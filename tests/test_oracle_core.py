"""Pins of the oracle's primitives against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each check is a hand-worked value
(tests/golden, each with its citation), a closed form, an invariant, a brute-force
loop on tiny inputs, or an independent library routine.
"""
import itertools
import json
import math
import os
import struct

import numpy as np
import pytest

from oracle import core
from tests.conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- BF16 decode

def test_bf16_canonical_round_trip():
    g = _golden("bf16.json")
    data = b"".join(bytes.fromhex(c["le_bytes"]) for c in g["canonical"])
    got = core.decode_bf16_bytes(data)
    want = np.array([c["value"] for c in g["canonical"]], dtype=np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_bf16_odd_length_rejected():
    g = _golden("bf16.json")
    with pytest.raises(core.OracleError, match="not even"):
        core.decode_bf16_bytes(bytes.fromhex(g["odd_length_bytes"]))


def test_bf16_misread_signature():
    # Reading two BF16 1.0 values as one F32 word gives 0x3f803f80, not 1.0: the
    # dtype-mismatch bug the pages guard against. The oracle's decode must not do that.
    g = _golden("bf16.json")
    two_ones = bytes.fromhex("803f803f")
    misread = struct.unpack("<f", two_ones)[0]
    assert struct.pack(">I", struct.unpack("<I", two_ones)[0]).hex() == g[
        "misread_two_bf16_ones_as_f32_bits"]
    assert misread == g["misread_value"] and misread != 1.0
    assert list(core.decode_bf16_bytes(two_ones)) == [1.0, 1.0]


def test_bf16_all_patterns_match_struct():
    # Every one of the 65536 patterns against Python's own unpacking of the F32 word
    # whose two low bytes are zero and whose two high bytes are the BF16 bytes.
    got = core.decode_bf16(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    for b in range(65536):
        ref = struct.unpack("<f", bytes([0, 0, b & 0xFF, b >> 8]))[0]
        g = float(got[b])
        if math.isnan(ref):
            assert math.isnan(g)
        else:
            assert g == ref and math.copysign(1.0, g) == math.copysign(1.0, ref)


# ---------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("case", _golden("rmsnorm.json")["cases"])
def test_rmsnorm_golden(case):
    y = core.rmsnorm(np.array(case["x"]), np.array(case["w"]), case["eps"], np.float64)
    assert np.allclose(y, case["y"], rtol=1e-12, atol=0)


def test_rmsnorm_scale_invariance_and_unit_rms():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64))
    w = np.ones(64)
    y = core.rmsnorm(x, w, 0.0, np.float64)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-12)
    y2 = core.rmsnorm(7.5 * x, w, 0.0, np.float64)
    assert np.allclose(y, y2, rtol=1e-12)
    # weight multiplies directly (no 1 + w)
    w3 = rng.standard_normal(64)
    assert np.allclose(core.rmsnorm(x, w3, 0.0, np.float64), y * w3, rtol=1e-12)


def test_head_rmsnorm_per_head():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 4 * 8))
    w = rng.standard_normal(8)
    y = core.head_rmsnorm(x, w, 4, 8, 1e-6, np.float64)
    for h in range(4):
        seg = x[:, h * 8:(h + 1) * 8]
        ref = seg / np.sqrt(np.mean(seg ** 2, axis=1, keepdims=True) + 1e-6) * w
        assert np.allclose(y[:, h * 8:(h + 1) * 8], ref, rtol=1e-12)
    # each head separately scale invariant: scaling head 2 only leaves the result unchanged
    x2 = x.copy()
    x2[:, 16:24] *= 3.0
    assert np.allclose(core.head_rmsnorm(x2, w, 4, 8, 0.0, np.float64),
                       core.head_rmsnorm(x, w, 4, 8, 0.0, np.float64), rtol=1e-12)


# ---------------------------------------------------------------- activations

def test_sigmoid_silu_special_values():
    assert core.sigmoid(0.0, np.float64) == 0.5
    assert core.silu(0.0, np.float64) == 0.0
    assert abs(core.silu(30.0, np.float64) - 30.0) < 1e-9
    assert abs(core.silu(-30.0, np.float64)) < 1e-9
    z = 1.3
    assert abs(core.silu(z, np.float64) - z / (1 + math.exp(-z))) < 1e-15


def test_linear_orientation():
    # W is [out, in]: y_o = sum_i W[o, i] x_i. A non-square, non-symmetric W pins the layout.
    W = np.array([[1.0, 2.0, 0.0], [0.0, -1.0, 4.0]], dtype=np.float32)
    bits = (W.view(np.uint32) >> 16).astype(np.uint16)
    x = np.array([1.0, 10.0, 100.0])
    assert np.array_equal(core.linear(x, bits, np.float64), [21.0, 390.0])


def test_swiglu_hand_example():
    # gate = [1, 0], up = [2, 3]: silu(1) * 2, silu(0) * 3 = 0; down = [[1, 1]] -> 2 * silu(1)
    f = lambda a: (np.array(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x = np.array([1.0, 0.0])
    wg = f([[1.0, 0.0], [0.0, 1.0]])
    wu = f([[2.0, 0.0], [3.0, 0.0]])
    wd = f([[1.0, 1.0]])
    want = 2.0 / (1.0 + math.exp(-1.0))
    assert abs(core.swiglu(x, wg, wu, wd, np.float64)[0] - want) < 1e-15


# ---------------------------------------------------------------- RoPE

@pytest.mark.parametrize("case", _golden("rope.json")["cases"])
def test_rope_golden(case):
    g = _golden("rope.json")
    y = core.rope(np.array(case["x"]).reshape(1, 1, 4), [case["pos"]], g["rotary_dim"],
                  g["theta"], np.float64)
    assert np.allclose(y.reshape(-1), case["y"], rtol=0, atol=1e-15)


def test_rope_invariants():
    rng = np.random.default_rng(2)
    d, r, theta = 16, 16, 1e6
    x = rng.standard_normal((1, 3, d))
    for p in (0, 1, 17, 4096, 32775):
        y = core.rope(x, [p], r, theta, np.float64)
        # norm of every rotated pair is preserved
        for i in range(r // 2):
            assert np.allclose(x[..., i] ** 2 + x[..., i + r // 2] ** 2,
                               y[..., i] ** 2 + y[..., i + r // 2] ** 2, rtol=1e-12)
    # R(p) R(q) = R(p + q)
    a = core.rope(core.rope(x, [5], r, theta, np.float64), [11], r, theta, np.float64)
    b = core.rope(x, [16], r, theta, np.float64)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
    # <R(p) q, R(s) k> depends only on p - s
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    dots = [np.sum(core.rope(q, [p], r, theta, np.float64) * core.rope(k, [p - 3], r, theta, np.float64))
            for p in (3, 10, 1000)]
    assert np.allclose(dots, dots[0], rtol=1e-10)


def test_rope_partial_rotary_passes_tail():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 2, 8))
    y = core.rope(x, [3, 9], 4, 1e4, np.float64)
    assert np.array_equal(y[..., 4:], x[..., 4:])
    assert not np.allclose(y[..., :4], x[..., :4])


# ---------------------------------------------------------------- SDPA

@pytest.mark.parametrize("case", _golden("sdpa.json")["cases"])
def test_sdpa_golden(case):
    o = core.sdpa(np.array(case["q"]), np.array(case["k"]), np.array(case["v"]), None, np.float64)
    assert np.allclose(o, case["o"], rtol=1e-14)


def _sdpa_loops(q, k, v, mask=None):
    T, nq, d = q.shape
    S, nkv, _ = k.shape
    rep = nq // nkv
    out = np.zeros((T, nq, d))
    for t in range(T):
        for h in range(nq):
            s = [sum(q[t, h, i] * k[j, h // rep, i] for i in range(d)) / math.sqrt(d) for j in range(S)]
            allowed = [j for j in range(S) if mask is None or mask[t, j]]
            m = max(s[j] for j in allowed)
            e = {j: math.exp(s[j] - m) for j in allowed}
            z = math.fsum(e.values())
            for i in range(d):
                out[t, h, i] = math.fsum(e[j] * v[j, h // rep, i] for j in allowed) / z
    return out


def test_sdpa_brute_force_gqa_and_mask():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((3, 4, 5))
    k = rng.standard_normal((6, 2, 5))
    v = rng.standard_normal((6, 2, 5))
    assert np.allclose(core.sdpa(q, k, v, None, np.float64), _sdpa_loops(q, k, v), rtol=1e-12)
    mask = rng.random((3, 6)) > 0.4
    mask[:, 0] = True
    assert np.allclose(core.sdpa(q, k, v, mask, np.float64), _sdpa_loops(q, k, v, mask), rtol=1e-12)


def test_sdpa_special_cases():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((2, 2, 4))
    k1 = rng.standard_normal((1, 1, 4))
    v1 = rng.standard_normal((1, 1, 4))
    # one key: output is that value row
    assert np.allclose(core.sdpa(q, k1, v1, None, np.float64), np.broadcast_to(v1, (2, 2, 4)))
    # all keys equal: output is the mean of V
    k = np.repeat(k1, 5, axis=0)
    v = rng.standard_normal((5, 1, 4))
    assert np.allclose(core.sdpa(q, k, v, None, np.float64), np.broadcast_to(v.mean(0), (2, 2, 4)))
    # GQA with each KV head repeated equals MHA
    kk = rng.standard_normal((5, 1, 4))
    vv = rng.standard_normal((5, 1, 4))
    a = core.sdpa(q, kk, vv, None, np.float64)
    b = core.sdpa(q, np.repeat(kk, 2, axis=1), np.repeat(vv, 2, axis=1), None, np.float64)
    assert np.allclose(a, b, rtol=1e-14)


# ---------------------------------------------------------------- argmax

def test_argmax_planted_and_ties():
    rng = np.random.default_rng(6)
    L = rng.standard_normal((4, 1000)).astype(np.float32)
    L[0, 777] = 10.0
    L[1, 5] = 9.0
    L[1, 600] = 9.0                    # tie: lowest index wins
    L[2, :] = 0.0                      # all equal: index 0, top2 == top1
    idx, t1, t2 = core.argmax_top2(L)
    assert list(idx[:3]) == [777, 5, 0]
    assert t1[1] == t2[1] == 9.0
    assert t2[2] == t1[2] == 0.0
    for r in range(4):
        best = max(range(1000), key=lambda j: (L[r, j], -j))
        assert idx[r] == best
        assert t2[r] == sorted(L[r])[-2]


def test_lm_head_argmax_chunked_matches_full_scan():
    rng = np.random.default_rng(7)
    W = rng.standard_normal((3000, 16)).astype(np.float32) * 0.02
    bits = (W.view(np.uint32) >> 16).astype(np.uint16)       # truncation: any valid bits
    Wd = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    x = rng.standard_normal((3, 16))
    idx, t1, t2 = core.lm_head_argmax(x, bits, np.float64, chunk=256)
    for r in range(3):
        logits = [math.fsum(Wd[v, j] * x[r, j] for j in range(16)) for v in range(3000)]
        order = sorted(range(3000), key=lambda v: (-logits[v], v))
        assert idx[r] == order[0]
        assert abs(t1[r] - logits[order[0]]) < 1e-12
        assert abs(t2[r] - logits[order[1]]) < 1e-12
    # a tie planted in two different chunks resolves to the lower index
    bits2 = bits.copy()
    one = (np.array([1.0], np.float32).view(np.uint32) >> 16).astype(np.uint16)[0]
    bits2[300, 0] = bits2[2900, 0] = one
    xx = np.zeros((1, 16))
    xx[0, 0] = 50.0
    i2, a, b = core.lm_head_argmax(xx, bits2, np.float64, chunk=256)
    assert i2[0] == 300 and a[0] == b[0] == 50.0


# ---------------------------------------------------------------- accept walk

@pytest.mark.parametrize("case", _golden("accept_walk.json")["cases"])
def test_accept_walk_golden(case):
    c, a, hit, rb = core.accept_walk(case["drafts"], case["target"], case["eos"])
    assert (c, a, hit, rb) == (case["committed"], case["accept"], case["hit_eos"], case["rollback"])


@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("eos", [(), (1,)])
def test_accept_walk_brute_force_invariants(K, eos):
    for drafts in itertools.product(range(3), repeat=K):
        for target in itertools.product(range(3), repeat=K + 1):
            c, a, hit, rb = core.accept_walk(drafts, target, eos)
            # a is the longest prefix on which drafts agree with the target
            assert all(drafts[i] == target[i] for i in range(a))
            assert a == K or drafts[a] != target[a]
            assert rb + a == K
            assert 1 <= len(c) <= K + 1
            full = list(drafts[:a]) + [target[a]]
            if hit:
                assert c[-1] in eos and all(t not in eos for t in c[:-1])
                assert c == full[:len(c)]
            else:
                assert c == full and all(t not in eos for t in c)


def test_accept_walk_requires_k_plus_one_targets():
    with pytest.raises(core.OracleError):
        core.accept_walk([1, 2], [1, 2], ())


@pytest.mark.parametrize("case", _golden("accept_walk.json")["rollback_cases"])
def test_kv_rollback_golden(case):
    if case.get("error"):
        with pytest.raises(core.OracleError):
            core.kv_rollback(case["seq_len"], case["n"])
    else:
        assert core.kv_rollback(case["seq_len"], case["n"]) == case["after"]


def test_round_bf16_hand_values_and_ties_to_even():
    one = 1.0
    assert core.round_bf16([one + 2.0 ** -8])[0] == one                  # halfway, even stays
    assert core.round_bf16([one + 3 * 2.0 ** -8])[0] == one + 2.0 ** -6   # halfway, odd rounds up
    assert core.round_bf16([one + 2.0 ** -8 + 2.0 ** -20])[0] == one + 2.0 ** -7
    assert core.round_bf16([-(one + 3 * 2.0 ** -8)])[0] == -(one + 2.0 ** -6)
    assert core.round_bf16([0.0, -0.0, 3.0])[0] == 0.0


def test_round_bf16_keeps_every_finite_bf16_value_and_matches_integer_rounding():
    from tests.oracle_fixtures import bf16_bits_rne
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = core.decode_bf16(bits)
    finite = np.isfinite(vals)
    assert np.array_equal(core.round_bf16(vals[finite]).view(np.uint32),
                          vals[finite].view(np.uint32))
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 100
    assert np.array_equal(core.round_bf16(x), core.decode_bf16(bf16_bits_rne(x)))
