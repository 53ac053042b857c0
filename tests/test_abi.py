"""The C ABI without a GPU: the library loads, exports every function include/dflash.h
declares, validates arguments on the host, and its host accept walk matches the oracle."""
import ctypes
import itertools
import os
import re

import pytest

from oracle import core
from tests.conftest import ROOT


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_drafter_dflash_gb300 import build, binding
    build.build()
    return binding


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "dflash.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char|void|uint64_t)\s*\*?\s*(\w+)\s*\(", src, re.M)
    return sorted(set(names))


def test_header_declares_the_round(L):
    names = _declared_functions()
    for must in ("dflash_block_forward", "lm_head_argmax", "accept_prefix_argmax",
                 "accept_prefix_argmax_host", "kv_rollback", "mtp_forward_draft",
                 "df_draft_round", "df_draft_round_host", "df_last_error"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    lib = L.lib()
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert lib.df_version() >= 100


def test_host_accept_walk_matches_oracle_brute_force(L):
    for K in (1, 2, 3, 4):
        for eos in ((), (1,)):
            for drafts in itertools.product(range(3), repeat=K):
                for target in itertools.product(range(3), repeat=K + 1):
                    got = L.accept_prefix_argmax_host(list(drafts), list(target), list(eos))
                    want = core.accept_walk(drafts, target, eos)
                    assert got == want, (drafts, target, eos)


def test_host_validation_errors(L):
    from speculative_decoding_drafter_dflash_gb300.workloads import TINY
    lib = L.lib()
    cfg = L.DFlashConfig(TINY.hidden, TINY.n_layers, TINY.n_q_heads, TINY.n_kv_heads,
                         TINY.head_dim, TINY.intermediate, TINY.vocab, TINY.n_target_layers, 0,
                         TINY.mask_id, 0, 1e-6, 1e6, 1.0)
    assert lib.df_dflash_workspace_bytes(ctypes.byref(cfg), 1, 5, 4) > 0
    bad = L.DFlashConfig.from_buffer_copy(cfg)
    bad.head_dim = 48                                    # not a multiple of 32
    assert lib.df_dflash_workspace_bytes(ctypes.byref(bad), 1, 5, 4) == 0
    assert lib.df_dflash_workspace_bytes(ctypes.byref(cfg), 1, 1, 4) == 0   # block < 2
    # NULL config / weights: rejected before any CUDA call
    rc = lib.dflash_block_forward(None, None, None, None, None, None, 0, 1, 5, None, None, 0,
                                  None, None)
    assert rc == L.DF_EINVAL and "config" in L.last_error()
    rc = lib.dflash_block_forward(ctypes.byref(bad), None, None, None, None, None, 0, 1, 5, None,
                                  None, 0, None, None)
    assert rc == L.DF_ESHAPE and "head_dim" in L.last_error()
    rc = lib.dflash_block_forward(ctypes.byref(cfg), None, None, None, None, None, 0, 1, 5, None,
                                  None, 0, None, None)
    assert rc == L.DF_EINVAL and "weights" in L.last_error()
    # lm_head: misaligned H and missing workspace
    assert lib.lm_head_argmax(None, None, 4, 12, 100, None, None, None, None, 0, None) == L.DF_ESHAPE
    assert lib.kv_rollback(None, None, 0, None, None) == L.DF_ESHAPE
    assert lib.accept_prefix_argmax(None, 0, None, 1, 0, None, 0, None, None, None, None, None,
                                    None) == L.DF_ESHAPE
    with pytest.raises(L.DFlashError):
        L.accept_prefix_argmax_host([], [1], [])


def test_workspace_queries_scale(L):
    from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15
    lib = L.lib()
    s = DFLASH_K15
    cfg = L.DFlashConfig(s.hidden, s.n_layers, s.n_q_heads, s.n_kv_heads, s.head_dim,
                         s.intermediate, s.vocab, s.n_target_layers, 0, s.mask_id, 0, 1e-6, 1e6, 1.0)
    w1 = lib.df_dflash_workspace_bytes(ctypes.byref(cfg), 1, 16, 16)
    w8 = lib.df_dflash_workspace_bytes(ctypes.byref(cfg), 8, 16, 16)
    assert 0 < w1 < w8 < 1 << 31
    assert lib.df_lm_head_workspace_bytes(16, 2816, 262144) > 2 * 16 * 2816 * 2


def test_binding_rejects_tensors_of_the_wrong_type_or_device(L):
    # The element size a kernel reads with comes from the entry point, not from the tensor: a
    # host tensor, or one of another dtype (a BF16 cache handed to the F32 attention), must stop
    # in the binding. Without a GPU every tensor is a host tensor: the first argument is named.
    import torch
    f32 = torch.zeros((1, 2, 2, 128))
    with pytest.raises(TypeError, match="^q: expected a contiguous CUDA"):
        L.attention(f32, f32.to(torch.bfloat16), f32, torch.zeros(1, dtype=torch.int32), f32,
                    torch.zeros(256, dtype=torch.uint8))
    with pytest.raises(TypeError, match="^W: expected a contiguous CUDA torch.bfloat16"):
        L.df_linear(torch.zeros((4, 8)), torch.zeros((2, 8)), torch.zeros((2, 4)),
                    torch.zeros(256, dtype=torch.uint8))
