"""Thin ctypes binding of libdflash.so: same names as the C ABI in include/dflash.h.

Argument marshalling only: torch tensors become device pointers, Python shapes become
the C structs, the current torch CUDA stream becomes the `cudaStream_t`. Every step of
the draft round runs in the library's CUDA kernels. There is no fallback: if the
library is missing, importing a call raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_int32, c_size_t, c_void_p
from typing import List, Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# DFLASH_LIB selects another build of the same library (the debug build, libdflash_debug.so).
LIB_PATH = os.environ.get("DFLASH_LIB") or os.path.join(_PKG, "libdflash.so")

DF_OK, DF_EINVAL, DF_ESHAPE, DF_ECAPACITY, DF_EWORKSPACE, DF_ECUDA, DF_ETIMEOUT = 0, -1, -2, -3, -4, -5, -6
STATUS_NAMES = {0: "DF_OK", -1: "DF_EINVAL", -2: "DF_ESHAPE", -3: "DF_ECAPACITY",
                -4: "DF_EWORKSPACE", -5: "DF_ECUDA", -6: "DF_ETIMEOUT"}


class DFlashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class DFlashConfig(ctypes.Structure):
    _fields_ = [("hidden", c_int32), ("n_layers", c_int32), ("n_q_heads", c_int32),
                ("n_kv_heads", c_int32), ("head_dim", c_int32), ("intermediate", c_int32),
                ("vocab", c_int32), ("n_target_layers", c_int32), ("rotary_dim", c_int32),
                ("mask_token_id", c_int32), ("causal_block", c_int32), ("rms_eps", c_float),
                ("rope_theta", c_float), ("embed_scale", c_float), ("kv_bf16", c_int32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("input_norm", "post_attn_norm", "q_norm", "k_norm", "wq",
                                        "wk", "wv", "wo", "w_gate", "w_up", "w_down")]


class DFlashWeights(ctypes.Structure):
    _fields_ = [("fc", c_void_p), ("hidden_norm", c_void_p), ("final_norm", c_void_p),
                ("layers", POINTER(LayerWeights)), ("embed", c_void_p), ("lm_head", c_void_p),
                ("tiled", c_void_p)]


class SyntheticVerifier(ctypes.Structure):
    _fields_ = [("ref", c_void_p), ("agree", c_void_p), ("table", c_void_p), ("n_comb", c_int32),
                ("sel", c_int32 * 16), ("max_len", c_int32)]


class KvCache(ctypes.Structure):
    _fields_ = [("k", POINTER(c_void_p)), ("v", POINTER(c_void_p)), ("seq_len", c_void_p),
                ("cap", c_int32), ("batch", c_int32), ("n_layers", c_int32)]


class MtpConfig(ctypes.Structure):
    _fields_ = [("hidden", c_int32), ("n_q_heads", c_int32), ("n_kv_heads", c_int32),
                ("head_dim", c_int32), ("vocab", c_int32), ("intermediate", c_int32),
                ("n_experts", c_int32), ("top_k", c_int32), ("expert_inter", c_int32),
                ("shared_inter", c_int32), ("rotary_dim", c_int32), ("rms_eps", c_float),
                ("rope_theta", c_float)]


class MtpWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in (
        "enorm", "hnorm", "eh_embed", "eh_hidden", "attn_norm", "post_attn_norm", "q_norm",
        "k_norm", "wq", "wk", "wv", "w_gate", "wo", "shared_head_norm", "embed", "lm_head",
        "w_gate_mlp", "w_up", "w_down", "router", "exp_gate", "exp_up", "exp_down",
        "sh_gate_mlp", "sh_up", "sh_down", "sh_expert_gate", "tiled")]


_lib = None

# (name, restype, argtypes)
_SIGS = [
    ("df_last_error", ctypes.c_char_p, []),
    ("df_version", c_int, []),
    ("df_kernel_launches", ctypes.c_uint64, []),
    ("df_profile_enable", c_int, [c_int]),
    ("df_profile_read", c_int, [c_void_p, c_int, ctypes.c_char_p, c_size_t]),
    ("df_dflash_workspace_bytes", c_size_t, [POINTER(DFlashConfig), c_int, c_int, c_int]),
    ("dflash_block_forward", c_int, [POINTER(DFlashConfig), POINTER(DFlashWeights), POINTER(KvCache),
                                     c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p,
                                     c_void_p, c_size_t, c_void_p, c_void_p]),
    ("df_lm_head_workspace_bytes", c_size_t, [c_int, c_int, c_int]),
    ("lm_head_argmax", c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p,
                               c_void_p, c_void_p, c_size_t, c_void_p]),
    ("lm_head_argmax_noalloc", c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p,
                                       c_void_p, c_void_p]),
    ("lm_head_argmax_tiled", c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_size_t, c_void_p]),
    ("df_dflash_tiled_bytes", c_size_t, [POINTER(DFlashConfig)]),
    ("df_dflash_tile_weights", c_int, [POINTER(DFlashConfig), POINTER(DFlashWeights), c_void_p,
                                       c_size_t, c_void_p]),
    ("df_tiled_matrix_bytes", c_size_t, [c_int, c_int]),
    ("df_mtp_tiled_bytes", c_size_t, [POINTER(MtpConfig), POINTER(MtpWeights)]),
    ("df_mtp_tile_weights", c_int, [POINTER(MtpConfig), POINTER(MtpWeights), c_void_p, c_size_t,
                                    c_void_p]),
    ("df_tile_matrix", c_int, [c_void_p, c_int, c_int, c_void_p, c_size_t, c_void_p]),
    ("df_linear_workspace_bytes", c_size_t, [c_int, c_int, c_int]),
    ("df_linear", c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_size_t,
                          c_void_p]),
    ("accept_prefix_argmax", c_int, [c_void_p, c_int, c_void_p, c_int, c_int, c_void_p, c_int,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    ("accept_prefix_argmax_host", c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_void_p,
                                          c_void_p, c_void_p, c_void_p, c_void_p]),
    ("kv_rollback", c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p]),
    ("df_draft_round", c_int, [POINTER(DFlashConfig), POINTER(DFlashWeights), POINTER(KvCache),
                               c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p,
                               c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                               c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
    ("df_draft_round_host_workspace_bytes", c_size_t, [POINTER(DFlashConfig), c_int, c_int, c_int,
                                                       c_int]),
    ("df_draft_round_host", c_int, [POINTER(DFlashConfig), POINTER(DFlashWeights),
                                    POINTER(KvCache), c_void_p, c_void_p, c_void_p, c_int, c_int,
                                    c_int, c_void_p, c_void_p, c_int, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_size_t, c_void_p]),
    ("df_mtp_workspace_bytes", c_size_t, [POINTER(MtpConfig), c_int]),
    ("mtp_forward_draft", c_int, [POINTER(MtpConfig), POINTER(MtpWeights), POINTER(KvCache),
                                  c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_size_t, c_void_p, c_void_p]),
    ("df_accept_stochastic_workspace_bytes", c_size_t, [c_int, c_int, c_int]),
    ("df_generate_workspace_bytes", c_size_t, [POINTER(DFlashConfig), c_int, c_int, c_int]),
    ("df_generate", c_int, [POINTER(DFlashConfig), POINTER(DFlashWeights), POINTER(KvCache),
                            POINTER(SyntheticVerifier), c_void_p, c_void_p, c_void_p, c_void_p,
                            c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p, c_int,
                            c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
    ("accept_stochastic", c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, c_float,
                                  c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p,
                                  c_void_p]),
    ("df_test_wait_hook", c_int, [ctypes.c_longlong, c_int]),
    ("df_trace_reset", c_int, []),
    ("df_trace_read", c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int]),
    ("df_sample_softmax_workspace_bytes", c_size_t, [c_int, c_int]),
    ("sample_softmax", c_int, [c_void_p, c_int, c_int, c_float, c_void_p, c_void_p, c_void_p,
                               c_size_t, c_void_p, c_void_p]),
    ("df_draft_round_stochastic_workspace_bytes", c_size_t, [POINTER(DFlashConfig), c_int, c_int,
                                                             c_int]),
    ("df_draft_round_stochastic", c_int, [POINTER(DFlashConfig), POINTER(DFlashWeights),
                                          POINTER(KvCache), c_void_p, c_void_p, c_void_p, c_int,
                                          c_int, c_int, c_void_p, c_float, c_void_p, c_void_p,
                                          c_void_p, c_void_p, c_int, c_void_p, c_void_p,
                                          c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                          c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
    ("mtp_forward_draft_sampled", c_int, [POINTER(MtpConfig), POINTER(MtpWeights),
                                          POINTER(KvCache), c_void_p, c_void_p, c_int, c_int,
                                          c_float, c_void_p, c_void_p, c_void_p, c_void_p,
                                          c_void_p, c_size_t, c_void_p, c_void_p]),
    ("df_attention_workspace_bytes", c_size_t, [c_int] * 6),
    ("df_attention", c_int, [c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p,
                             c_int, c_int, c_int, c_int, c_int, c_int, c_void_p, c_void_p,
                             c_size_t, c_void_p, c_void_p]),
    ("df_moe_workspace_bytes", c_size_t, [POINTER(MtpConfig), c_int]),
    ("df_moe_ffn", c_int, [POINTER(MtpConfig), POINTER(MtpWeights), c_void_p, c_int, c_void_p,
                           c_void_p, c_void_p, c_void_p, c_size_t, c_void_p, c_void_p]),
]


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m speculative_decoding_drafter_dflash_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in _SIGS:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def kernel_launches() -> int:
    return int(lib().df_kernel_launches())


def profile_enable(on: bool = True):
    _check(lib().df_profile_enable(1 if on else 0))


def profile_read(max_entries: int = 8192):
    """[(kernel name, microseconds)] of the launches recorded since profile_enable(True)."""
    us = (ctypes.c_float * max_entries)()
    buf = ctypes.create_string_buffer(64 * max_entries)
    n = lib().df_profile_read(us, max_entries, buf, len(buf))
    if n < 0:
        _check(n)
    names = buf.value.decode().split("\n")
    return [(names[i], float(us[i])) for i in range(n)]


def last_error() -> str:
    return lib().df_last_error().decode()


def _check(rc: int):
    if rc != DF_OK:
        raise DFlashError(rc, last_error())


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t: Optional[torch.Tensor], dtype, name: str):
    """Pointer of a contiguous CUDA tensor of `dtype` (None passes through). A tensor of another
    type, layout or device raises here rather than reaching a kernel that would read it with the
    wrong element size."""
    if t is None:
        return None
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA {dtype} tensor, got {t.dtype} on "
                        f"{t.device}" + ("" if t.is_contiguous() else " (not contiguous)"))
    return ctypes.c_void_p(t.data_ptr())


F32, I32, BF16 = torch.float32, torch.int32, torch.bfloat16


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


# ----------------------------------------------------------------------------- structs
class DFlashModel:
    """C structs for a DFlash drafter: config, weight pointers, KV cache. Keeps the tensors
    and ctypes arrays alive for the lifetime of the object."""

    def __init__(self, shape, weights, cache, embed_scale: float = 1.0, tiled: bool = True):
        """tiled: also lay the projection and lm_head weights out as tiles
        (df_dflash_tile_weights) and let the kernels read those; False reads the row-major
        matrices."""
        self.shape = shape
        self.cfg = DFlashConfig(shape.hidden, shape.n_layers, shape.n_q_heads, shape.n_kv_heads,
                                shape.head_dim, shape.intermediate, shape.vocab,
                                shape.n_target_layers, shape.rotary_dim, shape.mask_id,
                                shape.causal_block, shape.rms_eps, shape.rope_theta, embed_scale,
                                1 if getattr(shape, "kv_bf16", False) else 0)
        L = len(weights.layers)
        self._layers = (LayerWeights * L)()
        for i, lw in enumerate(weights.layers):
            self._layers[i] = LayerWeights(*(t.data_ptr() for t in (
                lw.input_norm, lw.post_norm, lw.q_norm, lw.k_norm, lw.wq, lw.wk, lw.wv, lw.wo,
                lw.wg, lw.wu, lw.wd)))
        self.weights = DFlashWeights(weights.fc.data_ptr(), weights.hidden_norm.data_ptr(),
                                     weights.final_norm.data_ptr(), self._layers,
                                     weights.embed.data_ptr(), weights.lm_head.data_ptr(), None)
        self._w = weights
        self._tiled = None
        if tiled:
            n = int(lib().df_dflash_tiled_bytes(ctypes.byref(self.cfg)))
            if n == 0:   # an invalid config: the tiling call reports why, with its code
                _check(lib().df_dflash_tile_weights(ctypes.byref(self.cfg),
                                                    ctypes.byref(self.weights), None, 0,
                                                    _stream(None)))
                _check(DF_EINVAL)
            buf, ptr = _aligned_buffer(n, weights.fc.device)
            _check(lib().df_dflash_tile_weights(ctypes.byref(self.cfg), ctypes.byref(self.weights),
                                                ptr, n, _stream(None)))
            torch.cuda.synchronize(weights.fc.device)
            self.weights.tiled = ptr
            self._tiled = buf
        self.set_cache(cache)

    def set_cache(self, cache):
        L = len(cache.k)
        want = BF16 if self.cfg.kv_bf16 else F32
        for i in range(L):
            _dev(cache.k[i], want, f"cache.k[{i}]")
            _dev(cache.v[i], want, f"cache.v[{i}]")
        _dev(cache.seq_len, I32, "cache.seq_len")
        self._k = (c_void_p * L)(*[t.data_ptr() for t in cache.k])
        self._v = (c_void_p * L)(*[t.data_ptr() for t in cache.v])
        self.cache_c = KvCache(self._k, self._v, cache.seq_len.data_ptr(), cache.cap,
                               cache.seq_len.shape[0], L)
        self._cache = cache

    def workspace_bytes(self, B: int, block: int, n_new_max: int) -> int:
        return int(lib().df_dflash_workspace_bytes(ctypes.byref(self.cfg), B, block, n_new_max))


def _aligned_buffer(nbytes: int, device, align: int = 1024):
    """A device byte buffer and the first `align`-aligned address in it with nbytes behind it."""
    buf = torch.empty(int(nbytes) + align, dtype=torch.uint8, device=device)
    ptr = (buf.data_ptr() + align - 1) // align * align
    return buf, ptr


class TiledMatrix:
    """The tiled copy of one BF16 [N, K] matrix (df_tile_matrix), e.g. an lm_head."""

    def __init__(self, W, stream=None):
        N, K = W.shape
        n = int(lib().df_tiled_matrix_bytes(N, K))
        self.buf, self.ptr = _aligned_buffer(n, W.device)
        self.N, self.K, self.nbytes = N, K, n
        _check(lib().df_tile_matrix(_dev(W, BF16, "W"), N, K, self.ptr, n, _stream(stream)))
        # complete before any projection reads it (projections prefetch weights ahead of their
        # predecessor kernels)
        torch.cuda.synchronize(W.device)

    def bytes_view(self) -> torch.Tensor:
        off = self.ptr - self.buf.data_ptr()
        return self.buf[off:off + self.nbytes]


def lm_head_argmax_tiled(Wt: TiledMatrix, X, idx, top1=None, top2=None, ws=None, stream=None):
    rows, H = X.shape
    if H != Wt.K:
        raise ValueError(f"X has {H} columns, the tiled matrix {Wt.K}")
    _check(lib().lm_head_argmax_tiled(Wt.ptr, _dev(X, F32, "X"), rows, H, Wt.N,
                                      _dev(idx, I32, "idx"), _dev(top1, F32, "top1"),
                                      _dev(top2, F32, "top2"), _p(ws),
                                      ws.numel() if ws is not None else 0, _stream(stream)))


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zeroed device workspace, 256-byte aligned (the caching allocator aligns to 512)."""
    t = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    assert t.data_ptr() % 256 == 0
    return t


# ----------------------------------------------------------------------------- calls
def dflash_block_forward(model: DFlashModel, block_ids, target_hidden_new, n_new, n_new_max: int,
                         h_final, ws, d_status=None, stream=None):
    B, block = block_ids.shape
    _check(lib().dflash_block_forward(ctypes.byref(model.cfg), ctypes.byref(model.weights),
                                      ctypes.byref(model.cache_c), _p(block_ids),
                                      _p(target_hidden_new), _p(n_new), n_new_max, B, block,
                                      _p(h_final), _p(ws), ws.numel(), _p(d_status),
                                      _stream(stream)))


def lm_head_workspace_bytes(rows: int, H: int, V: int) -> int:
    return int(lib().df_lm_head_workspace_bytes(rows, H, V))


def lm_head_argmax(W, X, idx, top1=None, top2=None, ws=None, stream=None):
    rows, H = X.shape
    V = W.shape[0]
    _check(lib().lm_head_argmax(_dev(W, BF16, "W"), _dev(X, F32, "X"), rows, H, V,
                                _dev(idx, I32, "idx"), _dev(top1, F32, "top1"),
                                _dev(top2, F32, "top2"), _p(ws),
                                ws.numel() if ws is not None else 0, _stream(stream)))


def linear_workspace_bytes(T: int, N: int, K: int) -> int:
    return int(lib().df_linear_workspace_bytes(T, N, K))


def df_linear(W, X, Y, ws, stream=None):
    T, K = X.shape
    N = W.shape[0]
    _check(lib().df_linear(_dev(W, BF16, "W"), _dev(X, F32, "X"), T, N, K, _dev(Y, F32, "Y"),
                           _p(ws), ws.numel(), _stream(stream)))


def lm_head_argmax_noalloc(W, X, idx, top1=None, top2=None, stream=None):
    """lm_head_argmax without a workspace (fixed scratch inside the library; see dflash.h)."""
    rows, H = X.shape
    V = W.shape[0]
    _check(lib().lm_head_argmax_noalloc(_dev(W, BF16, "W"), _dev(X, F32, "X"), rows, H, V,
                                        _dev(idx, I32, "idx"), _dev(top1, F32, "top1"),
                                        _dev(top2, F32, "top2"), _stream(stream)))


def accept_prefix_argmax(drafts, drafts_ld: int, target, K: int, eos, committed, n_committed,
                         accept_count, hit_eos, rollback, stream=None):
    B = target.shape[0]
    n_eos = 0 if eos is None else eos.numel()
    _check(lib().accept_prefix_argmax(_p(drafts), drafts_ld, _p(target), B, K, _p(eos), n_eos,
                                      _p(committed), _p(n_committed), _p(accept_count),
                                      _p(hit_eos), _p(rollback), _stream(stream)))


def accept_prefix_argmax_host(drafts: Sequence[int], target: Sequence[int], eos: Sequence[int]):
    """Host walk of one sequence; returns (committed list, accept_count, hit_eos, rollback)."""
    K = len(drafts)
    D = (c_int32 * max(K, 1))(*drafts)
    T = (c_int32 * (K + 1))(*target)
    E = (c_int32 * max(len(eos), 1))(*eos)
    C = (c_int32 * (K + 1))()
    nc, ac, he, rb = c_int32(), c_int32(), c_int32(), c_int32()
    _check(lib().accept_prefix_argmax_host(D, T, K, E if eos else None, len(eos), C,
                                           ctypes.byref(nc), ctypes.byref(ac), ctypes.byref(he),
                                           ctypes.byref(rb)))
    return list(C[:nc.value]), ac.value, he.value, rb.value


def kv_rollback(seq_len, n, d_status=None, stream=None):
    _check(lib().kv_rollback(_p(seq_len), _p(n), seq_len.shape[0], _p(d_status), _stream(stream)))


class RoundOutputs:
    """Device outputs of one draft round for B sequences and K drafts."""

    def __init__(self, B: int, K: int, device="cuda"):
        i32 = dict(dtype=torch.int32, device=device)
        self.argmax = torch.zeros((B, K + 1), **i32)
        self.committed = torch.zeros((B, K + 1), **i32)
        self.n_committed = torch.zeros(B, **i32)
        self.accept = torch.zeros(B, **i32)
        self.hit_eos = torch.zeros(B, **i32)
        self.rollback = torch.zeros(B, **i32)


def df_draft_round(model: DFlashModel, last_token, target_hidden_new, n_new, n_new_max: int, K: int,
                   target_argmax, eos, target_seq_len, out: RoundOutputs, ws, d_status=None,
                   stream=None):
    B = last_token.shape[0]
    n_eos = 0 if eos is None else eos.numel()
    _check(lib().df_draft_round(ctypes.byref(model.cfg), ctypes.byref(model.weights),
                                ctypes.byref(model.cache_c), _p(last_token), _p(target_hidden_new),
                                _p(n_new), n_new_max, B, K, _p(target_argmax), _p(eos), n_eos,
                                _p(target_seq_len), _p(out.argmax), _p(out.committed),
                                _p(out.n_committed), _p(out.accept), _p(out.hit_eos),
                                _p(out.rollback), _p(ws), ws.numel(), _p(d_status),
                                _stream(stream)))


def draft_round_host_workspace_bytes(model: DFlashModel, B: int, K: int, n_new_max: int,
                                     n_eos: int) -> int:
    return int(model.workspace_bytes(B, K + 1, n_new_max)
               + lib().df_draft_round_host_workspace_bytes(ctypes.byref(model.cfg), B, K,
                                                           n_new_max, n_eos))


def df_draft_round_host(model: DFlashModel, last_token, target_hidden_new, n_new, n_new_max: int,
                        K: int, target_argmax, eos, target_seq_len, host_out: dict, ws,
                        stream=None):
    """All tensor arguments are (pinned) HOST tensors; host_out holds host int32 tensors
    argmax/committed [B, K+1], n_committed/accept/hit_eos/rollback [B], status [1]."""
    B = last_token.shape[0]
    n_eos = 0 if eos is None else eos.numel()
    _check(lib().df_draft_round_host(
        ctypes.byref(model.cfg), ctypes.byref(model.weights), ctypes.byref(model.cache_c),
        _p(last_token), _p(target_hidden_new), _p(n_new), n_new_max, B, K, _p(target_argmax),
        _p(eos), n_eos, _p(target_seq_len), _p(host_out["argmax"]), _p(host_out["committed"]),
        _p(host_out["n_committed"]), _p(host_out["accept"]), _p(host_out["hit_eos"]),
        _p(host_out["rollback"]), _p(host_out["status"]), _p(ws), ws.numel(), _stream(stream)))


class MtpModel:
    """C structs of an MTP block: config + weight pointers + the one-layer KV slot."""

    def __init__(self, shape, w, cache, tiled: bool = True):
        """tiled: also lay the projection and lm_head weights out as tiles
        (df_mtp_tile_weights) and let the kernels read those."""
        self.shape = shape
        self.cfg = MtpConfig(shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                             shape.vocab, shape.intermediate, shape.n_experts, shape.top_k,
                             shape.expert_inter, shape.shared_inter, shape.rotary_dim,
                             shape.rms_eps, shape.rope_theta)
        ptr = lambda t: None if t is None else t.data_ptr()
        self.weights = MtpWeights(*[ptr(getattr(w, n)) for n in (
            "enorm", "hnorm", "eh_embed", "eh_hidden", "attn_norm", "post_norm", "q_norm",
            "k_norm", "wq", "wk", "wv", "w_gate", "wo", "shared_head_norm", "embed", "lm_head",
            "wg", "wu", "wd", "router", "exp_g", "exp_u", "exp_d", "sh_g", "sh_u", "sh_d",
            "sh_gate")], None)
        self._w = w
        self._tiled = None
        if tiled:
            n = int(lib().df_mtp_tiled_bytes(ctypes.byref(self.cfg), ctypes.byref(self.weights)))
            if n == 0:   # invalid config or weights: the tiling call reports why
                _check(lib().df_mtp_tile_weights(ctypes.byref(self.cfg),
                                                 ctypes.byref(self.weights), None, 0,
                                                 _stream(None)))
                _check(DF_EINVAL)
            buf, p_ = _aligned_buffer(n, w.lm_head.device)
            _check(lib().df_mtp_tile_weights(ctypes.byref(self.cfg), ctypes.byref(self.weights),
                                             p_, n, _stream(None)))
            torch.cuda.synchronize(w.lm_head.device)
            self.weights.tiled = p_
            self._tiled = buf
        self._k = (c_void_p * 1)(cache.k[0].data_ptr())
        self._v = (c_void_p * 1)(cache.v[0].data_ptr())
        self.cache_c = KvCache(self._k, self._v, cache.seq_len.data_ptr(), cache.cap,
                               cache.seq_len.shape[0], 1)
        self._cache = cache

    def workspace_bytes(self, B: int) -> int:
        return int(lib().df_mtp_workspace_bytes(ctypes.byref(self.cfg), B))

    def moe_workspace_bytes(self, T: int) -> int:
        return int(lib().df_moe_workspace_bytes(ctypes.byref(self.cfg), T))


def mtp_forward_draft(model: MtpModel, prev_hidden, token, n_steps: int, hidden_out, argmax_out,
                      ws, logits_out=None, d_status=None, stream=None):
    B = token.shape[0]
    _check(lib().mtp_forward_draft(ctypes.byref(model.cfg), ctypes.byref(model.weights),
                                   ctypes.byref(model.cache_c), _p(prev_hidden), _p(token), B,
                                   n_steps, _p(hidden_out), _p(argmax_out), _p(logits_out), _p(ws),
                                   ws.numel(), _p(d_status), _stream(stream)))


def mtp_forward_draft_sampled(model: MtpModel, prev_hidden, token, n_steps: int,
                              temperature: float, u_draft, hidden_out, draft_out, logits_out, ws,
                              d_status=None, stream=None):
    """The sampled MTP chain: u_draft [n_steps, B]; draft_out [n_steps, B] int32 and
    logits_out [n_steps, B, V] are outputs."""
    B = token.shape[0]
    _check(lib().mtp_forward_draft_sampled(
        ctypes.byref(model.cfg), ctypes.byref(model.weights), ctypes.byref(model.cache_c),
        _dev(prev_hidden, F32, "prev_hidden"), _dev(token, I32, "token"), B, n_steps,
        float(temperature), _dev(u_draft, F32, "u_draft"), _dev(hidden_out, F32, "hidden_out"),
        _dev(draft_out, I32, "draft_out"), _dev(logits_out, F32, "logits_out"), _p(ws),
        ws.numel(), _p(d_status), _stream(stream)))


def moe_ffn(model: MtpModel, x, out, ws, expert_ids=None, expert_w=None, d_status=None,
            stream=None):
    """The MoE FFN alone: out[T, H] from normalised rows x[T, H]; optional expert_ids
    [T, top_k] int32 and expert_w [T, top_k + 1] F32 outputs."""
    T = x.shape[0]
    _check(lib().df_moe_ffn(ctypes.byref(model.cfg), ctypes.byref(model.weights), _p(x), T,
                            _p(out), _p(expert_ids), _p(expert_w), _p(ws), ws.numel(),
                            _p(d_status), _stream(stream)))


def attention_workspace_bytes(B: int, blk: int, nq: int, nkv: int, d: int, cap: int) -> int:
    return int(lib().df_attention_workspace_bytes(B, blk, nq, nkv, d, cap))


def attention(q, cache_k, cache_v, seq_len, out, ws, kb=None, vb=None, causal_block=False,
              d_status=None, stream=None):
    """q [B, blk, nq, d]; cache_k/v [B, nkv, cap, d]; optional block keys kb/vb [B, nkv, blk, d];
    out [B, blk, nq, d]."""
    Bn, blk, nq, d = q.shape
    nkv, cap = cache_k.shape[1], cache_k.shape[2]
    _check(lib().df_attention(_dev(q, F32, "q"), _dev(cache_k, F32, "cache_k"),
                              _dev(cache_v, F32, "cache_v"), cap, _dev(seq_len, I32, "seq_len"),
                              _dev(kb, F32, "kb"), _dev(vb, F32, "vb"),
                              Bn, blk, nq, nkv, d, 1 if causal_block else 0,
                              _dev(out, F32, "out"), _p(ws),
                              ws.numel(), _p(d_status), _stream(stream)))


def accept_stochastic_workspace_bytes(B: int, K: int, V: int) -> int:
    return int(lib().df_accept_stochastic_workspace_bytes(B, K, V))


def accept_stochastic(draft_logits, target_logits, drafts, temperature: float, u_accept,
                      u_sample, eos, out: dict, ws, d_status=None, stream=None):
    """draft_logits [B, K, V], target_logits [B, K+1, V], drafts [B, K] int32, u_accept [B, K],
    u_sample [B]; out holds device int32 committed [B, K+1] and n_committed / accept /
    hit_eos / rollback [B]."""
    B, K, V = draft_logits.shape
    n_eos = 0 if eos is None else eos.numel()
    _check(lib().accept_stochastic(_p(draft_logits), _p(target_logits), V, _p(drafts), B, K,
                                   float(temperature), _p(u_accept), _p(u_sample), _p(eos), n_eos,
                                   _p(out["committed"]), _p(out["n_committed"]), _p(out["accept"]),
                                   _p(out["hit_eos"]), _p(out["rollback"]), _p(ws), ws.numel(),
                                   _p(d_status), _stream(stream)))


def trace_reset():
    _check(lib().df_trace_reset())


def trace_read(max_records: int = 1 << 20):
    """[(kernel id, SM, start ns, end ns)] of the CTAs recorded since trace_reset() (trace
    builds only)."""
    import numpy as np
    kid = np.zeros(max_records, np.uint32)
    sm = np.zeros(max_records, np.uint32)
    t0 = np.zeros(max_records, np.uint64)
    t1 = np.zeros(max_records, np.uint64)
    n = lib().df_trace_read(kid.ctypes.data, sm.ctypes.data, t0.ctypes.data, t1.ctypes.data,
                            max_records)
    if n < 0:
        _check(n)
    return kid[:n], sm[:n], t0[:n], t1[:n]


def test_wait_hook(wait_cycles: int, withhold_first: bool):
    """Failure-detection test hook of the projection kernel (see include/dflash.h)."""
    _check(lib().df_test_wait_hook(int(wait_cycles), 1 if withhold_first else 0))


def sample_softmax_workspace_bytes(R: int, V: int) -> int:
    return int(lib().df_sample_softmax_workspace_bytes(R, V))


def sample_softmax(logits, temperature: float, u, tokens, ws, d_status=None, stream=None):
    """logits [R, V] F32, u [R] F32 uniforms; tokens [R] int32 out: one draw per row from
    softmax(logits / T)."""
    R, V = logits.shape
    _check(lib().sample_softmax(_dev(logits, F32, "logits"), R, V, float(temperature),
                                _dev(u, F32, "u"), _dev(tokens, I32, "tokens"), _p(ws), ws.numel(),
                                _p(d_status), _stream(stream)))


def draft_round_stochastic_workspace_bytes(model: "DFlashModel", B: int, K: int,
                                           n_new_max: int) -> int:
    return int(lib().df_draft_round_stochastic_workspace_bytes(ctypes.byref(model.cfg), B, K,
                                                               n_new_max))


def df_draft_round_stochastic(model: "DFlashModel", last_token, target_hidden_new, n_new,
                              n_new_max: int, K: int, target_logits, temperature: float, u_draft,
                              u_accept, u_sample, eos, target_seq_len, logits_out, drafts_out,
                              out: "RoundOutputs", ws, d_status=None, stream=None):
    """The non-greedy round: target_logits [B, K+1, V]; u_draft, u_accept [B, K]; u_sample [B];
    logits_out [B, K+1, V] and drafts_out [B, K] are outputs, as are out.committed etc.
    (out.argmax is not written)."""
    B = last_token.shape[0]
    n_eos = 0 if eos is None else eos.numel()
    _check(lib().df_draft_round_stochastic(
        ctypes.byref(model.cfg), ctypes.byref(model.weights), ctypes.byref(model.cache_c),
        _dev(last_token, I32, "last_token"), _dev(target_hidden_new, F32, "target_hidden_new"),
        _dev(n_new, I32, "n_new"), n_new_max, B, K, _dev(target_logits, F32, "target_logits"),
        float(temperature), _dev(u_draft, F32, "u_draft"), _dev(u_accept, F32, "u_accept"),
        _dev(u_sample, F32, "u_sample"), _dev(eos, I32, "eos"), n_eos,
        _dev(target_seq_len, I32, "target_seq_len"), _dev(logits_out, F32, "logits_out"),
        _dev(drafts_out, I32, "drafts_out"), _p(out.committed), _p(out.n_committed),
        _p(out.accept), _p(out.hit_eos), _p(out.rollback), _p(ws), ws.numel(), _p(d_status),
        _stream(stream)))


def generate_workspace_bytes(model: "DFlashModel", B: int, K: int, n_new_max: int) -> int:
    return int(lib().df_generate_workspace_bytes(ctypes.byref(model.cfg), B, K, n_new_max))


def generate(model: "DFlashModel", ref, agree, table, sel, prior_cap, prior_len, out_tokens,
             out_len, prompt_len, max_new_tokens: int, max_rounds: int, K: int, n_new_max: int,
             eos, rounds, ws, accept_hist=None, d_status=None, stream=None):
    """The device generate loop (see include/dflash.h, df_generate). ref/agree [B, max_len],
    table [B, n_comb, max_len, H], sel: list of capture-layer indices of the drafter's target
    layers; the state tensors are device tensors updated in place."""
    B, max_len = ref.shape
    v = SyntheticVerifier()
    v.ref = ref.data_ptr()
    v.agree = None if agree is None else agree.data_ptr()
    v.table = table.data_ptr()
    v.n_comb = table.shape[1]
    for i, c in enumerate(sel):
        v.sel[i] = int(c)
    v.max_len = max_len
    n_eos = 0 if eos is None else eos.numel()
    _check(lib().df_generate(ctypes.byref(model.cfg), ctypes.byref(model.weights),
                             ctypes.byref(model.cache_c), ctypes.byref(v), _p(prior_cap),
                             _p(prior_len), _p(out_tokens), _p(out_len), _p(prompt_len),
                             max_new_tokens, max_rounds, B, K, n_new_max, _p(eos), n_eos,
                             _p(rounds), _p(accept_hist), _p(ws), ws.numel(), _p(d_status),
                             _stream(stream)))
