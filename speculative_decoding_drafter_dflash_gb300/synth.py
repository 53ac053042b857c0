"""Seeded synthetic inputs for a draft round (weights, KV cache, activations, targets).

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic. The same tensors feed the CUDA path and, copied to the
host, the CPU oracle. Draws come from one `torch.Generator` per call, on the
device the tensors are wanted on (Philox on CUDA, Mersenne Twister on CPU), so a
full-size workload of ~3 GB of weights is generated in milliseconds on the GPU.

Distributions (all seeded):
  * BF16 projection weights, embedding and lm_head tables: N(0, w_std) rounded
    to BF16 by round-to-nearest-even (torch's float->bfloat16 cast);
  * RMSNorm weights (F32): 1 + N(0, norm_std);
  * activations, target hidden rows and pre-filled KV rows (F32): N(0, 1);
  * router weights of an MoE block: N(0, 1/sqrt(H)), so router logits are ~N(0, 1);
  * last_token ~ U[2, V-1); target argmaxes agree with the drafts on a prefix whose
    length is geometric, P(a >= j) = p**j capped at K (or U{0..K} when p is None).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

from .workloads import DFlashShape, MtpShape


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(g, shape, std, device, dtype=torch.float32):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def bf16_to_u16(t: torch.Tensor) -> np.ndarray:
    """Host copy of a bfloat16 tensor's raw bit patterns (uint16)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy of a tensor (bf16 tensors come back as uint16 bit patterns)."""
    if t.dtype == torch.bfloat16:
        return bf16_to_u16(t)
    return t.detach().contiguous().cpu().numpy()


@dataclass
class LayerW:
    input_norm: torch.Tensor
    post_norm: torch.Tensor
    q_norm: torch.Tensor
    k_norm: torch.Tensor
    wq: torch.Tensor
    wk: torch.Tensor
    wv: torch.Tensor
    wo: torch.Tensor
    wg: torch.Tensor
    wu: torch.Tensor
    wd: torch.Tensor


@dataclass
class DFlashWeights:
    fc: torch.Tensor
    hidden_norm: torch.Tensor
    final_norm: torch.Tensor
    layers: List[LayerW]
    embed: torch.Tensor
    lm_head: torch.Tensor


@dataclass
class KvCache:
    k: List[torch.Tensor]        # per layer [B, n_kv, cap, d] F32
    v: List[torch.Tensor]
    seq_len: torch.Tensor        # [B] int32
    cap: int


@dataclass
class DFlashRoundInputs:
    last_token: torch.Tensor     # [B] int32
    block_ids: torch.Tensor      # [B, K+1] int32
    target_hidden: torch.Tensor  # [B, n_new_max, n_tl*H] F32
    n_new: torch.Tensor          # [B] int32
    n_new_max: int


def dflash_weights(s: DFlashShape, seed: int = 0, device="cpu") -> DFlashWeights:
    g = _gen(seed, device)
    H, I, bf = s.hidden, s.intermediate, torch.bfloat16

    def w(*shape):
        return _normal(g, shape, s.w_std, device, bf)

    def nrm(n):
        return 1.0 + _normal(g, (n,), s.norm_std, device)

    fc = w(H, s.fc_in)
    hidden_norm, final_norm = nrm(H), nrm(H)
    layers = []
    for _ in range(s.n_layers):
        layers.append(LayerW(input_norm=nrm(H), post_norm=nrm(H), q_norm=nrm(s.head_dim),
                             k_norm=nrm(s.head_dim), wq=w(s.q_total, H), wk=w(s.kv_total, H),
                             wv=w(s.kv_total, H), wo=w(H, s.q_total), wg=w(I, H), wu=w(I, H),
                             wd=w(H, I)))
    embed = w(s.vocab, H)
    lm_head = w(s.vocab, H)
    return DFlashWeights(fc, hidden_norm, final_norm, layers, embed, lm_head)


def kv_cache(n_layers: int, B: int, n_kv: int, d: int, filled: int, cap: int, seed: int,
             device="cpu", bf16: bool = False) -> KvCache:
    """Per-layer F32 (or BF16) K/V of `cap` positions; the first `filled` hold N(0,1) rows."""
    g = _gen(seed, device)
    ks, vs = [], []
    dt = torch.bfloat16 if bf16 else torch.float32
    for _ in range(n_layers):
        k = torch.zeros((B, n_kv, cap, d), device=device, dtype=dt)
        v = torch.zeros_like(k)
        if filled:
            k[:, :, :filled] = _normal(g, (B, n_kv, filled, d), 1.0, device).to(dt)
            v[:, :, :filled] = _normal(g, (B, n_kv, filled, d), 1.0, device).to(dt)
        ks.append(k)
        vs.append(v)
    seq = torch.full((B,), filled, device=device, dtype=torch.int32)
    return KvCache(ks, vs, seq, cap)


def dflash_cache(s: DFlashShape, seed: int = 1, device="cpu", extra: int = 0) -> KvCache:
    return kv_cache(s.n_layers, s.batch, s.n_kv_heads, s.head_dim, s.ctx,
                    s.ctx + s.block + extra, seed, device, bf16=s.kv_bf16)


def accept_lengths(n: int, K: int, p: Optional[float], seed: int) -> np.ndarray:
    """Accept counts in [0, K]: geometric P(a >= j) = p**j capped at K, or U{0..K} if p is None."""
    rng = np.random.default_rng(seed)
    if p is None:
        return rng.integers(0, K + 1, size=n).astype(np.int32)
    u = rng.random(n)
    a = np.floor(np.log(np.maximum(u, 1e-300)) / math.log(p)).astype(np.int64)
    return np.minimum(a, K).astype(np.int32)


def dflash_round_inputs(s: DFlashShape, n_new, seed: int = 2, device="cpu") -> DFlashRoundInputs:
    """Block ids [last_token, mask x K] and the new target-hidden rows of each sequence."""
    g = _gen(seed, device)
    B = s.batch
    n_new = torch.as_tensor(np.asarray(n_new, dtype=np.int32).reshape(B), device=device)
    n_new_max = int(n_new.max().item()) if B else 0
    last = torch.randint(2, s.vocab - 1, (B,), generator=g, device=device, dtype=torch.int64)
    last = last.to(torch.int32)
    block = torch.full((B, s.block), s.mask_id, device=device, dtype=torch.int32)
    block[:, 0] = last
    th = _normal(g, (B, max(n_new_max, 1), s.fc_in), 1.0, device)
    return DFlashRoundInputs(last, block, th, n_new, n_new_max)


def targets_from_drafts(drafts: np.ndarray, accept: np.ndarray, vocab: int, seed: int) -> np.ndarray:
    """Target argmaxes [B, K+1]: equal to the drafts on [0, a), a different id at a, uniform after."""
    rng = np.random.default_rng(seed)
    drafts = np.asarray(drafts, dtype=np.int64)
    B, K = drafts.shape
    t = rng.integers(0, vocab, size=(B, K + 1)).astype(np.int64)
    for b in range(B):
        a = int(accept[b])
        t[b, :a] = drafts[b, :a]
        if a < K:
            t[b, a] = (drafts[b, a] + 1 + rng.integers(0, vocab - 1)) % vocab
    return t.astype(np.int32)


@dataclass
class MtpWeights:
    enorm: torch.Tensor
    hnorm: torch.Tensor
    eh_embed: torch.Tensor      # [H, H] BF16 (applied to enorm(embed))
    eh_hidden: torch.Tensor     # [H, H] BF16 (applied to hnorm(prev_hidden))
    attn_norm: torch.Tensor
    post_norm: torch.Tensor
    q_norm: torch.Tensor
    k_norm: torch.Tensor
    wq: torch.Tensor
    wk: torch.Tensor
    wv: torch.Tensor
    w_gate: Optional[torch.Tensor]
    wo: torch.Tensor
    shared_head_norm: torch.Tensor
    embed: torch.Tensor
    lm_head: torch.Tensor
    # dense FFN
    wg: Optional[torch.Tensor] = None
    wu: Optional[torch.Tensor] = None
    wd: Optional[torch.Tensor] = None
    # MoE FFN
    router: Optional[torch.Tensor] = None       # [E, H] BF16
    exp_g: Optional[torch.Tensor] = None        # [E, Ie, H]
    exp_u: Optional[torch.Tensor] = None        # [E, Ie, H]
    exp_d: Optional[torch.Tensor] = None        # [E, H, Ie]
    sh_g: Optional[torch.Tensor] = None         # [Is, H]
    sh_u: Optional[torch.Tensor] = None
    sh_d: Optional[torch.Tensor] = None         # [H, Is]
    sh_gate: Optional[torch.Tensor] = None      # [1, H] BF16


def mtp_weights(s: MtpShape, seed: int = 0, device="cpu") -> MtpWeights:
    g = _gen(seed, device)
    H, bf = s.hidden, torch.bfloat16

    def w(*shape, std=None):
        return _normal(g, shape, s.w_std if std is None else std, device, bf)

    def nrm(n):
        return 1.0 + _normal(g, (n,), s.norm_std, device)

    mw = MtpWeights(enorm=nrm(H), hnorm=nrm(H), eh_embed=w(H, H), eh_hidden=w(H, H),
                    attn_norm=nrm(H), post_norm=nrm(H), q_norm=nrm(s.head_dim),
                    k_norm=nrm(s.head_dim), wq=w(s.q_total, H), wk=w(s.kv_total, H),
                    wv=w(s.kv_total, H), w_gate=w(s.q_total, H) if s.gate else None,
                    wo=w(H, s.q_total), shared_head_norm=nrm(H), embed=w(s.vocab, H),
                    lm_head=w(s.vocab, H))
    if s.moe:
        E, Ie, Is = s.n_experts, s.expert_inter, s.shared_inter
        mw.router = w(E, H, std=1.0 / math.sqrt(H))
        mw.exp_g, mw.exp_u, mw.exp_d = w(E, Ie, H), w(E, Ie, H), w(E, H, Ie)
        mw.sh_g, mw.sh_u, mw.sh_d = w(Is, H), w(Is, H), w(H, Is)
        mw.sh_gate = w(1, H)
    else:
        I = s.intermediate
        mw.wg, mw.wu, mw.wd = w(I, H), w(I, H), w(H, I)
    return mw


def mtp_cache(s: MtpShape, steps: int, seed: int = 1, device="cpu") -> KvCache:
    return kv_cache(1, s.batch, s.n_kv_heads, s.head_dim, s.kv_len, s.kv_len + steps, seed, device)


def mtp_inputs(s: MtpShape, seed: int = 2, device="cpu"):
    """prev_hidden [B, H] F32 ~ N(0,1) and the just-accepted token ids [B]."""
    g = _gen(seed, device)
    prev = _normal(g, (s.batch, s.hidden), 1.0, device)
    tok = torch.randint(2, s.vocab - 1, (s.batch,), generator=g, device=device,
                        dtype=torch.int64).to(torch.int32)
    return prev, tok
