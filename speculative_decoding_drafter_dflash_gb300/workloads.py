"""Shapes of the draft-round workloads this library is tested and measured on.

Each workload is a plain frozen dataclass of dimensions. Nothing here computes
anything of the method; `synth.py` turns a shape plus a seed into inputs.

DFlash drafter shapes follow the per-layer tensor list of hf2q's
`spec_decode/dflash/tensors.rs` (`DFlashLayerTensors`, `DFlashModelTensors`):
fc `[H, n_tl*H]`, q/k/v/o, gate/up/down, F32 norms. MTP shapes follow
`models/qwen35/mtp.rs` (`MtpWeights`, `MtpFullAttnWeightsGpu`, `MtpFfnWeightsGpu`).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Tuple


@dataclass(frozen=True)
class DFlashShape:
    name: str
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    K: int                      # drafts per round; the block is K+1 positions
    ctx: int                    # context rows already in the drafter KV cache
    n_target_layers: int        # target hiddens concatenated into the fc input
    batch: int = 1
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    rotary_dim: int = 0         # 0 means head_dim
    mask_token_id: int = -1     # -1 means vocab - 1
    eos_ids: Tuple[int, ...] = (1,)
    causal_block: int = 0       # 0: the K+1 block attends bidirectionally
    w_std: float = 0.02
    norm_std: float = 0.1
    accept_p: float = 0.6       # P(accept >= j) = p**j for the geometric target
    kv_bf16: bool = False       # BF16 KV cache (False: F32)

    @property
    def block(self) -> int:
        return self.K + 1

    @property
    def mask_id(self) -> int:
        return self.vocab - 1 if self.mask_token_id < 0 else self.mask_token_id

    @property
    def rot(self) -> int:
        return self.head_dim if self.rotary_dim == 0 else self.rotary_dim

    @property
    def q_total(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_total(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def fc_in(self) -> int:
        return self.n_target_layers * self.hidden

    def with_(self, **kw) -> "DFlashShape":
        return replace(self, **kw)

    def weight_bytes(self) -> int:
        """BF16 projection bytes + F32 norm bytes of the drafter (no embed/lm_head)."""
        H, I, L = self.hidden, self.intermediate, self.n_layers
        per_layer = 2 * (self.q_total * H + 2 * self.kv_total * H + H * self.q_total + 3 * I * H)
        per_layer += 4 * (2 * H + 2 * self.head_dim)
        return 2 * H * self.fc_in + 4 * 2 * H + L * per_layer


@dataclass(frozen=True)
class MtpShape:
    name: str
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int           # dense SwiGLU intermediate (0 for MoE)
    vocab: int
    kv_len: int                 # positions already in the MTP KV slot
    gate: bool = True           # sigmoid output gate present
    n_experts: int = 0          # 0: dense FFN
    top_k: int = 0
    expert_inter: int = 0
    shared_inter: int = 0
    batch: int = 1
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    rotary_dim: int = 0
    w_std: float = 0.02
    norm_std: float = 0.1

    @property
    def rot(self) -> int:
        return self.head_dim if self.rotary_dim == 0 else self.rotary_dim

    @property
    def q_total(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_total(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def moe(self) -> bool:
        return self.n_experts > 0

    def with_(self, **kw) -> "MtpShape":
        return replace(self, **kw)


# Tiny DFlash drafter round: parity case the oracle finishes in well under a second.
TINY = DFlashShape("dflash-tiny-h256-l1-k4-ctx64", hidden=256, n_layers=1, n_q_heads=4,
                   n_kv_heads=2, head_dim=64, intermediate=512, vocab=4096, K=4, ctx=64,
                   n_target_layers=2)

# DFlash-shaped drafter round, K=15 (block 16), context 4096: the measured workload.
DFLASH_K15 = DFlashShape("dflash-h2816-l5-k15-ctx4096", hidden=2816, n_layers=5, n_q_heads=16,
                         n_kv_heads=8, head_dim=128, intermediate=8192, vocab=262144, K=15,
                         ctx=4096, n_target_layers=5)

# Dense MTP single-token draft step (chained 1..3 steps).
MTP_DENSE = MtpShape("mtp-dense-h5120-kv8192", hidden=5120, n_q_heads=24, n_kv_heads=4,
                     head_dim=256, intermediate=17408, vocab=248320, kv_len=8192)

# MoE MTP single-token draft step: 256 experts, softmax top-8, one sigmoid-gated shared expert.
MTP_MOE = MtpShape("mtp-moe-h2048-e256-kv16384", hidden=2048, n_q_heads=16, n_kv_heads=2,
                   head_dim=256, intermediate=0, vocab=248320, kv_len=16384, n_experts=256,
                   top_k=8, expert_inter=512, shared_inter=512)

# Small MTP shapes the oracle runs in seconds (same structure, scaled down).
MTP_TINY = MtpShape("mtp-dense-tiny-h256", hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                    intermediate=512, vocab=4096, kv_len=40)
MTP_MOE_TINY = MtpShape("mtp-moe-tiny-h256-e16", hidden=256, n_q_heads=4, n_kv_heads=2,
                        head_dim=64, intermediate=0, vocab=4096, kv_len=40, n_experts=16,
                        top_k=4, expert_inter=128, shared_inter=128)


def sweep_shapes():
    """DFlash-shaped round sweep: K x context x batch."""
    out = []
    for K in (1, 3, 7, 15):
        for ctx in (1024, 8192, 32768):
            for B in (1, 8):
                out.append(DFLASH_K15.with_(name=f"dflash-h2816-k{K}-ctx{ctx}-b{B}", K=K, ctx=ctx,
                                            batch=B))
    return out
