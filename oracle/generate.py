"""Oracle of the multi-round DFlash generate loop with a synthetic verifier: test
infrastructure only.

qwen35_orchestrator.rs, `dispatch_qwen35_dflash_generate`, "Multi-round loop (Option A)":
per round (1) block [last_token, mask x K]; (2)-(3) the drafter's new context rows are the
committed positions it has not consumed yet (prior_ctx_len - drafter cache length), built by
`extract_drafter_concat` from the captured verifier hidden states: per position, the rows of
the drafter's target layers (a subset of the captured "combined" layers) concatenated; (4)-(5)
drafter forward and per-position argmax, drafts = argmax[1..]; (6) verify [last_token, drafts]
at start_pos = len(output) - 1 with a capture of K+1 positions; (7) greedy accept walk;
(8) rollback; (9) append the committed tokens, last_token = the last one, stop on EOS or when
len(output) - len(prompt) >= max_new_tokens; (10) `append_capture_positions`: the first
n_committed verify positions join the captured prefix. After the loop the output is truncated
to len(prompt) + max_new_tokens. Before the loop the page returns at once when the first token
(from the prefill) is an EOS id or max_new_tokens == 0.

The verifier is synthetic (the target model is out of scope): its captured hidden state of
capture layer c at position p is table[c, p]; its greedy token after position p + j of a
verify (j < K) is the draft x_j itself when agree[p + j] is set, else ref[p + j + 1]; after the
last verify position (j = K) it is ref[p + K + 1]. Every table is an input.
"""
from __future__ import annotations

import numpy as np

from .core import OracleError, accept_walk
from .dflash import dflash_block_forward
from .core import lm_head_argmax


def extract_drafter_concat(prior_cap, sel, start, stop):
    """Rows [start, stop) of the captured prefix, each the concatenation over the drafter's
    target layers (indices sel into the captured layers): [stop - start, len(sel) * H]."""
    if not 0 <= start <= stop <= prior_cap.shape[1]:
        raise OracleError("extract range outside the captured prefix")
    return np.concatenate([prior_cap[c, start:stop] for c in sel], axis=1)


def append_capture_positions(prior_cap, prior_len, verify_cap, n):
    """The first n verify positions join the captured prefix at prior_len; returns the new
    length."""
    if prior_len + n > prior_cap.shape[1] or n > verify_cap.shape[1]:
        raise OracleError("capture append out of range")
    prior_cap[:, prior_len:prior_len + n] = verify_cap[:, :n]
    return prior_len + n


def synthetic_verify(ref, agree, p0, drafts):
    """Greedy tokens of the synthetic verifier for the K+1 verify positions starting at p0."""
    K = len(drafts)
    out = []
    for j in range(K + 1):
        p = p0 + j
        if p + 1 >= len(ref):
            raise OracleError("reference sequence too short")
        out.append(int(drafts[j]) if j < K and agree[p] else int(ref[p + 1]))
    return out


def generate(cfg, w, cache_k, cache_v, cache_len0, out0, prompt_len, ref, agree, table, sel,
             max_new, K, eos, max_rounds, dt=np.float32):
    """One sequence. cache_k/cache_v: per layer [1, n_kv, cap, d] (updated in place);
    out0: prompt + first token; table [n_comb, max_len, H]; sel: drafter target layers as
    indices into the captured layers. Returns dict(out, rounds, accept (per round), cache_len,
    prior_len, gaps (per round, the smallest top-1/top-2 gap of the drafted positions))."""
    out = [int(t) for t in out0]
    eos = set(int(e) for e in eos)
    n_comb, max_len, H = table.shape
    prior_cap = np.zeros_like(table)
    prior_len = len(out) - 1                    # the prefill captured the prompt positions
    prior_cap[:, :prior_len] = table[:, :prior_len]
    cache_len = int(cache_len0)
    rounds, accepts, gaps = 0, [], []
    if out[-1] in eos or max_new == 0:              # the page returns prompt + first token
        return dict(out=out, rounds=0, accept=[], cache_len=cache_len, prior_len=prior_len,
                    gaps=[])
    while len(out) - prompt_len < max_new and rounds < max_rounds:
        rounds += 1
        if prior_len + 1 != len(out) or prior_len < cache_len:
            raise OracleError("captured prefix out of step with the output")
        n_new = prior_len - cache_len
        th = extract_drafter_concat(prior_cap, sel, cache_len, prior_len)[None]
        block = np.array([[out[-1]] + [cfg.mask_id] * K])
        h_final, seq = dflash_block_forward(cfg, w, cache_k, cache_v, [cache_len], block, th,
                                            [n_new], dt)
        cache_len = int(seq[0])
        idx, t1, t2 = lm_head_argmax(h_final[0], w["lm_head"], dt)
        drafts = [int(x) for x in idx[1:]]
        gaps.append(float(np.min(np.asarray(t1[1:]) - np.asarray(t2[1:]))))
        p0 = len(out) - 1
        target = synthetic_verify(ref, agree, p0, drafts)
        verify_cap = table[:, p0:p0 + K + 1]
        committed, a, hit, rb = accept_walk(drafts, target, eos)
        accepts.append(a)
        out.extend(committed)
        if hit or len(out) - prompt_len >= max_new:
            break
        prior_len = append_capture_positions(prior_cap, prior_len, verify_cap, len(committed))
    return dict(out=out[:prompt_len + max_new], rounds=rounds, accept=accepts,
                cache_len=cache_len, prior_len=prior_len, gaps=gaps)
