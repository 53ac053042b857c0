"""CPU oracle for one speculative-decoding draft round: TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct NumPy restatement of what the round computes,
written from hf2q 0.1.1's source pages (`models/qwen35/mtp.rs`,
`spec_decode/dflash/tensors.rs`, `spec_decode/dflash/qwen35_orchestrator.rs`).
Floating point is F32 over BF16-decoded weights, as those pages fix it
(BF16 projection weights, F32 activations/residuals/logits); every function
also runs in float64 (`dt=np.float64`) as a shadow to bound rounding.

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s cpu_baseline /
reference arm may import this package. The CUDA library never does, and this
package never imports the CUDA library: they share no code.

Pin status (what each function is checked against, in tests/test_oracle_*.py):
  decode_bf16            canonical round trip, odd length, misread signature, all 65536 patterns
  round_bf16             hand ties to even, every finite BF16 value kept, integer rounding rule
  BF16 KV cache          appended rows equal the F32 path's rows rounded to BF16
  rmsnorm / head_rmsnorm closed forms (constant vector, hand example), scale invariance, unit RMS
  rope                   hand example, norm preservation, R(p)R(q)=R(p+q), relative-position property
  sdpa                   brute-force float64 loops, one key, equal keys, GQA == MHA with repeated heads
  silu / sigmoid         special values
  argmax_top2            planted maxima, ties to the lowest index, brute-force scan
  accept_walk            hand examples + brute force over all short draft/target pairs
  kv_rollback            hand examples, overflow rejection
  qk_norm_rope           one-head hand example (norm first, then the turn)
  dflash forward / mtp   special cases with closed forms (zero projections, one key), whole-layer
                         closed forms with 2-dim heads (norm weights that do not commute with the
                         rotation fix "q/k norm, then RoPE"; identity / reversal projections; the
                         SwiGLU fed by the post-attention norm), float64 shadow, and planted slips
                         of the composition (norm order, FFN input norm, positions, eh halves,
                         gate placement, final-norm weight) that those pins catch
  moe routing            hand example, top-k weights sum to one, one-expert reduction to dense
  stochastic accept      hand draws, exact identity (committed token ~ target softmax) with a
                         planted wrong residual, Monte-Carlo run of the walk, greedy limit at
                         T -> 0 equals accept_walk, identical distributions accept everything
  generate loop          capture helpers by hand; output follows the verifier (the reference when
                         it never agrees), every draft accepted when it always agrees, budget
                         truncation, EOS stop, max_new_tokens == 0, prefix one behind the output
"""
