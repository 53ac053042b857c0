#!/usr/bin/env python
"""Benchmark: DFlash-shaped draft rounds per second on GB300 (K=15, block 16, H=2816, 5
layers, 16q/8kv x 128, SwiGLU 8192, vocab 262144, context 4096), batch 1 per GPU.

One step = one whole draft round through the C ABI (`df_draft_round`: embed gather, fc +
hidden_norm of the new context rows, 5 drafter layers, final norm, lm_head + fused argmax of
the 16 block rows, greedy accept walk, verifier KV rollback) followed by `kv_rollback` of the
drafter cache, so every replay sees the same state (stateless replays of 8 seeded round
variants whose new-context-row counts follow geometric acceptance, p = 0.6).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Prints one JSON line (rank 0). N > 1 runs under torchrun: one replica per GPU (the round
does not shard; no collective on the data path), value = all ranks' rounds / max elapsed.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft rounds/s (DFlash shape, K=15) & achieved HBM GB/s vs 8 TB/s"
N_VARIANTS = 8


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of CUDA graphs")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="bound on the oracle's CPU sample time")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--batch", type=int, default=1, help="sequences of --profile-case round, trace, layout, gemms and lm_head")
    ap.add_argument("--ctx", type=int, default=0, help="cache rows of --profile-case round")
    ap.add_argument("--vocab", type=int, default=0, help="lm_head rows of --profile-case lm_head and round")
    ap.add_argument("--layers", type=int, default=0, help="drafter layers of --profile-case round")
    ap.add_argument("--trace-dump", default=None, help="--profile-case trace: save the records")

    ap.add_argument("--profile-case", choices=["lm_head", "round", "gemms", "sweep", "sweep_bf16kv", "mtp",
                                                     "moe", "attn", "stochastic", "sampled", "generate", "trace",
                                                     "layout"],
                    default=None,
                    help="run a few launches of one case for an ncu capture and exit")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampled every 200 ms during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def round_bytes(s, n_new: int) -> int:
    """Algorithmic HBM bytes of one round: every weight once, KV read of the cache plus the
    appended rows, KV write of the appended rows, the new target hidden rows, embed rows."""
    H, d, nkv, L = s.hidden, s.head_dim, s.n_kv_heads, s.n_layers
    kv_row = nkv * d * (2 if getattr(s, "kv_bf16", False) else 4) * 2   # K and V
    w = s.weight_bytes() + 2 * s.vocab * H         # drafter + lm_head
    kv_read = L * (s.ctx + n_new) * kv_row
    kv_write = L * n_new * kv_row
    return w + kv_read + kv_write + n_new * s.fc_in * 4 + s.block * H * 2


def lm_head_bytes(s, rows: int) -> int:
    return 2 * s.vocab * s.hidden + 2 * 2 * rows * s.hidden


def variants(s):
    """Seeded round variants: accept counts a_v (geometric) and n_new_v = a_{v-1} + 1."""
    from speculative_decoding_drafter_dflash_gb300 import synth
    acc = synth.accept_lengths(N_VARIANTS, s.K, s.accept_p, seed=123)
    n_new = [int(acc[(v - 1) % N_VARIANTS]) + 1 for v in range(N_VARIANTS)]
    return acc, n_new


# ----------------------------------------------------------------------------- CPU oracle legs
def oracle_round_setup(s, w, cache, inputs):
    from speculative_decoding_drafter_dflash_gb300 import synth
    h = synth.host
    hw = dict(fc=h(w.fc), hidden_norm=h(w.hidden_norm), final_norm=h(w.final_norm),
              embed=h(w.embed), lm_head=h(w.lm_head),
              layers=[dict(input_norm=h(l.input_norm), post_norm=h(l.post_norm), q_norm=h(l.q_norm),
                           k_norm=h(l.k_norm), wq=h(l.wq), wk=h(l.wk), wv=h(l.wv), wo=h(l.wo),
                           wg=h(l.wg), wu=h(l.wu), wd=h(l.wd)) for l in w.layers])
    ks = [h(k) for k in cache.k]
    vs = [h(v) for v in cache.v]
    seq = h(cache.seq_len).copy()
    return hw, ks, vs, seq, [(h(i.block_ids), h(i.target_hidden), h(i.n_new)) for i in inputs]


def oracle_rounds(s, hw, ks, vs, seq, host_inputs, targets, n: int, budget_s: float):
    """Time up to n oracle rounds (stopping once budget_s is spent); returns (rounds, seconds)."""
    from oracle import dflash as odf
    done, t0 = 0, time.perf_counter()
    while done < n:
        v = done % len(host_inputs)
        ids, th, nn = host_inputs[v]
        odf.draft_round(s, hw, ks, vs, seq, ids, th, nn, targets[v], s.eos_ids, [1 << 30])
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return done, time.perf_counter() - t0


def _openblas():
    """numpy's OpenBLAS library handle, found among the loaded libraries (None if absent)."""
    import ctypes
    import re
    try:
        with open("/proc/self/maps") as f:
            libs = sorted(set(re.findall(r"(/\S*openblas\S*\.so\S*)", f.read())))
    except OSError:
        return None
    for path in libs:
        try:
            return ctypes.CDLL(path)
        except OSError:
            continue
    return None


def _blas_fn(kind: str):
    lib = _openblas()
    if lib is None:
        return None
    for name in (f"scipy_openblas_{kind}_num_threads64_", f"scipy_openblas_{kind}_num_threads",
                 f"openblas_{kind}_num_threads64_", f"openblas_{kind}_num_threads"):
        if hasattr(lib, name):
            return getattr(lib, name)
    return None


def blas_threads():
    """Threads numpy's BLAS uses now (None when it cannot be asked)."""
    import numpy  # noqa: F401  (loads the BLAS library)
    fn = _blas_fn("get")
    return int(fn()) if fn is not None else None


def set_blas_threads(n: int) -> bool:
    import numpy  # noqa: F401
    fn = _blas_fn("set")
    if fn is None:
        return False
    import ctypes
    fn.argtypes = [ctypes.c_int]
    fn(int(n))
    return True


def _median_ms(fn, want: int, budget_s: float):
    times, t_all = [], time.perf_counter()
    while len(times) < want:
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > budget_s:
            break
    return statistics.median(times) * 1e3, len(times)


def cpu_legs(dflash_state, budget_s: float, dev):
    """The CPU oracle on the tiny DFlash shape, the DFlash K=15 round and a 3-step dense MTP
    chain, with every core and with one BLAS thread (median ms of >= 3 rounds, >= 100 for the
    tiny shape, each leg bounded by budget_s). Inputs are drawn on the GPU and copied to the
    host, as for the main leg; dflash_state is the main leg's host state, reused."""
    from oracle import dflash as odf
    from oracle import mtp as omtp
    from speculative_decoding_drafter_dflash_gb300 import synth
    from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15, MTP_DENSE, TINY
    h = synth.host
    legs = {}
    # tiny DFlash round
    s = TINY
    w = synth.dflash_weights(s, seed=0, device=dev)
    cache = synth.dflash_cache(s, seed=1, device=dev)
    inp = synth.dflash_round_inputs(s, [3], seed=2, device=dev)
    hw, ks, vs, seq, hinp = oracle_round_setup(s, w, cache, [inp])
    ids, th, nn = hinp[0]
    tgt = np.zeros((1, s.block), dtype=np.int32)
    runs = {"tiny": (s.name, "round", 100,
                     lambda: odf.draft_round(s, hw, ks, vs, seq, ids, th, nn, tgt, s.eos_ids,
                                             [1 << 30]))}
    # DFlash K=15 round (the main leg's weights and inputs)
    s2 = DFLASH_K15
    hw2, ks2, vs2, seq2, hinp2, tg2 = dflash_state
    ids2, th2, nn2 = hinp2[0]
    runs["dflash"] = (s2.name, "round", 3,
                      lambda: odf.draft_round(s2, hw2, ks2, vs2, seq2, ids2, th2, nn2, tg2[0],
                                              s2.eos_ids, [1 << 30]))
    # dense MTP, one chain of 3 steps
    s3 = MTP_DENSE
    w3 = synth.mtp_weights(s3, seed=0, device=dev)
    hw3 = {n: (None if getattr(w3, n) is None else h(getattr(w3, n))) for n in (
        "enorm", "hnorm", "eh_embed", "eh_hidden", "attn_norm", "post_norm", "q_norm", "k_norm",
        "wq", "wk", "wv", "w_gate", "wo", "shared_head_norm", "embed", "lm_head", "wg", "wu", "wd",
        "router", "exp_g", "exp_u", "exp_d", "sh_g", "sh_u", "sh_d", "sh_gate")}
    del w3
    c3 = synth.mtp_cache(s3, 3, seed=1, device=dev)
    k3, v3, q3 = h(c3.k[0]), h(c3.v[0]), h(c3.seq_len).copy()
    p3, t3 = synth.mtp_inputs(s3, seed=2, device=dev)
    p3, t3 = h(p3), h(t3)
    del c3
    runs["mtp3"] = (s3.name, "3-step chain", 3,
                    lambda: omtp.mtp_forward_draft(s3, hw3, k3.copy(), v3.copy(), q3, p3, t3, 3))
    all_threads = blas_threads()
    for name, (wl, per, want, fn) in runs.items():
        leg = {"workload": wl, "per": per}
        fn()                                                   # warm-up
        for label, n in (("all_cores", all_threads), ("one_thread", 1)):
            if label == "one_thread" and not set_blas_threads(1):
                leg[label] = "unavailable: numpy's BLAS thread count cannot be set"
                continue
            ms, k = _median_ms(fn, want, budget_s)
            leg[label] = {"ms": round(ms, 3), "rounds": k, "blas_threads": blas_threads()}
            if all_threads:
                set_blas_threads(all_threads)
        legs[name] = leg
    return legs


def max_over_ranks(seconds: float, world: int, device=None) -> float:
    """The slowest rank's elapsed time (all ranks call this; a single rank returns its own)."""
    if world <= 1:
        return seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(steps_per_rank: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: every rank's rounds over the slowest rank's time (weak scaling:
    each rank runs its own replica on its own sequences)."""
    return steps_per_rank * world / max_seconds


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ----------------------------------------------------------------------------- native
def run_native(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from speculative_decoding_drafter_dflash_gb300 import binding as B
    from speculative_decoding_drafter_dflash_gb300 import synth
    from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15

    B.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    s = DFLASH_K15
    acc, n_new = variants(s)
    nmax = s.block
    w = synth.dflash_weights(s, seed=0, device=dev)
    cache = synth.dflash_cache(s, seed=1, device=dev)
    inputs = []
    for v in range(N_VARIANTS):
        inp = synth.dflash_round_inputs(s, [nmax], seed=10 + 100 * rank + v, device=dev)
        inp.n_new = torch.tensor([n_new[v]], dtype=torch.int32, device=dev)
        inputs.append(inp)
    model = B.DFlashModel(s, w, cache)
    ws = B.alloc_workspace(model.workspace_bytes(1, s.block, nmax), dev)
    out = B.RoundOutputs(1, s.K, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    eos = torch.tensor(s.eos_ids, dtype=torch.int32, device=dev)
    tsl = torch.full((1,), 1 << 30, dtype=torch.int32, device=dev)
    zero_tgt = torch.zeros((1, s.block), dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)

    def step(v, tgt):
        inp = inputs[v]
        B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new, nmax, s.K, tgt, eos,
                         tsl, out, ws, st, stream=stream)
        B.kv_rollback(cache.seq_len, inp.n_new, st, stream=stream)

    # Untimed pass: each variant's drafts define its synthetic target argmaxes.
    targets, drafts = [], []
    with torch.cuda.stream(stream):
        for v in range(N_VARIANTS):
            step(v, zero_tgt)
            stream.synchronize()
            d = out.argmax[0, 1:].cpu().numpy()
            drafts.append(d)
            t = synth.targets_from_drafts(d[None, :], np.array([acc[v]]), s.vocab, seed=50 + v)
            targets.append(torch.tensor(t, device=dev))
        # Check pass: drafts repeat bit-exactly and the accept walk lands on a_v.
        ok = True
        l0 = B.kernel_launches()
        for v in range(N_VARIANTS):
            step(v, targets[v])
            stream.synchronize()
            ok &= bool(np.array_equal(out.argmax[0, 1:].cpu().numpy(), drafts[v]))
            ok &= int(out.accept[0]) == int(acc[v]) and int(st.item()) == 0
        launches_per_step = (B.kernel_launches() - l0) // N_VARIANTS
    if not ok:
        raise RuntimeError("replayed rounds did not reproduce their drafts / accept counts")

    graphs = []
    if not args.no_graph:
        for v in range(N_VARIANTS):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(v, targets[v])
            graphs.append(g)

    def run(i):
        v = i % N_VARIANTS
        if graphs:
            graphs[v].replay()
        else:
            step(v, targets[v])

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            run(i)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            run(i)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    elapsed = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    if world > 1:
        dist.barrier()
    assert int(st.item()) == 0, "device status set during the timed region"
    rounds = args.steps * world
    value = job_rate(args.steps, world, elapsed)
    ms = elapsed / args.steps * 1e3
    avg_bytes = sum(round_bytes(s, n_new[i % N_VARIANTS]) for i in range(args.steps)) / args.steps
    hbm_peak, peak_kind = peaks()

    # Dominant kernel (lm_head + fused argmax over the 16 block rows): CUDA events around each
    # call on its launching stream, inputs resident, weights (1.48 GB) far larger than L2.
    rows = s.block
    X = torch.randn((rows, s.hidden), device=dev)
    idx = torch.empty(rows, dtype=torch.int32, device=dev)
    ws_lm = B.alloc_workspace(B.lm_head_workspace_bytes(rows, s.hidden, s.vocab), dev)
    Wt = B.TiledMatrix(w.lm_head)     # the tiled lm_head, as the round reads it
    torch.cuda.synchronize(dev)
    durs = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            B.lm_head_argmax_tiled(Wt, X, idx, ws=ws_lm, stream=stream)
        for i in range(max(args.steps, 10)):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            B.lm_head_argmax_tiled(Wt, X, idx, ws=ws_lm, stream=stream)
            b.record(stream)
            durs.append((a, b))
    torch.cuda.synchronize(dev)
    lm_s = statistics.mean(a.elapsed_time(b) for a, b in durs) / 1e3
    lm_ach = lm_head_bytes(s, rows) / lm_s / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "lm_head_argmax_traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tj = json.load(f)
        if tj.get("kernel_source_hash") == kernel_hash():
            traffic = tj.get("dram_bytes_per_launch")

    # End to end through the host-buffer entry point: pinned host inputs copied in, the round,
    # results copied back and the stream synchronised, every step.
    e2e = None
    if True:
        hin = []
        for v in range(N_VARIANTS):
            inp = inputs[v]
            hin.append(dict(last=inp.last_token.cpu().pin_memory(),
                            th=inp.target_hidden.cpu().pin_memory(),
                            nn=inp.n_new.cpu().pin_memory(), tgt=targets[v].cpu().pin_memory()))
        heos = eos.cpu().pin_memory()
        htsl = torch.full((1,), 1 << 30, dtype=torch.int32).pin_memory()
        hout = {k: torch.zeros(shape, dtype=torch.int32).pin_memory() for k, shape in (
            ("argmax", (1, s.block)), ("committed", (1, s.block)), ("n_committed", (1,)),
            ("accept", (1,)), ("hit_eos", (1,)), ("rollback", (1,)), ("status", (1,)))}
        ws_h = B.alloc_workspace(B.draft_round_host_workspace_bytes(model, 1, s.K, nmax, 1), dev)

        def host_step(i):
            v = i % N_VARIANTS
            h = hin[v]
            B.df_draft_round_host(model, h["last"], h["th"], h["nn"], nmax, s.K, h["tgt"], heos,
                                  htsl, hout, ws_h, stream=stream)
            B.kv_rollback(cache.seq_len, inputs[v].n_new, st, stream=stream)

        for i in range(args.warmup):
            host_step(i)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for i in range(args.steps):
            host_step(i)
        torch.cuda.synchronize(dev)
        e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
        assert int(hout["status"][0]) == 0
        h2d = sum(hin[i % N_VARIANTS]["last"].numel() * 4 + hin[i % N_VARIANTS]["th"].numel() * 4
                  + 4 + hin[i % N_VARIANTS]["tgt"].numel() * 4 + 4 + 4
                  for i in range(args.steps)) // args.steps
        d2h = sum(t.numel() * 4 for t in hout.values())
        e2e = {"value": round(rounds / e2e_s, 3), "unit": "rounds/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        hw, ks, vs, seq, hinp = oracle_round_setup(s, w, cache, inputs)
        tg = [t.cpu().numpy() for t in targets]
        oracle_rounds(s, hw, ks, vs, seq, hinp, tg, 1, 1e9)      # warm the BLAS / page cache
        n, secs = oracle_rounds(s, hw, ks, vs, seq, hinp, tg, 50, args.cpu_seconds)
        cpu = {"value": round(n / secs, 4), "unit": "rounds/s", "cores": cores(), "kind": "oracle",
               "sample": f"{n} full rounds of this workload by the NumPy F32 oracle ({secs:.1f} s)",
               "blas_threads": blas_threads(),
               "legs": cpu_legs((hw, ks, vs, seq, hinp, tg), max(3.0, args.cpu_seconds / 3), dev)}
        del hw, ks, vs

    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": round(value, 3), "unit": "rounds/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 hi/lo pair, f32 accumulate",
        "data": "synthetic",
        "config": {"workload": s.name, "batch_per_gpu": 1, "K": s.K, "block": s.block,
                   "ctx": s.ctx, "hidden": s.hidden, "layers": s.n_layers, "heads": "16q/8kv x 128",
                   "intermediate": s.intermediate, "vocab": s.vocab,
                   "weights": "bf16", "activations_kv": "f32", "accumulate": "f32",
                   "arithmetic": "bf16 weights x f32 activations carried into tcgen05 kind::f16 "
                                 "as a bf16 hi/lo pair (~16 mantissa bits); attention splits the "
                                 "f32 KV the same way (lo x lo dropped); f32 accumulate, softmax "
                                 "and norms",
                   "n_new_per_variant": n_new, "accept_per_variant": [int(a) for a in acc],
                   "l2": "no flush: each round streams 2.6 GB of weights, 20x the 129 MB L2",
                   "cuda_graph": not args.no_graph, "parallelism": f"replicas x{world}"},
        "positions_per_s": round(value * s.block, 1),
        "drafts_per_s": round(value * s.K, 1),
        "round_bytes": int(avg_bytes),
        "round_hbm_gbs": round(avg_bytes / (ms / 1e3) / 1e9, 1),
        "round_frac_of_8tbs": round(avg_bytes / (ms / 1e3) / 8e12, 4),
        "round_frac_of_measured_hbm": round(avg_bytes / (ms / 1e3) / 1e9 / hbm_peak, 4),
        "roofline": {"kernel": "lm_head_argmax_tiled (tiled lm_head x 16 block rows, fused argmax)",
                     "bound": "hbm", "achieved": round(lm_ach, 1), "peak": hbm_peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(lm_ach / hbm_peak, 4),
                     "traffic": traffic, "bytes_per_launch": lm_head_bytes(s, rows),
                     "avg_launch_us": round(lm_s * 1e6, 2)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches_per_step * args.steps),
        "launches_per_step": int(launches_per_step),
        "clocks": clk,
    }


LM_HEAD_SOURCES = ("k_gemm_tc.cu", "tc_ptx.cuh")


def kernel_hash(files=LM_HEAD_SOURCES):
    """Hash of the CUDA sources of the lm_head kernel: a stored traffic figure is only used for
    the kernel code it was taken on."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_drafter_dflash_gb300", "csrc")
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The oracle, as it stands, timed on this machine's host cores on the same workload."""
    if rank != 0:
        return None
    import torch

    from speculative_decoding_drafter_dflash_gb300 import synth
    from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15
    s = DFLASH_K15
    dev = "cuda" if torch.cuda.is_available() else "cpu"       # generation only
    acc, n_new = variants(s)
    w = synth.dflash_weights(s, seed=0, device=dev)
    cache = synth.dflash_cache(s, seed=1, device=dev)
    inputs = []
    for v in range(N_VARIANTS):
        inp = synth.dflash_round_inputs(s, [s.block], seed=10 + v, device=dev)
        inp.n_new = torch.tensor([n_new[v]], dtype=torch.int32, device=dev)
        inputs.append(inp)
    hw, ks, vs, seq, hinp = oracle_round_setup(s, w, cache, inputs)
    del w, cache, inputs
    # Each step is one full oracle round. The target row only steers the integer walk at the
    # end, so a fixed one leaves the timed arithmetic the same as with per-variant targets.
    tg = [np.zeros((1, s.block), dtype=np.int32)] * N_VARIANTS
    for i in range(args.warmup):
        oracle_rounds(s, hw, ks, vs, seq, [hinp[i % N_VARIANTS]], tg, 1, 1e9)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_rounds(s, hw, ks, vs, seq, [hinp[i % N_VARIANTS]], tg, 1, 1e9)
    secs = time.perf_counter() - t0
    value = args.steps / secs
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "rounds/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": s.name, "batch_per_gpu": 1, "K": s.K, "ctx": s.ctx},
        "cpu_baseline": {"value": round(value, 4), "unit": "rounds/s", "cores": cores(),
                         "kind": "oracle",
                         "sample": "one full round of the workload per step (NumPy F32 oracle)"},
        "e2e": {"value": round(value, 4), "unit": "rounds/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _graph_rate(run_once, steps: int, warmup: int = 3) -> float:
    """Capture run_once into a CUDA graph, replay it, return replays per second (CUDA events)."""
    import torch
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run_once(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run_once(stream)
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return steps / (e0.elapsed_time(e1) / 1e3)


def sweep_case(steps: int, kv_bf16: bool = False):
    """Draft rounds/s over K x context x batch at the DFlash shape (one line per case); with
    kv_bf16 the drafter's KV cache is BF16."""
    import torch

    from speculative_decoding_drafter_dflash_gb300 import binding as B
    from speculative_decoding_drafter_dflash_gb300 import synth
    from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15
    dev = torch.device("cuda", 0)
    hbm_peak, _ = peaks()
    w = synth.dflash_weights(DFLASH_K15, seed=0, device=dev)
    for ctx in (1024, 8192, 32768):
        for Bn in (1, 8):
            cache = None
            for K in (1, 3, 7, 15):
                s = DFLASH_K15.with_(K=K, ctx=ctx, batch=Bn, kv_bf16=kv_bf16)
                if cache is None or cache.cap < s.ctx + s.block:
                    cache = None
                    torch.cuda.empty_cache()
                    cache = synth.dflash_cache(s.with_(K=15), seed=1, device=dev)
                cache.seq_len.fill_(ctx)
                acc = synth.accept_lengths(Bn, K, s.accept_p, seed=7)
                n_new = [int(a) + 1 for a in acc]
                inp = synth.dflash_round_inputs(s, n_new, seed=3, device=dev)
                model = B.DFlashModel(s, w, cache)
                ws = B.alloc_workspace(model.workspace_bytes(Bn, s.block, inp.n_new_max), dev)
                out = B.RoundOutputs(Bn, K, dev)
                eos = torch.tensor(s.eos_ids, dtype=torch.int32, device=dev)
                tsl = torch.full((Bn,), 1 << 30, dtype=torch.int32, device=dev)
                tgt = torch.zeros((Bn, s.block), dtype=torch.int32, device=dev)

                def once(stream):
                    B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new,
                                     inp.n_new_max, K, tgt, eos, tsl, out, ws, stream=stream)
                    B.kv_rollback(cache.seq_len, inp.n_new, stream=stream)

                rate = _graph_rate(once, steps)
                nb = sum(round_bytes(s, n) for n in n_new) - (Bn - 1) * (s.weight_bytes() + 2 * s.vocab * s.hidden)
                print(json.dumps({"profile_case": "sweep", "kv": "bf16" if kv_bf16 else "f32",
                                  "K": K, "ctx": ctx, "batch": Bn,
                                  "rounds_per_s": round(rate, 1),
                                  "positions_per_s": round(rate * Bn * s.block, 1),
                                  "round_us": round(1e6 / rate, 1), "round_bytes": int(nb),
                                  "frac_of_measured_hbm": round(nb * rate / 1e9 / hbm_peak, 4)}),
                      flush=True)
                del ws, model, out


def mtp_step_weight_bytes(s) -> int:
    """Weight bytes one MTP step streams for one sequence: eh_proj, q/k/v(/gate)/o, the FFN
    (dense SwiGLU, or router + top_k experts + shared expert and its gate) and lm_head."""
    H = s.hidden
    attn = 2 * H * H + s.q_total * H * (3 if s.gate else 2) + 2 * s.kv_total * H
    if s.moe:
        ffn = s.n_experts * H + s.top_k * 3 * s.expert_inter * H + 3 * s.shared_inter * H + H
    else:
        ffn = 3 * s.intermediate * H
    return 2 * (attn + ffn + s.vocab * H)


def mtp_case(steps: int):
    """MTP chained draft (1..3 steps) at full size, dense and MoE FFN: steps/s and HBM
    fraction."""
    import torch

    from speculative_decoding_drafter_dflash_gb300 import binding as B
    from speculative_decoding_drafter_dflash_gb300 import synth
    from speculative_decoding_drafter_dflash_gb300.workloads import MTP_DENSE, MTP_MOE
    dev = torch.device("cuda", 0)
    hbm_peak, _ = peaks()
    for s in (MTP_DENSE, MTP_MOE):
        w = synth.mtp_weights(s, seed=0, device=dev)
        H, d = s.hidden, s.head_dim
        wbytes = mtp_step_weight_bytes(s)
        for n_steps in (1, 2, 3):
            cache = synth.mtp_cache(s, n_steps, seed=1, device=dev)
            prev, tok = synth.mtp_inputs(s, seed=2, device=dev)
            model = B.MtpModel(s, w, cache)
            ws = B.alloc_workspace(model.workspace_bytes(1), dev)
            hid = torch.empty((n_steps, 1, H), device=dev)
            am = torch.empty((n_steps, 1), dtype=torch.int32, device=dev)
            nback = torch.tensor([n_steps], dtype=torch.int32, device=dev)

            def once(stream):
                B.mtp_forward_draft(model, prev, tok, n_steps, hid, am, ws, stream=stream)
                B.kv_rollback(cache.seq_len, nback, stream=stream)

            rate = _graph_rate(once, steps)
            kv = sum((s.kv_len + i + 1) * s.n_kv_heads * d * 8 for i in range(n_steps))
            nb = n_steps * wbytes + kv
            print(json.dumps({"profile_case": "mtp", "workload": s.name, "n_steps": n_steps,
                              "drafts_per_s": round(rate * n_steps, 1),
                              "call_us": round(1e6 / rate, 1),
                              "step_us": round(1e6 / rate / n_steps, 1), "bytes_per_call": int(nb),
                              "frac_of_measured_hbm": round(nb * rate / 1e9 / hbm_peak, 4)}),
                  flush=True)
            del ws, model, cache
        del w
        torch.cuda.empty_cache()


def moe_case(steps: int):
    """The MoE FFN alone at full size (H=2048, 256 experts top-8, SwiGLU 512, shared expert)
    for 1 and 8 rows: weight bytes streamed over time. One MoE block is 57 MB, under L2, so
    each timed replay runs four blocks with their own weights (230 MB) in turn."""
    import torch

    from speculative_decoding_drafter_dflash_gb300 import binding as B
    from speculative_decoding_drafter_dflash_gb300 import synth
    from speculative_decoding_drafter_dflash_gb300.workloads import MTP_MOE
    dev = torch.device("cuda", 0)
    hbm_peak, _ = peaks()
    s = MTP_MOE.with_(vocab=1024)        # lm_head and embedding are not read here
    n_sets = 4
    models = [B.MtpModel(s, synth.mtp_weights(s, seed=i, device=dev),
                         synth.mtp_cache(s, 1, seed=1, device=dev)) for i in range(n_sets)]
    H = s.hidden
    g = torch.Generator(device=dev).manual_seed(5)
    for T in (1, 8):
        x = torch.randn((T, H), generator=g, device=dev)
        out = torch.empty_like(x)
        ids = [torch.empty((T, s.top_k), dtype=torch.int32, device=dev) for _ in models]
        ws = [B.alloc_workspace(m.moe_workspace_bytes(T), dev) for m in models]

        def once(stream):
            for m, i, w in zip(models, ids, ws):
                B.moe_ffn(m, x, out, w, i, stream=stream)

        rate = _graph_rate(once, steps) * n_sets
        torch.cuda.synchronize()
        distinct = sum(len(set(i.cpu().numpy().reshape(-1).tolist())) for i in ids) / n_sets
        nb = 2 * H * (s.n_experts + 1 + distinct * 3 * s.expert_inter + 3 * s.shared_inter)
        print(json.dumps({"profile_case": "moe", "workload": "moe-ffn-h2048-e256-top8-i512",
                          "rows": T, "distinct_experts": distinct, "call_us": round(1e6 / rate, 2),
                          "weight_bytes": int(nb),
                          "frac_of_measured_hbm": round(nb * rate / 1e9 / hbm_peak, 4)}),
              flush=True)


def attn_case(steps: int):
    """Split-KV attention alone on the drafter shapes: KV bytes read over time, each call timed
    with CUDA events after a 256 MB write that evicts L2."""
    import torch

    from speculative_decoding_drafter_dflash_gb300 import binding as B
    dev = torch.device("cuda", 0)
    hbm_peak, _ = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    g = torch.Generator(device=dev).manual_seed(0)
    cases = [("dflash-k15-ctx4096-b1", 1, 16, 16, 8, 128, 4096, True),
             ("dflash-k15-ctx32768-b1", 1, 16, 16, 8, 128, 32768, True),
             ("dflash-k15-ctx8192-b8", 8, 16, 16, 8, 128, 8192, True),
             ("mtp-dense-kv8192", 1, 1, 24, 4, 256, 8192, False),
             ("mtp-moe-kv16384", 1, 1, 16, 2, 256, 16384, False)]
    for name, Bn, blk, nq, nkv, d, ctx, blockk in cases:
        q = torch.randn((Bn, blk, nq, d), generator=g, device=dev)
        ck = torch.randn((Bn, nkv, ctx, d), generator=g, device=dev)
        cv = torch.randn((Bn, nkv, ctx, d), generator=g, device=dev)
        kb = torch.randn((Bn, nkv, blk, d), generator=g, device=dev) if blockk else None
        vb = torch.randn((Bn, nkv, blk, d), generator=g, device=dev) if blockk else None
        sl = torch.full((Bn,), ctx, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        ws = B.alloc_workspace(B.attention_workspace_bytes(Bn, blk, nq, nkv, d, ctx), dev)
        for _ in range(3):
            B.attention(q, ck, cv, sl, out, ws, kb, vb)
        times = []
        for _ in range(steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            B.attention(q, ck, cv, sl, out, ws, kb, vb)
            e1.record()
            times.append((e0, e1))
        torch.cuda.synchronize()
        us = statistics.median(a.elapsed_time(b) for a, b in times) * 1e3
        nb = 2 * Bn * nkv * (ctx + (blk if blockk else 0)) * d * 4 + 2 * q.numel() * 4
        B.profile_enable(True)
        B.attention(q, ck, cv, sl, out, ws, kb, vb)
        ks = [n for n, _ in B.profile_read()]
        B.profile_enable(False)
        print(json.dumps({"profile_case": "attn", "workload": name, "us": round(us, 2),
                          "bytes": int(nb), "gbs": round(nb / us / 1e3, 1),
                          "frac_of_measured_hbm": round(nb / us / 1e3 / hbm_peak, 4),
                          "kernels": ks}), flush=True)
        del q, ck, cv, kb, vb, out, ws


def stochastic_case(steps: int):
    """The stochastic accept step alone (K=15, V=262144, T=0.8) for 1 and 8 sequences: logit
    bytes read once over time, each call timed with CUDA events after an L2-evicting write."""
    import torch

    from speculative_decoding_drafter_dflash_gb300 import binding as B
    dev = torch.device("cuda", 0)
    hbm_peak, _ = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    g = torch.Generator(device=dev).manual_seed(0)
    K, V, T = 15, 262144, 0.8
    for Bn in (1, 8):
        tl = torch.randn((Bn, K + 1, V), generator=g, device=dev) * 2.0
        dl = (tl[:, :K] + torch.randn((Bn, K, V), generator=g, device=dev) * 0.5).contiguous()
        drafts = torch.argmax(dl, dim=-1).to(torch.int32).contiguous()
        ua = torch.rand((Bn, K), generator=g, device=dev)
        us = torch.rand((Bn,), generator=g, device=dev)
        eos = torch.tensor([1], dtype=torch.int32, device=dev)
        out = {k: torch.empty((Bn,), dtype=torch.int32, device=dev)
               for k in ("n_committed", "accept", "hit_eos", "rollback")}
        out["committed"] = torch.empty((Bn, K + 1), dtype=torch.int32, device=dev)
        ws = B.alloc_workspace(B.accept_stochastic_workspace_bytes(Bn, K, V), dev)
        for _ in range(3):
            B.accept_stochastic(dl, tl, drafts, T, ua, us, eos, out, ws)
        times = []
        for _ in range(steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            B.accept_stochastic(dl, tl, drafts, T, ua, us, eos, out, ws)
            e1.record()
            times.append((e0, e1))
        torch.cuda.synchronize()
        us_ = statistics.median(a.elapsed_time(b) for a, b in times) * 1e3
        nb = Bn * (2 * K + 1) * V * 4
        flush.fill_(1)
        B.profile_enable(True)          # one more call, each launch bracketed by events
        B.accept_stochastic(dl, tl, drafts, T, ua, us, eos, out, ws)
        torch.cuda.synchronize()
        per = [[n, round(t, 2)] for n, t in B.profile_read()]
        B.profile_enable(False)
        print(json.dumps({"profile_case": "stochastic", "workload": f"accept-k{K}-v{V}-b{Bn}",
                          "us": round(us_, 2), "logit_bytes": nb,
                          "gbs": round(nb / us_ / 1e3, 1),
                          "frac_of_measured_hbm": round(nb / us_ / 1e3 / hbm_peak, 4),
                          "mean_accept": float(out["accept"].float().mean()),
                          "per_launch_us_with_event_overhead": per}), flush=True)
        del tl, dl, ws


def sampled_case(steps: int):
    """The non-greedy path at full size: sample_softmax over the 15 drafter rows of a round
    (V=262144, after an L2-evicting write), the whole non-greedy DFlash round (K=15, ctx 4096,
    T=1) against the greedy round on the same inputs, both as CUDA graphs, and the sampled dense
    MTP chain (1 and 3 steps) against the argmax chain."""
    import torch

    from speculative_decoding_drafter_dflash_gb300 import binding as B
    from speculative_decoding_drafter_dflash_gb300 import synth
    from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15, MTP_DENSE
    dev = torch.device("cuda", 0)
    hbm_peak, _ = peaks()
    g = torch.Generator(device=dev).manual_seed(0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = DFLASH_K15
    K, V = s.K, s.vocab
    # sample_softmax alone
    lg = torch.randn((K, V), generator=g, device=dev)
    u = torch.rand((K,), generator=g, device=dev)
    tok = torch.empty((K,), dtype=torch.int32, device=dev)
    ws = B.alloc_workspace(B.sample_softmax_workspace_bytes(K, V), dev)
    for _ in range(3):
        B.sample_softmax(lg, 1.0, u, tok, ws)
    times = []
    for _ in range(steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        B.sample_softmax(lg, 1.0, u, tok, ws)
        e1.record()
        times.append((e0, e1))
    torch.cuda.synchronize()
    us_ = statistics.median(a.elapsed_time(b) for a, b in times) * 1e3
    nb = K * V * 4                # one pass over every logit (plus one 8 KB chunk per draw)
    flush.fill_(1)
    B.profile_enable(True)
    B.sample_softmax(lg, 1.0, u, tok, ws)
    torch.cuda.synchronize()
    per = [[n, round(t, 2)] for n, t in B.profile_read()]
    B.profile_enable(False)
    print(json.dumps({"profile_case": "sampled", "workload": f"sample-softmax-{K}x{V}",
                      "us": round(us_, 2), "bytes": nb, "gbs": round(nb / us_ / 1e3, 1),
                      "frac_of_measured_hbm": round(nb / us_ / 1e3 / hbm_peak, 4),
                      "per_launch_us_with_event_overhead": per}), flush=True)
    del lg, ws
    # the non-greedy round against the greedy round
    acc, n_new = variants(s)
    w = synth.dflash_weights(s, seed=0, device=dev)
    cache = synth.dflash_cache(s, seed=1, device=dev)
    model = B.DFlashModel(s, w, cache)
    inp = synth.dflash_round_inputs(s, [s.block], seed=10, device=dev)
    inp.n_new = torch.tensor([n_new[0]], dtype=torch.int32, device=dev)
    eos = torch.tensor(s.eos_ids, dtype=torch.int32, device=dev)
    tsl = torch.full((1,), 1 << 30, dtype=torch.int32, device=dev)
    out = B.RoundOutputs(1, K, dev)
    tl = torch.randn((1, K + 1, V), generator=g, device=dev)
    ud, ua = torch.rand((1, K), generator=g, device=dev), torch.rand((1, K), generator=g, device=dev)
    us = torch.rand((1,), generator=g, device=dev)
    logits = torch.empty((1, K + 1, V), device=dev)
    drafts = torch.empty((1, K), dtype=torch.int32, device=dev)
    ws_s = B.alloc_workspace(B.draft_round_stochastic_workspace_bytes(model, 1, K, s.block), dev)
    ws_g = B.alloc_workspace(model.workspace_bytes(1, s.block, s.block), dev)
    tgt = torch.zeros((1, s.block), dtype=torch.int32, device=dev)

    def stochastic(stream):
        B.df_draft_round_stochastic(model, inp.last_token, inp.target_hidden, inp.n_new, s.block,
                                    K, tl, 1.0, ud, ua, us, eos, tsl, logits, drafts, out, ws_s,
                                    stream=stream)
        B.kv_rollback(cache.seq_len, inp.n_new, stream=stream)

    def greedy(stream):
        B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new, s.block, K, tgt,
                         eos, tsl, out, ws_g, stream=stream)
        B.kv_rollback(cache.seq_len, inp.n_new, stream=stream)

    rs = _graph_rate(stochastic, steps)
    rg = _graph_rate(greedy, steps)
    print(json.dumps({"profile_case": "sampled", "workload": s.name, "round": "T=1 sampled drafts",
                      "rounds_per_s": round(rs, 1), "round_us": round(1e6 / rs, 1),
                      "greedy_rounds_per_s": round(rg, 1), "greedy_round_us": round(1e6 / rg, 1),
                      "extra_us": round(1e6 / rs - 1e6 / rg, 1)}), flush=True)
    del w, cache, model, ws_s, ws_g, logits, tl
    torch.cuda.empty_cache()
    # the sampled dense MTP chain against the argmax chain
    m = MTP_DENSE
    w = synth.mtp_weights(m, seed=0, device=dev)
    for n_steps in (1, 3):
        cache = synth.mtp_cache(m, n_steps, seed=1, device=dev)
        prev, tk = synth.mtp_inputs(m, seed=2, device=dev)
        model = B.MtpModel(m, w, cache)
        wsm = B.alloc_workspace(model.workspace_bytes(1), dev)
        hid = torch.empty((n_steps, 1, m.hidden), device=dev)
        am = torch.empty((n_steps, 1), dtype=torch.int32, device=dev)
        lgm = torch.empty((n_steps, 1, m.vocab), device=dev)
        um = torch.rand((n_steps, 1), generator=g, device=dev)
        nback = torch.tensor([n_steps], dtype=torch.int32, device=dev)

        def sampled(stream):
            B.mtp_forward_draft_sampled(model, prev, tk, n_steps, 1.0, um, hid, am, lgm, wsm,
                                        stream=stream)
            B.kv_rollback(cache.seq_len, nback, stream=stream)

        def argmax(stream):
            B.mtp_forward_draft(model, prev, tk, n_steps, hid, am, wsm, stream=stream)
            B.kv_rollback(cache.seq_len, nback, stream=stream)

        r1, r0 = _graph_rate(sampled, steps), _graph_rate(argmax, steps)
        print(json.dumps({"profile_case": "sampled", "workload": m.name, "n_steps": n_steps,
                          "sampled_call_us": round(1e6 / r1, 1), "argmax_call_us": round(1e6 / r0, 1),
                          "extra_us_per_step": round((1e6 / r1 - 1e6 / r0) / n_steps, 1)}),
              flush=True)
        del cache, model, wsm, lgm
    del w
    torch.cuda.empty_cache()


def generate_case(steps: int):
    """The device generate loop (one CUDA graph with a while node) on the DFlash K=15 shape:
    prompt 4096 tokens already in the drafter cache, 256 new tokens, a synthetic verifier that
    takes a draft with probability 0.6 per position. Tokens/s and time per round, CUDA events
    around each call (state reset outside the timed region)."""
    import torch

    from speculative_decoding_drafter_dflash_gb300 import binding as B
    from speculative_decoding_drafter_dflash_gb300 import synth
    from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15
    dev = torch.device("cuda", 0)
    s = DFLASH_K15
    K, prompt, max_new, n_comb = s.K, s.ctx, 256, s.n_target_layers + 1
    max_len = prompt + max_new + 2 * (K + 2)
    for Bn in (1, 4):
        w = synth.dflash_weights(s, seed=0, device=dev) if Bn == 1 else w
        cache = synth.kv_cache(s.n_layers, Bn, s.n_kv_heads, s.head_dim, prompt, max_len, 1, dev)
        seq0 = cache.seq_len.clone()
        g = torch.Generator(device=dev).manual_seed(2)
        ref = torch.randint(2, s.vocab - 2, (Bn, max_len), generator=g, device=dev,
                            dtype=torch.int32)
        agree = (torch.rand((Bn, max_len), generator=g, device=dev) < 0.6).to(torch.uint8)
        table = torch.randn((Bn, n_comb, max_len, s.hidden), generator=g, device=dev)
        prior = table.clone()
        model = B.DFlashModel(s, w, cache)
        n_new_max = K + 1
        ws = B.alloc_workspace(B.generate_workspace_bytes(model, Bn, K, n_new_max), dev)
        out = torch.zeros((Bn, max_len), dtype=torch.int32, device=dev)
        out[:, :prompt + 1] = ref[:, :prompt + 1]
        pl = torch.full((Bn,), prompt, dtype=torch.int32, device=dev)
        out_len, prior_len = pl + 1, pl.clone()
        rounds = torch.zeros(Bn, dtype=torch.int32, device=dev)
        eos = torch.tensor([1], dtype=torch.int32, device=dev)
        max_rounds = max_new
        times, toks, rnds = [], [], []
        for it in range(steps + 2):
            cache.seq_len.copy_(seq0)
            out_len.copy_(pl + 1)
            prior_len.copy_(pl)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            B.generate(model, ref, agree, table, list(range(s.n_target_layers)), prior, prior_len,
                       out, out_len, pl, max_new, max_rounds, K, n_new_max, eos, rounds, ws)
            e1.record()
            torch.cuda.synchronize()
            if it >= 2:                          # the first calls build and warm the graph
                times.append(e0.elapsed_time(e1))
                toks.append(int((out_len - pl).sum()))
                rnds.append(int(rounds.max()))
        ms = statistics.median(times)
        print(json.dumps({"profile_case": "generate", "workload": f"dflash-k15-ctx4096-b{Bn}-new256",
                          "ms_per_call": round(ms, 3), "tokens": toks[-1], "rounds": rnds[-1],
                          "tokens_per_s": round(toks[-1] / ms * 1e3, 1),
                          "us_per_round": round(ms * 1e3 / rnds[-1], 1),
                          "tokens_per_round": round(toks[-1] / Bn / rnds[-1], 3)}), flush=True)
        del cache, ws, table, prior


TRACE_MARK = 1000                # kids of the in-kernel trace marks: TRACE_MARK + phase
GEMM_MARKS = (11, 12, 13)        # phases marked by the projection kernel; the others by attention
TRACE_NAMES = {1: "rope_table", 2: "qk_rope", 3: "attn", 4: "attn_combine", 5: "seq_advance",
               6: "attn_tc", 15: "pack", 16: "pack", 17: "argmax_final", 18: "accept",
               19: "rollback", 20: "word_copy"}


def layout_case(args):
    """Row-major against tiled weights on the same GPU: the lm_head + argmax alone (20 launches
    after 3 warm-up, CUDA events) and the whole draft round as a CUDA graph (30 replays), both
    layouts alternated three times; --batch / --ctx set the round's workload."""
    import torch

    from speculative_decoding_drafter_dflash_gb300 import binding as B
    from speculative_decoding_drafter_dflash_gb300 import synth
    from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15
    dev = torch.device("cuda", 0)
    s = DFLASH_K15.with_(batch=args.batch, ctx=args.ctx or DFLASH_K15.ctx)
    w = synth.dflash_weights(s, seed=0, device=dev)
    res = {}
    rows = s.block
    X = torch.randn((rows, s.hidden), device=dev)
    idx = torch.empty(rows, dtype=torch.int32, device=dev)
    ws = B.alloc_workspace(B.lm_head_workspace_bytes(rows, s.hidden, s.vocab), dev)
    Wt = B.TiledMatrix(w.lm_head)

    def lm(tiled):
        if tiled:
            B.lm_head_argmax_tiled(Wt, X, idx, ws=ws)
        else:
            B.lm_head_argmax(w.lm_head, X, idx, ws=ws)

    for _ in range(3):
        for tiled in (False, True):
            for _ in range(3):
                lm(tiled)
            ev = []
            for _ in range(20):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                lm(tiled)
                b.record()
                ev.append((a, b))
            torch.cuda.synchronize()
            key = "lm_head_tiled_us" if tiled else "lm_head_rowmajor_us"
            res.setdefault(key, []).append(
                round(statistics.mean(x.elapsed_time(y) for x, y in ev) * 1e3, 2))
    del Wt
    inp = synth.dflash_round_inputs(s, [s.block] * s.batch, seed=10, device=dev)
    inp.n_new = torch.tensor([3] * s.batch, dtype=torch.int32, device=dev)
    eos = torch.tensor(s.eos_ids, dtype=torch.int32, device=dev)
    tsl = torch.full((s.batch,), 1 << 30, dtype=torch.int32, device=dev)
    tgt = torch.zeros((s.batch, s.block), dtype=torch.int32, device=dev)
    graphs, keep = {}, []
    for tiled in (False, True):
        cache = synth.dflash_cache(s, seed=1, device=dev)
        model = B.DFlashModel(s, w, cache, tiled=tiled)
        wsr = B.alloc_workspace(model.workspace_bytes(s.batch, s.block, s.block), dev)
        out = B.RoundOutputs(s.batch, s.K, dev)
        st = torch.cuda.Stream(dev)

        def step(model=model, wsr=wsr, out=out, cache=cache, st=st):
            B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new, s.block, s.K,
                             tgt, eos, tsl, out, wsr, stream=st)
            B.kv_rollback(cache.seq_len, inp.n_new, stream=st)

        with torch.cuda.stream(st):
            step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            step()
        graphs[tiled] = (g, st)
        keep.append((model, wsr, out, cache))
    for _ in range(3):
        for tiled in (False, True):
            g, st = graphs[tiled]
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(st):
                a.record(st)
                for _ in range(30):
                    g.replay()
                b.record(st)
            torch.cuda.synchronize()
            key = "round_tiled_us" if tiled else "round_rowmajor_us"
            res.setdefault(key, []).append(round(a.elapsed_time(b) * 1e3 / 30, 1))
    print(json.dumps({"profile_case": "layout", "workload": s.name, "batch": s.batch,
                      "ctx": s.ctx, **res}))


def trace_case(args):
    """In-graph timeline of the draft round from the trace build (per-CTA global-timer spans of
    every kernel): CUDA-graph rounds of the workload, each launch's first start, last end and the
    time it adds to the round's critical path, summed per kernel over the rounds' layers."""
    from speculative_decoding_drafter_dflash_gb300 import build as bld
    os.environ["DFLASH_LIB"] = bld.build(trace=True)
    import torch

    from speculative_decoding_drafter_dflash_gb300 import binding as B
    from speculative_decoding_drafter_dflash_gb300 import synth
    from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15
    s = DFLASH_K15.with_(batch=args.batch, ctx=args.ctx or DFLASH_K15.ctx)
    Bn, dev = s.batch, torch.device("cuda", 0)
    acc, n_new = variants(s)
    nmax = s.block
    w = synth.dflash_weights(s, seed=0, device=dev)
    cache = synth.dflash_cache(s, seed=1, device=dev)
    model = B.DFlashModel(s, w, cache)
    ws = B.alloc_workspace(model.workspace_bytes(Bn, s.block, nmax), dev)
    out = B.RoundOutputs(Bn, s.K, dev)
    eos = torch.tensor(s.eos_ids, dtype=torch.int32, device=dev)
    tsl = torch.full((Bn,), 1 << 30, dtype=torch.int32, device=dev)
    tgt = torch.zeros((Bn, s.block), dtype=torch.int32, device=dev)
    inp = synth.dflash_round_inputs(s, [nmax] * Bn, seed=10, device=dev)
    inp.n_new = torch.tensor([n_new[b % N_VARIANTS] for b in range(Bn)], dtype=torch.int32,
                             device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new, nmax, s.K, tgt, eos,
                         tsl, out, ws, stream=stream)
        B.kv_rollback(cache.seq_len, inp.n_new, stream=stream)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    B.profile_enable(True)                       # the launch names, in order, of one round
    with torch.cuda.stream(stream):
        step()
    names = [n for n, _ in B.profile_read()]
    B.profile_enable(False)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    rounds = max(3, min(args.steps, 20))
    B.trace_reset()
    for _ in range(rounds):
        g.replay()
    torch.cuda.synchronize()
    kid, sm, t0, t1 = B.trace_read()
    if args.trace_dump:
        np.savez(args.trace_dump, kid=kid, sm=sm, t0=t0, t1=t1, names=np.array(names))
    is_mark = kid >= TRACE_MARK
    mk, mt = kid[is_mark] - TRACE_MARK, t0[is_mark].astype(np.int64)
    kid, sm, t0, t1 = kid[~is_mark], sm[~is_mark], t0[~is_mark], t1[~is_mark]
    # Every kernel waits for its predecessor's grid to complete before its CTAs finish, so the
    # launches follow one another in the order of their CTAs' end times (their start times
    # interleave: a successor's CTAs become resident early and wait).
    order = np.argsort(t1, kind="stable")
    kid, t0, t1 = kid[order], t0[order].astype(np.int64), t1[order].astype(np.int64)
    groups = []                                  # [kid, first start, last end, ctas]
    for k, a, b in zip(kid.tolist(), t0.tolist(), t1.tolist()):
        if groups and groups[-1][0] == k:
            g_ = groups[-1]
            g_[1] = min(g_[1], a)
            g_[2] = max(g_[2], b)
            g_[3] += 1
        else:
            groups.append([k, a, b, 1])
    per = len(names)
    ok = len(groups) == per * rounds
    # Each launch is charged the time by which it moves the end of the timeline (the idle time
    # before it included), so the charges add up to the span of the replays.
    agg, crit_total, timeline = {}, 0.0, []
    prev_end = groups[0][1] if groups else 0
    for i, (k, a, b, n) in enumerate(groups):
        name = names[i % per] if ok else (TRACE_NAMES.get(k) or f"gemm_epi{(k - 100) // 2}")
        exposed = max(0, b - prev_end)
        if per <= i < 2 * per:                  # the second replay, launch by launch
            timeline.append({"launch": name, "ctas": n,
                             "first_start_us": round((a - groups[per][1]) / 1e3, 2),
                             "end_us": round((b - groups[per][1]) / 1e3, 2),
                             "after_previous_us": round(exposed / 1e3, 2)})
        prev_end = max(prev_end, b)
        e = agg.setdefault(name, [0, 0.0, 0.0, 0])
        e[0] += 1
        e[1] += (b - max(a, b - exposed)) / 1e3
        e[2] += exposed / 1e3
        e[3] = n
        crit_total += exposed / 1e3
    span = (groups[-1][2] - groups[0][1]) / 1e3 / rounds
    # Points inside the kernels (trace marks): each belongs to the first launch of its kernel
    # family that ends at or after it; reported as us after the end of the launch before that
    # one (median over CTAs and launches, and the median over launches of the last CTA's).
    phases = {}
    for fam, sel in (("attn", lambda k: k == 6), ("gemm", lambda k: k >= 100)):
        gi = [i for i, g_ in enumerate(groups) if sel(g_[0]) and i > 0]
        if not gi:
            continue
        ends = np.array([groups[i][2] for i in gi], dtype=np.int64)
        for ph in sorted(set(mk.tolist())):
            if (ph in GEMM_MARKS) != (fam == "gemm"):
                continue
            t = mt[mk == ph]
            j = np.searchsorted(ends, t, side="left")
            ok_ = j < len(gi)
            t, j = t[ok_], j[ok_]
            rel = {}
            for tt, jj in zip(t.tolist(), j.tolist()):
                i = gi[jj]
                name = names[i % per] if ok else fam
                rel.setdefault(name, {}).setdefault(i, []).append((tt - groups[i - 1][2]) / 1e3)
            for name, per_launch in rel.items():
                allv = [v for vs in per_launch.values() for v in vs]
                phases.setdefault(name, {})[str(ph)] = {
                    "median_us": round(float(np.median(allv)), 2),
                    "last_cta_us": round(float(np.median([max(vs) for vs in per_launch.values()])), 2)}
    table = {k: {"launches_per_round": v[0] // rounds, "span_us_each": round(v[1] / v[0], 2),
                 "critical_us_per_round": round(v[2] / rounds, 2), "ctas": v[3]}
             for k, v in sorted(agg.items(), key=lambda kv: -kv[1][2])}
    print(json.dumps({"profile_case": "trace", "workload": s.name, "batch": Bn, "ctx": s.ctx,
                      "rounds": rounds, "launches_per_round": per, "grouped_ok": ok,
                      "round_us": round(span, 1),
                      "critical_us_per_round": round(crit_total / rounds, 1), "kernels": table,
                      "phases_after_previous_launch": phases, "timeline": timeline}))


def profile_case(args):
    """A small, self-contained case for ncu: the full-size lm_head argmax (1.48 GB of weights,
    larger than L2) over the 16 block rows, 2 warm-up launches then 3 profiled ones; or one
    eager round of the workload."""
    if args.profile_case == "trace":              # loads the trace build: before the binding
        return trace_case(args)
    import torch

    from speculative_decoding_drafter_dflash_gb300 import binding as B
    from speculative_decoding_drafter_dflash_gb300.workloads import DFLASH_K15
    s = DFLASH_K15
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)
    if args.profile_case == "sweep":
        return sweep_case(args.steps)
    if args.profile_case == "sweep_bf16kv":
        return sweep_case(args.steps, kv_bf16=True)
    if args.profile_case == "mtp":
        return mtp_case(args.steps)
    if args.profile_case == "moe":
        return moe_case(args.steps)
    if args.profile_case == "attn":
        return attn_case(args.steps)
    if args.profile_case == "stochastic":
        return stochastic_case(args.steps)
    if args.profile_case == "generate":
        return generate_case(args.steps)
    if args.profile_case == "sampled":
        return sampled_case(args.steps)
    if args.profile_case == "layout":
        return layout_case(args)
    if args.profile_case == "lm_head":
        V = args.vocab or s.vocab
        rows = s.block * max(1, args.batch)          # --batch 8: the 128 rows of 8 sequences
        W = (torch.randn((V, s.hidden), generator=g, device=dev) * s.w_std).to(torch.bfloat16)
        X = torch.randn((rows, s.hidden), generator=g, device=dev)
        idx = torch.empty(rows, dtype=torch.int32, device=dev)
        ws = B.alloc_workspace(B.lm_head_workspace_bytes(rows, s.hidden, V), dev)
        Wt = B.TiledMatrix(W)          # the round reads the lm_head from its tiled copy
        for _ in range(5):
            B.lm_head_argmax_tiled(Wt, X, idx, ws=ws)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": "lm_head", "idx0": int(idx[0])}))
    elif args.profile_case == "gemms":
        # Every projection shape of one drafter layer (+ fc) timed alone with CUDA events, for
        # --batch sequences of 16 block rows (the QKV shape adds as many context rows); the
        # lm_head shape only at batch 1. --steps timed calls per shape after 3 warm-up calls.
        H, I, qt, kt = s.hidden, s.intermediate, s.q_total, s.kv_total
        b = max(1, args.batch)
        shapes = [("fc", 16 * b, H, s.fc_in), ("qkv", 32 * b, qt + 2 * kt, H), ("o", 16 * b, H, qt),
                  ("gate_up", 16 * b, 2 * I, H), ("down", 16 * b, H, I)]
        if b == 1:
            shapes.append(("lm_head_store", 16, s.vocab, H))
        res = {}
        for name, T, N, K in shapes:
            W = (torch.randn((N, K), generator=g, device=dev) * s.w_std).to(torch.bfloat16)
            X = torch.randn((T, K), generator=g, device=dev)
            Y = torch.empty((T, N), device=dev)
            ws = B.alloc_workspace(B.linear_workspace_bytes(T, N, K), dev)
            for _ in range(3):
                B.df_linear(W, X, Y, ws)
            evs = []
            for _ in range(max(1, min(args.steps, 20))):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                B.df_linear(W, X, Y, ws)
                e1.record()
                evs.append((e0, e1))
            torch.cuda.synchronize()
            us = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
            res[name] = {"T": T, "N": N, "K": K, "us": round(us, 2),
                         "weight_gbs": round(N * K * 2 / us / 1e3, 1)}
            del W, X, Y, ws
        print(json.dumps({"profile_case": "gemms", "sm_count": torch.cuda.get_device_properties(dev).multi_processor_count, **res}))
    else:
        # Per-kernel GPU time inside eager rounds of the workload (library event profiler);
        # --layers and --vocab shrink the model for captures that replay every kernel.
        from speculative_decoding_drafter_dflash_gb300 import synth
        s = s.with_(batch=args.batch, ctx=args.ctx or s.ctx, n_layers=args.layers or s.n_layers,
                    vocab=args.vocab or s.vocab)
        Bn = s.batch
        acc, n_new = variants(s)
        nmax = s.block
        w = synth.dflash_weights(s, seed=0, device=dev)
        cache = synth.dflash_cache(s, seed=1, device=dev)
        model = B.DFlashModel(s, w, cache)
        ws = B.alloc_workspace(model.workspace_bytes(Bn, s.block, nmax), dev)
        out = B.RoundOutputs(Bn, s.K, dev)
        eos = torch.tensor(s.eos_ids, dtype=torch.int32, device=dev)
        tsl = torch.full((Bn,), 1 << 30, dtype=torch.int32, device=dev)
        tgt = torch.zeros((Bn, s.block), dtype=torch.int32, device=dev)
        inputs = []
        for v in range(N_VARIANTS):
            inp = synth.dflash_round_inputs(s, [nmax] * Bn, seed=10 + v, device=dev)
            inp.n_new = torch.tensor([n_new[(v + b) % N_VARIANTS] for b in range(Bn)],
                                     dtype=torch.int32, device=dev)
            inputs.append(inp)

        def one(v):
            inp = inputs[v]
            B.df_draft_round(model, inp.last_token, inp.target_hidden, inp.n_new, nmax, s.K, tgt,
                             eos, tsl, out, ws)
            B.kv_rollback(cache.seq_len, inp.n_new)

        for v in range(3):
            one(v)
        torch.cuda.synchronize()
        rounds = 8
        B.profile_enable(True)
        for i in range(rounds):
            one(i % N_VARIANTS)
        rec = B.profile_read()
        B.profile_enable(False)
        agg = {}
        for name, us in rec:
            a = agg.setdefault(name, [0, 0.0])
            a[0] += 1
            a[1] += us
        total = sum(v[1] for v in agg.values()) / rounds
        table = {k: {"per_round": v[0] // rounds, "us_per_round": round(v[1] / rounds, 2),
                     "us_each": round(v[1] / v[0], 2), "share": round(v[1] / rounds / total, 4)}
                 for k, v in sorted(agg.items(), key=lambda kv: -kv[1][1])}
        print(json.dumps({"profile_case": "round", "rounds": rounds,
                          "kernel_us_per_round": round(total, 1), "kernels": table}))


def main():
    args = parse()
    if args.profile_case:
        profile_case(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            res = run_reference(args, rank, world)
        else:
            res = run_native(args, rank, world, local_rank)
        if res is not None:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
