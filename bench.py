"""Benchmark: layer-skip self-speculative greedy rounds on the 7B-shaped model.

Workload (one step = one whole round of the verification path):
  7B-shaped Llama decoder (32 layers, d 4096, 32 heads x 128, FFN 11008,
  vocab 32000), bf16 random-init N(0, 0.02) weights (13.5 GB), draft = first
  12 layers + LM head, verify = layers 12..31 reusing the draft's KV, chain
  k = 4, committed context 4096 per sequence (a seeded synthetic KV context,
  standing in for a prefilled random prompt), greedy acceptance, batch 1 (or
  --batch 8).  A round = spec_draft (k+1 first-12-layer passes, k LM heads) +
  spec_verify (layers 12..31 over k+1 rows, LM head, fused greedy acceptance)
  + kv_commit; the next round starts from the emitted token.

Metric: verified candidate tokens/s (k+1 per sequence per round, over the
whole round time) -- with accepted tokens/s, the verify-step-only rate and the
HBM roofline fraction of the dominant kernel (the tcgen05 GEMM) alongside.
Weights and KV (> L2) are re-streamed every round, so no L2 flush is needed.

--tree 4,2,2 runs greedy layer-skip tree rounds instead of chains: the draft
grows a 29-node token tree level by level (spec_draft_tree), verify runs
layers 12..31 over all nodes with the tree mask and fused greedy tree
acceptance, kv_commit compacts the accepted path.

--tree 4,2,2 --tree-mass 0.8 makes the tree's width follow the draft's
confidence (spec_draft_tree_dynamic): a node gets the fewest of its best draft
tokens whose draft probability reaches the mass, at most the level's
branching, one tree a sequence; the node counts are read back and
spec_verify_trees verifies each sequence's own tree.

--page 64 keeps the KV cache in 64-slot pages (page tables, pages taken before
each write and returned past the committed length at every commit).

--mode sample runs sampling rounds instead: draft tokens drawn from
softmax(draft logits / 0.8) with seeded uniforms (spec_draft_sample), target
rows at the same temperature cut to their top-p 0.9 nucleus (spec_probs),
rejection sampling (spec_accept) and kv_commit.

python bench.py [--gpus N] [--steps K] [--warmup W] [--batch B] [--mode greedy|sample] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified candidate tokens/s and accepted tokens/s @1 GB300; % HBM roofline"
WORKLOAD = "llama7b-shape layer-skip self-spec (draft 12/32 layers), chain k=4, ctx 4096, greedy"
K_DRAFT, CTX, SEED = 4, 4096, 4
TEMP, TOP_P = 0.8, 15099494 * 2.0 ** -24        # top-p 0.9 rounded down to a multiple of 2^-24


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--single-thread-sample", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--no-subs", action="store_true",
                    help="default run only: skip the sub-records of the other configurations")
    ap.add_argument("--layers", type=int, default=None,
                    help="fewer layers of the same shape (small case for profiler captures)")
    ap.add_argument("--exit-layer", type=int, default=None)
    ap.add_argument("--mode", default="greedy", choices=["greedy", "sample"],
                    help="chain workload: greedy acceptance, or sampling at temperature 0.8 with top-p 0.9")
    ap.add_argument("--page", type=int, default=0,
                    help="paged KV cache with pages of this many slots (a power of two, at least 64); 0: contiguous")
    ap.add_argument("--tree", default=None,
                    help="greedy layer-skip token tree instead of the chain, e.g. 4,2,2 (children per node by level)")
    ap.add_argument("--tree-mass", type=float, default=None,
                    help="with --tree: dynamic width, children of a node = its fewest best draft tokens whose "
                         "draft probability reaches this mass (at most the level's branching)")
    ap.add_argument("--workload", default="chain", choices=["chain", "adaptive", "tiny", "accept", "tree8"],
                    help="chain: k=4, ctx 4096, batch 1 (or --batch); adaptive: batch 32, contexts 512..8192, "
                         "per-sequence k in [2,16] from the confidence schedule")
    return ap.parse_args()


GEMM_SOURCES = ("gemm.cu", "attn_phase.cuh", "common.cuh", "model.cuh", "stats.cuh")


def gemm_source_sha256():
    """Hash of the sources the chain GEMM kernel is compiled from."""
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "speculative_decoding_verify_04_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def gemm_traffic_per_launch(avg_launch_bytes):
    """DRAM bytes of the average GEMM-chain launch of a round: the committed ncu
    summary (profiles/gemm_tc_kernel.llama7b_shapes.md) gives DRAM bytes over
    algorithmic bytes for the captured launches, applied to this run's average
    algorithmic bytes per launch (the launches move weights in proportion).
    None if the summary is absent or was taken on other kernel sources."""
    p = os.path.join(ROOT, "profiles", "gemm_tc_kernel.llama7b_shapes.md")
    if not os.path.exists(p):
        return None
    fields = {}
    for line in open(p):
        if ":" in line and line.split(":")[0] in ("traffic_over_algorithmic", "gemm_sources_sha256"):
            k, v = line.split(":", 1)
            fields[k] = v.strip()
    if fields.get("gemm_sources_sha256") != gemm_source_sha256() or "traffic_over_algorithmic" not in fields:
        return None
    return float(fields["traffic_over_algorithmic"]) * avg_launch_bytes


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle timing (sampled round, scaled)
class OracleRoundSample:
    """The float64 oracle on a bounded sample of one round, scaled to the round.

    Sample: one decoder layer of the 7B shape with 1 row (a draft pass) and
    with k+1 rows (a verify pass) over a ``ctx``-token context, and the LM head
    with 1 and k+1 rows.  A round is 5 x 12 one-row layer passes + 4 one-row
    heads + 20 (k+1)-row layer passes + one (k+1)-row head per sequence.  The
    weights and the context are built once; every ``run`` times the sample.
    """

    def __init__(self, k=K_DRAFT, ctx=CTX):
        import numpy as np
        import dataclasses
        from synthetic import SHAPES, make_weights, weights_to_numpy, make_kv_context
        from oracle.decoder import Decoder
        self.k, self.ctx = k, ctx
        self.shape = dataclasses.replace(SHAPES["llama7b"], n_layers=1, exit_layer=0)
        self.dec = Decoder(self.shape, weights_to_numpy(make_weights(self.shape, SEED, device="cpu")))
        kc, vc = make_kv_context(self.shape, 1, ctx, SEED, device="cpu")
        self.cache = self.dec.new_cache(ctx + k + 2)
        self.cache.load(kc[:, 0].float().numpy(), vc[:, 0].float().numpy())
        self.rng = np.random.default_rng(0)

    def _layer(self, rows):
        import numpy as np
        h = self.rng.standard_normal((rows, self.shape.d_model)) * 0.02
        pos = self.ctx + np.arange(rows)
        vis = [np.arange(self.ctx + r + 1) for r in range(rows)]
        t = time.perf_counter()
        self.dec.layer(0, h, pos, pos, vis, self.cache)
        return time.perf_counter() - t

    def _head(self, rows):
        h = self.rng.standard_normal((rows, self.shape.d_model))
        t = time.perf_counter()
        self.dec.logits(h)
        return time.perf_counter() - t

    def run(self, batch):
        """(seconds per round for ``batch`` sequences, sample description, threads)."""
        import torch
        k = self.k
        t1, t5, h1, h5 = self._layer(1), self._layer(k + 1), self._head(1), self._head(k + 1)
        per_seq = (k + 1) * 12 * t1 + k * h1 + 20 * t5 + h5
        threads = torch.get_num_threads()
        try:
            import threadpoolctl
            info = threadpoolctl.threadpool_info()
            threads = max([i.get("num_threads", 1) for i in info] + [1])
        except Exception:
            pass
        desc = (f"one 7B-shape layer at 1 and {k + 1} rows and the LM head at 1 and {k + 1} rows "
                f"over a {self.ctx}-token context, scaled to a round ({k + 1}x12 + 20 layer passes, {k + 1} heads)")
        return per_seq * batch, desc, threads


def oracle_round_sample(batch, k=K_DRAFT, ctx=CTX):
    return OracleRoundSample(k, ctx).run(batch)


class OracleVerifySample(OracleRoundSample):
    """The oracle's verify step on a bounded sample: one 7B-shape layer and the
    LM head at k+1 rows over a ``ctx``-token context, scaled to the 20 layers
    and the head of a verify step."""

    def run(self, batch):
        k = self.k
        t, h = self._layer(k + 1), self._head(k + 1)
        per_seq = 20 * t + h
        desc = (f"one 7B-shape layer and the LM head at {k + 1} rows over a {self.ctx}-token context, "
                f"scaled to a verify step (20 layers + head)")
        return per_seq * batch, desc, _blas_threads()


def _blas_threads():
    import torch
    threads = torch.get_num_threads()
    try:
        import threadpoolctl
        threads = max([i.get("num_threads", 1) for i in threadpoolctl.threadpool_info()] + [1])
    except Exception:
        pass
    return threads


class OracleFull:
    """The whole 7B-shaped oracle for the reference arm: all 32 layers (float64
    arithmetic over bf16 weights widened to float32, as the oracle stands), the
    4096-token synthetic context, and one draft's layer-12 states of the k+1
    candidate rows (setup, untimed).  ``verify_step`` runs layers 12..31 over the
    k+1 rows and the LM head, the unit of the metric; ``round`` a whole round
    (draft, verify, greedy acceptance, commit) from a fixed committed length."""

    def __init__(self, k=K_DRAFT, ctx=CTX):
        import numpy as np
        from synthetic import SHAPES, make_weights, weights_to_numpy, make_kv_context, make_tokens
        from oracle.decoder import Decoder
        from oracle import spec as OS
        self.k, self.ctx, self.OS = k, ctx, OS
        self.shape = SHAPES["llama7b"]
        w = make_weights(self.shape, SEED, device="cpu")
        self.dec = Decoder(self.shape, weights_to_numpy(w))
        del w
        kc, vc = make_kv_context(self.shape, 1, ctx, SEED * 1000, device="cpu")
        self.cache = self.dec.new_cache(ctx + k + 2)
        self.cache.load(kc[:, 0].float().numpy(), vc[:, 0].float().numpy())
        del kc, vc
        self.t0 = int(make_tokens(1, self.shape.vocab, SEED, "t0")[0])
        _, self.hL, _, _ = OS.draft(self.dec, self.cache, ctx, self.t0, k)
        # the rows' state entering each quarter of the verify layers (for the bounded steps)
        L, N = self.shape.exit_layer, self.shape.n_layers
        self.bounds = [L + (N - L) * q // 4 for q in range(5)]
        T = k + 1
        self.slots = ctx + np.arange(T)
        self.vis = OS.chain_visibility(ctx, T)
        self.h_at = [np.asarray(self.hL, dtype=np.float64)]
        for q in range(3):
            self.h_at.append(self.dec.run_layers(self.h_at[-1], self.bounds[q], self.bounds[q + 1], self.slots,
                                                 self.slots, self.vis, self.cache))

    def verify_step(self):
        t = time.perf_counter()
        self.OS.verify(self.dec, self.cache, self.ctx, self.hL, self.shape.exit_layer)
        return time.perf_counter() - t

    def verify_quarter(self, q):
        """A quarter of the verify step: its share of the layers from the state the
        earlier quarters leave (the fourth quarter adds the LM head)."""
        t = time.perf_counter()
        h = self.dec.run_layers(self.h_at[q], self.bounds[q], self.bounds[q + 1], self.slots, self.slots,
                                self.vis, self.cache)
        if q == 3:
            self.dec.logits(h)
        return time.perf_counter() - t

    def round(self):
        from oracle.accept import accept_greedy_chain, commit_chain
        t = time.perf_counter()
        d, hL, _, _ = self.OS.draft(self.dec, self.cache, self.ctx, self.t0, self.k)
        logits = self.OS.verify(self.dec, self.cache, self.ctx, hL, self.shape.exit_layer)
        a, _ = accept_greedy_chain(d, logits)
        commit_chain(self.ctx, a)                 # the committed length; the cache stays at ctx
        return time.perf_counter() - t


def oracle_tiny_generation():
    """Config 1 in full: the tiny f32 decoder's 64-token greedy speculative generation (seconds)."""
    from synthetic import SHAPES, make_weights, weights_to_numpy, make_tokens
    from oracle.decoder import Decoder
    from oracle import spec as OS
    shape = SHAPES["tiny"]
    dec = Decoder(shape, weights_to_numpy(make_weights(shape, 1, device="cpu")))
    t = time.perf_counter()
    OS.generate_greedy_spec(dec, make_tokens(32, shape.vocab, 1), 64, 4)
    return time.perf_counter() - t


def single_thread_sample():
    """Runs in a child process whose BLAS pool has one thread: the verify-step
    sample (one 7B layer and the head at k+1 rows) and config 1 in full."""
    sec, desc, thr = OracleVerifySample().run(1)
    print(json.dumps({"verify_step_s": sec, "sample": desc, "threads": thr, "tiny_generation_s": oracle_tiny_generation()}))


def run_reference(args):
    """The reference arm: the pages ship no code to install, so the reference is
    the oracle (oracle/, float64 numpy), unchanged, on this machine's host cores.
    One step = one complete verify step of the 7B-shaped configuration (layers
    12..31 over the k+1 candidate rows and the LM head over a 4096-token
    context), the unit of the metric.  Besides: one complete round, config 1 in
    full, and a single-thread run of a bounded sample beside the all-cores one."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if args.single_thread_sample:
        return single_thread_sample()
    cores = os.cpu_count()
    full = OracleFull()
    # bounded steps: step i runs quarter i mod 4 of the verify step (5 of its 20 layers, the
    # fourth with the LM head); the verify step's time is the sum of the quarters' means
    quarters = [[] for _ in range(4)]
    for i in range(args.warmup + args.steps):
        t = full.verify_quarter(i % 4)
        if i >= args.warmup:
            quarters[i % 4].append(t)
    for q in range(4):            # every quarter timed at least once
        if not quarters[q]:
            quarters[q].append(full.verify_quarter(q))
    per_step = sum(statistics.mean(x) for x in quarters)
    val = (K_DRAFT + 1) / per_step
    whole_verify_s = full.verify_step()
    round_s = full.round()
    del full
    tiny_all = oracle_tiny_generation()
    sample_all = OracleVerifySample().run(1)[0]
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    one = None
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--impl", "reference",
                            "--single-thread-sample"], env=env, capture_output=True, text=True, timeout=600)
        one = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as exc:          # reported, not fatal: the all-cores figures stand
        one = {"error": str(exc)[:200]}
    threads = _blas_threads()
    line = {
        "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": 0, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded random weights and KV context)",
        "config": {"workload": WORKLOAD, "batch": 1, "k": K_DRAFT, "ctx": CTX, "value": VALUE_DEF},
        "impl": "reference",
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": "the 7B-shaped verify step (layers 12..31 and the LM head over 5 rows, context "
                                   "4096): each timed step runs one quarter of it (5 layers, the fourth with the "
                                   "head), cycling; ms_per_step is the sum of the quarters' means",
                         "nproc": cores},
        "oracle_verify_step_whole_s": whole_verify_s,
        "oracle_round_s": round_s,
        "oracle_round_candidate_tokens_per_s": (K_DRAFT + 1) / round_s,
        "oracle_tiny_generation_s": tiny_all,
        "oracle_tiny_accepted_tokens_per_s": 64 / tiny_all,
        "single_thread_vs_all_cores": {
            "sample": "one 7B-shape layer and the LM head at 5 rows over a 4096-token context, scaled to a verify "
                      "step; and config 1's 64-token generation",
            "all_cores": {"threads": threads, "verify_step_s": sample_all, "tiny_generation_s": tiny_all},
            "one_thread": one},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_max(x, dist, device):
    """Max over ranks of a per-rank float: the job's time is its slowest rank's."""
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, seconds):
    """Whole-job throughput: each of `world` ranks processed `units_per_rank` units
    (independent replicas) within `seconds` (the slowest rank's time)."""
    return world * units_per_rank / seconds


def shard_range(n, world, rank):
    """Sequences [start, stop) of one global batch of ``n`` that rank ``rank`` of
    ``world`` runs: contiguous shares whose sizes differ by at most one, in rank
    order.  The batched workloads draw every input from streams keyed by the
    sequence's index in the global batch, so the shards of all ranks together
    are exactly the undivided batch."""
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


VALUE_DEF = ("verified candidate tokens/s: candidate rows verified per verify step over the verify step's device "
             "time (spec_verify: layers L..N-1 over every candidate row, the LM head and the fused acceptance); "
             "ms_per_step is the whole round (draft, verify, acceptance, commit)")
ADAPTIVE = ("llama7b-shape layer-skip self-spec (draft 12/32 layers), batch 32, contexts U{512..8192}, "
            "per-sequence k in [2,16] from the confidence schedule, greedy")
B_ADAPT, K_MIN, K_MAX, K_START, EMA_START = 32, 2, 16, 2, 0.5


def _timed(step, steps, warm, world, dist, local):
    """Warm-up, then ``steps`` calls of ``step`` between CUDA events on the
    current stream with SM clocks sampled; returns (seconds, clocks)."""
    import torch
    for _ in range(warm):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = Clocks(local)
    clocks.start()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    sec = e0.elapsed_time(e1) / 1e3
    if world > 1:
        sec = reduce_max(sec, dist, "cuda")
    return sec, clk


def _line(args, world, steps, warm, sec, value_units, dtype, config, extra):
    line = {"metric": METRIC, "value": job_rate(world, value_units, sec), "unit": "tokens/s", "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": sec * 1e3 / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic (seeded random-init weights and inputs; no dataset)", "config": config}
    line.update(extra)
    return line


def run_tiny(args, spec, world, rank, local, dist):
    """The tiny fp32 decoder (2 layers, d 256, 4 heads x 64, FFN 1024, vocab
    1024, draft = layer 0 + the LM head): one step = prefill a 32-token prompt,
    then greedy chain rounds of k = 4 until 64 tokens are out.  The host reads
    each round's accepted length (the stopping test): part of the step."""
    import torch
    from synthetic import SHAPES, make_weights, make_tokens
    shape = SHAPES["tiny"]
    k, n_prompt, n_new = 4, 32, 64
    w = make_weights(shape, 1 + rank, device="cuda")
    model = spec.Model(shape, w, max_rows=64, max_batch=1, max_position=256)
    del w
    prompt = torch.from_numpy(make_tokens(n_prompt, shape.vocab, 1 + rank)).cuda()
    cand = torch.empty((1, k + 1), dtype=torch.int32, device="cuda")
    hL = torch.empty((1, k + 1, shape.d_model), dtype=torch.float32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    t0 = torch.empty(1, dtype=torch.int32, device="cuda")
    acc_host = torch.empty(1, dtype=torch.int32).pin_memory()
    log = {"rounds": 0}
    kv = spec.KVCache(model, 1, n_prompt + n_new + k + 8)

    def generate():
        kv.set_lengths([0])
        spec.spec_prefill(model, kv, 0, prompt, None, t0)
        out = 1
        while out < n_new:
            spec.spec_draft(model, kv, t0, k, cand, hL)
            spec.spec_verify(model, kv, [k + 1], cand, k + 1, h_in=hL, h_stride=k + 1, acc_len=acc, next_tok=nxt)
            spec.kv_commit(kv, acc)
            t0.copy_(nxt)
            acc_host.copy_(acc)
            torch.cuda.current_stream().synchronize()
            out += int(acc_host.item()) + 1
            log["rounds"] += 1

    steps, warm = args.steps, args.warmup
    n0 = model.launch_count()
    sec, clk = _timed(generate, steps, warm, world, dist, local)
    rounds = log["rounds"] * steps // (steps + warm)
    launches = (model.launch_count() - n0) * steps // (steps + warm)
    if model.device_error():
        raise SystemExit("device error word set during the bench")
    hbm, peak_kind = peaks()
    d, F, V = shape.d_model, shape.d_ff, shape.vocab
    w_bytes = (shape.n_layers * (4 * d * d + 3 * F * d) + 2 * V * d) * 4
    achieved = rounds * w_bytes / sec / 1e9
    extra = {
        "accepted_tokens_per_s": job_rate(world, n_new * steps, sec),
        "rounds_per_step": rounds / steps,
        "roofline": {"bound": "hbm", "kernel": "whole generation (launch-bound: 10.5 MB of weights a round)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
                     "peak_source": peak_kind},
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": {"value": job_rate(world, n_new * steps, sec), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 4 * rounds // max(steps, 1),
                "note": "the step already reads every round's accepted length back to the host"},
    }
    line = _line(args, world, steps, warm, sec, rounds * (k + 1), "f32",
                 {"workload": "tiny fp32 decoder (2 layers, d 256, vocab 1024), prompt 32, 64 tokens, chain k=4 greedy",
                  "l2": "fits in L2 (launch-bound correctness workload)"}, extra)
    line["value_note"] = "verified candidate tokens/s over the whole generation; accepted_tokens_per_s = 64 per step"
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import spec as OS
        from oracle.decoder import Decoder
        from synthetic import weights_to_numpy
        dec = Decoder(shape, weights_to_numpy(make_weights(shape, 1, device="cpu")))
        tw = time.perf_counter()
        OS.generate_greedy_spec(dec, make_tokens(n_prompt, shape.vocab, 1), n_new, k)
        t = time.perf_counter() - tw
        line["cpu_baseline"] = {"value": n_new / t, "unit": "tokens/s (accepted)", "cores": os.cpu_count(),
                                "kind": "oracle", "sample": "one whole 64-token generation"}
    return line


def run_accept(args, spec, world, rank, local, dist):
    """The acceptance call alone: 256 sequences, k = 5, vocab 32000, p and q
    the softmax of N(0, 9) target logits and of those plus N(0, 1) noise, draft
    tokens drawn from q, one uniform a position plus one for the draw.  One
    step = one spec_accept over resident inputs (360 MB, larger than L2).
    Algorithmic bytes per sequence: the row(s) the draw reads (p_a and q_a
    after a rejection, p_k after k acceptances) plus one 32-byte sector of p
    and of q per ratio test."""
    import numpy as np
    import torch
    from synthetic import make_accept_inputs
    B, k, V = 256, 5, 32000          # sequences per rank; the global batch is world x 256
    first, _ = shard_range(B * world, world, rank)
    p, q, x, u = make_accept_inputs(B, k, V, seed=2, first=first)
    pg, qg = torch.from_numpy(p).cuda(), torch.from_numpy(q).cuda()
    xg, ug = torch.from_numpy(x.astype(np.int32)).cuda(), torch.from_numpy(u).cuda()
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    steps, warm = max(args.steps, 100), args.warmup
    sec, clk = _timed(lambda: spec.spec_accept(pg, qg, xg, ug, acc, nxt), steps, warm, world, dist, local)
    a = acc.cpu().numpy()
    alg = sum((2 if a[b] < k else 1) * V * 4 + 2 * min(int(a[b]) + 1, k) * 32 for b in range(B))
    hbm, peak_kind = peaks()
    achieved = alg / (sec / steps) / 1e9
    # e2e: the inputs copied in from pinned host memory every call, the decisions read back
    ph, qh = torch.from_numpy(p).pin_memory(), torch.from_numpy(q).pin_memory()
    xh, uh = torch.from_numpy(x.astype(np.int32)).pin_memory(), torch.from_numpy(u).pin_memory()
    oh = torch.empty((2, B), dtype=torch.int32).pin_memory()
    e_steps = 10
    torch.cuda.synchronize()
    tw = time.perf_counter()
    for _ in range(e_steps):
        pg.copy_(ph, non_blocking=True)
        qg.copy_(qh, non_blocking=True)
        xg.copy_(xh, non_blocking=True)
        ug.copy_(uh, non_blocking=True)
        spec.spec_accept(pg, qg, xg, ug, acc, nxt)
        oh[0].copy_(acc, non_blocking=True)
        oh[1].copy_(nxt, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - tw) / e_steps
    if world > 1:
        e2e_s = reduce_max(e2e_s, dist, "cuda")
    extra = {
        "sequences_per_s": job_rate(world, B * steps, sec),
        "mean_accepted": float(a.mean()),
        "roofline": {"bound": "hbm", "kernel": "accept_rows_kernel (one CTA of 1024 threads a sequence, two an SM)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
                     "peak_source": peak_kind, "algorithmic_bytes_per_launch": alg,
                     "dense_bytes_per_launch": B * (2 * k + 1) * V * 4},
        "gpu_launches": steps,
        "clocks": clk,
        "e2e": {"value": job_rate(world, B * k, e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": p.nbytes + q.nbytes + x.size * 4 + u.nbytes, "d2h_bytes_per_step": 8 * B},
    }
    line = _line(args, world, steps, warm, sec, B * k * steps, "f32",
                 {"workload": "acceptance alone: batch 256, k=5, vocab 32000, logits N(0,3^2), draft = target + N(0,1)",
                  "l2": "inputs larger than L2 (360 MB of p and q)",
                  "parallelism": "data parallel over sequences (one global batch, sharded)" if world > 1
                  else "single GPU"}, extra)
    line["value_note"] = "draft tokens decided per second"
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import accept as A
        n = 16
        tw = time.perf_counter()
        for b in range(n):
            A.accept_sampling_chain(p[b], q[b], x[b], u[b])
        t = (time.perf_counter() - tw) / n
        line["cpu_baseline"] = {"value": k / t, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} of the 256 sequences, one at a time"}
    return line


def run_tree8(args, spec, world, rank, local, dist):
    """Tree verification: 8-layer bf16 decoder (d 1024, 16 query / 4 KV heads
    x 64, FFN 2816, vocab 32000), a 2048-token random prompt prefilled, a
    29-node token tree [4, 2, 2] in level order, batch 1.  One step = one
    spec_verify over the tree from the embeddings (ancestor-only mask, depth
    positions, fused greedy longest-path acceptance) + kv_commit of the path."""
    import torch
    from synthetic import SHAPES, make_weights, make_tokens, tree_parents
    shape = SHAPES["tree8"]
    ctx = 2048
    par = [int(v) for v in tree_parents([4, 2, 2])]
    n = len(par)
    steps, warm = args.steps, args.warmup
    cap = ctx + (steps + warm + 4) * 4 + 2 * n
    w = make_weights(shape, 3 + rank, device="cuda")
    model = spec.Model(shape, w, max_rows=64, max_batch=1, max_position=cap + 8)
    del w
    kv = spec.KVCache(model, 1, cap)
    spec.spec_prefill(model, kv, 0, torch.from_numpy(make_tokens(ctx, shape.vocab, 3 + rank)).cuda())
    toks = torch.from_numpy(make_tokens(n, shape.vocab, 30 + rank, "tree")).cuda().view(1, n)
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    path = torch.empty((1, 64), dtype=torch.int32, device="cuda")

    def step():
        spec.spec_verify(model, kv, [n], toks, n, tree_parent=par, acc_len=acc, next_tok=nxt, path=path)
        spec.kv_commit(kv, acc, path)

    n0 = model.launch_count()
    sec, clk = _timed(step, steps, warm, world, dist, local)
    launches = (model.launch_count() - n0) * steps // (steps + warm)
    if model.device_error():
        raise SystemExit("device error word set during the bench")
    d, F, V = shape.d_model, shape.d_ff, shape.vocab
    qkv = (shape.n_heads + 2 * shape.n_kv_heads) * shape.head_dim
    w_bytes = shape.n_layers * (qkv * d + d * shape.n_heads * shape.head_dim + 3 * F * d) * 2 + V * d * 2
    kv_bytes = shape.n_layers * 2 * shape.n_kv_heads * shape.head_dim * 2 * (ctx + n)
    hbm, peak_kind = peaks()
    achieved = (w_bytes + kv_bytes) / (sec / steps) / 1e9
    # e2e: the tree's tokens from pinned host memory, the decision read back
    th = toks.cpu().pin_memory()
    oh = torch.empty((1, 66), dtype=torch.int32).pin_memory()
    e_steps = max(3, steps // 2)
    torch.cuda.synchronize()
    tw = time.perf_counter()
    for _ in range(e_steps):
        toks.copy_(th, non_blocking=True)
        step()
        oh[0, :64].copy_(path[0], non_blocking=True)
        oh[0, 64:65].copy_(acc, non_blocking=True)
        oh[0, 65:66].copy_(nxt, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - tw) / e_steps
    if world > 1:
        e2e_s = reduce_max(e2e_s, dist, "cuda")
    extra = {
        "roofline": {"bound": "hbm", "kernel": "whole verification step (GEMM chains + tree attention)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
                     "peak_source": peak_kind, "algorithmic_bytes_per_step": w_bytes + kv_bytes},
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": {"value": job_rate(world, n, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": 4 * n,
                "d2h_bytes_per_step": 4 * 66},
    }
    line = _line(args, world, steps, warm, sec, n * steps, "bf16",
                 {"workload": "tree verification: 8-layer bf16 d1024 GQA 16/4, vocab 32000, ctx 2048, tree [4,2,2]",
                  "l2": "weights 246 MB re-streamed each step (larger than L2)"}, extra)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import spec as OS
        from oracle.decoder import Decoder
        from synthetic import weights_to_numpy
        from synthetic import make_kv_context
        dec = Decoder(shape, weights_to_numpy(make_weights(shape, 3, device="cpu")))
        cache = dec.new_cache(ctx + n + 4)
        kc, vc = make_kv_context(shape, 1, ctx, 3, device="cpu")
        cache.load(kc[:, 0].float().numpy(), vc[:, 0].float().numpy())
        tw = time.perf_counter()
        OS.verify(dec, cache, ctx, dec.embed(toks[0].cpu().numpy()), 0, parents=par)
        t = time.perf_counter() - tw
        line["cpu_baseline"] = {"value": n / t, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": "one tree verification over a 2048-slot synthetic context"}
    return line


def run_adaptive(args, spec, world, rank, local, dist):
    """Adaptive-k rounds: every sequence verifies its own k_b + 1 rows; after
    the fused acceptance, the per-row top-1 / top-2 probabilities feed the
    schedule, which sets each sequence's next k on the device.  The host reads
    the new k back each round (the next call's row counts): that round trip is
    part of the step."""
    import torch
    from synthetic import SHAPES, make_weights, make_kv_context, make_tokens, make_ragged_contexts
    shape = SHAPES["llama7b"]
    B = B_ADAPT
    steps, warm = args.steps, args.warmup
    first, _ = shard_range(B * world, world, rank)
    lens = [int(x) for x in make_ragged_contexts(B * world, 512, 8192, seed=5)[first:first + B]]
    cap = max(lens) + (steps + warm + 2) * (K_MAX + 1) + 8
    w = make_weights(shape, SEED, device="cuda")
    model = spec.Model(shape, w, max_rows=B * (K_MAX + 1), max_batch=B, max_position=cap + 8)
    del w
    torch.cuda.empty_cache()
    kv = spec.KVCache(model, B, cap)
    for b in range(B):
        kc, vc = make_kv_context(shape, 1, lens[b], SEED * 1000 + first + b, device="cuda")
        kv.import_rows(b, 0, kc[:, 0].contiguous(), vc[:, 0].contiguous())
        del kc, vc
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    kv.set_lengths(lens)

    d = shape.d_model
    R = B * (K_MAX + 1)
    t0 = torch.from_numpy(make_tokens(B * world, shape.vocab, SEED, "t0")[first:first + B]).cuda()
    cand_buf = torch.empty(R, dtype=torch.int32, device="cuda")
    hl_buf = torch.empty(R * d, dtype=torch.float32, device="cuda")
    stats = torch.empty((R, 4), dtype=torch.float32, device="cuda")
    probs = torch.empty((R, 2), dtype=torch.float64, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    kn = torch.empty(B, dtype=torch.int32, device="cuda")
    conf = torch.empty(B, dtype=torch.float64, device="cuda")
    ema = torch.full((B,), EMA_START, dtype=torch.float64, device="cuda")
    k_cur = [K_START] * B
    stream = torch.cuda.current_stream()
    log = {"rows": 0, "accepted": 0, "verify_ms": 0.0, "kmax": 0}

    def round_(timed):
        kmax = max(k_cur)
        n_rows = [k + 1 for k in k_cur]
        T = sum(n_rows)
        cand = cand_buf[:B * (kmax + 1)].view(B, kmax + 1)
        hL = hl_buf[:B * (kmax + 1) * d].view(B, kmax + 1, d)
        spec.spec_draft(model, kv, t0, kmax, cand, hL)
        if timed:
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
        spec.spec_verify(model, kv, n_rows, cand, kmax + 1, h_in=hL, h_stride=kmax + 1, stats=stats[:T], acc_len=acc,
                         next_tok=nxt)
        if timed:
            ev1.record(stream)
        spec.spec_row_probs(stats[:T], probs[:T])
        spec.spec_schedule_k(probs[:T], n_rows, acc, ema, kn, conf, min_k=K_MIN, max_k=K_MAX)
        spec.kv_commit(kv, acc)
        t0.copy_(nxt)
        k_next = kn.tolist()                    # the next round's row counts (host)
        if timed:
            log["rows"] += T
            log["accepted"] += int(acc.sum().item()) + B
            log["verify_ms"] += ev0.elapsed_time(ev1)
            log["kmax"] = max(log["kmax"], kmax)
        k_cur[:] = k_next

    for _ in range(warm):
        round_(False)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = Clocks(local)
    clocks.start()
    n_launch0 = model.launch_count()
    torch.cuda.synchronize()
    tw0 = time.perf_counter()
    for _ in range(steps):
        round_(True)
    torch.cuda.synchronize()
    wall_s = time.perf_counter() - tw0
    launches = model.launch_count() - n_launch0
    clk = clocks.stop()
    err = model.device_error()
    if err:
        raise SystemExit(f"device error word {err} set during the bench")
    rows, accepted = log["rows"], log["accepted"]
    verify_s = log["verify_ms"] / 1e3
    model.profile(True)
    for _ in range(min(steps, 5)):
        round_(False)
    torch.cuda.synchronize()
    model.profile(False)
    g_ms, g_bytes, g_n = model.profile_read(0)
    if world > 1:
        wall_s = reduce_max(wall_s, dist, "cuda")
        verify_s = reduce_max(verify_s, dist, "cuda")
    hbm, peak_kind = peaks()
    g_avg_ms = g_ms / max(g_n, 1)
    achieved = g_bytes / max(g_n, 1) / (g_avg_ms / 1e3) / 1e9 if g_n else None
    # verify algorithmic bytes over the timed rounds: layers 12..31 + head weights per round, KV of layers 12..31
    F, V = shape.d_ff, shape.vocab
    layer_w = (4 * d * d + 3 * F * d) * 2
    n_ver = shape.n_layers - shape.exit_layer
    mean_ctx = sum(lens) / B + (steps + warm) * 0.5 * (K_START + 1)
    verify_bytes = steps * (n_ver * layer_w + V * d * 2) + n_ver * 2 * shape.n_kv_heads * shape.head_dim * 2 * mean_ctx * B * steps
    line = {
        "metric": METRIC,
        "value": job_rate(world, rows, verify_s),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warm,
        "ms_per_step": wall_s * 1e3 / steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded random-init weights and KV contexts; no dataset)",
        "config": {"workload": ADAPTIVE, "batch": B, "global_batch": B * world, "k_range": [K_MIN, K_MAX],
                   "ctx_range": [512, 8192], "value": VALUE_DEF,
                   "ctx_mean": sum(lens) / B, "exit_layer": shape.exit_layer, "n_layers": shape.n_layers,
                   "l2": "inputs larger than L2 (weights and ~45 GB of KV re-streamed each round)",
                   "parallelism": "data parallel over sequences" if world > 1 else "single GPU"},
        "round_candidate_tokens_per_s": job_rate(world, rows, wall_s),
        "accepted_tokens_per_s": job_rate(world, accepted, wall_s),
        "rows_per_round": rows / steps,
        "max_k_seen": log["kmax"],
        "verify_ms": verify_s * 1e3 / steps,
        "verify_bytes": verify_bytes / steps,
        "verify_candidate_tokens_per_s": job_rate(world, rows, verify_s),
        "verify_hbm_gbs": verify_bytes / verify_s / 1e9,
        "verify_hbm_frac": verify_bytes / verify_s / 1e9 / hbm,
        "roofline": {"bound": "hbm", "kernel": "gemm_tc_kernel (every launch of an instrumented pass of 5 rounds)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": (achieved / hbm) if achieved else None,
                     "traffic": None, "peak_source": peak_kind, "launches": g_n, "avg_launch_us": g_avg_ms * 1e3},
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": {"value": job_rate(world, rows, wall_s), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 4 * B,
                "note": "the timed rounds already read each round's k back to the host (the next call's row counts)"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        kbar = max(1, round(rows / steps / B) - 1)
        sec, desc, thr = oracle_round_sample(B, k=kbar, ctx=int(sum(lens) / B))
        line["cpu_baseline"] = {"value": B * (kbar + 1) / sec, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                                "sample": desc}
    return line


def run_chain(args, spec, world, rank, local, dist, batch=None):
    """The benchmark's main workload: layer-skip greedy (or sampling, tree) rounds
    on the 7B-shaped model at context 4096, ``batch`` (default ``--batch``)
    sequences a rank.  Returns the JSON line."""
    import torch
    from synthetic import SHAPES, make_weights, make_kv_context, make_tokens, make_uniforms
    import dataclasses
    shape = SHAPES["llama7b"]
    if args.layers is not None:
        shape = dataclasses.replace(shape, n_layers=args.layers,
                                    exit_layer=args.exit_layer if args.exit_layer is not None else args.layers // 2)
    B, k = (batch or args.batch), K_DRAFT
    first, _ = shard_range(B * world, world, rank)
    steps, warm = args.steps, args.warmup
    tree_arg = [int(x) for x in args.tree.split(",")] if args.tree else None
    n_cand = 1 + sum(math.prod(tree_arg[:i + 1]) for i in range(len(tree_arg))) if tree_arg else k + 1
    per_round = len(tree_arg) + 1 if tree_arg else k + 1         # most tokens a round commits
    rounds_total = warm + 2 * steps + max(3, steps // 2) + 1
    grow = rounds_total * per_round + n_cand + 8
    w = make_weights(shape, SEED, device="cuda")
    model = spec.Model(shape, w, max_rows=max(64, B * n_cand), max_batch=B, max_position=CTX + grow + 64)
    del w
    torch.cuda.empty_cache()
    kv = spec.KVCache(model, B, CTX + grow, page=args.page or None)
    for b in range(B):
        kc, vc = make_kv_context(shape, 1, CTX, SEED * 1000 + first + b, device="cuda")
        kv.import_rows(b, 0, kc[:, 0].contiguous(), vc[:, 0].contiguous())
        del kc, vc
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    kv.set_lengths([CTX] * B)

    t0 = torch.from_numpy(make_tokens(B * world, shape.vocab, SEED, "t0")[first:first + B]).cuda()
    cand = torch.empty((B, k + 1), dtype=torch.int32, device="cuda")
    hL = torch.empty((B, k + 1, shape.d_model), dtype=torch.float32, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    ev_v0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev_v1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    acc_log = torch.zeros((steps, B), dtype=torch.int32, device="cuda")
    tree = None
    if args.tree:
        from synthetic import tree_parents
        tree = [int(x) for x in tree_parents([int(x) for x in args.tree.split(",")])]
        if args.mode != "greedy":
            raise SystemExit("--tree takes greedy acceptance")
    assert n_cand == (len(tree) if tree else k + 1)
    if tree:
        tokens_t = torch.empty((B, n_cand), dtype=torch.int32, device="cuda")
        hL = torch.empty((B, n_cand, shape.d_model), dtype=torch.float32, device="cuda")
        tree_scratch = torch.empty((B * n_cand, shape.vocab), dtype=torch.float32, device="cuda")
        path = torch.empty((B, 64), dtype=torch.int32, device="cuda")
    dynamic = args.tree_mass is not None
    if dynamic:
        if not tree:
            raise SystemExit("--tree-mass needs --tree")
        parents_t = torch.empty((B, n_cand), dtype=torch.int32, device="cuda")
        n_nodes_t = torch.empty(B, dtype=torch.int32, device="cuda")
    nodes_log = []
    sampling = args.mode == "sample"
    V = shape.vocab
    if sampling:
        # every round's uniforms, resident before the timed region
        n_rounds = warm + 2 * steps + 1
        u_draft = torch.from_numpy(make_uniforms((n_rounds, B, k), SEED + rank, "u_draft")).cuda()
        u_acc = torch.from_numpy(make_uniforms((n_rounds, B, k + 1), SEED + rank, "u_accept")).cuda()
        q = torch.empty((B, k, V), dtype=torch.float32, device="cuda")
        logits = torch.empty((B * (k + 1), V), dtype=torch.float32, device="cuda")
        p = torch.empty_like(logits)
    rnd = [0]

    def draft(ud=None):
        if dynamic:
            spec.spec_draft_tree_dynamic(model, kv, t0, tree_arg, args.tree_mass, tokens_t, parents_t, n_nodes_t, hL,
                                         tree_scratch)
            return n_nodes_t.tolist()          # the node counts size the verify call (host)
        if tree:
            spec.spec_draft_tree(model, kv, t0, tree, tokens_t, hL, tree_scratch)
        elif sampling:
            spec.spec_draft_sample(model, kv, t0, k, TEMP, ud, cand, hL, q)
        else:
            spec.spec_draft(model, kv, t0, k, cand, hL)

    def verify(ua=None, n_host=None):
        if dynamic:
            spec.spec_verify_trees(model, kv, n_host, tokens_t, n_cand, parents_t, n_cand, h_in=hL, h_stride=n_cand,
                                   acc_len=acc, next_tok=nxt, path=path)
        elif tree:
            spec.spec_verify(model, kv, [n_cand] * B, tokens_t, n_cand, h_in=hL, h_stride=n_cand, tree_parent=tree,
                             acc_len=acc, next_tok=nxt, path=path)
        elif sampling:
            spec.spec_verify(model, kv, [k + 1] * B, cand, k + 1, h_in=hL, h_stride=k + 1, logits=logits)
            spec.spec_probs(logits, p, TEMP, TOP_P)
            spec.spec_accept(p.view(B, k + 1, V), q, cand[:, 1:], ua, acc, nxt)
        else:
            spec.spec_verify(model, kv, [k + 1] * B, cand, k + 1, h_in=hL, h_stride=k + 1, acc_len=acc,
                             next_tok=nxt)

    def step(i=None):
        j = rnd[0]
        rnd[0] += 1
        n_host = draft(u_draft[j] if sampling else None)
        if i is not None:
            ev_v0[i].record(stream)
            if dynamic:
                nodes_log.append(sum(n_host))
        verify(u_acc[j] if sampling else None, n_host)
        if i is not None:
            ev_v1[i].record(stream)
            acc_log[i].copy_(acc)
        spec.kv_commit(kv, acc, path if tree else None)
        t0.copy_(nxt)

    for _ in range(warm):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = Clocks(local)
    clocks.start()
    n_launch0 = model.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    launches = model.launch_count() - n_launch0
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    verify_ms = sum(ev_v0[i].elapsed_time(ev_v1[i]) for i in range(steps)) / steps
    accepted = int(acc_log.sum().item())
    # Instrumented pass of the same rounds: CUDA events around every GEMM and
    # attention launch (on the library's stream) give the per-launch durations
    # of the roofline.  Kept out of the timed region above because events
    # between kernels stop consecutive kernels from overlapping.
    model.profile(True)
    for i in range(steps):
        step()
    torch.cuda.synchronize()
    model.profile(False)
    g_ms, g_bytes, g_n = model.profile_read(0)
    a_ms, _, a_n = model.profile_read(1)
    err = model.device_error()
    if err:
        raise SystemExit(f"device error word {err} set during the bench")
    if world > 1:
        ms = reduce_max(ms, dist, "cuda")
        verify_ms = reduce_max(verify_ms, dist, "cuda")

    # e2e: the same rounds through the public API with the round's inputs (t0,
    # and in sampling mode its uniforms) copied in from pinned host memory and
    # its result read back each step
    t0_host = torch.empty(B, dtype=torch.int32).pin_memory()
    res_host = torch.empty((B, n_cand + 2), dtype=torch.int32).pin_memory()
    t0_host.copy_(t0.cpu())
    res_dev = torch.empty((B, n_cand + 2), dtype=torch.int32, device="cuda")
    e_steps = max(3, steps // 2)
    h2d = 4 * B
    if sampling:
        ud_host = make_uniforms((e_steps, B, k), SEED + rank, "u_draft_e2e")
        ua_host = make_uniforms((e_steps, B, k + 1), SEED + rank, "u_accept_e2e")
        ud_host, ua_host = torch.from_numpy(ud_host).pin_memory(), torch.from_numpy(ua_host).pin_memory()
        ud_dev, ua_dev = torch.empty_like(u_draft[0]), torch.empty_like(u_acc[0])
        h2d += 4 * B * k + 4 * B * (k + 1)
    torch.cuda.synchronize()
    e2e_cand = 0
    tw0 = time.perf_counter()
    for e in range(e_steps):
        t0.copy_(t0_host, non_blocking=True)
        if sampling:
            ud_dev.copy_(ud_host[e], non_blocking=True)
            ua_dev.copy_(ua_host[e], non_blocking=True)
        n_host = draft(ud_dev if sampling else None)
        e2e_cand += sum(n_host) if dynamic else B * n_cand
        verify(ua_dev if sampling else None, n_host)
        spec.kv_commit(kv, acc, path if tree else None)
        res_dev[:, :n_cand].copy_(tokens_t if tree else cand)
        res_dev[:, n_cand].copy_(acc)
        res_dev[:, n_cand + 1].copy_(nxt)
        res_host.copy_(res_dev, non_blocking=True)
        torch.cuda.synchronize()
        t0_host.copy_(res_host[:, n_cand + 1])
    e2e_s = (time.perf_counter() - tw0) / e_steps
    if world > 1:
        e2e_s = reduce_max(e2e_s, dist, "cuda")
    e2e_val = job_rate(world, e2e_cand / e_steps, e2e_s)

    hbm, peak_kind = peaks()
    # candidate rows verified a round: the full tree, or the dynamic trees' node counts
    cand_per_step = B * n_cand if not dynamic else sum(nodes_log) / len(nodes_log)
    value = job_rate(world, cand_per_step, verify_ms / 1e3)
    g_avg_ms = g_ms / max(g_n, 1)
    g_avg_bytes = g_bytes / max(g_n, 1)
    achieved = g_avg_bytes / (g_avg_ms / 1e3) / 1e9 if g_n else None
    # verify step algorithmic bytes: layers 12..31 + LM head weights + KV of layers 12..31 read once
    d, F, V = shape.d_model, shape.d_ff, shape.vocab
    layer_w = (3 * d * d + d * d + 2 * F * d + d * F) * 2
    n_ver = shape.n_layers - shape.exit_layer
    kv_bytes = n_ver * 2 * shape.n_kv_heads * shape.head_dim * 2 * (CTX + k + 1) * B
    verify_bytes = n_ver * layer_w + V * d * 2 + kv_bytes
    workload = WORKLOAD if not sampling else WORKLOAD.replace(
        "greedy", f"sampling (T {TEMP}, top-p {TOP_P:.7g}, rejection sampling)")
    if tree:
        workload = WORKLOAD.replace("chain k=4", f"token tree {args.tree} ({n_cand} nodes, layer-skip draft)")
    if dynamic:
        workload = WORKLOAD.replace("chain k=4", f"token tree up to {args.tree} ({n_cand} nodes) of dynamic width "
                                                 f"(confidence mass {args.tree_mass:g}), layer-skip draft")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warm,
        "ms_per_step": ms / steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded random-init weights and KV context; no dataset)",
        "config": {"workload": workload if args.layers is None else workload + f" (reduced: {shape.n_layers} layers)",
                   "value": VALUE_DEF,
                   "mode": args.mode,
                   "batch": B, "global_batch": B * world, "k": k if not tree else None, "tree": args.tree, "tree_mass": args.tree_mass,
                   "ctx": CTX,
                   "kv": f"paged, {args.page}-slot pages" if args.page else "contiguous", "exit_layer": shape.exit_layer, "n_layers": shape.n_layers,
                   "l2": "inputs larger than L2 (13.5 GB weights re-streamed each round)",
                   "parallelism": ("replicas (one sequence a rank)" if B == 1 else
                                   "data parallel over sequences (one global batch, sharded)") if world > 1
                   else "single GPU"},
        "round_candidate_tokens_per_s": job_rate(world, cand_per_step * steps, ms / 1e3),
        "accepted_tokens_per_s": world * (accepted + B * steps) / (ms / 1e3),
        "acceptance_rate": accepted / (B * steps * (per_round - 1)),
        "verify_ms": verify_ms,
        "verify_bytes": verify_bytes,
        "verify_candidate_tokens_per_s": world * cand_per_step / (verify_ms / 1e3),
        "verify_hbm_gbs": verify_bytes / (verify_ms / 1e3) / 1e9,
        "verify_hbm_frac": verify_bytes / (verify_ms / 1e3) / 1e9 / hbm,
        "roofline": {"bound": "hbm",
                     "kernel": "gemm_tc_kernel (tcgen05 skinny GEMM; every launch of an instrumented pass of the "
                               "same rounds)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": (achieved / hbm) if achieved else None,
                     "traffic": gemm_traffic_per_launch(g_avg_bytes) if args.layers is None and B == 1 else None,
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum over algorithmic bytes of "
                                       "the captured chain launches (profiles/gemm_tc_kernel.llama7b_shapes.md) "
                                       "times this run's algorithmic bytes per launch",
                     "peak_source": peak_kind, "launches": g_n, "avg_launch_us": g_avg_ms * 1e3,
                     "avg_launch_bytes": g_avg_bytes},
        "attention": {"launches": a_n, "total_ms_per_step": a_ms / steps},
        "mean_tree_nodes": (sum(nodes_log) / len(nodes_log) / B) if dynamic else None,
        "pdl": os.environ.get("SPEC_PDL", "1") != "0",
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": 4 * B * (n_cand + 2 + (1 if dynamic else 0)),
                "note": "candidate tokens over whole rounds through the public API, the round's inputs copied in "
                        "from pinned host memory and its tokens read back every round"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sec, desc, thr = OracleVerifySample().run(B)
        line["cpu_baseline"] = {"value": cand_per_step / sec, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                                "sample": desc}
    return line




SUBS = (("llama7b_chain_k4_ctx4096_batch8", "chain8"), ("llama7b_adaptive_k_batch32_ctx512_8192", "adaptive"),
        ("accept_batch256_k5_vocab32000", "accept"), ("tree8_d1024_ctx2048_tree422", "tree8"),
        ("tiny_fp32_64_tokens", "tiny"))
SUB_KEYS = ("value", "unit", "steps", "warmup", "ms_per_step", "higher_is_better", "dtype", "config", "value_note",
            "round_candidate_tokens_per_s", "accepted_tokens_per_s", "verify_ms", "verify_candidate_tokens_per_s",
            "verify_hbm_gbs", "verify_hbm_frac", "verify_bytes", "roofline", "attention", "mean_accepted",
            "sequences_per_s", "rows_per_round", "gpu_launches", "clocks", "e2e")


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    import argparse as _ap
    import gc
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verify_04_gb300 import spec
    runs = {"tiny": run_tiny, "accept": run_accept, "tree8": run_tree8, "adaptive": run_adaptive}
    if args.workload in runs:
        line = runs[args.workload](args, spec, world, rank, local, dist)
    else:
        line = run_chain(args, spec, world, rank, local, dist)
        default = (args.batch == 1 and args.mode == "greedy" and not args.tree and not args.page and
                   args.layers is None)
        if default and not args.no_subs:
            # the other configurations, each timed the same way (CUDA events on the
            # launching stream, warm-up first, clocks sampled), as sub-records of this line
            sub_args = _ap.Namespace(**vars(args))
            sub_args.steps, sub_args.warmup, sub_args.no_cpu_baseline = min(args.steps, 20), max(3, args.warmup), True
            subs = {}
            for name, kind in SUBS:
                gc.collect()
                torch.cuda.empty_cache()
                if kind == "chain8":
                    sub = run_chain(sub_args, spec, world, rank, local, dist, batch=8)
                else:
                    sub = runs[kind](sub_args, spec, world, rank, local, dist)
                subs[name] = {k2: sub[k2] for k2 in SUB_KEYS if k2 in sub}
            line["sub_workloads"] = subs
            line["gpu_launches_sub_workloads"] = sum(int(v.get("gpu_launches") or 0) for v in subs.values())
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
