#!/usr/bin/env python
"""Benchmark: constrained decode steps/s of the trie-constrained greedy decoder.

Default workload: the large single-sequence head (vocab 151,936, hidden 2,048
Gaussian bf16 tied embedding of 622 MB, the 42-tool catalog in constant
memory, k = 5, batch 1), queries cycled from the 1,000-query set.

One timed bench step = one tc_decode call: a captured CUDA graph that resets
the batch and runs the constrained decode step (mask, sparse head, argmax,
advance) until every sequence has stopped.  The reported value is decode
steps per second: loop iterations, each one step of the whole batch.

Timing: W untimed warm-up steps, then exactly K timed steps bracketed by a
barrier and torch.cuda.synchronize(); each step's device time is taken with
CUDA events on the launching stream around the graph launch only; between
steps (outside the events) the query's hidden states are copied into the
graph's input buffer (device to device) and L2 is flushed by writing a 512 MiB
buffer.  Max over ranks; ranks decode disjoint queries (weak scaling, no
collective on the data path).

Also printed: end-to-end rate through the same call with the inputs copied
from pinned host memory and the results read back inside the timed region;
the roofline of the step kernel (algorithmic bytes per launch over its
per-launch CUDA-event time); the dense-head comparison; the oracle timed on
the host cores; GPU clocks sampled during the timed region.

`--impl reference` times the CPU oracle on the same workload and metric.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from trie_constrained_decoding_gb300 import inputs as I  # noqa: E402

METRIC = "constrained decode steps/s"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FLUSH_BYTES = 512 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="large_head", choices=sorted(I.WORKLOADS))
    ap.add_argument("--head", choices=["sparse", "dense", "union", "dense_gemm"], default="sparse",
                    help="output head: sparse rows, dense GEMV + mask, union-of-legal-rows tcgen05 GEMM, "
                         "or full-vocabulary tcgen05 GEMM + mask")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-extras", action="store_true", help="skip the dense/host-loop/e2e/roofline passes")
    ap.add_argument("--residency", choices=["auto", "const", "global"], default=None,
                    help="grammar residency (default: the workload's)")
    ap.add_argument("--loop", choices=["graph", "host"], default="graph",
                    help="timed loop: the captured device-resident graph (default) or host-driven steps")
    ap.add_argument("--live-counts", action="store_true",
                    help="per-sequence live-count arrays instead of the read-only no-repeat state")
    ap.add_argument("--jump", action="store_true",
                    help="forced continuations: emit grammar-forced tokens without the head (sparse/dense heads)")
    ap.add_argument("--root-gemm", action="store_true",
                    help="sparse head with the first (root) step on the tcgen05 GEMM (TC_FLAG_ROOT_GEMM)")
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences per query batch (default: the workload's)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def sparse_kernel_name(max_fanout: int) -> str:
    """The sparse-step kernel the library launches for a grammar: the one-CTA
    kernel when no node has more than 32 edges."""
    return "sparse_step1_kernel" if max_fanout <= 32 else "sparse_step_kernel"


def source_code_sha256(*paths: str) -> str:
    """sha256 of source files' code, in order: `//` comments, surrounding
    blanks and empty lines removed, so that comment edits keep a capture valid."""
    import hashlib
    lines = []
    for path in paths:
        for line in open(path, encoding="utf-8").read().splitlines():
            code = line.split("//", 1)[0].strip()
            if code:
                lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def recorded_traffic(source: str, profile: str):
    """DRAM bytes per launch recorded by the last ncu capture of a kernel, or
    None when the kernel's source code has changed since that capture.
    `source` names the kernel's files, `+`-separated (the kernel file and the
    header of its shared types)."""
    try:
        text = open(os.path.join(ROOT, "profiles", profile)).read()
        want = source_code_sha256(*[os.path.join(ROOT, "trie_constrained_decoding_gb300", "csrc", f)
                                    for f in source.split("+")])
    except OSError:
        return None
    sha = traffic = None
    for line in text.splitlines():
        if line.startswith(f"source-code-sha256 {source}:"):
            sha = line.split(":", 1)[1].strip()
        if line.startswith("dram-bytes-per-launch:"):
            traffic = float(line.split(":", 1)[1])
    return traffic if sha == want else None


def physical_cores():
    """Physical cores of the host: distinct (package, core) pairs in sysfs, or None."""
    import re
    base = "/sys/devices/system/cpu"
    seen = set()
    try:
        names = os.listdir(base)
    except OSError:
        return None
    for d in names:
        if not re.fullmatch(r"cpu\d+", d):
            continue
        try:
            with open(os.path.join(base, d, "topology", "physical_package_id")) as f:
                pkg = f.read().strip()
            with open(os.path.join(base, d, "topology", "core_id")) as f:
                core = f.read().strip()
        except OSError:
            continue
        seen.add((pkg, core))
    return len(seen) or None


def host_cores():
    return {"logical_cpus": os.cpu_count(), "physical_cores": physical_cores(),
            "usable_cpus": len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else None}


def read_peaks():
    try:
        with open(PEAKS_PATH) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------- helpers

def query_ids(n_queries: int, rank: int, world: int, count: int):
    return [(rank + world * i) % n_queries for i in range(count)]


def aggregate_ranks(dist, dev_ms: float, steps: int, tokens: int, device: str):
    """Whole-job figures: the slowest rank's time and the steps/tokens of all ranks.

    Only timing scalars cross ranks; the decode itself has no collective."""
    import torch
    if dist is None:
        return dev_ms, float(steps), float(tokens)
    t_max = torch.tensor([dev_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t_max, op=dist.ReduceOp.MAX)
    sums = torch.tensor([float(steps), float(tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(sums, op=dist.ReduceOp.SUM)
    return float(t_max[0]), float(sums[0]), float(sums[1])


def host_hidden(w, qids):
    """bf16 bits [len(qids), steps, batch, hidden] of the queries' hidden states."""
    B = w.batch
    uniq = sorted(set(qids))
    start, stop = uniq[0], uniq[-1] + 1
    all_h = w.hidden_states(start * B, (stop - start) * B)       # [S, (stop-start)*B, H]
    S, _, H = all_h.shape
    all_h = all_h.reshape(S, stop - start, B, H).transpose(1, 0, 2, 3)
    return {q: np.ascontiguousarray(all_h[q - start]) for q in uniq}


def _oracle_batches(w, seconds: float, batches, hid_of, head: str):
    """Decode query batches in order with the oracle for about `seconds`;
    return (decode steps, tokens, batches decoded, seconds)."""
    from oracle import chars as C
    from oracle import decode as D
    from oracle import grammar as G
    if w.char_strings is not None:
        trie = C.CharGrammar(w.char_strings, w.char_vocab, w.sep_id, w.stop_id)
    else:
        trie = G.compile_catalog(w.catalog, w.sep_id, w.stop_id, w.vocab, max_fanout=w.max_fanout)
    emb = hid_of("emb")
    t0 = time.perf_counter()
    steps = tokens = done = 0
    i = 0
    while True:
        hid = hid_of(batches[i])
        lens = []
        for b in range(w.batch):
            toks, _, _ = D.greedy_decode(trie, w.k, emb, hid[:, b], w.max_steps, head=head)
            lens.append(len(toks))
        tokens += sum(lens)
        steps += max(lens)                  # lockstep: the batch steps until its longest sequence stops
        done += 1
        i = (i + 1) % len(batches)
        if time.perf_counter() - t0 >= seconds:
            break
    return steps, tokens, done, time.perf_counter() - t0


def oracle_baseline(w, seconds: float, head: str = "sparse"):
    """Greedy decode with the oracle on the host, one process, for about `seconds`."""
    emb = w.embedding()
    n_batches = max(1, min(w.n_queries // w.batch, max(1, 256 // w.batch)))
    hid = {q: w.hidden_states(q * w.batch, w.batch) for q in range(n_batches)}   # before the clock starts
    steps, tokens, done, dt = _oracle_batches(w, seconds, list(range(n_batches)),
                                              lambda q: emb if q == "emb" else hid[q], head)
    return {"value": steps / dt, "unit": "steps/s", "cores": 1, "kind": "oracle",
            "tokens_per_s": tokens / dt, "seconds": round(dt, 3),
            "sample": f"{done} query batches of '{w.name}' (batch {w.batch}), decoded in order by the "
                      f"fp64 oracle ({head} head), single process"}


def oracle_dense_steps(w, seconds: float):
    """The oracle's literal dense pipeline (every vocabulary logit, then the
    mask, then the argmax): first decode steps of successive queries, one
    process, for about `seconds` (at least one step)."""
    from oracle import chars as C
    from oracle import decode as D
    from oracle import grammar as G
    if w.char_strings is not None:
        trie = C.CharGrammar(w.char_strings, w.char_vocab, w.sep_id, w.stop_id)
    else:
        trie = G.compile_catalog(w.catalog, w.sep_id, w.stop_id, w.vocab, max_fanout=w.max_fanout)
    emb = w.embedding()
    hid = w.hidden_states(0, 8, steps=1)
    t0 = time.perf_counter()
    steps = 0
    while True:
        D.greedy_decode(trie, w.k, emb, hid[:, steps % 8], 1, head="dense")
        steps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": steps / dt, "unit": "steps/s", "cores": 1,
            "sample": f"first decode step of {steps} '{w.name}' queries, fp64 oracle, dense head"}


def _oracle_worker(name, shm_name, emb_shape, seconds, worker, n_workers, n_batches, head, ready, start, results):
    from multiprocessing import shared_memory
    shm = shared_memory.SharedMemory(name=shm_name)
    try:
        w = I.WORKLOADS[name]()
        emb = np.ndarray(emb_shape, dtype=np.uint16, buffer=shm.buf)
        mine = [q for q in range(n_batches) if q % n_workers == worker] or [worker % n_batches]
        hid = {q: w.hidden_states(q * w.batch, w.batch) for q in mine}
        ready.put(worker)
        start.wait()
        steps, tokens, done, dt = _oracle_batches(w, seconds, mine, lambda q: emb if q == "emb" else hid[q], head)
        results.put((worker, steps, tokens, done, dt))
    finally:
        del emb
        shm.close()


def oracle_pool_baseline(w, seconds: float, procs: int = 0, head: str = "sparse"):
    """The oracle as it stands on every host core: one spawned process per core,
    each decoding its own share of the query batches for about `seconds` (all
    released together); the rate is the sum of the processes' rates."""
    import multiprocessing as mp
    from multiprocessing import shared_memory
    procs = procs or os.cpu_count() or 1
    emb = w.embedding()
    n_batches = max(1, min(w.n_queries // w.batch, max(procs, 256 // w.batch)))
    shm = shared_memory.SharedMemory(create=True, size=emb.nbytes)
    try:
        np.ndarray(emb.shape, dtype=np.uint16, buffer=shm.buf)[...] = emb
        ctx = mp.get_context("spawn")
        ready, results, start = ctx.Queue(), ctx.Queue(), ctx.Event()
        ps = [ctx.Process(target=_oracle_worker, args=(w.name, shm.name, emb.shape, seconds, i, procs, n_batches,
                                                       head, ready, start, results)) for i in range(procs)]
        for p in ps:
            p.start()
        for _ in ps:
            ready.get(timeout=600)
        start.set()
        res = [results.get(timeout=600 + 4 * seconds) for _ in ps]
        for p in ps:
            p.join(timeout=60)
    finally:
        shm.close()
        shm.unlink()
    rate = sum(r[1] / r[4] for r in res)
    trate = sum(r[2] / r[4] for r in res)
    done = sum(r[3] for r in res)
    return {"value": rate, "unit": "steps/s", "cores": procs, "kind": "oracle", "tokens_per_s": trate,
            "sample": f"{done} query batches of '{w.name}' (batch {w.batch}) decoded by the fp64 oracle "
                      f"({head} head) in {procs} spawned processes (one per host core, "
                      f"os.cpu_count()={os.cpu_count()}), about {seconds:g} s each"}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = I.WORKLOADS[args.workload]()
    if args.batch:
        w.batch = args.batch
    # Each bench step decodes one query batch with the oracle; bounded so that
    # warm-up + steps finish within a few minutes.
    budget = min(120.0, max(5.0, 0.05 * (args.steps + args.warmup)))
    base = oracle_baseline(w, budget, head="sparse")
    line = {"metric": METRIC, "value": base["value"], "unit": "steps/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / base["value"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "batch": w.batch, "k": w.k, "vocab": w.vocab, "hidden": w.hidden,
                       "catalog": len(w.catalog), "note": "CPU oracle (plain Python + numpy fp64), one process: one stream of decode steps, as the GPU arm"},
            "cpu_baseline": dict({k: base[k] for k in ("value", "unit", "cores", "kind", "sample")},
                                 host=host_cores()),
            "e2e": {"value": base["value"], "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    from trie_constrained_decoding_gb300 import binding as tcd

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    stream = torch.cuda.current_stream()
    w = I.WORKLOADS[args.workload]()
    if args.batch:
        w.batch = args.batch
    head = {"sparse": tcd.HEAD_SPARSE, "dense": tcd.HEAD_DENSE, "union": tcd.HEAD_UNION_GEMM,
            "dense_gemm": tcd.HEAD_DENSE_GEMM}[args.head]
    if args.jump:
        head |= tcd.FLAG_JUMP_FORWARD
    if args.root_gemm:
        head |= tcd.FLAG_ROOT_GEMM
    B, S, H = w.batch, w.max_steps, w.hidden

    emb_bits = w.embedding()
    emb = torch.from_numpy(emb_bits.view(np.int16)).to(f"cuda:{dev}").view(torch.bfloat16)
    del emb_bits
    if w.char_strings is not None:
        trie = tcd.Trie.compile_chars(w.char_strings, w.char_vocab, w.sep_id, w.stop_id, w.vocab, w.max_fanout)
    else:
        trie = tcd.Trie.compile(w.catalog, w.sep_id, w.stop_id, w.vocab, w.max_fanout)
    tinfo = trie.info()
    ctx = tcd.Context(emb, max_batch=B, cand_cap=w.cand_cap)
    res = {"const": tcd.RES_CONST, "global": tcd.RES_GLOBAL, "auto": tcd.RES_AUTO}[args.residency or w.residency]
    ctx.bind(trie, res | (tcd.BIND_LIVE_COUNTS if args.live_counts else 0))
    state_mode = "live counts" if (args.live_counts or w.k > 8) else "read-only (rank ranges + banned set)"

    n_batches = max(1, min(w.n_queries // B, 2048 // B))
    K, W = args.steps, args.warmup
    qids = query_ids(n_batches, rank, world, K + W)
    hh = host_hidden(w, qids)
    dev_hidden = {q: torch.from_numpy(h.view(np.int16)).to(f"cuda:{dev}").view(torch.bfloat16)
                  for q, h in hh.items()}
    hid_buf = torch.empty((S, B, H), dtype=torch.bfloat16, device=f"cuda:{dev}")
    toks = torch.empty((B, S), dtype=torch.int32, device=f"cuda:{dev}")
    logits = torch.empty((B, S), dtype=torch.float32, device=f"cuda:{dev}")
    lens = torch.empty(B, dtype=torch.int32, device=f"cuda:{dev}")
    status = torch.empty(B, dtype=torch.int32, device=f"cuda:{dev}")
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=f"cuda:{dev}")

    def decode_one(q, ev=None):
        hid_buf.copy_(dev_hidden[q])
        flush.zero_()
        if ev is not None:
            ev[0].record(stream)
        run = ctx.decode if args.loop == "graph" else ctx.decode_host
        run(hid_buf, w.k, S, toks, logits, lens, status, head=head)
        if ev is not None:
            ev[1].record(stream)

    # Decode steps of each query batch, counted from an untimed decode of it
    # (the decode is deterministic): the steps until its last sequence
    # stopped, i.e. the head decisions of its longest-running sequence (forced
    # tokens ride along in the same step), plus the step in which a failing
    # sequence failed.  Idle launches after the last sequence stopped are not
    # steps.  The timed region's own counters are checked against these below.
    work = {}
    for q in sorted(set(qids)):
        decode_one(q)
        n = lens.cpu().numpy()
        lg = logits.cpu().numpy()
        stt = status.cpu().numpy()
        forced = np.array([int(np.isnan(lg[b, :n[b]]).sum()) for b in range(B)])
        work[q] = (int((n - forced + (stt != 0)).max()), int(n.sum()), int((n - forced).sum()), int(forced.sum()))
    # Clocks are sampled every 20 ms from the start of the warm-up to the end
    # of the timed region (a short timed region alone may fall between samples).
    sampler = ClockSampler(dev)
    sampler.start()
    time.sleep(0.05)
    for i in range(W):
        decode_one(qids[i])
    torch.cuda.synchronize()
    ctx.raise_on_error()
    ctx.stats(reset=True)

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(K):
        decode_one(qids[W + i], evs[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    clocks["window"] = "warm-up and timed region, nvidia-smi every 20 ms"
    dev_ms = sum(a.elapsed_time(b) for a, b in evs)
    st = ctx.stats(reset=True)
    ctx.raise_on_error()
    timed = [work[q] for q in qids[W:W + K]]
    decode_steps = sum(x[0] for x in timed)
    tokens = sum(x[1] for x in timed)
    # the timed decodes did exactly the counted work
    counted_ok = (st["seq_steps"] == sum(x[2] for x in timed) and st["forced"] == sum(x[3] for x in timed))
    gpu_launches = st["step_launches"] + st["reset_launches"]

    dev_ms_max, all_steps, all_tokens = aggregate_ranks(dist, dev_ms, decode_steps, tokens, f"cuda:{dev}")
    value = all_steps / (dev_ms_max / 1000.0)
    # Roofline in the regime of the headline: the timed graph loops' own
    # device time per decode step (reset, idle launches and loop control
    # included, so an upper bound of the step kernel's time) against the
    # algorithmic bytes of those steps (candidate rows + hidden states; the
    # union head: union rows + hidden states; dense heads: every row).
    hb = 2.0 * H
    base_head = head & ~(tcd.FLAG_JUMP_FORWARD | tcd.FLAG_FORCED_LOGITS | tcd.FLAG_ROOT_GEMM)
    if base_head == tcd.HEAD_SPARSE:
        algo = (st["cand_rows"] + st["seq_steps"]) * hb
    elif base_head == tcd.HEAD_UNION_GEMM:
        algo = (st["union_rows"] + st["seq_steps"]) * hb
    elif base_head == tcd.HEAD_DENSE:
        algo = st["seq_steps"] * (w.vocab + 1) * hb
    else:
        algo = decode_steps * w.vocab * hb + st["seq_steps"] * hb
    roof_graph = {"bound": "hbm", "achieved": algo / decode_steps / (dev_ms / decode_steps / 1000.0) / 1e9,
                  "unit": "GB/s", "algorithmic_bytes_per_launch": algo / decode_steps,
                  "us_per_launch": dev_ms * 1000.0 / decode_steps,
                  "regime": "graph loop of the timed region: device time per decode step (reset, idle launches "
                            "and loop control included), one step-kernel launch per decode step",
                  "candidates_per_sequence_step": st["cand_rows"] / max(1, st["seq_steps"])}

    extras = {}
    e2e = None
    per_launch = None
    if not args.no_extras:
        per_launch, extras = extra_passes(args, w, ctx, tcd, torch, stream, dev, dev_hidden, hh, qids[W:], head, flush,
                                    hid_buf, toks, logits, lens, status, tinfo["max_fanout"], work)
        e2e = extras.pop("e2e")
        if world == 1 and args.workload == "large_head" and head == tcd.HEAD_SPARSE:
            extras["heads_by_batch"] = heads_by_batch(tcd, torch, dev, stream, flush)

    if rank != 0:
        return 0
    peak, peak_kind = read_peaks()
    roof = dict(roof_graph, peak=peak, frac=roof_graph["achieved"] / peak, traffic=None,
                kernel={tcd.HEAD_SPARSE: sparse_kernel_name(tinfo["max_fanout"]),
                        tcd.HEAD_DENSE: "dense_step_kernel"}.get(base_head, "union_gemm_kernel"),
                peak_source=(f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)" if peak_kind == "measured"
                             else "fallback 6.8 TB/s"),
                per_launch_tc_step=per_launch)
    if base_head == tcd.HEAD_SPARSE and args.workload == "large_head":
        prof = f"{sparse_kernel_name(tinfo['max_fanout'])}_large_head.md"
        roof["traffic"] = recorded_traffic("step_kernels.cu+kernels.h", prof)
        roof["traffic_source"] = ("ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, cold caches, "
                                  f"profiles/{prof}" if roof["traffic"] is not None
                                  else "kernel source changed since the last ncu capture")
    cpu = None
    if world == 1 and not args.no_extras:
        # One process decodes one stream of query batches, as this bench does on
        # the GPU; the pool runs one such stream per host core (throughput of
        # independent streams, like a larger batch).
        one = oracle_baseline(w, args.cpu_seconds)
        pool = oracle_pool_baseline(w, args.cpu_seconds)
        cpu = {k: one[k] for k in ("value", "unit", "cores", "kind", "sample")}
        cpu["tokens_per_s"] = one["tokens_per_s"]
        cpu["host"] = host_cores()
        cpu["all_cores_pool"] = {k: pool[k] for k in ("value", "unit", "cores", "tokens_per_s", "sample")}
        if B == 1:   # the dense-logits-then-mask oracle, on a small subset (every vocabulary row per step)
            cpu["dense_head"] = oracle_dense_steps(w, min(6.0, args.cpu_seconds / 2))
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": dev_ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 x bf16 -> fp32 accumulate", "data": "synthetic (seeded; no dataset or weights)",
        "config": {"workload": w.name, "batch": B, "k": w.k, "vocab": w.vocab, "hidden": H,
                   "catalog_strings": len(w.catalog), "trie_nodes": tinfo["n_nodes"], "trie_edges": tinfo["n_edges"],
                   "max_fanout": tinfo["max_fanout"], "residency": ["auto", "const", "global"][ctx.residency()],
                   "head": args.head + (" (root step on the tcgen05 GEMM)" if args.root_gemm else ""),
                   "jump_forward": bool(args.jump), "no_repeat_state": state_mode,
                   "bench_step": "one tc_decode graph launch decoding one query batch to the end",
                   "decode_steps_per_bench_step": all_steps / (K * world),
                   "step_launches_per_bench_step": st["step_launches"] / K,
                   "timed_work_matches_count": counted_ok,
                   "tokens_per_s": all_tokens / (dev_ms_max / 1000.0),
                   "l2": "flushed between timed steps (512 MiB write outside the CUDA events)",
                   "wall_s_timed_region": round(t_wall, 3)},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = e2e
    line["roofline"] = roof
    if cpu is not None:
        line["cpu_baseline"] = cpu
    line["variants"] = extras
    print(json.dumps(line))
    ctx.close()
    if dist:
        dist.destroy_process_group()
    return 0


def head_rates(tcd, torch, dev, stream, flush, embs, name, heads, n_q, batch=None):
    """Decode n_q query batches of workload `name` (at `batch` sequences,
    default the workload's) with each of `heads`, through the graph loop with
    the main pass's exact step counting and L2 flushes.  Per head: decode
    steps/s, tokens/s and the algorithmic bytes of those steps over their
    device time (sparse: candidate rows; union: union rows once per step;
    dense GEMM: every vocabulary row once per step; all: each stepping
    sequence's hidden state)."""
    w = I.WORKLOADS[name]()
    if batch:
        w.batch = batch
    B, S, H = w.batch, w.max_steps, w.hidden
    key = (w.vocab, H, w.emb_kind)
    if key not in embs:
        bits = w.embedding()
        embs[key] = torch.from_numpy(bits.view(np.int16)).to(f"cuda:{dev}").view(torch.bfloat16)
        del bits
    if w.char_strings is not None:
        trie = tcd.Trie.compile_chars(w.char_strings, w.char_vocab, w.sep_id, w.stop_id, w.vocab, w.max_fanout)
    else:
        trie = tcd.Trie.compile(w.catalog, w.sep_id, w.stop_id, w.vocab, w.max_fanout)
    ctx = tcd.Context(embs[key], max_batch=B, cand_cap=w.cand_cap)
    ctx.bind(trie, {"const": tcd.RES_CONST, "global": tcd.RES_GLOBAL, "auto": tcd.RES_AUTO}[w.residency])
    qids = list(range(n_q))
    hh = host_hidden(w, qids)
    hid = {q: torch.from_numpy(h.view(np.int16)).to(f"cuda:{dev}").view(torch.bfloat16) for q, h in hh.items()}
    del hh
    # one input buffer: the captured decode graph is keyed by its arguments and reused
    buf = torch.empty((S, B, H), dtype=torch.bfloat16, device=f"cuda:{dev}")
    toks = torch.empty((B, S), dtype=torch.int32, device=f"cuda:{dev}")
    logits = torch.empty((B, S), dtype=torch.float32, device=f"cuda:{dev}")
    lens = torch.empty(B, dtype=torch.int32, device=f"cuda:{dev}")
    status = torch.empty(B, dtype=torch.int32, device=f"cuda:{dev}")
    out = {"workload": name, "batch": B, "k": w.k, "query_batches": n_q}
    for hname in heads:
        head = {"sparse": tcd.HEAD_SPARSE, "union": tcd.HEAD_UNION_GEMM, "dense_gemm": tcd.HEAD_DENSE_GEMM,
                "sparse_root_gemm": tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM}[hname]
        steps = {}
        for q in qids:        # untimed: the decode steps of each query batch under this head
            buf.copy_(hid[q])
            ctx.decode(buf, w.k, S, toks, logits, lens, status, head=head)
            n = lens.cpu().numpy()
            steps[q] = (int((n + (status.cpu().numpy() != 0)).max()), int(n.sum()))
        for q in qids[:2]:
            buf.copy_(hid[q])
            ctx.decode(buf, w.k, S, toks, logits, lens, status, head=head)
        torch.cuda.synchronize()
        ctx.raise_on_error()
        ctx.stats(reset=True)
        evs = []
        for q in qids:
            buf.copy_(hid[q])
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ctx.decode(buf, w.k, S, toks, logits, lens, status, head=head)
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        ctx.raise_on_error()
        st = ctx.stats(reset=True)
        sec = sum(a.elapsed_time(b) for a, b in evs) / 1000.0
        n_steps = sum(steps[q][0] for q in qids)
        n_tok = sum(steps[q][1] for q in qids)
        hid_bytes = st["seq_steps"] * 2.0 * H
        if hname in ("sparse", "sparse_root_gemm"):
            # (with the root step on the GEMM each root row is read once per step, not
            # once per sequence: these bytes count it per sequence, as the sparse head reads it)
            algo = st["cand_rows"] * 2.0 * H + hid_bytes
        elif hname == "union":
            algo = st["union_rows"] * 2.0 * H + hid_bytes
        else:
            algo = n_steps * w.vocab * 2.0 * H + hid_bytes
        r = {"steps_per_s": n_steps / sec, "tokens_per_s": n_tok / sec, "us_per_step": sec * 1e6 / n_steps,
             "timed_work_matches_count": st["seq_steps"] == n_tok, "algorithmic_gbs": algo / sec / 1e9,
             "candidates_per_sequence_step": st["cand_rows"] / max(1, st["seq_steps"])}
        if hname == "union":
            r["union_rows_per_step"] = st["union_rows"] / max(1, n_steps)
        if hname == "dense_gemm":
            r["tflops"] = n_steps * 2.0 * w.vocab * H * B / sec / 1e12
        out[hname] = r
    ctx.close()
    trie.close()
    del hid, buf
    return out


def heads_by_batch(tcd, torch, dev, stream, flush):
    """The constrained decode step at B=1 (large_head: sparse and union heads;
    the dense GEMV is the line's dense_head), at B=64 and B=256 with the sparse
    head, the union-of-legal-rows tcgen05 GEMM and the full-vocabulary tcgen05
    GEMM + mask (the 1000-tool catalog, hidden 4096), and the hex catalog (root
    fan-out 267) at B=16, 64 and 256 with the sparse and union heads: where the
    union of legal rows is large and shared, the GEMM reads each row once.
    `sparse_root_gemm`: the sparse head with the first (root) step on the
    tcgen05 GEMM (TC_FLAG_ROOT_GEMM), on the hex catalog and at B=256, timed
    right after the sparse head (the power-capped dense GEMM slows what
    follows it)."""
    embs = {}
    out = {
        "1": head_rates(tcd, torch, dev, stream, flush, embs, "large_head", ("sparse", "union"), 40),
        "64": head_rates(tcd, torch, dev, stream, flush, embs, "batched", ("sparse", "union", "dense_gemm"), 12),
        "256": head_rates(tcd, torch, dev, stream, flush, embs, "tensor_batch",
                          ("sparse", "sparse_root_gemm", "union", "dense_gemm"), 4),
    }
    hexes = {}
    for B, n_q in ((16, 8), (64, 4), (256, 2)):
        hexes[str(B)] = head_rates(tcd, torch, dev, stream, flush, embs, "unstructured",
                                   ("sparse", "sparse_root_gemm", "union"), n_q, batch=B)
    out["hex_catalog"] = hexes
    del embs
    return out


def extra_passes(args, w, ctx, tcd, torch, stream, dev, dev_hidden, hh, qids, head, flush, hid_buf, toks, logits,
                 lens, status, max_fanout, work):
    """Roofline of the step kernel, dense-head comparison, forced-continuation
    variant, loop floor, host loop and end-to-end rate."""
    B, S, H = w.batch, w.max_steps, w.hidden
    out = {}
    n_roof = min(len(qids), 200 if B == 1 else 8)
    flags = head & tcd.FLAG_JUMP_FORWARD
    head = head & ~(tcd.FLAG_JUMP_FORWARD | tcd.FLAG_ROOT_GEMM)  # the per-launch and host-loop passes run plain steps

    # --- step kernel alone: tc_step (same kernel body, host-argument form), one
    # event pair per launch; L2 flushed before every launch (cold) or not (warm).
    tok = torch.empty(B, dtype=torch.int32, device=f"cuda:{dev}")
    lg = torch.empty(B, dtype=torch.float32, device=f"cuda:{dev}")
    stt = torch.empty(B, dtype=torch.int32, device=f"cuda:{dev}")

    # steps each query needs (the graph loop's own count), so the step loop runs exactly those
    n_steps = {}
    for q in qids[:n_roof]:
        hid_buf.copy_(dev_hidden[q])
        ctx.decode(hid_buf, w.k, S, toks, logits, lens, status, head=head)
        n_steps[q] = int((lens + (status != 0).int()).max().item())

    def kernel_pass(cold: bool):
        pairs = []
        for q in qids[:n_roof]:
            hid_buf.copy_(dev_hidden[q])
            ctx.reset(B, w.k)
            for t in range(n_steps[q]):
                if cold:
                    flush.zero_()
                else:
                    torch.cuda._sleep(40000)   # keeps the GPU busy while the host enqueues the step
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                ctx.step(hid_buf[t], tok, lg, stt, head=head)
                b.record(stream)
                pairs.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in pairs]

    ctx.stats(reset=True)
    cold_ms = kernel_pass(True)
    st = ctx.stats(reset=True)
    launches = len(cold_ms)
    seq_steps = float(st["seq_steps"])
    cand_rows = float(st["cand_rows"])
    algo_bytes = cand_rows * 2 * H + seq_steps * 2 * H    # embedding rows gathered + hidden states read
    mean_ms = sum(cold_ms) / launches
    achieved = algo_bytes / launches / (mean_ms / 1000.0) / 1e9
    warm_ms = kernel_pass(False)
    warm_mean = sum(warm_ms) / len(warm_ms)
    roof = {"achieved_cold_gbs": achieved, "unit": "GB/s",
            "algorithmic_bytes_per_launch": algo_bytes / launches,
            "mean_launch_us_cold_l2": mean_ms * 1000.0, "mean_launch_us_warm_l2": warm_mean * 1000.0,
            "achieved_warm_gbs": algo_bytes / launches / (warm_mean / 1000.0) / 1e9,
            "candidates_per_sequence_step": cand_rows / max(1.0, seq_steps),
            "launches_timed": launches,
            "note": "side note, host-launched regime: per-launch CUDA events around tc_step (same kernel body "
                    "as the graph loop, plus host launch and event overhead); bytes = candidate rows x 2H + "
                    "hidden state 2H per sequence step"}

    # --- dense head + mask over the same queries (subset)
    if head in (tcd.HEAD_SPARSE, tcd.HEAD_UNION_GEMM):
        dense_head = tcd.HEAD_DENSE if B == 1 else tcd.HEAD_DENSE_GEMM
        n_dense = min(len(qids), 20 if B == 1 else 2)
        ctx.stats(reset=True)
        evs = []
        for q in qids[:n_dense]:
            hid_buf.copy_(dev_hidden[q])
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ctx.decode(hid_buf, w.k, S, toks, logits, lens, status, head=dense_head)
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        st = ctx.stats(reset=True)
        ms = sum(a.elapsed_time(b) for a, b in evs)
        out["dense_head"] = "dense GEMV + mask" if dense_head == tcd.HEAD_DENSE else "tcgen05 dense GEMM + mask"
        out["dense_head_steps_per_s"] = st["step_launches"] / (ms / 1000.0)
        # bytes of embedding the dense head must read per step: all V rows once
        # per sequence for the GEMV, once per step for the GEMM
        per_step = w.vocab * 2.0 * H
        reads = st["seq_steps"] * per_step if dense_head == tcd.HEAD_DENSE else st["step_launches"] * per_step
        out["dense_head_gbs"] = reads / (ms / 1000.0) / 1e9

    # --- host-driven loop (one synchronising read per step) over a subset
    n_host = min(len(qids), 100 if B == 1 else 4)
    ctx.stats(reset=True)
    t0 = time.perf_counter()
    for q in qids[:n_host]:
        hid_buf.copy_(dev_hidden[q])
        ctx.decode_host(hid_buf, w.k, S, toks, logits, lens, status, head=head)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    st = ctx.stats(reset=True)
    out["host_loop_steps_per_s_wall"] = st["step_launches"] / dt   # the host loop launches no idle steps

    # --- forced continuations (TC_FLAG_JUMP_FORWARD) against plain steps, same queries
    if head in (tcd.HEAD_SPARSE, tcd.HEAD_DENSE):
        n_j = min(len(qids), 500 if B == 1 else 16)
        rates = {}
        per_query = {}       # decode steps of each query under forced continuations (same with logits)
        for name, fl in (("plain", 0), ("jump_forward", tcd.FLAG_JUMP_FORWARD),
                         ("jump_forward_with_logits", tcd.FLAG_JUMP_FORWARD | tcd.FLAG_FORCED_LOGITS)):
            steps = toks_n = 0
            for q in sorted(set(qids[:n_j])):      # untimed: the exact step counts of each variant
                hid_buf.copy_(dev_hidden[q])
                ctx.decode(hid_buf, w.k, S, toks, logits, lens, status, head=head | fl)
            evs = []
            ctx.stats(reset=True)
            for q in qids[:n_j]:
                hid_buf.copy_(dev_hidden[q])
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                ctx.decode(hid_buf, w.k, S, toks, logits, lens, status, head=head | fl)
                e1.record(stream)
                evs.append((e0, e1))
                n = lens.cpu().numpy()
                lg = logits.cpu().numpy()
                forced = np.array([int(np.isnan(lg[b, :n[b]]).sum()) for b in range(B)])
                if name == "jump_forward":
                    per_query[q] = int((n - forced).max())
                # with logits the forced positions are not NaN: same decisions as jump_forward
                steps += per_query[q] if name == "jump_forward_with_logits" else int((n - forced).max())
                toks_n += int(n.sum())
            torch.cuda.synchronize()
            ms = sum(x.elapsed_time(y) for x, y in evs)
            st = ctx.stats(reset=True)
            rates[name] = {"steps_per_s": steps / (ms / 1000.0), "tokens_per_s": toks_n / (ms / 1000.0),
                           "forced_tokens": st["forced"], "head_decisions": st["seq_steps"]}
        out["forced_continuations"] = dict(rates, note=f"{n_j} query batches, L2 flushed before each decode; "
                                                        "a jump-forward step is one head decision plus the "
                                                        "forced span after it")

    # --- sampling (temperature 1, top-p 0.9) against the greedy argmax, same queries
    if head == tcd.HEAD_SPARSE:
        n_s = min(len(qids), 500 if B == 1 else 16)
        uq = {q: torch.from_numpy(w.uniforms(q * B, B)).to(f"cuda:{dev}") for q in sorted(set(qids[:n_s]))}
        rates = {}
        for name in ("greedy", "sampling"):
            steps = 0
            evs = []
            for q in qids[:n_s]:
                hid_buf.copy_(dev_hidden[q])
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if name == "greedy":
                    ctx.decode(hid_buf, w.k, S, toks, logits, lens, status, head=head)
                else:
                    ctx.decode_sample(hid_buf, w.k, S, uq[q], toks, logits, lens, status, temperature=1.0,
                                      top_k=0, top_p=0.9, head=head)
                e1.record(stream)
                evs.append((e0, e1))
                steps += int((lens + (status != 0).int()).max().item())
            torch.cuda.synchronize()
            ms = sum(x.elapsed_time(y) for x, y in evs)
            rates[name] = {"steps_per_s": steps / (ms / 1000.0)}
        out["sampling"] = dict(rates, note=f"{n_s} query batches, L2 flushed before each decode; sampling: "
                                           "temperature 1, top-p 0.9, seeded uniforms")

    # --- loop floor: the same graph loop with do-nothing kernels in the steps' place
    fl_ms, fl_n = tcd.loop_floor(dev, B, 256)
    out["loop_floor_us_per_launch"] = fl_ms * 1000.0 / fl_n

    # --- end to end through the C ABI with host buffers, as a serving loop
    # runs it: two buffer sets, so that the copies of one query (H2D of its
    # hidden states, D2H of its results packed in one block) overlap the
    # decode of the other on a second stream; every copy is inside the timed
    # region.
    n_e2e = min(len(qids), 500 if B == 1 else 8)
    pin_h = {q: torch.from_numpy(hh[q].view(np.int16)).view(torch.bfloat16).pin_memory() for q in qids[:n_e2e]}
    copy_stream = torch.cuda.Stream(device=dev)
    words = 2 * B * S + 2 * B          # toks | logits | lens | status, 4 bytes each

    class _Set:
        def __init__(self):
            self.hid = torch.empty((S, B, H), dtype=torch.bfloat16, device=f"cuda:{dev}")
            self.out = torch.empty(words, dtype=torch.int32, device=f"cuda:{dev}")
            self.toks = self.out[:B * S].view(B, S)
            self.logits = self.out[B * S:2 * B * S].view(torch.float32).view(B, S)
            self.lens = self.out[2 * B * S:2 * B * S + B]
            self.status = self.out[2 * B * S + B:]
            self.host = torch.empty(words, dtype=torch.int32).pin_memory()
            self.ev_in, self.ev_dec, self.ev_out = (torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event())

    sets = [_Set(), _Set()]

    def e2e_pass(qs):
        for i, q in enumerate(qs):
            st = sets[i % 2]
            copy_stream.wait_event(st.ev_dec)      # this set's hidden buffer is free again
            with torch.cuda.stream(copy_stream):
                st.hid.copy_(pin_h[q], non_blocking=True)
            st.ev_in.record(copy_stream)
            stream.wait_event(st.ev_in)
            stream.wait_event(st.ev_out)           # this set's outputs were read back
            ctx.decode(st.hid, w.k, S, st.toks, st.logits, st.lens, st.status, head=head | flags, stream=stream)
            st.ev_dec.record(stream)
            copy_stream.wait_event(st.ev_dec)
            with torch.cuda.stream(copy_stream):
                st.host.copy_(st.out, non_blocking=True)
            st.ev_out.record(copy_stream)

    e2e_pass(qids[:2])                             # (captures each set's decode graph, untimed)
    torch.cuda.synchronize()
    ctx.stats(reset=True)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    copy_stream.wait_event(a)
    e2e_pass(qids[:n_e2e])
    stream.wait_stream(copy_stream)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    ctx.stats(reset=True)
    h2d = S * B * H * 2
    d2h = words * 4
    e2e_steps = sum(work[q][0] for q in qids[:n_e2e])
    out["e2e"] = {"value": e2e_steps / (ms / 1000.0), "unit": "steps/s", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": d2h,
                  "note": "per bench step: pinned H2D of the query's hidden states, tc_decode, D2H of "
                          "tokens/logits/lengths/status (one packed block); two buffer sets, copies on a "
                          "second stream overlapping the other set's decode; CUDA events around the whole "
                          "sequence, L2 not flushed"}
    return roof, out


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
