"""Benchmark of the multi-adapter LoRA hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config stacked_gate_up] [--no-per-workload]

One step = lora_build_segments + lora_apply, made as the one public call
lora_build_and_apply, or for the MoE config build + gate/up delta + down
delta, over one batch of synthetic inputs already resident in HBM.  The
headline line is the largest single-GPU workload (the stacked gate/up
projection, 277 MB of algorithmic traffic per step); the same line carries a
per_workload map with every workload of the benchmark (decode, prefill,
stacked QKV / gate-up / down, MoE) measured the same way in the same run.
To keep L2 (129 MB) from serving the weights, every step uses the next of R
independent input sets (own adapter table, ids, x, y), with R * bytes-per-set
above 2x L2.  Steps are issued as CUDA-graph replays and timed with CUDA
events on the launching stream, bracketed by a barrier and a device
synchronize; rank 0 prints one JSON line.

Multi-GPU runs are independent replicas (the path has no exchange step):
every rank processes its own batches, the elapsed time is the max over ranks
and the value counts the tokens of all ranks.

--impl reference times the CPU oracle (plain C, fp64) on the host cores on
a bounded sample of the same workload; under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import re
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

METRIC = "LoRA-delta tokens/s at 1 GB300; achieved HBM GB/s or TC TFLOPS vs roofline"
L2_BYTES = 129 * 1024 * 1024
ENGINE_SRC = os.path.join(ROOT, "segmented_rank_gemm_lora_gb300", "csrc", "engine.cu")

CONFIGS = {
    "tiny": "M=64 tokens, K=256, N=512, 4 adapters ranks 8/16/16/32, ids uniform in -1..3, scale 2",
    "decode": "M=32 tokens (one per sequence), K=N=4096, 20 adapters ranks cycling 16/32/64, 10% ids -1, scale 2",
    "prefill": "16 requests, lengths ~ l^-1.2 on [16,512] (~1900 tokens), one adapter each, K=N=4096, "
               "16 adapters ranks cycling 16/32/64",
    "stacked_qkv": "M=1024 (512 decode + prefill runs), 32 adapters r=64, A=(3r,4096), B slices 4096/1024/1024",
    "stacked_gate_up": "M=1024 (512 decode + prefill runs), 32 adapters r=64, A=(2r,4096), B slices 14336/14336",
    "stacked_down": "M=1024 (512 decode + prefill runs), 32 adapters r=64, A=(r,14336), B 4096",
    "moe": "M=512, top-2 of 8 experts, hidden 4096, intermediate 14336, 8 adapters ranks 16/32/64, block_m 64",
}


def make_problem(config: str, seed: int, base: str = "random"):
    from segmented_rank_gemm_lora_gb300 import synth
    if config == "tiny":
        return synth.tiny(seed, y_base=base)
    if config == "decode":
        return synth.decode(seed, y_base=base)
    if config == "prefill":
        return synth.prefill(seed, y_base=base)
    if config.startswith("stacked_"):
        return synth.stacked(config[len("stacked_"):], seed, y_base=base)
    if config == "moe":
        return synth.moe(seed)
    raise ValueError(config)


def dense_algorithmic(p):
    """(bytes, flops) the method must move / do for one batch (true ranks, A and B read once)."""
    K, N = p.K, p.N
    active = sorted(set(int(i) for i in p.ids if 0 <= i < p.L))
    wbytes = sum(2 * (p.A[i].size + p.B[i].size) for i in active)
    Ma = int(sum(1 for i in p.ids if 0 <= i < p.L))
    nbytes = wbytes + Ma * (2 * K + 4 * N) + 4 * p.M
    flops = 0
    for i in active:
        m = int((p.ids == i).sum())
        flops += 2 * m * p.ranks[i] * (p.n_a * K + N)
    return nbytes, flops


def moe_algorithmic(p):
    """Gate/up + down deltas: A read once per used (adapter, expert) factor, x once per token,
    caches once per pair (read + write), cache2 read once per pair."""
    H, I, E, topk = p.H, p.I, p.E, p.topk
    pairs = [(int(p.ids[q // topk]), int(p.topk_ids.reshape(-1)[q])) for q in range(p.M * topk)]
    pairs = [(l, e) for l, e in pairs if 0 <= l < p.L]
    used_l = sorted(set(l for l, _ in pairs))
    used_le = sorted(set(pairs))
    wb = 0
    for l in used_l:
        wb += 2 * p.A_gu[l].shape[1] * p.A_gu[l].shape[2] * (p.A_gu[l].shape[0] if p.A_gu[l].shape[0] > 1 else 1)
        wb += 2 * p.B_d[l][0].size * (p.B_d[l].shape[0] if p.B_d[l].shape[0] > 1 else 1)
    for l, e in used_le:
        wb += 2 * p.B_gu[l][e if p.B_gu[l].shape[0] > 1 else 0].size
        wb += 2 * p.A_d[l][e if p.A_d[l].shape[0] > 1 else 0].size
    tokens = len(set(q // topk for q in range(p.M * topk) if 0 <= p.ids[q // topk] < p.L))
    P = len(pairs)
    nbytes = wb + tokens * 2 * H + P * (4 * 2 * I) + P * 2 * I + P * 4 * H + 4 * p.M + 4 * p.M * topk
    flops = sum(2 * p.ranks[l] * (H + 2 * I) + 2 * p.ranks[l] * (I + H) for l, _ in pairs)
    return nbytes, flops


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9], f[4]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        loaded = [r for r in rows if r[0] > 0.5 * r[1]] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# distributed helpers (replicas)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# traffic recorded by ncu for the current engine source (null if stale)
# ---------------------------------------------------------------------------
ENGINE_SOURCES = ("engine.cu", "stream.cu", "segments.cu", "common.cuh", "tc.cuh")
LINEAR_SOURCES = ("linear.cu", "linear.h", "common.cuh", "tc.cuh")


def engine_source_sha(names=ENGINE_SOURCES) -> str:
    """Hash of the kernels' code (the named csrc sources) with comments and blank space taken out, so that
    an edit of the comments alone does not retire the traffic counters taken on the same code."""
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "segmented_rank_gemm_lora_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(config: str):
    path = os.path.join(ROOT, "profiles", "engine_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path))
    except ValueError:
        return None
    entry = rec.get(config)
    sha = engine_source_sha({"linear_prefill": LINEAR_SOURCES, "embedding_decode": EMBED_SOURCES}.get(config, ENGINE_SOURCES))
    if not entry or entry.get("engine_sha") != sha:
        return None
    return entry.get("dram_bytes_per_launch")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------
def oracle_step(p):
    import oracle
    if hasattr(p, "A_gu"):
        oracle.moe_delta(p.ids, p.topk_ids, p.x, p.cache1, p.A_gu, p.B_gu, p.ranks, p.scales, p.E, True)
        oracle.moe_delta(p.ids, p.topk_ids, p.cache2, p.cache3, p.A_d, p.B_d, p.ranks, p.scales, p.E, False)
    else:
        oracle.lora_apply(p.ids, p.x, p.y_base, p.A, p.B, p.ranks, p.scales, p.slice_n, p.n_a)


def sample_problem(config: str, p, max_tokens: int):
    """A bounded sample of the workload: the first tokens of the batch, at most max_tokens and about
    5e7 multiply-adds of the oracle's per-token loops."""
    if hasattr(p, "A_gu"):
        return p, p.M
    per_token = max(1, (p.n_a * p.K + p.N) * max(p.ranks))
    max_tokens = max(8, min(max_tokens, int(5e7 // per_token)))
    if p.M <= max_tokens:
        return p, p.M
    from segmented_rank_gemm_lora_gb300 import synth
    q = synth.DenseProblem(**{**p.__dict__})
    q.ids, q.x, q.y_base, q.M = p.ids[:max_tokens], p.x[:max_tokens], p.y_base[:max_tokens], max_tokens
    return q, max_tokens


def host_cores() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _oracle_worker(config, warmup, steps, barrier, results):
    """One host core's share of an all-cores oracle run: untimed warm-up, then (after every worker is
    ready) `steps` samples, timed by the wall clock."""
    try:
        p = make_problem(config, 1000)
        q, tokens = sample_problem(config, p, 256)
        for _ in range(warmup):
            oracle_step(q)
        barrier.wait(timeout=600)
        t0 = time.time()
        for _ in range(steps):
            oracle_step(q)
        t1 = time.time()
        results.put((t0, t1, (tokens if not hasattr(q, "A_gu") else q.M) * steps))
    except Exception as exc:   # reported by the parent
        barrier.abort()
        results.put(("error", repr(exc)))


def oracle_all_cores(config: str, steps_per_worker, warmup: int = 1):
    """The oracle run on every host core at once (one spawned process per core, each on its own copy of
    the sample; tokens are independent, so this is the oracle over tokens in parallel).  Returns
    (tokens/s, wall seconds, workers); wall = last end - first start after a common barrier."""
    import multiprocessing as mp
    import queue
    import oracle
    oracle.build()   # once, before the workers load it
    ctx = mp.get_context("spawn")
    n = len(steps_per_worker)
    barrier, results = ctx.Barrier(n), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(config, warmup, k, barrier, results), daemon=True)
             for k in steps_per_worker]
    for pr in procs:
        pr.start()
    out = []
    try:
        for _ in range(n):
            out.append(results.get(timeout=900))
    except queue.Empty:
        out.append(("error", "an oracle worker did not report"))
    for pr in procs:
        pr.join(timeout=60)
        if pr.is_alive():
            pr.terminate()
    errs = [r for r in out if r[0] == "error"]
    if errs:
        raise RuntimeError("all-cores oracle run failed: %s" % errs[0][1])
    t0, t1 = min(r[0] for r in out), max(r[1] for r in out)
    return sum(r[2] for r in out) / max(t1 - t0, 1e-9), t1 - t0, n


def cpu_baseline(config: str, budget_s: float = 10.0):
    """The oracle on the host: single-threaded for about budget_s, then on every core at once with the
    same number of samples per core.  The all-cores figure is the baseline; the single-threaded one rides
    along."""
    import oracle
    oracle.build()
    p = make_problem(config, 1000)
    q, tokens = sample_problem(config, p, 256)
    t0 = time.perf_counter()
    oracle_step(q)
    one = time.perf_counter() - t0
    reps = max(1, min(100000, int(budget_s / max(one, 1e-6))))   # about budget_s of work, per leg
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(q)
    dt = time.perf_counter() - t0
    unit_tokens = tokens if not hasattr(q, "A_gu") else q.M
    single = {"value": unit_tokens * reps / dt, "cores": 1,
              "sample": "%d x one %s batch of %d tokens (first %d tokens of the batch), single-threaded C fp64"
                        % (reps, config, p.M, unit_tokens)}
    cores = host_cores()
    try:
        value, wall, n = oracle_all_cores(config, [reps] * cores)
    except RuntimeError as exc:
        return {"value": single["value"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "sample": single["sample"], "all_cores_error": str(exc)}
    return {"value": value, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": "%d processes x %d samples of one %s batch (first %d of its %d tokens), C fp64, "
                      "%.1f s wall" % (n, reps, config, unit_tokens, p.M, wall),
            "single_thread": single}


def run_reference(args, world, rank):
    if rank != 0:
        return
    p = make_problem(args.config, 1000)
    q, tokens = sample_problem(args.config, p, 256)
    # the K steps (and the W warm-up steps) spread over the host cores, one process each
    cores = min(host_cores(), max(1, args.steps))
    per = [args.steps // cores + (1 if i < args.steps % cores else 0) for i in range(cores)]
    value, dt, cores = oracle_all_cores(args.config, per, warmup=max(1, -(-args.warmup // cores)))
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "%s: %s" % (args.config, CONFIGS[args.config]),
                       "sample": "first %d tokens of each batch" % tokens},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": "%d steps of %d tokens over %d processes (one per host core), C fp64"
                                       % (args.steps, tokens, cores)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def _to_dev(a, torch, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _bf16_cpu(a, torch):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def _packed(torch, dev, parts):
    """One device buffer holding a step's inputs back to back (256-byte aligned), and a view of each, so
    that the end-to-end leg moves them host-to-device as one copy."""
    offs, total = [], 0
    for _, t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(total, dtype=torch.uint8, device=dev)
    views = {}
    for (name, t), o in zip(parts, offs):
        v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views[name] = v
    return buf, views


def build_sets(config, R, torch, lora, dev, first=0):
    sets = []
    for j in range(first, first + R):
        p = make_problem(config, 1000 + j)
        s = {"p": p}
        if hasattr(p, "A_gu"):
            s["gu"] = lora.lora_pack_weights([_to_dev(a, torch, dev) for a in p.A_gu],
                                             [_to_dev(b, torch, dev) for b in p.B_gu], p.ranks, p.scales, p.H,
                                             [2 * p.I], 1, E_A=p.A_gu[0].shape[0], E_B=p.B_gu[0].shape[0])
            s["dn"] = lora.lora_pack_weights([_to_dev(a, torch, dev) for a in p.A_d],
                                             [_to_dev(b, torch, dev) for b in p.B_d], p.ranks, p.scales, p.I,
                                             [p.H], 1, E_A=p.A_d[0].shape[0], E_B=p.B_d[0].shape[0])
            s["packed"], views = _packed(torch, dev, [
                ("ids", torch.from_numpy(p.ids)), ("tk", torch.from_numpy(p.topk_ids)), ("x", _bf16_cpu(p.x, torch)),
                ("c1", _bf16_cpu(p.cache1, torch)), ("c2", _bf16_cpu(p.cache2, torch)),
                ("c3", _bf16_cpu(p.cache3, torch))])
            s.update(views)
            s["ws"] = lora.Workspace(p.M, p.L, p.topk, p.E, p.block_m, device=dev)
            s["alg"] = moe_algorithmic(p)
            s["tokens"] = p.M
            s["bytes"] = sum(t.numel() * t.element_size() for t in (s["x"], s["c1"], s["c2"], s["c3"])) + \
                s["gu"].info().device_bytes + s["dn"].info().device_bytes
        else:
            s["table"] = lora.lora_pack_weights([_to_dev(a, torch, dev) for a in p.A],
                                                [_to_dev(b, torch, dev) for b in p.B], p.ranks, p.scales, p.K,
                                                p.slice_n, p.n_a)
            s["packed"], views = _packed(torch, dev, [("ids", torch.from_numpy(p.ids)), ("x", _bf16_cpu(p.x, torch)),
                                                      ("y", _bf16_cpu(p.y_base, torch))])
            s.update(views)
            s["ws"] = lora.Workspace(p.M, p.L, device=dev)
            # the rule lora_build_and_apply follows under the default options (lora.h): one launch when no
            # group can reach the tensor-core threshold (32 rows, 16 for A blocks over 128 rows)
            max_R = p.n_a * max(lora.lora_rank_padded(r) for r in p.ranks)
            s["fused"] = 0 < p.M <= (16 if max_R > 128 else 32)
            s["alg"] = dense_algorithmic(p)
            s["tokens"] = p.M
            s["bytes"] = s["x"].numel() * 2 + s["y"].numel() * 2 + s["table"].info().device_bytes
        sets.append(s)
    torch.cuda.synchronize()
    return sets


def step(s, lora, build=True):
    if "gu" in s:
        if build:
            lora.lora_build_segments(s["ws"], s["ids"], s["tk"])
        lora.lora_moe_delta(s["gu"], lora.LORA_MOE_GATE_UP, s["ws"], s["x"], s["c1"])
        lora.lora_moe_delta(s["dn"], lora.LORA_MOE_DOWN, s["ws"], s["c2"], s["c3"])
        return (1 if build else 0) + 2
    if build:
        # lora_build_segments + lora_apply as one public call: one launch for decode-sized batches
        lora.lora_build_and_apply(s["table"], s["ws"], s["ids"], s["x"], s["y"])
        return 1 if s["fused"] else 2
    lora.lora_apply(s["table"], s["ws"], s["x"], s["y"])
    return 1


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def measure(config, K, W, args, torch, lora, dev, world, e2e_steps, clocks=None):
    """One workload: K timed steps (build + apply, as CUDA-graph replays over R rotating input sets), the
    applies alone, and the end-to-end leg through host buffers.  Returns the numbers of one bench line."""
    sets = build_sets(config, 1, torch, lora, dev)
    per_set = sets[0]["bytes"]
    R = max(4, min(64, int(np.ceil(2.5 * L2_BYTES / max(per_set, 1)))))
    sets += build_sets(config, R - 1, torch, lora, dev, first=1)
    for s in sets:   # warm every set once eagerly (first launches set kernel attributes)
        step(s, lora)
    torch.cuda.synchronize()
    for s in sets:
        st = lora.lora_get_status(s["ws"])
        if st != lora.LORA_OK:
            raise RuntimeError("%s: device status %s" % (config, lora.STATUS[st]))

    stream = torch.cuda.Stream(device=dev)
    launches = {"n": 0}

    def steps_fn(n, build=True):
        def fn():
            c = 0
            for i in range(n):
                c += step(sets[i % R], lora, build)
            launches["n"] = c
        return fn

    # K steps are issued as replays of a graph of C = R steps (one rotation over the sets) plus one graph
    # with the remaining K mod C steps, so exactly K steps run in the timed region.
    C = R
    g_chunk = capture(torch, steps_fn(C), stream)
    launches_chunk = launches["n"]
    tail = K % C
    g_tail = capture(torch, steps_fn(tail), stream) if tail else None
    launches_tail = launches["n"] if tail else 0
    gpu_launches = (K // C) * launches_chunk + launches_tail
    g_apply = capture(torch, steps_fn(C, build=False), stream)

    def run_steps(n_chunks, with_tail):
        for _ in range(n_chunks):
            g_chunk.replay()
        if with_tail and g_tail is not None:
            g_tail.replay()

    # warm-up (W steps), and a load period so clock samples see a busy GPU
    if clocks is not None:
        clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(max(1, (W + C - 1) // C)):
            g_chunk.replay()
        torch.cuda.synchronize()
        t_end = time.perf_counter() + (args.load_seconds if clocks is not None else 0.0)
        while time.perf_counter() < t_end:
            run_steps(8, False)
            torch.cuda.synchronize()

    # timed region: exactly K steps
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        run_steps(K // C, True)
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    clk = clocks.stop() if clocks is not None else None
    ms_max = max_over_ranks(ms, world)

    # the applies alone: the same rotation without the segment builds
    reps = max(1, K // C)
    with torch.cuda.stream(stream):
        g_apply.replay()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(reps):
            g_apply.replay()
        a1.record(stream)
    torch.cuda.synchronize()
    apply_ms = a0.elapsed_time(a1) / (reps * C)
    moe = "gu" in sets[0]
    if moe:
        apply_ms /= 2.0     # two delta launches per step

    tokens_step = np.mean([sets[i % R]["tokens"] for i in range(K)])
    value = world * tokens_step * K / (ms_max / 1e3)
    alg_bytes = np.mean([sets[i % R]["alg"][0] for i in range(K)])
    alg_flops = np.mean([sets[i % R]["alg"][1] for i in range(K)])
    if moe:
        alg_bytes /= 2.0
        alg_flops /= 2.0
    hbm, tc, src = peaks()
    achieved = alg_bytes / (apply_ms / 1e3) / 1e9
    dense_small = (not moe) and sets[0]["fused"]
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": recorded_traffic(config),
                "kernel": "engine_kernel" if dense_small else "shrink_kernel + expand_kernel",
                "kernel_ms": apply_ms, "algorithmic_bytes": alg_bytes,
                "tflops": alg_flops / (apply_ms / 1e3) / 1e12, "peak_source": src + " (burst)"}
    e2e = run_e2e(args, sets, torch, lora, dev, stream, world, e2e_steps)
    out = {"value": value, "unit": "tokens/s", "ms_per_step": ms_max / K, "steps": K, "kernel_ms": apply_ms,
           "roofline": roofline, "e2e": e2e, "gpu_launches": gpu_launches, "clocks": clk,
           "step": ("build_segments + gate/up + down deltas" if moe else
                    "lora_build_and_apply (build_segments + apply; %s)" %
                    ("one launch" if dense_small else "build, shrink and expand launches")),
           "l2": "inputs larger than L2: %d rotating input sets, %.0f MB each" % (R, per_set / 1e6)}
    del sets, g_chunk, g_tail, g_apply
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


LINEAR_WORKLOAD = ("linear_prefill: the prefill batch through lora_linear (base projection x W^T with a random "
                   "bf16 W [4096][4096] and the LoRA delta in one kernel, y written, not read)")


def measure_linear(K, W, args, torch, lora, dev, e2e_steps):
    """The fused LoRA linear layer (lora_linear) on the prefill batch: K timed steps (build + linear) as
    CUDA-graph replays over rotating input sets (x, W, ids, table) larger than L2, the linear kernel alone,
    the same layer as a cuBLAS projection (torch.matmul) followed by lora_apply for comparison, and the
    end-to-end leg (x and ids in from pinned memory, y out)."""
    sets = []
    R = 7
    for j in range(R):
        p = make_problem("prefill", 1000 + j, base="zero")
        g = torch.Generator(device=dev).manual_seed(77 + j)
        s = {"p": p,
             "table": lora.lora_pack_weights([_to_dev(a, torch, dev) for a in p.A], [_to_dev(b, torch, dev) for b in p.B],
                                             p.ranks, p.scales, p.K, p.slice_n, p.n_a),
             "ws": lora.Workspace(p.M, p.L, device=dev),
             "ids": torch.from_numpy(p.ids).to(dev), "x": _to_dev(p.x, torch, dev),
             "W": (torch.randn(p.N, p.K, device=dev, generator=g) / p.K ** 0.5).to(torch.bfloat16),
             "y": torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev)}
        sets.append(s)
    torch.cuda.synchronize()

    def step(s, build=True, fused=True):
        if build:
            lora.lora_build_segments(s["ws"], s["ids"])
        if fused:
            lora.lora_linear(s["table"], s["ws"], s["x"], s["W"], s["y"])
        else:
            torch.matmul(s["x"], s["W"].t(), out=s["y"])
            lora.lora_apply(s["table"], s["ws"], s["x"], s["y"])

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):   # eager runs of both forms first (cuBLAS sets up outside any capture)
        for s in sets:
            step(s, fused=False)
            step(s)
    torch.cuda.synchronize()
    for s in sets:
        if lora.lora_get_status(s["ws"]) != lora.LORA_OK:
            raise RuntimeError("linear: device status")

    def graph(build, fused):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in sets:
                step(s, build, fused)
        return g

    def timed(g, reps):
        with torch.cuda.stream(stream):
            for _ in range(max(1, W // R + 1)):
                g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * R)

    reps = max(1, K // R)
    step_ms = timed(graph(True, True), reps)
    kernel_ms = timed(graph(False, True), reps)
    unfused_ms = timed(graph(False, False), reps)
    p = sets[0]["p"]
    _, lflops = dense_algorithmic(p)
    flops = 2.0 * p.M * p.N * p.K + lflops
    active = sorted(set(int(i) for i in p.ids if 0 <= i < p.L))
    # the active adapters' A and B, x and W read once, y written once, the ids
    nbytes = sum(2 * (p.A[i].size + p.B[i].size) for i in active) + 2 * (p.M * p.K + p.N * p.K + p.M * p.N) + 4 * p.M
    _, tc_peak, src = peaks()
    achieved = flops / (kernel_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s", "frac": achieved / tc_peak,
                "traffic": recorded_traffic("linear_prefill"), "kernel": "linear_kernel", "kernel_ms": kernel_ms, "algorithmic_bytes": nbytes,
                "algorithmic_flops": flops, "peak_source": src + " (burst)",
                "unfused_ms": unfused_ms, "unfused": "torch.matmul (cuBLAS) x W^T, then lora_apply on y"}
    # end to end: x and ids in from pinned memory, build + linear, y out; one step after another
    hx = [s["x"].cpu().pin_memory() for s in sets]
    hi = [s["ids"].cpu().pin_memory() for s in sets]
    hy = [torch.empty_like(s["y"], device="cpu", pin_memory=True) for s in sets]
    n = max(1, e2e_steps)
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            s = sets[i % R]
            s["x"].copy_(hx[i % R], non_blocking=True)
            s["ids"].copy_(hi[i % R], non_blocking=True)
            step(s)
            hy[i % R].copy_(s["y"], non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n
    tokens = p.M
    out = {"value": tokens / (step_ms / 1e3), "unit": "tokens/s", "ms_per_step": step_ms, "steps": reps * R,
           "kernel_ms": kernel_ms, "roofline": roofline,
           "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s", "steps": n,
                   "h2d_bytes_per_step": hx[0].numel() * 2 + hi[0].numel() * 4, "d2h_bytes_per_step": hy[0].numel() * 2,
                   "path": "public API calls with host-resident x and ids, one step after another on one stream"},
           "gpu_launches": 2 * reps * R, "workload": LINEAR_WORKLOAD}
    for s in sets:
        s["table"].destroy()
    del sets
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


EMBED_SOURCES = ("embedding.cu", "embedding.h", "common.cuh")
EMBED_WORKLOAD = ("embedding_decode: 32 tokens, 20 adapters (ranks cycling 16/32/64, 10% ids -1) over a 32768-entry "
                  "vocabulary, embedding width 4096, through lora_embedding_apply")


def measure_embedding(K, W, args, torch, lora, dev):
    """Embedding LoRA on a decode batch: K timed steps (build + lora_embedding_apply) as CUDA-graph replays over
    rotating input sets larger than L2, and the kernel alone; HBM roofline over the bytes the method moves."""
    from segmented_rank_gemm_lora_gb300 import synth
    V, N, R = 32768, 4096, 5
    sets = []
    for j in range(R):
        rng = np.random.default_rng(2000 + j)
        ids = synth.ids_decode(2000 + j)
        ranks = synth.cycle_ranks(20)
        A = [torch.randn(r, V, device=dev).to(torch.bfloat16) for r in ranks]
        B = [(torch.randn(N, r, device=dev) / r ** 0.5).to(torch.bfloat16) for r in ranks]
        s = {"ids": torch.from_numpy(ids).to(dev), "ids_np": ids, "ranks": ranks,
             "vocab": torch.from_numpy(rng.integers(0, V, len(ids)).astype(np.int32)).to(dev),
             "y": (torch.randn(len(ids), N, device=dev) * 4).to(torch.bfloat16),
             "table": lora.lora_pack_weights(A, B, ranks, [2.0] * len(ranks), V, [N], 1),
             "ws": lora.Workspace(len(ids), len(ranks), device=dev)}
        del A, B
        sets.append(s)
    stream = torch.cuda.Stream(device=dev)

    def step(s, build=True):
        if build:
            lora.lora_build_segments(s["ws"], s["ids"])
        lora.lora_embedding_apply(s["table"], s["ws"], s["vocab"], s["y"])

    with torch.cuda.stream(stream):
        for s in sets:
            step(s)
    torch.cuda.synchronize()
    for s in sets:
        if lora.lora_get_status(s["ws"]) != lora.LORA_OK:
            raise RuntimeError("embedding: device status")

    def timed(build, reps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for s in sets:
                step(s, build)
        with torch.cuda.stream(stream):
            for _ in range(max(1, W // R + 1)):
                g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * R)

    reps = max(1, K // R)
    step_ms = timed(True, reps)
    kernel_ms = timed(False, reps)
    ids, ranks = sets[0]["ids_np"], sets[0]["ranks"]
    active = sorted(set(int(i) for i in ids if i >= 0))
    Ma = int((ids >= 0).sum())
    # B once per active adapter, each token's A column (r values), y read and written, ids and vocabulary ids
    nbytes = sum(2 * N * ranks[i] for i in active) + sum(2 * ranks[int(i)] for i in ids if i >= 0) + Ma * 4 * N \
        + 8 * len(ids)
    hbm, _, src = peaks()
    achieved = nbytes / (kernel_ms / 1e3) / 1e9
    # end to end: ids, vocabulary ids and the base rows in from pinned memory, build + apply, rows out
    hi = [s["ids"].cpu().pin_memory() for s in sets]
    hv = [s["vocab"].cpu().pin_memory() for s in sets]
    hy = [s["y"].cpu().pin_memory() for s in sets]
    ho = [torch.empty_like(s["y"], device="cpu", pin_memory=True) for s in sets]
    n = 50
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            s = sets[i % R]
            s["ids"].copy_(hi[i % R], non_blocking=True)
            s["vocab"].copy_(hv[i % R], non_blocking=True)
            s["y"].copy_(hy[i % R], non_blocking=True)
            step(s)
            ho[i % R].copy_(s["y"], non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n
    e2e = {"value": len(ids) / (e2e_ms / 1e3), "unit": "tokens/s", "steps": n,
           "h2d_bytes_per_step": hi[0].numel() * 4 + hv[0].numel() * 4 + hy[0].numel() * 2,
           "d2h_bytes_per_step": ho[0].numel() * 2,
           "path": "public API calls with host-resident ids, vocabulary ids and base rows, one step after another"}
    out = {"value": len(ids) / (step_ms / 1e3), "unit": "tokens/s", "ms_per_step": step_ms, "steps": reps * R,
           "kernel_ms": kernel_ms,
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                        "traffic": recorded_traffic("embedding_decode"), "kernel": "embedding_kernel", "kernel_ms": kernel_ms,
                        "algorithmic_bytes": nbytes, "peak_source": src + " (burst)"},
           "e2e": e2e, "gpu_launches": 2 * reps * R, "workload": EMBED_WORKLOAD}
    for s in sets:
        s["table"].destroy()
    del sets
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


WORKLOADS = ("decode", "prefill", "stacked_qkv", "stacked_gate_up", "stacked_down", "moe")


def run_ours(args, world, rank, local):
    import torch
    from segmented_rank_gemm_lora_gb300 import lora
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lora.load()

    K, W = args.steps, args.warmup
    head = measure(args.config, K, W, args, torch, lora, dev, world, min(args.steps, args.e2e_steps),
                   clocks=ClockSampler(local))
    # every workload of the benchmark, measured the same way in the same run (fewer steps each)
    per = {}
    if args.per_workload:
        for name in WORKLOADS:
            r = head if name == args.config else measure(name, max(50, min(K, args.workload_steps)), W, args,
                                                         torch, lora, dev, world, min(args.workload_steps, 100))
            per[name] = {k: r[k] for k in ("value", "unit", "ms_per_step", "steps", "kernel_ms", "roofline", "e2e",
                                            "gpu_launches")}
            per[name]["workload"] = CONFIGS[name]
        per["linear_prefill"] = measure_linear(max(49, min(K, args.workload_steps)), W, args, torch, lora, dev,
                                               min(args.workload_steps, 20))
        per["embedding_decode"] = measure_embedding(max(50, min(K, args.workload_steps)), W, args, torch, lora, dev)

    cpu = cpu_baseline(args.config, args.cpu_seconds) if (rank == 0 and world == 1 and args.cpu_seconds > 0) else None
    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": K,
                "warmup": W, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": "%s: %s" % (args.config, CONFIGS[args.config]), "step": head["step"],
                           "l2": head["l2"], "parallelism": "replicas x%d" % world},
                "gpu_launches": head["gpu_launches"], "roofline": head["roofline"], "e2e": head["e2e"],
                "clocks": head["clocks"], "cpu_baseline": cpu, "per_workload": per}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, sets, torch, lora, dev, stream, world, e2e_steps):
    """Same metric through the public API with host-resident inputs: every step copies its inputs (ids, x
    and y_base, or the MoE caches) from pinned host memory, as one copy of the buffer they share on the
    device, builds, applies, and copies the result back."""
    R = len(sets)
    host = [{"packed": s["packed"].cpu().pin_memory()} for s in sets[:min(R, 8)]]
    outs = [{k: torch.empty_like(s[k], device="cpu", pin_memory=True) for k in (("c1", "c3") if "gu" in s else ("y",))}
            for s in sets[:min(R, 8)]]
    h2d = d2h = 0

    def one(i):
        nonlocal h2d, d2h
        s, h, o = sets[i % len(host)], host[i % len(host)], outs[i % len(host)]
        h2d = d2h = 0
        for k in h:
            s[k].copy_(h[k], non_blocking=True)
            h2d += h[k].numel() * h[k].element_size()
        step(s, lora)
        for k in o:
            o[k].copy_(s[k], non_blocking=True)
            d2h += o[k].numel() * o[k].element_size()

    K = max(1, e2e_steps)
    H = len(host)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # eager: every step's copies and calls issued from Python
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            one(i)
        torch.cuda.synchronize()
        barrier(world)
        e0.record(stream)
        for i in range(K):
            one(i)
        e1.record(stream)
    torch.cuda.synchronize()
    ms_eager = max_over_ranks(e0.elapsed_time(e1), world)
    # pipelined, as a serving loop runs it: each step's copy-in, compute and copy-out sit on three streams,
    # so step i+1's inputs travel while step i computes and step i-1's output returns; every step still
    # moves all of its bytes.  H consecutive steps (one per pinned host set) are captured once in a CUDA
    # graph with those cross-stream dependencies, and the graph is replayed.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fork = torch.cuda.Event()
        fork.record(stream)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        for j in range(H):
            sj, hj, oj = sets[j], host[j], outs[j]
            e_in, e_done = torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(s_in):
                for k in hj:
                    sj[k].copy_(hj[k], non_blocking=True)
                e_in.record(s_in)
            stream.wait_event(e_in)
            step(sj, lora)
            e_done.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e_done)
                for k in oj:
                    oj[k].copy_(sj[k], non_blocking=True)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
    # the host link makes this leg noisy from run to run: it is timed in five repeats, and the value is their
    # median, with the spread beside it
    reps = max(1, K // H)
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup // H)):
            g.replay()
    torch.cuda.synchronize()
    rep_ms = []
    for _ in range(5):
        barrier(world)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        rep_ms.append(max_over_ranks(e0.elapsed_time(e1), world))
    ms_pipe = float(np.median(rep_ms))
    tok_pipe = np.mean([sets[j]["tokens"] for j in range(H)])
    tok_serial = np.mean([sets[i % H]["tokens"] for i in range(K)])
    rate = lambda ms: world * tok_pipe * reps * H / (ms / 1e3)
    return {"value": rate(ms_pipe), "unit": "tokens/s",
            "spread": {"repeats": len(rep_ms), "median": rate(ms_pipe), "min": rate(max(rep_ms)),
                       "max": rate(min(rep_ms))},
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": reps * H,
            "path": "public API calls through the Python binding with host-resident inputs: per step, copy-in of "
                    "the inputs from pinned memory, build + apply, copy-out of the output to pinned memory, on "
                    "three streams so consecutive steps overlap; %d steps captured in one CUDA graph" % H,
            "serial_value": world * tok_serial * K / (ms_eager / 1e3),
            "serial_path": "the same calls one step after another on one stream, issued from Python"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--load-seconds", type=float, default=1.0)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="stacked_gate_up", choices=sorted(CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload-steps", type=int, default=1000,
                    help="timed steps of each per_workload entry (the headline workload uses --steps)")
    ap.add_argument("--no-per-workload", dest="per_workload", action="store_false")
    ap.add_argument("--linear-only", action="store_true",
                    help="measure only the fused LoRA linear layer (the per_workload linear_prefill entry) and "
                         "print it as one JSON line (for profiling that kernel)")
    ap.add_argument("--embedding-only", action="store_true",
                    help="measure only the embedding LoRA (the per_workload embedding_decode entry) and print it "
                         "as one JSON line (for profiling that kernel)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_env()
    if args.linear_only or args.embedding_only:
        import torch
        from segmented_rank_gemm_lora_gb300 import lora
        torch.cuda.set_device(local)
        lora.load()
        dev = torch.device("cuda", local)
        r = (measure_linear(args.steps, args.warmup, args, torch, lora, dev, args.e2e_steps) if args.linear_only
             else measure_embedding(args.steps, args.warmup, args, torch, lora, dev))
        print(json.dumps(r), flush=True)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
