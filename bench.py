"""Benchmark of the trellis MoE hot path on GB300.

Workload: one full MoE block of a Qwen3.6-35B-A3B-style Escha-W2 layer at
decode batch 1 (hidden 2048, 256 experts, top-8, gate_up 1024x2048 at K=3,
down 2048x512 at K=2, int8 w8a16 shared expert), seeded synthetic weights and
activations (x ~ N(0,1) in fp16; a fresh token every step, so the routed
experts change). One step = one MoE block forward of one token: router
(logits, top-8, softmax), input Hadamard transforms, fused trellis decode
GEMVs for gate_up and down, output transforms, SwiGLU, the int8 shared expert
and the combine, all in the library's kernels behind the C ABI, replayed from
a CUDA graph of 8 steps, which run as one escha_moe_blocks call: one launch
each of the router, gate_up and down/combine kernels over the 8 blocks'
slots (--path sequence: the same call held on the one-launch sequence kernel;
--path per-slot: one escha_moe_block call per step).

L2: inputs larger than L2. The benchmark cycles through 24 distinct layers of
this shape (about 6.5 GB of weights), one layer per step, so a step's weights
were last touched 23 steps (hundreds of MB of other traffic) earlier and come
from HBM, while the kernels' code stays cached as it would in a model.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from escha_synth import gen  # noqa: E402

METRIC = "MoE-layer tokens/s (decode batch 1), packed-expert HBM GB/s as a fraction of peak"
UNIT = "tokens/s"
WORKLOAD = ("Qwen3.6-35B-A3B-style Escha-W2 MoE block, decode batch 1: hidden 2048, 256 experts, top-8, "
            "gate_up 1024x2048 K=3, down 2048x512 K=2, int8 w8a16 shared expert 1024x2048/2048x512")
LAYER_SEED = 1002
X_SEED = 2002
HIDDEN, INTER, E, TOPK = 2048, 512, 256, 8
GU_CODE_BYTES = HIDDEN * 2 * INTER * 3 // 8  # per expert: 786,432
DN_CODE_BYTES = INTER * HIDDEN * 2 // 8  # per expert: 262,144
N_LAYERS = 24
STEPS_PER_GRAPH = 8
KERNELS_PER_STEP = 3  # router (+shared gate_up), gate_up (+top-k), down (+top-k, shared down, combine)


# Algorithmic bytes of one launch of the gate_up kernel at batch 1: 8 routed
# experts' codes, rin and rout, x once, the token's 256 f16 logits, the
# 8 x 1024 f32 outputs (the shared expert's gate_up runs in the router grid).
GATE_UP_KERNEL_BYTES = (TOPK * (GU_CODE_BYTES + HIDDEN * 2 + 2 * INTER * 2) + HIDDEN * 2 + E * 2
                        + TOPK * 2 * INTER * 4)


# Routed weights decoded by one launch of the gate_up kernel at batch 1, by a
# whole block (gate_up and down of 8 experts), and the issue peak of the GPU
# (warp-instructions per second: 152 SMs x 4 schedulers x 1 per clock).
GU_WEIGHTS = TOPK * HIDDEN * 2 * INTER
BLOCK_WEIGHTS = TOPK * (HIDDEN * 2 * INTER + INTER * HIDDEN)
ALU_OPS_PER_WEIGHT = 6  # the algorithm's minimum: window, hash multiply, and-xor, fp16 add, conversion, fma
ALU_PEAK_WARP_INSTR = 152 * 4 * 2.07e9
# Algorithmic bytes of the cooperative expert kernel of the batch-1 block: 8
# experts' codes, rin and rout of both projections, the shared expert's int8
# down rows and their scales, x, the logits, the shared gate_up outputs and
# the f32 output.
FUSED_KERNEL_BYTES = (TOPK * (GU_CODE_BYTES + DN_CODE_BYTES + (HIDDEN + 2 * INTER) * 2 + (INTER + HIDDEN) * 2)
                      + HIDDEN * INTER + HIDDEN * 4 + HIDDEN * 2 + E * 2 + 2 * INTER * 4 + HIDDEN * 4)
# Algorithmic bytes of one batch-1 block: 8 experts' codes, rin and rout of
# both projections, the router weights, the int8 shared expert (weights, row
# scales, gate vector), x in and the f32 output out.
BLOCK_BYTES = (TOPK * (GU_CODE_BYTES + DN_CODE_BYTES + (HIDDEN + 2 * INTER) * 2 + (INTER + HIDDEN) * 2)
               + E * HIDDEN * 2 + 3 * HIDDEN * INTER + (2 * INTER + HIDDEN) * 4 + HIDDEN * 2
               + HIDDEN * 2 + HIDDEN * 4)


def _profile_record(name: str, mode=None):
    """A committed ncu figure (profiles/<name>.json) of the bench mode `mode`,
    or None when it is another mode's or the kernel sources it depends on
    changed since the capture."""
    import hashlib

    p = os.path.join(ROOT, "profiles", name + ".json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    if rec.get("mode") != mode:
        return None
    h = hashlib.sha256()
    for src in rec["sources"]:
        with open(os.path.join(ROOT, "bit_trellis_quantized_gb300", "csrc", src), "rb") as f:
            h.update(f.read())
    return rec if h.hexdigest() == rec["sources_sha256"] else None


def measured_traffic(mode=None):
    """DRAM bytes per launch of the batch-1 block's dominant kernel in bench
    mode `mode` from the committed ncu capture, or None (another mode's, or
    the kernel sources changed since the capture)."""
    rec = _profile_record("traffic", mode)
    return rec["dram_bytes_per_launch"] if rec else None


def measured_instr_per_weight(mode=None):
    """Executed warp-instructions x 32 per decoded weight of the batch-1
    block's kernel (ncu smsp__inst_executed.sum over the launch, divided by
    the weights it decodes), or None without a current capture."""
    rec = _profile_record("traffic", mode)
    return rec.get("instructions_per_weight") if rec else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def replica_seeds(rank: int):
    """Seeds of one replica's layers and token stream: every rank runs its own
    independent stream (replicas, weak scaling)."""
    return LAYER_SEED + 1000 * rank, X_SEED + 100 * rank


def max_over_ranks(values, dist_mod=None, device=None):
    """Element-wise maximum of per-rank timings over all ranks (the slowest
    rank defines the job's time); identity on one process."""
    if dist_mod is None:
        return [float(v) for v in values]
    import torch

    tt = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist_mod.all_reduce(tt, op=dist_mod.ReduceOp.MAX)
    return [float(v) for v in tt.tolist()]


def aggregate_tokens_per_s(world_size: int, ms_per_step: float, tokens_per_step: int = 1) -> float:
    """Whole-job throughput: every rank processes tokens_per_step per step."""
    return world_size * tokens_per_step * 1e3 / ms_per_step


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed loops run."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # raw samples: $ESCHA_CLOCKS_DIR if set, else the system temp directory
        out_dir = os.environ.get("ESCHA_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"escha_clocks_rank{gpu_index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            # the timed loops start only once the sampler is producing samples
            t_end = time.time() + 5.0
            while time.time() < t_end and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
                time.sleep(0.01)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3][1:5]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(loaded), "power_w_max": max(r[2] for r in rows)}


def host_info():
    """Core count and CPU model of the host the oracle runs on."""
    import platform

    model = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k = line.split(":")[0].strip().lower()
                if k in ("model name", "cpu part", "hardware"):
                    model = line.split(":", 1)[1].strip() if k == "model name" else f"{platform.machine()} {k} " + \
                        line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"cpu_count": os.cpu_count(), "machine": platform.machine(), "cpu": model}


def _oracle_tokens(args):
    """Worker of the all-core leg: the oracle on a few tokens of the batch-1
    block (its own process, one thread)."""
    seed, x_seed, first, n = args
    from oracle import escha_oracle as o

    layer = o.MoeLayer(**gen.moe_layer(seed))
    xs = gen.fp16_normal(gen.rng(x_seed), (first + n, HIDDEN))
    for t in range(first, first + n):
        o.moe_block(layer, xs[t:t + 1], k=TOPK)
    return n


def r_skip_rates(layer, xs, o):
    """How often down_proj's 16-input strips are exactly zero on these tokens
    (oracle values): before its input Hadamard (h = SwiGLU of gate_up, where
    the gate/up prune mask zeroes channels) and after it (the x~ a tile-exact
    skip would test)."""
    pre = post = strips = 0
    ids, w, _ = o.route(xs, layer.Wg, TOPK)
    for b in range(xs.shape[0]):
        xv = o.f16_to_f64(xs[b].view(np.uint16))
        for j in range(TOPK):
            e = int(ids[b, j])
            y = o.trellis_gemv(None, xv, o.f16_to_f64(layer.gu_rin[e].view(np.uint16)),
                               o.f16_to_f64(layer.gu_rout[e].view(np.uint16)), W=layer.expert_weights("gu", e))
            h = o.swiglu(y)
            xt = o.input_transform(h, o.f16_to_f64(layer.dn_rin[e].view(np.uint16)))
            strips += h.size // 16
            pre += int(np.sum(np.all(h.reshape(-1, 16) == 0, axis=1)))
            post += int(np.sum(np.all(xt.reshape(-1, 16) == 0, axis=1)))
    return {"tokens": int(xs.shape[0]), "strips": strips, "zero_strips_before_hadamard": pre,
            "zero_strips_after_hadamard": post, "hit_rate": post / max(strips, 1),
            "note": "16-input strips of down_proj's input whose values are all exactly 0 (oracle, float64): after "
                    "the input Hadamard (what a tile-exact skip tests) and, for reference, before it"}


def cpu_baseline(seconds: float = 15.0, max_tokens: int = 8):
    """The CPU oracle as it stands, on the host cores, over a bounded sample
    of the same workload (whole tokens of the MoE block at batch 1): one
    thread, then every core (one process per core, tokens split over them,
    the same arithmetic)."""
    import multiprocessing as mp

    from oracle import escha_oracle as o

    d = gen.moe_layer(LAYER_SEED)
    layer = o.MoeLayer(**d)
    xs = gen.fp16_normal(gen.rng(X_SEED + 777), (max_tokens, HIDDEN))
    t0 = time.perf_counter()
    n = 0
    while n < max_tokens:
        o.moe_block(layer, xs[n:n + 1], k=TOPK)
        n += 1
        if time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    one = n / dt
    info = host_info()
    cores = max(1, int(info["cpu_count"] or 1))
    # all cores: each process decodes its tokens' experts itself, as the
    # one-thread leg does; 2 tokens per process
    per = 2
    jobs = [(LAYER_SEED, X_SEED + 999, i * per, per) for i in range(cores)]
    ctx = mp.get_context("spawn")
    t1 = time.perf_counter()
    with ctx.Pool(cores) as pool:
        done = sum(pool.map(_oracle_tokens, jobs))
    dt_all = time.perf_counter() - t1
    return {"value": one, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} tokens of the batch-1 MoE block through the numpy float64 oracle, one thread, "
                      f"{dt:.1f} s",
            "all_cores": {"value": done / dt_all, "unit": UNIT, "cores": cores,
                          "sample": f"{done} tokens, {per} per process on {cores} processes (spawned, one thread "
                                    f"each), {dt_all:.1f} s including process start-up"},
            "host": info,
            "r_skip": r_skip_rates(layer, xs[:min(n, 4)], o)}


def run_reference(args, rank):
    """The oracle on the host cores, as it stands: exactly args.steps timed
    steps after args.warmup untimed ones. A step is one eighth of a token
    (one of its 8 routed experts: gate_up, SwiGLU, down, weighted; the
    token's router runs at its first step, the shared expert and the combine
    at its last), so 8 steps are one token of the MoE block and the whole run
    stays within minutes; value = tokens per second = steps / 8 / time."""
    if rank != 0:
        return
    from oracle import escha_oracle as o

    d = gen.moe_layer(LAYER_SEED)
    layer = o.MoeLayer(**d)
    n_tok = -(-(args.warmup + args.steps) // TOPK) + 1
    xs = gen.fp16_normal(gen.rng(X_SEED), (n_tok, HIDDEN))
    state = {}

    def step(i):  # slot j of token t
        t, j = divmod(i, TOPK)
        if j == 0:
            ids, w, _ = o.route(xs[t:t + 1], layer.Wg, TOPK)
            state.update(ids=ids, w=w, acc=np.zeros(HIDDEN))
        xv = xs[t].astype(np.float64)
        state["acc"] += state["w"][0, j] * o.moe_expert(layer, state["ids"][0, j], xv)
        if j == TOPK - 1:
            state["out"] = state["acc"] + o.shared_expert(layer, xs[t:t + 1])[0]

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        step(i)
    elapsed = time.perf_counter() - t0
    ms = 1e3 * elapsed / args.steps
    value = args.steps / TOPK / elapsed
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": 1, "l2": "n/a (CPU)",
                       "step": "one routed expert of one token (8 steps = 1 token)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} steps = {args.steps / TOPK:g} tokens of the batch-1 MoE block "
                                       f"through the numpy float64 oracle, one thread, {elapsed:.1f} s"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, ws, rank, local):
    import torch

    from bit_trellis_quantized_gb300 import native
    from escha_synth.gen_torch import moe_layer_device

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    # NL distinct layers (~272 MB each): a step's weights were last touched
    # NL-1 steps earlier, far more than L2 holds, so they come from HBM.
    n_layers = args.layers
    layer_seed, x_seed = replica_seeds(rank)
    blocks = [native.MoeBlock(moe_layer_device(layer_seed + l, dev), device=dev, topk=TOPK)
              for l in range(n_layers)]
    # the steps of a graph run as one escha_moe_blocks call (by shape: the
    # per-slot kernels over all 8 blocks; --path sequence holds it on the
    # one-launch sequence kernel), or with --path per-slot as one
    # escha_moe_block call (three kernels) per step
    sequence = args.path in ("blocks", "sequence")  # one escha_moe_blocks call per graph
    native.lib()
    native.set_blocks_route(2 if args.path == "sequence" else 0)
    path = args.path if sequence else blocks[0].path(1)
    seq_ws = torch.empty(native.seq_workspace_bytes(blocks[:STEPS_PER_GRAPH]), dtype=torch.uint8, device=dev)
    n_total = args.warmup + args.steps
    xs_host = torch.from_numpy(gen.fp16_normal(gen.rng(x_seed), (n_total, HIDDEN))).pin_memory()
    xs = xs_host.to(dev)
    outs = torch.empty((n_total, HIDDEN), dtype=torch.float32, device=dev)
    ids_all = torch.empty((n_total, TOPK), dtype=torch.int32, device=dev)
    w_all = torch.empty((n_total, TOPK), dtype=torch.float32, device=dev)
    layer_of = [i % n_layers for i in range(n_total)]

    # One CUDA graph holds up to STEPS_PER_GRAPH consecutive steps (as a
    # model's decode graph holds its layers): whole graphs of warm-up steps,
    # then exactly args.steps timed steps (a shorter last graph when needed).
    # Like every kernel of the library, a step's first kernel is launched
    # programmatically: it loads router weights while the previous step's
    # last kernel finishes and waits for it before touching x or outputs.
    chunks = [(i0, STEPS_PER_GRAPH) for i0 in range(0, args.warmup, STEPS_PER_GRAPH)]
    chunks += [(i0, min(STEPS_PER_GRAPH, n_total - i0)) for i0 in range(args.warmup, n_total, STEPS_PER_GRAPH)]
    stream = torch.cuda.Stream(device=dev)

    def run_chunk(i0, n, events=None):
        """Steps i0 .. i0+n-1 on the current stream (events: four CUDA events
        recorded between the call's kernels)."""
        if sequence:
            idx = range(i0, i0 + n)
            native.moe_blocks([blocks[layer_of[i]] for i in idx], [xs[i] for i in idx], [outs[i] for i in idx],
                              ids=[ids_all[i] for i in idx], w=[w_all[i] for i in idx], ws=seq_ws, events=events)
        else:
            for i in range(i0, i0 + n):
                blocks[layer_of[i]](xs[i:i + 1], out=outs[i:i + 1], ids=ids_all[i:i + 1], w=w_all[i:i + 1])

    graphs = []
    with torch.cuda.stream(stream):
        for blk in blocks:  # workspaces sized and kernels loaded before capture
            blk(xs[0:1], out=outs[0:1], ids=ids_all[0:1], w=w_all[0:1])
        run_chunk(0, min(STEPS_PER_GRAPH, n_total))
        torch.cuda.synchronize()
        for i0, n in (chunks if not args.no_graph else []):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run_chunk(i0, n)
            graphs.append(g)
    torch.cuda.synchronize()
    n_warm_graphs = args.warmup // STEPS_PER_GRAPH

    with ClockSampler(local) as clk:
        # device-resident inputs: x already in HBM when the timed region starts
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            if args.no_graph:  # direct launches (for profilers)
                for i0, n in chunks[:n_warm_graphs]:
                    run_chunk(i0, n)
                barrier()
                t0.record(stream)
                for i0, n in chunks[n_warm_graphs:]:
                    run_chunk(i0, n)
                t1.record(stream)
                barrier()
            else:
                for g in graphs[:n_warm_graphs]:
                    g.replay()
                barrier()
                t0.record(stream)
                for g in graphs[n_warm_graphs:]:
                    g.replay()
                t1.record(stream)
                barrier()
        step_ms = t0.elapsed_time(t1) / args.steps

        # end to end through the public API: pinned host x in, out back to host.
        # Each group of steps (the chunks above) is one graph: its steps run on
        # the launch stream while a copy stream brings the next group's inputs
        # in from pinned host memory and sends the previous group's outputs
        # back, as a serving loop overlaps its I/O with compute. The timed
        # region also holds the first timed group's input copy and the last
        # group's output copy, so every timed step's input and output cross to
        # and from the host inside it.
        out_host = torch.empty((n_total, HIDDEN), dtype=torch.float32).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_groups = len(chunks)
        copy_stream = torch.cuda.Stream(device=dev)

        def h2d(gi):
            i0, n = chunks[gi]
            xs[i0:i0 + n].copy_(xs_host[i0:i0 + n], non_blocking=True)

        def d2h(gi):
            i0, n = chunks[gi]
            out_host[i0:i0 + n].copy_(outs[i0:i0 + n], non_blocking=True)

        def e2e_group(gi):
            i0, n = chunks[gi]
            fork, join = torch.cuda.Event(), torch.cuda.Event()
            fork.record(stream)
            copy_stream.wait_event(fork)
            with torch.cuda.stream(copy_stream):
                if gi + 1 < n_groups:
                    h2d(gi + 1)
                if gi > 0:
                    d2h(gi - 1)
                join.record(copy_stream)
            run_chunk(i0, n)
            stream.wait_event(join)

        e2e_graphs = []
        if not args.no_graph:
            with torch.cuda.stream(stream):
                for gi in range(n_groups):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        e2e_group(gi)
                    e2e_graphs.append(g)
            torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            h2d(0)
            for gi in range(n_warm_graphs):
                e2e_group(gi) if args.no_graph else e2e_graphs[gi].replay()
            barrier()
            e0.record(stream)
            h2d(n_warm_graphs)
            for gi in range(n_warm_graphs, n_groups):
                e2e_group(gi) if args.no_graph else e2e_graphs[gi].replay()
            d2h(n_groups - 1)
            e1.record(stream)
            barrier()
        # every timed step's output reached the host
        assert torch.equal(out_host[args.warmup:], outs[args.warmup:].cpu())
        e2e_ms = e0.elapsed_time(e1) / args.steps
        del e2e_graphs

        # per-kernel durations, timed live by events on the launch stream
        # between the kernels (the events serialise them): per call of up to
        # 8 steps the router, gate_up and down/combine kernels over all its
        # blocks (or the one sequence launch), or the three per-slot kernels
        # of each step
        if sequence:
            kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in chunks]
            with torch.cuda.stream(stream):
                for row in kev:  # torch creates the CUDA events lazily, at their first record
                    for e in row:
                        e.record(stream)
                barrier()
                for (i0, n), row in zip(chunks, kev):
                    run_chunk(i0, n, events=row)
                barrier()
            # (ms of each interval, steps) per timed call
            seq_launch = [([row[j].elapsed_time(row[j + 1]) for j in range(3)], n)
                          for (i0, n), row in list(zip(chunks, kev))[n_warm_graphs:]]
            phase = None
        else:
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_total)]
            with torch.cuda.stream(stream):
                for row in evs:  # torch creates the CUDA events lazily, at their first record
                    for e in row:
                        e.record(stream)
                torch.cuda.synchronize()
                handles = [(native.ctypes.c_void_p * 4)(*[e.cuda_event for e in row]) for row in evs]
                barrier()
                for i in range(n_total):
                    blk = blocks[layer_of[i]]
                    ws_t = blk.workspace(1)
                    native.check(native.lib().escha_moe_block_timed(
                        native.ctypes.byref(blk.layer), native.ptr(xs[i:i + 1]), 1, native.ptr(outs[i:i + 1]),
                        native.ptr(ids_all[i:i + 1]), native.ptr(w_all[i:i + 1]), native.ptr(ws_t), ws_t.numel(),
                        stream.cuda_stream, handles[i]))
                barrier()
            phase = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(3)]
                              for i in range(args.warmup, n_total)])
        status = int(seq_ws[:4].view(torch.int32).item()) if sequence else 0
    clocks = clk.summary()

    # max over ranks
    t_step, t_e2e = max_over_ranks([step_ms, e2e_ms], pg, dev)
    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return

    hbm, tflops, src = peaks()
    fused = path == native.ESCHA_PATH_FUSED
    blocks_mode = args.path == "blocks"
    if blocks_mode:
        # the dominant kernel: the gate_up kernel over the 8 blocks' slots of
        # one escha_moe_blocks call (calls of 8 steps; its work scales with n)
        full = [iv for iv, n in seq_launch if n == STEPS_PER_GRAPH] or [iv for iv, n in seq_launch]
        ph = np.array(full).mean(axis=0)  # router (+ shared gate_up), gate_up, down (+ shared down, combine) (ms)
        k_ms = float(ph[1])
        k_bytes, k_weights = STEPS_PER_GRAPH * GATE_UP_KERNEL_BYTES, STEPS_PER_GRAPH * GU_WEIGHTS
        k_name = (f"moe_gate_up_kernel<K=3> over {STEPS_PER_GRAPH} blocks' slots ({STEPS_PER_GRAPH * TOPK} "
                  f"(token, expert) pairs, each with its own layer's expert)")
        phase_ms = {"router+shared_gate_up": float(ph[0]), "gate_up": float(ph[1]),
                    "down+shared_down+combine": float(ph[2]),
                    "per_block_serialised": float(ph.sum() / STEPS_PER_GRAPH)}
    elif sequence:
        # the dominant kernel: the sequence kernel, per launch of n steps (n = 8
        # but for a shorter last launch); its work scales with n
        per_block = [iv[0] / n for iv, n in seq_launch]
        launch_ms = [iv[0] for iv, n in seq_launch if n == STEPS_PER_GRAPH] or [iv[0] for iv, n in seq_launch]
        k_ms = float(np.mean(launch_ms))
        k_bytes, k_weights = STEPS_PER_GRAPH * BLOCK_BYTES, STEPS_PER_GRAPH * BLOCK_WEIGHTS
        k_name = (f"moe_multi_kernel ({STEPS_PER_GRAPH} independent one-token blocks per launch: router, top-k, "
                  f"gate_up, down, shared expert, combine of each)")
        phase_ms = {"sequence_kernel_per_launch": k_ms, "per_block": float(np.mean(per_block))}
    elif fused:
        ph = phase.mean(axis=0)
        k_ms, k_bytes, k_weights = float(ph[1]), FUSED_KERNEL_BYTES, BLOCK_WEIGHTS
        k_name = f"moe_fused_kernel<3,2> (top-k, {TOPK} experts' gate_up and down, the shared expert's down rows, " \
                 f"combine; one cooperative grid)"
        phase_ms = {"router+shared_gate_up": float(ph[0]), "fused_experts": float(ph[1])}
    else:
        ph = phase.mean(axis=0)  # router (+shared gate_up), gate_up, down (+shared down, combine) (ms)
        k_ms, k_bytes, k_weights = float(ph[1]), GATE_UP_KERNEL_BYTES, GU_WEIGHTS
        k_name = "moe_gate_up_kernel<K=3> (8 routed experts)"
        phase_ms = {"router+shared_gate_up": float(ph[0]), "gate_up": float(ph[1]),
                    "down+shared_down+combine": float(ph[2])}
    achieved = k_bytes / (k_ms * 1e-3) / 1e9
    prof_mode = args.path if sequence else None  # the committed ncu record covers one mode's dominant kernel
    ipw = measured_instr_per_weight(prof_mode)
    ops = ipw if ipw else ALU_OPS_PER_WEIGHT
    routed_code_bytes = TOPK * (GU_CODE_BYTES + DN_CODE_BYTES)
    distinct = len({tuple(r) for r in ids_all[args.warmup:args.warmup + 16].cpu().numpy().tolist()})
    line = {
        "metric": METRIC, "value": aggregate_tokens_per_s(ws, t_step), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "dtype_note": "f32 arithmetic on fp16 weights decoded from 2/3-bit trellis codes (int8 shared expert)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 1, "tokens_per_step_per_gpu": 1,
                   "l2": f"inputs larger than L2: {n_layers} distinct MoE layers "
                         f"({n_layers * 272} MB) cycled, one per step, no flush",
                   "cuda_graph": ("none (direct launches)" if args.no_graph else
                                  f"up to {STEPS_PER_GRAPH} steps per graph") +
                                 ("; the steps of a graph as one escha_moe_blocks call: the router, gate_up and "
                                  "down kernels over all its blocks" if blocks_mode else
                                  "; the steps of a graph as one sequence launch (escha_moe_blocks)" if sequence else
                                  "; one escha_moe_block call per step (programmatic launches)"),
                   "parallelism": f"replicas x{ws} (independent token streams)"},
        # The dominant kernel is bound by instruction issue for the decode,
        # not by HBM: its roofline is the issue peak (152 SMs x 4 schedulers
        # x 1 warp-instruction per clock at the maximum SM clock) against the
        # warp-instructions its decoded weights cost: the instructions per
        # weight ncu counted on this kernel (smsp__inst_executed.sum over the
        # launch / weights decoded; profiles/traffic.json), else the
        # algorithm's 6 operations (16-bit window, hash multiply, and-xor,
        # fp16 add, conversion, f32 fma). `traffic` is the kernel's measured
        # DRAM bytes per launch.
        "roofline": {"bound": "alu", "achieved": k_weights * ops / 32 / (k_ms * 1e-3) / 1e12,
                     "peak": ALU_PEAK_WARP_INSTR / 1e12, "unit": "T warp-instructions/s",
                     "frac": k_weights * ops / 32 / (k_ms * 1e-3) / ALU_PEAK_WARP_INSTR,
                     "traffic": measured_traffic(prof_mode), "algorithmic_bytes_per_launch": k_bytes,
                     "kernel": k_name, "decoded_weights_per_launch": k_weights,
                     "instructions_per_weight": ops,
                     "instructions_per_weight_source": "ncu smsp__inst_executed.sum / weights (profiles/traffic.json)"
                     if ipw else "assumed: the algorithm's 6 operations per weight",
                     "ms_per_launch": k_ms, "peak_source": "derived: 152 SMs x 4 x 2.07e9 /s"},
        # the same launch against the measured HBM copy bandwidth
        "roofline_hbm": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": measured_traffic(prof_mode), "algorithmic_bytes_per_launch": k_bytes,
                         "ms_per_launch": k_ms, "peak_source": src},
        "packed_expert_gbs": routed_code_bytes / (t_step * 1e-3) / 1e9,
        "packed_expert_frac": routed_code_bytes / (t_step * 1e-3) / 1e9 / hbm,
        "phase_ms": phase_ms,
        "block_path": {"blocks": f"escha_moe_blocks: the per-slot kernels over {STEPS_PER_GRAPH} blocks' slots "
                                 f"(3 launches per {STEPS_PER_GRAPH} steps)",
                       "sequence": f"escha_moe_blocks: one cooperative launch per {STEPS_PER_GRAPH} steps",
                       native.ESCHA_PATH_FUSED: "router kernel + cooperative expert kernel per step",
                       native.ESCHA_PATH_SLOT: "per-slot (three kernels per step)"}.get(path, str(path)),
        "status_word": status,
        "gpu_launches": (3 if blocks_mode else 1) * len(chunks[n_warm_graphs:]) if sequence
        else (2 if fused else KERNELS_PER_STEP) * args.steps,
        "e2e": {"value": aggregate_tokens_per_s(ws, t_e2e), "unit": UNIT, "h2d_bytes_per_step": HIDDEN * 2,
                "d2h_bytes_per_step": HIDDEN * 4,
                "note": f"per group of up to {STEPS_PER_GRAPH} steps, one graph: the steps, and on a copy stream "
                        f"the next group's x in from pinned host memory and the previous group's outputs back "
                        f"to pinned host; the first timed input copy and the last output copy are in the timed "
                        f"region too"},
        "clocks": clocks,
        "routing_distinct_in_16_steps": distinct,
    }
    if ws == 1 and not args.no_extended:
        line["configs"] = extended(dev, blocks, hbm, tflops)
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def _time_graph(torch, stream, fn, reps: int, warm: int = 3, replays: int = 20):
    """ms per call of fn: the calls are captured once into a CUDA graph
    holding `reps` calls (fn(i) issues call i), replayed `warm` times, then
    `replays` times, each replay bracketed by CUDA events on the launching
    stream. Returns (median, min, max) over the replays, in ms per call."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn(0)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(reps):
                fn(i)
        for _ in range(warm):
            g.replay()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
        for a, b in evs:
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
    t = sorted(a.elapsed_time(b) / reps for a, b in evs)
    return statistics.median(t), t[0], t[-1]


def _stats(t):
    """{median, min, max} in microseconds of a (median, min, max) in ms."""
    return {"us_median": t[0] * 1e3, "us_min": t[1] * 1e3, "us_max": t[2] * 1e3}


def extended(dev, blocks, hbm, tflops):
    """The other workloads of the benchmark's configuration list, each with
    inputs larger than L2 (distinct weights cycled) unless stated:
    single projection at batch 1, the dense 5120 x 17408 linear at M = 1..2048,
    the MoE block at batch 8 / 16 / 64 / 256 and a
    2048-token prefill chunk, the int8 w8a16 shapes at M = 1 and 2048, and
    the 40-block stack at batch 1 / 8 / 128 and a 2048-token chunk."""
    import torch

    from bit_trellis_quantized_gb300 import native
    from escha_synth.gen_torch import moe_layer_device, projections_device

    stream = torch.cuda.Stream(device=dev)
    res = {}

    # single projection 1024x2048, K=2, batch 1: 1024 distinct projections (512 MB)
    P = 1024
    pj = projections_device(7001, dev, P)
    y = torch.empty((P, 1024), dtype=torch.float32, device=dev)
    t = _time_graph(torch, stream, lambda i: native.trellis_gemv(pj["codes"][i % P], pj["x"][i % P:i % P + 1],
                                                                 pj["rin"][i % P], pj["rout"][i % P],
                                                                 y=y[i % P:i % P + 1]), reps=P)
    ms = t[0]
    b = 2048 * 1024 * 2 // 8
    res["single_projection_1024x2048_k2_b1"] = {"us": ms * 1e3, **_stats(t), "packed_gbs": b / (ms * 1e-3) / 1e9,
                                               "frac_of_hbm": b / (ms * 1e-3) / 1e9 / hbm,
                                               "l2": f"{P} distinct projections ({P * b >> 20} MB) cycled"}
    # the same projection every call: its 512 KB of codes stay in L2
    t = _time_graph(torch, stream, lambda i: native.trellis_gemv(pj["codes"][0], pj["x"][0:1], pj["rin"][0],
                                                                 pj["rout"][0], y=y[0:1]), reps=256)
    res["single_projection_1024x2048_k2_b1_l2_resident"] = {
        "us": t[0] * 1e3, **_stats(t), "packed_gbs": b / (t[0] * 1e-3) / 1e9,
        "l2": "L2-resident: one projection, 256 calls per graph"}
    del pj, y

    # dense trellis linear 5120 -> 17408, K = 2 (a 27B-class gate_proj) with an
    # output bias: 8 distinct weights (178 MB packed) cycled; kt-major and
    # nt-major grids at M = 1, nt-major at M = 8, 64 and 2048
    n_in, n_out, nw = 5120, 17408, 8
    g = torch.Generator(device=dev).manual_seed(7101)
    codes = torch.randint(-32768, 32768, (nw, n_in // 16, n_out // 16, 32), dtype=torch.int16, device=dev,
                          generator=g)
    rin = (torch.randint(0, 2, (n_in,), device=dev, generator=g) * 2 - 1).to(torch.float16)
    rout = ((torch.rand(n_out, device=dev, generator=g) + 0.5)
            * (torch.randint(0, 2, (n_out,), device=dev, generator=g) * 2 - 1)).to(torch.float16)
    bias = torch.randn(n_out, device=dev, generator=g) * 8
    dn = {}
    packed = n_in * n_out * 2 // 8
    for nt_major, Ms in ((False, (1,)), (True, (1, 8, 64, 2048))):
        lins = [native.DenseLinear(codes[i], rin, rout, bias=bias, nt_major=nt_major) for i in range(nw)]
        for M in Ms:
            x = torch.randn((M, n_in), device=dev).to(torch.float16)
            y = torch.empty((M, n_out), dtype=torch.float32, device=dev)
            ws = torch.empty(lins[0].workspace_bytes(M), dtype=torch.uint8, device=dev)
            t = _time_graph(torch, stream, lambda i: lins[i % nw](x, y=y, ws=ws), reps=nw)
            ms = t[0]
            dn[f"{'nt' if nt_major else 'kt'}_major_m{M}"] = {
                "us": ms * 1e3, **_stats(t), "tokens_per_s": M / (ms * 1e-3), "packed_gbs": packed / (ms * 1e-3) / 1e9,
                "weight_fmas_per_s": float(M) * n_in * n_out / (ms * 1e-3)}
        del lins
    res["dense_linear_5120x17408_k2_bias"] = dn
    del codes
    torch.cuda.empty_cache()

    # MoE block at batch 1 through one escha_moe_block call per step (the
    # three per-slot kernels; the headline runs 8 steps per sequence launch)
    nl = len(blocks)
    mb = {}
    xs1 = torch.randn((nl, 1, HIDDEN), device=dev).to(torch.float16)
    out1 = torch.empty((1, HIDDEN), dtype=torch.float32, device=dev)
    t = _time_graph(torch, stream, lambda i: blocks[i % nl](xs1[i % nl], out=out1), reps=nl)
    mb["b1_per_slot_calls"] = {"tokens_per_s": 1 / (t[0] * 1e-3), "us_per_block": t[0] * 1e3, **_stats(t)}
    # one layer and one x every call: the 8 routed experts, the router and the
    # shared expert (12.6 MB) stay in L2
    t = _time_graph(torch, stream, lambda i: blocks[0](xs1[0], out=out1), reps=64)
    mb["b1_per_slot_calls_l2_resident"] = {"tokens_per_s": 1 / (t[0] * 1e-3), "us_per_block": t[0] * 1e3,
                                           **_stats(t), "l2": "L2-resident: one layer, one x, 64 calls per graph"}
    sws = torch.empty(native.seq_workspace_bytes([blocks[0]] * STEPS_PER_GRAPH), dtype=torch.uint8, device=dev)
    outs8 = torch.empty((STEPS_PER_GRAPH, HIDDEN), dtype=torch.float32, device=dev)
    t = _time_graph(torch, stream, lambda i: native.moe_blocks([blocks[0]] * STEPS_PER_GRAPH,
                                                               [xs1[0][0]] * STEPS_PER_GRAPH,
                                                               [outs8[j] for j in range(STEPS_PER_GRAPH)], ws=sws),
                    reps=16)
    mb["b1_blocks_l2_resident"] = {"tokens_per_s": STEPS_PER_GRAPH / (t[0] * 1e-3),
                                   "us_per_block": t[0] * 1e3 / STEPS_PER_GRAPH,
                                   **{k: v / STEPS_PER_GRAPH for k, v in _stats(t).items()},
                                   "l2": f"L2-resident: {STEPS_PER_GRAPH} blocks of one layer on one x per "
                                         "escha_moe_blocks call, 16 calls per graph"}
    del sws, outs8
    # MoE block at batch 8 / 16 (per-slot path), 64 / 256 / 2048 (grouped path)
    # over the headline's layers, fresh x per call
    for T in (8, 16, 64, 256, 2048):
        ws = torch.empty(max(native.lib().escha_moe_block_workspace(native.ctypes.byref(blocks[0].layer), T), 256),
                         dtype=torch.uint8, device=dev)
        reps = nl if T <= 256 else 8
        xs = torch.randn((reps, T, HIDDEN), device=dev).to(torch.float16)
        out = torch.empty((T, HIDDEN), dtype=torch.float32, device=dev)
        t = _time_graph(torch, stream, lambda i: blocks[i % nl](xs[i], out=out, ws=ws), reps=reps)
        ms = t[0]
        mb[f"b{T}" if T < 2048 else "prefill_2048"] = {"tokens_per_s": T / (ms * 1e-3), "us_per_block": ms * 1e3,
                                                       **_stats(t)}
        del ws, xs
    res["moe_block"] = mb

    # int8 w8a16: M = 1 (HBM) and M = 2048 (tensor cores), bf16 x
    i8 = {}
    for N, Kin in ((4096, 2048), (2048, 4096), (152064, 2048)):
        copies = max(1, (256 << 20) // (N * Kin))  # >= 256 MB of distinct weights at M = 1
        W = torch.randint(-127, 128, (copies, N, Kin), dtype=torch.int8, device=dev)
        s = torch.rand((copies, N), device=dev) * 9e-3 + 1e-3
        x1 = torch.randn((copies, 1, Kin), device=dev).to(torch.bfloat16)
        y1 = torch.empty((copies, 1, N), dtype=torch.float32, device=dev)
        t1 = _time_graph(torch, stream, lambda i: native.int8_w8a16_matvec(W[i % copies], s[i % copies],
                                                                           x1[i % copies], y=y1[i % copies]),
                         reps=max(copies, 8))
        ms1 = t1[0]
        M = 2048
        xm = torch.randn((M, Kin), device=dev).to(torch.bfloat16)
        ym = torch.empty((M, N), dtype=torch.float32, device=dev)
        t2 = _time_graph(torch, stream, lambda i: native.int8_w8a16_matvec(W[i % copies], s[i % copies], xm, y=ym),
                         reps=4)
        ms2 = t2[0]
        gbs = N * Kin / (ms1 * 1e-3) / 1e9
        tf = 2.0 * M * N * Kin / (ms2 * 1e-3) / 1e12
        i8[f"{N}x{Kin}"] = {"m1_us": ms1 * 1e3, "m1_us_min_max": [t1[1] * 1e3, t1[2] * 1e3], "m1_gbs": gbs,
                            "m1_frac_of_hbm": gbs / hbm, "m2048_us": ms2 * 1e3,
                            "m2048_us_min_max": [t2[1] * 1e3, t2[2] * 1e3], "m2048_tflops": tf,
                            "m2048_frac_of_bf16": tf / tflops}
        del W, s, x1, y1, xm, ym
    res["int8_w8a16"] = i8
    torch.cuda.empty_cache()

    # 40-block stack (K per projection from seed 5000 + block), ~10.6 GB
    sblocks = []
    for l in range(40):
        kg, kd = gen.stack_k(l)
        sblocks.append(native.MoeBlock(moe_layer_device(5000 + l, dev, k_gu=kg, k_dn=kd), device=dev))
    stack = native.MoeStack(sblocks)
    st = {}
    for T in ("1_sequence", 1, 8, 128, 2048):
        seq = T == "1_sequence"
        T = 1 if seq else T
        x0 = torch.randn((T, HIDDEN), device=dev)
        h = x0.clone()
        xb = torch.empty((T, HIDDEN), dtype=torch.float16, device=dev)
        ob = torch.empty((T, HIDDEN), dtype=torch.float32, device=dev)
        stack.workspace(T)
        t = _time_graph(torch, stream, lambda i: stack(h, xb, ob, sequence=seq), reps=2 if T == 2048 else 4)
        if seq:
            st["b1_one_launch"] = {"tokens_per_s": 1 / (t[0] * 1e-3), "ms_per_pass": t[0],
                                   "ms_per_pass_min_max": [t[1], t[2]],
                                   "note": "the 40 blocks as one escha_moe_stack launch (same bits as block by "
                                           "block, b1)"}
            continue
        ms = t[0]
        st[f"b{T}" if T < 2048 else "prefill_2048"] = {"tokens_per_s": T / (ms * 1e-3), "ms_per_pass": ms,
                                                       "ms_per_pass_min_max": [t[1], t[2]]}
    res["stack_40_blocks"] = st
    del stack, sblocks
    torch.cuda.empty_cache()
    return res


PROFILE_CASES = ("block_b1", "block_b8", "block_b64", "block_b256", "prefill_2048", "projection_b1",
                 "int8_m1", "int8_m2048", "int8_head_m2048", "dense_m1", "dense_m2048", "dense_split_m13")


def profile_case(name: str, reps: int):
    """One workload launched directly (no CUDA graph) `reps` times, for a
    profiler's launch list or a capture of one kernel; prints nothing timed."""
    import torch

    from bit_trellis_quantized_gb300 import native
    from escha_synth.gen_torch import moe_layer_device, projections_device

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if name.startswith("block_") or name == "prefill_2048":
        T = 2048 if name == "prefill_2048" else int(name.split("_b")[1])
        blk = native.MoeBlock(moe_layer_device(LAYER_SEED, dev), device=dev, topk=TOPK)
        xs = torch.randn((reps, T, HIDDEN), device=dev).to(torch.float16)
        out = torch.empty((T, HIDDEN), dtype=torch.float32, device=dev)
        for i in range(reps):
            blk(xs[i], out=out)
    elif name == "projection_b1":
        pj = projections_device(7001, dev, 64)
        y = torch.empty((64, 1024), dtype=torch.float32, device=dev)
        for i in range(reps):
            native.trellis_gemv(pj["codes"][i % 64], pj["x"][i % 64:i % 64 + 1], pj["rin"][i % 64],
                                pj["rout"][i % 64], y=y[i % 64:i % 64 + 1])
    elif name.startswith("dense_"):
        # 5120 -> 17408 K=2 at 1 or 2048 tokens; 17408 -> 5120 K=3 at 13 tokens (inputs split over CTAs)
        M = {"dense_m1": 1, "dense_m2048": 2048, "dense_split_m13": 13}[name]
        n_in, n_out, K = (17408, 5120, 3) if name == "dense_split_m13" else (5120, 17408, 2)
        codes = torch.randint(-32768, 32768, (n_in // 16, n_out // 16, 16 * K), dtype=torch.int16, device=dev)
        rin = (torch.randint(0, 2, (n_in,), device=dev) * 2 - 1).to(torch.float16)
        rout = (torch.rand(n_out, device=dev) + 0.5).to(torch.float16)
        lin = native.DenseLinear(codes, rin, rout, bias=torch.randn(n_out, device=dev), nt_major=True)
        x = torch.randn((M, n_in), device=dev).to(torch.float16)
        y = torch.empty((M, n_out), dtype=torch.float32, device=dev)
        for i in range(reps):
            lin(x, y=y)
    else:
        # int8 w8a16: 4096 x 2048 at 1 or 2048 tokens; the 152064 x 2048 head at 2048 tokens
        M = 1 if name == "int8_m1" else 2048
        N = 152064 if name == "int8_head_m2048" else 4096
        W = torch.randint(-127, 128, (N, 2048), dtype=torch.int8, device=dev)
        s = torch.rand(N, device=dev) * 9e-3 + 1e-3
        x = torch.randn((M, 2048), device=dev).to(torch.bfloat16)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        for i in range(reps):
            native.int8_w8a16_matvec(W, s, x, y=y)
    torch.cuda.synchronize()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extended", action="store_true", help="skip the other configurations (batched, prefill, "
                                                               "single projection, int8 shapes, 40-block stack)")
    ap.add_argument("--no-graph", action="store_true", help="launch the steps directly (for profilers)")
    ap.add_argument("--layers", type=int, default=N_LAYERS, help="distinct layers cycled through")
    ap.add_argument("--path", default="blocks", choices=["blocks", "sequence", "per-slot"],
                    help="the steps of a graph as one escha_moe_blocks call (by shape: the per-slot kernels over "
                         "all its blocks), the same call held on the sequence kernel, or one block call per step")
    ap.add_argument("--profile-case", help="comma-separated workloads (" + ", ".join(PROFILE_CASES) +
                                           ") run with direct launches (for profilers), then exit")
    ap.add_argument("--reps", type=int, default=3, help="launches of --profile-case")
    args = ap.parse_args()
    if args.profile_case:
        cases = args.profile_case.split(",")
        bad = [c for c in cases if c not in PROFILE_CASES]
        if bad:
            ap.error(f"unknown --profile-case {bad}; choose from {PROFILE_CASES}")
        for c in cases:
            profile_case(c, args.reps)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.steps < 1:
        args.steps = 1
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank)
        return
    # warm-up in whole graphs of STEPS_PER_GRAPH steps (at least the W asked
    # for); exactly args.steps timed steps
    args.warmup = -(-args.warmup // STEPS_PER_GRAPH) * STEPS_PER_GRAPH
    run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
