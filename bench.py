"""Benchmark: MLA decode over a paged latent KV cache on GB300.

One step = one full decode call through the C ABI (split-KV planner, paired
tcgen05 attention kernel, LSE merge of the split rows) over one batch of
synthetic inputs that are already resident in HBM.  Default workload: batch 64, Sq 1, seq_lens
drawn uniformly in [1, 32768] (seed 1003), bf16 cache with shuffled pages.

Printed (one JSON line): KV-tokens/s of the whole job, ms/step, the
roofline record of the attention kernel (timed alone with CUDA events on its
stream), an end-to-end number through the public API with host buffers, the
float64 oracle timed on the host cores on a bounded sample, and the SM
clocks sampled during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..9]
  (workloads 1..5: the dense configurations; 6: sparse top-2048 decode;
  7: the FP4 cache at the FP8 workload's shape; 8 and 9: the V4.1 FP8 and
  FP4 rows at that shape)
  python bench.py --impl reference ...   # the oracle arm (host cores)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import threading
import time

_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mla_latent_kv_05_gb300 import inputs as gen  # noqa: E402

METRIC = "MLA decode KV-tokens/s, HBM GB/s & TFLOP/s vs 1xGB300 roofline; us/call"
L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


# The sources the recorded DRAM counters depend on: the attention kernel and
# the headers it includes, and the planner (its partition sets the split
# partials the kernel writes).  The merge, W^UV and API files are not among
# them.
KERNEL_SOURCES = ("decode.cu", "decode.cuh", "common.cuh", "ptx.cuh", "plan.cu")


def kernel_source_hash():
    """Hash of the attention kernel's and planner's code: line comments and
    blank lines are dropped, so a comment-only edit keeps recorded counters
    valid."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_latent_kv_05_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in KERNEL_SOURCES:
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                lines = []
                for line in f:
                    code = line.split("//", 1)[0].rstrip() if not line.lstrip().startswith("#include") else line.rstrip()
                    if code.strip():
                        lines.append(code)
            h.update(name.encode() + "\n".join(lines).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: int, kind: str):
    """DRAM bytes per launch of the attention kernel from a committed ncu
    summary, only if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "decode_dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(f"{kind}:{workload}")
    if not rec or rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        smax = max(r["smax"] for r in rows)
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                          ("pcap", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in loaded):
                reasons.append(name)
        return {"sm_mhz": float(np.median([r["sm"] for r in loaded])), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded)}


def self_launch(gpus: int, argv) -> int:
    """`--gpus N` (N > 1) with no launcher around this process: start N ranks,
    one process per GPU, through torch.distributed.run on the loopback address
    and return its exit status. Each rank then sees RANK, LOCAL_RANK and
    WORLD_SIZE = N and runs the ordinary multi-rank path."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(gpus),
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def dist_setup(gpus: int | None = None):
    """Rank, world size and local rank from the launcher's environment.
    `--gpus N` must match the launcher's world size (a run with no launcher and
    N > 1 has already been re-started under one by `self_launch`), so a
    mismatch is an error rather than a silent one-GPU run."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if gpus is not None and gpus != world:
        raise SystemExit(f"bench.py: --gpus {gpus} but WORLD_SIZE={world}; launch N ranks with "
                         f"python -m torch.distributed.run --nproc-per-node {gpus} bench.py --gpus {gpus} ...")
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------- oracle arm
def oracle_sample(inp, budget_s: float, max_tokens_per_piece: int = 4096):
    """Time the float64 oracle (as it stands) on a bounded sample of the
    workload: whole (row, query) attentions over the first rows, each cut to
    at most `max_tokens_per_piece` tokens, until `budget_s` elapses.
    Returns (KV tokens processed, seconds, description)."""
    from oracle import mla_oracle
    raw = inp.kv_cache
    qa = inp.q_absorbed
    qr = inp.q_rope
    tokens = 0
    t0 = time.perf_counter()
    pieces = 0
    b = 0
    while time.perf_counter() - t0 < budget_s:
        bb = b % inp.batch
        n = min(int(inp.seq_lens[bb]), max_tokens_per_piece)
        if n > 0:
            pages = inp.block_table[bb, : (n + 63) // 64].long()
            sub = raw[pages]
            rows = mla_oracle.cache_rows(sub.double().numpy() if inp.kv_dtype == "bf16" else sub.numpy(),
                                         inp.kv_dtype)
            local_bt = np.arange(len(pages))
            g = mla_oracle.gather_rows(rows, local_bt, n)
            for i in range(inp.sq):
                mla_oracle.attend_latent(qa[bb, i].double().numpy(), qr[bb, i].double().numpy(), g, inp.scale)
            tokens += n
            pieces += 1
        b += 1
    dt = time.perf_counter() - t0
    return tokens, dt, f"{pieces} (row, all queries) attentions of <= {max_tokens_per_piece} tokens, 128 heads"


def oracle_sample_sparse(sp, budget_s: float):
    """The oracle on a bounded sample of a sparse workload: whole query rows
    (all listed tokens) in order until `budget_s` elapses."""
    from oracle import mla_oracle
    d = sp.dense
    flat = d.kv_cache.view(-1, d.kv_cache.shape[-1])
    tokens, pieces = 0, 0
    t0 = time.perf_counter()
    r = 0
    while time.perf_counter() - t0 < budget_s:
        b, i = divmod(r % (d.batch * d.sq), d.sq)
        s = sp.token_slots[b, i]
        s = s[s >= 0].long()
        rows = flat[s].double().numpy().reshape(1, -1, flat.shape[-1])
        g = mla_oracle.sparse_gather_rows(rows, np.arange(s.numel()))
        mla_oracle.attend_latent(d.q_absorbed[b, i].double().numpy(), d.q_rope[b, i].double().numpy(), g, d.scale)
        tokens += int(s.numel())
        pieces += 1
        r += 1
    dt = time.perf_counter() - t0
    return tokens, dt, f"{pieces} query rows with all their listed tokens (<= {sp.topk}), 128 heads"


def load_problem(workload: int):
    """(dense inputs, sparse inputs or None) of a workload."""
    if workload in gen.SPARSE_WORKLOADS:
        sp = gen.make_sparse_workload(workload)
        return sp.dense, sp
    return gen.make_workload(workload), None


def run_reference(args):
    world, rank, local = dist_setup(args.gpus)
    if rank != 0:
        return 0
    inp, sp = load_problem(args.workload)
    cfg = workload_config(args.workload, inp, sp)
    per_step = 0.01
    sample = (lambda b: oracle_sample_sparse(sp, b)) if sp is not None else (lambda b: oracle_sample(inp, b))
    for _ in range(args.warmup):
        sample(per_step)
    tot_tok, tot_s = 0, 0.0
    desc = ""
    for _ in range(args.steps):
        t, s, desc = sample(per_step)
        tot_tok += t
        tot_s += s
    value = tot_tok / tot_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "KV-tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": "KV-tokens/s", "cores": _CORES, "kind": "oracle",
                         "sample": f"per step: {desc}; ~{per_step}s of host work"},
        "e2e": {"value": value, "unit": "KV-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if args.workload == 1:
        line["cpu_baseline"]["unabsorbed"] = unabsorbed_sample(inp)
    print(json.dumps(line))
    return 0


def unabsorbed_sample(inp) -> dict:
    """The oracle's un-absorbed form (explicit per-head W^UK and W^UV, seeded
    N(0,1)/sqrt(512) weights, d_h = 128) on the oracle-sized workload's one
    query row, beside the absorbed form on the same row: what absorption
    saves on the host."""
    from oracle import mla_oracle
    rng = np.random.default_rng(7)
    H, d_h = int(inp.q_absorbed.shape[2]), 128
    n = int(inp.seq_lens[0])
    w_uk = rng.standard_normal((H, d_h, 512)) / np.sqrt(512)
    w_uv = rng.standard_normal((H, d_h, 512)) / np.sqrt(512)
    q_nope = rng.standard_normal((H, d_h))
    rows = mla_oracle.cache_rows(inp.kv_cache.double().numpy(), "bf16")
    g = mla_oracle.gather_rows(rows, inp.block_table[0].numpy(), n)
    qr = inp.q_rope[0, 0].double().numpy()
    t0 = time.perf_counter()
    mla_oracle.attend_unabsorbed(q_nope, qr, g[:, :512], g[:, 512:], w_uk, w_uv, inp.scale)
    t_un = time.perf_counter() - t0
    t0 = time.perf_counter()
    mla_oracle.attend_latent(mla_oracle.absorb_query(q_nope, w_uk), qr, g, inp.scale)
    t_abs = time.perf_counter() - t0
    return {"value": n / t_un, "unit": "KV-tokens/s", "absorbed_value": n / t_abs,
            "sample": f"one query row, {H} heads, {n} tokens; absorbed form on the same row for comparison"}


# ----------------------------------------------------------------- GPU arm
def workload_config(workload: int, inp, sp=None) -> dict:
    if sp is not None:
        c = gen.sparse_counts(sp)
        cache_bytes = inp.kv_cache.numel() * inp.kv_cache.element_size()
        return {"workload": gen.SPARSE_WORKLOADS[workload]["name"], "batch": inp.batch, "sq": inp.sq,
                "heads": int(inp.q_absorbed.shape[2]), "kv_dtype": inp.kv_dtype, "page_size": 64,
                "topk": sp.topk, "kv_tokens": c["kv_tokens"], "seed": gen.seed_for(workload),
                "l2": ("inputs larger than L2 (listed rows %.0f MB > 129 MB; KV cache %.0f MB)"
                       % (c["kv_bytes"] / 1e6, cache_bytes / 1e6)) if c["kv_bytes"] > L2_BYTES
                else "L2 flushed between steps"}
    c = gen.workload_counts(inp)
    return {"workload": gen.WORKLOADS[workload]["name"], "batch": inp.batch, "sq": inp.sq,
            "heads": int(inp.q_absorbed.shape[2]), "kv_dtype": inp.kv_dtype, "page_size": 64,
            "kv_tokens": c["kv_tokens"], "seed": gen.seed_for(workload),
            "l2": "inputs larger than L2 (KV cache %.0f MB > 129 MB)" % (c["kv_bytes"] / 1e6)
            if c["kv_bytes"] > L2_BYTES else "L2 flushed between steps"}


def run_ours(args):
    from mla_latent_kv_05_gb300 import binding
    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp, sp = load_problem(args.workload)
    q = inp.q_absorbed.to(dev)
    qr = inp.q_rope.to(dev)
    kv = inp.kv_cache.to(dev)
    out = torch.empty((inp.batch, inp.sq, 128, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((inp.batch, inp.sq, 128), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    if sp is not None:
        # sparse top-k decode: four launches per call (compaction, planner,
        # attention, merge); the per-step inputs are q, q_rope and the lists
        counts = gen.sparse_counts(sp)
        slots = sp.token_slots.to(dev)
        ws = binding.alloc_workspace_sparse(inp.batch, inp.sq, sp.topk, dev)
        launches = 4
        uploads = [(sp.token_slots.pin_memory(), slots)]

        def call(qb, qrb, extra, outb, lseb):
            binding.mla_decode_sparse_bf16(qb, qrb, kv, extra[0], inp.scale, out=outb, lse=lseb, workspace=ws)

        def step():
            call(q, qr, [slots], out, lse)
    else:
        counts = gen.workload_counts(inp)
        decode = {"bf16": binding.mla_decode_bf16, "fp8": binding.mla_decode_fp8,
                  "fp4": binding.mla_decode_fp4, "fp8v41": binding.mla_decode_fp8_v41,
                  "fp4v41": binding.mla_decode_fp4_v41}[inp.kv_dtype]
        bt = inp.block_table.to(dev)
        sl = inp.seq_lens.to(dev)
        ws = binding.alloc_workspace(inp.batch, inp.sq, dev)
        # planner, attention, merge (FP8, FP4: the exact pass after the f16
        # pass is a fourth launch, which returns at once unless needed)
        launches = 3 if inp.kv_dtype == "bf16" else 4
        uploads = [(inp.block_table.pin_memory(), bt), (inp.seq_lens.pin_memory(), sl)]

        def call(qb, qrb, extra, outb, lseb):
            decode(qb, qrb, kv, extra[0], extra[1], inp.scale, out=outb, lse=lseb, workspace=ws)

        def step():
            call(q, qr, [bt, sl], out, lse)
    flush = None
    if counts["kv_bytes"] <= L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    for _ in range(args.warmup):
        step()
    st = binding.mla_get_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {binding.status_string(st)}")

    # ---- timed region: K whole steps, barrier + sync on both sides
    kern_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    for a, b in kern_ev:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        t_start = time.perf_counter()
        for k in range(args.steps):
            if flush is not None:
                flush.zero_()
            step_ev[k][0].record(stream)
            step()
            step_ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        wall = time.perf_counter() - t_start
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    # The attention kernel alone, from a second pass of the same number of
    # steps with the library's profiling hook: its CUDA events bracket the
    # attention kernel on the call's stream.  (The hook makes that call
    # launch its three kernels without programmatic overlap, so it is kept
    # out of the timed steps above.)
    for k in range(args.steps):
        if flush is not None:
            flush.zero_()
        binding.mla_profile_next_decode(*kern_ev[k])
        step()
    torch.cuda.synchronize(dev)
    kern_ms = [a.elapsed_time(b) for a, b in kern_ev]
    st = binding.mla_get_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {binding.status_string(st)}")
    graph_us = None
    if args.workload == 1:
        # The oracle-sized call is launch-latency bound: also time it replayed
        # from a CUDA graph that captured one call (its three launches).
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record(stream)
        for _ in range(args.steps):
            g.replay()
        gb.record(stream)
        torch.cuda.synchronize(dev)
        graph_us = ga.elapsed_time(gb) * 1000.0 / args.steps
        if binding.mla_get_status(ws) != 0:
            raise RuntimeError("device status after the graph replays")
    total_ms = float(np.sum(step_ms))
    total_ms_max = max_over_ranks(total_ms, world, dev)
    tokens_all = sum_over_ranks(float(counts["kv_tokens"] * args.steps), world, dev)
    value = tokens_all / (total_ms_max / 1000.0)
    ms_per_step = total_ms_max / args.steps

    # ---- roofline of the attention kernel
    peaks = load_peaks()
    kern_s = float(np.mean(kern_ms)) / 1000.0
    bytes_alg = counts["bytes"]
    flops = counts["flops"]
    gbs = bytes_alg / kern_s / 1e9
    tfs = flops / kern_s / 1e12
    t_bytes = bytes_alg / (peaks["hbm"] * 1e9)
    t_flop = flops / (peaks["bf16"] * 1e12)
    if t_bytes >= t_flop:
        roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"]}
    else:
        roof = {"bound": "tensor", "achieved": tfs, "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": tfs / peaks["bf16"]}
    roof["traffic"] = recorded_traffic(args.workload, inp.kv_dtype)
    roof["peak_source"] = f"{peaks['source']} (MEASURED_PEAKS.json)" if peaks["source"] == "measured" else "fallback"
    roof["kernel_us"] = kern_s * 1e6
    roof["roofline_us"] = max(t_bytes, t_flop) * 1e6
    roof["roofline_frac_of_call"] = max(t_bytes, t_flop) / (ms_per_step / 1000.0)
    roof["hbm_gbs"] = gbs
    roof["tflops"] = tfs
    # the tensor pipe's share against the power-capped (sustained) GEMM rate
    roof["tensor_frac_of_sustained"] = tfs / peaks["bf16_sus"]

    # ---- end to end through the public API with pinned host buffers.
    # Every step uploads its inputs and reads its outputs back, pipelined the
    # way a serving loop would: two sets of device buffers, uploads on one
    # copy stream (overlapping the previous step's call), read-backs on
    # another (overlapping the next step's call), ordered by events.
    hq = inp.q_absorbed.pin_memory()
    hqr = inp.q_rope.pin_memory()
    e2e_steps = max(4, min(args.steps, 50))

    def make_set():
        return dict(q=torch.empty_like(q), qr=torch.empty_like(qr), extra=[torch.empty_like(d) for _, d in uploads],
                    out=torch.empty_like(out), lse=torch.empty_like(lse),
                    hout=torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                    hlse=torch.empty(lse.shape, dtype=lse.dtype).pin_memory())

    sets = [make_set(), make_set()]
    up_stream = torch.cuda.Stream(dev)
    down_stream = torch.cuda.Stream(dev)

    def run_e2e(n):
        ev_up = [torch.cuda.Event() for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_down = [torch.cuda.Event() for _ in range(n)]
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up_stream.wait_event(e0)
        down_stream.wait_event(e0)
        for k in range(n):
            st_ = sets[k % 2]
            with torch.cuda.stream(up_stream):
                if k >= 2:
                    up_stream.wait_event(ev_comp[k - 2])      # this set's inputs were last read by step k-2
                st_["q"].copy_(hq, non_blocking=True)
                st_["qr"].copy_(hqr, non_blocking=True)
                for (h, _), d in zip(uploads, st_["extra"]):
                    d.copy_(h, non_blocking=True)
                ev_up[k].record(up_stream)
            stream.wait_event(ev_up[k])
            if k >= 2:
                stream.wait_event(ev_down[k - 2])             # this set's outputs were last read back by step k-2
            call(st_["q"], st_["qr"], st_["extra"], st_["out"], st_["lse"])
            ev_comp[k].record(stream)
            with torch.cuda.stream(down_stream):
                down_stream.wait_event(ev_comp[k])
                st_["hout"].copy_(st_["out"], non_blocking=True)
                st_["hlse"].copy_(st_["lse"], non_blocking=True)
                ev_down[k].record(down_stream)
        stream.wait_event(ev_down[n - 1])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    run_e2e(2)
    barrier(world)
    e2e_ms = max_over_ranks(run_e2e(e2e_steps), world, dev)
    e2e_value = sum_over_ranks(float(counts["kv_tokens"] * e2e_steps), world, dev) / (e2e_ms / 1000.0)
    h2d = sum(t.numel() * t.element_size() for t in [hq, hqr] + [h for h, _ in uploads])
    d2h = sets[0]["hout"].numel() * sets[0]["hout"].element_size() + sets[0]["hlse"].numel() * sets[0]["hlse"].element_size()

    line = {
        "metric": METRIC, "value": value, "unit": "KV-tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_call": ms_per_step * 1000.0,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": inp.kv_dtype,
        "data": "synthetic", "config": workload_config(args.workload, inp, sp),
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "KV-tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": ("q, q_rope, the slot lists" if sp is not None else "q, q_rope, block_table, seq_lens")
                        + " uploaded and out, lse read back every step (copy streams, two buffer sets, "
                          "overlapping the neighbouring steps' calls); the KV cache stays resident in HBM"},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
        **({"graph_us_per_call": graph_us} if graph_us is not None else {}),
        "wall_s_timed_region": wall,
    }
    if rank == 0 and not args.no_cpu_baseline:
        tok, sec, desc = (oracle_sample_sparse(sp, args.cpu_seconds) if sp is not None
                          else oracle_sample(inp, args.cpu_seconds))
        line["cpu_baseline"] = {"value": tok / sec, "unit": "KV-tokens/s", "cores": _CORES, "kind": "oracle",
                                "sample": f"{desc}; {sec:.1f}s of host work"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_wuv(args):
    """Time the W^UV up-projection alone (mla_up_project_wuv) on `--wuv-rows`
    row counts: CUDA events on its stream, median of --steps calls after
    --warmup calls, an L2 flush (a 258 MB write) before each call.  One JSON
    line per row count, against the measured HBM roofline: algorithmic bytes
    = latent (rows x 128 x 512 bf16) + W^UV (128 x 128 x 512 bf16) + out
    (rows x 128 x 128 bf16); FLOPs = 2 x rows x 128 x 128 x 512."""
    from mla_latent_kv_05_gb300 import binding
    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    g = torch.Generator().manual_seed(7)
    w_uv = (torch.randn((128, 128, 512), generator=g) * 512 ** -0.5).to(torch.bfloat16).to(dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for rows in [int(x) for x in args.wuv_rows.split(",")]:
        lat = torch.randn((rows, 128, 512), generator=g).to(torch.bfloat16).to(dev)
        out = torch.empty((rows, 128, 128), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(256, dtype=torch.uint8, device=dev)
        for _ in range(args.warmup):
            binding.mla_up_project_wuv(lat, w_uv, out=out, workspace=ws)
        times = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            binding.mla_up_project_wuv(lat, w_uv, out=out, workspace=ws)
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b) * 1e-3)
        if binding.mla_get_status(ws) != 0:
            raise RuntimeError("device status after the W^UV calls")
        t = float(np.median(times))
        nbytes = 2 * (rows * 128 * 512 + 128 * 128 * 512 + rows * 128 * 128)
        flops = 2.0 * rows * 128 * 128 * 512
        gbs = nbytes / t / 1e9
        if rank == 0:
            print(json.dumps({"metric": "W^UV up-projection us/call", "value": t * 1e6, "unit": "us",
                              "higher_is_better": False, "rows": rows, "steps": args.steps,
                              "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
                              "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                                           "frac": gbs / peaks["hbm"], "tflops": flops / t / 1e12}}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=3, choices=sorted(gen.WORKLOADS) + sorted(gen.SPARSE_WORKLOADS))
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--wuv-rows", default=None,
                    help="time the W^UV up-projection alone on these row counts (e.g. 64,128,1024,4096)")
    args = ap.parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return self_launch(args.gpus, sys.argv[1:] if argv is None else list(argv))
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.wuv_rows:
        return run_wuv(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
