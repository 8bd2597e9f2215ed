"""Benchmark of the fused online-softmax attention path on GB300.

One step = one attention forward (rf_attn_fwd) over the grouped-query,
long-context causal prefill: B=1, Hq=64, Hkv=8, Sq=Sk=32768, d=128, bf16 in /
fp32 accumulate, inputs seeded-synthetic and resident in HBM (the largest
single-GPU configuration of the metric). The JSON line reports
  value      algorithmic TFLOP/s (4*d flops per visible query-key pair),
  e2e        the same metric through the public API with host buffers
             (pinned host -> device copies of Q, K, V and device -> host
             copies of O and LSE inside the timed region),
  roofline   the attention kernel against the measured dense bf16 peak,
  mha_prefill, tiny_fp32, decode, softmax, ...   the other workloads, each
             timed for at least MIN_SIDE_S seconds of launches,
  cpu_baseline  the float64 oracle on the host cores on a bounded sample.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 run under torch.distributed.run; each rank runs the full workload on
its own GPU (weak scaling, no collective on the data path) and the slowest
rank's time is reported for the aggregate.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from online_softmax_attention_rf_gb300 import inputs  # noqa: E402

WORKLOAD = "gqa_long"
# the metric as the workload statement names it; both arms print it verbatim
METRIC = "attn fwd TFLOP/s & % BF16 tensor peak (prefill); decode GB/s & % HBM peak"
# every secondary workload is timed for at least this long (clock sampling
# and a stable mean), whatever --steps says
MIN_SIDE_S = 0.5
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic per launch from ncu captures (summarised under profiles/), valid only for the
# kernel source they were taken on; any change to the source makes it null.
TRAFFIC = {
    # attn_tc_kernel<128, 0> on gqa_long: dram read 677.6 MB + write 505.0 MB
    "attn_tc_gqa_long": {"digest": "912cb81acc2699e7", "bytes": 1182629120,
                         "sources": ("attn_tc.cu", "rf_device.cuh")},
    # attn_tc_kernel<128, 0> on mha_prefill: dram read 404.3 MB + write 112.8 MB
    "attn_tc_mha_prefill": {"digest": "912cb81acc2699e7", "bytes": 517131008,
                            "sources": ("attn_tc.cu", "rf_device.cuh")},
    # attn_tc_kernel<64, 1> on two_level: dram read 289.3 MB + write 49.3 MB
    "attn_tc_two_level": {"digest": "912cb81acc2699e7", "bytes": 338543360,
                          "sources": ("attn_tc.cu", "rf_device.cuh")},
    # attn_tc_kernel<64, 0> on block_sparse: dram read 201.5 MB + write 49.8 MB
    "attn_tc_block_sparse": {"digest": "912cb81acc2699e7", "bytes": 251304960,
                             "sources": ("attn_tc.cu", "rf_device.cuh")},
    # attn_tc_kernel<64, 1> (the selected block-wise kernel) on scattered_short:
    # dram read 100.9 MB + write 12.9 MB
    "attn_tc_scattered_short": {"digest": "912cb81acc2699e7", "bytes": 113853952,
                                "sources": ("attn_tc.cu", "rf_device.cuh")},
    # softmax_rows kernels: dram__bytes_read.sum + dram__bytes_write.sum
    # (rows_64k: 1073.8 + 1013.9 MB; rows_1m, clusters of 8, three CTAs per SM,
    # second pass back to front: 1113.2 + 1014.5 MB)
    # (captured on digest 70553e06eb3b0b5c; the source since differs only in a
    # comment of the file header)
    "softmax_rows_64k": {"digest": "2ef0308bfe63e4af", "bytes": 2087659776,
                         "sources": ("softmax_rows.cu", "rf_device.cuh")},
    "softmax_rows_1m": {"digest": "2ef0308bfe63e4af", "bytes": 2127690752,
                        "sources": ("softmax_rows.cu", "rf_device.cuh")},
    # moe_route_kernel<float, 8>, row_moments_smem_kernel<float> and
    # inertia_kernel: dram__bytes_read.sum + dram__bytes_write.sum
    "moe_route": {"digest": "0079b63ed45830e3", "bytes": 139984384,
                  "sources": ("cascades.cu", "rf_device.cuh")},
    "row_moments": {"digest": "0079b63ed45830e3", "bytes": 1016576000,
                    "sources": ("cascades.cu", "rf_device.cuh")},
    "inertia": {"digest": "0079b63ed45830e3", "bytes": 1076683776,
                "sources": ("cascades.cu", "rf_device.cuh")},
    # fp8_gemm_kernel (persistent) and rowquant_kernel<bf16> on the 8192^3
    # workload: dram__bytes_read.sum + dram__bytes_write.sum
    "fp8_gemm": {"digest": "1bd446f9ea742eee", "bytes": 443226624,
                 "sources": ("fp8_gemm.cu", "rf_device.cuh")},
    "rowquant": {"digest": "1bd446f9ea742eee", "bytes": 167583744,
                 "sources": ("fp8_gemm.cu", "rf_device.cuh")},
    # mla_decode_kernel (persistent, 128-key tiles) on the MLA workload: dram
    # read 310.0 MB + write 7.6 MB (the merge kernel reads the partials)
    "mla_decode": {"digest": "bec3777b93cd0491", "bytes": 317687040,
                   "sources": ("mla_decode.cu", "rf_device.cuh")},
    # decode_partials_kernel<128, 4> on decode_splitk: dram read 4295.2 MB + write 6.1 MB
    "decode_partials_decode_splitk": {"digest": "e3c0faa2696296ac", "bytes": 4301298944,
                                      "sources": ("decode.cu", "rf_device.cuh")},
}


def traffic_for(key):
    """Recorded DRAM bytes per launch, or None once the kernel source changed."""
    t = TRAFFIC.get(key)
    return t["bytes"] if t and source_digest(*t["sources"]) == t["digest"] else None


def source_digest(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "online_softmax_attention_rf_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def visible_pairs(w, tile_mask=None):
    """Unmasked (query, key) pairs per head (the algorithmic work)."""
    Sq, Sk = w["Sq"], w["Sk"]
    if tile_mask is not None:
        rows = np.arange(Sq)
        total = 0
        T = w.get("tile", 128)
        for qt in range(tile_mask.shape[0]):
            r = rows[qt * T:(qt + 1) * T]
            for kt in np.nonzero(tile_mask[qt])[0]:
                keys = min(Sk, (kt + 1) * T) - kt * T
                if w["causal"]:
                    lim = np.minimum(Sk, r + 1 + Sk - Sq) - kt * T
                    total += int(np.clip(lim, 0, keys).sum())
                else:
                    total += len(r) * keys
        return total
    if w["causal"]:
        i = np.arange(Sq, dtype=np.int64)
        return int(np.clip(i + 1 + Sk - Sq, 0, Sk).sum())
    return Sq * Sk


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def max_over_ranks(dist, x):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


_INPUT_CACHE = {}


def cpu_oracle_sample(name, budget_s=12.0, start=0):
    """Time the float64 oracle on query-row blocks of the workload until the
    budget is spent; returns (TFLOP/s, seconds, blocks, cores).

    A block is ROW_BLOCK consecutive query rows of one head. For causal
    attention with Sq = Sk, rows [r0, r1) of a head see exactly keys [0, r1),
    so the oracle runs on q[r0:r1] against k, v[:r1] (bottom-right alignment
    makes that the same problem). Blocks are taken round-robin over heads and
    spread over the rows, starting at block `start`; the flops counted are
    the block's visible pairs, 4*d each."""
    import oracle
    w = inputs.WORKLOADS[name]
    if name not in _INPUT_CACHE:
        _INPUT_CACHE[name] = inputs.workload_inputs(name)
    q, k, v, scale, extras = _INPUT_CACHE[name]
    assert not extras and (not w["causal"] or w["Sq"] == w["Sk"])
    G = w["H"] // w["Hkv"]
    rb = oracle.three_pass.ROW_BLOCK
    nrb = -(-w["Sq"] // rb)
    heads = [(b, h) for b in range(w["B"]) for h in range(w["H"])]
    cores = len(os.sched_getaffinity(0))
    spent, flops, blocks = 0.0, 0.0, 0
    n = start
    while spent < budget_s:
        b, h = heads[n % len(heads)]
        r0 = ((n // len(heads)) * 37 + n) % nrb * rb      # spread over the rows
        r1 = min(w["Sq"], r0 + rb)
        kend = r1 if w["causal"] else w["Sk"]
        qb = q[b:b + 1, h:h + 1, r0:r1].double().numpy()
        kb = k[b:b + 1, h // G:h // G + 1, :kend].double().numpy()
        vb = v[b:b + 1, h // G:h // G + 1, :kend].double().numpy()
        t0 = time.perf_counter()
        oracle.attention(qb, kb, vb, scale, w["causal"])
        spent += time.perf_counter() - t0
        rows = np.arange(r0, r1, dtype=np.int64)
        pairs = int((rows + 1).sum()) if w["causal"] else (r1 - r0) * w["Sk"]
        flops += 4.0 * w["d"] * pairs
        blocks += 1
        n += 1
    return flops / spent / 1e12, spent, blocks, cores


def workload_config(name, world):
    w = inputs.WORKLOADS[name]
    return {"workload": name, "B": w["B"], "H": w["H"], "Hkv": w["Hkv"], "Sq": w["Sq"],
            "Sk": w["Sk"], "d": w["d"], "causal": w["causal"],
            "parallelism": "dp%d (independent replicas)" % world}


def run_reference(args, dist, rank):
    """The oracle as the reference arm, on the host cores."""
    if rank != 0:
        return
    for _ in range(args.warmup):
        cpu_oracle_sample(WORKLOAD, budget_s=1.0)
    t0 = time.perf_counter()
    vals, samples = [], []
    per_step = min(8.0, 150.0 / args.steps)
    cores = len(os.sched_getaffinity(0))
    for s in range(args.steps):
        v, dt, blocks, cores = cpu_oracle_sample(WORKLOAD, budget_s=per_step, start=1000 * s)
        vals.append(v)
        samples.append(blocks)
    elapsed = time.perf_counter() - t0
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * elapsed / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(WORKLOAD, 1),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "per step, %.1f s of 256-query-row blocks of the workload's "
                                   "heads (blocks per step: %s), float64 three-pass NumPy "
                                   "oracle; TFLOP/s over the blocks' visible pairs"
                                   % (per_step, samples)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_steps(fn, steps, warmup, stream, dist):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    total_ms = t_start.elapsed_time(t_end)
    per_launch = [a.elapsed_time(b) for a, b in ev]
    return total_ms, per_launch


def bench_prefill(name, args, dev, stream, peaks, peak_src, steps, warmup, dist=None, clk=None):
    """Dense or causal prefill of a named workload: exactly `steps` timed
    launches after `warmup`; returns (summary, inputs kept for e2e)."""
    from online_softmax_attention_rf_gb300 import api
    w = inputs.WORKLOADS[name]
    q_h, k_h, v_h, scale, _ = inputs.workload_inputs(name)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    flops = 4.0 * w["d"] * visible_pairs(w) * w["B"] * w["H"]

    def step():
        api.attn_fwd(q, k, v, scale, w["causal"], None, o, lse)

    if clk is not None:
        with clk:
            total_ms, per_launch = time_steps(step, steps, warmup, stream, dist)
    else:
        total_ms, per_launch = time_steps(step, steps, warmup, stream, dist)
    assert api.device_status() == 0
    att_ms = statistics.mean(per_launch)
    achieved = flops / (att_ms * 1e-3) / 1e12
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    out_bytes = o.numel() * o.element_size() + lse.numel() * 4
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "traffic": traffic_for("attn_tc_" + name),
                "algorithmic_bytes": in_bytes + out_bytes,
                "peak_source": "%s dense bf16 (burst)" % peak_src,
                "frac_sustained": achieved / peaks.get("bf16_tflops_sustained",
                                                       peaks["bf16_tflops"])}
    out = {"workload": name, "value": flops / (total_ms / steps * 1e-3) / 1e12,
           "unit": "TFLOP/s", "ms_per_step": total_ms / steps, "total_ms": total_ms,
           "flops_per_step": flops, "steps": steps, "roofline": roofline}
    del q, k, v, o, lse
    torch.cuda.empty_cache()
    return out, (q_h, k_h, v_h, scale, w)


def bench_tiny(args, dev, stream, peaks, peak_src):
    """The exact float32 case (B=H=1, S=128, d=64): launch latency in us."""
    from online_softmax_attention_rf_gb300 import api
    w = inputs.WORKLOADS["tiny_fp32"]
    q_h, k_h, v_h, scale, _ = inputs.workload_inputs("tiny_fp32")
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)

    def step():
        api.attn_fwd(q, k, v, scale, w["causal"], None, o, lse)

    total, per, n = time_side(step, args, stream)
    assert api.device_status() == 0
    us = 1000.0 * statistics.median(per)
    flops = 4.0 * w["d"] * visible_pairs(w)
    # the kernel alone: the same call captured once in a CUDA graph and
    # replayed, so that no host work sits between the two events
    graph_us, graph_note = None, None
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
            side.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                step()
        stream.wait_stream(side)
        reps = []
        for _ in range(args.warmup):
            g.replay()
        for _ in range(max(200, side_steps(args))):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            reps.append(a.elapsed_time(b))
        assert api.device_status() == 0
        graph_us = 1000.0 * statistics.median(reps)
    except Exception as e:  # the host-timed number above stands on its own
        graph_note = "graph capture failed: %s" % e
    return {"workload": "tiny_fp32 [B=1, H=1, S=128, d=64, f32, non-causal]", "value": us,
            "unit": "us", "ms_per_step": us / 1000.0, "launches": n,
            "mean_us": 1000.0 * statistics.mean(per),
            "graph_replay_us": graph_us, "graph_note": graph_note,
            "gflops": flops / (us * 1e-6) / 1e9,
            "note": "latency-bound parity case: value = median CUDA-event time of one call "
                    "through the binding (host argument handling and launch included, inputs "
                    "resident, 0.13 MB); graph_replay_us = the same launch replayed from a "
                    "CUDA graph (the kernel and the graph launch only)"}


def run_ours(args, dist, rank, world, local):
    from online_softmax_attention_rf_gb300 import api
    api.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    side = {"decode": bench_decode, "softmax": bench_softmax,
            "softmax_long": lambda *a: bench_softmax(*a, name="rows_1m"),
            "block_sparse": bench_block_sparse, "two_level": bench_two_level,
            "scattered": bench_scattered, "mla": bench_mla, "cascades": bench_cascades,
            "tiny": bench_tiny}
    if args.only in side:
        # one workload alone (used for profiling captures)
        out = side[args.only](args, dev, stream, peaks, peak_src)
        if rank == 0:
            print(json.dumps(out), flush=True)
        return
    if args.only == "mha_prefill":
        out, _ = bench_prefill("mha_prefill", args, dev, stream, peaks, peak_src, args.steps,
                               args.warmup)
        if rank == 0:
            print(json.dumps(out), flush=True)
        return

    # the headline: exactly K timed steps of the GQA long-context prefill
    clk = ClockSampler(local)
    head, (q_h, k_h, v_h, scale, w) = bench_prefill(WORKLOAD, args, dev, stream, peaks, peak_src,
                                                    args.steps, args.warmup, dist, clk)
    total_ms = max_over_ranks(dist, head["total_ms"])
    ms_step = total_ms / args.steps
    flops = head["flops_per_step"]
    value = flops * world / (ms_step * 1e-3) / 1e12
    if args.only == "prefill":
        if rank == 0:
            print(json.dumps({"workload": WORKLOAD, "value": value, "unit": "TFLOP/s",
                              "ms_per_step": ms_step, "roofline": head["roofline"],
                              "clocks": clk.summary()}), flush=True)
        return

    # end to end through the public API with host buffers: rf_attn_fwd_host
    # copies Q, K, V in and O, LSE out every step, pipelined with its kernels
    qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    op = torch.empty(q_h.shape, dtype=q_h.dtype).pin_memory()
    lp = torch.empty(q_h.shape[:3], dtype=torch.float32).pin_memory()
    ws = torch.empty(api.attn_fwd_host_workspace_bytes(w["B"], w["H"], w["Hkv"], w["Sq"], w["Sk"],
                                                       w["d"], q_h.dtype),
                     dtype=torch.uint8, device=dev)

    def e2e_step():
        api.attn_fwd_host(qp, kp, vp, scale, w["causal"], None, op, lp, workspace=ws, device=dev)

    n_e2e = max(3, min(args.steps, 50))
    e2e_total, _ = time_steps(e2e_step, n_e2e, 3, stream, dist)
    e2e_total = max_over_ranks(dist, e2e_total)
    e2e_ms = e2e_total / n_e2e
    h2d = sum(t.numel() * t.element_size() for t in (qp, kp, vp))
    d2h = op.numel() * op.element_size() + lp.numel() * lp.element_size()
    del qp, kp, vp, op, lp, ws, q_h, k_h, v_h
    torch.cuda.empty_cache()

    n_mha = max(args.steps, 1)
    mha, _ = bench_prefill("mha_prefill", args, dev, stream, peaks, peak_src, n_mha, args.warmup)
    # at least MIN_SIDE_S of launches for the sub-key as well
    est = mha["ms_per_step"]
    if n_mha * est < 1000.0 * args.min_side_s:
        mha, _ = bench_prefill("mha_prefill", args, dev, stream, peaks, peak_src,
                               int(math.ceil(1000.0 * args.min_side_s / est)), args.warmup)
    mha.pop("total_ms")
    tiny = bench_tiny(args, dev, stream, peaks, peak_src)
    decode = bench_decode(args, dev, stream, peaks, peak_src)
    softmax = bench_softmax(args, dev, stream, peaks, peak_src)
    softmax_long = bench_softmax(args, dev, stream, peaks, peak_src, "rows_1m")
    block_sparse = bench_block_sparse(args, dev, stream, peaks, peak_src)
    two_level = bench_two_level(args, dev, stream, peaks, peak_src)
    scattered = bench_scattered(args, dev, stream, peaks, peak_src)
    mla = bench_mla(args, dev, stream, peaks, peak_src)
    cascades = bench_cascades(args, dev, stream, peaks, peak_src)
    launches = args.steps          # one rf_attn_fwd kernel launch per timed step

    if rank != 0:
        return
    cpu_v, cpu_dt, cpu_blocks, cores = cpu_oracle_sample(WORKLOAD)
    config = workload_config(WORKLOAD, world)
    config["l2"] = ("inputs larger than L2 (Q, O = 537 MB each per step; K, V = 67 MB each, "
                    "re-read from L2 by the 8 query heads of a group)")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": config,
        "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "roofline": head["roofline"],
        "clocks": clk.summary(),
        "mha_prefill": mha,
        "tiny_fp32": tiny,
        "decode": decode,
        "softmax": softmax,
        "softmax_long": softmax_long,
        "block_sparse": block_sparse,
        "two_level": two_level,
        "scattered_short": scattered,
        "mla_decode": mla,
        "moe_route": cascades["moe_route"],
        "row_moments": cascades["row_moments"],
        "moment_of_inertia": cascades["moment_of_inertia"],
        "fp8_quant": cascades["fp8_quant"],
        "fp8_gemm": cascades["fp8_gemm"],
        "cpu_baseline": {"value": cpu_v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "%d blocks of 256 query rows of the workload's heads "
                                   "(%.1f s, float64 three-pass NumPy oracle); TFLOP/s over "
                                   "the blocks' visible pairs" % (cpu_blocks, cpu_dt)},
    }
    print(json.dumps(line), flush=True)


def time_side(fn, args, stream):
    """Times a secondary workload: at least side_steps(args) launches and at
    least args.min_side_s seconds of them; returns (total ms, per-launch ms, n)."""
    for _ in range(args.warmup):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(3):
        fn()
    b.record(stream)
    b.synchronize()
    est = max(a.elapsed_time(b) / 3.0, 1e-3)
    n = max(side_steps(args), min(20000, int(math.ceil(1000.0 * args.min_side_s / est))))
    total, per = time_steps(fn, n, 1, stream, None)
    return total, per, n


def side_steps(args):
    """Timed steps for the secondary workloads (decode, row softmax)."""
    return max(5, min(args.steps, 50))


def bench_decode(args, dev, stream, peaks, peak_src):
    from online_softmax_attention_rf_gb300 import api
    w = inputs.WORKLOADS["decode_splitk"]
    q_h, k_h, v_h, scale, _ = inputs.workload_inputs("decode_splitk")
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    ws = torch.empty(api.decode_workspace_bytes(w["B"], w["H"], w["nsplit"], w["d"]) // 4,
                     dtype=torch.float32, device=dev)
    algo = (k.numel() + v.numel() + q.numel() + o.numel()) * 2 + lse.numel() * 4

    def step():
        api.attn_decode_splitk(q, k, v, w["nsplit"], scale, ws, o, lse)

    # K and V (4.3 GB) are far larger than L2: no flush needed
    total, per = time_side(step, args, stream)[:2]
    ms = statistics.mean(per)
    gbs = algo / (ms * 1e-3) / 1e9
    assert api.device_status() == 0
    out = {"workload": "decode_splitk", "value": gbs, "unit": "GB/s", "ms_per_step": ms,
           "algorithmic_bytes": algo,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / peaks["hbm_gbs"], "frac_of_8TBs": gbs / 8000.0,
                        "traffic": traffic_for("decode_partials_decode_splitk"),
                        "peak_source": "%s HBM copy" % peak_src,
                        "note": "step = partials kernel + merge kernel; traffic is the "
                                "partials kernel's"}}
    del q, k, v, o, lse, ws
    torch.cuda.empty_cache()
    return out


def bench_block_sparse(args, dev, stream, peaks, peak_src):
    """Block-sparse attention (d = 64, 128 x 128 tiles: sliding window of 8
    tiles + 10 % of the other lower tiles, 1722 of 16384 per head)."""
    from online_softmax_attention_rf_gb300 import api
    w = inputs.WORKLOADS["block_sparse"]
    q_h, k_h, v_h, scale, extras = inputs.workload_inputs("block_sparse")
    tm = extras["tile_mask"]
    flops = 4.0 * w["d"] * visible_pairs(w, tm) * w["B"] * w["H"]
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    bm = api.BlockMask.from_dense(tm, device=dev)

    def step():
        api.attn_fwd(q, k, v, scale, w["causal"], bm, o, lse)

    # Q, O (268 MB) exceed L2; K and V of a head (4 MB) are re-read from L2
    total, per = time_side(step, args, stream)[:2]
    ms = statistics.mean(per)
    assert api.device_status() == 0
    tf = flops / (ms * 1e-3) / 1e12
    out = {"workload": "block_sparse [B=2, H=16, S=16384, d=64, 1722 of 16384 tiles per head]",
           "value": tf, "unit": "TFLOP/s", "ms_per_step": ms, "listed_tiles_per_head": int(tm.sum()),
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                        "traffic": traffic_for("attn_tc_block_sparse"),
                        "peak_source": "%s dense bf16 (burst)" % peak_src,
                        "note": "algorithmic flops count the listed tiles' pairs (non-causal)"}}
    del q, k, v, o, lse, bm
    torch.cuda.empty_cache()
    return out


def bench_scattered(args, dev, stream, peaks, peak_src):
    """Short sequences under a scattered element mask (STOF's row-wise
    kernel regime): both kernels timed, and the analytic selector's choice."""
    from online_softmax_attention_rf_gb300 import api
    w = inputs.WORKLOADS["scattered_short"]
    q_h, k_h, v_h, scale, extras = inputs.workload_inputs("scattered_short")
    em = extras["elem_mask"]
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    bm = api.BlockMask.from_dense_elements(em, device=dev)
    counts = api.selector_counts(w["B"], w["H"], w["Sq"], w["Sk"], False, bm, dev)
    choice = api.choose_kernel(w["B"], w["H"], w["Sq"], w["Sk"], w["d"], *counts, device=dev)
    est_block, est_row = api.estimate_us(w["B"], w["H"], w["Sq"], w["Sk"], w["d"], *counts,
                                         device=dev)
    flops = 4.0 * w["d"] * counts[2]
    times = {}
    for kern in ("block", "row"):
        def step(kern=kern):
            api.attn_fwd(q, k, v, scale, False, bm, o, lse, kernel=kern)

        # Q, K, V, O are 134 MB (above L2); K and V of a head (256 KB) are re-read
        _, per = time_side(step, args, stream)[:2]
        times[kern] = statistics.mean(per)
    assert api.device_status() == 0
    chosen = "row" if choice == api.RF_KERNEL_ROWWISE else "block"
    ms = times[chosen]
    tf = flops / (ms * 1e-3) / 1e12
    out = {"workload": "scattered_short [B=16, H=16, S=1024, d=64; window 16, 8 global, "
                       "1 % random keys]",
           "value": tf, "unit": "TFLOP/s (visible pairs)", "ms_per_step": ms,
           "selected_kernel": chosen, "ms_block": times["block"], "ms_row": times["row"],
           "model_us": {"block": est_block, "row": est_row},
           "listed_tiles": counts[0], "partial_tiles": counts[1], "visible_pairs": counts[2],
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                        "traffic": traffic_for("attn_tc_scattered_short") if chosen == "block"
                        else None,
                        "peak_source": "%s dense bf16 (burst)" % peak_src,
                        "note": "flops over visible pairs only"}}
    del q, k, v, o, lse, bm
    torch.cuda.empty_cache()
    return out


def bench_mla(args, dev, stream, peaks, peak_src):
    """MLA decode (absorbed form, B = 32, Sk = 8192, 128 heads, 576 / 512
    columns): partials on the tensor cores + the log-sum-exp merge."""
    from online_softmax_attention_rf_gb300 import api
    w = inputs.MLA_WORKLOADS["mla_decode"]
    q_h, kv_h = inputs.make_mla(w["B"], w["Sk"], w["seed"], w["amp"])
    q, kv = q_h.to(dev), kv_h.to(dev)
    o = torch.empty(w["B"], 128, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w["B"], 128, dtype=torch.float32, device=dev)
    nb = api.lib().rf_mla_decode_workspace_bytes(w["B"], w["nsplit"])
    ws = torch.empty(nb // 4, dtype=torch.float32, device=dev)

    def step():
        api.mla_decode(q, kv, w["nsplit"], w["scale"], ws, o, lse)

    # the latent cache (302 MB) is larger than L2: no flush needed
    _, per = time_side(step, args, stream)[:2]
    ms = statistics.mean(per)
    assert api.device_status() == 0
    flops = 2.0 * w["B"] * w["Sk"] * 128 * (576 + 512)
    algo = kv.numel() * 2 + q.numel() * 2 + o.numel() * 2 + lse.numel() * 4
    tf = flops / (ms * 1e-3) / 1e12
    out = {"workload": "mla_decode [B=32, Sk=8192, 128 heads, d_qk 576, d_v 512, 16 splits]",
           "value": tf, "unit": "TFLOP/s", "ms_per_step": ms,
           "gbs": algo / (ms * 1e-3) / 1e9, "algorithmic_bytes": algo,
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                        "hbm_frac": algo / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                        "traffic": traffic_for("mla_decode"),
                        "peak_source": "%s dense bf16 (burst)" % peak_src,
                        "note": "flops count Q K^T over 576 columns and P V over 512 once; "
                                "the two value halves recompute the scores (1.53x the MMAs)"}}
    del q, kv, o, lse, ws
    torch.cuda.empty_cache()
    return out


def bench_two_level(args, dev, stream, peaks, peak_src):
    """Attention under the two-level (element) mask workload; the device
    encoder of the mask is timed separately (once per mask)."""
    from online_softmax_attention_rf_gb300 import api
    w = inputs.WORKLOADS["two_level"]
    q_h, k_h, v_h, scale, extras = inputs.workload_inputs("two_level")
    em = extras["elem_mask"]
    pairs = int(em.sum())
    flops = 4.0 * w["d"] * pairs * w["B"] * w["H"]
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    bm = api.BlockMask.from_dense_elements(em, device=dev)
    # the device encoder alone, on the resident dense mask (one launch set)
    dense = torch.as_tensor(em).to(dev).to(torch.uint8).unsqueeze(0)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    api.blockmask_build_elements(dense, bm.row_ptr, bm.col_idx, bm.tile_bits, bm.bits)
    t1.record(stream)
    t1.synchronize()
    build_ms = t0.elapsed_time(t1)
    del dense
    nnz = int(bm.row_ptr[-1].item())
    n_partial = int((bm.tile_bits[:nnz] >= 0).sum().item())

    def step():
        api.attn_fwd(q, k, v, scale, False, bm, o, lse)

    # K and V of a head (4 MB) are re-read from L2 by its CTAs; Q, O (268 MB) exceed L2
    total, per = time_side(step, args, stream)[:2]
    ms = statistics.mean(per)
    assert api.device_status() == 0
    tf = flops / (ms * 1e-3) / 1e12
    out = {"workload": "two_level [B=2, H=16, S=16384, d=64, band 256 + 64 global tokens]",
           "value": tf, "unit": "TFLOP/s", "ms_per_step": ms, "visible_pairs_per_head": pairs,
           "listed_tiles_per_head": nnz, "partial_tiles_per_head": n_partial,
           "mask_build_ms": build_ms,
           "mask_build_note": "rf_blockmask_build_elements on the resident 16384 x 16384 uint8 mask",
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                        "traffic": traffic_for("attn_tc_two_level"),
                        "peak_source": "%s dense bf16 (burst)" % peak_src,
                        "note": "algorithmic flops count visible pairs only"}}
    del q, k, v, o, lse, bm
    torch.cuda.empty_cache()
    return out


def bench_softmax(args, dev, stream, peaks, peak_src, name="rows_64k"):
    from online_softmax_attention_rf_gb300 import api
    sw = inputs.SOFTMAX_WORKLOADS[name]
    x = inputs.make_rows(sw["rows"], sw["cols"], sw["seed"]).to(dev)
    y = torch.empty_like(x)
    algo = 2 * x.numel() * 4

    def step():
        api.softmax_rows(x, y)

    # x and y (2 GiB) are far larger than L2: no flush needed
    total, per = time_side(step, args, stream)[:2]
    ms = statistics.mean(per)
    gbs = algo / (ms * 1e-3) / 1e9
    assert api.device_status() == 0
    out = {"workload": "%s [%d x %d] f32" % (name, sw["rows"], sw["cols"]), "value": gbs,
           "unit": "GB/s", "ms_per_step": ms,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / peaks["hbm_gbs"], "frac_of_8TBs": gbs / 8000.0,
                        "traffic": traffic_for("softmax_" + name),
                        "peak_source": "%s HBM copy" % peak_src}}
    del x, y
    torch.cuda.empty_cache()
    return out


def bench_cascades(args, dev, stream, peaks, peak_src):
    """Other cascaded reductions: MoE top-k routing and row moments (both
    HBM-bound: each input element is read once, outputs written once)."""
    from online_softmax_attention_rf_gb300 import api
    out = {}
    c = inputs.CASCADE_WORKLOADS["moe_route"]
    x = inputs.make_logits(c["T"], c["E"], c["seed"], c["dtype"], c["amp"]).to(dev)
    idx = torch.empty(c["T"], c["k"], dtype=torch.int32, device=dev)
    w = torch.empty(c["T"], c["k"], dtype=torch.float32, device=dev)
    lse = torch.empty(c["T"], dtype=torch.float32, device=dev)
    algo = x.numel() * x.element_size() + idx.numel() * 4 + w.numel() * 4 + lse.numel() * 4

    def step_route():
        api.lib().rf_moe_route(x.data_ptr(), c["T"], c["E"], c["k"], int(c["renorm"]),
                               idx.data_ptr(), w.data_ptr(), lse.data_ptr(), api.RF_F32,
                               api._stream())

    # logits + outputs = 138 MB per step, larger than L2 (129 MB): no flush
    total, per = time_side(step_route, args, stream)[:2]
    ms = statistics.mean(per)
    assert api.device_status() == 0
    gbs = algo / (ms * 1e-3) / 1e9
    out["moe_route"] = {
        "workload": "moe_route [T=%d, E=%d, top %d, renorm] f32 logits" % (c["T"], c["E"], c["k"]),
        "value": c["T"] / (ms * 1e-3) / 1e9, "unit": "Gtokens/s", "ms_per_step": ms,
        "algorithmic_bytes": algo,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": traffic_for("moe_route"),
                     "peak_source": "%s HBM copy" % peak_src}}
    del x, idx, w, lse
    c = inputs.CASCADE_WORKLOADS["row_moments"]
    x = inputs.make_moment_rows(c["rows"], c["cols"], c["seed"], c["dtype"], c["amp"],
                                c["offset"]).to(dev)
    y = torch.empty_like(x)
    mean = torch.empty(c["rows"], dtype=torch.float32, device=dev)
    var = torch.empty_like(mean)
    algo = 2 * x.numel() * x.element_size() + 2 * mean.numel() * 4

    def step_moments():
        api.lib().rf_row_moments(x.data_ptr(), c["rows"], c["cols"], c["eps"], mean.data_ptr(),
                                 var.data_ptr(), y.data_ptr(), api.RF_F32, api._stream())

    # x and y (1 GiB) are far larger than L2: no flush needed
    total, per = time_side(step_moments, args, stream)[:2]
    ms = statistics.mean(per)
    assert api.device_status() == 0
    gbs = algo / (ms * 1e-3) / 1e9
    out["row_moments"] = {
        "workload": "row_moments [%d x %d] f32, normalised rows written" % (c["rows"], c["cols"]),
        "value": gbs, "unit": "GB/s", "ms_per_step": ms, "algorithmic_bytes": algo,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": traffic_for("row_moments"),
                     "peak_source": "%s HBM copy" % peak_src}}
    del x, y, mean, var
    c = inputs.CASCADE_WORKLOADS["inertia"]
    pts, ms = inputs.make_point_sets(c["sets"], c["n"], c["seed"], c["amp"], c["offset"])
    pts, ms = pts.to(dev), ms.to(dev)
    total = torch.empty(c["sets"], dtype=torch.float32, device=dev)
    centre = torch.empty(c["sets"], 3, dtype=torch.float32, device=dev)
    inertia = torch.empty_like(total)
    algo = pts.numel() * 4 + ms.numel() * 4 + c["sets"] * 5 * 4

    def step_inertia():
        api.lib().rf_moment_of_inertia(pts.data_ptr(), ms.data_ptr(), c["sets"], c["n"],
                                       total.data_ptr(), centre.data_ptr(), inertia.data_ptr(),
                                       api._stream())

    # points and masses (1.07 GB) are far larger than L2: no flush needed
    total_ms, per = time_side(step_inertia, args, stream)[:2]
    ms_ = statistics.mean(per)
    assert api.device_status() == 0
    gbs = algo / (ms_ * 1e-3) / 1e9
    out["moment_of_inertia"] = {
        "workload": "moment_of_inertia [%d sets x %d points, 3-D, f32 masses]" % (c["sets"],
                                                                               c["n"]),
        "value": gbs, "unit": "GB/s", "ms_per_step": ms_, "algorithmic_bytes": algo,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": traffic_for("inertia"),
                     "peak_source": "%s HBM copy" % peak_src}}
    del pts, ms, total, centre, inertia
    # FP8: per-row quantisation of the activations, then the GEMM over codes
    c = inputs.CASCADE_WORKLOADS["fp8_gemm"]
    a_h, w_h = inputs.make_gemm_operands(c["M"], c["N"], c["K"], c["seed"])
    a, wt = a_h.to(dev), w_h.to(dev)
    qa = torch.empty(c["M"], c["K"], dtype=torch.uint8, device=dev)
    sa = torch.empty(c["M"], dtype=torch.float32, device=dev)
    qw, sw = api.rowquant_e4m3(wt)            # weights: quantised once
    cm = torch.empty(c["M"], c["N"], dtype=torch.bfloat16, device=dev)

    def step_quant():
        api.lib().rf_rowquant_e4m3(a.data_ptr(), c["M"], c["K"], qa.data_ptr(), sa.data_ptr(),
                                   api.RF_BF16, api._stream())

    def step_gemm():
        api.lib().rf_fp8_gemm(qa.data_ptr(), sa.data_ptr(), qw.data_ptr(), sw.data_ptr(),
                              cm.data_ptr(), c["M"], c["N"], c["K"], api._stream())

    # A (128 MiB bf16) + codes (64 MiB) exceed L2 for the quantiser; the GEMM
    # reads 128 MiB of codes and writes 128 MiB of C per launch
    _, per_q = time_side(step_quant, args, stream)[:2]
    _, per_g = time_side(step_gemm, args, stream)[:2]
    assert api.device_status() == 0
    ms_q, ms_g = statistics.mean(per_q), statistics.mean(per_g)
    qbytes = a.numel() * 2 + qa.numel() + sa.numel() * 4
    flops = 2.0 * c["M"] * c["N"] * c["K"]
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    tf = flops / (ms_g * 1e-3) / 1e12
    out["fp8_quant"] = {
        "workload": "rowquant_e4m3 [%d x %d] bf16 -> E4M3 codes + row scales" % (c["M"], c["K"]),
        "value": qbytes / (ms_q * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms_q,
        "algorithmic_bytes": qbytes,
        "roofline": {"bound": "hbm", "achieved": qbytes / (ms_q * 1e-3) / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": qbytes / (ms_q * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "traffic": traffic_for("rowquant"), "peak_source": "%s HBM copy" % peak_src}}
    out["fp8_gemm"] = {
        "workload": "fp8_gemm E4M3 [M=%d, N=%d, K=%d] -> bf16, row and column scales" % (
            c["M"], c["N"], c["K"]),
        "value": tf, "unit": "TFLOP/s", "ms_per_step": ms_g, "ms_with_quant": ms_g + ms_q,
        "roofline": {"bound": "tensor", "achieved": tf, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": tf / fp8_peak, "traffic": traffic_for("fp8_gemm"),
                     "peak_source": "%s dense bf16 (burst) x 2, the nominal fp8/bf16 ratio"
                                    % peak_src}}
    del a, wt, qa, sa, qw, sw, cm
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--min-side-s", type=float, default=MIN_SIDE_S,
                    help="least time over which each secondary workload is timed (a launch "
                         "list capture sets 0: a few launches of each)")
    ap.add_argument("--only", choices=["all", "prefill", "mha_prefill", "tiny", "decode",
                                       "softmax", "softmax_long", "block_sparse", "two_level",
                                       "scattered", "mla", "cascades"],
                    default="all",
                    help="time one workload alone (for profiling); the default runs all")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dist, rank, world, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, dist, rank)
        else:
            run_ours(args, dist, rank, world, local)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
