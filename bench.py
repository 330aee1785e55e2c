"""Benchmark of the CSA2 FP4 decode step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 2] [--impl ours|reference]

Default workload (config 2): batched decode on a ratio-1 layer at 128K context,
32 sequences x 131,072 cached entries, 64 query heads x 512, 4-head indexer,
Top-512. One step = append the step's new token to every sequence (E2M1/E4M3 +
MXFP4 packing), score every cached entry with the indexer, select the exact
Top-512, gather/dequantise the selected entries and attend. Metric: decode
queries/s (one query = one sequence's step), whole job.

The cache (1.5 GB) is far larger than L2 (126 MB), so every step reads its
indexer keys from HBM. Timed steps run as CUDA graphs of 16 steps each; the
indexer scan of every step is bracketed by CUDA events inside the graph.

--impl reference times the CPU oracle (tests' reference implementation) on the
host cores, one sequence per step, on the same workload and metric.
Under torchrun every rank runs an independent replica on its own GPU (the path
shards by sequence; no collective); rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

SCAN_BYTES_PER_ENTRY = 68     # indexer key: 64 B codes + 4 B E8M0 scales
# DRAM read + write bytes per scanned entry of the streaming scan kernel, from one ncu
# capture of it on 16 x 131,072 entries (146.70 MB / 2,097,152 entries): the keys read
# once plus the score writes that reach DRAM during the launch. Traffic grows with the
# entries scanned, so a launch's traffic is this figure times its entries. Valid for the
# kernel as captured; it has to be measured again whenever the scan kernel changes.
SCAN_TRAFFIC_PER_ENTRY = 69.95
GATHER_BYTES_PER_ENTRY = 288  # latent: 256 B codes + 32 B E4M3 scales
STEPS_PER_GRAPH = 16
REFERENCE_BUDGET_S = 150.0   # longest timed run of the reference arm (the CPU oracle)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=4096)
    p.add_argument("--warmup", type=int, default=32)
    p.add_argument("--config", type=int, default=2)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=50)
    return p.parse_args()


# ----------------------------------------------------------------------------- dist
def dist_init(n):
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index):
        self.rows, self.err, self.proc, self.id = [], None, None, None
        try:
            self.id = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception as e:  # noqa: BLE001
            self.err = repr(e)

    def __enter__(self):
        import subprocess
        import tempfile
        self.out = tempfile.TemporaryFile(mode="w+")
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits", "-lms", "50"]
        if self.id:
            cmd += ["-i", self.id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception as e:  # noqa: BLE001
            self.err = repr(e)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait()
            self.out.seek(0)
            for line in self.out:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    self.rows.append(parts)

    def summary(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": self.err or "no samples"}
        sm = [v for v in (num(r[0]) for r in self.rows) if v is not None]
        mx = [v for v in (num(r[1]) for r in self.rows) if v is not None]
        reasons = sorted({n for r in self.rows for n, v in zip(self.NAMES, r[3:]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows), "sampler": "nvidia-smi -lms 50"}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


# ----------------------------------------------------------------------------- CPU oracle timing
def oracle_query_time(c, b, host_cache_rows, inputs, token):
    """Time one oracle decode query for sequence b: append the token, score, Top-512, attend."""
    from oracle import csa2 as O
    lc, ls, ic, isc = host_cache_rows
    q, q_idx, w = inputs
    t0 = time.perf_counter()
    new = O.encode_entries(token[0], token[1], 1)
    lc2 = np.concatenate([lc, new[0]])
    ls2 = np.concatenate([ls, new[1]])
    ic2 = np.concatenate([ic, new[2]])
    is2 = np.concatenate([isc, new[3]])
    keys = O.entry_keys(ic2, is2)
    s = O.indexer_scores(q_idx, w, keys)
    idx = O.topk_positions(s, 512)
    O.attend(q, lc2, ls2, idx)
    return time.perf_counter() - t0


def oracle_rows(c, b):
    from oracle import csa2 as O
    from fp4_compressed_kv_append_b300 import configs as CF
    lat, ikey = CF.source_tokens(c, b)
    lat, ikey = lat.cpu().numpy(), ikey.cpu().numpy()
    parts = [O.encode_entries(lat[i:i + 8192], ikey[i:i + 8192], 1) for i in range(0, len(lat), 8192)]
    return tuple(np.concatenate([p[j] for p in parts]) for j in range(4))


def oracle_inputs(c, b):
    from fp4_compressed_kv_append_b300 import workloads as WL
    q, q_idx, w = WL.queries(c["seed"], 0, c["B"], c["H"], dtype=c["dtype"], device="cuda")
    tok = WL.new_token(c["seed"], 0, c["B"], device="cuda")
    f = lambda t: t[b].float().cpu().numpy().astype(np.float64)  # noqa: E731
    return (f(q), f(q_idx), f(w)), (tok[0][b].cpu().numpy(), tok[1][b].cpu().numpy())


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:  # noqa: BLE001
        return os.cpu_count()


def cpu_baseline(c, budget_s=20.0):
    rows = oracle_rows(c, 0)
    inputs, token = oracle_inputs(c, 0)
    times = []
    t_end = time.perf_counter() + budget_s
    while time.perf_counter() < t_end and len(times) < 50:
        times.append(oracle_query_time(c, 0, rows, inputs, token))
    qps = 1.0 / statistics.median(times)
    return {"value": qps, "unit": "queries/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{len(times)} decode queries of sequence 0 ({c['tokens']} cached entries): append + "
                      f"score + Top-512 + attention, numpy float64, median time per query"}


# ----------------------------------------------------------------------------- main
def run_reference(args, rank, world):
    from fp4_compressed_kv_append_b300 import configs as CF
    if rank != 0:
        return
    c = CF.config(args.config)
    rows = oracle_rows(c, 0)
    inputs, token = oracle_inputs(c, 0)
    # one step = one oracle decode query of sequence 0 (about 0.3 s on the host cores);
    # the timed queries stop after REFERENCE_BUDGET_S so that any --steps ends within
    # a few minutes, and the rate comes from the queries timed
    for _ in range(min(args.warmup, 2)):
        oracle_query_time(c, 0, rows, inputs, token)
    times = []
    t_start = time.perf_counter()
    while len(times) < max(1, args.steps) and (not times or time.perf_counter() - t_start < REFERENCE_BUDGET_S):
        times.append(oracle_query_time(c, 0, rows, inputs, token))
    t, n = sum(times), len(times)
    value = n / t
    sample = (f"{n} decode queries of sequence 0 timed ({args.steps} steps asked; timing stops after "
              f"{REFERENCE_BUDGET_S:.0f} s): append + score + Top-512 + attention, numpy float64")
    line = {"impl": "reference", "metric": "decode queries/s", "value": value, "unit": "queries/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": c["name"], "sequences_per_step": 1,
                                            "entries": c["tokens"], "heads": c["H"], "topk": 512},
            "cpu_baseline": {"value": value, "unit": "queries/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local):
    import fp4_compressed_kv_append_b300 as K
    from fp4_compressed_kv_append_b300 import configs as CF
    from fp4_compressed_kv_append_b300 import workloads as WL

    torch.cuda.set_device(local)
    c = CF.config(args.config)
    if args.config != 2:
        raise SystemExit("the bench line is defined on config 2 (batched decode at 128K)")
    B, H, N0 = c["B"], c["H"], c["tokens"]
    n_graphs = max(1, -(-args.steps // STEPS_PER_GRAPH))
    K_steps = n_graphs * STEPS_PER_GRAPH
    warm_graphs = max(1, -(-args.warmup // STEPS_PER_GRAPH))
    # appends: device-timed graphs (+ warm-up and eager steps), then the e2e run's eager
    # warm-up, one untimed and the timed graph replays
    e2e_graphs = max(1, -(-args.e2e_steps // STEPS_PER_GRAPH))
    total_appends = (warm_graphs + n_graphs + 4) * STEPS_PER_GRAPH + (e2e_graphs + 2) * STEPS_PER_GRAPH
    wl = CF.DecodeWorkload(c, extra=total_appends)
    cache = wl.cache
    tok_lat, tok_key = WL.new_token(c["seed"], 0, B, device="cuda")

    def step(ev=None):
        """One decode step: append this step's token to every sequence, then the Full
        layer (indexer scan, cluster Top-512, gather + attention)."""
        K.kv_quant_append(tok_lat, tok_key, 1, cache)
        if ev is not None:
            K.set_scan_events(ev[0], ev[1])
        wl.step()
        if ev is not None:
            K.set_scan_events(None, None)

    # eager warm-up (sets kernel attributes before any capture), then graphs
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
          for _ in range(K_steps)]
    for a, b2 in ev:  # the hook takes raw event handles: create them on the device first
        a.record()
        b2.record()
    torch.cuda.synchronize()
    graphs = []
    l0 = K.launch_count()
    for gi in range(n_graphs + warm_graphs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for s in range(STEPS_PER_GRAPH):
                j = (gi - warm_graphs) * STEPS_PER_GRAPH + s
                step(ev[j] if j >= 0 else None)
        graphs.append(g)
    launches_per_step = (K.launch_count() - l0) / ((n_graphs + warm_graphs) * STEPS_PER_GRAPH)
    torch.cuda.synchronize()
    len_before = int(cache.len[0])
    for g in graphs[:warm_graphs]:
        g.replay()
    torch.cuda.synchronize()
    n_start = int(cache.len[0])
    assert K.sync_status() == 0

    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    with sampler:
        t0.record()
        for g in graphs[warm_graphs:]:
            g.replay()
        t1.record()
        torch.cuda.synchronize()
    barrier(world)
    ms = t0.elapsed_time(t1)
    ms = max_over_ranks(ms, world)
    st = K.sync_status()
    assert st == 0, f"device status {st}"
    scan_ms = [a.elapsed_time(b) for a, b in ev]
    scan_avg_ms = sum(scan_ms) / len(scan_ms)
    # entries scanned per step: the length after that step's append
    entries = [n_start + i + 1 for i in range(K_steps)]
    scan_bytes_avg = B * SCAN_BYTES_PER_ENTRY * sum(entries) / K_steps
    hbm_peak, peak_kind = peaks()
    achieved = scan_bytes_avg / (scan_avg_ms * 1e-3) / 1e9
    value = world * B * K_steps / (ms * 1e-3)
    step_bytes = B * (SCAN_BYTES_PER_ENTRY * sum(entries) / K_steps + GATHER_BYTES_PER_ENTRY * CF.TOPK)

    # ---- end to end through the public API with host buffers
    e2e = e2e_run(args, K, CF, wl, c, tok_lat, tok_key)

    line = {
        "metric": "decode queries/s", "value": value, "unit": "queries/s", "n_gpus": world,
        "steps": K_steps, "warmup": warm_graphs * STEPS_PER_GRAPH, "ms_per_step": ms / K_steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32 accumulate (fp4/fp8 cache, bf16 q)",
        "data": "synthetic",
        "config": {"workload": c["name"], "sequences": B, "entries": N0, "heads": H, "indexer_heads": 4,
                   "topk": CF.TOPK, "q_dtype": "bf16", "latents": "fp32 N(0,1) x LogNormal(0,1) per channel",
                   "step": "kv_quant_append of 1 token/seq + csa2_decode_step (indexer scan, cluster Top-512, "
                           "gather + sparse attention)",
                   "l2": "inputs larger than L2 (1.5 GB cache)", "parallelism": f"replicas x{world}",
                   "cuda_graphs": f"{STEPS_PER_GRAPH} steps per graph"},
        "step_algorithmic_bytes": step_bytes,
        "step_hbm_gbs": step_bytes / (ms / K_steps * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": "indexer scan", "achieved": achieved, "peak": hbm_peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "traffic": SCAN_TRAFFIC_PER_ENTRY * scan_bytes_avg / SCAN_BYTES_PER_ENTRY,
                     "scan_ms": scan_avg_ms, "bytes_per_launch": scan_bytes_avg},
        "gpu_launches": int(round(launches_per_step * K_steps)),
        "clocks": sampler.summary(),
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(c)
    if rank == 0:
        print(json.dumps(line), flush=True)


def e2e_run(args, K, CF, wl, c, tok_lat, tok_key):
    """The same step through the public API (kv_quant_append + csa2_decode_step) with
    pinned host buffers: every step copies its inputs (q, q_idx, w, the new token)
    host -> device and reads its attention output device -> host. The steps run in
    order on one compute stream (each step's append before its scan); the copies run
    on their own two streams into and out of two sets of device buffers, so a step's
    copies overlap the neighbouring steps' kernels (a serving loop's double buffering).
    """
    B, H = c["B"], c["H"]
    L0 = wl.layers[0]
    h_q = L0.q.cpu().pin_memory()
    h_qi = L0.q_idx.cpu().pin_memory()
    h_w = L0.w_idx.cpu().pin_memory()
    h_tl, h_tk = tok_lat.cpu().pin_memory(), tok_key.cpu().pin_memory()
    n_slots = 2
    slots = []
    for _ in range(n_slots):
        d = dict(q=torch.empty_like(L0.q), qi=torch.empty_like(L0.q_idx), w=torch.empty_like(L0.w_idx),
                 tl=torch.empty_like(tok_lat), tk=torch.empty_like(tok_key), out=torch.empty_like(L0.out),
                 h_out=torch.empty(B, H, 512, dtype=torch.float32).pin_memory())
        layer = K.Layer(L0.mode, d["q"], d["out"], cache=L0.cache, q_idx=d["qi"], w_idx=d["w"], pool=L0.pool,
                        idx_out=torch.empty_like(L0.idx_out))
        d["step"] = K.DecodeStep([layer], CF.TOPK, ws=wl.step.ws)  # steps are in order: one workspace
        slots.append(d)
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_qi, h_w, h_tl, h_tk))
    d2h = slots[0]["h_out"].numel() * 4
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(n_slots)]
    ev_comp = [torch.cuda.Event() for _ in range(n_slots)]
    ev_out = [torch.cuda.Event() for _ in range(n_slots)]

    def one(i):
        j = i % n_slots
        d = slots[j]
        with torch.cuda.stream(s_in):
            if i >= n_slots:
                s_in.wait_event(ev_comp[j])  # the slot's previous step has consumed its inputs
            d["q"].copy_(h_q, non_blocking=True)
            d["qi"].copy_(h_qi, non_blocking=True)
            d["w"].copy_(h_w, non_blocking=True)
            d["tl"].copy_(h_tl, non_blocking=True)
            d["tk"].copy_(h_tk, non_blocking=True)
            ev_in[j].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in[j])
            if i >= n_slots:
                s_comp.wait_event(ev_out[j])  # the slot's previous output has been read out
            K.kv_quant_append(d["tl"], d["tk"], 1, wl.cache)
            d["step"]()
            ev_comp[j].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[j])
            d["h_out"].copy_(d["out"], non_blocking=True)
            ev_out[j].record(s_out)

    for i in range(2 * n_slots):  # eager warm-up of the same sequence
        one(i)
    torch.cuda.synchronize()
    # STEPS_PER_GRAPH steps per CUDA graph (copies, appends and steps as captured
    # nodes on the three streams); replays are serialised on one stream
    cap = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for s in (s_in, s_comp, s_out):
            s.wait_stream(cap)
        for i in range(STEPS_PER_GRAPH):
            one(i)
        for s in (s_in, s_comp, s_out):
            cap.wait_stream(s)
    n_rep = max(1, -(-args.e2e_steps // STEPS_PER_GRAPH))
    g.replay()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_rep):
        g.replay()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert K.sync_status() == 0
    steps = n_rep * STEPS_PER_GRAPH
    return {"value": B * steps / dt, "unit": "queries/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "api": "kv_quant_append + csa2_decode_step, pinned host buffers, copies double-buffered on "
                   f"their own streams, {STEPS_PER_GRAPH} steps per CUDA graph",
            "steps": steps}


def main():
    args = parse()
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
