"""CSA2 decode benchmark: query-tokens/s at 128K context over 20 layers that
share one FP4 global KV (Full + HSI pool, 9 Reindex, 10 Reuse), batch 64 per
GPU, plus the HBM-roofline fraction of the dominant entry point.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

--workload decode-128k-b64-40L-ced times one decode step of the whole 40-layer
CED model instead (2 SWA layers, 3 encoder blocks of Full + 5 Reuse over three
2:1 copies, 5 decoder blocks over the per-position copy), each copy first
receiving its newest entry.

One JSON line on rank 0.  --impl reference times the fp64 CPU oracle (the
only other implementation there is) on the host cores, on a bounded sample.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 decode query-tokens/s at 128K ctx (indexer+top-k+attn); % of HBM roofline"
UNIT = "query-tokens/s"
WORKLOAD_INDEX = 2
FALLBACK_HBM_GBS = 6800.0
REF_BUDGET_S = 150
CPU_BUDGET_S = 12.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample-seqs", type=int, default=24)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="decode-128k-b64-20L",
                    help="decode-128k-b64-20L (the benchmark); decode-128k-b64-40L-ced (the 40-layer model "
                         "over four cache copies); prefill-chunk-8k-after-120k (8,192 queries); "
                         "profile-16k-b64-20L / profile-128k-b16-20L / profile-16k-b64-40L-ced / "
                         "profile-prefill-608-after-120k: smaller "
                         "shapes of the same kernels for ncu captures")
    return ap.parse_args()


def workload_of(name):
    """a Workload (one cache copy) or a Schedule (several)"""
    from synth.workloads import CED_40L, WORKLOADS, scaled, scaled_schedule
    wl = WORKLOADS[WORKLOAD_INDEX]
    if name == wl.name:
        return wl
    if name == "profile-16k-b64-20L":
        return scaled(wl, name=name, T=16384)
    if name == "profile-128k-b16-20L":
        return scaled(wl, name=name, B=16)
    if name == CED_40L.name:
        return CED_40L
    if name == WORKLOADS[4].name:
        return WORKLOADS[4]
    if name == "profile-prefill-608-after-120k":
        return scaled(WORKLOADS[4], name=name, chunk=608, T=122880 + 608)
    if name == "profile-16k-b64-40L-ced":
        return scaled_schedule(CED_40L, name=name, T=16384)
    raise SystemExit("unknown workload %r" % name)


def segments_of(wl):
    """the cache copies of a workload, each with the layers that read it"""
    return list(wl.segments) if hasattr(wl, "segments") else [wl]


def with_batch(wl, B):
    from synth.workloads import scaled, scaled_schedule
    return scaled_schedule(wl, B=B) if hasattr(wl, "segments") else scaled(wl, B=B)


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


FALLBACK_BF16_TFLOPS = 1900.0


def measured_peak(key="hbm_gbs"):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return (FALLBACK_HBM_GBS if key == "hbm_gbs" else FALLBACK_BF16_TFLOPS), "fallback"


def config_of(wl):
    segs = segments_of(wl)
    s0 = segs[0]
    cache_bytes = sum(s.B * s.n_entries * 360 for s in segs)
    if len(segs) == 1 and s0.chunk:
        layers = "chunk of %d positions written in the step; 1 Full layer, causal top-%d per query" % (s0.chunk, s0.k)
    elif len(segs) == 1:
        layers = "1 Full (+HSI pool 256x8), 9 Reindex, 10 Reuse"
    else:
        layers = ("40: SWA x2; 3 x [Full + Reuse x5] over three 2:1 copies; [Full (+HSI pool 256x8) + Reuse x3] "
                  "+ 4 x [Reindex + Reuse x3] over the per-position copy (projected indexer keys); every copy "
                  "written its newest entry in the step")
    cfg = {"workload": wl.name, "batch_per_gpu": s0.B, "context": s0.T, "layers": layers, "top_k": s0.k,
           "heads": s0.H, "indexer": "%d heads x %d FP4" % (s0.H_I, s0.d_I), "window": 128, "latent": 512,
           "l2": "inputs larger than L2 (%.2f GB FP4 cache per GPU)" % (cache_bytes / 1e9)}
    if len(segs) > 1:
        cfg["cache_bytes_per_token"] = cache_bytes / (s0.B * s0.T)
    return cfg


NOMINAL_HBM_GBS = 8000.0       # the nominal "about 8 TB/s" of HBM3e the target fraction is quoted against


def n_elig_decode(wl):
    """global entries a decode query at raw position T-1 may read: those lying
    wholly before its 128-row window (entry i covers raw positions ratio*i ..
    ratio*i + ratio - 1)"""
    return max(0, (wl.T - 1 - 127) // wl.ratio)


def attn_bytes_per_query(wl):
    """the gather of one query's attention: its k selected FP4 rows (256 B codes +
    32 B scales) and its 128 bf16 window rows"""
    return wl.k * 288 + 128 * 1024


def attn_extra_bytes_per_query(wl):
    """bytes the attention also moves that the algorithmic count leaves out: the
    query (H x 512 bf16), its k indices and the fp32 output (H x 512)"""
    return wl.H * 512 * 2 + wl.k * 4 + wl.H * 512 * 4


def op_bytes(wl):
    """algorithmic bytes each entry point must move in one step, over every copy:
    a Full scan its eligible keys (n_elig x 72 B), a Reindex its pool keys (pool
    x 72 B), an attention its gather (k x 288 B + 128 window rows x 1 KB; a
    window-only layer the window alone), a decode step's cache write the newest
    entry's hidden rows in (ratio x 1 KB) and the entry out (360 B)"""
    d = {}

    def add(name, n):
        d[name] = d.get(name, 0) + n

    for s in segments_of(wl):
        for mode in s.layers:
            if mode == "full":
                add("indexer_full", s.B * n_elig_decode(s) * 72)
            elif mode == "reindex":
                add("reindex", s.B * s.pool_len * 72)
            if mode == "swa":
                add("swa_attn", s.B * 128 * 1024)
            else:
                add("sparse_attn", s.B * attn_bytes_per_query(s))
        if s.new_entry:
            add("cache_write", s.B * (s.ratio * 1024 + 360))
    return d


def op_flops(wl):
    """the contractions of a chunked prefill, per step: the indexer's q.k over
    every (query, eligible entry, head) (2 d_I flops each) and the attention's
    two products per (query, head, key) over the 512-dim latent"""
    from synth.workloads import WINDOW
    d = {}
    for s in segments_of(wl):
        pos = s.q_positions()
        n_el = sum(max(0, (int(p) - (WINDOW - 1)) // s.ratio) for p in pos)
        d["indexer_full"] = d.get("indexer_full", 0) + s.B * n_el * s.H_I * s.d_I * 2
        d["sparse_attn"] = d.get("sparse_attn", 0) + s.B * s.n_q * s.H * (s.k + WINDOW) * 512 * 4
    return d


def tensor_roofline(wl, per_op, peak, peak_kind):
    """chunked prefill: the indexer is a contraction of 2 d_I flops per (query,
    entry, head), run on the tensor cores as fp16 MMAs; against the measured
    dense bf16 (= fp16) peak.  Its exact-score epilogue runs on the CUDA cores
    and sets the pace, so the fraction is small by construction"""
    fl = op_flops(wl)
    name = "indexer_full" if per_op["indexer_full"]["ms"] >= per_op["sparse_attn"]["ms"] else "sparse_attn"
    ach = fl[name] / (per_op[name]["ms"] * 1e-3) / 1e12
    return {"bound": "tensor", "kernel": name, "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
            "traffic": None, "flops_per_launch": fl[name] // per_op[name]["launches_per_step"],
            "launch_ms": per_op[name]["per_launch_ms"], "peak_kind": peak_kind,
            "flops": {k: v for k, v in fl.items()}}


def algorithmic_bytes(wl):
    return sum(op_bytes(wl).values())


def extra_bytes(wl):
    return sum(s.B * sum(m != "swa" for m in s.layers) * attn_extra_bytes_per_query(s) +
               s.B * sum(m == "swa" for m in s.layers) * s.H * 512 * 6 for s in segments_of(wl))


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from ncu captures: the
# attention on 64 queries, k = 512, 64 heads (it moves the same bytes at any context length); the
# decode Full scan at 128K context, 64 sequences (T).  Keyed by the SHA-256 of the kernel's source
# file at capture time: once the source changes the figure no longer describes the kernel and is
# reported as null.
MEASURED_TRAFFIC = {
    "sparse_attn": {"bytes": 24155863, "source_sha": "84a15cbef70dc54b",
                    "capture": "profiles/launches_decode-128k-b64-20L.md (k_sparse_attn_pair, 128K)"},
    "indexer_full": {"bytes": 317966720, "source_sha": "eb19be0a9b5c50a3", "T": 131072,
                     "capture": "profiles/launches_decode-128k-b64-20L.md (k_scan_full_tc, 128K)"},
}


def kernel_source_sha(name):
    import hashlib
    f = {"sparse_attn": "attn_pair.cu", "indexer_full": "indexer_tc.cu", "reindex": "reindex_tc.cu"}.get(name)
    if f is None:
        return None
    path = os.path.join(ROOT, "compressed_sparse_attention_decode_gb300", "csrc", f)
    with open(path, "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.rows = []
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
                for n, v in zip(names, r[4:8]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except Exception:
                pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- oracle timing

def oracle_caches(wl, b):
    import oracle
    return [oracle.sequence_cache(s, b) for s in segments_of(wl)]


def oracle_step(wl, b, caches, queries=None):
    """one sequence (or the given queries of it) through every layer of every copy"""
    import oracle
    for s, c in zip(segments_of(wl), caches):
        oracle.run_sequence(s, b, cache=c, queries=queries)


def oracle_units(wl):
    """the oracle's unit of timed work: a whole sequence when it has one query, else one query
    at a time, in a seeded order spread over the chunk (a sample stopped early stays
    representative); returns (queries argument, query-tokens) pairs"""
    if wl.n_q == 1:
        return [(None, 1)]
    import numpy as np
    order = np.argsort(np.random.default_rng(0).random(wl.n_q))
    return [([int(q)], 1) for q in order]


def cpu_baseline(wl, n_seqs, budget_s=CPU_BUDGET_S):
    """the oracle as it stands on the host cores: up to n_seqs sequences through all layers
    (each sequence's cache built just before it, outside the timed region), stopped once
    budget_s of timed work is done"""
    dt, tokens, seqs = 0.0, 0, 0
    for b in range(min(n_seqs, wl.B)):
        cache = oracle_caches(wl, b)
        seqs += 1
        for queries, n in oracle_units(wl):
            t0 = time.perf_counter()
            oracle_step(wl, b, cache, queries)
            dt += time.perf_counter() - t0
            tokens += n
            if dt >= budget_s:
                break
        if dt >= budget_s:
            break
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": tokens / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d query-tokens of %d sequences (of %d), all %d layers, %.1f s" % (
                tokens, seqs, wl.B, len(wl.layers), dt)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    wl = workload_of(args.workload)
    import oracle
    oracle.build()
    n = 1
    # a bounded sample: at most 4 sequences (caches built once, outside the
    # timed region), cycled; timing stops after REF_BUDGET_S so that any
    # --steps finishes within a few minutes
    seqs = list(range(min(4, wl.B, max(1, args.steps + args.warmup))))
    caches = {b: oracle_caches(wl, b) for b in seqs}
    units = oracle_units(wl)
    times = []
    t_start = time.perf_counter()
    for s in range(args.warmup + args.steps):
        b = seqs[s % len(seqs)]
        queries, n = units[(s // len(seqs)) % len(units)]
        t0 = time.perf_counter()
        oracle_step(wl, b, caches[b], queries)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
        if times and time.perf_counter() - t_start > REF_BUDGET_S:
            break
    total = sum(times)
    value = len(times) * n / total
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": len(times), "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "%s of %d per step (all %d layers), cycling over %d sequences, "
                                       "timing capped at %d s" % ("1 sequence" if wl.n_q == 1 else "1 query of 1 sequence",
                                                                  wl.B, len(wl.layers), len(seqs), REF_BUDGET_S)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our implementation

def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__
    __graft_entry__.build()
    import compressed_sparse_attention_decode_gb300 as csa
    from compressed_sparse_attention_decode_gb300.synthetic import HostInputs, build_schedule, build_step
    from compressed_sparse_attention_decode_gb300 import dist as cdist
    wl = workload_of(args.workload)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # replicas, batch-sharded: rank r owns sequences [64r, 64r+64) of a 64*N batch
    # (weak scaling, nothing exchanged on the data path)
    build = build_schedule if hasattr(wl, "segments") else build_step
    step = build(with_batch(wl, wl.B * world), seqs=cdist.shard(wl.B, rank, world))
    segs = getattr(step, "segments", [step])
    n0 = csa.csa2_launch_count()
    step.capture()
    launches_per_step = (csa.csa2_launch_count() - n0) // 2      # warm-up enqueue + captured enqueue
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step.run()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            step.run()
        ev1.record(stream)
        barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    tokens_per_step = wl.B * world * segments_of(wl)[0].n_q
    value = tokens_per_step / (ms * 1e-3)

    # per entry point device time (eager launches, events on the launching stream)
    per_op = measure_ops(step, stream, reps=max(3, min(args.steps, 20)))
    peak, peak_kind = measured_peak()
    if segments_of(wl)[0].chunk:
        roof = tensor_roofline(wl, per_op, *measured_peak("bf16_tflops"))
    else:
        roof = roofline(wl, per_op, peak, peak_kind)

    # end to end through the public API: every step copies its inputs from pinned host memory to the
    # device, runs, and copies its outputs (every layer's attention output) back.  Two buffer sets
    # alternate so that the copies of one step overlap the compute of the other (host->device and
    # device->host on their own streams; the steps themselves stay serial on the compute stream).
    hosts = [HostInputs(s) for s in segs]
    twin = step.twin()
    twin.capture()
    steps2 = (step, twin)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    parts = lambda st: getattr(st, "segments", [st])
    for st in steps2:                     # untimed: first-use allocations of the copy path
        with torch.cuda.stream(s_in):
            for h, sg in zip(hosts, parts(st)):
                h.copy_in(sg)
    torch.cuda.synchronize()
    # at least 30 steps, so that the two-buffer pipeline runs in its steady state
    n_e2e = max(30, min(args.steps, 300))
    n_e2e += n_e2e % 2                   # even: the last one runs on the twin buffers, checked below
    ev = lambda: torch.cuda.Event(enable_timing=True)
    e_in0, e_in1, e_c0, e_c1, e_o0, e_o1 = ([ev() for _ in range(n_e2e)] for _ in range(6))
    barrier()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        st = steps2[i % 2]
        if i >= 2:
            s_in.wait_event(e_c1[i - 2])          # step i-2 has read this buffer set's inputs
        e_in0[i].record(s_in)
        with torch.cuda.stream(s_in):
            for h, sg in zip(hosts, parts(st)):
                h.copy_in(sg)
        e_in1[i].record(s_in)
        stream.wait_event(e_in1[i])
        if i >= 2:
            stream.wait_event(e_o1[i - 2])        # the outputs of step i-2 have left this buffer set
        e_c0[i].record(stream)
        st.run()
        e_c1[i].record(stream)
        s_out.wait_event(e_c1[i])
        e_o0[i].record(s_out)
        with torch.cuda.stream(s_out):
            for h, sg in zip(hosts, parts(st)):
                h.out.copy_(sg.out, non_blocking=True)
        e_o1[i].record(s_out)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / n_e2e
    phase_ms = [sum(a.elapsed_time(b) for a, b in zip(x, y)) / n_e2e
                for x, y in ((e_in0, e_in1), (e_c0, e_c1), (e_o0, e_o1))]
    # the last end-to-end step's results against the graph step on the same inputs: the
    # indices must be identical and the attention outputs within the 2e-3 bound
    last = steps2[(n_e2e - 1) % 2]
    step.run()
    torch.cuda.synchronize()
    e2e_check = {"idx_identical": all(bool(torch.equal(a.idx, b.idx)) for a, b in zip(parts(last), segs))}
    err = 0.0
    for h, sg in zip(hosts, segs):
        ref_out = sg.out.cpu()
        den = ref_out.abs().amax(-1).clamp_min(1e-30)
        err = max(err, float(((h.out - ref_out).abs().amax(-1) / den).max()))
    e2e_check["out_max_rel_err"] = err
    if not (e2e_check["idx_identical"] and e2e_check["out_max_rel_err"] <= 2e-3):
        raise SystemExit("end-to-end step disagrees with the graph step: %r" % e2e_check)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([e2e_s], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": step_dtype(), "data": "synthetic", "config": config_of(wl),
                "roofline": roof,
                "step_roofline": {"algorithmic_bytes": algorithmic_bytes(wl), "extra_bytes": extra_bytes(wl),
                                  "achieved_gbs": algorithmic_bytes(wl) / (ms * 1e-3) / 1e9, "peak": peak,
                                  "frac": algorithmic_bytes(wl) / (ms * 1e-3) / 1e9 / peak,
                                  "frac_of_8tbs": algorithmic_bytes(wl) / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
                                  "note": "whole step: indexer-scan keys + gathered rows over the step time, against "
                                          "the %s copy peak (frac) and 8 TB/s (frac_of_8tbs); extra_bytes (queries, "
                                          "indices, fp32 outputs) are moved too but not counted" % peak_kind},
                "per_op_ms": {k: v["ms"] for k, v in per_op.items()},
                "e2e": {"value": tokens_per_step / e2e_s, "unit": UNIT,
                        "h2d_bytes_per_step": sum(h.h2d_bytes() for h in hosts),
                        "d2h_bytes_per_step": sum(h.d2h_bytes() for h in hosts), "h2d_ms": phase_ms[0], "step_ms": phase_ms[1],
                        "d2h_ms": phase_ms[2], "wall_ms": e2e_s * 1e3, "steps": n_e2e, "check": e2e_check,
                        "note": "per step: the step's own queries of every layer, newest window rows (and the "
                                "hidden rows of a newest entry) in, every layer's attention output out; copies of "
                                "one step overlap the compute of the other of two buffer sets"},
                "gpu_launches": launches_per_step * args.steps,
                "clocks": clk.summary()}
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, args.cpu_sample_seqs)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def step_dtype():
    return "u8 FP4 (E2M1, E4M3/16) cache; indexer int32+f64 exact; attention fp16 operands, fp32 accumulate"


def measure_ops(step, stream, reps):
    """device time of every entry point of one step: the calls an entry point
    makes in one step (in step order, on the step's own inputs) are captured as
    one CUDA graph, which is replayed reps times between CUDA events on the
    launching stream; no host launch time is inside the measurement"""
    import torch
    import compressed_sparse_attention_decode_gb300 as csa
    calls = {}

    def add(name, fn):
        calls.setdefault(name, []).append(fn)

    for sg in getattr(step, "segments", [step]):
        if sg.chunk_len:
            if sg.wik_codes is not None:
                add("cache_write", lambda sg=sg: csa.csa2_cache_write_projected(
                    sg.cache, sg.h_chunk, sg.chunk_pos, sg.w0, sg.w1, sg.wik_codes, sg.wik_scales))
            else:
                add("cache_write", lambda sg=sg: csa.csa2_cache_write(sg.cache, sg.h_chunk, sg.chunk_pos, sg.w0,
                                                                      sg.w1, sg.kraw_chunk))
        t = 0
        for l, mode in enumerate(sg.layers):
            idx_l = sg.layer_idx(l)
            if mode == "full":
                add("quantize_iq", lambda sg=sg, t=t: csa.csa2_quantize_fp4(sg.iq[t], sg.iq_codes, sg.iq_scales))
                add("indexer_full", lambda sg=sg, t=t, o=idx_l: csa.csa2_indexer_topk(
                    sg.cache, sg.iq_codes, sg.iq_scales, sg.w_head[t], sg.q_pos, sg.k,
                    sg.pool_blocks, sg.bs, idx_out=o, pool_out=sg.pool, ws=sg.ws_full))
                t += 1
            elif mode == "reindex":
                add("reindex", lambda sg=sg, t=t, o=idx_l: csa.csa2_reindex_f32(
                    sg.cache, sg.k, sg.iq[t], sg.w_head[t], sg.pool, idx_out=o, ws=sg.ws_re))
                t += 1
            # a Reuse layer launches nothing: its attention reads the latest indices in place
            add("swa_attn" if mode == "swa" else "sparse_attn",
                lambda sg=sg, l=l, i=idx_l: csa.csa2_sparse_attn(sg.cache, sg.q[l], sg.q_pos, i, sg.win[l],
                                                                 sg.swa_pos0, out=sg.out[l], ws=sg.ws_attn))
    out = {}
    for name, fns in calls.items():
        for fn in fns:               # eager warm-up of this entry point's calls
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for fn in fns:
                fn()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        out[name] = {"ms": ms, "per_launch_ms": ms / len(fns), "launches_per_step": len(fns)}
        del g
    step.run()                       # leave the step's outputs as one full step wrote them
    torch.cuda.synchronize()
    return out


def roofline(wl, per_op, peak, peak_kind):
    """HBM roofline of the entry point with the largest share of the step: its
    algorithmic bytes in one step (scan keys or gathered rows, every launch of
    it) over its device time in one step, against the measured copy peak and
    against the 8 TB/s of the target; per launch, both are divided by the
    launches, which leaves the ratio unchanged"""
    total = op_bytes(wl)
    extra = {"sparse_attn": sum(s.B * sum(m != "swa" for m in s.layers) * attn_extra_bytes_per_query(s)
                                for s in segments_of(wl))}
    name = max((n for n in per_op if n in total), key=lambda n: per_op[n]["ms"])
    n_launch = per_op[name]["launches_per_step"]
    ach = total[name] / (per_op[name]["ms"] * 1e-3) / 1e9
    traffic = None
    rec = MEASURED_TRAFFIC.get(name)
    s0 = segments_of(wl)[0]
    if rec and len(segments_of(wl)) == 1 and (s0.k, s0.H, s0.B, s0.n_q) == (512, 64, 64, 1) and \
            rec.get("T", s0.T) == s0.T and rec["source_sha"] == kernel_source_sha(name):
        traffic = rec["bytes"]
    return {"bound": "hbm", "kernel": name, "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
            "traffic": traffic, "bytes_per_launch": total[name] // n_launch,
            "extra_bytes_per_launch": extra.get(name, 0) // n_launch,
            "frac_of_8tbs": ach / NOMINAL_HBM_GBS,
            "launch_ms": per_op[name]["per_launch_ms"], "peak_kind": peak_kind}


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
