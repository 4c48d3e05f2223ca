"""Throughput of the DSA layer (fused Lightning Indexer → Top-K → sparse MLA attention).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode] [--impl ours|reference]

One step = one dsa_fused_forward over one batch of the workload (all of the
path's steps: scoring, head weighting, Top-K, gather, attention), inputs
resident in HBM.  L2 is flushed before every timed step, outside the step's
CUDA events: a 256 MB write, then a 256 MB read of another buffer, so that the
lines the write left dirty are written back before the step starts (a
write-only flush leaves L2 full of dirty lines whose write-back the step's first
kernel would pay for).  Prints one JSON line on rank 0.

Under torchrun (N > 1) every rank runs its own batch (seed offset by rank; the
sequences are independent, so no collective is on the data path): weak scaling,
value = all ranks' tokens ÷ the slowest rank's time.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (the only other arm this path has).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DSA tokens/sec (decode, prefill) on 1 GB300; % HBM and tensor-core roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch, from one ncu capture
# summarised under profiles/, valid only for the kernel sources it was taken with: a change to
# any of them (their hash differs) makes the figure unknown again.
MEASURED_TRAFFIC = {
    # (kernel, workload): (bytes per launch, sources, sha256 prefix of the sources); a kernel
    # whose sources changed since the capture reports null (profiles/ has the captures)
    ("indexer_topk_bf16", "decode"): (179_720_960, ("indexer_topk.cu", "tc_sm100.cuh", "dsa_internal.cuh"),
                    "002b3bb0257570c9"),
    ("sfa_tc", "decode"): (83_705_088, ("sfa_tc.cu", "tc_sm100.cuh", "dsa_internal.cuh"),
                    "98834c9a4a2eadfe"),
    ("sfa_tc", "prefill_8k"): (2_325_404_928, ("sfa_tc.cu", "tc_sm100.cuh", "dsa_internal.cuh"),
                    "98834c9a4a2eadfe"),
    ("topk_stream", "prefill_8k"): (33_431_040, ("topk_stream.cu", "tc_sm100.cuh", "dsa_internal.cuh"),
                    "5e134a9ae5e8b5fd"),
    ("indexer_tc_bf16_qb4", "prefill_8k"): (57_766_912, ("indexer_tc.cu", "tc_sm100.cuh", "dsa_internal.cuh"),
                    "25ff73549a3ca4b3"),
    # captured on the workload's first 16 of 128 sequences (--batch 16) and scaled by 8: the
    # key codes and their scales, read once, are 99 % of it and grow with the keys
    ("indexer_tc_mxfp8", "mxfp8_decode"): (2_255_173_632, ("indexer_tc.cu", "tc_sm100.cuh", "dsa_internal.cuh"),
                    "25ff73549a3ca4b3"),
    ("indexer_prolog", "decode"): (1_932_800, ("prolog.cu", "dsa_internal.cuh"), "45d03705f2200f27"),
}


def measured_traffic(kernel: str, workload: str):
    ent = MEASURED_TRAFFIC.get((kernel, workload))
    if ent is None:
        return None
    nbytes, files, digest = ent
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "sparse_attention_lightning_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return nbytes if h.hexdigest().startswith(digest) else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def describe(cfg) -> str:
    ql, kl = cfg.q_lens, cfg.k_lens
    lens = f"L={kl[0]}" if len(set(kl)) == 1 else f"L~[{min(kl)},{max(kl)}] (sum {sum(kl)})"
    return (f"{cfg.name}: B={cfg.num_seqs} T={sum(ql)} {lens} H_I={cfg.h_idx} d_I={cfg.d_idx} "
            f"H={cfg.h} d_c={cfg.d_c} d_rope={cfg.d_rope} top_k={cfg.top_k} "
            f"idx={cfg.idx_dtype} kv={cfg.kv_dtype}")


def positions(cfg):
    for T, L in zip(cfg.q_lens, cfg.k_lens):
        for i in range(T):
            yield L - T + i


def work_model(cfg):
    """Algorithmic bytes and flops of each stage (what the method must move/compute)."""
    es_i = {"f32": 4, "bf16": 2, "e4m3": 1, "mxfp8": 1}[cfg.idx_dtype]
    es_kv = {"f32": 4, "bf16": 2}[cfg.kv_dtype]
    es_o = {"f32": 4, "bf16": 2}[cfg.out_dtype]
    TQ, TK, D = cfg.total_q, cfg.total_k, cfg.d
    pairs = sum(p + 1 for p in positions(cfg))               # causal (query, key) pairs
    sel = sum(min(cfg.top_k, p + 1) for p in positions(cfg))  # selected (query, row) pairs
    scales = ((TK * 4 + TQ * cfg.h_idx * 4) if cfg.idx_dtype == "e4m3" else
              (TK + TQ * cfg.h_idx) * (cfg.d_idx // 32) if cfg.idx_dtype == "mxfp8" else 0)
    idx_b = TQ * cfg.top_k * 4
    indexer_bytes = TK * cfg.d_idx * es_i + TQ * cfg.h_idx * (cfg.d_idx * es_i + 4) + scales + idx_b
    sfa_bytes = TQ * cfg.h * D * es_kv + sel * D * es_kv + idx_b + TQ * cfg.h * (cfg.d_c * es_o + 4)
    return {
        "indexer": {"bytes": indexer_bytes, "flops": 2 * cfg.h_idx * cfg.d_idx * pairs},
        # Top-K reads each causal score once and writes the indices
        "topk": {"bytes": pairs * 4 + idx_b, "flops": 0},
        "sfa": {"bytes": sfa_bytes, "flops": 2 * cfg.h * (D + cfg.d_c) * sel},
        "pairs": pairs, "selected": sel,
    }


# Which stage each library kernel belongs to (for the roofline of the dominant kernel).
KERNEL_STAGE = {
    "indexer_scores_simt": "indexer", "indexer_tc_bf16": "indexer", "indexer_tc_fp8": "indexer",
    "indexer_tc_bf16_qb4": "indexer", "indexer_tc_fp8_qb4": "indexer",
    "indexer_topk_bf16": "indexer", "indexer_topk_fp8": "indexer", "indexer_tc_mxfp8": "indexer",
    "topk_rows": "topk", "topk_smem": "topk", "topk_stream": "topk",
    "sfa_simt": "sfa", "sfa_tc": "sfa",
}


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc:
            time.sleep(0.3)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_baseline(case, budget_s=(10.0, 30.0), rows=None):
    """Time the fp64 oracle on whole passes over `rows` until >= budget_s[0] seconds."""
    from oracle import dsa_oracle as O
    p = O.problem_from_case(case)
    rows = list(range(case.cfg.total_q)) if rows is None else list(rows)
    done, t0 = 0, time.perf_counter()
    passes = 0
    while True:
        for t in rows:
            p.forward_row(t)
            done += 1
            if time.perf_counter() - t0 > budget_s[1]:
                break
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s[0] or el > budget_s[1]:
            break
    return done, el, passes


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, cfg, case, rank):
    """The oracle arm: each step = the oracle over a bounded sample of query rows."""
    if rank != 0:
        return
    from oracle import dsa_oracle as O
    p = O.problem_from_case(case)
    n_sample = max(1, min(cfg.total_q, args.ref_rows))
    rows = list(range(n_sample))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        for t in rows:
            p.forward_row(t)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    el = sum(times)
    value = n_sample * len(times) / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(cfg), "sample_rows_per_step": n_sample},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                         "sample": f"first {n_sample} query rows of the workload per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "tiny_prefill", "prefill_8k", "prefill_64k", "fp8_decode",
                             "mxfp8_decode"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-rows", type=int, default=8, help="oracle rows per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling: keep only the workload's first N sequences (same shapes)")
    ap.add_argument("--extra", default="prefill_8k,fp8_decode,mxfp8_decode,prefill_64k",
                    help="other workloads timed after the primary one (N=1 only), reported "
                         "under \"workloads\"; empty for none")
    ap.add_argument("--page-size", type=int, default=0,
                    help="read the key caches through a block table of pages of this many rows "
                         "(pages in a seeded random order)")
    args = ap.parse_args()
    if args.impl == "reference":
        os.environ.setdefault("OPENBLAS_NUM_THREADS", str(cores()))
    if args.batch or args.page_size:
        args.extra = ""

    import torch
    import torch.distributed as dist

    from sparse_attention_lightning_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)

    cfg = W.workload(args.workload)
    if args.batch:
        import dataclasses
        cfg = dataclasses.replace(cfg, name=f"{cfg.name}_first{args.batch}",
                                  q_lens=list(cfg.q_lens[:args.batch]),
                                  k_lens=list(cfg.k_lens[:args.batch]))
    seed = W.WORKLOAD_SEEDS[args.workload] + 1000 * rank
    if args.impl == "reference":
        if rank == 0:
            case = W.make_case(cfg, seed)
            run_reference(args, cfg, case, rank)
        return

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import sparse_attention_lightning_gb300 as dsa
    dsa.lib()

    run = setup(dsa, W, cfg, seed, dev, args.page_size)
    case, d, P, ws, out, lse, idx, step = run
    res = time_steps(dsa, torch, dist, step, ws, dev, args.steps, args.warmup, world, local)
    step_ms, total_ms, records, clocks = res
    tokens = cfg.total_q * args.steps * world
    value = tokens / (total_ms / 1e3)
    roof, kernels = roofline(cfg, records, args.workload if not (args.batch or args.page_size)
                             else None, args.steps)

    # end to end through the public API: per-step inputs from pinned host memory, result back.
    # A serving loop overlaps transfers with compute: step i's inputs are copied in (copy-in
    # stream, one of two device input sets) while step i-1 computes, and step i-1's output
    # is copied out (copy-out stream, one of two device output buffers) while step i
    # computes; events order the reuse of each buffer.  Every step's copies are inside the
    # timed region (first copy-in to last copy-out).
    e2e = None
    if not args.no_e2e:
        keys_in = [k for k in ("q_idx", "w", "q", "q_scale") if k in case.tensors()]
        host_in = {k: case.tensors()[k].pin_memory() for k in keys_in}
        dev_in = [{k: torch.empty_like(d[k]) for k in keys_in} for _ in range(2)]
        dev_out = [torch.empty_like(out) for _ in range(2)]
        out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = out_h[0].numel() * out_h[0].element_size()
        s_c = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        n_all = args.warmup + args.steps
        in_done = [ev() for _ in range(n_all)]
        comp_done = [ev() for _ in range(n_all)]
        out_done = [ev() for _ in range(n_all)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def e2e_step(i):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])  # input set b is free
                for k in keys_in:
                    dev_in[b][k].copy_(host_in[k], non_blocking=True)
                in_done[i].record(s_in)
            s_c.wait_event(in_done[i])
            if i >= 2:
                s_c.wait_event(out_done[i - 2])        # output buffer b has been read out
            x = dict(d)
            x.update(dev_in[b])
            dsa.fused_forward(P, x["q_idx"], x["k_idx"], x["w"], x["q"], x["kv"],
                              x.get("q_scale"), x.get("k_scale"), out=dev_out[b], lse=lse,
                              idx=idx, ws=ws)
            comp_done[i].record(s_c)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                out_h[b].copy_(dev_out[b], non_blocking=True)
                out_done[i].record(s_out)

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        with torch.cuda.stream(s_in):
            t0.record(s_in)
        for i in range(args.warmup, n_all):
            e2e_step(i)
        with torch.cuda.stream(s_out):
            t1.record(s_out)
        torch.cuda.synchronize()
        e_ms = t0.elapsed_time(t1)
        e_t = torch.tensor([e_ms], dtype=torch.float64, device=dev)
        if world > 1:
            dist.all_reduce(e_t, op=dist.ReduceOp.MAX)
        e2e = {"value": tokens / (float(e_t.item()) / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "per-step query-side inputs (q_idx, w, q) host->device and out "
                       "device->host, overlapped with the neighbouring steps' compute on "
                       "copy streams (double-buffered); K/latent caches are device-resident "
                       "state; no L2 flush (the caches exceed L2)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, el, passes = oracle_baseline(case)
        cpu = {"value": n / el, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
               "sample": f"{n} query rows of this workload ({passes} pass(es) over its "
                         f"{cfg.total_q} rows), fp64 numpy on all {cores()} cores (BLAS "
                         f"threads); one_core: the same oracle with one BLAS thread",
               "seconds": el, "one_core": one_core_baseline(args.workload)}

    # the other workloads of the metric (prefill and FP8-indexer decode): each its own
    # timed steps, per-kernel roofline and clocks, on the same GPU after the primary one
    extra = {}
    if world == 1 and args.extra:
        del run, case, d, P, ws, out, lse, idx, step
        torch.cuda.empty_cache()
        for name in [x for x in args.extra.split(",") if x and x != args.workload]:
            ecfg = W.workload(name)
            erun = setup(dsa, W, ecfg, W.WORKLOAD_SEEDS[name], dev, 0)
            esteps = max(3, args.steps // 4)
            ems, etot, erec, eclk = time_steps(dsa, torch, dist, erun[-1], erun[3], dev, esteps,
                                               3, 1, local)
            eroof, ekern = roofline(ecfg, erec, name, esteps)
            extra[name] = {"value": ecfg.total_q * esteps / (etot / 1e3), "unit": "tokens/s",
                           "steps": esteps, "warmup": 3, "ms_per_step": etot / esteps,
                           "step_ms_median": statistics.median(ems), "workload": describe(ecfg),
                           "dtype": (ecfg.kv_dtype if ecfg.idx_dtype not in ("e4m3", "mxfp8")
                                     else ecfg.idx_dtype + "+bf16"),
                           "roofline": eroof, "kernels": ekern, "clocks": eclk,
                           "gpu_launches": len(erec)}
            del erun
            torch.cuda.empty_cache()
            if ecfg.idx_dtype in ("e4m3", "mxfp8"):
                extra[name]["topk_recall_vs_bf16"] = fp8_recall(dsa, W, ecfg,
                                                                W.WORKLOAD_SEEDS[name], dev)
                torch.cuda.empty_cache()
        # the indexer prolog (Q quantisation + head-weight projection, one launch) on the
        # query batches of the two decode workloads
        extra["indexer_prolog"] = {
            name: prolog_record(dsa, W, torch, dist, dev, local, name, W.WORKLOAD_SEEDS[name],
                                max(3, args.steps // 4))
            for name in ("decode", "fp8_decode")}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": (cfg.kv_dtype if cfg.idx_dtype not in ("e4m3", "mxfp8")
                      else cfg.idx_dtype + "+bf16"),
            "data": "synthetic (seeded N(0,1/sqrt(d)) values, w~U(0,1))",
            "config": {"workload": describe(cfg) + (f" paged={args.page_size}" if args.page_size
                                                    else ""),
                       "tokens_per_step_per_gpu": cfg.total_q,
                       "l2": "flushed before every timed step (256 MB write, then 256 MB read)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof, "kernels": kernels, "cpu_baseline": cpu,
            "clocks": clocks, "e2e": e2e, "gpu_launches": len(records),
            "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms),
            "workloads": extra or None,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def topk_recall(a, b):
    """Per-row recall of Top-K rows ``a`` against ``b`` (int32 [rows, k], -1 padded):
    |a ∩ b| / |b| over each row's valid entries (device tensors)."""
    import torch
    rows, k = b.shape
    big = 1 << 32
    base = torch.arange(rows, device=b.device, dtype=torch.int64)[:, None] * big
    va, vb = a >= 0, b >= 0
    hit = torch.isin((a.long() + base)[va], (b.long() + base)[vb])
    per = torch.zeros(rows, device=b.device, dtype=torch.float64)
    per.index_add_(0, torch.nonzero(va)[:, 0], hit.double())
    return per / vb.sum(1).clamp(min=1).double()


def fp8_recall(dsa, W, cfg, seed, dev, nseq=16):
    """Top-K recall of the quantised (FP8 or MXFP8) indexer against the bf16 indexer on the
    bf16 values it was quantised from (the same seeded streams), over the workload's first
    nseq sequences."""
    import dataclasses
    sub = W.first_sequences(cfg, nseq)
    res = {}
    for dt in (cfg.idx_dtype, "bf16"):
        c = dataclasses.replace(sub, idx_dtype=dt)
        case = W.make_case(c, seed, attention=False)
        d = {k: v.to(dev) for k, v in case.tensors().items() if v.numel()}
        P = dsa.Problem.from_config(c, d["cu_q"], d["cu_k"])
        res[dt], _ = dsa.fused_indexer(P, d["q_idx"], d["k_idx"], d["w"], d.get("q_scale"),
                                       d.get("k_scale"))
    r = topk_recall(res[cfg.idx_dtype], res["bf16"])
    return {"mean": float(r.mean()), "min": float(r.min()), "rows": int(r.numel()),
            "sample": f"the workload's first {nseq} sequences ({sub.total_k} keys)"}


def prolog_record(dsa, W, torch, dist, dev, local, name, seed, steps):
    """The indexer prolog on the query tokens of workload ``name``: timed like a step (L2 flushed before
    each), against HBM with its algorithmic bytes (bf16 q_proj, x and W_h read once; E4M3
    codes, per-head scales and fp32 weights written once)."""
    inp = {k: v.to(dev) for k, v in W.prolog_inputs(W.workload(name), seed).items()}
    T, h, d = inp["q_proj"].shape
    dm = inp["x"].shape[1]
    codes = torch.empty(T, h, d, dtype=torch.uint8, device=dev)
    scale = torch.empty(T, h, dtype=torch.float32, device=dev)
    w = torch.empty(T, h, dtype=torch.float32, device=dev)
    ws = dsa.Workspace(dev)

    def step():
        dsa.indexer_prolog(inp["q_proj"], inp["x"], inp["w_h"], codes, scale, w)

    ms, tot, rec, clk = time_steps(dsa, torch, dist, step, ws, dev, steps, 3, 1, local)
    alg = T * h * d * 2 + T * h * d + 2 * T * h * 4 + T * dm * 2 + h * dm * 2
    kms = statistics.mean(m for _, m in rec)
    peaks, src = load_peaks()
    ach = alg / (kms / 1e3) / 1e9
    return {"value": T * steps / (tot / 1e3), "unit": "tokens/s", "steps": steps, "warmup": 3,
            "ms_per_step": tot / steps, "step_ms_median": statistics.median(ms),
            "workload": f"indexer prolog: T={T} tokens, H_I={h}, d_I={d}, d_model={dm}, bf16 in, "
                        f"E4M3 codes + per-token scale + fp32 head weights out",
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                         "traffic": measured_traffic("indexer_prolog", name),
                         "kernel": "indexer_prolog", "algorithmic_bytes_per_launch": alg,
                         "kernel_ms": kms, "peak_source": f"{src} hbm_gbs"},
            "clocks": clk, "gpu_launches": len(rec)}


def setup(dsa, W, cfg, seed, dev, page_size):
    """Inputs of one workload on the device and a step that runs the DSA layer over them."""
    import torch
    case = W.make_case(cfg, seed)
    d = {k: v.to(dev) for k, v in case.tensors().items()}
    paging = {}
    if page_size:
        pk = W.paged_keys(case, page_size, seed)
        d.update({k: v.to(dev) for k, v in pk.tensors().items()})
        paging = dict(block_table=d["block_table"], page_size=page_size, num_pages=pk.num_pages)
    P = dsa.Problem.from_config(cfg, d["cu_q"], d["cu_k"], **paging)
    ws = dsa.Workspace(dev, P.workspace_size(5))
    out = torch.empty(cfg.total_q, cfg.h, cfg.d_c, dtype=torch.bfloat16 if cfg.out_dtype == "bf16"
                      else torch.float32, device=dev)
    lse = torch.empty(cfg.total_q, cfg.h, dtype=torch.float32, device=dev)
    idx = torch.empty(cfg.total_q, cfg.top_k, dtype=torch.int32, device=dev)

    def step():
        dsa.fused_forward(P, d["q_idx"], d["k_idx"], d["w"], d["q"], d["kv"], d.get("q_scale"),
                          d.get("k_scale"), out=out, lse=lse, idx=idx, ws=ws)

    return case, d, P, ws, out, lse, idx, step


def time_steps(dsa, torch, dist, step, ws, dev, steps, warmup, world, local):
    """Warm-up, then `steps` timed steps (CUDA events, L2 flushed before each, clocks sampled),
    then the same steps again with an event pair around every launch of the library."""
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)  # 256 MB > L2
    clean = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()                    # evicts the step's data
        torch.sum(clean, 0, out=sink)    # evicts the dirty flush lines (written back now)

    ws.clear_status()
    for _ in range(warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    flags = ws.status()
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} after warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # timed steps: no per-kernel events in the stream, so each kernel may start while the
    # one before it finishes (programmatic dependent launch)
    with ClockSampler(local) as clk:
        for i in range(steps):
            flush_l2()
            evs[i][0].record()
            step()
            evs[i][1].record()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # a second pass of the same steps with CUDA events around every launch (on its stream):
    # per-kernel durations for the roofline and the launch count
    with dsa.trace(capacity=512 * steps) as tr:  # row-chunked prefill: ~260 launches a step
        for i in range(steps):
            flush_l2()
            step()
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = sum(step_ms)
    t_max = torch.tensor([total_ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t_max, op=dist.ReduceOp.MAX)
    return step_ms, float(t_max.item()), tr.records, clk.summary()


def roofline(cfg, records, workload, steps):
    """The dominant kernel against its bound (bytes for decode-shaped problems and Top-K,
    tensor flops otherwise), and every kernel's share, mean time and achieved rate.  A stage
    that runs in several launches a step (row chunks) is measured by its time per step."""
    per_kernel = {}
    for name, ms in records:
        per_kernel.setdefault(name, []).append(ms)
    model = work_model(cfg)
    peaks, peak_src = load_peaks()
    dom = max(per_kernel, key=lambda k: sum(per_kernel[k]))
    dom_ms = sum(per_kernel[dom]) / steps
    stage = KERNEL_STAGE.get(dom, dom)
    decode_like = max(cfg.q_lens) == 1
    if decode_like or stage == "topk":
        alg = model[stage]["bytes"] if stage in model else cfg.total_q * cfg.top_k * 4
        achieved = alg / (dom_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": measured_traffic(dom, workload),
                "kernel": dom, "algorithmic_bytes_per_launch": alg,
                "peak_source": f"{peak_src} hbm_gbs"}
    else:
        alg = model[stage]["flops"]
        achieved = alg / (dom_ms / 1e3) / 1e12
        pk = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk, "unit": "TFLOP/s",
                "frac": achieved / pk, "traffic": measured_traffic(dom, workload), "kernel": dom,
                "algorithmic_flops_per_launch": alg, "peak_source": f"{peak_src} bf16_tflops"}
    roof["kernel_ms_per_step"] = dom_ms
    roof["launches_per_step"] = len(per_kernel[dom]) / steps
    total = sum(sum(x) for x in per_kernel.values())
    kernels = {k: {"launches": len(v), "ms_mean": statistics.mean(v), "share": sum(v) / total}
               for k, v in per_kernel.items()}
    # every kernel against its own bound (a chunked stage's launches share its work)
    for k, v in kernels.items():
        st = KERNEL_STAGE.get(k)
        if st not in model:
            continue
        ms = sum(per_kernel[k]) / steps  # this kernel's time per step
        if decode_like or st == "topk":
            ach = model[st]["bytes"] / (ms / 1e3) / 1e9
            v.update(achieved=ach, unit="GB/s", frac=ach / peaks["hbm_gbs"], ms_per_step=ms)
        else:
            ach = model[st]["flops"] / (ms / 1e3) / 1e12
            v.update(achieved=ach, unit="TFLOP/s", frac=ach / peaks["bf16_tflops"],
                     ms_per_step=ms)
    return roof, kernels


def one_core_baseline(workload):
    """The oracle arm of this workload with one BLAS thread, in a child process (the thread
    count of a BLAS library is fixed when it loads): tokens/s, or None if it failed."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        p = subprocess.run([sys.executable, os.path.abspath(__file__), "--impl", "reference",
                            "--workload", workload, "--steps", "2", "--warmup", "1",
                            "--ref-rows", "4"], capture_output=True, text=True, env=env,
                           timeout=600)
        return json.loads(p.stdout.strip().splitlines()[-1])["value"]
    except Exception:  # a missing number is reported as such
        return None


if __name__ == "__main__":
    main()
