"""Benchmark: MLA paged-KV decode on GB300, one JSON line on rank 0.

Workload: dense MLA decode, batch 64, s_q 1, h_q 128, d_qk 576, d_v 512,
bf16, 64-token pages, cache_seqlens uniform in [2048, 4096], random block
table over a 1.2x page pool, Q/KV ~ N(0, 1) (seeded, synthetic).

One step = one mla_decode_fwd call (split-KV attention kernel + combine
kernel) over that batch, inputs resident in HBM.  L2 is flushed (512 MiB
write) before every timed step, outside the timed events.
  value      = unique KV bytes read (sum_b L_b * 1152) / device time per step,
               GB/s, summed over ranks (each rank runs its own replica batch).
  e2e        = same metric through the public API with per-step inputs
               (Q, block table, seqlens) copied from pinned host memory,
               the scheduler run, the decode, and out/lse copied back.
  roofline   = the split-KV attention kernel alone (mla_decode_splits),
               KV bytes / its event-timed duration vs measured HBM bandwidth.
  cpu_baseline = the CPU fp64 oracle on a bounded sample of the same batch;
               its outputs also gate parity before anything is timed.
  workloads  = the other named workloads (tiny, long context, two-token
               causal, sparse FP8) timed the same way on one GPU: µs per
               decode + combine call and bytes read per second.
--impl reference times that oracle instead (the CPU reference arm).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "dense_b64_hq128_sk2048to4096"
METRIC = "MLA decode µs/call and achieved KV-read HBM GB/s (% of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["mla_paged_kv_gb300/csrc/decode_dense.cu", "mla_paged_kv_gb300/csrc/ptx.cuh",
                  "mla_paged_kv_gb300/csrc/common.cuh"]
PROFILE = os.path.join(ROOT, "profiles", "dense_decode_b64_hq128_sk2048to4096.md")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU oracle sample")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-other", action="store_true", help="skip timing the other named workloads")
    ap.add_argument("--other", default="", help="comma-separated subset of the other named workloads to time")
    return ap.parse_args()


def dist_setup(n):
    import torch
    if n <= 1 or "RANK" not in os.environ:
        return 0, 1, None
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    world = int(os.environ["WORLD_SIZE"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, dist


def max_over_ranks(x, dist, device):
    """The slowest rank's value (all ranks get it); x itself on a single process."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, bytes_per_rank, ms_slowest):
    """Whole-job GB/s: every rank processed its own batch in the slowest rank's time."""
    return world * bytes_per_rank / (ms_slowest * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak_tflops():
    """Burst cuBLAS bf16 TFLOP/s of MEASURED_PEAKS.json (a call is timed alone), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def source_sha():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it matches the kernel source."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram_bytes_per_launch_full_workload:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != source_sha():
        return None
    return float(m_b.group(1))


class ClockSampler:
    QUERY = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        # raw samples; the JSON line carries their summary
        self.path = os.path.join(os.environ.get("MLA_BENCH_OUT", os.path.join(ROOT, "bench_out")),
                                 f"clocks_{os.getpid()}.csv")

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self, bus_id=None):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        self.fh.close()
        rows = [r.split(", ") for r in open(self.path).read().strip().splitlines() if r.count(",") >= 9]
        if bus_id:
            mine = [r for r in rows if r[1].strip().lower().endswith(bus_id.lower()[-12:])]
            rows = mine or rows
        if not rows:
            return None
        idx0 = rows[0][0]
        rows = [r for r in rows if r[0] == idx0]
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        sm_max = max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        loaded = [s for s in sm if s > 0.5 * sm_max] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": sm_max,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_sample(case, budget_s, gpu_out=None, gpu_lse=None):
    """Time the fp64 oracle on whole requests until the budget is used; optionally gate parity."""
    import numpy as np
    from oracle import mla_oracle as orc
    q = case.q.double().numpy()
    kv = case.kv.float().numpy()
    bt = case.block_table.numpy()
    sl = case.cache_seqlens.numpy()
    done, kv_bytes, t_total = [], 0, 0.0
    errs = None
    n = 0
    while True:               # whole requests, cycling over the batch, until the budget is used
        b = n % case.batch
        n += 1
        t0 = time.perf_counter()
        out, lse = orc.dense_decode(q, kv, bt, sl, case.causal, case.scale, batches=[b])
        t_total += time.perf_counter() - t0
        done.append(b)
        kv_bytes += int(sl[b]) * 1152
        if gpu_out is not None and n <= case.batch:
            o = gpu_out[b].double().numpy()
            l = gpu_lse[b].double().numpy()
            ro, rl = out[b], lse[b]
            e = {"max_abs": float(np.abs(o - ro).max()),
                 "rel_fro": float(np.linalg.norm(o - ro) / np.linalg.norm(ro)),
                 "lse_abs": float(np.abs(l - rl).max())}
            errs = e if errs is None else {k: max(errs[k], e[k]) for k in e}
        if t_total >= budget_s and n >= min(case.batch, 1 if gpu_out is None else case.batch):
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"kv_bytes": kv_bytes, "seconds": t_total, "requests": done, "cores": cores, "errors": errs}


def cpu_model():
    """The host CPU's model name (/proc/cpuinfo; Arm hosts list an implementer/part instead)."""
    try:
        text = open("/proc/cpuinfo").read()
    except OSError:
        return None
    for key in ("model name", "Model", "cpu model"):
        m = re.search(rf"^{key}\s*:\s*(.+)$", text, flags=re.M)
        if m:
            return m.group(1).strip()
    parts = sorted(set(re.findall(r"^CPU part\s*:\s*(\S+)", text, flags=re.M)))
    impl = sorted(set(re.findall(r"^CPU implementer\s*:\s*(\S+)", text, flags=re.M)))
    if not parts:
        return None
    # Arm's published part numbers for the cores these hosts carry (implementer 0x41 = Arm)
    arm_parts = {"0xd4f": "Neoverse V2", "0xd40": "Neoverse V1", "0xd0c": "Neoverse N1", "0xd49": "Neoverse N2",
                 "0xd84": "Neoverse V3"}
    names = [arm_parts[p] for p in parts if impl == ["0x41"] and p in arm_parts]
    raw = f"implementer {','.join(impl)} part {','.join(parts)}"
    return f"{', '.join(names)} ({raw})" if names else raw


_ONE_THREAD_SCRIPT = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
from mla_paged_kv_gb300 import workloads as wl
from oracle import mla_oracle as orc
spec = json.loads(sys.argv[2]); kind = spec.pop("kind")
case = wl.dense_case(**spec)
q, kv = case.q.double().numpy(), case.kv.float().numpy()
bt, sl = case.block_table.numpy(), case.cache_seqlens.numpy()
t0 = time.perf_counter(); n = 0; nbytes = 0
while n < 1 or time.perf_counter() - t0 < float(sys.argv[3]):
    b = n % case.batch
    orc.dense_decode(q, kv, bt, sl, case.causal, case.scale, batches=[b])
    nbytes += int(sl[b]) * 1152; n += 1
print(json.dumps({"seconds": time.perf_counter() - t0, "kv_bytes": nbytes, "requests": n}))
"""


def cpu_oracle_one_thread(spec, budget_s):
    """The same oracle in a child process with every BLAS/OpenMP pool held to one thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               NUMEXPR_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    try:
        res = subprocess.run([sys.executable, "-c", _ONE_THREAD_SCRIPT, ROOT, json.dumps(spec), str(budget_s)],
                             capture_output=True, text=True, env=env, timeout=600)
        r = json.loads(res.stdout.strip().splitlines()[-1])
        return {"value": r["kv_bytes"] / r["seconds"] / 1e9, "unit": "GB/s", "cores": 1,
                "sample": f"{r['requests']} requests, {r['seconds']:.1f} s"}
    except Exception as e:  # the baseline is context; its absence must not stop the bench
        return {"value": None, "error": str(e)[-200:]}


def dense_flops(case):
    """2 * (576 + 512) flops per (query row, visible key): Q K^T and P V."""
    L = case.cache_seqlens.long()
    s_q, h_q = case.s_q, case.h_q
    vis = 0
    for i in range(s_q):
        vis += int((L - s_q + i + 1).clamp(min=0).sum()) if case.causal else int(L.sum())
    return 2.0 * (576 + 512) * h_q * vis


def stats_us(ms):
    return {"mean": 1e3 * statistics.mean(ms), "median": 1e3 * statistics.median(ms), "min": 1e3 * min(ms)}


OTHER_WORKLOADS = ["dense_b1_hq16_sk256_fp32out", "dense_b1_hq64_sk65536", "dense_b16_sq2causal_hq128_sk4096to8192",
                   "dense_b64_hq128_sk2048to4096_fp16", "dense_b32_hkv2_hq128_sk2048to4096",
                   "dense_fp8_b64_hq128_sk2048to4096",
                   "sparse_fp8_b16_hq128_topk2048", "sparse_fp8_b4_sq4_hq64_topk2048",
                   "sparse_fp8_b2_sq8_hq128_topk2048"]


def time_other_workloads(mla, wl, timed, steps, names=None):
    """µs per mla_decode_fwd / mla_sparse_fp8_decode_fwd call (L2 flushed before each) on the other workloads."""
    import torch
    res = {}
    for name in (names or OTHER_WORKLOADS):
        case = wl.make(name)
        sparse = name.startswith("sparse")
        fp8_dense = name.startswith("dense_fp8")
        q = case.q.cuda()
        B, s_q, h_q = case.batch, case.s_q, case.h_q
        out = torch.empty(B, s_q, h_q, 512, device="cuda",
                          dtype=torch.float32 if getattr(case, "out_fp32", False) else case.q.dtype)
        lse = torch.empty(B, s_q, h_q, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        if sparse:
            kv8, ind, tl = case.kv8.cuda(), case.indices.cuda(), case.topk_length.cuda()
            pl = mla.plan(tl.reshape(-1).contiguous(), B * s_q, h_q, sparse=True, default_length=ind.shape[2])

            def fn():
                mla.mla_sparse_fp8_decode_fwd(q, kv8, ind, tl, pl.sched, pl.split_offset, pl.num_parts,
                                              pl.workspace, out, lse, status, case.scale)
        elif fp8_dense:
            # the FP8 record cache through mla_decode_fwd (dtype FP8_RECORD: the
            # sparse kernel with the block table as its slot source, dense plan)
            kv8, bt, sl = case.kv8.cuda(), case.block_table.cuda(), case.cache_seqlens.cuda()
            pl = mla.plan(sl, B, s_q * h_q, num_parts=mla.mla_num_parts_dense(s_q, h_q, 1))

            def fn():
                mla.mla_decode_fwd(q, kv8, bt, sl, pl.sched, pl.split_offset, pl.num_parts, pl.workspace, out, lse,
                                   status, case.causal, case.scale)
        else:
            kv, bt, sl = case.kv.cuda(), case.block_table.cuda(), case.cache_seqlens.cuda()
            pl = mla.plan(sl, B, s_q * h_q, num_parts=mla.mla_num_parts_dense(s_q, h_q, case.h_kv))

            def fn():
                mla.mla_decode_fwd(q, kv, bt, sl, pl.sched, pl.split_offset, pl.num_parts, pl.workspace, out, lse,
                                   status, case.causal, case.scale)
        for _ in range(5):
            fn()
        ms = timed(fn, steps)
        mla.check_status(status, name)
        us = 1e3 * statistics.mean(ms)
        nbytes = case.kv_bytes()
        res[name] = {"us_per_call": us, "us_per_call_median": 1e3 * statistics.median(ms),
                     "us_per_call_min": 1e3 * min(ms), "gb_per_s": nbytes / (us * 1e-6) / 1e9,
                     "bytes_per_call": nbytes,
                     "bytes": ("valid records x 656" if sparse else "sum of cache_seqlens x 656" if fp8_dense
                               else "sum of cache_seqlens x 1152 x h_kv"),
                     "num_parts": pl.num_parts, "splits": int(pl.split_offset[-1].item())}
        if not sparse:
            fl = dense_flops(case)
            res[name]["tflops"] = fl / (us * 1e-6) / 1e12
            res[name]["pct_of_bf16_tensor_peak"] = 100.0 * res[name]["tflops"] / bf16_peak_tflops()
        if sparse:
            res[name + "_packed"] = time_packed(mla, case, q, kv8, ind, tl, pl, out, lse, status, timed, steps)
            # the same call under the request-local partition plan
            pl_local = mla.plan(tl.reshape(-1).contiguous(), B * s_q, h_q, sparse=True, default_length=ind.shape[2],
                                request_local=True)

            def fn_local():
                mla.mla_sparse_fp8_decode_fwd(q, kv8, ind, tl, pl_local.sched, pl_local.split_offset,
                                              pl_local.num_parts, pl_local.workspace, out, lse, status, case.scale)
            for _ in range(5):
                fn_local()
            us_local = 1e3 * statistics.mean(timed(fn_local, steps))
            mla.check_status(status, name + " request-local plan")
            res[name + "_request_local"] = {"us_per_call": us_local, "gb_per_s": nbytes / (us_local * 1e-6) / 1e9,
                                            "splits": int(pl_local.split_offset[-1].item())}
        del q, out, lse, fn
        torch.cuda.empty_cache()
    return res


def time_packed(mla, case, q, kv8, ind, tl, pl, out, lse, status, timed, steps):
    """Packed selected-KV path on the sparse workload: µs of the pack and of the
    packed attention (decode + combine), each timed alone with L2 flushed."""
    import torch
    B, s_q, topk = ind.shape
    packed = torch.empty(mla.mla_packed_kv_workspace_bytes(B * s_q, topk), dtype=torch.uint8, device="cuda")

    def pack():
        mla.mla_pack_selected_kv(kv8, ind, tl, packed, status)

    def attend():
        mla.mla_sparse_fp8_packed_decode_fwd(q, packed, topk, tl, pl.sched, pl.split_offset, pl.num_parts,
                                             pl.workspace, out, lse, status, case.scale)
    res = {}
    for key, fn in (("pack", pack), ("packed_attention", attend)):
        for _ in range(5):
            fn()
        res[key + "_us"] = 1e3 * statistics.mean(timed(fn, steps))
    mla.check_status(status, "packed path")
    nvalid = int((ind >= 0).sum().item())
    res["pack_bytes"] = nvalid * 656 * 2 + packed.numel() - nvalid * 656
    res["pack_gb_per_s"] = res["pack_bytes"] / (res["pack_us"] * 1e-6) / 1e9
    res["bytes_pack"] = "valid records read + whole packed workspace written"
    del packed
    return res


def run_reference(args):
    import torch
    from mla_paged_kv_gb300 import workloads as wl
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    case = wl.make(WORKLOAD)
    per_step = max(1.0, 60.0 / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        cpu_oracle_sample(case, per_step)
    secs, nbytes, reqs, cores = 0.0, 0, 0, 1
    for _ in range(args.steps):
        r = cpu_oracle_sample(case, per_step)
        secs += r["seconds"]
        nbytes += r["kv_bytes"]
        reqs += len(r["requests"])
        cores = r["cores"]
    gbs = nbytes / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 64, "s_q": 1, "h_q": 128, "seqlen": "uniform[2048,4096]",
                   "page_size": 64, "note": "each step = the CPU oracle on whole requests for about "
                                            f"{per_step:.1f} s (a bounded sample of the batch)"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{reqs} requests over {args.steps} steps, fp64 numpy oracle"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    import numpy as np
    import torch
    import mla_paged_kv_gb300 as mla
    from mla_paged_kv_gb300 import workloads as wl

    rank, world, dist = dist_setup(args.gpus)
    dev = torch.device("cuda", torch.cuda.current_device())
    spec = dict(wl.WORKLOADS[WORKLOAD])
    spec.pop("kind")
    spec["seed"] = spec["seed"] + 7919 * rank          # each rank its own replica batch
    case = wl.dense_case(**spec)
    B, s_q, h_q = case.batch, case.s_q, case.h_q
    kv_bytes = case.kv_bytes()

    q = case.q.to(dev)
    kv = case.kv.to(dev)
    bt = case.block_table.to(dev)
    sl = case.cache_seqlens.to(dev)
    pl = mla.plan(sl, B, s_q * h_q)
    out = torch.empty(B, s_q, h_q, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, s_q, h_q, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)

    def step(o=out, l=lse):
        mla.mla_decode_fwd(q, kv, bt, sl, pl.sched, pl.split_offset, pl.num_parts, pl.workspace, o, l, status,
                           case.causal, case.scale)

    # one checked call, then parity against the oracle sample (the CPU-baseline leg)
    step()
    torch.cuda.synchronize()
    mla.check_status(status, "mla_decode_fwd")
    cpu = None
    if rank == 0 and world == 1:
        cpu = cpu_oracle_sample(case, args.cpu_seconds, out.cpu(), lse.cpu())
        e = cpu["errors"]
        if not (e["max_abs"] <= 2e-2 and e["rel_fro"] <= 5e-3 and e["lse_abs"] <= 1e-3):
            print(json.dumps({"error": "parity check failed", "errors": e}))
            return 1

    def timed(fn, steps):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush.fill_(i & 255)
            starts[i].record()
            fn()
            ends[i].record()
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()

    # the clock sampler starts first (it sleeps while nvidia-smi comes up, and
    # an idle GPU lowers its clocks), then the warm-up steps bring the clocks
    # back before the timed ones
    sampler = ClockSampler()
    sampler.start()
    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    barrier()
    ms = timed(step, args.steps)
    barrier()
    bus = getattr(torch.cuda.get_device_properties(dev), "pci_bus_id", None)
    clocks = sampler.stop(bus if isinstance(bus, str) else None)
    mla.check_status(status, "timed loop")
    ms_step = max_over_ranks(sum(ms) / len(ms), dist, dev)

    # the split-KV attention kernel alone (roofline); its exported entry point
    def splits_only():
        mla.mla_decode_splits(q, kv, bt, sl, pl.sched, pl.split_offset, pl.num_parts, pl.workspace, out, lse,
                              status, case.causal, case.scale)
    for _ in range(3):
        splits_only()
    barrier()
    ms_k = timed(splits_only, args.steps)
    barrier()
    k_ms = statistics.mean(ms_k)

    # scheduler alone (computed once per batch, reused by every layer)
    sched_ms = statistics.mean(timed(lambda: mla.mla_get_metadata(sl, B, pl.num_parts, pl.sched, pl.split_offset),
                                     max(10, args.steps // 20)))

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        hq = case.q.pin_memory()
        hbt = case.block_table.pin_memory()
        hsl = case.cache_seqlens.pin_memory()
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

        side = torch.cuda.Stream()
        lens_in, plan_done = torch.cuda.Event(), torch.cuda.Event()

        def e2e_step():
            # lengths and block table first; the plan is computed on a second
            # stream while q crosses the host link, then the decode waits for it
            cur = torch.cuda.current_stream()
            sl.copy_(hsl, non_blocking=True)
            bt.copy_(hbt, non_blocking=True)
            lens_in.record(cur)
            side.wait_event(lens_in)
            with torch.cuda.stream(side):
                mla.mla_get_metadata(sl, B, pl.num_parts, pl.sched, pl.split_offset)
            plan_done.record(side)
            q.copy_(hq, non_blocking=True)
            cur.wait_event(plan_done)
            step()
            hout.copy_(out, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)
        for _ in range(3):
            e2e_step()
        barrier()
        ms_e = timed(e2e_step, max(20, args.steps // 10))
        barrier()
        e_ms = max_over_ranks(statistics.mean(ms_e), dist, dev)
        h2d = hq.numel() * 2 + hbt.numel() * 4 + hsl.numel() * 4
        d2h = hout.numel() * 2 + hlse.numel() * 4
        e2e = {"value": job_throughput(world, kv_bytes, e_ms), "unit": "GB/s", "us_per_call": 1e3 * e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "step": "lengths and block table to the device, plan on a second stream while q is copied, "
                       "decode + combine, out and lse back to pinned host memory"}
        mla.check_status(status, "e2e loop")

    other = None
    if world == 1 and not args.no_other:
        subset = [n for n in args.other.split(",") if n]
        unknown = [n for n in subset if n not in OTHER_WORKLOADS]
        if unknown:
            raise SystemExit(f"--other: unknown workload(s) {unknown}; known: {OTHER_WORKLOADS}")
        other = time_other_workloads(mla, wl, timed, max(20, min(200, args.steps // 10)), subset or None)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    peak, peak_kind = measured_peaks()
    achieved = kv_bytes / (k_ms * 1e-3) / 1e9
    traffic = profiled_traffic()
    line = {
        "metric": METRIC,
        "value": job_throughput(world, kv_bytes, ms_step),
        "unit": "GB/s",
        "us_per_call": 1e3 * ms_step,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/KV, random block table)",
        "config": {"workload": WORKLOAD, "batch": B, "s_q": s_q, "h_q": h_q, "d_qk": 576, "d_v": 512,
                   "seqlen": "uniform[2048,4096]", "page_size": 64, "kv_bytes_per_step": kv_bytes,
                   "num_parts": pl.num_parts, "l2": "flushed before every timed step (512 MiB write)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "us_per_call_stats": stats_us(ms),
        "kv_pct_of_hbm": 100.0 * (kv_bytes / (ms_step * 1e-3) / 1e9) / peak,
        "scheduler_us": 1e3 * sched_ms,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_kind, "kernel": "dense_decode_kernel (split-KV attention)",
                     "kernel_us": 1e3 * k_ms, "kernel_us_stats": stats_us(ms_k), "traffic": traffic},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    if other is not None:
        line["workloads"] = other
    if cpu is not None:
        line["cpu_baseline"] = {"value": cpu["kv_bytes"] / cpu["seconds"] / 1e9, "unit": "GB/s",
                                "cores": cpu["cores"], "kind": "oracle", "cpu_model": cpu_model(),
                                "one_thread": cpu_oracle_one_thread(dict(wl.WORKLOADS[WORKLOAD]),
                                                                    min(10.0, args.cpu_seconds)),
                                "sample": f"{len(cpu['requests'])} requests cycling over the {B} of the batch "
                                          f"({cpu['kv_bytes']} KV bytes), "
                                          f"fp64 numpy oracle, {cpu['seconds']:.1f} s",
                                "parity_errors": cpu["errors"]}
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
