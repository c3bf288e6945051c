"""Benchmark of the paged top-k sparse-MLA hot path on GB300.

One step = one call of the fused path (store of the step's new tokens ->
indexer scores -> top-k -> latent attention) for one layer over one batch of
the synthetic workload, inputs resident in HBM.  Default workload: the agentic
MTP decode batch at ~128K context (64 sequences x 4 query tokens, lognormal
contexts with median 142K, forked subagents sharing >= 96% of their blocks).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5] [--impl smla|reference]

Prints one JSON line.  --impl reference times the CPU oracle (the plain numpy
statement of the method) on a bounded sample of the same workload.  Under
torchrun each rank runs an independent replica (the path has no exchange
step), timing is the max over ranks, and value = all ranks' query tokens /
that time.
"""

import argparse
import hashlib
import datetime
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA decode tokens/s and HBM GB/s (% of GB300 peak) at 128K context"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = {
    "kvpack_store": "store.cu",
    "smla_index_scores": "indexer.cu",
    "smla_topk": "topk.cu",
    "smla_attend": "attend.cu",
}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def max_over_ranks(value, world, device="cuda"):
    """The largest of every rank's value (all ranks receive it); the value itself at world 1."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, steps, ms):
    """Units processed by all ranks per second over `steps` steps that took `ms` (max over ranks)."""
    return world * units_per_rank * steps / (ms / 1e3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ----------------------------------------------------------------------------- clocks
CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
CLOCK_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def summarise_clocks(lines, t0=None, t1=None):
    """Median SM clock, maximum SM clock and active throttle reasons of nvidia-smi samples.

    `lines` are rows of CLOCK_FIELDS (csv, noheader, nounits).  With a window [t0, t1] of host
    times (seconds since the epoch) only the samples taken inside it count; if none of them falls
    inside (or their timestamps cannot be read) every sample counts, and `in_window` says so.
    """
    rows = []
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 10:
            continue
        try:
            sm, mx = float(parts[2]), float(parts[3])
        except ValueError:
            continue
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            ts = None
        active = {nm for nm, val in zip(CLOCK_REASONS, parts[6:10]) if val.lower().startswith("active")}
        rows.append((ts, sm, mx, active))
    if not rows:
        return None
    inside = rows
    if t0 is not None and t1 is not None:
        inside = [r for r in rows if r[0] is not None and t0 <= r[0] <= t1]
    in_window = bool(inside) and t0 is not None
    use = inside if inside else rows
    reasons = set().union(*(r[3] for r in use))
    return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
            "reasons": sorted(reasons), "samples": len(use), "in_window": in_window}


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 50 ms, summarised over a marked window."""

    def __init__(self, device_index: int, csv_path=None):
        self.proc = None
        self.t0 = self.t1 = None
        self.path = csv_path or os.path.join(tempfile.gettempdir(), f"smla_clocks_{os.getpid()}.csv")
        try:
            os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(device_index), f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def start_window(self):
        self.t0 = time.time()

    def end_window(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            return summarise_clocks(f.readlines(), self.t0, self.t1)


# ----------------------------------------------------------------------------- launch count
LIB_KERNELS = ("kvpack_store_kernel", "index_scores_kernel", "topk_kernel", "attend_kernel", "split_merge_kernel",
               "topk_merge_kernel", "lse_merge_kernel")


def count_lib_kernels(names):
    """How many of the given kernel names are this library's kernels."""
    return sum(1 for n in names if any(k in n for k in LIB_KERNELS))


def count_step_launches(step_fn) -> int:
    """Kernels of this library that one call of step_fn launches (0 if the profiler saw none, or a
    CUDA tool such as ncu is attached to the process: the two would both subscribe to CUPTI)."""
    if os.environ.get("CUDA_INJECTION64_PATH"):
        return 0
    try:
        from torch.profiler import ProfilerActivity, profile
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            step_fn()
            torch.cuda.synchronize()
        return count_lib_kernels(e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA)
    except Exception:                       # profiler unavailable: the caller falls back to the formula
        return 0


def plausible_launches(profiled: int, n_groups: int):
    """(launches per fused step, how it was obtained).  The step launches the store once and, per query
    group, the indexer, the top-k and the attention, plus at most a second top-k pass and an attention
    merge; a profiled count outside that range is not taken."""
    base = 1 + 3 * n_groups
    if base <= profiled <= base + 2 * n_groups:
        return profiled, "profiled one step"
    note = f"; profiler count {profiled} outside [{base}, {base + 2 * n_groups}]" if profiled else ""
    return base, "formula: store + 3 launches per query group" + note


# ----------------------------------------------------------------------------- accounting
def accounting(wl, topk_host):
    """Algorithmic bytes / flops per step for each kernel (see the design notes)."""
    d = wl.dims
    bs = d.block_size
    seq_lens = wl.seq_lens.cpu().numpy().astype(np.int64)
    qsl = wl.query_start_loc.cpu().numpy().astype(np.int64)
    bt = wl.block_table.cpu().numpy().astype(np.int64)
    T = wl.n_tokens
    # positions of each query token
    pos = np.empty(T, np.int64)
    seq = np.empty(T, np.int64)
    for b in range(wl.batch):
        n_q = qsl[b + 1] - qsl[b]
        pos[qsl[b]:qsl[b + 1]] = seq_lens[b] - n_q + np.arange(n_q)
        seq[qsl[b]:qsl[b + 1]] = b
    visible = int((pos + 1).sum())
    # unique physical blocks read by the indexer (prefix-shared blocks once)
    blocks = set()
    logical_keys = 0
    for b in range(wl.batch):
        n = int(pos[qsl[b + 1] - 1] + 1)
        nb = (n + bs - 1) // bs
        blocks.update(bt[b, :nb].tolist())
        logical_keys += n
    uniq_keys = len(blocks) * bs
    idx_rec = d.key_bytes + 4          # cached key (E4M3, or packed E2M1) + its fp32 scale
    rec = ((d.d_latent + 4 * (d.d_latent // d.quant_tile) + 2 * d.d_rope) + 15) // 16 * 16
    q_idx_b = T * d.n_idx_heads * d.d_index + T * d.n_idx_heads * 4
    acct = {}
    acct["smla_index_scores"] = dict(
        bytes=uniq_keys * idx_rec + q_idx_b + 4 * visible,
        logical_bytes=logical_keys * idx_rec + q_idx_b + 4 * visible,
        flops=2.0 * visible * d.n_idx_heads * d.d_index, flop_dtype="fp8")
    acct["smla_topk"] = dict(bytes=4 * visible + 4 * T * d.top_k, flops=0.0, flop_dtype=None)
    valid = topk_host >= 0
    sel_slots = set()
    for t in range(T):
        j = topk_host[t][valid[t]].astype(np.int64)
        sl = bt[seq[t], j // bs] * bs + j % bs
        sel_slots.update(sl.tolist())
    n_sel = int(valid.sum())
    q_b = T * d.n_heads * (d.d_latent + d.d_rope) * 2
    out_b = T * d.n_heads * d.d_latent * 2 + T * d.n_heads * 4
    acct["smla_attend"] = dict(
        bytes=len(sel_slots) * rec + q_b + out_b + 4 * T * d.top_k,
        logical_bytes=n_sel * rec + q_b + out_b + 4 * T * d.top_k,
        flops=2.0 * n_sel * d.n_heads * (2 * d.d_latent + d.d_rope), flop_dtype="bf16")
    acct["kvpack_store"] = dict(bytes=T * (2 * d.d_latent + 2 * d.d_rope + d.key_bytes + 4 + 8) + T * (rec + idx_rec),
                                flops=0.0, flop_dtype=None)
    acct["_step"] = dict(bytes=sum(v["bytes"] for v in acct.values()),
                         logical_bytes=sum(v.get("logical_bytes", v["bytes"]) for k, v in acct.items()),
                         visible=visible, uniq_keys=uniq_keys, logical_keys=logical_keys, n_sel=n_sel,
                         uniq_sel=len(sel_slots))
    return acct


def traffic_table():
    """ncu DRAM bytes per launch recorded under profiles/, keyed by kernel source hash."""
    path = os.path.join(ROOT, "profiles", "dram_bytes_per-launch_all-kernels_agentic-mtp4-b64-ctx142k.txt")
    out = {}
    if not os.path.exists(path):
        return out
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if len(parts) >= 4:
            out[(parts[0], parts[1])] = (parts[2], float(parts[3]))   # (kernel, workload) -> (sha, bytes)
    return out


def source_sha(kernel):
    """Hash of the kernel's source file and the device headers every kernel includes."""
    csrc = os.path.join(ROOT, "paged_sparse_mla_gb300", "csrc")
    h = hashlib.sha256()
    for name in (KERNEL_SOURCES[kernel], "smla_device.cuh", "smla_internal.h"):
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import torch.distributed as dist
    import paged_sparse_mla_gb300 as smla
    from paged_sparse_mla_gb300 import build_lib
    from paged_sparse_mla_gb300.workloads import make_config

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if rank == 0:
        build_lib.build()
    if world > 1:
        dist.barrier()
    smla.lib()
    wl = make_config(args.workload, device="cuda", scale=args.scale, key_format=args.key_format)
    d = wl.dims
    lay = smla.layout_init(d.block_size, d.n_layers, d.d_latent, d.d_rope, d.quant_tile, d.d_index, wl.num_blocks,
                           d.key_format)
    prm = smla.make_params(d.n_heads, d.n_idx_heads, d.top_k, d.softmax_scale)
    pool = torch.zeros(lay.pool_bytes, dtype=torch.uint8, device="cuda")
    s = wl.cached_slots
    for c0 in range(0, s.numel(), 1 << 20):
        sl = s[c0:c0 + (1 << 20)].contiguous()
        smla.kvpack_store(lay, pool, 0, wl.slot_latent[sl].contiguous(), wl.slot_rope[sl].contiguous(),
                          wl.slot_idx_k[sl].contiguous(), wl.slot_idx_s[sl].contiguous(), sl)
    # the per-slot generator tensors are not needed any more
    wl.slot_latent = wl.slot_rope = wl.slot_idx_k = wl.slot_idx_s = None
    torch.cuda.empty_cache()
    T = wl.n_tokens
    ws = torch.empty(smla.workspace_size(lay, prm, T, wl.max_ctx), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    topk = torch.empty((T, d.top_k), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step(o=out, l=lse, q=wl.q, qpe=wl.q_pe, qi=wl.q_idx, w=wl.w, nl=wl.new_latent, nr=wl.new_rope,
             nk=wl.new_idx_k, ns=wl.new_idx_s, sm=wl.slot_mapping, bt=wl.block_table, sq=wl.seq_lens,
             qs=wl.query_start_loc):
        smla.smla_decode(lay, prm, pool, 0, nl, nr, nk, ns, sm, q, qpe, qi, w, bt, sq, qs, wl.max_q, wl.max_ctx,
                         o, l, ws, topk_idx_out=topk, stream=stream)

    stride = (wl.max_ctx + 3) // 4 * 4
    per_group = max(1, min(T, (512 << 20) // (stride * 4)))
    n_groups = math.ceil(T / per_group)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    err = smla.smla_get_last_error()
    if err != 0:
        raise RuntimeError(f"device error during warm-up: {smla.status_string(err)}")

    # ---------------- timed region: K fused steps ----------------
    clocks = ClockSampler(local_rank, args.clocks_csv) if rank == 0 else None
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(4_000_000)   # the host enqueues ahead of the GPU from the first step on
    if clocks:
        clocks.start_window()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if clocks:
        clocks.end_window()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    err = smla.smla_get_last_error()
    if err != 0:
        raise RuntimeError(f"device error in the timed region: {smla.status_string(err)}")
    ms_step = ms / args.steps
    value = whole_job_rate(T, world, args.steps, ms)

    # ---------------- per-kernel timing: same kernels, separate calls, events on the launch stream ----------------
    kern = {k: [] for k in ("kvpack_store", "smla_index_scores", "smla_topk", "smla_attend")}
    # one launch of each kernel over all query tokens (the fused call splits long prefill into groups)
    scores = torch.empty((T, stride), dtype=torch.float32, device="cuda")
    # the attention's split scratch, as the fused step gives it (small batches split rows over CTAs)
    att_ws_bytes = smla.attend_workspace_size(lay, prm, T)
    att_ws = torch.empty(max(att_ws_bytes, 1), dtype=torch.uint8, device="cuda") if att_ws_bytes else None
    topk_ws_bytes = smla.topk_workspace_size(prm, T)
    topk_ws = torch.empty(topk_ws_bytes, dtype=torch.uint8, device="cuda") if topk_ws_bytes else None
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for it in range(args.warmup + args.steps):
        # keep the GPU busy while the host enqueues the four launches, so no host gap lands between events
        torch.cuda._sleep(4_000_000)
        ev[0].record(stream)
        smla.kvpack_store(lay, pool, 0, wl.new_latent, wl.new_rope, wl.new_idx_k, wl.new_idx_s, wl.slot_mapping,
                          stream=stream)
        ev[1].record(stream)
        smla.smla_index_scores(lay, prm, pool, 0, wl.q_idx, wl.w, wl.block_table, wl.seq_lens,
                               wl.query_start_loc, wl.max_q, wl.max_ctx, scores, stream=stream)
        ev[2].record(stream)
        smla.smla_topk(prm, scores, wl.seq_lens, wl.query_start_loc, topk, stream=stream, workspace=topk_ws)
        ev[3].record(stream)
        smla.smla_attend(lay, prm, pool, 0, wl.q, wl.q_pe, topk, wl.block_table, wl.query_start_loc, out, lse,
                         stream=stream, workspace=att_ws)
        ev[4].record(stream)
        torch.cuda.synchronize()
        if it >= args.warmup:
            for k, (a, b) in zip(kern, [(0, 1), (1, 2), (2, 3), (3, 4)]):
                kern[k].append(ev[a].elapsed_time(ev[b]))
    kern_ms = {k: (sum(v) / len(v) if v else None) for k, v in kern.items()}
    del scores
    torch.cuda.empty_cache()

    # ---------------- end to end: host buffers in, results out, every step ----------------
    host_in = {n: getattr(wl, n).cpu().pin_memory() for n in
               ("new_latent", "new_rope", "new_idx_k", "new_idx_s", "slot_mapping", "q", "q_pe", "q_idx", "w",
                "block_table", "seq_lens", "query_start_loc")}
    # Two sets of device inputs/outputs: the copies of one step (inputs on `copy`, results on
    # `back`) overlap the neighbouring steps' kernels (on `stream`); every step still moves its own
    # inputs in and its own out/lse back inside the timed region.
    dev_in = [{n: torch.empty_like(v, device="cuda") for n, v in host_in.items()} for _ in range(2)]
    dev_out = [out, torch.empty_like(out)]
    dev_lse = [lse, torch.empty_like(lse)]
    host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    host_lse = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = host_out[0].numel() * host_out[0].element_size() + host_lse[0].numel() * host_lse[0].element_size()
    copy = torch.cuda.Stream()      # host -> device
    back = torch.cuda.Stream()      # device -> host (separate, so the next inputs need not wait for it)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):  # nothing to wait for before the first use of each buffer
        ev_done[b].record(stream)
        ev_read[b].record(back)

    def e2e_step(i):
        b = i & 1
        d = dev_in[b]
        copy.wait_event(ev_done[b])              # step i-2's kernels are done with these inputs
        with torch.cuda.stream(copy):
            for n, v in host_in.items():
                d[n].copy_(v, non_blocking=True)
        ev_in[b].record(copy)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_read[b])            # step i-2's results were read back
        smla.smla_decode(lay, prm, pool, 0, d["new_latent"], d["new_rope"], d["new_idx_k"], d["new_idx_s"],
                         d["slot_mapping"], d["q"], d["q_pe"], d["q_idx"], d["w"], d["block_table"],
                         d["seq_lens"], d["query_start_loc"], wl.max_q, wl.max_ctx, dev_out[b], dev_lse[b], ws,
                         topk_idx_out=topk, stream=stream)
        ev_done[b].record(stream)
        back.wait_event(ev_done[b])
        with torch.cuda.stream(back):
            host_out[b].copy_(dev_out[b], non_blocking=True)
            host_lse[b].copy_(dev_lse[b], non_blocking=True)
        ev_read[b].record(back)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0.record(copy)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(back)                              # after the last step's results are read back
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = whole_job_rate(T, world, args.steps, ms_e2e)

    if rank != 0:
        dist.destroy_process_group()
        return

    # launches of one fused step, counted by the profiler after all timing is done (the split paths
    # for small batches add a merge launch to the attention and a second pass to the top-k)
    launches_per_step, launches_how = plausible_launches(count_step_launches(step), n_groups)

    # ---------------- roofline of the dominant kernel ----------------
    acct = accounting(wl, topk.cpu().numpy())
    pk = peaks()
    tt = traffic_table()
    dominant = max((k for k in kern_ms if kern_ms[k] is not None), key=lambda k: kern_ms[k], default=None)
    roof = None
    kernels = {}
    for k, msk in kern_ms.items():
        if msk is None:
            continue
        a = acct[k]
        gbs = a["bytes"] / (msk / 1e3) / 1e9
        fl = a["flops"] / (msk / 1e3) / 1e12 if a["flops"] else 0.0
        kernels[k] = {"ms": round(msk, 4), "alg_bytes": a["bytes"], "alg_gbs": round(gbs, 1),
                      "hbm_frac": round(gbs / pk["hbm"], 3)}
        if a["flops"]:
            fpk = pk["bf16"] * (2.0 if a["flop_dtype"] == "fp8" else 1.0)
            kernels[k].update({"tflops": round(fl, 1), "tensor_frac": round(fl / fpk, 3),
                               "tensor_peak": f"{fpk:.0f} ({'2x ' if a['flop_dtype'] == 'fp8' else ''}bf16 of {pk['src']})"})
    if dominant is not None:
        a = acct[dominant]
        msk = kern_ms[dominant]
        t_hbm = a["bytes"] / (pk["hbm"] * 1e9)
        fpk = pk["bf16"] * (2.0 if a["flop_dtype"] == "fp8" else 1.0) if a["flops"] else None
        t_ten = a["flops"] / (fpk * 1e12) if fpk else 0.0
        wname = wl.name
        tr = tt.get((dominant, wname))
        # the recorded bytes are for the full-size workload of that name and the kernel source hashed
        traffic = tr[1] if tr is not None and tr[0] == source_sha(dominant) and args.scale == 1.0 else None
        if t_ten > t_hbm:
            ach = a["flops"] / (msk / 1e3) / 1e12
            roof = {"kernel": dominant, "bound": "tensor", "achieved": round(ach, 1), "peak": round(fpk, 1),
                    "unit": "TFLOP/s", "frac": round(ach / fpk, 4), "traffic": traffic,
                    "peak_source": f"{'2 x ' if a['flop_dtype'] == 'fp8' else ''}bf16 burst of {pk['src']} (fp8:bf16 nominal 2:1)"}
        else:
            ach = a["bytes"] / (msk / 1e3) / 1e9
            roof = {"kernel": dominant, "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm"], "unit": "GB/s",
                    "frac": round(ach / pk["hbm"], 4), "traffic": traffic, "peak_source": f"hbm copy of {pk['src']}"}
        roof["alg_bytes_per_launch"] = a["bytes"]
        roof["alg_flops_per_launch"] = a["flops"]

    step_b = acct["_step"]["bytes"]
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, budget_s=args.cpu_seconds, key_format=args.key_format)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8e4m3+bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "query_tokens": T, "max_q_per_seq": wl.max_q,
                   "mean_ctx": round(float(wl.seq_lens.float().mean()), 1), "max_ctx": wl.max_ctx,
                   "top_k": d.top_k, "heads": d.n_heads, "idx_heads": d.n_idx_heads, "block_size": d.block_size,
                   "pool_gb": round(lay.pool_bytes / 1e9, 3), "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {step_b / 1e6:.0f} MB unique per step > 129 MB",
                   "query_groups_per_step": n_groups, "context_scale": args.scale},
        "hbm_gbs": round(step_b / (ms_step / 1e3) / 1e9, 1),
        "hbm_frac": round(step_b / (ms_step / 1e3) / 1e9 / pk["hbm"], 4),
        "step_bytes": {"unique": step_b, "logical": acct["_step"]["logical_bytes"]},
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_how": f"{launches_per_step} per step ({launches_how}) x {args.steps} steps",
        "kernels": kernels,
        "roofline": roof,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- oracle (CPU) arm
class OracleSampler:
    """The CPU oracle on the query tokens of a workload.

    The workload is generated once, and each sampled sequence's cached context is written into its
    own oracle pool once, on first use (set-up, outside the timed region).  `run` then times the
    oracle's step over sequences taken in a fixed random order, cycling over the first `max_seqs`
    of them, until `budget_s` seconds of oracle work are done.  A sequence's query tokens go in
    slices of at most `max_rows` (all of a decode step's tokens; consecutive rows of a prefill
    chunk): the first slice of a pass over the sequence also stores its new tokens, and every slice
    runs the indexer, top-k and attention of its rows.
    """

    max_rows = 4

    def __init__(self, workload: int, max_seqs: int, key_format: str = "e4m3"):
        from paged_sparse_mla_gb300.workloads import make_config
        import oracle
        self.oracle = oracle
        self.wl = wl = make_config(workload, device="cpu", key_format=key_format)
        d = wl.dims
        self.lay = oracle.PoolLayout(d.block_size, d.n_layers, d.d_latent, d.d_rope, d.quant_tile, d.d_index,
                                     wl.num_blocks, d.key_format)
        self.order = [int(b) for b in np.random.default_rng(7).permutation(wl.batch)[:max_seqs]]
        self.qsl = self._npy(wl.query_start_loc)
        self.next = 0
        self.row_cursor = {}
        self.pools = {}
        self.args = dict(latent_new=self._bits(wl.new_latent), rope_new=self._bits(wl.new_rope),
                         idxk_new=self._npy(wl.new_idx_k), idxs_new=self._npy(wl.new_idx_s), q=self._bits(wl.q),
                         q_pe=self._bits(wl.q_pe), q_idx=self._npy(wl.q_idx), w=self._npy(wl.w),
                         block_table=self._npy(wl.block_table), seq_lens=self._npy(wl.seq_lens),
                         query_start_loc=self.qsl, top_k=d.top_k, sigma=d.softmax_scale)

    @staticmethod
    def _npy(t):
        return t.detach().cpu().numpy()

    @staticmethod
    def _bits(t):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    def _pool(self, b):
        """Oracle pool holding sequence b's cached context, and the slot mapping of its new tokens."""
        if b not in self.pools:
            wl, d, o = self.wl, self.wl.dims, self.oracle
            n_cached = int(wl.seq_lens[b]) - int(self.qsl[b + 1] - self.qsl[b])
            slots = o.context_slots(self._npy(wl.block_table)[b], n_cached, d.block_size)
            pool = np.zeros(self.lay.pool_bytes, dtype=np.uint8)
            for c0 in range(0, slots.size, 1 << 17):
                sc = torch.as_tensor(slots[c0:c0 + (1 << 17)])
                o.kvpack_store(self.lay, pool, 0, self._bits(wl.slot_latent[sc]), self._bits(wl.slot_rope[sc]),
                               self._npy(wl.slot_idx_k[sc]), self._npy(wl.slot_idx_s[sc]), sc.numpy())
            sm = self._npy(wl.slot_mapping).copy()
            keep = np.zeros(sm.shape, bool)
            keep[int(self.qsl[b]):int(self.qsl[b + 1])] = True
            sm[~keep] = -1                           # store this sequence's new tokens only
            self.pools[b] = (pool, sm)
        return self.pools[b]

    def run(self, budget_s: float):
        """(query tokens, seconds of oracle work, sequences) of one sample of about budget_s seconds."""
        done_tokens, spent, seqs = 0, 0.0, []
        while spent < budget_s:
            b = self.order[self.next % len(self.order)]
            pool, sm = self._pool(b)
            q0, q1 = int(self.qsl[b]), int(self.qsl[b + 1])
            r0 = self.row_cursor.get(b, 0)
            rows = list(range(q0 + r0, min(q1, q0 + r0 + self.max_rows)))
            store = sm if r0 == 0 else np.full_like(sm, -1)
            t0 = time.perf_counter()
            self.oracle.decode_step(self.lay, pool, 0, slot_mapping=store, rows=rows, **self.args)
            spent += time.perf_counter() - t0
            done_tokens += len(rows)
            if r0 + len(rows) >= q1 - q0:           # the sequence is done: the next one, from its start
                self.row_cursor[b] = 0
                self.next += 1
                seqs.append(b)
            else:
                self.row_cursor[b] = r0 + len(rows)
        return done_tokens, spent, seqs


def cpu_baseline(workload: int, budget_s: float, key_format: str = "e4m3"):
    sampler = OracleSampler(workload, max_seqs=64, key_format=key_format)
    n, spent, seqs = sampler.run(budget_s)
    cores = len(os.sched_getaffinity(0))
    return {"value": round(n / spent, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} query tokens of {sampler.wl.name} ({len(seqs)} sequences completed; query tokens in slices "
                      f"of at most {sampler.max_rows}), full store+indexer+top-k+attention per query token in numpy "
                      f"float64 ({spent:.1f} s); numpy BLAS may use all {cores} cores"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    # about two minutes of oracle work in all, split evenly over the warm-up and timed steps
    per_step = max(1.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    sampler = OracleSampler(args.workload, max_seqs=8, key_format=args.key_format)
    tok, spent_total, seqs_all = 0, 0.0, []
    for i in range(args.warmup + args.steps):
        n, spent, seqs = sampler.run(per_step)
        if i >= args.warmup:
            tok += n
            spent_total += spent
            seqs_all += seqs
    value = tok / spent_total
    cores = len(os.sched_getaffinity(0))
    name = sampler.wl.name
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "impl": "reference", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * spent_total / args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "sample_per_step_s": round(per_step, 2)},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"per step: query tokens of {name} in slices of at most {sampler.max_rows} "
                                   f"(cycling over {len(sampler.order)} sequences) until {per_step:.1f} s of "
                                   f"oracle work; {tok} query tokens in {spent_total:.1f} s"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ----------------------------------------------------------------------------- split-context (DCP) arm
def run_dcp(args):
    """--dcp N: the decode step split over N round-robin token shards on one GPU.

    A step = per shard (indexer scores, top-k) -> smla_dcp_topk_merge -> per shard
    attention -> smla_lse_merge, over every query token of a decode workload
    (one query token per sequence).  Prints one JSON line with tokens/s, the
    per-phase device times, the unsharded fused step on the same inputs for
    context, and the merge kernel's roofline.
    """
    import paged_sparse_mla_gb300 as smla
    from paged_sparse_mla_gb300 import build_lib
    from paged_sparse_mla_gb300.workloads import make_config, shard_pools

    torch.cuda.set_device(0)
    build_lib.build()
    smla.lib()
    n_sh = args.dcp
    wl = make_config(args.workload, device="cuda", scale=args.scale, key_format=args.key_format)
    if wl.max_q != 1:
        raise SystemExit("--dcp needs a decode workload with one query token per sequence (workloads 2 and 4)")
    d = wl.dims
    lay = smla.layout_init(d.block_size, d.n_layers, d.d_latent, d.d_rope, d.quant_tile, d.d_index, wl.num_blocks,
                           d.key_format)
    prm = smla.make_params(d.n_heads, d.n_idx_heads, d.top_k, d.softmax_scale)
    pool = torch.zeros(lay.pool_bytes, dtype=torch.uint8, device="cuda")
    s = wl.cached_slots
    for c0 in range(0, s.numel(), 1 << 20):
        sl = s[c0:c0 + (1 << 20)].contiguous()
        smla.kvpack_store(lay, pool, 0, wl.slot_latent[sl].contiguous(), wl.slot_rope[sl].contiguous(),
                          wl.slot_idx_k[sl].contiguous(), wl.slot_idx_s[sl].contiguous(), sl)
    smla.kvpack_store(lay, pool, 0, wl.new_latent, wl.new_rope, wl.new_idx_k, wl.new_idx_s, wl.slot_mapping)
    wl.slot_latent = wl.slot_rope = wl.slot_idx_k = wl.slot_idx_s = None
    shards = shard_pools(wl, lay, pool, n_sh, seed=17)
    torch.cuda.empty_cache()
    T, k = wl.n_tokens, d.top_k
    stride = max((x["max_ctx"] + 3) // 4 * 4 for x in shards)
    scores = torch.empty((n_sh, T, stride), dtype=torch.float32, device="cuda")
    topk = torch.empty((n_sh, T, k), dtype=torch.int32, device="cuda")
    sel = torch.empty((n_sh, T, k), dtype=torch.int32, device="cuda")
    parts = torch.empty((n_sh, T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    parts_lse = torch.empty((n_sh, T, d.n_heads), dtype=torch.float32, device="cuda")
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def phase_local():
        for r, x in enumerate(shards):
            smla.smla_index_scores(x["layout"], prm, x["pool"], 0, wl.q_idx, wl.w, x["block_table"], x["seq_lens"],
                                   wl.query_start_loc, 1, x["max_ctx"], scores[r], stream=stream)
            smla.smla_topk(prm, scores[r], x["seq_lens"], wl.query_start_loc, topk[r], stream=stream)

    def phase_merge():
        smla.smla_dcp_topk_merge(scores, topk, sel, stream=stream)

    def phase_attend():
        for r, x in enumerate(shards):
            smla.smla_attend(x["layout"], prm, x["pool"], 0, wl.q, wl.q_pe, sel[r], x["block_table"],
                             wl.query_start_loc, parts[r], parts_lse[r], stream=stream)

    def phase_lse():
        smla.smla_lse_merge(parts, parts_lse, out, lse, stream=stream)

    phases = [("local index+topk", phase_local), ("topk merge", phase_merge), ("attention", phase_attend),
              ("lse merge", phase_lse)]
    for _ in range(args.warmup):
        for _, f in phases:
            f()
    torch.cuda.synchronize()
    if smla.smla_get_last_error() != 0:
        raise RuntimeError("device error during warm-up")
    clocks = ClockSampler(0, args.clocks_csv)
    time.sleep(0.3)
    torch.cuda._sleep(4_000_000)
    marks = [[ev() for _ in range(len(phases) + 1)] for _ in range(args.steps)]
    clocks.start_window()
    for st in range(args.steps):
        marks[st][0].record(stream)
        for i, (_, f) in enumerate(phases):
            f()
            marks[st][i + 1].record(stream)
    torch.cuda.synchronize()
    clocks.end_window()
    clk = clocks.stop()
    if smla.smla_get_last_error() != 0:
        raise RuntimeError("device error in the timed region")
    ms_total = sum(marks[st][0].elapsed_time(marks[st][-1]) for st in range(args.steps))
    ph_ms = {name: statistics.median(marks[st][i].elapsed_time(marks[st][i + 1]) for st in range(args.steps))
             for i, (name, _) in enumerate(phases)}
    value = whole_job_rate(T, 1, args.steps, ms_total)
    # the unsharded fused step on the same inputs (context)
    ws = torch.empty(smla.workspace_size(lay, prm, T, wl.max_ctx), dtype=torch.uint8, device="cuda")
    o2 = torch.empty_like(out)
    l2 = torch.empty_like(lse)
    for _ in range(2):
        smla.smla_decode(lay, prm, pool, 0, None, None, None, None, None, wl.q, wl.q_pe, wl.q_idx, wl.w,
                         wl.block_table, wl.seq_lens, wl.query_start_loc, 1, wl.max_ctx, o2, l2, ws, stream=stream)
    a, b = ev(), ev()
    a.record(stream)
    for _ in range(args.steps):
        smla.smla_decode(lay, prm, pool, 0, None, None, None, None, None, wl.q, wl.q_pe, wl.q_idx, wl.w,
                         wl.block_table, wl.seq_lens, wl.query_start_loc, 1, wl.max_ctx, o2, l2, ws, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    ms_whole = a.elapsed_time(b) / args.steps
    pk = peaks()
    lse_bytes = n_sh * T * d.n_heads * (2 * d.d_latent + 4) + T * d.n_heads * (2 * d.d_latent + 4)
    ach = lse_bytes / (ph_ms["lse merge"] / 1e3) / 1e9
    line = {
        "metric": f"split-context sparse-MLA decode tokens/s, {n_sh} round-robin token shards on one GPU",
        "value": round(value, 1), "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_total / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8e4m3+bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": wl.name, "shards": n_sh, "batch": int(wl.seq_lens.numel()), "query_tokens": T,
                   "max_ctx": int(wl.max_ctx), "top_k": k, "l2": "inputs larger than L2"},
        "phases_ms": {k2: round(v, 4) for k2, v in ph_ms.items()},
        "unsharded_fused_ms": round(ms_whole, 4),
        "roofline": {"kernel": "smla_lse_merge", "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm"],
                     "unit": "GB/s", "frac": round(ach / pk["hbm"], 4), "traffic": None,
                     "alg_bytes_per_launch": lse_bytes},
        "clocks": clk,
    }
    print(json.dumps(line))


# ----------------------------------------------------------------------------- host-tier (HiSparse) arm
def run_hisparse(args):
    """--host-frac f: attention with the records of a fraction f of the blocks in pinned host memory.

    The step's selection comes from one fused call; then smla_attend (every record in HBM) and
    smla_attend_hisparse (records of the evicted blocks read from host memory over the CPU-GPU
    link) are timed on the same selection.  Prints one JSON line.
    """
    import paged_sparse_mla_gb300 as smla
    from paged_sparse_mla_gb300 import build_lib
    from paged_sparse_mla_gb300.workloads import make_config, evict_records

    torch.cuda.set_device(0)
    build_lib.build()
    smla.lib()
    wl = make_config(args.workload, device="cuda", scale=args.scale, key_format=args.key_format)
    d = wl.dims
    lay = smla.layout_init(d.block_size, d.n_layers, d.d_latent, d.d_rope, d.quant_tile, d.d_index, wl.num_blocks,
                           d.key_format)
    prm = smla.make_params(d.n_heads, d.n_idx_heads, d.top_k, d.softmax_scale)
    pool = torch.zeros(lay.pool_bytes, dtype=torch.uint8, device="cuda")
    s = wl.cached_slots
    for c0 in range(0, s.numel(), 1 << 20):
        sl = s[c0:c0 + (1 << 20)].contiguous()
        smla.kvpack_store(lay, pool, 0, wl.slot_latent[sl].contiguous(), wl.slot_rope[sl].contiguous(),
                          wl.slot_idx_k[sl].contiguous(), wl.slot_idx_s[sl].contiguous(), sl)
    wl.slot_latent = wl.slot_rope = wl.slot_idx_k = wl.slot_idx_s = None
    T = wl.n_tokens
    ws = torch.empty(smla.workspace_size(lay, prm, T, wl.max_ctx), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    topk = torch.empty((T, d.top_k), dtype=torch.int32, device="cuda")
    smla.smla_decode(lay, prm, pool, 0, wl.new_latent, wl.new_rope, wl.new_idx_k, wl.new_idx_s, wl.slot_mapping,
                     wl.q, wl.q_pe, wl.q_idx, wl.w, wl.block_table, wl.seq_lens, wl.query_start_loc, wl.max_q,
                     wl.max_ctx, out, lse, ws, topk_idx_out=topk)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(2_000_000)
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps

    ms_hbm = timed(lambda: smla.smla_attend(lay, prm, pool, 0, wl.q, wl.q_pe, topk, wl.block_table,
                                            wl.query_start_loc, out, lse, stream=stream))
    bt = wl.block_table.cpu().numpy()
    used = np.unique(bt[bt >= 0])
    rng = np.random.default_rng(29)
    moved = used[rng.random(used.size) < args.host_frac]
    host, hmap = evict_records(lay, pool, moved)
    clocks = ClockSampler(0, args.clocks_csv)
    time.sleep(0.3)
    clocks.start_window()
    ms_tier = timed(lambda: smla.smla_attend_hisparse(lay, prm, pool, 0, host, hmap, wl.q, wl.q_pe, topk,
                                                      wl.block_table, wl.query_start_loc, out, lse, stream=stream))
    clocks.end_window()
    clk = clocks.stop()
    if smla.smla_get_last_error() != 0:
        raise RuntimeError("device error in the timed region")
    # records read from the host tier per step: selected positions whose block was evicted
    tk = topk.cpu().numpy()
    qsl = wl.query_start_loc.cpu().numpy()
    seq = np.searchsorted(qsl, np.arange(T), side="right") - 1
    blk = np.where(tk >= 0, bt[seq[:, None], np.maximum(tk, 0) // d.block_size], -1)
    in_host = np.isin(blk, moved) & (tk >= 0)
    host_bytes = int(in_host.sum()) * lay.rec_stride
    line = {
        "metric": "sparse-MLA attention tokens/s with part of the KV records in host memory (host-tier gather)",
        "value": round(T / (ms_tier / 1e3), 1), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_tier, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8e4m3+bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": wl.name, "host_fraction_of_blocks": args.host_frac, "blocks_moved": int(moved.size),
                   "host_bytes_pinned": int(host.numel()), "query_tokens": T, "top_k": d.top_k},
        "attend_all_hbm_ms": round(ms_hbm, 4),
        "records_from_host_per_step": int(in_host.sum()), "host_bytes_per_step": host_bytes,
        "host_read_gbs_if_overlapped": round(host_bytes / (ms_tier / 1e3) / 1e9, 1),
        "clocks": clk,
    }
    print(json.dumps(line))


def run_topk_rows(args):
    """--topk-rows: smla_topk alone on score rows of the workload's query tokens (their visible lengths),
    drawn two ways: i.i.d. integer scores (the sampled threshold works: one streaming pass) and the same
    rows with the highest scores clustered on the most recent 6,000 positions (as recent turns would be),
    which overflows one warp's candidate list and takes the exact radix-select fallback over the whole
    row.  Prints one JSON line with both times."""
    import paged_sparse_mla_gb300 as smla
    from paged_sparse_mla_gb300 import build_lib
    from paged_sparse_mla_gb300.workloads import make_config

    torch.cuda.set_device(0)
    build_lib.build()
    smla.lib()
    wl = make_config(args.workload, device="cuda", scale=args.scale)
    d = wl.dims
    qsl = wl.query_start_loc.cpu().numpy()
    lens = wl.seq_lens.cpu().numpy()
    wl.slot_latent = wl.slot_rope = wl.slot_idx_k = wl.slot_idx_s = None
    T = int(qsl[-1])
    seq = np.searchsorted(qsl, np.arange(T), side="right") - 1
    n_vis = lens[seq] - (qsl[seq + 1] - qsl[seq]) + (np.arange(T) - qsl[seq]) + 1
    stride = (int(n_vis.max()) + 3) // 4 * 4
    gen = torch.Generator(device="cuda").manual_seed(77)
    base = (torch.randint(-60, 61, (T, stride), generator=gen, device="cuda").float() * 0.25)
    clustered = base.clone()
    cols = torch.arange(stride, device="cuda")[None, :]
    nv = torch.as_tensor(n_vis, device="cuda")[:, None]
    hot = (cols >= nv - 6000) & (cols < nv)
    clustered[hot] = 100.0 + torch.randint(0, 40, (int(hot.sum()),), generator=gen, device="cuda").float()
    prm = smla.make_params(d.n_heads, d.n_idx_heads, d.top_k, d.softmax_scale)
    sl = wl.seq_lens
    qs = wl.query_start_loc
    out = torch.empty((T, d.top_k), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def timed(scores):
        fn = lambda: smla.smla_topk(prm, scores, sl, qs, out, stream=stream)
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps

    clocks = ClockSampler(0, args.clocks_csv)
    time.sleep(0.3)
    clocks.start_window()
    ms_fast = timed(base)
    ms_slow = timed(clustered)
    clocks.end_window()
    clk = clocks.stop()
    if smla.smla_get_last_error() != 0:
        raise RuntimeError("device error in the timed region")
    line = {
        "metric": "top-k select time per launch: i.i.d. scores vs scores clustered on recent positions",
        "value": round(ms_slow, 4), "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_slow, 4), "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32 scores, int32 positions", "data": "synthetic",
        "config": {"workload": wl.name, "rows": T, "top_k": d.top_k, "mean_visible": round(float(n_vis.mean()), 1),
                   "max_visible": int(n_vis.max()), "cluster": "highest scores on the last 6,000 visible positions"},
        "iid_rows_ms": round(ms_fast, 4), "clustered_rows_ms": round(ms_slow, 4),
        "score_bytes_per_launch": int(n_vis.sum()) * 4,
        "clocks": clk,
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="smla", choices=["smla", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="where to keep the raw nvidia-smi clock samples (default: a file in the temp directory)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--host-frac", type=float, default=0.0,
                    help="host-tier arm: fraction of the blocks whose records live in pinned host memory")
    ap.add_argument("--dcp", type=int, default=0,
                    help="split-context arm: N round-robin token shards on one GPU (decode workloads 2 and 4)")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="shrink context lengths (profiler captures of a smaller case; not a bench line)")
    ap.add_argument("--fp4-keys", dest="key_format", action="store_const", const="e2m1", default="e4m3",
                    help="cache the indexer keys as packed FP4 E2M1 codes (workloads 2-5)")
    ap.add_argument("--topk-rows", action="store_true",
                    help="top-k arm: smla_topk alone on i.i.d. and on clustered score rows of the workload's shape")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.dcp > 0:
        run_dcp(args)
    elif args.host_frac > 0:
        run_hisparse(args)
    elif args.topk_rows:
        run_topk_rows(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
