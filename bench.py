"""Benchmark of the Engram hot path (hash -> gather/dequant -> wkv projection -> gate).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step is one pass of the whole path over one batch of the workload (default: the large
configuration, 16384 tokens of uniform ids over an FP8+E8M0 table of 201M rows (53 GB),
24 hash columns of 256, hidden 7168, hc 4).  Inputs are resident in HBM; the L2 is flushed
(512 MB write, then a 256 MB read) before every timed step; each step is timed with CUDA events
on the launching stream, per kernel as well.  Under torchrun every rank runs its own replica (the
path needs no exchange): weak scaling, max time over ranks.

--impl reference times the CPU oracle (oracle/) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from engram_synth import get_workload  # noqa: E402
from engram_synth.case import make_case, to_device  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_HBM_GBS = 7900.0          # HBM3e nominal; HBM fractions are also given against it
DEFAULT_WORKLOAD = "large_fp8_t16384"
L2_FLUSH_BYTES = 512 << 20
L2_FLUSH_READ_BYTES = 256 << 20

# DRAM bytes per launch of the dominant kernel from an ncu capture, keyed by kernel and
# workload, with the sha256 of the kernel's source at capture time (stale -> traffic null).
NCU_TRAFFIC: dict = {
    "project0@large_fp8_t16384": {"bytes": 4938854656 + 2314286592, "src_sha": "00fef9d6c5ea4026"},
    "project0@decode_fp8_t256": {"bytes": 254897920 + 3391232, "src_sha": "00fef9d6c5ea4026"},
    "project0@decode_fp8_t256@mxfp8": {"bytes": 131441664 + 3283200, "src_sha": "eb50e0f2c991739b",
                                       "src": "gemm_mx.cu"},
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(x: float, device) -> float:
    """The largest of a per-rank number over all ranks: the job takes as long as its slowest
    replica.  Identity outside torch.distributed."""
    if not torch.distributed.is_available() or not torch.distributed.is_initialized():
        return float(x)
    if torch.distributed.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, units_per_rank: int, ms: float) -> float:
    """Whole-job units/s when each of `world` replicas processes `units_per_rank` units and the
    slowest takes `ms` milliseconds."""
    return world * units_per_rank / (ms / 1e3)


def src_sha(name: str) -> str:
    with open(os.path.join(ROOT, "engram_gram_hash_02_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for r in csv.reader(io.StringIO(out)):
            if len(r) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(r[2]), float(r[3]), [x.strip() for x in r[6:10]], r[5].strip()))
            except Exception:
                continue
        inside = [x for x in rows if self.t0 - 1 <= x[0] <= self.t1 + 1] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for x in inside for i, v in enumerate(x[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([x[1] for x in inside])), "sm_max_mhz": max(x[2] for x in inside),
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------------------------------------------
# the CUDA path
# ------------------------------------------------------------------------------------------------

class Path:
    """Device-resident workload plus pre-marshalled C-ABI calls for each stage."""

    def __init__(self, w, device, table_rows=None, wkv="bf16", light=False):
        """light: only what the hash and the gather read and write (profiling one of them)."""
        import ctypes as C

        import engram_gram_hash_02_gb300 as E
        from engram_gram_hash_02_gb300 import binding as B
        self.E, self.C, self.B = E, C, B
        self.w, self.device = w, device
        if table_rows:
            # profiling only: primes near table_rows / cols, so the table holds about table_rows
            # rows and every hashed id stays inside it
            from dataclasses import replace
            w = replace(w, vocab_size=max(1024, int(table_rows) // w.cols))
            self.w = w
        primes, offsets, rows, mult = self._layout(E, w)
        self.light = light
        self.case = case = make_case(w, rows, device, with_weights=not light)
        b = case.batch
        self.pad = int(b["token_map"][w.pad_token_id])
        self.dims = E.make_dims(w.layers, w.max_ngram, w.n_heads, w.head_dim, w.hidden, w.hc, w.raw_vocab,
                                w.compressed_vocab, self.pad, w.eps, w.clamp)
        d = device
        self.input_ids = to_device(b["input_ids"], d)
        self.cu = to_device(b["cu_seqlens"], d)
        self.sid = to_device(b["sequence_ids"], d)
        self.mask = to_device(b["token_mask"], d)
        self.lookback = to_device(b["lookback_ids"], d)
        self.tables = E.HashTables(to_device(b["token_map"], d), to_device(mult, d), to_device(primes, d),
                                   to_device(offsets, d))
        self.mx = wkv == "mxfp8"
        if self.mx and any(t["fmt"] != "fp8" for t in case.tables):
            raise SystemExit("--wkv mxfp8 needs an FP8+E8M0 table (its rows are the projection's A operand)")
        self.layers = []
        for l, t in enumerate(case.tables):
            if light:
                self.layers.append(E.LayerWeights(t["fmt"], t["table"], t["scales"], t["num_rows"], None, None,
                                                  None))
                continue
            wkv_l, wsc = case.wkv[l], None
            if self.mx:                   # weight preparation, once, outside every timed region
                wkv_l, wsc = E.quantize_mxfp8(case.wkv[l])
            self.layers.append(E.LayerWeights(t["fmt"], t["table"], t["scales"], t["num_rows"], wkv_l,
                                              case.q_weight[l], case.k_weight[l], wkv_scales=wsc))
        self.streams = [s.clone() for s in case.streams]
        T, L, Cc, K, N = w.tokens, w.layers, w.cols, w.K, w.N
        self.ids = torch.empty((T, L, Cc), dtype=torch.int32, device=d)
        self.A = torch.empty((T, K), dtype=torch.bfloat16, device=d)
        if self.mx:                       # FP8 variant: codes [T, K] and scales [T, K/32] of the rows
            self.A_codes = torch.empty((T, K), dtype=torch.uint8, device=d)
            self.A_scales = torch.empty(E.mx_scale_shape(T, K), dtype=torch.uint8, device=d)
        self.kv = None if light else torch.empty((T, N), dtype=torch.float32, device=d)
        self.err = torch.zeros(1, dtype=torch.int32, device=d)
        self.gemm_ws = torch.empty(256 if light else max(256, E.project_workspace_bytes(T, K, N)),
                                   dtype=torch.uint8, device=d)
        self.table_rows = rows

    @staticmethod
    def _layout(E, w):
        primes, offsets, rows = E.engram_layout(w.vocab_size, w.layers, w.max_ngram, w.n_heads)
        mult = E.hash_multipliers(w.layer_ids, w.max_ngram, w.compressed_vocab)
        return primes, offsets, rows, mult

    def stage_calls(self, stream):
        """One closure per kernel launch of a step, in order, with arguments marshalled once."""
        lib, B, w, C = self.E.lib(), self.B, self.w, self.C
        p = B._ptr
        s = stream.cuda_stream
        T, L, Cc, K, N = w.tokens, w.layers, w.cols, w.K, w.N
        dims = self.dims
        S = self.cu.numel() - 1
        hash_args = (C.byref(dims), p(self.input_ids), T, p(self.cu), S, p(self.sid), p(self.mask),
                     p(self.lookback), p(self.tables.token_map), p(self.tables.multipliers),
                     p(self.tables.primes), p(self.tables.offsets), p(self.ids), p(self.err), s)
        calls = [("hash", lambda: lib.engram_hash(*hash_args))]
        for l, lw in enumerate(self.layers):
            if self.light:                # the hash and the gathers only
                if self.mx:
                    gc_args = (self.ids.data_ptr() + 4 * l * Cc, L * Cc, T, Cc, w.head_dim, p(lw.table),
                               p(lw.scales), int(lw.num_rows), p(self.A_codes), p(self.A_scales), p(self.err), s)
                    calls.append((f"gather{l}", lambda a=gc_args: lib.engram_gather_fp8_codes(*a)))
                else:
                    g_args = (B.TABLE_FORMATS[lw.fmt], self.ids.data_ptr() + 4 * l * Cc, L * Cc, T, Cc, w.head_dim,
                              p(lw.table), p(lw.scales), int(lw.num_rows), p(self.A), p(self.err), s)
                    calls.append((f"gather{l}", lambda a=g_args: lib.engram_gather_dequant(*a)))
                continue
            g_args = (B.TABLE_FORMATS[lw.fmt], self.ids.data_ptr() + 4 * l * Cc, L * Cc, T, Cc, w.head_dim,
                      p(lw.table), p(lw.scales), int(lw.num_rows), p(self.A), p(self.err), s)
            pr_args = (p(self.A), p(lw.wkv), p(self.kv), T, K, N, p(self.gemm_ws), self.gemm_ws.numel(), p(self.err), s)
            ga_args = (C.byref(dims), p(self.streams[l]), p(self.kv), p(lw.q_weight), p(lw.k_weight),
                       p(self.mask), T, p(self.err), s)
            if self.mx:
                gc_args = (self.ids.data_ptr() + 4 * l * Cc, L * Cc, T, Cc, w.head_dim, p(lw.table), p(lw.scales),
                           int(lw.num_rows), p(self.A_codes), p(self.A_scales), p(self.err), s)
                pm_args = (p(self.A_codes), p(self.A_scales), p(lw.wkv), p(lw.wkv_scales), p(self.kv), T, K, N,
                           p(self.err), s)
                calls.append((f"gather{l}", lambda a=gc_args: lib.engram_gather_fp8_codes(*a)))
                calls.append((f"project{l}", lambda a=pm_args: lib.engram_project_mxfp8(*a)))
            else:
                calls.append((f"gather{l}", lambda a=g_args: lib.engram_gather_dequant(*a)))
                calls.append((f"project{l}", lambda a=pr_args: lib.engram_project(*a)))
            calls.append((f"gate{l}", lambda a=ga_args: lib.engram_gate(*a)))
        return calls


# MXFP8 dense tensor peak, measured on this part (MEASURED_PEAKS.json holds no FP8 figure): cuBLAS
# through torch._scaled_mm, e4m3 x e4m3 with one E8M0 scale per 32 values, 8192^3, best of 10
# (burst) and back to back for 4 s (sustained). The nominal fp8 / bf16 ratio (4.5 / 2.25) times the
# measured bf16 peak would be 3847 TFLOP/s.
MXFP8_PEAK_TFLOPS = {"burst": 3282.7, "sustained": 3278.7}


def tensor_peak(peaks_d, mx: bool, kind: str = "burst") -> float:
    if mx:
        return MXFP8_PEAK_TFLOPS[kind]
    return peaks_d["bf16_tflops"] if kind == "burst" else peaks_d["bf16_tflops_sustained"]


def stage_model(w, name, peaks_d, mx: bool = False):
    """Algorithmic bytes / flops of one launch of a stage at workload w (``mx``: the FP8 variant,
    MXFP8 codes plus one scale byte per 32 values for both projection operands).

    ``bytes`` is what the method must move with kv in the model's dtype (bf16, 2 bytes per
    element); this library keeps kv in fp32, and the 2 extra bytes per kv element written by the
    projection and read by the gate are ``extra_bytes`` (not counted in ``bytes``)."""
    T, L, Cc, D, K, N, H, hc = w.tokens, w.layers, w.cols, w.head_dim, w.K, w.N, w.hidden, w.hc
    row = {"fp8": D + D // 32, "q2k": 84, "bf16": 2 * D}[w.table_format]
    op = (K + K // 32) if mx else 2 * K              # bytes of one operand row
    if name == "hash":
        return {"bytes": 8 * T + 4 * T * L * Cc, "flops": 0, "bound": "alu", "extra_bytes": 0}
    if name.startswith("gather"):
        return {"bytes": T * Cc * (row + 4) + T * op, "flops": 0, "bound": "hbm", "extra_bytes": 0}
    if name.startswith("project"):
        by = N * op + T * op + 2 * T * N
        fl = 2 * T * N * K
        t_hbm = by / (peaks_d["hbm_gbs"] * 1e9)
        t_tc = fl / (tensor_peak(peaks_d, mx) * 1e12)
        return {"bytes": by, "flops": fl, "bound": "hbm" if t_hbm >= t_tc else "tensor", "extra_bytes": 2 * T * N}
    if name.startswith("gate"):
        return {"bytes": 8 * hc * H * T + 2 * N * T + 4 * hc * H, "flops": 8 * hc * H * T, "bound": "hbm",
                "extra_bytes": 2 * T * N}
    raise ValueError(name)


def forward_launches(w, table_order: bool = False) -> int:
    """Kernels one engram_forward call launches: the hash (which also gathers the rows of up to 8
    leading FP8 layers), one gather launch per 8 remaining layers of the workload's one format,
    then per layer the projection and the gate. Table-order gathers: no rows from the hash, and four
    more launches per layer (clear, count, scan, scatter)."""
    fused = min(w.layers, 8) if w.table_format == "fp8" and not table_order else 0
    return 1 + -(-(w.layers - fused) // 8) + 2 * w.layers + (4 * w.layers if table_order else 0)


def kernel_src(name):
    for pre, src in (("hash", "hash.cu"), ("gather", "gather.cu"), ("project", "gemm.cu"), ("gate", "gate.cu")):
        if name.startswith(pre):
            return src
    return None


def run_ours(args, rank, world, device):
    w = get_workload(args.workload)
    path = Path(w, device, wkv=args.wkv)
    mx = path.mx
    stream = torch.cuda.current_stream()
    calls = path.stage_calls(stream)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    flush_read = torch.ones(L2_FLUSH_READ_BYTES // 4, dtype=torch.float32, device=device)

    def flush_l2(k):
        # write a buffer four times the L2, then read one twice its size: the L2 then holds none of
        # the step's data and no dirty line of the flush, whose write-back would otherwise land
        # inside the timed step
        flush.fill_(float(k))
        flush_read.sum()


    def step(evs=None):
        for i, (name, fn) in enumerate(calls):
            if evs is not None:
                evs[i].record(stream)
            rc = fn()
            if rc != 0:
                raise RuntimeError(f"{name} failed: {path.E.lib().engram_last_error().decode()}")
        if evs is not None:
            evs[len(calls)].record(stream)

    plan = path.E.ForwardPlan(path.dims, path.tables, path.layers, path.input_ids, path.streams,
                              cu_seqlens=path.cu, sequence_ids=path.sid, token_mask=path.mask,
                              lookback_ids=path.lookback, out_ids=path.ids, err=path.err)
    side = torch.cuda.Stream(device) if args.side_stream else None    # engram_forward2
    for _ in range(args.warmup):
        flush_l2(1)
        plan.run(stream, side)
        flush_l2(1)
        step()
    torch.cuda.synchronize()
    if path.err.item() != 0:
        raise RuntimeError(f"device error flag {path.err.item()} during warm-up")

    # timed region 1 (the headline): engram_forward, one C call per step; its kernels are chained
    # with programmatic dependent launch, so no event may sit between them
    fw = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    # timed region 2: the same kernels launched one by one, an event between each, for per-kernel times
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t0")
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush_l2(k)
        fw[k][0].record(stream)
        plan.run(stream, side)
        fw[k][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    for k in range(args.steps):
        flush_l2(k)
        step(ev[k])
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t1")
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    if path.err.item() != 0:
        raise RuntimeError(f"device error flag {path.err.item()} in the timed region")

    per_step = np.array([a.elapsed_time(b) for a, b in fw])                     # ms
    per_step_serial = np.array([e[0].elapsed_time(e[-1]) for e in ev])
    per_kernel = {name: float(np.mean([e[i].elapsed_time(e[i + 1]) for e in ev]))
                  for i, (name, _) in enumerate(calls)}
    ms = max_over_ranks(float(per_step.mean()), device)
    tokens = w.tokens * w.layers
    value = replica_throughput(world, tokens, ms)

    # ---- the FP8 operand variant on the same workload (wkv encoded as MXFP8 once) ------------
    variant = None
    if not mx and not args.no_variant and all(t["fmt"] == "fp8" for t in path.case.tables):
        variant = time_fp8_variant(args, path, stream, flush_l2, device)
        variant["ms"] = max_over_ranks(variant["ms"], device)
        variant["ms_per_step"] = round(variant["ms"], 5)

    # ---- end to end through the public API with host buffers -------------------------------
    e2e = run_e2e(args, path, stream, device) if not args.no_e2e else None
    if e2e is not None:
        e2e["ms"] = max_over_ranks(e2e["ms"], device)

    if rank != 0:
        return None
    pk, pk_kind = peaks()
    dom = max(per_kernel, key=per_kernel.get)
    model = stage_model(w, dom, pk, mx)
    t_s = per_kernel[dom] / 1e3
    if model["bound"] == "tensor":
        achieved, peak, unit = model["flops"] / t_s / 1e12, tensor_peak(pk, mx), "TFLOP/s"
    elif model["bound"] == "hbm":
        achieved, peak, unit = model["bytes"] / t_s / 1e9, pk["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = model["bytes"] / t_s / 1e9, None, "GB/s"
    key = f"{dom}@{w.name}" + ("@mxfp8" if mx else "")
    traffic = None
    rec = NCU_TRAFFIC.get(key)
    if rec and rec.get("src_sha") == src_sha(rec.get("src", kernel_src(dom))):
        traffic = rec["bytes"]
    stages = {}
    for name, t in per_kernel.items():
        m = stage_model(w, name, pk, mx)
        gbs = m["bytes"] / (t / 1e3) / 1e9
        stages[name] = {"us": round(t * 1e3, 2), "GB/s": round(gbs, 1), "bound": m["bound"]}
        if m["extra_bytes"]:
            stages[name]["GB/s_with_fp32_kv"] = round((m["bytes"] + m["extra_bytes"]) / (t / 1e3) / 1e9, 1)
        if m["flops"] and name.startswith("project"):
            tfs = m["flops"] / (t / 1e3) / 1e12
            stages[name]["TFLOP/s"] = round(tfs, 1)
            if m["bound"] == "tensor":
                stages[name]["frac"] = round(tfs / tensor_peak(pk, mx), 4)
        if m["bound"] == "hbm":
            stages[name]["frac"] = round(gbs / pk["hbm_gbs"], 4)
            stages[name]["frac_nominal"] = round(gbs / NOMINAL_HBM_GBS, 4)
    line = {
        "metric": "engram_tokens_per_s_per_layer",
        "value": round(value, 1),
        "unit": "tokens/s per layer",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "ms_per_step_kernels_serialised": round(float(per_step_serial.mean()), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 x e4m3 (MXFP8), fp32 accumulate" if mx else "bf16",
        "data": "synthetic (seeded; tables, weights and ids drawn on device)",
        "config": dict(workload_config(w, int(sum(path.table_rows)), "mxfp8" if mx else "bf16", world),
                       l2="flushed before every timed step (512 MB write, then a 256 MB read)",
                       **({"gate_fusion": args.gate_fusion} if args.gate_fusion else {}),
                       **({"side_stream": True} if args.side_stream else {}),
                       **({"operand_gather": True} if args.operand_gather else {}),
                       **({"gather_order": "table"} if args.gather_order else {}),
                       **({"gemm_tile": args.gemm_tile} if args.gemm_tile else {}),
                       **({"mx_tile": args.mx_tile} if args.mx_tile else {}),
                       **({"gate_form": args.gate_form} if args.gate_form else {})),
        "gpu_launches": args.steps * (forward_launches(w, bool(args.gather_order)) + len(calls)),
        "stages": stages,
        "roofline": roofline_entry(dom, model, achieved, peak, unit, pk, pk_kind, mx, traffic),
        "clocks": clocks,
        "wall_s_timed": round(wall, 4),
    }
    if e2e is not None:
        line["e2e"] = {"value": round(replica_throughput(world, tokens, e2e["ms"]), 1), "unit": "tokens/s per layer",
                       "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                       "ms_per_step": round(e2e["ms"], 5),
                       "pipelining": f"{e2e['slots']} buffer slots; copies in (token inputs packed in one pinned buffer, then the streams) / forward / copies out on 3 streams"}
    if variant is not None:
        line["variants"] = {"mxfp8_wkv": dict(variant, value=round(replica_throughput(world, tokens, variant["ms"]), 1),
                                              unit="tokens/s per layer")}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, path.case, args.cpu_tokens)
    return line


def time_fp8_variant(args, path, stream, flush_l2, device) -> dict:
    """engram_forward with every layer's wkv encoded as MXFP8 (engram_quantize_mxfp8, once, outside
    the timed region) and the FP8 table rows fed to the block-scaled projection: the same steps,
    L2 flush and events as the headline."""
    E = path.E
    layers = []
    for l, lw in enumerate(path.layers):
        codes, scales = E.quantize_mxfp8(path.case.wkv[l])
        layers.append(E.LayerWeights(lw.fmt, lw.table, lw.scales, lw.num_rows, codes, lw.q_weight, lw.k_weight,
                                     wkv_scales=scales))
    plan = E.ForwardPlan(path.dims, path.tables, layers, path.input_ids, path.streams, cu_seqlens=path.cu,
                         sequence_ids=path.sid, token_mask=path.mask, lookback_ids=path.lookback, err=path.err)
    for _ in range(args.warmup):
        flush_l2(1)
        plan.run(stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush_l2(k)
        ev[k][0].record(stream)
        plan.run(stream)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    if path.err.item() != 0:
        raise RuntimeError(f"device error flag {path.err.item()} in the FP8 variant")
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    return {"ms": ms, "ms_per_step": round(ms, 5), "dtype": "e4m3 x e4m3 (MXFP8), fp32 accumulate",
            "note": "wkv encoded once as MXFP8 (E8M0 scale per 32); the FP8 table rows are the projection's A operand"}


def roofline_entry(dom, model, achieved, peak, unit, pk, pk_kind, mx, traffic) -> dict:
    """The JSON line's roofline object for the dominant kernel: achieved against the measured peak
    (burst), plus the sustained tensor peak or the nominal HBM bandwidth for context."""
    r = {"kernel": dom, "bound": model["bound"], "achieved": round(achieved, 1), "peak": peak, "unit": unit,
         "frac": None if peak is None else round(achieved / peak, 4),
         "peak_source": (f"{pk_kind} (hbm_gbs, copy)" if unit == "GB/s" else
                         "measured (cuBLAS MXFP8 8192^3, burst)" if mx else f"{pk_kind} (bf16_tflops, burst)"),
         "algorithmic_bytes": model["bytes"], "algorithmic_flops": model["flops"],
         "extra_bytes_fp32_kv": model["extra_bytes"], "traffic": traffic}
    if unit == "TFLOP/s" and (mx or "bf16_tflops_sustained" in pk):
        sus = tensor_peak(pk, mx, "sustained")
        r["peak_sustained"] = sus
        r["frac_sustained"] = round(achieved / sus, 4)
    if unit == "GB/s":
        r["frac_nominal"] = round(achieved / NOMINAL_HBM_GBS, 4)
    return r


def run_only(args, device):
    """Run one stage alone (for short profiler captures); prints its mean time. ``forward`` runs
    engram_forward as a whole (its own kernels: the hash fused with the FP8 layers' gathers)."""
    w = get_workload(args.workload)
    if args.tokens:
        w = w.with_tokens((args.tokens,))
    path = Path(w, device, args.table_rows, wkv=args.wkv, light=args.only in ("hash", "gather"))
    w = path.w
    stream = torch.cuda.current_stream()
    all_calls = path.stage_calls(stream)
    if args.only == "forward":
        plan = path.E.ForwardPlan(path.dims, path.tables, path.layers, path.input_ids, path.streams,
                                  cu_seqlens=path.cu, sequence_ids=path.sid, token_mask=path.mask,
                                  lookback_ids=path.lookback, out_ids=path.ids, err=path.err)
        all_calls = [("forward", lambda: plan.run(stream) or 0)]
    calls = [(n, f) for n, f in all_calls if n.startswith(args.only)]
    for n, f in all_calls:                      # produce the stage's inputs once
        if n.startswith(args.only):
            break
        f()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        for _, f in calls:
            f()
    a.record(stream)
    for _ in range(args.steps):
        for _, f in calls:
            f()
    b.record(stream)
    b.synchronize()
    err = int(path.err.item())
    print(json.dumps({"profile_stage": args.only, "workload": w.name, "table_rows": args.table_rows,
                      "us_per_launch": round(a.elapsed_time(b) * 1e3 / max(1, args.steps * len(calls)), 2),
                      "err": err}))
    if err:
        raise SystemExit(f"device error flag {err}")


def run_e2e(args, path, stream, device, slots: int = 3):
    """engram_forward with per-step host->device copies of the inputs (pinned) and a
    device->host read of the updated streams, all inside the timed region. Steps are pipelined
    the way a serving loop runs them: `slots` sets of device buffers, copies in on one stream,
    the forward pass on the compute stream, copies out on a third, so step k+1's inputs move while
    step k computes and step k-1's result comes back. Every step copies its own inputs in and its
    own result out."""
    E, w = path.E, path.w
    names = [n for n in ("input_ids", "cu", "sid", "mask", "lookback") if getattr(path, n) is not None]
    # the token inputs travel packed in one pinned buffer (one copy per step instead of one per
    # tensor), each at a 256-byte aligned offset
    offs, size = {}, 0
    for n in names:
        offs[n] = size
        size += (getattr(path, n).numel() * getattr(path, n).element_size() + 255) // 256 * 256
    host_pack = torch.empty(size, dtype=torch.uint8).pin_memory()

    def views(pack, n):
        t = getattr(path, n)
        nb = t.numel() * t.element_size()
        return pack[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)

    for n in names:
        views(host_pack, n).copy_(getattr(path, n).cpu())
    host_in = {n: views(host_pack, n) for n in names}
    host_streams = [s.cpu().pin_memory() for s in path.case.streams]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    buf = []
    for _ in range(slots):
        dev_pack = torch.empty(size, dtype=torch.uint8, device=device)
        dev_in = {n: views(dev_pack, n) for n in names}
        dev_in["_pack"] = dev_pack
        dev_streams = [torch.empty_like(s) for s in path.streams]
        plan = E.ForwardPlan(path.dims, path.tables, path.layers, dev_in["input_ids"], dev_streams,
                             cu_seqlens=dev_in.get("cu"), sequence_ids=dev_in.get("sid"),
                             token_mask=dev_in.get("mask"), lookback_ids=dev_in.get("lookback"), err=path.err)
        out_host = [torch.empty_like(s).pin_memory() for s in host_streams]
        ev = {k: torch.cuda.Event() for k in ("in", "comp", "out")}
        buf.append({"in": dev_in, "streams": dev_streams, "plan": plan, "out": out_host, "ev": ev})
    h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + sum(
        s.numel() * s.element_size() for s in host_streams)           # bytes that carry data
    d2h = sum(s.numel() * s.element_size() for s in host_streams)
    for b in buf:
        b["ev"]["out"].record(s_out)

    def step(k):
        b = buf[k % slots]
        s_in.wait_event(b["ev"]["out"])          # this slot's previous result has been copied out
        with torch.cuda.stream(s_in):
            b["in"]["_pack"].copy_(host_pack, non_blocking=True)
            for l, hs in enumerate(host_streams):
                b["streams"][l].copy_(hs, non_blocking=True)
        b["ev"]["in"].record(s_in)
        stream.wait_event(b["ev"]["in"])
        b["plan"].run(stream)
        b["ev"]["comp"].record(stream)
        s_out.wait_event(b["ev"]["comp"])
        with torch.cuda.stream(s_out):
            for l, o in enumerate(b["out"]):
                o.copy_(b["streams"][l], non_blocking=True)
        b["ev"]["out"].record(s_out)

    for k in range(max(3, args.warmup)):
        step(k)
    torch.cuda.synchronize()
    n = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for k in range(n):
        step(k)
    s_out.wait_stream(s_in)
    s_out.wait_stream(stream)
    t1.record(s_out)
    t1.synchronize()
    # the last step's result equals a plain run's (same inputs every step)
    ref = [s.clone() for s in path.case.streams]
    chk = E.ForwardPlan(path.dims, path.tables, path.layers, path.input_ids, ref, cu_seqlens=path.cu,
                        sequence_ids=path.sid, token_mask=path.mask, lookback_ids=path.lookback, err=path.err)
    chk.run(stream)
    torch.cuda.synchronize()
    last = buf[(n - 1) % slots]["out"]
    if not all(torch.equal(o, r.cpu()) for o, r in zip(last, ref)):
        raise RuntimeError("pipelined end-to-end result differs from a plain forward pass")
    return {"ms": t0.elapsed_time(t1) / n, "h2d": int(h2d), "d2h": int(d2h), "slots": slots}


# ------------------------------------------------------------------------------------------------
# the CPU oracle (baseline line and reference arm)
# ------------------------------------------------------------------------------------------------

class OracleRunner:
    """The oracle on host copies of the workload: rows of the table are fetched once for the
    tokens in the sample, so each timed step runs the oracle's full path on them."""

    _BATCH_KEYS = ("input_ids", "token_map", "cu_seqlens", "sequence_ids", "token_mask", "lookback_ids")
    _LAYER_KEYS = ("need", "table", "scales", "wkv", "q", "k", "h")

    def save(self, path):
        """Write everything step() reads to an .npz (for a child process that times it)."""
        arrs = {"sel": self.sel}
        for k in self._BATCH_KEYS:
            if self.b.get(k) is not None:
                arrs["b_" + k] = self.b[k]
        for l, lay in enumerate(self.layers):
            arrs[f"fmt_{l}_{lay['fmt']}"] = np.zeros(0)
            for k in self._LAYER_KEYS:
                if lay[k] is not None:
                    arrs[f"l{l}_{k}"] = lay[k]
        np.savez(path, **arrs)

    @classmethod
    def load(cls, w, path):
        from oracle import engram_oracle as O
        r = cls.__new__(cls)
        r.O, r.w = O, w
        z = np.load(path)
        r.sel = z["sel"]
        r.b = {k: (z["b_" + k] if "b_" + k in z.files else None) for k in cls._BATCH_KEYS}
        r.pad = int(r.b["token_map"][w.pad_token_id])
        r.primes, r.offsets, _ = O.layout(w.vocab_size, w.layers, w.max_ngram, w.n_heads)
        r.mult = O.hash_multipliers(w.layer_ids, w.max_ngram, w.compressed_vocab)
        r.layers = []
        for l in range(w.layers):
            fmt = next(f.split("_", 2)[2] for f in z.files if f.startswith(f"fmt_{l}_"))
            lay = {"fmt": fmt}
            for k in cls._LAYER_KEYS:
                lay[k] = z[f"l{l}_{k}"] if f"l{l}_{k}" in z.files else None
            r.layers.append(lay)
        return r

    def __init__(self, w, case, n_tokens):
        from oracle import engram_oracle as O
        self.O, self.w = O, w
        b = case.batch
        self.b = b
        self.pad = int(b["token_map"][w.pad_token_id])
        self.primes, self.offsets, _ = O.layout(w.vocab_size, w.layers, w.max_ngram, w.n_heads)
        self.mult = O.hash_multipliers(w.layer_ids, w.max_ngram, w.compressed_vocab)
        win, _ = O.windows(b["input_ids"], b["token_map"], self.pad, w.max_ngram, b["cu_seqlens"],
                           b["sequence_ids"], b["token_mask"], b["lookback_ids"])
        ids = O.hash_ids(win, self.mult, self.primes, self.offsets, w.compressed_vocab)
        T = w.tokens
        n = min(n_tokens, T)
        self.sel = np.linspace(0, T - 1, n).round().astype(np.int64)
        self.layers = []
        for l, tab in enumerate(case.tables):
            need = np.unique(ids[self.sel, l, :].reshape(-1))
            idx = torch.from_numpy(need).to(tab["table"].device)
            t = tab["table"].index_select(0, idx).cpu()
            t_np = t.view(torch.int16).numpy().view(np.uint16) if tab["fmt"] == "bf16" else t.numpy()
            s_np = tab["scales"].index_select(0, idx).cpu().numpy() if tab["scales"] is not None else None
            self.layers.append({"fmt": tab["fmt"], "need": need, "table": t_np, "scales": s_np,
                                "wkv": case.wkv[l].cpu().view(torch.int16).numpy().view(np.uint16),
                                "q": case.q_weight[l].cpu().view(torch.int16).numpy().view(np.uint16),
                                "k": case.k_weight[l].cpu().view(torch.int16).numpy().view(np.uint16),
                                "h": case.streams[l].index_select(0, torch.from_numpy(self.sel).to(
                                    case.streams[l].device)).cpu().numpy()})

    def step(self):
        O, w, b = self.O, self.w, self.b
        win, _ = O.windows(b["input_ids"], b["token_map"], self.pad, w.max_ngram, b["cu_seqlens"],
                           b["sequence_ids"], b["token_mask"], b["lookback_ids"])
        ids = O.hash_ids(win, self.mult, self.primes, self.offsets, w.compressed_vocab)
        mask = b["token_mask"]
        for l, lay in enumerate(self.layers):
            sub = np.searchsorted(lay["need"], ids[self.sel, l, :])
            a_bits, _ = O.gather(lay["fmt"], lay["table"], lay["scales"], sub, len(lay["need"]), w.head_dim)
            kv = O.project(a_bits, lay["wkv"])
            O.gate(lay["h"], kv, lay["q"], lay["k"], w.eps, w.clamp, None if mask is None else mask[self.sel])


def time_oracle(r, seconds: float = 10.0, max_reps: int = 20):
    """Mean seconds per oracle pass: one warm pass (pages in the fp64 weights), then passes until
    `seconds` have gone by or `max_reps` passes ran."""
    r.step()
    t0 = time.perf_counter()
    reps = 0
    while True:
        r.step()
        reps += 1
        if time.perf_counter() - t0 > seconds or reps >= max_reps:
            break
    return (time.perf_counter() - t0) / reps, reps


BLAS_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                    "NUMEXPR_NUM_THREADS")


def cpu_child(args):
    """Child process of cpu_baseline: times the oracle state in args.cpu_child with the BLAS thread
    count its environment sets; prints one JSON line."""
    w = get_workload(args.workload)
    r = OracleRunner.load(w, args.cpu_child)
    dt, reps = time_oracle(r, args.cpu_seconds)
    print(json.dumps({"s_per_pass": dt, "reps": reps, "tokens": int(len(r.sel)), "layers": w.layers}))


def cpu_baseline(w, case, n_tokens, seconds: float = 10.0):
    """The oracle as it stands, on the host's cores: one run with one BLAS thread, one with a
    thread per core, each in a child process of its own (the thread count of numpy's BLAS is
    fixed when it loads). The same bounded token sample in both."""
    import tempfile
    r = OracleRunner(w, case, n_tokens)
    ncores = os.cpu_count() or 1
    runs = {}
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "oracle_state.npz")
        r.save(path)
        for label, threads in (("1_core", 1), ("all_cores", ncores)):
            env = dict(os.environ, **{k: str(threads) for k in BLAS_THREAD_VARS})
            env["CUDA_VISIBLE_DEVICES"] = ""          # the child never touches a GPU
            cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--workload", w.name,
                   "--cpu-child", path, "--cpu-seconds", str(seconds)]
            out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
            if out.returncode != 0:
                raise RuntimeError(f"oracle timing child failed: {out.stderr[-2000:]}")
            res = json.loads(out.stdout.strip().splitlines()[-1])
            runs[label] = {"value": round(res["tokens"] * res["layers"] / res["s_per_pass"], 2), "cores": threads,
                           "passes": res["reps"]}
    best = runs["all_cores"]
    return {"value": best["value"], "unit": "tokens/s per layer", "cores": best["cores"], "kind": "oracle",
            "one_core": runs["1_core"], "all_cores": runs["all_cores"],
            "sample": f"{len(r.sel)} of {w.tokens} tokens per pass (hash over all {w.tokens} tokens), "
                      f"numpy fp64; one child process with 1 BLAS thread and one with {ncores}"}


def workload_config(w, table_rows: int, wkv: str, world: int) -> dict:
    """The workload keys of the JSON line's config (both arms)."""
    return {"workload": w.name, "tokens": w.tokens, "layers": w.layers, "hash_cols": w.cols,
            "head_dim": w.head_dim, "table": w.table_format, "table_rows": table_rows, "hidden": w.hidden,
            "hc": w.hc, "K": w.K, "N": w.N, "wkv": wkv, "parallelism": f"replicas{world}"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = get_workload(args.workload)
    device = "cuda" if torch.cuda.is_available() else "cpu"
    from oracle import engram_oracle as O
    _, _, rows = O.layout(w.vocab_size, w.layers, w.max_ngram, w.n_heads)
    case = make_case(w, [int(r) for r in np.asarray(rows).reshape(-1)], device)
    r = OracleRunner(w, case, args.cpu_tokens)
    for _ in range(min(args.warmup, 3)):
        r.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r.step()
    dt = (time.perf_counter() - t0) / args.steps
    value = len(r.sel) * w.layers / dt
    return {
        "impl": "reference",
        "metric": "engram_tokens_per_s_per_layer",
        "value": round(value, 2),
        "unit": "tokens/s per layer",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": workload_config(w, int(np.asarray(rows).sum()), "bf16", world),
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s per layer", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"{len(r.sel)} of {w.tokens} tokens per step (hash over all), numpy fp64"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s per layer", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--wkv", choices=["bf16", "mxfp8"], default="bf16",
                    help="wkv format: bf16 (the workloads' own), or MXFP8 (the FP8 operand variant)")
    ap.add_argument("--operand-gather", action="store_true",
                    help="FP8 variant: the projection gathers its token rows from the table itself")
    ap.add_argument("--gemm-tile", type=int, default=0, help="tuning: force the bf16 projection's tile width")
    ap.add_argument("--mx-tile", type=int, default=0, help="tuning: force the MXFP8 projection's tile width")
    ap.add_argument("--gather-order", type=int, default=0, choices=[0, 1],
                    help="engram_forward's gathers: 0 token order, 1 table order (rows grouped by table region)")
    ap.add_argument("--side-stream", action="store_true",
                    help="engram_forward2: the later layers' gathers on a second stream")
    ap.add_argument("--gate-fusion", type=int, nargs="?", const=1, default=0, choices=[0, 1, 2],
                    help="engram_forward's gate: 1 key sums in the projection's epilogue, 2 the gate inside the "
                         "projection kernel, overlapped with it")
    ap.add_argument("--gate-form", type=int, choices=[0, 1, 2], default=0,
                    help="gate kernel: 0 automatic, 1 persistent, 2 one CTA per (token, stream) item")
    ap.add_argument("--cpu-tokens", type=int, default=32)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variant", action="store_true", help="skip the FP8 operand variant's line")
    ap.add_argument("--only", choices=["hash", "gather", "project", "gate", "forward"],
                    help="profiling: run one stage alone (forward: engram_forward as a whole)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling (--only): one sequence of this many tokens instead of the workload's")
    ap.add_argument("--table-rows", type=int, default=0,
                    help="profiling: shrink the table to about this many rows per layer")
    ap.add_argument("--cpu-child", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_child:
        cpu_child(args)
        return
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA device for --impl ours")
        torch.cuda.set_device(local)
        import engram_gram_hash_02_gb300 as E
        if args.gate_form:
            E.set_gate_form(args.gate_form)
        if args.gate_fusion:
            E.set_gate_fusion(args.gate_fusion)
        if args.operand_gather:
            E.set_operand_gather(True)
        if args.gather_order:
            E.set_gather_order(args.gather_order)
        if args.gemm_tile:
            E.set_gemm_tile(args.gemm_tile)
        if args.mx_tile:
            E.set_gemm_mx_tile(args.mx_tile)
        if args.only:
            run_only(args, torch.device("cuda", local))
            return
        line = run_ours(args, rank, world, torch.device("cuda", local))
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
