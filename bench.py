#!/usr/bin/env python3
"""Decode-attention benchmark: one JSON line on rank 0.

A step is one decode step of the attention block of a 36-layer model: the
step's RoPE cos/sin table (one launch, shared by every layer) and 36
back-to-back layer-steps (qdec_step: QK RMSNorm + NeoX RoPE + paged append +
split-KV GQA attention with the log-sum-exp merge, one kernel launch each),
each layer with its own KV pool, all layers sharing the block table.  Each
layer may start streaming its cached pages while the previous layer
finishes (programmatic dependent launch).  The launches are captured once in
CUDA graphs and replayed per step.

value   = KV GB/s: algorithmic bytes (KV read at token granularity plus the
          q/k/v inputs and the output) / device time, over all ranks.
e2e     = the same metric with, every step, the host->device copy of the
          step's new-token inputs and metadata from pinned memory and the
          device->host copy of the outputs inside the timed region.
roofline = the fused kernel against the measured HBM copy bandwidth.
cpu_baseline / --impl reference = the fp64 CPU oracle on a bounded sample.
--kv fp8 runs the same workload over an FP8 (E4M3) pool with per-(page,
plane, head) scales (qdec_step_fp8); its bytes count one byte per KV element
plus the scales read.
--qkv runs the block from hidden states instead: per layer the merged QKV
projection fused with norm, rotation and append (qdec_qkv_append_rope, a
random [(Hq+2Hkv)*128][hidden] weight per layer), then qdec_attn_decode
(split-KV attention and merge in one launch); its bytes add the weight and
the hidden states and drop q/k/v, and the roofline object describes the
projection kernel.

Multi-GPU: the path shards without any exchange, so N ranks run N
independent replicas (weak scaling); value sums their work over the slowest
rank's time.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from dataclasses import replace

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gqa_paged_kv_gb300 import workloads as wl  # noqa: E402

METRIC = "decode-attn µs/layer-step and KV GB/s (% of GB300 HBM peak) per batch×ctx"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PREFILL_METRIC = "prefill-attn TFLOP/s (causal, algorithmic) and µs/layer per prompt"
# the sources each roofline kernel is built from (its traffic entry below
# stays valid only while their hash matches)
_CSRC = "gqa_paged_kv_gb300/csrc/"
KERNEL_SOURCES = {
    "attention_kernel": tuple(_CSRC + f for f in ("qdec_kernels.cu", "qdec_internal.h",
                                                  "qdec_ptx.cuh", "qdec_ff.cuh")),
    "qkv_append_kernel": tuple(_CSRC + f for f in ("qdec_qkv.cu", "qdec_internal.h",
                                                   "qdec_ptx.cuh")),
    "prefill_attention_tc_kernel": tuple(_CSRC + f for f in ("qdec_prefill.cu",
                                                             "qdec_internal.h", "qdec_ptx.cuh",
                                                             "qdec_tc.cuh", "qdec_ff.cuh")),
}

# DRAM bytes per launch of the fused kernel measured with ncu (see
# profiles/), keyed by workload; used only while the kernel source hash
# still matches the one the counters were taken on.
TRAFFIC = {
    # the attention kernel (workload 5: the decode-mode kernel of the
    # two-launch step)
    "b8-ctx256to384-36layer":
        {"kernel_sha": "fec73a2c7746cf7a", "bytes_per_launch": 10899880},
    "b16-ctx256to384-chanscale-36layer":
        {"kernel_sha": "fec73a2c7746cf7a", "bytes_per_launch": 21779612},
    "b1-ctx8192-spikes-36layer":
        {"kernel_sha": "fec73a2c7746cf7a", "bytes_per_launch": 33636451},
    "b64-ragged128to16384-sharedpool-36layer":
        {"kernel_sha": "fec73a2c7746cf7a", "bytes_per_launch": 1038109092},
    "b64-ragged128to16384-sharedpool-36layer-fp8kv":
        {"kernel_sha": "fec73a2c7746cf7a", "bytes_per_launch": 524977074},
    # --prefill 2048: the causal prefill attention kernel (over an FP8 pool the
    # kernel that reads the dequantized workspace)
    "prefill-b1-prompt2048-36layer":
        {"kernel_sha": "7ac9fd35607ab740", "bytes_per_launch": 42005519},
    "prefill-b1-prompt2048-36layer-fp8kv":
        {"kernel_sha": "7ac9fd35607ab740", "bytes_per_launch": 42008950},
    # --qkv: the projection kernel
    "b8-ctx256to384-36layer-qkv2560":
        {"kernel_sha": "d083545efb834ee5", "bytes_per_launch": 31553438},
    "b64-ragged128to16384-sharedpool-36layer-qkv2560":
        {"kernel_sha": "d083545efb834ee5", "bytes_per_launch": 31908697},
}

# The CPU timings sample the first few layers of a workload (same shapes and
# lengths; fewer per-layer pools to materialise in host memory).
CPU_SAMPLE_LAYERS = 4
L2_BYTES_NOMINAL = 126 << 20


def kernel_sha(kernel: str = "attention_kernel") -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", type=int, default=5, choices=sorted(wl.WORKLOADS),
                    help="the headline workload (default 5, the largest; the others get one "
                         "record each in the line's `configs`)")
    ap.add_argument("--no-configs", action="store_true",
                    help="time the headline workload only")
    ap.add_argument("--plan-bound", type=int, default=0, metavar="TOKENS",
                    help="plan the step for contexts up to TOKENS (a model-wide bound) "
                         "instead of the workload's own maximum")
    ap.add_argument("--kv", choices=("bf16", "fp8"), default="bf16",
                    help="KV pool element type (fp8: E4M3 codes + per-page scales)")
    ap.add_argument("--qkv", action="store_true",
                    help="start each layer from hidden states: fused QKV projection + attention")
    ap.add_argument("--hidden", type=int, default=2560, help="hidden size for --qkv")
    ap.add_argument("--prefill", type=int, default=0, metavar="PROMPT",
                    help="chunked prefill instead of decode: one fresh prompt of PROMPT tokens "
                         "per layer (append + causal attention), metric TFLOP/s")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the 36 calls eagerly")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--two-call", action="store_true",
                    help="each layer as qdec_append_rope then qdec_attn_decode (step 4 and its "
                         "merge in one launch) instead of the one-launch qdec_step")
    ap.add_argument("--three-call", action="store_true",
                    help="each layer as qdec_append_rope, qdec_attn_split, qdec_attn_merge "
                         "(launched one after another) instead of the one-launch qdec_step")
    ap.add_argument("--no-overlap", action="store_true",
                    help="launch each layer only after the previous one completed")
    ap.add_argument("--fp8-in-kernel", action="store_true",
                    help="--prefill --kv fp8: convert the codes inside the attention kernel "
                         "instead of widening the pages once into a workspace")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: run fewer layers than the workload has")
    ap.add_argument("--pool-pages", type=int, default=0,
                    help="profiling only: a smaller pool per layer (it must still hold every "
                         "page the sequences reference; the work and traffic are the same)")
    return ap.parse_args()


# ------------------------------------------------------------------ infra --
class Dist:
    """One process per GPU (torchrun env vars).  The ranks run independent
    replicas of the workload: the only communication is the barrier around
    the timed region and the max of the elapsed times.  NCCL on GPUs, gloo
    where there are none (the CPU tests of this path)."""

    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.device = "cpu"
        if self.world > 1:
            import torch.distributed as dist
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local)
                self.device = f"cuda:{self.local}"
                dist.init_process_group("nccl", device_id=torch.device("cuda", self.local))
            else:
                dist.init_process_group("gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


class Clocks:
    """nvidia-smi samples of this GPU's clocks and throttle reasons."""
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.bus = None
        try:
            props = torch.cuda.get_device_properties(device)
            self.bus = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id,
                                             props.pci_device_id)
        except Exception:
            pass
        self.proc = None
        self.path = None

    def _cmd(self, loop_ms=None):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits"]
        if self.bus:
            cmd += ["-i", self.bus]
        if loop_ms:
            cmd += ["-lms", str(loop_ms)]
        return cmd

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(self._cmd(50), stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        rows = []
        try:
            snap = subprocess.run(self._cmd(), capture_output=True, text=True, timeout=20).stdout
        except (OSError, subprocess.SubprocessError):
            snap = ""
        if self.proc:
            self.proc.terminate()
            self.proc.wait(timeout=10)
        text = (open(self.path).read() if self.path else "") + snap
        for line in text.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append((float(f[2]), float(f[3]), f[5:]))
            except ValueError:
                continue
        if self.path:
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ("active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2])
                          if i > 0 and v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


def l2_bytes(dev=None) -> int:
    if dev is not None:
        n = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)
        if n:
            return int(n)
    return L2_BYTES_NOMINAL


def workload_name(spec, kv: str, qkv_hidden: int = 0, calls: int = 1) -> str:
    return (spec.name + ("-fp8kv" if kv == "fp8" else "")
            + (f"-qkv{qkv_hidden}" if qkv_hidden else "")
            + {1: "", 2: "-twocall", 3: "-threecall"}[calls])


def calls_per_layer(args) -> int:
    """Launches of one decode layer-step: qdec_step, or the two- or
    three-call decompositions."""
    return 3 if getattr(args, "three_call", False) else 2 if getattr(args, "two_call", False) else 1


def qkv_weight_bytes(spec, hidden: int) -> int:
    return (spec.num_q_heads + 2 * spec.num_kv_heads) * spec.head_dim * hidden * 2


def block_bytes_per_layer(w: wl.Workload, hidden: int) -> int:
    """--qkv: the weight, the hidden states, the KV read at token granularity
    and the output."""
    s = w.spec
    kv = w.algorithmic_bytes_per_layer() - s.batch * s.io_bytes_per_seq()
    return (qkv_weight_bytes(s, hidden) + s.batch * hidden * 2 + kv
            + s.batch * s.num_q_heads * s.head_dim * 2)


def workload_config(w: wl.Workload, args, world: int, l2: int = L2_BYTES_NOMINAL,
                    layers: int = 0) -> dict:
    """The `config` object of the JSON line (the same for both arms; the
    reference arm times a few layers of the workload and passes the full
    layer count as `layers`)."""
    spec, seq_lens_host = w.spec, w.seq_lens_host
    L = layers or spec.layers
    qkv_hidden = args.hidden if getattr(args, "qkv", False) else 0
    bytes_layer = (block_bytes_per_layer(w, qkv_hidden) if qkv_hidden
                   else w.algorithmic_bytes_per_layer())
    bytes_step = bytes_layer * L
    if bytes_step < 2 * l2:
        l2_note = (f"L2 flushed: a {2 * l2 / 2**20:.0f} MiB buffer is rewritten before each "
                   f"timed step (untimed); a step reads {bytes_step / 1e6:.1f} MB")
    elif spec.shared_pool:
        l2_note = (f"inputs larger than L2: {bytes_layer / 1e9:.3f} GB per layer-step from "
                   "one shared pool")
    else:
        l2_note = (f"inputs larger than L2: each step reads {bytes_step / 1e9:.3f} GB of KV "
                   f"across {L} per-layer pools")
    cfg = {"workload": workload_name(spec, w.kv, qkv_hidden), "batch": spec.batch,
            "ctx": f"{int(seq_lens_host.min())}-{int(seq_lens_host.max())}",
            "heads": f"{spec.num_q_heads}q/{spec.num_kv_heads}kv",
            "head_dim": spec.head_dim, "page_size": spec.page_size, "layers": L,
            "pool_pages_per_layer": spec.pool_pages,
            "kv_cache": ("E4M3 codes + fp32 scale per (page, plane, KV head)" if w.kv == "fp8"
                         else "bf16"),
            "kv_bytes_per_step": bytes_step,
            "l2": l2_note,
            "launch": ("eager" if args.no_graph else f"CUDA graphs: rope table + "
                       f"{L} {'qdec_step_fp8' if w.kv == 'fp8' else 'qdec_step'}")
                      + ("" if args.no_overlap else
                                            ", programmatic dependent launch"),
            "parallelism": f"replicas x{world}"}
    if qkv_hidden:
        cfg["hidden"] = qkv_hidden
        cfg["launch"] = (f"CUDA graphs: rope table + {L} x (qdec_qkv_append_rope, "
                         f"qdec_attn_decode)")
    elif calls_per_layer(args) == 3:
        sfx = "_fp8" if w.kv == "fp8" else ""
        cfg["workload"] = workload_name(spec, w.kv, 0, 3)
        cfg["launch"] = ("eager" if args.no_graph else "CUDA graphs") + (
            f": rope table + {L} x (qdec_append_rope{sfx}, qdec_attn_split{sfx}, "
            f"qdec_attn_merge), each launch after the previous one")
    elif calls_per_layer(args) == 2:
        sfx = "_fp8" if w.kv == "fp8" else ""
        cfg["workload"] = workload_name(spec, w.kv, 0, 2)
        cfg["launch"] = ("eager" if args.no_graph else "CUDA graphs") + (
            f": rope table + {L} x (qdec_append_rope{sfx}, qdec_attn_decode{sfx})"
            + ("" if args.no_overlap else ", programmatic dependent launch"))
    return cfg


# ------------------------------------------------------------ CPU oracle --
def oracle_sample(w: wl.Workload, seconds: float, per_seq: bool):
    """Time the fp64 oracle (as it stands, one thread) on a bounded sample of
    the workload: layer-steps in order (one sequence at a time when per_seq),
    until `seconds` have passed.  Returns (GB/s, description, steps, elapsed)."""
    import oracle
    B = w.spec.batch
    units = ([(l, [b]) for l in range(w.spec.layers) for b in range(B)] if per_seq
             else [(l, None) for l in range(w.spec.layers)])
    bytes_done, n, t_total = 0, 0, 0.0
    i = 0
    while t_total < seconds or n == 0:
        layer, seqs = units[i % len(units)]
        inp = wl.oracle_inputs(w, layer, seqs)
        t0 = time.perf_counter()
        oracle_layer(inp)
        t_total += time.perf_counter() - t0
        bytes_done += sample_bytes(w, inp["seq_lens"])
        n += 1
        i += 1
    what = "one sequence of one layer" if per_seq else "one layer (all sequences)"
    return bytes_done / t_total / 1e9, what, n, t_total


def oracle_layer(inp: dict):
    """One oracle layer-step on oracle_inputs (on a copy of the pool)."""
    import oracle
    args = (inp["q"], inp["k"], inp["v"], inp["w_q"], inp["w_k"], inp["positions"],
            inp["seq_lens"], inp["block_table"], inp["pool"].copy())
    if "kv_scale" in inp:
        oracle.decode_layer_fp8(*args, inp["kv_scale"], inp["rope_theta"], inp["eps"])
    else:
        oracle.decode_layer(*args, inp["rope_theta"], inp["eps"])


def sample_bytes(w: wl.Workload, seq_lens) -> int:
    """Algorithmic bytes of the given sequences of one layer-step."""
    s = w.spec
    sl = np.asarray(seq_lens, dtype=np.int64)
    io = len(sl) * s.io_bytes_per_seq()
    if w.kv == "fp8":
        pages = int(((sl + s.page_size - 1) // s.page_size).sum())
        return int(sl.sum()) * s.kv_bytes_per_token() // 2 + pages * 2 * s.num_kv_heads * 4 + io
    return int(sl.sum()) * s.kv_bytes_per_token() + io


def qkv_sample_bytes(w: wl.Workload, hidden: int, seq_lens) -> int:
    """--qkv: algorithmic bytes of the given sequences of one layer's block
    (the whole weight, their hidden states, KV and output)."""
    s = w.spec
    n = len(seq_lens)
    kv = sample_bytes(w, seq_lens) - n * s.io_bytes_per_seq()
    return qkv_weight_bytes(s, hidden) + n * hidden * 2 + kv + n * s.num_q_heads * s.head_dim * 2


def oracle_qkv_operands(w: wl.Workload, hidden: int):
    """Seeded hidden states [B][hidden] and one merged weight for the oracle
    (bf16 bits; the GPU arm's distributions, drawn on the host)."""
    s = w.spec
    gen = torch.Generator().manual_seed(s.seed + 11)
    x = torch.randn((s.batch, hidden), generator=gen).to(torch.bfloat16)
    rows = (s.num_q_heads + 2 * s.num_kv_heads) * s.head_dim
    wq = (torch.randn((rows, hidden), generator=gen) / hidden ** 0.5).to(torch.bfloat16)
    return wl.bf16_bits(x), wl.bf16_bits(wq)


def oracle_qkv_block(inp: dict, x, wqkv, seqs=None):
    """One oracle step of the --qkv block on oracle_inputs (a copy of the
    pool): projection fused with norm, rotation and append, then attention."""
    import math

    import oracle
    s_x = x if seqs is None else np.ascontiguousarray(x[seqs])
    pool = inp["pool"].copy()
    Hq = inp["q"].shape[1]
    res = oracle.qkv_append(s_x, wqkv, inp["w_q"], inp["w_k"], inp["positions"],
                            inp["seq_lens"], inp["block_table"], pool, inp["rope_theta"],
                            inp["eps"], Hq, pool.shape[2])
    oracle.attention(pool, inp["block_table"], inp["seq_lens"], res["q_rot"],
                     1 / math.sqrt(pool.shape[4]))


def oracle_qkv_sample(w: wl.Workload, hidden: int, seconds: float):
    """Time the oracle's --qkv block (one thread) on whole layers in order
    until `seconds` have passed.  Returns (GB/s, layers done, elapsed)."""
    x, wqkv = oracle_qkv_operands(w, hidden)
    bytes_done, n, t_total = 0, 0, 0.0
    while t_total < seconds or n == 0:
        inp = wl.oracle_inputs(w, n % w.spec.layers)
        t0 = time.perf_counter()
        oracle_qkv_block(inp, x, wqkv)
        t_total += time.perf_counter() - t0
        bytes_done += qkv_sample_bytes(w, hidden, inp["seq_lens"])
        n += 1
    return bytes_done / t_total / 1e9, n, t_total


def reference_device() -> str:
    """Where the reference arm synthesises its inputs: the GPU when there is
    one (drawing an 8 GiB pool there takes a second), else the host.  The
    oracle itself always runs on the host cores, on host copies."""
    return "cuda:0" if torch.cuda.is_available() else "cpu"


def run_reference(args, dist: Dist):
    """The reference arm: the CPU oracle, timed as it stands on the host."""
    if dist.rank != 0:
        return
    spec = wl.WORKLOADS[args.workload]
    w = wl.build(spec, reference_device(), layers=min(spec.layers, CPU_SAMPLE_LAYERS),
                 kv=args.kv)
    # a step is one sequence of one layer; the host copies of the steps'
    # inputs are made before the clock starts
    ops = oracle_qkv_operands(w, args.hidden) if args.qkv else None
    prepared = oracle_step_inputs(w, max(args.steps, args.warmup))
    oracle_run_steps(w, prepared[:args.warmup], ops, args.hidden)
    t0 = time.perf_counter()
    gbs_bytes = oracle_run_steps(w, prepared[:args.steps], ops, args.hidden)
    dt = time.perf_counter() - t0
    value = gbs_bytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": workload_config(w, args, 1, layers=spec.layers),
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} steps of one sequence x one layer"
                                   f"{' of the QKV block' if args.qkv else ''} "
                                   f"(layers 0-{w.spec.layers - 1} of the workload), "
                                   f"{dt:.1f} s"},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def oracle_step_inputs(w: wl.Workload, k: int):
    """Host inputs of k oracle steps of one sequence of one layer (sequences
    in order, then layers), as (inputs, sequence) pairs."""
    B = w.spec.batch
    out = []
    for i in range(k):
        layer, b = (i // B) % w.spec.layers, i % B
        out.append((wl.oracle_inputs(w, layer, [b]), b))
    return out


def oracle_run_steps(w: wl.Workload, prepared, qkv_ops=None, hidden: int = 0) -> int:
    """Run prepared oracle steps (of the --qkv block when qkv_ops holds its
    hidden states and weight); returns their bytes."""
    done = 0
    for inp, b in prepared:
        if qkv_ops is not None:
            oracle_qkv_block(inp, qkv_ops[0], qkv_ops[1], [b])
            done += qkv_sample_bytes(w, hidden, inp["seq_lens"])
        else:
            oracle_layer(inp)
            done += sample_bytes(w, inp["seq_lens"])
    return done


def oracle_steps(w: wl.Workload, k: int, qkv_ops=None, hidden: int = 0) -> int:
    """k oracle steps of one sequence of one layer; returns their bytes."""
    return oracle_run_steps(w, oracle_step_inputs(w, k), qkv_ops, hidden)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def balanced_parts(seq_lens, parts: int):
    """Sequence indices split into `parts` groups of about equal total length
    (longest first, each to the least loaded group)."""
    groups = [[] for _ in range(parts)]
    load = [0] * parts
    for b in sorted(range(len(seq_lens)), key=lambda i: -int(seq_lens[i])):
        j = load.index(min(load))
        groups[j].append(b)
        load[j] += int(seq_lens[b])
    return [sorted(g) for g in groups if g]


def oracle_sample_all_cores(w: wl.Workload, seconds: float, threads: int):
    """The same oracle on every host core: each layer-step's sequences are
    split into `threads` groups of about equal length and the oracle runs on
    each group in its own thread (the C oracle holds no shared state and the
    call releases the interpreter lock), until `seconds` have passed.
    Returns (GB/s, threads used, layer-steps, elapsed)."""
    from concurrent.futures import ThreadPoolExecutor
    groups = balanced_parts(w.seq_lens_host, threads)
    layers = list(range(min(2, w.spec.layers)))
    prepared = {l: [wl.oracle_inputs(w, l, g) for g in groups] for l in layers}
    bytes_done, n, t_total = 0, 0, 0.0
    with ThreadPoolExecutor(max_workers=len(groups)) as ex:
        while t_total < seconds or n == 0:
            parts = prepared[layers[n % len(layers)]]
            t0 = time.perf_counter()
            list(ex.map(oracle_layer, parts))
            t_total += time.perf_counter() - t0
            bytes_done += sample_bytes(w, w.seq_lens_host)
            n += 1
    return bytes_done / t_total / 1e9, len(groups), n, t_total


# -------------------------------------------------------------- our path --
# A model-wide plan bound for the graph-reuse records: the step is captured
# once for contexts up to this many tokens and replayed on shorter ones.
MODEL_SEQ_BOUND = 16384


class DecodeLayers:
    """Device buffers, shape and step function of one decode workload on
    this rank's GPU.  plan_bound > 0 plans (and sizes the block-table rows
    for) contexts up to plan_bound tokens instead of the workload's own
    maximum, as an engine that captures one graph for every length would."""

    def __init__(self, qdec, w: wl.Workload, args, stream, plan_bound: int = 0):
        self.qdec, self.w, self.args, self.stream = qdec, w, args, stream
        spec = w.spec
        P = spec.page_size
        mb = w.max_blocks
        self.block_table = w.block_table
        if plan_bound:
            mb = max(mb, (plan_bound + P - 1) // P)
            bt = torch.full((spec.batch, mb), -1, dtype=torch.int32, device=w.block_table.device)
            bt[:, :w.max_blocks] = w.block_table
            self.block_table = bt
        flags = 0 if args.no_overlap or calls_per_layer(args) == 3 else qdec.QDEC_LAUNCH_OVERLAP_PREVIOUS
        self.shape = qdec.Shape(batch=spec.batch, num_pages=spec.pool_pages,
                                max_blocks_per_seq=mb,
                                max_seq_len=max(plan_bound, w.max_blocks * P) if plan_bound
                                else mb * P,
                                num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                                head_dim=spec.head_dim, page_size=P, launch_flags=flags)
        self.ws = qdec.alloc_workspace(self.shape)
        self.rope = qdec.alloc_rope_table(self.shape)
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.out = torch.empty((spec.layers, spec.batch, spec.num_q_heads, spec.head_dim),
                               dtype=torch.bfloat16, device="cuda")
        self.q_rot = (torch.empty((spec.batch, spec.num_q_heads, spec.head_dim),
                                  dtype=torch.float32, device="cuda")
                      if args.three_call or args.two_call else None)

    def step_fn(self, qkv, seq_lens, positions, block_table, out_t):
        """One decode step (the rope table, then every layer) on these buffers."""
        qdec, w, shape, s = self.qdec, self.w, self.shape, self.stream
        Hq, Hkv = w.spec.num_q_heads, w.spec.num_kv_heads

        def fn():
            qdec.qdec_rope_table(shape, positions, self.rope, stream=s)
            for l in range(w.spec.layers):
                q, k, v = qkv[l, :, :Hq], qkv[l, :, Hq:Hq + Hkv], qkv[l, :, Hq + Hkv:]
                if self.args.three_call and w.kv == "fp8":
                    qdec.qdec_append_rope_fp8(shape, q, k, v, w.w_q[l], w.w_k[l], positions,
                                              seq_lens, block_table, w.pool8(l), w.scale(l),
                                              self.q_rot, self.err, stream=s, rope_table=self.rope)
                    qdec.qdec_attn_split_fp8(shape, self.q_rot, w.pool8(l), w.scale(l), block_table,
                                             seq_lens, self.ws, out_t[l], self.err, stream=s)
                    qdec.qdec_attn_merge(shape, seq_lens, self.ws, out_t[l], self.err, stream=s)
                elif self.args.two_call and w.kv == "fp8":
                    qdec.qdec_append_rope_fp8(shape, q, k, v, w.w_q[l], w.w_k[l], positions,
                                              seq_lens, block_table, w.pool8(l), w.scale(l),
                                              self.q_rot, self.err, stream=s, rope_table=self.rope)
                    qdec.qdec_attn_decode_fp8(shape, self.q_rot, w.pool8(l), w.scale(l),
                                              block_table, seq_lens, self.ws, out_t[l], self.err,
                                              stream=s)
                elif self.args.two_call:
                    qdec.qdec_append_rope(shape, q, k, v, w.w_q[l], w.w_k[l], positions, seq_lens,
                                          block_table, w.pool(l), self.q_rot, self.err, stream=s,
                                          rope_table=self.rope)
                    qdec.qdec_attn_decode(shape, self.q_rot, w.pool(l), block_table, seq_lens,
                                          self.ws, out_t[l], self.err, stream=s)
                elif self.args.three_call:
                    qdec.qdec_append_rope(shape, q, k, v, w.w_q[l], w.w_k[l], positions, seq_lens,
                                          block_table, w.pool(l), self.q_rot, self.err, stream=s,
                                          rope_table=self.rope)
                    qdec.qdec_attn_split(shape, self.q_rot, w.pool(l), block_table, seq_lens,
                                         self.ws, out_t[l], self.err, stream=s)
                    qdec.qdec_attn_merge(shape, seq_lens, self.ws, out_t[l], self.err, stream=s)
                elif w.kv == "fp8":
                    qdec.qdec_step_fp8(shape, qkv[l, :, :Hq], qkv[l, :, Hq:Hq + Hkv],
                                       qkv[l, :, Hq + Hkv:], w.w_q[l], w.w_k[l], positions,
                                       seq_lens, block_table, w.pool8(l), w.scale(l), self.ws,
                                       out_t[l], self.err, stream=s, rope_table=self.rope)
                else:
                    qdec.qdec_step(shape, qkv[l, :, :Hq], qkv[l, :, Hq:Hq + Hkv],
                                   qkv[l, :, Hq + Hkv:], w.w_q[l], w.w_k[l], positions,
                                   seq_lens, block_table, w.pool(l), self.ws, out_t[l],
                                   self.err, stream=s, rope_table=self.rope)
        return fn

    def default_step(self):
        w = self.w
        return self.step_fn(w.qkv, w.seq_lens, w.positions, self.block_table, self.out)

    def check(self):
        st, flags = self.qdec.qdec_check_error(self.err, self.stream)
        assert st == 0, f"device error flags {flags:#x}"


def capture(fn, stream):
    """fn once eagerly (it configures the kernels outside capture), then
    captured into a CUDA graph; returns the graph's replay."""
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            fn()
    capture.keep.append(g)
    return g.replay


capture.keep = []


def timed_steps(run, stream, steps: int, warmup: int, dist: Dist, flush=None, clocks=None):
    """warmup untimed steps, then exactly `steps` timed ones, bracketed by a
    barrier and a device synchronisation.  With `flush` (a buffer larger than
    L2) it is rewritten before every step, outside the per-step events, and
    the time is the sum of the steps; else the whole region.  Returns
    (this rank's ms, max over ranks of it, per-step ms)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if clocks:
        clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for k in range(steps):
            if flush is not None:
                flush.add_(1)   # evict the previous step's lines from L2 (not timed)
            starts[k].record(stream)
            run()
            ends[k].record(stream)
        e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    per = [a.elapsed_time(e) for a, e in zip(starts, ends)]
    t_ms = sum(per) if flush is not None else e0.elapsed_time(e1)
    return t_ms, dist.max(t_ms), per


def step_spread(per_ms, layers: int) -> dict:
    """Median and 10th / 90th percentiles (nearest rank) of the per-step
    CUDA-event times, as µs per layer-step."""
    xs = sorted(per_ms)
    if not xs:
        return {}

    def rank(f):
        return xs[min(len(xs) - 1, int(round(f * (len(xs) - 1))))] * 1e3 / layers

    return {"median": round(rank(0.5), 4), "p10": round(rank(0.1), 4),
            "p90": round(rank(0.9), 4)}


def l2_flush_buffer(bytes_step: int, l2: int):
    """A buffer of twice the L2 size when a step's inputs would fit in it."""
    if bytes_step < 2 * l2:
        return torch.empty(2 * l2 // 4, dtype=torch.int32, device="cuda")
    return None


def config_record(qdec, workload_id: int, args, dist: Dist, dev: int, peak: float) -> dict:
    """One bench record per workload (besides the headline line): µs per
    layer-step and GB/s of the graph-replayed step (the contract's timing),
    the same step launched from the host without a graph, for workload 1
    also L2-warm, and for the short-context workloads 2 and 4 also with the
    step planned for a model-wide bound of MODEL_SEQ_BOUND tokens."""
    spec = wl.WORKLOADS[workload_id]
    w = wl.build(spec, f"cuda:{dev}", kv=args.kv)
    L = w.spec.layers
    stream = torch.cuda.Stream()
    bytes_layer = w.algorithmic_bytes_per_layer()
    l2 = l2_bytes(dev)
    flush = l2_flush_buffer(bytes_layer * L, l2)

    def measure(layers: DecodeLayers, graph: bool, fl, with_clocks: bool):
        step = layers.default_step()
        run = capture(step, stream) if graph else step
        if not graph:
            with torch.cuda.stream(stream):
                step()   # first launch configures the kernels
        ck = Clocks(dev) if with_clocks else None
        t_ms, t_max, per = timed_steps(run, stream, args.steps, max(3, args.warmup), dist, fl, ck)
        layers.check()
        us = t_max / args.steps / L * 1e3
        rec = {"us_per_layer_step": round(us, 4), "spread": step_spread(per, L),
               "gbs": round(dist.world * bytes_layer / (us * 1e-6) / 1e9, 2),
               "frac_of_hbm": round(bytes_layer / (us * 1e-6) / 1e9 / peak, 4)}
        if ck:
            rec["clocks"] = ck.stop()
        return rec

    base = DecodeLayers(qdec, w, args, stream)
    rec = {"workload": workload_name(w.spec, w.kv), "layers": L,
           "bytes_per_layer_step": bytes_layer,
           "l2": "flushed before each step" if flush is not None else "inputs larger than L2",
           "plan": "exact bound (max_seq_len = the workload's block-table rows x 16)"}
    rec.update(measure(base, True, flush, True))
    rec["eager"] = measure(base, False, flush, False)
    if flush is not None:
        rec["l2_warm"] = measure(base, True, None, False)
    if workload_id in (2, 4) and w.spec.max_seq_len_bound < MODEL_SEQ_BOUND:
        bound = DecodeLayers(qdec, w, args, stream, plan_bound=MODEL_SEQ_BOUND)
        rec[f"plan_bound_{MODEL_SEQ_BOUND}"] = measure(bound, True, flush, False)
        del bound
    del base, w, flush
    capture.keep.clear()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def run_ours(args, dist: Dist):
    from gqa_paged_kv_gb300 import build as qbuild
    qbuild.build()
    from gqa_paged_kv_gb300 import qdec

    dev = dist.local
    torch.cuda.set_device(dev)
    spec = wl.WORKLOADS[args.workload]
    if args.pool_pages:
        spec = replace(spec, pool_pages=args.pool_pages)
    w = wl.build(spec, f"cuda:{dev}", layers=args.layers or None, kv=args.kv)
    spec = w.spec
    L = spec.layers
    stream = torch.cuda.Stream()
    layers = DecodeLayers(qdec, w, args, stream, plan_bound=args.plan_bound)
    shape, ws, rope, err, out = layers.shape, layers.ws, layers.rope, layers.err, layers.out
    torch.cuda.synchronize()

    Hq, Hkv = spec.num_q_heads, spec.num_kv_heads
    if args.qkv:
        assert w.kv == "bf16", "--qkv runs on a bf16 pool"
        # hidden states and one merged projection weight per layer (seeded)
        gen = torch.Generator(device="cuda").manual_seed(spec.seed + 11)
        step_in = torch.randn((L, spec.batch, args.hidden), generator=gen,
                              device="cuda").to(torch.bfloat16)
        w_qkv = torch.empty((L, (Hq + 2 * Hkv) * spec.head_dim, args.hidden),
                            dtype=torch.bfloat16, device="cuda")
        for l in range(L):
            w_row = (torch.randn(w_qkv.shape[1:], generator=gen, device="cuda")
                     / args.hidden ** 0.5).to(torch.bfloat16)
            qdec.qdec_qkv_pack_weights(shape, w_row, w_qkv[l])   # once, before any timing
        del w_row
        q_rot = torch.empty((spec.batch, Hq, spec.head_dim), dtype=torch.float32, device="cuda")
    else:
        step_in = w.qkv

    def step_fn(qkv, seq_lens, positions, block_table, out_t):
        """One decode step (the rope table, then the L layers) on these buffers."""
        if not args.qkv:
            return layers.step_fn(qkv, seq_lens, positions, block_table, out_t)

        def fn():
            qdec.qdec_rope_table(shape, positions, rope, stream=stream)
            for l in range(L):
                qdec.qdec_qkv_append_rope(shape, qkv[l], w_qkv[l], w.w_q[l], w.w_k[l], positions,
                                          seq_lens, block_table, w.pool(l), q_rot, rope, err,
                                          stream=stream)
                qdec.qdec_attn_decode(shape, q_rot, w.pool(l), block_table, seq_lens, ws,
                                      out_t[l], err, stream=stream)
        return fn

    def graph_of(fn):
        if args.no_graph:
            with torch.cuda.stream(stream):
                fn()   # the first launch configures the kernels
            return fn
        return capture(fn, stream)

    run = graph_of(step_fn(step_in, w.seq_lens, w.positions, layers.block_table, out))

    # Steps whose inputs fit in L2 twice over are timed L2-cold: a buffer
    # larger than L2 is rewritten before each one, outside the timed steps.
    l2 = l2_bytes(dev)
    bytes_layer = (block_bytes_per_layer(w, args.hidden) if args.qkv
                   else w.algorithmic_bytes_per_layer())
    flush = l2_flush_buffer(bytes_layer * L, l2)

    # ---- device-timed region (clocks sampled during it)
    clocks = Clocks(dev)
    t_ms, t_ms_max, per = timed_steps(run, stream, args.steps, args.warmup, dist, flush, clocks)
    ck = clocks.stop()
    layers.check()
    t_steps_ms = sum(per)

    bytes_step = bytes_layer * L
    ms_step = t_ms_max / args.steps
    value = dist.world * bytes_step * args.steps / (t_ms_max * 1e-3) / 1e9
    # per attention launch, this rank: the whole step (table kernel included)
    # over its L launches, so an upper bound of the launch's duration
    launch_us = t_steps_ms / args.steps / L * 1e3
    achieved = bytes_layer / (launch_us * 1e-6) / 1e9
    per_layer = calls_per_layer(args)
    # qdec_step itself runs in one launch or (bf16 pool, flat layout) two
    step_launches = qdec.qdec_step_launches(layers.shape, w.kv == "fp8") if per_layer == 1 else 0
    mode = {1: "fused" if step_launches == 1 else "decode", 2: "decode", 3: "split"}[per_layer]
    launches_layer = max(per_layer, step_launches)
    roof_bytes, roof_kernel = bytes_layer, (f"attention_kernel<{mode}, fp8>" if w.kv == "fp8"
                                            else f"attention_kernel<{mode}>")
    roof_how = (f"CUDA events around each step's graph (rope table + {launches_layer * L} "
                f"launches, gaps included) / {L}"
                + (f": the {launches_layer} launches of a layer together" if launches_layer > 1
                   else ""))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.qkv:
        # the projection kernel alone: a graph of its L launches, timed the same way
        gq = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(gq, stream=stream):
                for l in range(L):
                    qdec.qdec_qkv_append_rope(shape, step_in[l], w_qkv[l], w.w_q[l], w.w_k[l],
                                              w.positions, w.seq_lens, layers.block_table,
                                              w.pool(l), q_rot, rope, err, stream=stream)
            for _ in range(3):
                gq.replay()
            e0.record(stream)
            reps = max(10, args.steps // 4)
            for _ in range(reps):
                gq.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        launch_us = e0.elapsed_time(e1) / reps / L * 1e3
        roof_bytes = qkv_weight_bytes(spec, args.hidden) + spec.batch * args.hidden * 2
        achieved = roof_bytes / (launch_us * 1e-6) / 1e9
        roof_kernel = "qkv_append_kernel"
        roof_how = f"CUDA events around a graph of {L} projection launches, {reps} replays"
    peak, peak_kind = measured_peaks()

    # ---- end to end, over as many steps as the device-timed region: every
    # step copies its new-token inputs and metadata in from pinned host
    # memory and its outputs back.  Two sets of device buffers: a step's
    # input copies and its output copy run on their own streams, overlapping
    # the neighbouring steps' kernels.
    meta = [w.seq_lens, w.positions, layers.block_table]
    qkv_h = step_in.cpu().pin_memory()
    meta_h = [m.cpu().pin_memory() for m in meta]
    h2d = qkv_h.numel() * qkv_h.element_size() + sum(m.numel() * m.element_size() for m in meta_h)
    d2h = out.numel() * out.element_size()
    k_e2e = 0 if args.no_e2e else args.steps
    if k_e2e:
        sets = []
        for j in range(2):
            qkv_d = torch.empty_like(step_in)
            meta_d = [torch.empty_like(m) for m in meta]
            out_d = torch.empty_like(out)
            for d, h in zip([qkv_d] + meta_d, [qkv_h] + meta_h):
                d.copy_(h)
            fn = graph_of(step_fn(qkv_d, meta_d[0], meta_d[1], meta_d[2], out_d))
            sets.append(dict(qkv=qkv_d, meta=meta_d, out=out_d, run=fn,
                             out_h=torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                             loaded=torch.cuda.Event(), done=torch.cuda.Event()))
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        def e2e_step(k):
            b = sets[k & 1]
            with torch.cuda.stream(s_in):   # inputs of step k (set free once step k-2 ran)
                s_in.wait_event(b["done"])
                b["qkv"].copy_(qkv_h, non_blocking=True)
                for d, h in zip(b["meta"], meta_h):
                    d.copy_(h, non_blocking=True)
                b["loaded"].record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(b["loaded"])
                b["run"]()
                b["done"].record(stream)
            with torch.cuda.stream(s_out):  # outputs of step k
                s_out.wait_event(b["done"])
                b["out_h"].copy_(b["out"], non_blocking=True)

        for k in range(max(3, args.warmup)):
            e2e_step(k)
        torch.cuda.synchronize()
        dist.barrier()
        torch.cuda.synchronize()
        e0.record(s_in)
        for k in range(k_e2e):
            e2e_step(k)
        e1.record(s_out)
        torch.cuda.synchronize()
        dist.barrier()
        t_e2e = dist.max(e0.elapsed_time(e1))
    e2e_value = dist.world * bytes_step * k_e2e / (t_e2e * 1e-3) / 1e9 if k_e2e else None
    layers.check()

    traffic = None
    tr = TRAFFIC.get(workload_name(spec, w.kv, args.hidden if args.qkv else 0, per_layer))
    if tr and tr["kernel_sha"] == kernel_sha("qkv_append_kernel" if args.qkv
                                             else "attention_kernel"):
        traffic = tr["bytes_per_launch"]

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline and args.qkv:
        w_cpu = wl.build(spec, "cpu", layers=min(spec.layers, CPU_SAMPLE_LAYERS), kv=w.kv)
        gbs, n, secs = oracle_qkv_sample(w_cpu, args.hidden, args.cpu_seconds)
        cpu = {"value": round(gbs, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} x one layer (all sequences) of the QKV block of "
                         f"{workload_name(spec, w.kv, args.hidden)} "
                         f"(layers 0-{w_cpu.spec.layers - 1}), fp64, {secs:.1f} s"}
        del w_cpu
    elif dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        # host copies of the sampled layers come from the GPU workload (the
        # pages each layer references); the oracle runs on the host cores
        gbs, what, n, secs = oracle_sample(w, args.cpu_seconds, per_seq=False)
        cpu = {"value": round(gbs, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} x {what} of {workload_name(spec, w.kv)}, fp64, {secs:.1f} s"}
        gbs_all, used, n_all, secs_all = oracle_sample_all_cores(w, args.cpu_seconds,
                                                                host_cores())
        cpu["all_cores"] = {
            "value": round(gbs_all, 6), "unit": "GB/s", "cores": used, "kind": "oracle",
            "sample": f"{n_all} x one layer, its sequences split into {used} groups of about "
                      f"equal length, one oracle call per group on its own thread "
                      f"({host_cores()} host cores), fp64, {secs_all:.1f} s"}

    cfg = workload_config(w, args, dist.world, l2)
    if step_launches == 2:
        cfg["launch"] += (" (qdec_step runs as two launches here: the new-token kernel, then the "
                          "decode-mode attention as its programmatic dependent"
                          + ("; over an FP8 pool the new-token kernel starts after the previous "
                             "layer's attention has finished)" if w.kv == "fp8" else ")"))
    if args.plan_bound:
        cfg["plan"] = (f"planned for contexts up to {args.plan_bound} tokens (block-table rows "
                       f"of {layers.shape.max_blocks_per_seq} pages)")
    configs = []
    if (not args.qkv and not args.layers and not args.no_configs and not args.pool_pages
            and per_layer == 1):
        # the other workloads of the benchmark plan, each on its own (the
        # headline's buffers are released first)
        del layers, run, w, step_in, flush
        if k_e2e:
            del sets
        capture.keep.clear()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        for wid in sorted(wl.WORKLOADS):
            if wid != args.workload:
                configs.append(config_record(qdec, wid, args, dist, dev, peak))

    if dist.rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("e4m3 KV (e4m3 q.k and f16 p.v mma, f32 accumulate)" if args.kv == "fp8"
                      else "bf16"),
            "data": ("synthetic (seeded N(0,1) bf16 hidden states, N(0,1/hidden) bf16 merged "
                     "QKV weights and KV pages)" if args.qkv else
                     "synthetic (seeded N(0,1) bf16 q/k/v and KV pages"
                     + (", pages cast to E4M3 with amax/448 scales)" if args.kv == "fp8"
                        else ")")),
            "us_per_layer_step": round(ms_step * 1e3 / L, 4),
            "us_per_layer_step_spread": step_spread(per, L),
            "pct_of_hbm_peak": round(100 * value / dist.world / peak, 2),
            "config": cfg,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_kind == "measured" else "fallback",
                         "kernel": roof_kernel,
                         "launch_us": round(launch_us, 3),
                         "launch_us_how": roof_how,
                         "bytes_per_launch": roof_bytes},
            "e2e": {"value": e2e_value and round(e2e_value, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": k_e2e},
            "gpu_launches": ((2 * L if args.qkv else launches_layer * L) + 1) * args.steps,
            "clocks": ck,
            "cpu_baseline": cpu,
        }
        if configs:
            line["configs"] = configs
        print(json.dumps(line), flush=True)


def prefill_flops(seq_lens, chunks, Hq=32, D=128) -> int:
    """Algorithmic FLOPs of the causal attention of the chunks: per head,
    query row at token index t and each of its t+1 keys, 2 D for q.k and 2 D
    for p v."""
    tot = 0
    for L, n in zip(seq_lens, chunks):
        t = np.arange(L - n, L, dtype=np.int64)
        tot += int((t + 1).sum())
    return 4 * D * Hq * tot


def prefill_config(P: int, L: int, fp8: bool, widen: bool = True) -> dict:
    """The `config` object of a --prefill line (the same for both arms)."""
    if not fp8:
        launch = (f"CUDA graph: qdec_prefill_rope_table, then {L} x (qdec_prefill_append_rope, "
                  "qdec_prefill_attn), the attention a programmatic dependent of the append")
    elif widen:
        launch = (f"CUDA graph: qdec_prefill_rope_table, then {L} x "
                  "(qdec_prefill_append_rope_fp8, qdec_prefill_attn_fp8 with a workspace: the "
                  "pages dequantized to bf16 once, then the attention as a programmatic "
                  "dependent of that pass)")
    else:
        launch = (f"CUDA graph: qdec_prefill_rope_table, then {L} x "
                  "(qdec_prefill_append_rope_fp8, qdec_prefill_attn_fp8 without a workspace: "
                  "the codes converted inside the attention kernel)")
    return {"workload": f"prefill-b1-prompt{P}-{L}layer" + ("-fp8kv" if fp8 else ""),
            "batch": 1, "prompt": P, "layers": L, "heads": "32 q / 8 kv, head_dim 128, page 16",
            "launch": launch,
            "l2": "not flushed (compute-bound: each layer's K/V is re-read from L2 "
                  "by its query blocks by design)"}


def oracle_prefill_sample(P: int, fp8: bool):
    """A bounded sample of a --prefill step for the fp64 oracle: one layer of
    a fresh prompt of min(P, 256) tokens (append, then causal attention).
    Returns (run, flops, tokens); run() executes it on a fresh copy of the
    pool, the inputs being made once."""
    import math

    import oracle
    Pc = min(P, 256)
    if fp8:
        c, codes_h, sc_h = wl.prefill_case_fp8([Pc], [Pc], seed=1000, device="cpu")
        pool0, sc = codes_h.numpy().copy(), sc_h.numpy()
    else:
        c = wl.prefill_case([Pc], [Pc], seed=1000, device="cpu", poison=False)
        pool0, sc = wl.bf16_bits(c.pool).copy(), None
    bt, qo, sl = c.block_table.numpy(), c.qo_indptr.numpy(), c.seq_lens.numpy()
    ins = (wl.bf16_bits(c.q), wl.bf16_bits(c.k), wl.bf16_bits(c.v), wl.bf16_bits(c.w_q),
           wl.bf16_bits(c.w_k), c.positions.numpy(), qo, sl, bt)
    eps, scale = float(np.float32(1e-6)), 1 / math.sqrt(128)

    def run():
        pool = pool0.copy()
        if fp8:
            res = oracle.prefill_append_fp8(*ins, pool, sc, 1e6, eps)
            oracle.prefill_attention_fp8(pool, sc, bt, qo, sl, res["q_rot"], scale)
        else:
            res = oracle.prefill_append(*ins, pool, 1e6, eps)
            oracle.prefill_attention(pool, bt, qo, sl, res["q_rot"], scale)
    return run, prefill_flops([Pc], [Pc]), Pc


def run_reference_prefill(args, dist: Dist):
    """The reference arm of --prefill: the oracle on the host, each step one
    bounded sample of the workload (see oracle_prefill_sample)."""
    if dist.rank != 0:
        return
    P, L, fp8 = args.prefill, args.layers or 36, args.kv == "fp8"
    run, flops, Pc = oracle_prefill_sample(P, fp8)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = args.steps * flops / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 9),
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": prefill_config(P, L, fp8),
        "cpu_baseline": {"value": round(value, 9), "unit": "TFLOP/s", "cores": 1,
                         "kind": "oracle",
                         "sample": f"{args.steps} steps of one layer of a fresh {Pc}-token "
                                   f"prompt (append + causal attention), {dt:.1f} s"},
        "e2e": {"value": round(value, 9), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0}), flush=True)


def run_prefill(args, dist: Dist):
    """Chunked prefill: per layer one fresh prompt of args.prefill tokens
    (qdec_prefill_append_rope, then qdec_prefill_attn) over that layer's pool;
    a step = all layers, one CUDA graph."""
    from gqa_paged_kv_gb300 import build as qbuild
    qbuild.build()
    from gqa_paged_kv_gb300 import qdec

    dev = dist.local
    torch.cuda.set_device(dev)
    P = args.prefill
    L = args.layers or 36
    fp8 = args.kv == "fp8"
    widen = fp8 and not args.fp8_in_kernel
    name = prefill_config(P, L, fp8)["workload"]
    if fp8:   # E4M3 codes and per-(page, plane, head) scales of the same draws
        made = [wl.prefill_case_fp8([P], [P], seed=1000 + l, device="cuda") for l in range(L)]
        cases = [m[0] for m in made]
        pools8 = [(m[1], m[2]) for m in made]
    else:
        cases = [wl.prefill_case([P], [P], seed=1000 + l, device="cuda", poison=False)
                 for l in range(L)]
    c0 = cases[0]
    shape = qdec.Shape(batch=1, num_pages=c0.num_pages, max_blocks_per_seq=c0.max_blocks,
                       max_seq_len=c0.max_blocks * 16,
                       launch_flags=0 if args.no_overlap else qdec.QDEC_LAUNCH_OVERLAP_PREVIOUS)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_rot = torch.empty((P, 32, 128), dtype=torch.float32, device="cuda")
    out = torch.empty((L, P, 32, 128), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    flops_layer = prefill_flops([P], [P])
    # one workspace serves every layer: each call's widening waits for the
    # calls before it on the stream
    ws8 = (torch.empty(qdec.qdec_prefill_fp8_workspace_bytes(shape), dtype=torch.uint8,
                       device="cuda") if widen else None)

    # the chunk rows' RoPE angles, once per step for all layers (the same
    # positions in every layer)
    rope = qdec.alloc_prefill_rope_table(P)

    def step_fn(ins, outs):
        def fn():
            qdec.qdec_prefill_rope_table(shape, c0.positions, rope, stream=stream)
            for l, c in enumerate(cases):
                q, k, v = ins[l]
                if fp8:
                    codes, sc = pools8[l]
                    qdec.qdec_prefill_append_rope_fp8(shape, q, k, v, c.w_q, c.w_k, c.positions,
                                                      c.qo_indptr, c.seq_lens, c.block_table,
                                                      codes, sc, q_rot, err, stream=stream,
                                                      rope_table=rope)
                    qdec.qdec_prefill_attn_fp8(shape, q_rot, c.qo_indptr, c.seq_lens,
                                               c.block_table, codes, sc, outs[l], err,
                                               stream=stream, workspace=ws8)
                    continue
                qdec.qdec_prefill_append_rope(shape, q, k, v, c.w_q, c.w_k, c.positions,
                                              c.qo_indptr, c.seq_lens, c.block_table, c.pool,
                                              q_rot, err, stream=stream, rope_table=rope)
                qdec.qdec_prefill_attn(shape, q_rot, c.qo_indptr, c.seq_lens, c.block_table,
                                       c.pool, outs[l], err, stream=stream)
        return fn

    def graph_of(fn):
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                fn()
        return g

    ins = [(c.q, c.k, c.v) for c in cases]
    g = graph_of(step_fn(ins, out))
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
    stream.synchronize()
    st, flags = qdec.qdec_check_error(err, stream)
    assert st == 0, f"device error flags {flags:#x}"

    clocks = Clocks(dev)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    ck = clocks.stop()
    t_ms = dist.max(e0.elapsed_time(e1))
    ms_step = t_ms / args.steps
    value = dist.world * flops_layer * L * args.steps / (t_ms * 1e-3) / 1e12

    # the attention kernel alone: a graph of its L launches.  Over an FP8 pool
    # with a workspace each layer gets its own workspace, dequantized once
    # beforehand by a full call, and the timed calls are told the pages are
    # ready; the full call (dequantizing pass + attention) is timed as well.
    def attn_graph(fn):
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g_, stream=stream):
                fn()
        return g_

    def time_graph(g_, reps):
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_.replay()
            e0.record(stream)
            for _ in range(reps):
                g_.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps / L * 1e3

    def attn_calls(shape_, wss):
        def fn():
            for l, c in enumerate(cases):
                if fp8:
                    qdec.qdec_prefill_attn_fp8(shape_, q_rot, c.qo_indptr, c.seq_lens,
                                               c.block_table, *pools8[l], out[l], err,
                                               stream=stream, workspace=wss[l])
                else:
                    qdec.qdec_prefill_attn(shape_, q_rot, c.qo_indptr, c.seq_lens, c.block_table,
                                           c.pool, out[l], err, stream=stream)
        return fn

    reps = max(5, args.steps // 4)
    call_us = None
    if widen:
        call_us = time_graph(attn_graph(attn_calls(shape, [ws8] * L)), reps)
        ws_l = [torch.empty_like(ws8) for _ in range(L)]
        with torch.cuda.stream(stream):
            attn_calls(shape, ws_l)()
        ready = dataclasses.replace(
            shape, launch_flags=shape.launch_flags | qdec.QDEC_LAUNCH_PREFILL_PAGES_READY)
        launch_us = time_graph(attn_graph(attn_calls(ready, ws_l)), reps)
        del ws_l
    else:
        launch_us = time_graph(attn_graph(attn_calls(shape, [None] * L)), reps)
    achieved = flops_layer / (launch_us * 1e-6) / 1e12
    peak, peak_kind = measured_bf16_tflops()

    # end to end: each step's chunk q/k/v from pinned host memory, out back
    k_e2e = 0 if args.no_e2e else max(1, args.steps // 4)
    h2d = sum(t.numel() * t.element_size() for trip in ins for t in trip)
    d2h = out.numel() * out.element_size()
    e2e_value = None
    if k_e2e:
        host = [tuple(t.cpu().pin_memory() for t in trip) for trip in ins]
        dev_in = [tuple(torch.empty_like(t) for t in trip) for trip in ins]
        out_d = torch.empty_like(out)
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        ge = graph_of(step_fn(dev_in, out_d))

        def e2e_step():
            with torch.cuda.stream(stream):
                for hs, ds in zip(host, dev_in):
                    for h_, d_ in zip(hs, ds):
                        d_.copy_(h_, non_blocking=True)
                ge.replay()
                out_h.copy_(out_d, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        dist.barrier()
        e0.record(stream)
        for _ in range(k_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        e2e_value = dist.world * flops_layer * L * k_e2e / (dist.max(e0.elapsed_time(e1)) * 1e-3) / 1e12
    st, flags = qdec.qdec_check_error(err, stream)
    assert st == 0, f"device error flags {flags:#x}"

    tr = TRAFFIC.get(name)   # over an FP8 pool: counters of the workspace form
    traffic = (tr["bytes_per_launch"]
               if tr and tr["kernel_sha"] == kernel_sha("prefill_attention_tc_kernel")
               and widen == fp8 else None)

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        run, flops, Pc = oracle_prefill_sample(P, fp8)
        n, secs = 0, 0.0
        while secs < args.cpu_seconds or n == 0:
            t0 = time.perf_counter()
            run()
            secs += time.perf_counter() - t0
            n += 1
        cpu = {"value": round(n * flops / secs / 1e12, 9), "unit": "TFLOP/s", "cores": 1,
               "kind": "oracle",
               "sample": f"{n} x one layer of a fresh {Pc}-token prompt (append + causal "
                         f"attention), fp64, {secs:.1f} s"}

    if dist.rank == 0:
        line = {
            "metric": PREFILL_METRIC, "value": round(value, 3), "unit": "TFLOP/s",
            "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 6), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("e4m3 KV dequantized once to bf16 (code x scale) in a workspace, then "
                      "the bf16-pool attention (tcgen05 kind::f16 with bf16 operands, f32 "
                      "accumulators in tensor memory)" if widen else
                      "e4m3 KV converted exactly to f16 in shared memory (tcgen05 kind::f16 "
                      "with f16 operands, f32 accumulators in tensor memory)" if fp8 else
                      "bf16 (tcgen05 kind::f16 with bf16 operands, q rounded once to bf16, f32 "
                      "accumulators in tensor memory)"),
            "data": "synthetic (seeded N(0,1) bf16 q/k/v, U(0.5,1.5) norm weights)",
            "us_per_layer_step": round(ms_step * 1e3 / L, 3),
            "config": prefill_config(P, L, fp8, widen),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops, cuBLAS "
                                      f"burst)" if peak_kind == "measured" else "fallback",
                         "kernel": ("prefill_attention_tc_kernel<widened>"
                                    if widen else "prefill_attention_tc_kernel<fp8>" if fp8
                                    else "prefill_attention_tc_kernel<bf16>"),
                         "launch_us": round(launch_us, 3),
                         "launch_us_how": f"CUDA events around a graph of {L} attention "
                                          f"launches, {reps} replays" +
                                          (" (each layer's pages dequantized beforehand into "
                                           "its own workspace)" if widen else ""),
                         "call_us": call_us and round(call_us, 3),
                         "call_us_how": ("the same graph of full qdec_prefill_attn_fp8 calls "
                                         "(dequantizing pass + attention) on one shared "
                                         "workspace" if widen else None),
                         "flops_per_launch": flops_layer},
            "e2e": {"value": e2e_value and round(e2e_value, 3), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k_e2e},
            "gpu_launches": ((3 if widen else 2) * L + 1) * args.steps,
            "clocks": ck,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    dist = Dist()
    try:
        if args.impl == "reference":
            if args.prefill:
                run_reference_prefill(args, dist)
            else:
                run_reference(args, dist)
        elif args.prefill:
            run_prefill(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
