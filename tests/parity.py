"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI, run the oracle on the same seeded inputs, compare element by element.

Tolerances (stated for bf16 outputs of an fp32 pipeline against fp64):
  out     |gpu - ref| <= 2e-2 + 1e-2 |ref|        (ref: unrounded double)
  k slot  |gpu - ref| <= 1 bf16 ulp of ref         (ref: unrounded k_rot)
  v slot  bit-equal to the input v
  q_rot   |gpu - ref| <= 2e-5 (1 + |ref|)          (fp32 output, unrounded)
FP8 (E4M3) pools: the same out tolerance (the oracle attends over the exact
dequantized values, so only the kernel's arithmetic is measured); the K and V
codes of every appended slot bit-equal to the oracle's (both sides divide in
fp32 and round to E4M3 nearest-even with saturation).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from gqa_paged_kv_gb300 import workloads as wl

OUT_ATOL, OUT_RTOL = 2e-2, 1e-2
QROT_TOL = 2e-5


def qdec():
    from gqa_paged_kv_gb300 import qdec as q
    return q


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits, min normal 2^-126)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_bits_to_f64(wl.bf16_bits(t))


class Runner:
    """Device buffers for running a workload's layers through qdec_step."""

    def __init__(self, w: wl.Workload, num_ctas: int = 0, rope: bool = True,
                 overlap: bool = False):
        q = qdec()
        self.w = w
        self.shape = q.shape_for(w, num_ctas=num_ctas,
                                 launch_flags=q.QDEC_LAUNCH_OVERLAP_PREVIOUS if overlap else 0)
        self.ws = q.alloc_workspace(self.shape)
        self.rope = None
        if rope:
            self.rope = q.alloc_rope_table(self.shape)
            q.qdec_rope_table(self.shape, w.positions, self.rope)
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        s = w.spec
        self.out = torch.empty((s.layers, s.batch, s.num_q_heads, s.head_dim),
                               dtype=torch.bfloat16, device="cuda")
        self.q_rot = torch.empty((s.batch, s.num_q_heads, s.head_dim), dtype=torch.float32,
                                 device="cuda")

    def step(self, layer: int):
        q, w = qdec(), self.w
        if w.kv == "fp8":
            q.qdec_step_fp8(self.shape, w.q(layer), w.k(layer), w.v(layer), w.w_q[layer],
                            w.w_k[layer], w.positions, w.seq_lens, w.block_table, w.pool8(layer),
                            w.scale(layer), self.ws, self.out[layer], self.err,
                            rope_table=self.rope)
            return
        q.qdec_step(self.shape, w.q(layer), w.k(layer), w.v(layer), w.w_q[layer], w.w_k[layer],
                    w.positions, w.seq_lens, w.block_table, w.pool(layer), self.ws,
                    self.out[layer], self.err, rope_table=self.rope)

    def unfused(self, layer: int):
        q, w = qdec(), self.w
        if w.kv == "fp8":
            q.qdec_append_rope_fp8(self.shape, w.q(layer), w.k(layer), w.v(layer), w.w_q[layer],
                                   w.w_k[layer], w.positions, w.seq_lens, w.block_table,
                                   w.pool8(layer), w.scale(layer), self.q_rot, self.err,
                                   rope_table=self.rope)
            q.qdec_attn_split_fp8(self.shape, self.q_rot, w.pool8(layer), w.scale(layer),
                                  w.block_table, w.seq_lens, self.ws, self.out[layer], self.err)
        else:
            q.qdec_append_rope(self.shape, w.q(layer), w.k(layer), w.v(layer), w.w_q[layer],
                               w.w_k[layer], w.positions, w.seq_lens, w.block_table,
                               w.pool(layer), self.q_rot, self.err, rope_table=self.rope)
            q.qdec_attn_split(self.shape, self.q_rot, w.pool(layer), w.block_table, w.seq_lens,
                              self.ws, self.out[layer], self.err)
        q.qdec_attn_merge(self.shape, w.seq_lens, self.ws, self.out[layer], self.err)

    def two_calls(self, layer: int):
        """Steps 1-3 (qdec_append_rope) and then step 4 in one launch
        (qdec_attn_decode)."""
        q, w = qdec(), self.w
        if w.kv == "fp8":
            q.qdec_append_rope_fp8(self.shape, w.q(layer), w.k(layer), w.v(layer), w.w_q[layer],
                                   w.w_k[layer], w.positions, w.seq_lens, w.block_table,
                                   w.pool8(layer), w.scale(layer), self.q_rot, self.err,
                                   rope_table=self.rope)
            q.qdec_attn_decode_fp8(self.shape, self.q_rot, w.pool8(layer), w.scale(layer),
                                   w.block_table, w.seq_lens, self.ws, self.out[layer], self.err)
        else:
            q.qdec_append_rope(self.shape, w.q(layer), w.k(layer), w.v(layer), w.w_q[layer],
                               w.w_k[layer], w.positions, w.seq_lens, w.block_table,
                               w.pool(layer), self.q_rot, self.err, rope_table=self.rope)
            q.qdec_attn_decode(self.shape, self.q_rot, w.pool(layer), w.block_table, w.seq_lens,
                               self.ws, self.out[layer], self.err)

    def check_flags(self):
        st, flags = qdec().qdec_check_error(self.err)
        assert st == 0 and flags == 0, f"device error flags {flags:#x} (status {st})"


def run_oracle(inputs: dict) -> dict:
    """One layer on the oracle; `inputs` from workloads.oracle_inputs (pool copied)."""
    pool = inputs["pool"].copy()
    args = (inputs["q"], inputs["k"], inputs["v"], inputs["w_q"], inputs["w_k"],
            inputs["positions"], inputs["seq_lens"], inputs["block_table"], pool)
    if "kv_scale" in inputs:
        res = oracle.decode_layer_fp8(*args, inputs["kv_scale"], inputs["rope_theta"],
                                      float(np.float32(inputs["eps"])))
    else:
        res = oracle.decode_layer(*args, inputs["rope_theta"], float(np.float32(inputs["eps"])))
    res["pool_after"] = pool
    res["block_table"] = inputs["block_table"]
    return res


def assert_out_close(gpu: torch.Tensor, ref: np.ndarray, what: str = "out"):
    g = to_f64(gpu)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements out of tolerance, "
                           f"max err {err.max():.3e}")
    return float(err.max())


def assert_slots(w: wl.Workload, layer: int, seqs, res: dict):
    """The appended k rows are within 1 bf16 ulp of the unrounded oracle k_rot
    and the v rows carry v's bits; returns the count of k elements that are
    not bit-identical to the oracle's own rounding."""
    s = w.spec
    P = s.page_size
    pool = w.pool(layer)
    v_in = wl.bf16_bits(w.v(layer))
    not_exact = 0
    for i, b in enumerate(seqs):
        L = int(w.seq_lens_host[b])
        page = int(w.block_table_host[b, (L - 1) // P])
        row = wl.bf16_bits(pool[page, :, :, (L - 1) % P, :])       # [2][Hkv][D]
        k_ref = res["k_rot"][i]
        k_gpu = oracle.bf16_bits_to_f64(row[0])
        assert np.all(np.abs(k_gpu - k_ref) <= bf16_ulp(k_ref)), f"k slot seq {b}"
        not_exact += int(np.sum(row[0] != oracle.f64_to_bf16_bits(k_ref)))
        assert np.array_equal(row[1], v_in[b]), f"v slot seq {b}"
    assert not_exact == 0, f"{not_exact} k elements differ from the oracle's rounding"
    return not_exact


def assert_slots_fp8(w: wl.Workload, layer: int, seqs, res: dict):
    """The appended K and V codes of every (sequence, KV head) equal the
    oracle's (both quantize fp32(row) / scale with E4M3 nearest-even)."""
    P = w.spec.page_size
    pool = w.pool8(layer)
    for i, b in enumerate(seqs):
        L = int(w.seq_lens_host[b])
        page = int(w.block_table_host[b, (L - 1) // P])
        gpu = pool[page, :, :, (L - 1) % P, :].cpu().numpy()            # [2][Hkv][D] codes
        ref = res["pool_after"][res["block_table"][i, (L - 1) // P], :, :, (L - 1) % P, :]
        bad = np.argwhere(gpu != ref)
        assert bad.size == 0, (f"seq {b}: {len(bad)} slot codes differ, first "
                               f"(plane, head, dim) {tuple(bad[0])}: gpu {gpu[tuple(bad[0])]:#x} "
                               f"oracle {ref[tuple(bad[0])]:#x}")


def assert_slots_for(w: wl.Workload, layer: int, seqs, res: dict):
    """The appended slots, checked the way the workload's pool type defines them."""
    if w.kv == "fp8":
        return assert_slots_fp8(w, layer, seqs, res)
    return assert_slots(w, layer, seqs, res)


def step_call(shape, w: wl.Workload, layer: int, ws, out, err, rope=None):
    """One qdec_step / qdec_step_fp8 launch of `layer` with the given shape and buffers."""
    q = qdec()
    if w.kv == "fp8":
        q.qdec_step_fp8(shape, w.q(layer), w.k(layer), w.v(layer), w.w_q[layer], w.w_k[layer],
                        w.positions, w.seq_lens, w.block_table, w.pool8(layer), w.scale(layer),
                        ws, out, err, rope_table=rope)
    else:
        q.qdec_step(shape, w.q(layer), w.k(layer), w.v(layer), w.w_q[layer], w.w_k[layer],
                    w.positions, w.seq_lens, w.block_table, w.pool(layer), ws, out, err,
                    rope_table=rope)
