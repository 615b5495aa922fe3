"""Edge cases of the fused step against the oracle (marked gpu): the largest
batch the kernels take, a long context, RoPE positions other than L-1, and
rope_theta / eps / sm_scale other than the defaults, on bf16 and FP8 pools.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gqa_paged_kv_gb300 import workloads as wl
import parity

pytestmark = pytest.mark.gpu


KV = pytest.mark.parametrize("kv", ["bf16", "fp8"])


def _build(lens, seed, kv):
    pages = sum((l + 15) // 16 for l in lens) + 9
    spec = wl.custom(len(lens), lens, pool_pages=pages, seed=seed)
    return wl.build(spec, "cuda", poison=True, kv=kv)


@KV
@pytest.mark.parametrize("num_ctas", [0, 304], ids=["auto", "flat304"])
def test_largest_batch_1024_short_ragged(num_ctas, kv):
    rng = np.random.default_rng(51)
    lens = [int(x) for x in rng.integers(1, 41, size=1024)]
    w = _build(lens, seed=51, kv=kv)
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w, num_ctas=num_ctas)
    r.step(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots_for(w, 0, range(1024), ref)


@KV
def test_long_context_65536_tokens(kv):
    w = _build([65536], seed=52, kv=kv)
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w)
    r.step(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots_for(w, 0, [0], ref)


@KV
@pytest.mark.parametrize("rope", [True, False], ids=["rope_table", "in_kernel_angles"])
def test_positions_other_than_last_slot(rope, kv):
    w = _build([300, 17, 1000, 64], seed=53, kv=kv)
    w.positions.copy_(torch.tensor([0, 16383, 7, 123457], dtype=torch.int32))
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w, rope=rope)
    r.step(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots_for(w, 0, range(4), ref)


@KV
@pytest.mark.parametrize("theta,eps,scale", [(1.0e4, 1.0e-5, 0.05), (5.0e5, 1.0e-6, 0.2)])
def test_rope_theta_eps_and_scale_arguments(theta, eps, scale, kv):
    q = parity.qdec()
    w = _build([300, 17, 1000, 64], seed=54, kv=kv)
    inp = wl.oracle_inputs(w, 0)
    pool = inp["pool"].copy()
    args = (inp["q"], inp["k"], inp["v"], inp["w_q"], inp["w_k"], inp["positions"],
            inp["seq_lens"], inp["block_table"], pool)
    rest = (theta, float(np.float32(eps)), float(np.float32(scale)))
    if kv == "fp8":
        ref = oracle.decode_layer_fp8(*args, inp["kv_scale"], *rest)
    else:
        ref = oracle.decode_layer(*args, *rest)
    ref["pool_after"] = pool
    ref["block_table"] = inp["block_table"]
    shape = dataclasses.replace(q.shape_for(w), rope_theta=theta, eps=eps, sm_scale=scale)
    ws = q.alloc_workspace(shape)
    rope = q.alloc_rope_table(shape)
    q.qdec_rope_table(shape, w.positions, rope)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((4, 32, 128), dtype=torch.bfloat16, device="cuda")
    parity.step_call(shape, w, 0, ws, out, err, rope)
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0
    parity.assert_out_close(out, ref["out"])
    parity.assert_slots_for(w, 0, range(4), ref)
