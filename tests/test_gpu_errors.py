"""Device-side failure handling through the C ABI (marked gpu).

Bad block-table entries and sequence lengths are skipped and reported
through the error flag without a fault, the other sequences stay exact; a
wait that runs out (the withheld-tile test hook: a copy that is never
issued) ends the launch with a timeout status after a short budget, and the
next launch on the same device is exact again.  Every case runs on a bf16
and on an FP8 pool.
"""
import numpy as np
import pytest
import torch

from gqa_paged_kv_gb300 import workloads as wl
import parity

pytestmark = pytest.mark.gpu


KV = pytest.mark.parametrize("kv", ["bf16", "fp8"])


def _small(lens, seed, kv):
    pages = sum((l + 15) // 16 for l in lens) + 9
    spec = wl.custom(len(lens), lens, pool_pages=pages, seed=seed)
    return wl.build(spec, "cuda", poison=True, kv=kv)


@KV
@pytest.mark.parametrize("num_ctas", [0, 7], ids=["auto", "flat7"])
@pytest.mark.parametrize("bad_entry", [-1, 10 ** 6], ids=["negative", "beyond_pool"])
def test_bad_block_table_entry_is_flagged(num_ctas, bad_entry, kv):
    q = parity.qdec()
    w = _small([300, 200, 150], seed=41, kv=kv)
    good = [0, 2]
    ref = parity.run_oracle(wl.oracle_inputs(w, 0, good))
    w.block_table[1, 3] = bad_entry               # a middle page of sequence 1 (device copy)
    r = parity.Runner(w, num_ctas=num_ctas)
    r.step(0)
    st, flags = q.qdec_check_error(r.err)
    assert st == q.QDEC_ERR_DEVICE_BOUNDS and flags & q.QDEC_FLAG_BAD_PAGE, (st, flags)
    parity.assert_out_close(r.out[0][good], ref["out"])
    parity.assert_slots_for(w, 0, good, ref)


@KV
@pytest.mark.parametrize("num_ctas", [0, 7], ids=["auto", "flat7"])
@pytest.mark.parametrize("bad_len", [0, -5, 10 ** 6], ids=["zero", "negative", "too_long"])
def test_bad_sequence_length_is_flagged(num_ctas, bad_len, kv):
    q = parity.qdec()
    w = _small([300, 200, 150], seed=42, kv=kv)
    good = [0, 2]
    ref = parity.run_oracle(wl.oracle_inputs(w, 0, good))
    w.seq_lens[1] = bad_len                       # device copy only
    r = parity.Runner(w, num_ctas=num_ctas)
    r.step(0)
    st, flags = q.qdec_check_error(r.err)
    assert st == q.QDEC_ERR_DEVICE_BOUNDS and flags & q.QDEC_FLAG_BAD_SEQLEN, (st, flags)
    parity.assert_out_close(r.out[0][good], ref["out"])
    parity.assert_slots_for(w, 0, good, ref)


@KV
@pytest.mark.parametrize("num_ctas", [0, 5], ids=["auto", "flat5"])
def test_wait_that_runs_out_returns_timeout_and_device_stays_usable(num_ctas, kv):
    q = parity.qdec()
    w = _small([17, 1, 300, 64, 999], seed=43, kv=kv)
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w, num_ctas=num_ctas)
    shape = q.shape_for(w, num_ctas=num_ctas, launch_flags=q.QDEC_LAUNCH_TEST_WITHHOLD_TILE)
    ws = q.alloc_workspace(shape)
    out = torch.empty_like(r.out[0])
    parity.step_call(shape, w, 0, ws, out, r.err, r.rope)
    st, flags = q.qdec_check_error(r.err)
    assert st == q.QDEC_ERR_TIMEOUT and flags & q.QDEC_FLAG_TIMEOUT, (st, flags)
    # the same device, the normal launch: exact again
    r.step(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots_for(w, 0, range(5), ref)
