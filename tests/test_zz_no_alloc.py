"""qdec_step_static_scratch: the entry point for callers that cannot
allocate device memory (it uses the library's own fixed scratch array as the
workspace).  Its output must match qdec_step's on the same inputs, on two
calls in a row (the second one finds the first one's leftovers in the array).

This file is collected last on purpose, so that a failure here comes after
every other test has run; it also passes run alone in a fresh process."""
import pytest
import torch

from gqa_paged_kv_gb300 import workloads as wl
import parity

pytestmark = pytest.mark.gpu


def _run(lens, seed, num_ctas=0):
    from gqa_paged_kv_gb300 import qdec
    spec = wl.custom(len(lens), lens, pool_pages=sum((l + 15) // 16 for l in lens) + 5,
                     seed=seed)
    w_ref = wl.build(spec, "cuda", poison=True)
    w_new = wl.build(spec, "cuda", poison=True)   # same seed: identical inputs and pool
    shape = qdec.shape_for(w_ref, num_ctas=num_ctas)
    assert qdec.qdec_workspace_bytes(shape) <= qdec.QDEC_STATIC_SCRATCH_BYTES
    rope = qdec.alloc_rope_table(shape)
    qdec.qdec_rope_table(shape, w_ref.positions, rope)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    ws = qdec.alloc_workspace(shape)
    ref = torch.empty((w_ref.spec.batch, 32, 128), dtype=torch.bfloat16, device="cuda")
    qdec.qdec_step(shape, w_ref.q(0), w_ref.k(0), w_ref.v(0), w_ref.w_q[0], w_ref.w_k[0],
                   w_ref.positions, w_ref.seq_lens, w_ref.block_table, w_ref.pool(0), ws, ref,
                   err, rope_table=rope)
    outs = []
    for _ in range(2):
        out = torch.full((w_new.spec.batch, 32, 128), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        qdec.qdec_step_static_scratch(shape, w_new.q(0), w_new.k(0), w_new.v(0), w_new.w_q[0],
                                      w_new.w_k[0], w_new.positions, w_new.seq_lens,
                                      w_new.block_table, w_new.pool(0), out, err,
                                      rope_table=rope)
        outs.append(out)
    st, flags = qdec.qdec_check_error(err)
    assert st == 0 and flags == 0, f"device error {flags:#x} (status {st})"
    refd = parity.to_f64(ref)
    for out in outs:
        got = parity.to_f64(out)
        assert ((got - refd).__abs__() <= parity.OUT_ATOL + parity.OUT_RTOL * abs(refd)).all()
    # the appended key/value slots are bit-identical too (NaN poison compared as bits)
    assert torch.equal(w_ref.pool(0).view(torch.int16), w_new.pool(0).view(torch.int16))


@pytest.mark.parametrize("lens,num_ctas", [([17, 1, 300, 64, 16, 2, 999], 0),
                                           ([1000, 3, 2000], 9), ([513], 0)])
def test_static_scratch_matches_qdec_step_twice(lens, num_ctas):
    _run(lens, seed=31, num_ctas=num_ctas)


def test_static_scratch_rejects_shapes_beyond_its_size():
    from gqa_paged_kv_gb300 import qdec
    big = qdec.Shape(batch=1024, num_pages=1 << 20, max_blocks_per_seq=1024,
                     max_seq_len=16384)
    assert qdec.qdec_workspace_bytes(big) > qdec.QDEC_STATIC_SCRATCH_BYTES
    t = torch.empty((1024, 48, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qdec.QdecError) as e:
        qdec.qdec_step_static_scratch(big, t[:, :32], t[:, 32:40], t[:, 40:], t[0, 0],
                                      t[0, 1], t[0, 0], t[0, 0], t[0, 0], t, t)
    assert e.value.status == qdec.QDEC_ERR_WORKSPACE
