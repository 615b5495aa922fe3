"""qdec_step_static_scratch: the entry point for callers that cannot
allocate device memory (it uses the library's own fixed scratch array as the
workspace).  qdec_step is deterministic for a given shape, and this entry
point runs the same kernel with the same plan, so its output must equal
qdec_step's bit for bit on the same inputs: on two calls in a row, after a
call that gave up waiting (timeout test hook), and after a call of another
shape that left partial results where this call keeps its arrival counters
(which only the per-call clearing puts back to zero).

This file is collected last on purpose, so that a failure here comes after
every other test has run; it also passes run alone in a fresh process."""
import dataclasses

import pytest
import torch

from gqa_paged_kv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _qdec():
    from gqa_paged_kv_gb300 import qdec
    return qdec


class _Pair:
    """Two identical copies of one seeded workload (same seed: same inputs
    and pool); qdec_step runs on the first with a workspace it owns."""

    def __init__(self, lens, seed, num_ctas=0):
        q = _qdec()
        spec = wl.custom(len(lens), lens, pool_pages=sum((l + 15) // 16 for l in lens) + 5,
                         seed=seed)
        self.ref_w = wl.build(spec, "cuda", poison=True)
        self.new_w = wl.build(spec, "cuda", poison=True)
        self.shape = q.shape_for(self.ref_w, num_ctas=num_ctas)
        assert q.qdec_workspace_bytes(self.shape) <= q.QDEC_STATIC_SCRATCH_BYTES
        self.rope = q.alloc_rope_table(self.shape)
        q.qdec_rope_table(self.shape, self.ref_w.positions, self.rope)
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = q.alloc_workspace(self.shape)
        self.ref = self._out()
        w = self.ref_w
        q.qdec_step(self.shape, w.q(0), w.k(0), w.v(0), w.w_q[0], w.w_k[0], w.positions,
                    w.seq_lens, w.block_table, w.pool(0), ws, self.ref, self.err,
                    rope_table=self.rope)
        self.check(0)

    def _out(self):
        return torch.full((self.ref_w.spec.batch, 32, 128), float("nan"), dtype=torch.bfloat16,
                          device="cuda")

    def static(self, shape=None):
        """One qdec_step_static_scratch call on the second copy."""
        q = _qdec()
        w, out = self.new_w, self._out()
        q.qdec_step_static_scratch(shape or self.shape, w.q(0), w.k(0), w.v(0), w.w_q[0],
                                   w.w_k[0], w.positions, w.seq_lens, w.block_table, w.pool(0),
                                   out, self.err, rope_table=self.rope)
        return out

    def check(self, want_status):
        st, flags = _qdec().qdec_check_error(self.err)
        assert st == want_status, f"status {st}, flags {flags:#x}"

    def assert_equal(self, out):
        assert torch.equal(out.view(torch.int16), self.ref.view(torch.int16)), \
            "static-scratch output differs from qdec_step's"
        # the appended key/value slots are bit-identical too (NaN poison as bits)
        assert torch.equal(self.ref_w.pool(0).view(torch.int16),
                           self.new_w.pool(0).view(torch.int16))


@pytest.mark.parametrize("lens,num_ctas", [([17, 1, 300, 64, 16, 2, 999], 0),
                                           ([1000, 3, 2000], 9), ([513], 0)])
def test_static_scratch_matches_qdec_step_twice(lens, num_ctas):
    p = _Pair(lens, seed=31, num_ctas=num_ctas)
    outs = [p.static(), p.static()]
    p.check(0)
    for out in outs:
        p.assert_equal(out)


def test_static_scratch_after_a_call_that_timed_out():
    """A call whose first page tile is withheld gives up (QDEC_ERR_TIMEOUT);
    the next call through the same array is exact."""
    q = _qdec()
    p = _Pair([1000, 3, 2000, 40], seed=32, num_ctas=11)
    hooked = dataclasses.replace(p.shape, launch_flags=q.QDEC_LAUNCH_TEST_WITHHOLD_TILE)
    p.static(hooked)
    p.check(q.QDEC_ERR_TIMEOUT)
    out = p.static()
    p.check(0)
    p.assert_equal(out)


def test_static_scratch_after_a_call_that_left_partials_where_counters_go():
    """A one-sequence 8192-token call leaves split partials (their
    log-sum-exp values) 256 bytes into the array; a 16-sequence call on the
    flat layout keeps its 128 arrival counters in the first 512 bytes, so
    its counters start from those leftovers unless the call clears them."""
    first = _Pair([8192], seed=33)
    first.static()
    first.check(0)
    p = _Pair([17, 999, 300, 64, 16, 2, 513, 700, 1, 33, 250, 480, 96, 128, 1500, 45],
              seed=34, num_ctas=37)
    assert p.shape.batch * 8 * 4 > 256
    out = p.static()
    p.check(0)
    p.assert_equal(out)


def test_static_scratch_rejects_shapes_beyond_its_size():
    q = _qdec()
    big = q.Shape(batch=1024, num_pages=1 << 20, max_blocks_per_seq=1024, max_seq_len=16384)
    assert q.qdec_workspace_bytes(big) > q.QDEC_STATIC_SCRATCH_BYTES
    t = torch.empty((1024, 48, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q.QdecError) as e:
        q.qdec_step_static_scratch(big, t[:, :32], t[:, 32:40], t[:, 40:], t[0, 0],
                                   t[0, 1], t[0, 0], t[0, 0], t[0, 0], t, t)
    assert e.value.status == q.QDEC_ERR_WORKSPACE
