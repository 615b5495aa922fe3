"""Chunked prefill through the C ABI (marked gpu), against the oracle.

Each case appends a chunk of new tokens per sequence (qdec_prefill_append_rope)
and runs the causal paged attention of the chunk (qdec_prefill_attn); the
oracle runs the same two steps in fp64 on a host copy of the pool taken before
the append.  Checked: q_rot within the fp32 tolerance 2e-5 (1 + |ref|); every
appended key within 1 bf16 ulp of the oracle's unrounded k_rot and every
appended value bit-equal to v; out within 2e-2 + 1e-2 |ref|; nothing outside
the chunk's slots written.  Pools are NaN-poisoned past every sequence's last
token.  Cases: fresh prompts (no cached prefix), chunks after a cached prefix,
chunks that start and end inside a page and across many pages, chunks of one
token (equal to the decode step), empty chunks, ragged batches, positions
that differ from the token index, and malformed chunks (flagged, skipped).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gqa_paged_kv_gb300 import workloads as wl
import parity

pytestmark = pytest.mark.gpu


def _shape(c, B, launch_flags=0):
    q = parity.qdec()
    return q.Shape(batch=B, num_pages=c.num_pages, max_blocks_per_seq=c.max_blocks,
                   max_seq_len=c.max_blocks * 16, launch_flags=launch_flags)


def _run(c, B):
    q = parity.qdec()
    shape = _shape(c, B)
    T = c.q.shape[0]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_rot = torch.empty((T, 32, 128), dtype=torch.float32, device="cuda")
    out = torch.full((T, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    q.qdec_prefill_append_rope(shape, c.q, c.k, c.v, c.w_q, c.w_k, c.positions, c.qo_indptr,
                               c.seq_lens, c.block_table, c.pool, q_rot, err)
    q.qdec_prefill_attn(shape, q_rot, c.qo_indptr, c.seq_lens, c.block_table, c.pool, out, err)
    return q_rot, out, err


def _oracle(c):
    pool = wl.bf16_bits(c.pool).copy()
    res = oracle.prefill_append(wl.bf16_bits(c.q), wl.bf16_bits(c.k), wl.bf16_bits(c.v),
                                wl.bf16_bits(c.w_q), wl.bf16_bits(c.w_k),
                                c.positions.cpu().numpy(), c.qo_indptr.cpu().numpy(),
                                c.seq_lens.cpu().numpy(), c.block_table.cpu().numpy(), pool,
                                1e6, float(np.float32(1e-6)))
    out, _ = oracle.prefill_attention(pool, c.block_table.cpu().numpy(),
                                      c.qo_indptr.cpu().numpy(), c.seq_lens.cpu().numpy(),
                                      res["q_rot"], 1 / math.sqrt(128))
    res["out"], res["pool_after"] = out, pool
    return res


def _check(c, res, q_rot, out, pool_before):
    g = q_rot.double().cpu().numpy()
    qerr = np.abs(g - res["q_rot"])
    assert np.all(qerr <= parity.QROT_TOL * (1 + np.abs(res["q_rot"]))), qerr.max()
    parity.assert_out_close(out, res["out"])
    got = wl.bf16_bits(c.pool)
    qo, L = c.qo_indptr.cpu().numpy(), c.seq_lens.cpu().numpy()
    bt = c.block_table.cpu().numpy()
    changed = np.zeros(got.shape, bool)
    v_in = wl.bf16_bits(c.v)
    for b in range(len(L)):
        n = qo[b + 1] - qo[b]
        for j in range(n):
            r, t = qo[b] + j, L[b] - n + j
            page, off = bt[b, t // 16], t % 16
            k_ref = res["k_rot"][r]
            k_gpu = oracle.bf16_bits_to_f64(got[page, 0, :, off])
            assert np.all(np.abs(k_gpu - k_ref) <= parity.bf16_ulp(k_ref)), f"k slot row {r}"
            # and it is the nearest-even bf16 of the oracle's value, as in decode
            assert np.array_equal(got[page, 0, :, off], oracle.f64_to_bf16_bits(k_ref)), \
                f"k slot row {r} not the oracle's rounding"
            assert np.array_equal(got[page, 1, :, off], v_in[r]), f"v slot row {r}"
            changed[page, :, :, off] = True
    same = (got == pool_before) | (np.isnan(oracle.bf16_bits_to_f64(got)) &
                                   np.isnan(oracle.bf16_bits_to_f64(pool_before)))
    assert same[~changed].all(), "the append wrote outside the chunk's slots"


CASES = [
    ([37], [37]),                                  # a fresh prompt, ragged last page
    ([16], [16]),                                  # exactly one page
    ([300, 17, 1000], [20, 17, 1]),                # after a cached prefix; fresh; one token
    ([64, 65, 31], [48, 1, 15]),                   # chunks ending on / after / before a page edge
    ([500, 40, 77, 250], [0, 40, 33, 0]),          # empty chunks
    ([2048], [256]),                               # a long prefix and a multi-block chunk
    ([int(x) for x in np.random.default_rng(9).integers(1, 400, size=12)],
     [int(x) for x in np.random.default_rng(10).integers(0, 40, size=12)]),
]


@pytest.mark.parametrize("seq_lens,chunks", CASES, ids=lambda x: str(x)[:40])
def test_prefill_matches_oracle(seq_lens, chunks):
    chunks = [min(n, L) for L, n in zip(seq_lens, chunks)]
    c = wl.prefill_case(seq_lens, chunks, seed=sum(seq_lens) % 97)
    before = wl.bf16_bits(c.pool).copy()
    res = _oracle(c)
    q_rot, out, err = _run(c, len(seq_lens))
    st, flags = parity.qdec().qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    _check(c, res, q_rot, out, before)


def test_prefill_positions_differ_from_token_index():
    c = wl.prefill_case([90, 33], [30, 33], seed=5, pos_offset=1000)
    before = wl.bf16_bits(c.pool).copy()
    res = _oracle(c)
    q_rot, out, err = _run(c, 2)
    st, flags = parity.qdec().qdec_check_error(err)
    assert st == 0 and flags == 0
    _check(c, res, q_rot, out, before)


def test_prefill_chunk_of_one_equals_decode():
    """One token per sequence: the prefill pair gives the decode path's
    output (same q_rot).  The prefill kernel carries the softmax weights as
    bf16 (decode: bf16 hi + lo), so the two differ by at most about
    2^-9 max|v| (<= 8e-3 here) besides the final bf16 rounding."""
    q = parity.qdec()
    c = wl.prefill_case([300, 17, 1000, 64], [1, 1, 1, 1], seed=11)
    shape = _shape(c, 4)
    q_rot, out, err = _run(c, 4)
    ws = q.alloc_workspace(shape)
    out_d = torch.empty_like(out)
    q.qdec_attn_decode(shape, q_rot, c.pool, c.block_table, c.seq_lens, ws, out_d, err)
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0
    assert torch.allclose(out.float(), out_d.float(), rtol=2 ** -7, atol=8e-3)


def test_prefill_malformed_chunk_is_flagged():
    """A chunk longer than its sequence is skipped and flagged; the others
    are exact."""
    q = parity.qdec()
    c = wl.prefill_case([40, 50, 60], [10, 20, 30], seed=12)
    good = wl.prefill_case([40, 50, 60], [10, 20, 30], seed=12)
    res = _oracle(good)
    c.seq_lens[1] = 15                                  # chunk of 20 in 15 tokens (device copy)
    q_rot, out, err = _run(c, 3)
    st, flags = q.qdec_check_error(err)
    assert st == q.QDEC_ERR_DEVICE_BOUNDS and flags & q.QDEC_FLAG_BAD_SEQLEN, (st, flags)
    rows = np.r_[0:10, 30:60]
    parity.assert_out_close(out[rows], res["out"][rows])


def test_prefill_deterministic():
    c = wl.prefill_case([700, 129], [300, 129], seed=13)
    _, out1, _ = _run(c, 2)
    _, out2, _ = _run(c, 2)
    assert torch.equal(out1, out2)


@pytest.mark.parametrize("bad_entry", [-1, 10 ** 6], ids=["negative", "beyond_pool"])
def test_prefill_bad_page_is_flagged(bad_entry):
    """A block-table entry outside the pool in one sequence's chunk pages is
    flagged; the other sequences are exact."""
    q = parity.qdec()
    c = wl.prefill_case([60, 70, 80], [20, 30, 40], seed=14)
    good = wl.prefill_case([60, 70, 80], [20, 30, 40], seed=14)
    res = _oracle(good)
    c.block_table[1, 3] = bad_entry                     # a chunk page of sequence 1
    q_rot, out, err = _run(c, 3)
    st, flags = q.qdec_check_error(err)
    assert st == q.QDEC_ERR_DEVICE_BOUNDS and flags & q.QDEC_FLAG_BAD_PAGE, (st, flags)
    rows = np.r_[0:20, 50:90]
    parity.assert_out_close(out[rows], res["out"][rows])


def test_prefill_wait_that_runs_out_returns_timeout_and_device_stays_usable():
    """The test hook withholds every CTA's first page tile: the wait for it
    gives up, the call reports a timeout, and the next normal call on the
    same device and pool gives the verified result bit for bit."""
    q = parity.qdec()
    c = wl.prefill_case([300, 17, 1000], [20, 17, 200], seed=16)
    res = _oracle(c)
    q_rot, out, err = _run(c, 3)
    parity.assert_out_close(out, res["out"])
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    withheld = torch.empty_like(out)
    q.qdec_prefill_attn(_shape(c, 3, q.QDEC_LAUNCH_TEST_WITHHOLD_TILE), q_rot, c.qo_indptr,
                        c.seq_lens, c.block_table, c.pool, withheld, err)
    st, flags = q.qdec_check_error(err)
    assert st == q.QDEC_ERR_TIMEOUT and flags & q.QDEC_FLAG_TIMEOUT, (st, flags)
    again = torch.empty_like(out)
    q.qdec_prefill_attn(_shape(c, 3), q_rot, c.qo_indptr, c.seq_lens, c.block_table, c.pool,
                        again, err)
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    assert torch.equal(again, out)


# ------------------------------------------------------------------- FP8 pool --

def _fp8_workspace(shape):
    """A scratch for the widened-pages path, poisoned so a read of a byte the
    widening pass did not write shows up."""
    n = parity.qdec().qdec_prefill_fp8_workspace_bytes(shape)
    return torch.full((n,), 0x7F, dtype=torch.uint8, device="cuda")


def _run_fp8(c, codes, sc, B, widen=False):
    q = parity.qdec()
    shape = _shape(c, B)
    T = c.q.shape[0]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_rot = torch.empty((T, 32, 128), dtype=torch.float32, device="cuda")
    out = torch.full((T, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    q.qdec_prefill_append_rope_fp8(shape, c.q, c.k, c.v, c.w_q, c.w_k, c.positions, c.qo_indptr,
                                   c.seq_lens, c.block_table, codes, sc, q_rot, err)
    ws = _fp8_workspace(shape) if widen else None
    q.qdec_prefill_attn_fp8(shape, q_rot, c.qo_indptr, c.seq_lens, c.block_table, codes, sc, out,
                            err, workspace=ws)
    return q_rot, out, err


FP8_CASES = [([37], [37]), ([300, 17, 1000], [20, 17, 1]), ([64, 65, 31], [48, 1, 15]),
             ([500, 40, 77, 250], [0, 40, 33, 0]), ([2048], [200])]


@pytest.mark.parametrize("widen", [False, True], ids=["in-kernel", "widened"])
@pytest.mark.parametrize("seq_lens,chunks", FP8_CASES, ids=lambda x: str(x)[:40])
def test_prefill_fp8_matches_oracle(seq_lens, chunks, widen):
    """FP8 pool: q_rot and out as for bf16; the appended K and V codes equal
    the oracle's bit for bit (the bf16 key is the nearest-even rounding of the
    exact value on both sides; both divide in fp32 by the scale and round
    once); nothing outside the chunk's slots changes.  Both ways of reading
    the codes are checked: converted inside the attention kernel, and
    widened once into a caller's workspace beforehand."""
    c, codes, sc = wl.prefill_case_fp8(seq_lens, chunks, seed=sum(seq_lens) % 89)
    before = codes.cpu().numpy().copy()
    pool = before.copy()
    sc_h = sc.cpu().numpy()
    qo, L, bt = c.qo_indptr.cpu().numpy(), c.seq_lens.cpu().numpy(), c.block_table.cpu().numpy()
    res = oracle.prefill_append_fp8(wl.bf16_bits(c.q), wl.bf16_bits(c.k), wl.bf16_bits(c.v),
                                    wl.bf16_bits(c.w_q), wl.bf16_bits(c.w_k),
                                    c.positions.cpu().numpy(), qo, L, bt, pool, sc_h, 1e6,
                                    float(np.float32(1e-6)))
    ref_out, _ = oracle.prefill_attention_fp8(pool, sc_h, bt, qo, L, res["q_rot"],
                                              1 / math.sqrt(128))
    q_rot, out, err = _run_fp8(c, codes, sc, len(seq_lens), widen)
    st, flags = parity.qdec().qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    g = q_rot.double().cpu().numpy()
    assert np.all(np.abs(g - res["q_rot"]) <= parity.QROT_TOL * (1 + np.abs(res["q_rot"])))
    parity.assert_out_close(out, ref_out)
    got = codes.cpu().numpy()
    changed = np.zeros(got.shape, bool)
    for b in range(len(L)):
        n = qo[b + 1] - qo[b]
        for j in range(n):
            t = L[b] - n + j
            page, off = bt[b, t // 16], t % 16
            assert np.array_equal(got[page, 1, :, off], pool[page, 1, :, off]), f"V codes t={t}"
            assert np.array_equal(got[page, 0, :, off], pool[page, 0, :, off]), f"K codes t={t}"
            changed[page, :, :, off] = True
    assert np.array_equal(got[~changed], before[~changed]), "append touched another slot"


def _oracle_fp8(c, codes, sc):
    """The oracle's append over a host copy of the FP8 pool, then its
    attention over the appended pool."""
    pool = codes.cpu().numpy().copy()
    sc_h = sc.cpu().numpy()
    qo, L, bt = c.qo_indptr.cpu().numpy(), c.seq_lens.cpu().numpy(), c.block_table.cpu().numpy()
    res = oracle.prefill_append_fp8(wl.bf16_bits(c.q), wl.bf16_bits(c.k), wl.bf16_bits(c.v),
                                    wl.bf16_bits(c.w_q), wl.bf16_bits(c.w_k),
                                    c.positions.cpu().numpy(), qo, L, bt, pool, sc_h, 1e6,
                                    float(np.float32(1e-6)))
    ref_out, _ = oracle.prefill_attention_fp8(pool, sc_h, bt, qo, L, res["q_rot"],
                                              1 / math.sqrt(128))
    return ref_out


@pytest.mark.parametrize("seq_lens,chunks", [([300, 17, 1000], [20, 17, 1]),
                                             ([2048, 64, 5], [2048, 48, 5]),
                                             ([129, 4000], [129, 31])],
                         ids=lambda x: str(x)[:40])
def test_prefill_fp8_widened_equals_bf16_pool_of_the_dequantized_values(seq_lens, chunks):
    """The workspace path dequantizes each code once (code x scale in fp32,
    rounded to the nearest-even bf16) and then attends exactly as over a bf16
    pool: its output equals, bit for bit, the bf16-pool attention over a
    pool dequantized that way on the host, on a poisoned workspace.  The
    in-kernel conversion path (exact f16 codes, scales in the softmax) stays
    within the output tolerance of it."""
    q = parity.qdec()
    c, codes, sc = wl.prefill_case_fp8(seq_lens, chunks, seed=len(seq_lens) + sum(chunks) % 61)
    shape = _shape(c, len(seq_lens))
    q_rot, out, err = _run_fp8(c, codes, sc, len(seq_lens))
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    wide = torch.full_like(out, float("nan"))
    q.qdec_prefill_attn_fp8(shape, q_rot, c.qo_indptr, c.seq_lens, c.block_table, codes, sc,
                            wide, err, workspace=_fp8_workspace(shape))
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    vals = codes.cpu().view(torch.float8_e4m3fn).float() * sc.cpu()[..., None, None]
    pool16 = vals.to(torch.bfloat16).cuda()
    ref = torch.full_like(out, float("nan"))
    q.qdec_prefill_attn(shape, q_rot, c.qo_indptr, c.seq_lens, c.block_table, pool16, ref, err)
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    assert torch.equal(wide.view(torch.int16), ref.view(torch.int16))
    parity.assert_out_close(out, parity.to_f64(wide), "in-kernel vs workspace")


def test_prefill_fp8_pages_ready_attends_over_the_workspace_as_left():
    """With QDEC_LAUNCH_PREFILL_PAGES_READY the call skips the dequantizing
    pass and attends over what an earlier call left in the workspace: the
    same bits as that call, both as a plain launch and as a programmatic
    dependent."""
    q = parity.qdec()
    c, codes, sc = wl.prefill_case_fp8([700, 129, 40], [300, 129, 7], seed=19)
    shape = _shape(c, 3)
    T = c.q.shape[0]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_rot = torch.empty((T, 32, 128), dtype=torch.float32, device="cuda")
    q.qdec_prefill_append_rope_fp8(shape, c.q, c.k, c.v, c.w_q, c.w_k, c.positions, c.qo_indptr,
                                   c.seq_lens, c.block_table, codes, sc, q_rot, err)
    ws = _fp8_workspace(shape)
    first = torch.full((T, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    q.qdec_prefill_attn_fp8(shape, q_rot, c.qo_indptr, c.seq_lens, c.block_table, codes, sc,
                            first, err, workspace=ws)
    for extra in (0, q.QDEC_LAUNCH_OVERLAP_PREVIOUS):
        again = torch.full_like(first, float("nan"))
        q.qdec_prefill_attn_fp8(_shape(c, 3, q.QDEC_LAUNCH_PREFILL_PAGES_READY | extra), q_rot,
                                c.qo_indptr, c.seq_lens, c.block_table, codes, sc, again, err,
                                workspace=ws)
        st, flags = q.qdec_check_error(err)
        assert st == 0 and flags == 0, (st, flags)
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))


@pytest.mark.parametrize("widen", [False, True], ids=["in-kernel", "widened"])
def test_prefill_fp8_bad_prefix_page_is_flagged(widen):
    """A block-table entry outside the pool among one sequence's prefix pages
    (which the append does not touch) is flagged by the attention call; the
    other sequences are exact."""
    q = parity.qdec()
    c, codes, sc = wl.prefill_case_fp8([60, 70, 80], [20, 30, 40], seed=16)
    ref_out = _oracle_fp8(c, codes.clone(), sc)
    c.block_table[1, 0] = 10 ** 6                       # tokens 0-15 of sequence 1: prefix
    q_rot, out, err = _run_fp8(c, codes, sc, 3, widen)
    st, flags = q.qdec_check_error(err)
    assert st == q.QDEC_ERR_DEVICE_BOUNDS and flags & q.QDEC_FLAG_BAD_PAGE, (st, flags)
    rows = np.r_[0:20, 50:90]
    parity.assert_out_close(out[rows], ref_out[rows])


def test_prefill_fp8_widened_workspace_too_small_is_refused():
    """A workspace one alignment unit short is refused before any launch
    and the output is left untouched."""
    q = parity.qdec()
    c, codes, sc = wl.prefill_case_fp8([300, 17], [20, 17], seed=18)
    shape = _shape(c, 2)
    q_rot, out, err = _run_fp8(c, codes, sc, 2)
    short = _fp8_workspace(shape)[:-16]
    again = torch.full_like(out, float("nan"))
    with pytest.raises(q.QdecError) as e:
        q.qdec_prefill_attn_fp8(shape, q_rot, c.qo_indptr, c.seq_lens, c.block_table, codes, sc,
                                again, err, workspace=short)
    assert e.value.status == q.QDEC_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(again.float()).all()


@pytest.mark.parametrize("widen", [False, True], ids=["in-kernel", "widened"])
def test_prefill_fp8_wait_that_runs_out_returns_timeout_and_device_stays_usable(widen):
    """FP8 pool: as for bf16, the withheld tile's wait gives up with a timeout
    (the conversion barriers are never reached) and the next normal call
    gives the verified result bit for bit."""
    q = parity.qdec()
    c, codes, sc = wl.prefill_case_fp8([300, 17, 1000], [20, 17, 200], seed=17)
    q_rot, out, err = _run_fp8(c, codes, sc, 3, widen)
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    ws = _fp8_workspace(_shape(c, 3)) if widen else None
    withheld = torch.empty_like(out)
    q.qdec_prefill_attn_fp8(_shape(c, 3, q.QDEC_LAUNCH_TEST_WITHHOLD_TILE), q_rot, c.qo_indptr,
                            c.seq_lens, c.block_table, codes, sc, withheld, err, workspace=ws)
    st, flags = q.qdec_check_error(err)
    assert st == q.QDEC_ERR_TIMEOUT and flags & q.QDEC_FLAG_TIMEOUT, (st, flags)
    again = torch.empty_like(out)
    q.qdec_prefill_attn_fp8(_shape(c, 3), q_rot, c.qo_indptr, c.seq_lens, c.block_table, codes,
                            sc, again, err, workspace=ws)
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    assert torch.equal(again, out)


def test_prefill_fp8_chunk_of_one_equals_fp8_decode():
    """One token per sequence over an FP8 pool: the prefill pair and the FP8
    decode attention on the same appended pool agree closely."""
    q = parity.qdec()
    c, codes, sc = wl.prefill_case_fp8([300, 17, 1000, 64], [1, 1, 1, 1], seed=15)
    shape = _shape(c, 4)
    q_rot, out, err = _run_fp8(c, codes, sc, 4)
    ws = q.alloc_workspace(shape)
    out_d = torch.empty_like(out)
    q.qdec_attn_decode_fp8(shape, q_rot, codes, sc, c.block_table, c.seq_lens, ws, out_d, err)
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0
    assert torch.allclose(out.float(), out_d.float(), rtol=2 ** -7, atol=8e-3)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_prefill_rope_table_gives_the_same_bits(kv):
    """The append with the step's angle table (qdec_prefill_rope_table over
    the chunk rows' positions, away from the token index) writes the same
    q_rot and pool bits as the append that computes each row's angles
    itself: both take them from the same float-float routine."""
    q = parity.qdec()
    seq_lens, chunks = [300, 17, 1000], [20, 17, 200]
    outs = []
    for table in (False, True):
        if kv == "fp8":
            c, codes, sc = wl.prefill_case_fp8(seq_lens, chunks, seed=21, pos_offset=4093)
        else:
            c = wl.prefill_case(seq_lens, chunks, seed=21, pos_offset=4093)
        shape = _shape(c, 3)
        T = c.q.shape[0]
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        q_rot = torch.full((T, 32, 128), float("nan"), dtype=torch.float32, device="cuda")
        rope = None
        if table:
            rope = q.alloc_prefill_rope_table(T)
            q.qdec_prefill_rope_table(shape, c.positions, rope)
        if kv == "fp8":
            q.qdec_prefill_append_rope_fp8(shape, c.q, c.k, c.v, c.w_q, c.w_k, c.positions,
                                           c.qo_indptr, c.seq_lens, c.block_table, codes, sc,
                                           q_rot, err, rope_table=rope)
            pool = codes
        else:
            q.qdec_prefill_append_rope(shape, c.q, c.k, c.v, c.w_q, c.w_k, c.positions,
                                       c.qo_indptr, c.seq_lens, c.block_table, c.pool, q_rot, err,
                                       rope_table=rope)
            pool = c.pool
        st, flags = q.qdec_check_error(err)
        assert st == 0 and flags == 0, (st, flags)
        outs.append((q_rot.clone(), pool.clone()))
    assert torch.equal(outs[0][0].view(torch.int32), outs[1][0].view(torch.int32))
    assert torch.equal(outs[0][1].view(torch.uint8), outs[1][1].view(torch.uint8))


# ------------------------------------------------------------ full size --

@pytest.mark.parametrize("kv", ["bf16", "fp8", "fp8-workspace"])
def test_prefill_full_prompt_sampled(kv):
    """The benchmark's size: one fresh 2048-token prompt in one chunk, run as
    the benchmark runs it (over an FP8 pool both forms; the benchmark times
    the workspace form).  The oracle appends on its own copy of the pool
    (taken before the GPU runs) and gives q_rot for every row; the attention
    is compared on sampled rows: row r's causal attention is the (pinned)
    decode attention of the oracle's q_rot[r] over the first r + 1 tokens of
    the oracle-appended pool."""
    widen = kv == "fp8-workspace"
    kv = "fp8" if widen else kv
    P = 2048
    rows = np.array([0, 1, 15, 16, 17, 255, 1000, 1023, 1024, 2046, 2047])
    if kv == "fp8":
        c, codes, sc = wl.prefill_case_fp8([P], [P], seed=1000)
        pool = codes.cpu().numpy().copy()
        sc_h = sc.cpu().numpy()
    else:
        c = wl.prefill_case([P], [P], seed=1000, poison=True)
        pool = wl.bf16_bits(c.pool).copy()
    bt = c.block_table.cpu().numpy()
    qo, L = c.qo_indptr.cpu().numpy(), c.seq_lens.cpu().numpy()
    ins = (wl.bf16_bits(c.q), wl.bf16_bits(c.k), wl.bf16_bits(c.v), wl.bf16_bits(c.w_q),
           wl.bf16_bits(c.w_k), c.positions.cpu().numpy(), qo, L, bt)
    if kv == "fp8":
        ref = oracle.prefill_append_fp8(*ins, pool, sc_h, 1e6, float(np.float32(1e-6)))
        q_rot, out, err = _run_fp8(c, codes, sc, 1, widen)
    else:
        ref = oracle.prefill_append(*ins, pool, 1e6, float(np.float32(1e-6)))
        q_rot, out, err = _run(c, 1)
    st, flags = parity.qdec().qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    g = q_rot.double().cpu().numpy()
    assert np.all(np.abs(g - ref["q_rot"]) <= parity.QROT_TOL * (1 + np.abs(ref["q_rot"])))
    bt_r = np.repeat(bt, len(rows), axis=0)
    lens = (rows + 1).astype(np.int32)
    qr = np.ascontiguousarray(ref["q_rot"][rows])
    if kv == "fp8":
        ref_out, _ = oracle.attention_fp8(pool, sc_h, bt_r, lens, qr, 1 / math.sqrt(128))
    else:
        ref_out, _ = oracle.attention(pool, bt_r, lens, qr, 1 / math.sqrt(128))
    parity.assert_out_close(out[torch.as_tensor(rows, device="cuda")], ref_out)


def test_prefill_attention_as_a_programmatic_dependent_gives_the_same_bits():
    """With QDEC_LAUNCH_OVERLAP_PREVIOUS the tensor-core attention may start
    while the append before it finishes, waiting for it before it reads q_rot
    or the pool: several layers launched that way on one stream (each
    layer's append, then its attention) give the serial launches' bits."""
    q = parity.qdec()
    seq_lens, chunks = [300, 17, 1000, 2048], [20, 17, 200, 2048]
    layers = [wl.prefill_case(seq_lens, chunks, seed=40 + l) for l in range(3)]
    T = layers[0].q.shape[0]
    outs = []
    for flags in (0, q.QDEC_LAUNCH_OVERLAP_PREVIOUS):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        q_rot = torch.empty((T, 32, 128), dtype=torch.float32, device="cuda")
        out = torch.full((3, T, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        for l, c in enumerate(layers):
            pool = c.pool.clone()
            shape = _shape(c, len(seq_lens), flags)
            q.qdec_prefill_append_rope(shape, c.q, c.k, c.v, c.w_q, c.w_k, c.positions,
                                       c.qo_indptr, c.seq_lens, c.block_table, pool, q_rot, err)
            q.qdec_prefill_attn(shape, q_rot, c.qo_indptr, c.seq_lens, c.block_table, pool,
                                out[l], err)
        st, fl = q.qdec_check_error(err)
        assert st == 0 and fl == 0, (st, fl)
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_prefill_fp8_attention_as_a_programmatic_dependent_gives_the_same_bits():
    """The same over FP8 pools: the tensor-core attention launched as a
    programmatic dependent of each layer's append (it reads q_rot, the codes
    and the scales only after its wait) gives the serial launches' bits."""
    q = parity.qdec()
    seq_lens, chunks = [300, 17, 1000, 2048], [20, 17, 200, 2048]
    layers = [wl.prefill_case_fp8(seq_lens, chunks, seed=50 + l) for l in range(3)]
    T = layers[0][0].q.shape[0]
    outs = []
    for flags in (0, q.QDEC_LAUNCH_OVERLAP_PREVIOUS):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        q_rot = torch.empty((T, 32, 128), dtype=torch.float32, device="cuda")
        out = torch.full((3, T, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        for l, (c, codes, sc) in enumerate(layers):
            codes = codes.clone()
            shape = _shape(c, len(seq_lens), flags)
            q.qdec_prefill_append_rope_fp8(shape, c.q, c.k, c.v, c.w_q, c.w_k, c.positions,
                                           c.qo_indptr, c.seq_lens, c.block_table, codes, sc,
                                           q_rot, err)
            q.qdec_prefill_attn_fp8(shape, q_rot, c.qo_indptr, c.seq_lens, c.block_table, codes,
                                    sc, out[l], err)
        st, fl = q.qdec_check_error(err)
        assert st == 0 and fl == 0, (st, fl)
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
