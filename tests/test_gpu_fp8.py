"""FP8 (E4M3) KV pool: GPU vs oracle, element by element, through the C ABI
(marked gpu).

The pools hold the seeded bf16 draws as E4M3 codes with one fp32 scale per
(page, plane, KV head); NaN codes poison everything the attention must not
read.  The oracle attends over the exact dequantized values, so the out
tolerance is the bf16 path's; the appended K and V codes must equal the
oracle's bit for bit.  Cases mirror the bf16 suite: small ragged batches
with forced grids, the three-call path, a saturating page, overlapped and
graph-replayed layers, and the five benchmark workloads at full size.
"""
import numpy as np
import pytest
import torch

from gqa_paged_kv_gb300 import workloads as wl
import parity

pytestmark = pytest.mark.gpu

SMALL = [
    ([1], 0), ([2], 0), ([15, 16, 17], 0), ([31, 33, 1, 100], 0), ([1000], 0),
    ([17, 1, 300, 64, 16, 2, 999], 0),
    ([15, 16, 17], 1), ([31, 33, 1, 100], 3), ([1000, 1], 7), ([17, 1, 300, 64], 1000),
    ([513], 0), ([4096, 3, 777], 5), ([1056] * 6, 0), ([8192], 0),
]


def _small(lens, seed=41, hq=32, hkv=8, chan=False, spikes=0.0, layers=1, shared=True):
    pages = sum((l + 15) // 16 for l in lens) + 9
    spec = wl.custom(len(lens), lens, pool_pages=pages, seed=seed, num_q_heads=hq,
                     num_kv_heads=hkv, chan_scale=chan, spike_frac=spikes, layers=layers,
                     shared_pool=shared)
    return wl.build(spec, "cuda", poison=True, kv="fp8")


@pytest.mark.parametrize("rope", [True, False], ids=["rope_table", "in_kernel_angles"])
@pytest.mark.parametrize("lens,num_ctas", SMALL, ids=lambda x: str(x))
def test_step_small_fp8(lens, num_ctas, rope):
    w = _small(lens)
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w, num_ctas=num_ctas, rope=rope)
    r.step(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots_fp8(w, 0, range(len(lens)), ref)


@pytest.mark.parametrize("lens,num_ctas", SMALL[:8], ids=lambda x: str(x))
def test_unfused_three_calls_fp8(lens, num_ctas):
    w = _small(lens, seed=42)
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w, num_ctas=num_ctas)
    r.unfused(0)
    r.check_flags()
    q_rot = r.q_rot.double().cpu().numpy()
    err = np.abs(q_rot - ref["q_rot"])
    assert np.all(err <= parity.QROT_TOL * (1 + np.abs(ref["q_rot"]))), err.max()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots_fp8(w, 0, range(len(lens)), ref)


@pytest.mark.parametrize("lens,num_ctas", SMALL, ids=lambda x: str(x))
def test_append_then_decode_fp8(lens, num_ctas):
    """qdec_append_rope_fp8 followed by the one-launch qdec_attn_decode_fp8."""
    w = _small(lens, seed=44)
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w, num_ctas=num_ctas)
    r.two_calls(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots_fp8(w, 0, range(len(lens)), ref)
    torch.cuda.synchronize()
    n = w.spec.batch * w.spec.num_kv_heads
    assert torch.count_nonzero(r.ws[:4 * n].view(torch.int32)).item() == 0


@pytest.mark.parametrize("lens,num_ctas", [([5, 300, 17, 1000, 64, 3], 7),
                                           ([200 + 37 * i for i in range(30)], 0)],
                         ids=["forced_grid", "30_sequences"])
def test_two_launch_step_is_append_then_decode_fp8(lens, num_ctas):
    """Where qdec_step_fp8 runs as two launches (the flat layout: a forced
    grid, or 30 sequences = 240 segments) it is qdec_append_rope_fp8
    followed by qdec_attn_decode_fp8: the same bits, and the oracle's
    result."""
    q = parity.qdec()
    wa, wb = _small(lens, seed=46), _small(lens, seed=46)
    ra = parity.Runner(wa, num_ctas=num_ctas)
    rb = parity.Runner(wb, num_ctas=num_ctas)
    assert q.qdec_step_launches(ra.shape, fp8_pool=True) == 2
    ref = parity.run_oracle(wl.oracle_inputs(wa, 0))
    ra.step(0)
    rb.two_calls(0)
    ra.check_flags()
    rb.check_flags()
    assert torch.equal(ra.out[0].view(torch.int16), rb.out[0].view(torch.int16))
    assert torch.equal(wa.pool8(0), wb.pool8(0))
    parity.assert_out_close(ra.out[0], ref["out"])
    parity.assert_slots_fp8(wa, 0, range(len(lens)), ref)


def test_decode_overlapped_layers_match_serial_fp8():
    spec = wl.custom(5, [17, 1, 300, 64, 1000], pool_pages=120, layers=4, seed=45)
    w = wl.build(spec, "cuda", poison=True, kv="fp8")
    outs = []
    for overlap in (False, True):
        r = parity.Runner(w, overlap=overlap)
        for layer in range(4):
            r.two_calls(layer)
        r.check_flags()
        outs.append(r.out.clone())
    assert torch.equal(outs[0], outs[1])


def test_saturating_page_fp8():
    """Scales far too small for the new rows: the appended codes saturate at
    +-448 (0x7E / 0xFE) exactly where the oracle's do."""
    w = _small([17, 300, 1], seed=43)
    for b in range(3):
        L = int(w.seq_lens_host[b])
        page = int(w.block_table_host[b, (L - 1) // 16])
        w.scale(0)[page] = 1e-4
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w)
    r.step(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots_fp8(w, 0, range(3), ref)
    slot = w.pool8(0)[int(w.block_table_host[1, 299 // 16]), :, :, 299 % 16].cpu().numpy()
    assert np.mean((slot & 0x7F) == 0x7E) > 0.9


def test_channel_scales_and_spikes_small_fp8():
    w = _small([300, 1000, 37], seed=44, chan=True, spikes=0.01)
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w, num_ctas=5)
    r.step(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots_fp8(w, 0, range(3), ref)


def test_deterministic_bits_fp8():
    w = _small([17, 1, 300, 64, 16, 2, 999], seed=45)
    r = parity.Runner(w)
    r.step(0)
    a = r.out[0].clone()
    for _ in range(3):
        r.step(0)
        assert torch.equal(a, r.out[0])


def test_overlapped_layers_match_serial_layers_fp8():
    for shared in (False, True):
        w = _small([17, 1, 300, 64, 1000], seed=46, layers=6, shared=shared)
        outs = []
        for overlap in (False, True):
            r = parity.Runner(w, overlap=overlap)
            for layer in range(6):
                r.step(layer)
            r.check_flags()
            outs.append(r.out.clone())
        assert torch.equal(outs[0], outs[1])


def test_graph_capture_replays_identically_fp8():
    w = _small([17, 1, 300, 64], seed=47, layers=3, shared=False)
    r = parity.Runner(w)
    for layer in range(3):
        r.step(layer)
    torch.cuda.synchronize()
    eager = r.out.clone()
    r.out.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for layer in range(3):
                r.step(layer)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager, r.out)


def test_bad_page_flagged_fp8():
    w = _small([40, 17], seed=48)
    w.block_table[0, 1] = w.spec.pool_pages + 5
    r = parity.Runner(w)
    r.step(0)
    from gqa_paged_kv_gb300 import qdec
    st, flags = qdec.qdec_check_error(r.err)
    assert st == qdec.QDEC_ERR_DEVICE_BOUNDS and flags & qdec.QDEC_FLAG_BAD_PAGE
    # the other sequence is exact
    inputs = wl.oracle_inputs(w, 0, [1])
    ref = parity.run_oracle(inputs)
    parity.assert_out_close(r.out[0, 1:2], ref["out"])


# ------------------------------------------------------ benchmark workloads --

def _check_layers(w, layers, seqs=None):
    seqs = list(range(w.spec.batch)) if seqs is None else list(seqs)
    snaps = {l: wl.oracle_inputs(w, l, seqs) for l in layers}
    torch.cuda.synchronize()
    r = parity.Runner(w, overlap=True)
    for layer in range(w.spec.layers):
        r.step(layer)
    r.check_flags()
    sel = torch.as_tensor(seqs, device="cuda")
    for l in layers:
        ref = parity.run_oracle(snaps[l])
        parity.assert_out_close(r.out[l].index_select(0, sel), ref["out"], f"layer {l}")
        if w.spec.shared_pool and l != w.spec.layers - 1:
            continue  # later layers overwrote this layer's slot in the shared pool
        parity.assert_slots_fp8(w, l, seqs, ref)


def test_workload_1_full_fp8():
    _check_layers(wl.build(wl.WORKLOADS[1], "cuda", poison=True, kv="fp8"), [0])


@pytest.mark.parametrize("cid", [2, 3, 4])
def test_workloads_2_to_4_full_fp8(cid):
    _check_layers(wl.build(wl.WORKLOADS[cid], "cuda", poison=True, kv="fp8"), [0, 17, 35])


def test_workload_5_sampled_fp8():
    w = wl.build(wl.WORKLOADS[5], "cuda", poison=False, kv="fp8")
    lens = w.seq_lens_host
    order = np.argsort(lens)
    seqs = sorted(set([int(order[0]), int(order[1]), int(order[-1]), int(order[-2]),
                       int(order[len(order) // 2]), 0, 63]))
    _check_layers(w, [0, 35], seqs)
