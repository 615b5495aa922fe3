"""GPU vs oracle, element by element, through the C ABI (marked gpu).

Small cases span several page tiles, ragged last pages, forced grid sizes
(one CTA for everything, odd counts, more CTAs than tiles) and both the
fused single-launch step and the three-call path.  Pools are NaN-poisoned
wherever the attention must not read.  The five benchmark workloads run at
full size in the launch configuration the benchmark times; their outputs are
compared on every sequence of a few layers (sampled sequences for the
ragged 64-sequence batch).
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
    ([513], 0), ([4096, 3, 777], 5),
]


def _small(lens, seed=11, hq=32, hkv=8, chan=False, spikes=0.0):
    pages = sum((l + 15) // 16 for l in lens) + 9
    spec = wl.custom(len(lens), lens, pool_pages=pages, seed=seed, num_q_heads=hq,
                     num_kv_heads=hkv, chan_scale=chan, spike_frac=spikes)
    return wl.build(spec, "cuda", poison=True)


@pytest.mark.parametrize("rope", [True, False], ids=["rope_table", "in_kernel_angles"])
@pytest.mark.parametrize("lens,num_ctas", SMALL, ids=lambda x: str(x))
def test_step_small(lens, num_ctas, rope):
    w = _small(lens)
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w, num_ctas=num_ctas, rope=rope)
    r.step(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots(w, 0, range(len(lens)), ref)


@pytest.mark.parametrize("rope", [True, False], ids=["rope_table", "in_kernel_angles"])
@pytest.mark.parametrize("lens,num_ctas", SMALL[:8], ids=lambda x: str(x))
def test_unfused_three_calls(lens, num_ctas, rope):
    w = _small(lens, seed=12)
    inputs = wl.oracle_inputs(w, 0)
    ref = parity.run_oracle(inputs)
    r = parity.Runner(w, num_ctas=num_ctas, rope=rope)
    r.unfused(0)
    r.check_flags()
    q_rot = r.q_rot.double().cpu().numpy()
    err = np.abs(q_rot - ref["q_rot"])
    assert np.all(err <= parity.QROT_TOL * (1 + np.abs(ref["q_rot"]))), err.max()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots(w, 0, range(len(lens)), ref)


@pytest.mark.parametrize("lens,num_ctas", SMALL, ids=lambda x: str(x))
def test_append_then_decode(lens, num_ctas):
    """qdec_append_rope followed by the one-launch qdec_attn_decode (the
    fused step's work plan and in-kernel merge, q_rot read from memory)."""
    w = _small(lens, seed=14)
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w, num_ctas=num_ctas)
    r.two_calls(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots(w, 0, range(len(lens)), ref)
    torch.cuda.synchronize()
    n = w.spec.batch * w.spec.num_kv_heads
    assert torch.count_nonzero(r.ws[:4 * n].view(torch.int32)).item() == 0


def test_decode_equals_split_and_merge_closely():
    w = _small([17, 1, 300, 64, 16, 2, 999, 4096], seed=15)
    r = parity.Runner(w)
    r.unfused(0)
    a = r.out[0].float().clone()
    r.two_calls(0)
    r.check_flags()
    # the same q_rot and tile math; the pieces and merge order may differ
    assert torch.allclose(a, r.out[0].float(), rtol=2 ** -7, atol=1e-3)


@pytest.mark.parametrize("num_ctas", [0, 5])
def test_decode_overlapped_layers_match_serial(num_ctas):
    """qdec_attn_decode with the overlap flag after each append: no bit changes."""
    for shared in (False, True):
        spec = wl.custom(5, [17, 1, 300, 64, 1000], pool_pages=120, layers=4, seed=21,
                         shared_pool=shared)
        w = wl.build(spec, "cuda", poison=True)
        outs = []
        for overlap in (False, True):
            r = parity.Runner(w, num_ctas=num_ctas, overlap=overlap)
            for layer in range(4):
                r.two_calls(layer)
            r.check_flags()
            outs.append(r.out.clone())
        assert torch.equal(outs[0], outs[1])


def test_fused_equals_unfused_closely():
    w = _small([17, 1, 300, 64, 16, 2, 999], seed=13)
    r1 = parity.Runner(w)
    r1.step(0)
    a = r1.out[0].float().clone()
    r1.unfused(0)
    r1.check_flags()
    b = r1.out[0].float()
    # both round the same fp32 attention once to bf16; allow one bf16 step
    assert torch.allclose(a, b, rtol=2 ** -7, atol=1e-3)


def test_mqa_group_of_four_single_kv_head():
    w = _small([15, 16, 17, 200], seed=14, hq=4, hkv=1)
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w)
    r.step(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])
    parity.assert_slots(w, 0, range(4), ref)


def test_channel_scales_and_spikes_small():
    w = _small([300, 1000, 37], seed=15, chan=True, spikes=0.01)
    ref = parity.run_oracle(wl.oracle_inputs(w, 0))
    r = parity.Runner(w, num_ctas=5)
    r.step(0)
    r.check_flags()
    parity.assert_out_close(r.out[0], ref["out"])


def test_deterministic_bits():
    w = _small([17, 1, 300, 64, 16, 2, 999], seed=16)
    r = parity.Runner(w)
    r.step(0)
    a = r.out[0].clone()
    for _ in range(3):
        r.step(0)
        assert torch.equal(a, r.out[0])


def test_counters_return_to_zero():
    w = _small([1000, 3, 2000], seed=17)
    r = parity.Runner(w, num_ctas=9)
    r.step(0)
    torch.cuda.synchronize()
    n = w.spec.batch * w.spec.num_kv_heads
    assert torch.count_nonzero(r.ws[:4 * n].view(torch.int32)).item() == 0


def test_rope_table_values():
    """The table's float pairs carry cos/sin of pos * theta^(-2i/D) to ~1e-14."""
    w = _small([1, 17, 300, 16384], seed=19)
    r = parity.Runner(w)
    torch.cuda.synchronize()
    t = r.rope.view(torch.float32).view(4, 64, 4).double().cpu().numpy()
    pos = w.positions.cpu().numpy().astype(np.float64)
    inv = 1e6 ** (-2.0 * np.arange(64) / 128)
    ang = pos[:, None] * inv[None, :]
    assert np.max(np.abs(t[..., 0] + t[..., 1] - np.cos(ang))) < 1e-13
    assert np.max(np.abs(t[..., 2] + t[..., 3] - np.sin(ang))) < 1e-13


@pytest.mark.parametrize("lens,num_ctas", [([17, 1, 300, 64, 16, 2, 999], 7),
                                           ([int(x) for x in np.linspace(1, 3000, 30)], 0)])
def test_two_launch_step_is_append_then_decode(lens, num_ctas):
    """Where qdec_step runs as two launches (bf16 pool, flat layout: a forced
    grid, or 30 sequences = 240 segments, more than 60 % of the resident CTAs)
    it is qdec_append_rope followed by qdec_attn_decode: the same bits, and
    the oracle's result."""
    q = parity.qdec()
    spec = wl.custom(len(lens), lens, pool_pages=sum((l + 15) // 16 for l in lens) + 9, seed=23)
    wa, wb = wl.build(spec, "cuda", poison=True), wl.build(spec, "cuda", poison=True)
    ra = parity.Runner(wa, num_ctas=num_ctas)
    rb = parity.Runner(wb, num_ctas=num_ctas)
    assert q.qdec_step_launches(ra.shape) == 2
    ref = parity.run_oracle(wl.oracle_inputs(wa, 0))
    ra.step(0)
    rb.two_calls(0)
    ra.check_flags()
    rb.check_flags()
    assert torch.equal(ra.out[0].view(torch.int16), rb.out[0].view(torch.int16))
    assert torch.equal(wa.pool(0).view(torch.int16), wb.pool(0).view(torch.int16))
    parity.assert_out_close(ra.out[0], ref["out"])
    parity.assert_slots(wa, 0, range(len(lens)), ref)


def test_rope_table_values_at_large_positions():
    """The float pairs (double reduction by pi/2, float-float series) stay
    within 1e-13 of cos/sin of the double angle for positions far past any
    context, where the reduction takes out up to ~10^6 quarter turns; the
    bound adds pos x 2^-52 for a possible last-bit difference between the
    host's and numpy's theta^(-2i/D)."""
    q = parity.qdec()
    pos = torch.tensor([0, 1, 2, 3, 1023, 40960, 65535, 131071, 777777, 1 << 20],
                       dtype=torch.int32)
    B = pos.numel()
    shape = q.Shape(batch=B, num_pages=B, max_blocks_per_seq=1, max_seq_len=16)
    rope = q.alloc_rope_table(shape)
    q.qdec_rope_table(shape, pos.cuda(), rope)
    torch.cuda.synchronize()
    t = rope.view(torch.float32).view(B, 64, 4).double().cpu().numpy()
    p = pos.numpy().astype(np.float64)
    ang = p[:, None] * (1e6 ** (-2.0 * np.arange(64) / 128))[None, :]
    tol = 1e-13 + p[:, None] * 2.0 ** -52
    assert np.all(np.abs(t[..., 0] + t[..., 1] - np.cos(ang)) <= tol)
    assert np.all(np.abs(t[..., 2] + t[..., 3] - np.sin(ang)) <= tol)
    # the pairs are normalised: |lo| at most half an ulp of hi
    for k in (0, 2):
        hi, lo = t[..., k], t[..., k + 1]
        assert np.all(np.abs(lo) <= np.spacing(np.abs(hi).astype(np.float32)).astype(np.float64) / 2 + 1e-45)


@pytest.mark.parametrize("num_ctas", [0, 5])
def test_overlapped_layers_match_serial_layers(num_ctas):
    """Programmatic dependent launch of consecutive layers changes no bit,
    also when the layers share one pool (each layer rewrites the same slots)."""
    for shared in (False, True):
        spec = wl.custom(5, [17, 1, 300, 64, 1000], pool_pages=120, layers=6, seed=20,
                         shared_pool=shared)
        w = wl.build(spec, "cuda", poison=True)
        outs = []
        for overlap in (False, True):
            r = parity.Runner(w, num_ctas=num_ctas, overlap=overlap)
            for layer in range(6):
                r.step(layer)
            r.check_flags()
            outs.append(r.out.clone())
        assert torch.equal(outs[0], outs[1])


def test_graph_capture_replays_identically():
    spec = wl.custom(4, [17, 1, 300, 64], pool_pages=40, layers=3, seed=18)
    w = wl.build(spec, "cuda", poison=True)
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


# ------------------------------------------------------ benchmark workloads --

def _check_layers(w, layers, seqs=None, num_ctas=0):
    """Run every layer of w in order as the benchmark does (rope table, then
    overlapped layer launches); compare the given layers (pool snapshots
    taken before any layer ran)."""
    seqs = list(range(w.spec.batch)) if seqs is None else list(seqs)
    snaps = {l: wl.oracle_inputs(w, l, seqs) for l in layers}
    torch.cuda.synchronize()
    r = parity.Runner(w, num_ctas=num_ctas, overlap=True)
    for layer in range(w.spec.layers):
        r.step(layer)
    r.check_flags()
    sel = torch.as_tensor(seqs, device="cuda")
    for l in layers:
        ref = parity.run_oracle(snaps[l])
        parity.assert_out_close(r.out[l].index_select(0, sel), ref["out"], f"layer {l}")
        if w.spec.shared_pool and l != w.spec.layers - 1:
            continue  # later layers overwrote this layer's slot in the shared pool
        parity.assert_slots(w, l, seqs, ref)


def test_workload_1_full():
    w = wl.build(wl.WORKLOADS[1], "cuda", poison=True)
    _check_layers(w, [0])


@pytest.mark.parametrize("cid", [2, 3, 4])
def test_workloads_2_to_4_full(cid):
    w = wl.build(wl.WORKLOADS[cid], "cuda", poison=True)
    _check_layers(w, [0, 17, 35])


def test_workload_5_sampled():
    w = wl.build(wl.WORKLOADS[5], "cuda", poison=False)
    lens = w.seq_lens_host
    order = np.argsort(lens)
    seqs = sorted(set([int(order[0]), int(order[1]), int(order[-1]), int(order[-2]),
                       int(order[len(order) // 2]), 0, 63]))
    _check_layers(w, [0, 35], seqs)


_SHAPE_SWITCH = r"""
import sys, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from gqa_paged_kv_gb300 import workloads as wl
import parity

def make(lens, seed):
    pages = sum((l + 15) // 16 for l in lens) + 9
    return wl.build(wl.custom(len(lens), lens, pool_pages=pages, seed=seed), "cuda")

big = parity.Runner(make([1056] * 6, 31))    # 6 x 66 pages: clusters of 3-6, 12-slot ring
big.step(0); big.check_flags()
first = big.out[0].clone()
small = parity.Runner(make([20, 21], 32))    # first use of a smaller layout in this process
small.step(0); small.check_flags()
big.step(0); big.check_flags()               # the larger layout again
assert torch.equal(first, big.out[0])
print("ok")
"""


def test_shapes_with_different_shared_memory_alternate():
    """A shape whose launch needs more shared memory still launches after a
    shape needing less was planned for the first time in between."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = _SHAPE_SWITCH.format(root=os.path.dirname(here), tests=here)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
