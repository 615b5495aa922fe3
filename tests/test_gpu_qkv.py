"""The merged QKV projection fused with norm, rotation and append, through the
C ABI (marked gpu), against the oracle.  The GPU sums the projection in fp32,
so each element carries the fp32 dot-product error bound
    E_j = 2 * hidden * 2^-24 * sum_i |x_i w_ji|
(twice the first-order bound of a sum of `hidden` products), which the norm
and the rotation carry into q_rot and k_rot as r * max|w| * (E_i + E_(i+64)).
Checked: q_rot within the fp32 q_rot tolerance plus that bound; the appended
k and v within one bf16 ulp of the oracle's unrounded values plus that bound;
the rest of the pool untouched; the whole block (projection, then
qdec_attn_decode, or split attention and merge) within the out tolerance.
Batches of 1 to 70 rows (16-, 32-, 48- and 64-row tiles; two 64-row blocks),
hidden sizes 64 to 2560 (blocks of 64 split unevenly, some CTAs of a cluster
with none), NaN-poisoned pools.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gqa_paged_kv_gb300 import workloads as wl
import parity

pytestmark = pytest.mark.gpu


def _problem(lens, hidden, seed, hkv=8):
    pages = sum((l + 15) // 16 for l in lens) + 9
    spec = wl.custom(len(lens), lens, pool_pages=pages, seed=seed, num_q_heads=4 * hkv,
                     num_kv_heads=hkv)
    w = wl.build(spec, "cuda", poison=True)
    gen = torch.Generator(device="cuda").manual_seed(seed + 7)
    rows = (spec.num_q_heads + 2 * hkv) * spec.head_dim
    x = torch.randn((len(lens), hidden), generator=gen, device="cuda").to(torch.bfloat16)
    wqkv = (torch.randn((rows, hidden), generator=gen, device="cuda") /
            math.sqrt(hidden)).to(torch.bfloat16)
    return w, x, wqkv


def _run(w, x, wqkv, attn="decode"):
    q = parity.qdec()
    s = w.spec
    shape = q.shape_for(w)
    rope = q.alloc_rope_table(shape)
    q.qdec_rope_table(shape, w.positions, rope)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_rot = torch.empty((s.batch, s.num_q_heads, s.head_dim), dtype=torch.float32, device="cuda")
    packed = torch.empty_like(wqkv)
    q.qdec_qkv_pack_weights(shape, wqkv, packed)
    q.qdec_qkv_append_rope(shape, x, packed, w.w_q[0], w.w_k[0], w.positions, w.seq_lens,
                           w.block_table, w.pool(0), q_rot, rope, err)
    ws = q.alloc_workspace(shape)
    out = torch.empty((s.batch, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    if attn == "decode":
        q.qdec_attn_decode(shape, q_rot, w.pool(0), w.block_table, w.seq_lens, ws, out, err)
    else:
        q.qdec_attn_split(shape, q_rot, w.pool(0), w.block_table, w.seq_lens, ws, out, err)
        q.qdec_attn_merge(shape, w.seq_lens, ws, out, err)
    return q_rot, out, err


def _projection_bounds(w, x, wqkv, res):
    """Per-element error bounds of the fp32 projection: E for v, and E
    carried through norm + rotation for q_rot and k_rot."""
    s = w.spec
    D, Hq, Hkv = s.head_dim, s.num_q_heads, s.num_kv_heads
    xf = np.abs(oracle.bf16_bits_to_f64(wl.bf16_bits(x)))
    wf = np.abs(oracle.bf16_bits_to_f64(wl.bf16_bits(wqkv)))
    E = 2 * x.shape[1] * 2.0 ** -24 * (xf @ wf.T)          # [B][(Hq+2Hkv)*D]
    E = E.reshape(s.batch, Hq + 2 * Hkv, D)
    def rotated(Eh, rows, wmax):
        # r = 1/rms of the projected row, from the oracle's own values
        pair = Eh + np.concatenate([Eh[..., D // 2:], Eh[..., :D // 2]], axis=-1)
        return rows * wmax * pair
    inp = wl.oracle_inputs(w, 0)
    wq = np.abs(oracle.bf16_bits_to_f64(inp["w_q"])).max()
    wk = np.abs(oracle.bf16_bits_to_f64(inp["w_k"])).max()
    xq = oracle.bf16_bits_to_f64(wl.bf16_bits(x)) @ oracle.bf16_bits_to_f64(wl.bf16_bits(wqkv)).T
    xq = xq.reshape(s.batch, Hq + 2 * Hkv, D)
    r = 1 / np.sqrt((xq * xq).mean(axis=-1, keepdims=True) + float(np.float32(inp["eps"])))
    return {"q_rot": rotated(E[:, :Hq], r[:, :Hq], wq),
            "k_rot": rotated(E[:, Hq:Hq + Hkv], r[:, Hq:Hq + Hkv], wk),
            "v": E[:, Hq + Hkv:]}


def _oracle(w, x, wqkv):
    inp = wl.oracle_inputs(w, 0)
    pool = inp["pool"].copy()
    s = w.spec
    res = oracle.qkv_append(wl.bf16_bits(x), wl.bf16_bits(wqkv), inp["w_q"], inp["w_k"],
                            inp["positions"], inp["seq_lens"], inp["block_table"], pool,
                            inp["rope_theta"], float(np.float32(inp["eps"])), s.num_q_heads,
                            s.num_kv_heads)
    out, _ = oracle.attention(pool, inp["block_table"], inp["seq_lens"], res["q_rot"],
                              1 / math.sqrt(s.head_dim))
    res["out"] = out
    res["bound"] = _projection_bounds(w, x, wqkv, res)
    return res


def _check_slots(w, res):
    P = w.spec.page_size
    for b in range(w.spec.batch):
        L = int(w.seq_lens_host[b])
        page = int(w.block_table_host[b, (L - 1) // P])
        row = wl.bf16_bits(w.pool(0)[page, :, :, (L - 1) % P, :])
        for plane, key in ((0, "k_rot"), (1, "v")):
            ref = res[key][b]
            got = oracle.bf16_bits_to_f64(row[plane])
            excess = np.abs(got - ref) - parity.bf16_ulp(ref) - res["bound"][key][b]
            i = np.unravel_index(np.argmax(excess), excess.shape)
            assert excess[i] <= 0, (f"seq {b} plane {plane} at {i}: got {got[i]!r} ref {ref[i]!r} "
                                    f"ulp {parity.bf16_ulp(ref)[i]!r}; "
                                    f"{int((excess > 0).sum())} elements beyond 1 ulp")


@pytest.mark.parametrize("lens,hidden", [
    ([1], 64), ([17, 1, 300], 256), ([40] * 8, 2560), ([300, 17, 1000, 64], 2560),
    ([int(x) for x in np.random.default_rng(5).integers(1, 200, size=70)], 512),
    ([int(x) for x in np.random.default_rng(6).integers(1, 400, size=20)], 192),
    ([int(x) for x in np.random.default_rng(7).integers(1, 400, size=40)], 1280),
    ([int(x) for x in np.random.default_rng(8).integers(1, 100, size=64)], 320),
], ids=["b1-h64", "b3-h256", "b8-h2560", "b4-h2560", "b70-h512", "b20-h192", "b40-h1280",
        "b64-h320"])
def test_qkv_projection_matches_oracle(lens, hidden):
    w, x, wqkv = _problem(lens, hidden, seed=61)
    res = _oracle(w, x, wqkv)
    before = wl.bf16_bits(w.pool(0)).copy()
    q_rot, out, err = _run(w, x, wqkv)
    st, flags = parity.qdec().qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    g = q_rot.double().cpu().numpy()
    tol = parity.QROT_TOL * (1 + np.abs(res["q_rot"])) + res["bound"]["q_rot"]
    assert np.all(np.abs(g - res["q_rot"]) <= tol), np.abs(g - res["q_rot"]).max()
    _check_slots(w, res)
    parity.assert_out_close(out, res["out"])
    # only the append slots changed
    after = wl.bf16_bits(w.pool(0))
    P = w.spec.page_size
    mask = np.zeros(after.shape, bool)
    for b in range(w.spec.batch):
        L = int(w.seq_lens_host[b])
        mask[int(w.block_table_host[b, (L - 1) // P]), :, :, (L - 1) % P] = True
    same = (after == before) | (np.isnan(oracle.bf16_bits_to_f64(after)) &
                                np.isnan(oracle.bf16_bits_to_f64(before)))
    assert same[~mask].all(), "the projection wrote outside the append slots"


def test_qkv_then_split_and_merge():
    w, x, wqkv = _problem([300, 17, 1000, 64], 512, seed=64)
    res = _oracle(w, x, wqkv)
    _, out, err = _run(w, x, wqkv, attn="split")
    st, flags = parity.qdec().qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    parity.assert_out_close(out, res["out"])


def test_qkv_group_of_two_kv_heads():
    w, x, wqkv = _problem([33, 5, 16], 128, seed=62, hkv=2)
    res = _oracle(w, x, wqkv)
    q_rot, out, err = _run(w, x, wqkv)
    st, flags = parity.qdec().qdec_check_error(err)
    assert st == 0 and flags == 0
    _check_slots(w, res)
    parity.assert_out_close(out, res["out"])


def test_qkv_bad_page_is_flagged():
    q = parity.qdec()
    w, x, wqkv = _problem([40, 17], 256, seed=63)
    w.block_table[1, 1] = w.spec.pool_pages + 3   # the append page of sequence 1
    _, _, err = _run(w, x, wqkv)
    st, flags = q.qdec_check_error(err)
    assert st == q.QDEC_ERR_DEVICE_BOUNDS and flags & q.QDEC_FLAG_BAD_PAGE, (st, flags)


@pytest.mark.parametrize("shared", [False, True], ids=["per_layer_pools", "shared_pool"])
def test_qkv_block_overlapped_layers_match_serial(shared):
    """Layers of (qdec_qkv_append_rope, qdec_attn_decode) launched as
    programmatic dependents of each other change no bit of out or q_rot."""
    q = parity.qdec()
    lens, hidden, layers = [17, 1, 300, 64, 1000], 512, 4
    spec = wl.custom(len(lens), lens, pool_pages=120, layers=layers, seed=65, shared_pool=shared)
    w = wl.build(spec, "cuda", poison=True)
    s = w.spec
    gen = torch.Generator(device="cuda").manual_seed(66)
    rows = (s.num_q_heads + 2 * s.num_kv_heads) * s.head_dim
    xs = torch.randn((layers, s.batch, hidden), generator=gen, device="cuda").to(torch.bfloat16)
    packed = torch.empty((layers, rows, hidden), dtype=torch.bfloat16, device="cuda")
    for l in range(layers):
        wl_ = (torch.randn((rows, hidden), generator=gen, device="cuda") /
               math.sqrt(hidden)).to(torch.bfloat16)
        q.qdec_qkv_pack_weights(q.shape_for(w), wl_, packed[l])
    results = []
    for overlap in (False, True):
        shape = q.shape_for(w, launch_flags=q.QDEC_LAUNCH_OVERLAP_PREVIOUS if overlap else 0)
        rope = q.alloc_rope_table(shape)
        q.qdec_rope_table(shape, w.positions, rope)
        ws = q.alloc_workspace(shape)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        q_rot = torch.empty((s.batch, s.num_q_heads, s.head_dim), dtype=torch.float32,
                            device="cuda")
        out = torch.empty((layers, s.batch, s.num_q_heads, s.head_dim), dtype=torch.bfloat16,
                          device="cuda")
        for l in range(layers):
            q.qdec_qkv_append_rope(shape, xs[l], packed[l], w.w_q[l], w.w_k[l], w.positions,
                                   w.seq_lens, w.block_table, w.pool(l), q_rot, rope, err)
            q.qdec_attn_decode(shape, q_rot, w.pool(l), w.block_table, w.seq_lens, ws, out[l],
                               err)
        st, flags = q.qdec_check_error(err)
        assert st == 0 and flags == 0, (st, flags)
        results.append((out.clone(), q_rot.clone()))
    assert torch.equal(results[0][0], results[1][0])
    assert torch.equal(results[0][1], results[1][1])



# ------------------------------------------------------------------- FP8 pool --

@pytest.mark.parametrize("lens,hidden", [
    ([40] * 8, 2560),
    ([int(x) for x in np.random.default_rng(11).integers(1, 300, size=40)], 512),
], ids=["b8-h2560", "b40-h512"])
def test_qkv_fp8_pool_matches_oracle(lens, hidden):
    """The projection into an FP8 pool (both instantiations: one 16-row tile
    and a 48-row tile), then qdec_attn_decode_fp8.  q_rot as for bf16; the
    appended codes equal the oracle's, or sit one E4M3 step away on the rare
    elements where the kernel's bf16 row (within the fp32 dot-product bound
    plus one bf16 step of the exact value) straddles a rounding boundary from
    the oracle's; out within the out tolerance of the oracle's FP8 attention."""
    q = parity.qdec()
    pages = sum((l + 15) // 16 for l in lens) + 9
    spec = wl.custom(len(lens), lens, pool_pages=pages, seed=70)
    w = wl.build(spec, "cuda", poison=True, kv="fp8")
    s = w.spec
    gen = torch.Generator(device="cuda").manual_seed(71)
    rows = (s.num_q_heads + 2 * s.num_kv_heads) * s.head_dim
    x = torch.randn((len(lens), hidden), generator=gen, device="cuda").to(torch.bfloat16)
    wqkv = (torch.randn((rows, hidden), generator=gen, device="cuda") /
            math.sqrt(hidden)).to(torch.bfloat16)
    inp = wl.oracle_inputs(w, 0)
    pool = inp["pool"].copy()
    res = oracle.qkv_append_fp8(wl.bf16_bits(x), wl.bf16_bits(wqkv), inp["w_q"], inp["w_k"],
                                inp["positions"], inp["seq_lens"], inp["block_table"], pool,
                                inp["kv_scale"], inp["rope_theta"], float(np.float32(inp["eps"])),
                                s.num_q_heads, s.num_kv_heads)
    ref_out, _ = oracle.attention_fp8(pool, inp["kv_scale"], inp["block_table"],
                                      inp["seq_lens"], res["q_rot"], 1 / math.sqrt(s.head_dim))
    shape = q.shape_for(w)
    rope = q.alloc_rope_table(shape)
    q.qdec_rope_table(shape, w.positions, rope)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_rot = torch.empty((s.batch, s.num_q_heads, s.head_dim), dtype=torch.float32, device="cuda")
    packed = torch.empty_like(wqkv)
    q.qdec_qkv_pack_weights(shape, wqkv, packed)
    q.qdec_qkv_append_rope_fp8(shape, x, packed, w.w_q[0], w.w_k[0], w.positions, w.seq_lens,
                               w.block_table, w.pool8(0), w.scale(0), q_rot, rope, err)
    ws = q.alloc_workspace(shape)
    out = torch.empty((s.batch, s.num_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    q.qdec_attn_decode_fp8(shape, q_rot, w.pool8(0), w.scale(0), w.block_table, w.seq_lens, ws,
                           out, err)
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    bound = _projection_bounds(w, x, wqkv, res)
    g = q_rot.double().cpu().numpy()
    assert np.all(np.abs(g - res["q_rot"]) <=
                  parity.QROT_TOL * (1 + np.abs(res["q_rot"])) + bound["q_rot"])
    parity.assert_out_close(out, ref_out)
    got = w.pool8(0).cpu().numpy()
    P = s.page_size
    off_step = 0
    for b in range(s.batch):
        L = int(w.seq_lens_host[b])
        gpage = int(w.block_table_host[b, (L - 1) // P])
        opage = int(inp["block_table"][b, (L - 1) // P])
        gc = got[gpage, :, :, (L - 1) % P].astype(np.int32)
        oc = pool[opage, :, :, (L - 1) % P].astype(np.int32)
        diff = gc != oc
        assert np.all(((gc & 0x80) == (oc & 0x80)) | ~diff), f"code sign seq {b}"
        assert np.all(np.abs((gc & 0x7F) - (oc & 0x7F)) <= 1), f"codes seq {b}"
        off_step += int(diff.sum())
    assert off_step <= max(2, s.batch * 2 * s.num_kv_heads * s.head_dim // 100), off_step


@pytest.mark.parametrize("batch", [4, 20], ids=["mma_sync_rows16", "tcgen05_rows32"])
def test_qkv_wait_that_runs_out_returns_timeout_and_device_stays_usable(batch):
    """The test hook withholds every CTA's first stage of weight and hidden
    states: the wait for it gives up (the tensor-core variant still frees its
    tensor memory and every cluster still exchanges its partial sums), the
    call reports a timeout, and the next normal block on the same device
    gives the earlier result bit for bit."""
    q = parity.qdec()
    lens = [200 + 37 * i for i in range(batch)]
    w, x, wqkv = _problem(lens, 2560, seed=90 + batch)
    q_rot, out, err = _run(w, x, wqkv)
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    shape = q.shape_for(w, launch_flags=q.QDEC_LAUNCH_TEST_WITHHOLD_TILE)
    rope = q.alloc_rope_table(shape)
    q.qdec_rope_table(shape, w.positions, rope)
    packed = torch.empty_like(wqkv)
    q.qdec_qkv_pack_weights(shape, wqkv, packed)
    withheld = torch.empty_like(q_rot)
    q.qdec_qkv_append_rope(shape, x, packed, w.w_q[0], w.w_k[0], w.positions, w.seq_lens,
                           w.block_table, w.pool(0), withheld, rope, err)
    st, flags = q.qdec_check_error(err)
    assert st == q.QDEC_ERR_TIMEOUT and flags & q.QDEC_FLAG_TIMEOUT, (st, flags)
    q_rot2, out2, err = _run(w, x, wqkv)
    st, flags = q.qdec_check_error(err)
    assert st == 0 and flags == 0, (st, flags)
    assert torch.equal(q_rot2, q_rot) and torch.equal(out2, out)
