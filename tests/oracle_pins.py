"""Pins of the fp64 oracle against what the mathematics fixes.

Each ``pin_*`` takes an :class:`oracle.Oracle` and raises AssertionError if
the oracle disagrees with a closed form, an invariant, a special case that
reduces to a library routine, or brute force on tiny inputs.  The pages print
no worked numeric example for this path, so these are the oracle's anchors.

They are written so that a plausible slip anywhere in the oracle fails at
least one of them; ``test_oracle_mutants.py`` plants such slips in a copy of
the oracle source and checks exactly that.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch

import oracle as oracle_pkg
from oracle import OracleError


# ------------------------------------------------------------ tiny inputs --

def bits_of(x) -> np.ndarray:
    """bf16 bits of values that are exactly representable in bf16."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def random_bits(rng, shape, scale=1.0) -> np.ndarray:
    """Random bf16 bit patterns (normal draws truncated to bf16)."""
    f = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def f64(bits) -> np.ndarray:
    return oracle_pkg.bf16_bits_to_f64(bits)


class Paged:
    """A tiny paged problem: pool [pages][2][Hkv][P][D] plus block table."""

    def __init__(self, rng, seq_lens, Hq=8, Hkv=2, D=16, P=4, extra_pages=3, pool=None):
        self.seq_lens = np.asarray(seq_lens, np.int32)
        self.Hq, self.Hkv, self.D, self.P = Hq, Hkv, D, P
        n = (self.seq_lens + P - 1) // P
        self.mb = int(n.max())
        total = int(n.sum()) + extra_pages
        perm = rng.permutation(total)
        self.bt = np.full((len(seq_lens), self.mb), -1, np.int32)
        off = 0
        for b in range(len(seq_lens)):
            self.bt[b, :n[b]] = perm[off:off + n[b]]
            off += int(n[b])
        self.pool = random_bits(rng, (total, 2, Hkv, P, D)) if pool is None else pool
        self.q = rng.standard_normal((len(seq_lens), Hq, D))

    def gather(self, b, kv, g):
        """Contiguous [L][D] rows of sequence b, plane kv, head g (numpy indexing)."""
        L = int(self.seq_lens[b])
        t = np.arange(L)
        pages = self.bt[b, t // self.P]
        return f64(self.pool[pages, kv, g, t % self.P, :])


def _close(a, b, tol, what):
    a, b = np.asarray(a), np.asarray(b)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert np.all(np.isfinite(a)) and err <= tol, f"{what}: max |diff| {err:.3e} > {tol:.1e}"


# ------------------------------------------------------------------- bf16 --

def pin_bf16_roundtrip(orc):
    """Every finite bf16 pattern survives widening and re-rounding exactly."""
    for h in range(0, 1 << 16, 7):
        e = (h >> 7) & 0xFF
        if e == 0xFF:
            continue
        assert orc.double_to_bf16(orc.bf16_to_double(h)) == h, hex(h)


def pin_bf16_rne_matches_library(orc):
    """For binary32 inputs, the double->bf16 rounding equals torch's
    float32->bf16 conversion (round to nearest even) bit for bit."""
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(3000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-38).astype(np.float32),   # subnormal range
        (rng.standard_normal(1000) * 1e37).astype(np.float32),
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -133, 2 ** -134,
                  3.3e38, -3.3e38], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.f64_to_bf16_bits(x.astype(np.float64))
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first x={x[bad[0]]!r}"


def pin_bf16_single_rounding(orc):
    """Ties go to even; a double just above a tie rounds up (one rounding,
    not double rounding through binary32); overflow gives infinity."""
    assert orc.double_to_bf16(1 + 2 ** -8) == 0x3F80
    assert orc.double_to_bf16(1 + 3 * 2 ** -8) == 0x3F82
    assert orc.double_to_bf16(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert orc.double_to_bf16(-(1 + 2 ** -8 + 2 ** -40)) == 0xBF81
    assert orc.double_to_bf16(3.4e38) == 0x7F80
    assert orc.double_to_bf16(2.0 ** -133) == 0x0001
    assert orc.double_to_bf16(2.0 ** -134) == 0x0000


# ---------------------------------------------------------------- RMSNorm --

def pin_rmsnorm_closed_form(orc):
    x = np.array([1.0, 2.0, 3.0, 4.0])
    _close(orc.rmsnorm(x, np.ones(4), 0.0), x / math.sqrt(7.5), 1e-15, "rmsnorm [1,2,3,4]")
    w = np.array([1.0, 0.5, 2.0, 1.0])
    _close(orc.rmsnorm(x, w, 0.5), x * w / math.sqrt(8.0), 1e-15, "rmsnorm weighted, eps")


def pin_rmsnorm_invariants(orc):
    rng = np.random.default_rng(1)
    x = rng.standard_normal(128)
    y = orc.rmsnorm(x, np.ones(128), 0.0)
    _close(np.sqrt(np.mean(y * y)), 1.0, 1e-14, "unit RMS")
    _close(orc.rmsnorm(3.7 * x, np.ones(128), 0.0), y, 1e-14, "scale invariance")


def pin_rmsnorm_eps_inside_root(orc):
    x = np.full(4, 1e-3)
    # mean(x^2) = 1e-6; with eps = 1e-6 inside the root: 1e-3 / sqrt(2e-6)
    _close(orc.rmsnorm(x, np.ones(4), 1e-6), np.full(4, 1e-3 / math.sqrt(2e-6)), 1e-12,
           "eps inside the root")
    _close(orc.rmsnorm(np.zeros(4), np.ones(4), 1e-6), np.zeros(4), 0.0, "zero row")


# ------------------------------------------------------------------- RoPE --

def _rot2(x, a):
    R = np.array([[math.cos(a), -math.sin(a)], [math.sin(a), math.cos(a)]])
    return R @ np.asarray(x, float)


def pin_rope_2d_is_rotation(orc):
    """D = 2: one pair, frequency theta^0 = 1, so RoPE is the plane rotation
    by `pos` radians (counter-clockwise)."""
    _close(orc.rope_neox([1.0, 0.0], math.pi / 2, 1e6), [0.0, 1.0], 1e-15, "quarter turn")
    for pos in (0.3, 7.0, 1000.0):
        _close(orc.rope_neox([0.6, -1.2], pos, 1e6), _rot2([0.6, -1.2], pos), 1e-12, "2-D")


def pin_rope_d4_rotate_half_pairs(orc):
    """D = 4, theta = 10000: pair (0, 2) turns by pos, pair (1, 3) by
    pos * 10000^(-1/2) = pos / 100 (rotate-half pairing, not interleaved)."""
    x = np.array([0.5, -1.0, 2.0, 0.25])
    pos = 3.0
    y = orc.rope_neox(x, pos, 1e4)
    a = _rot2([x[0], x[2]], pos)
    b = _rot2([x[1], x[3]], pos / 100.0)
    _close(y, [a[0], b[0], a[1], b[1]], 1e-14, "D=4 pairs")


def pin_rope_invariants(orc):
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    _close(np.linalg.norm(orc.rope_neox(q, 12345, 1e6)), np.linalg.norm(q), 1e-12, "norm")
    _close(orc.rope_neox(q, 0, 1e6), q, 0.0, "pos 0 identity")
    _close(orc.rope_neox(orc.rope_neox(q, 777, 1e6), -777, 1e6), q, 1e-12, "R(p)R(-p)")
    for m, n, c in ((5, 2, 9), (100, 40, 1000), (0, 16383, 3)):
        d1 = orc.rope_neox(q, m, 1e6) @ orc.rope_neox(k, n, 1e6)
        d2 = orc.rope_neox(q, m + c, 1e6) @ orc.rope_neox(k, n + c, 1e6)
        _close(d1, d2, 1e-10, "relative position")


# -------------------------------------------------------------- attention --

def pin_attention_single_token(orc):
    """L = 1: softmax over one token is 1, so out = V_0 and lse = s_0."""
    rng = np.random.default_rng(3)
    pb = Paged(rng, [1, 1], Hq=8, Hkv=2, D=16, P=4)
    scale = 0.25
    out, lse = orc.attention(pb.pool, pb.bt, pb.seq_lens, pb.q, scale)
    for b in range(2):
        for h in range(8):
            g = h // 4
            K, V = pb.gather(b, 0, g), pb.gather(b, 1, g)
            _close(out[b, h], V[0], 1e-15, "out = V_0")
            _close(lse[b, h], scale * (pb.q[b, h] @ K[0]), 1e-13, "lse = s_0")


def pin_attention_equal_keys(orc):
    """All keys equal: uniform weights, out = mean of V, lse = s + ln L."""
    rng = np.random.default_rng(4)
    pb = Paged(rng, [13, 37], Hq=4, Hkv=1, D=16, P=4)
    krow = random_bits(rng, 16)
    pb.pool[:, 0] = krow
    out, lse = orc.attention(pb.pool, pb.bt, pb.seq_lens, pb.q, 0.3)
    for b, L in enumerate(pb.seq_lens):
        V = pb.gather(b, 1, 0)
        for h in range(4):
            _close(out[b, h], V.mean(axis=0), 1e-14, "mean of V")
            _close(lse[b, h], 0.3 * (pb.q[b, h] @ f64(krow)) + math.log(L), 1e-12, "lse")


def pin_attention_two_tokens(orc):
    """L = 2: out = sigma V_0 + (1 - sigma) V_1 with sigma = 1 / (1 + e^(s1 - s0))."""
    rng = np.random.default_rng(5)
    pb = Paged(rng, [2], Hq=4, Hkv=1, D=16, P=4)
    scale = 0.5
    out, lse = orc.attention(pb.pool, pb.bt, pb.seq_lens, pb.q, scale)
    K, V = pb.gather(0, 0, 0), pb.gather(0, 1, 0)
    for h in range(4):
        s0, s1 = scale * (pb.q[0, h] @ K[0]), scale * (pb.q[0, h] @ K[1])
        sig = 1.0 / (1.0 + math.exp(s1 - s0))
        _close(out[0, h], sig * V[0] + (1 - sig) * V[1], 1e-14, "two tokens")
        _close(lse[0, h], math.log(math.exp(s0) + math.exp(s1)), 1e-13, "two-token lse")


def pin_attention_dense_equivalence(orc):
    """Against dense contiguous attention: rows gathered with numpy indexing,
    scipy's softmax, numpy matmul.  Lengths straddle page boundaries."""
    rng = np.random.default_rng(6)
    pb = Paged(rng, [1, 3, 4, 5, 8, 15, 17, 40], Hq=8, Hkv=2, D=16, P=4)
    scale = 1 / 4
    out, lse = orc.attention(pb.pool, pb.bt, pb.seq_lens, pb.q, scale)
    for b in range(len(pb.seq_lens)):
        for h in range(8):
            g = h // 4
            K, V = pb.gather(b, 0, g), pb.gather(b, 1, g)
            s = scale * (K @ pb.q[b, h])
            _close(out[b, h], scipy.special.softmax(s) @ V, 1e-13, f"dense b={b} h={h}")
            _close(lse[b, h], scipy.special.logsumexp(s), 1e-12, "dense lse")


def pin_attention_page_relabel(orc):
    """Relabelling physical pages (pool and block table together) changes nothing."""
    rng = np.random.default_rng(8)
    pb = Paged(rng, [9, 30, 17], Hq=8, Hkv=2, D=16, P=4, extra_pages=5)
    out0, lse0 = orc.attention(pb.pool, pb.bt, pb.seq_lens, pb.q, 0.25)
    perm = rng.permutation(pb.pool.shape[0])
    pool2 = np.empty_like(pb.pool)
    pool2[perm] = pb.pool
    bt2 = np.where(pb.bt >= 0, perm[np.maximum(pb.bt, 0)], -1).astype(np.int32)
    out1, lse1 = orc.attention(pool2, bt2, pb.seq_lens, pb.q, 0.25)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1), "page relabel"


def pin_attention_token_permutation(orc):
    """Permuting (K_t, V_t) pairs jointly within a sequence changes nothing."""
    rng = np.random.default_rng(9)
    pb = Paged(rng, [23], Hq=4, Hkv=1, D=16, P=4)
    out0, lse0 = orc.attention(pb.pool, pb.bt, pb.seq_lens, pb.q, 0.25)
    L, P = 23, 4
    t = np.arange(L)
    rows = (pb.bt[0, t // P], t % P)
    K = pb.pool[rows[0], 0, 0, rows[1]].copy()
    V = pb.pool[rows[0], 1, 0, rows[1]].copy()
    pi = rng.permutation(L)
    pool2 = pb.pool.copy()
    pool2[rows[0], 0, 0, rows[1]] = K[pi]
    pool2[rows[0], 1, 0, rows[1]] = V[pi]
    out1, lse1 = orc.attention(pool2, pb.bt, pb.seq_lens, pb.q, 0.25)
    _close(out1, out0, 1e-13, "token permutation")
    _close(lse1, lse0, 1e-12, "token permutation lse")


def pin_attention_key_shift(orc):
    """K_t + c for one c shared by all tokens shifts every score by q.c: out unchanged."""
    rng = np.random.default_rng(10)
    pb = Paged(rng, [11, 29], Hq=4, Hkv=1, D=16, P=4)
    ints = rng.integers(-8, 8, size=pb.pool.shape).astype(np.float32) / 4
    pb.pool = bits_of(ints)
    out0, _ = orc.attention(pb.pool, pb.bt, pb.seq_lens, pb.q, 0.25)
    c = rng.integers(-4, 4, size=16).astype(np.float32)
    pool2 = pb.pool.copy()
    pool2[:, 0] = bits_of(ints[:, 0] + c)     # exact in bf16 (small quarter-integers)
    out1, _ = orc.attention(pool2, pb.bt, pb.seq_lens, pb.q, 0.25)
    _close(out1, out0, 1e-12, "key shift")


def pin_attention_value_affine(orc):
    """V -> a V + b gives out -> a out + b (weights sum to one)."""
    rng = np.random.default_rng(11)
    pb = Paged(rng, [7, 18], Hq=4, Hkv=1, D=16, P=4)
    ints = rng.integers(-8, 8, size=pb.pool.shape).astype(np.float32)
    pb.pool = bits_of(ints)
    out0, lse0 = orc.attention(pb.pool, pb.bt, pb.seq_lens, pb.q, 0.25)
    pool2 = pb.pool.copy()
    pool2[:, 1] = bits_of(2 * ints[:, 1] + 3)
    out1, lse1 = orc.attention(pool2, pb.bt, pb.seq_lens, pb.q, 0.25)
    _close(out1, 2 * out0 + 3, 1e-12, "value affine")
    _close(lse1, lse0, 0.0, "lse independent of V")


def pin_gqa_equals_replicated_mha(orc):
    """Hq = 8 over Hkv = 2 equals Hq = 8 over Hkv = 8 with KV head g copied to
    heads 4g..4g+3 (query head h reads KV head h / 4)."""
    rng = np.random.default_rng(12)
    pb = Paged(rng, [5, 21], Hq=8, Hkv=2, D=16, P=4)
    out0, lse0 = orc.attention(pb.pool, pb.bt, pb.seq_lens, pb.q, 0.25)
    rep = np.repeat(pb.pool, 4, axis=2)
    out1, lse1 = orc.attention(np.ascontiguousarray(rep), pb.bt, pb.seq_lens, pb.q, 0.25)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1), "GQA vs MHA"


def pin_split_merge_exact(orc):
    """Any chunking followed by the log-sum-exp merge equals the unsplit result."""
    rng = np.random.default_rng(13)
    pb = Paged(rng, [1, 16, 17, 45, 64], Hq=8, Hkv=2, D=16, P=4)
    out0, lse0 = orc.attention(pb.pool, pb.bt, pb.seq_lens, pb.q, 0.25)
    for chunk in (1, 2, 3, 16):
        out1, lse1 = orc.attention_split(pb.pool, pb.bt, pb.seq_lens, pb.q, 0.25, chunk)
        _close(out1, out0, 1e-13, f"split chunk={chunk}")
        _close(lse1, lse0, 1e-12, f"split lse chunk={chunk}")


def pin_nan_outside_context_is_ignored(orc):
    """NaN in slots past the end and in unreferenced pages never reaches out."""
    rng = np.random.default_rng(14)
    pb = Paged(rng, [6, 13], Hq=4, Hkv=1, D=16, P=4, extra_pages=2)
    out0, _ = orc.attention(pb.pool, pb.bt, pb.seq_lens, pb.q, 0.25)
    pool2 = pb.pool.copy()
    used = set(int(p) for p in pb.bt.ravel() if p >= 0)
    for p in range(pool2.shape[0]):
        if p not in used:
            pool2[p] = 0x7FC0
    for b, L in enumerate(pb.seq_lens):
        pool2[pb.bt[b, (L - 1) // 4], :, :, (L - 1) % 4 + 1:] = 0x7FC0
    out1, _ = orc.attention(pool2, pb.bt, pb.seq_lens, pb.q, 0.25)
    assert np.array_equal(out0, out1), "NaN poison"


def pin_errors(orc):
    rng = np.random.default_rng(15)
    pb = Paged(rng, [5], Hq=4, Hkv=1, D=16, P=4)
    bad = pb.bt.copy()
    bad[0, 1] = pb.pool.shape[0]
    for bt, sl in ((bad, pb.seq_lens), (pb.bt, np.array([0], np.int32)),
                   (pb.bt, np.array([pb.mb * 4 + 1], np.int32))):
        try:
            orc.attention(pb.pool, bt, sl, pb.q, 0.25)
        except OracleError:
            continue
        raise AssertionError("bad input accepted")


# ------------------------------------------------------------- layer-step --

def _layer_problem(rng, seq_lens, Hq=8, Hkv=2, D=16, P=4):
    pb = Paged(rng, seq_lens, Hq=Hq, Hkv=Hkv, D=D, P=P, extra_pages=4)
    B = len(seq_lens)
    q = random_bits(rng, (B, Hq, D))
    k = random_bits(rng, (B, Hkv, D))
    v = random_bits(rng, (B, Hkv, D))
    wq = bits_of((rng.integers(2, 6, D) / 4).astype(np.float32))
    wk = bits_of((rng.integers(2, 6, D) / 4).astype(np.float32))
    pos = (pb.seq_lens - 1).astype(np.int32)
    return pb, q, k, v, wq, wk, pos


def pin_layer_append_one_slot(orc):
    """The append changes exactly slot L-1 of every (sequence, KV head, plane):
    K gets bf16(k_rot) rounded to nearest even, V gets v's bits."""
    rng = np.random.default_rng(16)
    pb, q, k, v, wq, wk, pos = _layer_problem(rng, [1, 4, 5, 16, 22])
    before = pb.pool.copy()
    res = orc.decode_layer(q, k, v, wq, wk, pos, pb.seq_lens, pb.bt, pb.pool, 1e6, 1e-6)
    changed = np.zeros(before.shape, bool)
    for b, L in enumerate(pb.seq_lens):
        page, off = pb.bt[b, (L - 1) // 4], (L - 1) % 4
        for g in range(2):
            assert np.array_equal(pb.pool[page, 0, g, off], orc.f64_to_bf16_bits(res["k_rot"][b, g]))
            assert np.array_equal(pb.pool[page, 1, g, off], v[b, g])
        changed[page, :, :, off] = True
    assert np.array_equal(pb.pool[~changed], before[~changed]), "append touched another slot"


def pin_layer_composition(orc):
    """The layer-step is norm -> rope per row, append, then attention over the
    appended pool; and each stage uses the right weight vector."""
    rng = np.random.default_rng(17)
    pb, q, k, v, wq, wk, pos = _layer_problem(rng, [3, 17, 31])
    res = orc.decode_layer(q, k, v, wq, wk, pos, pb.seq_lens, pb.bt, pb.pool, 1e6, 1e-6)
    for b in range(3):
        for h in range(8):
            want = orc.rope_neox(orc.rmsnorm(f64(q[b, h]), f64(wq), 1e-6), pos[b], 1e6)
            _close(res["q_rot"][b, h], want, 0.0, "q_rot")
        for g in range(2):
            want = orc.rope_neox(orc.rmsnorm(f64(k[b, g]), f64(wk), 1e-6), pos[b], 1e6)
            _close(res["k_rot"][b, g], want, 0.0, "k_rot")
    out, lse = orc.attention(pb.pool, pb.bt, pb.seq_lens, res["q_rot"], 1 / math.sqrt(16))
    _close(res["out"], out, 0.0, "out after append")
    _close(res["lse"], lse, 0.0, "lse after append")


def pin_layer_new_token_attends_itself(orc):
    """L = 1: the only token is the new one, so out = v (exactly, as double)."""
    rng = np.random.default_rng(18)
    pb, q, k, v, wq, wk, pos = _layer_problem(rng, [1, 1])
    res = orc.decode_layer(q, k, v, wq, wk, pos, pb.seq_lens, pb.bt, pb.pool, 1e6, 1e-6)
    for b in range(2):
        for h in range(8):
            _close(res["out"][b, h], f64(v[b, h // 4]), 0.0, "out = v")


# -------------------------------------------------------------- fp8 (E4M3) --
# The format is the OCP 8-bit floating point E4M3 (bias 7, three mantissa
# bits, subnormals, NaN = S.1111.111, no infinity, largest finite 448).

def _torch_e4m3_values() -> np.ndarray:
    """Values of all 256 codes by PyTorch's float8_e4m3fn widening (a library
    implementation of the same format)."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def _e4m3_nearest(x: float, table: np.ndarray) -> int:
    """Brute force: the finite non-negative code nearest to |x| (ties to the
    code with even mantissa), magnitudes >= 448 saturate, sign copied."""
    if math.isnan(x):
        return 0x7F
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if a >= 448.0:
        return sign | 0x7E
    best_d, best_c = None, None
    for c in range(0x7F):
        d = abs(table[c] - a)
        if best_d is None or d < best_d or (d == best_d and c % 2 == 0):
            best_d, best_c = d, c
    return sign | best_c


def _fp8_codes(rng, shape, sigma=4.0) -> np.ndarray:
    """Random finite codes: normal draws cast by PyTorch (magnitudes < 448)."""
    x = np.clip(rng.standard_normal(shape) * sigma, -440, 440).astype(np.float32)
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_e4m3_decode_table(orc):
    """All 256 codes against the format's closed description and against
    PyTorch's widening."""
    vals = np.array([orc.e4m3_to_double(c) for c in range(256)])
    lib = _torch_e4m3_values()
    nan = np.isnan(vals)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF], "NaN patterns"
    assert np.array_equal(np.isnan(lib), nan) and np.array_equal(vals[~nan], lib[~nan]), \
        "differs from float8_e4m3fn"
    assert vals[0x7E] == 448 and vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6
    assert vals[0x38] == 1.0 and vals[0x39] == 1.125 and vals[0x30] == 0.5
    assert vals[0x80] == 0 and math.copysign(1.0, vals[0x80]) < 0, "negative zero"
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0), "codes 0x00..0x7E increase"
    assert np.array_equal(vals[0x80:0xFF], -pos), "sign bit negates"
    for k in range(-6, 8):   # eight equally spaced values per binade
        inb = pos[(pos >= 2.0 ** k) & (pos < 2.0 ** (k + 1))]
        assert np.array_equal(inb, 2.0 ** k * (1 + np.arange(8) / 8)), f"binade 2^{k}"
    assert np.array_equal(pos[pos >= 256], 256 * (1 + np.arange(7) / 8)), "top binade"
    assert np.array_equal(pos[(pos > 0) & (pos < 2.0 ** -6)], np.arange(1, 8) * 2.0 ** -9)


def pin_e4m3_encode_brute_force(orc):
    """Encoding equals the nearest code by exhaustive search (ties to even,
    saturation at 448) on every midpoint, every code and random values; and
    PyTorch's float8_e4m3fn cast where that cast does not overflow."""
    table = np.array([orc.e4m3_to_double(c) for c in range(0x7F)])
    mids = ((table[1:] + table[:-1]) / 2).astype(np.float32)
    rng = np.random.default_rng(19)
    xs = np.concatenate([
        table.astype(np.float32), mids, np.nextafter(mids, np.float32(0)),
        np.nextafter(mids, np.float32(1e3)),
        np.exp(rng.uniform(math.log(2.0 ** -12), math.log(600.0), 1500)).astype(np.float32),
        np.array([0.0, 448.0, 449.0, 463.99, 464.0, 465.0, 1e30, np.inf, 1e-40, 2.0 ** -10,
                  3 * 2.0 ** -10], np.float32)])
    xs = np.concatenate([xs, -xs, np.array([np.nan], np.float32)])
    got = orc.e4m3_codes(xs)
    for x, c in zip(xs, got):
        want = _e4m3_nearest(float(x), table)
        assert c == want, f"e4m3({float(x)!r}) = {c:#x}, nearest is {want:#x}"
    ok = np.abs(xs) < 464
    lib = torch.from_numpy(xs[ok]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[ok], lib), "differs from PyTorch's float8_e4m3fn cast"


def _fp8_pool(rng, pb, pow2: bool):
    pages, _, Hkv = pb.pool.shape[:3]
    codes = _fp8_codes(rng, pb.pool.shape)
    if pow2:
        sc = (2.0 ** rng.integers(-4, 3, size=(pages, 2, Hkv))).astype(np.float32)
    else:
        sc = rng.uniform(0.01, 0.5, size=(pages, 2, Hkv)).astype(np.float32)
    return codes, sc


def pin_fp8_attention_pow2_scales_equal_bf16(orc):
    """With power-of-two scales every element e4m3(code) * scale is exact in
    bf16, so FP8 attention must equal the (pinned) bf16 attention over the
    dequantized pool bit for bit."""
    rng = np.random.default_rng(20)
    pb = Paged(rng, [1, 3, 4, 5, 8, 15, 17, 40], Hq=8, Hkv=2, D=16, P=4)
    codes, sc = _fp8_pool(rng, pb, pow2=True)
    deq = _torch_e4m3_values()[codes] * sc[:, :, :, None, None]
    out0, lse0 = orc.attention(bits_of(deq.astype(np.float32)), pb.bt, pb.seq_lens, pb.q, 0.25)
    out1, lse1 = orc.attention_fp8(codes, sc, pb.bt, pb.seq_lens, pb.q, 0.25)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1), "fp8 vs bf16 attention"


def pin_fp8_attention_dense(orc):
    """General scales: against dense attention over rows dequantized with
    PyTorch's widening, one scale per (page, plane, head)."""
    rng = np.random.default_rng(21)
    pb = Paged(rng, [2, 7, 16, 33], Hq=8, Hkv=2, D=16, P=4)
    codes, sc = _fp8_pool(rng, pb, pow2=False)
    table = _torch_e4m3_values()
    out, lse = orc.attention_fp8(codes, sc, pb.bt, pb.seq_lens, pb.q, 0.25)
    for b, L in enumerate(pb.seq_lens):
        t = np.arange(L)
        pages, off = pb.bt[b, t // 4], t % 4
        for h in range(8):
            g = h // 4
            K = table[codes[pages, 0, g, off]] * sc[pages, 0, g][:, None].astype(np.float64)
            V = table[codes[pages, 1, g, off]] * sc[pages, 1, g][:, None].astype(np.float64)
            s = 0.25 * (K @ pb.q[b, h])
            _close(out[b, h], scipy.special.softmax(s) @ V, 1e-13, f"fp8 dense b={b} h={h}")
            _close(lse[b, h], scipy.special.logsumexp(s), 1e-12, "fp8 dense lse")


def pin_fp8_layer_append(orc):
    """The FP8 layer-step: the same q_rot/k_rot as the bf16 layer-step; the
    append changes exactly slot L-1 of every (sequence, plane, head), with
    K = nearest code of fp32(bf16(k_rot)) / scale and V = nearest code of
    fp32(v) / scale (fp32 division, brute-force rounding, saturation when
    the scale is too small); out and lse are the FP8 attention over the
    updated pool."""
    rng = np.random.default_rng(22)
    seq_lens = [1, 4, 5, 16, 22, 9, 31, 2]
    pb, q, k, v, wq, wk, pos = _layer_problem(rng, seq_lens, Hq=16, Hkv=4, D=32)
    codes, sc = _fp8_pool(rng, pb, pow2=False)
    sc[pb.bt[3, (16 - 1) // 4]] = 1e-4          # this page saturates
    before = codes.copy()
    res = orc.decode_layer_fp8(q, k, v, wq, wk, pos, pb.seq_lens, pb.bt, codes, sc, 1e6, 1e-6)
    ref = orc.decode_layer(q, k, v, wq, wk, pos, pb.seq_lens, pb.bt, pb.pool.copy(), 1e6, 1e-6)
    _close(res["q_rot"], ref["q_rot"], 0.0, "fp8 layer q_rot")
    _close(res["k_rot"], ref["k_rot"], 0.0, "fp8 layer k_rot")
    table = np.array([orc.e4m3_to_double(c) for c in range(0x7F)])
    changed = np.zeros(codes.shape, bool)
    saturated = 0
    for b, L in enumerate(pb.seq_lens):
        page, off = pb.bt[b, (L - 1) // 4], (L - 1) % 4
        for g in range(4):
            kf = f64(orc.f64_to_bf16_bits(ref["k_rot"][b, g])).astype(np.float32)
            vf = f64(v[b, g]).astype(np.float32)
            want_k = [_e4m3_nearest(float(x / sc[page, 0, g]), table) for x in kf]
            want_v = [_e4m3_nearest(float(x / sc[page, 1, g]), table) for x in vf]
            assert np.array_equal(codes[page, 0, g, off], want_k), f"K codes b={b} g={g}"
            assert np.array_equal(codes[page, 1, g, off], want_v), f"V codes b={b} g={g}"
            saturated += int(np.sum((codes[page, :, g, off] & 0x7F) == 0x7E))
        changed[page, :, :, off] = True
    assert saturated > 0, "the saturating page did not saturate"
    assert np.array_equal(codes[~changed], before[~changed]), "append touched another slot"
    out, lse = orc.attention_fp8(codes, sc, pb.bt, pb.seq_lens, res["q_rot"], 1 / math.sqrt(32))
    _close(res["out"], out, 0.0, "fp8 out after append")
    _close(res["lse"], lse, 0.0, "fp8 lse after append")


def pin_fp8_nan_codes_outside_context(orc):
    """NaN codes in slots past the end and in unreferenced pages never reach out."""
    rng = np.random.default_rng(23)
    pb = Paged(rng, [6, 13], Hq=4, Hkv=1, D=16, P=4, extra_pages=2)
    codes, sc = _fp8_pool(rng, pb, pow2=False)
    out0, _ = orc.attention_fp8(codes, sc, pb.bt, pb.seq_lens, pb.q, 0.25)
    c2 = codes.copy()
    used = set(int(p) for p in pb.bt.ravel() if p >= 0)
    for p in range(c2.shape[0]):
        if p not in used:
            c2[p] = 0x7F
    for b, L in enumerate(pb.seq_lens):
        c2[pb.bt[b, (L - 1) // 4], :, :, (L - 1) % 4 + 1:] = 0xFF
    out1, _ = orc.attention_fp8(c2, sc, pb.bt, pb.seq_lens, pb.q, 0.25)
    assert np.array_equal(out0, out1), "NaN codes"


# --------------------------------------------------------- QKV projection --

def _qkv_problem(rng, seq_lens, Hq=8, Hkv=2, D=16, hidden=24):
    pb, q, k, v, wq, wk, pos = _layer_problem(rng, seq_lens, Hq=Hq, Hkv=Hkv, D=D)
    B = len(seq_lens)
    x = random_bits(rng, (B, hidden))
    w = random_bits(rng, ((Hq + 2 * Hkv) * D, hidden), scale=0.2)
    return pb, x, w, wq, wk, pos


def pin_qkv_projection_is_the_matrix_product(orc):
    """q_rot and k_rot are norm + rotation (both pinned) of the rows of
    numpy's W @ x; v is the value rows of the same product."""
    rng = np.random.default_rng(24)
    Hq, Hkv, D = 8, 2, 16
    pb, x, w, wq, wk, pos = _qkv_problem(rng, [3, 17, 31])
    res = orc.qkv_append(x, w, wq, wk, pos, pb.seq_lens, pb.bt, pb.pool, 1e6, 1e-6, Hq, Hkv)
    for b in range(3):
        qkv = f64(w) @ f64(x[b])
        for h in range(Hq):
            want = orc.rope_neox(orc.rmsnorm(qkv[h * D:(h + 1) * D], f64(wq), 1e-6), pos[b], 1e6)
            _close(res["q_rot"][b, h], want, 1e-12, "qkv q_rot")
        for g in range(Hkv):
            row = qkv[(Hq + g) * D:(Hq + g + 1) * D]
            want = orc.rope_neox(orc.rmsnorm(row, f64(wk), 1e-6), pos[b], 1e6)
            _close(res["k_rot"][b, g], want, 1e-12, "qkv k_rot")
            _close(res["v"][b, g], qkv[(Hq + Hkv + g) * D:(Hq + Hkv + g + 1) * D], 1e-12, "qkv v")


def pin_qkv_one_hot_input_equals_the_layer_step(orc):
    """With x one-hot the projection picks one bf16 column of W exactly, so
    the fused projection must equal the (pinned) layer-step's steps 1-3 on
    those columns as q, k and v: the same q_rot, k_rot and pool bits."""
    rng = np.random.default_rng(25)
    Hq, Hkv, D, hidden = 8, 2, 16, 24
    pb, x, w, wq, wk, pos = _qkv_problem(rng, [1, 5, 16, 22], hidden=hidden)
    cols = rng.integers(0, hidden, size=4)
    x = np.zeros_like(x)
    x[np.arange(4), cols] = 0x3F80                      # 1.0 in bf16
    pool_a, pool_b = pb.pool.copy(), pb.pool.copy()
    res = orc.qkv_append(x, w, wq, wk, pos, pb.seq_lens, pb.bt, pool_a, 1e6, 1e-6, Hq, Hkv)
    picked = np.stack([w[:, c] for c in cols])           # [B][(Hq+2Hkv)*D] bf16 bits
    q = np.ascontiguousarray(picked[:, :Hq * D].reshape(4, Hq, D))
    k = np.ascontiguousarray(picked[:, Hq * D:(Hq + Hkv) * D].reshape(4, Hkv, D))
    v = np.ascontiguousarray(picked[:, (Hq + Hkv) * D:].reshape(4, Hkv, D))
    ref = orc.decode_layer(q, k, v, wq, wk, pos, pb.seq_lens, pb.bt, pool_b, 1e6, 1e-6)
    assert np.array_equal(res["q_rot"], ref["q_rot"]), "one-hot q_rot"
    assert np.array_equal(res["k_rot"], ref["k_rot"]), "one-hot k_rot"
    assert np.array_equal(pool_a, pool_b), "one-hot pool"


def pin_qkv_append_one_slot(orc):
    """Exactly slot L-1 of every (sequence, KV head, plane) changes: K gets
    bf16(k_rot), V gets bf16(v), both rounded once to nearest even."""
    rng = np.random.default_rng(26)
    Hq, Hkv = 8, 2
    pb, x, w, wq, wk, pos = _qkv_problem(rng, [1, 4, 5, 16, 22])
    before = pb.pool.copy()
    res = orc.qkv_append(x, w, wq, wk, pos, pb.seq_lens, pb.bt, pb.pool, 1e6, 1e-6, Hq, Hkv)
    changed = np.zeros(before.shape, bool)
    for b, L in enumerate(pb.seq_lens):
        page, off = pb.bt[b, (L - 1) // 4], (L - 1) % 4
        for g in range(Hkv):
            assert np.array_equal(pb.pool[page, 0, g, off], orc.f64_to_bf16_bits(res["k_rot"][b, g]))
            assert np.array_equal(pb.pool[page, 1, g, off], orc.f64_to_bf16_bits(res["v"][b, g]))
        changed[page, :, :, off] = True
    assert np.array_equal(pb.pool[~changed], before[~changed]), "append touched another slot"


# --------------------------------------------------------------- prefill --
# A chunk of n_b new tokens per sequence, packed by qo_indptr; chunk token j
# of sequence b is token t = L_b - n_b + j (L_b counted after the chunk).

def _prefill_problem(rng, seq_lens, chunks, Hq=8, Hkv=2, D=16, P=4, pos_offset=0):
    pb = Paged(rng, seq_lens, Hq=Hq, Hkv=Hkv, D=D, P=P, extra_pages=4)
    qo = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(qo[-1])
    q = random_bits(rng, (T, Hq, D))
    k = random_bits(rng, (T, Hkv, D))
    v = random_bits(rng, (T, Hkv, D))
    wq = bits_of((rng.integers(2, 6, D) / 4).astype(np.float32))
    wk = bits_of((rng.integers(2, 6, D) / 4).astype(np.float32))
    idx = np.concatenate([np.arange(L - n, L) for L, n in zip(seq_lens, chunks)]).astype(np.int32)
    return pb, qo, q, k, v, wq, wk, idx + pos_offset, idx


def pin_prefill_attention_dense_causal(orc):
    """Brute force on tiny inputs: gather each sequence's K and V densely and
    take softmax(q K^T / sqrt(D) + causal mask) V with numpy/scipy; chunk row
    j of sequence b sees keys 0 .. L_b - n_b + j."""
    rng = np.random.default_rng(31)
    seq_lens, chunks = [5, 9, 13, 4], [5, 3, 6, 1]
    pb, qo, *_ = _prefill_problem(rng, seq_lens, chunks)
    T = int(qo[-1])
    q_rot = rng.standard_normal((T, 8, 16))
    out, lse = orc.prefill_attention(pb.pool, pb.bt, qo, pb.seq_lens, q_rot, 0.25)
    for b, (L, n) in enumerate(zip(seq_lens, chunks)):
        for h in range(8):
            K, V = pb.gather(b, 0, h // 4), pb.gather(b, 1, h // 4)
            Q = q_rot[qo[b]:qo[b + 1], h]
            S = 0.25 * Q @ K.T
            mask = np.arange(L)[None, :] > (L - n + np.arange(n))[:, None]
            S[mask] = -np.inf
            _close(out[qo[b]:qo[b + 1], h], scipy.special.softmax(S, axis=1) @ V, 1e-12,
                   "causal out")
            _close(lse[qo[b]:qo[b + 1], h], scipy.special.logsumexp(S, axis=1), 1e-12,
                   "causal lse")


def pin_prefill_last_token_equals_decode(orc):
    """The chunk's last row attends to the whole sequence: the (pinned)
    decode attention of that row, bit for bit."""
    rng = np.random.default_rng(32)
    seq_lens, chunks = [7, 12, 3], [2, 5, 3]
    pb, qo, *_ = _prefill_problem(rng, seq_lens, chunks)
    q_rot = rng.standard_normal((int(qo[-1]), 8, 16))
    out, lse = orc.prefill_attention(pb.pool, pb.bt, qo, pb.seq_lens, q_rot, 0.3)
    last = qo[1:] - 1
    ref_out, ref_lse = orc.attention(pb.pool, pb.bt, pb.seq_lens,
                                     np.ascontiguousarray(q_rot[last]), 0.3)
    assert np.array_equal(out[last], ref_out) and np.array_equal(lse[last], ref_lse)


def pin_prefill_fresh_sequence_first_token_is_v(orc):
    """A sequence with no cached prefix (n_b = L_b): its first row attends
    only to token 0, so out = V_0 exactly and lse = the single score."""
    rng = np.random.default_rng(33)
    pb, qo, *_ = _prefill_problem(rng, [6, 8], [6, 3])
    q_rot = rng.standard_normal((int(qo[-1]), 8, 16))
    out, lse = orc.prefill_attention(pb.pool, pb.bt, qo, pb.seq_lens, q_rot, 0.25)
    for h in range(8):
        V0, K0 = pb.gather(0, 1, h // 4)[0], pb.gather(0, 0, h // 4)[0]
        _close(out[0, h], V0, 0.0, "first token out = v0")
        _close([lse[0, h]], [0.25 * q_rot[0, h] @ K0], 1e-12, "first token lse")


def pin_prefill_append_slots_and_rows(orc):
    """Norm and rotation of every chunk row at its own position (both
    pinned per row; positions differ from the token index here), and exactly
    the chunk's slots L-n .. L-1 change: K = bf16(k_rot), V = v's bits."""
    rng = np.random.default_rng(34)
    seq_lens, chunks = [5, 9, 13, 4], [5, 3, 6, 1]
    pb, qo, q, k, v, wq, wk, pos, idx = _prefill_problem(rng, seq_lens, chunks, pos_offset=7)
    before = pb.pool.copy()
    res = orc.prefill_append(q, k, v, wq, wk, pos, qo, pb.seq_lens, pb.bt, pb.pool, 1e6, 1e-6)
    changed = np.zeros(before.shape, bool)
    for b in range(len(seq_lens)):
        for r in range(qo[b], qo[b + 1]):
            for h in range(8):
                want = orc.rope_neox(orc.rmsnorm(f64(q[r, h]), f64(wq), 1e-6), pos[r], 1e6)
                _close(res["q_rot"][r, h], want, 0.0, "prefill q_rot")
            page, off = pb.bt[b, idx[r] // 4], idx[r] % 4
            for g in range(2):
                want = orc.rope_neox(orc.rmsnorm(f64(k[r, g]), f64(wk), 1e-6), pos[r], 1e6)
                _close(res["k_rot"][r, g], want, 0.0, "prefill k_rot")
                assert np.array_equal(pb.pool[page, 0, g, off], orc.f64_to_bf16_bits(want))
                assert np.array_equal(pb.pool[page, 1, g, off], v[r, g])
            changed[page, :, :, off] = True
    assert np.array_equal(pb.pool[~changed], before[~changed]), "append touched another slot"


def pin_prefill_chunk_of_one_is_the_decode_step(orc):
    """One new token per sequence: prefill append + attention is the
    (pinned) decode layer-step, bit for bit."""
    rng = np.random.default_rng(35)
    seq_lens = [3, 17, 31]
    pb, qo, q, k, v, wq, wk, pos, _ = _prefill_problem(rng, seq_lens, [1, 1, 1])
    pool_a, pool_b = pb.pool.copy(), pb.pool.copy()
    res = orc.prefill_append(q, k, v, wq, wk, pos, qo, pb.seq_lens, pb.bt, pool_a, 1e6, 1e-6)
    out, lse = orc.prefill_attention(pool_a, pb.bt, qo, pb.seq_lens, res["q_rot"], 0.25)
    ref = orc.decode_layer(q, k, v, wq, wk, pos, pb.seq_lens, pb.bt, pool_b, 1e6, 1e-6)
    assert np.array_equal(pool_a, pool_b) and np.array_equal(out, ref["out"])
    assert np.array_equal(lse, ref["lse"]) and np.array_equal(res["q_rot"], ref["q_rot"])


def pin_prefill_rejects_bad_chunks(orc):
    """A chunk longer than its sequence, a negative chunk or qo_indptr not
    starting at 0 is an error, not a silent read outside the sequence."""
    rng = np.random.default_rng(36)
    pb, qo, *_ = _prefill_problem(rng, [5, 9], [2, 3])
    for bad in ([0, 6, 9], [0, 2, 1], [1, 3, 5]):     # too long, negative, offset start
        q_rot = rng.standard_normal((bad[-1], 8, 16))
        try:
            orc.prefill_attention(pb.pool, pb.bt, np.array(bad, np.int32), pb.seq_lens, q_rot,
                                  0.25)
        except OracleError:
            continue
        raise AssertionError(f"qo_indptr {bad} accepted")


def pin_fp8_prefill_pow2_scales_equal_bf16(orc):
    """With power-of-two scales the dequantized pool is exact in bf16, so the
    FP8 causal prefill attention equals the (pinned) bf16 one bit for bit."""
    rng = np.random.default_rng(37)
    seq_lens, chunks = [5, 9, 13, 4], [5, 3, 6, 1]
    pb, qo, *_ = _prefill_problem(rng, seq_lens, chunks)
    codes, sc = _fp8_pool(rng, pb, pow2=True)
    deq = _torch_e4m3_values()[codes] * sc[:, :, :, None, None]
    q_rot = rng.standard_normal((int(qo[-1]), 8, 16))
    out0, lse0 = orc.prefill_attention(bits_of(deq.astype(np.float32)), pb.bt, qo,
                                       pb.seq_lens, q_rot, 0.25)
    out1, lse1 = orc.prefill_attention_fp8(codes, sc, pb.bt, qo, pb.seq_lens, q_rot, 0.25)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1), "fp8 vs bf16 prefill"


def pin_fp8_prefill_chunk_of_one_is_the_decode_step(orc):
    """One new token per sequence: the FP8 prefill append + attention is the
    (pinned) FP8 decode layer-step, codes and outputs bit for bit."""
    rng = np.random.default_rng(38)
    seq_lens = [3, 17, 31, 8]
    pb, qo, q, k, v, wq, wk, pos, _ = _prefill_problem(rng, seq_lens, [1, 1, 1, 1])
    codes, sc = _fp8_pool(rng, pb, pow2=False)
    sc[pb.bt[1, (17 - 1) // 4]] = 1e-4            # this page saturates
    a, b_ = codes.copy(), codes.copy()
    res = orc.prefill_append_fp8(q, k, v, wq, wk, pos, qo, pb.seq_lens, pb.bt, a, sc, 1e6, 1e-6)
    out, lse = orc.prefill_attention_fp8(a, sc, pb.bt, qo, pb.seq_lens, res["q_rot"], 0.25)
    ref = orc.decode_layer_fp8(q, k, v, wq, wk, pos, pb.seq_lens, pb.bt, b_, sc, 1e6, 1e-6)
    assert np.array_equal(a, b_), "fp8 prefill codes vs decode codes"
    assert np.array_equal(out, ref["out"]) and np.array_equal(lse, ref["lse"])


def pin_fp8_prefill_append_codes(orc):
    """Every chunk row's slot gets the nearest codes (brute force) of
    fp32(bf16(k_rot)) / scale_K and fp32(v) / scale_V, k_rot being the
    (pinned) bf16 prefill append's; no other slot changes."""
    rng = np.random.default_rng(39)
    seq_lens, chunks = [6, 9, 4], [4, 3, 4]
    pb, qo, q, k, v, wq, wk, pos, idx = _prefill_problem(rng, seq_lens, chunks, pos_offset=3)
    codes, sc = _fp8_pool(rng, pb, pow2=False)
    before = codes.copy()
    res = orc.prefill_append_fp8(q, k, v, wq, wk, pos, qo, pb.seq_lens, pb.bt, codes, sc, 1e6,
                                 1e-6)
    ref = orc.prefill_append(q, k, v, wq, wk, pos, qo, pb.seq_lens, pb.bt, pb.pool.copy(), 1e6,
                             1e-6)
    _close(res["k_rot"], ref["k_rot"], 0.0, "fp8 prefill k_rot")
    table = np.array([orc.e4m3_to_double(c) for c in range(0x7F)])
    changed = np.zeros(codes.shape, bool)
    for b in range(len(seq_lens)):
        for r in range(qo[b], qo[b + 1]):
            page, off = pb.bt[b, idx[r] // 4], idx[r] % 4
            for g in range(2):
                kf = f64(orc.f64_to_bf16_bits(ref["k_rot"][r, g])).astype(np.float32)
                vf = f64(v[r, g]).astype(np.float32)
                want_k = [_e4m3_nearest(float(x / sc[page, 0, g]), table) for x in kf]
                want_v = [_e4m3_nearest(float(x / sc[page, 1, g]), table) for x in vf]
                assert np.array_equal(codes[page, 0, g, off], want_k), f"K codes row {r}"
                assert np.array_equal(codes[page, 1, g, off], want_v), f"V codes row {r}"
            changed[page, :, :, off] = True
    assert np.array_equal(codes[~changed], before[~changed]), "append touched another slot"


def pin_qkv_fp8_append_codes(orc):
    """The projection into an FP8 pool: the same q_rot, k_rot and v as the
    (pinned) bf16 projection; slot L-1 of every (sequence, plane, head) gets
    the nearest codes (brute force) of the bf16 row the bf16 pool receives
    divided by the slot's scale in fp32, saturating where the scale is too
    small; no other slot changes."""
    rng = np.random.default_rng(40)
    Hq, Hkv = 8, 2
    pb, x, w, wq, wk, pos = _qkv_problem(rng, [1, 4, 5, 16, 22])
    codes, sc = _fp8_pool(rng, pb, pow2=False)
    sc[pb.bt[3, (16 - 1) // 4]] = 1e-4            # this page saturates
    before = codes.copy()
    res = orc.qkv_append_fp8(x, w, wq, wk, pos, pb.seq_lens, pb.bt, codes, sc, 1e6, 1e-6, Hq, Hkv)
    ref = orc.qkv_append(x, w, wq, wk, pos, pb.seq_lens, pb.bt, pb.pool.copy(), 1e6, 1e-6, Hq, Hkv)
    for key in ("q_rot", "k_rot", "v"):
        _close(res[key], ref[key], 0.0, f"qkv fp8 {key}")
    table = np.array([orc.e4m3_to_double(c) for c in range(0x7F)])
    changed = np.zeros(codes.shape, bool)
    saturated = 0
    for b, L in enumerate(pb.seq_lens):
        page, off = pb.bt[b, (L - 1) // 4], (L - 1) % 4
        for g in range(Hkv):
            for plane, key in ((0, "k_rot"), (1, "v")):
                row = f64(orc.f64_to_bf16_bits(ref[key][b, g])).astype(np.float32)
                want = [_e4m3_nearest(float(v_ / sc[page, plane, g]), table) for v_ in row]
                assert np.array_equal(codes[page, plane, g, off], want), f"codes b={b} {key}"
                saturated += int(np.sum((codes[page, plane, g, off] & 0x7F) == 0x7E))
        changed[page, :, :, off] = True
    assert saturated > 0, "the saturating page did not saturate"
    assert np.array_equal(codes[~changed], before[~changed]), "append touched another slot"


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
