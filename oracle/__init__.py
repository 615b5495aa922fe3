"""fp64 CPU oracle for the GQA paged-KV decode layer-step (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product path (the CUDA library
and its binding) never imports, links or executes it.

The arithmetic lives in ``qdec_oracle.c`` (plain C, double precision, one
thread); this module only compiles it with gcc and marshals numpy arrays
through ctypes.  bf16 tensors cross the boundary as their raw ``uint16`` bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "qdec_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")

_CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False, src: str = SOURCE, out: str = LIBRARY) -> str:
    """Compile the oracle with gcc (no FP contraction, so x86 and Arm round
    identically).  Returns the library path."""
    stale = (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


class OracleError(RuntimeError):
    pass


_RC = {-1: "block-table entry outside the pool", -2: "seq_len outside [1, max_blocks*P]",
       -3: "chunk_pages < 1", -4: "Hq not a multiple of Hkv, or odd head_dim"}


def _check(rc: int):
    if rc != 0:
        raise OracleError(_RC.get(rc, f"oracle error {rc}"))


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"expected raw bf16 bits (uint16), got {a.dtype}"
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


_D = ctypes.c_double
_U16 = ctypes.c_uint16
_I32 = ctypes.c_int32


class Oracle:
    """ctypes view of one compiled copy of qdec_oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp, u16p, i32p = (ctypes.POINTER(_D), ctypes.POINTER(_U16), ctypes.POINTER(_I32))
        ci = ctypes.c_int
        lib.oracle_bf16_to_double.argtypes = [_U16]
        lib.oracle_bf16_to_double.restype = _D
        lib.oracle_double_to_bf16.argtypes = [_D]
        lib.oracle_double_to_bf16.restype = _U16
        lib.oracle_rmsnorm.argtypes = [dp, dp, ci, _D, dp]
        lib.oracle_rmsnorm.restype = None
        lib.oracle_rope_neox.argtypes = [dp, ci, _D, _D, dp]
        lib.oracle_rope_neox.restype = None
        lib.oracle_attention.argtypes = [ci] * 7 + [u16p, i32p, i32p, dp, _D, dp, dp]
        lib.oracle_attention.restype = ci
        lib.oracle_attention_split.argtypes = [ci] * 7 + [u16p, i32p, i32p, dp, _D, ci, dp, dp]
        lib.oracle_attention_split.restype = ci
        lib.oracle_decode_layer.argtypes = ([ci] * 7 + [u16p] * 5 + [i32p] * 3 + [u16p]
                                            + [_D] * 3 + [dp] * 4)
        lib.oracle_decode_layer.restype = ci
        u8p, f32p = ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_float)
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = _D
        lib.oracle_float_to_e4m3_satfinite.argtypes = [ctypes.c_float]
        lib.oracle_float_to_e4m3_satfinite.restype = ctypes.c_uint8
        lib.oracle_attention_fp8.argtypes = [ci] * 7 + [u8p, f32p, i32p, i32p, dp, _D, dp, dp]
        lib.oracle_attention_fp8.restype = ci
        lib.oracle_decode_layer_fp8.argtypes = ([ci] * 7 + [u16p] * 5 + [i32p] * 3
                                                + [u8p, f32p] + [_D] * 3 + [dp] * 4)
        lib.oracle_decode_layer_fp8.restype = ci
        lib.oracle_qkv_append.argtypes = ([ci] * 8 + [u16p] * 4 + [i32p] * 3 + [u16p]
                                          + [_D] * 2 + [dp] * 3)
        lib.oracle_qkv_append.restype = ci
        lib.oracle_prefill_append.argtypes = ([ci] * 7 + [u16p] * 5 + [i32p] * 4 + [u16p]
                                              + [_D] * 2 + [dp] * 2)
        lib.oracle_prefill_append.restype = ci
        lib.oracle_prefill_attention.argtypes = ([ci] * 7 + [u16p] + [i32p] * 3 + [dp, _D]
                                                 + [dp] * 2)
        lib.oracle_prefill_attention.restype = ci
        lib.oracle_qkv_append_fp8.argtypes = ([ci] * 8 + [u16p] * 4 + [i32p] * 3 + [u8p, f32p]
                                              + [_D] * 2 + [dp] * 3)
        lib.oracle_qkv_append_fp8.restype = ci
        lib.oracle_prefill_append_fp8.argtypes = ([ci] * 7 + [u16p] * 5 + [i32p] * 4
                                                  + [u8p, f32p] + [_D] * 2 + [dp] * 2)
        lib.oracle_prefill_append_fp8.restype = ci
        lib.oracle_prefill_attention_fp8.argtypes = ([ci] * 7 + [u8p, f32p] + [i32p] * 3
                                                     + [dp, _D] + [dp] * 2)
        lib.oracle_prefill_attention_fp8.restype = ci
        self.lib = lib
        self.path = path

    # -------------------------------------------------------------- scalars
    def bf16_to_double(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(int(bits))

    def double_to_bf16(self, x: float) -> int:
        return int(self.lib.oracle_double_to_bf16(float(x)))

    def f64_to_bf16_bits(self, a) -> np.ndarray:
        """Round every element straight from double to bf16 (RNE)."""
        flat = np.asarray(a, dtype=np.float64).ravel()
        f = self.lib.oracle_double_to_bf16
        out = np.fromiter((f(float(x)) for x in flat), dtype=np.uint16, count=flat.size)
        return out.reshape(np.shape(a))

    # -------------------------------------------------------------- per row
    def rmsnorm(self, x, w, eps: float) -> np.ndarray:
        x, w = _f64(x), _f64(w)
        y = np.empty_like(x)
        self.lib.oracle_rmsnorm(_ptr(x, _D), _ptr(w, _D), x.size, float(eps), _ptr(y, _D))
        return y

    def rope_neox(self, x, pos: float, theta: float) -> np.ndarray:
        x = _f64(x)
        y = np.empty_like(x)
        self.lib.oracle_rope_neox(_ptr(x, _D), x.size, float(pos), float(theta), _ptr(y, _D))
        return y

    # ------------------------------------------------------------ attention
    @staticmethod
    def _dims(pool, block_table, q_rot):
        num_pages, two, Hkv, P, D = pool.shape
        assert two == 2
        B, Hq, D2 = q_rot.shape
        assert D2 == D
        return B, Hq, Hkv, D, P, num_pages, block_table.shape[1]

    def attention(self, pool, block_table, seq_lens, q_rot, scale: float):
        """Paged softmax attention with q_rot given (double [B][Hq][D]).
        Returns (out [B][Hq][D], lse [B][Hq]), both double."""
        pool, bt, sl, q = _u16(pool), _i32(block_table), _i32(seq_lens), _f64(q_rot)
        out = np.empty(q.shape, np.float64)
        lse = np.empty(q.shape[:2], np.float64)
        _check(self.lib.oracle_attention(*self._dims(pool, bt, q), _ptr(pool, _U16),
                                         _ptr(bt, _I32), _ptr(sl, _I32), _ptr(q, _D),
                                         float(scale), _ptr(out, _D), _ptr(lse, _D)))
        return out, lse

    def attention_split(self, pool, block_table, seq_lens, q_rot, scale: float,
                        chunk_pages: int):
        """Same as :meth:`attention`, through per-chunk partials and the LSE merge."""
        pool, bt, sl, q = _u16(pool), _i32(block_table), _i32(seq_lens), _f64(q_rot)
        out = np.empty(q.shape, np.float64)
        lse = np.empty(q.shape[:2], np.float64)
        _check(self.lib.oracle_attention_split(*self._dims(pool, bt, q), _ptr(pool, _U16),
                                               _ptr(bt, _I32), _ptr(sl, _I32), _ptr(q, _D),
                                               float(scale), int(chunk_pages),
                                               _ptr(out, _D), _ptr(lse, _D)))
        return out, lse

    def decode_layer(self, q, k, v, w_q, w_k, positions, seq_lens, block_table, pool,
                     rope_theta: float, eps: float, scale: float = 0.0):
        """One decode layer-step.  ``pool`` (uint16 [num_pages][2][Hkv][P][D])
        is updated in place by the append.  bf16 inputs are uint16 bit arrays:
        q [B][Hq][D], k/v [B][Hkv][D], w_q/w_k [D].

        Returns a dict of double arrays: q_rot, k_rot (unrounded), out, lse."""
        q, k, v = _u16(q), _u16(k), _u16(v)
        w_q, w_k = _u16(w_q), _u16(w_k)
        pos, sl, bt = _i32(positions), _i32(seq_lens), _i32(block_table)
        assert pool.dtype == np.uint16 and pool.flags["C_CONTIGUOUS"], \
            "pool must be a contiguous uint16 array"
        B, Hq, D = q.shape
        num_pages, _, Hkv, P, D2 = pool.shape
        assert D2 == D and k.shape == (B, Hkv, D) and v.shape == (B, Hkv, D)
        res = {"q_rot": np.empty((B, Hq, D)), "k_rot": np.empty((B, Hkv, D)),
               "out": np.empty((B, Hq, D)), "lse": np.empty((B, Hq))}
        _check(self.lib.oracle_decode_layer(
            B, Hq, Hkv, D, P, num_pages, bt.shape[1],
            _ptr(q, _U16), _ptr(k, _U16), _ptr(v, _U16), _ptr(w_q, _U16), _ptr(w_k, _U16),
            _ptr(pos, _I32), _ptr(sl, _I32), _ptr(bt, _I32), _ptr(pool, _U16),
            float(rope_theta), float(eps), float(scale),
            _ptr(res["q_rot"], _D), _ptr(res["k_rot"], _D), _ptr(res["out"], _D),
            _ptr(res["lse"], _D)))
        return res


    # ------------------------------------------------------------- fp8 KV
    def e4m3_to_double(self, code: int) -> float:
        return self.lib.oracle_e4m3_to_double(int(code))

    def float_to_e4m3(self, x: float) -> int:
        """E4M3 code of a binary32 value (nearest-even, saturating)."""
        return int(self.lib.oracle_float_to_e4m3_satfinite(float(x)))

    def e4m3_codes(self, a) -> np.ndarray:
        """float_to_e4m3 of every element (taken as binary32)."""
        flat = np.asarray(a, dtype=np.float32).ravel()
        f = self.lib.oracle_float_to_e4m3_satfinite
        out = np.fromiter((f(float(x)) for x in flat), dtype=np.uint8, count=flat.size)
        return out.reshape(np.shape(a))

    @staticmethod
    def _fp8_args(pool8, kv_scale):
        pool8 = np.ascontiguousarray(pool8)
        assert pool8.dtype == np.uint8, f"expected e4m3 codes (uint8), got {pool8.dtype}"
        sc = np.ascontiguousarray(kv_scale, dtype=np.float32)
        num_pages, two, Hkv = pool8.shape[:3]
        assert sc.shape == (num_pages, two, Hkv), (sc.shape, pool8.shape)
        return pool8, sc

    def attention_fp8(self, pool8, kv_scale, block_table, seq_lens, q_rot, scale: float):
        """:meth:`attention` over an FP8 pool (uint8 [pages][2][Hkv][P][D])
        with scales kv_scale (float32 [pages][2][Hkv])."""
        pool8, sc = self._fp8_args(pool8, kv_scale)
        bt, sl, q = _i32(block_table), _i32(seq_lens), _f64(q_rot)
        out = np.empty(q.shape, np.float64)
        lse = np.empty(q.shape[:2], np.float64)
        _check(self.lib.oracle_attention_fp8(
            *self._dims(pool8, bt, q), _ptr(pool8, ctypes.c_uint8), _ptr(sc, ctypes.c_float),
            _ptr(bt, _I32), _ptr(sl, _I32), _ptr(q, _D), float(scale), _ptr(out, _D),
            _ptr(lse, _D)))
        return out, lse

    def decode_layer_fp8(self, q, k, v, w_q, w_k, positions, seq_lens, block_table, pool8,
                         kv_scale, rope_theta: float, eps: float, scale: float = 0.0):
        """:meth:`decode_layer` with an FP8 pool; ``pool8`` (uint8, contiguous)
        is updated in place by the append, ``kv_scale`` is read only."""
        q, k, v = _u16(q), _u16(k), _u16(v)
        w_q, w_k = _u16(w_q), _u16(w_k)
        pos, sl, bt = _i32(positions), _i32(seq_lens), _i32(block_table)
        assert pool8.dtype == np.uint8 and pool8.flags["C_CONTIGUOUS"], \
            "pool8 must be a contiguous uint8 array"
        _, sc = self._fp8_args(pool8, kv_scale)
        B, Hq, D = q.shape
        num_pages, _, Hkv, P, D2 = pool8.shape
        assert D2 == D and k.shape == (B, Hkv, D) and v.shape == (B, Hkv, D)
        res = {"q_rot": np.empty((B, Hq, D)), "k_rot": np.empty((B, Hkv, D)),
               "out": np.empty((B, Hq, D)), "lse": np.empty((B, Hq))}
        _check(self.lib.oracle_decode_layer_fp8(
            B, Hq, Hkv, D, P, num_pages, bt.shape[1],
            _ptr(q, _U16), _ptr(k, _U16), _ptr(v, _U16), _ptr(w_q, _U16), _ptr(w_k, _U16),
            _ptr(pos, _I32), _ptr(sl, _I32), _ptr(bt, _I32), _ptr(pool8, ctypes.c_uint8),
            _ptr(sc, ctypes.c_float), float(rope_theta), float(eps), float(scale),
            _ptr(res["q_rot"], _D), _ptr(res["k_rot"], _D), _ptr(res["out"], _D),
            _ptr(res["lse"], _D)))
        return res


    # ------------------------------------------------------ QKV projection
    def qkv_append(self, x, w_qkv, w_q, w_k, positions, seq_lens, block_table, pool,
                   rope_theta: float, eps: float, num_q_heads: int, num_kv_heads: int):
        """The merged QKV projection fused with norm, rotation and append.
        x [B][hidden], w_qkv [(Hq+2Hkv)*D][hidden] (bf16 as uint16); ``pool``
        (uint16 [pages][2][Hkv][P][D]) is updated in place.  Returns double
        arrays q_rot [B][Hq][D], k_rot and v [B][Hkv][D] (unrounded)."""
        x, w, w_q, w_k = _u16(x), _u16(w_qkv), _u16(w_q), _u16(w_k)
        pos, sl, bt = _i32(positions), _i32(seq_lens), _i32(block_table)
        assert pool.dtype == np.uint16 and pool.flags["C_CONTIGUOUS"]
        B, hidden = x.shape
        num_pages, _, Hkv, P, D = pool.shape
        Hq = num_q_heads
        assert Hkv == num_kv_heads and w.shape == ((Hq + 2 * Hkv) * D, hidden)
        res = {"q_rot": np.empty((B, Hq, D)), "k_rot": np.empty((B, Hkv, D)),
               "v": np.empty((B, Hkv, D))}
        _check(self.lib.oracle_qkv_append(
            B, Hq, Hkv, D, P, num_pages, bt.shape[1], hidden,
            _ptr(x, _U16), _ptr(w, _U16), _ptr(w_q, _U16), _ptr(w_k, _U16),
            _ptr(pos, _I32), _ptr(sl, _I32), _ptr(bt, _I32), _ptr(pool, _U16),
            float(rope_theta), float(eps),
            _ptr(res["q_rot"], _D), _ptr(res["k_rot"], _D), _ptr(res["v"], _D)))
        return res


    def qkv_append_fp8(self, x, w_qkv, w_q, w_k, positions, seq_lens, block_table, pool8,
                       kv_scale, rope_theta: float, eps: float, num_q_heads: int,
                       num_kv_heads: int):
        """:meth:`qkv_append` with an FP8 pool (uint8, updated in place) and its
        scales (float32 [pages][2][Hkv], read only)."""
        x, w, w_q, w_k = _u16(x), _u16(w_qkv), _u16(w_q), _u16(w_k)
        pos, sl, bt = _i32(positions), _i32(seq_lens), _i32(block_table)
        assert pool8.dtype == np.uint8 and pool8.flags["C_CONTIGUOUS"]
        _, sc = self._fp8_args(pool8, kv_scale)
        B, hidden = x.shape
        num_pages, _, Hkv, P, D = pool8.shape
        Hq = num_q_heads
        assert Hkv == num_kv_heads and w.shape == ((Hq + 2 * Hkv) * D, hidden)
        res = {"q_rot": np.empty((B, Hq, D)), "k_rot": np.empty((B, Hkv, D)),
               "v": np.empty((B, Hkv, D))}
        _check(self.lib.oracle_qkv_append_fp8(
            B, Hq, Hkv, D, P, num_pages, bt.shape[1], hidden,
            _ptr(x, _U16), _ptr(w, _U16), _ptr(w_q, _U16), _ptr(w_k, _U16),
            _ptr(pos, _I32), _ptr(sl, _I32), _ptr(bt, _I32), _ptr(pool8, ctypes.c_uint8),
            _ptr(sc, ctypes.c_float), float(rope_theta), float(eps),
            _ptr(res["q_rot"], _D), _ptr(res["k_rot"], _D), _ptr(res["v"], _D)))
        return res

    # ------------------------------------------------------------- prefill
    def prefill_append(self, q, k, v, w_q, w_k, positions, qo_indptr, seq_lens, block_table,
                       pool, rope_theta: float, eps: float):
        """Norm, rotation and append of a chunk of tokens per sequence.
        q [T][Hq][D], k/v [T][Hkv][D] (bf16 as uint16), positions [T],
        qo_indptr [B+1], seq_lens [B] (after the chunk); ``pool`` updated in
        place.  Returns double arrays q_rot [T][Hq][D], k_rot [T][Hkv][D]."""
        q, k, v, w_q, w_k = _u16(q), _u16(k), _u16(v), _u16(w_q), _u16(w_k)
        pos, qo, sl, bt = _i32(positions), _i32(qo_indptr), _i32(seq_lens), _i32(block_table)
        assert pool.dtype == np.uint16 and pool.flags["C_CONTIGUOUS"]
        T, Hq, D = q.shape
        num_pages, _, Hkv, P, D2 = pool.shape
        B = sl.shape[0]
        assert D2 == D and k.shape == (T, Hkv, D) and v.shape == (T, Hkv, D)
        assert qo.shape == (B + 1,) and pos.shape == (T,) and qo[-1] == T
        res = {"q_rot": np.empty((T, Hq, D)), "k_rot": np.empty((T, Hkv, D))}
        _check(self.lib.oracle_prefill_append(
            B, Hq, Hkv, D, P, num_pages, bt.shape[1],
            _ptr(q, _U16), _ptr(k, _U16), _ptr(v, _U16), _ptr(w_q, _U16), _ptr(w_k, _U16),
            _ptr(pos, _I32), _ptr(qo, _I32), _ptr(sl, _I32), _ptr(bt, _I32), _ptr(pool, _U16),
            float(rope_theta), float(eps), _ptr(res["q_rot"], _D), _ptr(res["k_rot"], _D)))
        return res

    def prefill_attention(self, pool, block_table, qo_indptr, seq_lens, q_rot, scale: float):
        """Causal paged attention of the chunk rows q_rot (double [T][Hq][D]).
        Returns (out [T][Hq][D], lse [T][Hq]), both double."""
        pool, bt, qo, sl, q = (_u16(pool), _i32(block_table), _i32(qo_indptr), _i32(seq_lens),
                               _f64(q_rot))
        B = sl.shape[0]
        assert qo.shape == (B + 1,) and qo[-1] == q.shape[0]
        num_pages, _, Hkv, P, D = pool.shape
        out = np.empty(q.shape, np.float64)
        lse = np.empty(q.shape[:2], np.float64)
        _check(self.lib.oracle_prefill_attention(
            B, q.shape[1], Hkv, D, P, num_pages, bt.shape[1], _ptr(pool, _U16), _ptr(bt, _I32),
            _ptr(qo, _I32), _ptr(sl, _I32), _ptr(q, _D), float(scale), _ptr(out, _D),
            _ptr(lse, _D)))
        return out, lse


    def prefill_append_fp8(self, q, k, v, w_q, w_k, positions, qo_indptr, seq_lens,
                           block_table, pool8, kv_scale, rope_theta: float, eps: float):
        """:meth:`prefill_append` with an FP8 pool (uint8, updated in place)
        and its scales kv_scale (float32 [pages][2][Hkv], read only)."""
        q, k, v, w_q, w_k = _u16(q), _u16(k), _u16(v), _u16(w_q), _u16(w_k)
        pos, qo, sl, bt = _i32(positions), _i32(qo_indptr), _i32(seq_lens), _i32(block_table)
        assert pool8.dtype == np.uint8 and pool8.flags["C_CONTIGUOUS"]
        _, sc = self._fp8_args(pool8, kv_scale)
        T, Hq, D = q.shape
        num_pages, _, Hkv, P, D2 = pool8.shape
        B = sl.shape[0]
        assert D2 == D and k.shape == (T, Hkv, D) and qo.shape == (B + 1,) and qo[-1] == T
        res = {"q_rot": np.empty((T, Hq, D)), "k_rot": np.empty((T, Hkv, D))}
        _check(self.lib.oracle_prefill_append_fp8(
            B, Hq, Hkv, D, P, num_pages, bt.shape[1],
            _ptr(q, _U16), _ptr(k, _U16), _ptr(v, _U16), _ptr(w_q, _U16), _ptr(w_k, _U16),
            _ptr(pos, _I32), _ptr(qo, _I32), _ptr(sl, _I32), _ptr(bt, _I32),
            _ptr(pool8, ctypes.c_uint8), _ptr(sc, ctypes.c_float), float(rope_theta),
            float(eps), _ptr(res["q_rot"], _D), _ptr(res["k_rot"], _D)))
        return res

    def prefill_attention_fp8(self, pool8, kv_scale, block_table, qo_indptr, seq_lens, q_rot,
                              scale: float):
        """:meth:`prefill_attention` over an FP8 pool."""
        pool8, sc = self._fp8_args(pool8, kv_scale)
        bt, qo, sl, q = _i32(block_table), _i32(qo_indptr), _i32(seq_lens), _f64(q_rot)
        B = sl.shape[0]
        assert qo.shape == (B + 1,) and qo[-1] == q.shape[0]
        num_pages, _, Hkv, P, D = pool8.shape
        out = np.empty(q.shape, np.float64)
        lse = np.empty(q.shape[:2], np.float64)
        _check(self.lib.oracle_prefill_attention_fp8(
            B, q.shape[1], Hkv, D, P, num_pages, bt.shape[1], _ptr(pool8, ctypes.c_uint8),
            _ptr(sc, ctypes.c_float), _ptr(bt, _I32), _ptr(qo, _I32), _ptr(sl, _I32),
            _ptr(q, _D), float(scale), _ptr(out, _D), _ptr(lse, _D)))
        return out, lse


_default = None


def default() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def bf16_bits_to_f64(a) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a 16-bit shift: no rounding)."""
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(a) -> np.ndarray:
    return default().f64_to_bf16_bits(a)


def rmsnorm(x, w, eps):
    return default().rmsnorm(x, w, eps)


def rope_neox(x, pos, theta):
    return default().rope_neox(x, pos, theta)


def attention(pool, block_table, seq_lens, q_rot, scale):
    return default().attention(pool, block_table, seq_lens, q_rot, scale)


def attention_split(pool, block_table, seq_lens, q_rot, scale, chunk_pages):
    return default().attention_split(pool, block_table, seq_lens, q_rot, scale, chunk_pages)


def decode_layer(*args, **kwargs):
    return default().decode_layer(*args, **kwargs)


def attention_fp8(pool8, kv_scale, block_table, seq_lens, q_rot, scale):
    return default().attention_fp8(pool8, kv_scale, block_table, seq_lens, q_rot, scale)


def decode_layer_fp8(*args, **kwargs):
    return default().decode_layer_fp8(*args, **kwargs)


def qkv_append(*args, **kwargs):
    return default().qkv_append(*args, **kwargs)


def prefill_append(*args, **kwargs):
    return default().prefill_append(*args, **kwargs)


def prefill_attention(pool, block_table, qo_indptr, seq_lens, q_rot, scale):
    return default().prefill_attention(pool, block_table, qo_indptr, seq_lens, q_rot, scale)


def prefill_append_fp8(*args, **kwargs):
    return default().prefill_append_fp8(*args, **kwargs)


def prefill_attention_fp8(*args, **kwargs):
    return default().prefill_attention_fp8(*args, **kwargs)


def qkv_append_fp8(*args, **kwargs):
    return default().qkv_append_fp8(*args, **kwargs)
