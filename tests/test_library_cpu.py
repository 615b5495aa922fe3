"""libqdec on a machine without a GPU: it loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

from gqa_paged_kv_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q():
    qbuild.build()
    from gqa_paged_kv_gb300 import qdec
    return qdec


def declared_symbols():
    with open(os.path.join(ROOT, "include", "qdec.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(qdec_[a-z0-9_]+)\(", text)))


def test_exports_every_declared_symbol(q):
    lib = ctypes.CDLL(q.library_path())
    names = declared_symbols()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"{n} declared in qdec.h but not exported"
    assert set(names) == set(q.EXPORTS)


def test_version_and_status_strings(q):
    assert q.qdec_version() == 20000
    for st in range(7):
        assert q.status_string(st) and q.status_string(st) != "unknown status"
    assert q.status_string(99) == "unknown status"


def _shape(q, **kw):
    base = dict(batch=2, num_pages=64, max_blocks_per_seq=8, max_seq_len=128)
    base.update(kw)
    return q.Shape(**base)


def test_workspace_bytes_rejects_bad_shapes(q):
    lib = q._lib
    assert lib.qdec_workspace_bytes(None) == 0
    for kw, in [(dict(head_dim=64),), (dict(page_size=32),), (dict(num_q_heads=16),),
                (dict(batch=0),), (dict(batch=2000),), (dict(max_seq_len=129),),
                (dict(rope_theta=0.0),), (dict(eps=-1.0),), (dict(num_ctas=-1),)]:
        assert q.qdec_workspace_bytes(_shape(q, **kw)) == 0, kw


def test_step_launch_count(q):
    """qdec_step (either pool type) runs in one launch or, on the flat
    layout, two (the new-token kernel, then the decode-mode attention); bad
    shapes give 0.  The two-launch form keeps q_rot in the workspace, so the
    workspace is at least that large then."""
    assert q.qdec_step_launches(_shape(q, batch=0)) == 0
    assert q._lib.qdec_step_launches(None, 0) == 0
    for kw in (dict(), dict(batch=64, num_pages=4096, max_blocks_per_seq=64,
                            max_seq_len=1024), dict(num_ctas=7)):
        sh = _shape(q, **kw)
        for fp8 in (False, True):
            n = q.qdec_step_launches(sh, fp8_pool=fp8)
            assert n in (1, 2), kw
            if n == 2:
                assert q.qdec_workspace_bytes(sh) >= sh.batch * sh.num_q_heads * 128 * 4
    for fp8 in (False, True):  # forced grids are flat
        assert q.qdec_step_launches(_shape(q, num_ctas=7), fp8_pool=fp8) == 2


def test_entry_points_reject_null_and_misaligned_arguments(q):
    lib = q._lib
    sh = ctypes.byref(_shape(q).c())
    ok = ctypes.c_void_p(1 << 20)      # never dereferenced: rejected earlier
    bad = ctypes.c_void_p((1 << 20) + 2)
    z = ctypes.c_void_p(0)
    S = 48 * 128

    def step(shape=sh, qp=ok, qs=S, rope=z, ws=ok, ws_bytes=1 << 30, out=ok):
        # shape, q, q_stride, k, k_stride, v, v_stride, w_q, w_k, positions,
        # seq_lens, block_table, rope_table, kv_pool, workspace, bytes, out, err, stream
        return lib.qdec_step(shape, qp, qs, ok, S, ok, S, ok, ok, ok, ok, ok, rope, ok, ws,
                             ws_bytes, out, z, z)

    assert step(shape=None) == q.QDEC_ERR_INVALID_ARG
    assert step(qp=z) == q.QDEC_ERR_INVALID_ARG
    assert step(qp=bad) == q.QDEC_ERR_INVALID_ARG
    assert step(qs=S + 4) == q.QDEC_ERR_INVALID_ARG          # not a multiple of 8
    assert step(qs=16 * 128) == q.QDEC_ERR_INVALID_ARG       # shorter than the heads
    assert step(rope=bad) == q.QDEC_ERR_INVALID_ARG
    assert step(out=z) == q.QDEC_ERR_INVALID_ARG
    assert step(ws_bytes=16) == q.QDEC_ERR_WORKSPACE
    assert step(ws=z) == q.QDEC_ERR_WORKSPACE
    assert lib.qdec_attn_split(sh, ok, ok, ok, ok, z, 1 << 30, ok, z, z) == q.QDEC_ERR_WORKSPACE
    assert lib.qdec_attn_merge(sh, z, ok, 1 << 30, ok, z, z) == q.QDEC_ERR_INVALID_ARG
    # decode: workspace missing, q_rot missing or misaligned, out missing
    assert lib.qdec_attn_decode(sh, ok, ok, ok, ok, z, 1 << 30, ok, z, z) == q.QDEC_ERR_WORKSPACE
    assert lib.qdec_attn_decode(sh, z, ok, ok, ok, ok, 1 << 30, ok, z, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_attn_decode(sh, bad, ok, ok, ok, ok, 1 << 30, ok, z,
                                z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_attn_decode(sh, ok, ok, ok, ok, ok, 1 << 30, z, z, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_attn_decode(None, ok, ok, ok, ok, ok, 1 << 30, ok, z,
                                z) == q.QDEC_ERR_INVALID_ARG
    # prefill: missing qo_indptr / q_rot / out, misaligned q_rot, negative row count
    def pre_append(n=4, qo=ok, qr=ok, rt=z):
        return lib.qdec_prefill_append_rope(sh, n, ok, S, ok, S, ok, S, ok, ok, ok, rt, qo, ok, ok,
                                            ok, qr, z, z)
    assert pre_append(qo=z) == q.QDEC_ERR_INVALID_ARG
    assert pre_append(qr=z) == q.QDEC_ERR_INVALID_ARG
    assert pre_append(qr=bad) == q.QDEC_ERR_INVALID_ARG
    assert pre_append(n=-1) == q.QDEC_ERR_INVALID_ARG
    assert pre_append(rt=bad) == q.QDEC_ERR_INVALID_ARG   # a misaligned angle table
    # the prefill angle table: size, and missing or misaligned buffers
    assert lib.qdec_prefill_rope_table_bytes(2048) == 2048 * 64 * 16
    assert lib.qdec_prefill_rope_table_bytes(0) == 0 and lib.qdec_prefill_rope_table_bytes(-3) == 0
    assert lib.qdec_prefill_rope_table(sh, 4, z, ok, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_prefill_rope_table(sh, 4, ok, bad, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_prefill_rope_table(sh, -1, ok, ok, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_prefill_rope_table(None, 4, ok, ok, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_prefill_attn(sh, 4, z, ok, ok, ok, ok, ok, z, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_prefill_attn(sh, 4, ok, z, ok, ok, ok, ok, z, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_prefill_attn(sh, 4, ok, ok, ok, ok, ok, z, z, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_prefill_attn(sh, -2, ok, ok, ok, ok, ok, ok, z, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_prefill_attn(None, 4, ok, ok, ok, ok, ok, ok, z, z) == q.QDEC_ERR_INVALID_ARG
    # append without a q_rot output
    assert lib.qdec_append_rope(sh, ok, S, ok, S, ok, S, ok, ok, ok, ok, ok, z, ok, z, z,
                                z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_rope_table(sh, z, ok, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_rope_table(sh, ok, bad, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_check_error(None, z, None) == q.QDEC_ERR_INVALID_ARG
    # unsupported group size; unknown launch flag
    sh2 = ctypes.byref(_shape(q, num_q_heads=8, num_kv_heads=8).c())
    assert step(shape=sh2) == q.QDEC_ERR_UNSUPPORTED
    sh3 = ctypes.byref(_shape(q, launch_flags=4).c())
    assert step(shape=sh3) == q.QDEC_ERR_INVALID_ARG


def test_fp8_entry_points_reject_bad_arguments(q):
    """FP8 pool: null or misaligned scales, an odd number of KV heads."""
    lib = q._lib
    sh = ctypes.byref(_shape(q).c())
    ok = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p((1 << 20) + 4)
    z = ctypes.c_void_p(0)
    S = 48 * 128

    def step(shape=sh, pool=ok, scale=ok):
        # shape, q, q_stride, k, k_stride, v, v_stride, w_q, w_k, positions, seq_lens,
        # block_table, rope_table, pool, kv_scale, workspace, bytes, out, err, stream
        return lib.qdec_step_fp8(shape, ok, S, ok, S, ok, S, ok, ok, ok, ok, ok, z, pool, scale,
                                 ok, 16, ok, z, z)

    assert step(pool=z) == q.QDEC_ERR_INVALID_ARG
    assert step(pool=bad) == q.QDEC_ERR_INVALID_ARG
    assert step(scale=z) == q.QDEC_ERR_INVALID_ARG
    assert step(scale=bad) == q.QDEC_ERR_INVALID_ARG
    assert step() == q.QDEC_ERR_WORKSPACE                   # checks passed up to the workspace
    odd = ctypes.byref(_shape(q, num_q_heads=12, num_kv_heads=3).c())
    assert step(shape=odd) == q.QDEC_ERR_UNSUPPORTED
    assert lib.qdec_attn_split_fp8(odd, ok, ok, ok, ok, ok, ok, 1 << 30, ok, z,
                                   z) == q.QDEC_ERR_UNSUPPORTED
    assert lib.qdec_append_rope_fp8(sh, ok, S, ok, S, ok, S, ok, ok, ok, ok, ok, z, ok, z, ok, z,
                                    z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_attn_decode_fp8(odd, ok, ok, ok, ok, ok, ok, 1 << 30, ok, z,
                                    z) == q.QDEC_ERR_UNSUPPORTED
    assert lib.qdec_attn_decode_fp8(sh, ok, ok, z, ok, ok, ok, 1 << 30, ok, z,
                                    z) == q.QDEC_ERR_INVALID_ARG
    # prefill and the fused projection over an FP8 pool: scales required,
    # an odd number of KV heads unsupported
    assert lib.qdec_prefill_append_rope_fp8(sh, 4, ok, S, ok, S, ok, S, ok, ok, ok, z, ok, ok,
                                            ok, ok, z, ok, z, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_prefill_attn_fp8(odd, 4, ok, ok, ok, ok, ok, ok, z, 0, ok, z,
                                     z) == q.QDEC_ERR_UNSUPPORTED
    assert lib.qdec_prefill_attn_fp8(sh, 4, ok, ok, ok, ok, ok, bad, z, 0, ok, z,
                                     z) == q.QDEC_ERR_INVALID_ARG
    # the widening workspace: too small or misaligned is refused before any launch
    need = lib.qdec_prefill_fp8_workspace_bytes(sh)
    assert need > 0 and lib.qdec_prefill_fp8_workspace_bytes(None) == 0
    assert lib.qdec_prefill_attn_fp8(sh, 4, ok, ok, ok, ok, ok, ok, ok, need - 16, ok, z,
                                     z) == q.QDEC_ERR_WORKSPACE
    assert lib.qdec_prefill_attn_fp8(sh, 4, ok, ok, ok, ok, ok, ok, bad, need, ok, z,
                                     z) == q.QDEC_ERR_WORKSPACE
    assert lib.qdec_qkv_append_rope_fp8(sh, 256, ok, 256, ok, ok, ok, ok, ok, ok, ok, ok, z, ok,
                                        z, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_qkv_append_rope_fp8(odd, 256, ok, 256, ok, ok, ok, ok, ok, ok, ok, ok, ok, ok,
                                        z, z) == q.QDEC_ERR_UNSUPPORTED
    # one workspace size serves both pool types
    assert q.qdec_workspace_bytes(_shape(q, num_q_heads=12, num_kv_heads=3)) > 0


def test_rope_table_bytes(q):
    assert q.qdec_rope_table_bytes(_shape(q, batch=3)) == 3 * 64 * 16
    assert q.qdec_rope_table_bytes(_shape(q, head_dim=64)) == 0


def test_binding_refuses_host_tensors(q):
    """Every pointer the library takes is a device pointer: the Python
    binding refuses a host tensor (or anything that is not a tensor) before
    the library is entered."""
    import torch
    sh = _shape(q, batch=2)
    host = torch.zeros(64, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        q.qdec_rope_table(sh, host, host)
    with pytest.raises(ValueError, match="CUDA tensor"):
        q.qdec_check_error(host)
    with pytest.raises(ValueError, match="CUDA tensor"):
        q.qdec_attn_merge(sh, [1, 2], host, host)
    x = torch.zeros((2, 256), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        q.qdec_qkv_append_rope(sh, x, x, x, x, host, host, host, host, host, host)
