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
    return sorted(set(re.findall(r"\b(qdec_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(q):
    lib = ctypes.CDLL(q.library_path())
    names = declared_symbols()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"{n} declared in qdec.h but not exported"
    assert set(names) == set(q.EXPORTS)


def test_version_and_status_strings(q):
    assert q.qdec_version() == 10000
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


def test_entry_points_reject_null_and_misaligned_arguments(q):
    lib = q._lib
    sh = ctypes.byref(_shape(q).c())
    ok_ptr = ctypes.c_void_p(1 << 20)      # never dereferenced: rejected earlier
    bad_ptr = ctypes.c_void_p((1 << 20) + 2)
    z = ctypes.c_void_p(0)
    # null shape
    assert lib.qdec_step(None, *([z, 0] * 3), *([z] * 6), z, 0, z, z, z) == q.QDEC_ERR_INVALID_ARG
    # null q
    assert lib.qdec_step(sh, z, 48 * 128, ok_ptr, 48 * 128, ok_ptr, 48 * 128, *([ok_ptr] * 6),
                         ok_ptr, 1 << 30, ok_ptr, z, z) == q.QDEC_ERR_INVALID_ARG
    # misaligned q
    assert lib.qdec_step(sh, bad_ptr, 48 * 128, ok_ptr, 48 * 128, ok_ptr, 48 * 128,
                         *([ok_ptr] * 6), ok_ptr, 1 << 30, ok_ptr, z, z) == q.QDEC_ERR_INVALID_ARG
    # stride not a multiple of 8 / shorter than the heads
    assert lib.qdec_step(sh, ok_ptr, 48 * 128 + 4, ok_ptr, 48 * 128, ok_ptr, 48 * 128,
                         *([ok_ptr] * 6), ok_ptr, 1 << 30, ok_ptr, z, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_step(sh, ok_ptr, 16 * 128, ok_ptr, 48 * 128, ok_ptr, 48 * 128,
                         *([ok_ptr] * 6), ok_ptr, 1 << 30, ok_ptr, z, z) == q.QDEC_ERR_INVALID_ARG
    # workspace too small / missing
    assert lib.qdec_step(sh, *([ok_ptr, 48 * 128] * 3), *([ok_ptr] * 6), ok_ptr, 16, ok_ptr,
                         z, z) == q.QDEC_ERR_WORKSPACE
    assert lib.qdec_attn_split(sh, ok_ptr, ok_ptr, ok_ptr, ok_ptr, z, 1 << 30, ok_ptr, z,
                               z) == q.QDEC_ERR_WORKSPACE
    assert lib.qdec_attn_merge(sh, z, ok_ptr, 1 << 30, ok_ptr, z, z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_append_rope(sh, *([ok_ptr, 48 * 128] * 3), *([ok_ptr] * 6), z, z,
                                z) == q.QDEC_ERR_INVALID_ARG
    assert lib.qdec_check_error(None, z, None) == q.QDEC_ERR_INVALID_ARG
    # unsupported group size
    sh2 = ctypes.byref(_shape(q, num_q_heads=8, num_kv_heads=8).c())
    assert lib.qdec_step(sh2, *([ok_ptr, 48 * 128] * 3), *([ok_ptr] * 6), ok_ptr, 1 << 30,
                         ok_ptr, z, z) == q.QDEC_ERR_UNSUPPORTED
