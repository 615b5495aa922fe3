"""Python binding of libqdec (ctypes): argument marshalling only.

Every function here has the name of the C entry point it calls, takes torch
tensors that already live on the current CUDA device, passes their raw
pointers and the current stream, and raises :class:`QdecError` on a non-OK
status.  A tensor that is not on the current CUDA device is refused with
ValueError before the library is entered.  All arithmetic runs in the
library's kernels; if the library is missing or cannot be loaded, importing
this module fails.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libqdec.so")

QDEC_OK = 0
QDEC_ERR_INVALID_ARG = 1
QDEC_ERR_UNSUPPORTED = 2
QDEC_ERR_WORKSPACE = 3
QDEC_ERR_CUDA = 4
QDEC_ERR_DEVICE_BOUNDS = 5
QDEC_ERR_TIMEOUT = 6

QDEC_LAUNCH_OVERLAP_PREVIOUS = 1
QDEC_LAUNCH_PREFILL_PAGES_READY = 2

QDEC_FLAG_BAD_PAGE = 1
QDEC_FLAG_BAD_SEQLEN = 2
QDEC_FLAG_TIMEOUT = 4
QDEC_FLAG_BAD_INDEX = 8
QDEC_LAUNCH_TEST_WITHHOLD_TILE = 1 << 30

# Every symbol include/qdec.h declares.
EXPORTS = ("qdec_workspace_bytes", "qdec_step_launches", "qdec_workspace_init",
           "qdec_rope_table_bytes", "qdec_rope_table", "qdec_append_rope", "qdec_attn_split", "qdec_attn_merge",
           "qdec_attn_decode", "qdec_step", "qdec_qkv_append_rope", "qdec_qkv_pack_weights",
           "qdec_append_rope_fp8", "qdec_attn_split_fp8", "qdec_attn_decode_fp8",
           "qdec_prefill_append_rope", "qdec_prefill_attn", "qdec_prefill_append_rope_fp8",
           "qdec_prefill_attn_fp8", "qdec_prefill_fp8_workspace_bytes", "qdec_qkv_append_rope_fp8",
           "qdec_step_fp8", "qdec_prefill_rope_table_bytes", "qdec_prefill_rope_table",
           "qdec_step_static_scratch", "qdec_check_error", "qdec_status_string", "qdec_version")

QDEC_STATIC_SCRATCH_BYTES = 4 << 20


class QdecShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("eps", ctypes.c_float),
                ("sm_scale", ctypes.c_float), ("num_ctas", ctypes.c_int32),
                ("launch_flags", ctypes.c_int32)]


@dataclass
class Shape:
    batch: int
    num_pages: int
    max_blocks_per_seq: int
    max_seq_len: int
    num_q_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    page_size: int = 16
    rope_theta: float = 1.0e6
    eps: float = 1.0e-6
    sm_scale: float = 0.0
    num_ctas: int = 0
    launch_flags: int = 0

    def c(self) -> QdecShape:
        return QdecShape(self.batch, self.num_q_heads, self.num_kv_heads, self.head_dim,
                         self.page_size, self.num_pages, self.max_blocks_per_seq,
                         self.max_seq_len, self.rope_theta, self.eps, self.sm_scale,
                         self.num_ctas, self.launch_flags)


class QdecError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libqdec.so not built ({_LIB_PATH}); run gqa_paged_kv_gb300/build.py")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    sp = ctypes.POINTER(QdecShape)
    st = ctypes.c_int
    lib.qdec_workspace_bytes.argtypes = [sp]
    lib.qdec_workspace_bytes.restype = sz
    lib.qdec_step_launches.argtypes = [sp, ctypes.c_int]
    lib.qdec_step_launches.restype = ctypes.c_int
    lib.qdec_workspace_init.argtypes = [sp, vp, sz, vp]
    lib.qdec_workspace_init.restype = st
    lib.qdec_rope_table_bytes.argtypes = [sp]
    lib.qdec_rope_table_bytes.restype = sz
    lib.qdec_rope_table.argtypes = [sp, vp, vp, vp]
    lib.qdec_rope_table.restype = st
    lib.qdec_append_rope.argtypes = [sp, vp, i64, vp, i64, vp, i64, vp, vp, vp, vp, vp, vp, vp,
                                     vp, vp, vp]
    lib.qdec_append_rope.restype = st
    lib.qdec_attn_split.argtypes = [sp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    lib.qdec_attn_split.restype = st
    lib.qdec_attn_merge.argtypes = [sp, vp, vp, sz, vp, vp, vp]
    lib.qdec_attn_merge.restype = st
    lib.qdec_attn_decode.argtypes = [sp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    lib.qdec_attn_decode.restype = st
    lib.qdec_prefill_append_rope.argtypes = [sp, ctypes.c_int32, vp, i64, vp, i64, vp, i64, vp,
                                             vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.qdec_prefill_append_rope.restype = st
    lib.qdec_prefill_attn.argtypes = [sp, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.qdec_prefill_attn.restype = st
    lib.qdec_prefill_append_rope_fp8.argtypes = [sp, ctypes.c_int32, vp, i64, vp, i64, vp, i64,
                                                 vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.qdec_prefill_rope_table_bytes.argtypes = [ctypes.c_int32]
    lib.qdec_prefill_rope_table_bytes.restype = sz
    lib.qdec_prefill_rope_table.argtypes = [sp, ctypes.c_int32, vp, vp, vp]
    lib.qdec_prefill_rope_table.restype = st
    lib.qdec_prefill_append_rope_fp8.restype = st
    lib.qdec_prefill_attn_fp8.argtypes = [sp, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp, sz, vp,
                                          vp, vp]
    lib.qdec_prefill_attn_fp8.restype = st
    lib.qdec_prefill_fp8_workspace_bytes.argtypes = [sp]
    lib.qdec_prefill_fp8_workspace_bytes.restype = sz
    lib.qdec_step.argtypes = [sp, vp, i64, vp, i64, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                              vp, vp, vp]
    lib.qdec_step.restype = st
    lib.qdec_qkv_append_rope.argtypes = [sp, ctypes.c_int32, vp, i64, vp, vp, vp, vp, vp, vp, vp,
                                         vp, vp, vp, vp]
    lib.qdec_qkv_append_rope.restype = st
    lib.qdec_qkv_append_rope_fp8.argtypes = [sp, ctypes.c_int32, vp, i64, vp, vp, vp, vp, vp,
                                             vp, vp, vp, vp, vp, vp, vp]
    lib.qdec_qkv_append_rope_fp8.restype = st
    lib.qdec_qkv_pack_weights.argtypes = [sp, ctypes.c_int32, vp, vp, vp]
    lib.qdec_qkv_pack_weights.restype = st
    lib.qdec_append_rope_fp8.argtypes = [sp, vp, i64, vp, i64, vp, i64, vp, vp, vp, vp, vp, vp,
                                         vp, vp, vp, vp, vp]
    lib.qdec_append_rope_fp8.restype = st
    lib.qdec_attn_split_fp8.argtypes = [sp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    lib.qdec_attn_split_fp8.restype = st
    lib.qdec_attn_decode_fp8.argtypes = [sp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    lib.qdec_attn_decode_fp8.restype = st
    lib.qdec_step_fp8.argtypes = [sp, vp, i64, vp, i64, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                  vp, sz, vp, vp, vp]
    lib.qdec_step_fp8.restype = st
    lib.qdec_step_static_scratch.argtypes = [sp, vp, i64, vp, i64, vp, i64, vp, vp, vp, vp, vp,
                                             vp, vp, vp, vp, vp]
    lib.qdec_step_static_scratch.restype = st
    lib.qdec_check_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
    lib.qdec_check_error.restype = st
    lib.qdec_status_string.argtypes = [st]
    lib.qdec_status_string.restype = ctypes.c_char_p
    lib.qdec_version.argtypes = []
    lib.qdec_version.restype = ctypes.c_int32
    return lib


_lib = _load()


def library_path() -> str:
    return _LIB_PATH


def status_string(status: int) -> str:
    return _lib.qdec_status_string(int(status)).decode()


def qdec_version() -> int:
    return int(_lib.qdec_version())


def _ptr(t) -> int:
    """Device address of a tensor argument (None passes NULL where the C ABI
    allows it).  Every pointer the library takes is a device pointer on the
    current device, so a host tensor, or one on another GPU, is refused here
    rather than handed to a kernel as an address it cannot use."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got {type(t).__name__}"
                         + (f" on {t.device}" if isinstance(t, torch.Tensor) else ""))
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensor on {t.device}, but the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _rows(t: torch.Tensor, what: str) -> int:
    """Sequence stride (elements) of a [B][H][D] view whose head rows are contiguous."""
    if t.dtype != torch.bfloat16 or t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError(f"{what}: expected a bf16 [B][H][D] view with contiguous head rows")
    return t.stride(0)


def _raise(status: int, what: str):
    if status != QDEC_OK:
        raise QdecError(status, what)


def qdec_workspace_bytes(shape: Shape) -> int:
    return int(_lib.qdec_workspace_bytes(ctypes.byref(shape.c())))


def qdec_step_launches(shape: Shape, fp8_pool: bool = False) -> int:
    return int(_lib.qdec_step_launches(ctypes.byref(shape.c()), 1 if fp8_pool else 0))


def qdec_workspace_init(shape: Shape, workspace: torch.Tensor, stream=None):
    _raise(_lib.qdec_workspace_init(ctypes.byref(shape.c()), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _stream(stream)), "qdec_workspace_init")


def qdec_rope_table_bytes(shape: Shape) -> int:
    return int(_lib.qdec_rope_table_bytes(ctypes.byref(shape.c())))


def qdec_rope_table(shape: Shape, positions, rope_table, stream=None):
    _raise(_lib.qdec_rope_table(ctypes.byref(shape.c()), _ptr(positions), _ptr(rope_table),
                                _stream(stream)), "qdec_rope_table")


def qdec_append_rope(shape: Shape, q, k, v, q_norm_w, k_norm_w, positions, seq_lens,
                     block_table, kv_pool, q_rot, err_flag=None, stream=None, rope_table=None):
    _raise(_lib.qdec_append_rope(
        ctypes.byref(shape.c()), _ptr(q), _rows(q, "q"), _ptr(k), _rows(k, "k"), _ptr(v),
        _rows(v, "v"), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions), _ptr(seq_lens),
        _ptr(block_table), _ptr(rope_table), _ptr(kv_pool), _ptr(q_rot), _ptr(err_flag),
        _stream(stream)), "qdec_append_rope")


def qdec_attn_split(shape: Shape, q_rot, kv_pool, block_table, seq_lens, workspace, out,
                    err_flag=None, stream=None):
    _raise(_lib.qdec_attn_split(
        ctypes.byref(shape.c()), _ptr(q_rot), _ptr(kv_pool), _ptr(block_table), _ptr(seq_lens),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        _ptr(err_flag), _stream(stream)), "qdec_attn_split")


def qdec_attn_decode(shape: Shape, q_rot, kv_pool, block_table, seq_lens, workspace, out,
                     err_flag=None, stream=None):
    _raise(_lib.qdec_attn_decode(
        ctypes.byref(shape.c()), _ptr(q_rot), _ptr(kv_pool), _ptr(block_table), _ptr(seq_lens),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        _ptr(err_flag), _stream(stream)), "qdec_attn_decode")


def qdec_prefill_rope_table_bytes(num_tokens: int) -> int:
    return int(_lib.qdec_prefill_rope_table_bytes(num_tokens))


def qdec_prefill_rope_table(shape: Shape, positions, rope_table, stream=None):
    """The angles of the chunk rows at `positions` [T] into `rope_table`
    (qdec_prefill_rope_table_bytes(T) bytes)."""
    _raise(_lib.qdec_prefill_rope_table(ctypes.byref(shape.c()), positions.numel(),
                                        _ptr(positions), _ptr(rope_table), _stream(stream)),
           "qdec_prefill_rope_table")


def alloc_prefill_rope_table(num_tokens: int, device=None) -> torch.Tensor:
    """A device buffer for qdec_prefill_rope_table (caller owns it)."""
    return torch.empty(max(1, qdec_prefill_rope_table_bytes(num_tokens)), dtype=torch.uint8,
                       device=device or "cuda")


def qdec_prefill_append_rope(shape: Shape, q, k, v, q_norm_w, k_norm_w, positions, qo_indptr,
                             seq_lens, block_table, kv_pool, q_rot, err_flag=None, stream=None,
                             rope_table=None):
    """Chunk rows q [T][Hq][D], k/v [T][Hkv][D] (row-strided views allowed),
    positions [T], qo_indptr [B+1]; q_rot [T][Hq][D] float32 out; rope_table
    None or from qdec_prefill_rope_table over the same positions."""
    _raise(_lib.qdec_prefill_append_rope(
        ctypes.byref(shape.c()), q.shape[0], _ptr(q), _rows(q, "q"), _ptr(k), _rows(k, "k"),
        _ptr(v), _rows(v, "v"), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions),
        _ptr(rope_table), _ptr(qo_indptr),
        _ptr(seq_lens), _ptr(block_table), _ptr(kv_pool), _ptr(q_rot), _ptr(err_flag),
        _stream(stream)), "qdec_prefill_append_rope")


def qdec_prefill_attn(shape: Shape, q_rot, qo_indptr, seq_lens, block_table, kv_pool, out,
                      err_flag=None, stream=None):
    _raise(_lib.qdec_prefill_attn(
        ctypes.byref(shape.c()), q_rot.shape[0], _ptr(q_rot), _ptr(qo_indptr), _ptr(seq_lens),
        _ptr(block_table), _ptr(kv_pool), _ptr(out), _ptr(err_flag), _stream(stream)),
        "qdec_prefill_attn")


def qdec_prefill_append_rope_fp8(shape: Shape, q, k, v, q_norm_w, k_norm_w, positions, qo_indptr,
                                 seq_lens, block_table, kv_pool_fp8, kv_scale, q_rot,
                                 err_flag=None, stream=None, rope_table=None):
    pool, scale = _fp8_pool(kv_pool_fp8, kv_scale)
    _raise(_lib.qdec_prefill_append_rope_fp8(
        ctypes.byref(shape.c()), q.shape[0], _ptr(q), _rows(q, "q"), _ptr(k), _rows(k, "k"),
        _ptr(v), _rows(v, "v"), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions),
        _ptr(rope_table), _ptr(qo_indptr),
        _ptr(seq_lens), _ptr(block_table), pool, scale, _ptr(q_rot), _ptr(err_flag),
        _stream(stream)), "qdec_prefill_append_rope_fp8")


def qdec_prefill_attn_fp8(shape: Shape, q_rot, qo_indptr, seq_lens, block_table, kv_pool_fp8,
                          kv_scale, out, err_flag=None, stream=None, workspace=None):
    """workspace: None (each query block converts the codes it reads) or a
    device buffer of at least qdec_prefill_fp8_workspace_bytes(shape) bytes
    (the pages are dequantized to bf16 once, then attended as a bf16 pool)."""
    pool, scale = _fp8_pool(kv_pool_fp8, kv_scale)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _raise(_lib.qdec_prefill_attn_fp8(
        ctypes.byref(shape.c()), q_rot.shape[0], _ptr(q_rot), _ptr(qo_indptr), _ptr(seq_lens),
        _ptr(block_table), pool, scale, _ptr(workspace), nbytes, _ptr(out), _ptr(err_flag),
        _stream(stream)), "qdec_prefill_attn_fp8")


def qdec_prefill_fp8_workspace_bytes(shape: Shape) -> int:
    return int(_lib.qdec_prefill_fp8_workspace_bytes(ctypes.byref(shape.c())))


def qdec_attn_merge(shape: Shape, seq_lens, workspace, out, err_flag=None, stream=None):
    _raise(_lib.qdec_attn_merge(
        ctypes.byref(shape.c()), _ptr(seq_lens), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(err_flag),
        _stream(stream)), "qdec_attn_merge")


def qdec_step(shape: Shape, q, k, v, q_norm_w, k_norm_w, positions, seq_lens, block_table,
              kv_pool, workspace, out, err_flag=None, stream=None, rope_table=None):
    _raise(_lib.qdec_step(
        ctypes.byref(shape.c()), _ptr(q), _rows(q, "q"), _ptr(k), _rows(k, "k"), _ptr(v),
        _rows(v, "v"), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions), _ptr(seq_lens),
        _ptr(block_table), _ptr(rope_table), _ptr(kv_pool), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(err_flag),
        _stream(stream)), "qdec_step")


def qdec_qkv_pack_weights(shape: Shape, w_qkv, w_packed, stream=None):
    """Pack the row-major merged weight [(Hq+2Hkv)*D][hidden] for the projection."""
    _raise(_lib.qdec_qkv_pack_weights(ctypes.byref(shape.c()), int(w_qkv.shape[1]), _ptr(w_qkv),
                                      _ptr(w_packed), _stream(stream)), "qdec_qkv_pack_weights")


def qdec_qkv_append_rope(shape: Shape, x, w_packed, q_norm_w, k_norm_w, positions, seq_lens,
                         block_table, kv_pool, q_rot, rope_table, err_flag=None, stream=None):
    """The merged QKV projection of hidden states x [B][hidden] (weight packed
    by qdec_qkv_pack_weights) fused with norm, rotation and append."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x: expected a bf16 [B][hidden] view with contiguous rows")
    _raise(_lib.qdec_qkv_append_rope(
        ctypes.byref(shape.c()), int(x.shape[1]), _ptr(x), x.stride(0), _ptr(w_packed),
        _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions), _ptr(seq_lens), _ptr(block_table),
        _ptr(rope_table), _ptr(kv_pool), _ptr(q_rot), _ptr(err_flag), _stream(stream)),
        "qdec_qkv_append_rope")


def qdec_qkv_append_rope_fp8(shape: Shape, x, w_packed, q_norm_w, k_norm_w, positions, seq_lens,
                             block_table, kv_pool_fp8, kv_scale, q_rot, rope_table,
                             err_flag=None, stream=None):
    """qdec_qkv_append_rope into an FP8 pool (E4M3 codes, per-(page, plane,
    head) scales)."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x: expected a bf16 [B][hidden] view with contiguous rows")
    pool, scale = _fp8_pool(kv_pool_fp8, kv_scale)
    _raise(_lib.qdec_qkv_append_rope_fp8(
        ctypes.byref(shape.c()), int(x.shape[1]), _ptr(x), x.stride(0), _ptr(w_packed),
        _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions), _ptr(seq_lens), _ptr(block_table),
        _ptr(rope_table), pool, scale, _ptr(q_rot), _ptr(err_flag), _stream(stream)),
        "qdec_qkv_append_rope_fp8")


def _fp8_pool(pool, scale):
    if pool.dtype != torch.uint8 or scale.dtype != torch.float32:
        raise ValueError("FP8 pool: expected uint8 E4M3 codes and float32 scales")
    return _ptr(pool), _ptr(scale)


def qdec_append_rope_fp8(shape: Shape, q, k, v, q_norm_w, k_norm_w, positions, seq_lens,
                         block_table, kv_pool_fp8, kv_scale, q_rot, err_flag=None, stream=None,
                         rope_table=None):
    pool, scale = _fp8_pool(kv_pool_fp8, kv_scale)
    _raise(_lib.qdec_append_rope_fp8(
        ctypes.byref(shape.c()), _ptr(q), _rows(q, "q"), _ptr(k), _rows(k, "k"), _ptr(v),
        _rows(v, "v"), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions), _ptr(seq_lens),
        _ptr(block_table), _ptr(rope_table), pool, scale, _ptr(q_rot), _ptr(err_flag),
        _stream(stream)), "qdec_append_rope_fp8")


def qdec_attn_split_fp8(shape: Shape, q_rot, kv_pool_fp8, kv_scale, block_table, seq_lens,
                        workspace, out, err_flag=None, stream=None):
    pool, scale = _fp8_pool(kv_pool_fp8, kv_scale)
    _raise(_lib.qdec_attn_split_fp8(
        ctypes.byref(shape.c()), _ptr(q_rot), pool, scale, _ptr(block_table), _ptr(seq_lens),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        _ptr(err_flag), _stream(stream)), "qdec_attn_split_fp8")


def qdec_attn_decode_fp8(shape: Shape, q_rot, kv_pool_fp8, kv_scale, block_table, seq_lens,
                         workspace, out, err_flag=None, stream=None):
    pool, scale = _fp8_pool(kv_pool_fp8, kv_scale)
    _raise(_lib.qdec_attn_decode_fp8(
        ctypes.byref(shape.c()), _ptr(q_rot), pool, scale, _ptr(block_table), _ptr(seq_lens),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        _ptr(err_flag), _stream(stream)), "qdec_attn_decode_fp8")


def qdec_step_fp8(shape: Shape, q, k, v, q_norm_w, k_norm_w, positions, seq_lens, block_table,
                  kv_pool_fp8, kv_scale, workspace, out, err_flag=None, stream=None,
                  rope_table=None):
    pool, scale = _fp8_pool(kv_pool_fp8, kv_scale)
    _raise(_lib.qdec_step_fp8(
        ctypes.byref(shape.c()), _ptr(q), _rows(q, "q"), _ptr(k), _rows(k, "k"), _ptr(v),
        _rows(v, "v"), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions), _ptr(seq_lens),
        _ptr(block_table), _ptr(rope_table), pool, scale, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(err_flag),
        _stream(stream)), "qdec_step_fp8")


def qdec_step_static_scratch(shape: Shape, q, k, v, q_norm_w, k_norm_w, positions, seq_lens,
                             block_table, kv_pool, out, err_flag=None, stream=None,
                             rope_table=None):
    """qdec_step with the library's own fixed scratch array as the workspace
    (for callers that cannot allocate device memory)."""
    _raise(_lib.qdec_step_static_scratch(
        ctypes.byref(shape.c()), _ptr(q), _rows(q, "q"), _ptr(k), _rows(k, "k"), _ptr(v),
        _rows(v, "v"), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(positions), _ptr(seq_lens),
        _ptr(block_table), _ptr(rope_table), _ptr(kv_pool), _ptr(out), _ptr(err_flag),
        _stream(stream)), "qdec_step_static_scratch")


def qdec_check_error(err_flag, stream=None):
    """Synchronise, read and clear the device error flag: (status, flag bits)."""
    flags = ctypes.c_int32(0)
    st = _lib.qdec_check_error(_ptr(err_flag), _stream(stream), ctypes.byref(flags))
    return int(st), int(flags.value)


# ------------------------------------------------------------- conveniences --

def shape_for(workload, num_ctas: int = 0, launch_flags: int = 0) -> Shape:
    """The Shape of a workloads.Workload (one layer's pool)."""
    s = workload.spec
    return Shape(batch=s.batch, num_pages=s.pool_pages,
                 max_blocks_per_seq=workload.max_blocks,
                 max_seq_len=int(workload.max_blocks * s.page_size),
                 num_q_heads=s.num_q_heads, num_kv_heads=s.num_kv_heads,
                 head_dim=s.head_dim, page_size=s.page_size, num_ctas=num_ctas,
                 launch_flags=launch_flags)


def alloc_rope_table(shape: Shape, device=None) -> torch.Tensor:
    """A device buffer for qdec_rope_table (caller owns it)."""
    n = qdec_rope_table_bytes(shape)
    if n == 0:
        raise QdecError(QDEC_ERR_INVALID_ARG, "qdec_rope_table_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def alloc_workspace(shape: Shape, device=None, stream=None) -> torch.Tensor:
    """A zero-initialised workspace of the size `shape` needs (caller owns it)."""
    n = qdec_workspace_bytes(shape)
    if n == 0:
        raise QdecError(QDEC_ERR_INVALID_ARG, "qdec_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    qdec_workspace_init(shape, ws, stream)
    return ws
