"""Seeded synthetic decode workloads (inputs only: no attention arithmetic).

Both the CUDA path and the CPU oracle are fed from here; this module holds
none of the method's arithmetic.  Everything is drawn from seeded torch
generators:

* per-sequence metadata (context lengths, page assignment) from a CPU
  generator, so a workload's block table is identical on every machine;
* tensor values (new-token q/k/v, norm weights, cached K/V pages) from a
  generator on the target device, so multi-GiB pools are filled in HBM.

Cached pool contents are drawn directly (they stand for keys that were
normed and rotated when they were appended).  An FP8 (E4M3) variant of a
workload holds the same draws stored as codes: every (page, plane, KV head)
gets the scale amax/448 of its 16 x 128 values, and PyTorch's float8_e4m3fn
cast turns value/scale into codes.  That is input synthesis (a cache filled
by some earlier engine), not the path under test: the path's own
quantization is the append of the new token.  Five named workloads mirror
the decode workloads of the blog "GPU 算子与执行优化：从 26 到 100 token/s 的推理引擎破茧之路" (yuzheng310.github.io) (single stream,
concurrency 8 and 16, an 8K context) plus a ragged continuous-batching mix.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import numpy as np
import torch

NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 128
PAGE_SIZE = 16
ROPE_THETA = 1.0e6
EPS = 1.0e-6


@dataclass(frozen=True)
class WorkloadSpec:
    """Shape and value recipe of one decode workload."""
    name: str
    batch: int
    layers: int
    pool_pages: int            # pages per pool
    shared_pool: bool          # one pool for all layers (else one per layer)
    seq_len_kind: str          # "fixed" | "uniform" | "loguniform" | "list"
    seq_len_lo: int = 0
    seq_len_hi: int = 0
    seq_lens: tuple = ()       # used when seq_len_kind == "list"
    chan_scale: bool = False   # per-(KV head, channel) scale U(0.1, 4) on cached K and V
    spike_frac: float = 0.0    # fraction of cached (token, KV head) key rows scaled x8
    seed: int = 0
    num_q_heads: int = NUM_Q_HEADS
    num_kv_heads: int = NUM_KV_HEADS
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE
    max_blocks: int = 0        # block-table row stride; 0 = just enough

    @property
    def max_seq_len_bound(self) -> int:
        if self.seq_len_kind == "list":
            return max(self.seq_lens)
        return self.seq_len_hi

    def kv_bytes_per_token(self) -> int:
        return 2 * self.num_kv_heads * self.head_dim * 2

    def io_bytes_per_seq(self) -> int:
        """q, k, v in and out, bf16."""
        return 2 * self.head_dim * (self.num_q_heads + 2 * self.num_kv_heads + self.num_q_heads)


_SEED0 = 0x9E3779B9

# The five decode workloads (sizes fixed by the benchmark plan).
WORKLOADS = {
    1: WorkloadSpec("b1-ctx513-1layer", batch=1, layers=1, pool_pages=64, shared_pool=True,
                    seq_len_kind="fixed", seq_len_lo=513, seq_len_hi=513, seed=_SEED0 + 1),
    2: WorkloadSpec("b8-ctx256to384-36layer", batch=8, layers=36, pool_pages=4096,
                    shared_pool=False, seq_len_kind="uniform", seq_len_lo=256, seq_len_hi=384,
                    seed=_SEED0 + 2),
    3: WorkloadSpec("b16-ctx256to384-chanscale-36layer", batch=16, layers=36, pool_pages=4096,
                    shared_pool=False, seq_len_kind="uniform", seq_len_lo=256, seq_len_hi=384,
                    chan_scale=True, seed=_SEED0 + 3),
    4: WorkloadSpec("b1-ctx8192-spikes-36layer", batch=1, layers=36, pool_pages=1024,
                    shared_pool=False, seq_len_kind="fixed", seq_len_lo=8192, seq_len_hi=8192,
                    spike_frac=0.01, seed=_SEED0 + 4),
    5: WorkloadSpec("b64-ragged128to16384-sharedpool-36layer", batch=64, layers=36,
                    pool_pages=131072, shared_pool=True, seq_len_kind="loguniform",
                    seq_len_lo=128, seq_len_hi=16384, seed=_SEED0 + 5),
}


@dataclass
class Workload:
    spec: WorkloadSpec
    device: torch.device
    seq_lens: torch.Tensor        # int32 [B] (device)
    positions: torch.Tensor       # int32 [B] (device)
    block_table: torch.Tensor     # int32 [B][max_blocks] (device); unused entries -1
    qkv: torch.Tensor             # bf16 [layers][B][Hq + 2 Hkv][D] (device)
    w_q: torch.Tensor             # bf16 [layers][D]
    w_k: torch.Tensor             # bf16 [layers][D]
    pools: List[torch.Tensor] = field(default_factory=list)  # bf16 [pages][2][Hkv][P][D]
    seq_lens_host: np.ndarray = None
    block_table_host: np.ndarray = None
    kv: str = "bf16"              # "bf16" or "fp8"
    pools8: List[torch.Tensor] = field(default_factory=list)   # uint8 E4M3 [pages][2][Hkv][P][D]
    scales: List[torch.Tensor] = field(default_factory=list)   # float32 [pages][2][Hkv]

    # strided views of the fused qkv buffer, per layer
    def q(self, layer: int) -> torch.Tensor:
        return self.qkv[layer, :, :self.spec.num_q_heads]

    def k(self, layer: int) -> torch.Tensor:
        h = self.spec.num_q_heads
        return self.qkv[layer, :, h:h + self.spec.num_kv_heads]

    def v(self, layer: int) -> torch.Tensor:
        h = self.spec.num_q_heads + self.spec.num_kv_heads
        return self.qkv[layer, :, h:h + self.spec.num_kv_heads]

    def pool(self, layer: int) -> torch.Tensor:
        return self.pools[0] if self.spec.shared_pool else self.pools[layer]

    def pool8(self, layer: int) -> torch.Tensor:
        return self.pools8[0] if self.spec.shared_pool else self.pools8[layer]

    def scale(self, layer: int) -> torch.Tensor:
        return self.scales[0] if self.spec.shared_pool else self.scales[layer]

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    def algorithmic_bytes_per_layer(self) -> int:
        """KV read at token granularity plus q/k/v in and out (bf16); for an
        FP8 pool one byte per KV element plus the K and V scale of every
        (page, head) a sequence reads."""
        s = self.spec
        io = s.batch * s.io_bytes_per_seq()
        if self.kv == "fp8":
            pages = int(((self.seq_lens_host + s.page_size - 1) // s.page_size).sum())
            return (int(self.seq_lens_host.sum()) * s.kv_bytes_per_token() // 2
                    + pages * 2 * s.num_kv_heads * 4 + io)
        return int(self.seq_lens_host.sum()) * s.kv_bytes_per_token() + io


def draw_seq_lens(spec: WorkloadSpec, gen: torch.Generator) -> np.ndarray:
    B = spec.batch
    if spec.seq_len_kind == "fixed":
        return np.full(B, spec.seq_len_lo, np.int64)
    if spec.seq_len_kind == "list":
        assert len(spec.seq_lens) == B
        return np.asarray(spec.seq_lens, np.int64)
    if spec.seq_len_kind == "uniform":
        return torch.randint(spec.seq_len_lo, spec.seq_len_hi + 1, (B,), generator=gen).numpy()
    if spec.seq_len_kind == "loguniform":
        u = torch.rand(B, generator=gen, dtype=torch.float64).numpy()
        lo, hi = math.log(spec.seq_len_lo), math.log(spec.seq_len_hi)
        return np.clip(np.rint(np.exp(lo + u * (hi - lo))), spec.seq_len_lo,
                       spec.seq_len_hi).astype(np.int64)
    raise ValueError(spec.seq_len_kind)


def _fill_normal_bf16(t: torch.Tensor, gen: torch.Generator, chunk_elems: int = 1 << 27):
    """Fill a bf16 tensor with N(0,1) draws rounded to bf16, in chunks."""
    flat = t.view(-1)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(s + chunk_elems, flat.numel())
        flat[s:e] = torch.randn(e - s, generator=gen, device=t.device,
                                dtype=torch.float32).to(torch.bfloat16)


def build(spec: WorkloadSpec, device="cpu", poison: bool = False,
          layers: Optional[int] = None, kv: str = "bf16") -> Workload:
    """Materialise a workload.

    poison=True (tests): every pool element the attention must not read is
    NaN -- pages no sequence references, the slots past each sequence's end,
    and the append slot itself (it must be overwritten before it is read).
    kv="fp8": the pools are held as E4M3 codes plus per-(page, plane, head)
    scales (NaN poison becomes the NaN code 0x7F); `pools` is then empty.
    """
    assert kv in ("bf16", "fp8"), kv
    device = torch.device(device)
    nl = spec.layers if layers is None else layers
    spec = replace(spec, layers=nl)
    B, Hq, Hkv, D, P = (spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                        spec.page_size)
    gmeta = torch.Generator().manual_seed(spec.seed)
    gdev = torch.Generator(device=device).manual_seed(spec.seed + 1)

    seq_lens = draw_seq_lens(spec, gmeta)
    n_pages = (seq_lens + P - 1) // P
    max_blocks = spec.max_blocks or int(max(1, (spec.max_seq_len_bound + P - 1) // P))
    assert n_pages.max() <= max_blocks
    total = int(n_pages.sum())
    assert total <= spec.pool_pages, "pool too small for the drawn context lengths"
    perm = torch.randperm(spec.pool_pages, generator=gmeta).numpy()
    bt = np.full((B, max_blocks), -1, np.int32)
    off = 0
    for b in range(B):
        bt[b, :n_pages[b]] = perm[off:off + n_pages[b]]
        off += int(n_pages[b])

    qkv = torch.empty((nl, B, Hq + 2 * Hkv, D), dtype=torch.bfloat16, device=device)
    _fill_normal_bf16(qkv, gdev)
    w = (torch.rand((2, nl, D), generator=gdev, device=device) + 0.5).to(torch.bfloat16)

    npools = 1 if spec.shared_pool else nl
    pools, pools8, scales = [], [], []
    referenced = torch.zeros(spec.pool_pages, dtype=torch.bool)
    referenced[torch.from_numpy(perm[:total].astype(np.int64))] = True
    for _ in range(npools):
        pool = torch.empty((spec.pool_pages, 2, Hkv, P, D), dtype=torch.bfloat16, device=device)
        _fill_normal_bf16(pool, gdev)
        if spec.chan_scale:
            sc = torch.rand((2, Hkv, D), generator=gdev, device=device) * 3.9 + 0.1
            for plane in range(2):
                for s in range(0, spec.pool_pages, 4096):
                    blk = pool[s:s + 4096, plane].float() * sc[plane][None, :, None, :]
                    pool[s:s + 4096, plane] = blk.to(torch.bfloat16)
        if spec.spike_frac > 0:
            for s in range(0, spec.pool_pages, 4096):
                e = min(s + 4096, spec.pool_pages)
                m = torch.rand((e - s, Hkv, P), generator=gdev, device=device) < spec.spike_frac
                kp = pool[s:e, 0]
                kp[m] = kp[m] * 8  # a power of two: exact in bf16
        if kv == "fp8":
            codes, sc = _to_fp8(pool)
            del pool
            if poison:
                _poison(codes, referenced.to(device), bt, seq_lens, P, value=0x7F)
            pools8.append(codes)
            scales.append(sc)
            continue
        if poison:
            _poison(pool, referenced.to(device), bt, seq_lens, P)
        pools.append(pool)

    if spec.chan_scale:
        # the new value rows follow the scaled distribution of the cache
        sv = torch.rand((nl, Hkv, D), generator=gdev, device=device) * 3.9 + 0.1
        vv = qkv[:, :, Hq + Hkv:].float() * sv[:, None]
        qkv[:, :, Hq + Hkv:] = vv.to(torch.bfloat16)

    return Workload(
        spec=spec, device=device,
        seq_lens=torch.from_numpy(seq_lens.astype(np.int32)).to(device),
        positions=torch.from_numpy((seq_lens - 1).astype(np.int32)).to(device),
        block_table=torch.from_numpy(bt).to(device),
        qkv=qkv, w_q=w[0].contiguous(), w_k=w[1].contiguous(), pools=pools,
        seq_lens_host=seq_lens.astype(np.int64), block_table_host=bt, kv=kv, pools8=pools8,
        scales=scales)


def _to_fp8(pool: torch.Tensor, chunk: int = 4096):
    """E4M3 codes and per-(page, plane, head) scales amax/448 of a bf16 pool
    (PyTorch's float8_e4m3fn cast; magnitudes are at most 448 by construction)."""
    codes = torch.empty(pool.shape, dtype=torch.uint8, device=pool.device)
    sc = torch.empty(pool.shape[:3], dtype=torch.float32, device=pool.device)
    for s in range(0, pool.shape[0], chunk):
        x = pool[s:s + chunk].float()
        amax = x.abs().amax(dim=(3, 4))
        scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        y = (x / scale[..., None, None]).clamp(-448.0, 448.0)
        codes[s:s + chunk] = y.to(torch.float8_e4m3fn).view(torch.uint8)
        sc[s:s + chunk] = scale
    return codes, sc


def _poison(pool, referenced, bt, seq_lens, P, value=float("nan")):
    pool[~referenced] = value
    for b, L in enumerate(seq_lens):
        L = int(L)
        last = int(bt[b, (L - 1) // P])
        pool[last, :, :, (L - 1) % P:, :] = value   # the append slot and everything after it


def custom(batch: int, seq_lens, pool_pages: int, layers: int = 1, seed: int = 1234,
           num_q_heads: int = NUM_Q_HEADS, num_kv_heads: int = NUM_KV_HEADS,
           chan_scale: bool = False, spike_frac: float = 0.0, shared_pool: bool = True,
           max_blocks: int = 0, name: str = "custom") -> WorkloadSpec:
    """A workload with the given context lengths (tests and sweeps)."""
    return WorkloadSpec(name, batch=batch, layers=layers, pool_pages=pool_pages,
                        shared_pool=shared_pool, seq_len_kind="list",
                        seq_lens=tuple(int(x) for x in seq_lens), chan_scale=chan_scale,
                        spike_frac=spike_frac, seed=seed, num_q_heads=num_q_heads,
                        num_kv_heads=num_kv_heads, max_blocks=max_blocks)


# ------------------------------------------------------------ host views --

def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a numpy uint16 array (copied to host)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_inputs(w: Workload, layer: int, seqs=None):
    """Host copies of one layer's inputs for the oracle, restricted to the
    sequences `seqs` (all by default).  Only the pages those sequences
    reference are copied, renumbered 0..n-1 in block-table order (a pure
    relabelling of physical pages).  Call it BEFORE the layer runs on the
    GPU so the pool snapshot holds no GPU-written slot."""
    s = w.spec
    P = s.page_size
    seqs = list(range(s.batch)) if seqs is None else list(seqs)
    sl = w.seq_lens_host[seqs]
    n = (sl + P - 1) // P
    mb = int(n.max())
    pages = np.concatenate([w.block_table_host[b, :n[i]] for i, b in enumerate(seqs)])
    bt = np.full((len(seqs), mb), -1, np.int32)
    off = 0
    for i in range(len(seqs)):
        bt[i, :n[i]] = np.arange(off, off + n[i], dtype=np.int32)
        off += int(n[i])
    sel = torch.as_tensor(seqs, dtype=torch.long, device=w.qkv.device)
    extra = {}
    if w.kv == "fp8":
        pool = w.pool8(layer)
        idx = torch.from_numpy(pages.astype(np.int64)).to(pool.device)
        sub = np.ascontiguousarray(pool.index_select(0, idx).cpu().numpy())
        extra["kv_scale"] = np.ascontiguousarray(
            w.scale(layer).index_select(0, idx).cpu().numpy())
    else:
        pool = w.pool(layer)
        idx = torch.from_numpy(pages.astype(np.int64)).to(pool.device)
        sub = bf16_bits(pool.index_select(0, idx))
    return dict(extra,
        q=bf16_bits(w.q(layer).index_select(0, sel)),
        k=bf16_bits(w.k(layer).index_select(0, sel)),
        v=bf16_bits(w.v(layer).index_select(0, sel)),
        w_q=bf16_bits(w.w_q[layer]), w_k=bf16_bits(w.w_k[layer]),
        positions=w.positions.cpu().numpy()[seqs].astype(np.int32),
        seq_lens=sl.astype(np.int32),
        block_table=bt, pool=np.ascontiguousarray(sub),
        rope_theta=ROPE_THETA, eps=EPS)


# ------------------------------------------------------------ chunked prefill --

@dataclass
class PrefillCase:
    """A chunked-prefill input: B sequences of seq_lens[b] tokens (after the
    chunk), the last chunks[b] of them new, packed by qo_indptr."""
    seq_lens: torch.Tensor      # [B] int32
    qo_indptr: torch.Tensor     # [B+1] int32
    positions: torch.Tensor     # [T] int32 (RoPE positions of the chunk rows)
    block_table: torch.Tensor   # [B][max_blocks] int32
    pool: torch.Tensor          # [pages][2][Hkv][P][D] bf16
    q: torch.Tensor             # [T][Hq][D] bf16
    k: torch.Tensor             # [T][Hkv][D] bf16
    v: torch.Tensor             # [T][Hkv][D] bf16
    w_q: torch.Tensor           # [D] bf16
    w_k: torch.Tensor           # [D] bf16
    max_blocks: int
    num_pages: int


def prefill_case(seq_lens, chunks, seed: int = 7, device="cuda", poison: bool = True,
                 pos_offset: int = 0, num_q_heads: int = NUM_Q_HEADS,
                 num_kv_heads: int = NUM_KV_HEADS, extra_pages: int = 5) -> PrefillCase:
    """Seeded chunked-prefill input.  Every sequence's pages are a random
    permutation of one pool (plus unreferenced pages); tokens 0..L-n-1 hold
    N(0,1) cached K/V, the chunk's slots hold N(0,1) too (the append
    overwrites them); with poison every element past a sequence's last token
    and every unreferenced page is NaN.  Chunk q/k/v are N(0,1), the norm
    weights U(0.5, 1.5); positions = token index + pos_offset."""
    assert len(seq_lens) == len(chunks)
    gen = torch.Generator().manual_seed(seed)
    P, D = PAGE_SIZE, HEAD_DIM
    Hq, Hkv = num_q_heads, num_kv_heads
    L = np.asarray(seq_lens, np.int64)
    n = np.asarray(chunks, np.int64)
    npg = (L + P - 1) // P
    mb = int(max(1, npg.max()))
    total = int(npg.sum()) + extra_pages
    perm = torch.randperm(total, generator=gen).numpy()
    bt = np.full((len(L), mb), -1, np.int32)
    off = 0
    for b in range(len(L)):
        bt[b, :npg[b]] = perm[off:off + npg[b]]
        off += int(npg[b])
    pool = torch.randn((total, 2, Hkv, P, D), generator=gen).to(torch.bfloat16)
    if poison:
        used = np.zeros((total, P), bool)
        for b in range(len(L)):
            t = np.arange(L[b])
            used[bt[b, t // P], t % P] = True
        mask = torch.from_numpy(~used)[:, None, None, :, None].expand_as(pool)
        pool = pool.masked_fill(mask, float("nan"))
    qo = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    T = int(qo[-1])
    idx = np.concatenate([np.arange(Lb - nb, Lb) for Lb, nb in zip(L, n)] + [np.zeros(0)])
    mk = lambda *shape: torch.randn(shape, generator=gen).to(torch.bfloat16)
    w = lambda: (0.5 + torch.rand(D, generator=gen)).to(torch.bfloat16)
    return PrefillCase(
        seq_lens=torch.tensor(L, dtype=torch.int32, device=device),
        qo_indptr=torch.tensor(qo, dtype=torch.int32, device=device),
        positions=torch.tensor(idx.astype(np.int64) + pos_offset, dtype=torch.int32, device=device),
        block_table=torch.from_numpy(bt).to(device), pool=pool.to(device),
        q=mk(T, Hq, D).to(device), k=mk(T, Hkv, D).to(device), v=mk(T, Hkv, D).to(device),
        w_q=w().to(device), w_k=w().to(device), max_blocks=mb, num_pages=total)


def prefill_case_fp8(seq_lens, chunks, seed: int = 7, device="cuda", pos_offset: int = 0):
    """prefill_case held in an FP8 pool: the same draws as E4M3 codes with
    per-(page, plane, head) scales amax/448 (PyTorch's float8_e4m3fn cast);
    every element past a sequence's last token and every unreferenced page is
    the NaN code 0x7F.  Returns (case, codes, scales)."""
    c = prefill_case(seq_lens, chunks, seed=seed, device=device, poison=False,
                     pos_offset=pos_offset)
    codes, sc = _to_fp8(c.pool)
    P = PAGE_SIZE
    used = torch.zeros(codes.shape[0], P, dtype=torch.bool, device=codes.device)
    bt = c.block_table.cpu().numpy()
    for b, L in enumerate(seq_lens):
        t = torch.arange(int(L))
        used[torch.as_tensor(bt[b, (t // P).numpy()], device=codes.device),
             (t % P).to(codes.device)] = True
    codes.masked_fill_(~used[:, None, None, :, None].expand_as(codes), 0x7F)
    return c, codes, sc
