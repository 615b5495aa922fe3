"""One captured CUDA graph serves every context length (marked gpu).

The blog "GPU 算子与执行优化：从 26 到 100 token/s 的推理引擎破茧之路" keeps
per-step metadata (lengths, positions, block tables) in static buffers that
are rewritten in place outside the captured graph (part 5), and shows how a
graph captured with a fixed attention grid stops fitting long contexts (part
8, the fixed-CTA trap).  Here the step (RoPE table + three overlapped
layer-steps) is captured ONCE with a plan for contexts up to 16384 tokens;
then, for one set of lengths after another, the lengths, positions, block
table, new-token rows and pools are rewritten in place and the same graph is
replayed; every layer's output and appended slots are compared with the
oracle.  Lengths run from 1 to the bound, across page boundaries.  Batches of
one and four sequences (8 and 32 (sequence, KV head) segments) are planned on
the cluster layout, whose per-segment split follows the actual lengths; a
batch of 24 (192 segments, more than 60 % of the CTAs resident on a 152-SM
GPU) on the flat layout, so both layouts take every length.
"""
import numpy as np
import pytest
import torch

from gqa_paged_kv_gb300 import workloads as wl
import parity

pytestmark = pytest.mark.gpu

BOUND = 16384
PAGE = 16
MAX_BLOCKS = BOUND // PAGE
LAYERS = 3

_R = np.random.default_rng(77)
LENGTH_SETS = {
    1: [[1], [2], [16], [17], [300], [1024], [4097], [8192], [12345], [16383], [16384]],
    4: [[1, 2, 15, 16], [17, 300, 64, 1000], [16384, 1, 5000, 33], [8192, 8192, 8192, 8192],
        [513, 4097, 12000, 7], [16384, 16384, 16384, 16384]],
    24: [[1, 2, 15, 16, 17, 31, 32, 33] * 3,
         [16384, 1] + [int(x) for x in _R.integers(1, 400, 22)],
         [int(x) for x in np.exp(_R.uniform(0.0, np.log(16384), 24)).round().clip(1, 16384)],
         [384] * 24],
}


class _Static:
    """A workload whose buffers keep their addresses while their contents
    are rewritten for each new set of lengths."""

    def __init__(self, batch: int, kv: str, seed: int):
        self.pages = batch * MAX_BLOCKS + 8
        spec = wl.custom(batch, [BOUND] * batch, pool_pages=self.pages, layers=LAYERS,
                         seed=seed, shared_pool=False, max_blocks=MAX_BLOCKS)
        self.w = wl.build(spec, "cuda", kv=kv)
        self.gen = torch.Generator(device="cuda").manual_seed(seed + 100)
        self.rng = np.random.default_rng(seed)

    def load(self, lens):
        """New lengths, positions, block table (a fresh random page
        assignment), new-token rows and pool contents, written in place;
        every pool element the attention must not read is poisoned."""
        w, B = self.w, self.w.spec.batch
        lens = np.asarray(lens, np.int64)
        n = (lens + PAGE - 1) // PAGE
        perm = self.rng.permutation(self.pages)
        bt = np.full((B, MAX_BLOCKS), -1, np.int32)
        off = 0
        for b in range(B):
            bt[b, :n[b]] = perm[off:off + n[b]]
            off += int(n[b])
        referenced = torch.zeros(self.pages, dtype=torch.bool, device="cuda")
        referenced[torch.from_numpy(perm[:off].astype(np.int64)).cuda()] = True
        w.seq_lens.copy_(torch.from_numpy(lens.astype(np.int32)))
        w.positions.copy_(torch.from_numpy((lens - 1).astype(np.int32)))
        w.block_table.copy_(torch.from_numpy(bt))
        w.seq_lens_host = lens
        w.block_table_host = bt
        wl._fill_normal_bf16(w.qkv, self.gen)
        for l in range(LAYERS):
            fresh = torch.empty((self.pages, 2, 8, PAGE, 128), dtype=torch.bfloat16,
                                device="cuda")
            wl._fill_normal_bf16(fresh, self.gen)
            if w.kv == "fp8":
                codes, sc = wl._to_fp8(fresh)
                w.pools8[l].copy_(codes)
                w.scales[l].copy_(sc)
                wl._poison(w.pools8[l], referenced, bt, lens, PAGE, value=0x7F)
            else:
                w.pools[l].copy_(fresh)
                wl._poison(w.pools[l], referenced, bt, lens, PAGE)
            del fresh
        torch.cuda.synchronize()


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("batch", sorted(LENGTH_SETS))
def test_one_graph_serves_every_length(batch, kv):
    q = parity.qdec()
    st = _Static(batch, kv, seed=60 + batch)
    w = st.w
    shape = q.Shape(batch=batch, num_pages=st.pages, max_blocks_per_seq=MAX_BLOCKS,
                    max_seq_len=BOUND, launch_flags=q.QDEC_LAUNCH_OVERLAP_PREVIOUS)
    ws = q.alloc_workspace(shape)
    rope = q.alloc_rope_table(shape)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((LAYERS, batch, 32, 128), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        q.qdec_rope_table(shape, w.positions, rope, stream=stream)
        for l in range(LAYERS):
            if kv == "fp8":
                q.qdec_step_fp8(shape, w.q(l), w.k(l), w.v(l), w.w_q[l], w.w_k[l], w.positions,
                                w.seq_lens, w.block_table, w.pool8(l), w.scale(l), ws, out[l],
                                err, stream=stream, rope_table=rope)
            else:
                q.qdec_step(shape, w.q(l), w.k(l), w.v(l), w.w_q[l], w.w_k[l], w.positions,
                            w.seq_lens, w.block_table, w.pool(l), ws, out[l], err,
                            stream=stream, rope_table=rope)

    st.load(LENGTH_SETS[batch][0])
    with torch.cuda.stream(stream):
        step()          # configures the kernels outside capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            step()
    for lens in LENGTH_SETS[batch]:
        st.load(lens)
        snaps = [wl.oracle_inputs(w, l) for l in range(LAYERS)]   # before the replay writes
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        status, flags = q.qdec_check_error(err)
        assert status == 0 and flags == 0, f"lengths {lens}: device flags {flags:#x}"
        for l in range(LAYERS):
            ref = parity.run_oracle(snaps[l])
            parity.assert_out_close(out[l], ref["out"], f"lengths {lens}, layer {l}")
            parity.assert_slots_for(w, l, range(batch), ref)
