"""The synthetic workloads are built from the shapes the blog prints.

tests/golden/blog_workloads.json transcribes the blog's part-1 workload
table and model description (see the file's "source"); the pages print no
worked numeric example of the attention block itself.
"""
import json
import os

import numpy as np
import torch

from gqa_paged_kv_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "blog_workloads.json")


def _blog():
    with open(GOLDEN) as f:
        return json.load(f)


def test_model_dims_match_blog():
    g = _blog()
    for spec in wl.WORKLOADS.values():
        assert spec.num_q_heads == g["model"]["num_q_heads"]
        assert spec.num_kv_heads == g["model"]["num_kv_heads"]
        assert spec.page_size == g["page_size"]
        assert spec.layers in (1, g["model"]["layers"])


def test_workload_shapes_match_blog_table():
    w = _blog()["workloads"]
    s1, s2, s3, s4 = (wl.WORKLOADS[i] for i in (1, 2, 3, 4))
    # single stream: prompt 512 cached, plus the token being decoded
    assert (s1.batch, s1.seq_len_lo) == (w["A"]["concurrency"], w["A"]["prompt"] + 1)
    # concurrency 8 / 16: prompt 256 plus up to 128 generated tokens
    for s, k in ((s2, "B"), (s3, "C")):
        assert s.batch == w[k]["concurrency"]
        assert (s.seq_len_lo, s.seq_len_hi) == (w[k]["prompt"], w[k]["prompt"] + w[k]["gen"])
    # long-context single stream, past the blog's 2048 split threshold
    assert (s4.batch, s4.seq_len_lo) == (w["E"]["concurrency"], w["E"]["prompt"])
    assert s4.seq_len_lo > _blog()["split_threshold_ctx"]


def test_block_table_is_csr_equivalent():
    """The dense block table carries the blog's CSR page metadata (indptr,
    indices, last_page_len) exactly: rebuild one from the other."""
    w = wl.build(wl.custom(4, [1, 16, 17, 40], pool_pages=16), "cpu")
    P = w.spec.page_size
    n = (w.seq_lens_host + P - 1) // P
    indptr = np.concatenate([[0], np.cumsum(n)])
    indices = np.concatenate([w.block_table_host[b, :n[b]] for b in range(4)])
    last = w.seq_lens_host - (n - 1) * P
    assert list(last) == [1, 16, 1, 8]
    for b in range(4):
        row = indices[indptr[b]:indptr[b + 1]]
        assert np.array_equal(row, w.block_table_host[b, :n[b]])
        assert np.all(w.block_table_host[b, n[b]:] == -1)
    assert len(set(indices.tolist())) == len(indices), "pages shared between sequences"
