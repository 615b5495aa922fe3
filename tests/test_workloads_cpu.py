"""The seeded synthetic input recipe (no GPU): context-length recipes of the
five workloads, block tables, the key-row spikes of the 8K workload, the
per-channel K/V scales, the FP8 pools' per-(page, plane, head) scales, the
NaN poison the tests rely on, and the chunked-prefill inputs."""
import math

import numpy as np
import torch

from gqa_paged_kv_gb300 import workloads as wl


def _lens(i):
    spec = wl.WORKLOADS[i]
    return spec, wl.draw_seq_lens(spec, torch.Generator().manual_seed(spec.seed))


def test_context_length_recipes():
    spec, L = _lens(1)
    assert spec.batch == 1 and list(L) == [513]
    for i in (2, 3):
        spec, L = _lens(i)
        assert len(L) == spec.batch == (8 if i == 2 else 16)
        assert L.min() >= 256 and L.max() <= 384
    spec, L = _lens(4)
    assert list(L) == [8192]
    spec, L = _lens(5)
    assert len(L) == 64 and L.min() >= 128 and L.max() <= 16384
    # log-uniform: the logs spread over most of [ln 128, ln 16384]
    lo, hi = math.log(128), math.log(16384)
    u = (np.log(L) - lo) / (hi - lo)
    assert u.min() < 0.1 and u.max() > 0.9 and 0.3 < np.median(u) < 0.7
    # every pool holds its sequences' pages
    for i in range(1, 6):
        spec, L = _lens(i)
        assert int(((L + 15) // 16).sum()) <= spec.pool_pages


def test_lengths_are_deterministic():
    for i in range(1, 6):
        assert np.array_equal(_lens(i)[1], _lens(i)[1])


def test_block_tables_give_each_sequence_its_own_pages():
    spec = wl.custom(5, [1, 16, 17, 300, 33], pool_pages=64, seed=3)
    w = wl.build(spec, "cpu")
    bt, L = w.block_table_host, w.seq_lens_host
    used = []
    for b in range(5):
        n = (int(L[b]) + 15) // 16
        assert np.all(bt[b, :n] >= 0) and np.all(bt[b, :n] < 64) and np.all(bt[b, n:] == -1)
        used += list(bt[b, :n])
    assert len(used) == len(set(used))                     # no page shared
    assert np.array_equal(w.positions.numpy(), L - 1)


def test_spikes_scale_one_percent_of_key_rows_by_eight():
    w = wl.build(wl.WORKLOADS[4], "cpu", layers=1)
    pool = w.pools[0].float()                              # [pages][2][Hkv][P][D]
    row_max = pool.abs().amax(dim=-1)                      # [pages][2][Hkv][P]
    spiked_k = (row_max[:, 0] > 12).float().mean().item()  # N(0,1) rows never reach 12
    assert 0.009 < spiked_k < 0.011, spiked_k
    assert (row_max[:, 1] > 12).sum().item() == 0          # value rows are not spiked


def test_channel_scales_spread_the_key_and_value_columns():
    spec = wl.custom(2, [200, 300], pool_pages=256, seed=9, chan_scale=True)
    w = wl.build(spec, "cpu")
    pool = w.pools[0].float()
    for plane in range(2):
        std = pool[:, plane].permute(1, 3, 0, 2).reshape(8, 128, -1).std(dim=-1)  # [Hkv][D]
        assert std.min().item() > 0.08 and std.max().item() < 4.3
        assert std.max().item() / std.min().item() > 5


def test_fp8_pools_hold_the_same_draws_with_amax_scales():
    spec = wl.custom(3, [40, 17, 100], pool_pages=32, seed=21)
    wb = wl.build(spec, "cpu")
    w8 = wl.build(spec, "cpu", kv="fp8")
    x = wb.pools[0].float()
    sc = w8.scales[0]
    amax = x.abs().amax(dim=(3, 4))
    assert torch.equal(sc, torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)))
    dec = w8.pools8[0].view(torch.float8_e4m3fn).float() * sc[..., None, None]
    err = (dec - x).abs()
    bound = torch.maximum(x.abs() * 2.0 ** -4, sc[..., None, None] * 2.0 ** -10) * (1 + 1e-6)
    assert torch.all(err <= bound)


def test_poison_marks_exactly_what_attention_must_not_read():
    spec = wl.custom(3, [1, 17, 40], pool_pages=16, seed=5)
    w = wl.build(spec, "cpu", poison=True)
    pool = w.pools[0].float()
    bt, L = w.block_table_host, w.seq_lens_host
    live = torch.zeros(pool.shape, dtype=torch.bool)
    for b in range(3):
        for t in range(int(L[b]) - 1):                     # cached tokens only
            live[bt[b, t // 16], :, :, t % 16, :] = True
    assert torch.all(torch.isfinite(pool[live]))
    assert torch.all(torch.isnan(pool[~live]))
    w8 = wl.build(spec, "cpu", poison=True, kv="fp8")
    codes = w8.pools8[0]
    assert torch.all(codes[~live] == 0x7F) and torch.all(codes[live] != 0x7F)


def test_prefill_case_packs_the_last_tokens_of_each_sequence():
    L, n = [300, 17, 1000, 5], [20, 17, 0, 5]
    c = wl.prefill_case(L, n, seed=11, device="cpu", pos_offset=3)
    qo = c.qo_indptr.numpy()
    assert list(qo) == [0, 20, 37, 37, 42] and c.q.shape[0] == 42
    pos = c.positions.numpy()
    for b in range(4):
        assert list(pos[qo[b]:qo[b + 1]]) == list(range(L[b] - n[b] + 3, L[b] + 3))
    bt = c.block_table.numpy()
    used = [p for b in range(4) for p in bt[b, :(L[b] + 15) // 16]]
    assert len(used) == len(set(used)) and max(used) < c.num_pages
    assert c.num_pages == len(used) + 5                    # plus unreferenced pages
    pool = c.pool.float()
    for b in range(4):                                     # finite up to the last token only
        last = bt[b, (L[b] - 1) // 16]
        assert torch.all(torch.isfinite(pool[last, :, :, :(L[b] - 1) % 16 + 1]))
        assert torch.all(torch.isnan(pool[last, :, :, (L[b] - 1) % 16 + 1:]))
    free = sorted(set(range(c.num_pages)) - set(used))
    assert torch.all(torch.isnan(pool[free]))


def test_prefill_case_fp8_holds_the_same_draws():
    """The FP8 case is the bf16 case's draws: scales amax/448 of every
    (page, plane, head) block, codes within E4M3 rounding of the values up to
    each sequence's last token, the NaN code 0x7F everywhere else."""
    c, codes, sc = wl.prefill_case_fp8([40, 100], [40, 3], seed=13, device="cpu")
    ref = wl.prefill_case([40, 100], [40, 3], seed=13, device="cpu", poison=False)
    assert torch.equal(c.q, ref.q) and torch.equal(c.block_table, ref.block_table)
    x = ref.pool.float()
    amax = x.abs().amax(dim=(3, 4))
    assert torch.equal(sc, torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)))
    live = torch.zeros(x.shape, dtype=torch.bool)
    bt = c.block_table.numpy()
    for b, Lb in enumerate([40, 100]):
        for t in range(Lb):
            live[bt[b, t // 16], :, :, t % 16, :] = True
    assert torch.all(codes[~live] == 0x7F) and torch.all(codes[live] != 0x7F)
    dec = codes.view(torch.float8_e4m3fn).float() * sc[..., None, None]
    bound = torch.maximum(x.abs() * 2.0 ** -4, sc[..., None, None] * 2.0 ** -10) * (1 + 1e-6)
    assert torch.all((dec - x).abs()[live] <= bound[live])
