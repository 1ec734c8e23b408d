"""The seeded input generators (beam_decode_gb300/workload.py) against the input recipe: shapes
and sizes of the named workloads, distinct in-range catalogues with the stated code
distributions, reproducible per-tensor streams, and bfloat16 rounding checked against torch's
own conversion.  CPU only."""
import numpy as np
import pytest
import torch

from beam_decode_gb300 import workload as wl

QWEN3 = dict(n_layers=28, n_q_heads=16, n_kv_heads=8, head_dim=128, vocab=151936)


@pytest.mark.parametrize("name,R,T,W,L,items,dist", [
    ("page1", 64, 2000, 30, 5, 200_000, "uniform"),
    ("short", 16, 1000, 256, 3, 1_000_000, "zipf"),
    ("long", 8, 5000, 256, 3, 1_000_000, "uniform"),
])
def test_fixed_workloads_follow_the_recipe(name, R, T, W, L, items, dist):
    w = wl.make_workload(name)
    assert w.n_requests == R and w.ctx_lens == [T] * R and w.beam_widths == [W] * R
    assert w.n_levels == L and w.codes_per_level == 256 and w.n_items == [items] * R
    assert w.trie_dist == dist and w.shared_trie
    for k, v in QWEN3.items():
        assert getattr(w, k) == v
    assert w.code_base == w.vocab - L * 256  # the last L*C token ids are the codes
    assert w.seed == 1 and w.logit_std == 2.0


def test_tiny_workload():
    w = wl.make_workload("tiny")
    assert (w.n_layers, w.n_q_heads, w.n_kv_heads, w.head_dim, w.vocab) == (1, 2, 1, 64, 1024)
    assert (w.n_levels, w.codes_per_level, w.code_base) == (2, 16, 512)
    assert w.ctx_lens == [64] and w.beam_widths == [4] and w.n_items == [50] and w.seed == 0


def test_mixed_workload_ranges_and_reproducibility():
    w = wl.make_workload("mixed")
    assert w.n_requests == 32 and not w.shared_trie and w.trie_dist == "zipf"
    assert all(500 <= t <= 5000 for t in w.ctx_lens)
    assert set(w.beam_widths) <= {32, 64, 128, 256} and len(set(w.beam_widths)) > 1
    assert all(100_000 <= n <= 1_000_000 for n in w.n_items)
    assert 3 <= w.n_levels <= 5 and w.code_base == w.vocab - w.n_levels * 256
    w2 = wl.make_workload("mixed")
    assert (w.ctx_lens, w.beam_widths, w.n_items, w.n_levels) == (w2.ctx_lens, w2.beam_widths, w2.n_items,
                                                                  w2.n_levels)
    w3 = wl.make_workload("mixed", seed=2)
    assert w3.ctx_lens != w.ctx_lens


@pytest.mark.parametrize("dist", ["uniform", "zipf"])
def test_items_are_distinct_in_range_and_seeded(dist):
    a = wl.draw_items(20_000, 3, 64, dist, seed=5)
    assert a.shape == (20_000, 3) and a.dtype == np.int32
    assert a.min() >= 0 and a.max() < 64
    assert len(np.unique(a, axis=0)) == len(a)
    assert np.array_equal(a, wl.draw_items(20_000, 3, 64, dist, seed=5))
    assert not np.array_equal(a, wl.draw_items(20_000, 3, 64, dist, seed=5, stream=(1,)))


def test_code_distributions():
    n, C = 30_000, 256
    exp = n / C
    u = np.bincount(wl.draw_items(n, 3, C, "uniform", seed=3)[:, 0], minlength=C)
    z = np.bincount(wl.draw_items(n, 3, C, "zipf", seed=3)[:, 0], minlength=C)
    assert u.max() < 1.6 * exp and u.min() > 0.5 * exp   # flat
    assert z.max() > 8 * exp                             # one code dominates: Zipf(1.1) over 256 ranks
    assert (z > 0).sum() > C // 2                        # and the tail is still drawn


def test_items_refuse_more_than_the_code_space():
    with pytest.raises(ValueError):
        wl.draw_items(16 * 16 + 1, 2, 16, "uniform", seed=0)
    full = wl.draw_items(16 * 16, 2, 16, "uniform", seed=0)  # every tuple exactly once
    assert len(np.unique(full, axis=0)) == 256


def test_host_streams_are_reproducible_and_independent():
    a = wl.host_normal((4, 1000), seed=1, tag=wl.TAG_Q)
    assert a.dtype == np.float32
    assert np.array_equal(a, wl.host_normal((4, 1000), seed=1, tag=wl.TAG_Q))
    b = wl.host_normal((4, 1000), seed=1, tag=wl.TAG_CTX_K)
    assert abs(np.corrcoef(a.ravel(), b.ravel())[0, 1]) < 0.05
    s = wl.host_normal((200_000,), seed=1, tag=wl.TAG_LOGITS, std=2.0)
    assert abs(s.std() - 2.0) < 0.02 and abs(s.mean()) < 0.02


def test_device_streams_are_reproducible_per_layer():
    a = wl.device_normal((64, 8), 1, wl.TAG_Q, "cpu", sub=3)
    assert torch.equal(a, wl.device_normal((64, 8), 1, wl.TAG_Q, "cpu", sub=3))
    assert not torch.equal(a, wl.device_normal((64, 8), 1, wl.TAG_Q, "cpu", sub=4))
    assert wl.device_normal((4,), 1, wl.TAG_Q, "cpu", dtype=torch.bfloat16).dtype == torch.bfloat16


def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(100_000).astype(np.float32) * 7,
        # exact ties: a bf16 value plus half an ulp, with even and odd last kept bits
        (np.arange(1, 4001, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1e-40, -1e-40, 3.0e38, -3.0e38], dtype=np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = wl.round_to_bf16(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(wl.bf16_bits(got), (ref.view(np.uint32) >> 16).astype(np.uint16))
