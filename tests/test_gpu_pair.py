"""The two decode-attention kernels against the oracle.

gr_beam_set_attn_kernel forces either kernel: the single-CTA one (two 128-row
query tiles per CTA sharing whole K/V tiles) or the CTA-pair one (cta_group::2
MMAs with M = 256, each CTA of a pair holding half of every K/V tile).  The
same shapes run on both and are compared element-wise with the oracle's
float64 attention over the concatenated context + BeamKV sequence:
|gpu - ref| <= 1e-2 + 1e-2*|ref|.  Shapes: context lengths around the 64-key
half tiles and the 128-key tiles, one- and two-tile units, GQA groups 1..16,
units cut over several pairs and pairs running several jobs, two BeamKV
levels, a captured graph replayed, and the timeout path.
"""
import pytest

from beam_decode_gb300 import binding as B
from tests.harness import GraphStep, LockStep, Spec

pytestmark = pytest.mark.gpu

MODES = {1: "single", 2: "pair"}


def _run(spec, mode, steps=1):
    ls = LockStep(spec)
    ls.beam.set_attn_kernel(mode)
    assert ls.beam.attn_kernel() == MODES[mode]
    r0 = ls.topk_step()
    assert not r0["mismatch"], r0
    worst = 0.0
    for t in range(1, steps + 1):
        for layer in range(spec.n_layers):
            worst = max(worst, ls.attention(layer)["worst"])
        r = ls.topk_step()
        assert not r["mismatch"], (t, r)
    assert ls.beam.status() == 0
    return worst


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 128, 129, 1000, 4097])
def test_context_lengths_both_kernels(T, mode):
    spec = Spec(n_q_heads=4, n_kv_heads=2, head_dim=128, vocab=2048, n_levels=2, codes_per_level=64,
                code_base=1024, ctx_lens=[T], widths=[128], n_items=[2000], seed=T + 7 * mode)
    assert _run(spec, mode) <= 1.0


@pytest.mark.parametrize("G,W", [(1, 256), (2, 200), (4, 64), (8, 16), (2, 256), (16, 8), (16, 24), (2, 30),
                                 (2, 512), (1, 1000)])
def test_groups_and_widths_on_pairs(G, W):
    # one-tile units (W * G <= 128) leave the second CTA of the pair without rows
    Hkv = 2
    spec = Spec(n_q_heads=G * Hkv, n_kv_heads=Hkv, head_dim=128, vocab=2048, n_levels=2, codes_per_level=256,
                code_base=1024, ctx_lens=[777], widths=[W], n_items=[60000], seed=G * 1000 + W)
    assert _run(spec, 2) <= 1.0


@pytest.mark.parametrize("mode", [1, 2])
def test_cut_units_many_jobs_two_levels(mode):
    # 24 units over the pairs: units cut over several pairs (pieces and merges) and pairs that
    # run several jobs; two BeamKV levels (ancestry through BeamPath)
    spec = Spec(n_layers=2, n_q_heads=16, n_kv_heads=8, head_dim=128, vocab=8192, n_levels=3,
                codes_per_level=128, code_base=8192 - 384, ctx_lens=[3000, 1, 700, 6000],
                widths=[256, 5, 96, 128], n_items=[8000] * 4, seed=41 + mode)
    assert _run(spec, mode, steps=2) <= 1.0


def test_long_cut_unit_on_pairs():
    # one unit of 40,000 keys: cut over many pairs, every other pair publishes a piece of it
    spec = Spec(n_q_heads=2, n_kv_heads=1, head_dim=128, vocab=2048, n_levels=2, codes_per_level=64,
                code_base=1024, ctx_lens=[40000], widths=[128], n_items=[3000], seed=55)
    assert _run(spec, 2) <= 1.0


def test_captured_step_on_pairs():
    spec = Spec(n_layers=2, n_q_heads=16, n_kv_heads=8, head_dim=128, vocab=8192, n_levels=3,
                codes_per_level=256, code_base=8192 - 768, ctx_lens=[1500, 300], widths=[256, 128],
                n_items=[60000], seed=73)
    import torch
    ls = LockStep(spec)
    ls.beam.set_attn_kernel(2)
    assert ls.beam.attn_kernel() == "pair"
    assert not ls.topk_step()["mismatch"]
    g = GraphStep(ls)
    for t in (1, 2):
        res = g.replay()
        assert res["worst"] <= 1.0 and not res["mismatch"], (t, res)
    torch.cuda.synchronize()
    ls.beam.set_graph_mode(False)
    ls.beam.sync()
    assert ls.beam.status() == 0


def test_forced_timeout_on_pairs_and_context_survives():
    import torch
    spec = Spec(n_q_heads=4, n_kv_heads=2, head_dim=128, vocab=2048, codes_per_level=64, code_base=1024,
                ctx_lens=[2000], widths=[128], n_items=[3000], seed=32)
    ls = LockStep(spec)
    beam = ls.beam
    beam.set_attn_kernel(2)
    ls.topk_step()
    ls.write_beam_kv(1, 0)
    q = torch.randn((beam.rows, 4, 128), device="cuda").to(torch.bfloat16)
    out = torch.zeros_like(q)
    beam.set_wait_limit(-1)            # every pipeline wait gives up on its first failed check
    beam.decode_attn(0, q, out)
    torch.cuda.synchronize()
    assert beam.status(clear=True) == B.GR_ERR_TIMEOUT
    beam.set_wait_limit(0)             # back to the default limit: the same call now succeeds
    beam.rewind(1)
    res = ls.attention(0)
    assert res["worst"] <= 1.0, res
    assert beam.status() == 0


def test_pair_kernel_needs_head_dim_128():
    ls = LockStep(Spec())              # head_dim 64
    with pytest.raises(B.GrError) as e:
        ls.beam.set_attn_kernel(2)
    assert e.value.status == B.GR_ERR_UNSUPPORTED
    assert ls.beam.attn_kernel() == "single"
