"""Direct-pool-view CUDA-graph replay against the oracle.

The zhiding.cn recsys-examples article, section "语义ID生成式推荐专用推理框架",
names CUDA-graph replay of a step that works directly on the KV pools.  Here a
whole decode step (attention for every layer, the constrained top-K, the
BeamPath advance) is captured once in graph mode and replayed for the later
steps with fresh inputs; every replay is compared with the CPU oracle --
attention element-wise within 1e-2 + 1e-2*|ref|, the selection (parents,
tokens, scores) bit for bit under the float32 key contract -- and the final
beams with the oracle's results.
"""
import numpy as np
import pytest

from tests.harness import GraphStep, LockStep, Spec

pytestmark = pytest.mark.gpu


def _check_results(ls):
    for r in range(len(ls.spec.ctx_lens)):
        codes, items, scores = ls.gpu_results(r)
        exp = ls.obeams[r].results()
        assert len(codes) == len(exp), (r, len(codes), len(exp))
        for i, (tup, iid, sc) in enumerate(exp):
            assert tuple(int(c) for c in codes[i]) == tup, (r, i)
            assert int(items[i]) == iid
            assert np.float32(scores[i]).view(np.uint32) == np.float32(sc).view(np.uint32)


@pytest.mark.parametrize("spec", [
    # two requests of different context lengths; units cut over several CTAs
    Spec(n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=64, vocab=2048, n_levels=3, codes_per_level=32,
         code_base=2048 - 96, ctx_lens=[700, 1900], widths=[48, 64], n_items=[3000], seed=71),
    # Qwen3-1.7B head geometry (16 q / 8 KV heads, D 128), 256-code levels, two query tiles per unit
    Spec(n_layers=2, n_q_heads=16, n_kv_heads=8, head_dim=128, vocab=8192, n_levels=3, codes_per_level=256,
         code_base=8192 - 768, ctx_lens=[1000, 257], widths=[256, 96], n_items=[60000], seed=72),
], ids=["small", "qwen-heads"])
def test_captured_step_replays_match_oracle(spec):
    import torch
    ls = LockStep(spec)
    r0 = ls.topk_step(lse_mode=True)          # level 0, eager
    assert not r0["mismatch"], r0
    g = GraphStep(ls)
    for t in range(1, spec.n_levels):
        res = g.replay()
        assert res["worst"] <= 1.0, (t, res["worst"])
        assert not res["mismatch"], (t, res)
    torch.cuda.synchronize()
    ls.beam.set_graph_mode(False)
    ls.beam.sync()
    _check_results(ls)
    assert ls.beam.status() == 0
