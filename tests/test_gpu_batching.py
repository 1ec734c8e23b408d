"""Continuous batching and CUDA-graph replay through the C ABI.

GR-native continuous batching and direct-pool-view CUDA-graph replay are named
by the zhiding.cn recsys-examples article, section "语义ID生成式推荐专用推理框架":
requests of different lengths, widths, contexts and catalogues share one batch
at their own steps, a finished slot takes a new request, and a captured step
replays with every decision taken from device-resident state.  Every
comparison is against the CPU oracle, except graph replay, which must equal
the eager run of the same inputs bit for bit.
"""
import numpy as np
import pytest

from beam_decode_gb300 import binding as B
from beam_decode_gb300 import workload as wl
from tests.harness import MixedDriver, Occupant

pytestmark = pytest.mark.gpu


def test_mixed_lengths_in_one_batch():
    occ = [Occupant(ctx_len=200, width=16, n_levels=3, n_items=400, key=1),
           Occupant(ctx_len=130, width=40, n_levels=2, n_items=300, key=2),
           Occupant(ctx_len=70, width=8, n_levels=1, n_items=20, key=3)]
    d = MixedDriver(occ, [16, 40, 8])
    for k in range(3):
        r = d.step()
        assert r["worst"] <= 1.0 and not r["mismatch"], (k, r)
    assert sorted(d.finished) == [0, 1, 2]
    assert d.beam.status() == 0


def test_finished_slot_takes_new_request():
    occ = [Occupant(ctx_len=300, width=24, n_levels=2, n_items=500, key=11),   # slot 0 first
           Occupant(ctx_len=257, width=32, n_levels=3, n_items=800, key=12),   # slot 1 first
           Occupant(ctx_len=140, width=16, n_levels=3, n_items=600, key=13),   # into slot 0 (narrower)
           Occupant(ctx_len=64, width=24, n_levels=1, n_items=25, key=14)]     # into slot 1, one level
    d = MixedDriver(occ, [24, 32], head_dim=128, seed=51)
    plan = {2: [(0, 2)], 3: [(1, 3)]}   # batch step -> admissions made before it
    for k in range(5):
        for slot, o in plan.get(k, []):
            d.admit(slot, o)
        r = d.step()
        assert r["worst"] <= 1.0 and not r["mismatch"], (k, r)
    assert sorted(d.finished) == [0, 1, 2, 3]
    # a slot still decoding, a wider request or the middle of a step cannot admit
    d2 = MixedDriver(occ, [24, 32], seed=52)
    d2.step()
    with pytest.raises(B.GrError) as e:
        d2.admit(0, 2)
    assert e.value.status == B.GR_ERR_STATE
    d2.step()  # slot 0 finished
    with pytest.raises(B.GrError) as e:
        d2.beam.admit(0, d2.ctx_off[1], 10, 25, d2.gtries[1])
    assert e.value.status == B.GR_ERR_CAPACITY
    assert d.beam.status() == 0 and d2.beam.status() == 0


def test_many_narrow_requests_share_ctas():
    # 200 narrow requests (one query tile per unit, 1-4 key tiles) give far more units than
    # CTAs: the schedule packs several whole units into a CTA, so merging jobs follow one
    # another inside a CTA, each staging its BeamKV keys in the rings before the next loads
    widths = [8, 16, 32, 64]
    occ = [Occupant(ctx_len=90 + (37 * r) % 320, width=widths[r % 4], n_levels=2, n_items=60, key=100 + r)
           for r in range(200)]
    d = MixedDriver(occ, [o.width for o in occ], n_levels_max=2, seed=57)
    for k in range(2):
        r = d.step()
        assert r["worst"] <= 1.0 and not r["mismatch"], (k, r["worst"], r["mismatch"][:3])
    assert sorted(d.finished) == list(range(200))
    assert d.beam.status() == 0


def _batch(seed, device="cuda"):
    import torch
    L, NL, Hq, Hkv, D, V, C = 3, 2, 4, 2, 128, 4096, 64
    widths, ctx = [64, 200], [300, 700]
    items = [wl.draw_items(3000, L, C, "uniform", seed, stream=(r,)) for r in range(2)]
    tries = [B.Trie(it, codes_per_level=C, device=device) for it in items]
    off, offs = 3, []
    for T in ctx:
        offs.append(off)
        off += T + 5
    kc = torch.from_numpy(wl.round_to_bf16(wl.host_normal((NL, Hkv, off, D), seed, wl.TAG_CTX_K))).to(torch.bfloat16)
    vc = torch.from_numpy(wl.round_to_bf16(wl.host_normal((NL, Hkv, off, D), seed, wl.TAG_CTX_V))).to(torch.bfloat16)
    beam = B.Beam(NL, Hq, Hkv, D, V, V - L * C, L, C, kc.to(device), vc.to(device),
                  [(offs[r], ctx[r], widths[r], tries[r]) for r in range(2)], device=device)
    rows = beam.rows
    # BeamKV of both open levels, written straight into the pool
    for t in (1, 2):
        for layer in range(NL):
            k = wl.round_to_bf16(wl.host_normal((rows, Hkv, D), seed, wl.TAG_BEAM_K, sub=(t, layer)))
            v = wl.round_to_bf16(wl.host_normal((rows, Hkv, D), seed, wl.TAG_BEAM_V, sub=(t, layer)))
            beam.beam_k[layer, t - 1].copy_(torch.from_numpy(k).to(torch.bfloat16))
            beam.beam_v[layer, t - 1].copy_(torch.from_numpy(v).to(torch.bfloat16))
    q = {(t, l): torch.from_numpy(wl.round_to_bf16(wl.host_normal((rows, Hq, D), seed, wl.TAG_Q, sub=(t, l))))
         .to(torch.bfloat16).to(device) for t in (1, 2) for l in range(NL)}
    x = {t: torch.from_numpy(wl.host_normal((rows, V), seed, wl.TAG_LOGITS, sub=(t,), std=2.0)).to(device)
         for t in range(L)}
    return beam, q, x, NL


def test_captured_step_replays_like_eager():
    import torch
    # eager reference
    beam, q, x, NL = _batch(61)
    outs_e = {}
    beam.constrained_topk(x[0])
    beam.advance()
    for t in (1, 2):
        for l in range(NL):
            outs_e[(t, l)] = torch.empty_like(q[(t, l)])
            beam.decode_attn(l, q[(t, l)], outs_e[(t, l)])
        beam.constrained_topk(x[t])
        beam.advance()
    ref = [beam.results(r) for r in range(2)]
    # graph: step 0 eagerly, one warm-up step (then rewound), capture step 1, replay it twice
    g_beam, q, x, NL = _batch(61)
    g_beam.constrained_topk(x[0])
    g_beam.advance()
    q_st = [torch.empty_like(q[(1, l)]) for l in range(NL)]
    o_st = [torch.empty_like(q[(1, l)]) for l in range(NL)]
    x_st = torch.empty_like(x[1])
    for l in range(NL):
        q_st[l].copy_(q[(1, l)])
    x_st.copy_(x[1])
    for l in range(NL):
        g_beam.decode_attn(l, q_st[l], o_st[l])
    g_beam.constrained_topk(x_st)
    g_beam.advance()
    g_beam.rewind(1)
    torch.cuda.synchronize()
    g_beam.set_graph_mode(True)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for l in range(NL):
            g_beam.decode_attn(l, q_st[l], o_st[l])
        g_beam.constrained_topk(x_st)
        g_beam.advance()
    for t in (1, 2):
        for l in range(NL):
            q_st[l].copy_(q[(t, l)])
        x_st.copy_(x[t])
        graph.replay()
        for l in range(NL):
            assert torch.equal(o_st[l], outs_e[(t, l)]), (t, l)
    torch.cuda.synchronize()
    g_beam.set_graph_mode(False)
    g_beam.sync()
    assert [g_beam.request_step(r)[0] for r in range(2)] == [3, 3]
    for r in range(2):
        got = g_beam.results(r)
        for a, b in zip(got, ref[r]):
            assert np.array_equal(a, b)
    assert g_beam.status() == 0
