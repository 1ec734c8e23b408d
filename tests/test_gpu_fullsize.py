"""Parity at the benchmark's full size and launch configuration.

8 requests x context 5000 x beam 256, 28 layers, 16 q / 8 KV heads, head_dim
128, vocabulary 151,936, 3 levels x 256 codes, 1M items: the batch that
bench.py times.  The oracle checks, one by one, sampled attention rows (all
heads) of the first and last layer for the first and last request, and every
row of both top-K steps (bit-exact under the float32 key contract; the GPU's
own LSE within 1e-4 and the same selection).
"""
import numpy as np
import pytest

from tests.harness import ATOL, LP_TOL, RTOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def full():
    import torch
    from bench import DeviceBatch
    from beam_decode_gb300 import workload as wl
    w = wl.make_workload("long")
    b = DeviceBatch(w, "cuda")
    yield w, b
    del b
    torch.cuda.empty_cache()


def _oracle_beams(w, items):
    from oracle import OracleBeam, Trie
    trie = Trie(items[0], codes_per_level=w.codes_per_level)
    return [OracleBeam(trie, w.beam_widths[r], w.n_levels, w.codes_per_level, w.code_base, key_mode="f32")
            for r in range(w.n_requests)]


def test_fullsize_topk_and_attention(full):
    import torch
    from oracle import beam_attention, log_softmax_row
    w, b = full
    beam = b.beam
    obs = _oracle_beams(w, b.items)
    ro = beam.row_offsets
    # ---- step 0, bit-exact
    beam.rewind(0)
    x0 = b.logits[0].cpu().numpy()
    lse0 = np.zeros(b.rows, dtype=np.float32)
    for r in range(w.n_requests):
        row = x0[ro[r]]
        lse0[ro[r]] = np.float32(log_softmax_row(row)[1])
        obs[r].step(row[None], lse_in=[lse0[ro[r]]])
    beam.constrained_topk(b.logits[0], lse_in=torch.from_numpy(lse0).cuda())
    beam.advance()
    for r in range(w.n_requests):
        par, tok, nod, sc = beam.path(r, 0)
        assert np.array_equal(tok - w.code_base, np.array(obs[r].codes[0]))
        assert np.array_equal(sc.view(np.uint32), np.array(obs[r].scores[0], dtype=np.float32).view(np.uint32))
    # ---- step 1 attention (bench launch configuration), sampled rows checked one by one
    for l in range(w.n_layers):
        k, v = beam.kv_slot(l)
        k.copy_(b.new_k[l])
        v.copy_(b.new_v[l])
        beam.decode_attn(l, b.q[l], b.out[l])
    torch.cuda.synchronize()
    assert beam.status() == 0
    worst = 0.0
    for l in (0, w.n_layers - 1):
        out = b.out[l].float().cpu().numpy()
        q = b.q[l].float().cpu().numpy()
        nk = b.new_k[l].float().cpu().numpy()
        nv = b.new_v[l].float().cpu().numpy()
        for r in (0, w.n_requests - 1):
            T, o0, r0, W = w.ctx_lens[r], int(b.ctx_off[r]), ro[r], w.beam_widths[r]
            ck = b.ctx_k[l, :, o0:o0 + T].float().cpu().numpy()
            cv = b.ctx_v[l, :, o0:o0 + T].float().cpu().numpy()
            anc = obs[r].ancestry()
            beams = [0, 1, 63, 64, 127, 128, 200, obs[r].n_live() - 1]
            ref = beam_attention(q[r0:r0 + W], ck, cv, [nk[r0:r0 + W]], [nv[r0:r0 + W]], anc, beams=beams)
            got = out[r0 + np.array(beams)]
            worst = max(worst, float(np.max(np.abs(got - ref) / (ATOL + RTOL * np.abs(ref)))))
    assert worst <= 1.0, worst
    # ---- step 1 top-K, bit-exact on every row
    x1 = b.logits[1].cpu().numpy()
    lse1 = np.zeros(b.rows, dtype=np.float32)
    lse64 = np.zeros(b.rows)
    for r in range(w.n_requests):
        n = obs[r].n_live()
        rows = x1[ro[r]:ro[r] + n]
        l64 = np.array([log_softmax_row(rw)[1] for rw in rows])
        lse64[ro[r]:ro[r] + n] = l64
        lse1[ro[r]:ro[r] + n] = l64.astype(np.float32)
        obs[r].step(rows, lse_in=lse1[ro[r]:ro[r] + n])
    beam.constrained_topk(b.logits[1], lse_in=torch.from_numpy(lse1).cuda())
    beam.advance()
    for r in range(w.n_requests):
        par, tok, nod, sc = beam.path(r, 1)
        assert np.array_equal(par, np.array(obs[r].parents[1]))
        assert np.array_equal(tok - w.code_base - w.codes_per_level, np.array(obs[r].codes[1]))
        assert np.array_equal(sc.view(np.uint32), np.array(obs[r].scores[1], dtype=np.float32).view(np.uint32))
    # ---- the GPU's own LSE (the benchmark's mode): within 1e-4, same selection
    beam.rewind(1)
    lse_out = torch.full((b.rows,), float("nan"), device="cuda")
    beam.constrained_topk(b.logits[1], lse_out=lse_out)
    beam.advance()
    g = lse_out.cpu().numpy()
    live = np.isfinite(lse64) & (lse64 != 0)
    assert np.max(np.abs(g[live] - lse64[live])) <= LP_TOL
    for r in range(w.n_requests):
        par, tok, _, _ = beam.path(r, 1)
        assert np.array_equal(par, np.array(obs[r].parents[1]))
        assert np.array_equal(tok - w.code_base - w.codes_per_level, np.array(obs[r].codes[1]))
    assert beam.status() == 0


def test_fullsize_captured_step_matches_oracle(full):
    """The benchmark's own captured graph (bench.DeviceBatch.capture: rewind to step 1, 28
    attention layers, the top-K with the GPU's own LSE, advance), replayed once and checked
    against the oracle: sampled attention rows of the first and last layer for the first and
    last request, and every request's selection at level 1."""
    import torch
    from oracle import beam_attention, log_softmax_row
    w, b = full
    beam = b.beam
    obs = _oracle_beams(w, b.items)
    ro = beam.row_offsets
    # level 0 as in the benchmark's set-up, with the oracle's LSE so both sides hold the same beams
    beam.rewind(0)
    x0 = b.logits[0].cpu().numpy()
    lse0 = np.zeros(b.rows, dtype=np.float32)
    for r in range(w.n_requests):
        lse0[ro[r]] = np.float32(log_softmax_row(x0[ro[r]])[1])
        obs[r].step(x0[ro[r]][None], lse_in=[lse0[ro[r]]])
    beam.constrained_topk(b.logits[0], lse_in=torch.from_numpy(lse0).cuda())
    beam.advance()
    for l in range(w.n_layers):
        k, v = beam.kv_slot(l)
        k.copy_(b.new_k[l])
        v.copy_(b.new_v[l])
    b.capture()
    for l in range(w.n_layers):
        b.out[l].fill_(float("nan"))
    b.graph.replay()
    torch.cuda.synchronize()
    b.release()
    assert beam.status() == 0
    worst = 0.0
    for l in (0, w.n_layers - 1):
        out = b.out[l].float().cpu().numpy()
        q = b.q[l].float().cpu().numpy()
        nk = b.new_k[l].float().cpu().numpy()
        nv = b.new_v[l].float().cpu().numpy()
        for r in (0, w.n_requests - 1):
            T, o0, r0, W = w.ctx_lens[r], int(b.ctx_off[r]), ro[r], w.beam_widths[r]
            ck = b.ctx_k[l, :, o0:o0 + T].float().cpu().numpy()
            cv = b.ctx_v[l, :, o0:o0 + T].float().cpu().numpy()
            beams = [0, 5, 127, 128, 129, 250, obs[r].n_live() - 1]
            ref = beam_attention(q[r0:r0 + W], ck, cv, [nk[r0:r0 + W]], [nv[r0:r0 + W]], obs[r].ancestry(),
                                 beams=beams)
            got = out[r0 + np.array(beams)]
            worst = max(worst, float(np.max(np.abs(got - ref) / (ATOL + RTOL * np.abs(ref)))))
    assert worst <= 1.0, worst
    # level 1 from the GPU's own LSE: the same selection as the oracle's
    x1 = b.logits[1].cpu().numpy()
    for r in range(w.n_requests):
        n = obs[r].n_live()
        rows = x1[ro[r]:ro[r] + n]
        obs[r].step(rows, lse_in=np.array([log_softmax_row(rw)[1] for rw in rows], dtype=np.float32))
        par, tok, _, _ = beam.path(r, 1)
        assert np.array_equal(par, np.array(obs[r].parents[1])), r
        assert np.array_equal(tok - w.code_base - w.codes_per_level, np.array(obs[r].codes[1])), r
