"""gr_constrained_topk_noalloc: the constrained top-K for callers that cannot
allocate device memory (a plugin handed only its input and output tensors, a
service whose device memory is fixed at start-up).  Its scratch is a fixed
array inside the library; this test checks, through the C ABI, that two calls
in a row return the same selection as gr_constrained_topk on the same inputs,
and that sizes beyond the fixed scratch are refused.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest

from beam_decode_gb300 import binding as B
from tests.harness import LP_TOL, LockStep, Spec

pytestmark = pytest.mark.gpu


def _call(x, ld, n_rows, vocab, code_lo, n_codes, scores, mask, k, outs):
    import torch
    p, c, key, n = outs
    return B.lib().gr_constrained_topk_noalloc(
        x.data_ptr(), ld, n_rows, vocab, code_lo, n_codes, None if scores is None else scores.data_ptr(),
        mask.data_ptr(), k, p.data_ptr(), c.data_ptr(), key.data_ptr(), n.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_constrained_topk_twice():
    import torch
    C = 256
    spec = Spec(n_q_heads=2, n_kv_heads=1, head_dim=64, vocab=4096, n_levels=2, codes_per_level=C,
                code_base=4096 - 2 * C, ctx_lens=[8], widths=[64], n_items=[20000], seed=41)
    ls = LockStep(spec)
    ls.topk_step()                                   # level 0 through the existing path
    beam = ls.beam
    _, tok0, _, sc0 = beam.path(0, 0)
    n = len(tok0)
    code0 = tok0 - spec.code_base
    items = ls.items[0]
    mask = np.zeros((n, C // 32), dtype=np.uint32)
    for b in range(n):
        for c in np.unique(items[items[:, 0] == code0[b], 1]):
            mask[b, c >> 5] |= np.uint32(1) << np.uint32(c & 31)
    x = torch.from_numpy(ls.logits(1)).cuda()
    ld = x.shape[1]
    # existing entry point at step 1
    beam.constrained_topk(x)
    beam.advance()
    par1, tok1, _, sc1 = beam.path(0, 1)
    # the no-alloc entry point, twice, on the first n rows
    dmask = torch.from_numpy(mask.view(np.int32)).cuda()
    dscore = torch.from_numpy(sc0.astype(np.float32)).cuda()
    k = spec.widths[0]
    for _ in range(2):
        outs = (torch.full((k,), -1, dtype=torch.int32, device="cuda"),
                torch.full((k,), -1, dtype=torch.int32, device="cuda"),
                torch.full((k,), float("nan"), device="cuda"),
                torch.zeros(1, dtype=torch.int32, device="cuda"))
        st = _call(x, ld, n, spec.vocab, spec.code_base + C, C, dscore, dmask, k, outs)
        assert st == 0, B.lib().gr_last_error().decode()
        torch.cuda.synchronize()
        m = int(outs[3].item())
        assert m == len(par1)
        assert np.array_equal(outs[0].cpu().numpy()[:m], par1)
        assert np.array_equal(outs[1].cpu().numpy()[:m], tok1 - spec.code_base - C)
        assert np.max(np.abs(outs[2].cpu().numpy()[:m] - sc1)) <= LP_TOL


def test_noalloc_refuses_sizes_beyond_scratch():
    import torch
    x = torch.zeros((8, 1024), device="cuda")
    mask = torch.zeros((8, 32), dtype=torch.int32, device="cuda")
    outs = (torch.zeros(8, dtype=torch.int32, device="cuda"), torch.zeros(8, dtype=torch.int32, device="cuda"),
            torch.zeros(8, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda"))
    too_many_rows = B.GR_NOALLOC_MAX_CANDIDATES // 1024 + 1
    assert _call(x, 1024, too_many_rows, 1024, 0, 1024, None, mask, 8, outs) == B.GR_ERR_CAPACITY
    assert _call(x, 1024, 8, 1024, 0, 1024, None, mask, 2048, outs) == B.GR_ERR_CAPACITY
    assert _call(x, 1024, 8, 1024, 0, 2048, None, mask, 8, outs) == B.GR_ERR_CAPACITY
