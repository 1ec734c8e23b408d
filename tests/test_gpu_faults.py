"""Error paths through the C ABI on a GPU: call-order and argument errors are
returned synchronously; a NaN key is reported through the device status word;
a forced wait timeout inside the attention kernel is reported as
GR_ERR_TIMEOUT and leaves the CUDA context usable (no fault, trap or hang:
every wait is bounded and the kernel drains its own copies before returning)."""
import numpy as np
import pytest

from beam_decode_gb300 import binding as B
from tests.harness import LockStep, Spec

pytestmark = pytest.mark.gpu


def _code(fn, *a, **k):
    try:
        fn(*a, **k)
    except B.GrError as e:
        return e.status
    return 0


def test_call_order_and_arguments():
    import torch
    ls = LockStep(Spec(n_layers=2))
    beam = ls.beam
    q = torch.zeros((beam.rows, 2, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    x = torch.zeros((beam.rows, 1024), device="cuda")
    assert _code(beam.decode_attn, 0, q, out) == B.GR_ERR_STATE          # no attention at step 0
    assert _code(beam.advance) == B.GR_ERR_STATE                          # advance before top-K
    assert _code(beam.kv_slot, 0) == B.GR_ERR_STATE
    assert _code(beam.results, 0) == B.GR_ERR_STATE
    assert _code(beam.rewind, 1) == B.GR_ERR_STATE
    assert _code(beam.constrained_topk, x, ld=1022) == B.GR_ERR_INVALID_ARG
    assert _code(beam.constrained_topk, x[:, 1:], ld=1024) == B.GR_ERR_INVALID_ARG  # misaligned
    ls.topk_step()
    assert _code(beam.decode_attn, 2, q, out) == B.GR_ERR_INVALID_ARG     # layer out of range
    qm = torch.zeros(q.numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + q.numel()].view_as(q)
    assert _code(beam.decode_attn, 0, qm, out) == B.GR_ERR_INVALID_ARG    # misaligned q
    assert _code(beam.decode_attn, 0, q, out) == 0
    assert _code(beam.decode_attn, 0, q, out) == B.GR_ERR_STATE           # same layer twice
    assert _code(beam.constrained_topk, x) == 0
    assert _code(beam.decode_attn, 1, q, out) == B.GR_ERR_STATE           # attention after top-K
    assert _code(beam.constrained_topk, x) == B.GR_ERR_STATE              # top-K twice
    assert beam.status() == 0


def test_workspace_too_small():
    import ctypes
    import torch
    ls = LockStep(Spec())
    b = ls.beam
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    bufs = B.GrBuffers(b.ctx_k.data_ptr(), b.ctx_v.data_ptr(), b.beam_k.data_ptr(), b.beam_v.data_ptr(),
                       small.data_ptr(), small.numel())
    h = ctypes.c_void_p()
    st = B.lib().gr_beam_create(ctypes.byref(b.cfg), b.reqs, 1, ctypes.byref(bufs), None, ctypes.byref(h))
    assert st == B.GR_ERR_CAPACITY and not h.value


def test_duplicate_items_rejected():
    with pytest.raises(B.GrError) as e:
        B.Trie(np.array([[1, 2], [1, 2]], dtype=np.int32), codes_per_level=16)
    assert e.value.status == B.GR_ERR_INVALID_ARG


def test_nan_key_reported():
    def nan_logits(ls, t, x):
        x = x.copy()
        x[:, ls.spec.code_base:ls.spec.code_base + ls.spec.codes_per_level] = np.nan
        return x
    ls = LockStep(Spec(), logits_fn=nan_logits)
    import torch
    x = torch.from_numpy(ls.logits(0)).cuda()
    ls.beam.constrained_topk(x)
    ls.beam.advance()
    assert ls.beam.status(clear=True) == B.GR_ERR_DEVICE
    assert ls.beam.status() == 0


def test_forced_timeout_is_reported_and_context_survives():
    import torch
    spec = Spec(n_q_heads=4, n_kv_heads=2, head_dim=128, vocab=2048, codes_per_level=64, code_base=1024,
                ctx_lens=[2000], widths=[128], n_items=[3000], seed=31)
    ls = LockStep(spec)
    ls.topk_step()
    beam = ls.beam
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
