"""ctypes binding of libgrbeam (include/grbeam.h): argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels.  PyTorch
supplies device memory and the current CUDA stream.  If the shared library is
missing the import of this module still works, but the first call raises
``RuntimeError``: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libgrbeam.so")

GR_OK = 0
GR_ERR_INVALID_ARG = -1
GR_ERR_UNSUPPORTED = -2
GR_ERR_CAPACITY = -3
GR_ERR_STATE = -4
GR_ERR_CUDA = -5
GR_ERR_TIMEOUT = -6
GR_ERR_DEVICE = -7
GR_NOALLOC_MAX_CANDIDATES = 256 * 1024

KERNEL_ATTN = 0
KERNEL_LOGSOFTMAX = 1
KERNEL_TOPK = 2
KERNEL_ADVANCE = 3
KERNEL_RESULTS = 4
KERNEL_INIT = 5
KERNEL_KINDS = 6
KERNEL_NAMES = ["attn", "logsoftmax_gather", "topk_select", "advance", "results", "init"]

# exported symbols of include/grbeam.h
SYMBOLS = [
    "gr_trie_device_bytes", "gr_trie_create", "gr_trie_destroy",
    "gr_beam_workspace_bytes", "gr_beam_kv_bytes", "gr_attn_schedule", "gr_beam_create", "gr_beam_destroy",
    "gr_beam_rows", "gr_beam_step", "gr_beam_request_step", "gr_beam_kv_slot", "gr_beam_kv_slot_request",
    "gr_decode_attn", "gr_constrained_topk", "gr_beam_advance", "gr_beam_rewind", "gr_beam_admit",
    "gr_beam_set_graph_mode", "gr_beam_sync", "gr_beam_results", "gr_beam_path", "gr_beam_status",
    "gr_beam_set_timing", "gr_beam_kernel_stats", "gr_beam_set_wait_limit", "gr_beam_set_attn_kernel",
    "gr_beam_attn_kernel",
    "gr_constrained_topk_noalloc", "gr_status_str", "gr_last_error",
    "gr_score_workspace_bytes", "gr_score_create", "gr_score_destroy", "gr_score_rows", "gr_score_attn",
    "gr_score_labels", "gr_score_status",
]


class GrConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("vocab", ctypes.c_int), ("code_base", ctypes.c_int),
                ("n_levels", ctypes.c_int), ("codes_per_level", ctypes.c_int), ("pool_tokens", ctypes.c_int64)]


class GrRequest(ctypes.Structure):
    _fields_ = [("ctx_offset", ctypes.c_int64), ("ctx_len", ctypes.c_int), ("beam_width", ctypes.c_int),
                ("trie", ctypes.c_void_p)]


class GrBuffers(ctypes.Structure):
    _fields_ = [("ctx_k", ctypes.c_void_p), ("ctx_v", ctypes.c_void_p), ("beam_k", ctypes.c_void_p),
                ("beam_v", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class GrScoreConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("vocab", ctypes.c_int), ("pool_tokens", ctypes.c_int64),
                ("n_labels", ctypes.c_int), ("label_ids", ctypes.c_void_p)]


class GrScoreRequest(ctypes.Structure):
    _fields_ = [("ctx_offset", ctypes.c_int64), ("ctx_len", ctypes.c_int), ("n_candidates", ctypes.c_int),
                ("seg_lens", ctypes.c_void_p)]


class GrScoreBuffers(ctypes.Structure):
    _fields_ = [("ctx_k", ctypes.c_void_p), ("ctx_v", ctypes.c_void_p), ("seg_k", ctypes.c_void_p),
                ("seg_v", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class GrError(RuntimeError):
    def __init__(self, status: int, name: str, message: str):
        super().__init__(f"{name}: {message}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libgrbeam is not built ({LIB_PATH} missing): run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        c_int, c_i64, vp, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
        P = ctypes.POINTER
        sig = {
            "gr_trie_device_bytes": [vp, c_i64, c_int, c_int, P(sz)],
            "gr_trie_create": [vp, vp, c_i64, c_int, c_int, vp, sz, vp, P(vp)],
            "gr_trie_destroy": [vp],
            "gr_beam_workspace_bytes": [P(GrConfig), P(GrRequest), c_int, P(sz)],
            "gr_beam_kv_bytes": [P(GrConfig), P(GrRequest), c_int, P(sz)],
            "gr_attn_schedule": [P(GrConfig), vp, vp, c_int, c_int, c_int, P(c_int), P(c_int), P(c_int), vp, c_int, vp,
                                 c_int, vp, c_int],
            "gr_beam_create": [P(GrConfig), P(GrRequest), c_int, P(GrBuffers), vp, P(vp)],
            "gr_beam_destroy": [vp],
            "gr_beam_rows": [vp, P(c_int), vp],
            "gr_beam_step": [vp, P(c_int)],
            "gr_beam_request_step": [vp, c_int, P(c_int), P(c_int)],
            "gr_beam_kv_slot": [vp, c_int, P(vp), P(vp)],
            "gr_beam_kv_slot_request": [vp, c_int, c_int, P(vp), P(vp)],
            "gr_decode_attn": [vp, c_int, vp, vp, vp],
            "gr_constrained_topk": [vp, vp, c_i64, vp, vp, vp, vp],
            "gr_beam_advance": [vp, vp],
            "gr_beam_rewind": [vp, c_int, vp],
            "gr_beam_admit": [vp, c_int, P(GrRequest), vp],
            "gr_beam_set_graph_mode": [vp, c_int],
            "gr_beam_sync": [vp, vp],
            "gr_beam_results": [vp, c_int, vp, vp, vp, P(c_int), vp],
            "gr_beam_path": [vp, c_int, c_int, vp, vp, vp, vp, P(c_int), vp],
            "gr_beam_status": [vp, c_int, vp],
            "gr_beam_set_timing": [vp, c_int],
            "gr_beam_kernel_stats": [vp, c_int, P(c_i64), P(ctypes.c_double), c_int],
            "gr_beam_set_wait_limit": [vp, c_i64],
            "gr_beam_set_attn_kernel": [vp, c_int, vp],
            "gr_beam_attn_kernel": [vp, P(c_int)],
            "gr_constrained_topk_noalloc": [vp, c_i64, c_int, c_int, c_int, c_int, vp, vp, c_int, vp, vp, vp, vp,
                                            vp],
            "gr_score_workspace_bytes": [P(GrScoreConfig), P(GrScoreRequest), c_int, P(sz)],
            "gr_score_create": [P(GrScoreConfig), P(GrScoreRequest), c_int, P(GrScoreBuffers), vp, P(vp)],
            "gr_score_destroy": [vp],
            "gr_score_rows": [vp, P(c_int), vp, vp],
            "gr_score_attn": [vp, c_int, vp, vp, vp],
            "gr_score_labels": [vp, vp, c_i64, vp, vp, vp],
            "gr_score_status": [vp, c_int, vp],
            "gr_status_str": [c_int],
            "gr_last_error": [],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = c_int
        L.gr_status_str.restype = ctypes.c_char_p
        L.gr_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def check(status: int) -> None:
    if status != GR_OK:
        L = lib()
        raise GrError(status, L.gr_status_str(status).decode(), L.gr_last_error().decode())


def attn_schedule(n_q_heads: int, n_kv_heads: int, ctx_lens: Sequence[int], widths: Sequence[int],
                  n_sm: int, head_dim: int = 128, attn_kernel: int = 0) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """The attention schedule of a batch (gr_attn_schedule), host only: (units [n, 7], jobs [n, 4],
    ctas [n, 2]) int32 arrays with the columns the header lists.  attn_kernel: 0 automatic (the
    single-CTA kernel), 1 single-CTA, 2 the CTA-pair kernel (ctas are then CTA pairs)."""
    L = lib()
    cfg = GrConfig(n_layers=1, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, head_dim=head_dim, vocab=1, code_base=0,
                   n_levels=1, codes_per_level=1, pool_tokens=1)
    cl = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    bw = np.ascontiguousarray(widths, dtype=np.int32)
    nu, nj, nc = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    st = L.gr_attn_schedule(ctypes.byref(cfg), cl.ctypes.data, bw.ctypes.data, len(cl), n_sm, attn_kernel, ctypes.byref(nu),
                            ctypes.byref(nj), ctypes.byref(nc), None, 0, None, 0, None, 0)
    if st not in (GR_OK, GR_ERR_CAPACITY):
        check(st)
    units = np.zeros((nu.value, 7), np.int32)
    jobs = np.zeros((nj.value, 4), np.int32)
    ctas = np.zeros((nc.value, 2), np.int32)
    check(L.gr_attn_schedule(ctypes.byref(cfg), cl.ctypes.data, bw.ctypes.data, len(cl), n_sm, attn_kernel, ctypes.byref(nu),
                             ctypes.byref(nj), ctypes.byref(nc), units.ctypes.data, len(units), jobs.ctypes.data,
                             len(jobs), ctas.ctypes.data, len(ctas)))
    return units, jobs, ctas


def _stream_ptr(stream=None) -> ctypes.c_void_p:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


class Trie:
    """Item catalogue uploaded into a torch-owned device buffer."""

    def __init__(self, codes: np.ndarray, item_ids: Optional[np.ndarray] = None, codes_per_level: int = 256,
                 device="cuda"):
        import torch
        codes = np.ascontiguousarray(codes, dtype=np.int32)
        n, L = codes.shape
        self.n_levels, self.codes_per_level, self.n_items = L, codes_per_level, n
        ids = None if item_ids is None else np.ascontiguousarray(item_ids, dtype=np.int64)
        nbytes = ctypes.c_size_t()
        check(lib().gr_trie_device_bytes(codes.ctypes.data, n, L, codes_per_level, ctypes.byref(nbytes)))
        self.buffer = torch.empty(max(nbytes.value, 256), dtype=torch.uint8, device=device)
        h = ctypes.c_void_p()
        check(lib().gr_trie_create(codes.ctypes.data, None if ids is None else ids.ctypes.data, n, L,
                                   codes_per_level, self.buffer.data_ptr(), self.buffer.numel(), _stream_ptr(),
                                   ctypes.byref(h)))
        self.handle = h

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.gr_trie_destroy(self.handle)
            self.handle = None


class Beam:
    """One batch of requests being decoded (gr_beam handle + its device buffers)."""

    def __init__(self, n_layers: int, n_q_heads: int, n_kv_heads: int, head_dim: int, vocab: int,
                 code_base: int, n_levels: int, codes_per_level: int, ctx_k, ctx_v,
                 requests: Sequence[Tuple[int, int, int, Trie]], device="cuda"):
        """ctx_k / ctx_v: bf16 tensors [n_layers, n_kv_heads, pool_tokens, head_dim];
        requests: (ctx_offset, ctx_len, beam_width, trie) per request."""
        import torch
        assert ctx_k.dtype == torch.bfloat16 and ctx_v.dtype == torch.bfloat16
        assert ctx_k.is_contiguous() and ctx_v.is_contiguous()
        self.cfg = GrConfig(n_layers, n_q_heads, n_kv_heads, head_dim, vocab, code_base, n_levels,
                            codes_per_level, ctx_k.shape[2])
        n = len(requests)
        self.reqs = (GrRequest * n)(*[GrRequest(o, l, w, t.handle) for (o, l, w, t) in requests])
        self.tries = [t for (_, _, _, t) in requests]
        self.ctx_k, self.ctx_v = ctx_k, ctx_v
        self.n_requests = n
        self.widths = [w for (_, _, w, _) in requests]
        self.rows = sum(self.widths)
        ws = ctypes.c_size_t()
        check(lib().gr_beam_workspace_bytes(ctypes.byref(self.cfg), self.reqs, n, ctypes.byref(ws)))
        kvb = ctypes.c_size_t()
        check(lib().gr_beam_kv_bytes(ctypes.byref(self.cfg), self.reqs, n, ctypes.byref(kvb)))
        self.workspace = torch.empty(ws.value, dtype=torch.uint8, device=device)
        shape = (n_layers, max(n_levels - 1, 1), self.rows, n_kv_heads, head_dim)
        self.beam_k = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        self.beam_v = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        assert kvb.value <= self.beam_k.numel() * 2
        bufs = GrBuffers(ctx_k.data_ptr(), ctx_v.data_ptr(), self.beam_k.data_ptr(), self.beam_v.data_ptr(),
                         self.workspace.data_ptr(), self.workspace.numel())
        h = ctypes.c_void_p()
        check(lib().gr_beam_create(ctypes.byref(self.cfg), self.reqs, n, ctypes.byref(bufs), _stream_ptr(),
                                   ctypes.byref(h)))
        self.handle = h
        offs = (ctypes.c_int * (n + 1))()
        rows = ctypes.c_int()
        check(lib().gr_beam_rows(self.handle, ctypes.byref(rows), offs))
        self.row_offsets = list(offs)
        assert rows.value == self.rows

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.gr_beam_destroy(self.handle)
            self.handle = None

    # -- state -------------------------------------------------------------
    @property
    def step(self) -> int:
        s = ctypes.c_int()
        check(lib().gr_beam_step(self.handle, ctypes.byref(s)))
        return s.value

    def request_step(self, request: int) -> Tuple[int, int]:
        """(t_r, L_r) of one request (host copy; call sync() after graph replays)."""
        t, L = ctypes.c_int(), ctypes.c_int()
        check(lib().gr_beam_request_step(self.handle, request, ctypes.byref(t), ctypes.byref(L)))
        return t.value, L.value

    def kv_slot(self, layer: int, request: Optional[int] = None):
        """(k_new, v_new) views of the open BeamKV level: [rows, n_kv_heads, head_dim] for the
        whole batch (all requests at one step), or [W_r, ...] of one request at its own step."""
        k, v = ctypes.c_void_p(), ctypes.c_void_p()
        if request is None:
            check(lib().gr_beam_kv_slot(self.handle, layer, ctypes.byref(k), ctypes.byref(v)))
            t = max(self.request_step(r)[0] for r in range(self.n_requests)
                    if 1 <= self.request_step(r)[0] < self.request_step(r)[1])
            kk, vv = self.beam_k[layer, t - 1], self.beam_v[layer, t - 1]
        else:
            check(lib().gr_beam_kv_slot_request(self.handle, layer, request, ctypes.byref(k), ctypes.byref(v)))
            t = self.request_step(request)[0]
            r0, w = self.row_offsets[request], self.widths[request]
            kk, vv = self.beam_k[layer, t - 1, r0:r0 + w], self.beam_v[layer, t - 1, r0:r0 + w]
        assert kk.data_ptr() == k.value and vv.data_ptr() == v.value
        return kk, vv

    # -- hot path ------------------------------------------------------------
    def decode_attn(self, layer: int, q, out, stream=None) -> None:
        check(lib().gr_decode_attn(self.handle, layer, q.data_ptr(), out.data_ptr(), _stream_ptr(stream)))

    def constrained_topk(self, logits, ld: Optional[int] = None, logprobs_out=None, lse_out=None, lse_in=None,
                         stream=None) -> None:
        ld = logits.stride(0) if ld is None else ld
        check(lib().gr_constrained_topk(self.handle, logits.data_ptr(), ld, _ptr(logprobs_out), _ptr(lse_out),
                                        _ptr(lse_in), _stream_ptr(stream)))

    def advance(self, stream=None) -> None:
        check(lib().gr_beam_advance(self.handle, _stream_ptr(stream)))

    def rewind(self, step: int, stream=None) -> None:
        check(lib().gr_beam_rewind(self.handle, step, _stream_ptr(stream)))

    def admit(self, request: int, ctx_offset: int, ctx_len: int, beam_width: int, trie: "Trie", stream=None) -> None:
        """Slot `request` takes a new request (continuous batching); the slot's rows stay."""
        rq = GrRequest(ctx_offset, ctx_len, beam_width, trie.handle)
        check(lib().gr_beam_admit(self.handle, request, ctypes.byref(rq), _stream_ptr(stream)))
        self.tries[request] = trie  # keeps the catalogue's device buffer alive
        self.reqs[request] = rq

    def set_graph_mode(self, enable: bool) -> None:
        check(lib().gr_beam_set_graph_mode(self.handle, 1 if enable else 0))

    def sync(self, stream=None) -> None:
        check(lib().gr_beam_sync(self.handle, _stream_ptr(stream)))

    # -- reading back ----------------------------------------------------------
    def results(self, request: int, stream=None):
        """(codes int32 [n, L_r], item_ids int64 [n], scores float32 [n])."""
        W, L = self.widths[request], self.request_step(request)[1]
        codes = np.zeros((W, L), dtype=np.int32)
        items = np.zeros(W, dtype=np.int64)
        scores = np.zeros(W, dtype=np.float32)
        n = ctypes.c_int()
        check(lib().gr_beam_results(self.handle, request, codes.ctypes.data, items.ctypes.data,
                                    scores.ctypes.data, ctypes.byref(n), _stream_ptr(stream)))
        return codes[:n.value], items[:n.value], scores[:n.value]

    def path(self, request: int, level: int, stream=None):
        """BeamPath level: (parents, tokens, nodes, scores) of the beams it produced."""
        W = self.widths[request]
        par = np.zeros(W, dtype=np.int32)
        tok = np.zeros(W, dtype=np.int32)
        nod = np.zeros(W, dtype=np.int32)
        sc = np.zeros(W, dtype=np.float32)
        n = ctypes.c_int()
        check(lib().gr_beam_path(self.handle, request, level, par.ctypes.data, tok.ctypes.data, nod.ctypes.data,
                                 sc.ctypes.data, ctypes.byref(n), _stream_ptr(stream)))
        k = n.value
        return par[:k], tok[:k], nod[:k], sc[:k]

    def status(self, clear: bool = False, stream=None) -> int:
        """Device status as a gr_status code (does not raise)."""
        return lib().gr_beam_status(self.handle, 1 if clear else 0, _stream_ptr(stream))

    # -- measurement -----------------------------------------------------------------
    def set_timing(self, enable: bool) -> None:
        check(lib().gr_beam_set_timing(self.handle, 1 if enable else 0))

    def kernel_stats(self, kind: int, reset: bool = False) -> Tuple[int, float]:
        n = ctypes.c_int64()
        ms = ctypes.c_double()
        check(lib().gr_beam_kernel_stats(self.handle, kind, ctypes.byref(n), ctypes.byref(ms), 1 if reset else 0))
        return n.value, ms.value

    def set_wait_limit(self, ns: int) -> None:
        check(lib().gr_beam_set_wait_limit(self.handle, ns))

    def set_attn_kernel(self, mode: int) -> None:
        """0 automatic, 1 the single-CTA attention kernel, 2 the CTA-pair kernel (between steps)."""
        check(lib().gr_beam_set_attn_kernel(self.handle, mode, _stream_ptr()))

    def attn_kernel(self) -> str:
        v = ctypes.c_int(0)
        check(lib().gr_beam_attn_kernel(self.handle, ctypes.byref(v)))
        return "pair" if v.value else "single"


class Score:
    """Multi-item candidate scoring of one batch of requests (gr_score handle + its buffers)."""

    def __init__(self, n_layers: int, n_q_heads: int, n_kv_heads: int, head_dim: int, vocab: int,
                 label_ids: Sequence[int], ctx_k, ctx_v, requests: Sequence[Tuple[int, int, Sequence[int]]],
                 device="cuda"):
        """ctx_k / ctx_v: bf16 [n_layers, n_kv_heads, pool_tokens, head_dim];
        requests: (prefix ctx_offset, prefix ctx_len, tokens of each candidate) per request."""
        import torch
        self._labels = np.ascontiguousarray(label_ids, dtype=np.int32)
        self.cfg = GrScoreConfig(n_layers, n_q_heads, n_kv_heads, head_dim, vocab, ctx_k.shape[2],
                                 len(self._labels), self._labels.ctypes.data)
        self._segs = [np.ascontiguousarray(seg, dtype=np.int32) for (_, _, seg) in requests]
        n = len(requests)
        self.reqs = (GrScoreRequest * n)(*[GrScoreRequest(o, l, len(sg), sg.ctypes.data)
                                           for (o, l, _), sg in zip(requests, self._segs)])
        self.ctx_k, self.ctx_v = ctx_k, ctx_v
        self.n_requests = n
        self.n_labels = len(self._labels)
        ws = ctypes.c_size_t()
        check(lib().gr_score_workspace_bytes(ctypes.byref(self.cfg), self.reqs, n, ctypes.byref(ws)))
        self.rows = int(sum(int(sg.sum()) for sg in self._segs))
        self.n_candidates = int(sum(len(sg) for sg in self._segs))
        self.workspace = torch.empty(ws.value, dtype=torch.uint8, device=device)
        shape = (n_layers, self.rows, n_kv_heads, head_dim)
        self.seg_k = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        self.seg_v = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        bufs = GrScoreBuffers(ctx_k.data_ptr(), ctx_v.data_ptr(), self.seg_k.data_ptr(), self.seg_v.data_ptr(),
                              self.workspace.data_ptr(), self.workspace.numel())
        h = ctypes.c_void_p()
        check(lib().gr_score_create(ctypes.byref(self.cfg), self.reqs, n, ctypes.byref(bufs), _stream_ptr(),
                                    ctypes.byref(h)))
        self.handle = h
        rows = ctypes.c_int()
        ro, co = (ctypes.c_int * (n + 1))(), (ctypes.c_int * (n + 1))()
        check(lib().gr_score_rows(self.handle, ctypes.byref(rows), ro, co))
        assert rows.value == self.rows
        self.row_offsets, self.cand_offsets = list(ro), list(co)

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.gr_score_destroy(self.handle)
            self.handle = None

    def attn(self, layer: int, q, out, stream=None) -> None:
        check(lib().gr_score_attn(self.handle, layer, q.data_ptr(), out.data_ptr(), _stream_ptr(stream)))

    def labels(self, logits, ld: Optional[int] = None, ranking: bool = True, stream=None):
        """(log-probs float32 [n_candidates, n_labels], ranking int32 [n_candidates] or None)."""
        import torch
        ld = logits.stride(0) if ld is None else ld
        lp = torch.empty((self.n_candidates, self.n_labels), dtype=torch.float32, device=logits.device)
        rk = torch.empty(self.n_candidates, dtype=torch.int32, device=logits.device) if ranking else None
        check(lib().gr_score_labels(self.handle, logits.data_ptr(), ld, lp.data_ptr(), _ptr(rk),
                                    _stream_ptr(stream)))
        return lp, rk

    def status(self, clear: bool = False, stream=None) -> int:
        return lib().gr_score_status(self.handle, 1 if clear else 0, _stream_ptr(stream))
