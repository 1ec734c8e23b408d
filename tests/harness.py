"""Lock-step harness: the CUDA path (through the C ABI) and the CPU oracle are
fed the same seeded inputs, step by step, and their outputs compared.

Inputs come only from ``beam_decode_gb300.workload``; expected values come
only from ``oracle``.  Nothing computed by the CUDA path is fed to the oracle:
the oracle keeps its own beams, ancestry and BeamKV copy.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np

from beam_decode_gb300 import workload as wl
from oracle import OracleBeam, Trie as OTrie, beam_attention

ATOL = 1e-2   # attention: |gpu - ref| <= ATOL + RTOL*|ref| (bf16 K/V, fp32 accumulate)
RTOL = 1e-2
LP_TOL = 1e-4  # log-probabilities and log-sum-exp


@dataclasses.dataclass
class Spec:
    n_layers: int = 1
    n_q_heads: int = 2
    n_kv_heads: int = 1
    head_dim: int = 64
    vocab: int = 1024
    n_levels: int = 2
    codes_per_level: int = 16
    code_base: int = 512
    ctx_lens: List[int] = dataclasses.field(default_factory=lambda: [64])
    widths: List[int] = dataclasses.field(default_factory=lambda: [4])
    n_items: List[int] = dataclasses.field(default_factory=lambda: [50])
    trie_dist: str = "uniform"
    shared_trie: bool = True
    logit_std: float = 2.0
    ld_pad: int = 0
    seed: int = 0
    pool_gap: int = 7      # unused tokens between requests in the ContextKV pool
    q_std: float = 1.0     # queries ~ N(0, q_std^2): larger values make the running row max grow
                           # across key tiles, which exercises the online-softmax rescale

    @staticmethod
    def from_workload(w: wl.Workload, **over) -> "Spec":
        s = Spec(n_layers=w.n_layers, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
                 vocab=w.vocab, n_levels=w.n_levels, codes_per_level=w.codes_per_level, code_base=w.code_base,
                 ctx_lens=list(w.ctx_lens), widths=list(w.beam_widths), n_items=list(w.n_items),
                 trie_dist=w.trie_dist, shared_trie=w.shared_trie, logit_std=w.logit_std, seed=w.seed)
        for k, v in over.items():
            setattr(s, k, v)
        return s


def make_items(spec: Spec) -> List[np.ndarray]:
    if spec.shared_trie:
        it = wl.draw_items(spec.n_items[0], spec.n_levels, spec.codes_per_level, spec.trie_dist, spec.seed)
        return [it] * len(spec.ctx_lens)
    return [wl.draw_items(n, spec.n_levels, spec.codes_per_level, spec.trie_dist, spec.seed, stream=(r,))
            for r, n in enumerate(spec.n_items)]


class LockStep:
    """GPU batch + oracle beams over the same host-generated inputs."""

    def __init__(self, spec: Spec, device="cuda", key_mode="f32", logits_fn=None):
        import torch
        from beam_decode_gb300 import binding as B
        self.spec, self.device, self.torch, self.B = spec, device, torch, B
        self.logits_fn = logits_fn
        s = spec
        R = len(s.ctx_lens)
        self.items = make_items(s)
        # catalogues (GPU tries share the array when the catalogue is shared)
        cache: Dict[int, tuple] = {}
        self.gtries, self.otries = [], []
        for it in self.items:
            key = id(it)
            if key not in cache:
                cache[key] = (B.Trie(it, codes_per_level=s.codes_per_level, device=device),
                              OTrie(it, codes_per_level=s.codes_per_level))
            self.gtries.append(cache[key][0])
            self.otries.append(cache[key][1])
        # ContextKV pool with gaps between requests
        self.ctx_off = []
        off = 3
        for T in s.ctx_lens:
            self.ctx_off.append(off)
            off += T + s.pool_gap
        pool = off
        shp = (s.n_layers, s.n_kv_heads, pool, s.head_dim)
        self.ctx_k = wl.round_to_bf16(wl.host_normal(shp, s.seed, wl.TAG_CTX_K))
        self.ctx_v = wl.round_to_bf16(wl.host_normal(shp, s.seed, wl.TAG_CTX_V))
        tk = torch.from_numpy(self.ctx_k).to(torch.bfloat16).to(device)
        tv = torch.from_numpy(self.ctx_v).to(torch.bfloat16).to(device)
        reqs = [(self.ctx_off[r], s.ctx_lens[r], s.widths[r], self.gtries[r]) for r in range(R)]
        self.beam = B.Beam(s.n_layers, s.n_q_heads, s.n_kv_heads, s.head_dim, s.vocab, s.code_base, s.n_levels,
                           s.codes_per_level, tk, tv, reqs, device=device)
        self.row_off = self.beam.row_offsets
        self.obeams = [OracleBeam(self.otries[r], s.widths[r], s.n_levels, s.codes_per_level, s.code_base,
                                  key_mode=key_mode) for r in range(R)]
        # oracle copy of BeamKV: [layer][level] -> [rows, Hkv, D]
        self.obk = [[None] * max(s.n_levels - 1, 1) for _ in range(s.n_layers)]
        self.obv = [[None] * max(s.n_levels - 1, 1) for _ in range(s.n_layers)]
        self.t = 0

    # -- inputs -----------------------------------------------------------------
    def logits(self, t: int) -> np.ndarray:
        s = self.spec
        ld = s.vocab + s.ld_pad
        x = wl.host_normal((self.beam.rows, ld), s.seed, wl.TAG_LOGITS, sub=(t,), std=s.logit_std)
        if self.logits_fn is not None:
            x = np.ascontiguousarray(self.logits_fn(self, t, x), dtype=np.float32)
        return x

    def write_beam_kv(self, t: int, layer: int):
        s = self.spec
        shp = (self.beam.rows, s.n_kv_heads, s.head_dim)
        k = wl.round_to_bf16(wl.host_normal(shp, s.seed, wl.TAG_BEAM_K, sub=(t, layer)))
        v = wl.round_to_bf16(wl.host_normal(shp, s.seed, wl.TAG_BEAM_V, sub=(t, layer)))
        gk, gv = self.beam.kv_slot(layer)
        gk.copy_(self.torch.from_numpy(k).to(self.torch.bfloat16))
        gv.copy_(self.torch.from_numpy(v).to(self.torch.bfloat16))
        self.obk[layer][t - 1], self.obv[layer][t - 1] = k, v

    def queries(self, t: int, layer: int) -> np.ndarray:
        s = self.spec
        return wl.round_to_bf16(s.q_std * wl.host_normal((self.beam.rows, s.n_q_heads, s.head_dim), s.seed,
                                                         wl.TAG_Q, sub=(t, layer)))

    # -- one attention layer -------------------------------------------------------
    def attention(self, layer: int, requests=None, beams_per_request=None) -> Dict:
        """Run gr_decode_attn for `layer` at the current step; compare with the oracle.
        Returns the max violation ratio (<= 1 passes) and sizes compared."""
        torch = self.torch
        t = self.t
        self.write_beam_kv(t, layer)
        q = self.queries(t, layer)
        gq = torch.from_numpy(q).to(torch.bfloat16).to(self.device)
        gout = torch.full_like(gq, float("nan"))
        self.beam.decode_attn(layer, gq, gout)
        return self.compare_attention(layer, q, gout.float().cpu().numpy(), requests, beams_per_request)

    def compare_attention(self, layer: int, q: np.ndarray, out: np.ndarray, requests=None,
                          beams_per_request=None) -> Dict:
        """Element-wise check of one layer's attention output `out` [rows, Hq, D] against the
        oracle's float64 attention at the current step (the oracle's own beams and ancestry)."""
        s, t = self.spec, self.t
        worst, n = 0.0, 0
        reqs = range(len(s.ctx_lens)) if requests is None else requests
        for r in reqs:
            ob = self.obeams[r]
            n_live = ob.n_live()
            r0, T, o0 = self.row_off[r], s.ctx_lens[r], self.ctx_off[r]
            beams = list(range(n_live)) if beams_per_request is None else \
                [b for b in beams_per_request if b < n_live]
            anc = ob.ancestry()
            ck = self.ctx_k[layer, :, o0:o0 + T]
            cv = self.ctx_v[layer, :, o0:o0 + T]
            bk = [self.obk[layer][j][r0:r0 + s.widths[r]] for j in range(t)]
            bv = [self.obv[layer][j][r0:r0 + s.widths[r]] for j in range(t)]
            ref = beam_attention(q[r0:r0 + s.widths[r]], ck, cv, bk, bv, anc, beams=beams)
            got = out[r0 + np.array(beams)]
            viol = np.abs(got - ref) / (ATOL + RTOL * np.abs(ref))
            worst = max(worst, float(np.nanmax(viol)) if viol.size else 0.0)
            if np.isnan(got).any():
                worst = float("inf")
            n += viol.size
            # rows of dead beams are written as zeros
            dead = out[r0 + n_live:r0 + s.widths[r]]
            if dead.size and not np.all(dead == 0):
                worst = float("inf")
        return {"worst": worst, "n": n}

    # -- one top-K step ----------------------------------------------------------------
    def topk_step(self, lse_mode: bool = True) -> Dict:
        """gr_constrained_topk + gr_beam_advance vs the oracle step.
        lse_mode: pass the oracle's float32 LSE to the GPU (bit-exact contract)."""
        torch = self.torch
        s = self.spec
        x = self.logits(self.t)
        ld = x.shape[1]
        gx = torch.from_numpy(x).to(self.device)
        lp_out = torch.full((self.beam.rows, s.codes_per_level), float("nan"), device=self.device)
        lse_out = torch.full((self.beam.rows,), float("nan"), device=self.device)
        oinfo, lse32 = self.oracle_topk(x)   # oracle first: its float32 LSE is the GPU's lse_in
        lse_in = torch.from_numpy(np.nan_to_num(lse32, nan=0.0)).to(self.device) if lse_mode else None
        self.beam.constrained_topk(gx, ld=ld, logprobs_out=lp_out, lse_out=lse_out, lse_in=lse_in)
        self.beam.advance()
        return self.compare_topk(oinfo, lse_mode, lse_out.cpu().numpy(), lp_out.cpu().numpy())

    def oracle_lse(self, x: np.ndarray) -> np.ndarray:
        """The oracle's float64 log-sum-exp of every live row, rounded to float32 (NaN for
        rows that are not live); the oracle's state does not change."""
        from oracle import log_softmax_row
        s = self.spec
        lse32 = np.full(self.beam.rows, np.nan, dtype=np.float32)
        for r in range(len(s.ctx_lens)):
            r0, n = self.row_off[r], self.obeams[r].n_live()
            lse32[r0:r0 + n] = [log_softmax_row(rw)[1] for rw in x[r0:r0 + n, :s.vocab]]
        return lse32

    def oracle_topk(self, x: np.ndarray):
        """The oracle's step on the logit rows x (all requests, under the float32 key contract
        with its own LSE rounded to float32).  Returns (per-request step info, float32 LSE per
        row, NaN for rows that are not live)."""
        from oracle import log_softmax_row
        s = self.spec
        oinfo = []
        lse32 = np.full(self.beam.rows, np.nan, dtype=np.float32)
        for r in range(len(s.ctx_lens)):
            ob = self.obeams[r]
            n = ob.n_live()
            r0 = self.row_off[r]
            rows = x[r0:r0 + n, :s.vocab]
            lses = [log_softmax_row(rw)[1] for rw in rows]
            lse32[r0:r0 + n] = np.array(lses, dtype=np.float32)
            info = ob.step(rows, lse_in=lse32[r0:r0 + n])
            info["lse64"] = lses
            oinfo.append(info)
        return oinfo, lse32

    def compare_topk(self, oinfo, lse_mode: bool, lse_g=None, lp_g=None) -> Dict:
        """The GPU's BeamPath level t (read through gr_beam_path) against the oracle's step t:
        parents and tokens bit for bit, scores bit for bit under lse_in; the GPU's own LSE and
        log-probabilities (when given) within 1e-4 of float64."""
        s, t = self.spec, self.t
        res = {"lse_err": 0.0, "lp_err": 0.0, "mismatch": [], "n_sel": []}
        for r in range(len(s.ctx_lens)):
            info = oinfo[r]
            r0 = self.row_off[r]
            n = len(info["lse64"])
            if not lse_mode and lse_g is not None:
                res["lse_err"] = max(res["lse_err"], float(np.max(np.abs(lse_g[r0:r0 + n] - np.array(info["lse64"])))))
                ref_lp = info["logprobs"]
                fin = np.zeros(ref_lp.shape, dtype=bool)  # valid (beam, code) pairs per the oracle's trie
                for (_, _, b, c) in info["candidates"]:
                    fin[b, c] = True
                got = lp_g[r0:r0 + n]
                if not np.array_equal(np.isfinite(got), fin):
                    res["lp_err"] = float("inf")
                else:
                    res["lp_err"] = max(res["lp_err"], float(np.max(np.abs(got[fin] - ref_lp[fin]), initial=0.0)))
            par, tok, nod, sc = self.beam.path(r, t)
            ob = self.obeams[r]
            exp_par = np.array(ob.parents[t], dtype=np.int32)
            exp_tok = np.array([s.code_base + t * s.codes_per_level + c for c in ob.codes[t]], dtype=np.int32)
            exp_sc = np.array([float(v) for v in ob.scores[t]], dtype=np.float32)
            res["n_sel"].append(len(par))
            ok = (len(par) == len(exp_par) and np.array_equal(par, exp_par) and np.array_equal(tok, exp_tok))
            if lse_mode:
                ok = ok and np.array_equal(sc.view(np.uint32), exp_sc.view(np.uint32))
            if not ok:
                res["mismatch"].append(r)
        self.t += 1
        return res

    def gpu_results(self, r: int):
        return self.beam.results(r)


class GraphStep:
    """A whole decode step -- gr_decode_attn for every layer, gr_constrained_topk (with the
    oracle's float32 LSE through lse_in) and gr_beam_advance -- captured once as a CUDA graph
    in graph mode and replayed for the later steps, each replay checked against the oracle.

    Before a replay the host writes the step's inputs into the captured buffers: the BeamKV
    level of the codes chosen at the previous step (straight into the pool, as a model
    would), the queries of every layer, the logits and the LSE.  The oracle sees the same
    host arrays and keeps its own beams, ancestry and BeamKV copy."""

    def __init__(self, ls: LockStep):
        torch = ls.torch
        assert ls.t == 1, "capture after level 0 (the first step with attention)"
        self.ls = ls
        s, beam = ls.spec, ls.beam
        qs = (beam.rows, s.n_q_heads, s.head_dim)
        self.q = [torch.zeros(qs, dtype=torch.bfloat16, device=ls.device) for _ in range(s.n_layers)]
        self.out = [torch.zeros(qs, dtype=torch.bfloat16, device=ls.device) for _ in range(s.n_layers)]
        self.x = torch.zeros((beam.rows, s.vocab + s.ld_pad), device=ls.device)
        self.lse = torch.zeros((beam.rows,), device=ls.device)
        # one eager step first (one-time kernel set-up happens outside the capture), rewound
        self._enqueue()
        beam.rewind(1)
        torch.cuda.synchronize()
        beam.set_graph_mode(True)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._enqueue()

    def _enqueue(self):
        beam = self.ls.beam
        for layer in range(self.ls.spec.n_layers):
            beam.decode_attn(layer, self.q[layer], self.out[layer])
        beam.constrained_topk(self.x, ld=self.x.shape[1], lse_in=self.lse)
        beam.advance()

    def replay(self) -> Dict:
        """Replay the graph for the current step t and compare it with the oracle: every
        layer's attention element-wise, then the selection bit for bit."""
        ls, torch = self.ls, self.ls.torch
        s, t, beam = ls.spec, ls.t, ls.beam
        shp = (beam.rows, s.n_kv_heads, s.head_dim)
        qs = []
        for layer in range(s.n_layers):
            k = wl.round_to_bf16(wl.host_normal(shp, s.seed, wl.TAG_BEAM_K, sub=(t, layer)))
            v = wl.round_to_bf16(wl.host_normal(shp, s.seed, wl.TAG_BEAM_V, sub=(t, layer)))
            beam.beam_k[layer, t - 1].copy_(torch.from_numpy(k).to(torch.bfloat16))
            beam.beam_v[layer, t - 1].copy_(torch.from_numpy(v).to(torch.bfloat16))
            ls.obk[layer][t - 1], ls.obv[layer][t - 1] = k, v
            q = ls.queries(t, layer)
            self.q[layer].copy_(torch.from_numpy(q).to(torch.bfloat16))
            self.out[layer].fill_(float("nan"))
            qs.append(q)
        x = ls.logits(t)
        self.x.copy_(torch.from_numpy(x))
        self.lse.copy_(torch.from_numpy(np.nan_to_num(ls.oracle_lse(x), nan=0.0)))
        torch.cuda.synchronize()
        self.graph.replay()
        torch.cuda.synchronize()
        # attention against the oracle's state before its top-K step of level t
        worst = 0.0
        for layer in range(s.n_layers):
            a = ls.compare_attention(layer, qs[layer], self.out[layer].float().cpu().numpy())
            worst = max(worst, a["worst"])
        oinfo, _ = ls.oracle_topk(x)
        beam.sync()   # the host's copy of the device step state, for gr_beam_path
        res = ls.compare_topk(oinfo, lse_mode=True)
        res["worst"] = worst
        return res


@dataclasses.dataclass
class Occupant:
    """One request that holds a batch slot for a while (continuous batching)."""
    ctx_len: int
    width: int
    n_levels: int
    n_items: int
    key: int                 # seeds its catalogue and BeamKV streams


class MixedDriver:
    """Requests at their own steps: each slot holds one occupant (context, catalogue,
    length L_r, width); the batch advances with one call sequence per batch step while
    the occupants are at different levels, and a finished slot takes the next occupant
    (gr_beam_admit).  The GPU batch and one oracle beam per occupant see the same
    host-generated inputs; every comparison is against the oracle."""

    def __init__(self, occupants: List[Occupant], slot_widths: List[int], n_layers=2, n_q_heads=4, n_kv_heads=2,
                 head_dim=64, vocab=2048, codes_per_level=32, n_levels_max=3, seed=50, device="cuda"):
        import torch
        from beam_decode_gb300 import binding as B
        self.torch, self.B, self.device = torch, B, device
        self.NL, self.Hq, self.Hkv, self.D = n_layers, n_q_heads, n_kv_heads, head_dim
        self.V, self.C, self.Lmax, self.seed = vocab, codes_per_level, n_levels_max, seed
        self.code_base = vocab - n_levels_max * codes_per_level
        self.occ = list(occupants)
        # ContextKV pool: one region per occupant, gaps between them
        self.ctx_off, off = [], 5
        for o in self.occ:
            self.ctx_off.append(off)
            off += o.ctx_len + 9
        shp = (n_layers, n_kv_heads, off, head_dim)
        self.ctx_k = wl.round_to_bf16(wl.host_normal(shp, seed, wl.TAG_CTX_K))
        self.ctx_v = wl.round_to_bf16(wl.host_normal(shp, seed, wl.TAG_CTX_V))
        tk = torch.from_numpy(self.ctx_k).to(torch.bfloat16).to(device)
        tv = torch.from_numpy(self.ctx_v).to(torch.bfloat16).to(device)
        self.items = [wl.draw_items(o.n_items, o.n_levels, codes_per_level, "uniform", seed, stream=(o.key,))
                      for o in self.occ]
        self.gtries = [B.Trie(it, codes_per_level=codes_per_level, device=device) for it in self.items]
        self.otries = [OTrie(it, codes_per_level=codes_per_level) for it in self.items]
        self.slot_w = list(slot_widths)
        self.slot_occ = list(range(len(slot_widths)))   # occupant held by each slot
        reqs = [(self.ctx_off[i], self.occ[i].ctx_len, self.occ[i].width, self.gtries[i])
                for i in range(len(slot_widths))]
        # slots are created at their full widths (rows); the first occupants use them all
        assert all(self.occ[i].width == slot_widths[i] for i in range(len(slot_widths)))
        self.beam = B.Beam(n_layers, n_q_heads, n_kv_heads, head_dim, vocab, self.code_base, n_levels_max,
                           codes_per_level, tk, tv, reqs, device=device)
        self.row_off = self.beam.row_offsets
        self.rows = self.beam.rows
        self.obeam = {i: self._oracle(i) for i in range(len(slot_widths))}
        self.obk: Dict[int, Dict] = {}   # occupant -> {(layer, level): (k, v)}
        self.k = 0                       # batch steps so far
        self.finished: List[int] = []

    def _oracle(self, o):
        return OracleBeam(self.otries[o], self.occ[o].width, self.occ[o].n_levels, self.C, self.code_base,
                          key_mode="f32")

    def t(self, slot):
        return self.obeam[self.slot_occ[slot]].t

    def L(self, slot):
        return self.occ[self.slot_occ[slot]].n_levels

    def admit(self, slot, o):
        oc = self.occ[o]
        self.beam.admit(slot, self.ctx_off[o], oc.ctx_len, oc.width, self.gtries[o])
        self.slot_occ[slot] = o
        self.obeam[o] = self._oracle(o)

    def step(self, compare=True) -> Dict:
        torch = self.torch
        S = len(self.slot_w)
        attending = [s for s in range(S) if 1 <= self.t(s) < self.L(s)]
        decoding = [s for s in range(S) if self.t(s) < self.L(s)]
        worst = 0.0
        if attending:
            for layer in range(self.NL):
                for s in attending:
                    o, t = self.slot_occ[s], self.t(s)
                    shp = (self.slot_w[s], self.Hkv, self.D)
                    kk = wl.round_to_bf16(wl.host_normal(shp, self.seed, wl.TAG_BEAM_K, sub=(1000 + o, t - 1, layer)))
                    vv = wl.round_to_bf16(wl.host_normal(shp, self.seed, wl.TAG_BEAM_V, sub=(1000 + o, t - 1, layer)))
                    gk, gv = self.beam.kv_slot(layer, request=s)
                    gk.copy_(torch.from_numpy(kk).to(torch.bfloat16))
                    gv.copy_(torch.from_numpy(vv).to(torch.bfloat16))
                    self.obk.setdefault(o, {})[(layer, t - 1)] = (kk, vv)
                q = wl.round_to_bf16(wl.host_normal((self.rows, self.Hq, self.D), self.seed, wl.TAG_Q,
                                                    sub=(self.k, layer)))
                gq = torch.from_numpy(q).to(torch.bfloat16).to(self.device)
                gout = torch.full_like(gq, float("nan"))
                self.beam.decode_attn(layer, gq, gout)
                if not compare:
                    continue
                out = gout.float().cpu().numpy()
                for s in range(S):
                    r0, W = self.row_off[s], self.slot_w[s]
                    if s not in attending:  # rows of requests that do not attend are not written
                        if not np.all(np.isnan(out[r0:r0 + W])):
                            worst = float("inf")
                        continue
                    o, t = self.slot_occ[s], self.t(s)
                    ob = self.obeam[o]
                    n_live = ob.n_live()
                    T, c0 = self.occ[o].ctx_len, self.ctx_off[o]
                    bk = [self.obk[o][(layer, j)][0] for j in range(t)]
                    bv = [self.obk[o][(layer, j)][1] for j in range(t)]
                    ref = beam_attention(q[r0:r0 + W], self.ctx_k[layer, :, c0:c0 + T], self.ctx_v[layer, :, c0:c0 + T],
                                         bk, bv, ob.ancestry(), beams=list(range(n_live)))
                    got = out[r0:r0 + n_live]
                    viol = np.abs(got - ref) / (ATOL + RTOL * np.abs(ref))
                    worst = max(worst, float(np.max(viol)) if viol.size else 0.0)
                    # dead beams of the request are zeros; slot rows past its width are not written
                    w_occ = self.occ[o].width
                    if np.isnan(got).any() or not np.all(out[r0 + n_live:r0 + w_occ] == 0):
                        worst = float("inf")
        # top-K of every decoding request at its own level
        from oracle import log_softmax_row
        x = wl.host_normal((self.rows, self.V), self.seed, wl.TAG_LOGITS, sub=(self.k,), std=2.0)
        lse32 = np.zeros(self.rows, dtype=np.float32)
        for s in decoding:
            o, r0 = self.slot_occ[s], self.row_off[s]
            n = self.obeam[o].n_live()
            rows = x[r0:r0 + n]
            lse32[r0:r0 + n] = np.array([log_softmax_row(rw)[1] for rw in rows], dtype=np.float32)
            self.obeam[o].step(rows, lse_in=lse32[r0:r0 + n])
        self.beam.constrained_topk(torch.from_numpy(x).to(self.device),
                                   lse_in=torch.from_numpy(lse32).to(self.device))
        self.beam.advance()
        mismatch = []
        for s in decoding:
            o = self.slot_occ[s]
            ob = self.obeam[o]
            t = ob.t - 1
            par, tok, _, sc = self.beam.path(s, t)
            exp_tok = np.array([self.code_base + t * self.C + c for c in ob.codes[t]], dtype=np.int32)
            exp_sc = np.array([float(v) for v in ob.scores[t]], dtype=np.float32)
            if not (np.array_equal(par, np.array(ob.parents[t], dtype=np.int32)) and np.array_equal(tok, exp_tok)
                    and np.array_equal(sc.view(np.uint32), exp_sc.view(np.uint32))):
                mismatch.append((s, o, t))
            assert self.beam.request_step(s) == (ob.t, self.occ[o].n_levels)
            if ob.t == self.occ[o].n_levels:
                self.check_results(s)
                self.finished.append(o)
        self.k += 1
        return {"worst": worst, "mismatch": mismatch, "attending": attending, "decoding": decoding}

    def check_results(self, s):
        o = self.slot_occ[s]
        codes, items, scores = self.beam.results(s)
        exp = self.obeam[o].results()
        assert len(codes) == len(exp), (s, o)
        for i, (tup, iid, sc) in enumerate(exp):
            assert tuple(int(c) for c in codes[i]) == tup
            assert int(items[i]) == iid
            assert np.float32(scores[i]).view(np.uint32) == np.float32(sc).view(np.uint32)
