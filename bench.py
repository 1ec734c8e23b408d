"""Benchmark of one wide-beam semantic-ID decode step on GB300.

A step is one full-width decode step t = 1 over the whole batch: gr_decode_attn
for every layer (shared-context tensor-core attention + BeamKV combine), then
gr_constrained_topk (full-vocabulary log-softmax + item-constrained top-K) and
gr_beam_advance.  Each timed step first rewinds the handle to step 1 (host
state only), so every iteration decodes the same full-width step.

Workload (default): 8 requests x context 5000 x beam 256, Qwen3-1.7B attention
geometry (28 layers, 16 q / 8 KV heads, head_dim 128), vocabulary 151,936,
3 code levels x 256 codes, 1M uniform items -- the page's long-context shape
(zhiding.cn recsys-examples article, section "语义ID生成式推荐专用推理框架").
All tensors are synthetic (seeded normal bf16 Q/K/V, fp32 logits with std 2);
no model weights.  The ContextKV alone (4.6 GB) is larger than L2, so no
flush is needed between steps.

Prints one JSON line.  `--impl reference` times the CPU oracle instead on a
bounded sample of the same workload.
"""
from __future__ import annotations

import os

# the CPU oracle baseline is reported as single-threaded: pin BLAS before numpy loads
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from beam_decode_gb300 import workload as wl  # noqa: E402

METRIC = "GR beam decode-steps/s (ctx 5000, beam 256); attn TC % and HBM GB/s vs peak"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sust": d["bf16_tflops_sustained"],
                "src": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sust": 1700.0, "src": "fallback"}


# DRAM bytes (read + write) per launch of the attention kernel from one ncu capture, keyed
# by the sha256 of the kernel's sources it was taken on (the kernel file and the shared device
# code): (bytes per launch per request, note).  Sources without an entry report traffic null.
_ATTN_TRAFFIC = {
    "fcc55112ccee2c77": ((222.84e6 + 4.03e6) / 8,
                         "ncu capture of one launch at the long shapes (8 requests, one layer), per request"),
}


def _attn_traffic(w):
    import hashlib
    h = hashlib.sha256()
    for f in ("k_attn.cu", "attn_dev.cuh"):
        h.update(open(os.path.join(ROOT, "beam_decode_gb300", "csrc", f), "rb").read())
    key = h.hexdigest()[:16]
    if key not in _ATTN_TRAFFIC or w.name != "long" or len(set(w.ctx_lens)) != 1:
        return None
    per_req, _ = _ATTN_TRAFFIC[key]
    return per_req * w.n_requests


# ---------------------------------------------------------------------------
# device batch
# ---------------------------------------------------------------------------
class DeviceBatch:
    """Synthetic batch resident in HBM, decoded through the C ABI."""

    def __init__(self, w: wl.Workload, device="cuda"):
        import torch
        from beam_decode_gb300 import binding as B
        self.w, self.device, self.torch = w, device, torch
        R = w.n_requests
        items = wl.workload_items(w)
        tries = {}
        self.tries = []
        for it in items:
            if id(it) not in tries:
                tries[id(it)] = B.Trie(it, codes_per_level=w.codes_per_level, device=device)
            self.tries.append(tries[id(it)])
        self.items = items
        self.ctx_off = np.concatenate([[0], np.cumsum(w.ctx_lens)[:-1]]).astype(np.int64)
        pool = int(sum(w.ctx_lens))
        shp = (w.n_layers, w.n_kv_heads, pool, w.head_dim)
        self.ctx_k = torch.empty(shp, dtype=torch.bfloat16, device=device)
        self.ctx_v = torch.empty(shp, dtype=torch.bfloat16, device=device)
        for l in range(w.n_layers):  # layer by layer keeps the fp32 temporaries small
            self.ctx_k[l] = wl.device_normal(shp[1:], w.seed, wl.TAG_CTX_K, device, torch.bfloat16, sub=l)
            self.ctx_v[l] = wl.device_normal(shp[1:], w.seed, wl.TAG_CTX_V, device, torch.bfloat16, sub=l)
        reqs = [(int(self.ctx_off[r]), w.ctx_lens[r], w.beam_widths[r], self.tries[r]) for r in range(R)]
        self.beam = B.Beam(w.n_layers, w.n_q_heads, w.n_kv_heads, w.head_dim, w.vocab, w.code_base, w.n_levels,
                           w.codes_per_level, self.ctx_k, self.ctx_v, reqs, device=device)
        rows = self.beam.rows
        self.rows = rows
        qs = (rows, w.n_q_heads, w.head_dim)
        self.q = [wl.device_normal(qs, w.seed, wl.TAG_Q, device, torch.bfloat16, sub=l) for l in range(w.n_layers)]
        self.out = [torch.empty(qs, dtype=torch.bfloat16, device=device) for _ in range(w.n_layers)]
        self.logits = [wl.device_normal((rows, w.vocab), w.seed, wl.TAG_LOGITS, device, std=w.logit_std, sub=t)
                       for t in range(2)]
        kvs = (rows, w.n_kv_heads, w.head_dim)
        self.new_k = [wl.device_normal(kvs, w.seed, wl.TAG_BEAM_K, device, torch.bfloat16, sub=l)
                      for l in range(w.n_layers)]
        self.new_v = [wl.device_normal(kvs, w.seed, wl.TAG_BEAM_V, device, torch.bfloat16, sub=l)
                      for l in range(w.n_layers)]
        # step 0: level-0 codes from the prefill logits, then feed level-0 K/V
        self.beam.constrained_topk(self.logits[0])
        self.beam.advance()
        for l in range(w.n_layers):
            k, v = self.beam.kv_slot(l)
            k.copy_(self.new_k[l])
            v.copy_(self.new_v[l])
        torch.cuda.synchronize()

    def step(self):
        """One full-width decode step t = 1 (device-resident inputs)."""
        b = self.beam
        b.rewind(1)
        for l in range(self.w.n_layers):
            b.decode_attn(l, self.q[l], self.out[l])
        b.constrained_topk(self.logits[1])
        b.advance()

    def finish(self):
        """Decode the batch on to its last levels from the state a step leaves (the level just
        selected has no BeamKV yet): each further step writes that level's BeamKV, then runs
        attention, top-K and advance, until every request has reached its last level."""
        b, w = self.beam, self.w

        def unfinished():
            return any(t < L for t, L in (b.request_step(r) for r in range(w.n_requests)))

        while unfinished():
            for l in range(w.n_layers):
                k, v = b.kv_slot(l)
                k.copy_(self.new_k[l])
                v.copy_(self.new_v[l])
            for l in range(w.n_layers):
                b.decode_attn(l, self.q[l], self.out[l])
            b.constrained_topk(self.logits[1])
            b.advance()

    def capture(self):
        """Record the step once as a CUDA graph (graph mode: every decision inside comes from
        the device-resident step state); returns the library launches one replay makes."""
        torch = self.torch
        from beam_decode_gb300 import binding as B
        self.step()  # outside the capture: one-time kernel attribute setup
        torch.cuda.synchronize()
        for k in range(B.KERNEL_KINDS):
            self.beam.kernel_stats(k, reset=True)
        self.beam.set_graph_mode(True)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.step()
        return sum(self.beam.kernel_stats(k, reset=True)[0] for k in range(B.KERNEL_KINDS))

    def release(self):
        """Leave graph mode and reload the host's step state."""
        self.graph = None
        self.beam.set_graph_mode(False)
        self.beam.sync()

    # algorithmic work of one step
    def attn_flops(self) -> float:
        w = self.w
        return float(sum(4.0 * w.n_layers * w.n_q_heads * W * T * w.head_dim
                         for W, T in zip(w.beam_widths, w.ctx_lens)))

    def ctx_bytes_per_layer(self) -> float:
        w = self.w
        return float(sum(T for T in w.ctx_lens) * w.n_kv_heads * w.head_dim * 2 * 2)


# ---------------------------------------------------------------------------
# clocks sampling
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_step_seconds(w: wl.Workload, budget_s: float = 12.0):
    """Seconds per decode step of the CPU oracle, from a bounded sample:
    naive per-beam attention for a sample of (beam, layer) pairs of request 0
    and the constrained top-K of request 0 (full rows), scaled to the step."""
    from oracle import OracleBeam, Trie, beam_attention
    rng_seed = w.seed
    T, W, D = w.ctx_lens[0], w.beam_widths[0], w.head_dim
    ck = wl.round_to_bf16(wl.host_normal((w.n_kv_heads, T, D), rng_seed, wl.TAG_CTX_K)).astype(np.float64)
    cv = wl.round_to_bf16(wl.host_normal((w.n_kv_heads, T, D), rng_seed, wl.TAG_CTX_V)).astype(np.float64)
    q = wl.round_to_bf16(wl.host_normal((W, w.n_q_heads, D), rng_seed, wl.TAG_Q)).astype(np.float64)
    bk = [wl.round_to_bf16(wl.host_normal((W, w.n_kv_heads, D), rng_seed, wl.TAG_BEAM_K)).astype(np.float64)]
    bv = [wl.round_to_bf16(wl.host_normal((W, w.n_kv_heads, D), rng_seed, wl.TAG_BEAM_V)).astype(np.float64)]
    anc = [[b] for b in range(W)]
    t0 = time.perf_counter()
    n_att = 0
    while time.perf_counter() - t0 < budget_s * 0.5 and n_att < W:
        beam_attention(q, ck, cv, bk, bv, anc, beams=[n_att])
        n_att += 1
    att_s = (time.perf_counter() - t0) / n_att  # one (beam, layer): all q heads
    # top-K of one request at step 1 (full width) over the workload's whole catalogue
    items = wl.draw_items(w.n_items[0], w.n_levels, w.codes_per_level, w.trie_dist, w.seed)
    trie = Trie(items, codes_per_level=w.codes_per_level)
    ob = OracleBeam(trie, W, w.n_levels, w.codes_per_level, w.code_base)
    x0 = wl.host_normal((1, w.vocab), rng_seed, wl.TAG_LOGITS, std=w.logit_std)
    ob.step(x0)
    n1 = ob.n_live()
    x1 = wl.host_normal((n1, w.vocab), rng_seed, wl.TAG_LOGITS, sub=(1,), std=w.logit_std)
    t1 = time.perf_counter()
    ob.step(x1)
    topk_s = (time.perf_counter() - t1) * (W / max(n1, 1))
    per_step = (att_s * W * w.n_layers + topk_s) * w.n_requests
    sample = (f"oracle on request 0: naive float64 attention of {n_att} beams x {w.n_q_heads} heads at one layer "
              f"({att_s * 1e3:.1f} ms per beam-layer) scaled x{W} beams x{w.n_layers} layers x{w.n_requests} "
              f"requests; constrained top-K of {n1} live rows over {w.n_items[0]} items ({topk_s:.2f} s) "
              f"x{w.n_requests} requests")
    return per_step, sample


def batched_cpu_step_seconds(w: wl.Workload):
    """Seconds per decode step of a batched fp32 CPU implementation on every host core (a
    fairer CPU comparison than the naive oracle; reported beside it, never a parity check):
    one (request, layer) slice of the shared-context attention as GQA matmuls
    (all beams x query heads of a KV head against the request's context), scaled by the
    layers and requests, plus the full-vocab log-softmax, candidate gather and per-request
    top-K of one request's rows, scaled by the requests."""
    import torch
    threads = os.cpu_count() or 1
    old = torch.get_num_threads()
    torch.set_num_threads(threads)
    try:
        g = torch.Generator().manual_seed(w.seed * 1000 + 17)
        W, T, D, G = w.beam_widths[0], w.ctx_lens[0], w.head_dim, w.n_q_heads // w.n_kv_heads
        q = torch.randn(w.n_kv_heads, W * G, D, generator=g)
        k = torch.randn(w.n_kv_heads, T, D, generator=g)
        v = torch.randn(w.n_kv_heads, T, D, generator=g)
        x = torch.randn(W, w.vocab, generator=g) * w.logit_std
        score = torch.zeros(W)
        scale = 1.0 / D ** 0.5

        def attn():
            s = torch.matmul(q, k.transpose(1, 2)) * scale
            return torch.bmm(torch.softmax(s, dim=-1), v)

        def select():
            lp = torch.log_softmax(x, dim=-1)[:, w.code_base + w.codes_per_level:w.code_base + 2 * w.codes_per_level]
            return torch.topk((score[:, None] + lp).reshape(-1), W)

        attn(); select()  # warm the thread pool and allocator
        reps = 3
        t0 = time.perf_counter()
        for _ in range(reps):
            attn()
        att_s = (time.perf_counter() - t0) / reps
        t0 = time.perf_counter()
        for _ in range(reps):
            select()
        sel_s = (time.perf_counter() - t0) / reps
    finally:
        torch.set_num_threads(old)
    per_step = (att_s * w.n_layers + sel_s) * w.n_requests
    sample = (f"torch CPU fp32 on {threads} threads: attention of one (request, layer) slice "
              f"({att_s * 1e3:.1f} ms) x{w.n_layers} layers x{w.n_requests} requests; log-softmax + top-K of "
              f"{W} rows ({sel_s * 1e3:.1f} ms) x{w.n_requests} requests")
    return per_step, threads, sample


def workload_config(w):
    """The workload keys of the JSON line's config, the same for both arms."""
    return {"workload": w.name, "requests": w.n_requests, "ctx": w.ctx_lens[0], "beam": w.beam_widths[0],
            "layers": w.n_layers, "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
            "vocab": w.vocab, "levels": w.n_levels, "codes": w.codes_per_level, "items": w.n_items[0]}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    times = []
    sample = ""
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state
    for _ in range(max(args.steps, 1)):
        s, sample = oracle_step_seconds(w, budget_s=min(20.0, 60.0 / max(args.steps, 1)))
        times.append(s)
    sec = float(np.mean(times))
    value = 1.0 / sec
    line = {"metric": METRIC, "value": value, "unit": "steps/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(w), parallelism="oracle, one host core"),
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# replicas (N > 1): the path shards by request, so ranks decode independent
# batches and only the timing is reduced
# ---------------------------------------------------------------------------
def replica_workload(w, rank: int):
    """Each rank decodes its own batch of the same shape, seeded apart."""
    return w if rank == 0 else wl.make_workload(w.name, seed=w.seed + 1000 * rank)


def job_time_ms(ms_local: float, world: int, device) -> float:
    """The job's time is the slowest replica's: all-reduce MAX over the ranks."""
    if world == 1:
        return ms_local
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ms_per_step: float, world: int) -> float:
    """Whole-job throughput: every replica completes one step per ms_per_step."""
    return world * 1000.0 / ms_per_step


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args, w):
    import torch
    import torch.distributed as dist
    from beam_decode_gb300 import binding as B

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dev = f"cuda:{local}"
    w = replica_workload(w, rank)
    batch = DeviceBatch(w, dev)
    if args.attn_kernel != "auto":
        batch.beam.set_attn_kernel({"single": 1, "pair": 2}[args.attn_kernel])
    beam = batch.beam
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        batch.step()
    torch.cuda.synchronize()
    if beam.status() != 0:
        raise RuntimeError("device status error during warm-up")

    def timed(run_step, sample_clocks):
        clocks = Clocks(local) if sample_clocks else None
        if clocks:
            time.sleep(0.3)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            run_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        ck = clocks.stop() if clocks else None
        return job_time_ms(ms, world, dev), ck

    # eager launches, each bracketed by CUDA events on its stream: the per-kernel split
    for k in range(B.KERNEL_KINDS):
        beam.kernel_stats(k, reset=True)
    beam.set_timing(True)
    ms_eager, ck = timed(batch.step, args.no_graph)  # clocks here only when this is the headline
    beam.set_timing(False)
    stats = {B.KERNEL_NAMES[k]: beam.kernel_stats(k, reset=True) for k in range(B.KERNEL_KINDS)}
    ms = ms_eager
    launches = sum(n for (n, _) in stats.values())
    if not args.no_graph:
        # the headline: the same step captured once and replayed as a CUDA graph
        per_step = batch.capture()
        for _ in range(args.warmup):
            batch.graph.replay()
        ms, ck = timed(batch.graph.replay, True)
        launches = per_step * args.steps
        batch.release()
    # k_results runs once a decode is finished: decode the batch on to its last level and
    # time one results call per request (outside the timed step)
    batch.finish()
    beam.set_timing(True)
    for r in range(w.n_requests):
        beam.results(r)
    beam.set_timing(False)
    stats["results"] = beam.kernel_stats(B.KERNEL_NAMES.index("results"), reset=True)
    batch.step()  # back to the state a timed step leaves (level 1 selected)
    ms_per_step = ms / args.steps
    value = job_value(ms_per_step, world)
    st = beam.status()
    if st != 0:
        raise RuntimeError(f"device status error {st}")

    # roofline of the dominant kernel (shared-context attention)
    pk = _peaks()
    n_att, t_att = stats["attn"]
    att_ms = t_att / max(n_att, 1)
    flops_launch = batch.attn_flops() / w.n_layers
    achieved = flops_launch / (att_ms * 1e-3) / 1e12
    # the step runs at full SM clock (see "clocks"), so the burst GEMM rate is the ceiling;
    # the sustained (power-capped) rate is reported beside it.  The same launch against the HBM
    # roofline: one layer's ContextKV, each K/V row read once.  The bound reported is the one
    # the kernel is closer to (the tensor cores at wide beams, HBM at narrow ones).
    peak = pk["bf16"]
    attn_gbs = batch.ctx_bytes_per_layer() / (att_ms * 1e-3) / 1e9
    t_frac, h_frac = achieved / peak, attn_gbs / pk["hbm"]
    if t_frac >= h_frac:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": t_frac, "frac_of_sustained": achieved / pk["bf16_sust"],
                    "traffic": _attn_traffic(w), "kernel": "k_ctx_attn",
                    "peak_kind": f"{pk['src']} burst bf16", "hbm_frac": h_frac}
    else:
        roofline = {"bound": "hbm", "achieved": attn_gbs, "peak": pk["hbm"], "unit": "GB/s",
                    "frac": h_frac, "traffic": _attn_traffic(w), "kernel": "k_ctx_attn",
                    "peak_kind": f"{pk['src']} HBM copy", "tensor_frac": t_frac,
                    "algorithmic": "one layer's ContextKV, each K/V row once"}

    # end to end through the public API with host buffers
    e2e = run_e2e(args, batch) if (rank == 0 and not args.no_e2e) else None
    scoring = run_scoring(args, dev) if (rank == 0 and not args.no_scoring) else None

    per_kernel = {k: {"launches": n, "ms_per_launch": (t / n if n else 0.0), "ms_per_step": t / args.steps}
                  for k, (n, t) in stats.items() if n}
    hbm = small_kernel_hbm(batch, stats, pk)

    if rank == 0:
        cpu_s, sample = oracle_step_seconds(w, budget_s=12.0) if not args.no_cpu else (float("nan"), "skipped")
        cpu_batched = None
        if not args.no_cpu:
            bs, bthreads, bsample = batched_cpu_step_seconds(w)
            cpu_batched = {"value": 1.0 / bs, "unit": "steps/s", "cores": bthreads, "kind": "batched fp32 (torch CPU)",
                           "sample": bsample}
        line = {"metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": dict(workload_config(w),
                               l2="inputs larger than L2 (ContextKV %.2f GB)" % (batch.ctx_bytes_per_layer() * w.n_layers / 1e9),
                               parallelism=f"replicas{world}", cuda_graph=not args.no_graph,
                               attn_kernel=beam.attn_kernel()),
                "eager": {"value": job_value(ms_eager / args.steps, world), "unit": "steps/s",
                          "ms_per_step": ms_eager / args.steps},
                "roofline": roofline,
                "hbm_kernels": hbm,
                "kernels": per_kernel,
                "cpu_baseline": {"value": 1.0 / cpu_s if cpu_s == cpu_s else None, "unit": "steps/s", "cores": 1,
                                 "kind": "oracle", "sample": sample},
                "cpu_batched": cpu_batched,
                "e2e": e2e,
                "scoring": scoring,
                "gpu_launches": launches,
                "clocks": ck}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_scoring(args, device):
    """Multi-item candidate scoring at the pages' scoring size: each call scores 500
    candidates of one user; a batch of 8 calls with 2,000-token user prefixes and
    8-token candidates, Qwen3-1.7B attention geometry (28 layers).  One pass = 28
    masked-attention launches + label log-probs + ranking, inputs resident in HBM."""
    import torch
    from beam_decode_gb300 import binding as B
    NL, Hq, Hkv, D, V = 28, 16, 8, 128, 151936
    R, n_cand, seg, T = 8, 500, 8, 2000
    seed = 5
    shp = (NL, Hkv, R * T, D)
    ck = torch.empty(shp, dtype=torch.bfloat16, device=device)
    cv = torch.empty(shp, dtype=torch.bfloat16, device=device)
    for l in range(NL):
        ck[l] = wl.device_normal(shp[1:], seed, wl.TAG_CTX_K, device, torch.bfloat16, sub=l)
        cv[l] = wl.device_normal(shp[1:], seed, wl.TAG_CTX_V, device, torch.bfloat16, sub=l)
    sc = B.Score(NL, Hq, Hkv, D, V, [9454, 2753], ck, cv, [(r * T, T, [seg] * n_cand) for r in range(R)],
                 device=device)
    for l in range(NL):
        sc.seg_k[l] = wl.device_normal(sc.seg_k.shape[1:], seed, wl.TAG_BEAM_K, device, torch.bfloat16, sub=l)
        sc.seg_v[l] = wl.device_normal(sc.seg_v.shape[1:], seed, wl.TAG_BEAM_V, device, torch.bfloat16, sub=l)
    qs = (sc.rows, Hq, D)
    q = [wl.device_normal(qs, seed, wl.TAG_Q, device, torch.bfloat16, sub=l) for l in range(NL)]
    out = torch.empty(qs, dtype=torch.bfloat16, device=device)
    x = wl.device_normal((sc.n_candidates, V), seed, wl.TAG_LOGITS, device, std=2.0)
    stream = torch.cuda.current_stream()

    def one():
        for l in range(NL):
            sc.attn(l, q[l], out)
        return sc.labels(x)

    for _ in range(max(2, args.warmup)):
        one()
    torch.cuda.synchronize()
    steps = max(3, args.steps // 2)
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    att_ms = 0.0
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # the attention part alone
    e0.record(stream)
    for _ in range(steps):
        for l in range(NL):
            sc.attn(l, q[l], out)
    e2.record(stream)
    torch.cuda.synchronize()
    att_ms = e0.elapsed_time(e2) / steps
    if sc.status() != 0:
        raise RuntimeError("scoring: device status error")
    flops = 4.0 * NL * Hq * D * R * n_cand * seg * (T + (seg + 1) / 2.0)
    return {"workload": f"{R} calls x {n_cand} candidates x {seg} tokens, prefix {T}, 28 layers",
            "calls_per_s": R * 1000.0 / ms, "candidates_per_s": R * n_cand * 1000.0 / ms, "ms_per_pass": ms,
            "attn_ms_per_layer": att_ms / NL, "attn_TFLOP_s": flops / (att_ms * 1e-3) / 1e12,
            "labels_ms": ms - att_ms}


def small_kernel_hbm(batch, stats, pk):
    """Algorithmic HBM bytes / CUDA-event time per launch of the step's memory-bound kernels
    (the step is t = 1 at full width: n_live = W_r beams per request).  logsoftmax_gather
    reads every live row's fp32 logits once.  topk_select reads the C candidate keys of every
    live beam and writes W_r (parent, code, key) triples per request.  advance reads a beam's
    selection (parent, code, key), its parent's trie node, the node's child base and on
    average C/64 + 1 mask words below its code, and its parent's ancestry row (t entries);
    it writes parent, token, node, score and the ancestry row (t + 1 entries).  results (one
    launch per gr_beam_results call, after the batch is decoded to its last level L; each
    launch covers every request) reads each final beam's ancestry row, the L tokens it
    names, its node and leaf item and its score, and writes L codes, the item id and the
    score.  The small kernels are bound by launch latency, not bandwidth: their fractions
    say how far from the HBM roofline that leaves them."""
    w = batch.w
    C, L = w.codes_per_level, w.n_levels
    beams = float(sum(w.beam_widths))
    per_launch = {
        "logsoftmax_gather": batch.rows * w.vocab * 4.0,
        "topk_select": beams * C * 4.0 + beams * 12.0,
        "advance": beams * (12.0 + 4.0 + 4.0 + 4.0 * (C / 64 + 1) + 4.0 * 1 + 16.0 + 4.0 * 2),
        "results": beams * (8.0 * L + 4.0 + 8.0 + 4.0 + 4.0 * L + 8.0 + 4.0),
    }
    hbm = {}
    for k, byts in per_launch.items():
        n, t = stats.get(k, (0, 0.0))
        if n:
            gbs = byts / (t / n * 1e-3) / 1e9
            hbm[k] = {"GB_s": gbs, "frac": gbs / pk["hbm"], "bytes_per_launch": byts, "us_per_launch": t / n * 1e3}
    return hbm


def run_e2e(args, batch: DeviceBatch):
    """Same step through the public API with pinned host inputs copied in and the
    step's selection read back every step.  The copies run on their own stream,
    layer by layer, so that a layer's inputs arrive while earlier layers compute;
    events keep every device buffer from being overwritten before its consumer ran.
    The host issues the next step's copies before it reads the current step's
    selection back, so the copy stream never waits for the read-back: each timed
    step still holds one full set of input copies, one step and one read-back."""
    import torch
    w = batch.w
    beam = batch.beam
    NL = w.n_layers
    host_q = [q.cpu().pin_memory() for q in batch.q]
    host_k = [k.cpu().pin_memory() for k in batch.new_k]
    host_v = [v.cpu().pin_memory() for v in batch.new_v]
    host_x = batch.logits[1].cpu().pin_memory()
    dq = [torch.empty_like(q) for q in batch.q]
    dx = torch.empty_like(batch.logits[1])
    h2d = sum(t.numel() * t.element_size() for t in host_q + host_k + host_v) + host_x.numel() * 4
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    arrived = [torch.cuda.Event() for _ in range(NL + 1)]   # inputs of layer l (NL: logits) on the device
    used = [torch.cuda.Event() for _ in range(NL + 1)]      # the step's consumer of those buffers ran
    for e in used:
        e.record(comp)
    # BeamKV slots of level 0 (the open level at step 1) for every layer
    kv = [beam.kv_slot(l) for l in range(NL)]
    d2h = 0

    def copies():  # one step's inputs, host -> device
        with torch.cuda.stream(copy):
            for l in range(NL):
                copy.wait_event(used[l])
                kv[l][0].copy_(host_k[l], non_blocking=True)
                kv[l][1].copy_(host_v[l], non_blocking=True)
                dq[l].copy_(host_q[l], non_blocking=True)
                arrived[l].record(copy)
            copy.wait_event(used[NL])
            dx.copy_(host_x, non_blocking=True)
            arrived[NL].record(copy)

    def step():
        beam.rewind(1)
        for l in range(NL):
            comp.wait_event(arrived[l])
            beam.decode_attn(l, dq[l], batch.out[l])
            used[l].record(comp)
        comp.wait_event(arrived[NL])
        beam.constrained_topk(dx)
        used[NL].record(comp)
        beam.advance()

    def readback():
        nonlocal d2h
        n = 0
        for r in range(w.n_requests):  # the step's selection, read back (synchronises the step)
            par, tok, nod, sc = beam.path(r, 1)
            n += (par.nbytes + tok.nbytes + sc.nbytes)
        d2h = n

    copies()
    for _ in range(2):
        step()
        copies()
        readback()
    torch.cuda.synchronize()
    steps = max(3, args.steps // 4)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
        copies()
        readback()
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    # the host->device copy rate alone, for reading the number
    t1 = time.perf_counter()
    dx.copy_(host_x, non_blocking=True)
    torch.cuda.synchronize()
    gbs = host_x.numel() * 4 / (time.perf_counter() - t1) / 1e9
    return {"value": 1.0 / dt, "unit": "steps/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps, "h2d_GB_s_single_copy": gbs}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gr", choices=["gr", "reference"])
    ap.add_argument("--workload", default="long", choices=["tiny", "page1", "short", "long", "mixed"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of a replayed CUDA graph")
    ap.add_argument("--no-scoring", action="store_true", help="skip the multi-item scoring measurement")
    ap.add_argument("--requests", type=int, default=0,
                    help="keep only the first N requests of the workload (a smaller case for profiling)")
    ap.add_argument("--layers", type=int, default=0,
                    help="keep only the first N layers (a smaller case for profiling: same per-launch shapes)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--attn-kernel", default="auto", choices=["auto", "single", "pair"],
                    help="decode-attention kernel (auto: the library's choice)")
    args = ap.parse_args()
    w = wl.make_workload(args.workload)
    if args.requests:
        n = args.requests
        w.ctx_lens, w.beam_widths, w.n_items = w.ctx_lens[:n], w.beam_widths[:n], w.n_items[:n]
    if args.layers:
        w.n_layers = min(args.layers, w.n_layers)
    if args.impl == "reference":
        return run_reference(args, w)
    from beam_decode_gb300.build import build
    build()
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
