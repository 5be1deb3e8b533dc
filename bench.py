"""Benchmark of one batched speculation round on GB300.

Step = one pass of the whole round over one batch: Saguaro draft sampling,
lossless verification with the residual / bonus draw, outcome prediction
(top-F_k guesses) and the speculation-cache lookup, through the fused
``ssd_round`` call of the C ABI.  Workload: the Llama-3-vocabulary round
(B=32 sequences, K=5 draft tokens, V=128256, bf16 logits, Zipf-shaped target,
draft = target + N(0,1), T=1, C=1, fan-out (16,8,4,2,1,1) from budget 32).
Metric: seq-rounds/s (sequences verified+predicted per second).

Prints one JSON line.  Also reported on the same line: the roofline of the
dominant kernel (the HBM statistics pass), tree-masked branch attention on
its two workloads (GB/s against the HBM peak), the end-to-end figure through
host buffers, the CPU oracle on a bounded sample, and SM clocks sampled while
the GPU was under load.

``--impl reference`` times the fp64 CPU oracle (the reference arm) on the same
workload and metric; under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "verify+predict seq-rounds/s at V=128k"
UNIT = "seq-rounds/s"
L2_BYTES = 129 * 2 ** 20


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; sequences are independent units)
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def rank_seed(base: int, rank: int) -> int:
    """Each rank verifies its own batch of sequences (weak scaling)."""
    return base + 1000003 * rank


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# clocks sampled during the timed work
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, tag):
        self.marks.append((tag, time.time()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.lines:
            if t0 <= ts <= t1:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
def round_spec():
    from speculative_decoding_vocab_gb300 import workloads as w
    return w.llama3_round(T=1.0, B=32)


class RoundBuffers:
    """Inputs and outputs of one round resident on the device."""

    def __init__(self, spec, inp, device):
        import torch
        from speculative_decoding_vocab_gb300.binding import tensor
        self.spec = spec
        self.target = tensor(inp.target, device)
        self.draft = tensor(inp.draft, device)
        self.u_draft = torch.from_numpy(inp.u_draft).to(device)
        self.u_acc = torch.from_numpy(inp.u_acc).to(device)
        self.u_bonus = torch.from_numpy(inp.u_bonus).to(device)
        self.payload = torch.from_numpy(inp.payload).to(device)


def make_outputs(spec, device):
    import torch
    B, K = spec.B, spec.K
    sumF = int(sum(spec.F))
    i32 = dict(dtype=torch.int32, device=device)
    f32 = dict(dtype=torch.float32, device=device)
    return dict(d=torch.empty(B, K, **i32), qd=torch.empty(B, K, **f32),
                accept_len=torch.empty(B, **i32), out_tokens=torch.empty(B, K + 1, **i32),
                bonus=torch.empty(B, **i32), accept_prob=torch.empty(B, K, **f32),
                resid_mass=torch.empty(B, **f32), guess=torch.empty(B, sumF, **i32),
                guess_q=torch.empty(B, sumF, **f32), slot=torch.empty(B, **i32),
                next_tokens=torch.empty(B, K, **i32), hits=torch.zeros(1, **i32),
                near_ties=torch.zeros(1, **i32), status=torch.zeros(1, **i32))


def run_round(ssd, spec, buf, out, ws, pipelined=False):
    ssd.ssd_round(buf.target, buf.draft, spec.V, spec.F, spec.C, spec.T, buf.u_draft, buf.u_acc,
                  buf.u_bonus, out["d"], out["accept_len"], out["out_tokens"], out["bonus"],
                  payload=buf.payload, qd_out=out["qd"], accept_prob=out["accept_prob"],
                  resid_mass=out["resid_mass"], guess=out["guess"], guess_q=out["guess_q"],
                  slot=out["slot"], next_tokens=out["next_tokens"], hits=out["hits"],
                  status=out["status"], ws=ws, near_ties=out["near_ties"], pipelined=pipelined)


def kernels_per_round(spec) -> int:
    """Kernels of ours one ssd_round launches: the statistics pass (k_stats),
    the per-pair merges and draws (k_pair) and the residual units with the
    sequence finish (k_resid)."""
    return 3


def capture_graphs(calls, device):
    """One CUDA graph per zero-argument launch function (each replays a whole
    round's launches -- statistics, pair and residual kernels -- without host
    work in between)."""
    import torch
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        for fn in calls:
            fn()
    torch.cuda.current_stream(device).wait_stream(side)
    torch.cuda.synchronize(device)
    graphs = []
    for fn in calls:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append(g)
    torch.cuda.synchronize(device)
    return graphs


NSTREAMS = 6          # streams that independent rounds are issued on, round-robin
NBUF = 2 * NSTREAMS   # output/workspace sets: rounds in flight together never share one


def stream_chain(launch, device, nstreams=NSTREAMS):
    """chain(first, n) enqueues rounds first .. first+n-1, round q by launch(q)
    on stream q % nstreams, forked from and joined back into the current
    stream (so a CUDA graph captures it whole).  Rounds on one stream follow
    each other (pipelined: a round's statistics pass overlaps the previous
    round's tail); rounds on different streams are independent batches and
    overlap freely."""
    import torch
    streams = [torch.cuda.Stream(device) for _ in range(nstreams)]

    def chain(first, n):
        cur = torch.cuda.current_stream(device)
        for st in streams:
            st.wait_stream(cur)
        for q in range(first, first + n):
            with torch.cuda.stream(streams[q % nstreams]):
                launch(q)
        for st in streams:
            cur.wait_stream(st)

    return chain


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def bench_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from speculative_decoding_vocab_gb300 import build
    build.build()
    from speculative_decoding_vocab_gb300 import binding as ssd
    from speculative_decoding_vocab_gb300 import workloads as w

    spec = round_spec()
    inp = w.make_round(spec, seed=rank_seed(0, rank))
    # rotating input sets whose total exceeds L2 several times over
    per_set = w.round_bytes(spec)
    nsets = max(NBUF, int(np.ceil(3 * L2_BYTES / per_set)) + 1)
    sets = [RoundBuffers(spec, inp, device) for _ in range(nsets)]
    out = make_outputs(spec, device)
    ws = ssd.workspace(spec.B, spec.K, spec.V, spec.dtype, spec.F, device)
    stream = torch.cuda.current_stream(device)

    K, W = args.steps, args.warmup
    for i in range(W):
        run_round(ssd, spec, sets[i % nsets], out, ws)
    torch.cuda.synchronize()
    graphs = capture_graphs([lambda b=b: run_round(ssd, spec, b, out, ws) for b in sets], device)
    for i in range(W):
        graphs[i % nsets].replay()
    torch.cuda.synchronize()
    # the timed steps: rounds of independent batches (step q reads input set
    # q % nsets and writes output/workspace set q % NBUF) issued round-robin on
    # NSTREAMS streams with ssd_round_pipelined: on a stream, a round's
    # statistics pass overlaps the previous round's verification tail, and the
    # streams' rounds overlap each other; CUDA graphs of chain_n steps, and one
    # graph of the remainder
    outs = [make_outputs(spec, device) for _ in range(NBUF)]
    wss = [ssd.workspace(spec.B, spec.K, spec.V, spec.dtype, spec.F, device) for _ in range(NBUF)]
    chain_n = int(np.lcm(nsets, NBUF))
    chain_n *= max(1, 48 // chain_n)
    chain = stream_chain(lambda q: run_round(ssd, spec, sets[q % nsets], outs[q % NBUF], wss[q % NBUF],
                                             pipelined=True), device)
    chain(0, max(W, NBUF))
    torch.cuda.synchronize()
    g_chain = capture_graphs([lambda: chain(0, chain_n)], device)[0]
    rem = K % chain_n
    g_rem = capture_graphs([lambda: chain(0, rem)], device)[0] if rem else None
    for _ in range(max(1, W // chain_n + 1)):
        g_chain.replay()
    torch.cuda.synchronize()

    def timed_steps(n):
        """n steps: whole chains, then the remainder's graph."""
        for _ in range(n // chain_n):
            g_chain.replay()
        if n % chain_n:
            g_rem.replay()

    # the statistics kernel timed on its own stream with CUDA events (direct launches)
    nev = min(K, 256)
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(nev)]
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(nev)]
    for e in ev_b + ev_a:  # torch creates the CUDA event on its first record
        e.record(stream)
    torch.cuda.synchronize()
    for s in range(nev):
        ssd.ssd_set_timing_events(ev_b[s], ev_a[s])
        run_round(ssd, spec, sets[s % nsets], out, ws)
    ssd.ssd_set_timing_events(None, None)
    torch.cuda.synchronize()
    stats_ms = statistics.mean(b.elapsed_time(a) for b, a in zip(ev_b, ev_a))

    # clocks: sample while the GPU runs untimed rounds, the timed region, untimed rounds
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else local)
    sampler.start()
    t_load0 = time.time()
    settle = time.time() + 0.6
    i = 0
    while time.time() < settle:
        for _ in range(200):
            graphs[i % nsets].replay()
            i += 1
        torch.cuda.synchronize()

    # timed region: exactly K steps (pipelined rounds over the input sets)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for o in outs:
        o["near_ties"].zero_()
    barrier(device)
    torch.cuda.synchronize()
    start.record(stream)
    timed_steps(K)
    stop.record(stream)
    torch.cuda.synchronize()
    barrier(device)
    ms = start.elapsed_time(stop) / K
    ms = max_over_ranks(ms, device)
    near_k = sum(int(o["near_ties"].item()) for o in outs)  # the K timed rounds alone
    status = int(sum(int(o["status"].item()) for o in outs))
    same = all(torch.equal(o[k], out[k]) for o in outs
               for k in ("d", "accept_len", "out_tokens", "bonus", "guess", "slot", "next_tokens"))

    settle = time.time() + 0.6
    while time.time() < settle:
        for _ in range(200):
            graphs[i % nsets].replay()
            i += 1
        torch.cuda.synchronize()
    t_load1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_load0, t_load1)
    status += int(out["status"].item())
    # one round on its own (graph replays of single, non-overlapping rounds)
    for q in range(nsets):
        graphs[q].replay()
    lat_ms = _time_calls(lambda q: graphs[q % nsets].replay(), 100, stream)

    peaks = load_peaks()
    hbm_peak = peaks.get("hbm_gbs") or 6800.0
    alg_bytes = w.round_bytes(spec)
    achieved = alg_bytes / (stats_ms * 1e-3) / 1e9
    traffic = profiled_traffic("k_stats", spec.name)

    value = spec.B * world / (ms * 1e-3)
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded Zipf-shaped bf16 logits (-1.1 ln rank over a permutation + "
                "N(0,0.3^2)), draft = target + N(0,1); Philox4x32-10 uniforms",
        "config": {"workload": spec.name, "B": spec.B, "K": spec.K, "V": spec.V,
                   "input_dtype": "bf16", "T": spec.T, "C": spec.C, "F": list(spec.F),
                   "call": "ssd_round_pipelined (sample + verify + predict + lookup); steps are "
                           "independent batches (rotating input sets, own outputs and workspaces) issued "
                           f"round-robin on {NSTREAMS} streams: on a stream a step's statistics pass overlaps "
                           "the previous step's verification tail, and the streams' steps overlap; CUDA "
                           f"graphs of {chain_n} steps",
                   "l2": f"rotating {nsets} input sets, {nsets * per_set / 1e6:.0f} MB > 129 MB L2",
                   "parallelism": f"replicas x{world} (independent sequences per GPU)"},
        "roofline": {"kernel": "k_stats (register-resident segment statistics, one warp per 4 KiB)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                     "algorithmic_bytes": alg_bytes, "kernel_ms": round(stats_ms, 5),
                     "peak_source": "measured" if "hbm_gbs" in peaks else "fallback"},
        "gpu_launches": kernels_per_round(spec) * K,
        "round_latency_ms": round(lat_ms, 5),
        "round_latency_note": "one round alone (ssd_round, graph replays with nothing to overlap)",
        "outputs_equal_plain_round": bool(same),
        "clocks": clocks,
        "status_flags": status,
        "near_ties": {"count": near_k, "rounds": K, "sequences": K * spec.B,
                      "what": "draws within 1e-6 W of a bin edge and acceptance tests with "
                              "|u - p/q'| < 1e-6 (GPU fp32 count, ssd_round near_ties output)"},
    }
    result["step_roofline_frac"] = round(alg_bytes / (ms * 1e-3) / 1e9 / hbm_peak, 4)
    # secondary ceilings of a step: the exponentials (one per logit; none at T = 0) on the
    # special function units, against the HBM time of the logits
    n_exp = 0 if spec.T == 0 else 2 * (spec.K + 1) * spec.V * spec.B
    result["secondary_ceilings"] = {
        "exp_count": n_exp, "sfu_floor_ms": round(sfu_floor_ms(n_exp, device), 5),
        "hbm_floor_ms": round(alg_bytes / (hbm_peak * 1e9) * 1e3, 5),
        "note": "16 exponentials per clock per SM at the maximum SM clock; the round is HBM-bound"}
    if not args.no_extras:
        result["e2e"] = bench_e2e(ssd, spec, inp, device, K, W)
        result["branch_attention"] = bench_attention(ssd, device, hbm_peak)
        result["other_rounds"] = bench_other_rounds(ssd, w, device, hbm_peak)
        result["tiny_round"] = bench_tiny_round(ssd, w, device)
        result["round_analytics"] = bench_analytics(ssd, w, device, hbm_peak)
        result["saguaro_sample"] = bench_saguaro_sample(ssd, w, device, hbm_peak)
        result["miss_fallback"] = bench_fallback(ssd, w, device, hbm_peak)
        result["cache_fill"] = bench_cache_fill(ssd, w, device, hbm_peak)
        result["tree_verify"] = bench_tree(ssd, w, device, hbm_peak)
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(spec, inp, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bench_e2e(ssd, spec, inp, device, K, W):
    """The same metric through the public call with HOST buffers: every step
    copies that step's logits and uniforms from pinned host memory to the
    device, runs the round and reads the emitted tokens, accept lengths,
    bonus tokens and cache slots back.  Steps are pipelined over two device
    input buffers: the uploads run on a copy stream and step q + 1's upload
    overlaps step q's round and readback on the compute stream (the host link
    bounds the step, not the round)."""
    import torch
    from speculative_decoding_vocab_gb300.binding import pinned
    hin = dict(target=pinned(inp.target), draft=pinned(inp.draft),
               u_draft=torch.from_numpy(inp.u_draft).pin_memory(),
               u_acc=torch.from_numpy(inp.u_acc).pin_memory(),
               u_bonus=torch.from_numpy(inp.u_bonus).pin_memory(),
               payload=torch.from_numpy(inp.payload).pin_memory())
    bufs = [RoundBuffers(spec, inp, device) for _ in range(2)]
    outs = [make_outputs(spec, device) for _ in range(2)]
    wss = [ssd.workspace(spec.B, spec.K, spec.V, spec.dtype, spec.F, device) for _ in range(2)]
    keys = ("out_tokens", "accept_len", "bonus", "slot", "next_tokens")
    houts = [{k: torch.empty_like(outs[0][k], device="cpu").pin_memory() for k in keys} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in hin.values())
    d2h = sum(t.numel() * t.element_size() for t in houts[0].values())
    comp = torch.cuda.current_stream(device)
    copy = torch.cuda.Stream(device)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    for e in uploaded + consumed:  # torch creates the CUDA event on its first record
        e.record(comp)

    def step(q):
        i = q % 2
        with torch.cuda.stream(copy):
            copy.wait_event(consumed[i])  # round q - 2 has read buffer i
            for k in ("target", "draft", "u_draft", "u_acc", "u_bonus", "payload"):
                getattr(bufs[i], k).copy_(hin[k], non_blocking=True)
            uploaded[i].record(copy)
        comp.wait_event(uploaded[i])
        run_round(ssd, spec, bufs[i], outs[i], wss[i])
        consumed[i].record(comp)
        for k, t in houts[i].items():
            t.copy_(outs[i][k], non_blocking=True)

    for q in range(W):
        step(q)
    torch.cuda.synchronize()
    n = max(K // 4, 20)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    copy.wait_stream(comp)  # no upload of the timed steps starts before the start mark
    for q in range(n):
        step(q)
    b.record(comp)  # after the last round, which waited for the last upload, and its readback
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    same = all(torch.equal(houts[i][k], outs[i][k].cpu()) for i in range(2) for k in keys)
    return {"value": round(spec.B / (ms * 1e-3), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
            "steps": n, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "readback_ok": bool(same),
            "schedule": "uploads on a copy stream into two device input buffers; rounds and readbacks "
                        "on the compute stream; step q+1's upload overlaps step q's round"}


SFU_EXP_PER_CLK_PER_SM = 16  # ex2 results per clock per SM (the special function units)


def sfu_floor_ms(n_exp, device):
    """Time the special function units need for n_exp exponentials at the
    device's SM count and maximum SM clock (a secondary ceiling)."""
    import torch
    props = torch.cuda.get_device_properties(device)
    sms = props.multi_processor_count
    mhz = _max_sm_mhz()
    return n_exp / (SFU_EXP_PER_CLK_PER_SM * sms * mhz * 1e6) * 1e3


def _max_sm_mhz():
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits"],
                             capture_output=True, text=True, timeout=10).stdout.split()
        return float(out[0])
    except Exception:
        return 2070.0  # the GB300's maximum SM clock


def _time_calls(fn, n, stream):
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(n):
        fn(i)
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def device_attention_inputs(spec, device, seed):
    """Seeded attention inputs generated directly on the device (bench only)."""
    import torch
    from speculative_decoding_vocab_gb300 import workloads as w
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0xA77E]))
    parent1 = w.attn_tree(spec, rng)
    N = int(parent1.shape[0])
    Nq = N - spec.K if spec.tree == "fanout" else N
    nblk = (spec.L + N + w.PAGE - 1) // w.PAGE
    nb = spec.B * nblk
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    table = torch.randperm(nb, generator=g, device=device).to(torch.int32).view(spec.B, nblk)
    q = torch.randn(spec.B, Nq, spec.Hq, spec.d, generator=g, device=device).to(torch.bfloat16)
    kc = torch.randn(nb, spec.Hkv, w.PAGE, spec.d, generator=g, device=device).to(torch.bfloat16)
    vc = torch.randn(nb, spec.Hkv, w.PAGE, spec.d, generator=g, device=device).to(torch.bfloat16)
    prefix = torch.full((spec.B,), spec.L, dtype=torch.int32, device=device)
    parent = torch.from_numpy(np.broadcast_to(parent1, (spec.B, N)).copy()).to(device)
    return q, kc, vc, table, prefix, parent, N, Nq


def bench_attention(ssd, device, hbm_peak):
    import torch
    from speculative_decoding_vocab_gb300 import workloads as w
    res = {}
    stream = torch.cuda.current_stream(device)
    for spec in (w.draft_branch_attention(), w.verify_attention_at_scale()):
        q, kc, vc, table, prefix, parent, N, Nq = device_attention_inputs(spec, device, 7)
        # two copies of the caches so consecutive calls do not hit in L2 (config 4 is ~70 MB)
        kc2, vc2 = kc.clone(), vc.clone()
        out = torch.empty_like(q)
        st = torch.zeros(1, dtype=torch.int32, device=device)
        wsn = ssd.ssd_attention_workspace_size(spec.B, Nq, spec.Hq, spec.Hkv, spec.d, spec.L)
        aws = torch.empty(max(wsn, 256), dtype=torch.uint8, device=device)

        def call(i):
            ssd.ssd_branch_attention(q, kc if i % 2 == 0 else kc2, vc if i % 2 == 0 else vc2,
                                     table, prefix, parent, out, status=st, ws=aws)

        for i in range(3):
            call(i)
        # replayed as a CUDA graph of two calls (one per cache copy), so that the
        # host's per-call work (tensor maps, launch) never starves the GPU
        g = capture_graphs([lambda: (call(0), call(1))], device)[0]
        for _ in range(2):
            g.replay()
        n = 20 if spec.L > 4096 else 100
        ms = _time_calls(lambda i: g.replay(), n // 2, stream) / 2
        alg = w.attention_bytes(spec, N, Nq, [spec.L] * spec.B)
        vis_pairs = spec.B * spec.Hq * Nq * spec.L  # prefix keys
        par = parent[0].cpu().numpy()
        depth = 0
        for m in range(N - Nq, N):
            x = m
            while x >= 0:
                depth += 1
                x = par[x]
        vis_pairs += spec.B * spec.Hq * depth
        flops = 4 * spec.d * vis_pairs
        gbs = alg / (ms * 1e-3) / 1e9
        res[spec.name] = {"ms": round(ms, 4), "algorithmic_bytes": alg, "GB/s": round(gbs, 1),
                          "frac_of_hbm_peak": round(gbs / hbm_peak, 4),
                          "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 2),
                          "exp_count": vis_pairs,
                          "sfu_floor_ms": round(sfu_floor_ms(vis_pairs, device), 4),
                          # the binding floor: HBM bytes, bf16 tensor FLOPs (measured burst
                          # peak) or the exponentials, whichever takes longest
                          "frac_of_floor": round(max(alg / (hbm_peak * 1e9),
                                                     flops / ((load_peaks().get("bf16_tflops") or 1900.0) * 1e12),
                                                     sfu_floor_ms(vis_pairs, device) * 1e-3) / (ms * 1e-3), 4),
                          "kernel": "k_branch_attn_tc (tcgen05/TMEM + TMA)",
                          "status_flags": int(st.item())}
        del g, q, kc, vc, kc2, vc2, out
        torch.cuda.empty_cache()
    return res


def bench_tiny_round(ssd, w, device):
    """The tiny round (B=1, K=4, V=4096 fp32): latency-bound, so its figure is
    microseconds per round (graph replays over 64 seeded rounds)."""
    import torch
    spec = w.tiny_round()
    nsets = 64
    sets = [RoundBuffers(spec, w.make_round(spec, seed=0, rnd=r), device) for r in range(nsets)]
    out = make_outputs(spec, device)
    ws = ssd.workspace(spec.B, spec.K, spec.V, spec.dtype, spec.F, device)
    for i in range(3):
        run_round(ssd, spec, sets[i], out, ws)
    graphs = capture_graphs([lambda b=b: run_round(ssd, spec, b, out, ws) for b in sets], device)
    stream = torch.cuda.current_stream(device)
    ms = _time_calls(lambda i: graphs[i % nsets].replay(), 500, stream)
    return {"workload": spec.name, "us_per_round": round(ms * 1e3, 2),
            "seq_rounds_per_s": round(spec.B / (ms * 1e-3), 1),
            "note": "back-to-back graph replays of one round each (B = 1): latency, not bandwidth"}


def device_round_sets(spec, device, seed):
    """Zipf-shaped bf16 target/draft logits of ``spec`` generated on the device
    (bench only), copied into enough input sets that a rotation over them is
    larger than L2; returns (sets, nsets, bytes per set, uniforms)."""
    import torch
    from speculative_decoding_vocab_gb300 import workloads as w
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shape = (spec.B, spec.K + 1, spec.V)
    rank = torch.argsort(torch.rand(shape, generator=g, device=device), dim=-1).float() + 1
    zt = -spec.zipf_slope * torch.log(rank) + spec.target_noise * torch.randn(
        shape, generator=g, device=device)
    del rank
    zd = zt + spec.draft_noise * torch.randn(shape, generator=g, device=device)
    per = w.round_bytes(spec)
    nsets = max(2, int(np.ceil(3 * L2_BYTES / per)) + 1) if per < 2 * L2_BYTES else 1
    sets = [(zt.to(torch.bfloat16), zd.to(torch.bfloat16)) for _ in range(nsets)]
    del zt, zd
    u = torch.rand(3, spec.B, spec.K + 1, generator=g, device=device)
    uni = (u[0, :, :spec.K].contiguous(), u[1, :, :spec.K].contiguous(), u[2, :, 0].contiguous())
    return sets, nsets, per, uni


def bench_saguaro_sample(ssd, w, device, hbm_peak):
    """The draft's Saguaro draw alone (ssd_saguaro_sample: the K draft rows of
    every sequence, K V elem bytes per sequence) on the Llama-3 round (C = 1)
    and the large-batch Qwen-3 round (C = 0.5)."""
    import torch
    res = {}
    stream = torch.cuda.current_stream(device)
    for spec in (w.llama3_round(T=1.0, B=32), w.qwen3_round(C=0.5)):
        sets, nsets, per, (ud, _, _) = device_round_sets(spec, device, 17)
        B, K = spec.B, spec.K
        i32 = dict(dtype=torch.int32, device=device)
        d = torch.empty(B, K, **i32)
        qd = torch.empty(B, K, dtype=torch.float32, device=device)
        st = torch.zeros(1, **i32)
        ws = ssd.workspace(B, K, spec.V, spec.dtype, spec.F, device)

        def call(i):
            ssd.ssd_saguaro_sample(sets[i % nsets][1], spec.V, spec.F, spec.C, spec.T, ud, d, qd_out=qd,
                                   status=st, ws=ws)

        for i in range(3):
            call(i)
        g = capture_graphs([lambda: [call(i) for i in range(nsets)]], device)[0]
        g.replay()
        ms = _time_calls(lambda i: g.replay(), max(3, 60 // nsets), stream) / nsets
        alg = B * K * spec.V * 2  # the K draft rows of every sequence, bf16
        res[spec.name] = {"ms": round(ms, 4), "algorithmic_bytes": alg,
                          "frac_of_hbm_peak": round(alg / (ms * 1e-3) / 1e9 / hbm_peak, 4),
                          "seq_per_s": round(B / (ms * 1e-3), 1), "C": spec.C,
                          "status_flags": int(st.item())}
        del g, sets
        torch.cuda.empty_cache()
    return res


def bench_analytics(ssd, w, device, hbm_peak):
    """Exact round analytics (acceptance rates, accept-count distribution, hit
    rate, expected tokens) on the large-batch Qwen-3 round."""
    import torch
    spec = w.qwen3_round(C=0.5)
    stream = torch.cuda.current_stream(device)
    sets, nsets, per, _ = device_round_sets(spec, device, 13)
    B, K = spec.B, spec.K
    f32 = dict(dtype=torch.float32, device=device)
    pa, hr, et = torch.empty(B, K + 1, **f32), torch.empty(B, **f32), torch.empty(B, **f32)
    al, rw, hm = torch.empty(B, K, **f32), torch.empty(B, K, **f32), torch.empty(B, K + 1, **f32)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    ws = ssd.workspace(B, K, spec.V, spec.dtype, spec.F, device)

    def call(i):
        t, d = sets[i % nsets]
        ssd.ssd_round_analytics(t, d, spec.V, spec.F, spec.C, spec.T, pa, hr, et, alpha=al,
                                resid_w=rw, hit_mass=hm, status=st, ws=ws)

    for i in range(3):
        call(i)
    graphs = capture_graphs([lambda i=i: call(i) for i in range(nsets)], device)
    ms = _time_calls(lambda i: graphs[i % nsets].replay(), 50, stream)
    res = {"workload": spec.name, "ms": round(ms, 4),
           "seq_rounds_per_s": round(B / (ms * 1e-3), 1), "algorithmic_bytes": per,
           "frac_of_hbm_peak": round(per / (ms * 1e-3) / 1e9 / hbm_peak, 4),
           "mean_hit_rate": round(float(hr.mean().item()), 4),
           "mean_exp_tokens": round(float(et.mean().item()), 4), "status_flags": int(st.item())}
    del graphs, sets, ws
    torch.cuda.empty_cache()
    return res


def bench_cache_fill(ssd, w, device, hbm_peak):
    """The speculation-cache fill by branch decode on the Llama-3 vocabulary and
    the draft-attention tree: K decode steps, each a K/V append of the fed
    nodes, tree attention over the 2 Ki-token prefix and the tree, and the
    Saguaro draw of every branch's next token into the payload.  One CUDA graph
    per fill; the draws alone are timed for their HBM roofline."""
    import torch
    spec = w.llama3_fill()
    B, K, S, V, Hq, Hkv, d, L = spec.B, spec.K, spec.S, spec.V, spec.Hq, spec.Hkv, spec.d, spec.L
    stream = torch.cuda.current_stream(device)
    g = torch.Generator(device=device)
    g.manual_seed(23)
    logits = []
    for t in range(K):
        rank = torch.argsort(torch.rand(B, S, V, generator=g, device=device), dim=-1).float() + 1
        z = -1.1 * torch.log(rank) + torch.randn(B, S, V, generator=g, device=device)
        logits.append(z.to(torch.bfloat16))
        del rank, z
    u = torch.rand(K, B, S, generator=g, device=device)
    bf = dict(dtype=torch.bfloat16, device=device)
    kn = [torch.randn(B, S, Hkv, d, generator=g, device=device).to(torch.bfloat16) for _ in range(K)]
    vn = [torch.randn(B, S, Hkv, d, generator=g, device=device).to(torch.bfloat16) for _ in range(K)]
    q = [torch.randn(B, S, Hq, d, generator=g, device=device).to(torch.bfloat16) for _ in range(K)]
    N = K + K * S
    maxb = (L + N + 15) // 16
    nb = B * maxb
    table = torch.randperm(nb, generator=g, device=device).to(torch.int32).view(B, maxb)
    kc = torch.randn(nb, Hkv, 16, d, generator=g, device=device).to(torch.bfloat16)
    vc = torch.randn(nb, Hkv, 16, d, generator=g, device=device).to(torch.bfloat16)
    prefix = torch.full((B,), L, dtype=torch.int32, device=device)
    parents = [torch.from_numpy(np.broadcast_to(w.fill_tree(K, spec.F, t + 1),
                                                (B, K + (t + 1) * S)).copy()).to(device)
               for t in range(K)]
    out = torch.empty(B, S, Hq, d, **bf)
    wsn = ssd.ssd_attention_workspace_size(B, S, Hq, Hkv, d, L)
    wsa = torch.empty(max(wsn, 256), dtype=torch.uint8, device=device)
    wss = [ssd.fill_workspace(B, S, V, spec.dtype, spec.F[t], device) for t in range(K)]
    payload = torch.empty(B, S, K, dtype=torch.int32, device=device)
    tok = torch.empty(B, S, dtype=torch.int32, device=device)
    st = torch.zeros(1, dtype=torch.int32, device=device)

    def draw(t):
        ssd.ssd_fill_sample(logits[t], V, spec.F[t], spec.C, spec.T, u[t], tok, t=t, payload=payload,
                            status=st, ws=wss[t])

    def fill():
        for t in range(K):
            ssd.ssd_kv_append(kn[t], vn[t], kc, vc, table, prefix, K + t * S, status=st)
            ssd.ssd_branch_attention(q[t], kc, vc, table, prefix, parents[t], out, status=st, ws=wsa)
            draw(t)

    fill()
    gf = capture_graphs([fill], device)[0]
    gd = capture_graphs([lambda: [draw(t) for t in range(K)]], device)[0]
    for _ in range(3):
        gf.replay()
        gd.replay()
    ms = _time_calls(lambda i: gf.replay(), 20, stream)
    ms_draw = _time_calls(lambda i: gd.replay(), 20, stream)
    draw_bytes = K * B * S * V * 2
    res = {"workload": spec.name, "ms_per_fill": round(ms, 4),
           "branch_tokens_per_s": round(B * S * K / (ms * 1e-3), 1),
           "ms_draws": round(ms_draw, 4), "draw_bytes": draw_bytes,
           "draw_GB/s": round(draw_bytes / (ms_draw * 1e-3) / 1e9, 1),
           "draw_frac_of_hbm_peak": round(draw_bytes / (ms_draw * 1e-3) / 1e9 / hbm_peak, 4),
           "launches_per_fill": f"{K} x (1 append + 1-2 attention + 2 draw)", "status_flags": int(st.item()),
           "steps": f"{K} x (ssd_kv_append, ssd_branch_attention, ssd_fill_sample); "
                    f"{draw_bytes / 1e6:.0f} MB of draft logits per fill (> L2)"}
    del gf, gd, logits, kc, vc
    torch.cuda.empty_cache()
    return res


def bench_tree(ssd, w, device, hbm_peak):
    """Token-tree verification of the 28-node tree over the Llama-3 vocabulary:
    children drawn from the draft at their parent (torch.multinomial, setup
    only); four input copies rotate so the visited rows come from HBM."""
    import torch
    spec = w.llama3_tree()
    B, V, N = spec.B, spec.V, spec.N
    stream = torch.cuda.current_stream(device)
    g = torch.Generator(device=device)
    g.manual_seed(29)
    shape = (B, N + 1, V)
    rank = torch.argsort(torch.rand(shape, generator=g, device=device), dim=-1).float() + 1
    zt = -1.1 * torch.log(rank) + 0.3 * torch.randn(shape, generator=g, device=device)
    del rank
    zd = zt + spec.draft_noise * torch.randn(shape, generator=g, device=device)
    parent1 = w.tree_shape(spec.branching)
    rows = torch.from_numpy(parent1.astype(np.int64) + 1).to(device)
    probs = torch.softmax(zd[:, rows, :] / spec.T, dim=-1)  # [B, N, V]: q at each node's parent
    tok = torch.multinomial(probs.view(B * N, V), 1, generator=g).view(B, N).to(torch.int32)
    del probs
    par = torch.from_numpy(np.broadcast_to(parent1, (B, N)).copy()).to(device)
    ua = torch.rand(B, N, generator=g, device=device)
    ub = torch.rand(B, generator=g, device=device)
    nsets = 4
    sets = [(zt.to(torch.bfloat16), zd.to(torch.bfloat16)) for _ in range(nsets)]
    del zt, zd
    i32 = dict(dtype=torch.int32, device=device)
    acc, path, bon = torch.empty(B, **i32), torch.empty(B, N, **i32), torch.empty(B, **i32)
    st = torch.zeros(1, **i32)

    def call(i):
        t, d = sets[i % nsets]
        ssd.ssd_tree_verify(t, d, V, spec.T, par, tok, ua, ub, acc, path, bon, status=st)

    for i in range(nsets):
        call(i)
    gr = capture_graphs([lambda: [call(i) for i in range(nsets)]], device)[0]
    gr.replay()
    reps = 25
    ms = _time_calls(lambda i: gr.replay(), reps, stream) / nsets
    visited = int(acc.sum().item()) + B  # the rows of every visited node: accepted ones and the root
    alg = visited * 2 * V * 2
    res = {"workload": spec.name, "ms": round(ms, 4), "trees_per_s": round(B / (ms * 1e-3), 1),
           "mean_accept_len": round(visited / B - 1, 3), "algorithmic_bytes": alg,
           "GB/s": round(alg / (ms * 1e-3) / 1e9, 1),
           "frac_of_hbm_peak": round(alg / (ms * 1e-3) / 1e9 / hbm_peak, 4),
           "status_flags": int(st.item()),
           "kernel": "k_tree_walk (one 4-CTA cluster per sequence)",
           "timing": f"CUDA graph of {nsets} calls over input copies, replayed {reps} times"}
    del gr, sets
    torch.cuda.empty_cache()
    return res


def bench_fallback(ssd, w, device, hbm_peak):
    """The miss fallback on the large-batch Qwen-3 batch: the n-gram backup over
    1-8 Ki-token histories (the misses scan their histories; rotating copies
    larger than L2) and the batch plan."""
    import torch
    spec = w.qwen3_histories()
    stream = torch.cuda.current_stream(device)
    h = w.make_histories(spec, seed=21)
    per = h.hist.nbytes
    nsets = max(2, int(np.ceil(1.5 * L2_BYTES / per)) + 1)
    hist0 = torch.from_numpy(h.hist).to(device)
    sets = [hist0.clone() for _ in range(nsets)]
    del hist0
    hl = torch.from_numpy(h.hist_len).to(device)
    slot = torch.from_numpy(h.slot).to(device)
    u = torch.from_numpy(h.u_rand).to(device)
    nxt = torch.empty(spec.B, spec.K, dtype=torch.int32, device=device)
    mp = torch.empty(spec.B, dtype=torch.int32, device=device)
    st = torch.zeros(1, dtype=torch.int32, device=device)

    def call(i):
        ssd.ssd_ngram_backup(sets[i % nsets], hl, spec.n, spec.K, spec.V, u, nxt, slot=slot,
                             match_pos=mp, status=st)

    for i in range(3):
        call(i)
    # one graph holds a call per input copy, so the replays measure the device,
    # not the host's launch rate (one call is a few microseconds)
    g = capture_graphs([lambda: [call(i) for i in range(nsets)]], device)[0]
    g.replay()
    reps = 20
    ms = _time_calls(lambda i: g.replay(), reps, stream) / nsets
    m = mp.cpu().numpy()
    miss = h.slot < 0
    # algorithmic bytes: a miss reads its history from the end down to the match
    # (all of it without one), plus slot, length, uniforms, proposals, positions
    scanned = np.where(m >= 0, h.hist_len - np.maximum(m, 0), h.hist_len)[miss]
    alg = int(4 * scanned.sum() + 4 * spec.B * 3 + 8 * spec.K * miss.sum())
    res = {"workload": spec.name, "ms": round(ms, 4), "misses": int(miss.sum()),
           "matched": int((m[miss] >= 0).sum()), "algorithmic_bytes": alg,
           "GB/s": round(alg / (ms * 1e-3) / 1e9, 1),
           "frac_of_hbm_peak": round(alg / (ms * 1e-3) / 1e9 / hbm_peak, 4),
           "status_flags": int(st.item()), "kernel": "k_ngram_backup (one CTA per sequence)",
           "timing": f"CUDA graph of {nsets} calls over rotating history copies "
                     f"({nsets * per / 1e6:.0f} MB > L2), replayed {reps} times"}
    # the plan: one reduction over the batch
    p = torch.full((spec.B,), 0.9, dtype=torch.float32, device=device)
    e = torch.full((spec.B,), 3.0, dtype=torch.float32, device=device)
    best = torch.empty(1, dtype=torch.int32, device=device)
    thr = torch.empty(2, dtype=torch.float64, device=device)

    def plan(i):
        ssd.ssd_fallback_plan(p, e, 1.0, 0.5, [0.5, 0.02], [2.8, 1.0], throughput=thr, best=best,
                              status=st)

    for i in range(3):
        plan(i)
    gp = capture_graphs([lambda: [plan(i) for i in range(50)]], device)[0]
    gp.replay()
    res["plan_ms"] = round(_time_calls(lambda i: gp.replay(), 20, stream) / 50, 4)
    res["plan_best"] = int(best.item())
    del g, gp, sets
    torch.cuda.empty_cache()
    return res


def bench_other_rounds(ssd, w, device, hbm_peak):
    """The large-batch Qwen-3 round for each Saguaro C (with its cache hit rate),
    the at-scale Llama-3 round and the greedy Llama-3 round (seq-rounds/s)."""
    import torch
    res = {}
    stream = torch.cuda.current_stream(device)
    for spec in (w.qwen3_round(C=1.0), w.qwen3_round(C=0.5), w.qwen3_round(C=0.25),
                 w.llama3_round_at_scale(), w.llama3_round(T=0.0)):
        sets, nsets, per, (ud, ua, ub) = device_round_sets(spec, device, 11)
        out = make_outputs(spec, device)
        ws = ssd.workspace(spec.B, spec.K, spec.V, spec.dtype, spec.F, device)

        def call(i):
            t, d = sets[i % nsets]
            ssd.ssd_round(t, d, spec.V, spec.F, spec.C, spec.T, ud, ua, ub, out["d"],
                          out["accept_len"], out["out_tokens"], out["bonus"], guess=out["guess"],
                          slot=out["slot"], hits=out["hits"], status=out["status"], ws=ws)

        for i in range(3):
            call(i)
        graphs = capture_graphs([lambda i=i: call(i) for i in range(nsets)], device)
        ms = _time_calls(lambda i: graphs[i % nsets].replay(), 50, stream)
        hit_rate = int(out["hits"].item()) / spec.B
        del graphs
        # the same rounds as independent batches on NSTREAMS streams, pipelined
        # on each (as the headline steps): every round in flight reads its own
        # input copy and writes its own outputs and workspace
        psets = [sets[i % nsets] if i < nsets else (sets[0][0].clone(), sets[0][1].clone())
                 for i in range(max(nsets, NBUF))]
        npset = len(psets)
        pouts = [make_outputs(spec, device) for _ in range(NBUF)]
        pws = [ssd.workspace(spec.B, spec.K, spec.V, spec.dtype, spec.F, device) for _ in range(NBUF)]

        def plaunch(i):
            t, d = psets[i % npset]
            o = pouts[i % NBUF]
            ssd.ssd_round(t, d, spec.V, spec.F, spec.C, spec.T, ud, ua, ub, o["d"], o["accept_len"],
                          o["out_tokens"], o["bonus"], guess=o["guess"], slot=o["slot"],
                          hits=o["hits"], status=o["status"], ws=pws[i % NBUF], pipelined=True)

        pchain = stream_chain(plaunch, device)
        pn = int(np.lcm(npset, NBUF))
        pn *= max(1, 32 // pn)
        pchain(0, pn)
        gp = capture_graphs([lambda: pchain(0, pn)], device)[0]
        gp.replay()
        pms = _time_calls(lambda i: gp.replay(), max(3, 64 // pn), stream) / pn
        res[spec.name] = {"ms": round(ms, 4), "seq_rounds_per_s": round(spec.B / (ms * 1e-3), 1),
                          "algorithmic_bytes": per, "C": spec.C, "T": spec.T,
                          "frac_of_hbm_peak": round(per / (ms * 1e-3) / 1e9 / hbm_peak, 4),
                          "hit_rate": round(hit_rate, 4),
                          "streams_ms": round(pms, 4),
                          "streams_seq_rounds_per_s": round(spec.B / (pms * 1e-3), 1),
                          "streams_frac_of_hbm_peak": round(per / (pms * 1e-3) / 1e9 / hbm_peak, 4),
                          "streams_note": f"independent rounds on {NSTREAMS} streams, pipelined on each",
                          "status_flags": int(out["status"].item()) + sum(int(o["status"].item()) for o in pouts)}
        del gp, sets, psets, out, ws, pouts, pws
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline / reference arm)
# ---------------------------------------------------------------------------
def cpu_sample(spec, inp, nseq):
    from speculative_decoding_vocab_gb300 import workloads as w
    idx = np.arange(nseq) % spec.B
    sub = w.RoundSpec(**{**spec.__dict__, "B": nseq})
    return w.RoundInputs(sub, inp.target[idx], inp.draft[idx], inp.u_draft[idx], inp.u_acc[idx],
                         inp.u_bonus[idx], inp.payload[idx])


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        outp = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in outp.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def oracle_rounds(sub, cores: int):
    """The oracle's whole round over the sample's sequences, split over `cores`
    threads (its C functions release the GIL); returns the wall time."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    from speculative_decoding_vocab_gb300 import workloads as w
    B = sub.spec.B
    step = -(-B // cores)
    parts = []
    for lo in range(0, B, step):
        hi = min(B, lo + step)
        sp = w.RoundSpec(**{**sub.spec.__dict__, "B": hi - lo})
        parts.append(w.RoundInputs(sp, sub.target[lo:hi], sub.draft[lo:hi], sub.u_draft[lo:hi],
                                   sub.u_acc[lo:hi], sub.u_bonus[lo:hi], sub.payload[lo:hi]))
    t0 = time.perf_counter()
    if cores == 1:
        oracle.run_round(sub)
    else:
        with ThreadPoolExecutor(max_workers=cores) as ex:
            list(ex.map(oracle.run_round, parts))
    return time.perf_counter() - t0


def cpu_baseline(spec, inp, seconds):
    """The oracle timed on all host cores and on one core, on bounded samples
    of the workload (about `seconds` of one core's work for the one-core
    figure, a full batch of B sequences over all cores)."""
    import oracle
    oracle.build()
    cores = max(1, os.cpu_count() or 1)
    # calibrate on 2 sequences, then time a one-core sample sized to about `seconds`
    per_seq = oracle_rounds(cpu_sample(spec, inp, 2), 1) / 2
    n1 = int(max(2, min(spec.B, seconds / max(per_seq, 1e-6))))
    dt1 = oracle_rounds(cpu_sample(spec, inp, n1), 1)
    nall = spec.B if cores > 1 else n1
    dtall = oracle_rounds(cpu_sample(spec, inp, nall), cores) if cores > 1 else dt1
    return {"value": round(nall / dtall, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{nall} sequences of the {spec.name} round (full V, all K+1 rows; sample + "
                      f"verify + predict + lookup in fp64) over {cores} threads, {dtall:.1f} s",
            "one_core": {"value": round(n1 / dt1, 3), "unit": UNIT, "cores": 1,
                         "sample": f"{n1} sequences, {dt1:.1f} s"},
            "cpu_model": cpu_model(), "nproc": cores}


def bench_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from speculative_decoding_vocab_gb300 import workloads as w
    import oracle
    oracle.build()
    spec = round_spec()
    inp = w.make_round(spec, seed=0)
    cores = max(1, os.cpu_count() or 1)
    nseq = min(spec.B, args.ref_seqs * cores)
    sub = cpu_sample(spec, inp, nseq)
    for _ in range(args.warmup):
        oracle_rounds(cpu_sample(spec, inp, min(nseq, cores)), cores)
    dt = sum(oracle_rounds(sub, cores) for _ in range(args.steps)) / args.steps
    value = nseq / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same workload as our arm)",
        "config": {"workload": spec.name, "B": spec.B, "K": spec.K, "V": spec.V,
                   "input_dtype": "bf16", "T": spec.T, "C": spec.C, "F": list(spec.F),
                   "reference": f"fp64 CPU oracle (oracle/ssd_oracle.c) over {cores} host threads"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{nseq} sequences per step of the {spec.name} round",
                         "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary of this kernel on this
    workload, or None when no summary for the current kernel exists."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d.get(kernel, {}).get(workload)
    except (OSError, ValueError):
        return None


def probe(which):
    """A few calls of one workload and nothing else, for a profiler to capture
    (e.g. ncu -k regex:k_stats -s 2 -c 1 python bench.py --probe round)."""
    import torch
    from speculative_decoding_vocab_gb300 import build
    build.build()
    from speculative_decoding_vocab_gb300 import binding as ssd
    from speculative_decoding_vocab_gb300 import workloads as w
    device = torch.device("cuda", 0)
    if which == "round":
        spec = round_spec()
        inp = w.make_round(spec, seed=0)
        buf = RoundBuffers(spec, inp, device)
        out = make_outputs(spec, device)
        ws = ssd.workspace(spec.B, spec.K, spec.V, spec.dtype, spec.F, device)
        for _ in range(3):
            run_round(ssd, spec, buf, out, ws)
        torch.cuda.synchronize()
        print(json.dumps({"probe": which, "workload": spec.name, "status": int(out["status"].item())}))
        return
    if which == "fill":
        spec = w.llama3_fill()
        B, K, S, V = spec.B, spec.K, spec.S, spec.V
        logits = ssd.tensor(w.fill_step_logits(spec, 3, 1))
        u = torch.from_numpy(w.fill_uniforms(3, 0, 1, B, S)).to(device)
        kn, vn = (ssd.tensor(x) for x in w.fill_step_kv(spec, 3, 1))
        N = K + K * S
        maxb = (spec.L + N + 15) // 16
        table = torch.arange(B * maxb, dtype=torch.int32, device=device).view(B, maxb)
        kc = torch.zeros(B * maxb, spec.Hkv, 16, spec.d, dtype=torch.bfloat16, device=device)
        vc = torch.zeros_like(kc)
        prefix = torch.full((B,), spec.L, dtype=torch.int32, device=device)
        tok = torch.empty(B, S, dtype=torch.int32, device=device)
        payload = torch.empty(B, S, K, dtype=torch.int32, device=device)
        st = torch.zeros(1, dtype=torch.int32, device=device)
        ws = ssd.fill_workspace(B, S, V, spec.dtype, spec.F[1], device)
        for _ in range(3):
            ssd.ssd_kv_append(kn, vn, kc, vc, table, prefix, K + S, status=st)
            ssd.ssd_fill_sample(logits, V, spec.F[1], spec.C, spec.T, u, tok, t=1, payload=payload,
                                status=st, ws=ws)
        torch.cuda.synchronize()
        print(json.dumps({"probe": which, "workload": spec.name, "status": int(st.item())}))
        return
    if which == "tree":
        spec = w.llama3_tree()
        tgt, dft = w.tree_logits(spec, 5)
        parent1 = w.tree_shape(spec.branching)
        B, N = spec.B, spec.N
        rng = np.random.default_rng(6)
        tok = torch.from_numpy(rng.integers(0, 64, size=(B, N)).astype(np.int32)).to(device)
        par = torch.from_numpy(np.broadcast_to(parent1, (B, N)).copy()).to(device)
        ua, ub = w.tree_uniforms(5, 0, B, N)
        i32 = dict(dtype=torch.int32, device=device)
        acc, path, bon = torch.empty(B, **i32), torch.empty(B, N, **i32), torch.empty(B, **i32)
        st = torch.zeros(1, **i32)
        t, d = ssd.tensor(tgt), ssd.tensor(dft)
        for _ in range(3):
            ssd.ssd_tree_verify(t, d, spec.V, spec.T, par, tok, ssd.tensor(ua), ssd.tensor(ub), acc,
                                path, bon, status=st)
        torch.cuda.synchronize()
        print(json.dumps({"probe": which, "workload": spec.name, "status": int(st.item())}))
        return
    if which == "fallback":
        spec = w.qwen3_histories()
        h = w.make_histories(spec, seed=21)
        hist, hl = torch.from_numpy(h.hist).to(device), torch.from_numpy(h.hist_len).to(device)
        slot, u = torch.from_numpy(h.slot).to(device), torch.from_numpy(h.u_rand).to(device)
        nxt = torch.empty(spec.B, spec.K, dtype=torch.int32, device=device)
        st = torch.zeros(1, dtype=torch.int32, device=device)
        for _ in range(3):
            ssd.ssd_ngram_backup(hist, hl, spec.n, spec.K, spec.V, u, nxt, slot=slot, status=st)
        torch.cuda.synchronize()
        print(json.dumps({"probe": which, "workload": spec.name, "status": int(st.item())}))
        return
    spec = w.draft_branch_attention() if which == "attn-draft" else w.verify_attention_at_scale()
    q, kc, vc, table, prefix, parent, N, Nq = device_attention_inputs(spec, device, 7)
    out = torch.empty_like(q)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    wsn = ssd.ssd_attention_workspace_size(spec.B, Nq, spec.Hq, spec.Hkv, spec.d, spec.L)
    aws = torch.empty(max(wsn, 256), dtype=torch.uint8, device=device)
    for _ in range(3):
        ssd.ssd_branch_attention(q, kc, vc, table, prefix, parent, out, status=st, ws=aws)
    torch.cuda.synchronize()
    print(json.dumps({"probe": which, "workload": spec.name, "status": int(st.item())}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seqs", type=int, default=2,
                    help="reference arm: sequences per host core per step (capped at one batch)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-extras", action="store_true", help="skip e2e / attention / other rounds")
    ap.add_argument("--probe", choices=("round", "attn-draft", "attn-verify", "fallback", "tree", "fill"),
                    help="only run a few calls of one workload (for profilers) and exit")
    args = ap.parse_args(argv)
    if args.probe:
        probe(args.probe)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
