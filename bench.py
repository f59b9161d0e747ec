"""Benchmark of the GCA hot path on GB300.

Headline: one training step of the 128M-model workload (B=4 sequences of L=16384 tokens
= 256 chunks of 64, 12 heads x 64, landmark dim 768, k=8, Gumbel noise): causal
landmark retrieval, GCA forward, GCA backward (dQ, dK, dV, dscores) and the
landmark-score backward, all in this library's kernels, timed with CUDA events.
Secondary (same JSON line, key "decode"): decode-time retrieval at 16M context,
B=16 sequences x 262144 past chunk landmarks of dim 768, plus the GCA forward over the
8 retrieved chunks.  Further keys: "prefill_retrieval" (a 1M-token prefill: retrieval on
tensor cores, then with GCA's forward), "block_attention" (window attention and CCA,
forward and backward) and "encoder" (the chunk / landmark encoder).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

With N > 1 (launched by torch.distributed.run) every rank runs its own replica on its
own seed (the path shards by sequence; no collective on the data path) and rank 0
prints the job-wide throughput over the slowest rank's time.
`--impl reference` times the float64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import resource
import statistics
import sys
import threading
import time

import numpy as np

METRIC = "GCA fwd+bwd tokens/s at L=16K; landmark top-k GB/s at 16M ctx (1 GB300)"

def _by_path(fname, modname):
    """A module of the package loaded from its file: importing the package would load the
    CUDA library, which the oracle legs (and the reference arm) must not map."""
    import importlib.util
    if modname in sys.modules:
        return sys.modules[modname]
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "retrieval_sparse_attention_causal_gb300", fname)
    spec = importlib.util.spec_from_file_location(modname, path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod  # dataclasses resolve the module by name
    spec.loader.exec_module(mod)
    return mod


def _workloads():
    """The workload presets (sizes only)."""
    return _by_path("workloads.py", "gca_workloads")


def _synth():
    """The seeded input generators (no method arithmetic, no CUDA library)."""
    return _by_path("synth.py", "gca_synth")


_W = _workloads()
TRAIN_128M, DECODE_16M, PREFILL_1M, TRAIN_350M = _W.TRAIN_128M, _W.DECODE_16M, _W.PREFILL_1M, _W.TRAIN_350M_G2

B, NC, H, DH, D, K = TRAIN_128M.B, TRAIN_128M.n_chunks, TRAIN_128M.H, TRAIN_128M.dh, TRAIN_128M.D, TRAIN_128M.topk
L = TRAIN_128M.L
WORKLOAD = (f"GCA training step, 128M-model shape: B={B}, L={L} ({NC} chunks of 64), H={H} x dh={DH}, "
            f"landmark dim {D}, top-k {K}, Gumbel noise; retrieval + fwd + bwd + landmark grads")
DEC_B, DEC_NC = DECODE_16M.B, DECODE_16M.n_chunks
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(os.path.dirname(os.path.abspath(__file__)), "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML while running."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks"}

    def __init__(self, torch):
        self.samples, self.reasons, self.ok = [], set(), False
        self.max_mhz = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            prop = torch.cuda.get_device_properties(torch.cuda.current_device())
            bus = f"{getattr(prop, 'pci_domain_id', 0):08X}:{prop.pci_bus_id:02X}:{prop.pci_device_id:02X}.0"
            self.h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.nv, self.ok = nv, True
        except Exception:
            self.ok = False

    def _run(self):
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop:
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(0.005)

    def __enter__(self):
        self.stop = False
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        self.stop = True
        if self.ok:
            self.t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "note": "NVML unavailable" if not self.ok else "no sample in window"}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


# ----------------------------------------------------------------------------- flop model
def valid_slots(nC, k):
    """Valid (row, slot) pairs of one sequence in training: row r = c - 1 has min(k, r)
    candidates, for query chunks c = 1 .. nC-1."""
    return sum(min(k, r) for r in range(nC - 1))


def algorithmic_flops(B_, nC, H_, dh, k):
    """Per kernel launch.  Per valid (slot, head) unit: forward 4*64*64*dh (S = QK^T and
    PV); query-side backward 6*64*64*dh (S recompute, dPo = dO V^T, dQ); key-side
    backward 4*64*64*dh (dK, dV; its S/dPo recompute is not counted).  Whole step:
    14*64*64*dh per unit (forward + 2.5x forward)."""
    units = B_ * H_ * valid_slots(nC, k)
    u = 64 * 64 * dh
    return {"gca_fwd": 4 * u * units, "gca_bwd_q": 6 * u * units, "gca_bwd_kv": 4 * u * units,
            "step": 14 * u * units, "units": units}


def algorithmic_bytes(B_, nC, H_, dh, k, esize=2):
    """Per kernel launch, each tensor moved once (query and key chunks alike, nQ = nC):
    forward reads Q, K, V and writes O and the LSE rows; the query side reads Q, dO, K, V
    and the LSE rows and writes dQ and the D rows; the key side reads Q, dO, K, V, the LSE
    and D rows and writes dK, dV."""
    t = B_ * nC * 64 * H_ * dh * esize        # one [B][L][H][dh] tensor
    rows = B_ * nC * H_ * k * 64 * 4          # one f32 [B][nQ][H][k][64] row set
    return {"gca_fwd": 4 * t + rows, "gca_bwd_q": 5 * t + 2 * rows, "gca_bwd_kv": 6 * t + 2 * rows}


# ----------------------------------------------------------------------------- replicas
def max_over_ranks(ms: float, world: int, device=None) -> float:
    """Slowest rank's time (the job's time).  Works with any initialised backend: NCCL
    on GPUs, gloo in the CPU tests."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own replica of the workload (weak
    scaling), so the job does world x units per step in the slowest rank's time."""
    return units_per_rank * world / (ms_per_step / 1e3)


# Measured DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) on this
# workload, from the ncu captures summarised under profiles/. Each figure carries a
# fingerprint of the sources the kernel is built from at capture time; once the sources
# change, the figure no longer describes the kernel and the bench reports null.
KERNEL_SOURCES = {
    "gca_fwd": ("gca_fwd.cu", "tc.cuh", "common.cuh", "waits.cuh"),
    "gca_bwd_q": ("gca_bwd_tc.cu", "tc.cuh", "common.cuh", "waits.cuh"),
    "gca_bwd_kv": ("gca_bwd_tc.cu", "tc.cuh", "common.cuh", "waits.cuh"),
    "retrieve_stream": ("retrieve.cu", "common.cuh"),
    "retrieve_tc": ("retrieve_tc.cu", "tc.cuh", "tc_rows.cuh", "common.cuh"),
}
KNOWN_TRAFFIC = {  # kernel: (bytes per launch, source fingerprint at capture); profiles/gca_tc_kernels_128m.md
    "gca_fwd": (3.8405e+08, "c215969a10653850"),
    "gca_bwd_q": (5.1387e+08, "4f625c47e217a1eb"),
    "gca_bwd_kv": (7.0037e+08, "4f625c47e217a1eb"),
}
# profiles/retrieve_stream_decode_16m.md (B = 2 capture; traffic grows with the number of sequences)
STREAM_TRAFFIC_PER_SEQ = (805500928 / 2, "4efdb061233afa3e")


# profiles/retrieve_tc_prefill.md (8192-chunk capture: the two landmark tensors read once,
# nothing written back past L2; traffic grows with the number of chunks)
PREFILL_TRAFFIC_PER_CHUNK = (25219328 / 8192, "39d775d958d64b7d")


def source_fingerprint(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "retrieval_sparse_attention_causal_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def stream_traffic(nb: int):
    if STREAM_TRAFFIC_PER_SEQ is None:
        return None
    per_seq, fp = STREAM_TRAFFIC_PER_SEQ
    return round(per_seq * nb) if fp == source_fingerprint("retrieve_stream") else None


def prefill_traffic(nc: int):
    per_chunk, fp = PREFILL_TRAFFIC_PER_CHUNK
    return round(per_chunk * nc) if fp == source_fingerprint("retrieve_tc") else None


def measured_traffic(kernel: str, table=None):
    """Traffic per launch for `kernel` if it was captured from the current sources, else None."""
    entry = (table if table is not None else KNOWN_TRAFFIC).get(kernel)
    if entry is None:
        return None
    value, fp = entry
    return value if fp == source_fingerprint(kernel) else None


# ----------------------------------------------------------------------------- GPU arm
def gpu_arm(args):
    import torch
    import torch.distributed as dist

    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import retrieval_sparse_attention_causal_gb300 as gca
    from retrieval_sparse_attention_causal_gb300 import synth

    seed = args.seed + 1000 * rank
    bf = torch.bfloat16
    q = synth.device_normal(seed, synth.S_Q, (B, L, H, DH), 1 / 8, bf)
    k = synth.device_normal(seed, synth.S_K, (B, L, H, DH), 1 / 8, bf)
    v = synth.device_normal(seed, synth.S_V, (B, L, H, DH), 1 / 8, bf)
    do = synth.device_normal(seed, synth.S_DO, (B, L, H, DH), 1 / 8, bf)
    ql = synth.device_normal(seed, synth.S_QL, (B, NC, D), 1.0, bf)
    kl = synth.device_normal(seed, synth.S_KL, (B, NC, D), 1.0, bf)
    ws = gca.Workspace()
    out = dict(
        idx=torch.empty((B, NC, K), dtype=torch.int32, device="cuda"),
        sc=torch.empty((B, NC, K), dtype=torch.float32, device="cuda"),
        o=torch.empty_like(q), lse=torch.empty((B, NC, H, K, 64), dtype=torch.float32, device="cuda"),
        dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
        ds=torch.empty((B, NC, K), dtype=torch.float32, device="cuda"),
        dql=torch.empty((B, NC, D), dtype=torch.float32, device="cuda"),
        dkl=torch.empty((B, NC, D), dtype=torch.float32, device="cuda"))

    def step(i, q=q, k=k, v=v, do=do, ql=ql, kl=kl):
        gca.retrieve_topk(ql, kl, K, 0, True, seed + i, 0, ws=ws, idx=out["idx"], scores=out["sc"])
        gca.gca_forward(q, k, v, out["idx"], out["sc"], shift=1, ws=ws, out=out["o"], lse=out["lse"])
        gca.gca_backward(q, k, v, out["idx"], out["sc"], do, out["lse"], shift=1, ws=ws, dq=out["dq"],
                         dk=out["dk"], dv=out["dv"], dscores=out["ds"])
        gca.scores_backward(ql, kl, out["idx"], out["ds"], ws=ws, dq_out=out["dql"], dk_lmk=out["dkl"])

    def barrier():
        if world > 1:
            dist.barrier()

    def timed(fn, n):
        s = torch.cuda.current_stream()
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for i in range(n):
            fn(i)
        e1.record(s)
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(e0.elapsed_time(e1), world, "cuda")

    for i in range(args.warmup):
        step(i)
    ws.check()
    # The headline: the same step captured once as a CUDA graph (pipeline.TrainGraph) and
    # replayed; replay i draws the noise of seed + i, as step(i) does, and runs the same
    # six launches without the front-end gaps between separately issued ones.
    from retrieval_sparse_attention_causal_gb300 import pipeline
    gws = gca.Workspace()
    graph = pipeline.TrainGraph(lambda sd: pipeline.train_step(q, k, v, ql, kl, do, topk=K, seed_dev=sd, ws=gws),
                                seed=seed)

    def gstep(i):
        graph.replay()

    for i in range(args.warmup):
        gstep(i)
    gws.check()
    with ClockSampler(torch) as clk:
        reps = timed_repeats(timed, gstep, args.steps, args.min_seconds)
    gws.check()
    launches = graph.launches_per_replay * args.steps  # this library's kernels per timed region
    ms_step = statistics.median(reps) / args.steps
    tokens = B * L
    value = job_throughput(tokens, world, ms_step)
    # The same step issued launch by launch (train_step's calls, one by one).
    n0 = gca.launch_count()
    reps_e = timed_repeats(timed, step, args.steps, args.min_seconds)
    ms_eager = statistics.median(reps_e) / args.steps
    eager = {"ms_per_step": round(ms_eager, 4), "tokens_per_s": round(job_throughput(tokens, world, ms_eager), 1),
             "gpu_launches": int((gca.launch_count() - n0) // len(reps_e)), "timed_repeats": len(reps_e)}
    del graph

    # Per-kernel durations: the same loop again with event brackets around each launch.
    gca.profile_begin()
    timed(step, args.steps)
    prof = gca.profile_end()
    fl = algorithmic_flops(B, NC, H, DH, K)
    pk, src = peaks()
    kern = {n: {"launches": c, "avg_ms": t / c} for n, (c, t) in prof.items()}
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0]
    dom_flops = fl.get(dom)
    roof = None
    if dom_flops:
        avg_s = kern[dom]["avg_ms"] / 1e3
        ach = dom_flops / avg_s / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(ach, 2), "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(ach / pk["bf16_tflops"], 4), "traffic": measured_traffic(dom),
                "peak_source": f"{src} bf16 dense (burst)", "flops_per_launch": dom_flops}
        # The same launch against HBM: its algorithmic bytes over the measured copy rate.
        # (Both figures are algorithmic; at this shape the bytes take longer at peak than
        # the flops, i.e. the kernel's arithmetic intensity is below the ridge point.)
        by = algorithmic_bytes(B, NC, H, DH, K).get(dom)
        if by:
            gbs = by / avg_s / 1e9
            roof["hbm_view"] = {"bytes_per_launch": by, "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                                "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                                "flop_per_byte": round(dom_flops / by, 1),
                                "ridge_flop_per_byte": round(pk["bf16_tflops"] * 1e3 / pk["hbm_gbs"], 1)}
    step_tflops = fl["step"] / (ms_step / 1e3) / 1e12

    # The 350M-model step: two retrieval groups, the second group's query landmarks read
    # out of the first group's output.
    t350 = None if args.no_350m else train_350m_leg(args, torch, gca, synth, seed, timed, pk, src, clk_cls=ClockSampler)

    # The rest of the attention block at the same shape: sliding-window self-attention
    # (W = 512) and, as the ablation, chunked cross-attention over the same retrieval.
    blk = None if args.no_block else block_attn_leg(args, torch, gca, q, k, v, out, timed, pk)
    # The chunk / landmark encoder that produces K, V and the key landmarks.
    enc = None if args.no_encoder else encoder_leg(args, torch, gca, synth, timed, pk)
    # Retrieval for a 1M-token prefill (the scoring as a dense tensor-core product).
    pre = None if args.no_prefill else prefill_leg(args, torch, gca, synth, pk, src)

    # End to end through the public API from pinned host buffers.
    e2e = None
    if not args.no_e2e:
        e2e = e2e_leg(args, torch, gca, step_outputs_template=out, inputs=dict(q=q, k=k, v=v, do=do, ql=ql, kl=kl),
                      seed=seed, world=world, timed_barrier=barrier, tokens=tokens)
        # The same, reading back every result of the step (O, dQ, dK, dV, the landmark
        # gradients and the retrieval decision): inputs in, all results out.
        e2e["full_readback"] = e2e_leg(
            args, torch, gca, step_outputs_template=out, inputs=dict(q=q, k=k, v=v, do=do, ql=ql, kl=kl), seed=seed,
            world=world, timed_barrier=barrier, tokens=tokens,
            res=("idx", "sc", "ds", "o", "dq", "dk", "dv", "dql", "dkl"))

    dec = None if args.no_decode else decode_leg(args, torch, gca, synth, seed, pk, src, barrier, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(args.seed, budget_s=args.cpu_seconds)
        side = next_rows_cpu(args.seed)
        if dec is not None and dec.get("offload") is not None:
            dec["offload"]["cpu_baseline"] = side["decode"]
        if blk is not None:
            blk["window"]["cpu_baseline"] = side["window"]
            blk["cca"]["cpu_baseline"] = side["cca"]
            blk["cca"]["backward_cpu_baseline"] = side["cca_backward"]
        if enc is not None:
            enc["cpu_baseline"] = side["encoder"]
        if pre is not None:
            pre["cpu_baseline"] = side["prefill"]
        if t350 is not None:
            t350["cpu_baseline"] = cpu_baseline_350m(args.seed)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1)/8 Q/K/V/dO, N(0,1) landmarks)",
            "config": bench_config(world),
            "step_tflops_algorithmic": round(step_tflops, 2),
            "timed_repeats": {"n": len(reps), "ms_per_step_min": round(min(reps) / args.steps, 4),
                              "ms_per_step_max": round(max(reps) / args.steps, 4),
                              "ms_x_sm_mhz": (round(ms_step * clk.summary()["sm_mhz"], 1)
                                              if clk.summary().get("sm_mhz") else None)},
            "roofline": roof, "gpu_launches": int(launches), "clocks": clk.summary(),
            "step_issue": "one CUDA graph per step (pipeline.TrainGraph)", "eager": eager,
            "kernels": {n: round(x["avg_ms"], 5) for n, x in kern.items()},
            "e2e": e2e, "decode": dec, "train_350m": t350, "block_attention": blk, "encoder": enc,
            "prefill_retrieval": pre, "cpu_baseline": cpu,
        }
        # Compact copies of the secondary headlines, last on the line so that a reader of
        # the line's tail sees them.
        if t350 is not None:
            line["train_350m_headline"] = {
                "metric": "GCA fwd+bwd tokens/s, 350M shape, two groups", "tokens_per_s": t350["tokens_per_s"],
                "ms_per_step": t350["ms_per_step"], "gca_tflops_algorithmic": t350["tflops_algorithmic"],
                "gca_frac_of_bf16_peak": t350["frac_of_bf16_peak"],
                "cpu_baseline_tokens_per_s": (t350.get("cpu_baseline") or {}).get("value")}
        if dec is not None:
            line["decode_headline"] = {
                "metric": "landmark top-k GB/s at 16M ctx", "B": dec["batch"], "GBps": dec["value"],
                "ms_per_retrieval": dec["ms_per_retrieval"], "stream_kernel_GBps": dec["roofline"]["achieved"],
                "frac_of_hbm": dec["roofline"]["frac"], "peak_GBps": dec["roofline"]["peak"],
                "sweep_GBps": {b: x["GBps"] for b, x in dec["batch_sweep"].items()},
                "sweep_frac_of_hbm": {b: x["stream_kernel_frac_of_hbm"] for b, x in dec["batch_sweep"].items()}}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def timed_repeats(timed, fn, steps, min_seconds, max_repeats=500):
    """The K-step timed region (barrier + synchronize on both sides, CUDA events on the
    launching stream), repeated until at least `min_seconds` of timed work have run, so
    that a short step still gives a stable figure.  Returns the milliseconds of every
    repeat; the step time is their median over K."""
    reps = []
    while True:
        reps.append(timed(fn, steps))
        if sum(reps) >= min_seconds * 1e3 or len(reps) >= max_repeats:
            return reps


def bench_config(world):
    """The `config` object of the JSON line: the same for the GPU arm and the oracle arm."""
    return {"workload": WORKLOAD, "global_batch": B * world, "seq_len": L, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (Q, K, V, dO: 4 x 100.7 MB per step)"}


def e2e_leg(args, torch, gca, step_outputs_template, inputs, seed, world, timed_barrier, tokens,
            res=("idx", "sc", "ds")):
    """The training step end to end through the public API: every step copies its inputs
    from pinned host memory to the device and reads its result back: the retrieval
    decision (indices, scores) and the score gradients.  dQ, dK, dV and the landmark
    gradients stay on the device, where an optimizer would consume them.  Copies run on
    their own streams and overlap the previous/next step's compute (inputs and outputs
    are double-buffered); the timed region covers all of it."""
    res = list(res)
    hin = {n: t.cpu().pin_memory() for n, t in inputs.items()}
    din = [{n: torch.empty_like(t) for n, t in inputs.items()} for _ in range(2)]
    dout = [{n: torch.empty_like(t) for n, t in step_outputs_template.items()} for _ in range(2)]
    hout = [{n: torch.empty(step_outputs_template[n].shape, dtype=step_outputs_template[n].dtype, pin_memory=True)
             for n in res} for _ in range(2)]
    cs, h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ws = gca.Workspace()
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer set landed
    ev_comp = [torch.cuda.Event() for _ in range(2)]   # compute on buffer set done
    ev_out = [torch.cuda.Event() for _ in range(2)]    # results of buffer set copied out

    def copy_in(i):
        x = i & 1
        with torch.cuda.stream(h2d):
            h2d.wait_event(ev_comp[x])  # the compute that last read this set is done
            for n in hin:
                din[x][n].copy_(hin[n], non_blocking=True)
            ev_in[x].record(h2d)

    def compute(i):
        x = i & 1
        o, d = dout[x], din[x]
        with torch.cuda.stream(cs):
            cs.wait_event(ev_in[x])
            cs.wait_event(ev_out[x])  # the previous results of this set have been copied out
            gca.retrieve_topk(d["ql"], d["kl"], K, 0, True, seed + i, 0, ws=ws, idx=o["idx"], scores=o["sc"])
            gca.gca_forward(d["q"], d["k"], d["v"], o["idx"], o["sc"], shift=1, ws=ws, out=o["o"], lse=o["lse"])
            gca.gca_backward(d["q"], d["k"], d["v"], o["idx"], o["sc"], d["do"], o["lse"], shift=1, ws=ws,
                             dq=o["dq"], dk=o["dk"], dv=o["dv"], dscores=o["ds"])
            gca.scores_backward(d["ql"], d["kl"], o["idx"], o["ds"], ws=ws, dq_out=o["dql"], dk_lmk=o["dkl"])
            ev_comp[x].record(cs)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_comp[x])
            for n in res:
                hout[x][n].copy_(o[n], non_blocking=True)
            ev_out[x].record(d2h)

    def run(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)

    for e in ev_comp + ev_out:
        e.record(torch.cuda.current_stream())
    run(max(2, args.warmup // 2))
    torch.cuda.synchronize()
    timed_barrier()
    t0 = time.perf_counter()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(h2d)
    cs.wait_stream(h2d)
    d2h.wait_stream(h2d)
    run(args.steps)
    d2h.wait_stream(cs)
    h2d.wait_stream(d2h)
    end.record(h2d)
    torch.cuda.synchronize()
    ms_wall = (time.perf_counter() - t0) * 1e3
    timed_barrier()
    ms = max_over_ranks(start.elapsed_time(end), world, "cuda")
    ms_e = ms / args.steps
    return {"value": job_throughput(tokens, world, ms_e), "unit": "tokens/s", "ms_per_step": ms_e,
            "host_wall_ms_per_step": ms_wall / args.steps,
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin.values()),
            "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hout[0].values()),
            "overlap": "inputs of step i+1 and results of step i-1 move while step i computes",
            "d2h": ", ".join(RESULT_NAMES[n] for n in res) +
                   ("" if "dq" in res else "; dQ/dK/dV and landmark gradients stay on the device")}


RESULT_NAMES = {"idx": "retrieval indices", "sc": "retrieval scores", "ds": "score gradients", "o": "O",
                "dq": "dQ", "dk": "dK", "dv": "dV", "dql": "query-landmark gradients",
                "dkl": "key-landmark gradients"}


def decode_leg(args, torch, gca, synth, seed, pk, src, barrier, world):
    """Decode at 16M context: retrieval over 262144 landmarks per sequence (HBM-bound)
    and the GCA forward over the retrieved chunks; one K/V store shared by the batch."""
    bf = torch.bfloat16
    nb = args.decode_batch
    ql = synth.device_normal(seed, synth.S_QL, (nb, 1, D), 1.0, bf)
    kl = synth.device_normal(seed, synth.S_KL, (nb, DEC_NC, D), 1.0, bf)
    g = torch.Generator().manual_seed(seed)
    jstar = torch.randint(0, DEC_NC, (nb,), generator=g)
    for b in range(nb):
        kl[b, int(jstar[b])] = ql[b, 0]
    # K/V store of 262144 chunks x 64 tokens x 12 x 64 (25.8 GB each): a seeded 1 GiB
    # block tiled across the store.
    blk = synth.device_normal(seed, synth.S_K, (1 << 29,), 1 / 8, bf)
    kst = torch.empty((DEC_NC * 64, H, DH), dtype=bf, device="cuda")
    vst = torch.empty_like(kst)
    for t in (kst, vst):
        f = t.view(-1)
        for s in range(0, f.numel(), blk.numel()):
            n = min(blk.numel(), f.numel() - s)
            f[s:s + n].copy_(blk[:n])
    del blk
    qn = synth.device_normal(seed, synth.S_Q, (nb, 64, H, DH), 1 / 8, bf)
    ws = gca.Workspace()
    idx = torch.empty((nb, 1, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((nb, 1, K), dtype=torch.float32, device="cuda")
    o = torch.empty_like(qn)
    lse = torch.empty((nb, 1, H, K, 64), dtype=torch.float32, device="cuda")

    def retr(i):
        gca.retrieve_topk(ql, kl, K, DEC_NC, False, ws=ws, idx=idx, scores=sc)

    def full(i):
        retr(i)
        gca.gca_forward(qn, kst, vst, idx, sc, shift=0, kv_shared=True, ws=ws, out=o, lse=lse)

    for i in range(args.warmup):
        full(i)
    ws.check()
    ok = bool((idx[:, 0, 0].cpu() == jstar.to(torch.int32)).all())
    s = torch.cuda.current_stream()

    def time_loop(fn, n):
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for i in range(n):
            fn(i)
        e1.record(s)
        torch.cuda.synchronize()
        barrier()
        return e0.elapsed_time(e1) / n

    ms_r = time_loop(retr, args.steps)
    ms_f = time_loop(full, args.steps)
    gca.profile_begin()
    time_loop(retr, args.steps)
    prof = gca.profile_end()
    nbytes = nb * DEC_NC * D * 2
    rows_ms = prof["retrieve_stream"][1] / prof["retrieve_stream"][0]
    ach = nbytes / (rows_ms / 1e3) / 1e9
    # Batch sweep: the same retrieval over the first b sequences (every sequence's 402.7 MB
    # of landmarks is larger than L2, so each call streams from HBM).
    sweep = {}
    for nbs in (1, 2, 4, 8, 16):
        if nbs > nb:
            break
        qs, ks, ids, scs = ql[:nbs], kl[:nbs], idx[:nbs], sc[:nbs]

        def rs(i, qs=qs, ks=ks, ids=ids, scs=scs):
            gca.retrieve_topk(qs, ks, K, DEC_NC, False, ws=ws, idx=ids, scores=scs)

        for i in range(3):
            rs(i)
        ms_b = time_loop(rs, args.steps)
        gca.profile_begin()
        time_loop(rs, args.steps)
        pr = gca.profile_end()
        st_ms = pr["retrieve_stream"][1] / pr["retrieve_stream"][0]
        by = nbs * DEC_NC * D * 2
        sweep[str(nbs)] = {"ms_per_retrieval": round(ms_b, 4), "GBps": round(by / (ms_b / 1e3) / 1e9, 1),
                           "stream_kernel_ms": round(st_ms, 4),
                           "stream_kernel_GBps": round(by / (st_ms / 1e3) / 1e9, 1),
                           "stream_kernel_frac_of_hbm": round(by / (st_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)}
    # Batch 1: a decode step is a few short launches, so the host's launch cost matters.
    # The eager step against the same step captured once as a CUDA graph and replayed.
    from retrieval_sparse_attention_causal_gb300 import pipeline
    q1, ql1, kl1 = qn[:1], ql[:1], kl[:1]
    ws1 = gca.Workspace()

    def eager1(i):
        return pipeline.decode(q1, kst, vst, ql1, kl1, topk=K, kv_shared=True, ws=ws1)

    graph = pipeline.DecodeGraph(q1, kst, vst, ql1, kl1, topk=K, kv_shared=True)

    def graph1(i):
        graph.replay()

    for i in range(args.warmup):
        eager1(i)
        graph1(i)
    ms_e1 = time_loop(eager1, args.steps)
    ms_g1 = time_loop(graph1, args.steps)
    ref1 = eager1(0)
    graph1(0)
    torch.cuda.synchronize()
    batch1 = {"eager_ms_per_decode_chunk": round(ms_e1, 4), "graph_ms_per_decode_chunk": round(ms_g1, 4),
              "graph_equals_eager": bool(torch.equal(ref1["o"], graph.out["o"]) and
                                         torch.equal(ref1["idx"], graph.out["idx"]))}
    ws1.check()
    offload = None
    if not args.no_offload:
        offload = offload_leg(args, torch, gca, kst, vst, qn, ql, kl, ws, o, lse, idx, sc, time_loop)
    del kst, vst, graph
    return {"metric": "landmark top-k GB/s at 16M ctx", "value": round(nbytes * world / (ms_r / 1e3) / 1e9, 1),
            "unit": "GB/s", "batch": nb, "past_chunks": DEC_NC, "landmark_dim": D, "ms_per_retrieval": round(ms_r, 4),
            "ms_per_decode_chunk": round(ms_f, 4), "planted_chunk_found": ok,
            "roofline": {"kernel": "retrieve_stream", "bound": "hbm", "achieved": round(ach, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
                         "traffic": stream_traffic(nb), "peak_source": f"{src} copy bandwidth",
                         "bytes_per_launch": nbytes},
            "kernels": {n: round(t / c, 5) for n, (c, t) in prof.items()}, "batch_sweep": sweep, "batch1": batch1,
            "offload": offload}


def train_350m_leg(args, torch, gca, synth, seed, timed, pk, src, clk_cls):
    """The 350M-model training step: B = 8, L = 16384 (256 chunks), H = 16 x 64, D = 1024,
    k = 8 per group, Gumbel noise, two retrieval groups sharing K/V.  Per step: group 1's
    retrieval and forward; group 2's retrieval over landmarks read straight out of group 1's
    output at every chunk's last token (a strided view, no copy) and its forward; group 2's
    backward (dQ2, dK, dV, dscores); its landmark gradient added into group 1's output
    gradient at those tokens; group 1's backward accumulating into dK, dV; both groups'
    landmark gradients.  Group 1's output gradient buffer holds the upper layers' dO1; its
    chunk-last rows are restored from a saved copy before each step (4 MB), so that every
    step adds group 2's landmark gradient to the same dO1."""
    wl = TRAIN_350M
    b_, nc, h, dh, d, k = wl.B, wl.n_chunks, wl.H, wl.dh, wl.D, wl.topk
    bf = torch.bfloat16
    shape = (b_, wl.L, h, dh)
    q1, q2, kk, vv, do1, do2 = (synth.device_normal(seed, st, shape, wl.qkv_std, bf)
                                for st in (synth.S_Q, synth.S_Q2, synth.S_K, synth.S_V, synth.S_DO, synth.S_DO2))
    q1l, k1l, k2l = (synth.device_normal(seed, st, (b_, nc, d), 1.0, bf) for st in (synth.S_QL, synth.S_KL,
                                                                                     synth.S_KL2))
    from retrieval_sparse_attention_causal_gb300.pipeline import landmark_view
    last = landmark_view(do1)
    last_saved = last.clone()
    ws = gca.Workspace()
    f32, i32 = torch.float32, torch.int32
    o = {n: torch.empty((b_, nc, k), dtype=i32 if n.startswith("idx") else f32, device="cuda")
         for n in ("idx1", "s1", "idx2", "s2", "ds1", "ds2")}
    o.update({n: torch.empty_like(q1) for n in ("o1", "o2", "dq1", "dq2", "dk", "dv")})
    o.update({n: torch.empty((b_, nc, h, k, 64), dtype=f32, device="cuda") for n in ("lse1", "lse2")})
    o.update({n: torch.empty((b_, nc, d), dtype=f32, device="cuda") for n in ("dq1l", "dk1l", "dk2l")})
    q2l = landmark_view(o["o1"])

    def step(i, seed_dev=None):
        last.copy_(last_saved)
        gca.retrieve_topk(q1l, k1l, k, 0, True, seed + i, 0, ws=ws, idx=o["idx1"], scores=o["s1"], seed_dev=seed_dev)
        gca.gca_forward(q1, kk, vv, o["idx1"], o["s1"], shift=1, ws=ws, out=o["o1"], lse=o["lse1"])
        gca.retrieve_topk(q2l, k2l, k, 0, True, seed + i, 1, ws=ws, idx=o["idx2"], scores=o["s2"], seed_dev=seed_dev)
        gca.gca_forward(q2, kk, vv, o["idx2"], o["s2"], shift=1, ws=ws, out=o["o2"], lse=o["lse2"])
        gca.gca_backward(q2, kk, vv, o["idx2"], o["s2"], do2, o["lse2"], shift=1, ws=ws, dq=o["dq2"], dk=o["dk"],
                         dv=o["dv"], dscores=o["ds2"])
        gca.scores_backward(q2l, k2l, o["idx2"], o["ds2"], ws=ws, dq_out=last, accumulate=True, dk_lmk=o["dk2l"])
        gca.gca_backward(q1, kk, vv, o["idx1"], o["s1"], do1, o["lse1"], shift=1, ws=ws, dq=o["dq1"], dk=o["dk"],
                         dv=o["dv"], dscores=o["ds1"], accumulate_dkv=True)
        gca.scores_backward(q1l, k1l, o["idx1"], o["ds1"], ws=ws, dq_out=o["dq1l"], dk_lmk=o["dk1l"])

    for i in range(args.warmup):
        step(i)
    ws.check()
    # Timed as one CUDA graph per step (replay i draws the noise of seed + i), as the
    # 128M step is; the same step issued launch by launch is reported beside it.
    from retrieval_sparse_attention_causal_gb300 import pipeline
    graph = pipeline.TrainGraph(lambda sd: step(0, seed_dev=sd), seed=seed)

    def gstep(i):
        graph.replay()

    for i in range(args.warmup):
        gstep(i)
    with clk_cls(torch) as clk:
        reps = timed_repeats(timed, gstep, args.steps, args.min_seconds)
    ws.check()
    launches = graph.launches_per_replay * args.steps
    ms = statistics.median(reps) / args.steps
    n0 = gca.launch_count()
    reps_e = timed_repeats(timed, step, args.steps, args.min_seconds)
    ms_e = statistics.median(reps_e) / args.steps
    eager = {"ms_per_step": round(ms_e, 4), "tokens_per_s": round(b_ * wl.L / (ms_e / 1e3), 1),
             "gpu_launches": int((gca.launch_count() - n0) // len(reps_e))}
    del graph
    gca.profile_begin()
    timed(step, args.steps)
    prof = gca.profile_end()
    fl = algorithmic_flops(b_, nc, h, dh, k)  # one group
    per_group = {"gca_fwd": fl["gca_fwd"], "gca_bwd_q": fl["gca_bwd_q"], "gca_bwd_kv": fl["gca_bwd_kv"]}
    kern = {}
    for n, (c, t) in prof.items():
        row = {"launches_per_step": c // args.steps, "avg_ms": round(t / c, 5)}
        if n in per_group:
            tf = per_group[n] / (t / c / 1e3) / 1e12
            row["tflops_algorithmic"] = round(tf, 1)
            row["frac_of_bf16_peak"] = round(tf / pk["bf16_tflops"], 4)
        kern[n] = row
    step_fl = 2 * fl["step"]
    tf_step = step_fl / (ms / 1e3) / 1e12
    tokens = b_ * wl.L
    out = {"workload": f"{wl.name}: B={b_}, L={wl.L} ({nc} chunks), H={h} x dh={dh}, landmark dim {d}, top-k {k} "
                       f"per group, Gumbel noise",
           "tokens_per_s": round(tokens / (ms / 1e3), 1), "ms_per_step": round(ms, 4), "steps": args.steps,
           "timed_repeats": len(reps), "gpu_launches": int(launches), "clocks": clk.summary(),
           "step_issue": "one CUDA graph per step (pipeline.TrainGraph)", "eager": eager,
           "flops_algorithmic_per_step": step_fl, "tflops_algorithmic": round(tf_step, 1),
           "frac_of_bf16_peak": round(tf_step / pk["bf16_tflops"], 4),
           "peak_source": f"{src} bf16 dense (burst)", "kernels": kern,
           "l2": "inputs larger than L2 (Q1, Q2, K, V, dO1, dO2: 6 x 268 MB per step)",
           "not_ours": "one 4 MB torch copy per step restores dO1's chunk-last rows"}
    del q1, q2, kk, vv, do1, do2, o
    return out


def block_attn_leg(args, torch, gca, q, k, v, out, timed, pk):
    """Forward and backward of the sliding-window self-attention (W = 512) beside GCA (the
    forward accumulated onto GCA's output as in the attention block), and of CCA (one
    joint softmax over the same retrieved chunks), at the training shape.
    Algorithmic flops count the unmasked (query, key) pairs: 4 dh flops each forward (QK^T,
    PV) and 2.5 times that backward (S recompute, dO V^T, dQ, dK, dV)."""
    W = 512
    o = out["o"].clone()
    lse_w = torch.empty((B, NC, H, 64), dtype=torch.float32, device="cuda")
    o_c = torch.empty_like(q)
    lse_c = torch.empty((B, NC, H, 64), dtype=torch.float32, device="cuda")

    o_w = torch.empty_like(q)
    do = torch.empty_like(q).normal_(0.0, 0.125)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def win(i):
        gca.window_forward(q, k, v, window=W, out=o, lse=lse_w, accumulate=True)

    def win_bwd(i):
        gca.window_backward(q, k, v, o_w, do, lse_w, window=W, dq=dq, dk=dk, dv=dv)

    def cca(i):
        gca.cca_forward(q, k, v, out["idx"], shift=1, out=o_c, lse=lse_c)

    dqc, dkc, dvc = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def cca_bwd(i):
        gca.cca_backward(q, k, v, o_c, do, lse_c, out["idx"], shift=1, dq=dqc, dk=dkc, dv=dvc)

    gca.window_forward(q, k, v, window=W, out=o_w, lse=lse_w)  # the window attention's own output
    for i in range(args.warmup):
        win_bwd(i)
        win(i)
        cca(i)
        cca_bwd(i)
    ms_wb = timed(win_bwd, args.steps) / args.steps
    ms_w = timed(win, args.steps) / args.steps
    ms_c = timed(cca, args.steps) / args.steps
    ms_cb = timed(cca_bwd, args.steps) / args.steps
    t = torch.arange(L, dtype=torch.float64)
    pairs_w = float(torch.clamp(t + 1, max=W).sum()) * B * H
    valid = int((out["idx"][:, : NC - 1] >= 0).sum()) * H  # rows 0..nC-2 feed chunks 1..nC-1
    pairs_c = valid * 64 * 64
    fl_w, fl_c = pairs_w * 4 * DH, pairs_c * 4 * DH
    tok = B * L
    tf = lambda f, ms: f / (ms / 1e3) / 1e12
    peak = pk["bf16_tflops"]
    return {"window": {"window": W, "ms": round(ms_w, 4), "tokens_per_s": round(tok / (ms_w / 1e3), 1),
                       "tflops_algorithmic": round(tf(fl_w, ms_w), 1), "frac_of_bf16_peak": round(tf(fl_w, ms_w) / peak, 3),
                       "accumulated_onto_gca": True, "backward_ms": round(ms_wb, 4),
                       "backward_tflops_algorithmic": round(tf(2.5 * fl_w, ms_wb), 1),
                       "backward_frac_of_bf16_peak": round(tf(2.5 * fl_w, ms_wb) / peak, 3),
                       "fwd_bwd_tokens_per_s": round(tok / ((ms_w + ms_wb) / 1e3), 1)},
            "cca": {"ms": round(ms_c, 4), "tokens_per_s": round(tok / (ms_c / 1e3), 1),
                    "tflops_algorithmic": round(tf(fl_c, ms_c), 1), "frac_of_bf16_peak": round(tf(fl_c, ms_c) / peak, 3),
                    "backward_ms": round(ms_cb, 4),
                    "backward_tflops_algorithmic": round(tf(2.5 * fl_c, ms_cb), 1),
                    "backward_frac_of_bf16_peak": round(tf(2.5 * fl_c, ms_cb) / peak, 3),
                    "fwd_bwd_tokens_per_s": round(tok / ((ms_c + ms_cb) / 1e3), 1)}}


ENC_D, ENC_H = 768, 12  # the 128M model's width: the encoder's rows have d = H * 64 = 768


def prefill_flops(nc, d):
    """2 D flops per (query row, candidate) pair; row i has the i chunks before it."""
    return 2 * d * nc * (nc - 1) // 2


def prefill_leg(args, torch, gca, synth, pk, src):
    """Landmark retrieval for a 1M-token prefill: one sequence of 16384 chunks, D = 768,
    k = 8, no noise; every chunk's query landmark against all earlier chunks' landmarks.
    The two landmark tensors (25 MB each) fit in L2, so a 256 MB buffer is written before
    every call; the call's kernels are timed alone with CUDA events.  Reports the call's
    time, tokens/s (the prefill's tokens per call time) and the scoring kernel's
    algorithmic TFLOP/s against the measured bf16 peak; then the whole prefill (retrieval
    and GCA forward, `with_forward`)."""
    wl = PREFILL_1M
    nc, d, k = wl.n_chunks, wl.D, wl.topk
    ql = synth.device_normal(args.seed, synth.S_QL, (1, nc, d), 1.0, torch.bfloat16)
    kl = synth.device_normal(args.seed, synth.S_KL, (1, nc, d), 1.0, torch.bfloat16)
    ws = gca.Workspace()
    idx = torch.empty((1, nc, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((1, nc, k), dtype=torch.float32, device="cuda")
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")

    def call():
        gca.retrieve_topk(ql, kl, k, 0, False, ws=ws, idx=idx, scores=sc)

    for _ in range(max(3, args.warmup)):
        call()
    ws.check()
    n = 20
    torch.cuda.synchronize()
    gca.profile_begin()
    for _ in range(n):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    prof = gca.profile_end()
    ms = sum(t for _, t in prof.values()) / n
    dom = max(prof.items(), key=lambda kv: kv[1][1])[0]
    dom_ms = prof[dom][1] / prof[dom][0]
    fl = prefill_flops(nc, d)
    ach = fl / (dom_ms / 1e3) / 1e12

    # The whole prefill: the retrieval, then GCA's forward for every chunk over the chunks
    # its predecessor's landmark retrieved (Q/K/V of 1M tokens, 1.6 GB each, past L2).
    shape = (1, wl.L, wl.H, wl.dh)
    q, kk, vv = (synth.device_normal(args.seed, st, shape, wl.qkv_std, torch.bfloat16)
                 for st in (synth.S_Q, synth.S_K, synth.S_V))
    o = torch.empty_like(q)
    lse = torch.empty((1, nc, wl.H, k, 64), dtype=torch.float32, device="cuda")

    def full():
        call()
        gca.gca_forward(q, kk, vv, idx, sc, shift=1, ws=ws, out=o, lse=lse)

    for _ in range(3):
        full()
    ws.check()
    nf = 10
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(nf):
        full()
    e1.record()
    torch.cuda.synchronize()
    ms_full = e0.elapsed_time(e1) / nf
    gca.profile_begin()
    for _ in range(nf):
        full()
    torch.cuda.synchronize()
    fwd_ms = gca.profile_end()["gca_fwd"]
    fwd_ms = fwd_ms[1] / fwd_ms[0]
    af = algorithmic_flops(1, nc, wl.H, wl.dh, k)
    fl_fwd = af["gca_fwd"]
    # Bytes the forward must move at this size: the retrieved K and V chunk of every
    # (slot, head) unit (the 16384 chunks' consumers are spread over the whole sequence,
    # so L2 gives no reuse), plus Q and O of every chunk and head, plus the LSE rows.
    by_fwd = af["units"] * 2 * 64 * wl.dh * 2 + nc * wl.H * 2 * 64 * wl.dh * 2 + nc * wl.H * k * 64 * 4
    del q, kk, vv, o, lse
    return {"workload": f"{wl.name}: B=1, {nc} chunks, landmark dim {d}, top-k {k}, no noise",
            "ms": round(ms, 4), "tokens_per_s": round(wl.L / (ms / 1e3), 1),
            "kernels": {nm: round(t / c, 5) for nm, (c, t) in prof.items()},
            "l2": "256 MB buffer written before every call",
            "with_forward": {"ms": round(ms_full, 4), "tokens_per_s": round(wl.L / (ms_full / 1e3), 1),
                             "gca_fwd_ms": round(fwd_ms, 4),
                             "gca_fwd_tflops_algorithmic": round(fl_fwd / (fwd_ms / 1e3) / 1e12, 1),
                             "gca_fwd_frac_of_bf16_peak": round(fl_fwd / (fwd_ms / 1e3) / 1e12 / pk["bf16_tflops"], 3),
                             "gca_fwd_bytes_algorithmic": by_fwd,
                             "gca_fwd_gbs": round(by_fwd / (fwd_ms / 1e3) / 1e9, 1),
                             "gca_fwd_frac_of_hbm": round(by_fwd / (fwd_ms / 1e3) / 1e9 / pk["hbm_gbs"], 3),
                             "what": "retrieval + GCA forward of every chunk (H 12 x dh 64), next-chunk shift"},
            "roofline": {"kernel": dom, "bound": "tensor", "achieved": round(ach, 2), "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(ach / pk["bf16_tflops"], 4),
                         "traffic": prefill_traffic(nc) if dom == "retrieve_tc" else None,
                         "peak_source": f"{src} bf16 dense (burst)", "flops_per_launch": fl}}


def encoder_flops(nb, nc, d, h):
    """Algorithmic flops of one encoder pass, per kernel: 2 m n k for each GEMM over the
    rows it needs (every row of the layer; token rows only for the K/V transform) and
    4 * 65^2 * 64 per (chunk, head) for the in-chunk attention (QK^T and PV)."""
    m, mt = nb * nc * 65, nb * nc * 64
    return {"enc_qkv": 2 * m * d * 3 * d, "enc_attn": 4 * 65 * 65 * 64 * nb * nc * h, "enc_out": 2 * m * d * d,
            "enc_mlp1": 2 * m * d * 4 * d, "enc_mlp2": 2 * m * 4 * d * d, "enc_kv": 2 * mt * d * 2 * d}


def encoder_leg(args, torch, gca, synth, timed, pk):
    """The chunk / landmark encoder at the training shape (B = 4, 256 chunks of 64 tokens
    plus their LMK rows, d = 768, 12 heads): one pre-LN encoder layer over every chunk and
    the shared K/V transform, with synthetic weights (matrices N(0, 1/fan_in) in bf16,
    biases N(0, 0.02^2), LayerNorm gains 1).  Reports the pass time, tokens/s and per-kernel
    algorithmic TFLOP/s against the measured bf16 peak."""
    d, h = ENC_D, ENC_H
    x = synth.device_normal(args.seed, synth.S_ENC_X, (B, NC * 65, d), 1.0, torch.bfloat16)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(args.seed + 17)
    w = {}
    for n in gca.ENCODER_WEIGHTS:
        if n.startswith("w_"):
            rows, cols = {"w_qkv": (3 * d, d), "w_o": (d, d), "w_1": (4 * d, d), "w_2": (d, 4 * d), "w_kv": (2 * d, d)}[n]
            w[n] = (torch.randn((rows, cols), device="cuda", generator=gen) / cols ** 0.5).to(torch.bfloat16)
        else:
            size = {"b_qkv": 3 * d, "b_1": 4 * d}.get(n, d)
            w[n] = torch.ones(size, device="cuda") if n.endswith("_g") else 0.02 * torch.randn(size, device="cuda", generator=gen)
    ws = gca.Workspace()
    y = torch.empty_like(x)
    kk = torch.empty((B, NC * 64, d), dtype=torch.bfloat16, device="cuda")
    vv = torch.empty_like(kk)
    kl = torch.empty((B, NC, d), dtype=torch.bfloat16, device="cuda")

    def enc(i):
        gca.chunk_encoder(x, w, h, ws=ws, y=y, k=kk, v=vv, k_lmk=kl)

    for i in range(args.warmup):
        enc(i)
    ws.check()
    ms = timed(enc, args.steps) / args.steps
    gca.profile_begin()
    timed(enc, args.steps)
    prof = gca.profile_end()
    fl = encoder_flops(B, NC, d, h)
    kern = {}
    for n, (c, t) in prof.items():
        avg = t / c
        row = {"avg_ms": round(avg, 5)}
        if n in fl:
            row["tflops"] = round(fl[n] / (avg / 1e3) / 1e12, 1)
            row["frac_of_bf16_peak"] = round(fl[n] / (avg / 1e3) / 1e12 / pk["bf16_tflops"], 3)
        kern[n] = row
    total = sum(fl.values())
    return {"B": B, "chunks": NC, "d": d, "heads": h, "ms": round(ms, 4),
            "tokens_per_s": round(B * NC * 64 / (ms / 1e3), 1),
            "tflops_algorithmic": round(total / (ms / 1e3) / 1e12, 1), "kernels": kern}


def offload_leg(args, torch, gca, kst, vst, qn, ql, kl, ws, o, lse, idx, sc, time_loop):
    """Decode with the K/V store in pinned host memory (the inference offload): the same
    store as the device-resident decode copied to a pinned host buffer (2 x 25.8 GB, shared
    by the batch), then per step retrieval over the device landmarks, a GPU gather of the 8
    retrieved chunks per sequence from host memory, and the forward on the compact buffer.
    The output must equal the device-resident decode's bit for bit."""
    nb = qn.shape[0]
    kh = torch.empty(kst.shape, dtype=kst.dtype, pin_memory=True)
    vh = torch.empty(vst.shape, dtype=vst.dtype, pin_memory=True)
    kh.copy_(kst)
    vh.copy_(vst)
    torch.cuda.synchronize()
    kd = torch.empty((nb, K * 64, H, DH), dtype=kst.dtype, device="cuda")
    vd = torch.empty_like(kd)
    il = torch.empty_like(idx)
    o2 = torch.empty_like(o)
    lse2 = torch.empty_like(lse)

    def gather(i):
        gca.gather_chunks(kh, vh, idx, kv_shared=True, ws=ws, k_dst=kd, v_dst=vd, idx_local=il)

    def step(i):
        gca.retrieve_topk(ql, kl, K, DEC_NC, False, ws=ws, idx=idx, scores=sc)
        gather(i)
        gca.gca_forward(qn, kd, vd, il, sc, shift=0, ws=ws, out=o2, lse=lse2)

    for i in range(args.warmup):
        step(i)
    ws.check()
    same = bool(torch.equal(o, o2) and torch.equal(lse, lse2))
    ms_g = time_loop(gather, args.steps)
    ms_s = time_loop(step, args.steps)
    gbytes = nb * K * 2 * 64 * H * DH * 2  # K and V of the retrieved chunks
    del kh, vh
    return {"host_store_GB": round(2 * kst.numel() * kst.element_size() / 1e9, 1), "ms_per_decode_chunk": round(ms_s, 4),
            "gather_ms": round(ms_g, 4), "gather_bytes": gbytes, "gather_GBps": round(gbytes / (ms_g / 1e3) / 1e9, 1),
            "equals_device_decode": same}


def decode_retrieval_only(args):
    """Only the decode-time retrieval (no training step, no K/V store), for ncu captures
    of the landmark stream kernel; prints per-launch timings."""
    import torch
    import retrieval_sparse_attention_causal_gb300 as gca
    from retrieval_sparse_attention_causal_gb300 import synth
    bf = torch.bfloat16
    nb = args.decode_batch
    ql = synth.device_normal(args.seed, synth.S_QL, (nb, 1, D), 1.0, bf)
    kl = synth.device_normal(args.seed, synth.S_KL, (nb, DEC_NC, D), 1.0, bf)
    ws = gca.Workspace()
    idx = torch.empty((nb, 1, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((nb, 1, K), dtype=torch.float32, device="cuda")
    for _ in range(args.warmup + args.steps):
        gca.retrieve_topk(ql, kl, K, DEC_NC, False, ws=ws, idx=idx, scores=sc)
    torch.cuda.synchronize()
    ws.check()
    print(json.dumps({"decode_retrieval_only": True, "batch": nb, "launches": args.warmup + args.steps}))


def prefill_retrieval_only(args):
    """Only the prefill retrieval (one sequence of --prefill-chunks chunks, D = 768, k = 8,
    no noise), for ncu captures of the tensor-core scoring kernel."""
    import torch
    import retrieval_sparse_attention_causal_gb300 as gca
    from retrieval_sparse_attention_causal_gb300 import synth
    nc, d, k = args.prefill_chunks, PREFILL_1M.D, PREFILL_1M.topk
    ql = synth.device_normal(args.seed, synth.S_QL, (1, nc, d), 1.0, torch.bfloat16)
    kl = synth.device_normal(args.seed, synth.S_KL, (1, nc, d), 1.0, torch.bfloat16)
    ws = gca.Workspace()
    idx = torch.empty((1, nc, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((1, nc, k), dtype=torch.float32, device="cuda")
    for _ in range(args.warmup + args.steps):
        gca.retrieve_topk(ql, kl, k, 0, False, ws=ws, idx=idx, scores=sc)
    torch.cuda.synchronize()
    ws.check()
    print(json.dumps({"prefill_retrieval_only": True, "chunks": nc, "launches": args.warmup + args.steps}))


# ----------------------------------------------------------------------------- CPU oracle
def cpu_sample(seed, rows, budget_s=None):
    """The oracle on one sequence of the benchmarked workload, for query chunks
    1..rows (retrieval of their rows, GCA forward and backward, landmark gradients).
    Returns (tokens processed, seconds, cpu seconds)."""
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import oracle.gca_oracle as orc
    synth = _synth()

    x = synth.gca_inputs(seed, 1, NC, NC, H, DH, 1 / 8, "bf16")
    lm = synth.landmark_inputs(seed, 1, NC, NC, D, "bf16")
    r0 = resource.getrusage(resource.RUSAGE_SELF)
    t0 = time.perf_counter()
    idx, sc, _ = orc.retrieve_topk(lm["q_lmk"], lm["k_lmk"], K, 0, True, seed, rows=[(0, i) for i in range(rows)])
    ds_all = np.zeros((1, NC, K))
    done = 0
    for c in range(1, rows + 1):
        sl = slice(c * 64, (c + 1) * 64)
        orc.gca_chunk_forward(x["q"][0, sl], x["k"][0], x["v"][0], idx[0, c - 1], sc[0, c - 1])
        _, _, _, ds = orc.gca_chunk_backward(x["q"][0, sl], x["k"][0], x["v"][0], idx[0, c - 1], sc[0, c - 1],
                                             x["do"][0, sl])
        ds_all[0, c - 1] = ds
        done = c
        if budget_s and time.perf_counter() - t0 > budget_s:
            break
    orc.scores_backward(lm["q_lmk"][:, :done], lm["k_lmk"], idx[:, :done], ds_all[:, :done])
    dt = time.perf_counter() - t0
    r1 = resource.getrusage(resource.RUSAGE_SELF)
    cpu_s = (r1.ru_utime + r1.ru_stime) - (r0.ru_utime + r0.ru_stime)
    return done * 64, dt, cpu_s


def _cpu_timed(fn, min_s=1.5):
    """fn() repeated until min_s seconds have passed: (wall seconds per call, process CPU
    seconds per call, calls)."""
    r0 = resource.getrusage(resource.RUSAGE_SELF)
    t0 = time.perf_counter()
    n = 0
    while n == 0 or time.perf_counter() - t0 < min_s:
        fn()
        n += 1
    dt = time.perf_counter() - t0
    r1 = resource.getrusage(resource.RUSAGE_SELF)
    return dt / n, ((r1.ru_utime + r1.ru_stime) - (r0.ru_utime + r0.ru_stime)) / n, n


def next_rows_cpu(seed):
    """The oracle timed beside each leg of the rest of the method, on a bounded sample of
    that leg's workload (a few seconds each), in the leg's own unit."""
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import oracle.gca_oracle as orc
    synth = _synth()

    cores = len(os.sched_getaffinity(0))
    out = {}

    def entry(value, unit, t, sample):
        dt, cpu_s, n = t
        return {"value": round(value, 3), "unit": unit, "cores": cores, "threads_busy": round(cpu_s / dt, 2),
                "kind": "oracle", "sample": f"{sample}; float64 numpy; {dt:.3f} s wall per call, {n} calls"}

    # Decode at long context: retrieval over 32768 of one sequence's landmarks (1/8 of the
    # 16M-context row) and the forward over the 8 retrieved chunks.
    nk = DEC_NC // 8
    ql = synth.normal(seed, synth.S_QL, (1, 1, D), 1.0, "bf16")
    kl = synth.normal(seed, synth.S_KL, (1, nk, D), 1.0, "bf16")
    qn = synth.normal(seed, synth.S_Q, (64, H, DH), 1 / 8, "bf16")
    kc = synth.normal(seed, synth.S_K, (K * 64, H, DH), 1 / 8, "bf16")
    vc = synth.normal(seed, synth.S_V, (K * 64, H, DH), 1 / 8, "bf16")

    def dec():
        idx, sc, _ = orc.retrieve_topk(ql, kl, K, nk, False, 0)
        orc.gca_chunk_forward(qn, kc, vc, np.arange(K), sc[0, 0])  # on the compact buffer of the 8 chunks
    t = _cpu_timed(dec)
    out["decode"] = entry(nk * D * 2 / t[0] / 1e9, "GB/s", t,
                          f"one sequence: retrieval over {nk} landmarks x {D} (1/8 of the 16M-context row), "
                          f"forward over the {K} retrieved chunks")
    # Window attention W = 512, forward and backward, one sequence of 1024 tokens.
    lw = 1024
    q, k, v, do = (synth.normal(seed, st, (1, lw, H, DH), 1 / 8, "bf16")
                   for st in (synth.S_Q, synth.S_K, synth.S_V, synth.S_DO))
    t = _cpu_timed(lambda: (orc.swa_forward(q, k, v, 512), orc.swa_backward(q, k, v, do, 512)))
    out["window"] = entry(lw / t[0], "tokens/s", t, f"one sequence of {lw} tokens, 12 heads: forward + backward")
    # CCA forward: 16 query chunks of one sequence over its 256 chunks, 8 retrieved each.
    x = synth.gca_inputs(seed, 1, NC, NC, H, DH, 1 / 8, "bf16", with_grad=False)
    idx = np.stack([np.sort(synth.integers(seed, 40 + r, 0, max(r, 1), (K,))) if r >= K else
                    np.concatenate([np.arange(r), -np.ones(K - r, dtype=np.int64)]) for r in range(NC)])[None]
    nq = 16
    t = _cpu_timed(lambda: orc.cca_forward(x["q"], x["k"], x["v"], idx, 1, chunks=[(0, r) for r in range(1, nq + 1)]))
    out["cca"] = entry(nq * 64 / t[0], "tokens/s", t, f"{nq} query chunks of one sequence, {K} retrieved chunks each")
    sl = [slice(c * 64, (c + 1) * 64) for c in range(1, nq + 1)]
    dxo = synth.normal(seed, synth.S_DO, (1, NC * 64, H, DH), 1 / 8, "bf16")
    t = _cpu_timed(lambda: [orc.cca_chunk_backward(x["q"][0, s_], x["k"][0], x["v"][0], idx[0, c], dxo[0, s_])
                            for c, s_ in enumerate(sl)])
    out["cca_backward"] = entry(nq * 64 / t[0], "tokens/s", t,
                                f"{nq} query chunks of one sequence, {K} retrieved chunks each: backward")
    # Chunk encoder: 8 chunks (520 rows) of one sequence at d = 768.
    ne = 8
    xe = synth.encoder_inputs(seed, 1, ne, ENC_D, "bf16")
    pe = synth.encoder_params(seed, ENC_D, "bf16")
    t = _cpu_timed(lambda: orc.chunk_encoder_forward(xe, pe, ENC_H))
    out["encoder"] = entry(ne * 64 / t[0], "tokens/s", t, f"{ne} chunks of one sequence (their {ne * 65} rows), d = {ENC_D}")
    # Prefill retrieval: 16 query rows spread evenly over the 16384-chunk sequence (so that
    # their mean candidate count is the full prefill's), each against all its past chunks.
    pn, ns = PREFILL_1M.n_chunks, 16
    qp = synth.normal(seed, synth.S_QL, (1, pn, D), 1.0, "bf16")
    kp = synth.normal(seed, synth.S_KL, (1, pn, D), 1.0, "bf16")
    rows = [(0, (2 * r + 1) * pn // (2 * ns)) for r in range(ns)]
    t = _cpu_timed(lambda: orc.retrieve_topk(qp, kp, PREFILL_1M.topk, 0, False, 0, rows=rows))
    out["prefill"] = entry(ns * 64 / t[0], "tokens/s", t,
                           f"{ns} query rows spread evenly over one {pn}-chunk sequence, each against all its past chunks")
    return out


def cpu_baseline_350m(seed, budget_s=10.0):
    """The oracle on one sequence of the 350M-model two-group step, for query chunks
    1..n of both groups (group 2's landmark rows from the oracle's own group-1 output at
    those chunks), until the budget runs out.  Returns a cpu_baseline object in tokens/s
    (a token counted once for both groups, as on the GPU)."""
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import oracle.gca_oracle as orc
    synth = _synth()
    wl = TRAIN_350M
    nc, h, dh, d, k = wl.n_chunks, wl.H, wl.dh, wl.D, wl.topk
    x = synth.gca_inputs(seed, 1, nc, nc, h, dh, wl.qkv_std, "bf16")
    q2 = synth.normal(seed, synth.S_Q2, x["q"].shape, wl.qkv_std, "bf16")
    do2 = synth.normal(seed, synth.S_DO2, x["q"].shape, wl.qkv_std, "bf16")
    lm = synth.landmark_inputs(seed, 1, nc, nc, d, "bf16")
    k2l = synth.normal(seed, synth.S_KL2, (1, nc, d), 1.0, "bf16")
    r0 = resource.getrusage(resource.RUSAGE_SELF)
    t0 = time.perf_counter()
    done = 0
    q2l = np.zeros((1, nc, d))
    for c in range(1, nc):
        sl = slice(c * 64, (c + 1) * 64)
        i1, s1, _ = orc.retrieve_topk(lm["q_lmk"], lm["k_lmk"], k, 0, True, seed, 0, rows=[(0, c - 1)])
        o1, _, _ = orc.gca_chunk_forward(x["q"][0, sl], x["k"][0], x["v"][0], i1[0, c - 1], s1[0, c - 1])
        q2l[0, c] = synth.quantize(o1[63].reshape(d), "bf16")
        i2, s2, _ = orc.retrieve_topk(q2l, k2l, k, 0, True, seed, 1, rows=[(0, c - 1)])
        orc.gca_chunk_forward(q2[0, sl], x["k"][0], x["v"][0], i2[0, c - 1], s2[0, c - 1])
        _, _, _, ds2 = orc.gca_chunk_backward(q2[0, sl], x["k"][0], x["v"][0], i2[0, c - 1], s2[0, c - 1],
                                              do2[0, sl])
        _, _, _, ds1 = orc.gca_chunk_backward(x["q"][0, sl], x["k"][0], x["v"][0], i1[0, c - 1], s1[0, c - 1],
                                              x["do"][0, sl])
        orc.scores_backward(q2l[:, c - 1:c], k2l, i2[:, c - 1:c], ds2[None, None])
        orc.scores_backward(lm["q_lmk"][:, c - 1:c], lm["k_lmk"], i1[:, c - 1:c], ds1[None, None])
        done = c
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    r1 = resource.getrusage(resource.RUSAGE_SELF)
    cpu_s = (r1.ru_utime + r1.ru_stime) - (r0.ru_utime + r0.ru_stime)
    return {"value": round(done * 64 / dt, 2), "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
            "threads_busy": round(cpu_s / dt, 2), "kind": "oracle",
            "sample": f"one sequence of the 350M two-group step, query chunks 1..{done} ({done * 64} tokens) of both "
                      f"groups: retrieval rows, forward, backward, landmark gradients, float64 numpy; {dt:.1f} s wall"}


def cpu_baseline(seed, budget_s=20.0):
    tok, dt, cpu_s = cpu_sample(seed, NC - 1, budget_s)
    return {"value": round(tok / dt, 2), "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
            "threads_busy": round(cpu_s / dt, 2), "kind": "oracle",
            "sample": f"one sequence of the workload, query chunks 1..{tok // 64} ({tok} tokens): retrieval rows, "
                      f"GCA forward + backward, landmark gradients, float64 numpy; {dt:.1f} s wall"}


def reference_arm(args):
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    if rank != 0:
        return
    # Size each step so that warm-up + timed steps end within about two minutes.
    per_step = max(0.5, min(6.0, 120.0 / max(1, args.steps + args.warmup)))
    tok, dt, _ = cpu_sample(args.seed, NC - 1, per_step)
    rows = max(1, tok // 64)
    for i in range(args.warmup):
        cpu_sample(args.seed + i, rows)
    tot_t, tot_tok, tot_cpu = 0.0, 0, 0.0
    for i in range(args.steps):
        tk, d, c = cpu_sample(args.seed + i, rows)
        tot_t += d
        tot_tok += tk
        tot_cpu += c
    v = tot_tok / tot_t
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot_t / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(world),
            "cpu_baseline": {"value": round(v, 2), "unit": "tokens/s", "kind": "oracle",
                             "cores": len(os.sched_getaffinity(0)), "threads_busy": round(tot_cpu / tot_t, 2),
                             "sample": f"per step: one sequence, query chunks 1..{rows} ({rows * 64} tokens)"},
            "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--decode-batch", type=int, default=DEC_B)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-offload", action="store_true", help="skip the host-memory K/V store decode")
    ap.add_argument("--no-block", action="store_true", help="skip the window-attention and CCA leg")
    ap.add_argument("--no-encoder", action="store_true", help="skip the chunk / landmark encoder leg")
    ap.add_argument("--no-prefill", action="store_true", help="skip the 1M-token prefill retrieval leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-350m", action="store_true", help="skip the 350M-model two-group training step")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the K-step timed region until this much timed work has run (median reported)")
    ap.add_argument("--decode-retrieval-only", action="store_true",
                    help="run only the 16M-context landmark retrieval (for profiling captures)")
    ap.add_argument("--prefill-retrieval-only", action="store_true",
                    help="run only the prefill landmark retrieval (for profiling captures)")
    ap.add_argument("--prefill-chunks", type=int, default=PREFILL_1M.n_chunks)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
    elif args.decode_retrieval_only:
        decode_retrieval_only(args)
    elif args.prefill_retrieval_only:
        prefill_retrieval_only(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
