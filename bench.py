#!/usr/bin/env python
"""Benchmark: KDA chunked prefill forward on GB300, tokens/s and roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

One step is one ``kda_chunk_fwd`` call over one batch of synthetic inputs
(the whole hot path: gate cumsum, strip products, blocked solve, WY form,
state recurrence and output, final state). Inputs are resident in HBM when
the timed region starts; L2 is flushed (a 256 MiB write) between steps,
outside each step's CUDA events. ``value`` is whole-job tokens/s over all
ranks (weak scaling: every rank processes its own batch; the chains are
independent, so there is no collective on the data path).

Extra keys: ``roofline`` (HBM-bound: algorithmic bytes per launch / mean
launch time, against the measured copy bandwidth), ``e2e`` (the same metric
through the C ABI with pinned host buffers, every host-device transfer inside
the timed region),
``cpu_baseline`` (the fp64 oracle on the host cores, a bounded sample of the
same workload), ``clocks`` (nvidia-smi samples during the timed region) and
``gpu_launches`` (kernels this library launched in the timed region).

``--impl reference`` times the oracle instead (rank 0 only), each step a
bounded sample of the workload sized so the run ends within minutes.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s at T=8192,H=16,K=V=128 bf16; % of roofline (tensor/HBM)"
DECODE_METRIC = "KDA decode tokens/s ({n} sequences x {tn} tokens, H={h}, K=V=128, state in/out)"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "headline_4x2048_H16"
# Context only (another machine): the TPU report's fully optimised headline,
# T=8192 as 4x2048, H=16, K=V=128, BT=64, bf16: 2.62 ms.
PAGES_HEADLINE_TOKENS_PER_S = 8192 / 2.62e-3
# Algorithmic bytes per token-head with o counted as bf16 (q, k, v bf16 + g fp32
# + beta fp32 + o bf16 = 1540 B): the roofline's denominator. This library
# writes o in fp32 (for the parity bar), 256 B more per token-head; that
# widening is reported separately and not credited as useful traffic.
BYTES_PER_TOKEN_HEAD = 3 * 256 + 512 + 4 + 256
O_WIDENING_BYTES_PER_TOKEN_HEAD = 256
STATE_BYTES = 128 * 128 * 4
FLUSH_BYTES = 256 << 20


NORM_GATE_BYTES_PER_TOKEN_HEAD = 256  # the bf16 output gate read by the fused gated RMSNorm


def algorithmic_bytes(T, N, H, with_initial_state, with_final_state=True):
    return T * H * BYTES_PER_TOKEN_HEAD + N * H * STATE_BYTES * (int(with_initial_state) + int(with_final_state))


def algorithmic_flops(seqlens, H, K=128, V=128, BT=64):
    f = 0
    for L in seqlens:
        for c0 in range(0, L, BT):
            n = min(BT, L - c0)
            tri_in, tri_ex = n * (n + 1) // 2, n * (n - 1) // 2
            f += tri_in * 2 * K + tri_ex * 2 * K + tri_ex * 2 * (K + V) + 3 * 2 * n * K * V + tri_in * 2 * V
    return f * H


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples (200 ms) while running; keeps those inside [t0, t1]."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        inside = [s for t, s in self.samples if self.t0 is not None and self.t0 - 0.2 <= t <= self.t1 + 0.2]
        if not inside and self.samples:
            inside = [self.samples[-1][1]]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        mhz, mx, reasons = [], None, set()
        for s in inside:
            try:
                mhz.append(float(s[1]))
                mx = float(s[2])
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, s[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


def gpu_selector(dev) -> str:
    """nvidia-smi ignores CUDA_VISIBLE_DEVICES: address the GPU by UUID."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


KERNEL_SOURCES = {"kda_persistent_kernel": "kda_persistent.cu", "kda_decode_kernel": "kda_decode.cu"}


def source_stamp(kernel):
    from kda_chunked_prefill_gb300 import build as kbuild
    return kbuild.kernel_stamp(KERNEL_SOURCES[kernel])


def traffic_from_profile(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this exact kernel source and workload; otherwise None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        for e in d.get("entries", []):
            if e.get("workload") == workload and e.get("kernel") == kernel and e.get("source_stamp") == source_stamp(kernel):
                return float(e["dram_bytes_per_launch"])
    except (ValueError, KeyError, OSError):
        return None
    return None


def oracle_sample(inp, max_token_heads: int, cores: int):
    """A bounded sample of the workload for the oracle: whole (sequence, head)
    chains, the first heads of every sequence, trimmed to the token budget."""
    import numpy as np
    import torch
    T, H, _ = inp["q"].shape
    lens = inp["seqlens"]
    # heads: enough chains to occupy the cores, within the budget
    per_head = T
    heads = max(1, min(H, max_token_heads // max(per_head, 1)))
    if heads == 1 and per_head > max_token_heads:
        # a prefix of every sequence, one head
        frac = max_token_heads / per_head
        new_lens = [max(1, int(L * frac)) if L else 0 for L in lens]
    else:
        new_lens = list(lens)
    idx = np.concatenate([np.arange(s, s + nl) for s, nl in
                          zip(np.concatenate([[0], np.cumsum(lens)[:-1]]), new_lens)]).astype(np.int64)
    sel = list(range(heads))
    from kda_chunked_prefill_gb300 import inputs as kin
    cu = np.concatenate([[0], np.cumsum(new_lens)]).astype(np.int64)
    s0 = inp["initial_state"]
    args = dict(q=kin.to_f64(inp["q"][idx][:, sel]), k=kin.to_f64(inp["k"][idx][:, sel]),
                v=kin.to_f64(inp["v"][idx][:, sel]), g=kin.to_f64(inp["g"][idx][:, sel]),
                beta=kin.to_f64(inp["beta"][idx][:, sel]), cu=cu,
                s0=None if s0 is None else kin.to_f64(s0[:, sel]), scale=inp["scale"])
    tokens_equiv = int(cu[-1]) * heads / H  # tokens of all heads this sample is worth
    desc = f"{heads} of {H} heads x {len(new_lens)} sequences ({int(cu[-1])} tokens each head)"
    return args, tokens_equiv, desc


def run_oracle(args, threads):
    import oracle
    t = time.perf_counter()
    _, _, used = oracle.kda_recurrence(args["q"], args["k"], args["v"], args["g"], args["beta"], args["cu"],
                                       args["s0"], args["scale"], num_threads=threads, return_threads=True)
    return time.perf_counter() - t, used


def cpu_baseline(inp, target_s: float = 12.0):
    """The oracle as it stands, on the host cores, on a bounded sample."""
    cores = os.cpu_count() or 1
    T, H, _ = inp["q"].shape
    # calibrate on one head (a prefix if long)
    args, tok, _ = oracle_sample(inp, min(T, 4096), cores)
    dt, _ = run_oracle(args, 0)
    rate = tok * H / max(dt, 1e-6)  # token-heads per second
    budget = int(rate * target_s)
    args, tok, desc = oracle_sample(inp, max(1, budget), cores)
    dt, used = run_oracle(args, 0)
    return {"value": tok / dt, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"{desc}; {dt:.2f} s fp64 token recurrence", "seconds": round(dt, 3)}


def bench_reference(a, world, rank):
    """--impl reference: the oracle timed on the host cores, rank 0 only."""
    from kda_chunked_prefill_gb300 import inputs as kin
    if rank != 0:
        return None
    wl = kin.workloads()[a.workload]
    inp = kin.make_workload(wl)
    T, H, _ = inp["q"].shape
    cores = os.cpu_count() or 1
    args, tok, _ = oracle_sample(inp, min(T, 2048), cores)
    dt, _ = run_oracle(args, 0)
    rate = tok * H / max(dt, 1e-6)
    per_step = min(10.0, 120.0 / max(1, a.steps + a.warmup))
    args, tok, desc = oracle_sample(inp, max(1, int(rate * per_step)), cores)
    for _ in range(a.warmup):
        run_oracle(args, 0)
    times, used = [], 0
    for _ in range(a.steps):
        dt, used = run_oracle(args, 0)
        times.append(dt)
    total = sum(times)
    value = tok * a.steps / total
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * total / a.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(a.workload, inp),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": f"each step: {desc}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def workload_config(name, inp):
    T, H, D = inp["q"].shape
    return {"workload": name, "T": int(T), "num_seqs": len(inp["seqlens"]), "num_heads": int(H),
            "head_dim": int(D), "chunk": 64, "subblock": 16,
            "initial_state": "N(0,0.02)" if inp["initial_state"] is not None else "zeros (NULL)",
            "l2": "flushed between steps (256 MiB write outside the step events)",
            "seqlens": inp["seqlens"] if len(inp["seqlens"]) <= 16 else f"{len(inp['seqlens'])} varlen"}


def bench_gpu(a, world, rank, local):
    import torch
    import kda_chunked_prefill_gb300 as kda
    from kda_chunked_prefill_gb300 import inputs as kin

    kda.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    wl = kin.workloads()[a.workload]
    inp = kin.make_workload(wl)
    T, H, D = inp["q"].shape
    N = len(inp["seqlens"])
    d = {key: (None if inp[key] is None else inp[key].to(dev)) for key in
         ("q", "k", "v", "g", "beta", "cu_seqlens", "initial_state")}
    o = torch.empty(d["v"].shape, dtype=torch.float32, device=d["v"].device)
    fs = torch.empty((N, H, D, D), dtype=torch.float32, device=dev)
    norm_kw = {}
    if a.gated_norm:  # the output gate and weight of the fused gated RMSNorm of o
        nrm = kin.make_norm_inputs(T, H, seed=wl.seed + 1000)
        inp["norm_gate"] = nrm["gate"]
        d["norm_gate"] = nrm["gate"].to(dev)
        norm_kw = dict(norm_gate=d["norm_gate"], norm_weight=nrm["weight"].to(dev), norm_eps=nrm["eps"])
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    decode = wl.kind == "decode"

    split_ws = None
    split_L = 0
    if a.split:  # the split-sequence scan, with its planned segment length
        split_L = kda.split_plan(inp["cu_seqlens"], H)
        split_ws = torch.empty(max(1, kda.split_workspace_size(inp["cu_seqlens"], H, 0)), dtype=torch.uint8,
                               device=dev)

    def step():
        if a.split:
            kda.kda_chunk_fwd_split(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], inp["cu_seqlens"],
                                    d["initial_state"], inp["scale"], inp["lower_bound"], o, fs, None, stream,
                                    segment_chunks=0, workspace=split_ws)
        elif decode:
            kda.kda_decode_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], N, d["initial_state"], inp["scale"],
                               inp["lower_bound"], o, fs, None, stream)
        else:
            kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["initial_state"],
                              inp["scale"], inp["lower_bound"], o, fs, None, stream, raw_gates=a.raw_gates,
                              **norm_kw)

    for _ in range(max(3, a.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_selector(dev))
    sampler.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    barrier(world)
    torch.cuda.synchronize()
    sampler.t0 = time.perf_counter()
    for i in range(a.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    sampler.t1 = time.perf_counter()
    sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in ev]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world)
    ms_per_step = 1e3 * total_s / a.steps
    value = T * a.steps * world / total_s

    # e2e through the C ABI with pinned host buffers (every transfer inside the timed region)
    host = {key: (None if inp[key] is None else inp[key].pin_memory()) for key in
            ("q", "k", "v", "g", "beta", "cu_seqlens", "initial_state") + (("norm_gate",) if a.gated_norm else ())}
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    fs_h = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = o_h.numel() * o_h.element_size() + fs_h.numel() * fs_h.element_size()
    e2e_steps = max(3, min(a.steps, 100))

    plain_prefill = not (decode or a.split or a.gated_norm or a.raw_gates)
    if plain_prefill:
        # kda_chunk_fwd_host: the same call on the pinned host buffers, which
        # the kernel reads and writes in place
        hbuf = torch.empty(kda.host_buffer_size(inp["cu_seqlens"], H, inp["initial_state"] is not None, True),
                           dtype=torch.uint8, device=dev)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_step():
        if plain_prefill:
            kda.kda_chunk_fwd_host(host["q"], host["k"], host["v"], host["g"], host["beta"], inp["cu_seqlens"],
                                   host["initial_state"], inp["scale"], inp["lower_bound"], o_h, fs_h, hbuf,
                                   stream=stream, h2d_stream=s_in, d2h_stream=s_out)
            stream.synchronize()
            return
        for key, t in host.items():
            if t is not None:
                d[key].copy_(t, non_blocking=True)
        step()
        o_h.copy_(o, non_blocking=True)
        fs_h.copy_(fs, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    for _ in range(2):
        e2e_step()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    barrier(world)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = T * e2e_steps * world / e2e_s

    # roofline of the (single) kernel: algorithmic bytes per launch / mean launch time
    peaks = load_peaks()
    with_init = inp["initial_state"] is not None
    alg_bytes = algorithmic_bytes(T, N, H, with_init) + (T * H * NORM_GATE_BYTES_PER_TOKEN_HEAD if a.gated_norm else 0)
    mean_launch_s = (sum(step_ms) / len(step_ms)) / 1e3
    achieved_gbs = alg_bytes / mean_launch_s / 1e9
    extra_bytes = T * H * O_WIDENING_BYTES_PER_TOKEN_HEAD
    kernel = "kda_decode_kernel" if decode else "kda_persistent_kernel"
    traffic = None if (a.gated_norm or a.split) else traffic_from_profile(a.workload, kernel)
    if a.split and split_L > 0:
        kernel = "kda_persistent_kernel (two launches) + split combine"
    flops = 0.0 if decode else algorithmic_flops(inp["seqlens"], H)

    out = None
    if rank == 0:
        cpu = None
        if world == 1 and not a.no_cpu_baseline:
            cpu = cpu_baseline(inp)
        clocks = sampler.summary()
        out = {
            "metric": (DECODE_METRIC.format(n=N, tn=T // N, h=H) if decode else METRIC), "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": (value / world / PAGES_HEADLINE_TOKENS_PER_S) if a.workload == DEFAULT_WORKLOAD else None,
            "dtype": ("fp32 (bf16 q, k, v)" if decode else "bf16/fp16 (fp32 accumulate, fp32 state and o)"),
            "data": "synthetic", "config": dict(workload_config(a.workload, inp),
                                                **({"gates": "raw, activated in the kernel"} if a.raw_gates else {}),
                                                **({"output": "gated RMSNorm fused (bf16 gate, fp32 weight, eps 1e-5)"}
                                                   if a.gated_norm else {}),
                                                **({"split_segment_chunks": split_L} if a.split else {})),
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": traffic,
                         "kernel": kernel, "algorithmic_bytes_per_launch": alg_bytes,
                         "extra_bytes_per_launch": extra_bytes,
                         "extra_bytes_note": "o written as fp32 instead of bf16 (not counted in achieved/frac)",
                         "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, burst copy)",
                         "tensor_tflops": flops / mean_launch_s / 1e12,
                         "tensor_frac_of_bf16_peak": flops / mean_launch_s / 1e12 / peaks["bf16_tflops"]},
            "step_ms": {"median": statistics.median(step_ms), "p10": sorted(step_ms)[len(step_ms) // 10],
                        "p90": sorted(step_ms)[(9 * len(step_ms)) // 10]},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps,
                    "call": ("kda_chunk_fwd_host on pinned host buffers (one launch reads the inputs and writes "
                             "o and final_state in host memory over the CPU-GPU link; the byte counts are what "
                             "crosses it)" if plain_prefill else "host-to-device copies, the call, device-to-host copies")},
            "gpu_launches": a.steps * (1 if decode else (5 if split_L > 0 else kda.chunk_fwd_launches(N, T, H))),
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
    return out


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--raw-gates", action="store_true",
                   help="time kda_chunk_fwd_raw_gates (g and beta activated inside the kernel)")
    p.add_argument("--split", action="store_true",
                   help="time kda_chunk_fwd_split (the split-sequence scan, planned segment length)")
    p.add_argument("--gated-norm", action="store_true",
                   help="time kda_chunk_fwd_gated_norm (the gated RMSNorm of o fused into the output store)")
    a = p.parse_args()
    if sum(map(bool, (a.raw_gates, a.gated_norm, a.split))) > 1:
        p.error("--raw-gates, --gated-norm and --split are separate entry points")
    if a.warmup < 3:
        a.warmup = 3
    world, rank, local = dist_setup()
    if a.impl == "reference":
        out = bench_reference(a, world, rank)
    else:
        out = bench_gpu(a, world, rank, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
