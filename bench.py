"""Benchmark of the single-GPU MoE dispatch / grouped FFN / combine path.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME | --config 1..5] [--no-layer] [--cpu-full]

One step is one pass of the hot path over one batch: for the identity-expert
workloads (decode_dispatch_combine, skewed_dispatch_combine) that is
moe_dispatch followed by moe_combine; for the layer workloads it is moe_layer.
The default workload is decode_dispatch_combine: 16 partitions x 128 = 2048
tokens, H = 7168 bf16, 256 experts, top-8, shared expert, per-token mask
Bernoulli(0.9).  Inputs are seeded synthetic data (workloads.py recipe).

Timing: W untimed warm-up steps plus a ~2 s untimed soak (so the clock samples
see the GPU under load), then exactly K steps, each preceded by an untimed L2
flush (a 512 MiB write) and timed with CUDA events on the launching stream;
barrier + synchronize on both sides; max over ranks.  A second pass of K steps
with the library's per-kernel event profiling gives each kernel's average
duration for the roofline.  `timing` adds the median of the K step times and,
for the identity-expert workloads, the step hot in L2 (no flush) and the step
captured once as a CUDA graph and replayed (flushed and hot), so that launch
overhead shows separately; `dispatch_quant` times moe_dispatch_quant (int8 rows
and per-row scales) on the same inputs.  `e2e` repeats the step through the same C ABI
calls with pinned host inputs: host->device copies, the step, and the
device->host copy of the output are inside the timed region.  The same copy
loop is then timed without the kernels (`copies_only_ms_per_step`): the host
link's own time for a step's bytes, which bounds the end-to-end rate.

Under torchrun (N > 1) every rank runs the same workload on its own GPU with
its own seed and no collective on the data path (weak scaling, replicas).

The identity-expert workloads also report the full layer workload (8 x 2048
tokens, 128 experts, FFN 4096) as a secondary item, `full_layer`: tokens/s,
the grouped GEMMs against the measured bf16 peaks (burst and sustained), its
own clock samples and oracle baseline (--no-layer skips it).

cpu_baseline and --impl reference time the CPU oracle as it stands on every
host core (its threaded drivers only split tokens over threads): the whole
identity-expert workload per step, or a few tokens per thread through the
whole layer; under torchrun only rank 0 runs the reference arm.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from combine_route_count_prefix_gb300 import workloads as wl  # noqa: E402

METRIC = "MoE layer tokens/s; dispatch+combine HBM GB/s (% of peak), 1xGB300"
FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_dispatch_combine", choices=list(wl.WORKLOADS))
    ap.add_argument("--config", type=int, choices=sorted(wl.CONFIGS), default=None,
                    help="the benchmark configuration by number (1-5); overrides --workload")
    ap.add_argument("--no-layer", action="store_true",
                    help="skip the full layer workload (full_layer) that the identity-expert "
                         "workloads report as a secondary line item")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--tokens-per-partition", type=int, default=0,
                    help="override M (tokens per partition) of the workload")
    ap.add_argument("--experts", type=int, default=0, help="override E of the workload")
    ap.add_argument("--soak", type=float, default=2.0,
                    help="seconds of untimed steps before the timed region (clock samples)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--peak-probes", action="store_true",
                    help="build and run the probes (mma.sync int8, HBM copy, host link) and "
                         "print them beside the measured peaks; one JSON line")
    ap.add_argument("--cpu-full", action="store_true",
                    help="one GPU step, then the oracle over the whole workload on every host "
                         "core (timed) and every output token compared with it; one JSON line")
    ap.add_argument("--ffn-path", default="auto", choices=["auto", "large", "small", "large_pair"],
                    help="grouped-GEMM kernels of the layer workloads (auto: small-batch "
                         "kernels when T*K <= 128*E)")
    args = ap.parse_args()
    if args.config is not None:
        args.workload = wl.CONFIGS[args.config]
    return args


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        pmax = max(r["power"] for r in rows)
        load = [r for r in rows if r["power"] >= 0.5 * pmax] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(r["sm"] for r in load),
                    sm_max_mhz=max(r["smax"] for r in rows), reasons=sorted(reasons),
                    samples=len(rows), samples_under_load=len(load),
                    power_w_max=pmax)


# ------------------------------------------------------------------ helpers
def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "combine_route_count_prefix_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:12]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch recorded from an ncu capture in profiles/traffic.md,
    valid only while the kernel's source file is unchanged (hash match)."""
    p = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(p):
        return None
    for line in open(p):
        m = re.match(r"\|\s*(\S+)\s*\|\s*(\S+)\s*\|\s*(\S+)\s*\|\s*(\S+)\s*\|\s*([0-9.eE+]+)\s*\|", line)
        if not m or m.group(1) != kernel or m.group(2) != workload:
            continue
        src, h = m.group(3), m.group(4)
        if source_hash(src) != h:
            return None
        return float(m.group(5))
    return None


def bf16_dev(a, dev):
    import torch
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def identity_bytes(w, inp, R):
    """Algorithmic HBM bytes of dispatch and of combine (each byte the method
    must move once)."""
    T, K, H = w.num_tokens, w.topk, w.hidden
    mask = inp["mask"]
    act = np.ones((T, K), bool)
    if mask is not None:
        act &= (mask[:, None] if mask.ndim == 1 else mask).astype(bool)
    tok_active = int(act.any(axis=1).sum())
    mask_bytes = 0 if mask is None else mask.size
    row = H * 2
    dispatch_rows = tok_active * row + R * row + T * K * 4          # x once, rows once, route_row
    routing = T * K * 4 + mask_bytes + T * K * 4 + R * 12           # ids + mask, route_row, assist
    combine = R * row + T * row * (2 if inp["shared"] is not None else 1) + T * K * 8 + mask_bytes
    return dict(dispatch_rows=dispatch_rows, routing=routing, combine=combine,
                total=dispatch_rows + routing + combine)


def layer_row_bytes(w, inp, R):
    """HBM bytes of the layer's row kernels per launch, two ways: with each
    quantisation code counted as the int8 byte the method defines, and as the
    bytes the kernels move (codes stored as fp16 images, the GEMMs' operand
    format).  quant_scatter: x once per active token, the codes and per-row
    scales of R rows, route_row; quant2: g (fp32) read, codes and scales
    written; combine: y rows (bf16), the shared term, the output, route_row
    and probabilities."""
    T, K, H, Nh = w.num_tokens, w.topk, w.hidden, w.ffn // 2
    mask = inp["mask"]
    act = np.ones((T, K), bool)
    if mask is not None:
        act &= (mask[:, None] if mask.ndim == 1 else mask).astype(bool)
    tok_active = int(act.any(axis=1).sum())
    mask_bytes = 0 if mask is None else mask.size
    idx = T * K * 4 + mask_bytes
    comb = R * H * 2 + T * H * 2 * (2 if inp["shared"] is not None else 1) + T * K * 8 + mask_bytes
    return {
        "quant_scatter": {"int8_codes": tok_active * H * 2 + R * H + R * 4 + idx,
                          "as_moved": tok_active * H * 2 + R * H * 2 + R * 4 + idx},
        "quant2": {"int8_codes": R * Nh * 4 + R * Nh + R * 4,
                   "as_moved": R * Nh * 4 + R * Nh * 2 + R * 4},
        "combine": {"int8_codes": comb, "as_moved": comb},
    }


def row_kernel_fracs(row_bytes, prof, hbm_gbs):
    """Each profiled row kernel's mean launch time and its two byte counts
    (layer_row_bytes) against the HBM peak."""
    out = {}
    for name, nbytes in row_bytes.items():
        if name not in prof:
            continue
        k_us = prof[name][1] / prof[name][0] * 1e3
        out[name] = {"us": round(k_us, 3), "bytes_int8_codes": nbytes["int8_codes"],
                     "bytes_as_moved": nbytes["as_moved"],
                     "frac_int8_codes": nbytes["int8_codes"] / (k_us * 1e-6) / 1e9 / hbm_gbs,
                     "frac_as_moved": nbytes["as_moved"] / (k_us * 1e-6) / 1e9 / hbm_gbs}
    return out


def max_over_ranks(v, dist, device=None):
    """Largest value of v over all ranks (v itself without a process group)."""
    if dist is None:
        return float(v)
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank, world, ms_per_step):
    """Weak scaling: every rank processes its own tokens_per_rank per step;
    the job's rate is all ranks' tokens over the slowest rank's step time."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


# ------------------------------------------------------------------ reference arm (CPU oracle)
def host_cores():
    """Cores this process may run on (what `nproc` reports)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(w, inp, seed, threads):
    """A bounded sample of the workload for the CPU oracle on `threads`
    threads: returns (step callable returning tokens processed, description).
    Identity-expert workloads run whole (routing in one sequential pass, the
    row gather and the combine split by tokens over the threads); the layer
    workloads run a few tokens per thread through the whole layer."""
    import oracle
    oracle.build()
    if w.identity:
        T = w.num_tokens

        def step():
            oracle.dispatch_combine_identity(inp["x"], inp["ids"], inp["probs"], w.num_experts,
                                             w.num_partitions, mask=inp["mask"],
                                             shared=inp["shared"], threads=threads)
            return T
        return step, (f"the whole workload per step ({T} tokens, all {w.num_partitions} "
                      f"partitions): routing, row gather and combine, {threads} threads")
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=seed, threads=threads)
    n_tok = 2 * threads
    g = np.random.default_rng(seed + 7)
    state = {"i": 0}
    order = g.permutation(w.num_tokens).astype(np.int64)

    def step():
        i = state["i"]
        tok = np.sort(order[i: i + n_tok])
        state["i"] = (i + n_tok) % max(1, w.num_tokens - n_tok)
        oracle.layer_tokens(inp["x"], inp["ids"], inp["probs"], W1, S1, W2, S2, tok,
                            mask=inp["mask"], shared=inp["shared"], threads=threads)
        return n_tok
    return step, (f"{n_tok} tokens per step through the whole layer (each token's "
                  f"{w.topk} expert FFNs and combine; weights drawn by the input recipe), "
                  f"{threads} threads")


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = select_workload(args)
    inp = wl.make_inputs(w, seed=args.seed)
    threads = host_cores()
    step, sample = oracle_sample(w, inp, args.seed, threads)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    units = 0
    for _ in range(args.steps):
        units += step()
    dt = time.perf_counter() - t0
    value = units / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                         "nproc": host_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bf16_errors(got_bits, ref_bits):
    """Output errors in bf16 ulps taken at the oracle value's magnitude."""
    g = wl.bf16_bits_to_f32(got_bits).astype(np.float64)
    r = wl.bf16_bits_to_f32(ref_bits).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -126))) - 7)
    e = np.abs(g - r) / ulp
    tok_max = e.max(axis=1) if e.size else np.zeros(0)
    return {"tokens": int(got_bits.shape[0]), "max_ulp": float(e.max()) if e.size else 0.0,
            "rel_l2": float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)),
            "tokens_within_2_ulp": int((tok_max <= 2.0).sum()),
            "tokens_bit_exact": int((got_bits == ref_bits).all(axis=1).sum())}


def run_peak_probes():
    """The legacy int8 tensor instruction (mma.sync m16n8k32 s8, exact int32
    accumulation), a streaming copy and the host link (DMA in, out and both
    ways, and a kernel reading pinned host memory), measured on this GPU,
    beside the measured bf16 and HBM peaks the rooflines use."""
    import subprocess
    from combine_route_count_prefix_gb300 import build as bld
    src = os.path.join(ROOT, "combine_route_count_prefix_gb300", "probes", "peak_probes.cu")
    exe = os.path.join(bld.BUILD, "peak_probes")
    os.makedirs(bld.BUILD, exist_ok=True)
    r = subprocess.run([bld.nvcc(), *bld.ARCH, "-O3", "-std=c++17", "-o", exe, src],
                       capture_output=True, text=True)
    if r.returncode:
        raise RuntimeError(r.stderr[-2000:])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    if r.returncode:
        raise RuntimeError(r.stderr[-2000:])
    probe = json.loads(r.stdout.strip().splitlines()[-1])
    pk = peaks()
    line = {"peak_probes": probe, "measured_peaks": pk,
            "mma_sync_s8_vs_bf16_peak": probe["mma_sync_s8_tops"] / pk["bf16_tflops"],
            "copy_vs_hbm_peak": probe["copy_gbs"] / pk["hbm_gbs"]}
    print(json.dumps(line), flush=True)


def run_cpu_full(args):
    """The oracle once over the whole workload on every host core, timed, and
    every output token of one GPU step (the benchmark's launch configuration)
    compared with it."""
    import torch
    import oracle
    from combine_route_count_prefix_gb300 import binding as B
    B.lib()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = select_workload(args)
    T = w.num_tokens
    inp = wl.make_inputs(w, seed=args.seed)
    threads = host_cores()
    oracle.build()
    if w.identity:
        path = IdentityPath(B, w, inp, dev)
        path.step()
        torch.cuda.synchronize()
        got = path.out.view(torch.int16).cpu().numpy().view(np.uint16)
        del path
        t0 = time.perf_counter()
        _, _, ref = oracle.dispatch_combine_identity(
            inp["x"], inp["ids"], inp["probs"], w.num_experts, w.num_partitions,
            mask=inp["mask"], shared=inp["shared"], threads=threads)
        dt = time.perf_counter() - t0
        what = "routing, row gather and combine"
    else:
        path = LayerPath(B, w, inp, dev, args.seed, args.ffn_path)
        torch.cuda.synchronize()
        status = B.read_device_status(path.ws)
        got = path.out.view(torch.int16).cpu().numpy().view(np.uint16)
        del path
        torch.cuda.empty_cache()
        W1, S1, W2, S2 = wl.all_expert_weights(w, seed=args.seed, threads=threads)
        t0 = time.perf_counter()
        ref, ovf = oracle.layer_tokens(inp["x"], inp["ids"], inp["probs"], W1, S1, W2, S2,
                                       np.arange(T, dtype=np.int64), mask=inp["mask"],
                                       shared=inp["shared"], threads=threads)
        dt = time.perf_counter() - t0
        assert not ovf and status == 0
        what = f"every token through the whole layer ({w.topk} expert FFNs each, then combine)"
    line = {"cpu_full": {"workload": w.name, "config": workload_config(w), "kind": "oracle",
                         "value": T / dt, "unit": "tokens/s", "seconds": dt, "cores": threads,
                         "nproc": host_cores(), "run": f"the whole workload once: {what}"},
            "parity_full": bf16_errors(got, ref)}
    print(json.dumps(line), flush=True)


def workload_config(w):
    return {"workload": w.name, "tokens": w.num_tokens, "partitions": w.num_partitions,
            "hidden": w.hidden, "experts": w.num_experts, "topk": w.topk, "ffn": w.ffn,
            "mask": ["none", "per-token", "per-route"][w.mask_kind],
            "shared_expert": w.has_shared, "routing": w.routing,
            "l2": "flushed before every timed step (512 MiB write)"}


# ------------------------------------------------------------------ our arm
def cpu_baseline_sample(w, inp, seed, budget_s=10.0):
    """The oracle as it stands, on every host core, on a bounded sample of the
    same workload, repeated for about budget_s seconds."""
    threads = host_cores()
    step, sample = oracle_sample(w, inp, seed, threads)
    step()                                      # first call: library load, page-in
    t0 = time.perf_counter()
    units = reps = 0
    while True:
        units += step()
        reps += 1
        dt = time.perf_counter() - t0
        if dt > budget_s or reps >= 2000:
            break
    return {"value": units / dt, "unit": "tokens/s", "cores": threads, "nproc": host_cores(),
            "kind": "oracle", "sample": f"{sample}, repeated {reps}x over {dt:.1f} s"}


def select_workload(args):
    w = wl.WORKLOADS[args.workload]
    over = {}
    if args.tokens_per_partition:
        over["tokens_per_partition"] = args.tokens_per_partition
    if args.experts:
        over["num_experts"] = args.experts
    if over:
        suffix = "".join(f"_{k[:1]}{v}" for k, v in over.items())
        w = dataclasses.replace(w, name=w.name + suffix, **over)
    return w


def device_weights(w, dev, seed):
    """Expert weights of the input recipe (the same values the tests use),
    drawn on the host cores in parallel and copied to the device."""
    import torch
    W1, S1, W2, S2 = wl.all_expert_weights(w, seed=seed, threads=0)
    return (torch.from_numpy(W1).to(dev), torch.from_numpy(S1).to(dev),
            torch.from_numpy(W2).to(dev), torch.from_numpy(S2).to(dev))


class IdentityPath:
    """moe_dispatch + moe_combine with an identity expert (y = dispatched rows)."""

    def __init__(self, B, w, inp, dev):
        import torch
        self.B, self.w, self.inp = B, w, inp
        T, P, H, E = w.num_tokens, w.num_partitions, w.hidden, w.num_experts
        self.x = bf16_dev(inp["x"], dev)
        self.ids = torch.from_numpy(inp["ids"]).to(dev)
        self.probs = torch.from_numpy(inp["probs"]).to(dev)
        self.mask = None if inp["mask"] is None else torch.from_numpy(inp["mask"]).to(dev)
        self.shared = bf16_dev(inp["shared"], dev)
        self.d = B.dispatch(self.x, self.ids, E, P, mask=self.mask)
        self.ws = self.d["workspace"]
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

    def step(self, x=None, ids=None, probs=None, mask=None, shared=None, out=None):
        w, B, d = self.w, self.B, self.d
        x = self.x if x is None else x
        ids = self.ids if ids is None else ids
        probs = self.probs if probs is None else probs
        mask = self.mask if mask is None else mask
        shared = self.shared if shared is None else shared
        B.dispatch(x, ids, w.num_experts, w.num_partitions, mask=mask, ws=self.ws, out=d)
        B.combine(d["expand_x"], d["route_row"], probs, w.num_experts, w.num_partitions,
                  mask=mask, shared=shared, out=self.out if out is None else out)

    def rows(self):
        return int(self.d["expert_offsets"][-1].item())

    def roofline(self, prof, pk):
        by = identity_bytes(self.w, self.inp, self.rows())
        dom = max(("dispatch_rows", "combine"), key=lambda k: prof.get(k, (1, 0.0))[1])
        n, ms = prof[dom]
        us = ms / n * 1e3
        achieved = by[dom] / (us * 1e-6) / 1e9
        extra = {"hbm_gbs": None, "hbm_frac_of_peak": None}
        return dict(bound="hbm", kernel=dom, achieved=achieved, peak=pk["hbm_gbs"], unit="GB/s",
                    frac=achieved / pk["hbm_gbs"], traffic=recorded_traffic(dom, self.w.name),
                    algorithmic_bytes=by[dom],
                    algorithmic_unit="bytes per launch (each byte the step must move once)",
                    peak_source=pk["source"] + " hbm_gbs (burst copy)"), by["total"], extra

    def dtype(self):
        return "bf16"


class LayerPath:
    """moe_layer: routing, per-token int8 quantisation, grouped GEMM1 + SwiGLU,
    second quantisation, grouped GEMM2 + dequant, combine."""

    def __init__(self, B, w, inp, dev, seed, ffn_path="auto"):
        import torch
        self.B, self.w, self.inp = B, w, inp
        T, P, H, E, K, N = (w.num_tokens, w.num_partitions, w.hidden, w.num_experts, w.topk,
                            w.ffn)
        self.x = bf16_dev(inp["x"], dev)
        self.ids = torch.from_numpy(inp["ids"]).to(dev)
        self.probs = torch.from_numpy(inp["probs"]).to(dev)
        self.mask = None if inp["mask"] is None else torch.from_numpy(inp["mask"]).to(dev)
        self.shared = bf16_dev(inp["shared"], dev)
        self.shape = B.make_shape(T, P, H, E, K, N, w.mask_kind, w.has_shared, ffn_path=ffn_path)
        w1, self.s1, w2, self.s2 = device_weights(w, dev, seed)
        (self.o1, self.w1p), (self.o2, self.w2p) = B.pack_weights(self.shape, w1, w2)
        del w1, w2
        torch.cuda.synchronize()
        self.out, self.ws = B.layer(self.shape, self.x, self.ids, self.probs, self.w1p, self.s1,
                                    self.w2p, self.s2, mask=self.mask, shared=self.shared)

    def step(self, x=None, ids=None, probs=None, mask=None, shared=None, out=None):
        self.B.layer(self.shape, self.x if x is None else x, self.ids if ids is None else ids,
                     self.probs if probs is None else probs, self.w1p, self.s1, self.w2p, self.s2,
                     mask=self.mask if mask is None else mask,
                     shared=self.shared if shared is None else shared, ws=self.ws,
                     out=self.out if out is None else out)

    def rows(self):
        return int(self.B.stage_views(self.shape, self.ws)["expert_offsets"][-1].item())

    def roofline(self, prof, pk):
        w = self.w
        R = self.rows()
        H, N, Nh = w.hidden, w.ffn, w.ffn // 2
        small = "gemm1_swiglu_small" in prof
        sfx = "_small" if small else ("_pair" if "gemm1_swiglu_pair" in prof else "")
        g1, g2 = "gemm1_swiglu" + sfx, "gemm2_dequant" + sfx
        fl = {g1: 2.0 * R * H * N, g2: 2.0 * R * Nh * H}
        dom = max(fl, key=lambda k: prof.get(k, (1, 0.0))[1])
        n, ms = prof[dom]
        us = ms / n * 1e3
        extra = {"ffn_path": "small" if small else ("large_pair" if sfx else "large"),
                 "gemm_tflops": {k: fl[k] / (prof[k][1] / prof[k][0] * 1e-3) / 1e12 for k in fl},
                 "status": self.B.read_device_status(self.ws)}
        extra["row_kernels"] = row_kernel_fracs(layer_row_bytes(w, self.inp, R), prof, pk["hbm_gbs"])
        step_bytes = None
        if small:
            # few rows per expert: reading the int8 weights of every expert that
            # has rows bounds the time.  Algorithmic bytes per launch: those
            # weights, the int8 operand rows, and the stage's output.
            counts = self.B.stage_views(self.shape, self.ws)["expert_token_nums"].cpu().numpy()
            e_act = int((counts > 0).sum())
            by = {g1: e_act * N * H + R * H + R * Nh * 4, g2: e_act * H * Nh + R * Nh + R * H * 2}
            extra["gemm_hbm_gbs"] = {k: by[k] / (prof[k][1] / prof[k][0] * 1e-3) / 1e9 for k in by}
            achieved = by[dom] / (us * 1e-6) / 1e9
            return dict(bound="hbm", kernel=dom, achieved=achieved, peak=pk["hbm_gbs"], unit="GB/s",
                        frac=achieved / pk["hbm_gbs"], traffic=recorded_traffic(dom, w.name),
                        algorithmic_bytes=by[dom],
                        algorithmic_unit="int8 weights of the experts with rows + int8 rows + "
                        "stage output (g fp32 / y bf16) bytes per launch",
                        peak_source=pk["source"] + " hbm_gbs"), step_bytes, extra
        achieved = fl[dom] / (us * 1e-6) / 1e12
        extra["gemm_frac"] = {k: {"of_sustained": v / pk["bf16_tflops_sustained"],
                                  "of_burst": v / pk["bf16_tflops"]}
                              for k, v in extra["gemm_tflops"].items()}
        return dict(bound="tensor", kernel=dom, achieved=achieved,
                    peak=pk["bf16_tflops_sustained"], unit="TFLOP/s",
                    frac=achieved / pk["bf16_tflops_sustained"],
                    frac_of_burst=achieved / pk["bf16_tflops"], peak_burst=pk["bf16_tflops"],
                    peak_choice="sustained: the GEMMs run back to back inside a multi-ms "
                                "layer step after a soak, under the power cap",
                    traffic=recorded_traffic(dom, w.name), algorithmic_flops=fl[dom],
                    algorithmic_unit="2*R*H*N (GEMM1) or 2*R*(N/2)*H (GEMM2) flops per launch",
                    peak_source=pk["source"] + " bf16_tflops_sustained (cuBLAS bf16; the int8 "
                    "products run as exact fp16-image tcgen05 kind::f16 MMAs, whose dense rate "
                    "equals bf16's)"), step_bytes, extra

    def dtype(self):
        return "int8 GEMMs (exact, on fp16 images), fp32 epilogues, bf16 rows"


def run_layer_secondary(args, B, dev, stream, flush, pk, want_cpu):
    """The full layer workload (16384 tokens, 128 experts, FFN 4096) as a
    secondary line item: tokens/s, the grouped GEMMs' roofline against the
    burst and the sustained bf16 peaks, the clocks of its own timed region and
    its own oracle baseline."""
    import torch
    w = wl.WORKLOADS["full_layer"]
    inp = wl.make_inputs(w, seed=args.seed)
    path = LayerPath(B, w, inp, dev, args.seed, args.ffn_path)
    for _ in range(3):
        path.step()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    t_end = time.time() + max(args.soak, 1.0)          # untimed soak for the clock samples
    while time.time() < t_end:
        flush.fill_(1)
        path.step()
        torch.cuda.synchronize()
    steps = max(3, min(args.steps, 10))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.fill_(1)
        ev[i][0].record(stream)
        path.step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    B.profile_enable(True)
    for i in range(steps):
        flush.fill_(1)
        path.step()
    torch.cuda.synchronize()
    B.profile_enable(False)
    prof = B.profile_report()
    roofline, _, extra = path.roofline(prof, pk)
    roofline["per_kernel_us"] = {k: round(ms_ / n * 1e3, 3) for k, (n, ms_) in prof.items()}
    item = {"workload": w.name, "config": workload_config(w),
            "value": whole_job_tokens_per_s(w.num_tokens, 1, ms), "unit": "tokens/s",
            "ms_per_step": ms, "steps": steps, "roofline": roofline, "clocks": clk, **extra}
    del path
    torch.cuda.empty_cache()
    if want_cpu:
        item["cpu_baseline"] = cpu_baseline_sample(w, inp, args.seed, budget_s=8.0)
    return item


def quant_dispatch_item(B, path, w, inp, flush, stream, steps, pk):
    """moe_dispatch_quant (int8 rows + per-row dynamic scales) on the same
    inputs: its own event-timed calls, each after the L2 flush, and its HBM
    rate against the measured peak.  Algorithmic bytes: ids + mask, x once per
    token with an active route, R int8 rows + R scales, route_row, triplets."""
    import torch
    T, K, H = w.num_tokens, w.topk, w.hidden
    d = B.dispatch_quant(path.x, path.ids, w.num_experts, w.num_partitions, mask=path.mask)
    ws = d["workspace"]
    for _ in range(3):
        B.dispatch_quant(path.x, path.ids, w.num_experts, w.num_partitions, mask=path.mask, ws=ws, out=d)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush.fill_(1)
        ev[i][0].record(stream)
        B.dispatch_quant(path.x, path.ids, w.num_experts, w.num_partitions, mask=path.mask, ws=ws, out=d)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    us = float(np.mean([a.elapsed_time(b) for a, b in ev])) * 1e3
    R = int(d["expert_offsets"][-1].item())
    mask = inp["mask"]
    act = np.ones((T, K), bool)
    if mask is not None:
        act &= (mask[:, None] if mask.ndim == 1 else mask).astype(bool)
    tok_active = int(act.any(axis=1).sum())
    nbytes = (T * K * 4 + (0 if mask is None else mask.size) + tok_active * 2 * H + R * H + R * 4
              + T * K * 4 + R * 12)
    gbs = nbytes / (us * 1e-6) / 1e9
    # the quantising kernel alone (profiled pass of the same calls): x once per token read, the
    # route rows read, int8 rows + scales + triplets written
    B.profile_enable(True)
    for i in range(steps):
        flush.fill_(1)
        B.dispatch_quant(path.x, path.ids, w.num_experts, w.num_partitions, mask=path.mask, ws=ws, out=d)
    torch.cuda.synchronize()
    B.profile_enable(False)
    prof = B.profile_report()
    n, ms = prof.get("dispatch_quant", (1, 0.0))
    k_us = ms / max(n, 1) * 1e3
    k_bytes = tok_active * 2 * H + T * K * 4 + R * H + R * 4 + R * 12
    k_gbs = k_bytes / (k_us * 1e-6) / 1e9 if k_us > 0 else 0.0
    return {"us_per_call": us, "algorithmic_bytes": nbytes, "gbs": gbs,
            "frac_of_hbm_peak": gbs / pk["hbm_gbs"], "rows": R,
            "kernel_us": k_us, "kernel_algorithmic_bytes": k_bytes,
            "kernel_frac_of_hbm_peak": k_gbs / pk["hbm_gbs"],
            "per_kernel_us": {k: round(v[1] / v[0] * 1e3, 3) for k, v in prof.items()},
            "note": "routing + int8 rows + per-row scales; event-timed per call after an L2 flush "
                    "(the call's routing latency included); kernel_*: the quantising kernel alone, "
                    "from the library's per-kernel events"}


def timing_variants(path, flush, stream, steps):
    """The step without the L2 flush (hot L2), and the step captured once as a
    CUDA graph and replayed, with and without the flush, so that the launch
    overhead of the eager step shows separately.  Medians over `steps`."""
    import torch

    def timed(run, flush_each):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for i in range(steps):
            if flush_each:
                flush.fill_(1)
            ev[i][0].record(stream)
            run()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in ev]))

    out = {"hot_l2_ms": timed(path.step, False)}
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            path.step()
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        out["graph_ms"] = timed(g.replay, True)
        out["graph_hot_l2_ms"] = timed(g.replay, False)
    except Exception as exc:   # reported, not fatal: the eager numbers stand
        out["graph_error"] = str(exc)[:200]
    return out


def run_ours(args, rank, world, dist):
    import torch
    from combine_route_count_prefix_gb300 import binding as B

    B.lib()   # raises if the CUDA library was not built: there is no other path
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    w = select_workload(args)
    T, H = w.num_tokens, w.hidden
    inp = wl.make_inputs(w, seed=args.seed + rank)
    path = (IdentityPath(B, w, inp, dev) if w.identity
            else LayerPath(B, w, inp, dev, args.seed + rank, args.ffn_path))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        path.step()
    torch.cuda.synchronize()
    R = path.rows()
    clocks = ClockSampler(local)
    clocks.start()
    t_end = time.time() + args.soak                 # untimed soak for the clock samples
    while time.time() < t_end:
        for _ in range(10):
            flush.fill_(1)
            path.step()
        torch.cuda.synchronize()

    # ---------------- timed region
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    n0 = B.launch_count()
    for i in range(args.steps):
        flush.fill_(1)
        ev[i][0].record(stream)
        path.step()
        ev[i][1].record(stream)
    barrier()
    launches = B.launch_count() - n0
    ms = [a.elapsed_time(b) for a, b in ev]
    clk = clocks.stop()
    ms_step = max_over_ranks(float(np.mean(ms)), dist, dev)
    value = whole_job_tokens_per_s(T, world, ms_step)
    timing = {"median_ms": float(np.median(ms))}
    if w.identity:
        timing.update(timing_variants(path, flush, stream, args.steps))

    # ---------------- per-kernel durations (same K steps, profiled)
    B.profile_enable(True)
    for i in range(args.steps):
        flush.fill_(1)
        path.step()
    torch.cuda.synchronize()
    B.profile_enable(False)
    prof = B.profile_report()
    pk = peaks()
    roofline, step_bytes, extra = path.roofline(prof, pk)
    roofline["per_kernel_us"] = {k: round(ms_ / n * 1e3, 3) for k, (n, ms_) in prof.items()}
    roofline["per_kernel_grid"] = dict(B.LAST_GRIDS)
    quant_item = (quant_dispatch_item(B, path, w, inp, flush, stream, args.steps, pk)
                  if w.identity and w.hidden <= 8192 else None)

    # ---------------- end to end through the C ABI with pinned host buffers
    # Every step copies its inputs from pinned host memory and its output back.
    # As a serving loop would run it, the copies of neighbouring steps overlap
    # the current step's kernels on their own streams; the device tensors the
    # copies use are double-buffered, and events order each copy against the
    # steps that use the same buffer.  The L2 flush still precedes every step.
    def pin(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hx = pin(inp["x"].view(np.int16))
    hids, hprobs = pin(inp["ids"]), pin(inp["probs"])
    hmask = pin(inp["mask"])
    hshared = pin(None if inp["shared"] is None else inp["shared"].view(np.int16))
    hout = torch.empty((T, H), dtype=torch.int16).pin_memory()
    bufs = [dict(x=torch.empty((T, H), dtype=torch.int16, device=dev),
                 ids=torch.empty_like(path.ids), probs=torch.empty_like(path.probs),
                 mask=None if path.mask is None else torch.empty_like(path.mask),
                 shared=None if path.shared is None else torch.empty((T, H), dtype=torch.int16,
                                                                     device=dev),
                 out=torch.empty((T, H), dtype=torch.bfloat16, device=dev)) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (hx, hids, hprobs, hmask, hshared) if t is not None)
    d2h = hout.numel() * hout.element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(nsteps, start=None, end=None, compute=True):
        ev_in = [torch.cuda.Event() for _ in range(nsteps)]
        ev_comp = [torch.cuda.Event() for _ in range(nsteps)]
        ev_out = [torch.cuda.Event() for _ in range(nsteps)]
        if start is not None:
            start.record(s_in)
        for i in range(nsteps):
            b = bufs[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])    # step i-2 has read these inputs
                for name, src in (("x", hx), ("ids", hids), ("probs", hprobs), ("mask", hmask),
                                  ("shared", hshared)):
                    if src is not None:
                        b[name].copy_(src, non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])       # step i-2's output has been read back
            if compute:
                flush.fill_(1)
                path.step(b["x"].view(torch.bfloat16), b["ids"], b["probs"], b["mask"],
                          None if b["shared"] is None else b["shared"].view(torch.bfloat16),
                          out=b["out"])
            ev_comp[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                hout.copy_(b["out"].view(torch.int16), non_blocking=True)
                ev_out[i].record(s_out)
        if end is not None:
            end.record(s_out)

    e2e_run(3)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(args.steps, e0, e1)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, dev)
    # the same copies alone (same streams, bytes and ordering, no kernels): the
    # host link's own time for a step's inputs and output
    e2e_run(3, compute=False)
    barrier()
    e2e_run(args.steps, e0, e1, compute=False)
    barrier()
    link_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, dev)

    secondary = None
    if not args.no_layer and w.identity:
        secondary = run_layer_secondary(args, B, dev, stream, flush, pk,
                                        want_cpu=(world == 1 and not args.no_cpu_baseline))

    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(w, inp, args.seed)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": path.dtype(),
        "data": "synthetic", "config": workload_config(w),
        "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": whole_job_tokens_per_s(T, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copies_only_ms_per_step": link_ms, "frac_of_copies_only": link_ms / e2e_ms,
                "copies": "pinned host buffers; neighbouring steps' copies overlap compute on "
                          "their own streams (double-buffered device tensors)"},
        "gpu_launches": launches, "clocks": clk, "routed_rows": R,
        "timing": timing,
    }
    if step_bytes:
        gbs = step_bytes / (ms_step * 1e-3) / 1e9
        line["step_hbm_gbs"] = gbs
        line["step_hbm_frac_of_peak"] = gbs / pk["hbm_gbs"]
    line.update({k: v for k, v in extra.items() if v is not None})
    if secondary is not None:
        line["full_layer"] = secondary
    if quant_item is not None:
        line["dispatch_quant"] = quant_item
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            tdist.init_process_group("nccl")
            dist = tdist
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.cpu_full:
        if rank == 0 and world == 1:
            run_cpu_full(args)
    elif args.peak_probes:
        if rank == 0:
            run_peak_probes()
    else:
        run_ours(args, rank, world, dist)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
