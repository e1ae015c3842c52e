"""FP8 GEMM benchmark on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dense4096|cube256|proj|masked|smallm] [...]

One step = one pass of the hot path over one batch of synthetic input: one
FP8 GEMM (dense D = A.B^T, or the masked grouped MoE-decode GEMM) through
the C ABI.  Prints ONE JSON line (rank 0).  The default workload is the
dense 4096^3 E4M3 GEMM (FP32 accumulate, BF16 out) reported in TFLOP/s.

Multi-GPU: one process per GPU (torchrun); every rank runs its own shard of
the same shape (independent output slices, no data-path collective), so
scaling is weak; the timed region is bracketed by a barrier and a device
synchronise and the maximum time over ranks is reported.

--impl reference times the CPU oracle (the plain fp64 implementation the
tests compare against) on the host cores, on a bounded sample of the same
workload, and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "FP8 GEMM TFLOPS and % of roofline (tensor peak or HBM) on 1 GB300 vs CPU oracle"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0      # nominal dense FP8 : BF16 tensor-core rate on this part (4.5 : 2.25 PF)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

class Workload:
    """A named problem: shapes, input recipe, algorithmic FLOPs and bytes."""

    def __init__(self, name, kind, desc, **kw):
        self.name, self.kind, self.desc = name, kind, desc
        self.__dict__.update(kw)

    # algorithmic work of one step (padded MMA rows/columns are not counted)
    def flops(self, masked_m=None):
        if self.kind == "dense":
            return 2.0 * self.M * self.N * self.K
        return 2.0 * float(sum(masked_m)) * self.N * self.K

    def bytes(self, masked_m=None):
        ks = -(-self.K // self.gran) if self.gran else 0      # block-scale bytes per row
        if self.kind == "dense":
            return float(self.M * (self.K + ks) + self.N * (self.K + ks) + 2 * self.M * self.N)
        live = [m for m in masked_m if m > 0]
        return float(len(live) * self.N * (self.K + ks) + sum(live) * (self.K + ks) + 2 * sum(live) * self.N)


def make_workload(name: str, rank: int = 0) -> Workload:
    """A workload by name; a trailing ":bs" (":bs32") adds UE8M0 block scales
    per row per 128 (32) K elements: per-token scales for A, 128x128-block
    weight scales for B (each block's scale repeated over its rows)."""
    gran = 0
    if name.endswith(":bs") or name.endswith(":bs32"):
        base, tag = name.rsplit(":", 1)
        gran = 128 if tag == "bs" else 32
        w = _make_base_workload(base, rank)
        if w.kind == "contig":
            raise SystemExit("block scales are not supported with the contiguous grouped layout")
        w.name, w.gran = name, gran
        w.desc += ", block-scaled (UE8M0, 1x%d tokens, %s weights)" % (gran, "128x128" if gran == 128 else "1x32")
        if w.kind == "dense" and w.M > 128 and (w.flags & 3) != 1:
            w.kernel = "k_gemm_mn"
        return w
    w = _make_base_workload(name, rank)
    w.gran = gran
    return w


def _make_base_workload(name: str, rank: int = 0) -> Workload:
    import synth
    if name == "dense4096":
        return Workload(name, "dense", "dense GEMM M=N=K=4096, A,B E4M3 from N(0,1), FP32 accumulate, BF16 out",
                        M=4096, N=4096, K=4096, fa=synth.E4M3, fb=synth.E4M3, dist="normal", std=1.0,
                        seed=synth.seed_for(1, rank), bound="tensor", flags=0)
    if name == "cube256":
        return Workload(name, "dense", "dense GEMM M=N=K=256, A,B E4M3 from U[-2,2]",
                        M=256, N=256, K=256, fa=synth.E4M3, fb=synth.E4M3, dist="uniform", std=None,
                        seed=synth.seed_for(0, rank), bound="tensor", flags=0)
    if name.startswith("proj"):
        # proj:N:K[:e5m2]  -- M=8192 token projection shapes
        parts = name.split(":")
        N, K = int(parts[1]), int(parts[2])
        fb = synth.E5M2 if len(parts) > 3 and parts[3] == "e5m2" else synth.E4M3
        return Workload(name, "dense", "projection GEMM M=8192 N=%d K=%d, A E4M3, B %s, N(0,0.5)"
                        % (N, K, "E5M2" if fb else "E4M3"),
                        M=8192, N=N, K=K, fa=synth.E4M3, fb=fb, dist="normal", std=0.5,
                        seed=synth.seed_for(2, rank), bound="tensor", flags=0)
    if name == "masked" or name.startswith("masked:"):
        # masked[:swap|noswap|auto] -- the MoE-decode workload (SwapAB unless asked otherwise)
        mode = name.split(":")[1] if ":" in name else "swap"
        label = {"swap": "SwapAB", "noswap": "non-swapped", "auto": "library's choice"}[mode]
        return Workload(name, "masked", "masked grouped GEMM G=32 M_max=128 N=4096 K=7168, m_g~U{0..32}, "
                        "E4M3 N(0,0.5), %s" % label, G=32, M_max=128, N=4096, K=7168, fa=synth.E4M3,
                        fb=synth.E4M3, dist="normal", std=0.5, seed=synth.seed_for(3, rank), bound="hbm",
                        hint=32, flags={"swap": 1, "noswap": 2, "auto": 0}[mode])
    if name.startswith("grouped:"):
        # grouped:G:m:N:K[:swap|noswap|auto] -- masked grouped GEMM whose G groups
        # all hold m valid tokens (the aligned-M grouped benchmark shape)
        parts = name.split(":")
        G, m, N, K = int(parts[1]), int(parts[2]), int(parts[3]), int(parts[4])
        mode = parts[5] if len(parts) > 5 else "auto"
        label = {"swap": "SwapAB", "noswap": "non-swapped", "auto": "library's choice"}[mode]
        # tensor-bound above the ridge (~500 FLOP per byte), else HBM-bound
        bound = "tensor" if 2.0 * G * m * N * K / (G * N * K + G * m * K + 2.0 * G * m * N) > 500 else "hbm"
        return Workload(name, "masked", "masked grouped GEMM G=%d, m=%d tokens in every group, N=%d K=%d, "
                        "E4M3 N(0,0.5), %s" % (G, m, N, K, label), G=G, M_max=m, N=N, K=K, fa=synth.E4M3,
                        fb=synth.E4M3, dist="normal", std=0.5, seed=synth.seed_for(5, rank), bound=bound,
                        hint=m, flags={"swap": 1, "noswap": 2, "auto": 0}[mode], m_fixed=m)
    if name.startswith("contig:"):
        # contig:G:m:N:K[:swap|noswap|auto] -- contiguous grouped GEMM: the G
        # groups' m token rows each stored back to back in A [G*m, K]
        parts = name.split(":")
        G, m, N, K = int(parts[1]), int(parts[2]), int(parts[3]), int(parts[4])
        mode = parts[5] if len(parts) > 5 else "auto"
        label = {"swap": "SwapAB", "noswap": "non-swapped", "auto": "library's choice"}[mode]
        # tensor-bound above the ridge (~500 FLOP per byte), else HBM-bound
        bound = "tensor" if 2.0 * G * m * N * K / (G * N * K + G * m * K + 2.0 * G * m * N) > 500 else "hbm"
        return Workload(name, "contig", "contiguous grouped GEMM G=%d, m=%d token rows per group back to back, "
                        "N=%d K=%d, E4M3 N(0,0.5), %s" % (G, m, N, K, label), G=G, M_max=m, N=N, K=K,
                        fa=synth.E4M3, fb=synth.E4M3, dist="normal", std=0.5, seed=synth.seed_for(6, rank),
                        bound=bound, hint=m, flags={"swap": 1, "noswap": 2, "auto": 0}[mode], m_fixed=m)
    if name.startswith("smallm"):
        # smallm:M:N:K[:swap|noswap]
        parts = name.split(":")
        M, N, K = int(parts[1]), int(parts[2]), int(parts[3])
        mode = parts[4] if len(parts) > 4 else "auto"
        label = {"swap": "SwapAB", "noswap": "non-swapped", "auto": "library's choice"}[mode]
        return Workload(name, "dense", "small-M weight-streaming GEMM M=%d N=%d K=%d, E4M3 N(0,1), %s"
                        % (M, N, K, label),
                        M=M, N=N, K=K, fa=synth.E4M3, fb=synth.E4M3, dist="normal", std=1.0,
                        seed=synth.seed_for(4, rank), bound="hbm",
                        flags={"swap": 1, "noswap": 2, "auto": 0}[mode])
    raise SystemExit("unknown workload %r" % name)


def host_inputs(w: Workload):
    """Seeded FP8 codes (numpy) for one instance of the workload."""
    import numpy as np
    import synth
    if w.kind == "dense":
        if w.dist == "uniform":
            A = synth.uniform_fp8((w.M, w.K), w.seed, -2.0, 2.0, w.fa)
            B = synth.uniform_fp8((w.N, w.K), w.seed + 100, -2.0, 2.0, w.fb)
        else:
            A = synth.normal_fp8((w.M, w.K), w.seed, 0.0, w.std, w.fa)
            B = synth.normal_fp8((w.N, w.K), w.seed + 100, 0.0, w.std, w.fb)
        out = {"A": A, "B": B}
    elif w.kind == "contig":
        A = synth.normal_fp8((w.G * w.M_max, w.K), w.seed, 0.0, w.std, w.fa)
        B = synth.normal_fp8((w.G, w.N, w.K), w.seed + 100, 0.0, w.std, w.fb)
        mm = np.full(w.G, w.m_fixed, np.int32)
        out = {"A": A, "B": B, "masked_m": mm,
               "offsets": np.concatenate([[0], np.cumsum(mm)]).astype(np.int32)}
    else:
        A = synth.normal_fp8((w.G, w.M_max, w.K), w.seed, 0.0, w.std, w.fa)
        B = synth.normal_fp8((w.G, w.N, w.K), w.seed + 100, 0.0, w.std, w.fb)
        if getattr(w, "m_fixed", None) is not None:
            mm = np.full(w.G, w.m_fixed, np.int32)
        else:
            mm = synth.uniform_int(w.G, w.seed + 200, 0, 32).astype(np.int32)
        out = {"A": A, "B": B, "masked_m": mm}
    if w.gran:
        out.update(block_scales(w))
    return out


def block_scales(w: Workload):
    """Seeded UE8M0 codes in [120, 134]: sf_a [G, ks, lda] one per token row
    per K group; sf_b [G, ks, ldb] one per 128x128 weight block (gran 128) or
    per row per 32 K elements (gran 32), repeated over the block's rows."""
    import numpy as np
    import synth
    G = 1 if w.kind == "dense" else w.G
    rows = w.M if w.kind == "dense" else w.M_max
    ks = -(-w.K // w.gran)
    lda, ldb = -(-rows // 16) * 16, -(-w.N // 16) * 16
    sfa = synth.uniform_int(G * ks * lda, w.seed + 300, 120, 134).astype(np.uint8).reshape(G, ks, lda)
    if w.gran == 128:
        nb = -(-w.N // 128)
        blk = synth.uniform_int(G * ks * nb, w.seed + 301, 120, 134).astype(np.uint8).reshape(G, ks, nb)
        sfb = np.zeros((G, ks, ldb), np.uint8)
        sfb[:, :, :w.N] = np.repeat(blk, 128, axis=2)[:, :, :w.N]
    else:
        sfb = synth.uniform_int(G * ks * ldb, w.seed + 301, 120, 134).astype(np.uint8).reshape(G, ks, ldb)
    return {"sf_a": sfa, "sf_b": sfb}


# ---------------------------------------------------------------------------
# measurement helpers
# ---------------------------------------------------------------------------

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("kernels.cu", "ptx.cuh", "kernels.cuh", "api.cu"):
        with open(os.path.join(ROOT, "fp8_tensor_core_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KERNEL_NAMES = {0: "k_gemm_mn", 1: "k_gemm_mn2", 2: "k_gemm_swap"}


def planned_launch(w: Workload) -> dict:
    """The launch the library makes for the workload on the current device
    (kernel, tile, stages, split, issuers, SM sharing, token rows per copy,
    grid), from its planner."""
    import fp8_tensor_core_gb300 as fp8g
    if w.kind == "dense":
        return fp8g.fp8g_describe_plan(fp8g.LAYOUT_DENSE, 1, w.M, w.N, w.K, 0, w.gran or 0, w.flags)
    if w.kind == "contig":
        return fp8g.fp8g_describe_plan(fp8g.LAYOUT_CONTIGUOUS, w.G, w.G * w.M_max, w.N, w.K, w.hint, 0, w.flags)
    return fp8g.fp8g_describe_plan(fp8g.LAYOUT_MASKED, w.G, w.M_max, w.N, w.K, w.hint, w.gran or 0, w.flags)


def profiled_traffic(workload: str):
    """Per-launch DRAM bytes (read + write) of the dominant kernel from the
    committed ncu summary, valid only while the kernel sources are unchanged
    since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash()
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            if len(parts) >= 3 and parts[0] == workload and parts[1] == cur:
                return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples, timestamped on arrival."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [s.strip() for s in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        def parse(rows):
            sm = [float(r[0]) for _, r in rows if r and r[0].replace(".", "", 1).isdigit()]
            mx = [float(r[1]) for _, r in rows if len(r) > 1 and r[1].replace(".", "", 1).isdigit()]
            reasons = set()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for _, r in rows:
                for i, n in enumerate(names):
                    if len(r) > 4 + i and r[4 + i].lower().startswith("active"):
                        reasons.add(n)
            return sm, mx, sorted(reasons)
        inside = [s for s in self.samples if t0 <= s[0] <= t1 + 0.15]
        window = "timed"
        if len(inside) < 2:
            inside = [s for s in self.samples if s[0] <= t1 + 0.15]
            window = "warmup+timed"
        sm, mx, reasons = parse(inside)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sm), "window": window}


def dist_setup():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample(w: Workload, inp, budget_s: float, min_rows: int = 1):
    """Time the oracle on whole output rows of the workload until about
    `budget_s` seconds have been spent.  Returns (flops, seconds, cores,
    description)."""
    import numpy as np
    import oracle
    cores = oracle.default_threads()
    flops = 0.0
    t_start = time.perf_counter()
    if w.kind == "dense":
        A, B = inp["A"], inp["B"]
        rows, r0 = max(min_rows, 8), 0
        while r0 < w.M:
            r1 = min(w.M, r0 + rows)
            t = time.perf_counter()
            if w.gran:
                oracle.gemm_blockscaled(A[r0:r1], B, inp["sf_a"][0][:, r0:r1].copy(), inp["sf_b"][0], w.gran,
                                        fa=w.fa, fb=w.fb)
            else:
                oracle.gemm_nt(A[r0:r1], B, w.fa, w.fb)
            dt = time.perf_counter() - t
            flops += 2.0 * (r1 - r0) * w.N * w.K
            r0 = r1
            if time.perf_counter() - t_start >= budget_s:
                break
            rows = max(rows, int(rows * min(4.0, 0.5 * budget_s / max(dt, 1e-3))))
        secs = time.perf_counter() - t_start
        desc = "rows 0..%d of D (%d of %d rows, all N=%d columns, K=%d)" % (r0 - 1, r0, w.M, w.N, w.K)
        return flops, secs, cores, desc
    if w.kind == "contig":
        A, B, off = inp["A"], inp["B"], inp["offsets"]
        g_done = 0
        for g in range(w.G):
            if off[g + 1] > off[g]:
                oracle.gemm_nt(A[off[g]:off[g + 1]], B[g], w.fa, w.fb)
                flops += 2.0 * int(off[g + 1] - off[g]) * w.N * w.K
            g_done += 1
            if time.perf_counter() - t_start >= budget_s:
                break
        secs = time.perf_counter() - t_start
        return flops, secs, cores, "groups 0..%d of %d (all their rows)" % (g_done - 1, w.G)
    A, B, mm = inp["A"], inp["B"], inp["masked_m"]
    D0 = np.zeros((1, w.M_max, w.N), np.uint16)
    g_done = 0
    for g in range(w.G):
        if mm[g] == 0:
            g_done += 1
            continue
        if w.gran:
            oracle.gemm_blockscaled(A[g:g + 1], B[g:g + 1], inp["sf_a"][g:g + 1], inp["sf_b"][g:g + 1], w.gran,
                                    masked_m=mm[g:g + 1], D_init=D0, fa=w.fa, fb=w.fb)
        else:
            oracle.gemm_grouped_masked(A[g:g + 1], B[g:g + 1], mm[g:g + 1], D0, w.fa, w.fb)
        flops += 2.0 * int(mm[g]) * w.N * w.K
        g_done += 1
        if time.perf_counter() - t_start >= budget_s:
            break
    secs = time.perf_counter() - t_start
    return flops, secs, cores, "groups 0..%d of %d (all their valid rows)" % (g_done - 1, w.G)


def run_reference(args, w: Workload):
    """--impl reference: the CPU oracle timed on the host cores, each step a
    bounded sample (a block of output rows) of the workload."""
    rank, world, _ = dist_setup()
    if rank != 0:
        return 0
    import oracle
    inp = host_inputs(w)
    oracle.build()
    per_step_budget = max(0.05, min(2.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, inp, per_step_budget * 0.25)
    flops = secs = 0.0
    desc = ""
    cores = oracle.default_threads()
    for _ in range(args.steps):
        f, s, cores, desc = oracle_sample(w, inp, per_step_budget)
        flops += f
        secs += s
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.desc, "name": w.name},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "per step: " + desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args, w: Workload):
    import numpy as np
    import torch

    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", rank=rank, world_size=world, device_id=device)

    import fp8_tensor_core_gb300 as fp8g
    fp8g._lib.load()          # fails loudly if the CUDA library is not built
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 2**20)

    inp = host_inputs(w)
    stream = torch.cuda.current_stream(device)

    # Rotating device copies so that consecutive steps do not find their
    # operands in L2: sets x (inputs + output) >= 3 x L2.
    if w.kind == "dense":
        set_bytes = w.M * w.K + w.N * w.K + 2 * w.M * w.N
    elif w.kind == "contig":
        set_bytes = w.G * w.M_max * w.K + w.G * w.N * w.K + 2 * w.G * w.M_max * w.N
    else:
        set_bytes = w.G * w.M_max * w.K + w.G * w.N * w.K + 2 * w.G * w.M_max * w.N
    n_sets = max(1, math.ceil(3 * l2 / set_bytes))
    n_sets = min(n_sets, 64)
    sets = []
    A_h = torch.from_numpy(inp["A"]).pin_memory()
    B_h = torch.from_numpy(inp["B"]).pin_memory()
    sfa_h = torch.from_numpy(inp["sf_a"]).pin_memory() if w.gran else None
    sfb_h = torch.from_numpy(inp["sf_b"]).pin_memory() if w.gran else None
    for _ in range(n_sets):
        s = {"A": A_h.to(device), "B": B_h.to(device)}
        if w.gran:
            s["sfa"], s["sfb"] = sfa_h.to(device), sfb_h.to(device)
        if w.kind == "dense":
            s["D"] = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)
        elif w.kind == "contig":
            s["off"] = torch.from_numpy(inp["offsets"]).to(device)
            s["D"] = torch.empty((w.G * w.M_max, w.N), dtype=torch.bfloat16, device=device)
        else:
            s["mm"] = torch.from_numpy(inp["masked_m"]).to(device)
            s["D"] = torch.zeros((w.G, w.M_max, w.N), dtype=torch.bfloat16, device=device)
        sets.append(s)
    torch.cuda.synchronize(device)

    def call(s, strm):
        if w.kind == "dense" and w.gran:
            fp8g.fp8_gemm_nt_blockscaled(s["A"], s["B"], s["sfa"], s["sfb"], s["D"], sf_group_k=w.gran,
                                         a_dtype=w.fa, b_dtype=w.fb, flags=w.flags, stream=strm)
        elif w.kind == "dense":
            fp8g.fp8_gemm_nt(s["A"], s["B"], s["D"], a_dtype=w.fa, b_dtype=w.fb, flags=w.flags,
                             stream=strm)
        elif w.kind == "contig":
            fp8g.fp8_gemm_grouped_contiguous(s["A"], s["B"], s["off"], D=s["D"], max_m_hint=w.hint, a_dtype=w.fa,
                                             b_dtype=w.fb, flags=w.flags, stream=strm)
        elif w.gran:
            fp8g.fp8_gemm_grouped_masked_blockscaled(s["A"], s["B"], s["mm"], s["sfa"], s["sfb"], s["D"],
                                                     max_m_hint=w.hint, sf_group_k=w.gran, a_dtype=w.fa,
                                                     b_dtype=w.fb, flags=w.flags, stream=strm)
        else:
            fp8g.fp8_gemm_grouped_masked(s["A"], s["B"], s["mm"], s["D"], max_m_hint=w.hint,
                                         a_dtype=w.fa, b_dtype=w.fb, flags=w.flags, stream=strm)

    def step_on(i, strm):
        call(sets[i % n_sets], strm)

    def step(i):
        step_on(i, stream)

    sampler = ClockSampler("GPU-" + str(props.uuid)) if rank == 0 else None

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(device)
    st = fp8g.fp8g_get_device_status(stream)
    if st[0] != fp8g.OK:
        raise SystemExit("device status after warm-up: %s" % (st,))

    # ---- timed region: exactly K steps --------------------------------------
    # By default the K launches (the same C-ABI calls) are captured into one
    # CUDA graph and its replay is timed, so host launch gaps do not count;
    # --graph off times K direct launches with events around each.
    use_graph = args.graph != "off"
    graph = None
    if use_graph:
        gs = torch.cuda.Stream(device)
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            for i in range(2):            # warm the side stream too
                step_on(i, gs)
        gs.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for i in range(args.steps):
                step_on(args.warmup + i, gs)
        torch.cuda.synchronize(device)
        graph.replay()                    # upload / first replay, untimed
        torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(1 if use_graph else args.steps)]
    barrier(world, device)
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    if use_graph:
        ev[0][0].record(stream)
        graph.replay()
        ev[0][1].record(stream)
    else:
        for i in range(args.steps):
            ev[i][0].record(stream)
            step(args.warmup + i)
            ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    barrier(world, device)
    t_wall1 = time.time()
    total_ms = ev[0][0].elapsed_time(ev[-1][1])
    if use_graph:
        kernel_ms = total_ms / args.steps
    else:
        per_launch_ms = [a.elapsed_time(b) for a, b in ev]
        kernel_ms = sum(per_launch_ms) / len(per_launch_ms)
    st = fp8g.fp8g_get_device_status(stream)
    if st[0] != fp8g.OK:
        raise SystemExit("device status after timed region: %s" % (st,))
    total_ms_max = max_over_ranks(total_ms, world, device)
    kernel_ms_max = max_over_ranks(kernel_ms, world, device)
    if sampler:
        sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None

    mm = inp.get("masked_m")
    flops = w.flops(mm)
    algo_bytes = w.bytes(mm)
    value = world * args.steps * flops / (total_ms_max * 1e-3) / 1e12

    # ---- end to end through the public API, host buffers ---------------------
    # Every step copies its inputs in from pinned host memory, runs the GEMM
    # through the public API and copies the whole of D back.  Consecutive
    # steps rotate over --e2e-streams streams, each with its own device and
    # host buffers, so one step's copies overlap its neighbours' (the host
    # link moves ~210 GB/s one way, ~340 GB/s both ways at once).
    e2e = None
    if not args.no_e2e:
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        n_pipe = max(1, args.e2e_streams)
        mm_h = torch.from_numpy(inp["masked_m"]).pin_memory() if mm is not None and w.kind == "masked" else None
        off_h = torch.from_numpy(inp["offsets"]).pin_memory() if w.kind == "contig" else None
        pipe = []
        for k in range(n_pipe):
            if k < n_sets:
                s_k = sets[k]
            else:   # one more device set for this stream
                s_k = {key: torch.empty_like(v) for key, v in sets[0].items()}
            pipe.append({"set": s_k, "D_h": torch.empty(s_k["D"].shape, dtype=torch.bfloat16).pin_memory(),
                         "stream": stream if k == 0 else torch.cuda.Stream(device)})

        def e2e_step(i):
            p = pipe[i % n_pipe]
            s_k, strm = p["set"], p["stream"]
            with torch.cuda.stream(strm):
                s_k["A"].copy_(A_h, non_blocking=True)
                s_k["B"].copy_(B_h, non_blocking=True)
                if w.gran:
                    s_k["sfa"].copy_(sfa_h, non_blocking=True)
                    s_k["sfb"].copy_(sfb_h, non_blocking=True)
                if mm_h is not None:
                    s_k["mm"].copy_(mm_h, non_blocking=True)
                if off_h is not None:
                    s_k["off"].copy_(off_h, non_blocking=True)
                call(s_k, strm)
                p["D_h"].copy_(s_k["D"], non_blocking=True)

        for i in range(min(3, e2e_steps)):
            e2e_step(i)
        torch.cuda.synchronize(device)
        barrier(world, device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for p in pipe[1:]:
            p["stream"].wait_event(e0)
        for i in range(e2e_steps):
            e2e_step(i)
        for p in pipe[1:]:
            stream.wait_stream(p["stream"])
        e1.record(stream)
        torch.cuda.synchronize(device)
        st = fp8g.fp8g_get_device_status(stream)
        if st[0] != fp8g.OK:
            raise SystemExit("device status after the end-to-end run: %s" % (st,))
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, device)
        h2d = A_h.numel() + B_h.numel() + (mm_h.numel() * 4 if mm_h is not None else 0) + \
            (off_h.numel() * 4 if off_h is not None else 0)
        if w.gran:
            h2d += sfa_h.numel() + sfb_h.numel()
        d2h = pipe[0]["D_h"].numel() * 2
        e2e = {"value": world * e2e_steps * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
               "streams": n_pipe}

    # ---- roofline of the dominant kernel -----------------------------------------
    peaks, peak_src = load_peaks()
    if w.bound == "tensor":
        peak = FP8_PER_BF16 * peaks["bf16_tflops_sustained"]
        achieved = flops / (kernel_ms_max * 1e-3) / 1e12
        unit = "TFLOP/s"
        basis = ("FP8 = %g x %s BF16 sustained (%.1f TF/s; kernel timed back to back in a long loop)"
                 % (FP8_PER_BF16, peak_src, peaks["bf16_tflops_sustained"]))
    else:
        peak = peaks["hbm_gbs"]
        achieved = algo_bytes / (kernel_ms_max * 1e-3) / 1e9
        unit = "GB/s"
        basis = "%s HBM copy bandwidth" % peak_src
    traffic = profiled_traffic(w.name)
    plan = planned_launch(w)
    kernel_name = KERNEL_NAMES[plan["kernel"]]
    roof = {"bound": w.bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic, "kernel": kernel_name, "plan": plan,
            "peak_basis": basis, "algorithmic_flop": flops, "algorithmic_bytes": algo_bytes,
            "kernel_ms": kernel_ms_max}
    if w.bound == "tensor":
        roof["frac_of_nominal_4500"] = achieved / 4500.0
    else:
        roof["frac_of_nominal_8000"] = achieved / 8000.0

    # ---- CPU baseline (rank 0, N = 1 only) ----------------------------------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, s, cores, desc = oracle_sample(w, inp, args.cpu_budget)
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": desc + "; %.1f s" % s}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8_e4m3" if w.fb == 0 else "fp8_e4m3xe5m2", "data": "synthetic",
            "config": {"workload": w.desc, "name": w.name, "flags": hex(w.flags),
                       "l2": "%d rotating input+output sets of %.1f MB (>= 3x the %d MB L2)"
                             % (n_sets, set_bytes / 1e6, l2 >> 20),
                       "parallelism": "independent shard per GPU" if world > 1 else "single GPU"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "timing": "one CUDA graph of K launches" if use_graph else "K direct launches, events per launch",
            "clocks": clocks,
        }
        if w.kind == "masked":
            line["config"]["sum_masked_m"] = int(sum(mm))
            line["config"]["empty_groups"] = int(sum(1 for m in mm if m == 0))
        if w.kind == "contig":
            line["config"]["tokens"] = int(sum(mm))
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dense4096")
    ap.add_argument("--graph", choices=["on", "off"], default="on",
                    help="replay the K timed launches from one CUDA graph (off: K direct launches "
                         "with events around each)")
    ap.add_argument("--extra-flags", type=lambda v: int(v, 0), default=0,
                    help="tuning-override flag bits OR-ed into the call (FP8G_WHOLE_TILES 0x100, FP8G_TILE_N)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--e2e-streams", type=int, default=3,
                    help="streams the end-to-end steps alternate between (1 = strictly serial steps)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank, _, _ = dist_setup()
    w = make_workload(args.workload, rank)
    w.flags |= args.extra_flags
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
