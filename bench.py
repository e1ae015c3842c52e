"""FP8 GEMM benchmark on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dense4096|cube256|proj|masked|smallm] [...]

One step = one pass of the hot path over one batch of synthetic input: one
FP8 GEMM (dense D = A.B^T, or the masked grouped MoE-decode GEMM) through
the C ABI.  Prints ONE JSON line (rank 0).  The default workload is the
largest configuration, the dense 8192 x 18432 x 7168 E4M3 projection (FP32
accumulate, BF16 out), reported in TFLOP/s, with every other configuration
timed briefly in the line's per_config array.

--mma-microbench instead builds and runs bench_mma.cu: the tensor-core
instruction costs (plain and block-scaled MMAs, one or two issuers, with and
without the kernels' stage handshake, SM pairs, scale-set writes), one JSON
object per line.

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
    if name.startswith("dense:"):
        # dense:M:N:K[:e5m2] -- any dense shape, A and B from N(0,1)
        parts = name.split(":")
        M, N, K = int(parts[1]), int(parts[2]), int(parts[3])
        fb = synth.E5M2 if len(parts) > 4 and parts[4] == "e5m2" else synth.E4M3
        bound = "tensor" if 2.0 * M * N * K / (M * K + N * K + 2.0 * M * N) > 500 else "hbm"
        return Workload(name, "dense", "dense GEMM M=%d N=%d K=%d, A E4M3, B %s, N(0,1)"
                        % (M, N, K, "E5M2" if fb else "E4M3"), M=M, N=N, K=K, fa=synth.E4M3, fb=fb,
                        dist="normal", std=1.0, seed=synth.seed_for(7, rank), bound=bound, flags=0)
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
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        t_end = time.time() + 5.0          # nvidia-smi's first sample can take a second
        while not self.samples and time.time() < t_end and self.proc.poll() is None:
            time.sleep(0.02)

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

    def summary(self, t0: float, t1: float, t_warm: float = None):
        """Clocks in the timed region [t0, t1]; when that holds fewer than two
        samples (a short region), in [t_warm, t1] -- the warm-up launches of
        the same kernel and the timed region -- and without t_warm in
        everything sampled up to t1."""
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
        inside = [s for s in self.samples if t0 <= s[0] <= t1 + 0.05]
        window = "timed"
        if len(inside) < 2:
            lo = t_warm if t_warm is not None else 0.0
            inside = [s for s in self.samples if lo <= s[0] <= t1 + 0.05]
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

def oracle_sample(w: Workload, inp, budget_s: float, min_rows: int = 1, check_against=None):
    """Time the oracle on whole output rows (groups) of the workload until
    about `budget_s` seconds have been spent.  Returns (flops, seconds,
    cores, description, parity): with `check_against` (the device run's D
    as uint16 bits) every element the oracle computed is compared with it
    after the clock stops, within the acceptance rule (one BF16 ulp plus
    1e-6 * sum |a b|; masked padding rows bit for bit); parity is "ok ..."
    or a description of the first mismatch, None without a device D."""
    import numpy as np
    import oracle
    cores = oracle.default_threads()
    flops = 0.0
    pieces = []            # (what, reference D, absdot, device slice)
    t_start = time.perf_counter()
    if w.kind == "dense":
        A, B = inp["A"], inp["B"]
        rows, r0 = max(min_rows, 8), 0
        while r0 < w.M:
            r1 = min(w.M, r0 + rows)
            t = time.perf_counter()
            if w.gran:
                ref, absd, accb = oracle.gemm_blockscaled(A[r0:r1], B, inp["sf_a"][0][:, r0:r1].copy(),
                                                          inp["sf_b"][0], w.gran, fa=w.fa, fb=w.fb,
                                                          want_accbound=True)
            else:
                (ref, absd), accb = oracle.gemm_nt(A[r0:r1], B, w.fa, w.fb), None
            dt = time.perf_counter() - t
            if check_against is not None:
                pieces.append(("rows %d..%d" % (r0, r1 - 1), ref, absd, check_against[r0:r1], accb))
            flops += 2.0 * (r1 - r0) * w.N * w.K
            r0 = r1
            if time.perf_counter() - t_start >= budget_s:
                break
            rows = max(rows, int(rows * min(4.0, 0.5 * budget_s / max(dt, 1e-3))))
        secs = time.perf_counter() - t_start
        desc = "rows 0..%d of D (%d of %d rows, all N=%d columns, K=%d)" % (r0 - 1, r0, w.M, w.N, w.K)
    elif w.kind == "contig":
        A, B, off = inp["A"], inp["B"], inp["offsets"]
        g_done = 0
        for g in range(w.G):
            if off[g + 1] > off[g]:
                ref, absd = oracle.gemm_nt(A[off[g]:off[g + 1]], B[g], w.fa, w.fb)
                if check_against is not None:
                    pieces.append(("group %d" % g, ref, absd, check_against[off[g]:off[g + 1]], None))
                flops += 2.0 * int(off[g + 1] - off[g]) * w.N * w.K
            g_done += 1
            if time.perf_counter() - t_start >= budget_s:
                break
        secs = time.perf_counter() - t_start
        desc = "groups 0..%d of %d (all their rows)" % (g_done - 1, w.G)
    else:
        A, B, mm = inp["A"], inp["B"], inp["masked_m"]
        D0 = np.zeros((1, w.M_max, w.N), np.uint16)
        g_done = 0
        for g in range(w.G):
            if mm[g] == 0:
                g_done += 1
                continue
            if w.gran:
                ref, absd, accb = oracle.gemm_blockscaled(A[g:g + 1], B[g:g + 1], inp["sf_a"][g:g + 1],
                                                          inp["sf_b"][g:g + 1], w.gran, masked_m=mm[g:g + 1],
                                                          D_init=D0, fa=w.fa, fb=w.fb, want_accbound=True)
            else:
                (ref, absd), accb = oracle.gemm_grouped_masked(A[g:g + 1], B[g:g + 1], mm[g:g + 1], D0, w.fa,
                                                               w.fb), None
            if check_against is not None:
                m = int(mm[g])
                pieces.append(("group %d" % g, ref[0, :m], absd[0, :m], check_against[g, :m],
                               accb[0, :m] if accb is not None else None))
            flops += 2.0 * int(mm[g]) * w.N * w.K
            g_done += 1
            if time.perf_counter() - t_start >= budget_s:
                break
        secs = time.perf_counter() - t_start
        desc = "groups 0..%d of %d (all their valid rows)" % (g_done - 1, w.G)
    parity = None
    if check_against is not None:
        n = 0
        for what, ref, absd, got, accb in pieces:
            ok, rep = oracle.check_bf16(got, ref, absd, acc_bound=accb)
            if not ok:
                return flops, secs, cores, desc, "mismatch in %s: %s" % (what, rep)
            n += ref.size
        parity = "ok: %d elements of the device run's D (the sampled %s) match the oracle" % (
            n, "rows" if w.kind == "dense" else "groups")
    return flops, secs, cores, desc, parity


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
        f, s, cores, desc, _ = oracle_sample(w, inp, per_step_budget)
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

# The pages' configurations, each a bench workload: the per_config array of
# the JSON line times every one of them (configs 1-5; config 5 through both
# kernels, SwapAB and the non-swapped token tiles).
PER_CONFIG = ([("1", "cube256"), ("2", "dense4096")] +
              [("3", "proj:%s%s" % (nk, fmt)) for nk in ("7168:2048", "4096:7168", "18432:7168", "7168:18432")
               for fmt in ("", ":e5m2")] +
              [("4", "masked"), ("4", "masked:noswap")] +
              [("5", "smallm:%d:%s:%s" % (m, nk, mode)) for nk in ("24576:1536", "7168:16384")
               for m in (1, 8, 16, 32, 64) for mode in ("swap", "noswap")])
DEFAULT_WORKLOAD = "proj:18432:7168"      # the largest configuration (M=8192, N=18432, K=7168)
BURST_REGION_MS = 1000.0                  # timed regions shorter than this are compared with the burst peak


def set_bytes_of(w: Workload) -> int:
    if w.kind == "dense":
        return w.M * w.K + w.N * w.K + 2 * w.M * w.N
    return w.G * w.M_max * w.K + w.G * w.N * w.K + 2 * w.G * w.M_max * w.N


def device_sets(w: Workload, inp, device, l2: int, pinned=None):
    """Rotating device copies of the inputs and an output each, so that
    consecutive launches do not find their operands in L2: sets x (inputs +
    output) >= 3 x L2.  Returns (sets, host tensors)."""
    import torch
    n_sets = min(64, max(1, math.ceil(3 * l2 / set_bytes_of(w))))
    h = pinned or {}
    if not h:
        h["A"] = torch.from_numpy(inp["A"]).pin_memory()
        h["B"] = torch.from_numpy(inp["B"]).pin_memory()
        if w.gran:
            h["sfa"] = torch.from_numpy(inp["sf_a"]).pin_memory()
            h["sfb"] = torch.from_numpy(inp["sf_b"]).pin_memory()
    sets = []
    for _ in range(n_sets):
        s = {"A": h["A"].to(device), "B": h["B"].to(device)}
        if w.gran:
            s["sfa"], s["sfb"] = h["sfa"].to(device), h["sfb"].to(device)
        if w.kind == "dense":
            s["D"] = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)
        elif w.kind == "contig":
            s["off"] = torch.from_numpy(inp["offsets"]).to(device)
            s["D"] = torch.empty((w.G * w.M_max, w.N), dtype=torch.bfloat16, device=device)
        else:
            s["mm"] = torch.from_numpy(inp["masked_m"]).to(device)
            s["D"] = torch.zeros((w.G, w.M_max, w.N), dtype=torch.bfloat16, device=device)
        sets.append(s)
    return sets, h


def make_call(w: Workload):
    """The public-API call of one step on a device set."""
    import fp8_tensor_core_gb300 as fp8g

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
    return call


def check_status(where: str, stream=None):
    import fp8_tensor_core_gb300 as fp8g
    st = fp8g.fp8g_get_device_status(stream)
    if st[0] != fp8g.OK:
        raise SystemExit("device status %s: %s" % (where, st))


def timed_launches(call, sets, steps: int, warmup: int, device, stream, use_graph: bool, sync_world=None):
    """W warm-up launches, then exactly `steps` launches timed on the device
    with CUDA events on the launching stream: by default captured into one
    CUDA graph whose replay is timed (host launch gaps do not count), else
    direct launches with events around each.  Returns (total_ms, per-launch
    ms, wall-clock start and end of the timed region, wall-clock start of the
    warm-up)."""
    import torch
    t_warm = time.time()
    for i in range(warmup):
        call(sets[i % len(sets)], stream)
    torch.cuda.synchronize(device)
    check_status("after warm-up", stream)
    graph = None
    if use_graph:
        gs = torch.cuda.Stream(device)
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            for i in range(2):            # the side stream's own warm-up (its stream-K scratch)
                call(sets[i % len(sets)], gs)
        gs.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for i in range(steps):
                call(sets[(warmup + i) % len(sets)], gs)
        torch.cuda.synchronize(device)
        graph.replay()                    # upload / first replay, untimed
        torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(1 if use_graph else steps)]
    if sync_world:
        sync_world()
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    if use_graph:
        ev[0][0].record(stream)
        graph.replay()
        ev[0][1].record(stream)
    else:
        for i in range(steps):
            ev[i][0].record(stream)
            call(sets[(warmup + i) % len(sets)], stream)
            ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    if sync_world:
        sync_world()
    t_wall1 = time.time()
    total_ms = ev[0][0].elapsed_time(ev[-1][1])
    kernel_ms = total_ms / steps if use_graph else sum(a.elapsed_time(b) for a, b in ev) / steps
    check_status("after the timed launches", stream)
    return total_ms, kernel_ms, t_wall0, t_wall1, t_warm


def roofline_of(w: Workload, flops: float, algo_bytes: float, kernel_ms: float, region_ms: float, peaks, peak_src):
    """Achieved rate of the dominant kernel against its roofline: FP8 tensor
    peak (2 x the measured BF16 rate: the burst figure for timed regions
    under a second, the sustained one for longer) or the measured HBM copy
    bandwidth."""
    if w.bound == "tensor":
        burst = region_ms < BURST_REGION_MS
        bf16 = peaks["bf16_tflops"] if burst else peaks["bf16_tflops_sustained"]
        peak = FP8_PER_BF16 * bf16
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_basis": "FP8 = %g x %s BF16 %s (%.1f TF/s; timed region %.1f ms %s 1 s)"
                              % (FP8_PER_BF16, peak_src, "burst" if burst else "sustained", bf16, region_ms,
                                 "<" if burst else ">="),
                "frac_of_nominal_4500": achieved / 4500.0}
    else:
        achieved = algo_bytes / (kernel_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_basis": "%s HBM copy bandwidth" % peak_src,
                "frac_of_nominal_8000": achieved / 8000.0}
    roof.update({"algorithmic_flop": flops, "algorithmic_bytes": algo_bytes, "kernel_ms": kernel_ms})
    return roof


def host_us_per_call(w: Workload, s, stream, calls: int = 300) -> dict:
    """Host time of one enqueue through the C ABI from Python (pointers and
    sizes already marshalled; every call after the first finds its tensor
    maps in the library's cache), in a batch short of the launch queue's
    depth, and the floor of a ctypes call with as many arguments:
    fp8g_describe_plan (11 arguments, ~0.1 us of planning in C).  Their
    difference estimates the library's own cost per call, the CUDA launch
    included."""
    import ctypes
    import fp8_tensor_core_gb300 as fp8g
    lib = fp8g._lib.load()
    h = ctypes.c_void_p(stream.cuda_stream)
    if w.kind == "dense" and not w.gran:
        fn = lib.fp8_gemm_nt
        args = (s["A"].data_ptr(), s["B"].data_ptr(), s["D"].data_ptr(), w.M, w.N, w.K, w.fa, w.fb, w.flags, h)
    elif w.kind == "masked" and not w.gran:
        fn = lib.fp8_gemm_grouped_masked
        args = (s["A"].data_ptr(), s["B"].data_ptr(), s["D"].data_ptr(), s["mm"].data_ptr(), w.G, w.M_max, w.N, w.K,
                w.hint, w.fa, w.fb, w.flags, h)
    else:
        return {}
    import torch
    for _ in range(3):
        assert fn(*args) == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(calls):
        fn(*args)
    t1 = time.perf_counter()
    torch.cuda.synchronize()
    check_status("after the host-cost calls", stream)
    plan = fp8g._lib.Plan()
    pargs = (0, 1, 1, 256, 256, 0, 0, 0, 152, 232448, ctypes.byref(plan))
    t2 = time.perf_counter()
    for _ in range(calls):
        lib.fp8g_describe_plan(*pargs)
    t3 = time.perf_counter()
    host, floor = 1e6 * (t1 - t0) / calls, 1e6 * (t3 - t2) / calls
    return {"host_us_per_call": host, "ctypes_floor_us": floor, "c_abi_us_est": host - floor}


def run_per_config(device, stream, l2, peaks, peak_src, sampler, steps_tensor: int, steps_hbm: int,
                   use_graph: bool, known=None):
    """Every configuration of the pages through the same timing: kernel ms,
    achieved rate and roofline fraction (configs 3 in both B formats, config
    4 through SwapAB and token tiles, config 5 through both kernels with
    the automatic choice named)."""
    import torch
    import fp8_tensor_core_gb300 as fp8g
    out = []
    cache = {}
    for cfg, name in PER_CONFIG:
        if known and name in known:
            out.append(dict(known[name], config=cfg))
            continue
        w = make_workload(name)
        key = (w.kind, getattr(w, "M", None), w.N, w.K, w.fa, w.fb, w.seed, w.dist)
        inp = cache.get(key)
        if inp is None:
            inp = host_inputs(w)
            cache.clear()
            cache[key] = inp
        sets, _ = device_sets(w, inp, device, l2)
        call = make_call(w)
        steps = steps_tensor if w.bound == "tensor" else steps_hbm
        total_ms, kernel_ms, t0, t1, tw = timed_launches(call, sets, steps, 3, device, stream, use_graph)
        mm = inp.get("masked_m")
        roof = roofline_of(w, w.flops(mm), w.bytes(mm), kernel_ms, total_ms, peaks, peak_src)
        plan = planned_launch(w)
        e = {"config": cfg, "name": name, "kernel": KERNEL_NAMES[plan["kernel"]], "kernel_ms": kernel_ms,
             "achieved": roof["achieved"], "unit": roof["unit"], "frac": roof["frac"], "bound": roof["bound"],
             "steps": steps}
        if w.bound == "tensor":
            e["frac_of_nominal_4500"] = roof["frac_of_nominal_4500"]
        else:
            e["frac_of_nominal_8000"] = roof["frac_of_nominal_8000"]
            e["tflops"] = w.flops(mm) / (kernel_ms * 1e-3) / 1e12
        if name.startswith("smallm") or name.startswith("masked"):
            e.update(host_us_per_call(w, sets[0], stream))
        if name.startswith("smallm") and name.endswith(":swap"):
            base = name.rsplit(":", 1)[0]
            auto = planned_launch(make_workload(base))
            e["auto_picks"] = KERNEL_NAMES[auto["kernel"]]
        if sampler:
            c = sampler.summary(t0, t1, tw)
            if c["samples"]:
                e["sm_mhz"] = c["sm_mhz"]
        out.append(e)
        del sets
        torch.cuda.empty_cache()
    fp8g.fp8g_release_stream(stream)
    return out


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
    peaks, peak_src = load_peaks()

    # clock samples start now, so the sampler is running by the warm-up
    sampler = ClockSampler("GPU-" + str(props.uuid)) if rank == 0 else None
    inp = host_inputs(w)
    stream = torch.cuda.current_stream(device)
    sets, host = device_sets(w, inp, device, l2)
    n_sets = len(sets)
    torch.cuda.synchronize(device)
    call = make_call(w)

    # ---- timed region: exactly K steps --------------------------------------
    use_graph = args.graph != "off"
    total_ms, kernel_ms, t_wall0, t_wall1, t_warm = timed_launches(
        call, sets, args.steps, args.warmup, device, stream, use_graph,
        sync_world=lambda: barrier(world, device))
    total_ms_max = max_over_ranks(total_ms, world, device)
    kernel_ms_max = max_over_ranks(kernel_ms, world, device)
    clocks = sampler.summary(t_wall0, t_wall1, t_warm) if sampler else None

    mm = inp.get("masked_m")
    flops = w.flops(mm)
    algo_bytes = w.bytes(mm)
    value = world * args.steps * flops / (total_ms_max * 1e-3) / 1e12
    # The device-resident run's output (its last timed launch), kept on the
    # host before anything else writes the sets: the end-to-end output and
    # the oracle's sampled rows are compared with it.
    d_dev = sets[(args.warmup + args.steps - 1) % n_sets]["D"].view(torch.int16).cpu().numpy().view(np.uint16)

    # ---- end to end through the public API, host buffers ---------------------
    # Every step copies its inputs in from pinned host memory, runs the GEMM
    # through the public API and copies the whole of D back.  Consecutive
    # steps rotate over --e2e-streams streams, each with its own device and
    # host buffers (and its own stream-K scratch in the library), so one
    # step's copies overlap its neighbours' (the host link moves ~210 GB/s
    # one way, ~340 GB/s both ways at once).  Afterwards the last step's D,
    # as copied to the host, must equal the device-resident run's D bit for
    # bit (same inputs, same deterministic kernel).
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
                s_k["A"].copy_(host["A"], non_blocking=True)
                s_k["B"].copy_(host["B"], non_blocking=True)
                if w.gran:
                    s_k["sfa"].copy_(host["sfa"], non_blocking=True)
                    s_k["sfb"].copy_(host["sfb"], non_blocking=True)
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
        check_status("after the end-to-end run", stream)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, device)
        h2d = host["A"].numel() + host["B"].numel() + (mm_h.numel() * 4 if mm_h is not None else 0) + \
            (off_h.numel() * 4 if off_h is not None else 0)
        if w.gran:
            h2d += host["sfa"].numel() + host["sfb"].numel()
        d2h = pipe[0]["D_h"].numel() * 2
        # the last step's host copy against the device-resident run's output
        last = pipe[(e2e_steps - 1) % n_pipe]["D_h"].view(torch.int16).numpy().view(np.uint16)
        ref_dev = d_dev
        if w.kind == "masked":
            same = all(np.array_equal(last[g, :m], ref_dev[g, :m]) for g, m in enumerate(mm))
        elif w.kind == "contig":
            off = inp["offsets"]
            same = all(np.array_equal(last[off[g]:off[g + 1]], ref_dev[off[g]:off[g + 1]]) for g in range(w.G))
        else:
            same = np.array_equal(last, ref_dev)
        if not same:
            raise SystemExit("end-to-end output differs from the device-resident run's output")
        e2e = {"value": world * e2e_steps * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
               "streams": n_pipe, "check": "last step's D bit-identical to the device-resident run's D"}

    # ---- roofline of the dominant kernel -----------------------------------------
    roof = roofline_of(w, flops, algo_bytes, kernel_ms_max, total_ms_max, peaks, peak_src)
    plan = planned_launch(w)
    roof.update({"traffic": profiled_traffic(w.name), "kernel": KERNEL_NAMES[plan["kernel"]], "plan": plan})
    roof = {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")} | \
        {k: v for k, v in roof.items() if k not in ("bound", "achieved", "peak", "unit", "frac", "traffic")}

    # ---- CPU baseline (rank 0, N = 1 only) ----------------------------------------
    # The oracle, as it stands, on a bounded sample of the same workload; the
    # rows (groups) it computed are then compared with the device run's D.
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, s, cores, desc, parity = oracle_sample(w, inp, args.cpu_budget, check_against=d_dev)
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": desc + "; %.1f s" % s, "parity": parity}
        if not parity.startswith("ok"):
            raise SystemExit("device output differs from the oracle on the sampled rows: " + parity)

    per_config = None
    if rank == 0 and world == 1 and not args.no_per_config:
        del sets
        torch.cuda.empty_cache()
        known = {w.name: {"name": w.name, "kernel": roof["kernel"], "kernel_ms": kernel_ms_max,
                          "achieved": roof["achieved"], "unit": roof["unit"], "frac": roof["frac"],
                          "bound": roof["bound"], "steps": args.steps} |
                 ({"frac_of_nominal_4500": roof["frac_of_nominal_4500"]} if w.bound == "tensor" else
                  {"frac_of_nominal_8000": roof["frac_of_nominal_8000"]})}
        per_config = run_per_config(device, stream, l2, peaks, peak_src, sampler, args.per_config_steps,
                                    args.per_config_steps_hbm, use_graph, known=known)
    if sampler:
        sampler.stop()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8_e4m3" if w.fb == 0 else "fp8_e4m3xe5m2", "data": "synthetic",
            "config": {"workload": w.desc, "name": w.name, "flags": hex(w.flags),
                       "l2": "%d rotating input+output sets of %.1f MB (>= 3x the %d MB L2)"
                             % (n_sets, set_bytes_of(w) / 1e6, l2 >> 20),
                       "parallelism": "independent shard per GPU" if world > 1 else "single GPU"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "timing": "one CUDA graph of K launches" if use_graph else "K direct launches, events per launch",
            "clocks": clocks,
            "per_config": per_config,
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


def run_mma_microbench() -> int:
    """Compile bench_mma.cu for sm_103a next to the library and run it."""
    from fp8_tensor_core_gb300 import build as cuda_build
    os.makedirs(cuda_build.BUILD, exist_ok=True)
    exe = os.path.join(cuda_build.BUILD, "bench_mma")
    src = os.path.join(ROOT, "bench_mma.cu")
    cmd = [cuda_build.nvcc()] + cuda_build.ARCH + ["-O3", "-std=c++17", "-I", cuda_build.CSRC, "-o", exe, src]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        return r.returncode
    return subprocess.run([exe]).returncode


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
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
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config array (every configuration of the pages, timed briefly)")
    ap.add_argument("--per-config-steps", type=int, default=20,
                    help="timed launches per tensor-bound configuration in per_config")
    ap.add_argument("--per-config-steps-hbm", type=int, default=100,
                    help="timed launches per HBM-bound configuration in per_config")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--mma-microbench", action="store_true",
                    help="build and run bench_mma.cu (tensor-core instruction costs) instead of a GEMM")
    args = ap.parse_args(argv)
    if args.mma_microbench:
        return run_mma_microbench()
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
