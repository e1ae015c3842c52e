"""Host logic of bench.py: workload arithmetic, roofline inputs, and the
multi-rank path (max over ranks, barrier, per-rank shards) on world-size-2
gloo process groups on CPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

import __graft_entry__  # noqa: F401
import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_arithmetic.txt")


def golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            vals[k] = float(int(v, 16)) if v.startswith("0x") else float(v)
    return vals


def test_page_roofline_arithmetic():
    """Square GEMM intensity 2n/3 and the ridge point, as printed on the
    DeepGEMM page §2.2, from the bench's own FLOP and byte counts (bytes as
    the page counts them: one byte per element of A, B and C)."""
    g = golden()
    n = int(g["square_n"])
    w = bench.Workload("sq", "dense", "", M=n, N=n, K=n)
    flops = w.flops()
    page_bytes = 3.0 * n * n
    assert flops == 2.0 * n ** 3
    assert abs(flops / page_bytes - g["square_intensity_approx"]) < 5
    ridge = g["ridge_tflops"] * 1e12 / (g["ridge_tbs"] * 1e12)
    assert abs(ridge - g["ridge_approx"]) < 5


def test_page_tile_bytes():
    g = golden()
    assert 128 * 32 == g["tile_a_bytes"]
    assert 32 * 256 == g["tile_b_bytes"]
    assert 2 * (128 * 32 + 32 * 256) == g["double_buffer_bytes"]


def test_page_64bit_offset_example():
    """MLS page, Bug 1: the carry of a 64-bit add must not be lost."""
    g = golden()
    base, off = int(g["base"]), int(g["offset"])
    assert base + off == int(g["correct"])
    low_only = (base & ~0xFFFFFFFF) | ((base + off) & 0xFFFFFFFF)
    assert low_only == int(g["low_word_only"])
    assert int(g["correct"]) - low_only == int(g["delta"])


def test_page_m_utilisation():
    g = golden()
    assert g["natural_m"] / g["instr_m"] == g["utilisation"]


def test_workload_bytes_and_flops():
    w = bench.make_workload("masked")
    mm = [0, 5, 32, 0, 1]
    w.G = len(mm)
    assert w.flops(mm) == 2.0 * 38 * 4096 * 7168
    live = 3
    assert w.bytes(mm) == live * 4096 * 7168 + 38 * 7168 + 2 * 38 * 4096
    d = bench.make_workload("dense4096")
    assert d.bytes() == 4096 * 4096 * 4
    s = bench.make_workload("smallm:8:7168:16384:noswap")
    assert s.flags == 2 and s.M == 8
    p = bench.make_workload("proj:7168:18432:e5m2")
    assert p.fb == 1 and p.M == 8192


def test_shards_differ_per_rank():
    a = bench.make_workload("dense4096", rank=0)
    b = bench.make_workload("dense4096", rank=1)
    assert a.seed != b.seed


def test_traffic_lookup_tracks_kernel_sources(tmp_path, monkeypatch):
    h = bench.kernel_source_hash()
    assert len(h) == 16
    t = bench.profiled_traffic("dense4096")
    # valid only for the hash it was captured with
    lines = open(os.path.join(ROOT, "profiles", "traffic.txt")).read()
    if h in lines:
        assert t is not None
    else:
        assert t is None


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


_WORKER = r"""
import os, sys, json
sys.path.insert(0, %(root)r)
import torch.distributed as dist
import bench
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%(port)d",
                        rank=int(sys.argv[1]), world_size=2)
r = dist.get_rank()
bench.barrier(2)
m = bench.max_over_ranks(1.0 + 10.0 * r, 2)
w = bench.make_workload("dense4096", rank=r)
print(json.dumps({"rank": r, "max": m, "seed": w.seed}))
dist.destroy_process_group()
"""


def test_two_rank_gloo_max_and_barrier(tmp_path):
    port = _free_port()
    script = tmp_path / "w.py"
    script.write_text(_WORKER % {"root": ROOT, "port": port})
    procs = [subprocess.Popen([sys.executable, str(script), str(r)], stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    res = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    assert all(r["max"] == 11.0 for r in res)
    assert res[0]["seed"] != res[1]["seed"]


def test_reference_arm_rank1_does_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert p.returncode == 0
    assert p.stdout.strip() == ""


def test_reference_arm_line(tmp_path):
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "cube256", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    line = json.loads(p.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True


def test_workload_variants_parse():
    """masked:mode, grouped:G:m:N:K[:mode] and the :bs / :bs32 block-scale
    suffix give the documented shapes, flags, scale granularity and bytes."""
    m = bench.make_workload("masked:noswap")
    assert m.flags == 2 and m.G == 32 and m.hint == 32 and m.gran == 0
    assert bench.make_workload("masked").flags == 1 and bench.make_workload("masked:auto").flags == 0
    g = bench.make_workload("grouped:16:96:4096:7168:swap")
    assert (g.G, g.M_max, g.N, g.K, g.flags, g.hint) == (16, 96, 4096, 7168, 1, 96)
    inp = bench.host_inputs(g)
    assert inp["masked_m"].tolist() == [96] * 16
    b = bench.make_workload("dense4096:bs")
    assert b.gran == 128 and b.kernel == "k_gemm_mn" and b.name == "dense4096:bs"
    ks = 4096 // 128
    assert b.bytes() == 4096 * (4096 + ks) * 2 + 2 * 4096 * 4096
    b32 = bench.make_workload("smallm:16:7168:16384:swap:bs32")
    assert b32.gran == 32 and b32.M == 16 and b32.flags == 1
    c = bench.make_workload("contig:8:64:512:1024:noswap")
    assert (c.kind, c.G, c.M_max, c.N, c.K, c.flags, c.hint) == ("contig", 8, 64, 512, 1024, 2, 64)
    inp = bench.host_inputs(c)
    assert inp["A"].shape == (8 * 64, 1024) and inp["B"].shape == (8, 512, 1024)
    assert inp["offsets"].tolist() == [64 * g for g in range(9)]
    assert c.flops(inp["masked_m"]) == 2.0 * 8 * 64 * 512 * 1024
    assert c.bytes(inp["masked_m"]) == 8 * 512 * 1024 + 8 * 64 * 1024 + 2 * 8 * 64 * 512
    with pytest.raises(SystemExit):
        bench.make_workload("contig:8:64:512:1024:bs")


def test_block_scale_recipe():
    """Per-token scales vary per row; weight scales are constant over each
    128x128 block (gran 128); all codes in [120, 134]; ld is padded to 16."""
    import numpy as np
    w = bench.make_workload("masked:bs")
    w.G = 3                                  # a small instance of the same recipe
    sc = bench.block_scales(w)
    sfa, sfb = sc["sf_a"], sc["sf_b"]
    assert sfa.shape == (3, 7168 // 128, 128) and sfb.shape == (3, 7168 // 128, 4096)
    assert sfa.min() >= 120 and sfa.max() <= 134 and sfb.min() >= 120 and sfb.max() <= 134
    blocks = sfb.reshape(3, 56, 32, 128)
    assert np.all(blocks == blocks[..., :1])          # one code per 128 rows
    assert len(np.unique(sfa[0, 0])) > 1
    w32 = bench.make_workload("smallm:1:7168:16384:bs32")
    sc32 = bench.block_scales(w32)
    assert sc32["sf_a"].shape == (1, 16384 // 32, 16) and sc32["sf_b"].shape == (1, 512, 7168)


def test_planned_launch_names_the_kernel(monkeypatch):
    """The bench line's kernel comes from the library's planner (here for a
    described GB300, so no device is needed)."""
    from fp8_tensor_core_gb300 import build as cuda_build
    import fp8_tensor_core_gb300 as fp8g
    cuda_build.build()
    real = fp8g.fp8g_describe_plan
    monkeypatch.setattr(fp8g, "fp8g_describe_plan",
                        lambda *a, **k: real(*a, sms=152, smem_optin=232448))
    for name, kernel in [("dense4096", "k_gemm_mn2"), ("masked", "k_gemm_swap"), ("masked:noswap", "k_gemm_mn"),
                         ("smallm:1:24576:1536", "k_gemm_mn"), ("smallm:16:7168:16384", "k_gemm_swap"),
                         ("contig:32:256:4096:7168", "k_gemm_mn2"), ("dense4096:bs", "k_gemm_mn"),
                         ("grouped:16:160:4096:7168:auto", "k_gemm_swap")]:
        plan = bench.planned_launch(bench.make_workload(name))
        assert bench.KERNEL_NAMES[plan["kernel"]] == kernel, (name, plan)


def test_mma_microbench_builds(tmp_path):
    """bench_mma.cu (bench.py --mma-microbench) compiles for sm_103a against
    the library's PTX wrappers (no GPU needed to build it)."""
    from fp8_tensor_core_gb300 import build as cuda_build
    out = tmp_path / "bench_mma"
    cmd = [cuda_build.nvcc()] + cuda_build.ARCH + ["-O3", "-std=c++17", "-I", cuda_build.CSRC, "-o", str(out),
                                                   os.path.join(ROOT, "bench_mma.cu")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert out.exists()
