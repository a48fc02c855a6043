"""The benchmark's JSON line: one line with the keys and types the benchmark
contract asks for -- on the CPU through the reference arm (`bench.py --impl
reference`, which times the oracle and needs no GPU), and on a GPU through a
short run of the CUDA path."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(*extra):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "1",
           "--workload", "tiny_n512_h256_e16_k2", *extra]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_line_has_the_contract_keys():
    d = run_reference()
    assert d["impl"] == "reference"
    for k, t in [("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                 ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                 ("dtype", str), ("data", str), ("config", dict), ("cpu_baseline", dict), ("e2e", dict)]:
        assert isinstance(d[k], t), k
    assert d["vs_baseline"] is None
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny_n512_h256_e16_k2"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert d["value"] > 0 and d["higher_is_better"] is True


def test_reference_line_names_the_variant():
    d = run_reference("--residual", "--route-stats")
    assert "residual" in d["config"]["combine"]
    assert "moe_route_stats" in d["config"]["route"]


def test_reference_arm_under_torchrun_prints_one_line():
    # the launch used for N > 1: rank 0 alone runs the reference arm and prints
    # its line, the other rank exits 0 without work (no GPU, no process group)
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1",
           "--workload", "tiny_n512_h256_e16_k2"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


@pytest.mark.gpu
def test_gpu_line_has_the_contract_keys():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5", "--warmup", "3", "--no-cpu-baseline",
           "--e2e-steps", "16", "--no-torch-naive"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["value"] > 0
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert "traffic" in r
    c = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(c)
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    # the default workload is the largest one: route, the dispatch's metadata launch,
    # the row copy in a launch of its own (>= 256 MiB) and the combine
    import moe_inputs as mi
    assert d["config"]["workload"] == mi.BENCH_WORKLOAD == "skewed_zipf_n65536_h4096_e64_k2"
    assert d["gpu_launches"] == 4 * d["steps"]
    assert d["roofline"]["kernel"] in ("route", "dispatch", "combine")
    assert d["roofline"]["traffic_source"].startswith("profiles/dram_traffic.csv")


@pytest.mark.gpu
def test_gpu_line_of_the_fused_workload():
    # at N=2048, H=1024 the router runs split-K and route + dispatch is one launch:
    # two kernels per step
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "n2048_h1024_e64_k2", "--steps", "5",
           "--warmup", "3", "--no-cpu-baseline", "--e2e-steps", "16", "--no-torch-naive"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["gpu_launches"] == 2 * d["steps"]
    assert "route_dispatch" in d["kernels"] and d["kernels"]["route_dispatch"]["launches"] == 1
    assert d["roofline"]["kernel"] in ("route_dispatch", "combine")


GPU_VARIANTS = {
    "apart": (["--apart"], lambda c: c["calls"] == "moe_route, moe_dispatch, moe_combine"),
    "residual": (["--residual"], lambda c: "residual" in c["combine"]),
    "route_stats": (["--route-stats"], lambda c: "moe_route_stats" in c["route"]),
    "ue8m0": (["--workload", "moe_layer_n16384_h2048_e128_k8_fp8", "--scale-format", "ue8m0"],
              lambda c: c["fp8_scales"] == "ue8m0"),
    "ep": (["--workload", "n4096_h2048_e64_k4", "--ep-size", "4"], lambda c: "ep_size 4" in c["dispatch"]),
}


@pytest.mark.gpu
@pytest.mark.parametrize("variant", sorted(GPU_VARIANTS))
def test_gpu_variant_lines(variant):
    # every bench variant still runs end to end and names itself in its config
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    extra, names_itself = GPU_VARIANTS[variant]
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5", "--warmup", "3", "--no-cpu-baseline",
           "--e2e-steps", "8", "--no-torch-naive", *extra]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert names_itself(d["config"]), d["config"]
    assert d["value"] > 0 and d["e2e"]["value"] > 0 and d["gpu_launches"] >= 2 * d["steps"]
    r = d["roofline"]
    assert r["peak"] > 0 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9


def test_source_digest_ignores_comments_only():
    import bench
    a = 'int f(int x) { // add one\n  return x + 1; /* done */ }\nconst char *s = "// kept";\n'
    b = '/* header */\nint f(int x) {\n    return x + 1;\n}\nconst char *s = "// kept";  // trailing\n'
    c = 'int f(int x) { return x + 2; }\nconst char *s = "// kept";\n'
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)
    assert '"// kept"' in bench.code_only(a)
    for k in ("route", "dispatch", "combine", "route_dispatch"):
        assert len(bench.source_digest(k)) == 16


def test_record_traffic_parses_an_ncu_log(tmp_path):
    # the traffic table is written from ncu's own CSV log: per call the smallest of its
    # launches, the dispatch call as its counting-sort launch plus the permute launch that
    # follows it, units converted, every row stamped with the kernel source's digest
    import bench
    import moe_inputs as mi
    hdr = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",'
           '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"')

    def launch(i, name, rd, wr, unit="byte"):
        row = f'"{i}","1","python3","h","{name}","1","7","(1, 1, 1)","(1, 1, 1)","0","10.3","m",'
        return [row + f'"dram__bytes_read.sum","{unit}","{rd}"', row + f'"dram__bytes_write.sum","{unit}","{wr}"',
                row + '"gpu__time_duration.sum","ns","1000"']

    rows = ["==PROF== Connected", hdr]
    rows += launch(0, "void route_tc_kernel<2, 0, 0>(CUtensorMap_st)", 1000, 10)
    rows += launch(1, "void dispatch_fused_kernel<0, 0, 1>(FusedParams)", 5, 0)
    rows += launch(2, "void permute_kernel<1, 0, 16>(const uint4 *)", 200, 400)
    rows += launch(3, "void combine_kernel<2, 8, 0>(const uint4 *)", 0.5, 0.25, unit="Kbyte")
    rows += launch(4, "void route_tc_kernel<2, 0, 0>(CUtensorMap_st)", 990, 10)
    log = tmp_path / "launches.csv"
    log.write_text("\n".join(rows) + "\n")
    table = tmp_path / "traffic.csv"
    table.write_text("kernel,workload,dram_bytes_per_launch,source_digest,read,write,algorithmic_bytes,capture\n"
                     "route,other,1,x,1,0,1,old\n")
    w = mi.WORKLOADS["tiny_n512_h256_e16_k2"]
    calls = bench.record_traffic(str(log), w, str(table))
    assert calls == {"route": (990.0, 10.0), "dispatch": (205.0, 400.0), "combine": (500.0, 250.0)}
    assert bench.ncu_traffic("route", w.name, str(table)) == 1000.0
    assert bench.ncu_traffic("dispatch", w.name, str(table)) == 605.0
    assert bench.ncu_traffic("combine", w.name, str(table)) == 750.0
    assert bench.ncu_traffic("route", "other", str(table)) is None      # digest "x" is not the source's
    assert "route,other,1,x,1,0,1,old" in table.read_text()             # other workloads' rows kept
