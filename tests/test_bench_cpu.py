"""Host-side checks of bench.py: the reference arm's JSON line (the oracle
timed on this host's cores), its behaviour under a two-rank torchrun (rank
0 alone prints), and the slowest-rank aggregation over a two-rank gloo
process group.  No GPU is used."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

SMALL = ["--config", "q06_layer_b1_ctx1024", "--steps", "1", "--warmup", "0"]


def _json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"] + SMALL,
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1, r.stdout
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 1
    assert d["config"]["workload"] == "q06_layer_b1_ctx1024"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    # the same oracle on one thread, reported beside the all-cores figure
    st = cb["single_thread"]
    assert st["cores"] == 1 and st["unit"] == "GB/s" and st["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert abs(d["ms_per_step"] * 1e-3 * d["value"] * 1e9 - _algo_bytes("q06_layer_b1_ctx1024")) \
        < 1e-6 * _algo_bytes("q06_layer_b1_ctx1024")


def _algo_bytes(name):
    from pdl_persistent_megakernel_gb300 import bytes_model, synth
    return bytes_model.algorithmic_bytes(synth.CONFIGS[name])["total"]


def test_reference_arm_two_ranks_rank0_prints():
    """Under torchrun with two ranks the reference arm runs on rank 0 only:
    one JSON line, both ranks exit 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29631",
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"] + SMALL
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def _max_rank(rank, ws, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    q.put((rank, bench.max_over_ranks(10.0 + 5.0 * rank, ws)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    """The per-schedule and end-to-end times are the slowest rank's."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_max_rank, args=(r, 2, 29632, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = dict(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 15.0, 1: 15.0}


def test_max_over_ranks_single():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_sources_hash_gates_traffic():
    """The DRAM traffic figure in profiles/traffic.json is used only while the
    device sources hash to the value recorded with it."""
    import bench
    h = bench.kernel_sources_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        tj = json.load(f)
    assert {"workload", "kernel", "bytes_per_launch", "sources_sha256_16"} <= set(tj)


def test_trace_timeline_from_a_synthetic_table():
    """bench.py --trace summarises a trace table: times from the earliest
    share start, medians and maxima per slot, per-unit time of the loop, and
    None for slots a share never stamps (a norm has no unit loop)."""
    import numpy as np
    import bench
    ops = [("add_rmsnorm1", 2, 0), ("o_proj", 3, 0)]
    tr = np.zeros((2, 4, 8), dtype=np.uint64)
    base = 10_000_000
    # norm shares: start, dependency release, exit, one unit each
    tr[0, 0, [0, 1, 4, 5]] = [base, base + 500, base + 3000, 1]
    tr[0, 1, [0, 1, 4, 5]] = [base + 100, base + 600, base + 3500, 1]
    # projection shares: 5 units, first and last unit 4 us apart (1 us each)
    for c in range(3):
        s = base + 4000 + 100 * c
        tr[1, c] = [s, s + 200, s + 1000, s + 5000, s + 7000, 5, s + 6000, 0]
    tl = bench.trace_timeline(tr, ops)
    norm, proj = tl["ops"]
    assert norm["start_min"] == 0.0 and norm["end_max"] == 3.5
    assert norm["first_med"] is None and norm["loop_end_max"] is None
    assert norm["units"] == 2 and norm["us_per_unit_med"] is None
    assert proj["start_min"] == 4.0 and proj["start_max"] == 4.2 and proj["deps_med"] == 4.3
    assert proj["us_per_unit_med"] == 1.0 and proj["units"] == 15
    assert proj["reduce_max"] == 10.2 and proj["end_max"] == 11.2 and tl["span_us"] == 11.2


def test_single_thread_sample_is_bounded():
    """The one-thread oracle sample is skipped, with the estimate stated,
    when the all-cores time x threads is over the limit."""
    import bench
    st = bench.single_thread_baseline(None, None, None, 1e9, sec_all=4.0, threads_all=16)
    assert st["value"] is None and st["cores"] == 1 and "skipped" in st["sample"]


def test_l2_auto_streams_only_workloads_twice_the_l2():
    """--l2 auto runs steps back to back only when one step reads at least
    1.5 times the L2 size (the Q8 FP8 layer at M = 16, ctx 8192: 260.7 MB); a
    smaller step (the Q0.6B layer at batch 1: 35.7 MB) gets the clean flush.
    Nothing is allocated before the first call."""
    import bench
    from pdl_persistent_megakernel_gb300 import bytes_model, synth
    big = bytes_model.algorithmic_bytes(synth.CONFIGS["q8_layer_m16_ctx8192_fp8"])["total"]
    small = bytes_model.algorithmic_bytes(synth.CONFIGS["q06_layer_b1_ctx1024"])["total"]
    assert big >= 1.5 * 132.2e6 > small
    f = bench.L2Flush("auto", "cpu", big)
    assert f.mode == "stream" and f.w is None
    f()
    assert f.w is None
    g = bench.L2Flush("auto", "cpu", small)
    assert g.mode == "clean" and g.w is None
    assert bench.L2Flush("auto", "cpu").mode == "clean"
    assert bench.L2Flush("flush", "cpu", big).mode == "flush"
    assert "1.5 times" in f.describe() and "read of another buffer" in g.describe()
