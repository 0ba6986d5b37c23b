"""The multi-GPU bench path on CPU: two gloo ranks, no GPU.

The bench runs one replica of the workload per rank (the attention problems are
independent, so there is no data exchange) and reports the whole job: every
rank's FLOPs over the slowest rank's time.  These tests drive the helpers that
do that across two real processes, and check that only rank 0 of the reference
arm does any work.
"""

import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = [2.0, 3.5][rank]  # rank 1 is the slower replica
        ms_max = bench.max_over_ranks(local_ms, dist, "cpu")
        value = bench.whole_job_tflops(1.0e12, world, ms_max)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms_max": ms_max, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_slowest_time_and_total_work(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r in res:
        assert r["ms_max"] == 3.5                         # max over ranks, seen by every rank
        assert r["value"] == pytest.approx(2 * 1.0e12 / 3.5e-3 / 1e12)  # both ranks' FLOPs / slowest time


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(1.25, None, "cpu") == 1.25
    assert bench.whole_job_tflops(2.0e12, 1, 1.0) == pytest.approx(2000.0)


def _ref_rank_main(rank, world, out_dir):
    sys.path.insert(0, ROOT)
    import argparse
    import contextlib
    import io

    import bench
    from online_softmax_14_b300.inputs import Workload

    w = Workload("tiny_causal", "bf16", 1, 2, 128, 64, True)
    args = argparse.Namespace(seed=0, steps=2, warmup=1, ref_budget_s=1.0)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, w, rank, world)
    with open(os.path.join(out_dir, f"ref{rank}.txt"), "w") as f:
        f.write(buf.getvalue())


def test_reference_arm_runs_on_rank0_only(tmp_path):
    mp.start_processes(_ref_rank_main, args=(2, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    out0 = (tmp_path / "ref0.txt").read_text().strip().splitlines()
    out1 = (tmp_path / "ref1.txt").read_text().strip()
    assert out1 == ""                                     # other ranks exit without work
    line = json.loads(out0[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_forward_source_digest_covers_kernel_and_launch_only():
    """The digest that guards the recorded DRAM traffic covers the forward's
    headers and the host functions that shape its launch: the text of such a
    function is extracted up to its matching brace, and a function that is not
    there contributes nothing."""
    import bench

    src = "int a() { return 1; }\nfa_status launch_tc(int x) {\n  if (x) { return 2; }\n  return 3;\n}\nint b() {}\n"
    assert bench._function_text(src, "fa_status launch_tc(") == (
        "fa_status launch_tc(int x) {\n  if (x) { return 2; }\n  return 3;\n}")
    assert bench._function_text(src, "int missing(") == ""
    digest = bench.kernel_src_digest()
    assert len(digest) == 16 and int(digest, 16) >= 0
    # every host function the digest names is present in the library source
    lib = open(os.path.join(ROOT, "online_softmax_14_b300", "csrc", "fa_lib.cu"), encoding="utf-8").read()
    for head in bench.FWD_HOST_FUNCTIONS:
        assert bench._function_text(lib, head).startswith(head)


def test_recorded_forward_traffic_matches_the_current_sources():
    """The DRAM traffic bench.py reports for the headline workload was captured
    with ncu on the forward sources as they are now: a change to the forward's
    headers or launch code without a new capture fails here rather than
    silently turning the reported traffic into null."""
    import bench

    rec = bench.NCU_TRAFFIC["bf16_causal_B2_H32_N8192_d128"]
    assert rec["src_digest"] == bench.kernel_src_digest()
    # the algorithmic bytes of that workload are 539 MB; the capture is within 10 %
    assert 539e6 <= rec["bytes"] <= 1.1 * 539e6
