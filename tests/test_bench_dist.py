"""The multi-rank side of bench.py on CPU: two gloo ranks (no GPU), checking
the barrier, the max over ranks of the step time and the whole-job value."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    r, local, w = bench.dist_env()
    assert (r, local, w) == (rank, rank, world)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    ms = 2.0 + rank  # rank 1 is the slower one
    ms_max, value = bench.whole_job(1e9, ms, w, torch.device("cpu"), 1e9)
    out[rank] = (ms_max, value)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        for p in procs:
            if p.is_alive():
                p.kill()
                pytest.fail("a rank did not finish")
            assert p.exitcode == 0
        res = dict(out)
    # both ranks see the slower rank's 3 ms; 2 ranks x 1 GB each per 3 ms = 666.7 GB/s
    for r in range(world):
        ms_max, value = res[r]
        assert ms_max == pytest.approx(3.0)
        assert value == pytest.approx(2 * 1e9 / 3e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    import bench

    ms_max, value = bench.whole_job(5e12, 10.0, 1, torch.device("cpu"), 1e12)
    assert ms_max == 10.0 and value == pytest.approx(500.0)


def test_bench_launch_count_follows_the_library_split_plan():
    """bench.py counts one launch per decode call when a KV head's splits fit a
    cluster (<= 8) and two otherwise; its copy of the split plan must agree with
    the library's, read back here from the workspace size the library asks for
    (no GPU: the library plans for 148 SMs when it cannot query the device)."""
    import bench
    import streaming_attention_gb300 as sa
    from streaming_attention_gb300 import build as B
    from streaming_attention_gb300.inputs import DECODE_GQA

    B.build()

    def splits_from_workspace(w):
        nb = sa.attn_workspace_bytes_ex(w.B, w.Hq, w.Hkv, w.M, w.N, w.D, w.causal, w.window, sa.PATH_DECODE)
        rows, D = w.B * w.Hq * w.M, w.D
        up = lambda x: (x + 255) // 256 * 256  # noqa: E731
        for S in range(1, 4097):
            if 2 * up(rows * S * 4) + up(rows * S * D * 4) == nb:
                return S
        raise AssertionError(f"no split count gives {nb} bytes")

    # the SM count the library plans for: the device's, or 148 without one
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148
    cases = [DECODE_GQA, DECODE_GQA.with_(B=1, Hkv=1, Hq=8, N=9000, window=0),
             DECODE_GQA.with_(B=2, Hkv=2, Hq=8, N=1000, window=0)]
    for w in cases:
        assert bench.decode_splits(w, sms) == splits_from_workspace(w), w
    assert bench.path_launches("decode", DECODE_GQA, sms) == 1
    assert bench.path_launches("decode", cases[1], sms) == 2
    assert bench.path_launches("prefill_or_simt", DECODE_GQA, sms) == 1


def _run_bench(args, env_extra=None):
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, **(env_extra or {}))
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=root, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    return [json.loads(ln) for ln in lines]


@pytest.mark.parametrize("workload,unit", [("tiny_b1_h2_64x64_d64_bf16", "TFLOP/s"),
                                           ("decode_gqa_b8_hq32_hkv8_m1_n8192_w4096_d128_bf16", "GB/s")])
def test_reference_arm_prints_one_contract_line(workload, unit):
    """The reference arm (the FP64 oracle on the host cores) needs no GPU: one
    JSON line with the contract's keys, in the unit of the workload's metric."""
    (line,) = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-seconds", "1",
                          "--workload", workload])
    assert line["impl"] == "reference" and line["unit"] == unit and line["value"] > 0
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling", "dtype",
                "data", "config"):
        assert key in line, key
    assert line["steps"] == 1 and line["warmup"] == 3 and line["vs_baseline"] is None
    assert line["config"]["workload"] == workload
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    assert _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-seconds", "1",
                       "--workload", "tiny_b1_h2_64x64_d64_bf16"], {"RANK": "1", "WORLD_SIZE": "2"}) == []
