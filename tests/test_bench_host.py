"""Host-side logic of bench.py that needs no GPU: pair counts, clock parsing, and the max over
ranks of the multi-replica run (two gloo ranks on the CPU)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_pair_counts():
    assert bench.logical_pairs(100_000, 100_000) == 3 * 10**10
    assert bench.evaluated_pairs(100_000, 100_000) == 10**10 + 2 * (100_000 * 99_999 // 2)


def test_clock_summary_parses_nvidia_smi_lines():
    cs = bench.ClockSampler(0, None)
    cs.lines = ["0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active",
                "0, 1965, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
                "0, 300, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = cs.summary()
    assert s["sm_max_mhz"] == 2070 and s["sm_mhz"] == pytest.approx(2017.5) and s["reasons"] == ["sw_power_cap"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    out = bench.reduce_max([1.0 + rank, 10.0 - rank], world)
    bench.barrier(world)
    q.put((rank, out))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = dict(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
    assert res[0] == res[1] == [2.0, 10.0]


def test_option_arguments_parse_to_library_options():
    import bench
    assert bench.parse_options([]) == {}
    assert bench.parse_options(["exact=0", "layout=3"]) == {"exact": 0, "layout": 3}
    with pytest.raises(SystemExit):
        bench.parse_options(["exact"])


def test_kernel_hash_ignores_comments_but_not_code():
    import bench
    a = 'int f() { return 1; } // one\n/* block */\nconst char* s = "a//b";\n'
    b = 'int f() { return 1; }\n\n// another comment\nconst char* s = "a//b";   \n'
    c = 'int f() { return 2; }\nconst char* s = "a//b";\n'
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)
    assert '"a//b"' in bench.code_only(a)


def test_reference_arm_prints_the_contract_line():
    # the reference arm times the fp64 oracle on the host cores; it needs no GPU
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--ref-rows", "10"], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 3
    assert line["unit"] == "Gpairs/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("pages-shape-100k")
    # both arms print the same workload description (launch facts go elsewhere in our arm)
    import synth
    c = synth.config(1)
    assert line["config"] == bench.bench_config(c, line["config"]["workload"], {})
    assert "grid" not in line["config"] and "threads" not in line["config"]


def test_executed_roofline_from_a_record():
    rec = {"per_launch": {"DD": {"thread_inst_executed": 1.0e11}, "DR": {"thread_inst_executed": 2.0e11},
                          "RR": {"thread_inst_executed": 1.0e11}}, "issue_active_pct": 88.0}
    # 4e11 instructions in 10 ms = 40 T inst/s
    r = bench.executed_roofline(rec, 10.0, 3.2e11, 40.0)
    assert r["achieved"] == pytest.approx(40.0) and r["frac"] == pytest.approx(1.0)
    assert r["inst_overhead"] == pytest.approx(1.25) and r["ncu_issue_active_pct"] == 88.0
    assert bench.executed_roofline(None, 10.0, 1.0, 40.0) is None
    assert bench.executed_roofline({"per_launch": {"DD": {}}}, 10.0, 1.0, 40.0) is None
