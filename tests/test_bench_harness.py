"""bench.py host logic: timing harness (1 and 2 gloo ranks) and workload arithmetic."""

import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
import synth


def test_dense_flops_of_the_128k_prefill():
    w = synth.WORKLOADS["prefill_128k_gqa8"]
    assert bench.prefill_dense_flops(w) == 4.0 * 64 * 128 * (131072 * 131073 // 2)
    assert abs(bench.prefill_dense_flops(w) - 2.8147e14) / 2.8147e14 < 1e-3
    w0 = synth.WORKLOADS["prefill_1k_d64"]
    assert bench.prefill_dense_flops(w0) == 4.0 * 64 * (1024 * 1025 // 2)
    wn = w0.with_(causal=False, Sq=100, Skv=300)
    assert bench.prefill_dense_flops(wn) == 4.0 * 64 * 100 * 300
    wc = w0.with_(Sq=100, Skv=300)  # bottom-right aligned: query i sees 201 + i keys
    assert bench.prefill_dense_flops(wc) == 4.0 * 64 * sum(201 + i for i in range(100))


def test_exec_flops_and_decode_bytes():
    w = synth.WORKLOADS["prefill_128k_gqa8"]
    per = 2 * 128 * 128 * 128
    assert bench.prefill_exec_flops(w, 10, 4, 128, 128) == per * 10 + per * 6
    wd = synth.WORKLOADS["decode_128k_gqa8"]
    nblk = 8 * 8 * 2048
    dense = bench.decode_bytes(wd, nblk, 16)
    k_bytes = 8 * 8 * 131072 * 128 * 2
    assert dense > 2 * k_bytes and dense < 2 * k_bytes * 1.01
    assert bench.decode_bytes(wd, 0, 16) < 0.51 * dense


def test_timed_loop_single_process():
    calls = []
    sec, wall = bench.timed_loop(lambda i: calls.append(i), 4, 3, lambda: None, lambda: 1.25,
                                 False)
    assert calls == [0, 1, 2, 0, 1, 2, 3]
    assert sec == 1.25 and wall >= 0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    steps = []
    sec, _ = bench.timed_loop(lambda i: steps.append(i), 5, 3, lambda: None,
                              lambda: 1.0 + rank, True)
    ws, r, lr = bench.dist_env()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"sec": sec, "steps": len(steps), "env": [ws, r, lr]}, f)
    dist.destroy_process_group()


def test_timed_loop_two_gloo_ranks_take_the_max(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert d["sec"] == 2.0           # max over ranks of (1 + rank)
        assert d["steps"] == 8           # warm-up + timed
        assert d["env"] == [2, r, r]


def test_reference_arm_non_zero_rank_exits_quietly(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_oracle_line(capsys):
    # the reference arm times the oracle on the host: one JSON line, no GPU needed
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0",
                       "--ref-budget", "0.01"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert "9 splits" in line["cpu_baseline"]["sample"]
    # the same config object as our arm's, at the step's thresholds and split count
    assert line["config"] == bench.workload_config(bench.PREFILL_LAMBDA, bench.DECODE_LAMBDA,
                                                   bench.DECODE_SPLITS, 1)


def test_reference_arm_loads_no_library():
    # the oracle arm is self-contained: it imports neither the package nor libskipsm.so
    import subprocess
    import sys
    code = ("import sys, bench; bench.main(['--impl', 'reference', '--steps', '1', '--warmup', "
            "'0', '--ref-budget', '0.01']); "
            "assert 'block_sparse_long_softmax_b300' not in sys.modules, 'package imported'; "
            "maps = open('/proc/self/maps').read(); assert 'libskipsm' not in maps, 'lib loaded'")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]


def test_kernel_source_hash_ignores_comments_only():
    src = 'int f() { // a\n  return 1; /* b */ }\nconst char* s = "// kept";\n'
    same = 'int f() { // another\n  return 1; /* c\n d */ }\nconst char* s = "// kept";\n'
    other = 'int f() { // a\n  return 2; /* b */ }\nconst char* s = "// kept";\n'
    strip = bench._strip_comments
    assert strip(src) == strip(same)
    assert strip(src) != strip(other)
    assert '"// kept"' in strip(src)
