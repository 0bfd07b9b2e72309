"""Host-side logic of bench.py on CPU: the max-over-ranks aggregation with
two gloo ranks, the reference (oracle) arm's JSON line, and the work model."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(1.5 + rank, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


def test_reference_arm_prints_one_json_line():
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_work_model():
    P = bench.PREFILL
    dense, per_pair = bench.prefill_flops(P)
    assert dense == 4.0 * 128 * 32 * 16384 * 16385 / 2
    assert per_pair == 2.0 * 128 * 128 * 128
    assert bench.traversed_pairs(P) == 32 * 128 * 129 // 2
    D = bench.DECODE
    n_blocks = D.B * D.Hkv * (D.L // D.Bc)
    full = bench.decode_bytes(D, n_blocks, n_blocks)
    assert full == 2 * D.B * D.Hkv * D.L * D.dk * 2 + D.B * D.Hq * D.dk * 2 + \
        D.B * D.Hq * D.n_splits * (D.dv + 1) * 4
    assert bench.tile_visible_pairs(P, 0) == 128 * 129 / 2


def test_rejects_too_few_warmups():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_gpus_flag_drives_the_world_size():
    """--gpus N outside torchrun relaunches one process per GPU under
    torch.distributed.run; inside torchrun it must match WORLD_SIZE."""
    assert bench.launch_plan(1, {}, []) == ("run", 1)
    assert bench.launch_plan(4, {"WORLD_SIZE": "4"}, []) == ("run", 4)
    plan, why = bench.launch_plan(8, {"WORLD_SIZE": "2"}, [])
    assert plan == "error" and "WORLD_SIZE=2" in why
    assert bench.launch_plan(0, {}, [])[0] == "error"
    plan, cmd = bench.launch_plan(2, {}, ["--gpus", "2", "--steps", "3"])
    assert plan == "relaunch"
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=2" in cmd and "127.0.0.1" in cmd
    assert cmd[-4:] == ["--gpus", "2", "--steps", "3"]
    assert cmd[-5].endswith("bench.py")
