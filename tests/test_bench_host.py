"""Host-side checks of bench.py: the algorithmic byte model of each op, and
the max-over-ranks timing reduction run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from inputgen.workloads import WORKLOADS

# algorithmic bytes per op (read x and w, write y / read x, dy, w, write dx
# and the parameter gradient), as in the measurement plan's table
EXPECTED = {
    "c1": (26_256, 52_112),
    "c2": (134_217_732, 201_326_600),
    "c3": (2_149_584_896, 4_297_072_640),
    "c4": (2_181_038_336, 4_328_522_240),
    "c5": (1_074_020_352, 2_148_024_320),
}


@pytest.mark.parametrize("name", sorted(EXPECTED))
def test_byte_model(name):
    wl = WORKLOADS[name]
    assert (bench.op_bytes(wl, "fwd"), bench.op_bytes(wl, "bwd")) == EXPECTED[name]


def test_step_composition():
    ops = bench.steps_ops(bench.ORDER_FWD)
    assert ops[:4] == [("c2", "fwd"), ("c3", "fwd"), ("c4", "fwd"), ("c5", "fwd")]
    assert ops[4:] == [("c5", "bwd"), ("c4", "bwd"), ("c3", "bwd"), ("c2", "bwd")]
    total = sum(bench.op_bytes(WORKLOADS[n], op) for n, op in ops)
    assert total == sum(sum(EXPECTED[n]) for n in ["c2", "c3", "c4", "c5"])
    assert sum(bench.KERNELS_PER_OP[bench.op_name(WORKLOADS[n], op)] for n, op in ops) == 12


def test_scaled_workloads():
    s = bench.scaled_workloads(0.125)
    assert s["c4"].N == (1 << 24) // 8 and s["c4"].D == 64 and s["c1"].N == 12
    assert bench.scaled_workloads(1.0) is WORKLOADS


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info() == (rank, world, rank)
        v = bench.max_over_ranks(10.0 * (rank + 1), device="cpu")
        out[rank] = v
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(3.5) == 3.5


def test_traffic_records_keyed_by_operator_sources(tmp_path, monkeypatch):
    # every record names a known operator and carries that operator's hash
    # format; a change to one operator's kernel file voids only its records
    import json
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    ops = {k.split(":")[0].rsplit("_", 1)[0] for k in t if not k.startswith("_")}
    assert ops <= set(bench.OP_SOURCES)
    for k, e in t.items():
        if not k.startswith("_"):
            assert len(e["source_hash"]) == 16 and int(e["source_hash"], 16) >= 0
            assert e["dram_bytes_per_launch"] > 0 and e["algorithmic_bytes"] > 0
    src = os.path.join(bench.ROOT, "backward_ws_fwd_gb300", "csrc")
    fake = tmp_path / "backward_ws_fwd_gb300" / "csrc"
    fake.mkdir(parents=True)
    for name in os.listdir(src):
        (fake / name).write_bytes(open(os.path.join(src, name), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = {op: bench.source_hash(op) for op in bench.OP_SOURCES}
    # comments and layout are not code: the records stay valid
    (fake / "norm.cu").write_bytes(b"// a comment\n/* and a block */\n" +
                                   (fake / "norm.cu").read_bytes() + b"\n\n   \n")
    assert {op: bench.source_hash(op) for op in bench.OP_SOURCES} == before
    (fake / "norm.cu").write_bytes((fake / "norm.cu").read_bytes() + b"\nstatic int edit;\n")
    after = {op: bench.source_hash(op) for op in bench.OP_SOURCES}
    assert {op for op in before if before[op] != after[op]} == {"rmsnorm", "layernorm"}
    (fake / "wsf_device.cuh").write_bytes((fake / "wsf_device.cuh").read_bytes() +
                                          b"\nstatic int edit2;\n")
    final = {op: bench.source_hash(op) for op in bench.OP_SOURCES}
    assert all(final[op] != after[op] for op in bench.OP_SOURCES)
    # a "//" inside a string literal is code
    (fake / "ws.cu").write_bytes((fake / "ws.cu").read_bytes() + b'\nconst char* u = "a//b";\n')
    h1 = bench.source_hash("ws")
    (fake / "ws.cu").write_bytes((fake / "ws.cu").read_bytes().replace(b'"a//b"', b'"a//c"'))
    assert bench.source_hash("ws") != h1


def test_reference_arm_line_contract():
    # the reference arm is the fp64 oracle on the host cores: it needs no
    # GPU, and its one JSON line carries the fields of the benchmark contract
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=300, cwd=bench.ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"]
