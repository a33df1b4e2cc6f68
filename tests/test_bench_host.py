"""Host-side logic of bench.py on the CPU: the multi-rank timing aggregation
(barrier + max over ranks, whole-job throughput) with two gloo ranks, and the
byte accounting of the roofline."""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    t = bench.max_over_ranks(1.0 + rank, world)          # rank 1 is the slow one
    v = bench.whole_job_value(1e9, 10, world, t)
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in out:
        assert t == 2.0                        # max over ranks, seen by every rank
        assert abs(v - 1e9 * 10 * 2 / 2.0 / 1e9) < 1e-9


def test_algorithmic_bytes():
    # square decode layer, M=8: Wq + s_w + X bf16 + Y bf16
    assert bench.algorithmic_bytes(8, 5120, 5120) == 26214400 + 6400 + 81920 + 81920
    # vocab layer, M=8
    assert bench.algorithmic_bytes(8, 248320, 5120) == 1271398400 + 310400 + 81920 + 3973120
    assert bench.bf16_bytes(8, 248320, 5120) == 2542796800 + 81920 + 3973120
    assert bench.whole_job_value(26384640, 1000, 1, 0.005) == 26384640 * 1000 / 0.005 / 1e9


def test_decode_pass_accounting():
    """One decode pass: 64 GEMMs of each of the four layer shapes, in cycling
    order, then the output layer; the step's algorithmic bytes are the sum of
    the 257 GEMMs' bytes (22.4 GB of weights)."""
    shapes = bench.pass_layers_shapes()
    assert len(shapes) == 257 and shapes[-1] == (248320, 5120)
    assert shapes[:4] == [(5120, 5120), (34816, 5120), (5120, 17408), (7168, 5120)]
    assert all(shapes.count(s) == 64 for s in bench.PASS_SHAPES)
    weights = sum(N * K for N, K in shapes)
    assert weights == 64 * (5120 * 5120 + 34816 * 5120 + 5120 * 17408 + 7168 * 5120) + 248320 * 5120
    assert abs(weights / 1e9 - 22.41) < 0.01
    assert bench.pass_bytes(8) == sum(bench.algorithmic_bytes(8, N, K) for N, K in shapes)


def test_workload_configs():
    """Both arms of the JSON line name the decode pass with the same config
    (one helper builds it); ``mx_<layer>`` is the same layer in the MX variant,
    whose bytes count one scale byte per 32 K per weight row instead of the
    fp32 block scales and activation scales."""
    c = bench.pass_workload(8)
    assert c["M"] == 8 and c["gemms_per_step"] == 257
    assert c["weight_bytes"] == sum(N * K for N, K in bench.pass_layers_shapes())
    assert c["workload"].startswith("decode_pass M=8: 256 GEMMs cycling 5120x5120, 34816x5120")
    assert bench.workload("mx_square_decode", 512) == dict(bench.workload("square_decode"), M=512)
    assert bench.workload("mx_mlp_up") == bench.workload("mlp_up")
    assert bench.mx_bytes(8, 5120, 5120) == 26214400 + 26214400 // 32 + 81920 + 81920
