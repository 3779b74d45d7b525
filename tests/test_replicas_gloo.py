"""The multi-GPU path is N independent replicas (the hot path has no exchange
between GPUs): the benchmark's only cross-rank logic is the max over ranks
of the timed region and the whole-job throughput.  Checked here with two
gloo ranks on the CPU."""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [7.5, 9.25][rank]  # rank 1 is the slow replica
        m = bench.max_over_ranks(ms, world, device="cpu")
        out[rank] = (m, bench.replica_throughput(32768, 10, world, m))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:  # no fork of a threaded process
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 9.25
    assert abs(res[0][1] - 32768 * 2 * 10 / 9.25e-3) < 1e-6 * res[0][1]


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.replica_throughput(100, 4, 1, 2.0) == 100 * 4 / 2e-3


def test_recorded_traffic_only_for_the_profiled_source(tmp_path, monkeypatch):
    import json
    prof = tmp_path / "profiles"
    prof.mkdir()
    src = tmp_path / "k.cu"
    src.write_text("head // K-BEGIN kernel v1 // K-END tail")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sl = [{"file": "k.cu", "begin": "// K-BEGIN", "end": "// K-END"}]
    rec = {"k": {"traffic_bytes_per_launch": 123, "source": sl,
                 "source_sha256": bench._source_digest(sl)}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("k") == 123
    src.write_text("other head // K-BEGIN kernel v1 // K-END other tail")  # unrelated edit
    assert bench.recorded_traffic("k") == 123
    src.write_text("head // K-BEGIN kernel v2 // K-END tail")  # the kernel itself changed
    assert bench.recorded_traffic("k") is None
    assert bench.recorded_traffic("other") is None
