"""The replicas-only multi-GPU path of bench.py, run as two gloo ranks on the CPU.

Each rank times its own batches; the job's throughput is the tokens of all ranks over the
slowest rank's time, and every rank draws different batches (weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, ms_of_rank, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(ms_of_rank[rank], dist)
        idx, _, _ = bench.workload_cases("decode", rank, 1, 64, layer_range=range(0))
        dist.barrier()
        q.put((rank, ms, idx.tolist()))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_distinct_batches():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ms_of_rank = [3.0, 5.0]
    procs = [ctx.Process(target=_worker, args=(r, world, port, ms_of_rank, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[1] for o in out] == [5.0, 5.0]  # every rank sees the slowest rank's time
    assert out[0][2] != out[1][2]  # replicas draw different batches
    assert bench.job_tokens_per_s(world, 64 * 32, 100, 5.0) == pytest.approx(2 * 64 * 32 * 100 / 5e-3)


def test_single_process_helpers():
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.rank_seed_offset(0) == 0 and bench.rank_seed_offset(1) != 0


def test_profile_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    # an ncu summary carries the hash of the GEMM source it was taken on; the bench reports
    # its DRAM bytes only while that source is unchanged
    import hashlib

    csrc = tmp_path / "adapter_gemm_segment_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = b"// a kernel source\n"
    (csrc / "gemm_tc.cu").write_bytes(src)
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = hashlib.sha256(src).hexdigest()[:16]
    (prof / "gemm_decode_decode.md").write_text(
        f"# summary\n- gemm_tc.cu sha256[:16]: {sha}\n- dram bytes per launch (full workload): 35937024\n")
    (prof / "gemm_prefill_prefill.md").write_text(
        "- gemm_tc.cu sha256[:16]: 0000000000000000\n- dram bytes per launch (full workload): 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_profile_traffic("gemm_decode_decode") == 35937024.0
    assert bench.read_profile_traffic("gemm_prefill_prefill") is None  # taken on another source
    assert bench.read_profile_traffic("no_such_profile") is None


def test_algorithmic_bytes_and_flops_hand_worked():
    # 6 tokens, idx [-1, 0, 0, 2, -1, 5]: D = 3 distinct adapters, n_L = 4 LoRA tokens;
    # h_in 10, h_out 7, r_max 4, 2-byte elements
    a = bench.algorithmic_case([-1, 0, 0, 2, -1, 5], 10, 7, 4)
    assert (a["D"], a["n_L"]) == (3, 4)
    W, A_D, B_D, xy = 7 * 10 * 2, 3 * 4 * 10 * 2, 3 * 7 * 4 * 2, 6 * (10 + 7) * 2
    assert a["linear_bytes"] == W + A_D + B_D + xy == 752
    assert a["gemm_bytes"] == W + B_D + xy == 512
    assert a["linear_flops"] == 2 * 6 * 10 * 7 + 2 * 4 * 4 * (10 + 7) == 1384
    assert a["gemm_flops"] == 2 * 6 * 10 * 7 + 2 * 4 * 4 * 7 == 1064


def test_algorithmic_bytes_match_the_decode_figure():
    # decode q_proj: 64 tokens, 4096 x 4096 fp16, r_max 8, 27 adapters touched:
    # 33.55 MB of W + 3.54 MB of adapters + 1.05 MB of x and y
    idx = [k % 27 for k in range(64)]
    a = bench.algorithmic_case(idx, 4096, 4096, 8)
    assert a["D"] == 27 and a["n_L"] == 64
    assert abs(a["linear_bytes"] / 1e6 - (33.554 + 3.539 + 1.049)) < 0.01


def test_job_throughput_counts_every_rank():
    assert bench.job_tokens_per_s(1, 1000, 10, 5.0) == 1000 * 10 / 5e-3
    assert bench.job_tokens_per_s(4, 1000, 10, 5.0) == 4 * 1000 * 10 / 5e-3
