"""Host-side logic of bench.py (CPU only): the metric's formula, clock-sample parsing and the
max-over-ranks reduction of a world-size-2 gloo group."""

import os
import socket

import torch.multiprocessing as mp

import bench


def test_formula_flops_headline():
    up, attn = bench.formula_flops(1, 4096, 128, 6292480)
    assert up == 2 * 4096 * 128 * 512 * 256                      # 137.4 GF
    assert attn == 2 * 128 * 6292480 * 320                        # 515.5 GF
    assert abs((up + attn) / 1e9 - 652.9) < 0.1


def test_clock_parse():
    lines = [
        "0, 1905, 2032, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1800, 2032, 1100.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 300, 2032, 100.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ]
    s = bench.ClockSampler.parse(lines)
    assert s["samples"] == 3 and s["sm_max_mhz"] == 2032
    assert s["reasons"] == ["sw_power_cap"]
    assert s["sm_mhz"] in (1800, 1852.5, 1905)                  # median of the loaded samples


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(dist)
    q.put((rank, bench.max_over_ranks(1.0 + rank * 2.5, dist)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 3.5, 1: 3.5}


def test_profiled_traffic_tracks_kernel_sources(tmp_path, monkeypatch):
    # the committed headline capture is reported only while the kernel sources are the ones it
    # measured; another workload or a changed source hash gives None
    assert bench.profiled_traffic("tiny") is None
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "sparse_attn_headline.md").write_text(
        "x\ntraffic: kernel=sparse_attn_kernel dram_bytes_per_launch=123 sources_sha256=%s\n"
        % bench.kernel_sources_sha256(bench.ATTENTION_SOURCES))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_sources_sha256", lambda files=None: "0" * 64)
    assert bench.profiled_traffic("headline") is None
    (prof / "sparse_attn_headline.md").write_text(
        "traffic: kernel=sparse_attn_kernel dram_bytes_per_launch=123 sources_sha256=%s\n" % ("0" * 64))
    assert bench.profiled_traffic("headline") == 123


def test_source_hash_ignores_comments_not_code():
    # the capture's hash follows the kernels' code: a comment or whitespace edit keeps it, a code
    # edit changes it
    a = bench._code_only("int x = 1; // one\n/* block\n comment */  float y;\n")
    b = bench._code_only("int x = 1;   // the value one\nfloat   y; /* other */\n")
    c = bench._code_only("int x = 2; // one\nfloat y;\n")
    assert a == b == "intx=1;floaty;"
    assert c != a


def test_hardware_mma_flops_headline():
    # attention: 528 causal key blocks per head (32 query tiles), 24 UMMAs of 128x128x16 each
    gemm, attn = bench.hardware_mma_flops(1, 4096, 128)
    assert attn == 128 * 528 * 24 * 2 * 128 * 128 * 16            # 850.4 GF
    assert gemm == 32 * 128 * 2 * 32 * 2 * 128 * 128 * 16           # 137.4 GF, the formula's up-projection
    up, _ = bench.formula_flops(1, 4096, 128, 6292480)
    assert gemm == up
    # a ragged tail pads the last tile to 128 rows
    g2, a2 = bench.hardware_mma_flops(2, 130, 3)
    assert a2 == 2 * 3 * 3 * 24 * 2 * 128 * 128 * 16 and g2 == 2 * 2 * 3 * 2 * 32 * 2 * 128 * 128 * 16
