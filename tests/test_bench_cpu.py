"""Host-side logic of bench.py, on the CPU: algorithmic byte counts, the traffic
record's source check, clock-reason decoding, and the replica path (max over
ranks, barriers) with two gloo ranks."""
import hashlib
import os
import socket

import pytest

import bench


def test_layer_and_model_bytes():
    # packed bytes of the four layer matrices (dual, 18 B per 32 weights)
    assert [bench.matrix_bytes(N, K) for _, N, K in bench.LAYER] == [20643840, 17694720, 100270080, 50135040]
    # + 2 B per activation and 4 B per output at M = 1
    assert bench.step_bytes(bench.LAYER) == sum(
        N * K // 32 * 18 + 2 * K + 4 * N for _, N, K in bench.LAYER)
    mats = [("x", N, K) for _ in range(bench.N_LAYERS) for (_, N, K) in bench.LAYER] + [bench.LM_HEAD]
    assert bench.weight_bytes(mats) == 12517539840
    assert bench.matrix_bytes(7168, 5120, variant=1) == 7168 * 160 * 17


def test_layout_map_per_tensor_role():
    lay = bench.parse_layouts("gate_up=fast,down=fast")
    assert lay == {"qkv": 0, "o": 0, "gate_up": 1, "down": 1, "lm_head": 0}
    assert bench.parse_layouts("") == {r: 0 for r in bench.ROLES}
    for bad in ("ffn=fast", "qkv=fp8", "qkv"):
        with pytest.raises(SystemExit):
            bench.parse_layouts(bad)
    assert bench.role_of("l12.gate_up") == "gate_up" and bench.role_of("lm_head") == "lm_head"
    # mixed step bytes: each matrix at its own block size
    mats = [("l0.qkv", 7168, 5120), ("l0.gate_up", 34816, 5120)]
    got = sum(bench.step_bytes([m], lay[bench.role_of(m[0])]) for m in mats)
    assert got == 7168 * 160 * 18 + 34816 * 160 * 17 + 2 * 5120 * 2 + 4 * (7168 + 34816)


def test_gate_up_bytes():
    # the fused product reads the 2I x K matrix of the layer's gate+up, one x, writes I outputs
    I, K = bench.GATE_UP
    assert 2 * I == 34816
    assert bench.gate_up_bytes(I, K) == 34816 * (K // 32) * 18 + 2 * K + 4 * I
    assert bench.gate_up_bytes(I, K, M=4) == bench.matrix_bytes(2 * I, K) + 8 * K + 16 * I


def test_attention_bytes():
    # K and V rows of 4 dual blocks (72 B) per token and KV head, q fp16 in, out fp32
    assert bench.attention_bytes(1, 32768) == 2 * 8 * 32768 * 72 + 2 * 40 * 128 + 4 * 40 * 128
    assert bench.attention_bytes(16, 4096, variant=1) == 2 * 16 * 8 * 4096 * 68 + 6 * 16 * 40 * 128


def test_quantize_bytes():
    assert bench.quantize_bytes(34816, 5120) == 2 * 34816 * 5120 + 34816 * 160 * 18


def test_traffic_record_needs_the_measured_source(tmp_path, monkeypatch):
    src = tmp_path / "gemv.cu"
    src.write_text("kernel v1\n")
    host = tmp_path / "api.cu"
    host.write_text("grid v1\n")
    rec = tmp_path / "rec.md"
    sha = hashlib.sha256(b"kernel v1\ngrid v1\n").hexdigest()
    rec.write_text(f"notes\nsource_sha256: {sha}\ndram_bytes_per_launch: qkv=10, o=20, gate_up=30, down=40\n")
    monkeypatch.setattr(bench, "GEMV_SOURCES", (str(src), str(host)))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    assert bench.gemv_traffic() == {"qkv": 10, "o": 20, "gate_up": 30, "down": 40}
    host.write_text("grid v2\n")  # launch sizing changed since the capture: no traffic figure
    assert bench.gemv_traffic() is None
    host.write_text("grid v1\n")
    src.write_text("kernel v2\n")  # kernel changed since the capture: no traffic figure
    assert bench.gemv_traffic() is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.md"))
    assert bench.gemv_traffic() is None


def test_clock_summary_decodes_reasons():
    c = bench.ClockSampler()
    assert c.summary()["samples"] == 0
    c.samples = [(2070.0, 0), (1980.0, 0x4), (2070.0, 0x40)]
    c.max_mhz = 2070.0
    s = c.summary()
    assert s["sm_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_peaks_read_the_measured_file():
    hbm, bf16, bf16_s, kind = bench.peaks()
    if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):
        assert kind == "measured" and hbm > 1000 and bf16 > 100
    else:
        assert kind == "fallback"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(1.5 + rank, w)
    bench.barrier(w)
    dist.destroy_process_group()


def test_replicas_take_the_max_over_ranks():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    if torch.cuda.is_available():
        pytest.skip("the gloo replica test runs on CPU-only hosts")
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_layer_passes_replay_whole_rotations_and_count_exactly():
    """run_steps(n, first) replays exactly n passes, copy (first + i) % copies for
    pass i: whole rotations from the multi-pass graph, the rest one by one."""
    import bench

    class G:
        def __init__(self, log, tag):
            self.log, self.tag = log, tag

        def replay(self):
            self.log.append(self.tag)

    for copies in (2, 3, 4):
        for first in range(0, 2 * copies + 1):
            for n in range(0, 3 * copies + 2):
                log = []
                step = type("S", (), {})()
                step.copies = copies
                step.multi = G(log, "multi")
                step.graphs = [G(log, r) for r in range(copies)]
                bench.GemvStep.run_steps(step, n, first)
                passes = []
                for tag in log:
                    passes.extend(range(copies) if tag == "multi" else [tag])
                assert passes == [(first + i) % copies for i in range(n)], (copies, first, n, log)


def test_read_ceiling_kernel_builds_and_exports():
    # the benchmark's plain-read ceiling kernel: a separate measurement library
    import ctypes

    import ceiling
    L = ctypes.CDLL(ceiling.build())
    for sym in ("readceil_launch", "readceil_prepare", "readceil_smem"):
        assert hasattr(L, sym), sym
    L.readceil_smem.restype = ctypes.c_size_t
    for chunk, warps, per_sm, stages in ceiling.CONFIGS:
        smem = L.readceil_smem(chunk, warps, stages)
        assert smem == warps * stages * (chunk + 8)
        assert smem * per_sm <= 228 * 1024 and smem <= ceiling.MAX_SMEM  # the CTAs of a config fit on an SM
        assert chunk % 512 == 0
