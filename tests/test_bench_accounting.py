"""The bench's roofline arithmetic against closed-form sizes of the layer:
algorithmic bytes (every selected expert's record read once, the router
weights, x in and out) and FLOPs (2 H E per token for the router, 6 H I per
(token, expert) pair for gate/up/down), plus its launch and throughput
accounting. CPU only."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from w4a16_routed_expert_gb300 import synth  # noqa: E402


def _payload(H, I, G):
    """Codes + scales of one expert record (no alignment padding)."""
    return 3 * H * I // 2 + 2 * I * (-(-H // G)) * 2 + H * (-(-I // G)) * 2


def test_olmoe_batch1_layer_bytes():
    s = synth.OLMOE
    b, f, per = bench.algorithmic(s, 1, 8)
    assert _payload(2048, 1024, 128) == 3_244_032
    assert b["layer"] == 8 * 3_244_032 + 64 * 2048 * 4 + 2 * 2048 * 2 == 26_484_736
    assert per["gate_up_per_expert"] == 2_162_688 and per["down_per_expert"] == 1_081_344
    assert f["layer"] == 2 * 2048 * 64 + 8 * 6 * 2048 * 1024


def test_prefill_flops_make_it_tensor_bound():
    s = synth.OLMOE
    b, f, _ = bench.algorithmic(s, 8192, 64)
    assert f["layer"] == 2 * 8192 * 2048 * 64 + 8192 * 8 * 6 * 2048 * 1024
    assert f["gate_up"] == 8192 * 8 * 4 * 2048 * 1024 and f["down"] == 8192 * 8 * 2 * 2048 * 1024
    # about 827 GFLOP against about 0.2 GB: the FLOPs set the roofline time
    assert abs(f["layer"] / 1e9 - 826.8) < 1.0
    peaks = bench._peaks()
    assert f["layer"] / (peaks["bf16_tflops"] * 1e12) > b["layer"] / (peaks["hbm_gbs"] * 1e9)


def test_many_experts_batch1_includes_shared_expert_and_router():
    s = synth.MANY_EXPERTS
    b, f, _ = bench.algorithmic(s, 1, 10)
    rec = _payload(2048, 512, 128)
    assert rec == 1_622_016
    assert b["layer"] == 11 * rec + 512 * 2048 * 4 + 2 * 2048 * 2
    assert f["layer"] == 2 * 2048 * 512 + 11 * 6 * 2048 * 512


@pytest.mark.parametrize("T,gmin,expect", [(8, 48, 4), (16, 48, 4), (17, 48, 6), (47, 48, 6), (48, 48, 7),
                                           (8192, 48, 7)])
def test_multi_kernel_launch_count(T, gmin, expect):
    # routing (1 kernel up to 16 tokens, else 3) + experts (2 GEMV or gather + 2 GEMM) + combine
    assert bench.launches_per_multi_kernel_forward(T, gmin) == expect


def test_replica_throughput():
    assert bench.replica_throughput(1, 1, 0.025) == pytest.approx(40_000.0)
    assert bench.replica_throughput(16, 4, 0.1) == pytest.approx(640_000.0)


def test_parity_record_flags_planted_errors():
    """The bench's parity record against hand-made GPU results: exact ids
    and outputs within the bound pass; a wrong id on a decided token, or an
    output off by more than the bound, fails; near-tie tokens are counted and
    not compared."""
    import numpy as np
    shape = synth.OLMOE
    ids = np.tile(np.arange(8), (4, 1))
    out = np.ones((4, 16))
    ref = dict(ids=ids.copy(), out=out.copy(), rows=np.arange(4), near=np.array([2]))
    ok = bench.parity_record(shape, ref, ids.copy(), out + 1e-3)
    assert ok["pass"] and ok["near_ties"] == 1 and ok["rows_compared"] == 3
    assert ok["max_err_over_bound"] == pytest.approx(0.5)
    bad_ids = ids.copy()
    bad_ids[1, 0] = 9
    assert not bench.parity_record(shape, ref, bad_ids, out)["pass"]
    near_ids = ids.copy()
    near_ids[2, 0] = 9  # token 2 is a near tie: not compared
    assert bench.parity_record(shape, ref, near_ids, out)["pass"]
    bad_out = out.copy()
    bad_out[3, 5] += 3e-3
    assert not bench.parity_record(shape, ref, ids, bad_out)["pass"]


def test_parity_rows_cover_small_batches_and_sample_large_ones():
    import numpy as np
    assert bench._parity_rows(1).tolist() == [0]
    assert bench._parity_rows(64).tolist() == list(range(64))
    r = bench._parity_rows(8192)
    assert len(r) == 64 and r[0] == 0 and r[-1] == 8191 and (np.diff(r) > 0).all()


def test_traffic_is_reported_only_for_unchanged_sources(tmp_path, monkeypatch):
    """A recorded DRAM-traffic figure is returned while the kernel's sources
    hash to the recorded state, and None once any of them changes."""
    csrc = tmp_path / "w4a16_routed_expert_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES["gemm"]:
        (csrc / f).write_text(f"// {f}\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    files = [f"w4a16_routed_expert_gb300/csrc/{f}" for f in bench.KERNEL_SOURCES["gemm"]]
    rec = {"w": {"gate_up": {"dram_bytes_per_launch": 123, "source_sha": bench.source_hash(*files)}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.kernel_traffic("w", "gate_up", True) == 123
    assert bench.kernel_traffic("w", "down", True) is None
    (csrc / "tc.cuh").write_text("// changed\n")
    assert bench.kernel_traffic("w", "gate_up", True) is None
