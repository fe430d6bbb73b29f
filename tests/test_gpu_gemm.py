"""Prefill path: the tensor-core grouped GEMM (tcgen05, TMEM accumulators,
TMA-loaded INT4 tiles dequantised in shared memory) against the oracle and
against the register-dequant GEMV path."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from w4a16_routed_expert_gb300 import capi, synth  # noqa: E402

import gpu_harness as GH  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    capi.lib()


GEMM_CASES = [
    # (id, shape, seed, T, codes)
    ("tiny-T40", synth.TINY, 30, 40, "quantized"),
    ("tiny-uniform-T130", synth.TINY, 31, 130, "uniform"),
    ("shared-G64-T50", synth.LayerShape(512, 384, 16, 3, 64, False, has_shared=True), 32, 50, "uniform"),
    ("wide-2880-T33", synth.LayerShape(2880, 2880, 8, 4, 128, True), 33, 33, "uniform"),
    ("olmoe-T300", synth.OLMOE, 34, 300, "quantized"),
]


@pytest.mark.parametrize("name,shape,seed,T,codes", GEMM_CASES, ids=[c[0] for c in GEMM_CASES])
def test_gemm_path_matches_oracle(name, shape, seed, T, codes, monkeypatch):
    monkeypatch.setenv("MOE_GEMM_MIN_TOKENS", "1")
    lay = synth.make_layer(shape, seed=seed, codes=codes)
    x = synth.make_tokens(shape.hidden, T, seed=seed)
    ml = GH.upload(lay, max_tokens=T)
    g = GH.run(ml, x)
    ml.close()
    rep = GH.compare(lay, x, g)
    print(name, rep)


def test_gemm_and_gemv_paths_agree(monkeypatch):
    shape = synth.LayerShape(512, 384, 16, 3, 64, True, has_shared=True)
    lay = synth.make_layer(shape, seed=35, codes="uniform")
    x = synth.make_tokens(shape.hidden, 70, seed=35)
    monkeypatch.setenv("MOE_GEMM_MIN_TOKENS", "1")
    a = GH.upload(lay, max_tokens=70)
    ga = GH.run(a, x)
    a.close()
    monkeypatch.setenv("MOE_GEMM_MIN_TOKENS", "1000000")
    b = GH.upload(lay, max_tokens=70)
    gb = GH.run(b, x)
    b.close()
    assert np.array_equal(ga["ids"], gb["ids"]) and np.array_equal(ga["perm"], gb["perm"])
    # the GEMM rounds each dequantised weight to FP16; the GEMV keeps exact
    # products: the outputs agree within the layer tolerance
    err = np.abs(ga["out"] - gb["out"])
    assert (err <= GH.TOL * np.maximum(1, np.abs(gb["out"]))).all(), err.max()


def test_prefill_8192_tokens_every_row():
    """The 8192-token prefill in the launch configuration the benchmark
    times: every output row and the whole routing against the oracle."""
    shape = synth.OLMOE
    T = 8192
    lay = synth.make_layer(shape, seed=1)
    x = synth.make_tokens(shape.hidden, T, seed=1)
    ml = GH.upload(lay, max_tokens=T)
    g = GH.run(ml, x)
    ml.close()
    rep = GH.compare(lay, x, g)
    assert rep["rows_compared"] == T


def test_many_experts_T256_gemm_every_row(monkeypatch):
    monkeypatch.setenv("MOE_GEMM_MIN_TOKENS", "1")
    shape = synth.MANY_EXPERTS
    lay = synth.make_layer(shape, seed=3)
    x = synth.make_tokens(shape.hidden, 256, seed=3)
    ml = GH.upload(lay, max_tokens=256)
    g = GH.run(ml, x)
    ml.close()
    GH.compare(lay, x, g)


def test_partial_residency_on_the_gemm_path(monkeypatch):
    monkeypatch.setenv("MOE_GEMM_MIN_TOKENS", "1")
    shape = synth.LayerShape(512, 384, 24, 3, 128, True, has_shared=True)
    lay = synth.make_layer(shape, seed=36, codes="uniform")
    x = synth.make_tokens(shape.hidden, 60, seed=36)
    full = GH.upload(lay, max_tokens=60)
    gf = GH.run(full, x)
    full.close()
    from test_gpu_residency import _partial
    ml, _ = _partial(lay, 5, 60)
    gp = GH.run(ml, x)
    ml.close()
    assert np.array_equal(gp["out"], gf["out"])
