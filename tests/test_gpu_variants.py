"""Format variants against the oracle, every row: group size 32, asymmetric
zero points (w = (q - z) * s), a shared expert gated per token by
sigmoid(x . w_gate), alone and together, on the grouped-GEMV path (small
batches, one token included), the tensor-core GEMM path (large batches) and
partial residency."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from w4a16_routed_expert_gb300 import capi, synth  # noqa: E402
from w4a16_routed_expert_gb300.layer import MoELayer  # noqa: E402

import gpu_harness as GH  # noqa: E402

G32 = synth.LayerShape(256, 256, 16, 4, 32, True)
ZP = synth.LayerShape(512, 384, 24, 3, 128, True, zero_points=True)
GATED = synth.LayerShape(512, 256, 32, 4, 64, False, has_shared=True, shared_gate=True)
ALL = synth.LayerShape(256, 512, 16, 2, 32, True, has_shared=True, zero_points=True, shared_gate=True)
OLMOE_ZP32 = synth.LayerShape(2048, 1024, 64, 8, 32, False, zero_points=True)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    capi.lib()


CASES = [
    ("g32", G32, "uniform", (1, 7, 64)),
    ("zp-g128", ZP, "quantized", (1, 9, 96)),
    ("zp-uniform", ZP, "uniform", (2, 64)),
    ("gated-g64", GATED, "uniform", (1, 16, 80)),
    ("all", ALL, "uniform", (1, 5, 128)),
    ("all-quantized", ALL, "quantized", (3, 64)),
]


@pytest.mark.parametrize("name,shape,codes,Ts", CASES, ids=[c[0] for c in CASES])
def test_variant_matches_oracle_every_row(name, shape, codes, Ts):
    lay = synth.make_layer(shape, seed=41, codes=codes)
    assert lay.records.shape[1] == capi.lib().moe_record_bytes_zp(
        shape.hidden, shape.intermediate, shape.group_size, int(shape.zero_points))
    ml = GH.upload(lay, max_tokens=max(Ts))
    for T in Ts:
        x = synth.make_tokens(shape.hidden, T, seed=41 + T)
        g = GH.run(ml, x)
        GH.compare(lay, x, g)
    ml.close()


@pytest.mark.parametrize("T", [1, 256])
def test_olmoe_size_zero_points_g32(T):
    lay = synth.make_layer(OLMOE_ZP32, seed=42)
    ml = GH.upload(lay, max_tokens=T)
    x = synth.make_tokens(OLMOE_ZP32.hidden, T, seed=42)
    GH.compare(lay, x, GH.run(ml, x))
    ml.close()


def test_variants_repeatable():
    lay = synth.make_layer(ALL, seed=43, codes="uniform")
    ml = GH.upload(lay, max_tokens=64)
    for T in (1, 64):
        x = synth.make_tokens(ALL.hidden, T, seed=43)
        a, b = GH.run(ml, x), GH.run(ml, x)
        assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["w"], b["w"])
    ml.close()


def test_variants_under_partial_residency():
    lay = synth.make_layer(ALL, seed=44, codes="uniform")
    full = GH.upload(lay, max_tokens=64)
    host = torch.from_numpy(lay.records[lay.expert_to_slot]).contiguous().pin_memory()
    dev = torch.device("cuda")
    s = ALL
    part = MoELayer(hidden=s.hidden, intermediate=s.intermediate, num_experts=s.num_experts, top_k=s.top_k,
                    group_size=s.group_size, renormalize=s.renormalize, has_shared=s.has_shared, max_tokens=64,
                    router_w=torch.from_numpy(lay.router_w).to(dev), num_slots=5, spare_slots=2,
                    host_backing=host, zero_points=True, shared_gate=torch.from_numpy(lay.shared_gate).to(dev))
    for T in (1, 6, 64):
        x = synth.make_tokens(s.hidden, T, seed=44 + T)
        gp, gf = GH.run(part, x), GH.run(full, x)
        GH.compare(lay, x, gp)
        if T > 1:  # same kernels, same bits (one token: the same multi-kernel path as well)
            assert np.array_equal(gp["out"], gf["out"]), T
    part.close()
    full.close()


def test_gate_without_shared_expert_is_rejected():
    shape = synth.LayerShape(256, 256, 8, 2, 64, True)
    lay = synth.make_layer(shape, seed=45, codes="uniform")
    dev = torch.device("cuda")
    with pytest.raises(capi.MoEError) as ei:
        MoELayer(hidden=256, intermediate=256, num_experts=8, top_k=2, group_size=64, renormalize=True,
                 max_tokens=4, router_w=torch.from_numpy(lay.router_w).to(dev),
                 pool=torch.from_numpy(lay.records).to(dev),
                 expert_to_slot=torch.from_numpy(lay.expert_to_slot.astype(np.int32)).to(dev),
                 shared_gate=torch.zeros(256, device=dev))
    assert ei.value.status == capi.MOE_ERR_INVALID_ARG
