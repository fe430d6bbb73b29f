"""The routing entry point that allocates no device memory.

Some callers cannot allocate device memory (a runtime that owns every device
byte, a fixed arena, a plug-in handed only its buffers); they route tokens
through moe_route_topk_static, whose scratch is a static device array. This
checks it through the C ABI against the layer's own forward (the existing
entry point) on two calls in a row, and that it rejects sizes beyond its
limits. Collected last so that a failure here comes after every other test.
"""
import ctypes

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


def _static_route(x, lay, stream):
    s = lay.shape
    dev = torch.device("cuda")
    T = x.shape[0]
    xd = torch.from_numpy(x).to(dev)
    rw = torch.from_numpy(lay.router_w).to(dev)
    rb = torch.from_numpy(lay.router_bias).to(dev) if lay.router_bias is not None else None
    ids = torch.full((T, s.top_k), -1, dtype=torch.int32, device=dev)
    w = torch.full((T, s.top_k), float("nan"), dtype=torch.float32, device=dev)
    st = capi.lib().moe_route_topk_static(xd.data_ptr(), T, s.hidden, rw.data_ptr(),
                                          rb.data_ptr() if rb is not None else None, s.num_experts, s.top_k,
                                          int(s.renormalize), ids.data_ptr(), w.data_ptr(), stream.cuda_stream)
    capi.check(st, "moe_route_topk_static")
    stream.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("shape,seed,T", [(synth.OLMOE, 40, 1), (synth.MANY_EXPERTS, 41, 16),
                                          (synth.LayerShape(256, 128, 8, 2, 64, True), 42, 7)])
def test_static_routing_matches_the_layer_forward_twice(shape, seed, T):
    lay = synth.make_layer(shape, seed=seed)
    ml = GH.upload(lay, max_tokens=T)
    stream = GH.stream()
    for call in range(2):  # two calls in a row share (and reuse) the static scratch
        x = synth.make_tokens(shape.hidden, T, seed=seed * 10 + call)
        ref = GH.run(ml, x)
        ids, w = _static_route(x, lay, stream)
        assert np.array_equal(ids, ref["ids"]), call
        np.testing.assert_allclose(w, ref["w"], rtol=2e-5, atol=1e-7)
    ml.close()


def test_static_routing_rejects_sizes_beyond_its_limits():
    lib = capi.lib()
    p = ctypes.c_void_p(16)
    assert lib.moe_route_topk_static(p, 17, 2048, p, None, 64, 8, 0, p, p, None) == capi.MOE_ERR_INVALID_ARG
    assert "T must be" in capi.last_error()
    assert lib.moe_route_topk_static(p, 1, 2048, p, None, 2048, 8, 0, p, p, None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk_static(p, 1, 2048, p, None, 64, 33, 0, p, p, None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk_static(p, 0, 2048, p, None, 64, 8, 0, p, p, None) == capi.MOE_OK
