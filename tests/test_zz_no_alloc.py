"""The routing entry point that allocates no device memory.

Some callers cannot allocate device memory (a runtime that owns every device
byte, a fixed arena, a plug-in handed only its buffers); they route tokens
through moe_route_topk_static, whose scratch is a static device array. This
checks it through the C ABI against the CPU oracle and against the layer's
own forward (the existing entry point) on two calls in a row, at its largest
sizes (16 tokens, 1024 experts, top-32: the biggest carve of the static
scratch and a shared-memory request above 48 KB), that repeated calls leave
the device's allocated memory unchanged, and that it rejects sizes beyond
its limits. Collected last so that a failure here comes after every other
test.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import moe_oracle as O  # noqa: E402
from w4a16_routed_expert_gb300 import capi, synth  # noqa: E402

import gpu_harness as GH  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    capi.lib()


def _static_route(x, lay, stream):
    s = lay.shape
    return _static_route_raw(x, lay.router_w, lay.router_bias, s.num_experts, s.top_k, s.renormalize, stream)


def _static_route_raw(x, router_w, router_bias, E, k, renorm, stream):
    dev = torch.device("cuda")
    T, H = x.shape
    xd = torch.from_numpy(x).to(dev)
    rw = torch.from_numpy(router_w).to(dev)
    rb = torch.from_numpy(router_bias).to(dev) if router_bias is not None else None
    ids = torch.full((T, k), -1, dtype=torch.int32, device=dev)
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
    st = capi.lib().moe_route_topk_static(xd.data_ptr(), T, H, rw.data_ptr(),
                                          rb.data_ptr() if rb is not None else None, E, k,
                                          int(renorm), ids.data_ptr(), w.data_ptr(), stream.cuda_stream)
    capi.check(st, "moe_route_topk_static")
    stream.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


def _against_oracle(x, router_w, router_bias, k, renorm, ids, w):
    """ids bit-exact on tokens whose routing is decided beyond the near-tie
    margin; weights against the oracle's FP64 softmax taken at the returned
    ids (every token)."""
    L = O.router_logits(x, router_w, router_bias)
    p = O.softmax_rows(L)
    ref = O.select_topk_fast(L, k)
    near = set(O.near_tie_tokens(L, k, GH.TIE_EPS).tolist())
    decided = [t for t in range(x.shape[0]) if t not in near]
    assert np.array_equal(ids[decided], ref[decided])
    for t in near:  # still a valid top-k within the margin
        assert sorted(set(ids[t].tolist())) == sorted(ids[t].tolist())
        kth = np.sort(L[t])[::-1][k - 1]
        assert (L[t, ids[t]] >= kth - GH.TIE_EPS).all()
    np.testing.assert_allclose(w, O.routing_weights(p, ids.astype(np.int64), renorm), rtol=2e-5, atol=1e-7)
    return len(near)


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
        _against_oracle(x, lay.router_w, lay.router_bias, shape.top_k, shape.renormalize, ids, w)
    ml.close()


@pytest.mark.parametrize("E,k,T,renorm", [(1024, 32, 16, True), (1024, 32, 16, False), (600, 10, 13, True),
                                          (64, 8, 1, False)])
def test_static_routing_at_its_limits_matches_the_oracle(E, k, T, renorm):
    """Largest sizes the entry point takes: 16 tokens, 1024 experts (the
    32-values-per-lane selection), top-32, twice in a row."""
    H = 2048
    rng = np.random.default_rng(E + k + T)
    # a wider router than the workloads' keeps most tokens clear of near ties
    router_w = (rng.standard_normal((E, H)) * 0.2).astype(np.float32)
    bias = (-1.1 * np.log1p(np.arange(E))).astype(np.float32) if E == 600 else None
    stream = GH.stream()
    for call in range(2):
        x = synth.make_tokens(H, T, seed=900 + call + E)
        ids, w = _static_route_raw(x, router_w, bias, E, k, renorm, stream)
        assert ids.min() >= 0 and ids.max() < E
        _against_oracle(x, router_w, bias, k, renorm, ids, w)


def test_static_routing_allocates_nothing():
    """After a first call (which may load the library's code and its static
    array onto the device), further calls change neither the caching
    allocator's count nor the device's free memory."""
    E, k, T, H = 1024, 32, 16, 2048
    rng = np.random.default_rng(5)
    router_w = (rng.standard_normal((E, H)) * 0.2).astype(np.float32)
    dev = torch.device("cuda")
    x = torch.from_numpy(synth.make_tokens(H, T, seed=5)).to(dev)
    rw = torch.from_numpy(router_w).to(dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    stream = GH.stream()
    lib = capi.lib()

    def call():
        st = lib.moe_route_topk_static(x.data_ptr(), T, H, rw.data_ptr(), None, E, k, 1, ids.data_ptr(),
                                       w.data_ptr(), stream.cuda_stream)
        capi.check(st, "moe_route_topk_static")

    call()
    stream.synchronize()
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(20):
        call()
    stream.synchronize()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)


def test_static_routing_rejects_sizes_beyond_its_limits():
    lib = capi.lib()
    p = ctypes.c_void_p(16)
    assert lib.moe_route_topk_static(p, 17, 2048, p, None, 64, 8, 0, p, p, None) == capi.MOE_ERR_INVALID_ARG
    assert "T must be" in capi.last_error()
    assert lib.moe_route_topk_static(p, 1, 2048, p, None, 2048, 8, 0, p, p, None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk_static(p, 1, 2048, p, None, 64, 33, 0, p, p, None) == capi.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk_static(p, 0, 2048, p, None, 64, 8, 0, p, p, None) == capi.MOE_OK
