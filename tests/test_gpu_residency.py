"""Partially resident slot pool on the GPU: same results as full residency
(bit-exact) and as the oracle, the pool bookkeeping counters, the host copy
never written, and a host-side injected copy failure."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from w4a16_routed_expert_gb300 import capi, synth  # noqa: E402
from w4a16_routed_expert_gb300.layer import MoELayer  # noqa: E402

import gpu_harness as GH  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    capi.lib()


def _partial(lay, slots, max_tokens, spares=0, policy=0, pinned=False, staging=0):
    s = lay.shape
    host = torch.from_numpy(lay.records[lay.expert_to_slot]).contiguous()  # expert order
    if pinned:
        host = host.pin_memory()
    dev = torch.device("cuda")
    ml = MoELayer(hidden=s.hidden, intermediate=s.intermediate, num_experts=s.num_experts, top_k=s.top_k,
                  group_size=s.group_size, renormalize=s.renormalize, has_shared=s.has_shared,
                  max_tokens=max_tokens, router_w=torch.from_numpy(lay.router_w).to(dev),
                  router_bias=torch.from_numpy(lay.router_bias).to(dev) if lay.router_bias is not None else None,
                  num_slots=slots, host_backing=host, spare_slots=spares, cache_policy=policy,
                  staging_records=staging)
    return ml, host


@pytest.mark.parametrize("shape,slots,T", [
    (synth.LayerShape(256, 256, 16, 2, 64, True), 4, 8),
    (synth.LayerShape(512, 384, 24, 3, 128, True, has_shared=True), 5, 12),
    (synth.LayerShape(2880, 2880, 12, 4, 128, True), 4, 6),
])
def test_partial_matches_full_and_oracle(shape, slots, T):
    lay = synth.make_layer(shape, seed=21, codes="uniform")
    x = synth.make_tokens(shape.hidden, T, seed=21)
    full = GH.upload(lay, max_tokens=T)
    gf = GH.run(full, x)
    full.close()
    ml, host = _partial(lay, slots, T)
    before = host.numpy().copy()
    g1 = GH.run(ml, x)
    g2 = GH.run(ml, x)
    st = ml.stats()
    for key in ("out", "ids", "w", "perm", "counts"):
        assert np.array_equal(g1[key], gf[key]) and np.array_equal(g2[key], gf[key]), key
    GH.compare(lay, x, g1)
    demanded = int((g1["counts"] > 0).sum()) + (1 if shape.has_shared else 0)
    assert st.forward_calls == 2 and st.tokens == 2 * T
    assert st.expert_hits + st.expert_misses == 2 * demanded
    assert st.h2d_bytes == st.expert_misses * lay.records.shape[1]
    assert st.d2h_expert_bytes == 0
    assert st.waves >= 2 * -(-demanded // slots)
    # the second call finds at least the previous call's last wave resident
    assert st.expert_hits >= min(slots, demanded) - 0
    assert np.array_equal(host.numpy(), before), "host backing was written"
    ml.close()


def test_injected_copy_failure_keeps_a_consistent_pool(monkeypatch):
    shape = synth.LayerShape(256, 256, 16, 2, 64, True)
    lay = synth.make_layer(shape, seed=22, codes="uniform")
    x = synth.make_tokens(shape.hidden, 8, seed=22)
    monkeypatch.setenv("MOE_FAULT_INJECT", "h2d_fail")
    ml, host = _partial(lay, 4, 8)
    with pytest.raises(capi.MoEError) as ei:
        GH.run(ml, x)
    assert ei.value.status == capi.MOE_ERR_CUDA and "injected" in str(ei.value)
    # the injection is one-shot; the next forward is correct
    g = GH.run(ml, x)
    GH.compare(lay, x, g)
    ml.close()


def test_capacity_shortfall_fails_at_create():
    shape = synth.LayerShape(256, 256, 16, 4, 64, True)
    lay = synth.make_layer(shape, seed=23)
    with pytest.raises(capi.MoEError) as ei:
        _partial(lay, 3, 4)
    assert ei.value.status == capi.MOE_ERR_CAPACITY


POLICIES = [capi.MOE_POLICY_LRU, capi.MOE_POLICY_LFU, capi.MOE_POLICY_LRU_FREQ]


@pytest.mark.parametrize("policy", POLICIES)
@pytest.mark.parametrize("spares", [0, 3, 5])
@pytest.mark.parametrize("pinned", [False, True])
def test_every_policy_matches_full_residency(policy, spares, pinned):
    """Horizon RunMap report, "Partial-residency contract": whichever experts
    the policy keeps, a forward reads complete published copies, so the
    outputs are the full-residency outputs bit for bit; misses go through
    the pinned staging buffers only when the host copy is pageable."""
    shape = synth.LayerShape(512, 384, 24, 3, 128, True, has_shared=True)
    lay = synth.make_layer(shape, seed=25, codes="uniform")
    full = GH.upload(lay, max_tokens=12)
    ml, host = _partial(lay, 5, 12, spares=spares, policy=policy, pinned=pinned, staging=2)
    before = host.numpy().copy()
    gens = 0
    for call in range(3):
        x = synth.make_tokens(shape.hidden, 12, seed=250 + call)
        gf = GH.run(full, x)
        g = GH.run(ml, x)
        for key in ("out", "ids", "w", "perm", "counts"):
            assert np.array_equal(g[key], gf[key]), (call, key)
        st = ml.stats()
        assert st.generations >= gens and st.faulted == 0
        gens = st.generations
    st = ml.stats()
    assert st.h2d_bytes == st.expert_misses * lay.records.shape[1]
    assert st.staged_copies == (0 if pinned else st.expert_misses)
    assert st.d2h_expert_bytes == 0
    assert np.array_equal(host.numpy(), before), "host backing was written"
    full.close()
    ml.close()


def test_failure_after_publication_faults_the_cache(monkeypatch):
    shape = synth.LayerShape(256, 256, 16, 2, 64, True)
    lay = synth.make_layer(shape, seed=26, codes="uniform")
    x = synth.make_tokens(shape.hidden, 8, seed=26)
    monkeypatch.setenv("MOE_FAULT_INJECT", "after_publish")
    ml, _ = _partial(lay, 4, 8)
    with pytest.raises(capi.MoEError) as ei:
        GH.run(ml, x)
    assert ei.value.status == capi.MOE_ERR_CUDA and "faulted" in str(ei.value)
    assert ml.stats().faulted == 1
    with pytest.raises(capi.MoEError) as ei:  # every later forward fails
        GH.run(ml, x)
    assert "faulted" in str(ei.value)
    ml.close()


def test_partial_residency_full_size_every_row():
    """The 2880-wide layer at its full size (128 experts, top-4 renormalised,
    32 resident slots filled from host backing of all 128 experts), 256
    tokens: every demanded expert is copied in over several waves. Every
    output row and the whole routing against the oracle."""
    shape = synth.GPTOSS_LIKE
    T = 256
    lay = synth.make_layer(shape, seed=4)
    x = synth.make_tokens(shape.hidden, T, seed=4)
    ml, host = _partial(lay, 32, T)
    g = GH.run(ml, x)
    st = ml.stats()
    ml.close()
    rep = GH.compare(lay, x, g)
    assert rep["rows_compared"] == T
    demanded = int((g["counts"] > 0).sum())
    assert st.expert_hits + st.expert_misses == demanded
    assert st.waves >= -(-demanded // 32)
    assert st.h2d_bytes == st.expert_misses * lay.records.shape[1]
    assert st.d2h_expert_bytes == 0
