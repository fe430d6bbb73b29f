"""Next-layer router prefetch on partially resident stacks (moe-stream,
"Findings": the next layer's router run early on the current state guesses
its experts). A prefetch changes only which experts are resident when a
forward starts, never a result: outputs with and without prefetches are
bit-identical; a guess made from the forward's own input is exact, so that
forward misses nothing; every counter adds up."""
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


def _partial(lay, slots, max_tokens, spares=0, policy=0, add_residual=False):
    s = lay.shape
    host = torch.from_numpy(lay.records[lay.expert_to_slot]).contiguous().pin_memory()
    dev = torch.device("cuda")
    return MoELayer(hidden=s.hidden, intermediate=s.intermediate, num_experts=s.num_experts, top_k=s.top_k,
                    group_size=s.group_size, renormalize=s.renormalize, has_shared=s.has_shared,
                    max_tokens=max_tokens, router_w=torch.from_numpy(lay.router_w).to(dev),
                    router_bias=torch.from_numpy(lay.router_bias).to(dev) if lay.router_bias is not None else None,
                    num_slots=slots, host_backing=host, spare_slots=spares, cache_policy=policy,
                    add_residual=add_residual)


def _run_stack(layers, x0, steps, prefetch):
    """Residual stack: each layer's output feeds the next; with `prefetch`,
    layer l+1's experts are guessed from layer l's input right after layer
    l's forward is enqueued. Returns every layer's output of every step."""
    outs = []
    x = x0
    for step in range(steps):
        xin = x
        per = []
        for l, m in enumerate(layers):
            y = m.forward(xin)
            if prefetch and l + 1 < len(layers):
                layers[l + 1].prefetch(xin)
            per.append(y)
            xin = y
        torch.cuda.synchronize()
        outs.append([p.cpu().numpy() for p in per])
        # next step: last output at unit RMS per token plus a small change
        y = xin.float()
        y = y * torch.rsqrt(y.square().mean(dim=1, keepdim=True).clamp_min(1e-12))
        x = (y + 0.1 * torch.randn(y.shape, generator=torch.Generator(device="cuda").manual_seed(step),
                                   device="cuda")).half()
    return outs


@pytest.mark.parametrize("shape,slots,spares,policy,T", [
    (synth.LayerShape(512, 384, 24, 3, 128, True), 6, 2, 0, 1),
    (synth.LayerShape(512, 384, 24, 3, 128, True, has_shared=True), 8, 0, 2, 4),
    (synth.LayerShape(256, 256, 32, 4, 64, False), 12, 4, 1, 16),
])
def test_prefetch_leaves_results_bit_identical(shape, slots, spares, policy, T):
    lays = [synth.make_layer(shape, seed=synth.stack_layer_seed(31, l)) for l in range(4)]
    x0 = torch.from_numpy(synth.make_tokens(shape.hidden, T, seed=31)).cuda()
    plain = [_partial(l, slots, T, spares, policy, add_residual=True) for l in lays]
    pref = [_partial(l, slots, T, spares, policy, add_residual=True) for l in lays]
    steps = 5
    a = _run_stack(plain, x0, steps, prefetch=False)
    b = _run_stack(pref, x0, steps, prefetch=True)
    for step in range(steps):
        for l in range(len(lays)):
            assert np.isfinite(a[step][l]).all(), (step, l)
            assert np.array_equal(a[step][l], b[step][l]), (step, l)
    for l, m in enumerate(pref):
        st = m.stats()
        assert st.prefetch_calls == (steps if l > 0 else 0)
        assert st.prefetch_used <= st.prefetched
        assert st.faulted == 0 and st.d2h_expert_bytes == 0
        # every copied expert is a miss of a forward or a prefetched guess
        assert st.h2d_bytes == (st.expert_misses + st.prefetched) * lays[l].records.shape[1]
    for m in plain:
        assert m.stats().prefetched == 0
    for m in plain + pref:
        m.close()


@pytest.mark.parametrize("T", [1, 3])
def test_a_guess_from_the_forwards_own_input_is_exact(T):
    # Guessing with the very input of the forward routes exactly as the
    # forward does: with every demanded expert fitting in the pool (at most
    # 3 tokens x top-3 + the shared expert = 10 of 12 slots), the
    # forward finds all of them resident and every copied guess is used.
    shape = synth.LayerShape(512, 384, 24, 3, 128, True, has_shared=True)
    lay = synth.make_layer(shape, seed=32, codes="uniform")
    full = GH.upload(lay, max_tokens=T)
    m = _partial(lay, 12, T)
    for step in range(4):
        x = synth.make_tokens(shape.hidden, T, seed=320 + step)
        xd = torch.from_numpy(x).cuda()
        s0 = m.stats()
        m.prefetch(xd)
        torch.cuda.synchronize()
        s1 = m.stats()
        g = GH.run(m, x)
        s2 = m.stats()
        demanded = int((g["counts"] > 0).sum()) + 1
        assert demanded <= 12
        assert s2.expert_misses == s1.expert_misses == s0.expert_misses
        assert s2.expert_hits - s1.expert_hits == demanded
        assert s2.prefetch_used - s0.prefetch_used == s1.prefetched - s0.prefetched
        gf = GH.run(full, x)
        for key in ("ids", "counts"):
            assert np.array_equal(g[key], gf[key]), (step, key)
        GH.compare(lay, x, g)
    full.close()
    m.close()


def test_prefetch_edge_cases():
    shape = synth.LayerShape(256, 256, 16, 2, 64, True)
    lay = synth.make_layer(shape, seed=33, codes="uniform")
    m = _partial(lay, 4, 8)
    x = torch.from_numpy(synth.make_tokens(shape.hidden, 8, seed=33)).cuda()
    m.prefetch(x[:0])  # T = 0: nothing
    assert m.stats().prefetch_calls == 0
    with pytest.raises(capi.MoEError) as ei:
        capi.check(capi.moe_layer_prefetch(m.handle, x.data_ptr(), 9, None), "prefetch")
    assert ei.value.status == capi.MOE_ERR_INVALID_ARG
    # more guessed experts than slots: at most num_slots are copied
    m.prefetch(x)
    torch.cuda.synchronize()
    st = m.stats()
    assert st.prefetch_calls == 1 and 0 < st.prefetched <= 4
    g = GH.run(m, synth.make_tokens(shape.hidden, 8, seed=33))
    GH.compare(lay, synth.make_tokens(shape.hidden, 8, seed=33), g)
    m.close()
    # full residency: a no-op
    f = GH.upload(lay, max_tokens=8)
    capi.check(capi.moe_layer_prefetch(f.handle, x.data_ptr(), 8, None), "prefetch")
    assert f.stats().prefetch_calls == 0
    f.close()


def test_a_failed_prefetch_is_reported_once_and_leaves_the_cache_consistent(monkeypatch):
    # host-side injection: the planning thread aborts the guess's copies
    # before publication; the next forward reports it, the one after is
    # correct and nothing the guess would have loaded became resident
    monkeypatch.setenv("MOE_FAULT_INJECT", "prefetch_fail")
    shape = synth.LayerShape(256, 256, 16, 2, 64, True)
    lay = synth.make_layer(shape, seed=34, codes="uniform")
    m = _partial(lay, 6, 4)
    x = synth.make_tokens(shape.hidden, 4, seed=34)
    m.prefetch(torch.from_numpy(x).cuda())
    with pytest.raises(capi.MoEError) as ei:
        GH.run(m, x)
    assert ei.value.status == capi.MOE_ERR_CUDA and "prefetch" in str(ei.value)
    st = m.stats()
    assert st.prefetch_calls == 1 and st.prefetched == 0 and st.h2d_bytes == 0
    g = GH.run(m, x)
    GH.compare(lay, x, g)
    assert m.stats().faulted == 0
    m.close()


def test_prefetch_through_the_staging_ring_of_a_pageable_backing():
    # a pageable host copy goes through a small ring of pinned staging
    # buffers, shared by the forwards and the prefetch thread (which the next
    # forward waits for): results bit-identical to a pinned backing
    shape = synth.LayerShape(512, 384, 24, 3, 128, True)
    lays = [synth.make_layer(shape, seed=synth.stack_layer_seed(35, l)) for l in range(3)]
    dev = torch.device("cuda")

    def make(lay, pinned):
        host = torch.from_numpy(lay.records[lay.expert_to_slot]).contiguous()
        if pinned:
            host = host.pin_memory()
        return MoELayer(hidden=shape.hidden, intermediate=shape.intermediate, num_experts=shape.num_experts,
                        top_k=shape.top_k, group_size=shape.group_size, renormalize=shape.renormalize,
                        max_tokens=4, router_w=torch.from_numpy(lay.router_w).to(dev), num_slots=6, spare_slots=2,
                        host_backing=host, staging_records=2, add_residual=True)

    x0 = torch.from_numpy(synth.make_tokens(shape.hidden, 4, seed=35)).cuda()
    pageable = [make(l, False) for l in lays]
    pinned = [make(l, True) for l in lays]
    a = _run_stack(pageable, x0, 4, prefetch=True)
    b = _run_stack(pinned, x0, 4, prefetch=False)
    for step in range(4):
        for l in range(3):
            assert np.array_equal(a[step][l], b[step][l]), (step, l)
    st = pageable[1].stats()
    assert st.staged_copies > 0 and st.prefetch_calls == 4 and st.faulted == 0
    for m in pageable + pinned:
        m.close()
