"""Stacked layers with a residual stream (16 OLMoE-shaped layers):
x_{l+1} = fp16(x_l + fp16(layer_l(x_l))), next step's input = last output +
N(0, 0.1) (the literal recipe, finite over the steps run here). Checked
teacher-forced: every layer and every token against the oracle fed the GPU's
own input to that layer, for the layers' own forwards and for the stack
handle (one launch for the whole stack at one token)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import moe_oracle as O  # noqa: E402
from w4a16_routed_expert_gb300 import capi, synth  # noqa: E402
from w4a16_routed_expert_gb300.layer import MoEStack  # noqa: E402

import gpu_harness as GH  # noqa: E402

LAYERS = 16


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    capi.lib()


@pytest.fixture(scope="module")
def stack_layers():
    return [synth.make_layer(synth.OLMOE, seed=synth.stack_layer_seed(2, l)) for l in range(LAYERS)]


@pytest.mark.parametrize("T,steps,checked", [(1, 2, range(LAYERS)), (64, 1, range(LAYERS))])
def test_stack_teacher_forced(stack_layers, T, steps, checked):
    shape = synth.OLMOE
    mls = [GH.upload(lay, max_tokens=T, add_residual=True) for lay in stack_layers]
    x = synth.make_tokens(shape.hidden, T, seed=77)
    kw = GH.oracle_kw(shape)
    for step in range(steps):
        xin = x
        for l in range(LAYERS):
            g = GH.run(mls[l], xin)
            xout = g["out"].astype(np.float16)
            if l in checked:
                lay = stack_layers[l]
                ref = O.moe_forward(xin, lay.router_w, None, lay.records, lay.expert_to_slot, **kw)
                toks = np.arange(T)
                near = set(O.near_tie_tokens(ref["logits"], shape.top_k).tolist())
                for i, t in enumerate(toks):
                    if int(t) in near:
                        continue
                    layer_out = ref["out"][i]
                    expect = O.residual_add(xin[t:t + 1], layer_out.astype(np.float16)[None, :])[0].astype(np.float64)
                    got = xout[t].astype(np.float64)
                    # the residual is rounded twice in FP16: allow the layer
                    # tolerance plus one FP16 unit of the result
                    tol = GH.TOL * np.maximum(1, np.abs(layer_out)) + np.abs(expect) * 2.0 ** -10
                    assert (np.abs(got - expect) <= tol).all(), (step, l, int(t))
            xin = xout
        noise = synth.make_noise(shape.hidden, T, seed=2, step=step)
        x = (xin.astype(np.float32) + noise).astype(np.float16)
    for m in mls:
        m.close()


def _check_layer(lay, shape, xin, xout, step, l):
    """Teacher-forced check of one layer's output rows against the oracle
    fed the same input (near-tie tokens excluded)."""
    kw = GH.oracle_kw(shape)
    ref = O.moe_forward(xin, lay.router_w, lay.router_bias, lay.records, lay.expert_to_slot, **kw)
    near = set(O.near_tie_tokens(ref["logits"], shape.top_k).tolist())
    for t in range(xin.shape[0]):
        if t in near:
            continue
        layer_out = ref["out"][t]
        expect = O.residual_add(xin[t:t + 1], layer_out.astype(np.float16)[None, :])[0].astype(np.float64)
        got = xout[t].astype(np.float64)
        tol = GH.TOL * np.maximum(1, np.abs(layer_out)) + np.abs(expect) * 2.0 ** -10
        assert (np.abs(got - expect) <= tol).all(), (step, l, t)
    return ref, near


def _stack_run(st, x_np, n, T):
    dev = torch.device("cuda")
    x = torch.from_numpy(x_np).to(dev)
    states = torch.full((max(n - 1, 1), T, x.shape[1]), float("nan"), dtype=torch.float16, device=dev)
    out = torch.full_like(x, float("nan"))
    s = GH.stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        st.forward(x, out=out, states=states if n > 1 else None)
        st.sync()
    ins = [x_np] + [states[l].cpu().numpy() for l in range(n - 1)]
    outs = [states[l].cpu().numpy() for l in range(n - 1)] + [out.cpu().numpy()]
    return ins, outs


def test_stack_kernel_teacher_forced(stack_layers):
    # one launch per step for all 16 layers; two steps of the literal recipe
    shape = synth.OLMOE
    mls = [GH.upload(lay, max_tokens=1, add_residual=True) for lay in stack_layers]
    st = MoEStack(mls)
    assert st.single_launch
    x = synth.make_tokens(shape.hidden, 1, seed=78)
    for step in range(2):
        ins, outs = _stack_run(st, x, LAYERS, 1)
        for l in range(LAYERS):
            assert np.isfinite(outs[l]).all(), (step, l)
            ref, near = _check_layer(stack_layers[l], shape, ins[l], outs[l], step, l)
            # the layer's own routing of this forward: its experts, unless near a tie
            counts = mls[l].routing(1)[0].cpu().numpy()
            if 0 not in near:
                want = np.zeros(shape.num_experts, dtype=np.int64)
                want[ref["ids"][0]] = 1
                assert np.array_equal(counts, want), (step, l)
        noise = synth.make_noise(shape.hidden, 1, seed=2, step=step)
        x = (outs[-1].astype(np.float32) + noise).astype(np.float16)
    st.close()
    for m in mls:
        m.close()


def test_stack_kernel_repeatable_and_counted(stack_layers):
    shape = synth.OLMOE
    mls = [GH.upload(lay, max_tokens=1, add_residual=True) for lay in stack_layers[:6]]
    st = MoEStack(mls)
    x = synth.make_tokens(shape.hidden, 1, seed=79)
    a = _stack_run(st, x, 6, 1)
    b = _stack_run(st, x, 6, 1)
    for l in range(6):
        assert np.array_equal(a[1][l], b[1][l]), l
    for m in mls:
        s_ = m.stats()
        assert s_.forward_calls == 2 and s_.tokens == 2
    st.close()
    for m in mls:
        m.close()


@pytest.mark.parametrize("shape,n", [
    (synth.LayerShape(256, 128, 8, 2, 64, True, has_shared=True), 3),
    (synth.LayerShape(512, 256, 128, 6, 128, False), 2),
    (synth.LayerShape(256, 256, 16, 4, 64, True), 1),
])
def test_stack_kernel_other_shapes(shape, n):
    lays = [synth.make_layer(shape, seed=synth.stack_layer_seed(5, l)) for l in range(n)]
    mls = [GH.upload(lay, max_tokens=1, add_residual=True) for lay in lays]
    st = MoEStack(mls)
    assert st.single_launch
    x = synth.make_tokens(shape.hidden, 1, seed=80)
    ins, outs = _stack_run(st, x, n, 1)
    for l in range(n):
        _check_layer(lays[l], shape, ins[l], outs[l], 0, l)
    st.close()
    for m in mls:
        m.close()


@pytest.mark.parametrize("T,single_off", [(4, False), (1, True)])
def test_stack_of_layer_forwards_matches_the_layers(stack_layers, monkeypatch, T, single_off):
    # without the stack kernel the stack runs each layer's own forward: the
    # same bits as calling the layers one after another
    if single_off:
        monkeypatch.setenv("MOE_STACK1", "0")
    shape = synth.OLMOE
    n = 4
    mls = [GH.upload(lay, max_tokens=T, add_residual=True) for lay in stack_layers[:n]]
    st = MoEStack(mls)
    assert st.single_launch == (not single_off)  # eligibility; a T > 1 call runs the layers
    x = synth.make_tokens(shape.hidden, T, seed=81)
    ins, outs = _stack_run(st, x, n, T)
    xin = x
    for l in range(n):
        g = GH.run(mls[l], xin)
        assert np.array_equal(g["out"].astype(np.float16), outs[l]), l
        xin = g["out"].astype(np.float16)
    st.close()
    for m in mls:
        m.close()
