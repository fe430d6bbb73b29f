"""Stacked layers with a residual stream (16 OLMoE-shaped layers):
x_{l+1} = fp16(x_l + fp16(layer_l(x_l))), next step's input = last output +
N(0, 0.1) (the literal recipe, finite over the steps run here). Checked
teacher-forced: every layer and every token against the oracle fed the GPU's
own input to that layer."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import moe_oracle as O  # noqa: E402
from w4a16_routed_expert_gb300 import capi, synth  # noqa: E402

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
