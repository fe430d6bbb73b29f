"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle."""
import json
import os

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


# ----------------------------------------------------------------------------
# hand-worked two-expert layer, embedded at a size the kernels run
# ----------------------------------------------------------------------------

def _embed_fixture(fx, case, H=128, I=128, G=64):
    """The 4-wide / 2-wide fixture padded with zero weights (code 8) to H=128,
    I=128, one scale per row (each fixture row's non-zero weights share one
    scale)."""
    Gs = fx["G"]
    recs = []
    for ex in fx["experts"]:
        mats = []
        for name, (n, kdim, N, K) in (("gate", (2, 4, I, H)), ("up", (2, 4, I, H)), ("down", (4, 2, H, I))):
            codes = np.array(ex[name + "_codes"])
            scales = np.array(ex[name + "_scales"], dtype=np.float64)
            q = np.full((N, K), 8, dtype=np.uint8)
            s = np.ones((N, -(-K // G)), dtype=np.float16)
            for r in range(n):
                w = (codes[r] - 8) * np.repeat(scales[r], Gs)[:kdim]
                nz = [gi for gi in range(scales.shape[1])
                      if scales[r, gi] != 0 and (codes[r, gi * Gs:(gi + 1) * Gs] != 8).any()]
                sr = scales[r, nz[0]] if nz else 1.0
                qq = w / sr + 8
                assert np.allclose(qq, np.rint(qq)) and (qq >= 0).all() and (qq <= 15).all()
                q[r, :kdim] = np.rint(qq).astype(np.uint8)
                s[r, 0] = sr
            mats.append((q, s))
        (gq, gs), (uq, us), (dq, ds) = mats
        recs.append(synth.pack_record(H, I, G, gq, uq, dq, gs, us, ds))
    recs = np.stack(recs)
    rw = np.zeros((2, H), dtype=np.float32)
    rw[:, :4] = np.array(case["router_w"], dtype=np.float32)
    x = np.zeros((2, H), dtype=np.float16)
    x[:, :4] = np.array(fx["x"], dtype=np.float16)
    shape = synth.LayerShape(H, I, 2, case["k"], G, case["renormalize"])
    lay = synth.Layer(shape, rw, None, recs[::-1].copy(), np.array([1, 0], dtype=np.int32))
    return lay, x


@pytest.mark.parametrize("case", ["tie", "k1", "k2"])
def test_hand_worked_two_expert_layer(golden_dir, case):
    with open(os.path.join(golden_dir, "two_expert_h4.json")) as f:
        fx = json.load(f)
    c = [c for c in fx["cases"] if c["name"] == case][0]
    lay, x = _embed_fixture(fx, c)
    ml = GH.upload(lay, max_tokens=4)
    g = GH.run(ml, x)
    assert g["ids"].tolist() == c["ids"]
    np.testing.assert_allclose(g["w"], c["weights"], rtol=1e-6)
    assert g["counts"].tolist() == c["counts"] and g["offsets"].tolist() == c["offsets"]
    assert g["perm"].tolist() == c["perm"] and g["inv_perm"].tolist() == c["inv_perm"]
    expect = np.zeros((2, 128))
    expect[:, :4] = np.array(c["out"])
    assert (np.abs(g["out"] - expect) <= GH.TOL * np.maximum(1, np.abs(expect))).all()
    ml.close()


# ----------------------------------------------------------------------------
# seeded synthetic layers against the oracle
# ----------------------------------------------------------------------------

PARITY_CASES = [
    # (id, shape, seed, T, codes)
    ("tiny-T4", synth.TINY, 0, 4, "quantized"),
    ("tiny-uniform-T7", synth.TINY, 1, 7, "uniform"),
    ("olmoe-T1", synth.OLMOE, 1, 1, "quantized"),
    ("olmoe-T4", synth.OLMOE, 1, 4, "quantized"),
    ("olmoe-T16", synth.OLMOE, 1, 16, "quantized"),
    ("many-experts-T1", synth.MANY_EXPERTS, 3, 1, "quantized"),
    ("many-experts-T16", synth.MANY_EXPERTS, 3, 16, "quantized"),
    ("wide-2880-T3", synth.LayerShape(2880, 2880, 8, 4, 128, True), 4, 3, "uniform"),
    ("k1-E1", synth.LayerShape(256, 256, 1, 1, 128, True), 5, 5, "uniform"),
    ("shared-G64-T9", synth.LayerShape(512, 384, 16, 3, 64, False, has_shared=True), 6, 9, "uniform"),
]


@pytest.mark.parametrize("name,shape,seed,T,codes", PARITY_CASES, ids=[c[0] for c in PARITY_CASES])
def test_parity_small_batches(name, shape, seed, T, codes):
    lay = synth.make_layer(shape, seed=seed, codes=codes)
    x = synth.make_tokens(shape.hidden, T, seed=seed)
    ml = GH.upload(lay, max_tokens=max(T, 16))
    g = GH.run(ml, x)
    rep = GH.compare(lay, x, g)
    print(name, rep)
    ml.close()


@pytest.mark.parametrize("T", [17, 64, 200])
def test_parity_multi_chunk_routing(T):
    """T > 16 takes the multi-kernel routing path (32-token chunks, ragged
    last chunk); every output row checked."""
    shape = synth.OLMOE
    lay = synth.make_layer(shape, seed=7)
    x = synth.make_tokens(shape.hidden, T, seed=7)
    ml = GH.upload(lay, max_tokens=T)
    g = GH.run(ml, x)
    GH.compare(lay, x, g)
    ml.close()


def test_many_experts_T256_every_row():
    """The 256-token many-expert batch in the launch configuration the
    benchmark times (the library's own path choice): every row."""
    shape = synth.MANY_EXPERTS
    lay = synth.make_layer(shape, seed=3)
    x = synth.make_tokens(shape.hidden, 256, seed=3)
    ml = GH.upload(lay, max_tokens=256)
    g = GH.run(ml, x)
    rep = GH.compare(lay, x, g)
    assert rep["rows_compared"] == 256
    ml.close()


def test_exact_ties_go_to_lowest_id():
    # duplicated router rows: experts 2/5 and 3/6 always tie exactly
    shape = synth.LayerShape(256, 128, 8, 3, 64, True)
    lay = synth.make_layer(shape, seed=8)
    lay.router_w[5] = lay.router_w[2]
    lay.router_w[6] = lay.router_w[3]
    x = synth.make_tokens(256, 16, seed=8)
    ml = GH.upload(lay, max_tokens=16)
    g = GH.run(ml, x)
    ref = O.moe_forward(x, lay.router_w, None, lay.records, lay.expert_to_slot, **GH.oracle_kw(shape))
    # identical rows give identical logits on both sides: the tie is exact
    assert np.array_equal(g["ids"], ref["ids"])
    for t in range(16):
        row = g["ids"][t].tolist()
        for lo, hi in ((2, 5), (3, 6)):
            if hi in row:
                assert lo in row and row.index(lo) < row.index(hi), (t, row)
    ml.close()


def test_zero_tokens_is_a_no_op():
    shape = synth.TINY
    lay = synth.make_layer(shape, seed=0)
    ml = GH.upload(lay, max_tokens=4)
    x = torch.zeros((0, shape.hidden), dtype=torch.float16, device="cuda")
    out = torch.zeros((0, shape.hidden), dtype=torch.float16, device="cuda")
    ml.forward(x, out=out)
    ml.sync()
    ml.close()


def test_too_many_tokens_is_rejected():
    shape = synth.TINY
    lay = synth.make_layer(shape, seed=0)
    ml = GH.upload(lay, max_tokens=4)
    x = torch.zeros((5, shape.hidden), dtype=torch.float16, device="cuda")
    with pytest.raises(capi.MoEError) as ei:
        ml.forward(x)
    assert ei.value.status == capi.MOE_ERR_INVALID_ARG
    ml.close()


def test_max_tokens_exactly():
    shape = synth.OLMOE
    lay = synth.make_layer(shape, seed=9)
    x = synth.make_tokens(shape.hidden, 16, seed=9)
    ml = GH.upload(lay, max_tokens=16)
    g = GH.run(ml, x)
    GH.compare(lay, x, g)
    ml.close()


def test_residual_add_matches_two_step_definition():
    shape = synth.OLMOE
    lay = synth.make_layer(shape, seed=10)
    x = synth.make_tokens(shape.hidden, 4, seed=10)
    ml = GH.upload(lay, max_tokens=4)
    plain = GH.run(ml, x)["out"].astype(np.float16)
    ml.close()
    mr = GH.upload(lay, max_tokens=4, add_residual=True)
    fused = GH.run(mr, x)["out"].astype(np.float16)
    mr.close()
    # fused residual == fp16(x + fp16(layer(x))) computed from the plain run
    assert np.array_equal(fused, O.residual_add(x, plain))


def test_zero_scales_give_exact_zero():
    shape = synth.OLMOE
    lay = synth.make_layer(shape, seed=11)
    offs, _ = O.record_layout(shape.hidden, shape.intermediate, shape.group_size)
    for name in ("gate_s", "up_s", "down_s"):
        o, n = offs[name]
        lay.records[:, o:o + n] = 0
    x = synth.make_tokens(shape.hidden, 3, seed=11)
    ml = GH.upload(lay, max_tokens=4)
    g = GH.run(ml, x)
    assert (g["out"] == 0).all()
    ml.close()


def test_repeatable_bit_for_bit_and_pdl_independent(monkeypatch):
    shape = synth.MANY_EXPERTS
    lay = synth.make_layer(shape, seed=12)
    x = synth.make_tokens(shape.hidden, 16, seed=12)
    ml = GH.upload(lay, max_tokens=16)
    a = GH.run(ml, x)
    b = GH.run(ml, x)
    ml.close()
    monkeypatch.setenv("MOE_PDL", "0")
    ml2 = GH.upload(lay, max_tokens=16)
    c = GH.run(ml2, x)
    ml2.close()
    for key in ("out", "ids", "w", "perm"):
        assert np.array_equal(a[key], b[key]) and np.array_equal(a[key], c[key]), key


@pytest.mark.parametrize("T,pinned", [(1, "all"), (4, "all"), (16, "all"), (24, "all"), (4, "none"), (1, "x-only")])
def test_forward_host_buffers_match_device_forward(T, pinned):
    # mapped (page-locked) buffers up to 16 tokens are read / written in
    # place by the kernels; pageable ones, a mix, or more tokens go through
    # the staging copies: the same bits every way
    shape = synth.OLMOE
    lay = synth.make_layer(shape, seed=13)
    x = synth.make_tokens(shape.hidden, T, seed=13)
    ml = GH.upload(lay, max_tokens=T)
    dev = GH.run(ml, x)

    def buf(t, pin):
        return t.pin_memory() if pin else t

    xh = buf(torch.from_numpy(x), pinned in ("all", "x-only"))
    oh = buf(torch.full(xh.shape, float("nan"), dtype=torch.float16), pinned == "all")
    ih = buf(torch.full((T, shape.top_k), -1, dtype=torch.int32), pinned == "all")
    wh = buf(torch.full((T, shape.top_k), float("nan"), dtype=torch.float32), pinned == "all")
    for _ in range(2):
        ml.forward_host(xh, oh, ih, wh)
        ml.sync()
        assert np.array_equal(oh.float().numpy(), dev["out"])
        assert np.array_equal(ih.numpy(), dev["ids"]) and np.array_equal(wh.numpy(), dev["w"])
    ml.close()


@pytest.mark.parametrize("shape,seed,T", [(synth.OLMOE, 50, 1), (synth.OLMOE, 51, 4), (synth.OLMOE, 52, 16),
                                          (synth.MANY_EXPERTS, 53, 1), (synth.MANY_EXPERTS, 54, 16),
                                          (synth.TINY, 55, 3)])
def test_single_launch_decode_matches_multi_kernel_path(shape, seed, T, monkeypatch):
    """The one-launch decode path (T <= 16) against the routing / GEMV /
    combine kernels: both compute the logits with the same function and the
    experts with the same work items, so every output is bit-identical."""
    lay = synth.make_layer(shape, seed=seed)
    x = synth.make_tokens(shape.hidden, T, seed=seed)
    monkeypatch.setenv("MOE_DECODE1", "0")  # batch 1 too: this compares the two kernels below
    monkeypatch.setenv("MOE_MEGAKERNEL_MAX_T", "16")  # the one-launch path for every T here
    mk = GH.upload(lay, max_tokens=T)
    a = GH.run(mk, x)
    b2 = GH.run(mk, x)
    mk.close()
    monkeypatch.setenv("MOE_MEGAKERNEL", "0")
    mm = GH.upload(lay, max_tokens=T)
    b = GH.run(mm, x)
    mm.close()
    GH.compare(lay, x, a)
    for key in ("out", "ids", "w", "perm", "counts", "offsets"):
        assert np.array_equal(a[key], b2[key]), key  # repeatable across launches (counters reset)
    for key in ("out", "ids", "w", "perm", "inv_perm", "counts", "offsets"):
        assert np.array_equal(a[key], b[key]), key


BATCH1_CASES = [
    ("olmoe", synth.OLMOE, 60, "quantized"),
    ("many-experts", synth.MANY_EXPERTS, 61, "quantized"),
    ("tiny-uniform", synth.TINY, 62, "uniform"),
    ("shared-G64", synth.LayerShape(512, 384, 16, 3, 64, False, has_shared=True), 63, "uniform"),
    ("k1-E1", synth.LayerShape(256, 256, 1, 1, 128, True), 64, "uniform"),
    ("E1024-k32", synth.LayerShape(256, 128, 1024, 32, 64, True, router_std=0.2), 65, "uniform"),
]


@pytest.mark.parametrize("name,shape,seed,codes", BATCH1_CASES, ids=[c[0] for c in BATCH1_CASES])
def test_batch1_kernel_matches_oracle_and_the_other_paths(name, shape, seed, codes, monkeypatch):
    """One token takes the batch-1 kernel (every CTA's share of the bytes
    requested at once, the combine local to each CTA): against the oracle,
    repeatable bit for bit across launches, the same routing bits as the
    single-launch small-batch kernel and the multi-kernel path (the logits
    and the softmax use the same FP32 arithmetic), and outputs that agree
    with theirs within the layer tolerance (the per-group partial sums are
    added in another order)."""
    lay = synth.make_layer(shape, seed=seed, codes=codes)
    ml = GH.upload(lay, max_tokens=4)
    for call in range(3):
        x = synth.make_tokens(shape.hidden, 1, seed=seed * 10 + call)
        a = GH.run(ml, x)
        a2 = GH.run(ml, x)
        GH.compare(lay, x, a)
        for key in ("out", "ids", "w", "perm", "inv_perm", "counts", "offsets"):
            assert np.array_equal(a[key], a2[key]), key
        for env in ({"MOE_DECODE1": "0"}, {"MOE_DECODE1": "0", "MOE_MEGAKERNEL": "0"}):
            for kv in env.items():
                monkeypatch.setenv(*kv)
            other = GH.upload(lay, max_tokens=4)
            b = GH.run(other, x)
            other.close()
            for kv in env:
                monkeypatch.delenv(kv)
            for key in ("ids", "w", "perm", "inv_perm", "counts", "offsets"):
                assert np.array_equal(a[key], b[key]), (env, key)
            err = np.abs(a["out"] - b["out"])
            assert (err <= GH.TOL * np.maximum(1, np.abs(b["out"]))).all(), (env, err.max())
    ml.close()
