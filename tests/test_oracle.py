"""Pins of the CPU oracle to facts that do not come from the oracle itself:
hand-written bytes, a hand-worked two-expert layer, brute-force orderings,
library routines, closed-form sizes printed on the pages, special cases and
invariants. CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from w4a16_routed_expert_gb300 import synth


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# record format
# ----------------------------------------------------------------------------

def test_unpack_hand_written_bytes(golden_dir):
    fx = _load(golden_dir, "nibble_bytes.json")
    raw = np.array(fx["bytes"], dtype=np.uint8)
    q = O.unpack_codes(raw, 1, 8)
    assert q[0].tolist() == fx["codes"]
    w = O.dequantize(q, np.full((1, 1), fx["scale"], dtype=np.float16), 8)
    assert w[0].tolist() == fx["weights"]


def test_dequantize_ragged_last_group():
    # K = 6, G = 4: codes 0..3 use scale 0, codes 4..5 use scale 1 (ragged group)
    q = np.array([[9, 10, 7, 8, 12, 0]])
    s = np.array([[2.0, -0.25]], dtype=np.float16)
    w = O.dequantize(q, s, 4)
    assert w[0].tolist() == [2.0, 4.0, -2.0, 0.0, -1.0, 2.0]


def test_record_sizes_closed_form():
    # OLMoE-shaped expert: 3 matrices of 2048 x 1024 codes + 128-code groups
    offs, rb = O.record_layout(2048, 1024, 128)
    assert rb == 3 * 2048 * 1024 // 2 + 3 * 2 * 2048 * 1024 // 128 == 3_244_032
    assert synth.record_bytes(2048, 1024, 128) == rb
    # many-expert layer (intermediate 512) and the tiny layer
    assert O.record_layout(2048, 512, 128)[1] == 1_622_016
    assert O.record_layout(256, 128, 64)[1] == 52_224
    # H = I = 2880, G = 128: 23 groups per row, the last one 64 codes wide;
    # payload 12,839,040 B, padded to 256-byte sections
    offs, rb = O.record_layout(2880, 2880, 128)
    payload = sum(n for (_, n) in offs.values())
    assert payload == 12_839_040 and rb == 12_839_424
    assert synth.section_layout(2880, 2880, 128)["payload_bytes"] == payload
    for name, (o, n) in offs.items():
        assert o % 256 == 0
        assert synth.section_layout(2880, 2880, 128)[name] == (o, n)


def test_expert_sizes_match_pages():
    # moe-stream, "Method": each of the 1,024 OLMoE experts is a 12.6 MB file
    # (BF16, 3 x 2048 x 1024 parameters); "Speed against memory": 13 GB of
    # experts.
    params = 3 * 2048 * 1024
    assert round(params * 2 / 1e6, 1) == 12.6
    assert round(1024 * params * 2 / 1e9) == 13
    # F51 Nitro-MoE, "The simulator": gpt-oss-120B, 128 experts, 12.61 MiB
    # per expert in MXFP4 (4.25 bits per parameter), hidden = intermediate =
    # 2880.
    assert round(3 * 2880 * 2880 * 4.25 / 8 / 2**20, 2) == 12.61
    # stacked OLMoE-shaped workload: 16 layers x 64 experts of INT4 codes
    # come to about 3.2 GB.
    assert round(16 * 64 * params / 2 / 1e9, 1) == 3.2


def test_synth_pack_roundtrip_through_oracle_unpack():
    rng = np.random.default_rng(3)
    q = rng.integers(0, 16, size=(5, 64), dtype=np.uint8)
    raw = synth.pack_nibbles(q)
    assert np.array_equal(O.unpack_codes(raw, 5, 64), q)


# ----------------------------------------------------------------------------
# hand-worked two-expert layer
# ----------------------------------------------------------------------------

def _fixture_records(fx, shared_from=None):
    H, I, G = fx["H"], fx["I"], fx["G"]
    recs = []
    srcs = list(fx["experts"])
    if shared_from is not None:
        srcs.append(fx["experts"][shared_from])
    for ex in srcs:
        recs.append(synth.pack_record(
            H, I, G,
            np.array(ex["gate_codes"]), np.array(ex["up_codes"]), np.array(ex["down_codes"]),
            np.array(ex["gate_scales"], dtype=np.float16), np.array(ex["up_scales"], dtype=np.float16),
            np.array(ex["down_scales"], dtype=np.float16)))
    return np.stack(recs)


@pytest.mark.parametrize("case", ["tie", "k1", "k2"])
def test_two_expert_hand_worked(golden_dir, case):
    fx = _load(golden_dir, "two_expert_h4.json")
    c = [c for c in fx["cases"] if c["name"] == case][0]
    recs = _fixture_records(fx)
    # store the records in swapped slots to exercise the indirection
    recs = recs[::-1].copy()
    e2s = np.array([1, 0])
    x = np.array(fx["x"], dtype=np.float16)
    r = O.moe_forward(x, np.array(c["router_w"], dtype=np.float32), None, recs, e2s,
                      H=fx["H"], I=fx["I"], E=fx["E"], k=c["k"], G=fx["G"],
                      renormalize=c["renormalize"])
    assert r["ids"].tolist() == c["ids"]
    np.testing.assert_allclose(r["weights"], c["weights"], rtol=1e-14, atol=0)
    assert r["counts"].tolist() == c["counts"]
    assert r["offsets"].tolist() == c["offsets"]
    assert r["perm"].tolist() == c["perm"]
    assert r["inv_perm"].tolist() == c["inv_perm"]
    np.testing.assert_allclose(r["out"], c["out"], rtol=1e-14, atol=1e-15)


def test_two_expert_per_expert_outputs(golden_dir):
    fx = _load(golden_dir, "two_expert_h4.json")
    recs = _fixture_records(fx)
    x = np.array(fx["x"], dtype=np.float16)
    for e, ex in enumerate(fx["experts"]):
        wg, wu, wd = O.expert_matrices(recs[e], fx["H"], fx["I"], fx["G"])
        np.testing.assert_allclose(O.expert_ffn(wg, wu, wd, x), ex["y"], rtol=1e-14, atol=1e-15)


def test_two_expert_shared_expert(golden_dir):
    # shared expert = a third record with expert 0's weights, weight 1, run on
    # every token: out = routed out + y_0(x)
    fx = _load(golden_dir, "two_expert_h4.json")
    recs = _fixture_records(fx, shared_from=0)
    c = [c for c in fx["cases"] if c["name"] == "k1"][0]
    x = np.array(fx["x"], dtype=np.float16)
    r = O.moe_forward(x, np.array(c["router_w"], dtype=np.float32), None, recs, np.arange(3),
                      H=fx["H"], I=fx["I"], E=2, k=1, G=fx["G"], renormalize=True, has_shared=True)
    np.testing.assert_allclose(r["out"], np.array(c["out"]) + np.array(fx["experts"][0]["y"]),
                               rtol=1e-14, atol=1e-15)


# ----------------------------------------------------------------------------
# routing
# ----------------------------------------------------------------------------

def test_topk_against_full_sort_with_ties():
    rng = np.random.default_rng(7)
    for E, k in ((8, 2), (16, 5), (64, 8), (7, 7)):
        L = rng.integers(-3, 4, size=(40, E)).astype(np.float64)  # many exact ties
        # brute force: full order by (logit descending, id ascending)
        ref = np.array([sorted(range(E), key=lambda e: (-row[e], e))[:k] for row in L])
        assert np.array_equal(O.select_topk(L, k), ref)
        assert np.array_equal(O.select_topk_fast(L, k), ref)


def test_topk_non_finite_logits_hand_worked():
    # NaN ranks below every number (as -inf); equal keys go to the lower id.
    # Row 0 keys: [-inf, 1, -inf, 1, -inf, 3] -> 5, then 1 and 3 (tie, lower
    # id first), then the lowest id among the -inf keys, 0.
    # Row 1: every logit NaN -> all keys equal -> ids 0, 1, 2, 3.
    # Row 2: +inf beats every number; -inf and NaN tie below them.
    nan, inf = np.nan, np.inf
    L = np.array([[nan, 1.0, nan, 1.0, -inf, 3.0],
                  [nan, nan, nan, nan, nan, nan],
                  [-inf, nan, inf, 0.5, inf, -2.0]])
    expect = [[5, 1, 3, 0], [0, 1, 2, 3], [2, 4, 3, 5]]
    assert O.select_topk(L, 4).tolist() == expect
    assert O.select_topk_fast(L, 4).tolist() == expect
    # the fast path must not re-take an entry when every remaining key is -inf
    L2 = np.array([[-inf, -inf, 7.0, -inf]])
    assert O.select_topk_fast(L2, 4).tolist() == [[2, 0, 1, 3]]
    assert O.select_topk(L2, 4).tolist() == [[2, 0, 1, 3]]


def test_softmax_and_silu_against_library():
    rng = np.random.default_rng(1)
    L = rng.normal(0, 3, size=(20, 33))
    ref = torch.softmax(torch.from_numpy(L), dim=1).numpy()
    np.testing.assert_allclose(O.softmax_rows(L), ref, rtol=1e-13, atol=0)
    z = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(O.silu(z), torch.nn.functional.silu(torch.from_numpy(z)).numpy(),
                               rtol=1e-13, atol=1e-300)


def test_router_zero_special_case():
    x = synth.make_tokens(64, 5, seed=2)
    for renorm in (False, True):
        L = O.router_logits(x, np.zeros((16, 64), dtype=np.float32))
        p = O.softmax_rows(L)
        ids = O.select_topk_fast(L, 4)
        assert (ids == np.arange(4)).all()
        w = O.routing_weights(p, ids, renorm)
        np.testing.assert_allclose(w, 1 / 4 if renorm else 1 / 16, rtol=1e-15)


def test_router_logits_against_integer_arithmetic():
    # integer-valued inputs: the logits are exact integers
    rng = np.random.default_rng(4)
    x = rng.integers(-4, 5, size=(6, 32)).astype(np.float16)
    wr = rng.integers(-3, 4, size=(5, 32)).astype(np.float32)
    b = np.arange(5, dtype=np.float32)
    L = O.router_logits(x, wr, b)
    ref = [[sum(int(x[t, h]) * int(wr[e, h]) for h in range(32)) + e for e in range(5)] for t in range(6)]
    assert L.tolist() == ref


def test_routing_weight_invariants():
    shape = synth.TINY
    lay = synth.make_layer(shape, seed=0)
    x = synth.make_tokens(shape.hidden, 50, seed=0)
    L = O.router_logits(x, lay.router_w)
    p = O.softmax_rows(L)
    ids = O.select_topk_fast(L, shape.top_k)
    wr = O.routing_weights(p, ids, True)
    np.testing.assert_allclose(wr.sum(axis=1), 1.0, rtol=1e-14)
    wn = O.routing_weights(p, ids, False)
    assert (wn.sum(axis=1) <= 1.0 + 1e-15).all()
    # rank order: weights non-increasing along j
    assert (np.diff(wn, axis=1) <= 0).all()


def test_near_tie_detection():
    L = np.array([[3.0, 2.0, 1.0, 0.0], [3.0, 1.0005, 1.0, 0.0], [3.0, 2.0, 2.0, 0.0]])
    # k = 2: row 1 has 1.0005 vs 1.0 at the k / k+1 boundary, row 2 an exact tie
    assert O.near_tie_tokens(L, 2).tolist() == [1, 2]
    # k = 1: row 2's boundary is 3 vs 2 (no tie); rank-adjacent gaps k..k+1 only
    assert O.near_tie_tokens(L, 1).tolist() == []
    assert O.near_tie_tokens(L, 3).tolist() == [1, 2]


# ----------------------------------------------------------------------------
# permutation
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("T,k,E", [(1, 8, 64), (37, 2, 8), (200, 10, 513), (0, 4, 16)])
def test_permutation_invariants(T, k, E):
    rng = np.random.default_rng(T + k + E)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]) if T else np.zeros((0, k), int)
    counts, offsets, perm, inv = O.counting_sort(ids, E)
    flat = ids.reshape(-1)
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert (np.diff(offsets) == counts).all() and (counts >= 0).all()
    # bit-exact against a stable library sort
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(perm[inv], np.arange(T * k))
    assert np.array_equal(inv[perm], np.arange(T * k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert (flat[seg] == e).all() and (np.diff(seg) > 0).all()


# ----------------------------------------------------------------------------
# whole layer
# ----------------------------------------------------------------------------

def _kw(shape, k=None):
    return dict(H=shape.hidden, I=shape.intermediate, E=shape.num_experts, k=k or shape.top_k,
                G=shape.group_size, renormalize=shape.renormalize, has_shared=shape.has_shared)


@pytest.mark.parametrize("codes", ["quantized", "uniform"])
def test_oracle_matches_dense_masked_bruteforce(codes):
    shape = synth.TINY
    lay = synth.make_layer(shape, seed=0, codes=codes)
    x = synth.make_tokens(shape.hidden, 4, seed=0)
    r = O.moe_forward(x, lay.router_w, None, lay.records, lay.expert_to_slot, **_kw(shape))
    dense, sel = O.dense_masked_forward(x, lay.router_w, None, lay.records, lay.expert_to_slot, **_kw(shape))
    assert np.array_equal(r["ids"], sel)
    np.testing.assert_allclose(r["out"], dense, rtol=1e-12, atol=1e-14)


def test_oracle_matches_bruteforce_with_shared_and_bias():
    shape = synth.LayerShape(64, 32, 12, 3, 64, True, has_shared=True, zipf_s=1.1)
    lay = synth.make_layer(shape, seed=5, codes="uniform")
    x = synth.make_tokens(64, 9, seed=5)
    r = O.moe_forward(x, lay.router_w, lay.router_bias, lay.records, lay.expert_to_slot, **_kw(shape))
    dense, sel = O.dense_masked_forward(x, lay.router_w, lay.router_bias, lay.records,
                                        lay.expert_to_slot, **_kw(shape))
    assert np.array_equal(r["ids"], sel)
    np.testing.assert_allclose(r["out"], dense, rtol=1e-12, atol=1e-14)


def test_single_expert_reduces_to_dense_swiglu_ffn():
    # E = 1, k = 1, renormalised: the layer is a plain SwiGLU FFN on the
    # dequantised matrices; checked with torch's own silu and matmul.
    shape = synth.LayerShape(64, 96, 1, 1, 64, True)
    lay = synth.make_layer(shape, seed=11, codes="uniform")
    x = synth.make_tokens(64, 7, seed=11)
    r = O.moe_forward(x, lay.router_w, None, lay.records, lay.expert_to_slot, **_kw(shape))
    wg, wu, wd = (torch.from_numpy(m) for m in O.expert_matrices(lay.records[lay.expert_to_slot[0]], 64, 96, 64))
    xt = torch.from_numpy(x.astype(np.float64))
    ref = (torch.nn.functional.silu(xt @ wg.T) * (xt @ wu.T)) @ wd.T
    np.testing.assert_allclose(r["out"], ref.numpy(), rtol=1e-12, atol=1e-14)


def test_zero_input_and_zero_scales_give_zero():
    shape = synth.TINY
    lay = synth.make_layer(shape, seed=1)
    x0 = np.zeros((3, shape.hidden), dtype=np.float16)
    r = O.moe_forward(x0, lay.router_w, None, lay.records, lay.expert_to_slot, **_kw(shape))
    assert (r["out"] == 0).all()
    # all scales zero -> every weight zero -> output zero for any input
    recs = lay.records.copy()
    offs, _ = O.record_layout(shape.hidden, shape.intermediate, shape.group_size)
    for name in ("gate_s", "up_s", "down_s"):
        o, n = offs[name]
        recs[:, o:o + n] = 0
    x = synth.make_tokens(shape.hidden, 3, seed=1)
    r = O.moe_forward(x, lay.router_w, None, recs, lay.expert_to_slot, **_kw(shape))
    assert (r["out"] == 0).all()


def test_token_subset_matches_full_batch():
    shape = synth.LayerShape(64, 64, 8, 2, 64, False)
    lay = synth.make_layer(shape, seed=9)
    x = synth.make_tokens(64, 12, seed=9)
    full = O.moe_forward(x, lay.router_w, None, lay.records, lay.expert_to_slot, **_kw(shape))
    sub = O.moe_forward(x, lay.router_w, None, lay.records, lay.expert_to_slot, tokens=[3, 7, 11],
                        **_kw(shape))
    # equal up to the matmul's blocking order
    np.testing.assert_allclose(sub["out"], full["out"][[3, 7, 11]], rtol=1e-12, atol=1e-16)


def test_residual_add_rounds_once():
    x = np.array([[1.0, 2048.0]], dtype=np.float16)
    o = np.array([[0.5, 1.0]], dtype=np.float16)
    # 2048 + 1 = 2049 is not an fp16 value; round-half-even gives 2048
    assert O.residual_add(x, o).tolist() == [[1.5, 2048.0]]


@pytest.mark.parametrize("mistake", ["no_zero_point", "swapped_nibbles", "ties_high", "transposed_down"])
def test_planted_mistakes_are_caught(golden_dir, mistake, monkeypatch):
    """A plausible mistake planted in the oracle must fail the hand-worked pin."""
    fx = _load(golden_dir, "two_expert_h4.json")
    if mistake == "no_zero_point":
        monkeypatch.setattr(O, "dequantize", lambda q, s, G, zeros=None: q.astype(np.float64)
                            * np.asarray(s, np.float16).astype(np.float64)[:, np.arange(q.shape[1]) // G])
    elif mistake == "swapped_nibbles":
        orig = O.unpack_codes
        monkeypatch.setattr(O, "unpack_codes", lambda raw, N, K: orig(raw, N, K).reshape(N, K // 2, 2)[:, :, ::-1].reshape(N, K))
    elif mistake == "ties_high":
        def ties_to_highest(L, k):
            nudged = L + 1e-9 * np.arange(L.shape[1])
            return np.argsort(-nudged, axis=1, kind="stable")[:, :k]
        monkeypatch.setattr(O, "select_topk_fast", ties_to_highest)
    elif mistake == "transposed_down":
        orig = O.expert_ffn
        monkeypatch.setattr(O, "expert_ffn", lambda wg, wu, wd, x: orig(wg, wu, wd.T.reshape(wd.shape), x))
    caught = False
    for c in fx["cases"]:
        recs = _fixture_records(fx)
        x = np.array(fx["x"], dtype=np.float16)
        r = O.moe_forward(x, np.array(c["router_w"], dtype=np.float32), None, recs, np.arange(2),
                          H=fx["H"], I=fx["I"], E=fx["E"], k=c["k"], G=fx["G"], renormalize=c["renormalize"])
        if r["ids"].tolist() != c["ids"] or not np.allclose(r["out"], c["out"], rtol=1e-12, atol=1e-14):
            caught = True
    assert caught


# ----------------------------------------------------------------------------
# variants: asymmetric zero points, G = 32, sigmoid-gated shared expert
# ----------------------------------------------------------------------------

def test_zero_point_record_hand_built(golden_dir):
    fx = _load(golden_dir, "zero_point_record.json")
    H, I, G = fx["H"], fx["I"], fx["G"]
    offs, size = O.record_layout(H, I, G, zero_points=True)
    assert {k: v[0] for k, v in offs.items()} == fx["offsets"] and size == fx["record_bytes"]
    rec = np.zeros(size, dtype=np.uint8)
    o = fx["offsets"]

    def put(name, arr, dtype):
        b = np.asarray(arr, dtype=dtype).reshape(-1).view(np.uint8)
        rec[o[name]:o[name] + b.size] = b

    put("gate_q", fx["gate_q_bytes"], np.uint8)
    put("up_q", fx["up_q_bytes"], np.uint8)
    put("down_q", fx["down_q_bytes"], np.uint8)
    put("gate_s", fx["gate_s"], np.float16)
    put("up_s", fx["up_s"], np.float16)
    put("down_s", fx["down_s"], np.float16)
    put("gate_z", fx["gate_z"], np.uint8)
    put("up_z", fx["up_z"], np.uint8)
    put("down_z", fx["down_z"], np.uint8)
    wg, wu, wd = O.expert_matrices(rec, H, I, G, zero_points=True)
    assert wg.tolist() == fx["gate_w"]
    assert wu.tolist() == fx["up_w"]
    assert wd.tolist() == fx["down_w"]
    # the same bytes read without zero points: zero point 8 everywhere
    q = O.unpack_codes(np.array(fx["gate_q_bytes"], dtype=np.uint8), I, H)
    assert q.tolist() == fx["gate_codes"]


def test_zero_point_8_is_the_symmetric_format():
    rng = np.random.default_rng(3)
    q = rng.integers(0, 16, size=(5, 96))
    s = rng.uniform(-1, 1, size=(5, 3)).astype(np.float16)
    a = O.dequantize(q, s, 32)
    b = O.dequantize(q, s, 32, zeros=np.full((5, 3), 8, dtype=np.uint8))
    assert np.array_equal(a, b)
    # and a zero point z shifts every weight of its group by (8 - z) * s
    z = rng.integers(0, 16, size=(5, 3)).astype(np.uint8)
    c = O.dequantize(q, s, 32, zeros=z)
    shift = (8.0 - z.astype(np.float64)) * s.astype(np.float64)
    assert np.allclose(c - a, np.repeat(shift, 32, axis=1), rtol=0, atol=1e-12)


@pytest.mark.parametrize("K", [128, 96])
def test_g32_with_paired_scales_is_g64(K):
    # groups of 32 whose scales (and zero points) agree in pairs are groups
    # of 64: the G = 32 reading reduces to the pinned G = 64 one (K = 96:
    # the last G = 64 group is the ragged 32 codes)
    rng = np.random.default_rng(4)
    q = rng.integers(0, 16, size=(4, K))
    s64 = rng.uniform(-2, 2, size=(4, -(-K // 64))).astype(np.float16)
    z64 = rng.integers(0, 16, size=s64.shape).astype(np.uint8)
    s32 = np.repeat(s64, 2, axis=1)[:, :K // 32]
    z32 = np.repeat(z64, 2, axis=1)[:, :K // 32]
    assert np.array_equal(O.dequantize(q, s32, 32), O.dequantize(q, s64, 64))
    assert np.array_equal(O.dequantize(q, s32, 32, z32), O.dequantize(q, s64, 64, z64))
    # one different scale in the second half changes exactly those 32 codes
    s32b = s32.copy()
    s32b[0, 1] = np.float16(float(s32[0, 1]) + 1.0)
    d = O.dequantize(q, s32b, 32) != O.dequantize(q, s32, 32)
    assert not d[1:].any() and not d[0, :32].any() and not d[0, 64:].any()


def test_shared_gate_weight_hand_worked():
    # sigmoid(ln 3) = 3 / (3 + 1) = 0.75; sigmoid(0) = 0.5; no gate -> 1
    x = np.array([[math.log(3.0), 5.0], [0.0, 0.0]])
    g = np.array([1.0, 0.0])
    assert np.allclose(O.shared_gate_weight(x, g), [0.75, 0.5], rtol=0, atol=1e-15)
    assert O.shared_gate_weight(x, None).tolist() == [1.0, 1.0]


def _gated_layer(zero_points):
    shape = synth.LayerShape(64, 32, 6, 2, 32, True, has_shared=True, zero_points=zero_points, shared_gate=True)
    return shape, synth.make_layer(shape, seed=12, codes="uniform")


@pytest.mark.parametrize("zero_points", [False, True])
def test_shared_gate_special_cases(zero_points):
    shape, lay = _gated_layer(zero_points)
    x = synth.make_tokens(shape.hidden, 5, seed=12)
    kw = dict(H=shape.hidden, I=shape.intermediate, E=shape.num_experts, k=shape.top_k, G=shape.group_size,
              renormalize=shape.renormalize, zero_points=zero_points)
    args = (x, lay.router_w, None, lay.records, lay.expert_to_slot)
    routed = O.moe_forward(*args, has_shared=False, **kw)["out"]
    full = O.moe_forward(*args, has_shared=True, **kw)["out"]
    # a zero gate vector: every token takes half the shared expert
    half = O.moe_forward(*args, has_shared=True, shared_gate=np.zeros(shape.hidden), **kw)["out"]
    assert np.allclose(half, routed + 0.5 * (full - routed), rtol=1e-12, atol=1e-15)
    # a gate that saturates: weight 1 (to the last bits of float64)
    big = np.full(shape.hidden, 1e3) * np.sign(x.astype(np.float64).sum(axis=0) + 1e-9)
    sat = O.moe_forward(*args, has_shared=True, shared_gate=big, **kw)["out"]
    gw = O.shared_gate_weight(x, big)
    ok = gw > 1 - 1e-12
    assert ok.any() and np.allclose(sat[ok], full[ok], rtol=1e-10, atol=1e-14)
    # brute force (every expert on every token, a dense mask) agrees
    dense, _ = O.dense_masked_forward(*args, has_shared=True, shared_gate=lay.shared_gate, **kw)
    ref = O.moe_forward(*args, has_shared=True, shared_gate=lay.shared_gate, **kw)["out"]
    assert np.allclose(dense, ref, rtol=1e-12, atol=1e-14)


def test_asymmetric_quantiser_round_trips_within_half_a_step():
    # the generator's asymmetric quantiser: every weight within half a scale
    # step of (q - z) * s (clipping aside), using the oracle's dequantisation
    rng = np.random.default_rng(5)
    w = rng.standard_normal((6, 96)).astype(np.float32) * np.float32(0.02)
    q, s, z = synth.quantize_int4_asym(w, 32)
    wd = O.dequantize(q, s, 32, zeros=z)
    step = np.repeat(s.astype(np.float64), 32, axis=1)
    assert (np.abs(wd - w) <= 0.5 * step + 1e-6).all()


@pytest.mark.parametrize("mistake", ["zero_point_ignored", "zero_point_sign", "gate_ignored", "gate_sign"])
def test_planted_variant_mistakes_are_caught(golden_dir, mistake, monkeypatch):
    """A plausible mistake planted in the variants' oracle code fails a pin."""
    orig_dq, orig_gate = O.dequantize, O.shared_gate_weight
    if mistake == "zero_point_ignored":
        monkeypatch.setattr(O, "dequantize", lambda q, s, G, zeros=None: orig_dq(q, s, G))
    elif mistake == "zero_point_sign":
        monkeypatch.setattr(O, "dequantize", lambda q, s, G, zeros=None: orig_dq(
            q, s, G, None if zeros is None else (16 - np.asarray(zeros, dtype=np.int64)) % 16))
    elif mistake == "gate_ignored":
        monkeypatch.setattr(O, "shared_gate_weight", lambda x, g: orig_gate(x, None))
    elif mistake == "gate_sign":
        monkeypatch.setattr(O, "shared_gate_weight", lambda x, g: orig_gate(x, None if g is None else -np.asarray(g)))
    with pytest.raises(AssertionError):
        if mistake.startswith("zero_point"):
            test_zero_point_record_hand_built(golden_dir)
        else:
            test_shared_gate_weight_hand_worked()
