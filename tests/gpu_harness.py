"""Shared helpers of the GPU parity tests: upload a synthetic layer, run it
through the C ABI, and compare with the CPU oracle.

Acceptance: expert ids bit-exact for tokens whose k-th and (k+1)-th logits
(and adjacent selected logits) differ by more than 1e-3; counts / offsets /
perm / inv_perm bit-exact against the counting sort of the GPU's ids (and
against the oracle's when no token is a near tie); routing weights within
FP32 rounding; outputs within |gpu - oracle| <= 2e-3 * max(1, |oracle|).
Near-tie tokens are checked against the oracle recomputed with the GPU's ids.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O
from w4a16_routed_expert_gb300 import synth
from w4a16_routed_expert_gb300.layer import MoELayer

TOL = 2e-3
TIE_EPS = 1e-3
_STREAM = None
# one entry per compare() call of the session: test id, tokens compared,
# near-tie tokens (reported separately; the routing check skips them), worst
# error over its bound. Printed at the end of the run (tests/conftest.py).
REPORTS = []


def stream():
    """A created (non-default) stream, so launches use programmatic
    dependent launch as in production."""
    global _STREAM
    if _STREAM is None:
        _STREAM = torch.cuda.Stream()
    return _STREAM


def oracle_kw(shape):
    return dict(H=shape.hidden, I=shape.intermediate, E=shape.num_experts, k=shape.top_k,
                G=shape.group_size, renormalize=shape.renormalize, has_shared=shape.has_shared,
                zero_points=shape.zero_points)


def upload(lay: synth.Layer, max_tokens: int, add_residual: bool = False) -> MoELayer:
    s = lay.shape
    dev = torch.device("cuda")
    pool = torch.from_numpy(lay.records).to(dev)
    e2s = torch.from_numpy(lay.expert_to_slot.astype(np.int32)).to(dev)
    rw = torch.from_numpy(lay.router_w).to(dev)
    rb = torch.from_numpy(lay.router_bias).to(dev) if lay.router_bias is not None else None
    gate = torch.from_numpy(lay.shared_gate).to(dev) if lay.shared_gate is not None else None
    return MoELayer(hidden=s.hidden, intermediate=s.intermediate, num_experts=s.num_experts, top_k=s.top_k,
                    group_size=s.group_size, renormalize=s.renormalize, has_shared=s.has_shared,
                    max_tokens=max_tokens, router_w=rw, router_bias=rb, pool=pool, expert_to_slot=e2s,
                    num_slots=pool.shape[0], add_residual=add_residual, zero_points=s.zero_points,
                    shared_gate=gate)


def run(ml: MoELayer, x_np: np.ndarray):
    dev = torch.device("cuda")
    x = torch.from_numpy(x_np).to(dev)
    T = x.shape[0]
    k = ml.top_k
    ids = torch.full((T, k), -1, dtype=torch.int32, device=dev)
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
    out = torch.full_like(x, float("nan"))
    s = stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ml.forward(x, out=out, ids=ids, w=w)
        counts, offsets, perm, inv = ml.routing(T)
        ml.sync()
    return dict(out=out.float().cpu().numpy().astype(np.float64), ids=ids.cpu().numpy().astype(np.int64),
                w=w.cpu().numpy().astype(np.float64), counts=counts.cpu().numpy(), offsets=offsets.cpu().numpy(),
                perm=perm.cpu().numpy(), inv_perm=inv.cpu().numpy())


def compare(lay: synth.Layer, x_np: np.ndarray, g: dict, tokens=None, tol: float = TOL):
    """Assert the acceptance criteria; returns a small report dict."""
    s = lay.shape
    kw = oracle_kw(s)
    T = x_np.shape[0]
    ref = O.moe_forward(x_np, lay.router_w, lay.router_bias, lay.records, lay.expert_to_slot,
                        tokens=tokens, shared_gate=lay.shared_gate, **kw)
    near = set(O.near_tie_tokens(ref["logits"], s.top_k, TIE_EPS).tolist())
    decided = np.array([t for t in range(T) if t not in near], dtype=np.int64)
    # routing: ids bit-exact where decided
    assert np.array_equal(g["ids"][decided], ref["ids"][decided]), "expert ids differ on decided tokens"
    # permutation bit-exact against the counting sort of the GPU's own ids
    c, o, p, ip = O.counting_sort(g["ids"], s.num_experts)
    assert np.array_equal(g["counts"], c) and np.array_equal(g["offsets"], o)
    assert np.array_equal(g["perm"], p) and np.array_equal(g["inv_perm"], ip)
    if not near:
        assert np.array_equal(g["counts"], ref["counts"]) and np.array_equal(g["perm"], ref["perm"])
        assert np.array_equal(g["offsets"], ref["offsets"]) and np.array_equal(g["inv_perm"], ref["inv_perm"])
    # routing weights: FP32 softmax vs FP64
    w_ref = O.routing_weights(ref["probs"], g["ids"], s.renormalize)
    np.testing.assert_allclose(g["w"], w_ref, rtol=2e-5, atol=1e-7)
    # outputs
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    out_ref = ref["out"].copy()
    nt_rows = [i for i, t in enumerate(toks) if int(t) in near]
    if nt_rows:
        sub = toks[nt_rows]
        out_ref[nt_rows] = O.expert_combine(x_np, g["ids"], w_ref, lay.records, lay.expert_to_slot,
                                            H=s.hidden, I=s.intermediate, E=s.num_experts, k=s.top_k,
                                            G=s.group_size, has_shared=s.has_shared, tokens=sub,
                                            zero_points=s.zero_points, shared_gate=lay.shared_gate)
    got = g["out"][toks]
    err = np.abs(got - out_ref)
    bound = tol * np.maximum(1.0, np.abs(out_ref))
    worst = float((err / bound).max()) if err.size else 0.0
    assert np.isfinite(got).all(), "non-finite outputs"
    assert (err <= bound).all(), f"max err/bound {worst:.3f}, max abs err {err.max():.3e}"
    rep = dict(tokens=int(T), rows_compared=int(len(toks)), near_ties=len(near), worst_ratio=worst,
               max_abs_err=float(err.max()) if err.size else 0.0)
    import os
    REPORTS.append(dict(test=os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], **rep))
    return rep
