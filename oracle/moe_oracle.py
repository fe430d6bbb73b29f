"""CPU oracle of the W4A16 routed-expert MoE layer — TEST INFRASTRUCTURE.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this module. The product path (the CUDA library and its binding) never
calls it and shares no code with it; this file imports nothing from the
package.

Plain, slow, obviously-correct NumPy in float64, one function per step of the
layer, each step written in the order the layer defines it:

1. router logits ``L = x W_r^T (+ b)``                       -> router_logits
2. softmax over all E experts                                -> softmax_rows
3. top-k, ties to the lowest expert id, rank order; NaN logits rank as -inf
                                                              -> select_topk
4. routing weights (softmax value, optionally renormalised)   -> routing_weights
5. counting-sort permutation by expert                        -> counting_sort
6. expert FFN ``y = W_d (silu(W_g x) * (W_u x))`` on dequantised INT4 weights
                                                              -> expert_ffn
7. weighted combine ``out = sum_j w_j y_j (+ g y_shared)``   -> moe_forward

Variants (readings of this library; the pages print none of them): an
asymmetric zero point per group, ``w = (q - z) * s`` with z a code 0..15
stored one per byte in three more record sections (gate_z, up_z, down_z);
any group size G (32, 64, 128); a shared expert gated per token by
``g = sigmoid(x . w_gate)`` (weight 1 without a gate vector).

Sources (page title, section):
* Horizon RunMap report, "Architecture invariants" / "What is implemented" /
  "The complete execution path" step 2: routed experts stored as INT4 qpacked
  data with FP16 scales, executed with FP16 activations; routing selects the
  experts each token needs.
* moe-stream, "Terms used here" and "Method": a router picks 8 of 64 experts
  per token at each layer (the OLMoE shape).
* F51 Nitro-MoE, "The thesis": 10 routed experts plus one shared expert.
The pages give no formulas for the layer; where they are silent this oracle
takes the plain readings that the layer's specification states: zero point 8,
one FP16 scale per G codes along K, SwiGLU ``silu(g) * u``, softmax over all
experts, ties to the lowest id, shared expert with weight 1.

Record layout (its own reading of the canonical format): sections gate_q,
up_q, down_q, gate_s, up_s, down_s, each starting on a 256-byte boundary;
codes row-major with K contiguous, low nibble = even k.
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------
# expert record
# ----------------------------------------------------------------------------

def _align256(v: int) -> int:
    return -(-v // 256) * 256


def record_layout(H: int, I: int, G: int, zero_points: bool = False):
    """Section offsets of one expert record and the padded record size; with
    zero points, three byte-per-group sections follow the scales."""
    groups_h = -(-H // G)
    groups_i = -(-I // G)
    order = (("gate_q", I * (H // 2)), ("up_q", I * (H // 2)), ("down_q", H * (I // 2)),
             ("gate_s", 2 * I * groups_h), ("up_s", 2 * I * groups_h), ("down_s", 2 * H * groups_i))
    if zero_points:
        order = order + (("gate_z", I * groups_h), ("up_z", I * groups_h), ("down_z", H * groups_i))
    offs = {}
    cur = 0
    for name, nbytes in order:
        cur = _align256(cur)
        offs[name] = (cur, nbytes)
        cur += nbytes
    return offs, _align256(cur)


def unpack_codes(raw: np.ndarray, N: int, K: int) -> np.ndarray:
    """Bytes of an [N][K] code matrix -> integer codes 0..15.

    Byte b of a row holds code k = 2b in its low four bits and k = 2b + 1 in
    its high four bits."""
    raw = np.asarray(raw, dtype=np.uint8).reshape(N, K // 2)
    q = np.empty((N, K), dtype=np.uint8)
    q[:, 0::2] = raw % 16
    q[:, 1::2] = raw // 16
    return q


def dequantize(q: np.ndarray, scales: np.ndarray, G: int, zeros=None) -> np.ndarray:
    """w[n, k] = (q[n, k] - z[n, k // G]) * s[n, k // G] in float64, z = 8
    when no zero points are given."""
    N, K = q.shape
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    w = np.asarray(q).astype(np.float64)
    for gi in range(s.shape[1]):
        z = 8.0 if zeros is None else np.asarray(zeros)[:, gi:gi + 1].astype(np.float64)
        w[:, gi * G:(gi + 1) * G] = (w[:, gi * G:(gi + 1) * G] - z) * s[:, gi:gi + 1]
    return w


def expert_matrices(record: np.ndarray, H: int, I: int, G: int, zero_points: bool = False):
    """Dequantised (W_gate [I][H], W_up [I][H], W_down [H][I]) of one record."""
    offs, _ = record_layout(H, I, G, zero_points)
    rec = np.asarray(record, dtype=np.uint8).reshape(-1)

    def sect(name):
        o, n = offs[name]
        return rec[o:o + n]

    def zeros(name, n, ng):
        return sect(name).reshape(n, ng) if zero_points else None

    gh, gi = -(-H // G), -(-I // G)
    wg = dequantize(unpack_codes(sect("gate_q"), I, H), sect("gate_s").view(np.float16).reshape(I, gh), G,
                    zeros("gate_z", I, gh))
    wu = dequantize(unpack_codes(sect("up_q"), I, H), sect("up_s").view(np.float16).reshape(I, gh), G,
                    zeros("up_z", I, gh))
    wd = dequantize(unpack_codes(sect("down_q"), H, I), sect("down_s").view(np.float16).reshape(H, gi), G,
                    zeros("down_z", H, gi))
    return wg, wu, wd


# ----------------------------------------------------------------------------
# routing
# ----------------------------------------------------------------------------

def router_logits(x: np.ndarray, router_w: np.ndarray, router_bias=None) -> np.ndarray:
    """L[t, e] = sum_h x[t, h] * W_r[e, h]  (+ b[e]) in float64."""
    L = np.asarray(x, dtype=np.float64) @ np.asarray(router_w, dtype=np.float64).T
    if router_bias is not None:
        L = L + np.asarray(router_bias, dtype=np.float64)[None, :]
    return L


def softmax_rows(L: np.ndarray) -> np.ndarray:
    """Softmax over all experts of each row, with the row max subtracted."""
    m = L.max(axis=1, keepdims=True)
    z = np.exp(L - m)
    return z / z.sum(axis=1, keepdims=True)


def selection_key(L: np.ndarray) -> np.ndarray:
    """Key a logit is ranked by: the logit itself, with NaN ranked below
    every number (as -inf). The pages say nothing about non-finite values;
    this reading keeps the order (key descending, id ascending) total for
    any input."""
    L = np.asarray(L, dtype=np.float64)
    return np.where(np.isnan(L), -np.inf, L)


def select_topk(L: np.ndarray, k: int) -> np.ndarray:
    """k rounds of selection: each round takes the largest remaining key
    (selection_key), the lowest expert id among equal keys. Result in rank
    order."""
    K = selection_key(L)
    T, E = K.shape
    ids = np.empty((T, k), dtype=np.int64)
    for t in range(T):
        taken = np.zeros(E, dtype=bool)
        for j in range(k):
            best = -1
            for e in range(E):
                if taken[e]:
                    continue
                if best < 0 or K[t, e] > K[t, best]:
                    best = e
            ids[t, j] = best
            taken[best] = True
    return ids


def select_topk_fast(L: np.ndarray, k: int) -> np.ndarray:
    """Same selection as select_topk, vectorised over tokens: a stable sort
    of the negated keys keeps equal keys in ascending id order (every key is
    a number or -inf, so the negation is exact)."""
    order = np.argsort(-selection_key(L), axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def routing_weights(p: np.ndarray, ids: np.ndarray, renormalize: bool) -> np.ndarray:
    """w[t, j] = p[t, ids[t, j]], divided by the sum over the selected experts
    when renormalising."""
    w = np.take_along_axis(p, ids, axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return w


def counting_sort(ids: np.ndarray, E: int):
    """Counting sort of the flat (token, rank) pairs f = t*k + j by expert.

    counts[e]   = number of pairs routed to e
    offsets     = exclusive prefix sum of counts, offsets[E] = T*k
    perm[p]     = flat index at sorted position p (ascending f within an expert)
    inv_perm[f] = sorted position of flat index f
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    n = flat.size
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:E].copy()
    perm = np.empty(n, dtype=np.int64)
    inv_perm = np.empty(n, dtype=np.int64)
    for f in range(n):
        e = flat[f]
        perm[cursor[e]] = f
        inv_perm[f] = cursor[e]
        cursor[e] += 1
    return counts, offsets, perm, inv_perm


# ----------------------------------------------------------------------------
# expert FFN and combine
# ----------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def shared_gate_weight(x: np.ndarray, gate_w) -> np.ndarray:
    """Per-token weight of the shared expert: sigmoid(x . w_gate) in float64,
    1 for every token without a gate vector."""
    x64 = np.asarray(x, dtype=np.float64)
    if gate_w is None:
        return np.ones(x64.shape[0])
    z = x64 @ np.asarray(gate_w, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def expert_ffn(wg: np.ndarray, wu: np.ndarray, wd: np.ndarray, xrows: np.ndarray) -> np.ndarray:
    """SwiGLU expert: y = W_d (silu(W_g x) * (W_u x)) for each row of xrows."""
    x64 = np.asarray(xrows, dtype=np.float64)
    g = x64 @ wg.T
    u = x64 @ wu.T
    h = silu(g) * u
    return h @ wd.T


def moe_forward(x, router_w, router_bias, records, expert_to_slot, *, H, I, E, k, G,
                renormalize, has_shared=False, tokens=None, zero_points=False, shared_gate=None):
    """Whole layer for the tokens in ``tokens`` (default: all).

    Routing (logits, softmax, selection, weights, permutation) is computed for
    every token of the batch; expert outputs and the combine only for the
    requested tokens. Returns a dict of float64 / int64 arrays."""
    x = np.asarray(x)
    T = x.shape[0]
    L = router_logits(x, router_w, router_bias)
    p = softmax_rows(L)
    ids = select_topk_fast(L, k)
    w = routing_weights(p, ids, renormalize)
    counts, offsets, perm, inv_perm = counting_sort(ids, E)
    if tokens is None:
        tokens = np.arange(T)
    out = expert_combine(x, ids, w, records, expert_to_slot, H=H, I=I, E=E, k=k, G=G,
                         has_shared=has_shared, tokens=tokens, zero_points=zero_points,
                         shared_gate=shared_gate)
    return dict(out=out, logits=L, probs=p, ids=ids, weights=w, counts=counts,
                offsets=offsets, perm=perm, inv_perm=inv_perm)


def expert_combine(x, ids, w, records, expert_to_slot, *, H, I, E, k, G, has_shared=False, tokens=None,
                   zero_points=False, shared_gate=None):
    """out[t] = sum_j w[t, j] * y_{ids[t, j]}(x[t]) (+ g_t y_shared(x[t])) for
    the requested tokens, given the routing (ids, w) of the whole batch; g_t
    from shared_gate_weight."""
    x = np.asarray(x)
    ids = np.asarray(ids)
    w = np.asarray(w, dtype=np.float64)
    if tokens is None:
        tokens = np.arange(x.shape[0])
    tokens = np.asarray(tokens, dtype=np.int64)
    out = np.zeros((tokens.size, H), dtype=np.float64)
    used = sorted(set(int(e) for e in ids[tokens].reshape(-1)))
    for e in used:
        wg, wu, wd = expert_matrices(records[int(expert_to_slot[e])], H, I, G, zero_points)
        for j in range(k):
            rows = np.nonzero(ids[tokens, j] == e)[0]
            if rows.size == 0:
                continue
            y = expert_ffn(wg, wu, wd, x[tokens[rows]])
            out[rows] += w[tokens[rows], j][:, None] * y
    if has_shared:
        wg, wu, wd = expert_matrices(records[int(expert_to_slot[E])], H, I, G, zero_points)
        out += shared_gate_weight(x[tokens], shared_gate)[:, None] * expert_ffn(wg, wu, wd, x[tokens])
    return out


def dense_masked_forward(x, router_w, router_bias, records, expert_to_slot, *, H, I, E, k, G,
                         renormalize, has_shared=False, zero_points=False, shared_gate=None):
    """Brute force: every expert runs on every token; a [T][E] mask-weight
    matrix (zero for experts a token did not select) combines them."""
    x = np.asarray(x)
    T = x.shape[0]
    L = router_logits(x, router_w, router_bias)
    p = softmax_rows(L)
    # full descending order of each row, lower id first among equals
    order = np.lexsort((np.broadcast_to(np.arange(E), (T, E)), -L), axis=1)
    sel = order[:, :k]
    M = np.zeros((T, E), dtype=np.float64)
    for t in range(T):
        ps = p[t, sel[t]]
        if renormalize:
            ps = ps / ps.sum()
        M[t, sel[t]] = ps
    Y = np.zeros((E, T, H), dtype=np.float64)
    for e in range(E):
        wg, wu, wd = expert_matrices(records[int(expert_to_slot[e])], H, I, G, zero_points)
        Y[e] = expert_ffn(wg, wu, wd, x)
    out = np.einsum("te,eth->th", M, Y)
    if has_shared:
        wg, wu, wd = expert_matrices(records[int(expert_to_slot[E])], H, I, G, zero_points)
        ys = expert_ffn(wg, wu, wd, x)
        for t in range(T):
            gate = 1.0
            if shared_gate is not None:
                gate = 1.0 / (1.0 + np.exp(-float(np.dot(x[t].astype(np.float64),
                                                         np.asarray(shared_gate, dtype=np.float64)))))
            out[t] = out[t] + gate * ys[t]
    return out, sel


def residual_add(x_fp16: np.ndarray, out_fp16: np.ndarray) -> np.ndarray:
    """Residual stream update between stacked layers: fp16(x + moe(x)), with
    the layer output taken at its FP16 value."""
    return (np.asarray(x_fp16, dtype=np.float64) + np.asarray(out_fp16, dtype=np.float64)).astype(np.float16)


def near_tie_tokens(L: np.ndarray, k: int, eps: float = 1e-3) -> np.ndarray:
    """Tokens whose routing is not decided beyond eps: the gap between the
    k-th and (k+1)-th largest logits, or between two adjacent selected
    logits, is at most eps."""
    s = -np.sort(-np.asarray(L, dtype=np.float64), axis=1)
    E = s.shape[1]
    upto = min(k + 1, E)
    gaps = s[:, :upto - 1] - s[:, 1:upto]
    return np.nonzero((gaps <= eps).any(axis=1))[0]
