"""Seeded synthetic inputs for the W4A16 routed-expert MoE layer.

This module is the one piece shared by the CPU oracle's tests and the CUDA
path: it draws activations, router weights and expert weights, quantises the
expert weights to unsigned INT4 codes with FP16 group scales (an offline
preparation step, not part of the layer's forward computation) and packs them
into the canonical qpacked expert record. It performs none of the layer's own
arithmetic (no router logits, softmax, selection, permutation, expert FFN or
combine).

Canonical expert record (one contiguous record per expert, so that one copy
moves everything an expert needs — the "one read brings everything it needs"
file layout of the moe-stream page, section "Method"):

    gate_q | up_q | down_q | gate_s | up_s | down_s

* ``gate_q``/``up_q``: INT4 codes of the [I][H] gate and up projections,
  ``down_q``: codes of the [H][I] down projection. Row-major, K (the
  reduction axis) contiguous, two codes per byte: the low nibble holds the even
  k, the high nibble the odd k. Row stride K/2 bytes.
* ``*_s``: FP16 scales, [N][ceil(K/G)] row-major, one per G consecutive codes
  along K; the last group of a row covers the remaining K mod G codes.
* The dequantised weight is ``(q - 8) * s`` (unsigned 4-bit, zero point 8),
  or, for a layer with zero points, ``(q - z) * s`` with one code z per
  group stored as one byte in three more sections after the scales:
  ``gate_z | up_z | down_z``, each [N][ceil(K/G)].
* Each section starts on a 256-byte boundary; the record size is rounded up to
  a multiple of 256 bytes.

Horizon RunMap report, "Architecture invariants" and "What is implemented":
routed experts are kept compact as INT4 qpacked data with FP16 scales and run
with FP16 activations; the pages do not print a byte layout, so the layout
above is this library's own definition.
"""
from __future__ import annotations

import dataclasses
import os
from typing import Optional

import numpy as np

SECTION_ALIGN = 256


def _round_up(v: int, a: int) -> int:
    return (v + a - 1) // a * a


@dataclasses.dataclass(frozen=True)
class LayerShape:
    hidden: int
    intermediate: int
    num_experts: int
    top_k: int
    group_size: int
    renormalize: bool
    has_shared: bool = False
    router_std: float = 0.02
    expert_std: float = 0.02
    zipf_s: float = 0.0  # >0: add -zipf_s*ln(e+1) to expert e's logit
    zero_points: bool = False  # asymmetric quantisation, a zero code per group
    shared_gate: bool = False  # the shared expert gated per token by sigmoid(x . w_gate)

    @property
    def n_records(self) -> int:
        return self.num_experts + (1 if self.has_shared else 0)


# Workloads named by what they are (shapes from the pages plus the stated
# synthetic recipe).
TINY = LayerShape(256, 128, 8, 2, 64, True, router_std=0.05)
OLMOE = LayerShape(2048, 1024, 64, 8, 128, False)
MANY_EXPERTS = LayerShape(2048, 512, 512, 10, 128, True, has_shared=True, zipf_s=1.1)
GPTOSS_LIKE = LayerShape(2880, 2880, 128, 4, 128, True)


def section_layout(H: int, I: int, G: int, zero_points: bool = False) -> dict:
    """Byte offset and size of each section of the canonical record."""
    ng_h = -(-H // G)
    ng_i = -(-I // G)
    sizes = [
        ("gate_q", I * H // 2),
        ("up_q", I * H // 2),
        ("down_q", H * I // 2),
        ("gate_s", I * ng_h * 2),
        ("up_s", I * ng_h * 2),
        ("down_s", H * ng_i * 2),
    ]
    if zero_points:
        sizes += [("gate_z", I * ng_h), ("up_z", I * ng_h), ("down_z", H * ng_i)]
    out = {}
    off = 0
    for name, size in sizes:
        off = _round_up(off, SECTION_ALIGN)
        out[name] = (off, size)
        off += size
    out["record_bytes"] = _round_up(off, SECTION_ALIGN)
    out["payload_bytes"] = sum(s for _, s in sizes)
    return out


def record_bytes(H: int, I: int, G: int, zero_points: bool = False) -> int:
    return section_layout(H, I, G, zero_points)["record_bytes"]


def quantize_int4(w: np.ndarray, G: int):
    """Symmetric-range INT4 quantisation with zero point 8 (data preparation).

    scale = fp16(max|w| / 7) per group of G along K (1.0 for an all-zero
    group); code = clip(rint(w / scale) + 8, 0, 15).
    """
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    ng = -(-K // G)
    pad = ng * G - K
    wp = np.pad(w, ((0, 0), (0, pad))) if pad else w
    wg = wp.reshape(N, ng, G)
    amax = np.abs(wg).max(axis=2)
    s16 = (amax / np.float32(7.0)).astype(np.float16)
    s16[amax == 0] = np.float16(1.0)
    s32 = s16.astype(np.float32)
    q = np.rint(wg / s32[:, :, None]) + 8.0
    q = np.clip(q, 0, 15).astype(np.uint8).reshape(N, ng * G)[:, :K]
    return np.ascontiguousarray(q), s16


def quantize_int4_asym(w: np.ndarray, G: int):
    """Asymmetric INT4 quantisation (data preparation): per group of G along
    K, scale = fp16((max - min) / 15) (1.0 for a constant group), zero code
    z = clip(rint(-min / scale), 0, 15), code = clip(rint(w / scale) + z, 0, 15)."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    ng = -(-K // G)
    pad = ng * G - K
    # padding repeats each row's last value, so it leaves min / max alone
    wp = np.pad(w, ((0, 0), (0, pad)), mode="edge") if pad else w
    wg = wp.reshape(N, ng, G)
    lo, hi = wg.min(axis=2), wg.max(axis=2)
    s16 = ((hi - lo) / np.float32(15.0)).astype(np.float16)
    s16[s16 == 0] = np.float16(1.0)
    s32 = s16.astype(np.float32)
    z = np.clip(np.rint(-lo / s32), 0, 15).astype(np.uint8)
    q = np.clip(np.rint(wg / s32[:, :, None]) + z[:, :, None], 0, 15).astype(np.uint8).reshape(N, ng * G)[:, :K]
    return np.ascontiguousarray(q), s16, np.ascontiguousarray(z)


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """[N][K] codes in 0..15 -> [N][K/2] bytes, low nibble = even k."""
    q = np.asarray(q, dtype=np.uint8)
    assert q.shape[1] % 2 == 0
    return np.ascontiguousarray((q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)).astype(np.uint8)


def pack_record(H, I, G, gate_q, up_q, down_q, gate_s, up_s, down_s, gate_z=None, up_z=None,
                down_z=None) -> np.ndarray:
    zp = gate_z is not None
    lay = section_layout(H, I, G, zp)
    rec = np.zeros(lay["record_bytes"], dtype=np.uint8)
    parts = {
        "gate_q": pack_nibbles(gate_q),
        "up_q": pack_nibbles(up_q),
        "down_q": pack_nibbles(down_q),
        "gate_s": np.ascontiguousarray(gate_s, dtype=np.float16).view(np.uint8),
        "up_s": np.ascontiguousarray(up_s, dtype=np.float16).view(np.uint8),
        "down_s": np.ascontiguousarray(down_s, dtype=np.float16).view(np.uint8),
    }
    if zp:
        parts.update(gate_z=np.ascontiguousarray(gate_z, dtype=np.uint8),
                     up_z=np.ascontiguousarray(up_z, dtype=np.uint8),
                     down_z=np.ascontiguousarray(down_z, dtype=np.uint8))
    for name, arr in parts.items():
        off, size = lay[name]
        flat = arr.reshape(-1)
        assert flat.size == size, (name, flat.size, size)
        rec[off:off + size] = flat
    return rec


def _expert_codes(shape: LayerShape, rng: np.random.Generator, codes: str):
    H, I, G = shape.hidden, shape.intermediate, shape.group_size
    mats = []
    for (n, k) in ((I, H), (I, H), (H, I)):
        if codes == "quantized":
            w = rng.standard_normal((n, k), dtype=np.float32) * np.float32(shape.expert_std)
            mats.append(quantize_int4_asym(w, G) if shape.zero_points else quantize_int4(w, G))
        elif codes == "uniform":
            # every code 0..15 equally likely; scales spread over a range so
            # that no single scale dominates (exercises q = 0 and q = 15).
            q = rng.integers(0, 16, size=(n, k), dtype=np.uint8)
            ng = -(-k // G)
            s = (rng.uniform(0.5, 1.5, size=(n, ng)) * (shape.expert_std / 4.6)).astype(np.float16)
            if shape.zero_points:
                mats.append((q, s, rng.integers(0, 16, size=(n, ng), dtype=np.uint8)))
            else:
                mats.append((q, s))
        else:
            raise ValueError(codes)
    if shape.zero_points:
        (gq, gs, gz), (uq, us, uz), (dq, ds, dz) = mats
        return gq, uq, dq, gs, us, ds, gz, uz, dz
    (gq, gs), (uq, us), (dq, ds) = mats
    return gq, uq, dq, gs, us, ds


@dataclasses.dataclass
class Layer:
    shape: LayerShape
    router_w: np.ndarray            # fp32 [E][H]
    router_bias: Optional[np.ndarray]  # fp32 [E] or None
    records: np.ndarray             # uint8 [n_slots][record_bytes], in slot order
    expert_to_slot: np.ndarray      # int32 [n_records]
    shared_gate: Optional[np.ndarray] = None  # fp32 [H] gate vector of the shared expert, or None


def _expert_record(args):
    shape, child, codes = args
    rng = np.random.default_rng(child)
    return pack_record(shape.hidden, shape.intermediate, shape.group_size, *_expert_codes(shape, rng, codes))


def make_layer(shape: LayerShape, seed: int, codes: str = "quantized",
               shuffle_slots: bool = True, extra_slots: int = 0, workers: Optional[int] = None) -> Layer:
    """Draw one layer. Expert e's draws come from its own child seed, so any
    expert can be regenerated alone (and records can be drawn in parallel
    worker processes with identical results). Records are stored in slot
    order through a random expert_to_slot permutation (identity if
    shuffle_slots is False); ``extra_slots`` appends unused slots filled with
    0xFF bytes."""
    E = shape.num_experts
    nrec = shape.n_records
    children = np.random.SeedSequence(seed).spawn(3 + nrec)
    rng_router = np.random.default_rng(children[1])
    router_w = rng_router.standard_normal((E, shape.hidden), dtype=np.float32) * np.float32(shape.router_std)
    bias = None
    if shape.zipf_s > 0:
        bias = (-shape.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))).astype(np.float32)
    n_slots = nrec + extra_slots
    if shuffle_slots:
        slot_of = np.random.default_rng(children[2]).permutation(n_slots)[:nrec].astype(np.int32)
    else:
        slot_of = np.arange(nrec, dtype=np.int32)
    rb = record_bytes(shape.hidden, shape.intermediate, shape.group_size, shape.zero_points)
    records = np.full((n_slots, rb), 0xFF, dtype=np.uint8)
    jobs = [(shape, children[3 + e], codes) for e in range(nrec)]
    weights_per_layer = nrec * 3 * shape.hidden * shape.intermediate
    if workers is None:
        workers = min(os.cpu_count() or 1, 16) if weights_per_layer > 64 * 2**20 else 1
    if workers > 1:
        import concurrent.futures
        import multiprocessing
        ctx = multiprocessing.get_context("spawn")
        with concurrent.futures.ProcessPoolExecutor(max_workers=workers, mp_context=ctx) as ex:
            for e, rec in enumerate(ex.map(_expert_record, jobs, chunksize=max(1, nrec // (4 * workers)))):
                records[slot_of[e]] = rec
    else:
        for e, job in enumerate(jobs):
            records[slot_of[e]] = _expert_record(job)
    gate = None
    if shape.shared_gate and shape.has_shared:
        gate = (np.random.default_rng(np.random.SeedSequence(seed).spawn(4 + nrec)[3 + nrec])
                .standard_normal(shape.hidden, dtype=np.float32) * np.float32(shape.router_std))
    return Layer(shape, router_w, bias, records, slot_of, gate)


def make_tokens(H: int, T: int, seed: int, std: float = 1.0) -> np.ndarray:
    """FP16 activations ~ N(0, std), [T][H]."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x70C5]))
    return (rng.standard_normal((T, H), dtype=np.float32) * np.float32(std)).astype(np.float16)


def make_noise(H: int, T: int, seed: int, step: int, std: float = 0.1) -> np.ndarray:
    """Per-step residual-stream noise for the stacked-layer decode workload."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 1000 + step]))
    return (rng.standard_normal((T, H), dtype=np.float32) * np.float32(std))


def stack_layer_seed(seed: int, layer: int) -> int:
    """Seed of layer ``layer`` in the stacked workload (distinct per layer)."""
    return int(np.random.SeedSequence([seed, layer]).generate_state(1)[0])
