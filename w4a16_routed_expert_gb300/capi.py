"""ctypes binding of include/moe_layer.h — argument marshalling only.

Every entry point has the same name as in the header. The library is loaded
on first use; if it has not been built this raises instead of falling back
to anything else.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_w4a16.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_OOM = 2
MOE_ERR_CUDA = 3
MOE_ERR_UNSUPPORTED = 4
MOE_ERR_CAPACITY = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_INTERNAL = 7
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_OOM", 3: "MOE_ERR_CUDA",
                4: "MOE_ERR_UNSUPPORTED", 5: "MOE_ERR_CAPACITY", 6: "MOE_ERR_TIMEOUT",
                7: "MOE_ERR_INTERNAL"}

MOE_RESIDENCY_FULL = 0
MOE_RESIDENCY_PARTIAL = 1


class moe_layer_config_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "intermediate", "num_experts", "top_k", "group_size", "renormalize",
        "has_shared_expert", "max_tokens", "num_slots", "residency", "add_residual", "spare_slots",
        "staging_records", "cache_policy", "zero_points")]


class moe_layer_weights_t(ctypes.Structure):
    _fields_ = [("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("slot_pool", ctypes.c_void_p), ("expert_to_slot", ctypes.c_void_p),
                ("host_backing", ctypes.c_void_p), ("shared_gate", ctypes.c_void_p)]


class moe_layer_stats_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "forward_calls", "tokens", "expert_hits", "expert_misses", "h2d_bytes",
        "d2h_expert_bytes", "waves", "generations", "evictions", "staged_copies")] + [
        ("faulted", ctypes.c_int32), ("reserved", ctypes.c_int32)] + [
        (n, ctypes.c_uint64) for n in ("prefetch_calls", "prefetched", "prefetch_used")]


class moe_layer_profile_t(ctypes.Structure):
    _fields_ = [("route_ms", ctypes.c_float), ("gate_up_ms", ctypes.c_float), ("down_ms", ctypes.c_float),
                ("combine_ms", ctypes.c_float), ("total_ms", ctypes.c_float),
                ("active_experts", ctypes.c_int32), ("tokens", ctypes.c_int32), ("single_launch", ctypes.c_int32)]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {message}")


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32

# name -> (restype, argtypes)
PROTOTYPES = {
    "moe_abi_version": (_I32, []),
    "moe_record_bytes": (ctypes.c_size_t, [_I32, _I32, _I32]),
    "moe_record_bytes_zp": (ctypes.c_size_t, [_I32, _I32, _I32, _I32]),
    "moe_record_section": (_I32, [_I32, _I32, _I32, _I32, ctypes.POINTER(ctypes.c_size_t),
                                  ctypes.POINTER(ctypes.c_size_t)]),
    "moe_layer_create": (_I32, [ctypes.POINTER(moe_layer_config_t), ctypes.POINTER(moe_layer_weights_t),
                                ctypes.POINTER(_P)]),
    "moe_layer_forward": (_I32, [_P, _P, _I32, _P, _P, _P, _P]),
    "moe_layer_forward_host": (_I32, [_P, _P, _I32, _P, _P, _P, _P]),
    "moe_layer_prefetch": (_I32, [_P, _P, _I32, _P]),
    "moe_stack_create": (_I32, [ctypes.POINTER(_P), _I32, ctypes.POINTER(_P)]),
    "moe_stack_forward": (_I32, [_P, _P, _I32, _P, _P, _P]),
    "moe_stack_sync": (_I32, [_P, _P]),
    "moe_stack_single_launch": (_I32, [_P]),
    "moe_stack_destroy": (_I32, [_P]),
    "moe_layer_routing": (_I32, [_P, _P, _P, _P, _P, _P]),
    "moe_layer_sync": (_I32, [_P, _P]),
    "moe_layer_get_stats": (_I32, [_P, ctypes.POINTER(moe_layer_stats_t)]),
    "moe_layer_set_profiling": (_I32, [_P, _I32]),
    "moe_layer_get_trace": (_I32, [_P, ctypes.POINTER(ctypes.c_uint64), _I32, ctypes.POINTER(_I32)]),
    "moe_layer_get_gemm_stats": (_I32, [_P, ctypes.POINTER(ctypes.c_uint64), _I32, ctypes.POINTER(_I32)]),
    "moe_layer_get_profile": (_I32, [_P, ctypes.POINTER(moe_layer_profile_t)]),
    "moe_layer_destroy": (_I32, [_P]),
    "moe_layer_last_error": (ctypes.c_char_p, [ctypes.c_void_p]),
    "moe_route_topk_static": (_I32, [_P, _I32, _I32, _P, _P, _I32, _I32, _I32, _P, _P, _P]),
    # include/moe_residency.h
    "moe_slot_planner_create": (_P, [_I32, _I32]),
    "moe_slot_planner_plan": (_I32, [_P, ctypes.POINTER(_I32), _I32, _I32, ctypes.POINTER(_I32),
                                     ctypes.POINTER(_I32), ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "moe_slot_planner_slot_of": (_I32, [_P, _I32]),
    "moe_slot_planner_invalidate": (None, [_P, _I32]),
    "moe_slot_planner_destroy": (None, [_P]),
    "moe_expert_cache_create": (_P, [_I32, _I32, _I32, _I32]),
    "moe_expert_cache_access": (_I32, [_P, ctypes.POINTER(_I32), _I32, _I32, ctypes.POINTER(_I32),
                                       ctypes.POINTER(_I32), ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "moe_expert_cache_row_of": (_I32, [_P, _I32]),
    "moe_expert_cache_stats": (_I32, [_P, ctypes.POINTER(ctypes.c_uint64)]),
    "moe_expert_cache_prefetch": (_I32, [_P, ctypes.POINTER(_I32), _I32]),
    "moe_expert_cache_prefetch_stats": (_I32, [_P, ctypes.POINTER(ctypes.c_uint64)]),
    "moe_expert_cache_destroy": (None, [_P]),
}

MOE_PLAN_HITS_FIRST = 0
MOE_PLAN_FIXED_ORDER_LRU = 1
MOE_CACHE_LRU = 0
MOE_CACHE_LFU = 1
MOE_CACHE_LRU_FREQ = 2
# moe_cache_policy_t of moe_layer_config_t (same values)
MOE_POLICY_LRU, MOE_POLICY_LFU, MOE_POLICY_LRU_FREQ = 0, 1, 2


class ExpertCache:
    """Host-side model of the partially resident expert cache (no GPU)."""

    def __init__(self, n_records: int, capacity: int, spare_rows: int = 0, policy: int = MOE_CACHE_LRU):
        self.n_records = n_records
        self.h = lib().moe_expert_cache_create(n_records, capacity, spare_rows, policy)
        if not self.h:
            raise ValueError("invalid cache parameters")

    def access(self, demanded, abort_txn: int = -1):
        d = [int(e) for e in demanded]
        n = len(d)
        arr = (_I32 * max(n, 1))(*d)
        txn = (_I32 * max(n, 1))()
        row = (_I32 * max(n, 1))()
        hit = (_I32 * max(n, 1))()
        nt = _I32()
        rc = lib().moe_expert_cache_access(self.h, arr, n, abort_txn, txn, row, hit, ctypes.byref(nt))
        if rc < 0:
            raise ValueError("invalid access")
        return dict(experts=d, txn=list(txn)[:n], row=list(row)[:n], hit=list(hit)[:n], n_txn=nt.value,
                    aborted=rc == 1)

    def row_of(self, e: int) -> int:
        return lib().moe_expert_cache_row_of(self.h, e)

    def prefetch(self, guessed) -> int:
        g = [int(e) for e in guessed]
        arr = (_I32 * max(len(g), 1))(*g)
        rc = lib().moe_expert_cache_prefetch(self.h, arr, len(g))
        if rc < 0:
            raise ValueError("invalid prefetch")
        return rc

    def prefetch_stats(self):
        out = (ctypes.c_uint64 * 2)()
        lib().moe_expert_cache_prefetch_stats(self.h, out)
        return dict(prefetched=out[0], used=out[1])

    def stats(self):
        out = (ctypes.c_uint64 * 5)()
        lib().moe_expert_cache_stats(self.h, out)
        return dict(hits=out[0], misses=out[1], evictions=out[2], generations=out[3], decays=out[4])

    def close(self):
        if self.h:
            lib().moe_expert_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class SlotPlanner:
    """Host-side slot planner of the partially resident pool (no GPU)."""

    def __init__(self, n_records: int, num_slots: int):
        self.n_records = n_records
        self.h = lib().moe_slot_planner_create(n_records, num_slots)
        if not self.h:
            raise ValueError("invalid planner size")

    def plan(self, demanded, policy=MOE_PLAN_HITS_FIRST):
        d = sorted(int(e) for e in demanded)
        n = len(d)
        arr = (_I32 * max(n, 1))(*d)
        wave = (_I32 * max(n, 1))()
        slot = (_I32 * max(n, 1))()
        hit = (_I32 * max(n, 1))()
        nw = _I32()
        rc = lib().moe_slot_planner_plan(self.h, arr, n, policy, wave, slot, hit, ctypes.byref(nw))
        if rc != 0:
            raise ValueError("invalid plan request")
        return dict(experts=d, wave=list(wave)[:n], slot=list(slot)[:n], hit=list(hit)[:n], n_waves=nw.value)

    def slot_of(self, e: int) -> int:
        return lib().moe_slot_planner_slot_of(self.h, e)

    def invalidate(self, slot: int) -> None:
        lib().moe_slot_planner_invalidate(self.h, slot)

    def close(self):
        if self.h:
            lib().moe_slot_planner_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run w4a16_routed_expert_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def last_error() -> str:
    return lib().moe_layer_last_error(None).decode()


def check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoEError(status, where, last_error())


def record_bytes(hidden: int, intermediate: int, group_size: int) -> int:
    return int(lib().moe_record_bytes(hidden, intermediate, group_size))


def record_section(hidden: int, intermediate: int, group_size: int, section: int):
    off, size = ctypes.c_size_t(), ctypes.c_size_t()
    check(lib().moe_record_section(hidden, intermediate, group_size, section, ctypes.byref(off),
                                   ctypes.byref(size)), "moe_record_section")
    return off.value, size.value


def moe_layer_create(config: moe_layer_config_t, weights: moe_layer_weights_t) -> int:
    h = _P()
    check(lib().moe_layer_create(ctypes.byref(config), ctypes.byref(weights), ctypes.byref(h)),
          "moe_layer_create")
    return h.value


def moe_layer_forward(h, x, T, out, ids, w, stream) -> int:
    return lib().moe_layer_forward(h, x, T, out, ids, w, stream)


def moe_layer_forward_host(h, x, T, out, ids, w, stream) -> int:
    return lib().moe_layer_forward_host(h, x, T, out, ids, w, stream)


def moe_layer_prefetch(h, x, T, stream) -> int:
    return lib().moe_layer_prefetch(h, x, T, stream)


def moe_layer_routing(h, counts, offsets, perm, inv_perm, stream) -> int:
    return lib().moe_layer_routing(h, counts, offsets, perm, inv_perm, stream)


def moe_layer_sync(h, stream) -> int:
    return lib().moe_layer_sync(h, stream)


def moe_layer_get_stats(h) -> moe_layer_stats_t:
    st = moe_layer_stats_t()
    check(lib().moe_layer_get_stats(h, ctypes.byref(st)), "moe_layer_get_stats")
    return st


def moe_layer_set_profiling(h, enable: bool) -> None:
    check(lib().moe_layer_set_profiling(h, int(bool(enable))), "moe_layer_set_profiling")


def moe_layer_get_profile(h) -> moe_layer_profile_t:
    p = moe_layer_profile_t()
    check(lib().moe_layer_get_profile(h, ctypes.byref(p)), "moe_layer_get_profile")
    return p


TRACE_STAMPS = 32


def moe_layer_get_trace(h, max_stamps: int = 1024 * TRACE_STAMPS):
    buf = (ctypes.c_uint64 * max_stamps)()
    n = _I32()
    check(lib().moe_layer_get_trace(h, buf, max_stamps, ctypes.byref(n)), "moe_layer_get_trace")
    return list(buf)[:n.value]


GEMM_STATS = 9


def moe_layer_get_gemm_stats(h, max_values: int = 2 * 1024 * GEMM_STATS):
    buf = (ctypes.c_uint64 * max_values)()
    n = _I32()
    check(lib().moe_layer_get_gemm_stats(h, buf, max_values, ctypes.byref(n)), "moe_layer_get_gemm_stats")
    return list(buf)[:n.value]


def moe_layer_destroy(h) -> int:
    return lib().moe_layer_destroy(h)
