"""MoELayer: a torch-tensor convenience wrapper over the C ABI.

PyTorch only provides device memory and streams here; every step of the
layer runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import capi


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream_handle(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class MoELayer:
    """One routed-expert layer bound to device-resident weights.

    router_w: cuda fp32 [E][H]; router_bias: cuda fp32 [E] or None;
    pool: cuda uint8 [num_slots][record_bytes] (full residency) ;
    expert_to_slot: cuda int32 [E (+1)];
    host_backing: cpu uint8 [E (+1)][record_bytes] (partial residency; pageable
    memory is copied through the library's pinned staging buffers);
    spare_slots / staging_records / cache_policy: partial residency, see
    moe_layer_config_t; zero_points: records with zero-point sections;
    shared_gate: cuda fp32 [H] gate vector of the shared expert, or None.
    """

    def __init__(self, *, hidden, intermediate, num_experts, top_k, group_size, renormalize,
                 has_shared=False, max_tokens, router_w, router_bias=None, pool=None,
                 expert_to_slot=None, num_slots=None, host_backing=None, add_residual=False, spare_slots=0,
                 staging_records=0, cache_policy=0, zero_points=False, shared_gate=None):
        partial = host_backing is not None
        self.cfg = capi.moe_layer_config_t(
            hidden=hidden, intermediate=intermediate, num_experts=num_experts, top_k=top_k,
            group_size=group_size, renormalize=int(bool(renormalize)), has_shared_expert=int(bool(has_shared)),
            max_tokens=max_tokens,
            num_slots=int(num_slots if num_slots is not None else (pool.shape[0] if pool is not None else 0)),
            residency=capi.MOE_RESIDENCY_PARTIAL if partial else capi.MOE_RESIDENCY_FULL,
            add_residual=int(bool(add_residual)), spare_slots=int(spare_slots),
            staging_records=int(staging_records), cache_policy=int(cache_policy),
            zero_points=int(bool(zero_points)))
        self.weights = capi.moe_layer_weights_t(
            router_w=_ptr(router_w), router_bias=_ptr(router_bias),
            slot_pool=None if partial else _ptr(pool), expert_to_slot=None if partial else _ptr(expert_to_slot),
            host_backing=_ptr(host_backing) if partial else None, shared_gate=_ptr(shared_gate))
        # keep the borrowed buffers alive for the handle's lifetime
        self._keep = (router_w, router_bias, pool, expert_to_slot, host_backing, shared_gate)
        self.hidden, self.top_k, self.num_experts = hidden, top_k, num_experts
        self.handle = capi.moe_layer_create(self.cfg, self.weights)

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, ids: Optional[torch.Tensor] = None,
                w: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        capi.check(capi.moe_layer_forward(self.handle, _ptr(x), T, _ptr(out), _ptr(ids), _ptr(w),
                                          _stream_handle(stream)), "moe_layer_forward")
        return out

    def forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor, ids_host=None, w_host=None, stream=None):
        capi.check(capi.moe_layer_forward_host(self.handle, _ptr(x_host), x_host.shape[0], _ptr(out_host),
                                               _ptr(ids_host), _ptr(w_host), _stream_handle(stream)),
                   "moe_layer_forward_host")
        return out_host

    def prefetch(self, x: torch.Tensor, stream=None):
        """Guess this layer's experts from x (e.g. the previous layer's input)
        and start copying them into the pool (partial residency only)."""
        capi.check(capi.moe_layer_prefetch(self.handle, _ptr(x), x.shape[0], _stream_handle(stream)),
                   "moe_layer_prefetch")

    def routing(self, T: int, stream=None):
        dev = torch.device("cuda")
        E, k = self.num_experts, self.top_k
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
        inv = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
        capi.check(capi.moe_layer_routing(self.handle, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
                                          _stream_handle(stream)), "moe_layer_routing")
        return counts, offsets, perm[:T * k], inv[:T * k]

    def sync(self, stream=None):
        capi.check(capi.moe_layer_sync(self.handle, _stream_handle(stream)), "moe_layer_sync")

    def set_profiling(self, enable: bool = True):
        capi.moe_layer_set_profiling(self.handle, enable)

    def profile(self):
        return capi.moe_layer_get_profile(self.handle)

    def stats(self):
        return capi.moe_layer_get_stats(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            capi.moe_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoEStack:
    """Layers run one after another on one stream: x_{l+1} = layer_l(x_l).

    Borrows the MoELayer objects (keep them alive while the stack lives).
    A one-token forward over fully resident layers of one shape runs as a
    single kernel launch (``single_launch``)."""

    def __init__(self, layers):
        self._layers = list(layers)
        arr = (capi._P * len(self._layers))(*[l.handle for l in self._layers])
        h = capi._P()
        capi.check(capi.lib().moe_stack_create(arr, len(self._layers), ctypes.byref(h)), "moe_stack_create")
        self.handle = h.value
        self.hidden = self._layers[0].hidden

    @property
    def single_launch(self) -> bool:
        return bool(capi.lib().moe_stack_single_launch(self.handle))

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, states: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(x)
        capi.check(capi.lib().moe_stack_forward(self.handle, _ptr(x), x.shape[0], _ptr(out), _ptr(states),
                                                _stream_handle(stream)), "moe_stack_forward")
        return out

    def sync(self, stream=None):
        capi.check(capi.lib().moe_stack_sync(self.handle, _stream_handle(stream)), "moe_stack_sync")

    def close(self):
        if getattr(self, "handle", None):
            capi.lib().moe_stack_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
