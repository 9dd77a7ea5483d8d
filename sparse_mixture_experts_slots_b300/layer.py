"""Thin PyTorch binding of the C ABI: allocation of outputs with torch and
argument marshalling.  Every step of the layer runs in the CUDA library.
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional

import torch

from . import _lib
from ._lib import SwitchConfig, SwitchRouteOut, check


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


@dataclasses.dataclass
class RouteResult:
    """Device tensors filled by switch_route (see switch_route_out in the header)."""
    expert: torch.Tensor          # [N] int32
    slot: torch.Tensor            # [N] int32
    keep: torch.Tensor            # [N] uint8
    gate: torch.Tensor            # [N] float32
    row: torch.Tensor             # [N] int32
    raw_count: torch.Tensor       # [G, E] int32
    accepted_count: torch.Tensor  # [G, E] int32
    P: torch.Tensor               # [G, E] float32
    balance: torch.Tensor         # [G] float32
    aux_loss_per_group: torch.Tensor  # [G] float32
    aux_loss: torch.Tensor        # [1] float32
    expert_rows: torch.Tensor     # [E] int32
    probs: Optional[torch.Tensor] = None   # [N, E] float32
    logits: Optional[torch.Tensor] = None  # [N, E] float32
    z_loss_per_group: Optional[torch.Tensor] = None  # [G] float32, router z-loss (unweighted)
    z_loss: Optional[torch.Tensor] = None            # [1] float32, mean over groups
    # top-2 routing only: the second choices
    expert2: Optional[torch.Tensor] = None           # [N] int32
    slot2: Optional[torch.Tensor] = None             # [N] int32
    keep2: Optional[torch.Tensor] = None             # [N] uint8
    gate2: Optional[torch.Tensor] = None             # [N] float32
    row2: Optional[torch.Tensor] = None              # [N] int32
    raw2_count: Optional[torch.Tensor] = None        # [G, E] int32
    accepted2_count: Optional[torch.Tensor] = None   # [G, E] int32

    def c_struct(self) -> SwitchRouteOut:
        return SwitchRouteOut(*[_ptr(getattr(self, n)) for n in _lib.ROUTE_FIELDS])


class SwitchMoE:
    """One top-1 Switch layer configuration bound to a library handle (and its workspace)."""

    def __init__(self, G: int, T: int, d_model: int, d_ff: int, E: int, capacity_factor: float = 1.0, *,
                 dtype: torch.dtype = torch.bfloat16, alpha: float = 0.01, capacity_override: int = 0,
                 write_probs: bool = False, write_logits: bool = False, debug_bounds: bool = False,
                 profile: bool = False, top_k: int = 1, training: bool = False, test_stall: bool = False,
                 test_discard: bool = False, device=None):
        self.lib = _lib.load()
        if dtype not in (torch.bfloat16, torch.float32):
            raise ValueError("dtype must be torch.bfloat16 or torch.float32")
        self.dtype = dtype
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        flags = ((_lib.FLAG_WRITE_PROBS if write_probs else 0) | (_lib.FLAG_WRITE_LOGITS if write_logits else 0)
                 | (_lib.FLAG_DEBUG_BOUNDS if debug_bounds else 0) | (_lib.FLAG_PROFILE if profile else 0)
                 | (_lib.FLAG_TOP2 if top_k == 2 else 0) | (_lib.FLAG_TRAINING if training else 0)
                 | (_lib.FLAG_TEST_STALL if test_stall else 0) | (_lib.FLAG_TEST_DISCARD if test_discard else 0))
        if top_k not in (1, 2):
            raise ValueError("top_k must be 1 or 2")
        self.top_k = top_k
        self.cfg = SwitchConfig(G, T, d_model, d_ff, E, float(capacity_factor), int(capacity_override),
                                float(alpha), _lib.SWITCH_BF16 if dtype == torch.bfloat16 else _lib.SWITCH_F32,
                                flags)
        self.G, self.T, self.d_model, self.d_ff, self.E = G, T, d_model, d_ff, E
        self.N = G * T
        self.C = int(self.lib.switch_capacity(ctypes.byref(self.cfg)))
        self.block_rows = int(self.lib.switch_expert_block_rows(ctypes.byref(self.cfg)))
        if self.C < 0:
            check(_lib.SWITCH_ERR_INVALID_ARG, "switch config")
        self.write_probs, self.write_logits = write_probs, write_logits
        self._h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            check(self.lib.switch_create(ctypes.byref(self.cfg), ctypes.byref(self._h)), "switch_create")

    # ------------------------------------------------------------------ lifetime
    def close(self) -> None:
        if self._h:
            check(self.lib.switch_destroy(self._h), "switch_destroy")
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------ buffers
    def alloc_route(self) -> RouteResult:
        dev, N, G, E = self.device, self.N, self.G, self.E
        i32, f32 = torch.int32, torch.float32
        return RouteResult(
            expert=torch.empty(N, dtype=i32, device=dev), slot=torch.empty(N, dtype=i32, device=dev),
            keep=torch.empty(N, dtype=torch.uint8, device=dev), gate=torch.empty(N, dtype=f32, device=dev),
            row=torch.empty(N, dtype=i32, device=dev),
            raw_count=torch.empty(G, E, dtype=i32, device=dev), accepted_count=torch.empty(G, E, dtype=i32, device=dev),
            P=torch.empty(G, E, dtype=f32, device=dev), balance=torch.empty(G, dtype=f32, device=dev),
            aux_loss_per_group=torch.empty(G, dtype=f32, device=dev), aux_loss=torch.empty(1, dtype=f32, device=dev),
            expert_rows=torch.empty(E, dtype=i32, device=dev),
            probs=torch.empty(N, E, dtype=f32, device=dev) if self.write_probs else None,
            logits=torch.empty(N, E, dtype=f32, device=dev) if self.write_logits else None,
            z_loss_per_group=torch.empty(G, dtype=f32, device=dev), z_loss=torch.empty(1, dtype=f32, device=dev),
            **({} if self.top_k == 1 else dict(
                expert2=torch.empty(N, dtype=i32, device=dev), slot2=torch.empty(N, dtype=i32, device=dev),
                keep2=torch.empty(N, dtype=torch.uint8, device=dev), gate2=torch.empty(N, dtype=f32, device=dev),
                row2=torch.empty(N, dtype=i32, device=dev), raw2_count=torch.empty(G, E, dtype=i32, device=dev),
                accepted2_count=torch.empty(G, E, dtype=i32, device=dev))))

    def alloc_expert_buffer(self, width: Optional[int] = None) -> torch.Tensor:
        return torch.empty(self.E, self.block_rows, width or self.d_model, dtype=self.dtype, device=self.device)

    # ------------------------------------------------------------------ stages
    def prepare_router(self, Wr, stream=None) -> None:
        """Split the router weights once (bfloat16 activations); later calls may pass Wr=None."""
        check(self.lib.switch_prepare_router(self._h, _ptr(Wr), _stream(stream)), "switch_prepare_router")

    def set_sm_budget(self, route_ctas: int = 0, ffn_ctas: int = 0) -> None:
        """Cap the CTAs of the persistent router and FFN kernels (0: as many as fit), so two
        layers on two streams can run their router and FFN side by side on disjoint SMs."""
        check(self.lib.switch_set_sm_budget(self._h, int(route_ctas), int(ffn_ctas)), "switch_set_sm_budget")

    def route(self, x, Wr, br=None, out: Optional[RouteResult] = None, stream=None) -> RouteResult:
        r = out or self.alloc_route()
        cs = r.c_struct()
        check(self.lib.switch_route(self._h, _ptr(x), _ptr(Wr), _ptr(br), ctypes.byref(cs), _stream(stream)),
              "switch_route")
        return r

    def dispatch(self, x, r: RouteResult, xe: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        xe = self.alloc_expert_buffer() if xe is None else xe
        cs = r.c_struct()
        check(self.lib.switch_dispatch(self._h, _ptr(x), ctypes.byref(cs), _ptr(xe), _stream(stream)),
              "switch_dispatch")
        return xe

    def expert_ffn(self, xe, W1, b1, W2, b2, expert_rows, ye: Optional[torch.Tensor] = None,
                   stream=None) -> torch.Tensor:
        ye = self.alloc_expert_buffer() if ye is None else ye
        check(self.lib.switch_expert_ffn(self._h, _ptr(xe), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2),
                                         _ptr(expert_rows), _ptr(ye), _stream(stream)), "switch_expert_ffn")
        return ye

    def combine(self, ye, r: RouteResult, x_residual=None, y: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
        y = torch.empty(self.N, self.d_model, dtype=self.dtype, device=self.device) if y is None else y
        cs = r.c_struct()
        check(self.lib.switch_combine(self._h, _ptr(ye), ctypes.byref(cs), _ptr(x_residual), _ptr(y),
                                      _stream(stream)), "switch_combine")
        return y

    def forward(self, x, Wr, br, W1, b1, W2, b2, x_residual=None, r: Optional[RouteResult] = None,
                y: Optional[torch.Tensor] = None, stream=None):
        """The whole layer; returns (y, route results)."""
        r = r or self.alloc_route()
        y = torch.empty(self.N, self.d_model, dtype=self.dtype, device=self.device) if y is None else y
        cs = r.c_struct()
        check(self.lib.switch_forward(self._h, _ptr(x), _ptr(Wr), _ptr(br), _ptr(W1), _ptr(b1), _ptr(W2),
                                      _ptr(b2), ctypes.byref(cs), _ptr(x_residual), _ptr(y), _stream(stream)),
              "switch_forward")
        return y, r

    def forward_host(self, x_host, Wr, br, W1, b1, W2, b2, y_host, aux_host=None, residual: bool = False,
                     r: Optional[RouteResult] = None, done=None, stream=None) -> RouteResult:
        """The whole layer on host activations: x_host, y_host [N, d] CPU tensors (page-locked
        for asynchronous copies), aux_host a float32 CPU tensor of one element or None.
        done: a torch.cuda.Event recorded after the copy out (the stream then does not wait
        for it); without one the stream waits for the copy out.  Returns the route results."""
        r = r or self.alloc_route()
        if x_host.device.type != "cpu" or y_host.device.type != "cpu":
            raise ValueError("forward_host takes CPU tensors for x_host and y_host")
        if aux_host is not None and (aux_host.device.type != "cpu" or aux_host.dtype != torch.float32):
            raise ValueError("aux_host must be a float32 CPU tensor")
        ev = None
        if done is not None:
            if not done.cuda_event:  # torch creates its events on first record
                done.record(torch.cuda.current_stream(self.device))
            ev = ctypes.c_void_p(done.cuda_event)
        cs = r.c_struct()
        check(self.lib.switch_forward_host(self._h, _ptr(x_host), _ptr(Wr), _ptr(br), _ptr(W1), _ptr(b1), _ptr(W2),
                                           _ptr(b2), ctypes.byref(cs), 1 if residual else 0, _ptr(y_host),
                                           _ptr(aux_host), ev, _stream(stream)),
              "switch_forward_host")
        return r

    def backward(self, x, Wr, W1, W2, r: RouteResult, dy, w_aux: float = 0.0, w_z: float = 0.0,
                 residual: bool = False, out: Optional[dict] = None, stream=None) -> dict:
        """Float32 gradients of sum(dy * y) + w_aux * aux_loss + w_z * z_loss for the last
        forward on this layer (constructed with training=True): dx, dWr, dbr, dW1, db1, dW2, db2.
        out: float32 tensors of those names to write into (allocated when None)."""
        dev, f32 = self.device, torch.float32
        E, d, F, N = self.E, self.d_model, self.d_ff, self.N
        g = out if out is not None else dict(
            dx=torch.empty(N, d, dtype=f32, device=dev), dWr=torch.empty(E, d, dtype=f32, device=dev),
            dbr=torch.empty(E, dtype=f32, device=dev), dW1=torch.empty(E, F, d, dtype=f32, device=dev),
            db1=torch.empty(E, F, dtype=f32, device=dev), dW2=torch.empty(E, d, F, dtype=f32, device=dev),
            db2=torch.empty(E, d, dtype=f32, device=dev))
        cs = r.c_struct()
        check(self.lib.switch_backward(self._h, _ptr(x), _ptr(Wr), _ptr(W1), _ptr(W2), ctypes.byref(cs), _ptr(dy),
                                       float(w_aux), float(w_z), 1 if residual else 0, _ptr(g["dx"]), _ptr(g["dWr"]),
                                       _ptr(g["dbr"]), _ptr(g["dW1"]), _ptr(g["db1"]), _ptr(g["dW2"]),
                                       _ptr(g["db2"]), _stream(stream)),
              "switch_backward")
        return g

    # ------------------------------------------------------------------ host-side reads
    def get_stats(self, r: RouteResult, stream=None) -> dict:
        GE = self.G * self.E
        aux = ctypes.c_float()
        raw = (ctypes.c_int32 * GE)()
        acc = (ctypes.c_int32 * GE)()
        dropped = ctypes.c_int64()
        cs = r.c_struct()
        check(self.lib.switch_get_stats(self._h, ctypes.byref(cs), _stream(stream), ctypes.byref(aux), raw, acc,
                                        ctypes.byref(dropped)), "switch_get_stats")
        return {"aux_loss": aux.value, "raw_count": list(raw), "accepted_count": list(acc),
                "dropped": dropped.value}

    def sync_status(self, stream=None) -> None:
        check(self.lib.switch_sync_status(self._h, _stream(stream)), "device status")

    def stage_ms(self) -> list:
        ms = (ctypes.c_float * 5)()
        check(self.lib.switch_stage_ms(self._h, ms, 5), "switch_stage_ms")
        return list(ms)

    def last_launch_count(self) -> int:
        return int(self.lib.switch_last_launch_count(self._h))
