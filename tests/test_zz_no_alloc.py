"""switch_route_static, the routing step without a handle, against switch_route.

Some callers cannot allocate device memory once they are running (work recorded into
an already-instantiated CUDA graph, a latency-critical loop where cudaMalloc may block
or fail, an embedding without an allocator).  For them the library exposes one
handle-free routing call whose scratch is a fixed array inside the library.  This test
calls it through the C ABI, twice in a row on the same inputs, and checks every output
against switch_route on a handle: integers bit-exact, floats within the parity tests'
relative tolerance.  It runs last (file name) and needs nothing from the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from gen import LayerShape, WORKLOADS, make_inputs, workload_seed
import parity as P

pytestmark = pytest.mark.gpu

SHAPES = {
    "ragged-groups": (LayerShape("ragged-groups", 2, 300, 256, 384, 8, 1.0), dict(router_bias_std=0.1), 7),
    "fp32-toy": (WORKLOADS["tiny-e16-fp32"], {}, workload_seed("tiny-e16-fp32")),
    "switch-base": (WORKLOADS["switch-base-e128"], {}, workload_seed("switch-base-e128")),
    "many-experts": (WORKLOADS["many-experts-e2048"], {}, workload_seed("many-experts-e2048")),
}


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _same(a, b, name):
    if a is None:
        return
    if a.is_floating_point():
        P.rel_close(P.to_np(a), P.to_np(b), what=name)
    else:
        assert torch.equal(a, b), name


@pytest.mark.parametrize("name", list(SHAPES))
def test_static_route_matches_handle_route(name):
    shape, kw, seed = SHAPES[name]
    inp = make_inputs(shape, seed, "cuda", with_experts=False, **kw)
    layer = P.make_layer(shape, write_probs=shape.N * shape.E <= (1 << 24))
    lib = layer.lib
    stream = torch.cuda.current_stream().cuda_stream
    ref = layer.route(inp["x"], inp["Wr"], inp["br"])
    layer.sync_status()
    ptr = lambda t: None if t is None else t.data_ptr()
    for call in range(2):  # the second call reuses the array the first one left behind
        got = layer.alloc_route()
        cs = got.c_struct()
        st = lib.switch_route_static(ctypes.byref(layer.cfg), ptr(inp["x"]), ptr(inp["Wr"]), ptr(inp["br"]),
                                     ctypes.byref(cs), stream)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        for field in ("expert", "slot", "keep", "row", "raw_count", "accepted_count", "expert_rows", "gate", "P",
                      "balance", "aux_loss_per_group", "aux_loss", "probs"):
            _same(getattr(got, field), getattr(ref, field), f"call {call}: {field}")


def test_static_route_rejects_oversized_and_invalid():
    from sparse_mixture_experts_slots_b300 import _lib
    lib = _lib.load()
    big = _lib.SwitchConfig(1, 1 << 20, 64, 128, 64, 1.0, 0, 0.01, _lib.SWITCH_F32, 0)  # 256 MiB of logits
    out = _lib.SwitchRouteOut(*([ctypes.c_void_p(16)] * 12 + [None, None]))
    assert lib.switch_route_static(ctypes.byref(big), ctypes.c_void_p(16), ctypes.c_void_p(16), None,
                                   ctypes.byref(out), None) == _lib.SWITCH_ERR_UNSUPPORTED
    bad = _lib.SwitchConfig(1, 64, 64, 128, 0, 1.0, 0, 0.01, _lib.SWITCH_BF16, 0)  # E = 0
    assert lib.switch_route_static(ctypes.byref(bad), ctypes.c_void_p(16), ctypes.c_void_p(16), None,
                                   ctypes.byref(out), None) == _lib.SWITCH_ERR_INVALID_ARG
