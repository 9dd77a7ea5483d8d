"""CPU-only checks of the C ABI: the library loads, exports every declared entry
point, and its host-side logic (capacity rule, config validation) behaves.
No compute call is made here (there is no GPU)."""
import ctypes
import os
import re

import pytest

from oracle import switch_oracle as so
from gen import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "switch_moe.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_mixture_experts_slots_b300 import _lib
    return _lib.load()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    return re.findall(r"SWITCH_API\s+[\w\s\*]+?\b(switch_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for n in ("switch_create", "switch_destroy", "switch_route", "switch_dispatch", "switch_expert_ffn",
              "switch_combine", "switch_forward", "switch_get_stats", "switch_capacity"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from sparse_mixture_experts_slots_b300 import _lib
    names = declared_functions()
    assert len(names) == len(set(names))
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature"
    assert set(_lib.SIGNATURES) == set(names)


def _cfg(G=1, T=64, d=128, F=256, E=4, c=1.0, override=0, dtype=1):
    from sparse_mixture_experts_slots_b300._lib import SwitchConfig
    return SwitchConfig(G, T, d, F, E, c, override, 0.01, dtype, 0)


def test_struct_layout():
    from sparse_mixture_experts_slots_b300._lib import SwitchConfig, SwitchRouteOut
    assert ctypes.sizeof(SwitchConfig) == 48
    assert SwitchConfig.capacity_factor.offset == 24
    # the binding's fields are the header struct's pointer fields, in the same order
    text = open(HEADER, encoding="utf-8").read()
    body = re.search(r"typedef struct \{((?:(?!typedef).)*?)\} switch_route_out;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    header_fields = re.findall(r"\*\s*(\w+)\s*;", body)
    assert [n for n, _ in SwitchRouteOut._fields_] == header_fields
    assert ctypes.sizeof(SwitchRouteOut) == len(header_fields) * 8


def test_capacity_matches_oracle_rule(lib):
    for name, s in WORKLOADS.items():
        cfg = _cfg(s.G, s.T, s.d_model, s.d_ff, s.E, s.capacity_factor, 0, 0 if s.dtype == "f32" else 1)
        assert lib.switch_capacity(ctypes.byref(cfg)) == so.capacity(s.capacity_factor, s.T, s.E), name
    for (c, T, E) in [(1.1, 100, 10), (1.0, 10, 3), (0.5, 64, 4), (1.25, 64, 4), (1.0, 7, 8), (3.0, 5, 1)]:
        cfg = _cfg(T=T, E=E, c=c)
        assert lib.switch_capacity(ctypes.byref(cfg)) == so.capacity(c, T, E)
    cfg = _cfg(T=64, E=4, override=8)
    assert lib.switch_capacity(ctypes.byref(cfg)) == 8


def test_block_rows(lib):
    # G groups x min(C, T) rows per expert block
    assert lib.switch_expert_block_rows(ctypes.byref(_cfg(G=8, T=4096, E=64, c=1.25))) == 8 * 80
    assert lib.switch_expert_block_rows(ctypes.byref(_cfg(G=2, T=5, E=1, c=3.0))) == 2 * 5


@pytest.mark.parametrize("bad", [
    dict(G=0), dict(T=-1), dict(E=0), dict(E=4096), dict(c=0.0), dict(c=-1.0), dict(override=-2),
    dict(d=100), dict(F=20), dict(dtype=7), dict(d=0),
])
def test_invalid_configs_rejected_on_host(lib, bad):
    kw = dict(G=1, T=64, d=128, F=256, E=4, c=1.0, override=0, dtype=1)
    kw.update(bad)
    cfg = _cfg(**kw)
    assert lib.switch_capacity(ctypes.byref(cfg)) == -1
    h = ctypes.c_void_p()
    assert lib.switch_create(ctypes.byref(cfg), ctypes.byref(h)) == 1  # SWITCH_ERR_INVALID_ARG
    assert not h.value


def test_fp32_alignment_rule(lib):
    # d * 4 bytes must be a multiple of 16: d = 48 ok (the toy model), d = 50 not
    assert lib.switch_capacity(ctypes.byref(_cfg(d=48, F=32, dtype=0))) > 0
    assert lib.switch_capacity(ctypes.byref(_cfg(d=50, F=32, dtype=0))) == -1


def test_null_arguments_rejected(lib):
    assert lib.switch_destroy(None) == 1
    assert lib.switch_route(None, None, None, None, None, None) == 1
    assert lib.switch_forward(None, None, None, None, None, None, None, None, None, None, None, None) == 1
    assert lib.switch_create(None, None) == 1
    assert lib.switch_prepare_router(None, None, None) == 1
    assert lib.switch_set_sm_budget(None, 0, 0) == 1


def test_status_strings(lib):
    for s in range(7):
        assert lib.switch_status_string(s)
    from sparse_mixture_experts_slots_b300 import SwitchError
    e = SwitchError(1, "x")
    assert "invalid argument" in str(e)


def test_top2_capacity_and_config(lib):
    from sparse_mixture_experts_slots_b300._lib import FLAG_TOP2, SwitchConfig
    for (c, T, E) in [(1.0, 64, 4), (1.25, 4096, 64), (1.1, 100, 10), (0.5, 7, 3)]:
        cfg = SwitchConfig(1, T, 128, 256, E, c, 0, 0.01, 1, FLAG_TOP2)
        assert lib.switch_capacity(ctypes.byref(cfg)) == so.capacity(2 * c, T, E)
    one = SwitchConfig(1, 64, 128, 256, 1, 1.0, 0, 0.01, 1, FLAG_TOP2)  # top-2 needs two experts
    assert lib.switch_capacity(ctypes.byref(one)) == -1


def test_flag_constants_match_the_header():
    from sparse_mixture_experts_slots_b300 import _lib
    text = open(HEADER, encoding="utf-8").read()
    flags = {m.group(1): int(m.group(2), 16) for m in re.finditer(r"#define SWITCH_FLAG_(\w+)\s+0x([0-9a-fA-F]+)u", text)}
    assert flags, "no SWITCH_FLAG_ definitions found"
    for name, value in flags.items():
        assert getattr(_lib, "FLAG_" + name) == value, name
    assert len(set(flags.values())) == len(flags), "flag bits overlap"
