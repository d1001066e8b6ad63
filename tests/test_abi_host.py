"""Host-side checks of libmoe that need no GPU: the library loads, exports every symbol that
include/moe.h declares, and its host-only logic (config validation, workspace layout) behaves."""
import ctypes
import os
import re

import pytest

import tile_level_copy_gb300 as tlc
from tile_level_copy_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    return set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text))


def test_header_declares_the_binding_exports():
    assert declared_symbols() == set(tlc.EXPORTS)


def test_header_constants_match_the_binding():
    """Every MOE_ flag, error code, trace slot and stage event the header defines has the same value
    in the binding (trace slots and events drop the MOE_ prefix there)."""
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    defs = re.findall(r"#define\s+(MOE_\w+)\s+\(?(-?(?:0x[0-9a-fA-F]+|\d+))u?\)?\s*(?:/\*|$)", text, re.M)
    assert len(defs) > 30
    for name, val in defs:
        attr = name[4:] if name.startswith(("MOE_TRACE_", "MOE_EV_")) else name
        assert hasattr(tlc, attr), name
        assert getattr(tlc, attr) == int(val, 0), name


def test_library_exports_every_declared_symbol(built_library):
    for name in declared_symbols():
        assert hasattr(built_library, name), name
    # the library exports nothing else with C linkage besides the moe_ API
    nm = os.popen(f"nm -D --defined-only {tlc.LIB_PATH}").read()
    exported = {ln.split()[-1] for ln in nm.splitlines() if " T " in ln}
    assert declared_symbols() <= exported
    assert {s for s in exported if s.startswith("moe_")} == declared_symbols()


def cfg_of(name, **kw):
    return tlc.Config.from_workload(inputs.WORKLOADS[name], **kw)


@pytest.mark.parametrize("name", ["tiny", "mixtral", "skew", "fine"])
def test_layout_regions_are_aligned_and_disjoint(name):
    cfg = cfg_of(name)
    L = tlc.workspace_layout(cfg)
    assert L["bytes"] == tlc.workspace_size(cfg)
    w = inputs.WORKLOADS[name]
    TK, G = w.T * w.topk, w.E * w.R
    assert L["P_max"] == -(-(TK + min(G, TK) * (w.tile_M - 1)) // w.tile_M) * w.tile_M
    assert L["MT_max"] * w.tile_M == L["P_max"]
    # compact GEMM input rows: every expert's run padded to the 128-row UMMA tile
    assert L["PC_max"] == -(-(TK + min(w.E, TK) * 127) // 128) * 128 and L["IU_max"] * 128 == L["PC_max"]
    assert (w.T // w.R) % L["chunk_tokens"] == 0 and L["chunk_tokens"] <= 128
    offs = sorted(L[r] for r in tlc.LAYOUT_REGIONS)
    assert all(o % 1024 == 0 for o in offs)
    assert len(set(offs)) == len(offs) and offs[-1] < L["bytes"]
    ws_view_sizes = {"Xc": L["PC_max"] * w.d * 2, "Hc": L["PC_max"] * w.ffn * 2, "Yp": L["P_max"] * w.d * 2,
                     "Ret": TK * w.d * 2, "items_up": L["IU_max"] * 8, "tile_crow": L["MT_max"] * 4}
    for r, n in ws_view_sizes.items():
        nxt = min(o for o in offs if o > L[r]) if L[r] != offs[-1] else L["bytes"]
        assert nxt - L[r] >= n


@pytest.mark.parametrize("bad", [
    dict(d=100), dict(ffn=200), dict(topk=9, E=16), dict(topk=5, E=4), dict(R=3), dict(tile_M=32),
    dict(mgb=0), dict(mgb=5), dict(E=300), dict(T=0), dict(E=256, R=8),
])
def test_invalid_configs_are_rejected(bad):
    cfg = cfg_of("tiny", **{})
    for k_, v in bad.items():
        setattr(cfg, k_, v)
    with pytest.raises(tlc.MoEError) as ei:
        tlc.workspace_size(cfg)
    assert ei.value.code == tlc.MOE_ERR_ARG
    assert len(str(ei.value)) > 20


def test_reserved_fields_must_be_zero(built_library):
    c = cfg_of("tiny").to_c()
    c.reserved[1] = 1
    n = ctypes.c_size_t()
    assert built_library.moe_workspace_size(ctypes.byref(c), ctypes.byref(n)) == tlc.MOE_ERR_ARG


def test_null_arguments_are_rejected(built_library):
    n = ctypes.c_size_t()
    assert built_library.moe_workspace_size(None, ctypes.byref(n)) == tlc.MOE_ERR_ARG
    c = cfg_of("tiny").to_c()
    assert built_library.moe_workspace_size(ctypes.byref(c), None) == tlc.MOE_ERR_ARG
    # a NULL workspace is refused before any CUDA call
    rc = built_library.moe_forward(ctypes.byref(c), None, None, None, None, None, None, None, 0, None)
    assert rc == tlc.MOE_ERR_ARG


def test_workspace_size_grows_with_tokens():
    small = tlc.workspace_size(cfg_of("mixtral", ))
    cfg = cfg_of("mixtral")
    cfg.T = 8192
    assert tlc.workspace_size(cfg) > small


def test_static_entry_point_rejects_null_pointers_without_a_gpu(built_library):
    """moe_route_static checks its config and pointers before any CUDA call."""
    c = cfg_of("tiny").to_c()
    assert built_library.moe_route_static(ctypes.byref(c), None, None, None, None, None, None, None) == tlc.MOE_ERR_ARG
    assert b"NULL" in built_library.moe_last_error()
    c.R = 3  # T % R != 0
    one = ctypes.c_void_p(16)
    assert built_library.moe_route_static(ctypes.byref(c), one, one, one, one, one, one, None) == tlc.MOE_ERR_ARG


def test_negative_tail_window_is_rejected():
    cfg = cfg_of("tiny", tail_window=-1)
    with pytest.raises(tlc.MoEError) as ei:
        tlc.workspace_size(cfg)
    assert ei.value.code == tlc.MOE_ERR_ARG
