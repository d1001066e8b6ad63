"""moe_route_static, the entry point that allocates nothing.

Some callers cannot allocate device memory (an allocator callback, a plugin whose host owns all
device memory, a serving runtime with a fixed pool), so they cannot hand moe_plan a workspace. For
them moe_route_static keeps its scratch in a file-scope device array inside the library. This test
calls it through the C ABI twice in a row and checks each result against moe_plan's, which runs the
same kernels on a caller-allocated workspace. It lives in a file that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import tile_level_copy_gb300 as tlc
from tile_level_copy_gb300 import inputs

pytestmark = pytest.mark.gpu


def via_moe_plan(cfg, logits):
    ws = tlc.Workspace(cfg)
    idx = torch.empty(cfg.T, cfg.topk, dtype=torch.int32, device="cuda")
    gate = torch.empty(cfg.T, cfg.topk, dtype=torch.float32, device="cuda")
    tlc.plan(cfg, logits, None, ws, idx, gate)
    torch.cuda.synchronize()
    return {"idx": idx.cpu(), "gate": gate.cpu(), "slot": ws.view("slot").cpu(),
            "ret_slot": ws.view("ret_slot").cpu(), "offsets": ws.view("offsets").cpu()}


def via_static(cfg, logits):
    T, k, G = cfg.T, cfg.topk, cfg.E * cfg.R
    out = {"idx": torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
           "gate": torch.full((T, k), -7.0, dtype=torch.float32, device="cuda"),
           "slot": torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
           "ret_slot": torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
           "offsets": torch.full((G + 1,), -7, dtype=torch.int32, device="cuda")}
    c = cfg.to_c()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = tlc.lib().moe_route_static(ctypes.byref(c), p(logits), p(out["idx"]), p(out["gate"]), p(out["slot"]),
                                    p(out["ret_slot"]), p(out["offsets"]), stream)
    assert rc == tlc.MOE_OK, tlc.lib().moe_last_error()
    torch.cuda.synchronize()
    return {n: t.cpu() for n, t in out.items()}


def test_static_scratch_plan_matches_workspace_plan_twice():
    for name, seed in (("fine", 1), ("skew", 2)):  # two calls in a row, different shapes
        w = inputs.WORKLOADS[name]
        cfg = tlc.Config.from_workload(w, flags=tlc.MOE_PLAN_SKIP_PERMUTE)
        logits = torch.from_numpy(inputs.make_logits(w, seed)).cuda()
        want = via_moe_plan(cfg, logits)
        got = via_static(cfg, logits)
        for n in ("idx", "slot", "ret_slot", "offsets"):
            assert torch.equal(got[n], want[n]), n
        np.testing.assert_allclose(got["gate"].numpy(), want["gate"].numpy(), rtol=0, atol=0)


def test_static_scratch_rejects_configs_beyond_its_size():
    cfg = tlc.Config(T=131072, d=128, ffn=128, E=64, topk=8, R=8, tile_M=128)
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    c = cfg.to_c()
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = tlc.lib().moe_route_static(ctypes.byref(c), p, p, p, p, p, p, None)
    assert rc == tlc.MOE_ERR_ARG
    assert b"static scratch" in tlc.lib().moe_last_error()
