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
        rc, detail = tlc.status(cfg, None)  # the static call's own status words
        assert rc == tlc.MOE_OK, (rc, detail, tlc.lib().moe_last_error())


def test_static_scratch_ignores_the_permute_flag():
    """cfg.flags has no effect on the static entry point: with and without MOE_PLAN_SKIP_PERMUTE the
    routing and row layout are the same, and equal to moe_plan's."""
    w = inputs.WORKLOADS["skew"]
    logits = torch.from_numpy(inputs.make_logits(w, 3)).cuda()
    with_flag = via_static(tlc.Config.from_workload(w, flags=tlc.MOE_PLAN_SKIP_PERMUTE), logits)
    cfg0 = tlc.Config.from_workload(w, flags=0)
    without = via_static(cfg0, logits)
    want = via_moe_plan(tlc.Config.from_workload(w, flags=tlc.MOE_PLAN_SKIP_PERMUTE), logits)
    for n in ("idx", "gate", "slot", "ret_slot", "offsets"):
        assert torch.equal(with_flag[n], without[n]), n
        assert torch.equal(without[n], want[n]), n
    assert tlc.status(cfg0, None)[0] == tlc.MOE_OK


def test_static_scratch_reports_a_failed_plan_check():
    """A plan that fails its device-side bounds check is reported to the caller of the static entry
    point through moe_status(cfg, NULL): the test hook MOE_TEST_PLAN_FAIL makes the plan kernel report
    one (detail -3); the next call without the hook clears it. The workspace path reports the same."""
    w = inputs.WORKLOADS["fine"]
    logits = torch.from_numpy(inputs.make_logits(w, 5)).cuda()
    bad = tlc.Config.from_workload(w, flags=tlc.MOE_TEST_PLAN_FAIL)
    via_static(bad, logits)
    rc, detail = tlc.status(bad, None)
    assert rc == tlc.MOE_ERR_PLAN and detail == -3
    assert b"plan" in tlc.lib().moe_last_error()
    good = tlc.Config.from_workload(w)
    via_static(good, logits)
    assert tlc.status(good, None) == (tlc.MOE_OK, 0)
    bad_ws = tlc.Config.from_workload(w, flags=tlc.MOE_TEST_PLAN_FAIL | tlc.MOE_PLAN_SKIP_PERMUTE)
    ws = tlc.Workspace(bad_ws)
    tlc.plan(bad_ws, logits, None, ws)
    assert tlc.status(bad_ws, ws) == (tlc.MOE_ERR_PLAN, -3)


def test_static_scratch_rejects_configs_beyond_its_size():
    cfg = tlc.Config(T=131072, d=128, ffn=128, E=64, topk=8, R=8, tile_M=128)
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    c = cfg.to_c()
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = tlc.lib().moe_route_static(ctypes.byref(c), p, p, p, p, p, p, None)
    assert rc == tlc.MOE_ERR_ARG
    assert b"static scratch" in tlc.lib().moe_last_error()
    assert tlc.status(cfg, None)[0] == tlc.MOE_ERR_ARG  # nor can its status be read
