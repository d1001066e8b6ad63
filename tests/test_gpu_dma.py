"""The return copy on the copy engines (moe_forward_dma).

No consumer SMs: the down-projection runs on every SM and publishes, per completed band, a record in
pinned host memory; the calling thread issues one device-to-device cudaMemcpyAsync per ready band on
a copy stream, and the combine waits for that stream. Bar: out and Ret bitwise equal to the
GEMM-then-copy path on the same inputs (the copies move the same bytes), over several calls in a row
with different inputs; the argument checks; a GEMM that stops early is reported, not waited for.
"""
import ctypes

import pytest
import torch

import tile_level_copy_gb300 as tlc
from tile_level_copy_gb300 import inputs
from tests.gpu_util import Layer, small

pytestmark = pytest.mark.gpu

PAIR = tlc.MOE_PAIR_UMMA


def host_rec_for(cfg):
    n = tlc.dma_host_bytes(cfg)
    return torch.zeros((n + 15) // 16 * 4, dtype=torch.int32).pin_memory()


@pytest.mark.parametrize("name", ["tiny", "mixtral", "skew", "fine"])
@pytest.mark.parametrize("flags", [PAIR, 0], ids=["pairs", "single"])
def test_dma_copy_equals_sequential(name, flags):
    w = small(name)
    L = Layer(w, seed=1, cfg_kw=dict(consumer_ctas=4, flags=flags))
    want = L.run(sequential=True)
    ret_seq = L.ws.view("Ret").clone()
    rec = host_rec_for(L.cfg)
    for _ in range(2):  # the second call's records must not be confused with the first's
        L.ws.view("Ret").zero_()
        L.out.zero_()
        tlc.forward_dma(L.cfg, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws, rec)
        assert tlc.status(L.cfg, L.ws)[0] == tlc.MOE_OK
        assert torch.equal(L.out, want)
        assert torch.equal(L.ws.view("Ret"), ret_seq)


@pytest.mark.parametrize("window", [0, 20, 1 << 20])
@pytest.mark.parametrize("flags", [PAIR, 0], ids=["pairs", "single"])
def test_dma_copy_with_direct_tail(flags, window):
    """MOE_DIRECT_TAIL on the copy-engine path: the bands the window's items complete are written into
    Ret by the epilogue and their records carry 0 rows (no copy issued); out and Ret stay equal to the
    GEMM-then-copy path, and those bands' Yp rows (zeroed first) stay untouched."""
    w = small("skew")
    L = Layer(w, seed=5, cfg_kw=dict(consumer_ctas=4, flags=flags))
    want = L.run(sequential=True)
    ret_seq = L.ws.view("Ret").clone()
    cfg = tlc.Config.from_workload(w, consumer_ctas=4, flags=flags | tlc.MOE_DIRECT_TAIL, tail_window=window)
    rec = host_rec_for(cfg)
    L.ws.view("Ret").zero_()
    L.ws.view("Yp").zero_()
    tlc.forward_dma(cfg, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws, rec)
    assert tlc.status(cfg, L.ws)[0] == tlc.MOE_OK
    assert torch.equal(L.out, want)
    assert torch.equal(L.ws.view("Ret"), ret_seq)
    MT = int(L.ws.view("meta")[1].item())
    valid = rec[4:4 + 4 * MT].view(MT, 4)[:, 2].tolist()
    tiles = L.ws.view("tiles").cpu().numpy()[:MT]
    Yp = L.ws.view("Yp").view(torch.int16).cpu().numpy()
    zero_rows = [m for m in range(MT) if valid[m] == 0]
    for m in range(MT):  # a record says 0 rows exactly for the bands left out of Yp
        row0, v = int(tiles[m, 2]), int(tiles[m, 3])
        assert (valid[m] == 0) == (not Yp[row0:row0 + v].any()), m
        assert valid[m] in (0, v)
    if window == 20:
        assert 0 < len(zero_rows) < MT
    else:  # a huge window, or one wave: the small layer has fewer tiles than that
        assert len(zero_rows) == MT


def test_dma_copy_calls_in_a_row_with_new_inputs_and_events():
    """Three calls with different routing on one workspace and one record buffer; each output equals
    the sequential path's of its own inputs; the copy-done event follows the down-projection's."""
    w = small("skew")
    L = Layer(w, seed=0, cfg_kw=dict(consumer_ctas=4, flags=PAIR))
    rec = host_rec_for(L.cfg)
    for seed in (3, 4, 5):
        lg = torch.from_numpy(inputs.make_logits(w, seed)).cuda()
        x = inputs.make_x(w, seed).cuda()
        tlc.forward(L.cfg, lg, x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws, sequential=True)
        want = L.out.clone()
        L.out.zero_()
        ev = tlc.stage_events()
        tlc.forward_dma(L.cfg, lg, x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws, rec, events=ev)
        torch.cuda.synchronize()
        assert torch.equal(L.out, want)
        assert ev[tlc.EV_DOWN].elapsed_time(ev[tlc.EV_END]) > 0
        assert ev[tlc.EV_BEGIN].elapsed_time(ev[tlc.EV_COPIED]) > 0


@pytest.mark.slow
def test_dma_copy_full_size_mixtral():
    import bench
    w = inputs.WORKLOADS["mixtral"]
    L = Layer(w, seed=0, cfg_kw=dict(consumer_ctas=4, flags=bench.default_flags(False)))
    want = L.run(sequential=True)
    ret_seq = L.ws.view("Ret").clone()
    L.ws.view("Ret").zero_()
    rec = host_rec_for(L.cfg)
    tlc.forward_dma(L.cfg, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws, rec)
    assert tlc.status(L.cfg, L.ws)[0] == tlc.MOE_OK
    assert torch.equal(L.out, want)
    assert torch.equal(L.ws.view("Ret"), ret_seq)


def test_dma_copy_argument_checks():
    w = small("tiny")
    L = Layer(w, seed=0)
    rec = host_rec_for(L.cfg)
    W = L.W
    with pytest.raises(tlc.MoEError) as ei:  # too small
        tlc.forward_dma(L.cfg, L.logits, L.x, W["W1"], W["W3"], W["W2"], L.out, L.ws, rec[:4])
    assert ei.value.code == tlc.MOE_ERR_ARG
    with pytest.raises(ValueError):  # not pinned
        tlc.forward_dma(L.cfg, L.logits, L.x, W["W1"], W["W3"], W["W2"], L.out, L.ws, torch.zeros_like(rec))
    # a stream being captured into a graph is refused before anything is enqueued
    s = torch.cuda.Stream()
    c = L.cfg.to_c()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rc = tlc.lib().moe_forward_dma(ctypes.byref(c), p(L.logits), p(L.x), p(W["W1"]), p(W["W3"]), p(W["W2"]),
                                       p(L.out), L.ws.ptr, L.ws.nbytes, p(rec), rec.numel() * 4, None,
                                       ctypes.c_void_p(s.cuda_stream))
    assert rc == tlc.MOE_ERR_ARG
    assert b"graph" in tlc.lib().moe_last_error()


def test_dma_copy_reports_a_stopped_gemm_and_context_survives():
    """The pair GEMMs stop early (test hook: rank 1's loads stall until the bounded waits run out): the
    call sees the stream finish with band records missing and returns MOE_ERR_TIMEOUT instead of
    waiting; the next call is correct."""
    w = small("mixtral")
    L = Layer(w, seed=2, cfg_kw=dict(consumer_ctas=4, flags=PAIR))
    want = L.run(sequential=True)
    rec = host_rec_for(L.cfg)
    bad = tlc.Config.from_workload(w, consumer_ctas=4, flags=PAIR | tlc.MOE_TEST_STALL_PIPE1, timeout_us=20000)
    with pytest.raises(tlc.MoEError) as ei:
        tlc.forward_dma(bad, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws, rec)
    assert ei.value.code == tlc.MOE_ERR_TIMEOUT
    assert tlc.status(bad, L.ws)[0] == tlc.MOE_ERR_TIMEOUT
    tlc.forward_dma(L.cfg, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws, rec)
    assert tlc.status(L.cfg, L.ws)[0] == tlc.MOE_OK
    assert torch.equal(L.out, want)
