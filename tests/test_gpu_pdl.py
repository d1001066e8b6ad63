"""Programmatic dependent launch between the layer's kernels (MOE_PDL).

Each kernel after the first may start its prologue while the previous one finishes, and waits on the
GPU (griddepcontrol.wait) before it reads that kernel's outputs. Bar: the layer output, Hc and Ret
bitwise equal to the same layer launched without it, overlapped and sequential, eager and replayed
from a CUDA graph, for the CTA-pair, single-CTA and copy-warp configurations.
"""
import pytest
import torch

import tile_level_copy_gb300 as tlc
from tile_level_copy_gb300 import inputs
from tests.gpu_util import Layer, small

pytestmark = pytest.mark.gpu

PDL = tlc.MOE_PDL
CONFIGS = [(4, tlc.MOE_PAIR_UMMA | tlc.MOE_TAIL_ASSIST | tlc.MOE_DIRECT_TAIL), (8, tlc.MOE_TAIL_ASSIST),
           (0, tlc.MOE_COPY_WARPS | tlc.MOE_TAIL_ASSIST), (4, tlc.MOE_PAIR_UMMA | tlc.MOE_FUSED_GEMMS),
           (4, tlc.MOE_PAIR_UMMA | tlc.MOE_FUSED_DISPATCH)]
IDS = ["pairs-direct", "single", "copywarps", "fused-gemms", "fused-dispatch"]


@pytest.mark.parametrize("name", ["tiny", "mixtral", "skew", "fine"])
@pytest.mark.parametrize("consumers,flags", CONFIGS, ids=IDS)
def test_pdl_equals_serial_launches(name, consumers, flags):
    L = Layer(small(name), seed=7)
    for seq in (False, True):
        base = tlc.Config.from_workload(L.w, consumer_ctas=consumers, flags=flags, timeout_us=500000)
        want = L.run(sequential=seq, cfg=base)
        ret = L.ws.view("Ret").clone()
        L.ws.view("Ret").zero_()
        got = L.run(sequential=seq, cfg=tlc.Config.from_workload(L.w, consumer_ctas=consumers, flags=flags | PDL,
                                                                  timeout_us=500000))
        assert torch.equal(got, want)
        assert torch.equal(L.ws.view("Ret"), ret)


def test_pdl_in_a_replayed_graph():
    """Three steps captured in one graph with programmatic edges, replayed twice: every step's
    output equals the serial launches'."""
    w = small("mixtral")
    L = Layer(w, seed=9)
    cfg = tlc.Config.from_workload(w, consumer_ctas=4, flags=tlc.MOE_PAIR_UMMA | tlc.MOE_TAIL_ASSIST |
                                   tlc.MOE_DIRECT_TAIL | PDL)
    want = L.run(sequential=False, cfg=tlc.Config.from_workload(w, consumer_ctas=4, flags=cfg.flags & ~PDL))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        L.run(sequential=False, cfg=cfg)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            tlc.forward(cfg, L.logits, L.x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws)
    for _ in range(2):
        L.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert tlc.status(cfg, L.ws)[0] == tlc.MOE_OK
        assert torch.equal(L.out, want)


@pytest.mark.parametrize("consumers,flags", CONFIGS, ids=IDS)
def test_back_to_back_layers_with_different_routings(consumers, flags):
    """Sixteen calls on two alternating inputs (different routings, so different layouts, work items
    and bands), enqueued back to back on one stream with no other work between them, each into its
    own output: every output equals its input's result from a call run alone. A call that read a
    layout, a plan table, a flag or a return row of the call before it would differ."""
    w = small("mixtral")
    L = Layer(w, seed=4)
    ins = [(L.logits, L.x), (torch.from_numpy(inputs.make_logits(w, 21)).cuda(), inputs.make_x(w, 21).cuda())]
    cfg = tlc.Config.from_workload(w, consumer_ctas=consumers, flags=flags | PDL)
    want = []
    for lg, x in ins:
        tlc.forward(cfg, lg, x, L.W["W1"], L.W["W3"], L.W["W2"], L.out, L.ws)
        assert tlc.status(cfg, L.ws)[0] == tlc.MOE_OK
        want.append(L.out.clone())
    assert not torch.equal(want[0], want[1])
    outs = [torch.full_like(L.out, float("nan")) for _ in range(16)]
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        lg, x = ins[i % 2]
        tlc.forward(cfg, lg, x, L.W["W1"], L.W["W3"], L.W["W2"], o, L.ws)
    assert tlc.status(cfg, L.ws)[0] == tlc.MOE_OK
    for i, o in enumerate(outs):
        assert torch.equal(o, want[i % 2]), i


@pytest.mark.parametrize("name", ["mixtral", "fine"])
def test_pdl_full_size_in_the_bench_configuration(name):
    import bench
    c, warps = bench.DEFAULT_COPY[name]
    L = Layer(inputs.WORKLOADS[name], seed=3)
    flags = bench.default_flags(warps) & ~PDL
    want = L.run(sequential=False, cfg=tlc.Config.from_workload(L.w, consumer_ctas=c, flags=flags))
    got = L.run(sequential=False, cfg=tlc.Config.from_workload(L.w, consumer_ctas=c, flags=flags | PDL))
    assert torch.equal(got, want)
