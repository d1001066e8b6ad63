"""Fused dispatch (MOE_FUSED_DISPATCH): the permute's row copies inside the SwiGLU GEMM.

The SwiGLU GEMM's epilogue warps copy the token rows into the compact rows Xc expert by expert and
release a per-expert row count; the TMA threads acquire it before loading an expert's rows. Bar: Xc,
Hc and the layer output bitwise equal to the separate permute launch's on the same inputs (the same
bytes reach the same rows, and the GEMM is unchanged), for the CTA-pair and single-CTA kernels, on the
four workloads' reduced shapes, degenerate shapes and the full sizes in the bench's configuration.
"""
import pytest
import torch

import tile_level_copy_gb300 as tlc
from tile_level_copy_gb300 import inputs
from tests.gpu_util import Layer, small

pytestmark = pytest.mark.gpu

FD = tlc.MOE_FUSED_DISPATCH


def compare(L: Layer, flags, consumers=4):
    cfg = tlc.Config.from_workload(L.w, consumer_ctas=consumers, flags=flags, timeout_us=500000)
    want = L.run(sequential=False, cfg=cfg)
    PC = int(L.ws.view("meta")[9].item())
    xc, hc = L.ws.view("Xc")[:PC].clone(), L.ws.view("Hc")[:PC].clone()
    L.ws.view("Xc").fill_(7)  # rows the dispatch does not write would show
    got = L.run(sequential=False, cfg=tlc.Config.from_workload(L.w, consumer_ctas=consumers, flags=flags | FD,
                                                                timeout_us=500000))
    assert torch.equal(L.ws.view("Xc")[:PC], xc)
    assert torch.equal(L.ws.view("Hc")[:PC], hc)
    assert torch.equal(got, want)
    assert int(L.ws.view("xrows").sum().item()) == PC  # every compact row counted once


@pytest.mark.parametrize("name", ["tiny", "mixtral", "skew", "fine"])
@pytest.mark.parametrize("flags", [tlc.MOE_PAIR_UMMA | tlc.MOE_TAIL_ASSIST, tlc.MOE_TAIL_ASSIST],
                         ids=["pairs", "single"])
def test_fused_dispatch_equals_separate_permute(name, flags):
    compare(Layer(small(name), seed=3), flags)


@pytest.mark.parametrize("shape", [dict(T=8, d=128, ffn=128, E=1, topk=1, R=1, tile_M=64),
                                   dict(T=1000, d=256, ffn=256, E=256, topk=8, R=4, tile_M=128),
                                   dict(T=64, d=384, ffn=128, E=16, topk=1, R=64, tile_M=128)],
                         ids=["one-expert", "E256-k8", "one-token-per-owner"])
def test_fused_dispatch_edge_shapes(shape):
    compare(Layer(inputs.Workload("edge", **shape), seed=4), tlc.MOE_PAIR_UMMA | tlc.MOE_TAIL_ASSIST)


@pytest.mark.parametrize("name", ["mixtral", "skew", "fine"])
def test_fused_dispatch_full_size_in_the_bench_configuration(name):
    import bench
    c, warps = bench.DEFAULT_COPY[name]
    compare(Layer(inputs.WORKLOADS[name], seed=2), bench.default_flags(warps), consumers=c)
