"""SM clock counters of the expert-GEMM launches (trace slots 8-11).

CTA 0 of each GEMM launch adds its SM's cycle count and the global-timer nanoseconds of one span (from
the end of its wait for the previous kernel to the end of its tiles) to a pair of counters that the
plan kernel leaves alone, so they sum over calls until the caller zeroes them. Bar: untouched by a
plan-only call; after layers, both GEMMs' counters grow with every call and their ratio is a clock the
part can run at, for the CTA-pair, single-CTA and fused-GEMM launches, overlapped and sequential.
"""
import pytest
import torch

import tile_level_copy_gb300 as tlc
from tests.gpu_util import Layer, small

pytestmark = pytest.mark.gpu

CONFIGS = [(4, tlc.MOE_PAIR_UMMA | tlc.MOE_TAIL_ASSIST | tlc.MOE_DIRECT_TAIL | tlc.MOE_PDL),
           (8, tlc.MOE_TAIL_ASSIST), (4, tlc.MOE_PAIR_UMMA | tlc.MOE_FUSED_GEMMS)]
SLOTS = slice(tlc.TRACE_UP_CYCLES, tlc.TRACE_DOWN_NS + 1)


def counters(ws):
    return [int(v) for v in ws.view("trace")[SLOTS].cpu()]


@pytest.mark.parametrize("consumers,flags", CONFIGS, ids=["pairs", "single", "fused-gemms"])
@pytest.mark.parametrize("sequential", [False, True], ids=["overlapped", "sequential"])
def test_clock_counters(consumers, flags, sequential):
    L = Layer(small("mixtral"), seed=3)
    cfg = tlc.Config.from_workload(L.w, consumer_ctas=consumers, flags=flags)
    L.run(sequential=sequential, cfg=cfg)  # warm-up
    L.ws.view("trace")[SLOTS].zero_()
    tlc.plan(cfg, L.logits, L.x, L.ws)
    torch.cuda.synchronize()
    assert counters(L.ws) == [0, 0, 0, 0]
    prev = [0, 0, 0, 0]
    fused = bool(flags & tlc.MOE_FUSED_GEMMS) and not sequential
    for _ in range(3):
        L.run(sequential=sequential, cfg=cfg)
        now = counters(L.ws)
        up_c, up_ns, dn_c, dn_ns = now
        assert up_c > prev[0] and up_ns > prev[1]
        if fused:  # one launch for both GEMMs: its span counts as the SwiGLU GEMM's
            assert dn_c == 0 and dn_ns == 0
        else:
            assert dn_c > prev[2] and dn_ns > prev[3]
        prev = now
    for c, ns in ((prev[0], prev[1]), (prev[2], prev[3])):
        if ns:
            assert 200.0 < 1000.0 * c / ns < 2600.0, (c, ns)
