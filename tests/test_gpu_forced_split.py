"""The layer under schedules planned for other SM counts.

The K-split plan depends on the SM count: each count gives other CTA ranges,
other contributors per 128-row tile and so another summation order in the
fixed-order reduction.  Every such order is a correct result (the tolerance
of the layer covers any order of the fp32 sums), and each is reproducible bit
for bit.  Run through a test hook of the library that plans for a given SM
count; CTAs beyond the device's capacity run in later waves, which the
schedule allows because no CTA ever waits for another.
"""
import ctypes

import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
from fp8_block_scaled_token_gb300 import synth
from tests.gpu_helpers import Ran, check_y, oracle_layer

pytestmark = pytest.mark.gpu

SM_COUNTS = (1, 37, 76, 152, 300)


def ws_size(M, N, K, sms):
    sz = ctypes.c_size_t(0)
    rc = fb.lib().fp8bs_testhook_workspace_size_sms(M, N, K, sms, ctypes.byref(sz))
    assert rc == 0, fb.status_string(rc)
    return sz.value


def fused_sms(x, wq, ws, y, work, N, sms, flags=0):
    M, K = x.shape
    rc = fb.lib().fp8bs_testhook_gemm_fused_sms(x.data_ptr(), x.stride(0), wq.data_ptr(), ws.data_ptr(),
                                                y.data_ptr(), M, N, K, work.data_ptr(), work.numel(), flags, sms,
                                                torch.cuda.current_stream().cuda_stream)
    assert rc == 0, fb.status_string(rc)


@pytest.mark.parametrize("M,N,K", [(8, 5120, 5120), (1, 5120, 5120), (13, 300, 1280), (64, 1024, 2048),
                                   (8, 256, 512)])
def test_forced_sm_counts_within_tolerance_and_reproducible(M, N, K):
    x_cpu = synth.activations(M, K, seed=M + 900, outlier_p=0.001)
    w_cpu = synth.weights(N, K, seed=M + 901, outlier_p=0.01)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w, tiled=True)
    ref = oracle_layer(x_cpu, w_cpu)
    outs = {}
    for sms in SM_COUNTS:
        work = fb.make_workspace(ws_size(M, N, K, sms))
        ys = []
        for _ in range(3):
            y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            with Ran() as r:
                fused_sms(x, wq, ws, y, work, N, sms, fb.FLAG_WEIGHTS_TILED)
            assert sum(r.launched().values()) in (1, 2)
            ys.append(y)
        for y in ys[1:]:
            assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16)), "sms=%d not reproducible" % sms
        check_y(ys[0], ref["y"], ref["bound"], "M=%d N=%d K=%d sms=%d" % (M, N, K, sms))
        assert fb.workspace_status(work) == 0
        s = fb.gemm_schedule(M, N, K, sms)
        counters = work[1024:1024 + 4 * s["token_tiles"] * ((N + 127) // 128)]
        assert not counters.any(), "arrival counters must be back at zero"
        outs[sms] = ys[0]
    # the device's own SM count gives exactly the public entry point's result
    dev_sms = torch.cuda.get_device_properties(0).multi_processor_count
    if dev_sms in outs:
        y_pub = fb.fp8_blockscaled_gemm_fused(x, wq, ws, n=N)
        torch.cuda.synchronize()
        assert torch.equal(y_pub.view(torch.int16), outs[dev_sms].view(torch.int16))
