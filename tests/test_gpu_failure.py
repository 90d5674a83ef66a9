"""Failure detection on the GPU without a fault: every wait in the kernels is a bounded
mbarrier poll that records WQ_ERR_TIMEOUT and returns.  wq_selftest_timeout runs that path on a
barrier nothing arrives on; the status is reported once, and the context stays usable."""
import pytest
import torch

from bit_weight_quantized_matmul_gb300 import workloads as wl
from oracle import linear as L
from oracle import quant as Q
from tests.gpu_common import wq, need_gpu, REL_L2_TOL
from tests.helpers import rel_l2

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    need_gpu()
    m = wq()
    assert m.last_device_status() == 0
    m.selftest_timeout(2000)
    assert m.last_device_status() == m.WQ_ERR_TIMEOUT
    assert m.last_device_status() == 0  # read once, then cleared
    # the context still runs the hot path correctly
    N, K, M = 256, 512, 4
    W = wl.weight(7, N, K)
    packed, scales = m.pack("nf4", torch.from_numpy(W).cuda())
    x = wl.activations(7, M, K)
    y = m.linear(x.cuda(), packed, scales, "nf4", N, K)
    torch.cuda.synchronize()
    assert m.last_device_status() == 0
    want = L.linear_w4a16(wl.bf16_as_f32(x), Q.PACK["nf4"](W), None)
    assert rel_l2(y.float().cpu().numpy(), want) <= REL_L2_TOL


def test_selftest_rejects_bad_poll_counts():
    need_gpu()
    m = wq()
    for polls in (0, (1 << 20) + 1):
        with pytest.raises(m.WQError):
            m.selftest_timeout(polls)
