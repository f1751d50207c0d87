"""Failure handling on the GPU without a fault: a bounded device wait that runs out. The
library's self-test kernel waits on an mbarrier phase that nothing completes; the wait gives
up after about a second, records GDR_ERR_TIMEOUT in the workspace status word, and the
context stays usable (a chunked forward afterwards is still correct)."""
import time

import pytest
import torch

import gated_delta_rule_31_gb300 as gdr
import oracle
from gated_delta_rule_31_gb300.synth import Shape, make_inputs
from tests.util import BF16_TOL, cuda_device, rel_err, to_dev

pytestmark = pytest.mark.gpu
TIMEOUT = 5  # GDR_ERR_TIMEOUT


def test_wait_expiry_is_reported_and_the_context_stays_usable():
    dev = cuda_device()
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    t0 = time.perf_counter()
    gdr.selftest_wait_expiry(ws)
    assert gdr.workspace_status(ws) == TIMEOUT  # synchronises: the kernel has returned
    elapsed = time.perf_counter() - t0
    assert 0.2 < elapsed < 20.0, elapsed
    assert gdr.workspace_status(ws) == 0  # read and cleared
    x = make_inputs(Shape(1, 130, 1, 2, 128, 128), dtype=torch.bfloat16, seed=3)
    d = to_dev(x, dev)
    o, ht = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    assert rel_err(o, ro) <= BF16_TOL and rel_err(ht, rht) <= BF16_TOL


def test_wait_expiry_argument_checks():
    dev = cuda_device()
    with pytest.raises(gdr.GdrError):
        gdr.selftest_wait_expiry(torch.empty(128, dtype=torch.uint8, device=dev))
