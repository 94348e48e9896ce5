"""Failure detection on the GPU without a fault: a bounded device-side wait that nothing completes
runs out, the library reports RELATION_ERR_DEVICE_TIMEOUT through its status word, and the context
stays usable (a normal forward afterwards still matches the oracle)."""
import time

import numpy as np
import pytest
import torch

import oracle
from relation_token_mixing_gb300 import binding as rb
from relation_token_mixing_gb300 import inputs as rin

pytestmark = pytest.mark.gpu

RELATION_ERR_DEVICE_TIMEOUT = 6


def test_expired_wait_is_reported_and_the_context_stays_usable():
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    t0 = time.perf_counter()
    rb.relation_selftest_wait_timeout(100)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert rb.relation_check_device_status() == RELATION_ERR_DEVICE_TIMEOUT
    assert rb.relation_check_device_status() == 0  # reading clears the word
    assert 0.09 <= dt < 5.0, dt                     # it waited its limit, then returned

    w = rin.Workload("after_timeout", 1, 2, 200, 64, torch.bfloat16, 1.0, 0.5, True, 1.0)
    x = rin.make(w)
    Y, L = rb.fwd(x["P1"].cuda(), x["P2"].cuda(), x["V"].cuda(), w.tau_S, w.lam, True)
    torch.cuda.synchronize()
    assert rb.relation_check_device_status() == 0
    Yr, _ = oracle.fwd(x["P1"], x["P2"], x["V"], w.tau_S, w.lam, True)
    vmax = float(x["V"].abs().max())
    assert float(np.max(np.abs(Y.float().cpu().numpy() - Yr))) <= 1e-2 * vmax
