"""Failure detection without a GPU fault: a wait that nothing completes runs
into its limit, the kernel reports DSA_DEVERR_TIMEOUT and returns, and the
context keeps working (a real call afterwards matches the oracle)."""

import time

import numpy as np
import pytest

import oracle
from deepseek_v4_top_gb300 import inputs as I

from gpu_helpers import compare, run

pytestmark = pytest.mark.gpu


def test_a_wait_that_nothing_completes_reports_a_timeout():
    import __graft_entry__
    __graft_entry__.build()
    import torch
    from deepseek_v4_top_gb300 import dsa
    torch.cuda.set_device(0)
    assert dsa.dsa_get_device_error() == 0
    t0 = time.time()
    dsa.dsa_selftest_wait_limit()
    code = dsa.dsa_get_device_error()          # synchronises: the kernel has returned
    waited = time.time() - t0
    assert code == dsa.DSA_DEVERR_TIMEOUT
    assert 1.0 < waited < 30.0
    assert dsa.dsa_get_device_error() == 0     # the word was cleared by the read
    case = I.prefill(rows=8, N=1024, first_pos=900)
    got, code = run(case)
    assert code == 0
    ref, _ = oracle.attn(case)
    compare(case, got, ref)
