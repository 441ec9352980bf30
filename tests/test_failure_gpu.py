"""Failure detection on the GPU without a fault: a bounded device wait that expires
(on a barrier nothing completes) raises the sticky status word, the host reads
HLA_ERR_TIMEOUT from hla_sync_status once, and the context stays usable."""
import numpy as np
import pytest
import torch

import causal_prefix_scan_gb300 as hla
import oracle
from causal_prefix_scan_gb300 import workloads as W
from gpu_helpers import TOL_BF16, assert_parity, run_forward, run_oracle

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_once_and_context_survives():
    hla.hla_sync_status()  # clean start
    stream = torch.cuda.Stream()
    hla.hla_selftest_expired_wait(stream)
    with pytest.raises(hla.HlaError) as ei:
        hla.hla_sync_status(stream)
    assert ei.value.status == hla.HLA_ERR_TIMEOUT
    hla.hla_sync_status(stream)  # reported once, then clear
    # the context still computes correctly
    w = W.Workload("after_timeout", 1, 2, 200, 64, 64, 64, "bf16", "l2", seed=51)
    x = W.make_inputs(w)
    o, st = run_forward(x, "bf16", 64)
    o_ref, st_ref = run_oracle(x)
    assert_parity(o, o_ref, st, st_ref, tol=TOL_BF16, what="forward after an expired wait")
