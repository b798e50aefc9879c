"""The failure path of the pipelines' bounded waits, on the GPU without a fault: a kernel waits on
an mbarrier that nothing completes, gives up after its limit, sets the timeout bit and returns;
the host reads DSA_ERR_TIMEOUT through the error word, and the next calls on the same context
compute correct results."""
import pytest
import torch

import indexer_top_sparse_paged_gb300 as dsa
import workloads as W
from cases import small_spec
from gpu_helpers import Dev, assert_index_parity

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_reports_a_timeout_and_the_context_stays_usable():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    dsa.selftest_wait_timeout(ws)
    bits = dsa.ctypes.c_int32(0)
    st = dsa.lib().dsa_read_error(dsa._p(ws), dsa.ctypes.byref(bits), dsa._stream())
    assert st == 6 and bits.value == 0x4  # DSA_ERR_TIMEOUT, DSA_FAULT_TIMEOUT
    # read_error cleared the word; a second read is clean
    assert dsa.read_error(ws) == 0
    # the context still computes
    case = W.generate(small_spec("bf16", [3000, 700], 256), seed=901)
    dev = Dev(case)
    idx = dev.indexer()
    assert dev.faults() == 0
    assert_index_parity(case, idx)
