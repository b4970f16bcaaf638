"""Failure detection without a GPU fault.

Every wait of the decode kernels' copy pipeline has a time limit; when it
runs out the kernel raises ATTN_DEV_WAIT_TIMEOUT in the caller's status word
and winds down instead of hanging.  Here a wait is made to run out on a
barrier that nothing arrives at (attn_selftest_wait_timeout), and the CUDA
context must still serve a normal decode call afterwards.  Contract
violations on the device (bad page ids, bad lengths) are covered in
test_parity.py; host-side argument errors in test_boundary.py.
"""

import ctypes
import time

import pytest
import torch

import paged_decode_attention_gb300 as pda
from workloads import make_case

from _helpers import assert_within_tolerance, oracle_full

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def test_a_wait_that_runs_out_reports_a_timeout_and_leaves_the_context_usable(cuda_lib):
    lib = pda.load()
    fn = lib.attn_selftest_wait_timeout
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.perf_counter()
    assert fn(status.data_ptr(), torch.cuda.current_stream(DEV).cuda_stream) == 0
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == pda.DEV_WAIT_TIMEOUT
    assert 0.5 < waited < 30.0  # the 1 s limit ran out; nothing hung
    # the context still works
    case = make_case("global", [5, 700], seed=991)
    g = case.to(DEV)
    status.zero_()
    o = pda.attn_decode_global(g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                               max_seq_len=g.max_seq_len, out_dtype=torch.float32, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_within_tolerance(o.double().cpu().numpy(), oracle_full(case), "after timeout")


def test_selftest_rejects_a_missing_status_word(cuda_lib):
    fn = pda.load().attn_selftest_wait_timeout
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert fn(None, None) == 1
