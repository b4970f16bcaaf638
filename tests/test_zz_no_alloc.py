"""attn_decode_sliding_noalloc: the sliding-window decode for callers that
cannot allocate device memory (no workspace argument; the library's own
built-in scratch array holds the partial results).

Called through the C ABI with ctypes, twice in a row on different inputs (the
second call runs on whatever the first left in the shared scratch), and
compared both with the fp64 oracle and with attn_decode_sliding given a
workspace, within the parity tolerance of the other tests.  A call with many
forced splits followed by one with the automatic plan checks that a call
never reads partial rows left by an earlier call's layout; the same kernels
given a workspace whose partial rows are NaN check that only the counters at
its head need to start at zero.  This file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

import paged_decode_attention_gb300 as pda
from workloads import make_case

from _helpers import ATOL, RTOL, assert_within_tolerance, oracle_full

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _noalloc(lib):
    fn = lib.attn_decode_sliding_noalloc
    fn.restype = ctypes.c_int32
    c_i32, c_i64, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    fn.argtypes = [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,       # q k_pool v_pool block_table seq_lens o
                   c_i32, c_i32, c_i64, c_i32, c_i32, c_i32,  # batch max_blocks num_pages max_seq_len window out_dtype
                   c_i32, c_vp, c_vp]                         # num_splits status stream
    return fn


def _call_noalloc(fn, case, o, status, num_splits=0):
    stream = torch.cuda.current_stream(DEV).cuda_stream
    return fn(case.q.data_ptr(), case.k_pool.data_ptr(), case.v_pool.data_ptr(),
              case.block_table.data_ptr(), case.seq_lens.data_ptr(), o.data_ptr(),
              case.B, case.max_blocks, case.num_pages, case.max_seq_len, case.window,
              1 if o.dtype == torch.float32 else 0, num_splits, status.data_ptr(), stream)


def test_noalloc_matches_the_workspace_entry_point_on_two_calls(cuda_lib):
    fn = _noalloc(pda.load())
    cases = [make_case("sliding", [1, 17, 300, 1100, 5000, 0, 2047], seed=901).to(DEV),
             make_case("sliding", [2048, 33, 1024, 7, 4096], seed=902, window_only=True).to(DEV)]
    for i, case in enumerate(cases):
        ref = pda.attn_decode_sliding(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                                      window=case.window, max_seq_len=case.max_seq_len,
                                      out_dtype=torch.float32)
        o = torch.full_like(ref, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        st = _call_noalloc(fn, case, o, status)
        assert st == 0, pda.attn_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got, want = o.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.isfinite(got).all(), "call %d" % i
        assert np.all(np.abs(got - want) <= ATOL + RTOL * np.abs(want)), "call %d" % i
        assert_within_tolerance(got, oracle_full(case), "no-alloc call %d against the oracle" % i)


def test_noalloc_after_a_call_with_another_split_layout(cuda_lib):
    """Many forced splits leave partial rows all over the scratch; the next
    calls (automatic plan, other lengths; split sequences merged inside the
    decode kernel, with its arrival counters in the scratch, then by the
    combine kernel) must not read any of them."""
    fn = _noalloc(pda.load())
    first = make_case("sliding", [1100, 3000, 17, 2500], seed=904).to(DEV)
    lens = torch.randint(1, 3000, (48,), generator=torch.Generator().manual_seed(907)).tolist()
    second = make_case("sliding", lens, seed=905).to(DEV)
    third = make_case("sliding", [5, 1024, 1500, 40, 777, 2049], seed=908).to(DEV)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    launches = [pda.attn_decode_launches(pda.KIND_SLIDING, c.B, c.max_seq_len, c.window, ns, sms)
                for c, ns in ((first, 200), (second, 0), (third, 0))]
    assert launches == [2, 1, 2]
    for case, ns in ((first, 200), (second, 0), (third, 0)):
        o = torch.full((case.B, 16, 256), float("nan"), dtype=torch.float32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        assert _call_noalloc(fn, case, o, status, num_splits=ns) == 0, pda.attn_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_within_tolerance(o.double().cpu().numpy(), oracle_full(case), "no-alloc, %d splits" % ns)


def test_the_kernels_read_only_rows_their_call_wrote(cuda_lib):
    """The workspace entry point given a workspace whose partial rows are NaN
    (the kernels the no-alloc entry point runs): a read of any row this call
    did not write would turn the output into NaN."""
    case = make_case("sliding", [1, 17, 300, 1100, 5000, 0, 2047], seed=906).to(DEV)
    for ns in (0, 64):
        ws_bytes = pda.attn_decode_workspace_size(pda.KIND_SLIDING, case.B, case.max_seq_len, case.window, ns)
        ws = torch.full(((ws_bytes + 3) // 4,), float("nan"), dtype=torch.float32, device=DEV).view(torch.uint8)
        ws[:pda.WORKSPACE_ZERO_BYTES].zero_()  # the arrival counters; the partial rows stay NaN
        o = pda.attn_decode_sliding(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                                    window=case.window, max_seq_len=case.max_seq_len, out_dtype=torch.float32,
                                    workspace=ws, num_splits=ns)
        torch.cuda.synchronize()
        assert_within_tolerance(o.double().cpu().numpy(), oracle_full(case), "NaN workspace, %d splits" % ns)


def test_noalloc_rejects_a_plan_beyond_its_scratch(cuda_lib):
    fn = _noalloc(pda.load())
    case = make_case("sliding", [1024] * 256, seed=903, window_only=True).to(DEV)
    o = torch.empty((256, 16, 256), dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    # 1024 blocks per KV head need (1024 + 256) * 16 rows of partials: more than 8 MiB
    st = _call_noalloc(fn, case, o, status, num_splits=1024)
    assert st == 2  # ATTN_ERR_UNSUPPORTED
    assert "scratch" in pda.attn_last_error()
