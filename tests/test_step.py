"""A whole decode step recorded once and launched as one CUDA graph
(attn_step_*), through the C ABI.

The graph replays the very kernels of the direct calls with the same
arguments, so its outputs must equal the direct calls' outputs bitwise, and
the direct calls are themselves checked against the oracle elsewhere.  The
step is launched again after its inputs change in place, on a side stream,
and with a bad page id.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_gb300 as pda
from workloads import PAGE_SIZE, bits, key_weight, make_append_case, make_case

from _helpers import assert_within_tolerance, oracle_full

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _layer_inputs(seed):
    """One sliding layer (append, then decode over the appended cache), one
    global layer and one global layer over a values-only cache."""
    positions = [0, 16, 333, 1023, 1024, 2500]
    app = make_append_case("sliding", positions, seed=seed, full_cache=True).to(DEV)
    seq_lens = torch.tensor([p + 1 for p in positions], dtype=torch.int32, device=DEV)
    glob = make_case("global", [17, 700, 3000], seed=seed + 1).to(DEV)
    shared = make_case("global", [1, 1500, 4097], seed=seed + 2).to(DEV)
    w_k = key_weight(512, seed + 3, device=DEV)
    return app, seq_lens, glob, shared, w_k


def _record(step, app, seq_lens, glob, shared, w_k, status):
    c = app.cache
    q = step.add_kv_append_sliding(app.qkv, app.w_q, app.w_k, c.block_table, app.positions, c.k_pool, c.v_pool,
                                   status=status)
    o1 = step.add_decode_sliding(q, c.k_pool, c.v_pool, c.block_table, seq_lens, window=c.window,
                                 out_dtype=torch.float32, status=status)
    o2 = step.add_decode_global(glob.q, glob.k_pool, glob.v_pool, glob.block_table, glob.seq_lens,
                                max_seq_len=glob.max_seq_len, out_dtype=torch.float32, status=status)
    o3 = step.add_decode_global_shared(shared.q, shared.v_pool, w_k, shared.block_table, shared.seq_lens,
                                       max_seq_len=shared.max_seq_len, out_dtype=torch.float32, status=status)
    return o1, o2, o3


def _direct(app, seq_lens, glob, shared, w_k, status):
    c = app.cache
    q = pda.attn_kv_append_sliding(app.qkv, app.w_q, app.w_k, c.block_table, app.positions, c.k_pool, c.v_pool,
                                   status=status)
    o1 = pda.attn_decode_sliding(q, c.k_pool, c.v_pool, c.block_table, seq_lens, window=c.window,
                                 out_dtype=torch.float32, status=status)
    o2 = pda.attn_decode_global(glob.q, glob.k_pool, glob.v_pool, glob.block_table, glob.seq_lens,
                                max_seq_len=glob.max_seq_len, out_dtype=torch.float32, status=status)
    o3 = pda.attn_decode_global_shared(shared.q, shared.v_pool, w_k, shared.block_table, shared.seq_lens,
                                       max_seq_len=shared.max_seq_len, out_dtype=torch.float32, status=status)
    torch.cuda.synchronize()
    return o1, o2, o3


@pytest.mark.parametrize("mode", ["graph", "direct", "auto"])
def test_step_equals_the_direct_calls_bitwise(cuda_lib, mode):
    a = _layer_inputs(1300)
    b = _layer_inputs(1300)  # the same inputs, for the direct calls
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    step = pda.Step()
    outs = _record(step, *a, status)
    # append 1, sliding decode 1 or 2 (the plan's choice), global decodes 2 each
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    c = a[0].cache
    sliding = pda.attn_decode_launches(pda.KIND_SLIDING, c.B, c.max_blocks * PAGE_SIZE, c.window, 0, sms)
    assert step.num_calls == 4 and step.num_kernels == 1 + sliding + 2 + 2
    for o in outs:  # recording and finalizing launch nothing
        o.fill_(7.0)
    torch.cuda.synchronize()
    step.finalize(mode)
    torch.cuda.synchronize()
    assert all(torch.all(o == 7.0) for o in outs)
    # six or seven kernels: auto takes the graph
    assert step.launch_mode == ("graph" if mode == "auto" else mode)
    step.launch()
    torch.cuda.synchronize()
    want = _direct(*b, torch.zeros(1, dtype=torch.int32, device=DEV))
    assert int(status.item()) == 0
    for got, ref in zip(outs, want):
        assert torch.equal(got, ref)
    # the appended cache rows too
    assert torch.equal(a[0].cache.k_pool, b[0].cache.k_pool) and torch.equal(a[0].cache.v_pool, b[0].cache.v_pool)
    # and the global call against the oracle
    assert_within_tolerance(outs[1].double().cpu().numpy(), oracle_full(a[2].to("cpu")), "step global")
    step.close()


@pytest.mark.parametrize("mode", ["graph", "direct"])
def test_step_follows_inputs_changed_in_place(cuda_lib, mode):
    app, seq_lens, glob, shared, w_k = _layer_inputs(1310)
    other = make_case("global", [17, 700, 3000], seed=1399).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    step = pda.Step()
    _, o2, o3 = _record(step, app, seq_lens, glob, shared, w_k, status)
    step.finalize(mode)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step.launch(s)
    s.synchronize()
    first = o2.clone()
    # next step: a new query in the same buffer, one sequence one token shorter
    glob.q.copy_(other.q)
    glob.seq_lens[2] -= 1
    step.launch(s)
    s.synchronize()
    want = pda.attn_decode_global(glob.q, glob.k_pool, glob.v_pool, glob.block_table, glob.seq_lens,
                                  max_seq_len=glob.max_seq_len, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o2, want) and not torch.equal(o2, first)
    assert int(status.item()) == 0
    step.close()


@pytest.mark.parametrize("mode", ["graph", "direct"])
def test_step_reports_device_status(cuda_lib, mode):
    case = make_case("global", [100, 40], seed=1320).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    step = pda.Step()
    step.add_decode_global(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, status=status)
    step.finalize(mode)
    step.launch()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    case.block_table[1, 0] = case.num_pages + 5
    step.launch()
    torch.cuda.synchronize()
    assert int(status.item()) & pda.DEV_BAD_PAGE
    step.close()


def test_step_rejects_calls_after_finalize(cuda_lib):
    case = make_case("global", [40], seed=1330).to(DEV)
    step = pda.Step()
    step.add_decode_global(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens)
    step.finalize()
    with pytest.raises(pda.AttnDecodeError, match="finalized"):
        step.add_decode_global(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens)
    with pytest.raises(pda.AttnDecodeError, match="WORKSPACE"):
        pda.Step().add_decode_global(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                                     workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    step.close()


def test_step_with_a_values_only_global_layer(cuda_lib):
    """A global layer over a values-only cache inside a step: the append writes V only and the
    decode rebuilds the keys; both match the direct calls bitwise and the oracle's append and decode."""
    positions = [0, 16, 333, 1023, 1024, 2500]
    a = make_append_case("global", positions, seed=1340, full_cache=True).to(DEV)
    b = make_append_case("global", positions, seed=1340, full_cache=True).to(DEV)
    seq_lens = torch.tensor([p + 1 for p in positions], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    step = pda.Step()
    q = step.add_kv_append_global(a.qkv, a.w_q, a.w_k, a.cache.block_table, a.positions, None, a.cache.v_pool,
                                  status=status)
    o = step.add_decode_global_shared(q, a.cache.v_pool, a.w_k, a.cache.block_table, seq_lens,
                                      out_dtype=torch.float32, status=status)
    step.finalize()
    step.launch()
    qb = pda.attn_kv_append_global(b.qkv, b.w_q, b.w_k, b.cache.block_table, b.positions, None, b.cache.v_pool)
    ob = pda.attn_decode_global_shared(qb, b.cache.v_pool, b.w_k, b.cache.block_table, seq_lens,
                                       out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(q, qb) and torch.equal(a.cache.v_pool, b.cache.v_pool) and torch.equal(o, ob)
    want = oracle.decode_paged_shared(bits(q), bits(a.cache.v_pool), bits(a.w_k), a.cache.block_table.cpu().numpy(),
                                      seq_lens.cpu().numpy(), 0, 1.0e6, 64)
    assert_within_tolerance(o.double().cpu().numpy(), want, "step values-only layer")
    step.close()


def test_one_call_step_launches_directly_back_to_back(cuda_lib):
    """A one-call step takes the direct mode by default; many launches in a row,
    with the inputs rotating between two buffers, equal the direct calls each time."""
    cases = [make_case("global", [5, 700, 2049, 8192], seed=1350 + i).to(DEV) for i in range(2)]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    steps, outs = [], []
    for c in cases:
        st = pda.Step()
        outs.append(st.add_decode_global(c.q, c.k_pool, c.v_pool, c.block_table, c.seq_lens,
                                         max_seq_len=c.max_seq_len, out_dtype=torch.float32, status=status))
        st.finalize()
        assert st.launch_mode == "direct"
        steps.append(st)
    want = [pda.attn_decode_global(c.q, c.k_pool, c.v_pool, c.block_table, c.seq_lens, max_seq_len=c.max_seq_len,
                                   out_dtype=torch.float32) for c in cases]
    s = torch.cuda.Stream()
    for _ in range(3):
        for k in range(20):
            steps[k % 2].launch(s)
        s.synchronize()
        assert int(status.item()) == 0
        for got, ref in zip(outs, want):
            assert torch.equal(got, ref)
    for st in steps:
        st.close()
