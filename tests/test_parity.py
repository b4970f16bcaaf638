"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Tolerance |o - ref| <= 2e-2 + 2e-2 |ref| (bf16 inputs, fp32 accumulation).
Block-table indexing is checked exactly: every slot the decode query may not
read is NaN (see ``workloads``), -1 pages carry no data at all, and the
device status word must stay 0 (no page outside [0, num_pages) was fetched).
"""

import numpy as np
import pytest
import torch

import paged_decode_attention_gb300 as pda
from workloads import PAGE_SIZE, config_case, make_case

from _helpers import assert_within_tolerance, oracle_full, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def run(case, out_dtype=torch.float32, num_splits=0, status=None, **kw):
    fn = pda.attn_decode_sliding if case.kind == "sliding" else pda.attn_decode_global
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = fn(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, window=case.window,
           max_seq_len=case.max_seq_len, out_dtype=out_dtype, num_splits=num_splits, status=status, **kw)
    torch.cuda.synchronize()
    return o, int(status.item())


def check_case(case, label, num_splits=0, out_dtype=torch.float32, want=None):
    if want is None:
        want = oracle_full(case)
    g = case.to(DEV)
    o, st = run(g, out_dtype=out_dtype, num_splits=num_splits)
    assert st == 0, "%s: device status %d" % (label, st)
    return assert_within_tolerance(o.double().cpu().numpy(), want, label), o


# ---------------------------------------------------------------------------
# the workloads at oracle-friendly sizes, in full
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_tiny_sliding_decode(cuda_lib, out_dtype):
    case = config_case(1)
    check_case(case, "tiny sliding", out_dtype=out_dtype)


def test_global_decode_b8(cuda_lib):
    case = config_case(2)
    check_case(case, "global B=8")


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_edge_lengths(cuda_lib, kind):
    # empty, single position, page edges, window edges, ragged tails
    lens = [0, 1, 2, 15, 16, 17, 31, 32, 33, 1023, 1024, 1025, 1039, 1040, 1041, 2047]
    case = make_case(kind, lens, seed=77)
    err, o = check_case(case, "%s edges" % kind)
    assert torch.all(o[0] == 0)


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_window_only_pages_with_unmapped_prefix(cuda_lib, kind):
    lens = [1024, 1025, 1040, 2047, 3000, 4096, 5000, 17]
    case = make_case(kind, lens, seed=78, window=1024, window_only=True)
    assert (case.block_table[4, :100] == -1).all()
    check_case(case, "%s window-only" % kind)


@pytest.mark.parametrize("window", [1, 7, 16, 100, 1000])
def test_global_with_a_window(cuda_lib, window):
    case = make_case("global", [1, 40, 999, 2100], seed=79, window=window)
    check_case(case, "global w=%d" % window)


@pytest.mark.parametrize("window", [1, 5, 16, 17, 333, 2048])
def test_sliding_other_windows(cuda_lib, window):
    case = make_case("sliding", [1, 40, 999, 2100], seed=80, window=window)
    check_case(case, "sliding w=%d" % window)


# ---------------------------------------------------------------------------
# splits, determinism, output type, paging
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_split_count_does_not_change_the_result(cuda_lib, kind):
    # Sliding: fp32 throughout, so splits only regroup fp32 sums.  Global: P is
    # rounded to bf16 against each split's own running max, so two split
    # counts may differ by up to 2 * 2^-9 * max|v| (|v| <= 8 here).
    tol = dict(rtol=1e-5, atol=1e-6) if kind == "sliding" else dict(rtol=0, atol=2 * 2.0**-9 * 8)
    # Every split count is also held to the oracle at the parity tolerance.
    case = make_case(kind, [3, 700, 1100, 5000], seed=81).to(DEV)
    want = oracle_full(case)
    ref, _ = run(case, num_splits=1)
    assert_within_tolerance(ref.double().cpu().numpy(), want, "%s one split" % kind)
    for ns in (2, 7, 64, 1000):
        o, st = run(case, num_splits=ns)
        assert st == 0
        np.testing.assert_allclose(o.cpu().numpy(), ref.cpu().numpy(), **tol)
        assert_within_tolerance(o.double().cpu().numpy(), want, "%s %d splits" % (kind, ns))


def test_in_grid_merge_matches_the_oracle_and_leaves_its_counters_zero(cuda_lib):
    """Sliding calls whose plan expects few blocks per sequence merge their split
    sequences inside the decode kernel (the last block of each sequence reads
    the others' partials); the others keep the combine kernel.  Either way
    every split count, empty sequences among them, matches the oracle, the
    counters at the head of the workspace are zero again after each call, and a
    workspace whose partial rows hold a previous layout's data gives the same
    output."""
    case = make_case("sliding", [0, 1, 17, 300, 1100, 5000, 0, 2047, 1024, 16], seed=95).to(DEV)
    # one long sequence among empty ones: the plan expects short spans to be rare, and its
    # 65 pages fall on about 17 blocks, whose last one merges them all
    lone = make_case("sliding", [1100] + [0] * 15, seed=96).to(DEV)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    for case, ns in ((case, 0), (case, 3), (case, 40), (case, 300), (case, 1000), (lone, 0)):
        want = oracle_full(case)
        in_grid = pda.attn_decode_launches(pda.KIND_SLIDING, case.B, case.max_seq_len, case.window, ns, sms) == 1
        assert in_grid == (ns <= 40)
        need = pda.attn_decode_workspace_size(pda.KIND_SLIDING, case.B, case.max_seq_len, case.window, ns)
        ws = pda.new_workspace(need, DEV)
        outs = []
        for _ in range(2):  # the second call finds the first one's partial rows in place
            status = torch.zeros(1, dtype=torch.int32, device=DEV)
            o = pda.attn_decode_sliding(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                                        window=case.window, max_seq_len=case.max_seq_len, out_dtype=torch.float32,
                                        workspace=ws, num_splits=ns, status=status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert int(torch.count_nonzero(ws[:pda.WORKSPACE_ZERO_BYTES])) == 0, "counters left nonzero"
            outs.append(o)
        assert torch.equal(outs[0], outs[1])
        assert_within_tolerance(outs[0].double().cpu().numpy(), want, "B=%d, %d splits" % (case.B, ns))
        empty = [b for b, L in enumerate(case.seq_lens_host) if L == 0]
        assert all(torch.all(outs[0][b] == 0) for b in empty)


def test_a_workspace_whose_counters_were_not_zeroed_is_reported(cuda_lib):
    """Counters that start far above zero (a workspace head never zeroed) raise
    ATTN_DEV_INTERNAL instead of going unnoticed; nothing waits on them."""
    lens = torch.randint(1, 3000, (48,), generator=torch.Generator().manual_seed(97)).tolist()
    case = make_case("sliding", lens, seed=98).to(DEV)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert pda.attn_decode_launches(pda.KIND_SLIDING, case.B, case.max_seq_len, case.window, 0, sms) == 1
    need = pda.attn_decode_workspace_size(pda.KIND_SLIDING, case.B, case.max_seq_len, case.window)
    ws = torch.full((need,), 0x7F, dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pda.attn_decode_sliding(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, window=case.window,
                            max_seq_len=case.max_seq_len, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pda.DEV_INTERNAL


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_deterministic_and_bf16_is_rounded_fp32(cuda_lib, kind):
    case = make_case(kind, [5, 300, 1100], seed=82).to(DEV)
    a, _ = run(case)
    b, _ = run(case)
    assert torch.equal(a, b)
    h, _ = run(case, out_dtype=torch.bfloat16)
    assert torch.equal(h, a.to(torch.bfloat16))


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_paging_is_a_relabelling_bitwise(cuda_lib, kind):
    a = make_case(kind, [3, 16, 17, 700, 1500], seed=83)
    P = a.num_pages
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(9))
    b = make_case(kind, [3, 16, 17, 700, 1500], seed=83)
    b.k_pool = torch.empty_like(a.k_pool)
    b.v_pool = torch.empty_like(a.v_pool)
    b.k_pool[perm] = a.k_pool
    b.v_pool[perm] = a.v_pool
    bt = a.block_table.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    b.block_table = bt
    oa, _ = run(a.to(DEV))
    ob, _ = run(b.to(DEV))
    assert torch.equal(oa, ob)


def test_query_head_reads_kv_head_h_over_G(cuda_lib):
    for kind in ("sliding", "global"):
        case = make_case(kind, [37, 1100], seed=84)
        case.q.zero_()
        nan = torch.isnan(case.v_pool)
        for c in range(case.Hkv):
            case.v_pool[:, :, c, :] = float(c + 1)
        case.v_pool[nan] = float("nan")
        o, st = run(case.to(DEV))
        assert st == 0
        G = case.Hq // case.Hkv
        for h in range(case.Hq):
            assert torch.all(o[:, h, :] == float(h // G + 1)), (kind, h)


def test_dominant_logit_selects_its_value_row(cuda_lib):
    for kind in ("sliding", "global"):
        case = make_case(kind, [333], seed=85)
        L, j = 333, 300
        case.q.zero_()
        case.q[0, :, 0] = 64.0
        bt = case.block_table
        nan = torch.isnan(case.k_pool)
        case.k_pool.zero_()
        case.k_pool[nan] = float("nan")
        case.k_pool[bt[0, j // PAGE_SIZE], j % PAGE_SIZE, :, 0] = 64.0
        o, st = run(case.to(DEV))
        assert st == 0
        vj = case.v_pool[bt[0, j // PAGE_SIZE], j % PAGE_SIZE].float()
        G = case.Hq // case.Hkv
        for h in range(case.Hq):
            assert torch.equal(o[0, h].cpu(), vj[h // G]), (kind, h)


def test_shared_k_and_v_pool(cuda_lib):
    case = make_case("global", [50, 600], seed=86)
    case.v_pool = case.k_pool
    check_case(case, "k_pool is v_pool")


def test_non_default_stream_and_preallocated_workspace(cuda_lib):
    case = make_case("global", [4000, 10], seed=87).to(DEV)
    need = pda.attn_decode_workspace_size(pda.KIND_GLOBAL, case.B, case.max_seq_len, 0)
    assert need > 0
    ws = pda.new_workspace(need, DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o = pda.attn_decode_global(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                                   max_seq_len=case.max_seq_len, out_dtype=torch.float32, workspace=ws,
                                   stream=s)
    s.synchronize()
    assert_within_tolerance(o.double().cpu().numpy(), oracle_full(case), "side stream")
    with pytest.raises(pda.AttnDecodeError, match="WORKSPACE"):
        pda.attn_decode_global(case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens,
                               max_seq_len=case.max_seq_len, workspace=ws[: need // 2])


# ---------------------------------------------------------------------------
# device-side contract checks (no fault: out-of-range pages are zero-filled)
# ---------------------------------------------------------------------------

def test_out_of_range_page_id_is_flagged_not_read(cuda_lib):
    for kind in ("sliding", "global"):
        case = make_case(kind, [100, 40], seed=88).to(DEV)
        case.block_table[0, 2] = -1
        case.block_table[1, 0] = case.num_pages + 5
        _, st = run(case)
        assert st & pda.DEV_BAD_PAGE


def test_seq_len_beyond_block_table_is_flagged_and_clamped(cuda_lib):
    case = make_case("global", [40, 40], seed=89).to(DEV)
    case.seq_lens[1] = case.max_blocks * PAGE_SIZE + 100
    case.seq_lens_host[1] = case.max_blocks * PAGE_SIZE
    _, st = run(case)
    assert st & pda.DEV_BAD_SEQ_LEN


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times:
# sampled rows against the oracle
# ---------------------------------------------------------------------------

def _full_size(case, n_rows, seed, label):
    o, st = run(case)
    assert st == 0, "%s: device status %d" % (label, st)
    rows = sample_rows(case, n_rows, seed)
    want = oracle_rows(case, rows)
    got = o.reshape(-1, case.D)[rows].double().cpu().numpy()
    return assert_within_tolerance(got, want, label)


@pytest.mark.slow
def test_sliding_b256_window_only_full_size(cuda_lib):
    case = config_case(3, device=DEV)
    _full_size(case, 96, 1, "sliding B=256")


@pytest.mark.slow
@pytest.mark.parametrize("variant", [None, "b"])
def test_long_context_global_full_size(cuda_lib, variant):
    case = config_case(4, device=DEV, variant=variant)
    _full_size(case, 24, 2, "global long %s" % variant)


@pytest.mark.slow
@pytest.mark.parametrize("layer", [4, 5])
def test_decode_step_mix_layers_full_size(cuda_lib, layer):
    case = config_case(5, device=DEV, layer=layer)
    _full_size(case, 48, 3, "mix layer %d" % layer)


def test_prepared_call_matches_the_one_shot_call(cuda_lib):
    for kind in ("sliding", "global"):
        case = make_case(kind, [17, 1500, 300], seed=92).to(DEV)
        ref, _ = run(case)
        prep = (pda.prepare_decode_sliding if kind == "sliding" else pda.prepare_decode_global)(
            case.q, case.k_pool, case.v_pool, case.block_table, case.seq_lens, window=case.window,
            max_seq_len=case.max_seq_len, out_dtype=torch.float32)
        s = torch.cuda.Stream()
        for _ in range(2):  # a prepared call is reusable
            o = prep.run(s)
            s.synchronize()
            assert torch.equal(o, ref)
