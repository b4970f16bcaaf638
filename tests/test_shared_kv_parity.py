"""Decode over a values-only global cache (attn_decode_global_shared) vs the
fp64 oracle (``oracle.decode_paged_shared``), through the C ABI.

The cache holds V only; the kernel rebuilds each visible key as
bf16(rope(V * w_k)) (Gemma-4-12B model page, "What to watch for": values =
keys).  The oracle rebuilds it in fp64 with one rounding, so a rebuilt key may
sit one bf16 step away from the oracle's; the outputs are compared with the
decode tolerance |o - ref| <= 2e-2 + 2e-2 |ref|.  Every slot the query may not
read is NaN, so a key rebuilt from the wrong slot, or a rotation at the wrong
position, shows.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_gb300 as pda
from workloads import GLOBAL, PAGE_SIZE, ROPE, DecodeCase, bits, config_case, key_weight, make_append_case, make_case

from _helpers import assert_within_tolerance, sample_rows

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
THETA, PAIRS = ROPE["global"]["theta"], ROPE["global"]["pairs"]


def run(case, w_k, out_dtype=torch.float32, num_splits=0, status=None):
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = pda.attn_decode_global_shared(case.q, case.v_pool, w_k.to(DEV), case.block_table, case.seq_lens,
                                      window=case.window, max_seq_len=case.max_seq_len, out_dtype=out_dtype,
                                      num_splits=num_splits, status=status)
    torch.cuda.synchronize()
    return o, int(status.item())


def oracle_shared(case, w_k, rows=None):
    return oracle.decode_paged_shared(bits(case.q), bits(case.v_pool), bits(w_k), case.block_table.cpu().numpy(),
                                      case.seq_lens.cpu().numpy(), case.window, THETA, PAIRS, rows=rows, threads=16)


def check(case, w_k, label, **kw):
    g = case.to(DEV)
    o, st = run(g, w_k, **kw)
    assert st == 0, "%s: device status %d" % (label, st)
    want = oracle_shared(case, w_k)
    return assert_within_tolerance(o.double().cpu().numpy(), want, label), o


def test_edge_lengths(cuda_lib):
    lens = [0, 1, 2, 15, 16, 17, 31, 32, 33, 1023, 1024, 1025, 1039, 1040, 1041, 2047]
    case = make_case("global", lens, seed=1201)
    _, o = check(case, key_weight(512, 1), "edges")
    assert torch.all(o[0] == 0)


def test_global_decode_b8_workload(cuda_lib):
    check(config_case(2), key_weight(512, 2), "global B=8")


@pytest.mark.parametrize("window", [1, 7, 16, 100, 1000])
def test_with_a_window(cuda_lib, window):
    case = make_case("global", [1, 40, 999, 2100], seed=1203, window=window)
    check(case, key_weight(512, 3), "window %d" % window)


@pytest.mark.parametrize("num_splits", [1, 3, 64, 1000])
def test_forced_splits(cuda_lib, num_splits):
    case = make_case("global", [3, 700, 1100, 5000], seed=1204)
    check(case, key_weight(512, 4), "splits %d" % num_splits, num_splits=num_splits)


def test_bf16_output_is_the_rounded_fp32_output(cuda_lib):
    case = make_case("global", [5, 300, 1100], seed=1205).to(DEV)
    w = key_weight(512, 5)
    a, _ = run(case, w)
    b, _ = run(case, w)
    assert torch.equal(a, b)
    h, _ = run(case, w, out_dtype=torch.bfloat16)
    assert torch.equal(h, a.to(torch.bfloat16))


def test_unit_weight_reads_v_as_keys_beyond_the_rotated_dims(cuda_lib):
    # w_k = 1 and q zero outside dims [64, 256) + [320, 512): the logits are
    # <q, V> over unrotated dims only, so the result equals the separate-cache
    # decode with k_pool = v_pool (bitwise: the same bf16 operands and order
    # of MMAs are not guaranteed, so within a tight bound)
    case = make_case("global", [40, 1500, 777], seed=1206)
    case.q[:, :, :64] = 0
    case.q[:, :, 256:320] = 0
    g = case.to(DEV)
    ones = torch.ones(512, dtype=torch.bfloat16)
    o, st = run(g, ones)
    assert st == 0
    ref = pda.attn_decode_global(g.q, g.v_pool, g.v_pool, g.block_table, g.seq_lens, out_dtype=torch.float32)
    torch.cuda.synchronize()
    np.testing.assert_allclose(o.cpu().numpy(), ref.cpu().numpy(), rtol=0, atol=2 * 2.0 ** -9 * 8)


def test_matches_the_separate_cache_with_the_oracles_keys(cuda_lib):
    # the oracle's rebuilt keys fed to attn_decode_global: both paths agree
    case = make_case("global", [17, 2000, 4097], seed=1207)
    w = key_weight(512, 7)
    k = oracle.rebuild_keys(bits(case.v_pool), bits(w), case.block_table.numpy(), case.seq_lens.numpy(), 0, THETA,
                            PAIRS)
    g = case.to(DEV)
    k_dev = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).to(DEV)
    sep = pda.attn_decode_global(g.q, k_dev, g.v_pool, g.block_table, g.seq_lens, out_dtype=torch.float32)
    o, st = run(g, w)
    assert st == 0
    want = oracle_shared(case, w)
    assert_within_tolerance(sep.double().cpu().numpy(), want, "separate cache, oracle keys")
    assert_within_tolerance(o.double().cpu().numpy(), want, "values-only cache")


def test_paging_is_a_relabelling_bitwise(cuda_lib):
    lens = [3, 16, 17, 700, 1500]
    a = make_case("global", lens, seed=1208)
    perm = torch.randperm(a.num_pages, generator=torch.Generator().manual_seed(9))
    v = torch.empty_like(a.v_pool)
    v[perm] = a.v_pool
    bt = a.block_table.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    b = DecodeCase("global", a.q, a.k_pool, v, bt, a.seq_lens, a.window, a.seq_lens_host)
    w = key_weight(512, 8)
    oa, _ = run(a.to(DEV), w)
    ob, _ = run(b.to(DEV), w)
    assert torch.equal(oa, ob)


def test_out_of_range_page_is_flagged(cuda_lib):
    case = make_case("global", [100, 40], seed=1209).to(DEV)
    case.block_table[0, 2] = -1
    case.block_table[1, 0] = case.num_pages + 5
    _, st = run(case, key_weight(512, 9))
    assert st & pda.DEV_BAD_PAGE


def test_argument_validation(cuda_lib):
    case = make_case("global", [40], seed=1210).to(DEV)
    with pytest.raises(ValueError):
        pda.attn_decode_global_shared(case.q, case.v_pool, torch.ones(256, dtype=torch.bfloat16, device=DEV),
                                      case.block_table, case.seq_lens)
    lib = pda.load()
    o = torch.empty((1, 16, 512), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    rc = lib.attn_decode_global_shared(case.q.data_ptr(), case.v_pool.data_ptr(), None,
                                       case.block_table.data_ptr(), case.seq_lens.data_ptr(), o.data_ptr(), 1,
                                       case.block_table.shape[1], case.num_pages, 40, 0, pda.OUT_BF16, 0,
                                       ws.data_ptr(), ws.numel(), None, None)
    assert rc == 1 and "w_k" in pda.attn_last_error()


def test_values_only_append_then_decode(cuda_lib):
    """attn_kv_append_global with k_pool = None writes the same V rows as with
    a key pool, and the values-only decode over them matches the oracle's
    append followed by its values-only decode."""
    positions = [0, 16, 333, 1023, 1024, 2500]
    case = make_append_case("global", positions, seed=1211, full_cache=True)
    g = case.to(DEV)
    v_only = g.cache.v_pool.clone()
    q = pda.attn_kv_append_global(g.qkv, g.w_q, g.w_k, g.cache.block_table, g.positions, None, v_only)
    q2 = pda.attn_kv_append_global(g.qkv, g.w_q, g.w_k, g.cache.block_table, g.positions, g.cache.k_pool,
                                   g.cache.v_pool)
    torch.cuda.synchronize()
    assert torch.equal(q, q2)
    assert torch.equal(v_only, g.cache.v_pool)
    seq_lens = torch.tensor([p + 1 for p in positions], dtype=torch.int32, device=DEV)
    o = pda.attn_decode_global_shared(q, v_only, g.w_k, g.cache.block_table, seq_lens, out_dtype=torch.float32)
    torch.cuda.synchronize()
    want = oracle.decode_paged_shared(bits(q), bits(v_only), bits(case.w_k), case.cache.block_table.numpy(),
                                      np.array([p + 1 for p in positions], dtype=np.int32), 0, THETA, PAIRS)
    assert_within_tolerance(o.double().cpu().numpy(), want, "values-only append then decode")


# ---------------------------------------------------------------------------
# full-size workloads in the benchmark's launch configuration: sampled rows
# ---------------------------------------------------------------------------

def _oracle_rows_shared(case, w_k, rows):
    """Oracle on flat rows, copying only the pages of the sequences involved."""
    Hq = case.Hq
    seqs = sorted(set(int(r) // Hq for r in rows))
    sel = torch.tensor(seqs, dtype=torch.long, device=case.block_table.device)
    bt = case.block_table.index_select(0, sel)
    mapped = bt >= 0
    uniq = torch.unique(bt[mapped].long())
    new_bt = torch.full_like(bt, -1)
    new_bt[mapped] = torch.searchsorted(uniq, bt[mapped].long()).to(torch.int32)
    v = case.v_pool.index_select(0, uniq)
    pos = {s: i for i, s in enumerate(seqs)}
    sub_rows = [pos[int(r) // Hq] * Hq + int(r) % Hq for r in rows]
    return oracle.decode_paged_shared(bits(case.q.index_select(0, sel)), bits(v), bits(w_k), new_bt.cpu().numpy(),
                                      case.seq_lens.index_select(0, sel).cpu().numpy(), case.window, THETA, PAIRS,
                                      rows=sub_rows, threads=16)


@pytest.mark.slow
@pytest.mark.parametrize("variant", [None, "b"])
def test_long_context_full_size(cuda_lib, variant):
    case = config_case(4, device=DEV, variant=variant)
    w = key_weight(512, 12)
    o, st = run(case, w)
    assert st == 0
    rows = sample_rows(case, 24, 2)
    want = _oracle_rows_shared(case, w, rows)
    got = o.reshape(-1, case.D)[rows].double().cpu().numpy()
    assert_within_tolerance(got, want, "values-only long context %s" % variant)


@pytest.mark.slow
def test_decode_step_mix_global_layer_full_size(cuda_lib):
    # a global layer of the 48-layer step: B = 64, lengths log-uniform in [16, 262144]
    case = config_case(5, device=DEV, layer=5)
    w = key_weight(512, 13)
    o, st = run(case, w)
    assert st == 0
    rows = sample_rows(case, 48, 3)
    want = _oracle_rows_shared(case, w, rows)
    got = o.reshape(-1, case.D)[rows].double().cpu().numpy()
    assert_within_tolerance(got, want, "values-only step mix")
