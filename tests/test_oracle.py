"""Pins for the fp64 oracle, checked against what the pages and mathematics fix.

None of these compares the oracle with itself: each pin is a closed form, an
invariant of the definitions, or the literal dense definition evaluated
independently (``oracle.dense``).  Sources (Gemma-4-12B model page and Op
Specs page): Attention.lean ``softmax`` / ``causalGQA`` / ``slidingGQA`` /
``decodeGQA``; the attn.core rows of the compute graph; the shape domain
(page size 16).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import dense
from workloads import PAGE_SIZE, bits, make_case


def bf16_to_f64(u16):
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x):
    """Exact only for values representable in bf16 (used to build test inputs)."""
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(np.asarray(x, dtype=np.float32))), "not bf16-exact"
    return t.view(torch.int16).numpy().view(np.uint16)


def run(case, rows=None, threads=1, window=None):
    return oracle.decode_paged(bits(case.q), bits(case.k_pool), bits(case.v_pool),
                               case.block_table.numpy(), case.seq_lens.numpy(),
                               case.window if window is None else window,
                               rows=rows, threads=threads)


def dense_kv(case, b):
    """Unpage sequence b: k, v as [L, Hkv, D] float64, by reading the block table."""
    L = case.seq_lens_host[b]
    kb, vb, bt = bits(case.k_pool), bits(case.v_pool), case.block_table.numpy()
    ks, vs = [], []
    for l in range(L):
        page = bt[b, l // PAGE_SIZE]
        ks.append(bf16_to_f64(kb[page, l % PAGE_SIZE]))
        vs.append(bf16_to_f64(vb[page, l % PAGE_SIZE]))
    Hkv, D = case.Hkv, case.D
    if not ks:
        return np.zeros((0, Hkv, D)), np.zeros((0, Hkv, D))
    return np.stack(ks), np.stack(vs)


def small_case(seq_lens, seed, Hq=4, Hkv=2, D=8, window=0, kind="global", poison=False, **kw):
    return make_case(kind, seq_lens, seed, "cpu", window=window, Hq=Hq, Hkv=Hkv, D=D,
                     poison=poison, **kw)


# ---------------------------------------------------------------------------
# decode = causalGQA at position L-1, sliding decode = slidingGQA at L-1
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (4, 1), (2, 2), (16, 8)])
def test_decode_equals_last_row_of_dense_causal_gqa(Hq, Hkv):
    D = 8 if Hq < 16 else 16
    case = small_case([1, 7, 16, 17, 33], seed=11 + Hq + Hkv, Hq=Hq, Hkv=Hkv, D=D)
    got = run(case)
    G = Hq // Hkv
    for b, L in enumerate(case.seq_lens_host):
        k, v = dense_kv(case, b)
        q = bf16_to_f64(bits(case.q)[b]).reshape(Hkv, G, D)
        full = dense.causal_gqa(1.0, list(range(L)), np.broadcast_to(q, (L, Hkv, G, D)), k, v)
        want = full[L - 1].reshape(Hq, D)
        np.testing.assert_allclose(got[b], want, rtol=1e-12, atol=1e-14)
        # and the decodeGQA form itself
        np.testing.assert_allclose(got[b], dense.decode_gqa(1.0, q, k, v).reshape(Hq, D),
                                   rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("window", [1, 3, 5, 16, 17, 31])
def test_sliding_decode_equals_last_row_of_dense_sliding_gqa(window):
    case = small_case([1, 2, 6, 16, 17, 40], seed=200 + window, window=window, kind="sliding",
                      Hq=4, Hkv=2, D=8)
    got = run(case)
    for b, L in enumerate(case.seq_lens_host):
        k, v = dense_kv(case, b)
        q = bf16_to_f64(bits(case.q)[b]).reshape(2, 2, 8)
        full = dense.sliding_gqa(1.0, window, list(range(L)), np.broadcast_to(q, (L, 2, 2, 8)), k, v)
        np.testing.assert_allclose(got[b], full[L - 1].reshape(4, 8), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(got[b], dense.sliding_decode_gqa(1.0, window, q, k, v).reshape(4, 8),
                                   rtol=1e-12, atol=1e-14)


def test_gemma_shapes_tiny_lengths_match_dense():
    """Full Gemma head shapes (16/8 x 256 and 16/1 x 512) at a few short lengths."""
    for kind, lens, win in (("sliding", [1, 5, 19], 1024), ("sliding", [12], 4), ("global", [1, 3, 18], 0)):
        case = make_case(kind, lens, seed=7, window=win, poison=False)
        got = run(case)
        G = case.Hq // case.Hkv
        for b, L in enumerate(lens):
            k, v = dense_kv(case, b)
            q = bf16_to_f64(bits(case.q)[b]).reshape(case.Hkv, G, case.D)
            want = dense.sliding_decode_gqa(1.0, win, q, k, v) if win > 0 else dense.decode_gqa(1.0, q, k, v)
            np.testing.assert_allclose(got[b], want.reshape(case.Hq, case.D), rtol=1e-11, atol=1e-13)


def test_sliding_equals_full_decode_when_L_le_window():
    # slidingGQA: p < l + w holds for every l >= 0 when L <= w
    lens = [1, 9, 64, 100]
    case = make_case("sliding", lens, seed=3, window=100, poison=False)
    a = run(case, window=100)
    b = run(case, window=0)
    assert np.array_equal(a, b)
    # and it differs once L > w (the window then drops keys)
    c = run(case, window=50)
    assert not np.allclose(c[3], b[3])


# ---------------------------------------------------------------------------
# closed forms of the softmax
# ---------------------------------------------------------------------------

def test_zero_query_gives_mean_of_visible_value_rows():
    # q = 0 => every logit is 0 => softmax is uniform over the visible set
    lens = [1, 5, 16, 17, 40, 41]
    for window in (0, 7, 16, 33):
        case = small_case(lens, seed=5 + window, window=window, poison=True, kind="sliding")
        case.q.zero_()
        got = run(case)
        G = case.Hq // case.Hkv
        for b, L in enumerate(lens):
            lo = max(0, L - window) if window > 0 else 0
            _, v = dense_kv(case, b)
            mean = v[lo:L].mean(axis=0)  # [Hkv, D]
            for h in range(case.Hq):
                np.testing.assert_allclose(got[b, h], mean[h // G], rtol=1e-14, atol=1e-15)


def test_single_cached_position_returns_its_value_row():
    case = make_case("sliding", [1, 1], seed=9)
    got = run(case)
    vb = bits(case.v_pool)
    bt = case.block_table.numpy()
    for b in range(2):
        for h in range(16):
            np.testing.assert_array_equal(got[b, h], bf16_to_f64(vb[bt[b, 0], 0, h // 2]))


def test_dominant_logit_selects_its_value_row():
    # q = 64 e_0 and k_j[0] = 64 for one j, all other keys 0: logit 4096 vs 0,
    # so o = v_j up to a relative weight e^-4096 (below double precision)
    L, j = 37, 23
    case = small_case([L], seed=13, Hq=4, Hkv=2, D=8, poison=False)
    case.q.zero_()
    case.q[0, :, 0] = 64.0
    bt = case.block_table.numpy()
    case.k_pool.zero_()
    case.k_pool[bt[0, j // PAGE_SIZE], j % PAGE_SIZE, :, 0] = 64.0
    got = run(case)
    vj = bf16_to_f64(bits(case.v_pool)[bt[0, j // PAGE_SIZE], j % PAGE_SIZE])
    for h in range(4):
        np.testing.assert_array_equal(got[0, h], vj[h // 2])
    # flipping the sign of q makes j the only *least* likely key: the rest share evenly
    case.q[0, :, 0] = -64.0
    got = run(case)
    _, v = dense_kv(case, 0)
    others = np.delete(v, j, axis=0).mean(axis=0)
    for h in range(4):
        np.testing.assert_allclose(got[0, h], others[h // 2], rtol=1e-13, atol=1e-14)


def test_two_positions_closed_form():
    # L = 2: o = (e^{s0} v0 + e^{s1} v1) / (e^{s0} + e^{s1}), logits set through exact bf16 values
    case = small_case([2], seed=17, Hq=2, Hkv=1, D=4, poison=False)
    q = np.array([[1.0, 0.5, 0.0, -2.0], [0.25, 0.0, 3.0, 1.0]])
    k = np.array([[2.0, -1.0, 0.5, 0.25], [-0.5, 4.0, 1.0, -1.0]])
    v = np.array([[1.0, 2.0, 3.0, 4.0], [-8.0, 0.5, 0.125, 16.0]])
    case.q[0] = torch.tensor(q, dtype=torch.bfloat16)
    bt = case.block_table.numpy()
    case.k_pool[bt[0, 0], 0:2, 0] = torch.tensor(k, dtype=torch.bfloat16)
    case.v_pool[bt[0, 0], 0:2, 0] = torch.tensor(v, dtype=torch.bfloat16)
    got = run(case)
    for h in range(2):
        s0 = float(np.dot(q[h], k[0]))
        s1 = float(np.dot(q[h], k[1]))
        w0, w1 = math.exp(s0), math.exp(s1)
        want = (w0 * v[0] + w1 * v[1]) / (w0 + w1)
        np.testing.assert_allclose(got[0, h], want, rtol=1e-15, atol=1e-15)


def test_empty_sequence_gives_zeros():
    case = make_case("global", [0, 3], seed=19)
    got = run(case)
    assert np.array_equal(got[0], np.zeros((16, 512)))
    assert np.isfinite(got[1]).all()


# ---------------------------------------------------------------------------
# invariants: window edges, head mapping, paging
# ---------------------------------------------------------------------------

def test_keys_outside_the_window_have_no_effect():
    lens = [5, 40, 77]
    window = 20
    case = small_case(lens, seed=23, window=window, kind="sliding", poison=False)
    base = run(case)
    bt = case.block_table.numpy()
    g = torch.Generator().manual_seed(99)
    for b, L in enumerate(lens):
        lo = max(0, L - window)
        for l in list(range(0, lo)) + list(range(L, bt.shape[1] * PAGE_SIZE)):
            page = bt[b, l // PAGE_SIZE]
            if page >= 0:
                case.k_pool[page, l % PAGE_SIZE] = 100 * torch.randn(case.k_pool.shape[2:], generator=g)
                case.v_pool[page, l % PAGE_SIZE] = 100 * torch.randn(case.v_pool.shape[2:], generator=g)
    assert np.array_equal(run(case), base)
    # and a key inside the window does have an effect
    L = lens[2]
    page = bt[2, (L - 1) // PAGE_SIZE]
    case.v_pool[page, (L - 1) % PAGE_SIZE] += 1.0
    assert not np.array_equal(run(case)[2], base[2])


def test_nan_poisoned_invisible_slots_do_not_reach_the_output():
    case = make_case("sliding", [1, 17, 300, 1100], seed=1001, poison=True)
    got = run(case)
    assert np.isfinite(got).all()
    case3 = make_case("sliding", [1024, 1030, 2047], seed=31, window_only=True, poison=True)
    assert (case3.block_table.numpy()[2, :63] == -1).all()  # L=2047: lo=1023, first page 63
    assert np.isfinite(run(case3)).all()


def test_query_head_h_reads_kv_head_h_over_G():
    # q = 0 and V constant per KV head (value c+1): head h must return (h // G) + 1
    for Hq, Hkv in ((16, 8), (16, 1), (8, 4)):
        case = small_case([21, 3], seed=29, Hq=Hq, Hkv=Hkv, D=8, poison=True, kind="sliding",
                          window=0)
        case.q.zero_()
        nan_mask = torch.isnan(case.v_pool)
        for c in range(Hkv):
            case.v_pool[:, :, c, :] = float(c + 1)
        case.v_pool[nan_mask] = float("nan")
        got = run(case)
        G = Hq // Hkv
        for h in range(Hq):
            assert np.all(got[:, h, :] == float(h // G + 1))


def test_paging_is_a_relabelling():
    # the same logical cache under two page permutations gives the identical result
    lens = [3, 16, 17, 50]
    a = make_case("sliding", lens, seed=37, window=0, Hq=4, Hkv=2, D=8, poison=True)
    b = make_case("sliding", lens, seed=37, window=0, Hq=4, Hkv=2, D=8, poison=True)
    # relabel b: move every page of a through a fresh permutation
    P = a.num_pages
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(5))
    b.k_pool = torch.empty_like(a.k_pool)
    b.v_pool = torch.empty_like(a.v_pool)
    b.k_pool[perm] = a.k_pool
    b.v_pool[perm] = a.v_pool
    bt = a.block_table.clone()
    mapped = bt >= 0
    bt[mapped] = perm[bt[mapped].long()].to(torch.int32)
    b.block_table = bt
    assert not torch.equal(a.block_table, b.block_table)
    assert np.array_equal(run(a), run(b))


def test_row_subset_and_threads_agree_with_full_run():
    case = make_case("global", [5, 100, 33], seed=41)
    full = run(case)
    rows = [0, 17, 47, 20]
    sub = run(case, rows=rows, threads=3)
    for i, r in enumerate(rows):
        assert np.array_equal(sub[i], full.reshape(-1, 512)[r])


def test_unmapped_visible_page_is_an_error():
    case = make_case("global", [40], seed=43)
    case.block_table[0, 1] = -1
    with pytest.raises(oracle.OracleError):
        run(case)
    case = make_case("global", [40], seed=43)
    case.block_table[0, 2] = case.num_pages  # out of range
    with pytest.raises(oracle.OracleError):
        run(case)


def test_golden_fixture_reproduces():
    """tests/golden/decode_small.json: frozen bf16 inputs and the oracle's outputs."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "decode_small.json")
    for c in json.load(open(path)):
        B = len(c["seq_lens"])
        q = np.array(c["q_bits"], dtype=np.uint16).reshape(B, c["Hq"], c["D"])
        shape = (c["num_pages"], c["page_size"], c["Hkv"], c["D"])
        k = np.array(c["k_bits"], dtype=np.uint16).reshape(shape)
        v = np.array(c["v_bits"], dtype=np.uint16).reshape(shape)
        bt = np.array(c["block_table"], dtype=np.int32)
        sl = np.array(c["seq_lens"], dtype=np.int32)
        got = oracle.decode_paged(q, k, v, bt, sl, c["window"])
        want = np.array([float.fromhex(x) for x in c["o"]]).reshape(got.shape)
        np.testing.assert_allclose(got, want, rtol=1e-14, atol=0)
