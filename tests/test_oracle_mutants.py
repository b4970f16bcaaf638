"""Planted mistakes in a copy of the C oracle must be caught by the pins.

Each mutant is a plausible slip (a wrong window edge, head index, sign,
operand, page slot, missing term) applied textually to a temporary copy of
``oracle/oracle.c``, compiled with gcc into a temp directory, and run through
a battery of the same pins as ``test_oracle.py`` (dense Lean definitions,
closed forms).  The unmodified source must pass the battery and every mutant
must fail it.  Nothing here touches a GPU.
"""

import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle import dense
from workloads import PAGE_SIZE, bits, make_case

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "window_edge_off_by_one": ("lo = L - j->window;", "lo = L - j->window + 1;"),
    "head_map_modulo": ("const int c = h / G;", "const int c = h % j->Hkv;"),
    "no_normalisation": ("o[d] /= Z;", "o[d] /= 1.0;"),
    "softmax_sign": ("logit[i] = exp(logit[i] - m);", "logit[i] = exp(m - logit[i]);"),
    "no_max_subtraction": ("logit[i] = exp(logit[i] - m);", "logit[i] = exp(logit[i]);"),
    "slot_from_page_index": ("return phys * j->page_size + (l % j->page_size);",
                             "return phys * j->page_size + (page % j->page_size);"),
    "logits_read_v_pool": ("const uint16_t* kv = j->k_pool + (r * j->Hkv + c) * D;",
                           "const uint16_t* kv = j->v_pool + (r * j->Hkv + c) * D;"),
    "query_of_wrong_head": ("attend_one_row(j, b, h, j->q + ((int64_t)b * j->Hq + h) * j->D, L, o, logit)",
                            "attend_one_row(j, b, h, j->q + ((int64_t)b * j->Hq + h / (j->Hq / j->Hkv)) * j->D, L, o, logit)"),
    "denominator_drops_last_term": ("    Z += logit[i];", "    Z += (i + 1 < n) ? logit[i] : 0.0;"),
}


def _build(tmp_path, name, replace=None):
    src = open(SRC).read()
    if replace is not None:
        old, new = replace
        assert src.count(old) >= 1, "mutation anchor missing: %s" % old
        src = src.replace(old, new)
    c = tmp_path / ("%s.c" % name)
    so = tmp_path / ("lib%s.so" % name)
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so), str(c), "-lm"],
                   check=True)
    return str(so)


def _f64(u16):
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _run(case, lib):
    return oracle.decode_paged(bits(case.q), bits(case.k_pool), bits(case.v_pool),
                               case.block_table.numpy(), case.seq_lens.numpy(), case.window,
                               lib_path=lib)


def _dense_kv(case, b):
    L = case.seq_lens_host[b]
    kb, vb, bt = bits(case.k_pool), bits(case.v_pool), case.block_table.numpy()
    k = np.stack([_f64(kb[bt[b, l // PAGE_SIZE], l % PAGE_SIZE]) for l in range(L)])
    v = np.stack([_f64(vb[bt[b, l // PAGE_SIZE], l % PAGE_SIZE]) for l in range(L)])
    return k, v


def battery(lib):
    """The pins, as a list of (name, passed) pairs."""
    out = []

    def check(name, fn):
        try:
            out.append((name, bool(fn())))
        except Exception:
            out.append((name, False))

    # dense slidingGQA / decodeGQA at the last position
    def dense_pin(window, Hq, Hkv):
        case = make_case("sliding", [1, 6, 17, 40], 300 + window + Hq, window=window, Hq=Hq, Hkv=Hkv,
                         D=8, poison=True)
        got = _run(case, lib)
        G = Hq // Hkv
        for b, L in enumerate(case.seq_lens_host):
            k, v = _dense_kv(case, b)
            q = _f64(bits(case.q)[b]).reshape(Hkv, G, 8)
            want = dense.sliding_decode_gqa(1.0, window, q, k, v) if window > 0 else dense.decode_gqa(1.0, q, k, v)
            if not np.allclose(got[b], want.reshape(Hq, 8), rtol=1e-12, atol=1e-14):
                return False
        return True

    check("dense_sliding_w5", lambda: dense_pin(5, 4, 2))
    check("dense_causal", lambda: dense_pin(0, 4, 1))
    check("dense_gqa_8_4", lambda: dense_pin(0, 8, 4))

    # dominant logit 4096 selects its row
    def dominant():
        case = make_case("global", [37], 13, Hq=4, Hkv=2, D=8, poison=False)
        case.q.zero_()
        case.q[0, :, 0] = 64.0
        bt = case.block_table.numpy()
        case.k_pool.zero_()
        case.k_pool[bt[0, 1], 7, :, 0] = 64.0
        got = _run(case, lib)
        vj = _f64(bits(case.v_pool)[bt[0, 1], 7])
        return all(np.array_equal(got[0, h], vj[h // 2]) for h in range(4))

    check("dominant_logit", dominant)

    # q = 0 gives the mean of the visible rows
    def mean_pin():
        case = make_case("sliding", [3, 33], 21, window=20, Hq=4, Hkv=2, D=8, poison=True)
        case.q.zero_()
        got = _run(case, lib)
        for b, L in enumerate(case.seq_lens_host):
            _, v = _dense_kv(case, b)
            mean = v[max(0, L - 20):L].mean(axis=0)
            if not all(np.allclose(got[b, h], mean[h // 2], rtol=1e-14) for h in range(4)):
                return False
        return True

    check("zero_query_mean", mean_pin)

    # two-position closed form
    def two_pos():
        case = make_case("global", [2], 17, Hq=2, Hkv=1, D=4, poison=False)
        q = np.array([[1.0, 0.5, 0.0, -2.0], [0.25, 0.0, 3.0, 1.0]])
        k = np.array([[2.0, -1.0, 0.5, 0.25], [-0.5, 4.0, 1.0, -1.0]])
        v = np.array([[1.0, 2.0, 3.0, 4.0], [-8.0, 0.5, 0.125, 16.0]])
        case.q[0] = torch.tensor(q, dtype=torch.bfloat16)
        bt = case.block_table.numpy()
        case.k_pool[bt[0, 0], 0:2, 0] = torch.tensor(k, dtype=torch.bfloat16)
        case.v_pool[bt[0, 0], 0:2, 0] = torch.tensor(v, dtype=torch.bfloat16)
        got = _run(case, lib)
        for h in range(2):
            w0, w1 = math.exp(np.dot(q[h], k[0])), math.exp(np.dot(q[h], k[1]))
            if not np.allclose(got[0, h], (w0 * v[0] + w1 * v[1]) / (w0 + w1), rtol=1e-15):
                return False
        return True

    check("two_positions", two_pos)
    return out


def test_unmodified_oracle_passes_the_battery(tmp_path):
    lib = _build(tmp_path, "clean")
    res = battery(lib)
    assert all(ok for _, ok in res), res


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    lib = _build(tmp_path, name, MUTANTS[name])
    res = battery(lib)
    failed = [n for n, ok in res if not ok]
    assert failed, "mutant %s passed every pin" % name
