"""The C ABI without a GPU: the library loads, exports what the header declares,
plans splits by plain arithmetic, and rejects bad arguments before launching.
"""

import ctypes
import os
import re

import pytest

import paged_decode_attention_gb300 as pda
from paged_decode_attention_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
HEADERS = sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pda.load()


def declared_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_operations():
    names = declared_functions()
    for n in ("attn_decode_sliding", "attn_decode_global", "attn_decode_plan",
              "attn_decode_workspace_size", "attn_last_error", "attn_abi_version",
              "attn_decode_global_shared", "attn_step_create", "attn_step_launch"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), "symbol %s declared in include/ but not exported" % n


def test_binding_covers_the_exports(lib):
    assert set(pda.EXPORTS) <= set(declared_functions())


def test_abi_version(lib):
    assert lib.attn_abi_version() == 1


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "attn_decode.h"\n#include "attn_step.h"\n'
                   'int main(void){attn_step* s = 0; return ATTN_OK + attn_step_num_calls(s);}\n')
    import subprocess
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-c", str(src), "-o", str(tmp_path / "use.o")], check=True)


# ---------------------------------------------------------------------------
# split plan (pure host arithmetic)
# ---------------------------------------------------------------------------

def _workspace(gx, batch, D):
    def a256(x):
        return (x + 255) // 256 * 256
    rows = (gx + batch) * 16
    return pda.WORKSPACE_ZERO_BYTES + a256(rows * D * 4) + a256(rows * 8)


def test_plan_fills_one_wave(lib):
    # sliding: 3 blocks per SM x 152 SMs over 8 KV-head columns; global: 2 per SM
    gx, ws = pda.attn_decode_plan(pda.KIND_SLIDING, 256, 32768, 1024)
    assert gx == 152 * 3 // 8
    assert ws == _workspace(gx, 256, 256)
    gx, ws = pda.attn_decode_plan(pda.KIND_GLOBAL, 4, 262144, 0)
    assert gx == 304
    assert ws == _workspace(304, 4, 512)


def test_plan_small_problems_launch_fewer_blocks(lib):
    # 2 sequences of at most 10 pages, 4 pages per block at least -> 5 blocks
    gx, _ = pda.attn_decode_plan(pda.KIND_GLOBAL, 2, 160, 0)
    assert gx == 5
    # a window bounds a sequence's visible pages at ceil(w/16) + 1 = 65
    gx, _ = pda.attn_decode_plan(pda.KIND_SLIDING, 1, 262144, 1024)
    assert gx == 17  # ceil(65 / 4)
    gx, ws = pda.attn_decode_plan(pda.KIND_SLIDING, 2, 0, 1024)
    assert gx == 1 and ws == _workspace(1, 2, 256)


def test_split_sequences_merge_in_the_grid_when_few_blocks_share_one(lib):
    K = pda.KIND_SLIDING
    # sliding, window 1024: at most 65 visible pages, spans of at least 4 pages -> at most 18 blocks;
    # with 256 sequences the spans are long, so 2 or 3 blocks share one
    assert pda.attn_decode_launches(K, 256, 32768, 1024) == 1
    assert pda.attn_decode_launches(K, 64, 262144, 1024) == 1
    # a window of 1456 spans at most 92 pages, (92 - 1) // 4 + 2 = 24 blocks: the bound; 1457 does not fit
    assert pda.attn_decode_launches(K, 256, 262144, 1456) == 1
    assert pda.attn_decode_launches(K, 256, 262144, 1457) == 2
    # max_seq_len caps the pages too: 1472 positions are 92 pages
    assert pda.attn_decode_launches(K, 256, 1472, 100000) == 1
    assert pda.attn_decode_launches(K, 256, 1473, 100000) == 2
    # few short-spanned blocks: 4 sequences of up to 65 pages over 57 blocks would put about 15 blocks on
    # one sequence, whose last block would read 14 partials: the combine kernel is faster there
    assert pda.attn_decode_launches(K, 4, 1100, 1024) == 2
    assert pda.attn_decode_launches(K, 10, 5000, 1024, num_splits=40) == 1
    assert pda.attn_decode_launches(K, 10, 5000, 1024, num_splits=300) == 2
    # the SM count sizes the grid: one SM holds 3 blocks over 8 columns, so spans are long
    assert pda.attn_decode_launches(K, 4, 1100, 1024, num_sms=1) == 1
    # global layers keep the combine kernel
    assert pda.attn_decode_launches(pda.KIND_GLOBAL, 8, 8192, 0) == 2
    with pytest.raises(pda.AttnDecodeError):
        pda.attn_decode_launches(K, 0, 100, 1024)


def test_plan_respects_forced_block_counts(lib):
    assert pda.attn_decode_plan(pda.KIND_GLOBAL, 2, 160, 0, num_splits=7)[0] == 7
    assert pda.attn_decode_plan(pda.KIND_GLOBAL, 2, 160, 0, num_splits=1)[0] == 1
    assert pda.attn_decode_plan(pda.KIND_SLIDING, 1, 262144, 1024, num_splits=1000)[0] == 1000
    # the combine kernel merges at most 1024 partials per row
    assert pda.attn_decode_plan(pda.KIND_GLOBAL, 1, 262144, 0, num_splits=5000)[0] == 1024


def test_plan_rejects_bad_arguments(lib):
    with pytest.raises(pda.AttnDecodeError):
        pda.attn_decode_plan(7, 1, 16, 0)
    with pytest.raises(pda.AttnDecodeError):
        pda.attn_decode_plan(pda.KIND_GLOBAL, 0, 16, 0)
    with pytest.raises(pda.AttnDecodeError):
        pda.attn_decode_plan(pda.KIND_GLOBAL, 1, 16, 0, num_sms=0)


# ---------------------------------------------------------------------------
# host validation: returns an error code and launches nothing
# ---------------------------------------------------------------------------

FAKE = 1 << 20  # an aligned, never dereferenced address


def call(lib, name="attn_decode_sliding", **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, o=FAKE, batch=4, max_blocks=70,
             num_pages=300, max_seq_len=1100, window=1024, out_dtype=0, num_splits=0,
             ws=None, ws_bytes=0, status=None, stream=None)
    a.update(kw)
    fn = getattr(lib, name)
    return fn(a["q"], a["k"], a["v"], a["bt"], a["sl"], a["o"], a["batch"], a["max_blocks"],
              a["num_pages"], a["max_seq_len"], a["window"], a["out_dtype"], a["num_splits"],
              a["ws"], a["ws_bytes"], a["status"], a["stream"])


# attn_decode_global_shared takes (q, kv_pool, w_k, ...): k is its pool, v its w_k
@pytest.mark.parametrize("name", ["attn_decode_sliding", "attn_decode_global", "attn_decode_global_shared"])
@pytest.mark.parametrize("bad,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(bt=None), 1), (dict(sl=None), 1),
    (dict(o=None), 1), (dict(q=FAKE + 8), 1), (dict(v=FAKE + 8), 1), (dict(o=FAKE + 2), 1),
    (dict(status=FAKE + 2), 1),
    (dict(batch=0), 1), (dict(batch=257), 2), (dict(max_blocks=0), 1), (dict(num_pages=0), 1),
    (dict(num_pages=1 << 27), 2), (dict(max_seq_len=-1), 1), (dict(max_seq_len=70 * 16 + 1), 1),
    (dict(max_blocks=20000, max_seq_len=262145), 2), (dict(out_dtype=2), 1), (dict(num_splits=-1), 1),
])
def test_invalid_arguments_are_rejected_before_launch(lib, name, bad, code):
    assert call(lib, name, **bad) == code
    assert pda.attn_last_error() != ""


def test_sliding_requires_a_positive_window(lib):
    assert call(lib, "attn_decode_sliding", window=0) == 1
    assert call(lib, "attn_decode_sliding", window=-5) == 1
    assert "window" in pda.attn_last_error()


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 16, 256, dtype=torch.bfloat16)
    pool = torch.zeros(2, 16, 8, 256, dtype=torch.bfloat16)
    bt = torch.zeros(1, 1, dtype=torch.int32)
    sl = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        pda.attn_decode_sliding(q, pool, pool, bt, sl)


# ---------------------------------------------------------------------------
# whole-step object: recording validates each call; nothing needs a GPU until
# a valid call queries the device
# ---------------------------------------------------------------------------

def _step_add(lib, step, name, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, sl=FAKE, o=FAKE, batch=4, max_blocks=70,
             num_pages=300, max_seq_len=1100, window=1024, out_dtype=0, num_splits=0,
             ws=None, ws_bytes=0, status=None)
    a.update(kw)
    return getattr(lib, name)(step, a["q"], a["k"], a["v"], a["bt"], a["sl"], a["o"], a["batch"], a["max_blocks"],
                              a["num_pages"], a["max_seq_len"], a["window"], a["out_dtype"], a["num_splits"],
                              a["ws"], a["ws_bytes"], a["status"])


@pytest.mark.parametrize("name", ["attn_step_add_decode_sliding", "attn_step_add_decode_global",
                                  "attn_step_add_decode_global_shared"])
@pytest.mark.parametrize("bad,code", [(dict(q=None), 1), (dict(o=FAKE + 2), 1), (dict(batch=257), 2),
                                      (dict(num_splits=-1), 1), (dict(out_dtype=7), 1)])
def test_step_rejects_a_bad_call_and_records_nothing(lib, name, bad, code):
    h = ctypes.c_void_p()
    assert lib.attn_step_create(ctypes.byref(h)) == 0
    try:
        assert _step_add(lib, h, name, **bad) == code
        assert pda.attn_last_error() != ""
        assert lib.attn_step_num_calls(h) == 0 and lib.attn_step_num_kernels(h) == 0
    finally:
        lib.attn_step_destroy(h)


def test_step_without_calls_or_handle(lib):
    h = ctypes.c_void_p()
    assert lib.attn_step_create(ctypes.byref(h)) == 0
    try:
        assert lib.attn_step_finalize(h) == 1 and "no calls" in pda.attn_last_error()
        assert lib.attn_step_launch(h, None) == 1 and "not finalized" in pda.attn_last_error()
    finally:
        lib.attn_step_destroy(h)
    assert lib.attn_step_create(None) == 1
    assert lib.attn_step_finalize(None) == 1
    assert lib.attn_step_launch(None, None) == 1
    assert lib.attn_step_num_calls(None) == 0
    lib.attn_step_destroy(None)  # ignored


def test_step_launch_mode_is_checked_and_kept(lib):
    h = ctypes.c_void_p()
    assert lib.attn_step_create(ctypes.byref(h)) == 0
    try:
        assert lib.attn_step_launch_mode(h) == pda.STEP_LAUNCH_AUTO
        assert lib.attn_step_set_launch_mode(h, 7) == 1 and "unknown mode" in pda.attn_last_error()
        assert lib.attn_step_set_launch_mode(h, -1) == 1
        assert lib.attn_step_launch_mode(h) == pda.STEP_LAUNCH_AUTO
        for m in (pda.STEP_LAUNCH_DIRECT, pda.STEP_LAUNCH_GRAPH):
            assert lib.attn_step_set_launch_mode(h, m) == 0 and lib.attn_step_launch_mode(h) == m
    finally:
        lib.attn_step_destroy(h)
    assert lib.attn_step_set_launch_mode(None, 0) == 1
    assert lib.attn_step_launch_mode(None) == -1
    with pytest.raises(ValueError):
        pda.Step().finalize("sometimes")


def test_step_append_validation(lib):
    h = ctypes.c_void_p()
    assert lib.attn_step_create(ctypes.byref(h)) == 0
    try:
        # sliding needs a key pool; a batch outside the domain is refused
        assert lib.attn_step_add_kv_append_sliding(h, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 4, 70, 300,
                                                   None) == 1
        assert lib.attn_step_add_kv_append_global(h, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 0, 70, 300,
                                                  None) == 2
        # a values-only global append passes the host checks (no device query) and is recorded
        assert lib.attn_step_add_kv_append_global(h, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 4, 70, 300,
                                                  None) == 0
        assert lib.attn_step_num_calls(h) == 1 and lib.attn_step_num_kernels(h) == 1
    finally:
        lib.attn_step_destroy(h)


def test_step_binding_refuses_cpu_tensors_and_empty_finalize(lib):
    import torch
    step = pda.Step()
    q = torch.zeros(1, 16, 512, dtype=torch.bfloat16)
    pool = torch.zeros(2, 16, 1, 512, dtype=torch.bfloat16)
    bt = torch.zeros(1, 1, dtype=torch.int32)
    sl = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        step.add_decode_global(q, pool, pool, bt, sl)
    assert step.num_calls == 0
    with pytest.raises(pda.AttnDecodeError):
        step.finalize()
    step.close()
    step.close()  # idempotent
