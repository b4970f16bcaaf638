"""fp64 CPU oracle for paged decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never links, loads or calls it, and this package
never imports the CUDA library.

* ``decode_paged`` -- the paged decode oracle in ``oracle.c`` (plain C,
  double precision, pthreads over output rows), called through ctypes.
* ``prefill_paged`` -- multi-query (prefill) attention over the paged cache:
  each query row is the decode of its sequence cut at the query's position
  (``oracle.c``).
* ``decode_paged_shared`` -- the global-layer decode over a cache that stores
  values only: keys rebuilt as rope(V * w_k), rounded once to bf16
  (``oracle.c``), then ``decode_paged``.
* ``qkv_append``   -- the per-head norms, RoPE and paged KV-cache append of
  one new token per sequence (``oracle.c``, double precision).
* ``dense``        -- the literal Lean definitions over unpaged arrays, for
  tiny cases (see ``dense.py``).

Inputs are numpy arrays: bf16 tensors are passed as their uint16 bit patterns.
"""

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

ERRORS = {
    0: "ok",
    1: "invalid argument",
    2: "seq_len negative or beyond the block table",
    3: "a visible position maps to an unmapped or out-of-range page",
    4: "out of memory",
}


class OracleError(RuntimeError):
    pass


def build(force=False):
    """Compile oracle.c with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_libs = {}


def _load(lib_path=None):
    key = lib_path or "default"
    if key not in _libs:
        lib = ctypes.CDLL(lib_path or build())
        fn = lib.oracle_decode_paged
        fn.restype = ctypes.c_int
        fn.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # q, k_pool, v_pool
            ctypes.c_void_p, ctypes.c_void_p,                    # block_table, seq_lens
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,  # B Hq Hkv D
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,      # page_size max_blocks num_pages
            ctypes.c_int32,                                      # window
            ctypes.c_void_p, ctypes.c_int32,                     # rows, n_rows
            ctypes.c_void_p, ctypes.c_int32,                     # out, n_threads
        ]
        fp = lib.oracle_prefill_paged
        fp.restype = ctypes.c_int
        fp.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # q, k_pool, v_pool
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # block_table, seq_lens, cu_q
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,  # B Hq Hkv D
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,      # page_size max_blocks num_pages
            ctypes.c_int32,                                      # window
            ctypes.c_void_p, ctypes.c_int32,                     # rows, n_rows
            ctypes.c_void_p, ctypes.c_int32,                     # out, n_threads
        ]
        fr = lib.oracle_rebuild_keys
        fr.restype = ctypes.c_int
        fr.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # v_pool w_k block_table seq_lens
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,      # B Hkv D page_size
            ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,                      # max_blocks num_pages window
            ctypes.c_double, ctypes.c_int32, ctypes.c_void_p,                    # theta rope_pairs k_out
        ]
        fa = lib.oracle_qkv_append
        fa.restype = ctypes.c_int
        fa.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # qkv, w_q, w_k
            ctypes.c_void_p, ctypes.c_void_p,                    # block_table, positions
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,  # B Hq Hkv D shared
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,      # page_size max_blocks num_pages
            ctypes.c_double, ctypes.c_int32, ctypes.c_double,    # theta, rope_pairs, eps
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,  # q_out, k_pool, v_pool
        ]
        _libs[key] = lib
    return _libs[key]


def _as(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError("expected %s, got %s" % (dtype, a.dtype))
    return a


def decode_paged(q_bits, k_bits, v_bits, block_table, seq_lens, window, page_size=16,
                 rows=None, threads=1, lib_path=None):
    """Paged decode attention in fp64.

    q_bits      uint16 [B, Hq, D]                     (bf16 bit patterns)
    k_bits      uint16 [num_pages, page_size, Hkv, D]
    v_bits      uint16 [num_pages, page_size, Hkv, D]
    block_table int32  [B, max_blocks]
    seq_lens    int32  [B]
    window      > 0 sliding window, <= 0 none
    rows        None (all B*Hq rows) or a sequence of flat b*Hq + h indices
    lib_path    another build of oracle.c to call (the tests' planted-mistake checks)
    returns     float64 [B, Hq, D], or [len(rows), D] when rows is given
    """
    q_bits = _as(q_bits, np.uint16)
    k_bits = _as(k_bits, np.uint16)
    v_bits = _as(v_bits, np.uint16)
    block_table = _as(block_table, np.int32)
    seq_lens = _as(seq_lens, np.int32)
    B, Hq, D = q_bits.shape
    num_pages, ps, Hkv, Dk = k_bits.shape
    if ps != page_size or Dk != D or v_bits.shape != k_bits.shape:
        raise ValueError("pool shape does not match q / page_size")
    if block_table.ndim != 2 or block_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("block_table / seq_lens shape")
    max_blocks = block_table.shape[1]
    if rows is None:
        rows_arr, n_rows, out = None, 0, np.zeros((B, Hq, D), dtype=np.float64)
    else:
        rows_arr = _as(np.asarray(rows, dtype=np.int32), np.int32)
        n_rows = len(rows_arr)
        out = np.zeros((n_rows, D), dtype=np.float64)
    st = _load(lib_path).oracle_decode_paged(
        q_bits.ctypes.data, k_bits.ctypes.data, v_bits.ctypes.data,
        block_table.ctypes.data, seq_lens.ctypes.data,
        B, Hq, Hkv, D, page_size, max_blocks, num_pages, int(window),
        None if rows_arr is None else rows_arr.ctypes.data, n_rows,
        out.ctypes.data, int(threads),
    )
    if st != 0:
        raise OracleError(ERRORS.get(st, "error %d" % st))
    return out


def prefill_paged(q_bits, k_bits, v_bits, block_table, seq_lens, cu_q, window, page_size=16,
                  rows=None, threads=1, lib_path=None):
    """Multi-query attention over the paged cache, fp64.

    q_bits      uint16 [T, Hq, D], the queries of every sequence packed in order
    cu_q        int32 [B+1]: sequence b owns rows cu_q[b] .. cu_q[b+1]-1, the
                last n = cu_q[b+1] - cu_q[b] of its L = seq_lens[b] tokens, so its
                query i sits at position L - n + i
    rows        None (all T*Hq rows) or flat t*Hq + h indices
    returns     float64 [T, Hq, D], or [len(rows), D]
    The other arguments are as for decode_paged.
    """
    q_bits = _as(q_bits, np.uint16)
    k_bits = _as(k_bits, np.uint16)
    v_bits = _as(v_bits, np.uint16)
    block_table = _as(block_table, np.int32)
    seq_lens = _as(seq_lens, np.int32)
    cu_q = _as(cu_q, np.int32)
    T, Hq, D = q_bits.shape
    num_pages, ps, Hkv, Dk = k_bits.shape
    B = seq_lens.shape[0]
    if ps != page_size or Dk != D or v_bits.shape != k_bits.shape:
        raise ValueError("pool shape does not match q / page_size")
    if block_table.ndim != 2 or block_table.shape[0] != B or cu_q.shape != (B + 1,) or cu_q[-1] != T:
        raise ValueError("block_table / cu_q shape")
    if rows is None:
        rows_arr, n_rows, out = None, 0, np.zeros((T, Hq, D), dtype=np.float64)
    else:
        rows_arr = _as(np.asarray(rows, dtype=np.int32), np.int32)
        n_rows = len(rows_arr)
        out = np.zeros((n_rows, D), dtype=np.float64)
    st = _load(lib_path).oracle_prefill_paged(
        q_bits.ctypes.data, k_bits.ctypes.data, v_bits.ctypes.data,
        block_table.ctypes.data, seq_lens.ctypes.data, cu_q.ctypes.data,
        B, Hq, Hkv, D, page_size, block_table.shape[1], num_pages, int(window),
        None if rows_arr is None else rows_arr.ctypes.data, n_rows,
        out.ctypes.data, int(threads),
    )
    if st != 0:
        raise OracleError(ERRORS.get(st, "error %d" % st))
    return out


def rebuild_keys(v_bits, wk_bits, block_table, seq_lens, window, theta, rope_pairs, k_init=None, page_size=16,
                 lib_path=None):
    """Keys of a values-only cache: K = bf16(rope(V * w_k)) at every visible
    position (fp64, one rounding).  Returns uint16 [num_pages, page_size, Hkv, D]:
    k_init (default: all NaN) with the visible slots written."""
    v_bits = _as(v_bits, np.uint16)
    wk_bits = _as(wk_bits, np.uint16)
    block_table = _as(block_table, np.int32)
    seq_lens = _as(seq_lens, np.int32)
    num_pages, ps, Hkv, D = v_bits.shape
    if ps != page_size or wk_bits.shape != (D,) or block_table.shape[0] != seq_lens.shape[0]:
        raise ValueError("shapes")
    k = np.full(v_bits.shape, 0x7FC0, dtype=np.uint16) if k_init is None else _as(k_init, np.uint16).copy()
    st = _load(lib_path).oracle_rebuild_keys(
        v_bits.ctypes.data, wk_bits.ctypes.data, block_table.ctypes.data, seq_lens.ctypes.data,
        seq_lens.shape[0], Hkv, D, page_size, block_table.shape[1], num_pages, int(window), float(theta),
        int(rope_pairs), k.ctypes.data)
    if st != 0:
        raise OracleError("oracle_rebuild_keys: %s" % ERRORS.get(st, st))
    return k


def decode_paged_shared(q_bits, v_bits, wk_bits, block_table, seq_lens, window, theta, rope_pairs, page_size=16,
                        rows=None, threads=1, lib_path=None):
    """decode_paged over a values-only cache: the keys are rebuild_keys(...)."""
    k = rebuild_keys(v_bits, wk_bits, block_table, seq_lens, window, theta, rope_pairs, page_size=page_size,
                     lib_path=lib_path)
    return decode_paged(q_bits, k, v_bits, block_table, seq_lens, window, page_size=page_size, rows=rows,
                        threads=threads, lib_path=lib_path)


def qkv_append(qkv_bits, wq_bits, wk_bits, block_table, positions, q_out, k_pool, v_pool, *, Hq, Hkv, D,
               shared_kv, theta, rope_pairs, eps=1e-6, page_size=16, lib_path=None):
    """Norms, RoPE and cache append of one token per sequence, fp64, rounded once to bf16.

    qkv_bits    uint16 [B, Hq*D + (D if shared_kv else 2*Hkv*D)]   (bf16 bit patterns)
    wq_bits, wk_bits  uint16 [D]   qk_norm weights of q and k
    block_table int32 [B, max_blocks];  positions int32 [B] (each token's position)
    q_out       uint16 [B, Hq, D], written
    k_pool, v_pool  uint16 [num_pages, page_size, Hkv, D]; each token's slot is written
    Raises OracleError on a position beyond the table or an unmapped page.
    """
    qkv_bits = _as(qkv_bits, np.uint16)
    wq_bits = _as(wq_bits, np.uint16)
    wk_bits = _as(wk_bits, np.uint16)
    block_table = _as(block_table, np.int32)
    positions = _as(positions, np.int32)
    for name, arr in (("q_out", q_out), ("k_pool", k_pool), ("v_pool", v_pool)):
        if arr.dtype != np.uint16 or not arr.flags["C_CONTIGUOUS"] or not arr.flags["WRITEABLE"]:
            raise TypeError("%s must be a writeable C-contiguous uint16 array" % name)
    B = qkv_bits.shape[0]
    row_len = Hq * D + (D if shared_kv else 2 * Hkv * D)
    if qkv_bits.shape != (B, row_len) or wq_bits.shape != (D,) or wk_bits.shape != (D,):
        raise ValueError("qkv / weight shape")
    if q_out.shape != (B, Hq, D) or positions.shape != (B,) or block_table.shape[0] != B:
        raise ValueError("q_out / positions / block_table shape")
    num_pages = k_pool.shape[0]
    if k_pool.shape != (num_pages, page_size, Hkv, D) or v_pool.shape != k_pool.shape:
        raise ValueError("pool shape")
    st = _load(lib_path).oracle_qkv_append(
        qkv_bits.ctypes.data, wq_bits.ctypes.data, wk_bits.ctypes.data, block_table.ctypes.data,
        positions.ctypes.data, B, Hq, Hkv, D, int(bool(shared_kv)), page_size, block_table.shape[1],
        num_pages, float(theta), int(rope_pairs), float(eps), q_out.ctypes.data, k_pool.ctypes.data,
        v_pool.ctypes.data)
    if st != 0:
        raise OracleError("oracle_qkv_append: %s" % ERRORS.get(st, st))
    return q_out, k_pool, v_pool
