"""Paged decode attention for the Gemma-4-12B text path on GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/attn_decode.h``; every
function here only checks and marshals arguments (torch tensors -> device
pointers) and calls the library of the same name.  All arithmetic runs in
the CUDA kernels of ``libattn_decode.so``; there is no CPU path.  The library
is built in-tree by ``_build.build()`` (or ``__graft_entry__.build()``); when
it is missing, ``load()`` raises instead of falling back to anything.

    attn_decode_sliding(q, k_pool, v_pool, block_table, seq_lens, ...)  -> o
    attn_decode_global(q, k_pool, v_pool, block_table, seq_lens, ...)   -> o
"""

import ctypes
import os

import torch

from . import _build

__all__ = [
    "attn_decode_sliding", "attn_decode_global", "attn_decode_global_shared", "attn_decode_plan",
    "attn_decode_workspace_size", "attn_decode_launches", "new_workspace", "WORKSPACE_ZERO_BYTES",
    "PreparedDecode", "prepare_decode_sliding", "prepare_decode_global", "prepare_decode_global_shared", "Step",
    "attn_last_error", "load", "library_path", "AttnDecodeError",
    "KIND_SLIDING", "KIND_GLOBAL", "DEV_WAIT_TIMEOUT", "DEV_BAD_PAGE", "DEV_BAD_SEQ_LEN",
]

ATTN_OK = 0
ERROR_NAMES = {1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_WORKSPACE",
               4: "ATTN_ERR_CUDA"}
OUT_BF16, OUT_F32 = 0, 1
KIND_SLIDING, KIND_GLOBAL = 0, 1
DEV_WAIT_TIMEOUT, DEV_BAD_PAGE, DEV_BAD_SEQ_LEN, DEV_INTERNAL = 1, 2, 4, 8
PAGE_SIZE = 16
WORKSPACE_ZERO_BYTES = 8192  # ATTN_WORKSPACE_ZERO_BYTES: zero before a workspace's first use, kept zero
SHAPES = {KIND_SLIDING: (16, 8, 256), KIND_GLOBAL: (16, 1, 512)}  # Hq, Hkv, D

EXPORTS = ("attn_decode_sliding", "attn_decode_global", "attn_decode_global_shared", "attn_decode_plan",
           "attn_decode_workspace_size", "attn_decode_launches", "attn_kv_append_sliding", "attn_kv_append_global",
           "attn_prefill_sliding", "attn_prefill_global",
           "attn_step_create", "attn_step_destroy", "attn_step_add_decode_sliding", "attn_step_add_decode_global",
           "attn_step_add_decode_global_shared", "attn_step_add_kv_append_sliding", "attn_step_add_kv_append_global",
           "attn_step_num_calls", "attn_step_num_kernels", "attn_step_set_launch_mode", "attn_step_launch_mode",
           "attn_step_finalize", "attn_step_launch", "attn_last_error", "attn_abi_version")
# attn_step launch modes (attn_step.h)
STEP_LAUNCH_AUTO, STEP_LAUNCH_GRAPH, STEP_LAUNCH_DIRECT = 0, 1, 2
STEP_LAUNCH_MODES = {"auto": STEP_LAUNCH_AUTO, "graph": STEP_LAUNCH_GRAPH, "direct": STEP_LAUNCH_DIRECT}
APPEND_ROW = {KIND_SLIDING: 16 * 256 + 2 * 8 * 256, KIND_GLOBAL: 16 * 512 + 512}  # qkv row length


class AttnDecodeError(RuntimeError):
    def __init__(self, code, message):
        super().__init__("%s: %s" % (ERROR_NAMES.get(code, "error %d" % code), message))
        self.code = code


_lib = None


def library_path():
    return _build.LIB_PATH


def load(path=None):
    """Load libattn_decode.so (built in-tree); raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError("CUDA library %s is not built; run __graft_entry__.build() "
                           "(there is no CPU fallback)" % p)
    lib = ctypes.CDLL(p)
    c_i32, c_i64, c_vp, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    call = [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,       # q k_pool v_pool block_table seq_lens o
            c_i32, c_i32, c_i64, c_i32, c_i32, c_i32,  # batch max_blocks num_pages max_seq_len window out_dtype
            c_i32, c_vp, c_sz, c_vp, c_vp]             # num_splits workspace workspace_bytes status stream
    for name in ("attn_decode_sliding", "attn_decode_global"):
        fn = getattr(lib, name)
        fn.restype = c_i32
        fn.argtypes = call
    lib.attn_decode_global_shared.restype = c_i32
    lib.attn_decode_global_shared.argtypes = call[:2] + [c_vp] + call[3:]  # q kv_pool w_k block_table ...
    lib.attn_decode_plan.restype = c_i32
    lib.attn_decode_plan.argtypes = [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32,
                                     ctypes.POINTER(c_i32), ctypes.POINTER(c_sz)]
    lib.attn_decode_workspace_size.restype = c_sz
    lib.attn_decode_workspace_size.argtypes = [c_i32, c_i32, c_i32, c_i32, c_i32]
    lib.attn_decode_launches.restype = c_i32
    lib.attn_decode_launches.argtypes = [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32]
    app = [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,  # qkv w_q w_k block_table positions q_out k_pool v_pool
           c_i32, c_i32, c_i64, c_vp, c_vp]                 # batch max_blocks num_pages status stream
    for name in ("attn_kv_append_sliding", "attn_kv_append_global"):
        fn = getattr(lib, name)
        fn.restype = c_i32
        fn.argtypes = app
    pre = [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,  # q k_pool v_pool block_table seq_lens cu_q o
           c_i32, c_i32, c_i32, c_i32, c_i64,          # batch total_q max_q max_blocks num_pages
           c_i32, c_i32, c_vp, c_vp]                   # window out_dtype status stream
    for name in ("attn_prefill_sliding", "attn_prefill_global"):
        fn = getattr(lib, name)
        fn.restype = c_i32
        fn.argtypes = pre
    c_step = ctypes.c_void_p
    lib.attn_step_create.restype = c_i32
    lib.attn_step_create.argtypes = [ctypes.POINTER(c_step)]
    lib.attn_step_destroy.restype = None
    lib.attn_step_destroy.argtypes = [c_step]
    for name in ("attn_step_add_decode_sliding", "attn_step_add_decode_global", "attn_step_add_decode_global_shared"):
        fn = getattr(lib, name)
        fn.restype = c_i32
        fn.argtypes = [c_step] + call[:-1]
    for name in ("attn_step_add_kv_append_sliding", "attn_step_add_kv_append_global"):
        fn = getattr(lib, name)
        fn.restype = c_i32
        fn.argtypes = [c_step] + app[:-1]
    for name in ("attn_step_num_calls", "attn_step_num_kernels", "attn_step_finalize"):
        fn = getattr(lib, name)
        fn.restype = c_i32
        fn.argtypes = [c_step]
    lib.attn_step_set_launch_mode.restype = c_i32
    lib.attn_step_set_launch_mode.argtypes = [c_step, c_i32]
    lib.attn_step_launch_mode.restype = c_i32
    lib.attn_step_launch_mode.argtypes = [c_step]
    lib.attn_step_launch.restype = c_i32
    lib.attn_step_launch.argtypes = [c_step, c_vp]
    lib.attn_selftest_delayed_copy.restype = c_i32
    lib.attn_selftest_delayed_copy.argtypes = [c_vp, c_vp, c_i64, c_i32, c_vp]
    lib.attn_last_error.restype = ctypes.c_char_p
    lib.attn_last_error.argtypes = []
    lib.attn_abi_version.restype = c_i32
    lib.attn_abi_version.argtypes = []
    if path is None:
        _lib = lib
    return lib


def attn_last_error():
    return load().attn_last_error().decode()


def attn_decode_plan(kind, batch, max_seq_len, window, num_splits=0, num_sms=152):
    """(num_splits, workspace_bytes) the library would use; pure host arithmetic."""
    lib = load()
    ns = ctypes.c_int32(0)
    ws = ctypes.c_size_t(0)
    st = lib.attn_decode_plan(kind, batch, max_seq_len, window, num_splits, num_sms,
                              ctypes.byref(ns), ctypes.byref(ws))
    if st != ATTN_OK:
        raise AttnDecodeError(st, attn_last_error())
    return ns.value, ws.value


def attn_decode_workspace_size(kind, batch, max_seq_len, window, num_splits=0):
    """Workspace bytes for the current CUDA device."""
    lib = load()
    n = lib.attn_decode_workspace_size(kind, batch, max_seq_len, window, num_splits)
    err = attn_last_error()
    if n == 0 and err:
        raise AttnDecodeError(1, err)
    return n


def attn_decode_launches(kind, batch, max_seq_len, window, num_splits=0, num_sms=152):
    """Kernels one decode call launches: 1 (split sequences merged in the decode kernel) or 2 (and a combine)."""
    n = load().attn_decode_launches(kind, batch, max_seq_len, window, num_splits, num_sms)
    if n < 0:
        raise AttnDecodeError(1, attn_last_error())
    return n


def new_workspace(nbytes, device):
    """A decode workspace of nbytes: its first WORKSPACE_ZERO_BYTES zeroed, as a first use requires."""
    ws = torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)
    ws[:WORKSPACE_ZERO_BYTES].zero_()
    return ws


def _ptr(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device.type != "cuda":
        raise ValueError("%s must be a CUDA tensor (there is no CPU path)" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t.data_ptr()


def _decode_args(kind, q, k_pool, v_pool, block_table, seq_lens, o, window, max_seq_len, out_dtype,
                 num_splits, workspace, status, w_k=None):
    """Checked, marshalled arguments of one decode call (everything but the stream).

    Returns (args, keep, o, fn_name): the C arguments, the tensors they point
    into (to be kept alive), the output tensor and the C entry point."""
    Hq, Hkv, D = SHAPES[kind]
    if q.dim() != 3:
        raise ValueError("q must be [batch, %d, %d]" % (Hq, D))
    batch = q.shape[0]
    if k_pool.dim() != 4:
        raise ValueError("k_pool must be [num_pages, 16, %d, %d]" % (Hkv, D))
    num_pages = k_pool.shape[0]
    if block_table.dim() != 2:
        raise ValueError("block_table must be [batch, max_blocks]")
    max_blocks = block_table.shape[1]
    args_q = _ptr(q, "q", torch.bfloat16, (batch, Hq, D))
    args_k = _ptr(k_pool, "k_pool", torch.bfloat16, (num_pages, PAGE_SIZE, Hkv, D))
    args_v = _ptr(v_pool, "v_pool", torch.bfloat16, (num_pages, PAGE_SIZE, Hkv, D))
    if w_k is not None:
        args_v = _ptr(w_k, "w_k", torch.bfloat16, (D,))
    args_bt = _ptr(block_table, "block_table", torch.int32, (batch, max_blocks))
    args_sl = _ptr(seq_lens, "seq_lens", torch.int32, (batch,))
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out_dtype must be torch.bfloat16 or torch.float32")
    if o is None:
        o = torch.empty((batch, Hq, D), dtype=out_dtype, device=q.device)
    args_o = _ptr(o, "o", o.dtype, (batch, Hq, D))
    if max_seq_len is None:
        max_seq_len = max_blocks * PAGE_SIZE
    if workspace is None:
        with torch.cuda.device(q.device):
            need = attn_decode_workspace_size(kind, batch, max_seq_len, window, num_splits)
        workspace = new_workspace(need, q.device)
    ws_ptr = _ptr(workspace, "workspace", torch.uint8)
    st_ptr = None if status is None else _ptr(status, "status", torch.int32, (1,))
    fn_name = ("attn_decode_sliding" if kind == KIND_SLIDING else
               "attn_decode_global" if w_k is None else "attn_decode_global_shared")
    args = (args_q, args_k, args_v, args_bt, args_sl, args_o, batch, max_blocks, num_pages, int(max_seq_len),
            int(window), OUT_F32 if o.dtype == torch.float32 else OUT_BF16, int(num_splits), ws_ptr,
            workspace.numel(), st_ptr)
    keep = (q, k_pool, v_pool, block_table, seq_lens, o, workspace, status, w_k)
    return args, keep, o, fn_name


def _stream_ptr(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _call(kind, q, k_pool, v_pool, block_table, seq_lens, o, window, max_seq_len, out_dtype,
          num_splits, workspace, status, stream, w_k=None):
    args, _, o, fn_name = _decode_args(kind, q, k_pool, v_pool, block_table, seq_lens, o, window, max_seq_len,
                                       out_dtype, num_splits, workspace, status, w_k)
    s_ptr = _stream_ptr(stream, q.device)
    with torch.cuda.device(q.device):
        st = getattr(load(), fn_name)(*args, s_ptr)
    if st != ATTN_OK:
        raise AttnDecodeError(st, attn_last_error())
    return o


class PreparedDecode:
    """A decode call whose arguments are checked and marshalled once.

    For a serving loop that calls the same buffers every step: construction
    validates the tensors exactly as the one-shot functions do and keeps their
    device pointers; ``run(stream)`` then costs one C call.  The tensors must
    stay alive and in place (the object keeps references to them); their
    contents may change between runs.
    """

    def __init__(self, kind, q, k_pool, v_pool, block_table, seq_lens, o=None, *, window, max_seq_len=None,
                 out_dtype=torch.bfloat16, num_splits=0, workspace=None, status=None, w_k=None):
        self._args, self._keep, self.o, fn_name = _decode_args(
            kind, q, k_pool, v_pool, block_table, seq_lens, o, window, max_seq_len, out_dtype, num_splits,
            workspace, status, w_k)
        self._fn = getattr(load(), fn_name)

    def run(self, stream):
        """Enqueue the call on `stream` (a torch.cuda.Stream or a raw cudaStream_t); returns o."""
        s_ptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        st = self._fn(*self._args, s_ptr)
        if st != ATTN_OK:
            raise AttnDecodeError(st, attn_last_error())
        return self.o


class Step:
    """The attention calls of a decode step, recorded once and replayed with one call.

    ``add_*`` take the arguments of the one-shot function of the same name
    (minus the stream), validate them at once and return the call's output
    tensor (o, or q_out for the appends).  ``finalize(mode)`` records the
    calls' kernel launches, in the order added, on the current CUDA device;
    ``launch(stream)`` then enqueues the whole step with one C call: one CUDA
    graph launch (mode "graph"), or the recorded launches back to back (mode
    "direct"); "auto" picks direct for steps of up to two calls.  The tensors
    are used in place (the object keeps references to them); their contents
    may change between launches.
    """

    def __init__(self):
        self._lib = load()
        h = ctypes.c_void_p()
        self._check(self._lib.attn_step_create(ctypes.byref(h)))
        self._h = h
        self._keep = []
        self.device = None

    def _check(self, rc):
        if rc != ATTN_OK:
            raise AttnDecodeError(rc, attn_last_error())

    def _add_decode(self, kind, fn_name, q, k_pool, v_pool, block_table, seq_lens, o, window, max_seq_len=None,
                    out_dtype=torch.bfloat16, num_splits=0, workspace=None, status=None, w_k=None):
        args, keep, o, name = _decode_args(kind, q, k_pool, v_pool, block_table, seq_lens, o, window, max_seq_len,
                                           out_dtype, num_splits, workspace, status, w_k)
        with torch.cuda.device(q.device):
            self._check(getattr(self._lib, fn_name)(self._h, *args))
        self._keep.append(keep)
        self.device = q.device
        return o

    def add_decode_sliding(self, q, k_pool, v_pool, block_table, seq_lens, o=None, *, window=1024, **kw):
        return self._add_decode(KIND_SLIDING, "attn_step_add_decode_sliding", q, k_pool, v_pool, block_table,
                                seq_lens, o, window, **kw)

    def add_decode_global(self, q, k_pool, v_pool, block_table, seq_lens, o=None, *, window=0, **kw):
        return self._add_decode(KIND_GLOBAL, "attn_step_add_decode_global", q, k_pool, v_pool, block_table,
                                seq_lens, o, window, **kw)

    def add_decode_global_shared(self, q, kv_pool, w_k, block_table, seq_lens, o=None, *, window=0, **kw):
        return self._add_decode(KIND_GLOBAL, "attn_step_add_decode_global_shared", q, kv_pool, kv_pool, block_table,
                                seq_lens, o, window, w_k=w_k, **kw)

    def _add_append(self, kind, fn_name, qkv, w_q, w_k, block_table, positions, k_pool, v_pool, q_out, status):
        args, keep, q_out, _ = _append_args(kind, qkv, w_q, w_k, block_table, positions, k_pool, v_pool, q_out,
                                            status)
        with torch.cuda.device(qkv.device):
            self._check(getattr(self._lib, fn_name)(self._h, *args))
        self._keep.append(keep)
        self.device = qkv.device
        return q_out

    def add_kv_append_sliding(self, qkv, w_q, w_k, block_table, positions, k_pool, v_pool, q_out=None, *,
                              status=None):
        return self._add_append(KIND_SLIDING, "attn_step_add_kv_append_sliding", qkv, w_q, w_k, block_table,
                                positions, k_pool, v_pool, q_out, status)

    def add_kv_append_global(self, qkv, w_q, w_k, block_table, positions, k_pool, v_pool, q_out=None, *,
                             status=None):
        return self._add_append(KIND_GLOBAL, "attn_step_add_kv_append_global", qkv, w_q, w_k, block_table,
                                positions, k_pool, v_pool, q_out, status)

    @property
    def num_calls(self):
        return self._lib.attn_step_num_calls(self._h)

    @property
    def num_kernels(self):
        return self._lib.attn_step_num_kernels(self._h)

    def finalize(self, mode="auto"):
        """Record the step's launches; mode is "auto", "graph" or "direct"."""
        if mode not in STEP_LAUNCH_MODES:
            raise ValueError("mode must be one of %s" % ", ".join(STEP_LAUNCH_MODES))
        if self.device is None:
            raise AttnDecodeError(1, "no calls recorded")
        self._check(self._lib.attn_step_set_launch_mode(self._h, STEP_LAUNCH_MODES[mode]))
        with torch.cuda.device(self.device):
            self._check(self._lib.attn_step_finalize(self._h))
        return self

    @property
    def launch_mode(self):
        """"graph" or "direct" once finalized (before: the mode requested)."""
        m = self._lib.attn_step_launch_mode(self._h)
        return {v: k for k, v in STEP_LAUNCH_MODES.items()}.get(m)

    def launch(self, stream=None):
        """Enqueue the whole step on `stream` (default: the current stream of its device)."""
        self._check(self._lib.attn_step_launch(self._h, _stream_ptr(stream, self.device)))

    def close(self):
        if self._h is not None and self._h.value:
            self._lib.attn_step_destroy(self._h)
        self._h = None
        self._keep = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def prepare_decode_sliding(q, k_pool, v_pool, block_table, seq_lens, o=None, *, window=1024, **kw):
    """PreparedDecode for attn_decode_sliding (same arguments, minus the stream)."""
    return PreparedDecode(KIND_SLIDING, q, k_pool, v_pool, block_table, seq_lens, o, window=window, **kw)


def prepare_decode_global(q, k_pool, v_pool, block_table, seq_lens, o=None, *, window=0, **kw):
    """PreparedDecode for attn_decode_global (same arguments, minus the stream)."""
    return PreparedDecode(KIND_GLOBAL, q, k_pool, v_pool, block_table, seq_lens, o, window=window, **kw)


def prepare_decode_global_shared(q, kv_pool, w_k, block_table, seq_lens, o=None, *, window=0, **kw):
    """PreparedDecode for attn_decode_global_shared (same arguments, minus the stream)."""
    return PreparedDecode(KIND_GLOBAL, q, kv_pool, kv_pool, block_table, seq_lens, o, window=window, w_k=w_k, **kw)


def attn_decode_sliding(q, k_pool, v_pool, block_table, seq_lens, o=None, *, window=1024,
                        max_seq_len=None, out_dtype=torch.bfloat16, num_splits=0, workspace=None,
                        status=None, stream=None):
    """slidingDecodeGQA: q [B,16,256], pools [P,16,8,256] bf16 -> o [B,16,256].

    max_seq_len: host bound on seq_lens for the split plan (default max_blocks*16).
    workspace:   uint8 CUDA tensor of at least attn_decode_workspace_size(...) bytes whose first
                 WORKSPACE_ZERO_BYTES were zero at its first use (new_workspace); allocated per
                 call when None.
    status:      optional int32 [1] CUDA tensor receiving ATTN_DEV_* bits.
    """
    return _call(KIND_SLIDING, q, k_pool, v_pool, block_table, seq_lens, o, window, max_seq_len,
                 out_dtype, num_splits, workspace, status, stream)


def attn_decode_global(q, k_pool, v_pool, block_table, seq_lens, o=None, *, window=0,
                       max_seq_len=None, out_dtype=torch.bfloat16, num_splits=0, workspace=None,
                       status=None, stream=None):
    """decodeGQA: q [B,16,512], pools [P,16,1,512] bf16 -> o [B,16,512] (window <= 0: none)."""
    return _call(KIND_GLOBAL, q, k_pool, v_pool, block_table, seq_lens, o, window, max_seq_len,
                 out_dtype, num_splits, workspace, status, stream)


def attn_decode_global_shared(q, kv_pool, w_k, block_table, seq_lens, o=None, *, window=0,
                              max_seq_len=None, out_dtype=torch.bfloat16, num_splits=0, workspace=None,
                              status=None, stream=None):
    """decodeGQA over a values-only cache: kv_pool [P,16,1,512] holds V; keys are
    rebuilt in the kernel as bf16(rope(V * w_k)), w_k [512] bf16.  Otherwise as
    attn_decode_global."""
    return _call(KIND_GLOBAL, q, kv_pool, kv_pool, block_table, seq_lens, o, window, max_seq_len,
                 out_dtype, num_splits, workspace, status, stream, w_k=w_k)


def _append_args(kind, qkv, w_q, w_k, block_table, positions, k_pool, v_pool, q_out, status):
    """Checked, marshalled arguments of one append call: (args, keep, q_out, fn_name)."""
    Hq, Hkv, D = SHAPES[kind]
    batch, max_blocks, num_pages = qkv.shape[0], block_table.shape[1], v_pool.shape[0]
    args = [_ptr(qkv, "qkv", torch.bfloat16, (batch, APPEND_ROW[kind])),
            _ptr(w_q, "w_q", torch.bfloat16, (D,)),
            _ptr(w_k, "w_k", torch.bfloat16, (D,)),
            _ptr(block_table, "block_table", torch.int32, (batch, max_blocks)),
            _ptr(positions, "positions", torch.int32, (batch,))]
    if q_out is None:
        q_out = torch.empty((batch, Hq, D), dtype=torch.bfloat16, device=qkv.device)
    args += [_ptr(q_out, "q_out", torch.bfloat16, (batch, Hq, D)),
             None if k_pool is None and kind == KIND_GLOBAL else
             _ptr(k_pool, "k_pool", torch.bfloat16, (num_pages, PAGE_SIZE, Hkv, D)),
             _ptr(v_pool, "v_pool", torch.bfloat16, (num_pages, PAGE_SIZE, Hkv, D))]
    st_ptr = None if status is None else _ptr(status, "status", torch.int32, (1,))
    args += [batch, max_blocks, num_pages, st_ptr]
    fn_name = "attn_kv_append_sliding" if kind == KIND_SLIDING else "attn_kv_append_global"
    keep = (qkv, w_q, w_k, block_table, positions, q_out, k_pool, v_pool, status)
    return tuple(args), keep, q_out, fn_name


def _append(kind, qkv, w_q, w_k, block_table, positions, k_pool, v_pool, q_out, status, stream):
    args, _, q_out, fn_name = _append_args(kind, qkv, w_q, w_k, block_table, positions, k_pool, v_pool, q_out,
                                           status)
    rc = getattr(load(), fn_name)(*args, _stream_ptr(stream, qkv.device))
    if rc != ATTN_OK:
        raise AttnDecodeError(rc, attn_last_error())
    return q_out


def attn_kv_append_sliding(qkv, w_q, w_k, block_table, positions, k_pool, v_pool, q_out=None, *, status=None,
                           stream=None):
    """Norms, RoPE and cache append of one token per sequence (sliding layers).

    qkv [B, 8192] bf16 = [q 16x256 | k 8x256 | v 8x256]; w_q, w_k [256] bf16;
    positions [B] int32.  Writes each token's key and value into k_pool /
    v_pool at page block_table[b, pos/16], row pos % 16; returns q_out [B,16,256].
    """
    return _append(KIND_SLIDING, qkv, w_q, w_k, block_table, positions, k_pool, v_pool, q_out, status, stream)


def attn_kv_append_global(qkv, w_q, w_k, block_table, positions, k_pool, v_pool, q_out=None, *, status=None,
                          stream=None):
    """Norms, RoPE and cache append of one token per sequence (global layers).

    qkv [B, 8704] bf16 = [q 16x512 | x 512], x giving both key and value
    (values = keys); w_q, w_k [512] bf16.  Returns q_out [B,16,512].
    k_pool None: a values-only cache (attn_decode_global_shared); only V is written.
    """
    return _append(KIND_GLOBAL, qkv, w_q, w_k, block_table, positions, k_pool, v_pool, q_out, status, stream)



def _prefill(kind, q, k_pool, v_pool, block_table, seq_lens, cu_q, o, max_q, window, out_dtype, status, stream):
    Hq, Hkv, D = SHAPES[kind]
    if q.dim() != 3:
        raise ValueError("q must be [total_q, %d, %d]" % (Hq, D))
    total_q, batch = q.shape[0], seq_lens.shape[0]
    num_pages, max_blocks = k_pool.shape[0], block_table.shape[1]
    if max_q is None:
        counts = (cu_q[1:] - cu_q[:-1]).cpu()   # host bound for the grid (synchronises)
        max_q = int(counts.max().item()) if counts.numel() else 0
    if o is None:
        o = torch.empty((total_q, Hq, D), dtype=out_dtype, device=q.device)
    code = {torch.bfloat16: OUT_BF16, torch.float32: OUT_F32}.get(o.dtype)
    if code is None:
        raise ValueError("o must be bf16 or fp32")
    args = [_ptr(q, "q", torch.bfloat16, (total_q, Hq, D)),
            _ptr(k_pool, "k_pool", torch.bfloat16, (num_pages, PAGE_SIZE, Hkv, D)),
            _ptr(v_pool, "v_pool", torch.bfloat16, (num_pages, PAGE_SIZE, Hkv, D)),
            _ptr(block_table, "block_table", torch.int32, (batch, max_blocks)),
            _ptr(seq_lens, "seq_lens", torch.int32, (batch,)),
            _ptr(cu_q, "cu_q", torch.int32, (batch + 1,)),
            _ptr(o, "o", o.dtype, (total_q, Hq, D))]
    st_ptr = None if status is None else _ptr(status, "status", torch.int32, (1,))
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    s_ptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    lib = load()
    fn = lib.attn_prefill_sliding if kind == KIND_SLIDING else lib.attn_prefill_global
    rc = fn(*args, batch, total_q, int(max_q), max_blocks, num_pages, int(window), code, st_ptr, s_ptr)
    if rc != ATTN_OK:
        raise AttnDecodeError(rc, attn_last_error())
    return o


def attn_prefill_sliding(q, k_pool, v_pool, block_table, seq_lens, cu_q, o=None, *, max_q=None, window=1024,
                         out_dtype=torch.bfloat16, status=None, stream=None):
    """slidingGQA for the last n tokens of each sequence (n = cu_q[b+1] - cu_q[b]):
    q [total_q,16,256] packed by sequence, pools as for the decode -> o [total_q,16,256].
    max_q: host bound on n (read from cu_q, with a synchronisation, when None)."""
    return _prefill(KIND_SLIDING, q, k_pool, v_pool, block_table, seq_lens, cu_q, o, max_q, window, out_dtype,
                    status, stream)


def attn_prefill_global(q, k_pool, v_pool, block_table, seq_lens, cu_q, o=None, *, max_q=None, window=0,
                        out_dtype=torch.bfloat16, status=None, stream=None):
    """causalGQA for the last n tokens of each sequence: q [total_q,16,512] -> o [total_q,16,512]."""
    return _prefill(KIND_GLOBAL, q, k_pool, v_pool, block_table, seq_lens, cu_q, o, max_q, window, out_dtype,
                    status, stream)

def selftest_delayed_copy(dst, src, delay_ns=5000, stream=None):
    """attn_selftest_delayed_copy: copy src into dst (same-size int32 CUDA tensors)
    from a kernel that lets the next kernel launch first and copies after
    delay_ns.  For tests of the launch order."""
    if dst.dtype != torch.int32 or src.dtype != torch.int32 or dst.shape != src.shape:
        raise ValueError("dst and src must be int32 tensors of one shape")
    if not (dst.is_cuda and src.is_cuda and dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("dst and src must be contiguous CUDA tensors")
    if stream is None:
        stream = torch.cuda.current_stream(dst.device)
    s_ptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    rc = load().attn_selftest_delayed_copy(dst.data_ptr(), src.data_ptr(), dst.numel() * 4, int(delay_ns), s_ptr)
    if rc != ATTN_OK:
        raise AttnDecodeError(rc, attn_last_error())
