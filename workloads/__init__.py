"""Seeded synthetic inputs for paged decode attention.

This module is shared by the tests, the oracle checks and the benchmark; it
holds none of the attention arithmetic (no logits, softmax or weighted sums),
only the recipe that makes the inputs:

* Activations are drawn per head as N(0, 1), rounded to bf16 (the output of a
  bf16 projection), then RMS-normalised in fp32 and rounded back to bf16 with
  round-to-nearest-even.  q and k use the weighted norm ``x / rms(x) * w`` with
  one weight vector of length D per tensor, w ~ N(1, 0.1); v uses the unit
  norm ``x / rms(x)`` (Norm.lean ``rmsnorm`` / ``rmsnormUnit``; Gemma-4-12B
  model page, attn.qk_norm / attn.v_norm, eps 1e-6).
* Global layers keep one cache projection for K and V ("values = keys",
  ``attention_k_eq_v``): K = rmsnorm(x) * w_k and V = rmsnormUnit(x) of the same x.
* RoPE is not applied: a rotation of q and k changes no step of the kernel.
* The cache is a pool of pages of 16 token rows, [num_pages, 16, Hkv, D]
  (Gemma-4-12B shape domain: page size 16).  Physical page ids are a seeded
  random permutation; page 0 and the last page are guard pages.  Every slot
  that the decode query must not read (guard pages, slots past L - 1 in the
  last page, and positions before the window) is filled with bf16 NaN, so a
  read of any of them turns the output into NaN.
* ``window_only=True`` allocates only the pages that hold the last ``window``
  positions; earlier block-table entries are -1.

Every case is produced from ``torch.Generator(device).manual_seed(seed)``; a
case made on the CPU and one made on a GPU differ (different generators) but
each side of a comparison always reads the same realised tensors.
"""

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE_SIZE = 16
EPS = 1e-6
BF16_NAN_BITS = 0x7FC0

# Gemma-4-12B attention shapes (model page, "What to watch for" and attn.core rows)
SLIDING = dict(Hq=16, Hkv=8, D=256, window=1024)
GLOBAL = dict(Hq=16, Hkv=1, D=512, window=0)

N_LAYERS = 48  # layer i is global iff i % 6 == 5

# attn.rope per layer type (model page, "What to watch for" and the attn.rope
# rows): theta, and the number of active pairs (i, i + D/2)
ROPE = {"sliding": dict(theta=1.0e4, pairs=128), "global": dict(theta=1.0e6, pairs=64)}


def is_global_layer(i):
    return i % 6 == 5


@dataclass
class DecodeCase:
    """One decode-attention call: device tensors plus the host facts about them."""
    kind: str                 # "sliding" or "global"
    q: torch.Tensor           # bf16 [B, Hq, D]
    k_pool: torch.Tensor      # bf16 [num_pages, 16, Hkv, D]
    v_pool: torch.Tensor      # bf16 [num_pages, 16, Hkv, D]
    block_table: torch.Tensor  # int32 [B, max_blocks], -1 = unmapped
    seq_lens: torch.Tensor    # int32 [B]
    window: int               # > 0 sliding window, <= 0 none
    seq_lens_host: list = field(default_factory=list)
    seed: int = 0

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def Hkv(self):
        return self.k_pool.shape[2]

    @property
    def num_pages(self):
        return self.k_pool.shape[0]

    @property
    def max_blocks(self):
        return self.block_table.shape[1]

    @property
    def max_seq_len(self):
        return max(self.seq_lens_host) if self.seq_lens_host else 0

    def visible_positions(self):
        """Number of visible positions per sequence (host ints)."""
        w = self.window
        return [min(L, w) if w > 0 else L for L in self.seq_lens_host]

    def to(self, device):
        return DecodeCase(self.kind, self.q.to(device), self.k_pool.to(device),
                          self.v_pool.to(device), self.block_table.to(device),
                          self.seq_lens.to(device), self.window, list(self.seq_lens_host),
                          self.seed)


def bits(t):
    """uint16 numpy view of a bf16 tensor (bit patterns, for the oracle)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _rms_normalise(x, w=None):
    """x / sqrt(mean(x^2) + eps) [* w] over the last axis, in fp32."""
    x = x.float()
    y = x * torch.rsqrt(x.pow(2).mean(dim=-1, keepdim=True) + EPS)
    if w is not None:
        y = y * w.float()
    return y


def _randn_bf16(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def _norm_weight(D, gen, device):
    return (1.0 + 0.1 * torch.randn(D, generator=gen, device=device)).to(torch.bfloat16)


def key_weight(D, seed, device="cpu"):
    """A seeded qk_norm weight w_k ~ N(1, 0.1), bf16 [D] (values-only cache cases)."""
    return _norm_weight(D, torch.Generator(device=device).manual_seed(int(seed)), device)


def _allocated_pages(L, window, window_only):
    """Logical page indices that hold a cached position this call may need."""
    if L <= 0:
        return []
    last = (L - 1) // PAGE_SIZE
    first = 0
    if window_only and window > 0:
        first = max(0, L - window) // PAGE_SIZE
    return list(range(first, last + 1))


def make_case(kind, seq_lens, seed, device="cpu", window=None, window_only=False,
              k_eq_v=None, poison=True, max_blocks=None, Hq=None, Hkv=None, D=None,
              chunk_rows=1 << 22, layout_seed=None):
    """Build one decode case.

    kind        "sliding" (16/8 heads, D=256, window 1024) or "global" (16/1, D=512, no window)
    seq_lens    list of ints, one per sequence
    window      overrides the kind's window (> 0 sliding rule, <= 0 none)
    window_only allocate only the pages of the last `window` positions (-1 elsewhere)
    k_eq_v      K and V from one projection (default: True for global)
    poison      NaN-fill every slot the decode query must not read
    max_blocks  block-table width (default ceil(max(seq_lens)/16), at least 1)
    Hq/Hkv/D    override the head shape (tests of the oracle only)
    layout_seed seeds the page layout (block table) instead of `seed`: cases
                with the same lengths, window rule and layout_seed share one
                block table, as the layers of one cache layout do in a step
    """
    shape = dict(SLIDING if kind == "sliding" else GLOBAL)
    if window is not None:
        shape["window"] = window
    Hq = Hq or shape["Hq"]
    Hkv = Hkv or shape["Hkv"]
    D = D or shape["D"]
    window = shape["window"]
    if k_eq_v is None:
        k_eq_v = kind == "global"
    seq_lens = [int(L) for L in seq_lens]
    B = len(seq_lens)
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))

    max_L = max(seq_lens) if seq_lens else 0
    if max_blocks is None:
        max_blocks = max(1, -(-max_L // PAGE_SIZE))

    # logical pages per sequence, then a seeded permutation of physical ids 1..P-2
    alloc = [_allocated_pages(L, window, window_only) for L in seq_lens]
    n_alloc = sum(len(a) for a in alloc)
    num_pages = n_alloc + 2
    lseed = int(seed if layout_seed is None else layout_seed)
    perm = torch.randperm(n_alloc, generator=torch.Generator().manual_seed(lseed + 7)) + 1
    block_table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    i = 0
    for b, pages in enumerate(alloc):
        if pages:
            block_table[b, pages] = perm[i:i + len(pages)].to(torch.int32)
            i += len(pages)

    # weights (one length-D vector per tensor, shared by all heads)
    w_q = _norm_weight(D, gen, device)
    w_k = _norm_weight(D, gen, device)

    q = _rms_normalise(_randn_bf16((B, Hq, D), gen, device), w_q).to(torch.bfloat16)

    rows = num_pages * PAGE_SIZE * Hkv
    k_pool = torch.empty((rows, D), dtype=torch.bfloat16, device=device)
    v_pool = torch.empty((rows, D), dtype=torch.bfloat16, device=device)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = _randn_bf16((r1 - r0, D), gen, device)
        k_pool[r0:r1] = _rms_normalise(x, w_k).to(torch.bfloat16)
        if not k_eq_v:
            x = _randn_bf16((r1 - r0, D), gen, device)
        v_pool[r0:r1] = _rms_normalise(x).to(torch.bfloat16)
    k_pool = k_pool.view(num_pages, PAGE_SIZE, Hkv, D)
    v_pool = v_pool.view(num_pages, PAGE_SIZE, Hkv, D)

    if poison:
        _poison(k_pool, v_pool, block_table, seq_lens, window)

    return DecodeCase(kind, q, k_pool, v_pool, block_table.to(device),
                      torch.tensor(seq_lens, dtype=torch.int32, device=device), window,
                      list(seq_lens), int(seed))


def _poison(k_pool, v_pool, block_table, seq_lens, window):
    """NaN-fill every pool slot that no decode query of this case may read."""
    num_pages = k_pool.shape[0]
    visible = torch.zeros(num_pages * PAGE_SIZE, dtype=torch.bool)
    bt = block_table
    for b, L in enumerate(seq_lens):
        if L <= 0:
            continue
        lo = max(0, L - window) if window > 0 else 0
        pos = torch.arange(lo, L)
        phys = bt[b, pos // PAGE_SIZE].long()
        visible[phys * PAGE_SIZE + pos % PAGE_SIZE] = True
    dead = (~visible).nonzero().flatten().to(k_pool.device)
    nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
    kf = k_pool.view(num_pages * PAGE_SIZE, -1)
    vf = v_pool.view(num_pages * PAGE_SIZE, -1)
    kf.index_fill_(0, dead, nan)
    vf.index_fill_(0, dead, nan)


# ---------------------------------------------------------------------------
# The five workloads (seed 1000*cfg + layer)
# ---------------------------------------------------------------------------

def _uniform_ints(lo, hi, n, seed):
    g = torch.Generator().manual_seed(int(seed))
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def config_seq_lens(cfg, variant=None):
    """Host seq_lens of workload `cfg` (1..5), drawn from its own seed."""
    if cfg == 1:
        return [1, 17, 300, 1100]
    if cfg == 2:
        return _uniform_ints(1, 8192, 8, 1000 * cfg)
    if cfg == 3:
        return _uniform_ints(1024, 32768, 256, 1000 * cfg)
    if cfg == 4:
        return [262144] * 4 if variant == "b" else [131072] * 16
    if cfg == 5:
        g = torch.Generator().manual_seed(1000 * cfg)
        u = torch.rand(64, generator=g, dtype=torch.float64)
        lo, hi = math.log(16), math.log(262144)
        return [int(math.floor(math.exp(lo + (hi - lo) * x))) for x in u.tolist()]
    raise ValueError("unknown workload %r" % (cfg,))


def config_case(cfg, device="cpu", variant=None, layer=0, poison=True, seed_offset=0):
    """One call of workload `cfg`.  For cfg 5, `layer` picks the layer (0..47).

    seed_offset draws a different cache and query with the same lengths (the
    benchmark's rotating input sets)."""
    L = config_seq_lens(cfg, variant)
    seed = 1000 * cfg + layer + seed_offset
    if cfg == 1:
        return make_case("sliding", L, seed, device, poison=poison)
    if cfg == 2:
        return make_case("global", L, seed, device, poison=poison)
    if cfg == 3:
        return make_case("sliding", L, seed, device, window_only=True, poison=poison)
    if cfg == 4:
        return make_case("global", L, seed, device, poison=poison)
    if cfg == 5:
        # every layer of one type has its own cache and queries but the same
        # page layout (one block table per layer type, the layout of the
        # type's first layer: 0 sliding, 5 global)
        first = 5 if is_global_layer(layer) else 0
        layout = 1000 * cfg + first + seed_offset
        if is_global_layer(layer):
            return make_case("global", L, seed, device, poison=poison, layout_seed=layout)
        return make_case("sliding", L, seed, device, window_only=True, poison=poison, layout_seed=layout)
    raise ValueError("unknown workload %r" % (cfg,))


WORKLOADS = {
    1: "tiny sliding decode: B=4, seq_lens {1,17,300,1100}, 16/8 heads, D=256, window 1024",
    2: "global decode: B=8, seq_lens U[1,8192], 16/1 heads, D=512, no window",
    3: "sliding decode: B=256, seq_lens U[1024,32768], 16/8 heads, D=256, window 1024, window-only pages",
    4: "long-context global decode: B=16 x 131072 (variant b: B=4 x 262144), 16/1 heads, D=512",
    5: "Gemma-4-12B decode-step mix: B=64, seq_lens log-uniform [16,262144], 40 sliding + 8 global layers",
}


# ---------------------------------------------------------------------------
# One new token per sequence for the norm + RoPE + cache-append step
# ---------------------------------------------------------------------------

@dataclass
class AppendCase:
    """The attn.qkv_proj output of one new token per sequence, the qk_norm
    weights, the token positions, and a cache whose pages cover them."""
    kind: str
    qkv: torch.Tensor        # bf16 [B, Hq*D + 2*Hkv*D] (sliding) or [B, Hq*D + D] (global)
    w_q: torch.Tensor        # bf16 [D]
    w_k: torch.Tensor        # bf16 [D]
    positions: torch.Tensor  # int32 [B]
    cache: DecodeCase        # block table and pools; seq_lens = positions + 1

    @property
    def shared_kv(self):
        return self.kind == "global"

    def to(self, device):
        return AppendCase(self.kind, self.qkv.to(device), self.w_q.to(device), self.w_k.to(device),
                          self.positions.to(device), self.cache.to(device))


def append_row_len(kind):
    shape = SLIDING if kind == "sliding" else GLOBAL
    return shape["Hq"] * shape["D"] + (shape["D"] if kind == "global" else 2 * shape["Hkv"] * shape["D"])


def make_append_case(kind, positions, seed, device="cpu", scale=1.0, full_cache=False):
    """Tokens at `positions` (one per sequence), and a cache filled like
    make_case (no poison, so every other slot keeps a known value) whose pages
    cover each token's position: with full_cache every position 0..pos (for a
    decode after the append), else only the token's own page.
    qkv ~ N(0, scale^2) in bf16."""
    positions = [int(p) for p in positions]
    cache = make_case(kind, [p + 1 for p in positions], seed, device=device, poison=False,
                      **({} if full_cache else dict(window=1, window_only=True)))
    shape = SLIDING if kind == "sliding" else GLOBAL
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(int(seed) + 11)
    qkv = (scale * torch.randn((len(positions), append_row_len(kind)), generator=gen, device=device)).to(torch.bfloat16)
    w_q = _norm_weight(shape["D"], gen, device)
    w_k = _norm_weight(shape["D"], gen, device)
    return AppendCase(kind, qkv, w_q, w_k, torch.tensor(positions, dtype=torch.int32, device=device), cache)


# ---------------------------------------------------------------------------
# Multi-query (prefill) cases: the last q_len[b] tokens of each sequence query
# the paged cache, which already holds their keys and values
# ---------------------------------------------------------------------------

@dataclass
class PrefillCase:
    """Packed queries q [T, Hq, D] (sequence b owns rows cu_q[b] .. cu_q[b+1]-1,
    its last q_lens[b] tokens) and the paged cache they attend to."""
    kind: str
    q: torch.Tensor       # bf16 [T, Hq, D]
    cu_q: torch.Tensor    # int32 [B+1]
    q_lens: list
    cache: DecodeCase     # pools, block table, seq_lens (= every cached token), window

    @property
    def T(self):
        return self.q.shape[0]

    def to(self, device):
        return PrefillCase(self.kind, self.q.to(device), self.cu_q.to(device), list(self.q_lens),
                           self.cache.to(device))


def _poison_outside(k_pool, v_pool, block_table, first, seq_lens):
    """NaN-fill every pool slot outside positions [first[b], L_b) of every sequence."""
    num_pages = k_pool.shape[0]
    keep = torch.zeros(num_pages * PAGE_SIZE, dtype=torch.bool)
    for b, L in enumerate(seq_lens):
        if L <= first[b]:
            continue
        pos = torch.arange(first[b], L)
        phys = block_table[b, pos // PAGE_SIZE].long()
        keep[phys * PAGE_SIZE + pos % PAGE_SIZE] = True
    dead = (~keep).nonzero().flatten().to(k_pool.device)
    nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
    k_pool.view(num_pages * PAGE_SIZE, -1).index_fill_(0, dead, nan)
    v_pool.view(num_pages * PAGE_SIZE, -1).index_fill_(0, dead, nan)


def make_prefill_case(kind, seq_lens, q_lens, seed, device="cpu", window=None, window_only=False, poison=True,
                      Hq=None, Hkv=None, D=None):
    """Sequences of seq_lens[b] cached tokens whose last q_lens[b] (1 <= q_len <= L,
    or 0 for none) are queries.  The cache is built as by make_case; with
    window_only only the pages the queries can see are allocated.  With poison
    every slot no query may read is NaN: positions before the first query's
    window, and the unused tail of the last page.  q is rms-normalised times a
    weight vector, like the decode's q."""
    assert len(seq_lens) == len(q_lens) and all(0 <= n <= L for n, L in zip(q_lens, seq_lens))
    shape = dict(SLIDING if kind == "sliding" else GLOBAL)
    w = shape["window"] if window is None else window
    n_max = max(q_lens) if q_lens else 0
    # allocate as for one query whose window reaches back to the first query's
    alloc_window = w + max(n_max, 1) - 1 if w > 0 else w
    cache = make_case(kind, seq_lens, seed, device=device, window=alloc_window, window_only=window_only,
                      poison=False, Hq=Hq, Hkv=Hkv, D=D)
    cache.window = w
    if poison:
        first = [max(0, L - n - w + 1) if w > 0 else 0 for L, n in zip(seq_lens, q_lens)]
        _poison_outside(cache.k_pool, cache.v_pool, cache.block_table.cpu(), first, seq_lens)
    Hq_, D_ = cache.q.shape[1], cache.q.shape[2]
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(int(seed) + 23)
    T = sum(q_lens)
    w_q = _norm_weight(D_, gen, device)
    q = _rms_normalise(_randn_bf16((T, Hq_, D_), gen, device), w_q).to(torch.bfloat16)
    cu = [0]
    for n in q_lens:
        cu.append(cu[-1] + int(n))
    return PrefillCase(kind, q, torch.tensor(cu, dtype=torch.int32, device=device), [int(n) for n in q_lens], cache)
