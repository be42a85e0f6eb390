"""Seeded synthetic inputs for prefix-shared KV attention.

This module only draws numbers and lays out index tables: Q/K/V values (fp32 N(0,1) rounded to
bf16, round-to-nearest-even), the random order in which pool slots are handed out, token ids and
request lengths.  It holds none of the method's arithmetic, so the fp64 oracle and the CUDA path
can both be fed from it without sharing any code that computes attention.

Workload shapes follow the pages' workloads:

* a shared system prompt followed by short per-user questions (prefix-caching comparison page,
  section on the 1,000-token common prefix and the 40-token question);
* shared prefixes of 2,000 and 16,000 tokens at sharing degree 16 (BatchLLM explainer, Global
  Prefix Sharing and the micro-benchmark table);
* a three-level radix tree (system prompt -> branches -> leaves) as in the RadixAttention tree
  figures of the SGLang explainer.

Every pool is "page size 1": each token owns one slot of ``[pool_size, num_kv_heads, head_dim]``
and slots are handed out in a random permutation, so neighbouring tokens never sit in
neighbouring slots.  Token ids of cached runs are drawn from [0, 16000) and those of new runs from
[16000, 32000), so a new token can never extend a cached match by chance.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

HEAD_DIM = 128
CACHED_TOKEN_RANGE = (0, 16000)
NEW_TOKEN_RANGE = (16000, 32000)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), round-to-nearest-even (inputs are finite)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_b = b.reshape(-1)
    flat_o = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_b.size, step):
        bb = flat_b[s:s + step]
        flat_o[s:s + step] = ((bb + (0x7FFF + ((bb >> 16) & 1))) >> 16).astype(np.uint16)
    return out


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32))


@dataclass
class Run:
    """A run of consecutive token positions and the pool slots holding their KV."""
    slots: np.ndarray            # int32 [n]
    tokens: np.ndarray           # int32 [n]
    cached: bool                 # True: KV already in the pool; False: stored during the step
    k: Optional[np.ndarray] = None   # uint16 [n, Hkv, d] for new runs
    v: Optional[np.ndarray] = None

    def __len__(self) -> int:
        return int(self.slots.shape[0])


@dataclass
class ExtendBatch:
    req_idx: np.ndarray          # int32 [B]   row of req_to_token for each request
    prefix_len: np.ndarray       # int32 [B]   cached tokens before the new ones
    extend_len: np.ndarray       # int32 [B]   new tokens
    cu_q: np.ndarray             # int32 [B+1] row offsets of each request in q/o
    q: np.ndarray                # uint16 [sum(extend_len), Hq, d]
    group_of_req: np.ndarray     # int32 [B]   -1 = no declared shared prefix
    group_prefix_len: np.ndarray  # int32 [G]
    tokens: List[np.ndarray] = field(default_factory=list)  # full token ids per request
    group_parent: Optional[np.ndarray] = None  # int32 [G], -1 = root; None = one level


@dataclass
class DecodeBatch:
    req_idx: np.ndarray          # int32 [B]
    seq_len: np.ndarray          # int32 [B]   keys 0..seq_len-1, the current token included
    q: np.ndarray                # uint16 [B, Hq, d]
    group_of_req: np.ndarray     # int32 [B]
    group_prefix_len: np.ndarray  # int32 [G]
    group_parent: Optional[np.ndarray] = None  # int32 [G], -1 = root; None = one level


@dataclass
class Step:
    store_slots: np.ndarray      # int32 [T]
    k_new: np.ndarray            # uint16 [T, Hkv, d]
    v_new: np.ndarray
    extend: Optional[ExtendBatch] = None
    decode: Optional[DecodeBatch] = None


@dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    softmax_scale: float
    pool_size: int
    req_to_token: np.ndarray     # int32 [R, W]
    k_pool: np.ndarray           # uint16 [P, Hkv, d], cached KV present, all else zero
    v_pool: np.ndarray
    steps: List[Step]
    cached_sequences: List[tuple] = field(default_factory=list)  # (tokens, slots) held by a cache
    recipe: str = ""


class Builder:
    """Allocates runs in a randomly permuted pool and assembles req_to_token rows.  page = 1: every
    token a random slot; page > 1: a run takes whole pages (slots page * P + i) drawn in a random
    page order, its last page possibly part-filled (block-granular pools)."""

    def __init__(self, rng: np.random.Generator, num_q_heads: int, num_kv_heads: int,
                 pool_size: int, head_dim: int = HEAD_DIM, page: int = 1, values: bool = True):
        # values=False: the same slots, lengths, tokens, new tokens' KV and queries, but no cached
        # KV is drawn or written into pools (structure-only checks of full-size workloads without
        # allocating their pools; device runs whose pools are filled on the GPU)
        self.values = values
        self.rng = rng
        # the values come from streams of their own, seeded from the structure stream: one for the
        # cached KV (not drawn at all by structure-only builds), one for the new tokens' KV and the
        # queries; so values=False changes no other draw and builds in a fraction of the time
        s_cached, s_new = rng.integers(0, 2 ** 63, size=2)
        self.crng = np.random.default_rng(int(s_cached))
        self.nrng = np.random.default_rng(int(s_new))
        self.hq, self.hkv, self.d = num_q_heads, num_kv_heads, head_dim
        self.pool_size = pool_size
        self.page = page
        self.perm = rng.permutation(pool_size // page).astype(np.int32)
        self.next = 0
        pool_rows = pool_size if values else 0
        self.k_pool = np.zeros((pool_rows, num_kv_heads, head_dim), dtype=np.uint16)
        self.v_pool = np.zeros((pool_rows, num_kv_heads, head_dim), dtype=np.uint16)
        self.rows: List[np.ndarray] = []

    def _alloc(self, n: int) -> np.ndarray:
        P = self.page
        pages = (n + P - 1) // P
        if self.next + pages > self.perm.shape[0]:
            raise ValueError(f"pool of {self.pool_size} slots exhausted")
        first = self.perm[self.next:self.next + pages].astype(np.int64)
        self.next += pages
        return (first[:, None] * P + np.arange(P)[None, :]).reshape(-1)[:n].astype(np.int32)

    def cached(self, n: int) -> Run:
        slots = self._alloc(n)
        tokens = self.rng.integers(*CACHED_TOKEN_RANGE, size=n).astype(np.int32)
        if self.values:
            shape = (n, self.hkv, self.d)
            self.k_pool[slots] = normal_bf16(self.crng, shape)
            self.v_pool[slots] = normal_bf16(self.crng, shape)
        return Run(slots, tokens, True)

    def new(self, n: int) -> Run:
        slots = self._alloc(n)
        tokens = self.rng.integers(*NEW_TOKEN_RANGE, size=n).astype(np.int32)
        shape = (n, self.hkv, self.d)
        return Run(slots, tokens, False, normal_bf16(self.nrng, shape),
                   normal_bf16(self.nrng, shape))

    def row(self, runs: Sequence[Run]) -> int:
        self.rows.append(np.concatenate([r.slots for r in runs]).astype(np.int32)
                         if runs else np.zeros(0, np.int32))
        return len(self.rows) - 1

    def q(self, n_rows: int) -> np.ndarray:
        return normal_bf16(self.nrng, (n_rows, self.hq, self.d))

    def finish(self, name: str, steps_spec, cached_sequences, recipe: str) -> Workload:
        """steps_spec: list of (new_runs, extend_spec, decode_spec) with row ids; rows are then
        placed at randomly permuted req_to_token indices."""
        n_rows = len(self.rows)
        width = max([len(r) for r in self.rows] + [1])
        table_rows = max(n_rows, 1)  # the library wants a table of at least one row
        width = (width + 15) // 16 * 16
        row_perm = self.rng.permutation(n_rows).astype(np.int32)
        r2t = np.zeros((table_rows, width), dtype=np.int32)
        for i, r in enumerate(self.rows):
            r2t[row_perm[i], :len(r)] = r
        steps = []
        for new_runs, ext, dec in steps_spec:
            if new_runs:
                slots = np.concatenate([r.slots for r in new_runs]).astype(np.int32)
                kn = np.concatenate([r.k for r in new_runs])
                vn = np.concatenate([r.v for r in new_runs])
            else:
                slots = np.zeros(0, np.int32)
                kn = np.zeros((0, self.hkv, self.d), np.uint16)
                vn = kn.copy()
            e = d = None
            if ext is not None:
                rows, pl, el, grp, gpl, toks = ext[:6]
                epar = np.asarray(ext[6], np.int32) if len(ext) > 6 else None
                el = np.asarray(el, np.int32)
                cu = np.zeros(len(el) + 1, np.int32)
                cu[1:] = np.cumsum(el)
                e = ExtendBatch(row_perm[np.asarray(rows, np.int64)].astype(np.int32),
                                np.asarray(pl, np.int32), el, cu, self.q(int(cu[-1])),
                                np.asarray(grp, np.int32), np.asarray(gpl, np.int32), toks, epar)
            if dec is not None:
                rows, sl, grp, gpl = dec[:4]
                dpar = np.asarray(dec[4], np.int32) if len(dec) > 4 else None
                d = DecodeBatch(row_perm[np.asarray(rows, np.int64)].astype(np.int32),
                                np.asarray(sl, np.int32), self.q(len(rows)),
                                np.asarray(grp, np.int32), np.asarray(gpl, np.int32), dpar)
            steps.append(Step(slots, kn, vn, e, d))
        return Workload(name, self.hq, self.hkv, self.d, 1.0 / float(np.sqrt(self.d)),
                        self.pool_size, r2t, self.k_pool, self.v_pool, steps,
                        cached_sequences, recipe)


def _tokens(runs: Sequence[Run]) -> np.ndarray:
    return np.concatenate([r.tokens for r in runs]).astype(np.int32)


def _slots(runs: Sequence[Run]) -> np.ndarray:
    return np.concatenate([r.slots for r in runs]).astype(np.int32)


# --------------------------------------------------------------------------------------------
# Generic shapes used by the named workloads and by the parity tests.
# --------------------------------------------------------------------------------------------

def extend_workload(seed: int, num_q_heads: int, num_kv_heads: int, *, n_groups: int,
                    members: int, prefix: int, ext_lo: int, ext_hi: int,
                    own_cached_hi: int = 0, ungrouped: int = 0, ungrouped_prefix: int = 0,
                    pool_size: Optional[int] = None, name: str = "extend",
                    values: bool = True) -> Workload:
    """Groups of `members` requests share a cached `prefix`; each request may also hold
    U[0, own_cached_hi] cached tokens of its own, then extends U[ext_lo, ext_hi] new tokens.
    `ungrouped` more requests have their own cached prefix of `ungrouped_prefix` tokens."""
    rng = np.random.default_rng(seed)
    n_req = n_groups * members + ungrouped
    ext = rng.integers(ext_lo, ext_hi + 1, size=n_req)
    own = rng.integers(0, own_cached_hi + 1, size=n_req) if own_cached_hi > 0 else np.zeros(n_req, np.int64)
    need = n_groups * prefix + int(ext.sum()) + int(own.sum()) + ungrouped * ungrouped_prefix
    P = pool_size if pool_size is not None else max(4096, 1 << int(np.ceil(np.log2(need * 1.25 + 1))))
    b = Builder(rng, num_q_heads, num_kv_heads, P, values=values)
    rows, pl, grp, toks, new_runs, cached_seqs = [], [], [], [], [], []
    gpl = []
    i = 0
    for g in range(n_groups):
        pre = b.cached(prefix) if prefix > 0 else None
        gpl.append(prefix)
        if pre is not None:
            cached_seqs.append((pre.tokens.copy(), pre.slots.copy()))
        for _ in range(members):
            runs = [pre] if pre is not None else []
            if own[i] > 0:
                runs.append(b.cached(int(own[i])))
                cached_seqs.append((_tokens(runs), _slots(runs)))
            nr = b.new(int(ext[i]))
            new_runs.append(nr)
            rows.append(b.row(runs + [nr]))
            pl.append(sum(len(r) for r in runs))
            grp.append(g)
            toks.append(_tokens(runs + [nr]))
            i += 1
    for _ in range(ungrouped):
        runs = [b.cached(ungrouped_prefix)] if ungrouped_prefix > 0 else []
        if runs:
            cached_seqs.append((_tokens(runs), _slots(runs)))
        nr = b.new(int(ext[i]))
        new_runs.append(nr)
        rows.append(b.row(runs + [nr]))
        pl.append(ungrouped_prefix)
        grp.append(-1)
        toks.append(_tokens(runs + [nr]))
        i += 1
    recipe = (f"seed {seed}; Hq={num_q_heads} Hkv={num_kv_heads} d=128; {n_groups} groups x "
              f"{members} requests on a cached {prefix}-token prefix; own cached U[0,{own_cached_hi}];"
              f" new U[{ext_lo},{ext_hi}]; {ungrouped} ungrouped (prefix {ungrouped_prefix});"
              f" pool {P} slots, random permutation")
    return b.finish(name, [(new_runs, (rows, pl, [len(r) for r in new_runs], grp, gpl, toks), None)],
                    cached_seqs, recipe)


def decode_workload(seed: int, num_q_heads: int, num_kv_heads: int, *, n_groups: int,
                    members: int, prefix: int, dist_lo: int, dist_hi: int,
                    ungrouped: int = 0, min_pool: int = 0, name: str = "decode",
                    values: bool = True) -> Workload:
    """Groups of `members` requests share a cached `prefix`; each request holds U[dist_lo,
    dist_hi] distinct tokens of which the last is the current token (stored in the step).
    `ungrouped` more requests hold only distinct tokens."""
    rng = np.random.default_rng(seed)
    n_req = n_groups * members + ungrouped
    dist = rng.integers(dist_lo, dist_hi + 1, size=n_req)
    need = n_groups * prefix + int(dist.sum())
    P = max(min_pool, need) if min_pool else max(4096, 1 << int(np.ceil(np.log2(need * 1.25 + 1))))
    b = Builder(rng, num_q_heads, num_kv_heads, P, values=values)
    rows, sl, grp, gpl, new_runs, cached_seqs = [], [], [], [], [], []
    i = 0
    for g in range(n_groups):
        pre = b.cached(prefix) if prefix > 0 else None
        gpl.append(prefix)
        if pre is not None:
            cached_seqs.append((pre.tokens.copy(), pre.slots.copy()))
        for _ in range(members):
            runs = [pre] if pre is not None else []
            if dist[i] > 1:
                runs.append(b.cached(int(dist[i]) - 1))
            cur = b.new(1)
            new_runs.append(cur)
            rows.append(b.row(runs + [cur]))
            sl.append(prefix + int(dist[i]))
            grp.append(g)
            i += 1
    for _ in range(ungrouped):
        runs = [b.cached(int(dist[i]) - 1)] if dist[i] > 1 else []
        cur = b.new(1)
        new_runs.append(cur)
        rows.append(b.row(runs + [cur]))
        sl.append(int(dist[i]))
        grp.append(-1)
        i += 1
    recipe = (f"seed {seed}; Hq={num_q_heads} Hkv={num_kv_heads} d=128; {n_groups} groups x "
              f"{members} requests on a cached {prefix}-token prefix; distinct U[{dist_lo},{dist_hi}]"
              f" incl. the current token; {ungrouped} ungrouped; pool {P} slots, random permutation")
    return b.finish(name, [(new_runs, None, (rows, sl, grp, gpl))], cached_seqs, recipe)


def paged_workload(seed: int, num_q_heads: int, num_kv_heads: int, *, page: int, prefix: int,
                   n_req: int, ext_lo: int, ext_hi: int, name: str = "paged",
                   values: bool = True) -> Workload:
    """Block-granular pool (prefix-caching comparison page: vLLM keeps KV in blocks and reuses only
    whole blocks).  n_req requests share a cached `prefix` of which only floor(prefix / page) *
    page tokens -- whole pages -- are reused; each request recomputes the rest of the prefix and
    its U[ext_lo, ext_hi] new tokens in pages of its own (one extend step), then decodes one token
    (a second step)."""
    rng = np.random.default_rng(seed)
    shared = prefix // page * page
    ext = rng.integers(ext_lo, ext_hi + 1, size=n_req)
    need_pages = shared // page + int(sum((prefix - shared + e + 1 + page - 1) // page + 1 for e in ext))
    P = max(4096, 1 << int(np.ceil(np.log2(need_pages * page * 1.25 + 1))))
    b = Builder(rng, num_q_heads, num_kv_heads, P, page=page, values=values)
    pre = b.cached(shared) if shared > 0 else None
    cached_seqs = [(pre.tokens.copy(), pre.slots.copy())] if pre is not None else []
    new_runs, rows, pl, el, toks, cur_runs = [], [], [], [], [], []
    for i in range(n_req):
        nr = b.new(prefix - shared + int(ext[i]))
        new_runs.append(nr)
        runs = ([pre] if pre is not None else []) + [nr]
        rows.append(b.row(runs))
        pl.append(shared)
        el.append(int(len(nr)))
        toks.append(_tokens(runs))
    d_rows, d_sl, d_runs = [], [], []
    for i in range(n_req):
        cur = b.new(1)
        d_runs.append(cur)
        runs = ([pre] if pre is not None else []) + [new_runs[i], cur]
        d_rows.append(b.row(runs))
        d_sl.append(shared + len(new_runs[i]) + 1)
    grp = [0 if shared > 0 else -1] * n_req
    steps = [(new_runs, (rows, pl, el, grp, [shared], toks), None),
             (d_runs, None, (d_rows, d_sl, grp, [shared]))]
    recipe = (f"seed {seed}; Hq={num_q_heads} Hkv={num_kv_heads} d=128; pages of {page} slots in "
              f"random page order; {n_req} requests on a {prefix}-token prefix of which {shared} "
              f"(whole pages) are reused; extend U[{ext_lo},{ext_hi}] new tokens, then one decode "
              f"step; pool {P} slots")
    return b.finish(name, steps, cached_seqs, recipe)


def tree_workload(seed: int, num_q_heads: int, num_kv_heads: int, *, depth: int, fanout: int,
                  seg_lo: int, seg_hi: int, p_empty: float, n_decode: int, tail_hi: int,
                  n_extend: int, own_hi: int, ext_lo: int, ext_hi: int,
                  name: str = "tree", values: bool = True) -> Workload:
    """A random radix tree of cached segments (a node's segment U[seg_lo, seg_hi] tokens, empty
    with probability p_empty; 1..fanout children per node down to `depth` levels) declared as a
    group forest.  Decode requests sit on random nodes with U[0, tail_hi] cached tokens of their
    own plus the current token; extend requests sit on random nodes with U[0, own_hi] cached tokens
    of their own and U[ext_lo, ext_hi] new ones."""
    rng = np.random.default_rng(seed)
    parent, seg_len = [-1], [int(rng.integers(seg_lo, seg_hi + 1))]
    frontier = [0]
    for _ in range(depth - 1):
        nxt = []
        for nd in frontier:
            for _ in range(int(rng.integers(1, fanout + 1))):
                parent.append(nd)
                seg_len.append(0 if rng.random() < p_empty else int(rng.integers(seg_lo, seg_hi + 1)))
                nxt.append(len(parent) - 1)
        frontier = nxt
    n_nodes = len(parent)
    dec_node = rng.integers(0, n_nodes, size=n_decode)
    dec_tail = rng.integers(0, tail_hi + 1, size=n_decode)
    ext_node = rng.integers(0, n_nodes, size=n_extend)
    ext_own = rng.integers(0, own_hi + 1, size=n_extend)
    ext_new = rng.integers(ext_lo, ext_hi + 1, size=n_extend)
    need = sum(seg_len) + int(dec_tail.sum()) + n_decode + int(ext_own.sum()) + int(ext_new.sum())
    P = max(4096, 1 << int(np.ceil(np.log2(need * 1.25 + 1))))
    b = Builder(rng, num_q_heads, num_kv_heads, P, values=values)
    runs = [b.cached(n) if n > 0 else None for n in seg_len]
    plen = []
    for nd in range(n_nodes):
        plen.append((plen[parent[nd]] if parent[nd] >= 0 else 0) + seg_len[nd])

    def path(nd):
        out = []
        while nd >= 0:
            if runs[nd] is not None:
                out.append(runs[nd])
            nd = parent[nd]
        return out[::-1]

    cached_seqs = [(_tokens(path(nd)), _slots(path(nd))) for nd in range(n_nodes) if plen[nd] > 0]
    new_runs = []
    e_rows, e_pl, e_el, e_grp, e_toks = [], [], [], [], []
    for i in range(n_extend):
        nd = int(ext_node[i])
        rr = path(nd) + ([b.cached(int(ext_own[i]))] if ext_own[i] > 0 else [])
        nr = b.new(int(ext_new[i]))
        new_runs.append(nr)
        e_rows.append(b.row(rr + [nr]))
        e_pl.append(plen[nd] + int(ext_own[i]))
        e_el.append(int(ext_new[i]))
        e_grp.append(nd)
        e_toks.append(_tokens(rr + [nr]))
    d_rows, d_sl, d_grp = [], [], []
    for i in range(n_decode):
        nd = int(dec_node[i])
        rr = path(nd) + ([b.cached(int(dec_tail[i]))] if dec_tail[i] > 0 else [])
        cur = b.new(1)
        new_runs.append(cur)
        d_rows.append(b.row(rr + [cur]))
        d_sl.append(plen[nd] + int(dec_tail[i]) + 1)
        d_grp.append(nd)
    step = (new_runs, (e_rows, e_pl, e_el, e_grp, plen, e_toks, parent) if n_extend else None,
            (d_rows, d_sl, d_grp, plen, parent) if n_decode else None)
    recipe = (f"seed {seed}; Hq={num_q_heads} Hkv={num_kv_heads} d=128; radix tree of {n_nodes} "
              f"nodes, depth {depth}, fanout 1..{fanout}, segments U[{seg_lo},{seg_hi}] (empty "
              f"with p={p_empty}); {n_decode} decode on random nodes, tail U[0,{tail_hi}] + current; "
              f"{n_extend} extend, own U[0,{own_hi}], new U[{ext_lo},{ext_hi}]; pool {P} slots")
    return b.finish(name, [step], cached_seqs, recipe)


# --------------------------------------------------------------------------------------------
# The five named workloads.
# --------------------------------------------------------------------------------------------

def chunked_prefill_workload(seed: int, num_q_heads: int, num_kv_heads: int, *, system: int,
                             prompt: int, chunk: int, n_decode: int, tail_lo: int, tail_hi: int,
                             name: str = "chunked-prefill", values: bool = True) -> Workload:
    """Mixed token batching with chunked prefill: after a cached system prompt of `system` tokens,
    one request's `prompt`-token prompt is prefilled `chunk` tokens per step; in every step
    `n_decode` running requests (the same system prompt, then an own cached tail of U[tail_lo,
    tail_hi] tokens) decode one token each.  A chunk is an extend whose prefix is the system prompt
    plus the chunks before it, so each step's extend attends over everything already computed."""
    rng = np.random.default_rng(seed)
    n_steps = (prompt + chunk - 1) // chunk
    pool = system + prompt + n_decode * (tail_hi + n_steps) + 64
    pool = max(4096, (pool + 1023) // 1024 * 1024)
    b = Builder(rng, num_q_heads, num_kv_heads, pool, values=values)
    sp = b.cached(system)
    chunks = [b.new(min(chunk, prompt - i * chunk)) for i in range(n_steps)]
    tails = [b.cached(int(rng.integers(tail_lo, tail_hi + 1))) for _ in range(n_decode)]
    dec_new = [[b.new(1) for _ in range(n_steps)] for _ in range(n_decode)]
    long_row = b.row([sp] + chunks)
    dec_rows = [b.row([sp, tails[j]] + dec_new[j]) for j in range(n_decode)]
    steps = []
    for st in range(n_steps):
        done = system + sum(len(c.slots) for c in chunks[:st])
        new_runs = [chunks[st]] + [dec_new[j][st] for j in range(n_decode)]
        ext = ([long_row], [done], [len(chunks[st].slots)], [0], [done],
               [_tokens([sp] + chunks[:st + 1])])
        seq = [system + len(tails[j].slots) + st + 1 for j in range(n_decode)]
        dec = (dec_rows, seq, [0] * n_decode, [system]) if n_decode else None
        steps.append((new_runs, ext, dec))
    cached = [(sp.tokens.copy(), sp.slots.copy())]
    for j in range(n_decode):
        cached.append((_tokens([sp, tails[j]]), _slots([sp, tails[j]])))
    return b.finish(name, steps, cached,
                    f"seed {seed}; Hq={num_q_heads} Hkv={num_kv_heads} d=128; cached system prompt "
                    f"{system}; one {prompt}-token prompt prefilled {chunk} tokens per step over "
                    f"{n_steps} steps; {n_decode} decode requests (system prompt + own tail "
                    f"U[{tail_lo},{tail_hi}]) decode one token per step; pool {pool} slots, "
                    f"random permutation")


def llama3_chunked_prefill(seed: int = 1006, values: bool = True) -> Workload:
    """32 q / 8 kv heads; a 6144-token prompt prefilled 2048 tokens per step beside 64 decode
    requests on a shared 1024-token system prompt (own tails U[200,1000])."""
    return chunked_prefill_workload(seed, 32, 8, system=1024, prompt=6144, chunk=2048,
                                    n_decode=64, tail_lo=200, tail_hi=1000,
                                    name="llama3-chunked-prefill-6144x2048-64dec",
                                    values=values)


def tiny(seed: int = 1001, values: bool = True) -> Workload:
    """8 q / 2 kv heads; one cached 1000-token prefix in a 4096-slot pool; 4 requests extend 40
    new tokens each (causal), then 8 decode steps of one token per request."""
    rng = np.random.default_rng(seed)
    b = Builder(rng, 8, 2, 4096, values=values)
    pre = b.cached(1000)
    ext = [b.new(40) for _ in range(4)]
    dec = [[b.new(1) for _ in range(8)] for _ in range(4)]
    rows = [b.row([pre, ext[i]] + dec[i]) for i in range(4)]
    toks = [_tokens([pre, ext[i]]) for i in range(4)]
    steps = [(ext, (rows, [1000] * 4, [40] * 4, [0] * 4, [1000], toks), None)]
    for s in range(8):
        steps.append(([dec[i][s] for i in range(4)], None,
                      (rows, [1041 + s] * 4, [0] * 4, [1000])))
    return b.finish("tiny-8q2kv-p1000", steps, [(pre.tokens.copy(), pre.slots.copy())],
                    f"seed {seed}; Hq=8 Hkv=2 d=128; cached prefix 1000; 4 x 40 extend; "
                    f"8 decode steps; pool 4096 slots, random permutation")


def llama7b_extend(seed: int = 1002, values: bool = True) -> Workload:
    """32/32 heads; 4 groups x 16 requests on a cached 2000-token prefix; each extends U[40,200]."""
    return extend_workload(seed, 32, 32, n_groups=4, members=16, prefix=2000, ext_lo=40,
                           ext_hi=200, pool_size=32768, name="llama7b-extend-4x16-p2000",
                           values=values)


def llama7b_paged(seed: int = 1007, values: bool = True) -> Workload:
    """The extend workload's shape on a block-granular pool: 32/32 heads, pages of 16 slots in
    random page order; 64 requests on a 2000-token prefix (all of it whole pages, so all reused),
    each extending U[40,200] new tokens in pages of its own; then one decode step."""
    return paged_workload(seed, 32, 32, page=16, prefix=2000, n_req=64, ext_lo=40, ext_hi=200,
                          name="llama7b-paged16-64-p2000", values=values)


def llama7b_decode_hf(seed: int = 1003, values: bool = True) -> Workload:
    """32/32 heads; 16 groups x 16 requests on a 2000-token prefix; distinct U[100,500]."""
    return decode_workload(seed, 32, 32, n_groups=16, members=16, prefix=2000, dist_lo=100,
                           dist_hi=500, name="llama7b-decode-16x16-p2000", values=values)


def llama3_gqa_decode(seed: int = 1004, values: bool = True) -> Workload:
    """32 q / 8 kv heads; 16 groups x 16 requests on a 16000-token prefix; distinct U[200,1000];
    pool of at least 409,600 slots."""
    return decode_workload(seed, 32, 8, n_groups=16, members=16, prefix=16000, dist_lo=200,
                           dist_hi=1000, min_pool=409600, name="llama3-gqa-decode-16x16-p16000",
                           values=values)


def radix_mixed(seed: int = 1005, tree: bool = True, values: bool = True) -> Workload:
    """Radix tree 1000 -> 8 x 500 -> 4 x 200 per branch (32 leaves).  One step: 16 leaf requests
    extend 64 tokens; 8 cache misses run a 1500-token full prefill; 40 decode requests, request j on
    leaf j mod 32 with its own tail of U[1,32] tokens (the last one current).
    tree=True declares the radix tree as groups (root = system prompt, 8 branch nodes, 32 leaf
    nodes for decode; extend requests belong to their branch node); tree=False declares only the
    system prompt, one level."""
    rng = np.random.default_rng(seed)
    tails = rng.integers(1, 33, size=40)
    b = Builder(rng, 32, 32, 32768, values=values)
    sysp = b.cached(1000)
    branch = [b.cached(500) for _ in range(8)]
    leaf = [b.cached(200) for _ in range(32)]
    paths = [[sysp, branch[k // 4], leaf[k]] for k in range(32)]
    cached_seqs = [(_tokens(p), _slots(p)) for p in paths]
    new_runs, e_rows, e_pl, e_el, e_grp, e_toks = [], [], [], [], [], []
    for k in range(16):
        nr = b.new(64)
        new_runs.append(nr)
        e_rows.append(b.row(paths[k] + [nr]))
        e_pl.append(1700); e_el.append(64); e_grp.append(0)
        e_toks.append(_tokens(paths[k] + [nr]))
    for _ in range(8):
        nr = b.new(1500)
        new_runs.append(nr)
        e_rows.append(b.row([nr]))
        e_pl.append(0); e_el.append(1500); e_grp.append(-1)
        e_toks.append(nr.tokens.copy())
    d_rows, d_sl = [], []
    for j in range(40):
        runs = list(paths[j % 32])
        if tails[j] > 1:
            tail = b.cached(int(tails[j]) - 1)
            runs.append(tail)
            cached_seqs.append((_tokens(runs), _slots(runs)))
        cur = b.new(1)
        new_runs.append(cur)
        d_rows.append(b.row(runs + [cur]))
        d_sl.append(1700 + int(tails[j]))
    if tree:
        # groups: 0 root [0,1000), 1..8 branch b [1000,1500), 9..40 leaf k [1500,1700)
        gpl = [1000] + [1500] * 8 + [1700] * 32
        par = [-1] + [0] * 8 + [1 + k // 4 for k in range(32)]
        e_spec = (e_rows, e_pl, e_el, [1 + k // 4 for k in range(16)] + [-1] * 8, gpl, e_toks, par)
        d_spec = (d_rows, d_sl, [9 + j % 32 for j in range(40)], gpl, par)
    else:
        e_spec = (e_rows, e_pl, e_el, e_grp, [1000], e_toks)
        d_spec = (d_rows, d_sl, [0] * 40, [1000])
    step = (new_runs, e_spec, d_spec)
    return b.finish("radix-mixed-1000-8x500-32x200" + ("" if tree else "-1level"), [step],
                    cached_seqs,
                    f"seed {seed}; Hq=Hkv=32 d=128; tree 1000 -> 8x500 -> 32x200; 16 extend "
                    f"(p=1700, E=64) + 8 miss (p=0, E=1500) + 40 decode (tail U[1,32]); "
                    + ("groups = the radix tree (system prompt, branches, leaves)" if tree else
                       "shared-prefix groups at the 1000-token system prompt only")
                    + "; pool 32768 slots")


NAMED = {
    "tiny": tiny,
    "extend": llama7b_extend,
    "decode": llama7b_decode_hf,
    "gqa-decode": llama3_gqa_decode,
    "radix-mixed": radix_mixed,
    "radix-mixed-1level": lambda values=True: radix_mixed(tree=False, values=values),
    "chunked-prefill": llama3_chunked_prefill,
    "paged": llama7b_paged,
}
