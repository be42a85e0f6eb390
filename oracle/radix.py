"""Oracle for prefix matching on a token-granular (page size 1) KV cache.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages' prefix match walks a radix tree from the root and returns the matched token count and
the KV pages of the matched tokens, reusing their KV and computing only the rest (SGLang explainer,
"主要な操作: プレフィックスマッチング").  A hit needs agreement from the very first token; the
number of tokens saved is the leading matched count floored to the engine's match unit: 16-token
blocks in vLLM, 1-token pages in SGLang (prefix-caching comparison page, "要点" and the worked
example of the 1,000-token common prefix: 992 at unit 16, 1,000 at unit 1).

The oracle is the plain definition rather than a radix tree: an uncompressed trie with one node
per token, each node holding the slot of that token's KV.  A stored prefix keeps the slots of the
first sequence that stored it (later sequences reuse the cached KV, as a radix tree insert would).
match() returns the longest stored prefix of the query, floored to the unit.
"""
from __future__ import annotations


class PrefixStore:
    def __init__(self):
        self._root = {}          # token -> [slot, children dict]
        self._n = 0

    def insert(self, tokens, slots):
        node = self._root
        for t, s in zip(tokens, slots):
            t = int(t)
            if t not in node:
                node[t] = [int(s), {}]
                self._n += 1
            node = node[t][1]

    def _walk(self, tokens):
        node, slots = self._root, []
        for t in tokens:
            nxt = node.get(int(t))
            if nxt is None:
                break
            slots.append(nxt[0])
            node = nxt[1]
        return slots

    def longest(self, tokens) -> int:
        return len(self._walk(tokens))

    def match(self, tokens, unit: int = 1):
        """(tokens saved at `unit`, their slots)."""
        if unit < 1:
            raise ValueError("match unit must be >= 1")
        slots = self._walk(tokens)
        saved = (len(slots) // unit) * unit
        return saved, slots[:saved]

    def __len__(self):
        return self._n


class LRURadixCache:
    """Plain model of the radix cache's memory management, for checking the library's.

    Pages: SGLang explainer, "LRU退避" (when memory runs short, free the least recently accessed
    leaves of the radix tree, recursively, starting with leaves whose reference count is 0, so
    caches in use stay protected); SGLang paper notes §3 (LRU on leaf nodes; a node is reclaimed
    only when its reference count is 0; the cache shares one memory pool with the running
    requests) and Figure 3 (nine steps of inserts, reuse, splits and evictions).

    Readings (the pages do not fix these details): a logical clock advances on every insert and
    every acquire, and stamps the nodes on that call's path; an acquire splits the edge at the
    end of the prefix it saves, so that exactly those tokens form the held nodes; among leaves of
    equal age the node created first goes first.  The tree is a list-based radix tree; every
    search is a linear scan.
    """

    class _Node:
        def __init__(self, toks, slots, parent, last, nid):
            self.toks, self.slots, self.kids = list(toks), list(slots), []
            self.parent, self.last, self.ref, self.id = parent, last, 0, nid

    def __init__(self):
        self._clock = 0
        self._ids = 0
        self.root = self._Node([], [], None, 0, 0)

    def _new(self, toks, slots, parent, last):
        self._ids += 1
        return self._Node(toks, slots, parent, last, self._ids)

    def _child(self, node, tok):
        for k in node.kids:
            if k.toks[0] == tok:
                return k
        return None

    def _split(self, node, c):
        """node keeps toks[c:]; a new node with toks[:c] takes its place under its parent."""
        inner = self._new(node.toks[:c], node.slots[:c], node.parent, node.last)
        inner.ref = node.ref
        pa = node.parent
        pa.kids[pa.kids.index(node)] = inner
        node.toks, node.slots, node.parent = node.toks[c:], node.slots[c:], inner
        inner.kids.append(node)
        return inner

    @staticmethod
    def _common(a, b):
        i = 0
        while i < len(a) and i < len(b) and a[i] == b[i]:
            i += 1
        return i

    def _walk(self, tokens):
        """matched token count and their slots (no changes)."""
        node, pos, slots = self.root, 0, []
        while pos < len(tokens):
            k = self._child(node, tokens[pos])
            if k is None:
                break
            c = self._common(tokens[pos:], k.toks)
            slots += k.slots[:c]
            pos += c
            if c < len(k.toks):
                break
            node = k
        return pos, slots

    def insert(self, tokens, slots):
        tokens, slots = [int(t) for t in tokens], [int(s) for s in slots]
        self._clock += 1
        node, pos = self.root, 0
        while pos < len(tokens):
            k = self._child(node, tokens[pos])
            if k is None:
                node.kids.append(self._new(tokens[pos:], slots[pos:], node, self._clock))
                return len(tokens) - pos
            c = self._common(tokens[pos:], k.toks)
            if c < len(k.toks):
                k = self._split(k, c)
            k.last = self._clock
            pos += c
            node = k
        return 0

    def acquire(self, tokens, unit=1, lock=True):
        tokens = [int(t) for t in tokens]
        m, slots = self._walk(tokens)
        s = m // unit * unit
        self._clock += 1
        node, pos = self.root, 0
        while pos < s:
            k = self._child(node, tokens[pos])
            if s - pos < len(k.toks):
                k = self._split(k, s - pos)
            k.last = self._clock
            if lock:
                k.ref += 1
            pos += len(k.toks)
            node = k
        return s, slots[:s]

    def release(self, tokens):
        tokens = [int(t) for t in tokens]
        node, pos, path = self.root, 0, []
        while pos < len(tokens):
            k = self._child(node, tokens[pos])
            if k is None or tokens[pos:pos + len(k.toks)] != k.toks or k.ref < 1:
                raise ValueError("not a held path")
            path.append(k)
            pos += len(k.toks)
            node = k
        for k in path:
            k.ref -= 1

    def _nodes(self):
        out, stack = [], list(self.root.kids)
        while stack:
            k = stack.pop()
            out.append(k)
            stack += k.kids
        return out

    def evict(self, n_tokens):
        """Slots freed, in eviction order: repeatedly the least recently used unheld leaf."""
        freed = []
        while len(freed) < n_tokens:
            leaves = [k for k in self._nodes() if not k.kids and k.ref == 0]
            if not leaves:
                break
            k = min(leaves, key=lambda x: (x.last, x.id))
            freed += k.slots
            k.parent.kids.remove(k)
        return freed

    def stats(self):
        nodes = self._nodes()
        return sum(len(k.toks) for k in nodes), len(nodes)

    def match(self, tokens, unit=1):
        m, slots = self._walk([int(t) for t in tokens])
        s = m // unit * unit
        return s, slots[:s]


def edge_tokens(sequences) -> int:
    """Tokens on the edges of the batch's radix tree = the batch's distinct prefixes: the least a
    batch must compute, each edge's KV once (SGLang paper notes, App. A.3, proof of Theorem 3.1)."""
    return len({tuple(q[:i + 1]) for q in sequences for i in range(len(q))})


def computed_tokens(sequences, order, capacity) -> int:
    """Prefill tokens computed when the batch runs in `order` through an LRU radix cache of
    `capacity` tokens: each request reuses its cached prefix (held while it runs), computes the
    rest, and enters the cache, the least recently used unheld leaves making room."""
    cache = LRURadixCache()
    total = 0
    slot = 0
    for r in order:
        q = [int(t) for t in sequences[r]]
        hit, _ = cache.acquire(q, 1, True)
        need = len(q) - hit
        over = cache.stats()[0] + need - capacity
        if over > 0:
            cache.evict(over)
        cache.insert(q, list(range(slot, slot + len(q))))
        slot += len(q)
        cache.release(q[:hit])
        total += need
    return total


def longest_prefix_first(sequences, capacity):
    """Order chosen online: next the waiting request with the longest cached prefix (ties: lower
    index), with the cache of computed_tokens (SGLang paper notes, §3: longest-shared-prefix-first
    instead of first-come-first-served)."""
    cache = LRURadixCache()
    waiting = list(range(len(sequences)))
    order, slot = [], 0
    while waiting:
        best = max(waiting, key=lambda r: (cache.match(sequences[r])[0], -r))
        waiting.remove(best)
        order.append(best)
        q = [int(t) for t in sequences[best]]
        hit, _ = cache.acquire(q, 1, True)
        over = cache.stats()[0] + len(q) - hit - capacity
        if over > 0:
            cache.evict(over)
        cache.insert(q, list(range(slot, slot + len(q))))
        slot += len(q)
        cache.release(q[:hit])
    return order
