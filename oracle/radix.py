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
