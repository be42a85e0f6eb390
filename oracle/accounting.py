"""Oracle for the pages' token-accounting closed forms.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""
from __future__ import annotations


def compute_reduction(l_prefix: float, l_new: float) -> float:
    """Fraction of prefill compute removed by a cache hit on an l_prefix-token prefix followed by
    l_new new tokens: l_prefix / (l_prefix + l_new) (SGLang explainer, "キャッシュヒット率の定量的
    効果", Reduction formula)."""
    return l_prefix / (l_prefix + l_new)


def token_saving_ratio(n_processed: float, n_logical: float) -> float:
    """BatchLLM token-saving ratio, percent: (1 - processed / logical) * 100 (BatchLLM explainer,
    Global Prefix Sharing, Equation 2)."""
    return (1.0 - n_processed / n_logical) * 100.0


def hit_rate(cached_prompt_tokens: float, prompt_tokens: float) -> float:
    """Cache hit rate = cached prompt tokens / prompt tokens (SGLang paper notes §3,
    cache-aware scheduling, definition)."""
    return cached_prompt_tokens / prompt_tokens


def optimal_hit_rate(tree_edge_tokens: float, prefill_tokens_total: float) -> float:
    """Hit rate when every tree edge's KV is computed exactly once (DFS order, Theorem 3.1):
    1 - C / sum over requests of prefill tokens, C = total tokens on the tree's edges
    (SGLang paper notes, App. A.3)."""
    return 1.0 - tree_edge_tokens / prefill_tokens_total


def merge_gain(leaves: int, tokens: int) -> int:
    """BatchLLM merge gain of a grandchild node: (leaves - 1) * tokens (BatchLLM explainer,
    Global Prefix Sharing, merge criterion)."""
    return (leaves - 1) * tokens
