"""fp64 oracle: page-1 KV pool scatter and attention with a cached prefix.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain float64 numpy; a matrix product is
used as a library step and nothing is blocked, fused or reordered.

What is computed, and where the pages fix it
--------------------------------------------
* The KV cache lives on the GPU in pages of one token; a tree node refers to the pages of its
  tokens (SGLang explainer, "RadixAttention: Radix Tree による KV キャッシュ管理"; LMSYS blog
  translation, RadixAttention backend; SGLang paper notes §3, cache storage).  So a request's keys
  are the pool rows named, position by position, by its row of the request->slot table.
* The KV of a token depends only on the tokens before it, so a request whose first p tokens are
  cached attends exactly as if it had recomputed them (SGLang paper notes, App. A.1; prefix-caching
  comparison page: prefix caching does not change the model's output).  Extend therefore computes
  causal attention of the new tokens over [cached prefix + new tokens]; only the unmatched part is
  computed (SGLang explainer, prefix matching: "only the unmatched part is newly computed").
* Decode is one query per request over all of its keys (prefix-caching comparison page, the
  definitions of prefill and decode).  Horizontal fusion splits those keys into the shared prefix
  and the request's own part and computes them in different thread blocks (BatchLLM explainer,
  Horizontal Fusion); the parts are recombined by the log-sum-exp merge below.  Grouping never
  changes the result, so the oracle ignores it and attends over the full row.

Readings where the pages are silent: scale 1/sqrt(d); query head h uses KV head h // (Hq/Hkv);
LSE is the natural log of sum_j exp(scale q.k_j); the current decode token attends to itself; new
row i of an extend (0-based) sees key positions 0 .. prefix_len + i.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def store_kv(k_pool: np.ndarray, v_pool: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
             slots: np.ndarray):
    """Page-1 pool scatter: the KV of new token t goes to pool row slots[t].  Bit copies."""
    k = k_pool.copy()
    v = v_pool.copy()
    for t in range(len(slots)):
        k[slots[t]] = k_new[t]
        v[slots[t]] = v_new[t]
    return k, v


def attend(q: np.ndarray, keys: np.ndarray, vals: np.ndarray, visible: np.ndarray, scale: float):
    """softmax attention of query rows over key rows, per the definition.

    q [n, d], keys [L, d], vals [L, d] float64; visible [n, L] bool.
    Returns o [n, d] = sum_j softmax_j(scale q.k_j) v_j over visible j, and
    lse [n] = log sum_j exp(scale q.k_j).  A row with no visible key gets o = 0, lse = -inf.
    """
    n, L = visible.shape
    s = scale * (q @ keys.T)
    s = np.where(visible, s, -np.inf)
    o = np.zeros((n, q.shape[1]))
    lse = np.full(n, -np.inf)
    has = visible.any(axis=1)
    if has.any():
        sh = s[has]
        m = sh.max(axis=1, keepdims=True)
        p = np.exp(sh - m)
        l = p.sum(axis=1, keepdims=True)
        o[has] = (p @ vals) / l
        lse[has] = (m + np.log(l))[:, 0]
    return o, lse


def _gather(pool_bits: np.ndarray, slots: np.ndarray) -> np.ndarray:
    return bf16_to_f64(pool_bits[np.asarray(slots, dtype=np.int64)])


def extend(q, k_pool, v_pool, req_to_token, req_idx, prefix_len, extend_len, cu_q, scale,
           requests=None):
    """Extend (prefill with a cached prefix) attention.

    q [sum E, Hq, d] bf16 bits with request r's new rows at cu_q[r]..cu_q[r+1];
    k_pool, v_pool [P, Hkv, d] bf16 bits (the new tokens' KV already stored);
    request r's key positions 0 .. prefix_len[r] + extend_len[r] - 1 live in pool rows
    req_to_token[req_idx[r], j].  New row i of request r sees positions j <= prefix_len[r] + i.
    Returns o [sum E, Hq, d], lse [sum E, Hq] float64; rows of requests not listed in `requests`
    are NaN.
    """
    n_rows, hq, d = q.shape
    hkv = k_pool.shape[1]
    gq = hq // hkv
    o = np.full((n_rows, hq, d), np.nan)
    lse = np.full((n_rows, hq), np.nan)
    reqs = range(len(req_idx)) if requests is None else requests
    for r in reqs:
        p, e = int(prefix_len[r]), int(extend_len[r])
        if e == 0:
            continue
        L = p + e
        slots = req_to_token[req_idx[r], :L]
        K = _gather(k_pool, slots)
        V = _gather(v_pool, slots)
        rows = slice(int(cu_q[r]), int(cu_q[r]) + e)
        Q = bf16_to_f64(q[rows])
        visible = np.arange(L)[None, :] <= (p + np.arange(e))[:, None]
        for h in range(hq):
            o[rows, h], lse[rows, h] = attend(Q[:, h], K[:, h // gq], V[:, h // gq], visible, scale)
    return o, lse


def decode(q, k_pool, v_pool, req_to_token, req_idx, seq_len, scale, requests=None):
    """Decode attention: request b's single query (q[b]) over key positions 0 .. seq_len[b]-1,
    the current token included.  Returns o [B, Hq, d], lse [B, Hq]; unlisted requests NaN."""
    B, hq, d = q.shape
    hkv = k_pool.shape[1]
    gq = hq // hkv
    o = np.full((B, hq, d), np.nan)
    lse = np.full((B, hq), np.nan)
    reqs = range(B) if requests is None else requests
    for b in reqs:
        L = int(seq_len[b])
        slots = req_to_token[req_idx[b], :L]
        K = _gather(k_pool, slots)
        V = _gather(v_pool, slots)
        Q = bf16_to_f64(q[b])
        visible = np.ones((1, L), dtype=bool)
        for h in range(hq):
            ob, lb = attend(Q[h][None, :], K[:, h // gq], V[:, h // gq], visible, scale)
            o[b, h], lse[b, h] = ob[0], lb[0]
    return o, lse


def merge(parts):
    """Log-sum-exp merge of attention results over disjoint key partitions.

    parts: list of (o [..., d], lse [...]) computed over disjoint key sets of the same query.
    Softmax over the union weights partition i by exp(lse_i - lse), lse = log sum_i exp(lse_i);
    an empty partition (lse = -inf) contributes nothing.
    """
    lses = np.stack([np.asarray(p[1], dtype=np.float64) for p in parts])
    os_ = np.stack([np.asarray(p[0], dtype=np.float64) for p in parts])
    m = lses.max(axis=0)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lses - safe_m)                       # exp(-inf) = 0 for empty parts
    tot = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(tot > 0, safe_m + np.log(tot), -np.inf)
        o = np.where((tot > 0)[..., None], (w[..., None] * os_).sum(axis=0) / tot[..., None], 0.0)
    return o, lse
