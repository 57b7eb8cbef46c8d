"""Dense causal attention on contiguous K/V in float64 — the textbook form.

Test infrastructure (see the package docstring).  This is what the paged
oracle must reduce to once the pages are gathered into one contiguous history:
"vLLM 推理全流程深度解析", prefill section (causal mask: lower triangle kept,
upper triangle -inf) and decode section (a single query against all cached
keys), with the chunk offset of "Tour: One forward pass", stop 3
(seq_len = num_computed + query_len).
"""
import numpy as np


def dense_causal_attention(q, k, v, ctx: int, scale: float):
    """q: [n, hq, d], k/v: [ctx + n, hkv, d] (any real dtype), float64 out.

    Query row i sits at position ctx + i and sees keys 0 .. ctx + i.  Query
    head h reads KV head h // (hq // hkv)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, hq, d = q.shape
    L, hkv, _ = k.shape
    assert L == ctx + n and hq % hkv == 0
    group = hq // hkv
    kh = np.repeat(k, group, axis=1)   # [L, hq, d]; head h -> kv head h // group
    vh = np.repeat(v, group, axis=1)
    s = np.einsum("ihd,jhd->hij", q, kh) * scale
    visible = np.arange(L)[None, :] <= (ctx + np.arange(n))[:, None]
    s = np.where(visible[None, :, :], s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    return np.einsum("hij,jhd->ihd", p, vh)
