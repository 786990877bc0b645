"""Dense per-request causal GQA attention in float64.

Sources:
* "AI Infra入门干货总结：大模型是如何高效推理的", section "Attention Module
  (以标准GQA + RoPE为例)": attention runs per request (requests are separated
  by cu_seqlens / query_start_loc); Q is [query_lens, num_heads, head_dim] and
  K, V are [seq_lens, num_kv_heads, head_dim] - the request's whole history;
  decode has query_lens = 1.  The Flash-Decoding remark at the end of the page
  (cross-SM normalisation by log-sum-exp) defines `lse_combine`.
* "Chunked Prefill 与 Preemption", section "Chunked Prefill：改变调度粒度，
  不改变 causal 结果": for a chunk [a, b) the cache holds positions 0..b-1 and
  query i attends key j iff j <= i (mask 0 for j <= i, -inf for j > i).

Readings where the pages are silent:
* GQA head map: query head h uses KV head h // G with G = H / Hkv
  (contiguous groups; the pages only say "standard GQA").
* The query at step row i of request r sits at absolute position
  num_computed[r] + i; seq_lens[r] = num_computed[r] + query_len[r] is the KV
  length after this step's writes.

K and V here are each request's own logical history in position order; they
never pass through the paged layout.  Inputs of any float type are converted
exactly to float64 before any arithmetic.
"""

from __future__ import annotations

import torch


def _f64(x) -> torch.Tensor:
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float64)
    return torch.as_tensor(x, dtype=torch.float64)


def causal_attention_request(q, k, v, num_computed: int, scale: float) -> torch.Tensor:
    """Attention of one request's query rows over its history.

    q: [n, H, D]; k, v: [>= num_computed + n, Hkv, D].
    Row i is at absolute position p = num_computed + i and sees keys 0..p.
    Returns float64 [n, H, D].
    """
    n, num_heads, head_dim = q.shape
    num_kv_heads = k.shape[1]
    if num_heads % num_kv_heads:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    group = num_heads // num_kv_heads
    length = num_computed + n
    if k.shape[0] < length or v.shape[0] < length:
        raise ValueError("history shorter than num_computed + query_len")
    out = torch.empty((n, num_heads, head_dim), dtype=torch.float64)
    if n == 0:
        return out
    pos = num_computed + torch.arange(n)
    keys = torch.arange(length)
    masked = keys[None, :] > pos[:, None]                  # j > p  ->  -inf
    qd = _f64(q)
    for g in range(num_kv_heads):
        kg = _f64(k[:length, g, :])                        # [L, D]
        vg = _f64(v[:length, g, :])
        for h in range(g * group, (g + 1) * group):        # heads of this KV head
            logits = scale * (qd[:, h, :] @ kg.T)          # [n, L]
            logits = logits.masked_fill(masked, float("-inf"))
            m = logits.max(dim=1, keepdim=True).values
            w = torch.exp(logits - m)
            out[:, h, :] = (w @ vg) / w.sum(dim=1, keepdim=True)
    return out


def paged_attention_varlen(q, histories, query_start_loc, seq_lens, num_computed_tokens,
                           scale: float, rows=None) -> torch.Tensor:
    """Attention for a flattened batch.

    q: [T, H, D], requests concatenated; query_start_loc: [R + 1] prefix sums of
    the query lengths; histories[r] = (k_r, v_r), the request's logical K/V of
    length >= seq_lens[r].  `rows`, if given, restricts the work to those
    requests (other rows of the result are left as NaN).
    Returns float64 [T, H, D].
    """
    T, H, D = q.shape
    out = torch.full((T, H, D), float("nan"), dtype=torch.float64)
    R = len(seq_lens)
    for r in (range(R) if rows is None else rows):
        a, b = int(query_start_loc[r]), int(query_start_loc[r + 1])
        nc = int(num_computed_tokens[r])
        if int(seq_lens[r]) != nc + (b - a):
            raise ValueError(f"request {r}: seq_len {int(seq_lens[r])} != num_computed {nc} + query_len {b - a}")
        if b == a:
            continue
        k_r, v_r = histories[r]
        out[a:b] = causal_attention_request(q[a:b], k_r, v_r, nc, scale)
    return out


# -- split-KV partials and their log-sum-exp merge ------------------------------
def split_partial(q_row, k, v, key_range, scale: float):
    """Unnormalised partial of one query row over keys [lo, hi) for every head.

    q_row: [H, D]; k, v: [L, Hkv, D].  Returns (m [H], l [H], o [H, D]) with
    m = max logit, l = sum exp(logit - m), o = sum exp(logit - m) * V.
    """
    lo, hi = key_range
    H, D = q_row.shape
    group = H // k.shape[1]
    qd = _f64(q_row)
    m = torch.empty(H, dtype=torch.float64)
    l = torch.empty(H, dtype=torch.float64)
    o = torch.empty((H, D), dtype=torch.float64)
    for h in range(H):
        g = h // group
        logits = scale * (_f64(k[lo:hi, g, :]) @ qd[h])
        m[h] = logits.max()
        w = torch.exp(logits - m[h])
        l[h] = w.sum()
        o[h] = w @ _f64(v[lo:hi, g, :])
    return m, l, o


def lse_combine(ms, ls, os):
    """Merge split partials: M = max_s m_s; out = sum_s e^(m_s - M) o_s divided by
    sum_s e^(m_s - M) l_s.  ms, ls: [S, H]; os: [S, H, D]."""
    ms, ls, os = _f64(ms), _f64(ls), _f64(os)
    big = ms.max(dim=0).values
    wgt = torch.exp(ms - big)                 # [S, H]
    num = (wgt[:, :, None] * os).sum(dim=0)
    den = (wgt * ls).sum(dim=0)
    return num / den[:, None]
