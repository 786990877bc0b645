"""Pins of the float64 attention oracle against things the pages and the
mathematics fix: torch's own scaled-dot-product attention on full prefills,
the chunked-equals-full trace, closed forms and pure-Python brute force."""

import json
import math
import os
import random

import pytest
import torch
import torch.nn.functional as F

from oracle import attention as oa

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _sdpa_full_prefill(q, k, v, scale):
    """Library reference for a full prefill ([n, H, D] / [n, Hkv, D], fp64)."""
    H, Hkv = q.shape[1], k.shape[1]
    G = H // Hkv
    qq = q.permute(1, 0, 2).double()
    kk = k.permute(1, 0, 2).double().repeat_interleave(G, dim=0)   # head h -> KV head h // G
    vv = v.permute(1, 0, 2).double().repeat_interleave(G, dim=0)
    out = F.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=scale)
    return out.permute(1, 0, 2)


@pytest.mark.parametrize("n,H,Hkv,D", [(1, 4, 2, 8), (7, 2, 2, 4), (33, 8, 2, 16), (64, 4, 1, 32)])
def test_full_prefill_matches_sdpa(n, H, Hkv, D):
    g = torch.Generator().manual_seed(n * 1000 + H)
    q = torch.randn(n, H, D, generator=g)
    k = torch.randn(n, Hkv, D, generator=g)
    v = torch.randn(n, Hkv, D, generator=g)
    scale = 1.0 / math.sqrt(D)
    ours = oa.causal_attention_request(q, k, v, 0, scale)
    ref = _sdpa_full_prefill(q, k, v, scale)
    assert torch.allclose(ours, ref, rtol=1e-12, atol=1e-13)


def test_chunked_equals_full_trace():
    g = json.load(open(os.path.join(GOLD, "chunked_prefill_trace.json")))
    _, H, T, D = g["qkv_shape"]
    gen = torch.Generator().manual_seed(g["seed"])
    q = torch.randn(T, H, D, generator=gen)
    k = torch.randn(T, H, D, generator=gen)
    v = torch.randn(T, H, D, generator=gen)
    scale = 1.0 / math.sqrt(D)
    full = oa.causal_attention_request(q, k, v, 0, scale)
    parts, trace = [], []
    C = g["chunk_size"]
    for a in range(0, T, C):
        b = min(a + C, T)
        # the cache holds positions 0..b-1 when chunk [a, b) runs
        parts.append(oa.causal_attention_request(q[a:b], k[:b], v[:b], a, scale))
        trace.append([a, b, [1, H, b, D]])
    assert trace == g["trace"]
    chunked = torch.cat(parts)
    assert torch.allclose(chunked, full, rtol=0, atol=1e-14)
    assert torch.allclose(chunked, full, rtol=g["rtol"], atol=g["atol"])
    assert torch.allclose(full, _sdpa_full_prefill(q, k, v, scale), rtol=1e-12, atol=1e-13)


def test_single_key_returns_its_value():
    q = torch.randn(1, 6, 16)
    k = torch.randn(1, 3, 16)
    v = torch.randn(1, 3, 16)
    out = oa.causal_attention_request(q, k, v, 0, 0.3)
    for h in range(6):
        assert torch.allclose(out[0, h], v[0, h // 2].double(), atol=1e-15)


def test_equal_keys_average_values():
    # every visible key identical -> uniform weights -> mean of visible values
    n_hist, n, D = 10, 4, 8
    k = torch.randn(1, 1, D).expand(n_hist + n, 1, D).clone()
    v = torch.randn(n_hist + n, 1, D)
    q = torch.randn(n, 2, D)
    out = oa.causal_attention_request(q, k, v, n_hist, 0.7)
    for i in range(n):
        p = n_hist + i
        mean = v[:p + 1, 0].double().mean(dim=0)
        assert torch.allclose(out[i, 0], mean, atol=1e-14)
        assert torch.allclose(out[i, 1], mean, atol=1e-14)


def test_aligned_query_selects_value():
    # orthonormal keys, q = c * K_j with large c: weight of key j -> 1
    D = 16
    basis = torch.eye(D)
    k = basis[:6].reshape(6, 1, D)
    v = torch.randn(6, 1, D)
    for j in range(6):
        q = (40.0 * basis[j]).reshape(1, 1, D)
        out = oa.causal_attention_request(q, k, v, 5, 1.0)
        assert torch.allclose(out[0, 0], v[j, 0].double(), atol=1e-15)


def test_two_key_closed_form_fixes_scale_and_sign():
    # query at position 1 over keys 0 and 1:
    # out = (v0 + e^(s (q.k1 - q.k0)) v1) / (1 + e^(s (q.k1 - q.k0)))
    q = torch.tensor([[[0.5, -1.0, 2.0]]])
    k = torch.tensor([[[1.0, 0.0, 0.5]], [[-0.5, 1.5, 1.0]]])
    v = torch.tensor([[[1.0, 2.0, 3.0]], [[-4.0, 0.0, 6.0]]])
    s = 0.37
    a = math.exp(s * ((0.5 * -0.5 + -1.0 * 1.5 + 2.0 * 1.0) - (0.5 * 1.0 + 0.0 + 2.0 * 0.5)))
    want = [(v0 + a * v1) / (1 + a) for v0, v1 in zip([1.0, 2.0, 3.0], [-4.0, 0.0, 6.0])]
    out = oa.causal_attention_request(q, k, v, 1, s)
    assert torch.allclose(out[0, 0], torch.tensor(want, dtype=torch.float64), atol=1e-15)


def test_gqa_head_map():
    # V of KV head g is the constant g: query head h must read KV head h // G
    H, Hkv, D, L = 8, 2, 4, 5
    k = torch.randn(L, Hkv, D)
    v = torch.stack([torch.full((L, D), float(g)) for g in range(Hkv)], dim=1)
    q = torch.randn(2, H, D)
    out = oa.causal_attention_request(q, k, v, L - 2, 0.5)
    for h in range(H):
        assert torch.allclose(out[:, h], torch.full((2, D), float(h // (H // Hkv)), dtype=torch.float64))


def _brute_force(q, k, v, nc, scale):
    n, H, D = q.shape
    Hkv = k.shape[1]
    G = H // Hkv
    out = [[[0.0] * D for _ in range(H)] for _ in range(n)]
    for i in range(n):
        p = nc + i
        for h in range(H):
            g = h // G
            w = [math.exp(scale * sum(float(q[i, h, d]) * float(k[j, g, d]) for d in range(D)))
                 for j in range(p + 1)]
            z = sum(w)
            for d in range(D):
                out[i][h][d] = sum(w[j] * float(v[j, g, d]) for j in range(p + 1)) / z
    return torch.tensor(out, dtype=torch.float64)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(seed):
    rng = random.Random(seed)
    Hkv = rng.choice([1, 2])
    H = Hkv * rng.choice([1, 2, 3])
    D = rng.choice([2, 3, 5])
    nc = rng.randint(0, 6)
    n = rng.randint(1, 4)
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(n, H, D, generator=g)
    k = torch.randn(nc + n + rng.randint(0, 3), Hkv, D, generator=g)   # extra rows must be ignored
    v = torch.randn(k.shape, generator=g)
    scale = rng.uniform(0.1, 1.0)
    assert torch.allclose(oa.causal_attention_request(q, k, v, nc, scale),
                          _brute_force(q, k, v, nc, scale), atol=1e-12)


def test_varlen_isolates_requests():
    g = torch.Generator().manual_seed(5)
    H, Hkv, D = 4, 2, 8
    qlens, ncs = [3, 1, 0, 5], [0, 9, 4, 2]
    hist = [(torch.randn(nc + ql, Hkv, D, generator=g), torch.randn(nc + ql, Hkv, D, generator=g))
            for ql, nc in zip(qlens, ncs)]
    q = torch.randn(sum(qlens), H, D, generator=g)
    qsl = [0]
    for ql in qlens:
        qsl.append(qsl[-1] + ql)
    seq = [nc + ql for nc, ql in zip(ncs, qlens)]
    out = oa.paged_attention_varlen(q, hist, qsl, seq, ncs, 0.4)
    for r in range(4):
        a, b = qsl[r], qsl[r + 1]
        if b > a:
            want = _brute_force(q[a:b], hist[r][0], hist[r][1], ncs[r], 0.4)
            assert torch.allclose(out[a:b], want, atol=1e-12)
    with pytest.raises(ValueError):
        oa.paged_attention_varlen(q, hist, qsl, [s + 1 for s in seq], ncs, 0.4)


@pytest.mark.parametrize("nsplit", [1, 2, 3, 7])
def test_lse_combine_split_invariance(nsplit):
    g = torch.Generator().manual_seed(nsplit)
    H, Hkv, D, L = 8, 2, 16, 50
    q = torch.randn(H, D, generator=g)
    k = torch.randn(L, Hkv, D, generator=g) * 3
    v = torch.randn(L, Hkv, D, generator=g)
    cuts = sorted(random.Random(nsplit).sample(range(1, L), nsplit - 1))
    bounds = list(zip([0] + cuts, cuts + [L]))
    parts = [oa.split_partial(q, k, v, rng_, 0.25) for rng_ in bounds]
    ms = torch.stack([p[0] for p in parts])
    ls = torch.stack([p[1] for p in parts])
    os_ = torch.stack([p[2] for p in parts])
    combined = oa.lse_combine(ms, ls, os_)
    full = oa.causal_attention_request(q[None], k, v, L - 1, 0.25)[0]
    assert torch.allclose(combined, full, atol=1e-13)
