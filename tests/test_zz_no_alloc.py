"""The workspace-free attention entry point, for callers that cannot allocate
device memory at the point where they run attention (an engine plugin whose
enqueue step must not allocate, a server whose free HBM all went to the KV
pool).  It is called through the C ABI and must agree with the
workspace-taking entry point within the bf16 tolerance the other tests use,
on two calls in a row (the shared scratch array keeps the previous call's
contents, so the second call checks that it is cleared correctly).

This file sorts last so that a run stopping at its first failure has already
run every other test.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

from tests.gpu_support import BF16_MAX_ABS, BF16_REL

pytestmark = pytest.mark.gpu


def _noalloc(pkv, q, kc, vc, bt, qsl, seq, nc, out, max_q, err):
    T, H, D = q.shape
    nb, bs, hkv, _ = kc.shape
    return pkv.lib().pkv_paged_attention_varlen_noalloc(
        q.data_ptr(), q.stride(0), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), bt.stride(0),
        qsl.data_ptr(), seq.data_ptr(), nc.data_ptr(), ctypes.c_float(1.0 / math.sqrt(D)),
        out.data_ptr(), out.stride(0), T, int(seq.shape[0]), nb, bs, H, hkv, D, pkv.PKV_BF16,
        max_q, err.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_on_two_calls():
    from paged_kv_cache_36_gb300 import build
    build.build()
    import paged_kv_cache_36_gb300 as pkv

    g = torch.Generator().manual_seed(127)
    H, Hkv, D, B = 32, 8, 128, 16
    # long decodes (several splits each, so the scratch's counters and partials
    # are used), a short decode, and a prefill chunk of 40 tokens
    ctx = [6000, 17, 3100, 9000]
    chunk_nc, chunk_len = 200, 40
    seq = ctx + [chunk_nc + chunk_len]
    qlens = [1, 1, 1, 1, chunk_len]
    counts = [(s + B - 1) // B for s in seq]
    nb = sum(counts) + 16
    perm = torch.randperm(nb, generator=g).numpy()
    bt = np.full((len(seq), max(counts)), -1, np.int32)
    at = 0
    for r, c in enumerate(counts):
        bt[r, :c] = perm[at:at + c]
        at += c
    kc = torch.randn(nb, B, Hkv, D, generator=g).to(torch.bfloat16).cuda()
    vc = torch.randn(nb, B, Hkv, D, generator=g).to(torch.bfloat16).cuda()
    T = sum(qlens)
    q = torch.randn(T, H, D, generator=g).to(torch.bfloat16).cuda()
    qsl = torch.tensor(np.concatenate([[0], np.cumsum(qlens)]), dtype=torch.int32, device="cuda")
    seq_t = torch.tensor(seq, dtype=torch.int32, device="cuda")
    nc_t = torch.tensor([s - l for s, l in zip(seq, qlens)], dtype=torch.int32, device="cuda")
    bt_t = torch.from_numpy(bt).cuda()

    ref = pkv.paged_attention_varlen(q, kc, vc, bt_t, qsl, seq_t, nc_t, 1.0 / math.sqrt(D),
                                     max_query_len=chunk_len)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        rc = _noalloc(pkv, q, kc, vc, bt_t, qsl, seq_t, nc_t, out, chunk_len, err)
        assert rc == 0, pkv.lib().pkv_last_error()
        torch.cuda.synchronize()
        assert err.item() == 0, f"call {call}: error word {err.item()}"
        d = (out.double() - ref.double()).cpu()
        assert torch.isfinite(out).all(), f"call {call}"
        assert d.abs().max().item() <= BF16_MAX_ABS, f"call {call}"
        assert (torch.linalg.norm(d) / torch.linalg.norm(ref.double().cpu())).item() <= BF16_REL


def test_noalloc_rejects_a_batch_beyond_the_static_scratch():
    from paged_kv_cache_36_gb300 import build
    build.build()
    import paged_kv_cache_36_gb300 as pkv
    q = torch.zeros(1, 32, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    i32 = torch.zeros(4, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = pkv.lib()
    # 100000 requests need far more than 16 MiB of split scratch
    rc = L.pkv_paged_attention_varlen_noalloc(
        q.data_ptr(), q.stride(0), kc.data_ptr(), kc.data_ptr(), i32.data_ptr(), 1, i32.data_ptr(),
        i32.data_ptr(), i32.data_ptr(), ctypes.c_float(0.1), q.data_ptr(), q.stride(0), 1, 100000,
        1, 16, 32, 8, 128, pkv.PKV_BF16, 1, err.data_ptr(), None)
    assert rc == -3 and b"static array" in L.pkv_last_error()
