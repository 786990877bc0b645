"""The workspace-free attention entry point, for callers that cannot allocate
device memory at the point where they run attention (an engine plugin whose
enqueue step must not allocate, a server whose free HBM all went to the KV
pool).  It is called through the C ABI.

Every call shares one scratch array that keeps the previous call's contents,
so the test drives it through a sequence of calls:
  1. a call whose block table holds an out-of-range block id: the kernels'
     bounds check sets PKV_ERR_BLOCK_ID in the scratch's error word, which
     the call copies to the caller's error word;
  2. the large batch, clean: the error word must come back 0 (the entry
     clears what the previous call left), and the output must match the
     workspace-taking entry point and the float64 oracle;
  3. a small batch (one long decode split over many CTAs, one short one);
  4. the large batch again.
Each clean call is compared with the workspace-taking entry point and with
the oracle over the requests' logical histories, within the bf16 tolerance
the other tests use.

This file sorts last so that a run stopping at its first failure has already
run every other test.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

from oracle import attention as oa
from tests.gpu_support import BF16_MAX_ABS, BF16_REL, compare

pytestmark = pytest.mark.gpu

H, HKV, D, B = 32, 8, 128, 16
PKV_ERR_BLOCK_ID = 1


def _noalloc(pkv, q, kc, vc, bt, qsl, seq, nc, out, max_q, err):
    T = q.shape[0]
    nb = kc.shape[0]
    return pkv.lib().pkv_paged_attention_varlen_noalloc(
        q.data_ptr(), q.stride(0), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), bt.stride(0),
        qsl.data_ptr(), seq.data_ptr(), nc.data_ptr(), ctypes.c_float(1.0 / math.sqrt(D)),
        out.data_ptr(), out.stride(0), T, int(seq.shape[0]), nb, B, H, HKV, D, pkv.PKV_BF16,
        max_q, err.data_ptr(), torch.cuda.current_stream().cuda_stream)


class _Batch:
    """Requests with logical K/V histories (host, bf16) placed in a shared
    paged cache through their block tables."""

    def __init__(self, g, seq, qlens, kc, vc, free_blocks):
        self.seq, self.qlens = seq, qlens
        self.nc = [s - l for s, l in zip(seq, qlens)]
        counts = [(s + B - 1) // B for s in seq]
        self.bt = np.full((len(seq), max(counts)), -1, np.int32)
        self.hist = []
        for r, (s, c) in enumerate(zip(seq, counts)):
            blocks = [free_blocks.pop() for _ in range(c)]
            self.bt[r, :c] = blocks
            k = torch.randn(s, HKV, D, generator=g).to(torch.bfloat16)
            v = torch.randn(s, HKV, D, generator=g).to(torch.bfloat16)
            pos = np.arange(s)
            slots = torch.from_numpy(np.asarray(blocks)[pos // B] * B + pos % B).cuda()
            kc.view(-1, HKV, D)[slots] = k.cuda()
            vc.view(-1, HKV, D)[slots] = v.cuda()
            self.hist.append((k, v))
        T = sum(qlens)
        self.q_host = torch.randn(T, H, D, generator=g).to(torch.bfloat16)
        self.q = self.q_host.cuda()
        self.qsl_host = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
        self.qsl = torch.from_numpy(self.qsl_host).cuda()
        self.seq_t = torch.tensor(seq, dtype=torch.int32, device="cuda")
        self.nc_t = torch.tensor(self.nc, dtype=torch.int32, device="cuda")
        self.bt_t = torch.from_numpy(self.bt).cuda()
        self.max_q = max(qlens)

    def oracle(self):
        return oa.paged_attention_varlen(self.q_host, self.hist, self.qsl_host, self.seq,
                                         self.nc, 1.0 / math.sqrt(D))


def test_noalloc_sequence_of_calls_matches_workspace_entry_and_oracle():
    from paged_kv_cache_36_gb300 import build
    build.build()
    import paged_kv_cache_36_gb300 as pkv

    g = torch.Generator().manual_seed(127)
    nb = 4096
    kc = torch.zeros(nb, B, HKV, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    free_blocks = list(torch.randperm(nb, generator=g).tolist())
    # long decodes (several splits each, so the scratch's counters and partials
    # are used), a short decode, and a prefill chunk of 40 tokens
    large = _Batch(g, [6000, 17, 3100, 9000, 240], [1, 1, 1, 1, 40], kc, vc, free_blocks)
    small = _Batch(g, [20000, 33], [1, 1], kc, vc, free_blocks)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    # 1. dirty the scratch: a block id past the pool trips the bounds check
    bad_bt = large.bt_t.clone()
    bad_bt[0, 3] = nb + 5
    out = torch.empty_like(large.q)
    rc = _noalloc(pkv, large.q, kc, vc, bad_bt, large.qsl, large.seq_t, large.nc_t, out,
                  large.max_q, err)
    assert rc == 0, pkv.lib().pkv_last_error()
    torch.cuda.synchronize()
    assert err.item() & PKV_ERR_BLOCK_ID, f"error word {err.item()}"

    # 2-4. clean calls of different batch sizes on the dirty scratch
    for step, b in enumerate([large, small, large]):
        ref = pkv.paged_attention_varlen(b.q, kc, vc, b.bt_t, b.qsl, b.seq_t, b.nc_t,
                                         1.0 / math.sqrt(D), max_query_len=b.max_q)
        err.fill_(-1)
        out = torch.full_like(b.q, float("nan"))
        rc = _noalloc(pkv, b.q, kc, vc, b.bt_t, b.qsl, b.seq_t, b.nc_t, out, b.max_q, err)
        assert rc == 0, pkv.lib().pkv_last_error()
        torch.cuda.synchronize()
        assert err.item() == 0, f"call {step + 2}: error word {err.item()}"
        assert torch.isfinite(out).all(), f"call {step + 2}"
        d = (out.double() - ref.double()).cpu()
        assert d.abs().max().item() <= BF16_MAX_ABS, f"call {step + 2}"
        assert (torch.linalg.norm(d) / torch.linalg.norm(ref.double().cpu())).item() <= BF16_REL
        compare(out, b.oracle(), b.qsl_host, torch.bfloat16)


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
