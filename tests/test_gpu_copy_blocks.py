"""GPU parity of copy_blocks: whole-block copies, bit for bit, within one pool
(copy-on-write pairs listed by the allocator), between two device pools, and
between the device pool and a pool in pinned host memory."""

import numpy as np
import pytest
import torch

from oracle.allocator import NaiveAllocator
from workloads.generators import randn_fp32, random_block_placement

pytestmark = pytest.mark.gpu


def _pkv():
    import paged_kv_cache_36_gb300 as pkv
    return pkv


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _pool(nb, name, dtype=torch.bfloat16, hkv=8, d=128):
    return randn_fp32((nb, 16, hkv, d), name, "k", dtype=dtype), \
        randn_fp32((nb, 16, hkv, d), name, "v", dtype=dtype)


def _oracle_copy(sk, sv, dk, dv, pairs):
    dk, dv = dk.clone(), dv.clone()
    for s, d in pairs:
        dk[d] = sk[s]
        dv[d] = sv[s]
    return dk, dv


def test_copy_on_write_pairs_from_the_allocator():
    """A forked request writes into its shared partial block: the pairs the
    allocator lists are copied before the write."""
    nb = 64
    a = NaiveAllocator(nb, 16)
    for r in range(6):
        assert a.reserve([(r, 16 * (r + 1) + 5)])
        a.commit()
        a.fork(r, 100 + r)
    assert a.reserve([(100 + r, 3) for r in range(6)])
    pairs = a.pending_copies()
    assert len(pairs) == 6
    k, v = _pool(nb, "cow")
    dk, dv = k.cuda(), v.cuda()
    dpairs = torch.tensor(pairs, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _pkv().copy_blocks(dk, dv, dk, dv, dpairs, error_word=err)
    torch.cuda.synchronize()
    wk, wv = _oracle_copy(k, v, k, v, pairs)
    assert err.item() == 0
    assert torch.equal(_bits(dk.cpu()), _bits(wk)) and torch.equal(_bits(dv.cpu()), _bits(wv))


@pytest.mark.parametrize("dtype,hkv,d", [(torch.bfloat16, 8, 128), (torch.float32, 2, 64),
                                         (torch.bfloat16, 1, 64)])
def test_between_device_pools(dtype, hkv, d):
    ns, nd, n = 300, 200, 150
    sk, sv = _pool(ns, "src", dtype, hkv, d)
    dk, dv = _pool(nd, "dst", dtype, hkv, d)
    src = random_block_placement(ns, [n], "pairs", "src")[0]
    dst = random_block_placement(nd, [n], "pairs", "dst")[0]
    pairs = np.stack([src, dst], axis=1).astype(np.int32)
    gk, gv = dk.cuda(), dv.cuda()
    _pkv().copy_blocks(sk.cuda(), sv.cuda(), gk, gv, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    wk, wv = _oracle_copy(sk, sv, dk, dv, pairs.tolist())
    assert torch.equal(_bits(gk.cpu()), _bits(wk)) and torch.equal(_bits(gv.cpu()), _bits(wv))


def test_device_to_pinned_host_and_back():
    """Offload 500 scattered blocks to a pinned host pool and reload them to
    other places: both directions bit-exact."""
    nd, nh, n = 2048, 600, 500
    k, v = _pool(nd, "swap")
    dk, dv = k.cuda(), v.cuda()
    hk = torch.zeros((nh, 16, 8, 128), dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_src = random_block_placement(nd, [n], "swap", "out_src")[0]
    out_dst = random_block_placement(nh, [n], "swap", "out_dst")[0]
    out_pairs = np.stack([out_src, out_dst], axis=1).astype(np.int32)
    pkv = _pkv()
    pkv.copy_blocks(dk, dv, hk, hv, torch.from_numpy(out_pairs).cuda())
    torch.cuda.synchronize()
    wk, wv = _oracle_copy(k, v, torch.zeros_like(hk), torch.zeros_like(hv), out_pairs.tolist())
    assert torch.equal(_bits(hk), _bits(wk)) and torch.equal(_bits(hv), _bits(wv))
    # reload into blocks the offloaded ones do not occupy
    free = np.setdiff1d(np.arange(nd), out_src)[:n]
    in_pairs = np.stack([out_dst, free], axis=1).astype(np.int32)
    pkv.copy_blocks(hk, hv, dk, dv, torch.from_numpy(in_pairs).cuda())
    torch.cuda.synchronize()
    assert torch.equal(_bits(dk.cpu()[free]), _bits(k[out_src]))
    assert torch.equal(_bits(dv.cpu()[free]), _bits(v[out_src]))


def test_bad_pairs_are_skipped_and_flagged():
    nb = 32
    k, v = _pool(nb, "bad", hkv=2, d=64)
    dk, dv = k.cuda(), v.cuda()
    pairs = [(1, 2), (40, 3), (4, -1), (5, 6)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv = _pkv()
    pkv.copy_blocks(dk, dv, dk, dv, torch.tensor(pairs, dtype=torch.int32, device="cuda"),
                    error_word=err)
    torch.cuda.synchronize()
    assert err.item() == pkv.ERR_BLOCK_ID
    wk, wv = _oracle_copy(k, v, k, v, [(1, 2), (5, 6)])
    assert torch.equal(_bits(dk.cpu()), _bits(wk)) and torch.equal(_bits(dv.cpu()), _bits(wv))
    # no pairs: nothing launched
    pkv.copy_blocks(dk, dv, dk, dv, torch.empty((0, 2), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
