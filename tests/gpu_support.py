"""Shared set-up for the GPU parity tests: upload synthetic workloads into a
paged cache, run the library, and compare with the oracle.

Test plumbing only.  The history of each request is placed in the cache with
torch indexing at slots computed by the oracle; this step's new tokens go
through the library's reshape_and_cache.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import paged_kv_cache_36_gb300 as pkv
from oracle import attention as oa
from oracle import paging

BF16_MAX_ABS = 2e-2
BF16_REL = 1e-2
F32_MAX_ABS = 1e-5


def history_slots(blocks, positions, block_size=16) -> np.ndarray:
    """Oracle slots of absolute positions of one request (vectorised form of
    oracle.paging.slot_index, checked against it on a sample)."""
    blocks = np.asarray(blocks, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    out = blocks[positions // block_size] * block_size + positions % block_size
    for p in positions[:: max(1, len(positions) // 7)][:8]:
        assert out[int(np.searchsorted(positions, p))] == paging.slot_index(blocks, int(p), block_size)
    return out


class Batch:
    """One step of the flattened batch, on the device."""

    def __init__(self, kv, blocks, num_blocks, query_len, num_computed, q, num_heads, dtype,
                 device="cuda", block_size=16):
        self.kv, self.blocks = kv, blocks
        self.R = len(query_len)
        self.query_len = np.asarray(query_len, np.int64)
        self.num_computed = np.asarray(num_computed, np.int64)
        self.seq = self.num_computed + self.query_len
        self.H, self.Hkv, self.D = num_heads, kv.key.shape[1], kv.key.shape[2]
        self.num_blocks, self.block_size = num_blocks, block_size
        self.dtype, self.device = dtype, device
        self.q_host = q
        self.qsl_host = np.concatenate([[0], np.cumsum(self.query_len)]).astype(np.int32)
        width = max(1, max((len(b) for b in blocks), default=1))
        bt = np.full((self.R, width), -1, np.int32)
        for r, b in enumerate(blocks):
            bt[r, :len(b)] = b
        self.bt_host = bt
        self.T = int(self.qsl_host[-1])

    def alloc_cache(self):
        shape = (self.num_blocks, self.block_size, self.Hkv, self.D)
        self.key_cache = torch.empty(shape, dtype=self.dtype, device=self.device)
        self.value_cache = torch.empty(shape, dtype=self.dtype, device=self.device)
        return self

    def fill_history(self, chunk_tokens=1 << 20):
        """Write positions [0, num_computed) of every request (plumbing)."""
        kf = self.key_cache.view(-1, self.Hkv, self.D)
        vf = self.value_cache.view(-1, self.Hkv, self.D)
        slots, rows = [], []
        for r in range(self.R):
            n = int(self.num_computed[r])
            if n == 0:
                continue
            slots.append(history_slots(self.blocks[r], np.arange(n), self.block_size))
            o = int(self.kv.offsets[r])
            rows.append((o, n))
        if not slots:
            return self
        for (o, n), s in zip(rows, slots):
            st = torch.from_numpy(s).to(self.device)
            for a in range(0, n, chunk_tokens):
                b = min(n, a + chunk_tokens)
                kf[st[a:b]] = self.kv.key[o + a:o + b].to(self.device, self.dtype)
                vf[st[a:b]] = self.kv.value[o + a:o + b].to(self.device, self.dtype)
        return self

    def new_tokens(self):
        """K/V rows of this step's tokens in batch order, and their oracle slots."""
        ks, vs, slots = [], [], []
        rows = [list(b) for b in self.blocks]
        for r in range(self.R):
            o, nc, ql = int(self.kv.offsets[r]), int(self.num_computed[r]), int(self.query_len[r])
            ks.append(self.kv.key[o + nc:o + nc + ql])
            vs.append(self.kv.value[o + nc:o + nc + ql])
        slots = paging.slot_mapping(rows, self.query_len, self.num_computed, self.block_size) \
            if self.T < 4096 else np.concatenate(
                [history_slots(self.blocks[r], np.arange(int(self.num_computed[r]), int(self.seq[r])),
                               self.block_size) for r in range(self.R)]).tolist()
        return torch.cat(ks), torch.cat(vs), slots

    def upload_metadata(self):
        d = self.device
        self.q = self.q_host.to(d, self.dtype)
        self.block_table = torch.from_numpy(self.bt_host).to(d)
        self.qsl = torch.from_numpy(self.qsl_host).to(d)
        self.seq_lens = torch.from_numpy(self.seq.astype(np.int32)).to(d)
        self.nc = torch.from_numpy(self.num_computed.astype(np.int32)).to(d)
        self.slot_mapping = torch.from_numpy(
            pkv.build_slot_mapping(self.bt_host, self.qsl_host, self.num_computed, self.block_size)).to(d)
        return self

    def write_new_tokens(self, error_word=None):
        k, v, _ = self.new_tokens()
        self.k_new = k.to(self.device, self.dtype)
        self.v_new = v.to(self.device, self.dtype)
        pkv.reshape_and_cache(self.k_new, self.v_new, self.key_cache, self.value_cache,
                              self.slot_mapping, error_word=error_word)
        return self

    def attention(self, workspace=None, out=None, check_error_word=True):
        self.workspace = workspace if workspace is not None else pkv.new_workspace(self.R, self.H, self.D)
        out = pkv.paged_attention_varlen(
            self.q, self.key_cache, self.value_cache, self.block_table, self.qsl, self.seq_lens,
            self.nc, 1.0 / math.sqrt(self.D), out=out, workspace=self.workspace,
            max_query_len=int(self.query_len.max()) if self.R else 0)
        if check_error_word:
            assert pkv.read_error_word(self.workspace) == 0, "kernel error word set"
        return out

    def oracle(self, rows=None):
        hist = [(self.kv.k(r), self.kv.v(r)) for r in range(self.R)]
        return oa.paged_attention_varlen(self.q_host, hist, self.qsl_host, self.seq,
                                         self.num_computed, 1.0 / math.sqrt(self.D), rows=rows)


def compare(got: torch.Tensor, ref: torch.Tensor, qsl, dtype, rows=None):
    """Asserts the tolerance for dtype over all rows of the chosen requests and
    per request; returns (max_abs, rel)."""
    got = got.detach().double().cpu()
    R = len(qsl) - 1
    reqs = range(R) if rows is None else rows
    sel = torch.cat([torch.arange(int(qsl[r]), int(qsl[r + 1])) for r in reqs]) if R else torch.arange(0)
    g, f = got[sel], ref[sel]
    assert torch.isfinite(g).all(), "non-finite output"
    max_abs = (g - f).abs().max().item() if g.numel() else 0.0
    rel = (torch.linalg.norm(g - f) / torch.linalg.norm(f)).item() if g.numel() else 0.0
    if dtype == torch.float32:
        assert max_abs <= F32_MAX_ABS, max_abs
        return max_abs, rel
    assert max_abs <= BF16_MAX_ABS, max_abs
    assert rel <= BF16_REL, rel
    for r in reqs:
        a, b = int(qsl[r]), int(qsl[r + 1])
        if b > a:
            d = got[a:b] - ref[a:b]
            assert d.abs().max().item() <= BF16_MAX_ABS, (r, d.abs().max().item())
            assert (torch.linalg.norm(d) / torch.linalg.norm(ref[a:b])).item() <= BF16_REL, r
    return max_abs, rel


def host_buffer_is_device_mapped(t: torch.Tensor) -> bool:
    """True when the CUDA runtime reports t's storage as host memory that the
    device addresses at the same pointer (pinned memory under unified
    addressing), so a kernel may store to it."""
    import ctypes

    class _Attr(ctypes.Structure):
        # cudaPointerAttributes: type, device, devicePointer, hostPointer and
        # long reserved[8], with spare room past it
        _fields_ = [("type", ctypes.c_int), ("device", ctypes.c_int),
                    ("devicePointer", ctypes.c_void_p), ("hostPointer", ctypes.c_void_p),
                    ("reserved", ctypes.c_long * 8), ("spare", ctypes.c_char * 256)]

    rt = None
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            continue
    if rt is None:
        return False
    rt.cudaPointerGetAttributes.argtypes = [ctypes.POINTER(_Attr), ctypes.c_void_p]
    rt.cudaPointerGetAttributes.restype = ctypes.c_int
    a = _Attr()
    if rt.cudaPointerGetAttributes(ctypes.byref(a), ctypes.c_void_p(t.data_ptr())) != 0:
        return False
    return a.type == 1 and a.devicePointer == t.data_ptr()  # cudaMemoryTypeHost
