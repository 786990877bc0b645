"""PagedAttention over a flattened, variable-length token batch on one GB300.

Thin Python binding of libpkv.so: every function marshals arguments into the
C ABI declared in include/pkv.h and calls it; all computation runs in the
library (CUDA kernels for sm_103a, C++ host code).  PyTorch is used only to
hand over device pointers and the current CUDA stream.  If the library is not
built, importing the binding's entry points raises ImportError.
"""

from __future__ import annotations

import ctypes as C

import numpy as np

from . import _ffi
from ._ffi import (ERR_BLOCK_ID, ERR_METADATA, ERR_POSITION, ERR_SLOT, ERR_TIMEOUT,  # noqa: F401
                   PKV_BF16, PKV_F32)

__all__ = [
    "PkvError", "lib", "reshape_and_cache", "rope_reshape_and_cache", "copy_blocks",
    "attention_workspace_bytes", "new_workspace",
    "paged_attention_varlen", "reshape_and_cache_paged_attention", "read_error_word",
    "PreparedCall", "prepare_reshape_and_cache_paged_attention",
    "build_slot_mapping", "Allocator", "Scheduler",
]

_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        _lib = _ffi.load()
    return _lib


class PkvError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = lib().pkv_last_error().decode(errors="replace")
        super().__init__(f"{where}: {_ffi.ERRORS.get(code, code)}: {msg}")
        self.code = code


def _check(code: int, where: str) -> int:
    if code < 0:
        raise PkvError(code, where)
    return code


# ---------------------------------------------------------------------------
# device entry points (torch tensors in, no computation here)
# ---------------------------------------------------------------------------
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return PKV_F32
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream_ptr(stream) -> int | None:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _token_stride(t) -> int:
    # [tokens, heads, dim] with heads and dim contiguous (one stride() call:
    # per-dimension stride(i) calls cost several times more host time)
    st = t.stride()
    if len(st) != 3 or st[2] != 1 or st[1] != t.shape[2]:
        raise ValueError("expected [tokens, heads, head_dim] with contiguous heads and dims")
    return st[0]


def _row_stride(block_table) -> int:
    st = block_table.stride()
    if len(st) != 2 or st[1] != 1:
        raise ValueError("block_table must be [R, max_blocks] with unit inner stride")
    return st[0]


def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, error_word=None,
                      stream=None) -> None:
    """Scatter key/value [T, Hkv, D] into the caches [NB, B, Hkv, D] at slot_mapping[T] (int64)."""
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    nb, bs, hkv, d = key_cache.shape
    code = lib().pkv_reshape_and_cache(
        key.data_ptr(), value.data_ptr(), _token_stride(key), _token_stride(value),
        key_cache.data_ptr(), value_cache.data_ptr(), slot_mapping.data_ptr(),
        int(slot_mapping.shape[0]), nb, bs, hkv, d, _dtype_code(key_cache),
        error_word.data_ptr() if error_word is not None else None, _stream_ptr(stream))
    _check(code, "reshape_and_cache")


def rope_reshape_and_cache(positions, query, key, value, key_cache, value_cache, slot_mapping,
                           cos_sin_cache, rotary_dim: int | None = None, is_neox: bool = True,
                           key_out=None, error_word=None, stream=None) -> None:
    """Rotate query [T, H, D] in place and key [T, Hkv, D] by cos_sin_cache[positions]
    (float32 [max_position, rotary_dim]), and scatter the rotated key and value
    into the caches [NB, B, Hkv, D] at slot_mapping (int64 [T]).  key_out, if
    given, receives the rotated key too (it may be `key`)."""
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()
            and cos_sin_cache.is_contiguous()):
        raise ValueError("caches and cos_sin_cache must be contiguous")
    import torch
    if cos_sin_cache.dtype != torch.float32 or cos_sin_cache.dim() != 2:
        raise TypeError("cos_sin_cache must be float32 [max_position, rotary_dim]")
    if positions.dtype != torch.int64 or slot_mapping.dtype != torch.int64:
        raise TypeError("positions and slot_mapping must be int64")
    nb, bs, hkv, d = key_cache.shape
    rd = int(cos_sin_cache.shape[1]) if rotary_dim is None else int(rotary_dim)
    if rd != cos_sin_cache.shape[1]:
        raise ValueError("rotary_dim must equal cos_sin_cache.shape[1]")
    ks = _token_stride(key)
    if key_out is not None and _token_stride(key_out) != ks:
        raise ValueError("key_out must have key's token stride")
    code = lib().pkv_rope_reshape_and_cache(
        positions.data_ptr(), query.data_ptr(), _token_stride(query), int(query.shape[1]),
        key.data_ptr(), ks, key_out.data_ptr() if key_out is not None else None,
        value.data_ptr(), _token_stride(value), key_cache.data_ptr(), value_cache.data_ptr(),
        slot_mapping.data_ptr(), cos_sin_cache.data_ptr(), int(cos_sin_cache.shape[0]), rd,
        int(bool(is_neox)), int(positions.shape[0]), nb, bs, hkv, d, _dtype_code(key_cache),
        error_word.data_ptr() if error_word is not None else None, _stream_ptr(stream))
    _check(code, "rope_reshape_and_cache")


def copy_blocks(src_key_cache, src_value_cache, dst_key_cache, dst_value_cache, block_pairs,
                error_word=None, stream=None) -> None:
    """Copy whole blocks: dst[pairs[i, 1]] = src[pairs[i, 0]] for K and V.  Pools are
    [num_blocks, block_size, Hkv, D] tensors (device, or pinned host memory the
    device can map); block_pairs is int32 [n, 2] (device or pinned host)."""
    for t in (src_key_cache, src_value_cache, dst_key_cache, dst_value_cache, block_pairs):
        if not t.is_contiguous():
            raise ValueError("pools and block_pairs must be contiguous")
    if src_key_cache.shape[1:] != dst_key_cache.shape[1:] or \
            src_key_cache.dtype != dst_key_cache.dtype:
        raise ValueError("source and destination pools must have the same block shape and dtype")
    block_bytes = src_key_cache[0].numel() * src_key_cache.element_size()
    code = lib().pkv_copy_blocks(
        src_key_cache.data_ptr(), src_value_cache.data_ptr(), dst_key_cache.data_ptr(),
        dst_value_cache.data_ptr(), block_pairs.data_ptr(), int(block_pairs.shape[0]),
        int(src_key_cache.shape[0]), int(dst_key_cache.shape[0]), block_bytes,
        error_word.data_ptr() if error_word is not None else None, _stream_ptr(stream))
    _check(code, "copy_blocks")


def attention_workspace_bytes(num_reqs: int, num_heads: int, head_dim: int) -> int:
    return int(lib().pkv_attention_workspace_bytes(num_reqs, num_heads, head_dim))


def new_workspace(num_reqs: int, num_heads: int, head_dim: int, device="cuda"):
    """A zero-filled workspace large enough for batches of up to num_reqs requests."""
    import torch
    n = attention_workspace_bytes(num_reqs, num_heads, head_dim)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def read_error_word(workspace) -> int:
    """The PKV_ERR_* bits the kernels recorded in this workspace (synchronises)."""
    return int(workspace[:4].view(dtype=__import__("torch").int32).item()) & 0xFFFFFFFF


def paged_attention_varlen(q, key_cache, value_cache, block_table, query_start_loc, seq_lens,
                           num_computed_tokens, scale: float, out=None, workspace=None,
                           max_query_len: int = 0, stream=None):
    """Causal GQA attention of the flattened batch q [T, H, D] over the paged caches.

    block_table int32 [R, max_blocks]; query_start_loc int32 [R + 1]; seq_lens,
    num_computed_tokens int32 [R].  Returns out [T, H, D]: a CUDA tensor, or
    a pinned CPU tensor that the kernels store into directly.
    """
    import torch
    T, H, D = q.shape
    nb, bs, hkv, d2 = key_cache.shape
    R = int(seq_lens.shape[0])
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = new_workspace(R, H, D, q.device)
    code = lib().pkv_paged_attention_varlen(
        q.data_ptr(), _token_stride(q), key_cache.data_ptr(), value_cache.data_ptr(),
        block_table.data_ptr(), _row_stride(block_table), query_start_loc.data_ptr(),
        seq_lens.data_ptr(), num_computed_tokens.data_ptr(), float(scale), out.data_ptr(),
        _token_stride(out), T, R, nb, bs, H, hkv, D, _dtype_code(q), int(max_query_len),
        workspace.data_ptr(), workspace.nbytes, _stream_ptr(stream))
    _check(code, "paged_attention_varlen")
    return out


def reshape_and_cache_paged_attention(key, value, slot_mapping, q, key_cache, value_cache,
                                      block_table, query_start_loc, seq_lens, num_computed_tokens,
                                      scale: float, out=None, workspace=None,
                                      max_query_len: int = 0, stream=None):
    """reshape_and_cache of key/value [T, Hkv, D] at slot_mapping (int64 [T]),
    then paged_attention_varlen of q [T, H, D]; one kernel for any bf16
    step.  Returns out [T, H, D]: a CUDA tensor, or a pinned CPU tensor that
    the kernels store into directly."""
    import torch
    T, H, D = q.shape
    nb, bs, hkv, _ = key_cache.shape
    R = int(seq_lens.shape[0])
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = new_workspace(R, H, D, q.device)
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    code = lib().pkv_reshape_and_cache_paged_attention(
        key.data_ptr(), _token_stride(key), value.data_ptr(), _token_stride(value),
        slot_mapping.data_ptr(), q.data_ptr(), _token_stride(q), key_cache.data_ptr(),
        value_cache.data_ptr(), block_table.data_ptr(), _row_stride(block_table),
        query_start_loc.data_ptr(), seq_lens.data_ptr(), num_computed_tokens.data_ptr(),
        float(scale), out.data_ptr(), _token_stride(out), T, R, nb, bs, H, hkv, D, _dtype_code(q),
        int(max_query_len), workspace.data_ptr(), workspace.nbytes, _stream_ptr(stream))
    _check(code, "reshape_and_cache_paged_attention")
    return out


class PreparedCall:
    """A C-ABI call whose arguments were marshalled once.  Calling it makes the
    same library call again, on the stream resolved at preparation: for a
    serving loop whose buffers stay in place from step to step, this leaves
    out the per-call Python work (pointer, stride and stream lookups).  The
    library still validates every call.  The tensors it was prepared from are
    kept alive; their storage and shapes must not change."""

    __slots__ = ("_fn", "_args", "_keep", "_where")

    def __init__(self, fn, args, keep, where):
        self._fn, self._args, self._keep, self._where = fn, args, keep, where

    def __call__(self):
        code = self._fn(*self._args)
        if code < 0:
            raise PkvError(code, self._where)
        return self._keep[0]


def prepare_reshape_and_cache_paged_attention(key, value, slot_mapping, q, key_cache,
                                              value_cache, block_table, query_start_loc,
                                              seq_lens, num_computed_tokens, scale: float, out,
                                              workspace, max_query_len: int = 0, stream=None):
    """reshape_and_cache_paged_attention with its arguments marshalled once;
    returns a PreparedCall that issues the call (and returns out) each time it
    is called.  out and workspace are required: they are part of the state the
    calls reuse."""
    import torch
    T, H, D = q.shape
    nb, bs, hkv, _ = key_cache.shape
    R = int(seq_lens.shape[0])
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    args = (key.data_ptr(), _token_stride(key), value.data_ptr(), _token_stride(value),
            slot_mapping.data_ptr(), q.data_ptr(), _token_stride(q), key_cache.data_ptr(),
            value_cache.data_ptr(), block_table.data_ptr(), _row_stride(block_table),
            query_start_loc.data_ptr(), seq_lens.data_ptr(), num_computed_tokens.data_ptr(),
            float(scale), out.data_ptr(), _token_stride(out), T, R, nb, bs, H, hkv, D,
            _dtype_code(q), int(max_query_len), workspace.data_ptr(), workspace.nbytes,
            _stream_ptr(stream))
    keep = (out, key, value, slot_mapping, q, key_cache, value_cache, block_table,
            query_start_loc, seq_lens, num_computed_tokens, workspace)
    return PreparedCall(lib().pkv_reshape_and_cache_paged_attention, args, keep,
                        "reshape_and_cache_paged_attention")


# ---------------------------------------------------------------------------
# host entry points (numpy arrays)
# ---------------------------------------------------------------------------
def _ptr(a: np.ndarray) -> int:
    # the address as an int (ctypes passes it as void*); cheaper than data_as
    return a.ctypes.data


def build_slot_mapping(block_table: np.ndarray, query_start_loc, num_computed_tokens,
                       block_size: int, out: np.ndarray | None = None) -> np.ndarray:
    """slot_mapping (int64 [num_tokens]) of the step, built on the host; `out`,
    if given, is a C-contiguous int64 array of num_tokens entries (for instance
    a view of a pinned staging buffer) written in place."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    nc = np.ascontiguousarray(num_computed_tokens, dtype=np.int32)
    n = int(qsl[-1]) if len(qsl) else 0
    if out is None:
        out = np.empty(n, dtype=np.int64)
    elif out.dtype != np.int64 or out.shape != (n,) or not out.flags.c_contiguous:
        raise ValueError(f"out must be a contiguous int64 array of {n} entries")
    _check(lib().pkv_build_slot_mapping(_ptr(bt), bt.shape[1], _ptr(qsl), _ptr(nc), len(nc),
                                        block_size, _ptr(out), n), "build_slot_mapping")
    return out


class Allocator:
    """Reserve / commit / rollback block allocator (host)."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_req: int | None = None,
                 _handle=None, num_cpu_blocks: int = 0):
        self._own = _handle is None
        self.num_blocks = num_blocks
        self.num_cpu_blocks = num_cpu_blocks
        self._h = _handle or lib().pkv_alloc_create_with_cpu_pool(
            num_blocks, block_size, max_blocks_per_req or num_blocks, num_cpu_blocks)
        if not self._h:
            raise PkvError(-1, "pkv_alloc_create")

    def __del__(self):
        if getattr(self, "_own", False) and self._h:
            lib().pkv_alloc_destroy(self._h)
            self._h = None

    def reserve(self, plan) -> bool:
        """plan: [(req_id, new_tokens)].  False if the blocks are not there."""
        ids = np.array([r for r, _ in plan], dtype=np.int32)
        toks = np.array([s for _, s in plan], dtype=np.int32)
        code = lib().pkv_alloc_reserve(self._h, len(ids), _ptr(ids), _ptr(toks))
        if code == -4:
            return False
        _check(code, "reserve")
        return True

    def commit(self):
        _check(lib().pkv_alloc_commit(self._h), "commit")

    def rollback(self):
        _check(lib().pkv_alloc_rollback(self._h), "rollback")

    def free_request(self, req: int) -> int:
        return _check(lib().pkv_alloc_free_request(self._h, req), "free_request")

    def stats(self) -> dict:
        s = _ffi.AllocStats()
        _check(lib().pkv_alloc_get_stats(self._h, C.byref(s)), "stats")
        return {n: getattr(s, n) for n, _ in s._fields_}

    def table(self, req: int) -> list[int]:
        buf = np.empty(self.num_blocks, dtype=np.int32)
        n = _check(lib().pkv_alloc_table(self._h, req, _ptr(buf), len(buf)), "table")
        return buf[:n].tolist()

    def held_tokens(self, req: int) -> int:
        return int(lib().pkv_alloc_held_tokens(self._h, req))

    def free_list(self) -> list[int]:
        buf = np.empty(self.num_blocks, dtype=np.int32)
        n = _check(lib().pkv_alloc_free_list(self._h, _ptr(buf), len(buf)), "free_list")
        return buf[:n].tolist()

    def check(self):
        _check(lib().pkv_alloc_check(self._h), "check")

    # -- prefix sharing --------------------------------------------------------
    def match_prefix(self, req: int, namespace: int, tokens) -> int:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        return _check(lib().pkv_alloc_match_prefix(self._h, req, namespace, _ptr(t), len(t)),
                      "match_prefix")

    def peek_prefix(self, namespace: int, tokens) -> tuple[int, int]:
        """(matched tokens, how many matched blocks are cached now)."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        cached = C.c_int32(0)
        n = _check(lib().pkv_alloc_peek_prefix(self._h, namespace, _ptr(t), len(t),
                                               C.byref(cached)), "peek_prefix")
        return n, cached.value

    def fork(self, parent: int, child: int) -> None:
        _check(lib().pkv_alloc_fork(self._h, parent, child), "fork")

    def pending_copies(self) -> list[tuple[int, int]]:
        buf = np.empty(2 * max(1, self.num_blocks), dtype=np.int32)
        n = _check(lib().pkv_alloc_pending_copies(self._h, _ptr(buf), len(buf) // 2),
                   "pending_copies")
        return [(int(buf[2 * i]), int(buf[2 * i + 1])) for i in range(n)]

    def prefix_stats(self) -> dict:
        s = _ffi.PrefixStats()
        _check(lib().pkv_alloc_get_prefix_stats(self._h, C.byref(s)), "prefix_stats")
        return {n: getattr(s, n) for n, _ in s._fields_}

    def ref_count(self, block: int) -> int:
        return _check(lib().pkv_alloc_ref_count(self._h, block), "ref_count")

    def cached_list(self) -> list[int]:
        buf = np.empty(self.num_blocks, dtype=np.int32)
        n = _check(lib().pkv_alloc_cached_list(self._h, _ptr(buf), len(buf)), "cached_list")
        return buf[:n].tolist()

    def available(self) -> int:
        return int(lib().pkv_alloc_available(self._h))

    # -- swapping ----------------------------------------------------------------
    def swap_out(self, req: int):
        """([(gpu, cpu)], released) or None if the CPU pool is too small."""
        buf = np.empty(2 * max(1, self.num_blocks), dtype=np.int32)
        rel = C.c_int32(0)
        n = lib().pkv_alloc_swap_out(self._h, req, _ptr(buf), len(buf) // 2, C.byref(rel))
        if n == -4:
            return None
        _check(n, "swap_out")
        return [(int(buf[2 * i]), int(buf[2 * i + 1])) for i in range(n)], rel.value

    def swap_in_status(self, req: int) -> str:
        st = _check(lib().pkv_alloc_swap_in_status(self._h, req), "swap_in_status")
        return ("ok", "later", "never")[st]

    def swap_in(self, req: int) -> list[tuple[int, int]]:
        buf = np.empty(2 * max(1, self.num_blocks), dtype=np.int32)
        n = _check(lib().pkv_alloc_swap_in(self._h, req, _ptr(buf), len(buf) // 2), "swap_in")
        return [(int(buf[2 * i]), int(buf[2 * i + 1])) for i in range(n)]

    def swapped_blocks(self, req: int):
        """(CPU blocks, T_i) of a swapped request, or ([], 0)."""
        buf = np.empty(max(1, self.num_cpu_blocks), dtype=np.int32)
        tok = C.c_int64(0)
        n = _check(lib().pkv_alloc_swapped_blocks(self._h, req, _ptr(buf), len(buf),
                                                  C.byref(tok)), "swapped_blocks")
        return buf[:n].tolist(), tok.value

    def cpu_free_list(self) -> list[int]:
        buf = np.empty(max(1, self.num_cpu_blocks), dtype=np.int32)
        n = _check(lib().pkv_alloc_cpu_free_list(self._h, _ptr(buf), len(buf)), "cpu_free_list")
        return buf[:n].tolist()


class Scheduler:
    """Continuous-batching scheduler with recompute preemption (host)."""

    def __init__(self, max_num_seqs, max_num_batched_tokens, chunk_size, max_model_len,
                 block_size, num_blocks, max_blocks_per_req, artificial_preempt_prob=0.0,
                 artificial_preempt_max=0, artificial_seed=0, preemption_mode="recompute",
                 num_cpu_blocks=0):
        if preemption_mode not in ("recompute", "swap"):
            raise ValueError("preemption_mode must be 'recompute' or 'swap'")
        swap = preemption_mode == "swap"
        cfg = _ffi.SchedConfig(max_num_seqs, max_num_batched_tokens, chunk_size, max_model_len,
                               block_size, num_blocks, max_blocks_per_req, artificial_preempt_max,
                               artificial_preempt_prob, artificial_seed, 1 if swap else 0,
                               num_cpu_blocks)
        self._h = lib().pkv_sched_create(C.byref(cfg))
        if not self._h:
            raise PkvError(-1, "pkv_sched_create")
        self.num_blocks = num_blocks
        self.max_blocks_per_req = max_blocks_per_req
        self.allocator = Allocator(num_blocks, block_size, _handle=lib().pkv_sched_allocator(self._h),
                                   num_cpu_blocks=num_cpu_blocks if swap else 0)
        self.info = _ffi.StepInfo()

    def __del__(self):
        if getattr(self, "_h", None):
            lib().pkv_sched_destroy(self._h)
            self._h = None

    def add_request(self, req_id: int, prompt_len: int, max_output: int, namespace: int = 0,
                    tokens=None) -> bool:
        """Queue a request; with `tokens` (its prompt's token ids) it takes part in
        prefix sharing within `namespace`."""
        if tokens is None:
            code = lib().pkv_sched_add_request(self._h, req_id, prompt_len, max_output)
        else:
            t = np.ascontiguousarray(tokens, dtype=np.int32)
            if len(t) != prompt_len:
                return False
            code = lib().pkv_sched_add_request_tokens(self._h, req_id, prompt_len, max_output,
                                                      namespace, _ptr(t))
        return bool(_check(code, "add_request"))

    def step(self) -> dict:
        _check(lib().pkv_sched_step(self._h, C.byref(self.info)), "step")
        i = self.info
        n = i.num_reqs
        ids = np.empty(n, np.int32)
        toks = np.empty(n, np.int32)
        before = np.empty(n, np.int32)
        lib().pkv_sched_plan(self._h, _ptr(ids), _ptr(toks), _ptr(before), n)
        pre = np.empty(max(i.num_preempted, 1), np.int32)
        adm = np.empty(max(i.num_admitted, 1), np.int32)
        lib().pkv_sched_preempted(self._h, _ptr(pre), len(pre))
        lib().pkv_sched_admitted(self._h, _ptr(adm), len(adm))
        no, ni = C.c_int32(0), C.c_int32(0)
        _check(lib().pkv_sched_swaps(self._h, None, 0, C.byref(no), None, 0, C.byref(ni)), "swaps")
        outp = np.empty(2 * max(1, no.value), np.int32)
        inp = np.empty(2 * max(1, ni.value), np.int32)
        _check(lib().pkv_sched_swaps(self._h, _ptr(outp), no.value, C.byref(no), _ptr(inp),
                                     ni.value, C.byref(ni)), "swaps")
        cap = 1 << 12
        so, si, ig = (np.empty(cap, np.int32) for _ in range(3))
        nso, nsi, nig = C.c_int32(0), C.c_int32(0), C.c_int32(0)
        _check(lib().pkv_sched_swap_events(self._h, _ptr(so), C.byref(nso), _ptr(si),
                                           C.byref(nsi), _ptr(ig), C.byref(nig), cap), "swap_events")
        return {"entries": list(zip(ids.tolist(), toks.tolist(), before.tolist())),
                "preempted": pre[:i.num_preempted].tolist(), "admitted": adm[:i.num_admitted].tolist(),
                "swap_out_pairs": [tuple(x) for x in outp[:2 * no.value].reshape(-1, 2).tolist()],
                "swap_in_pairs": [tuple(x) for x in inp[:2 * ni.value].reshape(-1, 2).tolist()],
                "swapped_out": so[:nso.value].tolist(), "swapped_in": si[:nsi.value].tolist(),
                "ignored": ig[:nig.value].tolist(),
                "num_tokens": int(i.num_tokens), "max_blocks": int(i.max_blocks),
                "max_query_len": int(i.max_query_len)}

    def build_metadata(self, block_table, query_start_loc, seq_lens, num_computed, slot_mapping):
        """Fill caller-owned numpy buffers (e.g. views of pinned host tensors)."""
        _check(lib().pkv_sched_build_metadata(
            self._h, _ptr(block_table), block_table.shape[1], _ptr(query_start_loc),
            _ptr(seq_lens), _ptr(num_computed), _ptr(slot_mapping)), "build_metadata")

    def metadata(self, stride: int | None = None):
        i = self.info
        stride = stride or max(int(i.max_blocks), 1)
        bt = np.empty((i.num_reqs, stride), np.int32)
        qsl = np.empty(i.num_reqs + 1, np.int32)
        seq = np.empty(i.num_reqs, np.int32)
        nc = np.empty(i.num_reqs, np.int32)
        slots = np.empty(int(i.num_tokens), np.int64)
        self.build_metadata(bt, qsl, seq, nc, slots)
        return bt, qsl, seq, nc, slots

    def finish_step(self, executed_ok: bool) -> list[int]:
        buf = np.empty(1024, np.int32)
        n = _check(lib().pkv_sched_finish_step(self._h, 1 if executed_ok else 0, _ptr(buf),
                                               len(buf)), "finish_step")
        return buf[:min(n, len(buf))].tolist()

    def request(self, req_id: int) -> dict | None:
        st = _ffi.RequestState()
        code = lib().pkv_sched_request(self._h, req_id, C.byref(st))
        if code == -6:
            return None
        _check(code, "request")
        return {n: getattr(st, n) for n, _ in st._fields_ if n != "pad_"}

    def queues(self):
        cap = 1 << 16
        run = np.empty(cap, np.int32)
        wait = np.empty(cap, np.int32)
        nr, nw = C.c_int32(0), C.c_int32(0)
        _check(lib().pkv_sched_queues(self._h, _ptr(run), C.byref(nr), _ptr(wait), C.byref(nw),
                                      cap), "queues")
        return run[:nr.value].tolist(), wait[:nw.value].tolist()

    def swapped_queue(self) -> list[int]:
        cap = 1 << 16
        buf = np.empty(cap, np.int32)
        n = C.c_int32(0)
        _check(lib().pkv_sched_swapped_queue(self._h, _ptr(buf), C.byref(n), cap), "swapped_queue")
        return buf[:n.value].tolist()

    def counters(self) -> dict:
        out = (C.c_int64 * 4)()
        _check(lib().pkv_sched_counters(self._h, out), "counters")
        return {"preemptions": out[0], "recomputed_tokens": out[1], "finished": out[2],
                "inject_left": out[3]}
