"""The C-ABI library loads and exports every entry point include/pkv.h declares
(no GPU needed: nothing here launches a kernel)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_symbols():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(pkv_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def libpkv():
    from paged_kv_cache_36_gb300 import build
    return ctypes.CDLL(build.build())


def test_header_declares_entry_points():
    names = declared_symbols()
    for must in ["pkv_reshape_and_cache", "pkv_paged_attention_varlen",
                 "pkv_attention_workspace_bytes", "pkv_alloc_reserve", "pkv_alloc_commit",
                 "pkv_alloc_rollback", "pkv_sched_step", "pkv_build_slot_mapping"]:
        assert must in names


def test_every_declared_symbol_is_exported(libpkv):
    missing = [n for n in declared_symbols() if not hasattr(libpkv, n)]
    assert not missing, missing


def test_binding_signatures_cover_header():
    from paged_kv_cache_36_gb300 import _ffi
    assert set(declared_symbols()) <= set(_ffi.SIGNATURES)


def test_version_and_error_string(libpkv):
    import paged_kv_cache_36_gb300 as pkv
    assert pkv.lib().pkv_version() >= 1
    # a host-side error sets the thread-local message
    assert pkv.lib().pkv_alloc_commit(None) == -1
    assert b"null handle" in pkv.lib().pkv_last_error()


def test_bad_arguments_rejected_without_gpu(libpkv):
    import paged_kv_cache_36_gb300 as pkv
    L = pkv.lib()
    # block_size other than 16 is refused before any CUDA call
    rc = L.pkv_paged_attention_varlen(None, 0, None, None, None, 0, None, None, None, 1.0, None,
                                      0, 1, 1, 16, 8, 4, 2, 64, 1, 0, None, 0, None)
    assert rc == -2
    rc = L.pkv_reshape_and_cache(None, None, 0, 0, None, None, None, 1, 16, 16, 2, 64, 7, None, None)
    assert rc == -2


def test_rope_argument_checks(libpkv):
    """Host-side validation of the fused RoPE entry point (nothing launches)."""
    import paged_kv_cache_36_gb300 as pkv
    from paged_kv_cache_36_gb300 import _ffi
    lib = pkv.lib()
    f = lib.pkv_rope_reshape_and_cache

    def call(rd=128, neox=1, T=0, D=128, dtype=_ffi.PKV_BF16, max_pos=16):
        return f(None, None, 32 * D, 32, None, 8 * D, None, None, 8 * D, None, None, None, None,
                 max_pos, rd, neox, T, 64, 16, 8, D, dtype, None, None)

    assert call() == 0                                   # zero tokens: nothing to do
    assert call(rd=127) == -1                            # odd rotary_dim
    assert call(rd=256) == -1                            # rotary_dim > head_dim
    assert call(rd=0) == -1
    assert call(max_pos=0) == -1
    assert call(dtype=5) == -2                           # unknown dtype
    assert call(rd=8, neox=1) == -2                      # NeoX half of 4 bf16 = 8 bytes
    assert call(rd=8, neox=0) == 0                       # interleaved 8 bf16 = 16 bytes
    assert call(T=3) == -1                               # null pointers with tokens to do
    assert b"null pointer" in lib.pkv_last_error()


def test_prepared_call_matches_the_eager_call_without_gpu(libpkv):
    """The prepared form passes the same arguments as the eager binding: on a
    machine without a GPU both fail the same way (block_size 8 is refused
    before any CUDA call), and the prepared call raises on every call."""
    import torch
    import paged_kv_cache_36_gb300 as pkv
    T, H, Hkv, D, R, NB = 4, 8, 2, 64, 2, 16
    q = torch.zeros(T, H, D, dtype=torch.bfloat16)
    kc = torch.zeros(NB, 8, Hkv, D, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    k = torch.zeros(T, Hkv, D, dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    slots = torch.zeros(T, dtype=torch.int64)
    bt = torch.zeros(R, 4, dtype=torch.int32)
    qsl = torch.tensor([0, 2, 4], dtype=torch.int32)
    seq = torch.tensor([2, 2], dtype=torch.int32)
    nc = torch.zeros(R, dtype=torch.int32)
    out = torch.empty_like(q)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)

    class _S:  # a stand-in stream object (no CUDA here)
        cuda_stream = 0

    args = (k, v, slots, q, kc, vc, bt, qsl, seq, nc, 0.125)
    with pytest.raises(pkv.PkvError) as eager:
        pkv.reshape_and_cache_paged_attention(*args, out=out, workspace=ws, max_query_len=2,
                                              stream=_S())
    call = pkv.prepare_reshape_and_cache_paged_attention(*args, out=out, workspace=ws,
                                                         max_query_len=2, stream=_S())
    for _ in range(2):
        with pytest.raises(pkv.PkvError) as prepared:
            call()
        assert prepared.value.code == eager.value.code
        assert "block_size" in str(prepared.value)
