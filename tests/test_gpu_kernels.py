"""GPU parity of reshape_and_cache and paged_attention_varlen against the oracle.

Bit-exact cache images for reshape_and_cache; float tolerances for attention:
max-abs <= 1e-5 in float32; max-abs <= 2e-2 and relative Frobenius error
<= 1e-2 (overall and per request) in bfloat16.
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import paging
from tests.gpu_support import Batch, compare
from workloads import configs
from workloads.configs import KVHistory
from workloads.generators import randn_fp32, random_block_placement, uniform_int

pytestmark = pytest.mark.gpu


def _pkv():
    import paged_kv_cache_36_gb300 as pkv
    return pkv


def _sub_history(tensors_k, tensors_v):
    lengths = np.array([k.shape[0] for k in tensors_k], np.int64)
    offsets = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
    return KVHistory(torch.cat(tensors_k), torch.cat(tensors_v), lengths, offsets)


# ---------------------------------------------------------------- reshape_and_cache
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("hkv,d", [(2, 64), (8, 128)])
def test_reshape_and_cache_bit_exact(dtype, hkv, d):
    pkv = _pkv()
    NB, B, T = 64, 16, 300
    g = torch.Generator().manual_seed(7)
    key = torch.randn(T, hkv, d, generator=g).to(dtype)
    value = torch.randn(T, hkv, d, generator=g).to(dtype)
    slots = torch.randperm(NB * B, generator=g)[:T].to(torch.int64)
    slots[::17] = -1                                          # padding tokens
    kc_ref = torch.randn(NB, B, hkv, d, generator=g).to(dtype)
    vc_ref = torch.randn(NB, B, hkv, d, generator=g).to(dtype)
    kc, vc = kc_ref.cuda(), vc_ref.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.reshape_and_cache(key.cuda(), value.cuda(), kc, vc, slots.cuda(), error_word=err)
    paging.write_cache(kc_ref, vc_ref, key, value, slots.tolist())
    torch.cuda.synchronize()
    assert torch.equal(kc.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       kc_ref.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    assert torch.equal(vc.cpu(), vc_ref)
    assert err.item() == 0


def test_reshape_and_cache_strided_input_and_bad_slot():
    pkv = _pkv()
    NB, B, hkv, d, T = 8, 16, 2, 64, 40
    qkv = torch.randn(T, 3 * hkv, d, dtype=torch.bfloat16)     # fused rows: K, V are strided views
    key, value = qkv[:, hkv:2 * hkv], qkv[:, 2 * hkv:]
    slots = torch.arange(T, dtype=torch.int64)
    slots[5] = NB * B + 3                                       # past the pool: skipped and flagged
    kc = torch.zeros(NB, B, hkv, d, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    kg, vg = kc.cuda(), vc.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qg = qkv.cuda()
    pkv.reshape_and_cache(qg[:, hkv:2 * hkv], qg[:, 2 * hkv:], kg, vg, slots.cuda(), error_word=err)
    good = [int(s) if i != 5 else -1 for i, s in enumerate(slots)]
    paging.write_cache(kc, vc, key, value, good)
    torch.cuda.synchronize()
    assert torch.equal(kg.cpu(), kc) and torch.equal(vg.cpu(), vc)
    assert err.item() & pkv.ERR_SLOT


# ---------------------------------------------------------------- tiny config
def _tiny_batch(case, reqs, query_len, num_computed, dtype):
    """Batch over requests `reqs` of the tiny case (their own histories)."""
    kv = _sub_history([case.kv.k(r) for r in reqs], [case.kv.v(r) for r in reqs])
    q = torch.cat([case.q[r][nc:nc + ql] for r, nc, ql in zip(reqs, num_computed, query_len)])
    blocks = [np.array(case.block_tables[r], np.int32) for r in reqs]
    b = Batch(kv, blocks, case.num_blocks, query_len, num_computed, q, case.num_heads, dtype)
    return b


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_tiny_decode_step(dtype):
    case = configs.tiny_fp32_case(dtype)
    # request 0: 40 tokens, query at position 39 (slot 199); request 1: 20 tokens, position 19 (slot 115)
    b = _tiny_batch(case, [0, 1], [1, 1], [39, 19], dtype).alloc_cache().fill_history().upload_metadata()
    assert b.slot_mapping.tolist() == [199, 115]
    b.write_new_tokens()
    out = b.attention()
    compare(out, b.oracle(), b.qsl_host, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_tiny_chunked_prefill_equals_full(dtype):
    case = configs.tiny_fp32_case(dtype)
    pkv = _pkv()
    shape = (case.num_blocks, 16, case.num_kv_heads, case.head_dim)
    kc = torch.empty(shape, dtype=dtype, device="cuda")
    vc = torch.empty_like(kc)
    chunks = []
    for a, e in [(0, 3), (3, 6), (6, 7)]:
        b = _tiny_batch(case, [1], [e - a], [a], dtype)
        b.key_cache, b.value_cache = kc, vc                # the cache carries over between chunks
        b.upload_metadata()
        assert b.slot_mapping.tolist() == list(range(48 + a, 48 + e))
        b.write_new_tokens()
        chunks.append(b.attention().clone())
        compare(chunks[-1], b.oracle(), b.qsl_host, dtype)
    full_b = _tiny_batch(case, [1], [7], [0], dtype).alloc_cache().upload_metadata().write_new_tokens()
    full = full_b.attention()
    chunked = torch.cat(chunks)
    ref = full_b.oracle()
    compare(chunked, ref, full_b.qsl_host, dtype)
    compare(full, ref, full_b.qsl_host, dtype)
    if dtype == torch.float32:
        assert (chunked - full).abs().max().item() <= 1e-5


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_tiny_mixed_step(dtype):
    case = configs.tiny_fp32_case(dtype)
    # request 0 decodes at position 39 while request 1 runs chunk [3, 6)
    b = _tiny_batch(case, [0, 1], [1, 3], [39, 3], dtype).alloc_cache().fill_history().upload_metadata()
    assert b.slot_mapping.tolist() == [199, 51, 52, 53]
    b.write_new_tokens()
    compare(b.attention(), b.oracle(), b.qsl_host, dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_tiny_alternative_readings(dtype):
    """The other readings of the tiny configuration: (a) request 0 holds 40
    cached tokens and decodes at position 40 (slot 200); (b) request 1's last
    7 of 20 tokens run in chunks (13,16), (16,19), (19,20) over 13 cached
    ones, and their concatenated outputs equal one 7-token chunk."""
    case = configs.tiny_fp32_case(dtype)
    h, hkv, d = case.num_heads, case.num_kv_heads, case.head_dim
    # (a) a 41-token history for request 0
    k41 = randn_fp32((41, hkv, d), "tiny_alt", "k", dtype=dtype)
    v41 = randn_fp32((41, hkv, d), "tiny_alt", "v", dtype=dtype)
    q41 = randn_fp32((1, h, d), "tiny_alt", "q", dtype=dtype)
    kv = KVHistory(k41, v41, np.array([41], np.int64), np.array([0], np.int64))
    b = Batch(kv, [np.array([5, 8, 12], np.int32)], case.num_blocks, [1], [40], q41, h, dtype)
    b.alloc_cache().fill_history().upload_metadata()
    assert b.slot_mapping.tolist() == [200]
    b.write_new_tokens()
    compare(b.attention(), b.oracle(), b.qsl_host, dtype)
    # (b) chunks over request 1's positions [13, 20)
    shape = (case.num_blocks, 16, hkv, d)
    kc = torch.empty(shape, dtype=dtype, device="cuda")
    vc = torch.empty_like(kc)
    outs = []
    for i, (a, e) in enumerate([(13, 16), (16, 19), (19, 20)]):
        bb = _tiny_batch(case, [1], [e - a], [a], dtype)
        bb.key_cache, bb.value_cache = kc, vc
        if i == 0:
            bb.fill_history()                              # positions 0..12
        bb.upload_metadata()
        assert bb.slot_mapping.tolist() == {13: [61, 62, 63], 16: [112, 113, 114], 19: [115]}[a]
        bb.write_new_tokens()
        outs.append(bb.attention().clone())
        compare(outs[-1], bb.oracle(), bb.qsl_host, dtype)
    whole = _tiny_batch(case, [1], [7], [13], dtype).alloc_cache().fill_history()
    whole.upload_metadata().write_new_tokens()
    ref = whole.oracle()
    compare(torch.cat(outs), ref, whole.qsl_host, dtype)
    compare(whole.attention(), ref, whole.qsl_host, dtype)


# ---------------------------------------------------------------- random varlen batches
CASES = [
    # (H, Hkv, D, query lens, num_computed) - several tiles, ragged tails, empty requests
    (32, 8, 128, [1, 1, 1, 1, 1, 1], [0, 15, 16, 17, 250, 1031]),
    (32, 8, 128, [1, 37, 0, 1, 130, 1], [700, 0, 5, 3000, 300, 44]),
    (8, 8, 64, [1, 5, 1, 64], [100, 30, 1, 0]),
    (16, 2, 128, [1, 1, 2, 1], [513, 2, 77, 4095]),
    (64, 8, 128, [1, 1, 9], [2000, 31, 100]),
    (4, 1, 64, [1, 20, 1], [63, 16, 1000]),
    # prefill rows spanning several query tiles, with ragged last tiles and
    # query-tile counts that are not a multiple of 2 or 4
    (32, 8, 128, [70, 1, 45], [0, 10, 1000]),
    (32, 8, 128, [300, 129, 1, 64], [0, 2500, 40, 7]),
    (16, 4, 64, [200, 33], [5, 100]),
    (64, 8, 128, [100, 1], [3000, 5]),
    (16, 8, 128, [150], [17]),
    (32, 2, 128, [40, 1], [60, 9]),
    # one query tile per request (single-CTA tiles) over long histories
    (32, 8, 128, [32, 1, 17], [1500, 20, 3000]),
    (8, 8, 64, [128, 1], [2000, 700]),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_random_varlen_bf16(case):
    H, Hkv, D, qlens, ncs = CASES[case]
    name = f"varlen{case}"
    seq = [a + b for a, b in zip(qlens, ncs)]
    counts = [max(1, (s + 15) // 16) for s in seq]
    NB = 4 * sum(counts) + 8
    blocks = random_block_placement(NB, counts, name, "placement")
    lengths = np.array(seq, np.int64)
    offsets = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
    n = int(lengths.sum())
    kv = KVHistory(randn_fp32((n, Hkv, D), name, "k", dtype=torch.bfloat16),
                   randn_fp32((n, Hkv, D), name, "v", dtype=torch.bfloat16), lengths, offsets)
    q = randn_fp32((sum(qlens), H, D), name, "q", dtype=torch.bfloat16)
    b = Batch(kv, blocks, NB, qlens, ncs, q, H, torch.bfloat16).alloc_cache().fill_history()
    b.upload_metadata().write_new_tokens()
    compare(b.attention(), b.oracle(), b.qsl_host, torch.bfloat16)


def _repeat_case(name, qlens, ncs, H=32, Hkv=8, D=128, reps=12):
    seq = [a + b for a, b in zip(qlens, ncs)]
    counts = [(s + 15) // 16 for s in seq]
    NB = sum(counts) + 64
    blocks = random_block_placement(NB, counts, name, "placement")
    lengths = np.array(seq, np.int64)
    offsets = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
    n = int(lengths.sum())
    kv = KVHistory(randn_fp32((n, Hkv, D), name, "k", dtype=torch.bfloat16),
                   randn_fp32((n, Hkv, D), name, "v", dtype=torch.bfloat16), lengths, offsets)
    q = randn_fp32((sum(qlens), H, D), name, "q", dtype=torch.bfloat16)
    b = Batch(kv, blocks, NB, qlens, ncs, q, H, torch.bfloat16).alloc_cache().fill_history()
    b.upload_metadata().write_new_tokens()
    ws = _pkv().new_workspace(b.R, H, D)
    first = b.attention(ws).clone()
    compare(first, b.oracle(), b.qsl_host, torch.bfloat16)
    for _ in range(reps):
        again = b.attention(ws)
        assert torch.equal(again, first), "output changed between identical calls"


def test_repeated_single_tile_requests_over_long_histories():
    """96 requests of one query tile each (32 tokens, 4 query heads per KV
    head) over 1000-3000 computed tokens: one CTA per tile, many key tiles.
    Every call must match the oracle bit for bit with the first; the softmax
    warps here can run two key tiles ahead of the PV products, which is what
    the epilogue's wait must tolerate."""
    R = 96
    ncs = uniform_int(1000, 3000, R, "repeat1", "nc").tolist()
    _repeat_case("repeat1", [32] * R, ncs)


def test_repeated_long_chunk():
    """The 512-token chunk at [1536, 2048) repeated: every CTA's tile plan and
    barrier phases must give the same bits on every call."""
    _repeat_case("repeat2", [512], [1536])


def test_workspace_reuse_and_error_word():
    pkv = _pkv()
    H, Hkv, D = 32, 8, 128
    name = "reuse"
    ctx = [3000, 200, 4096, 17]
    counts = [(c + 15) // 16 for c in ctx]
    NB = sum(counts) + 4
    blocks = random_block_placement(NB, counts, name, "placement")
    lengths = np.array(ctx, np.int64)
    offsets = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
    kv = KVHistory(randn_fp32((int(lengths.sum()), Hkv, D), name, "k", dtype=torch.bfloat16),
                   randn_fp32((int(lengths.sum()), Hkv, D), name, "v", dtype=torch.bfloat16),
                   lengths, offsets)
    q = randn_fp32((4, H, D), name, "q", dtype=torch.bfloat16)
    b = Batch(kv, blocks, NB, [1] * 4, [c - 1 for c in ctx], q, H, torch.bfloat16)
    b.alloc_cache().fill_history().upload_metadata().write_new_tokens()
    ws = pkv.new_workspace(64, H, D)
    first = b.attention(workspace=ws).clone()
    second = b.attention(workspace=ws).clone()
    assert torch.equal(first, second)                 # split counters were left at zero
    compare(first, b.oracle(), b.qsl_host, torch.bfloat16)
    assert pkv.read_error_word(ws) == 0
    # an out-of-range block id is reported, not faulted on (TMA reads zeros there)
    bad = b.block_table.clone()
    bad[1, 0] = NB + 5
    pkv.paged_attention_varlen(b.q, b.key_cache, b.value_cache, bad, b.qsl, b.seq_lens, b.nc,
                               1 / math.sqrt(D), workspace=ws, max_query_len=1)
    assert pkv.read_error_word(ws) & pkv.ERR_BLOCK_ID
    ws.zero_()
    third = b.attention(workspace=ws)
    assert torch.equal(first, third)


def test_workspace_shared_across_batch_sizes():
    # one workspace serves batches of different sizes in any order: the split
    # counters must not move with the batch size
    pkv = _pkv()
    H, Hkv, D = 32, 8, 128
    batches = []
    for i, ctx in enumerate([[3000, 5000, 800, 4000, 2500, 9000, 700, 6000, 100, 3300],
                             [7000, 90, 4100], [1500] * 12 + [8000, 12000]]):
        name = f"shared_ws_{i}"
        counts = [(c + 15) // 16 for c in ctx]
        NB = sum(counts) + 4
        blocks = random_block_placement(NB, counts, name, "placement")
        lengths = np.array(ctx, np.int64)
        offsets = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
        kv = KVHistory(randn_fp32((int(lengths.sum()), Hkv, D), name, "k", dtype=torch.bfloat16),
                       randn_fp32((int(lengths.sum()), Hkv, D), name, "v", dtype=torch.bfloat16),
                       lengths, offsets)
        q = randn_fp32((len(ctx), H, D), name, "q", dtype=torch.bfloat16)
        b = Batch(kv, blocks, NB, [1] * len(ctx), [c - 1 for c in ctx], q, H, torch.bfloat16)
        batches.append(b.alloc_cache().fill_history().upload_metadata().write_new_tokens())
    fresh = [b.attention().clone() for b in batches]
    ws = pkv.new_workspace(256, H, D)
    for order in [0, 1, 2, 1, 0, 2, 2, 1]:
        got = batches[order].attention(workspace=ws)
        assert torch.equal(got, fresh[order]), order
    compare(fresh[2], batches[2].oracle(), batches[2].qsl_host, torch.bfloat16)


# ---------------------------------------------------------------- full-size configs
def _decode_cfg_batch(cfg):
    return Batch(cfg.kv, cfg.blocks, cfg.num_blocks, np.ones(len(cfg.context), np.int64),
                 cfg.context - 1, cfg.q, cfg.num_heads, cfg.dtype)


def test_decode_llama8b_64_requests():
    cfg = configs.decode_batch_llama8b()
    b = _decode_cfg_batch(cfg).alloc_cache().fill_history().upload_metadata().write_new_tokens()
    out = b.attention()
    compare(out, b.oracle(), b.qsl_host, torch.bfloat16)


def test_mixed_chunk512_beside_256_decodes():
    cfg = configs.mixed_chunked_step()
    b = Batch(cfg.kv, cfg.blocks, cfg.num_blocks, cfg.query_len, cfg.num_computed, cfg.q,
              cfg.num_heads, cfg.dtype).alloc_cache().fill_history().upload_metadata()
    b.write_new_tokens()
    # this step's 768 new tokens landed bit-exactly at their slots
    _, _, slots = b.new_tokens()
    got = b.key_cache.view(-1, b.Hkv, b.D)[torch.tensor(slots, device="cuda")]
    assert torch.equal(got, b.k_new)
    out = b.attention()
    compare(out, b.oracle(), b.qsl_host, torch.bfloat16)


@pytest.mark.slow
def test_long_decode_llama70b_8x131072():
    cfg = configs.long_decode_llama70b()
    b = _decode_cfg_batch(cfg).alloc_cache().fill_history().upload_metadata().write_new_tokens()
    out = b.attention()
    compare(out, b.oracle(), b.qsl_host, torch.bfloat16)


def test_validate_mode_reports_kernel_error_bits(monkeypatch):
    """PKV_VALIDATE=1: an inconsistent seq_len (metadata error bit) makes the
    call itself fail; without it the call succeeds and the bit waits in the
    error word."""
    pkv = _pkv()
    case = configs.tiny_fp32_case(torch.bfloat16)
    b = _tiny_batch(case, [0, 1], [1, 1], [39, 19], torch.bfloat16).alloc_cache().fill_history()
    b.upload_metadata().write_new_tokens()
    monkeypatch.setenv("PKV_VALIDATE", "1")
    b.attention()                                          # consistent: passes validation
    b.seq_lens[1] += 5                                     # seq_len != num_computed + 1
    ws = pkv.new_workspace(b.R, b.H, b.D)
    with pytest.raises(pkv.PkvError, match="error bits 0x4"):
        pkv.paged_attention_varlen(b.q, b.key_cache, b.value_cache, b.block_table, b.qsl,
                                   b.seq_lens, b.nc, 0.125, workspace=ws, max_query_len=1)
    monkeypatch.delenv("PKV_VALIDATE")
    ws = pkv.new_workspace(b.R, b.H, b.D)
    pkv.paged_attention_varlen(b.q, b.key_cache, b.value_cache, b.block_table, b.qsl,
                               b.seq_lens, b.nc, 0.125, workspace=ws, max_query_len=1)
    assert pkv.read_error_word(ws) & pkv.ERR_METADATA
