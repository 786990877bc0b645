"""GPU parity of reshape_and_cache + paged_attention_varlen in one call.

For bf16 the two run as one kernel.  A decode row's CTA writes the token's
K/V row to its slot and uses it in place of the cache's copy; the prefill
CTAs write the rows of their own query tiles and meet at a counter in the
workspace before reading K/V.  Outputs and cache image must equal those of
the two separate calls bit for bit (the same bf16 values meet the same
arithmetic), and match the oracle within the bf16 tolerance; float32 steps
run the two kernels one after the other and must equal the separate calls
too.
"""

import math

import numpy as np
import pytest
import torch

from tests.gpu_support import Batch, compare, host_buffer_is_device_mapped
from workloads import configs
from workloads.configs import KVHistory
from workloads.generators import randn_fp32, random_block_placement

pytestmark = pytest.mark.gpu


def _pkv():
    import paged_kv_cache_36_gb300 as pkv
    return pkv


def _batch(name, H, Hkv, D, qlens, ncs, dtype=torch.bfloat16, spare=8):
    seq = [a + b for a, b in zip(qlens, ncs)]
    counts = [max(1, (s + 15) // 16) for s in seq]
    NB = 2 * sum(counts) + spare
    blocks = random_block_placement(NB, counts, name, "placement")
    lengths = np.array(seq, np.int64)
    offsets = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
    n = int(lengths.sum())
    kv = KVHistory(randn_fp32((n, Hkv, D), name, "k", dtype=dtype),
                   randn_fp32((n, Hkv, D), name, "v", dtype=dtype), lengths, offsets)
    q = randn_fp32((sum(qlens), H, D), name, "q", dtype=dtype)
    b = Batch(kv, blocks, NB, qlens, ncs, q, H, dtype).alloc_cache().fill_history().upload_metadata()
    k, v, _ = b.new_tokens()
    b.k_new, b.v_new = k.to("cuda", dtype), v.to("cuda", dtype)
    return b


def _fused(b, slot_mapping=None, workspace=None):
    pkv = _pkv()
    ws = workspace if workspace is not None else pkv.new_workspace(b.R, b.H, b.D)
    out = pkv.reshape_and_cache_paged_attention(
        b.k_new, b.v_new, b.slot_mapping if slot_mapping is None else slot_mapping, b.q,
        b.key_cache, b.value_cache, b.block_table, b.qsl, b.seq_lens, b.nc,
        1.0 / math.sqrt(b.D), workspace=ws, max_query_len=int(b.query_len.max()))
    return out, ws


def _check_against_two_calls(b):
    pkv = _pkv()
    kc0, vc0 = b.key_cache.clone(), b.value_cache.clone()
    out, ws = _fused(b)
    torch.cuda.synchronize()
    assert pkv.read_error_word(ws) == 0
    fused_out = out.clone()
    kc1, vc1 = b.key_cache.clone(), b.value_cache.clone()
    # the same step as two calls, on the cache as it was before
    b.key_cache.copy_(kc0)
    b.value_cache.copy_(vc0)
    pkv.reshape_and_cache(b.k_new, b.v_new, b.key_cache, b.value_cache, b.slot_mapping)
    two = b.attention()
    # bit patterns: slots never written hold whatever the allocation had, NaNs included
    same = [torch.equal(x.view(torch.int16 if x.element_size() == 2 else torch.int32),
                        y.view(torch.int16 if y.element_size() == 2 else torch.int32))
            for x, y in ((b.key_cache, kc1), (b.value_cache, vc1))]
    assert all(same), "cache images differ"
    assert torch.equal(fused_out, two), "outputs differ from the two separate calls"
    compare(fused_out, b.oracle(), b.qsl_host, b.dtype)


def test_fused_decode_llama8b_64_requests():
    cfg = configs.decode_batch_llama8b()
    b = Batch(cfg.kv, cfg.blocks, cfg.num_blocks, np.ones(len(cfg.context), np.int64),
              cfg.context - 1, cfg.q, cfg.num_heads, cfg.dtype).alloc_cache().fill_history()
    b.upload_metadata()
    k, v, _ = b.new_tokens()
    b.k_new, b.v_new = k.to("cuda", b.dtype), v.to("cuda", b.dtype)
    _check_against_two_calls(b)


# (H, Hkv, D, contexts): seq_len % 16 in {0, 1, other}, a context of 1 (only
# the new token), GQA groups 1 to 16, head_dim 64 and 128
FUSED_CASES = [
    (32, 8, 128, [1, 16, 17, 33, 4096, 250, 4095, 2]),
    (8, 8, 64, [1, 64, 65, 1000]),
    (64, 4, 128, [300, 17, 16, 2048]),
    (16, 8, 128, [5000, 31, 1, 48]),
    (16, 1, 64, [129, 7, 3000]),
]


@pytest.mark.parametrize("case", range(len(FUSED_CASES)))
def test_fused_decode_random_shapes(case):
    H, Hkv, D, ctx = FUSED_CASES[case]
    b = _batch(f"fused{case}", H, Hkv, D, [1] * len(ctx), [c - 1 for c in ctx])
    _check_against_two_calls(b)


def test_fused_entry_with_prefill_rows_and_float32():
    # bf16 prefill rows: one kernel; float32: reshape_and_cache runs first
    b = _batch("fusedmix", 32, 8, 128, [1, 300, 1, 40], [999, 20, 15, 0])
    _check_against_two_calls(b)
    b = _batch("fusedf32", 4, 2, 64, [1, 7, 1], [39, 0, 19], dtype=torch.float32)
    _check_against_two_calls(b)


# (H, Hkv, D, query lengths, histories): a 512-token chunk beside decodes, a
# chunk starting inside a block, prompts only (many prefill CTAs meet), query
# lengths below one tile's tokens, GQA groups 1 to 16, head_dim 64
FUSED_MIXED_CASES = [
    (32, 8, 128, [512] + [1] * 24, [1536] + [int(x) for x in np.linspace(200, 6000, 24)]),
    (32, 8, 128, [37, 1, 1, 200], [1003, 77, 16, 5]),
    (32, 8, 128, [300] * 12, [0] * 12),
    (16, 8, 128, [2, 3, 1, 5], [14, 0, 40, 11]),
    (8, 8, 64, [130, 1, 64], [60, 500, 0]),
    (64, 4, 128, [97, 1, 33], [31, 1000, 200]),
    (16, 1, 64, [250, 1], [1, 3000]),
]


@pytest.mark.parametrize("case", range(len(FUSED_MIXED_CASES)))
def test_fused_mixed_and_prefill_steps(case):
    H, Hkv, D, qlens, ncs = FUSED_MIXED_CASES[case]
    b = _batch(f"fusedmixed{case}", H, Hkv, D, qlens, ncs)
    _check_against_two_calls(b)


def test_fused_chunked_prefill_steps_reuse_one_workspace():
    """A 700-token prompt prefilled in chunks of 256, 256 and 188 while three
    requests decode, on one cache and one workspace: each step through the
    fused call against the oracle (the prefill CTAs' meeting counter must be
    back at zero after every call), then the cache image."""
    pkv = _pkv()
    H, Hkv, D, name = 32, 8, 128, "fusedchunks"
    prompt, chunks = 700, [256, 256, 188]
    ctx0 = [90, 17, 2500]
    steps = len(chunks)
    final = [prompt] + [c + steps - 1 for c in ctx0]
    R = len(final)
    counts = [(f + 15) // 16 for f in final]
    NB = 2 * sum(counts) + 8
    blocks = random_block_placement(NB, counts, name, "placement")
    lengths = np.array(final, np.int64)
    offsets = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
    n = int(lengths.sum())
    kv = KVHistory(randn_fp32((n, Hkv, D), name, "k", dtype=torch.bfloat16),
                   randn_fp32((n, Hkv, D), name, "v", dtype=torch.bfloat16), lengths, offsets)
    qall = randn_fp32((steps, max(chunks) + R - 1, H, D), name, "q", dtype=torch.bfloat16)
    ws = pkv.new_workspace(R, H, D)
    cache = None
    done = 0
    for s in range(steps):
        qlens = [chunks[s]] + [1] * (R - 1)
        ncs = [done] + [c - 1 + s for c in ctx0]
        b = Batch(kv, blocks, NB, qlens, ncs, qall[s, :sum(qlens)], H, torch.bfloat16)
        if cache is None:
            # the decode requests' histories; the prompt has none yet
            b.alloc_cache().fill_history()
            cache = (b.key_cache, b.value_cache)
        b.key_cache, b.value_cache = cache
        b.upload_metadata()
        k, v, _ = b.new_tokens()
        b.k_new, b.v_new = k.to("cuda", b.dtype), v.to("cuda", b.dtype)
        out, _ = _fused(b, workspace=ws)
        torch.cuda.synchronize()
        assert pkv.read_error_word(ws) == 0, s
        compare(out, b.oracle(), b.qsl_host, b.dtype)
        # the prefill CTAs' meeting counter (header words 1 and 2) is back at zero
        assert ws[4:12].count_nonzero().item() == 0, s
        done += chunks[s]
    kf = cache[0].view(-1, Hkv, D)
    slots = [int(blocks[0][p // 16]) * 16 + p % 16 for p in range(prompt)]
    assert torch.equal(kf[torch.tensor(slots, device="cuda")].cpu(), kv.k(0)[:prompt])


def test_fused_prefill_slot_mismatch_sets_metadata_bit():
    pkv = _pkv()
    b = _batch("fusedbadp", 32, 8, 128, [1, 40, 1], [40, 17, 300], spare=64)
    bad = b.slot_mapping.clone()
    used = set(int(x) for row in b.blocks for x in row)
    spare_block = next(i for i in range(b.num_blocks) if i not in used)
    bad[5] = spare_block * 16 + 3  # a token of the prefill row
    out, ws = _fused(b, slot_mapping=bad)
    torch.cuda.synchronize()
    assert pkv.read_error_word(ws) & pkv.ERR_METADATA
    kf = b.key_cache.view(-1, b.Hkv, b.D)
    assert torch.equal(kf[bad[5]], b.k_new[5])
    # the decode requests are unaffected
    ref = b.oracle()
    compare(out, ref, b.qsl_host, b.dtype, rows=[0, 2])


def test_fused_decode_repeated_steps():
    """Ten decode steps in a row through the fused call on one cache, each
    appending a token to every request; every step against the oracle."""
    pkv = _pkv()
    H, Hkv, D, steps, name = 32, 8, 128, 10, "fusedrep"
    ctx0 = [100, 15, 16, 1777, 2]
    R = len(ctx0)
    final = [c + steps - 1 for c in ctx0]
    counts = [(f + 15) // 16 for f in final]
    NB = 2 * sum(counts) + 8
    blocks = random_block_placement(NB, counts, name, "placement")
    lengths = np.array(final, np.int64)
    offsets = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
    n = int(lengths.sum())
    kv = KVHistory(randn_fp32((n, Hkv, D), name, "k", dtype=torch.bfloat16),
                   randn_fp32((n, Hkv, D), name, "v", dtype=torch.bfloat16), lengths, offsets)
    qs = randn_fp32((steps, R, H, D), name, "q", dtype=torch.bfloat16)
    first = Batch(kv, blocks, NB, [1] * R, [c - 1 for c in ctx0], qs[0], H, torch.bfloat16)
    first.alloc_cache().fill_history()
    ws = pkv.new_workspace(R, H, D)
    for s in range(steps):
        b = Batch(kv, blocks, NB, [1] * R, [c - 1 + s for c in ctx0], qs[s], H, torch.bfloat16)
        b.key_cache, b.value_cache = first.key_cache, first.value_cache
        b.upload_metadata()
        k, v, _ = b.new_tokens()
        b.k_new, b.v_new = k.to("cuda", b.dtype), v.to("cuda", b.dtype)
        out, _ = _fused(b, workspace=ws)
        compare(out, b.oracle(), b.qsl_host, b.dtype)
    assert pkv.read_error_word(ws) == 0
    # the cache now holds every request's whole history, written step by step
    kf = first.key_cache.view(-1, Hkv, D)
    for r in range(R):
        slots = [int(blocks[r][p // 16]) * 16 + p % 16 for p in range(ctx0[r] - 1, final[r])]
        assert torch.equal(kf[torch.tensor(slots, device="cuda")].cpu(),
                           kv.k(r)[ctx0[r] - 1:final[r]])


def test_fused_decode_slot_mismatch_sets_metadata_bit():
    pkv = _pkv()
    b = _batch("fusedbad", 32, 8, 128, [1, 1, 1], [40, 17, 300], spare=64)
    bad = b.slot_mapping.clone()
    used = set(int(x) for row in b.blocks for x in row)
    spare_block = next(i for i in range(b.num_blocks) if i not in used)
    bad[1] = spare_block * 16 + 3
    out, ws = _fused(b, slot_mapping=bad)
    torch.cuda.synchronize()
    assert pkv.read_error_word(ws) & pkv.ERR_METADATA
    # reshape_and_cache semantics: the row still went to the given slot
    kf = b.key_cache.view(-1, b.Hkv, b.D)
    assert torch.equal(kf[bad[1]], b.k_new[1])
    # the other requests are unaffected
    ref = b.oracle()
    compare(out, ref, b.qsl_host, b.dtype, rows=[0, 2])


@pytest.mark.parametrize("kind", ["decode", "mixed", "float32"])
def test_fused_step_writes_out_into_pinned_host_memory(kind):
    """out may be pinned host memory that the device maps at its host address:
    the kernels only store to out, so the result lands in host memory without
    a device-to-host copy.  The same step with out on the device and with out
    in pinned host memory: equal bit for bit, and within the oracle's
    tolerance (the decode kernel, the mixed-batch kernel with both roles, and
    the float32 path)."""
    pkv = _pkv()
    if kind == "decode":
        H, Hkv, D, ctx = FUSED_CASES[0]
        b = _batch("pinnedout_dec", H, Hkv, D, [1] * len(ctx), [c - 1 for c in ctx])
    elif kind == "mixed":
        H, Hkv, D, qlens, ncs = FUSED_MIXED_CASES[1]
        b = _batch("pinnedout_mix", H, Hkv, D, qlens, ncs)
    else:
        b = _batch("pinnedout_f32", 4, 2, 64, [1, 7, 1], [39, 0, 19], dtype=torch.float32)
    host_out = torch.full(tuple(b.q.shape), float("nan"), dtype=b.q.dtype).pin_memory()
    if not host_buffer_is_device_mapped(host_out):
        pytest.skip("pinned host memory is not device-mapped at its host address here")
    kc0, vc0 = b.key_cache.clone(), b.value_cache.clone()
    dev_out, ws = _fused(b)
    torch.cuda.synchronize()
    assert pkv.read_error_word(ws) == 0
    b.key_cache.copy_(kc0)
    b.value_cache.copy_(vc0)
    ws2 = pkv.new_workspace(b.R, b.H, b.D)
    got = pkv.reshape_and_cache_paged_attention(
        b.k_new, b.v_new, b.slot_mapping, b.q, b.key_cache, b.value_cache, b.block_table,
        b.qsl, b.seq_lens, b.nc, 1.0 / math.sqrt(b.D), out=host_out, workspace=ws2,
        max_query_len=int(b.query_len.max()))
    torch.cuda.synchronize()
    assert got is host_out
    assert pkv.read_error_word(ws2) == 0
    assert torch.equal(host_out, dev_out.cpu())
    compare(host_out, b.oracle(), b.qsl_host, b.dtype)


def test_prepared_call_llama8b_decode_into_pinned_host_memory():
    """The end-to-end step as bench.py times it: the Llama-3-8B decode batch
    (64 requests, contexts 128-4096) through the binding's prepared call,
    with out in pinned host memory, called twice in a row (the second call
    writes the same new rows again); both results against the oracle."""
    pkv = _pkv()
    cfg = configs.decode_batch_llama8b()
    b = Batch(cfg.kv, cfg.blocks, cfg.num_blocks, np.ones(len(cfg.context), np.int64),
              cfg.context - 1, cfg.q, cfg.num_heads, cfg.dtype).alloc_cache().fill_history()
    b.upload_metadata()
    k, v, _ = b.new_tokens()
    b.k_new, b.v_new = k.to("cuda", b.dtype), v.to("cuda", b.dtype)
    host_out = torch.full(tuple(b.q.shape), float("nan"), dtype=b.q.dtype).pin_memory()
    if not host_buffer_is_device_mapped(host_out):
        pytest.skip("pinned host memory is not device-mapped at its host address here")
    ws = pkv.new_workspace(b.R, b.H, b.D)
    call = pkv.prepare_reshape_and_cache_paged_attention(
        b.k_new, b.v_new, b.slot_mapping, b.q, b.key_cache, b.value_cache, b.block_table, b.qsl,
        b.seq_lens, b.nc, 1.0 / math.sqrt(b.D), out=host_out, workspace=ws, max_query_len=1)
    ref = b.oracle()
    first = call()
    torch.cuda.synchronize()
    assert first is host_out
    assert pkv.read_error_word(ws) == 0
    compare(host_out, ref, b.qsl_host, b.dtype)
    saved = host_out.clone()
    host_out.fill_(float("nan"))
    call()
    torch.cuda.synchronize()
    assert pkv.read_error_word(ws) == 0
    assert torch.equal(host_out, saved)
