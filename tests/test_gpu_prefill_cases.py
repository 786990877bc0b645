"""More prefill batches on the GPU against the oracle: query tiles over long
histories, ragged tiles (odd tile counts, 2-3 token requests, a single
partial tile), batches with fewer tiles than the GPU has SMs, prompts from an
empty cache, and every query-head group size the kernel takes (G = 1, 2, 4,
16), each compared with the float64 oracle at the bf16 tolerances, and
repeated calls compared bit for bit.
"""

import numpy as np
import pytest
import torch

from tests.gpu_support import Batch, compare
from workloads.configs import KVHistory
from workloads.generators import randn_fp32, random_block_placement

pytestmark = pytest.mark.gpu


def _batch(name, qlens, ncs, H=32, Hkv=8, D=128):
    seq = [a + b for a, b in zip(qlens, ncs)]
    counts = [max(1, (s + 15) // 16) for s in seq]
    NB = sum(counts) + 64
    blocks = random_block_placement(NB, counts, name, "placement")
    lengths = np.array(seq, np.int64)
    offsets = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
    n = int(lengths.sum())
    kv = KVHistory(randn_fp32((n, Hkv, D), name, "k", dtype=torch.bfloat16),
                   randn_fp32((n, Hkv, D), name, "v", dtype=torch.bfloat16), lengths, offsets)
    q = randn_fp32((sum(qlens), H, D), name, "q", dtype=torch.bfloat16)
    b = Batch(kv, blocks, NB, qlens, ncs, q, H, torch.bfloat16).alloc_cache().fill_history()
    return b.upload_metadata().write_new_tokens()


CASES = {
    # one 64-token slice per KV head over a 16000-token history (126 key tiles)
    "long_history_short_chunk": ([64], [16000]),
    # the mixed step's chunk beside decodes of several lengths
    "chunk_and_decodes": ([512, 1, 1, 1, 1], [1536, 3000, 17, 8000, 250]),
    # ragged prefills: odd tile counts, 2-3 token requests, one request a
    # single partial tile
    "ragged": ([2, 3, 45, 97, 130, 1, 33], [0, 500, 1000, 7, 4000, 60, 2000]),
    # far fewer tiles than SMs: one 2-token prefill
    "tiny": ([2], [40]),
    # a 300-token chunk and a 40-token prompt beside two decodes
    "few_tiles": ([1, 300, 1, 40], [999, 20, 15, 0]),
    # several long prompts from an empty cache (many tiles per CTA)
    "prompts": ([1024, 777, 1500], [0, 0, 0]),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_prefill_case_matches_oracle(case):
    qlens, ncs = CASES[case]
    b = _batch(f"split_{case}", qlens, ncs)
    ws = torch.zeros(_pkv().attention_workspace_bytes(b.R, b.H, b.D), dtype=torch.uint8,
                     device="cuda")
    first = b.attention(workspace=ws).clone()
    compare(first, b.oracle(), b.qsl_host, torch.bfloat16)
    for _ in range(3):
        assert torch.equal(b.attention(workspace=ws), first)


@pytest.mark.parametrize("H,Hkv,D", [(8, 8, 64), (16, 8, 128), (32, 2, 128), (16, 4, 64)])
def test_prefill_across_group_sizes(H, Hkv, D):
    """G = 1, 2, 16, 4: 128, 64, 8 and 32 query tokens per 128-row tile."""
    qlens, ncs = [300, 1, 70, 5], [2100, 900, 0, 3000]
    b = _batch(f"split_g{H // Hkv}_d{D}", qlens, ncs, H=H, Hkv=Hkv, D=D)
    compare(b.attention(), b.oracle(), b.qsl_host, torch.bfloat16)


def _pkv():
    import paged_kv_cache_36_gb300 as pkv
    return pkv


@pytest.mark.parametrize("bad", ["prefill_row", "only_prefill_row", "decode_row"])
def test_mixed_call_with_a_bad_row(bad):
    """One kernel serves both kinds of rows: a row whose seq_len disagrees with
    num_computed + query length sets the metadata bit and is skipped, and the
    other rows still match the oracle (whichever role the bad row belongs to,
    including a call whose only prefill row is bad)."""
    pkv = _pkv()
    if bad == "only_prefill_row":
        qlens, ncs, victim = [1, 200, 1], [700, 300, 90], 1
    elif bad == "prefill_row":
        qlens, ncs, victim = [1, 200, 64, 1], [700, 300, 1000, 90], 1
    else:
        qlens, ncs, victim = [1, 200, 64, 1], [700, 300, 1000, 90], 3
    b = _batch(f"badrow_{bad}", qlens, ncs)
    ref = b.oracle()
    b.seq_lens[victim] += 3
    ws = pkv.new_workspace(b.R, b.H, b.D)
    out = pkv.paged_attention_varlen(b.q, b.key_cache, b.value_cache, b.block_table, b.qsl,
                                     b.seq_lens, b.nc, 1.0 / np.sqrt(b.D), workspace=ws,
                                     max_query_len=int(max(qlens)))
    torch.cuda.synchronize()
    assert pkv.read_error_word(ws) & pkv.ERR_METADATA
    rows = [r for r in range(b.R) if r != victim]
    compare(out, ref, b.qsl_host, torch.bfloat16, rows=rows)
