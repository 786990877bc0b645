"""GPU parity of the prefill path where each CTA walks many tiles: eight
2048-token prompts in one call, and one 16384-token prompt (query tiles of 1
to 128 key tiles, block-table batches that wrap many times).

The full oracle over these batches would take minutes in float64, so query
rows are sampled (first and last rows, tile and block edges, random rows).
The oracle of a row at absolute position p is the dense causal attention of
that one query over keys 0..p of its request: the same definition as a query
of length 1 after p computed tokens.  Tolerances as everywhere in bf16:
max-abs <= 2e-2 and relative Frobenius error <= 1e-2 over the sampled rows.
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention as oa
from tests.gpu_support import BF16_MAX_ABS, BF16_REL, Batch
from workloads.configs import KVHistory
from workloads.generators import randn_fp32, random_block_placement, uniform_int

pytestmark = pytest.mark.gpu


def _sampled_rows(prompt: int, name: str, n_random: int) -> list[int]:
    edges = [0, 1, 15, 16, 31, 32, 127, 128, 129, prompt // 2, prompt - 129, prompt - 128,
             prompt - 2, prompt - 1]
    rnd = uniform_int(0, prompt - 1, n_random, name, "rows").tolist()
    return sorted({int(r) for r in edges + rnd if 0 <= r < prompt})


def _check_prompts(name: str, nreq: int, prompt: int, n_random: int):
    H, Hkv, D = 32, 8, 128
    counts = [prompt // 16] * nreq
    NB = 2 * sum(counts) + 16
    blocks = random_block_placement(NB, counts, name, "placement")
    n = nreq * prompt
    lengths = np.full(nreq, prompt, np.int64)
    offsets = (np.arange(nreq) * prompt).astype(np.int64)
    kv = KVHistory(randn_fp32((n, Hkv, D), name, "k", dtype=torch.bfloat16),
                   randn_fp32((n, Hkv, D), name, "v", dtype=torch.bfloat16), lengths, offsets)
    q = randn_fp32((n, H, D), name, "q", dtype=torch.bfloat16)
    b = Batch(kv, blocks, NB, [prompt] * nreq, [0] * nreq, q, H, torch.bfloat16)
    b.alloc_cache().fill_history().upload_metadata().write_new_tokens()
    out = b.attention().double().cpu()
    assert torch.isfinite(out).all()
    scale = 1.0 / math.sqrt(D)
    got, ref = [], []
    for r in range(nreq):
        k, v = kv.k(r), kv.v(r)
        for p in _sampled_rows(prompt, f"{name} {r}", n_random):
            t = r * prompt + p
            ref.append(oa.causal_attention_request(q[t:t + 1], k, v, p, scale)[0])
            got.append(out[t])
    got, ref = torch.stack(got), torch.stack(ref)
    d = got - ref
    assert d.abs().max().item() <= BF16_MAX_ABS, d.abs().max().item()
    assert (torch.linalg.norm(d) / torch.linalg.norm(ref)).item() <= BF16_REL


def test_eight_prompts_of_2048_tokens_in_one_call():
    _check_prompts("prefill8x2048", 8, 2048, 10)


def test_one_prompt_of_16384_tokens():
    _check_prompts("prefill16384", 1, 16384, 40)
