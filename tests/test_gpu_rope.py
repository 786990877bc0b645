"""GPU parity of the fused RoPE + reshape_and_cache against the oracle.

Tolerances, derived from the arithmetic (the kernel works in float32 on
exact float32 / bfloat16 inputs and an exact float32 table; u = 2^-24):
* every output element of a rotation pair (x, y) with angle (c, s) is
  x c - y s or y c + x s; one product rounded and one fused multiply-add give
  an error <= 2u (|x c| + |y s|) in float32, bounded here by
  2^-22 (|x c| + |y s|);
* a bfloat16 result adds its round-to-nearest-even step, <= 2^-8 of the
  magnitude, so the bound is 2^-8 |exact| + 2^-21 (|x c| + |y s|);
* pass-through dimensions, V, addressing and untouched slots are bit-exact.
"""


import numpy as np
import pytest
import torch

from oracle import rope
from tests.gpu_support import Batch, compare
from workloads.configs import KVHistory
from workloads.generators import (randn_fp32, random_block_placement, rope_cos_sin_table,
                                  uniform_int)

pytestmark = pytest.mark.gpu


def _pkv():
    import paged_kv_cache_36_gb300 as pkv
    return pkv


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _magnitude(x, positions, table, rd, is_neox):
    """|x_a c| + |x_b s| for both elements of every pair; 0 outside rotary_dim."""
    x = x.detach().to("cpu", torch.float64).numpy()
    tab = table.detach().to("cpu", torch.float64).numpy()[np.asarray(positions)]
    half = rd // 2
    c, s = np.abs(tab[:, None, :half]), np.abs(tab[:, None, half:rd])
    a, b = rope.pair_indices(rd, is_neox)
    m = np.zeros_like(x)
    m[..., a] = np.abs(x[..., a]) * c + np.abs(x[..., b]) * s
    m[..., b] = np.abs(x[..., b]) * c + np.abs(x[..., a]) * s
    return m


def _assert_rotated(got, exact, mag, dtype, what):
    """got (device or host tensor) against the float64 oracle under the bound."""
    g = got.detach().to("cpu", torch.float64).numpy()
    if dtype == torch.bfloat16:
        bound = np.where(mag > 0, 2.0 ** -8 * np.abs(exact) + 2.0 ** -21 * mag, 0.0)
    else:
        bound = np.where(mag > 0, 2.0 ** -22 * mag, 0.0)
    err = np.abs(g - exact)
    bad = err > bound
    assert not bad.any(), (what, int(bad.sum()), float(err[bad].max()), np.argwhere(bad)[:4])
    if dtype == torch.bfloat16 and exact.size:
        # almost every element is the correctly rounded value
        rne = torch.from_numpy(exact).to(torch.float32).to(torch.bfloat16).double().numpy()
        assert (g == rne).mean() > 0.995, (what, float((g == rne).mean()))


def _case(T, H, Hkv, D, rd, dtype, NB, B=16, max_pos=4096, name="rope", pad_every=17):
    q = randn_fp32((T, H, D), name, "q", dtype=dtype)
    k = randn_fp32((T, Hkv, D), name, "k", dtype=dtype)
    v = randn_fp32((T, Hkv, D), name, "v", dtype=dtype)
    pos = uniform_int(0, max_pos - 1, T, name, "pos")
    slots = random_block_placement(NB * B, [T], name, "slots")[0].astype(np.int64)
    if pad_every:
        slots[::pad_every] = -1
    table = rope_cos_sin_table(max_pos, rd)
    kc = randn_fp32((NB, B, Hkv, D), name, "kc", dtype=dtype)
    vc = randn_fp32((NB, B, Hkv, D), name, "vc", dtype=dtype)
    return q, k, v, pos, slots, table, kc, vc


def _run_and_check(T, H, Hkv, D, rd, dtype, is_neox, NB=64, name="rope", key_out_mode=None):
    pkv = _pkv()
    q, k, v, pos, slots, table, kc, vc = _case(T, H, Hkv, D, rd, dtype, NB, name=name)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    dkc, dvc = kc.cuda(), vc.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    key_out = None
    if key_out_mode == "inplace":
        key_out = dk
    elif key_out_mode == "separate":
        key_out = torch.zeros_like(dk)
    pkv.rope_reshape_and_cache(torch.from_numpy(pos).cuda(), dq, dk, dv, dkc, dvc,
                               torch.from_numpy(slots).cuda(), table.cuda(), rd,
                               is_neox=is_neox, key_out=key_out, error_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    # oracle
    kc64 = kc.double().numpy().copy()
    vc64 = vc.double().numpy().copy()
    q_rot, k_rot = rope.rope_reshape_and_cache(pos, q, k, v, kc64, vc64, slots, table, rd, is_neox)
    mq = _magnitude(q, pos, table, rd, is_neox)
    mk = _magnitude(k, pos, table, rd, is_neox)
    _assert_rotated(dq, q_rot, mq, dtype, "query")
    # the cache: rotated K rows at the addressed slots, everything else untouched
    mkc = np.zeros_like(kc64)
    B = kc.shape[1]
    for t, s in enumerate(slots):
        if s >= 0:
            mkc[s // B, s % B] = mk[t]
    _assert_rotated(dkc, kc64, mkc, dtype, "key_cache")
    assert torch.equal(_bits(dvc.cpu()), _bits(torch.from_numpy(vc64).to(dtype))), "value_cache"
    live = slots >= 0
    untouched = np.ones(kc.shape[0] * B, bool)
    untouched[slots[live]] = False
    kflat, vflat = dkc.cpu().view(-1, Hkv, D), dvc.cpu().view(-1, Hkv, D)
    idx = torch.from_numpy(np.nonzero(untouched)[0])
    assert torch.equal(_bits(kflat[idx]), _bits(kc.view(-1, Hkv, D)[idx]))
    assert torch.equal(_bits(vflat[idx]), _bits(vc.view(-1, Hkv, D)[idx]))
    # pass-through dimensions of Q are bit-exact
    assert torch.equal(_bits(dq.cpu()[..., rd:].contiguous()), _bits(q[..., rd:].contiguous()))
    if key_out is not None:
        _assert_rotated(key_out, k_rot, mk, dtype, "key_out")
        # key_out equals what went into the cache, bit for bit
        rows = torch.from_numpy(slots[live])
        assert torch.equal(_bits(key_out.cpu()[torch.from_numpy(np.nonzero(live)[0])]),
                           _bits(kflat[rows]))
    else:
        assert torch.equal(_bits(dk.cpu()), _bits(k)), "key must be left unchanged"


@pytest.mark.parametrize("T", [300, 1500])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("is_neox", [True, False])
@pytest.mark.parametrize("H,Hkv,D,rd", [(32, 8, 128, 128), (8, 2, 128, 64), (4, 1, 64, 64),
                                        (6, 2, 64, 32), (8, 2, 128, 48)])
def test_rope_reshape_and_cache_parity(T, dtype, is_neox, H, Hkv, D, rd):
    # 300 tokens take the staged form (one to a few tokens per CTA, a ragged
    # split), 1500 the one-warp-per-token form (a ragged last block of 8
    # warps); rotary_dim 48 (3 or 6 items per head) always takes the warp
    # form.  Every 17th token is a padding token.
    _run_and_check(T, H, Hkv, D, rd, dtype, is_neox, NB=(T + 15) // 16 + 48,
                   name=f"rope{T}_{H}_{D}_{rd}")


@pytest.mark.parametrize("is_neox", [True, False])
def test_rope_rows_too_large_for_the_ring(is_neox):
    """128 query heads of 256 dims (64 KiB of Q per token in bf16): three
    ring stages do not fit in shared memory, the warp form takes over."""
    _run_and_check(45, 128, 8, 256, 256, torch.bfloat16, is_neox, NB=8, name="ropebig")


def test_rope_many_tokens_per_cta():
    """160000 tokens of 8 + 2 heads (the one-warp-per-token form, each warp
    looping over many tokens).  V rows and untouched slots are checked bit
    for bit, Q and K of 2048 sampled tokens against the oracle."""
    T, H, Hkv, D, NB, B = 160000, 8, 2, 128, 10240, 16
    _large_case_check("ropemany", T, H, Hkv, D, NB, B,
                      uniform_int(0, 4095, T, "ropemany", "pos"), 4096,
                      random_block_placement(NB * B, [T], "ropemany", "slots")[0].astype(np.int64))


@pytest.mark.parametrize("mode", ["inplace", "separate"])
def test_rope_key_out(mode):
    _run_and_check(77, 16, 4, 128, 128, torch.bfloat16, True, name="rope_keyout", key_out_mode=mode)
    _run_and_check(1100, 16, 4, 128, 128, torch.bfloat16, True, NB=120, name="rope_keyout_w",
                   key_out_mode=mode)


def test_rope_one_token_and_empty():
    pkv = _pkv()
    _run_and_check(1, 32, 8, 128, 128, torch.bfloat16, True, name="rope_one")
    # zero tokens: nothing is launched, nothing is touched
    kc = torch.ones(4, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.ones_like(kc)
    e = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    eq = torch.empty(0, 32, 128, dtype=torch.bfloat16, device="cuda")
    none = torch.empty(0, dtype=torch.int64, device="cuda")
    pkv.rope_reshape_and_cache(none, eq, e, e, kc, vc, none,
                               rope_cos_sin_table(16, 128).cuda(), 128)
    torch.cuda.synchronize()
    assert bool((kc == 1).all()) and bool((vc == 1).all())


@pytest.mark.parametrize("T,NB", [(40, 8), (1200, 80)])
def test_rope_bad_position_and_slot(T, NB):
    """A position outside the table leaves its token untouched and flags
    PKV_ERR_POSITION; a slot past the pool is skipped and flags PKV_ERR_SLOT
    (the token's Q is still rotated).  Both forms (40 and 1200 tokens)."""
    pkv = _pkv()
    H, Hkv, D, B, max_pos = 8, 2, 128, 16, 64
    q = randn_fp32((T, H, D), "ropebad", "q", dtype=torch.bfloat16)
    k = randn_fp32((T, Hkv, D), "ropebad", "k", dtype=torch.bfloat16)
    v = randn_fp32((T, Hkv, D), "ropebad", "v", dtype=torch.bfloat16)
    pos = uniform_int(0, max_pos - 1, T, "ropebad", "pos")
    pos[3], pos[9] = max_pos, -1
    slots = np.arange(T, dtype=np.int64)
    slots[20] = NB * B + 5
    table = rope_cos_sin_table(max_pos, D)
    kc = torch.zeros(NB, B, Hkv, D, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    dq, dkc, dvc = q.cuda(), kc.cuda(), vc.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.rope_reshape_and_cache(torch.from_numpy(pos).cuda(), dq, k.cuda(), v.cuda(), dkc, dvc,
                               torch.from_numpy(slots).cuda(), table.cuda(), D, error_word=err)
    torch.cuda.synchronize()
    assert err.item() == pkv.ERR_POSITION | pkv.ERR_SLOT
    good = np.ones(T, bool)
    good[[3, 9]] = False
    # untouched tokens: Q unchanged, their slots unwritten
    assert torch.equal(_bits(dq.cpu()[3]), _bits(q[3])) and torch.equal(_bits(dq.cpu()[9]), _bits(q[9]))
    assert bool((dkc.cpu().view(-1, Hkv, D)[[3, 9]] == 0).all())
    # the rest as the oracle says, with slot 20 skipped
    ok = np.nonzero(good)[0]
    s_or = slots.copy()
    s_or[20] = -1
    kc64 = kc.double().numpy().copy()
    vc64 = vc.double().numpy().copy()
    q_rot, _ = rope.rope_reshape_and_cache(pos[ok], q[ok], k[ok], v[ok], kc64, vc64, s_or[ok],
                                           table, D, True)
    _assert_rotated(dq.cpu()[ok], q_rot, _magnitude(q[ok], pos[ok], table, D, True),
                    torch.bfloat16, "query")
    mk = _magnitude(k[ok], pos[ok], table, D, True)
    mkc = np.zeros_like(kc64)
    for i, t in enumerate(ok):
        s = s_or[t]
        if s >= 0:
            mkc[s // B, s % B] = mk[i]
    _assert_rotated(dkc, kc64, mkc, torch.bfloat16, "key_cache")
    assert torch.equal(_bits(dvc.cpu()), _bits(torch.from_numpy(vc64).to(torch.bfloat16)))


def _large_case_check(name, T, H, Hkv, D, NB, B, pos, max_pos, slots, sample_n=2048):
    pkv = _pkv()
    q = randn_fp32((T, H, D), name, "q", dtype=torch.bfloat16)
    k = randn_fp32((T, Hkv, D), name, "k", dtype=torch.bfloat16)
    v = randn_fp32((T, Hkv, D), name, "v", dtype=torch.bfloat16)
    table = rope_cos_sin_table(max_pos, D)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    dkc = torch.zeros(NB, B, Hkv, D, dtype=torch.bfloat16, device="cuda")
    dvc = torch.zeros_like(dkc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dslots = torch.from_numpy(slots).cuda()
    pkv.rope_reshape_and_cache(torch.from_numpy(pos).cuda(), dq, dk, dv, dkc, dvc, dslots,
                               table.cuda(), D, error_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    vflat, kflat = dvc.view(-1, Hkv, D), dkc.view(-1, Hkv, D)
    assert torch.equal(_bits(vflat[dslots]), _bits(dv))
    mask = torch.ones(NB * B, dtype=torch.bool, device="cuda")
    mask[dslots] = False
    assert not bool(_bits(kflat[mask]).any()) and not bool(_bits(vflat[mask]).any())
    assert torch.equal(_bits(dk), _bits(k.cuda())), "key must be left unchanged"
    sample = np.sort(np.random.default_rng(5).choice(T, sample_n, replace=False))
    q_rot = rope.apply_rope(q[sample], pos[sample], table, D, True)
    k_rot = rope.apply_rope(k[sample], pos[sample], table, D, True)
    _assert_rotated(dq.cpu()[sample], q_rot, _magnitude(q[sample], pos[sample], table, D, True),
                    torch.bfloat16, "query")
    _assert_rotated(kflat[dslots[torch.from_numpy(sample).cuda()]], k_rot,
                    _magnitude(k[sample], pos[sample], table, D, True), torch.bfloat16, "key")


def test_rope_full_size_llama8b_prefill_chunk():
    """8192 tokens of Llama-3-8B (32 query heads, 8 KV heads, head_dim 128,
    NeoX pairing, bf16) scattered over a 4096-block pool, positions in four
    2048-token chunks at depths up to 122047: every V row and every untouched
    slot checked bit for bit, Q and K of 1024 sampled tokens against the
    oracle."""
    T, NB, B = 8192, 4096, 16
    starts = [0, 2048, 30000, 120000]
    pos = np.concatenate([np.arange(s, s + 2048) for s in starts]).astype(np.int64)
    blocks = random_block_placement(NB, [128] * 4, "rope8192", "placement")
    slots = np.concatenate([b.astype(np.int64)[np.arange(2048) // B] * B + np.arange(2048) % B
                            for b in blocks])
    _large_case_check("rope8192", T, 32, 8, 128, NB, B, pos, 131072, slots, sample_n=1024)


# ---------------------------------------------------------------- followed by attention
ATTN_CASES = [
    # (H, Hkv, D, query lens, num computed)
    (32, 8, 128, [1] * 24, None),                 # decode only: the decode kernel follows directly
    (32, 8, 128, [1, 70, 1, 33, 1], [500, 0, 2000, 100, 40]),  # mixed: prefill then decode
    (16, 4, 64, [1, 1, 1], [10, 300, 1000]),
]


@pytest.mark.parametrize("case", range(len(ATTN_CASES)))
def test_rope_then_attention(case):
    """The fused op followed directly by paged_attention_varlen on the same
    stream: the attention kernels must see the rotated Q and K."""
    H, Hkv, D, qlens, ncs = ATTN_CASES[case]
    name = f"ropeattn{case}"
    if ncs is None:
        ncs = uniform_int(100, 3000, len(qlens), name, "nc").tolist()
    seq = [a + b for a, b in zip(qlens, ncs)]
    counts = [(s + 15) // 16 for s in seq]
    NB = 2 * sum(counts) + 8
    blocks = random_block_placement(NB, counts, name, "placement")
    lengths = np.array(seq, np.int64)
    offsets = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
    n = int(lengths.sum())
    # history rows (positions < num_computed) are taken as already rotated
    key = randn_fp32((n, Hkv, D), name, "k", dtype=torch.bfloat16)
    value = randn_fp32((n, Hkv, D), name, "v", dtype=torch.bfloat16)
    q = randn_fp32((sum(qlens), H, D), name, "q", dtype=torch.bfloat16)
    max_pos = max(seq) + 1
    table = rope_cos_sin_table(max_pos, D)
    positions = np.concatenate([np.arange(nc, nc + ql) for nc, ql in zip(ncs, qlens)]).astype(np.int64)
    # the oracle's view: rotated Q and new K, rounded to the cache type
    new_rows = np.concatenate([np.arange(o + nc, o + nc + ql) for o, nc, ql in zip(offsets, ncs, qlens)])
    k_new = key[torch.from_numpy(new_rows)]
    q_rot = torch.from_numpy(rope.apply_rope(q, positions, table, D, True)).to(torch.bfloat16)
    k_rot = torch.from_numpy(rope.apply_rope(k_new, positions, table, D, True)).to(torch.bfloat16)
    key_or = key.clone()
    key_or[torch.from_numpy(new_rows)] = k_rot
    b = Batch(KVHistory(key_or, value, lengths, offsets), blocks, NB, qlens, ncs, q_rot, H,
              torch.bfloat16).alloc_cache().fill_history().upload_metadata()
    # the device gets the unrotated Q and K
    dq = q.cuda()
    b.q = dq
    v_new = value[torch.from_numpy(new_rows)]
    pkv = _pkv()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.rope_reshape_and_cache(torch.from_numpy(positions).cuda(), dq, k_new.cuda(), v_new.cuda(),
                               b.key_cache, b.value_cache, b.slot_mapping, table.cuda(), D,
                               error_word=err)
    out = b.attention()
    assert err.item() == 0
    compare(out, b.oracle(), b.qsl_host, torch.bfloat16)
