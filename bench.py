"""Benchmark of the paged-attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the hot path over one batch that is already resident
in HBM: reshape_and_cache of the step's new tokens, then paged attention over
the whole batch, made as one call (reshape_and_cache_paged_attention), which
for this decode-only batch is one kernel; the same steps as two calls are
reported beside it (`step_forms`).  The headline workload is the Llama-3-8B decode batch (64
requests, one query each, contexts uniform on [128, 4096], 32/8/128 heads,
block_size 16, blocks drawn from a 65536-block pool).  It is reported as
algorithmic HBM bytes per second:

    bytes/step = sum(ctx) * 2 * Hkv * D * 2          (K and V history read once)
               + 2 * T * H * D * 2                   (q read, out written)
               + 4 * sum(ceil(ctx / 16))             (block_table entries)
               + T * (2 * Hkv * D * 2) * 2 + 8 * T   (reshape_and_cache read+write, slots)

Consecutive timed steps rotate over four copies of the batch placed on
disjoint blocks of the pool, so no step reads data the previous step left in
L2 (0.55 GB per step against a 129 MB L2).

The JSON line also carries the mixed chunked-prefill step (one 512-token
chunk at [1536, 2048) plus 256 decodes) as tokens/s/layer, the decode
kernel's roofline (CUDA events on its stream over the timed region), an
end-to-end figure through the public API from pinned host buffers, GPU clocks
sampled during the timed region, and the CPU oracle on a bounded sample.

With --gpus N > 1 (under torch.distributed.run) every rank runs an
independent replica on its own GPU - the path has no cross-GPU exchange - and
rank 0 prints the aggregate over ranks with the max time over ranks.
"""

from __future__ import annotations

import argparse
import functools
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn decode HBM GB/s (% of peak); mixed-batch attention tokens/s/layer"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
CHUNK_COPIES = 20


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        busy = [s for s in sm if s >= 0.5 * max(sm)]
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def source_sha(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_cache_36_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profile(kernel: str, sources, units: float):
    """dram bytes per launch from the committed ncu summary, scaled to `units`,
    or None when the kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f).get(kernel)
    if not t or t.get("source_sha") != source_sha(sources):
        return None
    return t["dram_bytes_per_unit"] * units


# ---------------------------------------------------------------------------
# workloads on the device
# ---------------------------------------------------------------------------
class DeviceStep:
    """One batch resident on the device, runnable as a step of the hot path."""

    def __init__(self, pkv, kc, vc, q, k_new, v_new, blocks, qlens, ncs, num_heads, device):
        self.pkv = pkv
        self.kc, self.vc = kc, vc
        self.R = len(qlens)
        self.H = num_heads
        self.D = kc.shape[3]
        qlens = np.asarray(qlens, np.int64)
        ncs = np.asarray(ncs, np.int64)
        self.qlens, self.ncs, self.seq = qlens, ncs, ncs + qlens
        width = max(len(b) for b in blocks)
        bt = np.full((self.R, width), -1, np.int32)
        for r, b in enumerate(blocks):
            bt[r, :len(b)] = b
        self.bt_host = bt
        self.qsl_host = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
        self.seq_host = self.seq.astype(np.int32)
        self.nc_host = ncs.astype(np.int32)
        self.slots_host = pkv.build_slot_mapping(bt, self.qsl_host, self.nc_host, 16)
        self.q = q.to(device)
        self.k_new, self.v_new = k_new.to(device), v_new.to(device)
        self.block_table = torch.from_numpy(bt).to(device)
        self.qsl = torch.from_numpy(self.qsl_host).to(device)
        self.seq_lens = torch.from_numpy(self.seq_host).to(device)
        self.nc = torch.from_numpy(self.nc_host).to(device)
        self.slots = torch.from_numpy(self.slots_host).to(device)
        self.out = torch.empty_like(self.q)
        self.ws = pkv.new_workspace(self.R, self.H, self.D, device)
        self.fuse = False
        self.max_q = int(qlens.max())
        self.scale = 1.0 / math.sqrt(self.D)
        self.T = int(qlens.sum())
        hkv = kc.shape[2]
        kv_tok = 2 * hkv * self.D * 2
        self.attn_bytes = int(self.seq.sum()) * kv_tok + 2 * self.T * self.H * self.D * 2 + \
            4 * int(((self.seq + 15) // 16).sum())
        self.k1_bytes = self.T * kv_tok * 2 + 8 * self.T
        self.decode_rows = qlens == 1
        self.decode_bytes = int(self.seq[self.decode_rows].sum()) * kv_tok + \
            2 * int(self.decode_rows.sum()) * self.H * self.D * 2 + \
            4 * int(((self.seq[self.decode_rows] + 15) // 16).sum())
        # causal prefill flops of the rows with query length > 1
        fl = 0
        for r in np.nonzero(~self.decode_rows)[0]:
            for_p = np.arange(ncs[r], ncs[r] + qlens[r], dtype=np.float64) + 1.0
            fl += 4.0 * self.D * self.H * float(for_p.sum())
        self.prefill_flops = fl

    def k1(self):
        self.pkv.reshape_and_cache(self.k_new, self.v_new, self.kc, self.vc, self.slots)

    def attn(self):
        self.pkv.paged_attention_varlen(self.q, self.kc, self.vc, self.block_table, self.qsl,
                                        self.seq_lens, self.nc, self.scale, out=self.out,
                                        workspace=self.ws, max_query_len=self.max_q)

    def fused(self):
        """reshape_and_cache + attention in one call (one kernel for a decode-only step)."""
        self.pkv.reshape_and_cache_paged_attention(
            self.k_new, self.v_new, self.slots, self.q, self.kc, self.vc, self.block_table,
            self.qsl, self.seq_lens, self.nc, self.scale, out=self.out, workspace=self.ws,
            max_query_len=self.max_q)

    def step(self):
        if self.fuse:
            self.fused()
        else:
            self.k1()
            self.attn()


def build_decode_steps(pkv, device, replicas=4):
    """The Llama-3-8B decode batch on `replicas` disjoint placements of the pool."""
    from workloads import configs
    from workloads.generators import random_block_placement
    cfg = configs.decode_batch_llama8b()
    counts = [len(b) for b in cfg.blocks]
    all_blocks = random_block_placement(cfg.num_blocks, counts * replicas, cfg.name, "bench")
    shape = (cfg.num_blocks, 16, cfg.num_kv_heads, cfg.head_dim)
    kc = torch.empty(shape, dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    kf, vf = kc.view(-1, cfg.num_kv_heads, cfg.head_dim), vc.view(-1, cfg.num_kv_heads, cfg.head_dim)
    steps = []
    R = len(cfg.context)
    for rep in range(replicas):
        blocks = all_blocks[rep * R:(rep + 1) * R]
        slots = []
        for r in range(R):
            b = blocks[r].astype(np.int64)
            p = np.arange(int(cfg.context[r]) - 1)
            slots.append(b[p // 16] * 16 + p % 16)
        s = torch.from_numpy(np.concatenate(slots)).to(device)
        hist_rows = np.concatenate([np.arange(int(cfg.kv.offsets[r]),
                                              int(cfg.kv.offsets[r] + cfg.context[r] - 1))
                                    for r in range(R)])
        hr = torch.from_numpy(hist_rows)
        kf[s] = cfg.kv.key[hr].to(device)
        vf[s] = cfg.kv.value[hr].to(device)
        last = torch.from_numpy((cfg.kv.offsets + cfg.context - 1).astype(np.int64))
        steps.append(DeviceStep(pkv, kc, vc, cfg.q, cfg.kv.key[last], cfg.kv.value[last], blocks,
                                np.ones(R, np.int64), cfg.context - 1, cfg.num_heads, device))
    return cfg, steps


def build_mixed_step(pkv, device, with_prefill_alone=False, **mix):
    """The mixed chunked-prefill step (the 512-token chunk at [1536, 2048)
    beside 256 decodes by default, or the mix the
    keyword arguments of configs.mixed_chunked_step give) as one fused call,
    the same step's decodes alone and, on request, its prefill request
    alone."""
    from workloads import configs
    cfg = configs.mixed_chunked_step(**mix)
    shape = (cfg.num_blocks, 16, cfg.num_kv_heads, cfg.head_dim)
    kc = torch.empty(shape, dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    kf, vf = kc.view(-1, cfg.num_kv_heads, cfg.head_dim), vc.view(-1, cfg.num_kv_heads, cfg.head_dim)
    R = len(cfg.query_len)
    slots, rows, knew, vnew = [], [], [], []
    for r in range(R):
        b = cfg.blocks[r].astype(np.int64)
        p = np.arange(int(cfg.num_computed[r]))
        slots.append(b[p // 16] * 16 + p % 16)
        rows.append(np.arange(int(cfg.kv.offsets[r]), int(cfg.kv.offsets[r] + cfg.num_computed[r])))
        o = int(cfg.kv.offsets[r] + cfg.num_computed[r])
        knew.append(cfg.kv.key[o:o + int(cfg.query_len[r])])
        vnew.append(cfg.kv.value[o:o + int(cfg.query_len[r])])
    s = torch.from_numpy(np.concatenate(slots)).to(device)
    hr = torch.from_numpy(np.concatenate(rows))
    kf[s] = cfg.kv.key[hr].to(device)
    vf[s] = cfg.kv.value[hr].to(device)
    step = DeviceStep(pkv, kc, vc, cfg.q, torch.cat(knew), torch.cat(vnew), cfg.blocks,
                      cfg.query_len, cfg.num_computed, cfg.num_heads, device)
    # the same step without its prefill request (request 0): the 256 decodes alone
    q0 = int(cfg.query_len[0])
    decodes = DeviceStep(pkv, kc, vc, cfg.q[q0:], torch.cat(knew[1:]), torch.cat(vnew[1:]),
                         cfg.blocks[1:], cfg.query_len[1:], cfg.num_computed[1:], cfg.num_heads,
                         device)
    # each step is one call of the fused entry: the cache write and the
    # attention in one kernel
    step.fuse = decodes.fuse = True
    if not with_prefill_alone:
        return cfg, step, decodes
    prefill = DeviceStep(pkv, kc, vc, cfg.q[:q0], knew[0], vnew[0], cfg.blocks[:1],
                         cfg.query_len[:1], cfg.num_computed[:1], cfg.num_heads, device)
    prefill.fuse = True
    return cfg, step, decodes, prefill


def build_prefill_chunks(pkv, device, copies=CHUNK_COPIES, pool_blocks=4096, from_start=False):
    """The mixed step's 512-token prefill chunk at [1536, 2048) alone (or, with
    from_start, the whole 2048-token prompt as one prefill), in its own
    4096-block cache: `copies` placements of the request's 128 blocks on
    disjoint random blocks (8.4 MB of K/V each, 168 MB for 20 against a
    129 MB L2), so consecutive calls do not find the previous call's K/V in
    L2."""
    from workloads import configs
    from workloads.generators import random_block_placement
    cfg = configs.mixed_chunked_step()
    nc, ql = int(cfg.num_computed[0]), int(cfg.query_len[0])
    if from_start:
        nc, ql = 0, nc + ql
    n0 = (nc + ql + 15) // 16
    placements = random_block_placement(pool_blocks, [n0] * copies, cfg.name, "chunk copies")
    shape = (pool_blocks, 16, cfg.num_kv_heads, cfg.head_dim)
    kc = torch.empty(shape, dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    kf, vf = kc.view(-1, cfg.num_kv_heads, cfg.head_dim), vc.view(-1, cfg.num_kv_heads, cfg.head_dim)
    o = int(cfg.kv.offsets[0])
    # the history and the chunk's own new keys (as reshape_and_cache leaves them)
    hist_k = cfg.kv.key[o:o + nc + ql].to(device)
    hist_v = cfg.kv.value[o:o + nc + ql].to(device)
    p = np.arange(nc + ql)
    chunks = []
    for blk in placements:
        b = blk.astype(np.int64)
        s = torch.from_numpy(b[p // 16] * 16 + p % 16).to(device)
        kf[s] = hist_k
        vf[s] = hist_v
        q = cfg.q[:ql] if ql <= cfg.q.shape[0] else cfg.q[:1].expand(ql, -1, -1).contiguous()
        chunks.append(DeviceStep(pkv, kc, vc, q, cfg.kv.key[o + nc:o + nc + ql],
                                 cfg.kv.value[o + nc:o + nc + ql], [blk], np.array([ql]),
                                 np.array([nc]), cfg.num_heads, device))
    return chunks


@functools.lru_cache(maxsize=None)
def _cudart():
    import ctypes
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            lib = ctypes.CDLL(name)
        except OSError:
            continue
        lib.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_int, ctypes.c_void_p]
        lib.cudaMemcpyAsync.restype = ctypes.c_int
        return lib
    return None


def host_mapped(t) -> bool:
    """True when the CUDA runtime reports t's storage as host memory that the
    device addresses at the same pointer (pinned memory under unified
    addressing), so a kernel may store to it."""
    import ctypes

    class Attr(ctypes.Structure):
        # cudaPointerAttributes: type, device, devicePointer, hostPointer and
        # long reserved[8], with spare room past it
        _fields_ = [("type", ctypes.c_int), ("device", ctypes.c_int),
                    ("devicePointer", ctypes.c_void_p), ("hostPointer", ctypes.c_void_p),
                    ("reserved", ctypes.c_long * 8), ("spare", ctypes.c_char * 256)]

    rt = _cudart()
    if rt is None:
        return False
    rt.cudaPointerGetAttributes.argtypes = [ctypes.POINTER(Attr), ctypes.c_void_p]
    rt.cudaPointerGetAttributes.restype = ctypes.c_int
    a = Attr()
    if rt.cudaPointerGetAttributes(ctypes.byref(a), ctypes.c_void_p(t.data_ptr())) != 0:
        return False
    return a.type == 1 and a.devicePointer == t.data_ptr()  # cudaMemoryTypeHost


def cuda_copy_async():
    """copy(dst, src, nbytes, stream) of two tensors, one of them pinned host
    memory: cudaMemcpyAsync through the CUDA runtime (cudaMemcpyDefault
    infers the direction), or torch's copy_ if the runtime cannot be
    loaded."""
    rt = _cudart()
    if rt is None:
        def copy(dst, src, nbytes, stream):
            dst.view(torch.uint8).view(-1)[:nbytes].copy_(
                src.view(torch.uint8).view(-1)[:nbytes], non_blocking=True)
        return copy

    def copy(dst, src, nbytes, stream):
        rc = rt.cudaMemcpyAsync(dst.data_ptr(), src.data_ptr(), nbytes, 4, stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(f"cudaMemcpyAsync failed: {rc}")
    return copy


def graph_time(calls, reps=5):
    """Captures calls (a list of callables) in one CUDA graph and returns the
    median over `reps` replays of the replay time per call, in ms: GPU time
    without the host's per-call launch work."""
    cur = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(cur)
    with torch.cuda.stream(side):
        for c in calls[:3]:
            c()
    cur.wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in calls:
            c()
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        g.replay()
        b.record(cur)
        b.synchronize()
        times.append(a.elapsed_time(b) / len(calls))
    del g
    return statistics.median(times)


def _rounded(obj):
    """Floats to 6 significant digits, so that the headline line stays short."""
    if isinstance(obj, float):
        return float(f"{obj:.6g}")
    if isinstance(obj, dict):
        return {k: _rounded(v) for k, v in obj.items()}
    if isinstance(obj, (list, tuple)):
        return [_rounded(v) for v in obj]
    return obj


def combine_ranks(ms: float, units: float, dist=None, device="cpu") -> tuple[float, float]:
    """Whole-job figures of a replicas run: the slowest rank's time and the
    units (bytes or tokens) all ranks processed.  Every rank runs its own
    replica, so this is the only exchange; without a process group the
    rank's own figures come back unchanged."""
    if dist is None:
        return ms, units
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def event_time(fn, n, stream):
    """Mean device time of fn over n calls, between two events (ms)."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        fn()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / n


def build_long_decode(pkv, device, pool=1 << 20):
    """The long-context decode call: 8 decodes over 131072-token histories,
    Llama-3-70B heads (64/8/128), blocks scattered over a pool of `pool`
    blocks (2^20 = 68.7 GB by default); only the used blocks are filled.
    Returns the caches, the step and the generator that filled them (later
    measurements draw from it)."""
    from workloads import configs
    cfg = configs.long_decode_llama70b(pool=pool)
    H, Hkv, D = cfg.num_heads, cfg.num_kv_heads, cfg.head_dim
    nb = cfg.num_blocks
    kc = torch.empty((nb, 16, Hkv, D), dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    used = torch.from_numpy(np.concatenate(cfg.blocks).astype(np.int64)).to(device)
    g = torch.Generator(device=device)
    g.manual_seed(127)
    for c in (kc, vc):
        for part in used.split(8192):
            c[part] = torch.randn((part.numel(), 16, Hkv, D), generator=g, device=device,
                                  dtype=torch.float32).to(torch.bfloat16)
    R = len(cfg.context)
    q = torch.randn((R, H, D), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    step = DeviceStep(pkv, kc, vc, q.cpu(), q.cpu()[:, :Hkv], q.cpu()[:, :Hkv], cfg.blocks,
                      np.ones(R, np.int64), cfg.context - 1, H, device)
    return kc, vc, step, g


def extra_measurements(pkv, device, stream, hbm_peak, bf16_peak):
    """Supporting measurements beside the headline: the long-context decode
    (8 x 131072-token histories), the 300-step continuous-batching trace per step,
    reshape_and_cache at 8192 tokens with and without the fused RoPE of Q and
    K, and the prefill kernel on a 2048-token prompt, on 8 such prompts in one
    call and on one 16384-token prompt."""
    from workloads import configs, trace_spec, generate_arrivals
    from workloads.generators import random_block_placement
    res = {}
    # ---- long-context decode: 8 decodes over 131072-token histories, 2^20-block pool ----
    kc, vc, step, g = build_long_decode(pkv, device)
    for _ in range(3):
        step.attn()
    ms = event_time(step.attn, 20, stream)
    res["long_decode"] = {
        "workload": "Llama-3-70B heads (64/8/128): 8 decodes x 131072-token contexts, "
                    "2^20-block pool (68.7 GB), random placement",
        "ms_per_launch": ms, "gbs": step.decode_bytes / (ms * 1e-3) / 1e9,
        "frac_of_hbm_peak": step.decode_bytes / (ms * 1e-3) / 1e9 / hbm_peak,
        "algorithmic_bytes_per_launch": step.decode_bytes,
    }
    del kc, vc, step
    torch.cuda.empty_cache()
    # ---- reshape_and_cache at 8192 tokens (inputs rotate over 4 batches) ----
    T, Hkv, D = 8192, 8, 128
    nbk = 4 * T // 16 + 64
    kc = torch.empty((nbk, 16, Hkv, D), dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    blocks = random_block_placement(nbk, [T // 16] * 4, "bench", "k1 8192")
    batches = []
    for bi in range(4):
        b = blocks[bi].astype(np.int64)
        slots = torch.from_numpy((b[:, None] * 16 + np.arange(16)[None, :]).reshape(-1)).to(device)
        kn = torch.randn((T, Hkv, D), generator=g, device=device).to(torch.bfloat16)
        vn = torch.randn((T, Hkv, D), generator=g, device=device).to(torch.bfloat16)
        batches.append((kn, vn, slots))
    it = [0]
    def k1():
        kn, vn, slots = batches[it[0] % 4]
        it[0] += 1
        pkv.reshape_and_cache(kn, vn, kc, vc, slots)
    for _ in range(8):
        k1()
    ms_eager = event_time(k1, 40, stream)

    def k1_b(b):
        kn, vn, slots = batches[b]
        pkv.reshape_and_cache(kn, vn, kc, vc, slots)
    # graph-timed: an eager call's host work is close to the kernel's time
    ms = graph_time([functools.partial(k1_b, c % 4) for c in range(40)])
    k1_bytes = T * (2 * Hkv * D * 2) * 2 + 8 * T
    res["reshape_and_cache_8192"] = {
        "workload": "8192 new tokens, 8 KV heads x 128 dims bf16, whole 16-token blocks, "
                    "4 rotating batches (268 MB of inputs and targets)",
        "ms_per_launch": ms, "gbs": k1_bytes / (ms * 1e-3) / 1e9,
        "frac_of_hbm_peak": k1_bytes / (ms * 1e-3) / 1e9 / hbm_peak,
        "algorithmic_bytes_per_launch": k1_bytes,
        "ms_per_launch_eager": ms_eager,
        "timing": "CUDA graph of 40 launches over the 4 batches; eager: CUDA events around 40 "
                  "back-to-back binding calls",
        "traffic": traffic_from_profile("reshape_and_cache", ["reshape_and_cache.cu"], 1.0),
    }
    # ---- the same scatter fused with RoPE of Q (32 heads) and K ----
    from workloads.generators import rope_cos_sin_table
    H = 32
    max_pos = 131072
    table = rope_cos_sin_table(max_pos, D).to(device)
    starts = [0, 2048, 30000, 120000]  # four 2048-token chunks at different depths
    pos = torch.from_numpy(np.concatenate([np.arange(a, a + 2048) for a in starts])).to(device)
    qs = [torch.randn((T, H, D), generator=g, device=device).to(torch.bfloat16) for _ in range(4)]
    it = [0]
    def rope_k1():
        kn, vn, slots = batches[it[0] % 4]
        pkv.rope_reshape_and_cache(pos, qs[it[0] % 4], kn, vn, kc, vc, slots, table, D)
        it[0] += 1
    for _ in range(8):
        rope_k1()
    ms_rope_eager = event_time(rope_k1, 40, stream)

    def rope_b(b):
        kn, vn, slots = batches[b]
        pkv.rope_reshape_and_cache(pos, qs[b], kn, vn, kc, vc, slots, table, D)
    ms = graph_time([functools.partial(rope_b, c % 4) for c in range(40)])
    rope_bytes = T * (2 * H * D * 2 + 2 * (2 * Hkv * D * 2) + D * 4 + 16)
    # the same kernel at a decode step's size: 64 tokens (the staged form),
    # graph-timed since a call's host work outlasts the kernel
    def rope_64(b):
        kn, vn, slots = batches[b]
        pkv.rope_reshape_and_cache(pos[:64], qs[b][:64], kn[:64], vn[:64], kc, vc, slots[:64],
                                   table, D)
    ms64 = graph_time([functools.partial(rope_64, c % 4) for c in range(100)])
    res["rope_reshape_and_cache_8192"] = {
        "workload": "8192 new tokens of Llama-3-8B (32 query heads, 8 KV heads, head_dim 128, "
                    "bf16, NeoX pairing), positions in four 2048-token chunks, Q rotated in "
                    "place, rotated K and V scattered to whole 16-token blocks, 4 rotating "
                    "batches (800 MB of inputs and targets)",
        "ms_per_launch": ms, "gbs": rope_bytes / (ms * 1e-3) / 1e9,
        "frac_of_hbm_peak": rope_bytes / (ms * 1e-3) / 1e9 / hbm_peak,
        "algorithmic_bytes_per_launch": rope_bytes,
        "bytes_per_token": "Q read + write 16384, K and V read + cache write 8192, "
                           "table row 512, position + slot 16",
        "ms_per_launch_64_tokens": ms64,
        "timing_64_tokens": "CUDA graph of 100 launches over 4 batches (L2-warm inputs)",
        "ms_per_launch_eager": ms_rope_eager,
        "timing": "CUDA graph of 40 launches over the 4 batches; eager: CUDA events around 40 "
                  "back-to-back binding calls",
    }
    del kc, vc, batches, qs, table
    torch.cuda.empty_cache()
    # ---- the prefill kernel on a 2048-token prompt from an empty cache ----
    prompts = build_prefill_chunks(pkv, device, from_start=True)
    ms = graph_time([c.attn for c in prompts] * 5)
    fl = prompts[0].prefill_flops
    res["prefill_2048"] = {
        "workload": "one 2048-token prompt from an empty cache, Llama-3-8B heads, "
                    "20 rotating placements (graph-timed)",
        "ms_per_call": ms, "tflops": fl / (ms * 1e-3) / 1e12,
        "frac_of_bf16_peak": fl / (ms * 1e-3) / 1e12 / bf16_peak, "flops": fl,
    }
    del prompts
    torch.cuda.empty_cache()
    # ---- the prefill kernel where its start and end are amortised: many
    # tiles per CTA (8 prompts of 2048 tokens in one call) and one long
    # prompt (16384 tokens, causal tiles of 1 to 128 key tiles) ----
    for key, nreq, plen in (("prefill_8x2048", 8, 2048), ("prefill_16384", 1, 16384)):
        copies = 4
        nblk = plen // 16
        pool = nreq * nblk * copies
        places = random_block_placement(pool, [nblk] * (nreq * copies), "bench", key)
        kc = torch.randn((pool, 16, 8, 128), generator=g, device=device).to(torch.bfloat16)
        vc = torch.randn((pool, 16, 8, 128), generator=g, device=device).to(torch.bfloat16)
        calls = []
        for c in range(copies):
            q = torch.randn((nreq * plen, 32, 128), generator=g, device=device).to(torch.bfloat16)
            calls.append(DeviceStep(pkv, kc, vc, q, q[:0, :8], q[:0, :8],
                                    places[c * nreq:(c + 1) * nreq], np.full(nreq, plen),
                                    np.zeros(nreq, np.int64), 32, device))
        ms = graph_time([c.attn for c in calls] * 2)
        fl = calls[0].prefill_flops
        res[key] = {
            "workload": f"{nreq} prompt(s) of {plen} tokens from an empty cache in one call, "
                        f"Llama-3-8B heads, {copies} rotating placements "
                        f"({copies * nreq * plen * 4096 / 1e6:.0f} MB of K/V; graph-timed)",
            "ms_per_call": ms, "tflops": fl / (ms * 1e-3) / 1e12,
            "frac_of_bf16_peak": fl / (ms * 1e-3) / 1e12 / bf16_peak, "flops": fl,
            "error_word": pkv.read_error_word(calls[0].ws),
        }
        del calls, kc, vc, q
        torch.cuda.empty_cache()
    # ---- whole-block copies: copy-on-write within the pool, offload to and
    # reload from pinned host memory (the GPU drives the CPU-GPU link) ----
    nbp, n = 16384, 4096
    kc = torch.randn((nbp, 16, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    vc = torch.randn((nbp, 16, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    hk = torch.empty((n, 16, Hkv, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    blk = random_block_placement(nbp, [2 * n], "bench", "copy blocks")[0].astype(np.int32)
    cow = torch.from_numpy(np.stack([blk[:n], blk[n:]], axis=1)).to(device)
    out_p = torch.from_numpy(np.stack([blk[:n], np.arange(n, dtype=np.int32)], axis=1)).to(device)
    in_p = torch.from_numpy(np.stack([np.arange(n, dtype=np.int32), blk[n:]], axis=1)).to(device)
    copy_bytes = 2 * n * 16 * Hkv * D * 2   # K and V blocks moved
    res_copy = {"workload": "4096 scattered blocks of Llama-3-8B shape (K+V, 256 MiB moved), "
                            "from a 16384-block pool", "bytes_per_call": copy_bytes}
    for name, args in (("device_to_device", (kc, vc, kc, vc, cow)),
                       ("device_to_host", (kc, vc, hk, hv, out_p)),
                       ("host_to_device", (hk, hv, kc, vc, in_p))):
        for _ in range(3):
            pkv.copy_blocks(*args)
        ms = event_time(lambda: pkv.copy_blocks(*args), 10, stream)
        res_copy[name] = {"ms": ms, "gbs": copy_bytes / (ms * 1e-3) / 1e9}
    res_copy["device_to_device"]["frac_of_hbm_peak"] = \
        2 * copy_bytes / (res_copy["device_to_device"]["ms"] * 1e-3) / 1e9 / hbm_peak
    res_copy["device_to_device"]["traffic"] = traffic_from_profile("copy_blocks",
                                                                   ["copy_blocks.cu"], 1.0)
    # the link's own rate: the copy engines moving the same bytes contiguously
    dk, dv = kc[:n], vc[:n]
    link = {}
    for name, fn in (("device_to_host", lambda: (hk.copy_(dk, non_blocking=True),
                                                 hv.copy_(dv, non_blocking=True))),
                     ("host_to_device", lambda: (dk.copy_(hk, non_blocking=True),
                                                 dv.copy_(hv, non_blocking=True)))):
        for _ in range(3):
            fn()
        link[name] = copy_bytes / (event_time(fn, 10, stream) * 1e-3) / 1e9
        res_copy[name]["link_memcpy_gbs"] = link[name]
        res_copy[name]["frac_of_link"] = res_copy[name]["gbs"] / link[name]
    res["copy_blocks"] = res_copy
    del kc, vc, hk, hv
    torch.cuda.empty_cache()
    # ---- the base trace with swap preemption (block moves in the timed step) ----
    spec = trace_spec()
    H, Hkv, D, B = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    ncpu = 4096
    sched = pkv.Scheduler(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                          spec.max_model_len, B, spec.num_blocks, spec.max_model_len // B,
                          preemption_mode="swap", num_cpu_blocks=ncpu)
    kc = torch.zeros((spec.num_blocks, B, Hkv, D), dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    hk = torch.zeros((ncpu, B, Hkv, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    ws = pkv.new_workspace(spec.max_num_seqs, H, D, device)
    budget = spec.max_num_batched_tokens
    qp = torch.randn((budget, H, D), generator=g, device=device).to(torch.bfloat16)
    kp = torch.randn((budget, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    vp = torch.randn((budget, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    by_step = {}
    for a in generate_arrivals(spec):
        by_step.setdefault(a.step, []).append(a)
    toks_done, ms_total, moved_blocks, ms_moves = 0, 0.0, 0, 0.0
    for st in range(spec.steps):
        for a in by_step.get(st, []):
            sched.add_request(a.req_id, a.prompt_len, a.max_output)
        plan = sched.step()
        bt, qsl, seq, nc, slots = sched.metadata()
        T = int(qsl[-1])
        dev = [torch.from_numpy(x).to(device) for x in (bt, qsl, seq, nc, slots)]
        outp = torch.tensor(plan["swap_out_pairs"], dtype=torch.int32).reshape(-1, 2).to(device)
        inp = torch.tensor(plan["swap_in_pairs"], dtype=torch.int32).reshape(-1, 2).to(device)
        a_ev, m_ev, b_ev = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a_ev.record(stream)
        if outp.shape[0]:
            pkv.copy_blocks(kc, vc, hk, hv, outp)
        if inp.shape[0]:
            pkv.copy_blocks(hk, hv, kc, vc, inp)
        m_ev.record(stream)
        if T:
            pkv.reshape_and_cache(kp[:T], vp[:T], kc, vc, dev[4])
            pkv.paged_attention_varlen(qp[:T], kc, vc, dev[0], dev[1], dev[2], dev[3],
                                       1.0 / math.sqrt(D), workspace=ws,
                                       max_query_len=plan["max_query_len"])
        b_ev.record(stream)
        b_ev.synchronize()
        toks_done += T
        ms_total += a_ev.elapsed_time(b_ev)
        ms_moves += a_ev.elapsed_time(m_ev)
        moved_blocks += outp.shape[0] + inp.shape[0]
        sched.finish_step(True)
    cnt = sched.counters()
    block_bytes = 2 * B * Hkv * D * 2
    res["trace_swap"] = {
        "workload": "the 300-step trace above with swap preemption and a 4096-block pinned "
                    "host pool; swap-outs then swap-ins run with copy_blocks inside each "
                    "step's timed region",
        "tokens": toks_done, "tokens_per_s_per_layer": toks_done / (ms_total * 1e-3),
        "preemptions": int(cnt["preemptions"]), "recomputed_tokens": int(cnt["recomputed_tokens"]),
        "blocks_moved": int(moved_blocks), "ms_moving_blocks": ms_moves,
        "moved_gbs": moved_blocks * block_bytes / max(ms_moves * 1e-3, 1e-9) / 1e9,
    }
    # the swap round trip of one 4096-token request against the page's bound
    nreq = 256                                           # blocks of 16 tokens
    blk = torch.arange(nreq, dtype=torch.int32, device=device)
    pairs = torch.stack([blk, blk], 1).contiguous()
    for _ in range(3):
        pkv.copy_blocks(kc, vc, hk, hv, pairs)
        pkv.copy_blocks(hk, hv, kc, vc, pairs)
    rt = event_time(lambda: (pkv.copy_blocks(kc, vc, hk, hv, pairs),
                             pkv.copy_blocks(hk, hv, kc, vc, pairs)), 20, stream)
    one_way = event_time(lambda: pkv.copy_blocks(kc, vc, hk, hv, pairs), 20, stream)
    payload = nreq * block_bytes
    res["swap_roundtrip_4096_tokens"] = {
        "payload_bytes": payload, "measured_ms": rt,
        "bound_ms_from_one_way_bandwidth": 2 * payload / (payload / (one_way * 1e-3)) * 1e3,
        "note": "bound = 2 * payload / beta (page: Chunked Prefill 与 Preemption), beta = the "
                "measured one-way copy rate of the same blocks",
    }
    del kc, vc, hk, hv, ws, sched
    torch.cuda.empty_cache()
    # ---- the trace with shared system prompts (prefix sharing on) ----
    from workloads import generate_prefix_arrivals
    spec = trace_spec()
    H, Hkv, D, B = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    sched = pkv.Scheduler(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                          spec.max_model_len, B, spec.num_blocks, spec.max_model_len // B)
    kc = torch.zeros((spec.num_blocks, B, Hkv, D), dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    ws = pkv.new_workspace(spec.max_num_seqs, H, D, device)
    budget = spec.max_num_batched_tokens
    qp = torch.randn((budget, H, D), generator=g, device=device).to(torch.bfloat16)
    kp = torch.randn((budget, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    vp = torch.randn((budget, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    by_step = {}
    for a in generate_prefix_arrivals(spec):
        by_step.setdefault(a.step, []).append(a)
    toks_done, ms_total = 0, 0.0
    for st in range(spec.steps):
        for a in by_step.get(st, []):
            sched.add_request(a.req_id, a.prompt_len, a.max_output, a.namespace, a.tokens)
        plan = sched.step()
        bt, qsl, seq, nc, slots = sched.metadata()
        T = int(qsl[-1])
        if T:
            dev = [torch.from_numpy(x).to(device) for x in (bt, qsl, seq, nc, slots)]
            a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_ev.record(stream)
            pkv.reshape_and_cache(kp[:T], vp[:T], kc, vc, dev[4])
            pkv.paged_attention_varlen(qp[:T], kc, vc, dev[0], dev[1], dev[2], dev[3],
                                       1.0 / math.sqrt(D), workspace=ws,
                                       max_query_len=plan["max_query_len"])
            b_ev.record(stream)
            b_ev.synchronize()
            toks_done += T
            ms_total += a_ev.elapsed_time(b_ev)
        sched.finish_step(True)
    pst = sched.allocator.prefix_stats()
    res["prefix_trace"] = {
        "workload": "300-step trace, 75 % of prompts = one of 8 shared system prompts "
                    "(popularity 1/(k+1), median 1536 tokens, 2 namespaces) + a private part "
                    "(median 256), C++ scheduler with the prefix index, 16384-block pool",
        "tokens_computed": toks_done, "prefix_tokens_matched": int(pst["matched_tokens"]),
        "lookups": int(pst["lookups"]), "hits": int(pst["hits"]),
        "evictions": int(pst["evictions"]),
        "tokens_per_s_per_layer": toks_done / (ms_total * 1e-3),
        "prompt_tokens_served_per_s_per_layer": (toks_done + pst["matched_tokens"]) / (ms_total * 1e-3),
        "preemptions": int(sched.counters()["preemptions"]),
        "timing": "CUDA events around reshape_and_cache + paged_attention_varlen of each step",
    }
    del kc, vc, ws, sched
    torch.cuda.empty_cache()
    # ---- the 300-step trace, per step (C++ scheduler, device-random K/V/Q) ----
    spec = trace_spec()
    H, Hkv, D, B = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    sched = pkv.Scheduler(spec.max_num_seqs, spec.max_num_batched_tokens, spec.chunk_size,
                          spec.max_model_len, B, spec.num_blocks, spec.max_model_len // B)
    kc = torch.zeros((spec.num_blocks, B, Hkv, D), dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    ws = pkv.new_workspace(spec.max_num_seqs, H, D, device)
    budget = spec.max_num_batched_tokens
    qp = torch.randn((budget, H, D), generator=g, device=device).to(torch.bfloat16)
    kp = torch.randn((budget, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    vp = torch.randn((budget, Hkv, D), generator=g, device=device).to(torch.bfloat16)
    by_step = {}
    for a in generate_arrivals(spec):
        by_step.setdefault(a.step, []).append(a)
    per_step = []
    for st in range(spec.steps):
        for a in by_step.get(st, []):
            sched.add_request(a.req_id, a.prompt_len, a.max_output)
        plan = sched.step()
        bt, qsl, seq, nc, slots = sched.metadata()
        T = int(qsl[-1])
        if T:
            dev = [torch.from_numpy(x).to(device) for x in (bt, qsl, seq, nc, slots)]
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            pkv.reshape_and_cache(kp[:T], vp[:T], kc, vc, dev[4])
            pkv.paged_attention_varlen(qp[:T], kc, vc, dev[0], dev[1], dev[2], dev[3],
                                       1.0 / math.sqrt(D), workspace=ws,
                                       max_query_len=plan["max_query_len"])
            b.record(stream)
            b.synchronize()
            per_step.append((T, a.elapsed_time(b)))
        sched.finish_step(True)
    toks = np.array([t for t, _ in per_step], np.float64)
    mss = np.array([m for _, m in per_step], np.float64)
    rate = toks / (mss * 1e-3)
    hist, edges = np.histogram(rate, bins=10)
    res["trace"] = {
        "workload": "300-step continuous-batching trace (Poisson arrivals, log-normal prompts, "
                    "geometric outputs, budget 8192, chunk 512, 16384-block pool), C++ scheduler",
        "steps_with_tokens": len(per_step), "tokens": int(toks.sum()),
        "tokens_per_s_per_layer": float(toks.sum() / (mss.sum() * 1e-3)),
        "per_step_tokens_per_s": {"mean": float(rate.mean()), "p10": float(np.percentile(rate, 10)),
                                  "median": float(np.median(rate)),
                                  "p90": float(np.percentile(rate, 90))},
        "per_step_histogram": {"counts": hist.tolist(), "edges": [float(e) for e in edges]},
        "preemptions": int(sched.counters()["preemptions"]),
        "timing": "CUDA events around reshape_and_cache + paged_attention_varlen of each step",
    }
    del kc, vc, ws
    torch.cuda.empty_cache()
    # ---- the mixed batch as one kernel on two other mixes: the step against
    # its decodes alone and its prefill request alone (each one fused call
    # per step, eager, back to back) ----
    mixes = {
        "prefill_heavy": dict(num_decodes=64, chunk_start=0, chunk_end=2048, ctx_lo=128,
                              ctx_hi=4096, pool=65536),
        "small_chunk": dict(num_decodes=256, chunk_start=1920, chunk_end=2048),
    }
    res["mixed_batches"] = {}
    for name, mix in mixes.items():
        _, mstep, mdec, mpre = build_mixed_step(pkv, device, with_prefill_alone=True, **mix)
        times = {}
        for key, obj in (("mixed", mstep), ("decodes_alone", mdec), ("prefill_alone", mpre)):
            for _ in range(5):
                obj.step()
            tot, _ = time_loop([obj], 40, stream)
            times[key] = tot / 40
        res["mixed_batches"][name] = {
            "workload": f"{mix['chunk_end'] - mix['chunk_start']}-token chunk at "
                        f"[{mix['chunk_start']},{mix['chunk_end']}) + {mix['num_decodes']} decodes",
            "ms_per_step": times["mixed"], "decodes_alone_ms": times["decodes_alone"],
            "prefill_alone_ms": times["prefill_alone"],
            "sum_of_parts_ms": times["decodes_alone"] + times["prefill_alone"],
        }
        del mstep, mdec, mpre
        torch.cuda.empty_cache()
    return res


def time_loop(fn_list, steps, stream, per_call=None):
    """Runs fn_list[i % len] for `steps` iterations between two events; if
    per_call is given, also brackets the attention launch with events each
    step (the whole step when it is one fused call).
    Returns (total ms, [per-call ms])."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = []
    start.record(stream)
    for i in range(steps):
        s = fn_list[i % len(fn_list)]
        if per_call is None:
            s.step()
        else:
            if not s.fuse:
                s.k1()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if s.fuse:
                s.fused()
            else:
                s.attn()
            b.record(stream)
            marks.append((a, b))
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end), [a.elapsed_time(b) for a, b in marks]


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------
class OracleDecode:
    """The CPU oracle on the headline decode batch, one request at a time: the
    reshape_and_cache scatter of the request's new token and its float64
    attention over the whole history."""

    def __init__(self):
        from workloads import configs
        cfg = configs.decode_batch_llama8b()
        self.cfg = cfg
        self.R = len(cfg.context)
        hkv, d = cfg.num_kv_heads, cfg.head_dim
        self.kv_tok = 2 * hkv * d * 2
        self.kc = torch.zeros(8, 16, hkv, d, dtype=torch.bfloat16)   # scratch image for the scatter
        self.vc = torch.zeros_like(self.kc)
        self.next = 0

    def request_bytes(self, r):
        c = int(self.cfg.context[r])
        H, d = self.cfg.num_heads, self.cfg.head_dim
        return c * self.kv_tok + 2 * H * d * 2 + 4 * ((c + 15) // 16) + 2 * self.kv_tok + 8

    def run_request(self, r):
        from oracle import attention as oa
        from oracle import paging
        cfg = self.cfg
        c = int(cfg.context[r])
        row = [0] * ((c + 15) // 16)
        row[-1] = 7                                  # the last logical block maps to image block 7
        slot = paging.slot_mapping([row], [1], [c - 1], 16)
        paging.write_cache(self.kc, self.vc, cfg.kv.k(r)[-1:], cfg.kv.v(r)[-1:], slot)
        oa.paged_attention_varlen(cfg.q[r:r + 1], [(cfg.kv.k(r), cfg.kv.v(r))], [0, 1], [c],
                                  [c - 1], 1.0 / math.sqrt(cfg.head_dim))

    def sample(self, budget_s):
        """Requests in rotation until budget_s has passed (at least one).
        Returns (bytes, seconds, requests)."""
        t0 = time.perf_counter()
        nbytes, n = 0, 0
        while n == 0 or time.perf_counter() - t0 < budget_s:
            r = self.next
            self.next = (self.next + 1) % self.R
            self.run_request(r)
            nbytes += self.request_bytes(r)
            n += 1
        return nbytes, time.perf_counter() - t0, n


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on the host cores, each step a bounded
    sample (whole requests in rotation) sized so the run ends within minutes."""
    if rank != 0:
        return
    torch.set_num_threads(os.cpu_count() or 1)
    o = OracleDecode()
    per_step_budget = min(1.0, 150.0 / (args.steps + args.warmup))
    for _ in range(args.warmup):
        o.sample(per_step_budget)
    tot_b, tot_t, tot_n = 0, 0.0, 0
    for _ in range(args.steps):
        b, t, n = o.sample(per_step_budget)
        tot_b, tot_t, tot_n = tot_b + b, tot_t + t, tot_n + n
    value = tot_b / tot_t / 1e9
    line = {
        "metric": METRIC, "impl": "reference", "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "Llama-3-8B decode batch: 64 requests x 1 query, contexts U[128,4096] "
                               "(seed 127), 32 query / 8 KV heads, head_dim 128, block_size 16, "
                               "blocks from a 65536-block pool",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": torch.get_num_threads(),
                         "kind": "oracle",
                         "sample": f"{tot_n} requests of the batch in rotation over {args.steps} "
                                   f"steps ({tot_t:.1f} s): reshape_and_cache scatter of the new "
                                   f"token + float64 attention over the history"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="primary timed steps only (no e2e, secondary or CPU legs), for ncu")
    ap.add_argument("--profile-prefill", action="store_true",
                    help="only --steps calls of the 512-token chunk (rotating placements), for ncu")
    ap.add_argument("--profile-mixed", action="store_true",
                    help="only --steps mixed chunked-prefill steps, for ncu")
    ap.add_argument("--profile-rope", action="store_true",
                    help="only --steps calls of the fused RoPE + cache write at 8192 tokens, for ncu")
    ap.add_argument("--profile-k1", action="store_true",
                    help="only --steps reshape_and_cache calls of 8192 tokens (4 rotating "
                         "batches), for ncu")
    ap.add_argument("--profile-long-decode", action="store_true",
                    help="only --steps calls of the long-context decode (8 x 131072-token "
                         "contexts, Llama-3-70B heads) in a pool that just holds them "
                         "(66560 blocks, 4.4 GB), for ncu")
    ap.add_argument("--profile-copy", action="store_true",
                    help="only --steps copy_blocks calls of 4096 scattered block pairs within "
                         "a 16384-block pool, for ncu")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_36_gb300 as pkv

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    hbm_peak, bf16_peak, bf16_sust, peak_kind = peaks()
    stream = torch.cuda.current_stream()
    if args.profile_rope:
        from workloads.generators import random_block_placement, rope_cos_sin_table
        T, H, Hkv, D = 8192, 32, 8, 128
        g = torch.Generator(device=device)
        g.manual_seed(127)
        nbk = 4 * T // 16 + 64
        kc = torch.empty((nbk, 16, Hkv, D), dtype=torch.bfloat16, device=device)
        vc = torch.empty_like(kc)
        table = rope_cos_sin_table(131072, D).to(device)
        pos = torch.from_numpy(np.concatenate([np.arange(a, a + 2048)
                                               for a in (0, 2048, 30000, 120000)])).to(device)
        batches = []
        for b in random_block_placement(nbk, [T // 16] * 4, "bench", "k1 8192"):
            b = b.astype(np.int64)
            slots = torch.from_numpy((b[:, None] * 16 + np.arange(16)[None, :]).reshape(-1)).to(device)
            batches.append((torch.randn((T, H, D), generator=g, device=device).to(torch.bfloat16),
                            torch.randn((T, Hkv, D), generator=g, device=device).to(torch.bfloat16),
                            torch.randn((T, Hkv, D), generator=g, device=device).to(torch.bfloat16),
                            slots))
        err = torch.zeros(1, dtype=torch.int32, device=device)
        for i in range(args.warmup + args.steps):
            q, k, v, slots = batches[i % 4]
            pkv.rope_reshape_and_cache(pos, q, k, v, kc, vc, slots, table, D, error_word=err)
        torch.cuda.synchronize()
        print(json.dumps({"profile_rope_calls": args.warmup + args.steps,
                          "error_word": int(err.item())}))
        return

    if args.profile_k1 or args.profile_copy:
        from workloads.generators import random_block_placement
        Hkv, D = 8, 128
        g = torch.Generator(device=device)
        g.manual_seed(127)
        err = torch.zeros(1, dtype=torch.int32, device=device)
        if args.profile_k1:
            T = 8192
            nbk = 4 * T // 16 + 64
            kc = torch.empty((nbk, 16, Hkv, D), dtype=torch.bfloat16, device=device)
            vc = torch.empty_like(kc)
            calls = []
            for b in random_block_placement(nbk, [T // 16] * 4, "bench", "k1 8192"):
                b = b.astype(np.int64)
                slots = torch.from_numpy((b[:, None] * 16 + np.arange(16)[None, :])
                                         .reshape(-1)).to(device)
                calls.append((torch.randn((T, Hkv, D), generator=g, device=device)
                              .to(torch.bfloat16),
                              torch.randn((T, Hkv, D), generator=g, device=device)
                              .to(torch.bfloat16), kc, vc, slots))
            for i in range(args.warmup + args.steps):
                pkv.reshape_and_cache(*calls[i % 4], error_word=err)
        else:
            nbp, n = 16384, 4096
            kc = torch.randn((nbp, 16, Hkv, D), generator=g, device=device).to(torch.bfloat16)
            vc = torch.randn((nbp, 16, Hkv, D), generator=g, device=device).to(torch.bfloat16)
            blk = random_block_placement(nbp, [2 * n], "bench", "copy blocks")[0].astype(np.int32)
            pairs = torch.from_numpy(np.stack([blk[:n], blk[n:]], axis=1)).to(device)
            for _ in range(args.warmup + args.steps):
                pkv.copy_blocks(kc, vc, kc, vc, pairs, error_word=err)
        torch.cuda.synchronize()
        print(json.dumps({"profile_calls": args.warmup + args.steps, "error_word": int(err.item())}))
        return

    if args.profile_long_decode:
        _, _, step, _ = build_long_decode(pkv, device, pool=8 * 131072 // 16 + 1024)
        for _ in range(args.warmup + args.steps):
            step.attn()
        torch.cuda.synchronize()
        print(json.dumps({"profile_long_decode_calls": args.warmup + args.steps,
                          "algorithmic_bytes_per_launch": step.decode_bytes,
                          "error_word": pkv.read_error_word(step.ws)}))
        return

    if args.profile_mixed:
        _, mstep, _ = build_mixed_step(pkv, device)
        for _ in range(args.warmup + args.steps):
            mstep.step()
        torch.cuda.synchronize()
        print(json.dumps({"profile_mixed_steps": args.warmup + args.steps,
                          "error_word": pkv.read_error_word(mstep.ws)}))
        return

    if args.profile_prefill:
        chunks = build_prefill_chunks(pkv, device)
        for i in range(args.warmup + args.steps):
            chunks[i % len(chunks)].attn()
        torch.cuda.synchronize()
        print(json.dumps({"profile_prefill_calls": args.warmup + args.steps,
                          "error_word": pkv.read_error_word(chunks[0].ws)}))
        return

    cfg, steps = build_decode_steps(pkv, device)
    for s in steps:  # the cache write and the attention as one kernel
        s.fuse = True
    for i in range(args.warmup):
        steps[i % len(steps)].step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        total_ms, _ = time_loop(steps, args.steps, stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    step_bytes = steps[0].attn_bytes + steps[0].k1_bytes
    total_ms, job_bytes = combine_ranks(total_ms, float(step_bytes) * args.steps, dist, device)
    if dist:
        dist.barrier()
    ms_per_step = total_ms / args.steps
    value = job_bytes / (total_ms * 1e-3) / 1e9
    # One kernel per step, launched back to back on `stream`: the events
    # around the K launches give its average launch time.  Consecutive
    # launches overlap only in the next launch's metadata prologue (its
    # loads wait for the previous grid to complete).
    attn_avg_ms = total_ms / args.steps
    # the fused kernel's algorithmic bytes: the decode reads plus the cache write
    kernel_bytes = steps[0].decode_bytes + steps[0].k1_bytes
    decode_gbs = kernel_bytes / (attn_avg_ms * 1e-3) / 1e9
    traffic = traffic_from_profile("decode_splitkv", ["decode_splitkv.cu", "decode_core.cuh"], 1.0)
    # the same steps as two calls (reshape_and_cache, then attention), as one
    # call again, and as one call with events around each launch, for comparison
    forms = None
    if not args.profile:
        forms = {}
        for fuse, key in ((False, "two_calls_ms_per_step"), (True, "one_call_ms_per_step")):
            for s in steps:
                s.fuse = fuse
            for i in range(args.warmup):
                steps[i % len(steps)].step()
            n = max(100, min(args.steps, 2000))
            tot, _ = time_loop(steps, n, stream)
            forms[key] = tot / n
        # each launch bracketed by its own events, which also keeps the next
        # launch's prologue from overlapping it
        _, marks = time_loop(steps, n, stream, per_call=True)
        forms["one_call_isolated_ms"] = statistics.mean(marks)
        forms["timing"] = ("CUDA events around the whole loop (two_calls, one_call) or around "
                           "each call (one_call_isolated); same steps and placements")
        for s in steps:
            s.fuse = True

    if args.profile:
        args.no_secondary = args.no_cpu_baseline = True
    # ---- end to end through the public API, from pinned host buffers ----
    # The step's inputs (q, the new K/V rows, block table, query_start_loc,
    # seq_lens, num_computed and the slot mapping built on the host) sit in one
    # pinned staging buffer and go to the device in one copy.  Two staging
    # buffers (host and device) alternate: while the GPU runs step i, the host
    # builds step i + 1's slot mapping and the copy of step i + 1's inputs runs
    # on a second stream.  The output goes to pinned host memory: the kernel
    # stores it there itself over the host link when the device maps that
    # memory at its host address (GB300's Grace host), else one D2H copy
    # brings it back.
    s0 = steps[0]
    parts = [("q", s0.q.cpu()), ("k_new", s0.k_new.cpu()), ("v_new", s0.v_new.cpu()),
             ("bt", torch.from_numpy(s0.bt_host)), ("qsl", torch.from_numpy(s0.qsl_host)),
             ("seq", torch.from_numpy(s0.seq_host)), ("nc", torch.from_numpy(s0.nc_host)),
             ("slots", torch.empty(s0.T, dtype=torch.int64))]
    layout, total = {}, 0
    for name, t in parts:
        nbytes = t.numel() * t.element_size()
        layout[name] = (total, nbytes, t.dtype, tuple(t.shape))
        total += (nbytes + 255) // 256 * 256
    stage_hosts = [torch.empty(total, dtype=torch.uint8).pin_memory() for _ in range(2)]
    stage_devs = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(2)]
    stage_host, stage_dev = stage_hosts[0], stage_devs[0]

    def view(buf, name):
        off, nbytes, dtype, shape = layout[name]
        return buf[off:off + nbytes].view(dtype).view(shape)

    hosts = [{name: view(sh, name) for name, _ in parts} for sh in stage_hosts]
    devs = [{name: view(sd, name) for name, _ in parts} for sd in stage_devs]
    dev = devs[0]
    for host in hosts:
        for name, t in parts[:-1]:
            host[name].copy_(t)
    out_host = torch.empty_like(hosts[0]["q"]).pin_memory()
    out_direct = host_mapped(out_host)
    h2d = total
    d2h = out_host.numel() * out_host.element_size()
    slots_outs = [host["slots"].numpy() for host in hosts]
    copy_async = cuda_copy_async()
    e2e_stream = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]

    def stage_in(i):
        # step i's inputs: slot_mapping (a2) on the host, then one H2D copy
        # on the copy stream
        b = i & 1
        pkv.build_slot_mapping(s0.bt_host, s0.qsl_host, s0.nc_host, 16, out=slots_outs[b])
        copy_async(stage_devs[b], stage_hosts[b], total, copy_stream)
        h2d_done[b].record(copy_stream)

    # the call on each staging buffer, its arguments marshalled once (the
    # binding's prepared form; the library validates every call)
    calls = [pkv.prepare_reshape_and_cache_paged_attention(
        d["k_new"], d["v_new"], d["slots"], d["q"], s0.kc, s0.vc, d["bt"], d["qsl"], d["seq"],
        d["nc"], s0.scale, out=out_host if out_direct else s0.out, workspace=s0.ws,
        max_query_len=1, stream=e2e_stream)
        for d in devs]

    def e2e_step(i):
        # step i's call once its inputs have landed, then step i + 1's inputs
        # staged while the GPU runs it, then (unless the kernel wrote out to
        # host memory itself) the D2H of out, and a sync
        b = i & 1
        e2e_stream.wait_event(h2d_done[b])
        calls[b]()
        stage_in(i + 1)
        if not out_direct:
            copy_async(out_host, s0.out, d2h, e2e_stream)
        e2e_stream.synchronize()

    stage_in(0)
    for i in range(args.warmup):
        e2e_step(i)
    e2e_n = 3 if args.profile else max(50, min(args.steps, 1000))
    step_ends = [0.0] * (e2e_n + 1)
    # the collector runs before the timed steps and not during them (as
    # timeit does): a full pass over the interpreter's objects takes a few
    # hundred ms, which would land on whichever step triggered it
    gc.collect()
    gc.disable()
    try:
        t0 = step_ends[0] = time.perf_counter()
        for i in range(e2e_n):
            e2e_step(args.warmup + i)
            step_ends[i + 1] = time.perf_counter()
    finally:
        gc.enable()
    e2e_ms = (step_ends[-1] - t0) * 1e3 / e2e_n
    # each step's wall time, so that a stall of the host shows as one slow
    # step rather than as a slower mean
    walls = np.sort(np.diff(np.array(step_ends)) * 1e3)
    e2e_spread = {"median_ms": float(walls[len(walls) // 2]),
                  "p99_ms": float(walls[min(len(walls) - 1, int(len(walls) * 0.99))]),
                  "max_ms": float(walls[-1]), "steps": e2e_n}
    e2e_ms, e2e_bytes = combine_ranks(e2e_ms, float(step_bytes), dist, device)
    e2e_value = e2e_bytes / (e2e_ms * 1e-3) / 1e9
    # The same step with its device work (H2D, the call, D2H) captured once in
    # a CUDA graph and replayed each step after the host has written the
    # step's inputs into the pinned staging buffer: what is left of the
    # host's per-call launch work.
    e2e_graph = None
    if not args.profile:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            stage_dev.copy_(stage_host, non_blocking=True)
            pkv.reshape_and_cache_paged_attention(
                dev["k_new"], dev["v_new"], dev["slots"], dev["q"], s0.kc, s0.vc, dev["bt"],
                dev["qsl"], dev["seq"], dev["nc"], s0.scale, out=s0.out, workspace=s0.ws,
                max_query_len=1)
            out_host.copy_(s0.out, non_blocking=True)
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()

        def e2e_graph_step():
            pkv.build_slot_mapping(s0.bt_host, s0.qsl_host, s0.nc_host, 16, out=slots_outs[0])
            g.replay()
            cur.synchronize()

        for _ in range(args.warmup):
            e2e_graph_step()
        gc.collect()
        gc.disable()
        try:
            t0 = time.perf_counter()
            for _ in range(e2e_n):
                e2e_graph_step()
            gms = (time.perf_counter() - t0) * 1e3 / e2e_n
        finally:
            gc.enable()
        gms, gbytes = combine_ranks(gms, float(step_bytes), dist, device)
        e2e_graph = {"value": gbytes / (gms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": gms,
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                     "path": "host slot_mapping build into the pinned staging buffer -> replay "
                             "of a CUDA graph holding the H2D copy, "
                             "reshape_and_cache_paged_attention and the D2H copy -> stream sync"}
        del g

    # ---- secondary: the mixed chunked-prefill step ----
    secondary = None
    if not args.no_secondary:
        mcfg, mstep, mdec = build_mixed_step(pkv, device)
        chunks = build_prefill_chunks(pkv, device)
        for i in range(args.warmup):
            mstep.step()
            chunks[i % len(chunks)].attn()
        n2 = max(20, min(args.steps // 10, 300))
        tot, _ = time_loop([mstep], n2, stream)
        mixed_ms, mixed_tokens = combine_ranks(tot / n2, float(mstep.T), dist, device)
        # the step's 256 decodes alone (their cache write and attention), to
        # show what the prefill chunk adds to the step
        for _ in range(args.warmup):
            mdec.step()
        tot_d, _ = time_loop([mdec], n2, stream)
        decodes_only_ms = tot_d / n2
        # one call per placement: the chunk alone (a call with no decode row
        # puts every CTA of the varlen kernel in the prefill role), each a
        # programmatic dependent of the call before it
        chunk_ms = graph_time([c.attn for c in chunks] * 5)
        chunk_tflops = mstep.prefill_flops / (chunk_ms * 1e-3) / 1e12
        secondary = {
            "metric": "mixed-batch attention tokens/s/layer",
            "value": mixed_tokens / (mixed_ms * 1e-3), "unit": "tokens/s/layer",
            "ms_per_step": mixed_ms,
            "workload": "512-token prefill chunk at [1536,2048) + 256 decodes (ctx U[256,8192]), "
                        "Llama-3-8B heads, 131072-block pool",
            "prefill_chunk_ms": chunk_ms,
            "prefill_tflops": chunk_tflops,
            "prefill_roofline": {
                "kernel": "varlen_attention_kernel", "bound": "tensor", "achieved": chunk_tflops,
                "peak": bf16_peak, "unit": "TFLOP/s", "frac": chunk_tflops / bf16_peak,
                "peak_kind": peak_kind, "algorithmic_flops_per_launch": mstep.prefill_flops,
                "avg_launch_ms": chunk_ms,
                "timing": f"CUDA graph of {5 * CHUNK_COPIES} calls rotating over {CHUNK_COPIES} "
                          f"disjoint placements of the chunk in a 4096-block cache (168 MB of "
                          f"K/V > L2), back to back; per call: the varlen kernel, all CTAs prefill",
            },
            "decodes_only_ms_per_step": decodes_only_ms,
            "prefill_chunk_cost_in_step_ms": mixed_ms - decodes_only_ms,
            "decodes_only_gbs": (mdec.decode_bytes + mdec.k1_bytes) / (decodes_only_ms * 1e-3) / 1e9,
        }
        del mstep, mdec, chunks

    extra = None
    if not args.no_secondary:
        extra = extra_measurements(pkv, device, stream, hbm_peak, bf16_peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        torch.set_num_threads(os.cpu_count() or 1)
        o = OracleDecode()
        nbytes, dt, n = o.sample(12.0)
        cpu = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": torch.get_num_threads(),
               "kind": "oracle", "cpu_model": cpu_model(),
               "sample": f"{n} requests of the headline batch in rotation ({dt:.1f} s): "
                         f"reshape_and_cache scatter of the new token + float64 attention"}
        # the same oracle on one core, over a shorter sample
        torch.set_num_threads(1)
        nb1, dt1, n1 = o.sample(4.0)
        cpu["single_thread"] = {"value": nb1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                                "sample": f"{n1} requests ({dt1:.1f} s)"}
        torch.set_num_threads(os.cpu_count() or 1)

    if rank == 0:
        clk = clocks.summary()
        # Everything measured, in full, on a line of its own first; the
        # headline line comes last and stays short, so that a reader of the
        # end of the output sees all of it.
        details = {
            "bench_details": {
                "roofline_decode": {"timing": "CUDA events on the launching stream around the "
                                              "timed region's back-to-back launches (one per step)",
                                    "peak_kind": peak_kind},
                "e2e": {"path": "per step: reshape_and_cache_paged_attention once the step's "
                                "inputs have landed (one H2D copy of a pinned staging buffer "
                                "holding all of them, issued during the previous step on a copy "
                                "stream after the host built its slot_mapping; the call in the "
                                "binding's prepared form) -> the next step's "
                                "slot_mapping and H2D while this one runs -> out into pinned "
                                "host memory -> stream sync; K H2D copies in K timed steps; "
                                "Python's cyclic collector run before the timed steps and off "
                                "during them",
                        "out_to_host": ("stored by the kernel into device-mapped pinned host "
                                        "memory over the host link (no D2H copy)"
                                        if out_direct else "one D2H copy per step"),
                        "step_wall_times": e2e_spread, "graph": e2e_graph},
                "secondary": secondary,
                "extra": extra,
                "cpu_baseline": cpu,
                "step_forms": forms,
                "wall_s_timed": wall,
            }
        }
        print(json.dumps(details), flush=True)
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "pct_of_hbm_peak": 100.0 * value / world / hbm_peak,
            "config": {
                "workload": "Llama-3-8B decode: 64 reqs x 1 query, ctx U[128,4096], 32/8 heads, "
                            "D 128, block 16, 65536-block pool",
                "l2": "inputs > L2: 4 disjoint placements (0.55 GB each)",
                "parallelism": f"replicas x{world}",
            },
            "roofline": {"kernel": "decode_splitkv_kernel", "bound": "hbm",
                         "achieved": decode_gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": decode_gbs / hbm_peak,
                         "algorithmic_bytes_per_launch": kernel_bytes,
                         "avg_launch_ms": attn_avg_ms, "traffic": traffic},
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "cpu_baseline": None if cpu is None else {
                "value": cpu["value"], "unit": cpu["unit"], "cores": cpu["cores"],
                "kind": cpu["kind"], "sample": "headline batch in rotation, 12 s"},
            "gpu_launches": args.steps,
            "clocks": clk,
        }
        if secondary is not None:
            pr = secondary["prefill_roofline"]
            line["mixed_tokens_per_s_per_layer"] = {
                "value": secondary["value"], "ms_per_step": secondary["ms_per_step"],
                "workload": "512-token chunk + 256 decodes"}
            line["prefill_roofline"] = {
                "kernel": pr["kernel"], "bound": "tensor", "achieved": pr["achieved"],
                "peak": pr["peak"], "unit": "TFLOP/s", "frac": pr["frac"],
                "avg_launch_ms": pr["avg_launch_ms"]}
        print(json.dumps(_rounded(line)), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
