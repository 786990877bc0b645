"""ctypes declarations of libpkv.so (the C ABI in include/pkv.h).

Loading fails loudly: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpkv.so")

PKV_OK = 0
ERRORS = {
    -1: "PKV_E_INVALID", -2: "PKV_E_UNSUPPORTED", -3: "PKV_E_WORKSPACE", -4: "PKV_E_NO_BLOCKS",
    -5: "PKV_E_STATE", -6: "PKV_E_UNKNOWN_REQ", -7: "PKV_E_CUDA", -8: "PKV_E_CAPACITY",
}
PKV_F32, PKV_BF16 = 0, 1
ERR_BLOCK_ID, ERR_SLOT, ERR_METADATA, ERR_TIMEOUT, ERR_POSITION = 1, 2, 4, 8, 16

i32, i64, u32, u64, f32, f64 = C.c_int32, C.c_int64, C.c_uint32, C.c_uint64, C.c_float, C.c_double
vp, sz = C.c_void_p, C.c_size_t
P_i32, P_i64 = C.POINTER(i32), C.POINTER(i64)


class AllocStats(C.Structure):
    _fields_ = [(n, i64) for n in ("capacity", "free", "reserved", "committed", "num_requests",
                                   "tail_waste", "alloc_failures", "peak_used")]


class PrefixStats(C.Structure):
    _fields_ = [(n, i64) for n in ("lookups", "hits", "matched_tokens", "evictions", "cow_copies",
                                   "indexed", "shared", "cached")]


class SchedConfig(C.Structure):
    _fields_ = [("max_num_seqs", i32), ("max_num_batched_tokens", i32), ("chunk_size", i32),
                ("max_model_len", i32), ("block_size", i32), ("num_blocks", i32),
                ("max_blocks_per_req", i32), ("artificial_preempt_max", i32),
                ("artificial_preempt_prob", f64), ("artificial_seed", u64),
                ("preemption_mode", i32), ("num_cpu_blocks", i32)]


class StepInfo(C.Structure):
    _fields_ = [("num_reqs", i32), ("num_preempted", i32), ("num_admitted", i32),
                ("max_blocks", i32), ("num_tokens", i64), ("max_query_len", i32), ("pad_", i32)]


class RequestState(C.Structure):
    _fields_ = [("status", i32), ("prompt_len", i32), ("max_output", i32), ("outputs", i32),
                ("num_tokens", i64), ("num_computed", i64), ("preemptions", i32), ("pad_", i32)]


# name -> (restype, argtypes)
SIGNATURES = {
    "pkv_last_error": (C.c_char_p, []),
    "pkv_version": (C.c_int, []),
    "pkv_reshape_and_cache": (C.c_int, [vp, vp, i64, i64, vp, vp, vp, i64, i64, i32, i32, i32,
                                        i32, vp, vp]),
    "pkv_rope_reshape_and_cache": (C.c_int, [vp, vp, i64, i32, vp, i64, vp, vp, i64, vp, vp,
                                             vp, vp, i64, i32, i32, i64, i64, i32, i32, i32,
                                             i32, vp, vp]),
    "pkv_copy_blocks": (C.c_int, [vp, vp, vp, vp, vp, i32, i64, i64, i64, vp, vp]),
    "pkv_attention_workspace_bytes": (sz, [i32, i32, i32]),
    "pkv_paged_attention_varlen": (C.c_int, [vp, i64, vp, vp, vp, i32, vp, vp, vp, f32, vp, i64,
                                             i64, i32, i64, i32, i32, i32, i32, i32, i32, vp, sz,
                                             vp]),
    "pkv_reshape_and_cache_paged_attention": (C.c_int, [vp, i64, vp, i64, vp, vp, i64, vp, vp,
                                                        vp, i32, vp, vp, vp, f32, vp, i64, i64,
                                                        i32, i64, i32, i32, i32, i32, i32, i32,
                                                        vp, sz, vp]),
    "pkv_paged_attention_varlen_noalloc": (C.c_int, [vp, i64, vp, vp, vp, i32, vp, vp, vp, f32,
                                                     vp, i64, i64, i32, i64, i32, i32, i32, i32,
                                                     i32, i32, vp, vp]),
    "pkv_build_slot_mapping": (C.c_int, [vp, i32, vp, vp, i32, i32, vp, i64]),
    "pkv_alloc_create": (vp, [i32, i32, i32]),
    "pkv_alloc_destroy": (None, [vp]),
    "pkv_alloc_reserve": (C.c_int, [vp, i32, vp, vp]),
    "pkv_alloc_commit": (C.c_int, [vp]),
    "pkv_alloc_rollback": (C.c_int, [vp]),
    "pkv_alloc_free_request": (C.c_int, [vp, i32]),
    "pkv_alloc_get_stats": (C.c_int, [vp, C.POINTER(AllocStats)]),
    "pkv_alloc_table": (C.c_int, [vp, i32, vp, i32]),
    "pkv_alloc_held_tokens": (i64, [vp, i32]),
    "pkv_alloc_free_list": (C.c_int, [vp, vp, i32]),
    "pkv_alloc_check": (C.c_int, [vp]),
    "pkv_alloc_match_prefix": (C.c_int, [vp, i32, u64, vp, i32]),
    "pkv_alloc_peek_prefix": (C.c_int, [vp, u64, vp, i32, vp]),
    "pkv_alloc_fork": (C.c_int, [vp, i32, i32]),
    "pkv_alloc_pending_copies": (C.c_int, [vp, vp, i32]),
    "pkv_alloc_get_prefix_stats": (C.c_int, [vp, C.POINTER(PrefixStats)]),
    "pkv_alloc_ref_count": (C.c_int, [vp, i32]),
    "pkv_alloc_cached_list": (C.c_int, [vp, vp, i32]),
    "pkv_alloc_available": (i64, [vp]),
    "pkv_alloc_create_with_cpu_pool": (vp, [i32, i32, i32, i32]),
    "pkv_alloc_swap_out": (C.c_int, [vp, i32, vp, i32, vp]),
    "pkv_alloc_swap_in_status": (C.c_int, [vp, i32]),
    "pkv_alloc_swap_in": (C.c_int, [vp, i32, vp, i32]),
    "pkv_alloc_swapped_blocks": (C.c_int, [vp, i32, vp, i32, vp]),
    "pkv_alloc_cpu_free_list": (C.c_int, [vp, vp, i32]),
    "pkv_sched_create": (vp, [C.POINTER(SchedConfig)]),
    "pkv_sched_destroy": (None, [vp]),
    "pkv_sched_add_request": (C.c_int, [vp, i32, i32, i32]),
    "pkv_sched_add_request_tokens": (C.c_int, [vp, i32, i32, i32, u64, vp]),
    "pkv_sched_step": (C.c_int, [vp, C.POINTER(StepInfo)]),
    "pkv_sched_plan": (C.c_int, [vp, vp, vp, vp, i32]),
    "pkv_sched_preempted": (C.c_int, [vp, vp, i32]),
    "pkv_sched_admitted": (C.c_int, [vp, vp, i32]),
    "pkv_sched_swaps": (C.c_int, [vp, vp, i32, vp, vp, i32, vp]),
    "pkv_sched_swap_events": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, i32]),
    "pkv_sched_build_metadata": (C.c_int, [vp, vp, i32, vp, vp, vp, vp]),
    "pkv_sched_finish_step": (C.c_int, [vp, i32, vp, i32]),
    "pkv_sched_request": (C.c_int, [vp, i32, C.POINTER(RequestState)]),
    "pkv_sched_queues": (C.c_int, [vp, vp, vp, vp, vp, i32]),
    "pkv_sched_swapped_queue": (C.c_int, [vp, vp, vp, i32]),
    "pkv_sched_counters": (C.c_int, [vp, P_i64]),
    "pkv_sched_allocator": (vp, [vp]),
}


def load(path: str = LIB_PATH) -> C.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libpkv.so is not built ({path}); run "
                          "`python -m paged_kv_cache_36_gb300.build`")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib
