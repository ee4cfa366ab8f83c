"""Thin ctypes binding of libpkv (include/pkv.h): argument marshalling only, same names as the C ABI.

Every step of the path runs in the library's CUDA kernels.  If ``libpkv.so`` is missing this module raises;
there is no fallback of any kind.  Tensors are passed as torch tensors (their ``data_ptr()``) or raw ints.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_OUT_OF_RANGE = 2
PKV_ERR_UNSUPPORTED = 3
PKV_ERR_CUDA = 4
PKV_ERR_NO_BLOCKS = 5
PKV_ERR_NOT_FOUND = 6

PKV_DEVERR_SLOT_RANGE = 0x1
PKV_DEVERR_BLOCK_RANGE = 0x2
PKV_DEVERR_ROW_META = 0x4
PKV_DEVERR_QSL = 0x8
PKV_DEVERR_WAIT_TIMEOUT = 0x10

PKV_ALLOC_ON_DEMAND = 0
PKV_ALLOC_RESERVE = 1
PKV_UNIT_PASS = 0
PKV_UNIT_REQUEST = 1

PKV_KV_F16 = 0
PKV_KV_E4M3 = 1

DEFAULT_SPLIT_BLOCKS = 32  # pkv_config.split_blocks = 0 selects this many blocks per split-K partition

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


class pkv_config(ctypes.Structure):
    _fields_ = [("num_layers", _i32), ("num_q_heads", _i32), ("num_kv_heads", _i32), ("head_dim", _i32),
                ("block_size", _i32), ("num_blocks", _i32), ("split_blocks", _i32), ("kv_dtype", _i32)]


class pkv_sched_config(ctypes.Structure):
    _fields_ = [("max_num_seqs", _i32), ("token_budget", _i32), ("block_size", _i32), ("num_blocks", _i32)]


class pkv_step(ctypes.Structure):
    _fields_ = [("num_seqs", _i32), ("num_tokens", _i32), ("max_blocks_per_seq", _i32),
                ("req_ids", ctypes.POINTER(_i64)), ("q_lens", ctypes.POINTER(_i32)),
                ("context_lens", ctypes.POINTER(_i32)), ("query_start_loc", ctypes.POINTER(_i32)),
                ("block_tables", ctypes.POINTER(_i32)), ("slot_mapping", ctypes.POINTER(_i64)),
                ("num_preempted", _i32), ("preempted", ctypes.POINTER(_i64)),
                ("num_admitted", _i32), ("admitted", ctypes.POINTER(_i64)),
                ("num_finished", _i32), ("finished", ctypes.POINTER(_i64))]


class pkv_sched_stats(ctypes.Structure):
    _fields_ = [("steps", _i64), ("preemptions", _i64), ("recomputed_tokens", _i64),
                ("recomputed_prompt_tokens", _i64), ("max_batch", _i64), ("batch_sum", _i64),
                ("tokens_scheduled", _i64), ("running", _i32), ("waiting", _i32), ("free_blocks", _i32),
                ("live_tokens", _i64), ("held_slots", _i64), ("prefix_hit_tokens", _i64)]


# name -> (restype, argtypes); the list every exported symbol of include/pkv.h
SIGNATURES = {
    "pkv_pool_bytes": (_sz, [ctypes.POINTER(pkv_config)]),
    "pkv_pool_init": (ctypes.c_int, [ctypes.POINTER(pkv_config), _p, _sz, ctypes.POINTER(_p)]),
    "pkv_pool_destroy": (None, [_p]),
    "pkv_pool_layer_ptr": (_p, [_p, _i32, _i32]),
    "pkv_pool_scales_ptr": (_p, [_p, _i32]),
    "pkv_pool_check": (ctypes.c_int, [_p, ctypes.POINTER(_i32), _i32]),
    "pkv_slot_mapping": (ctypes.c_int, [_p, _p, _i32, _p, _p, _i32, _i32, _p, _p]),
    "pkv_append": (ctypes.c_int, [_p, _i32, _p, _p, _p, _i32, _p]),
    "pkv_attention_workspace_bytes": (_sz, [_p, _i32, _i32, _i32]),
    "pkv_attention_plan": (ctypes.c_int, [_p, _p, _p, _i32, _i32, _i32, _p, _sz, _p]),
    "pkv_attention": (ctypes.c_int, [_p, _i32, _p, _p, _i32, _p, _p, _i32, _i32, _p, _p, _sz, _p]),
    "pkv_attention_noalloc": (ctypes.c_int, [_p, _i32, _p, _p, _i32, _p, _p, _i32, _i32, _p, _p]),
    "pkv_attention_append": (ctypes.c_int, [_p, _i32, _p, _p, _p, _p, _p, _i32, _p, _p, _i32, _i32, _p, _p, _sz,
                                            _p]),
    "pkv_debug_expire_wait": (ctypes.c_int, [_p, _i64, _p]),
    "pkv_last_launch_count": (_i32, [_p]),
    "pkv_last_error": (ctypes.c_char_p, []),
    "pkv_sched_create": (ctypes.c_int, [ctypes.POINTER(pkv_sched_config), _p, ctypes.POINTER(_p)]),
    "pkv_sched_destroy": (None, [_p]),
    "pkv_sched_add": (ctypes.c_int, [_p, _i64, _i32, _i32]),
    "pkv_sched_add_declared": (ctypes.c_int, [_p, _i64, _i32, _i32, _i32]),
    "pkv_sched_set_policy": (ctypes.c_int, [_p, _i32, _i32]),
    "pkv_sched_set_prefix_caching": (ctypes.c_int, [_p, _i32]),
    "pkv_sched_step": (ctypes.c_int, [_p, ctypes.POINTER(pkv_step)]),
    "pkv_sched_abort": (ctypes.c_int, [_p, _i64]),
    "pkv_sched_set_max_num_seqs": (ctypes.c_int, [_p, _i32]),
    "pkv_sched_get_stats": (None, [_p, ctypes.POINTER(pkv_sched_stats)]),
    "pkv_sched_done": (_i32, [_p]),
    "pkv_sched_free_list": (_i32, [_p, ctypes.POINTER(_i32), _i32]),
}

_lib = None


class PkvError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


def load():
    """Load libpkv.so (built by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status: int, fn: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, fn, load().pkv_last_error().decode())


# ---- C-ABI mirrors (same names) ---------------------------------------------------------------------

def pkv_pool_bytes(cfg: pkv_config) -> int:
    return load().pkv_pool_bytes(ctypes.byref(cfg))


def pkv_pool_init(cfg: pkv_config, dev_cache, nbytes: int) -> int:
    h = _p()
    _check(load().pkv_pool_init(ctypes.byref(cfg), _ptr(dev_cache), nbytes, ctypes.byref(h)), "pkv_pool_init")
    return h.value


def pkv_pool_destroy(pool: int) -> None:
    load().pkv_pool_destroy(pool)


def pkv_pool_layer_ptr(pool: int, layer: int, kv: int) -> int:
    return load().pkv_pool_layer_ptr(pool, layer, kv) or 0


def pkv_pool_scales_ptr(pool: int, layer: int) -> int:
    return load().pkv_pool_scales_ptr(pool, layer) or 0


def pkv_pool_check(pool: int, clear: bool = True) -> int:
    bits = _i32(0)
    _check(load().pkv_pool_check(pool, ctypes.byref(bits), 1 if clear else 0), "pkv_pool_check")
    return bits.value


def pkv_slot_mapping(pool: int, block_tables, max_blocks_per_seq: int, context_lens, query_start_loc,
                     num_seqs: int, num_tokens: int, slot_mapping, stream=None) -> None:
    _check(load().pkv_slot_mapping(pool, _ptr(block_tables), max_blocks_per_seq, _ptr(context_lens),
                                   _ptr(query_start_loc), num_seqs, num_tokens, _ptr(slot_mapping),
                                   _stream(stream)), "pkv_slot_mapping")


def pkv_append(pool: int, layer: int, k, v, slot_mapping, num_tokens: int, stream=None) -> None:
    _check(load().pkv_append(pool, layer, _ptr(k), _ptr(v), _ptr(slot_mapping), num_tokens, _stream(stream)),
           "pkv_append")


def pkv_attention_workspace_bytes(pool: int, num_seqs: int, num_tokens: int, max_blocks_per_seq: int) -> int:
    return load().pkv_attention_workspace_bytes(pool, num_seqs, num_tokens, max_blocks_per_seq)


def pkv_attention_plan(pool: int, context_lens, query_start_loc, num_seqs: int, num_tokens: int,
                       max_blocks_per_seq: int, workspace, workspace_bytes: int, stream=None) -> None:
    _check(load().pkv_attention_plan(pool, _ptr(context_lens), _ptr(query_start_loc), num_seqs, num_tokens,
                                     max_blocks_per_seq, _ptr(workspace), workspace_bytes, _stream(stream)),
           "pkv_attention_plan")


def pkv_attention(pool: int, layer: int, q, block_tables, max_blocks_per_seq: int, context_lens, query_start_loc,
                  num_seqs: int, num_tokens: int, out, workspace, workspace_bytes: int, stream=None) -> None:
    _check(load().pkv_attention(pool, layer, _ptr(q), _ptr(block_tables), max_blocks_per_seq, _ptr(context_lens),
                                _ptr(query_start_loc), num_seqs, num_tokens, _ptr(out), _ptr(workspace),
                                workspace_bytes, _stream(stream)), "pkv_attention")


def pkv_attention_append(pool: int, layer: int, q, k, v, slot_mapping, block_tables, max_blocks_per_seq: int,
                         context_lens, query_start_loc, num_seqs: int, num_tokens: int, out, workspace,
                         workspace_bytes: int, stream=None) -> None:
    _check(load().pkv_attention_append(pool, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(block_tables),
                                       max_blocks_per_seq, _ptr(context_lens), _ptr(query_start_loc), num_seqs,
                                       num_tokens, _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)),
           "pkv_attention_append")


def pkv_debug_expire_wait(pool: int, limit_ns: int, stream=None) -> None:
    """Test hook (needs PKV_TEST_HOOKS=1): a bounded on-chip wait that runs out after limit_ns."""
    _check(load().pkv_debug_expire_wait(pool, limit_ns, _stream(stream)), "pkv_debug_expire_wait")


def pkv_attention_noalloc(pool: int, layer: int, q, block_tables, max_blocks_per_seq: int, context_lens,
                          query_start_loc, num_seqs: int, num_tokens: int, out, stream=None) -> None:
    _check(load().pkv_attention_noalloc(pool, layer, _ptr(q), _ptr(block_tables), max_blocks_per_seq,
                                        _ptr(context_lens), _ptr(query_start_loc), num_seqs, num_tokens, _ptr(out),
                                        _stream(stream)), "pkv_attention_noalloc")


PKV_NOALLOC_SCRATCH_BYTES = 16 << 20


def pkv_last_launch_count(pool: int) -> int:
    return load().pkv_last_launch_count(pool)


def pkv_last_error() -> str:
    return load().pkv_last_error().decode()


# ---- convenience wrappers over the same calls ---------------------------------------------------------

class Pool:
    """A cache pool backed by one torch uint8 device buffer of pkv_pool_bytes(cfg) bytes."""

    def __init__(self, num_layers, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size=16, split_blocks=0,
                 device="cuda", kv_dtype=PKV_KV_F16):
        import torch
        self.cfg = pkv_config(num_layers, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, split_blocks,
                              kv_dtype)
        nbytes = pkv_pool_bytes(self.cfg)
        if nbytes == 0:
            raise PkvError(PKV_ERR_INVALID_ARG, "pkv_pool_bytes", pkv_last_error())
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.handle = pkv_pool_init(self.cfg, self.buffer, nbytes)

    @property
    def is_8bit(self) -> bool:
        return self.cfg.kv_dtype == PKV_KV_E4M3

    def layer(self, layer: int, kv: int):
        """torch view [num_blocks, Hkv, bs, d] of one layer's K (kv=0) or V (kv=1) pool: fp16 values, or uint8
        E4M3 codes for an 8-bit cache."""
        return self.cache_view()[layer, kv]

    def cache_view(self):
        """torch view [L, 2, num_blocks, Hkv, bs, d] of the whole cache (fp16, or uint8 codes)."""
        import torch
        c = self.cfg
        n = 2 * c.num_layers * c.num_blocks * c.num_kv_heads * c.block_size * c.head_dim
        if self.is_8bit:
            v = self.buffer[:n]
        else:
            v = self.buffer[: n * 2].view(torch.float16)
        return v.view(c.num_layers, 2, c.num_blocks, c.num_kv_heads, c.block_size, c.head_dim)

    def scales_view(self):
        """8-bit cache: torch uint8 view [L, num_blocks, Hkv, 2 (K, V), bs] of the scale bytes."""
        c = self.cfg
        assert self.is_8bit, "an fp16 cache has no scales"
        off = 2 * c.num_layers * c.num_blocks * c.num_kv_heads * c.block_size * c.head_dim
        n = 2 * c.num_layers * c.num_blocks * c.num_kv_heads * c.block_size
        return self.buffer[off:off + n].view(c.num_layers, c.num_blocks, c.num_kv_heads, 2, c.block_size)

    def check(self, clear: bool = True) -> int:
        return pkv_pool_check(self.handle, clear)

    def close(self):
        if self.handle:
            pkv_pool_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Scheduler:
    """The C++ host scheduler (pkv_sched_*), returning numpy copies of each pass's batch."""

    def __init__(self, max_num_seqs: int, token_budget: int, block_size: int, num_blocks: int, free_order=None,
                 alloc: int = 0, unit: int = 0, prefix_caching: bool = False):
        lib = load()
        cfg = pkv_sched_config(max_num_seqs, token_budget, block_size, num_blocks)
        h = _p()
        arr = None
        if free_order is not None:
            arr = np.ascontiguousarray(np.asarray(free_order, dtype=np.int32))
        _check(lib.pkv_sched_create(ctypes.byref(cfg), arr.ctypes.data if arr is not None else None, ctypes.byref(h)),
               "pkv_sched_create")
        self.handle = h.value
        if alloc or unit:
            _check(lib.pkv_sched_set_policy(self.handle, alloc, unit), "pkv_sched_set_policy")
        if prefix_caching:
            _check(lib.pkv_sched_set_prefix_caching(self.handle, 1), "pkv_sched_set_prefix_caching")

    def add(self, req_id: int, prompt_len: int, max_output: int, declared_output: Optional[int] = None) -> None:
        if declared_output is None:
            _check(load().pkv_sched_add(self.handle, req_id, prompt_len, max_output), "pkv_sched_add")
        else:
            _check(load().pkv_sched_add_declared(self.handle, req_id, prompt_len, max_output, declared_output),
                   "pkv_sched_add_declared")

    def step(self) -> dict:
        st = pkv_step()
        _check(load().pkv_sched_step(self.handle, ctypes.byref(st)), "pkv_sched_step")
        B, T, W = st.num_seqs, st.num_tokens, st.max_blocks_per_seq

        def arr(ptr, n, dt):
            if n == 0:
                return np.zeros(0, dtype=dt)
            return np.ctypeslib.as_array(ptr, shape=(n,)).astype(dt, copy=True)

        return {
            "req_ids": arr(st.req_ids, B, np.int64), "q_lens": arr(st.q_lens, B, np.int32),
            "context_lens": arr(st.context_lens, B, np.int32),
            "query_start_loc": arr(st.query_start_loc, B + 1, np.int32),
            "block_tables": arr(st.block_tables, B * W, np.int32).reshape(B, W),
            "slot_mapping": arr(st.slot_mapping, T, np.int64), "max_blocks_per_seq": W,
            "preempted": arr(st.preempted, st.num_preempted, np.int64).tolist(),
            "admitted": arr(st.admitted, st.num_admitted, np.int64).tolist(),
            "finished": arr(st.finished, st.num_finished, np.int64).tolist(),
        }

    def abort(self, req_id: int) -> None:
        _check(load().pkv_sched_abort(self.handle, req_id), "pkv_sched_abort")

    def set_max_num_seqs(self, n: int) -> None:
        _check(load().pkv_sched_set_max_num_seqs(self.handle, n), "pkv_sched_set_max_num_seqs")

    def stats(self) -> dict:
        s = pkv_sched_stats()
        load().pkv_sched_get_stats(self.handle, ctypes.byref(s))
        return {f: getattr(s, f) for f, _ in pkv_sched_stats._fields_}

    def done(self) -> bool:
        return bool(load().pkv_sched_done(self.handle))

    def free_list(self) -> list:
        n = load().pkv_sched_free_list(self.handle, None, 0)
        buf = (_i32 * max(n, 1))()
        load().pkv_sched_free_list(self.handle, buf, n)
        return list(buf[:n])

    def close(self):
        if self.handle:
            load().pkv_sched_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
