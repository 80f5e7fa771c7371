"""Thin Python binding of the C ABI in include/gdn.h (argument marshalling only).

The functions keep the C names and argument order; device buffers are passed as torch
tensors (or raw integer addresses) and streams as torch.cuda.Stream (or raw handles).
Every computation happens in libgdn.so; there is no Python or CPU fallback. Importing
this module does not load the library; the first call does, and fails loudly if it was
not built (python -m packed_linear_attention_gb300.build).
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID_ARGUMENT = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_WORKSPACE_TOO_SMALL = 3
GDN_ERR_CUDA = 4
GDN_ERR_DEVICE_TIMEOUT = 5
GDN_ERR_POOL_EXHAUSTED = 6
GDN_ERR_BUSY = 7
GDN_F32 = 0
GDN_BF16 = 1
GDN_GATES_DIRECT = 0
GDN_GATES_RAW = 1
KERNEL_AUTO = 0
KERNEL_RECURRENT = 1
KERNEL_CHUNKED_PIPELINED = 2
KERNEL_CHUNKED_THROUGHPUT = 3

# every symbol include/gdn.h declares
EXPORTS = (
    "gdn_abi_version", "gdn_status_string", "gdn_handle_create", "gdn_handle_destroy",
    "gdn_pool_info", "gdn_set_kernel_preference", "gdn_prefill_workspace_size",
    "gdn_prefill_packed", "gdn_read_device_status", "gdn_checkpoint_copy",
    "gdn_checkpoint_copy_query", "gdn_checkpoint_copy_wait", "gdn_decode_step",
    "gdn_ckpt_position", "gdn_mixed_budget", "gdn_prefill_worklist_host",
    "gdn_prefill_packed_noalloc", "gdn_prefill_packed_async", "gdn_prefill_async_query",
    "gdn_prefill_async_wait", "gdn_prefill_async_join", "gdn_prefill_split_workspace_size",
    "gdn_prefill_packed_split", "gdn_prefill_packed_host", "gdn_prefill_host_workspace_size",
    "gdn_chunked_schedule", "gdn_set_test_hook", "gdn_prefill_packed_pool",
    "gdn_prefill_launch_count", "gdn_prefill_packed_snapshot", "gdn_checkpoint_copy_event",
    "gdn_checkpoint_copy_join", "gdn_noalloc_read_status", "gdn_noalloc_set_test_hook",
    "gdn_split_segment_auto",
)


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class gdn_prefill_buffers(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in
                ("q", "k", "v", "a", "beta", "initial_state", "o", "ckpt_states",
                 "final_states")]


class gdn_config(ctypes.Structure):
    _fields_ = [("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_dim_k", ctypes.c_int32), ("head_dim_v", ctypes.c_int32),
                ("chunk_size", ctypes.c_int32), ("scale", ctypes.c_float),
                ("qk_l2norm", ctypes.c_int32), ("io_dtype", ctypes.c_int32),
                ("gate_mode", ctypes.c_int32), ("a_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libgdn.so (once) and declare the prototypes."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m packed_linear_attention_gb300.build`")
        lib = ctypes.CDLL(path)
        P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        CFG = ctypes.POINTER(gdn_config)
        IP = ctypes.POINTER(ctypes.c_int32)
        sig = {
            "gdn_abi_version": (I32, []),
            "gdn_status_string": (ctypes.c_char_p, [I32]),
            "gdn_handle_create": (I32, [I32, SZ, ctypes.POINTER(P)]),
            "gdn_handle_destroy": (I32, [P]),
            "gdn_pool_info": (I32, [P, ctypes.POINTER(P), ctypes.POINTER(SZ)]),
            "gdn_set_kernel_preference": (I32, [P, I32]),
            "gdn_chunked_schedule": (I32, [I32, IP, I32, I32, IP]),
            "gdn_set_test_hook": (I32, [P, I32]),
            "gdn_prefill_workspace_size": (I32, [CFG, I32, IP, IP, ctypes.POINTER(SZ)]),
            "gdn_prefill_packed": (I32, [P, CFG, I32, IP, P, P, P, P, P, P, IP, IP, P, P, P,
                                         P, SZ, P]),
            "gdn_prefill_packed_pool": (I32, [P, CFG, I32, IP, P, P, P, P, P, P, I32, IP, IP,
                                              IP, IP, P, P, P, SZ, P]),
            "gdn_prefill_launch_count": (I32, [P, IP]),
            "gdn_prefill_packed_snapshot": (I32, [P, CFG, I32, IP, P, P, P, P, P, P, IP, IP, P,
                                                  P, P, SZ, P, SZ, P]),
            "gdn_checkpoint_copy_event": (I32, [P, ctypes.POINTER(P)]),
            "gdn_checkpoint_copy_join": (I32, [P, P]),
            "gdn_noalloc_read_status": (I32, [IP, P]),
            "gdn_split_segment_auto": (I32, [I32, IP, I32, I32, IP]),
            "gdn_noalloc_set_test_hook": (I32, [I32]),
            "gdn_prefill_split_workspace_size": (I32, [CFG, I32, IP, IP, IP, I32,
                                                       ctypes.POINTER(ctypes.c_size_t)]),
            "gdn_prefill_packed_split": (I32, [P, CFG, I32, IP, P, P, P, P, P, P, IP, IP, P, P,
                                               P, I32, P, SZ, P]),
            "gdn_prefill_host_workspace_size": (I32, [CFG, I32, IP, IP, I32,
                                                      ctypes.POINTER(ctypes.c_size_t)]),
            "gdn_prefill_packed_host": (I32, [P, CFG, I32, IP, IP, IP,
                                              ctypes.POINTER(gdn_prefill_buffers),
                                              ctypes.POINTER(gdn_prefill_buffers), I32, P, SZ,
                                              P]),
            "gdn_read_device_status": (I32, [P, IP, P]),
            "gdn_prefill_packed_noalloc": (I32, [CFG, I32, IP, P, P, P, P, P, P, IP, IP, P, P,
                                                 P, P]),
            "gdn_prefill_worklist_host": (I32, [P, CFG, I32, IP, IP, IP, P, SZ,
                                                ctypes.POINTER(SZ)]),
            "gdn_prefill_packed_async": (I32, [P, CFG, I32, IP, P, P, P, P, P, P, IP, IP, P, P,
                                               P, P, SZ, P]),
            "gdn_prefill_async_query": (I32, [P]),
            "gdn_prefill_async_wait": (I32, [P]),
            "gdn_prefill_async_join": (I32, [P, P]),
            "gdn_checkpoint_copy": (I32, [P, P, SZ, SZ, P]),
            "gdn_checkpoint_copy_query": (I32, [P]),
            "gdn_checkpoint_copy_wait": (I32, [P]),
            "gdn_decode_step": (I32, [P, CFG, I32, P, P, P, P, P, P, I32, P, P, P]),
            "gdn_ckpt_position": (I32, [I32, I32, I32]),
            "gdn_mixed_budget": (I32, [I32, IP, I32, I32, IP]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != GDN_OK:
        raise GdnError(status, where)


def _addr(x) -> int | None:
    """Device address of a tensor (or an int address, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    return x.data_ptr() or None


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None


def _i32(a) -> ctypes.Array | None:
    if a is None:
        return None
    arr = np.ascontiguousarray(a, dtype=np.int32)
    return (ctypes.c_int32 * max(1, arr.size))(*arr.tolist())


def make_config(num_k_heads, num_v_heads, head_dim, *, scale=None, io_dtype=GDN_BF16,
                chunk_size=64, qk_l2norm=True, a_log=None, dt_bias=None) -> gdn_config:
    """Layer config; passing a_log and dt_bias (device tensors of H_v floats) selects raw
    gate inputs (GDN_GATES_RAW). The tensors must outlive every call using the config."""
    raw = a_log is not None or dt_bias is not None
    return gdn_config(int(num_k_heads), int(num_v_heads), int(head_dim), int(head_dim),
                      int(chunk_size), float(scale if scale is not None else head_dim ** -0.5),
                      1 if qk_l2norm else 0, int(io_dtype),
                      GDN_GATES_RAW if raw else GDN_GATES_DIRECT, _addr(a_log), _addr(dt_bias))


# ---- C entry points, same names -----------------------------------------------------------

def gdn_abi_version() -> int:
    return int(load().gdn_abi_version())


def gdn_handle_create(device: int = 0, pinned_pool_bytes: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(load().gdn_handle_create(int(device), int(pinned_pool_bytes), ctypes.byref(h)),
           "gdn_handle_create")
    return h.value


def gdn_handle_destroy(handle: int) -> None:
    _check(load().gdn_handle_destroy(handle), "gdn_handle_destroy")


def gdn_pool_info(handle: int) -> tuple[int, int]:
    p, n = ctypes.c_void_p(), ctypes.c_size_t()
    _check(load().gdn_pool_info(handle, ctypes.byref(p), ctypes.byref(n)), "gdn_pool_info")
    return p.value or 0, n.value


def gdn_set_kernel_preference(handle: int, preference: int) -> None:
    _check(load().gdn_set_kernel_preference(handle, int(preference)),
           "gdn_set_kernel_preference")


def gdn_set_test_hook(handle: int, hook: int) -> None:
    """1: the chunked kernels leave out every unit's first q/k copy, so that its first
    bounded wait runs out (the device timeout path, without a fault); 0: off."""
    _check(load().gdn_set_test_hook(handle, int(hook)), "gdn_set_test_hook")


def gdn_chunked_schedule(cu_seqlens, num_v_heads: int, num_sms: int) -> int:
    """The chunked schedule the automatic choice takes for this pack: KERNEL_CHUNKED_PIPELINED
    or KERNEL_CHUNKED_THROUGHPUT."""
    out = ctypes.c_int32()
    _check(load().gdn_chunked_schedule(len(cu_seqlens) - 1, _i32(cu_seqlens), int(num_v_heads),
                                       int(num_sms), ctypes.byref(out)), "gdn_chunked_schedule")
    return out.value


def gdn_split_segment_auto(cu_seqlens, num_v_heads: int, num_sms: int) -> int:
    """The segment length the cost model picks for gdn_prefill_packed_split (0: no split)."""
    out = ctypes.c_int32()
    _check(load().gdn_split_segment_auto(len(cu_seqlens) - 1, _i32(cu_seqlens),
                                         int(num_v_heads), int(num_sms), ctypes.byref(out)),
           "gdn_split_segment_auto")
    return out.value


def gdn_prefill_workspace_size(cfg: gdn_config, cu_seqlens, ckpt_cu=None) -> int:
    n = ctypes.c_size_t()
    num_seqs = len(cu_seqlens) - 1
    _check(load().gdn_prefill_workspace_size(ctypes.byref(cfg), num_seqs, _i32(cu_seqlens),
                                             _i32(ckpt_cu), ctypes.byref(n)),
           "gdn_prefill_workspace_size")
    return n.value


def gdn_prefill_packed(handle, cfg, cu_seqlens, q, k, v, a, beta, initial_state, ckpt_cu,
                       ckpt_pos, o, ckpt_states, final_states, workspace, workspace_bytes,
                       stream=None, *, raise_on_error=True) -> int:
    num_seqs = len(cu_seqlens) - 1
    st = load().gdn_prefill_packed(
        handle, ctypes.byref(cfg), num_seqs, _i32(cu_seqlens), _addr(q), _addr(k), _addr(v),
        _addr(a), _addr(beta), _addr(initial_state), _i32(ckpt_cu), _i32(ckpt_pos),
        _addr(o), _addr(ckpt_states), _addr(final_states), _addr(workspace),
        int(workspace_bytes), _stream(stream))
    if raise_on_error:
        _check(st, "gdn_prefill_packed")
    return st


def gdn_prefill_packed_pool(handle, cfg, cu_seqlens, q, k, v, a, beta, state_pool,
                            num_slots, slot_idx, start_zero, ckpt_cu, ckpt_pos, o, ckpt_states,
                            workspace, workspace_bytes, stream=None, *,
                            raise_on_error=True) -> int:
    """Prefill whose prompts read and write their states in place in a pool:
    state_pool[slot_idx[n]] (host int32 list); start_zero[n] != 0 starts prompt n from zeros."""
    num_seqs = len(cu_seqlens) - 1
    st = load().gdn_prefill_packed_pool(
        handle, ctypes.byref(cfg), num_seqs, _i32(cu_seqlens), _addr(q), _addr(k), _addr(v),
        _addr(a), _addr(beta), _addr(state_pool), int(num_slots), _i32(slot_idx),
        _i32(start_zero), _i32(ckpt_cu), _i32(ckpt_pos), _addr(o), _addr(ckpt_states),
        _addr(workspace), int(workspace_bytes), _stream(stream))
    if raise_on_error:
        _check(st, "gdn_prefill_packed_pool")
    return st


def gdn_prefill_launch_count(handle) -> int:
    """Kernels enqueued by the handle's last prefill call."""
    n = ctypes.c_int32()
    _check(load().gdn_prefill_launch_count(handle, ctypes.byref(n)), "gdn_prefill_launch_count")
    return n.value


def gdn_prefill_split_workspace_size(cfg: gdn_config, cu_seqlens, ckpt_cu=None, ckpt_pos=None,
                                     segment_len: int = 4096) -> int:
    n = ctypes.c_size_t()
    _check(load().gdn_prefill_split_workspace_size(ctypes.byref(cfg), len(cu_seqlens) - 1,
                                                   _i32(cu_seqlens), _i32(ckpt_cu),
                                                   _i32(ckpt_pos), int(segment_len),
                                                   ctypes.byref(n)),
           "gdn_prefill_split_workspace_size")
    return n.value


def gdn_prefill_packed_split(handle, cfg, cu_seqlens, q, k, v, a, beta, initial_state, ckpt_cu,
                             ckpt_pos, o, ckpt_states, final_states, segment_len, workspace,
                             workspace_bytes, stream=None, *, raise_on_error=True) -> int:
    """gdn_prefill_packed with prompts longer than segment_len cut into parallel segments."""
    st = load().gdn_prefill_packed_split(
        handle, ctypes.byref(cfg), len(cu_seqlens) - 1, _i32(cu_seqlens), _addr(q), _addr(k),
        _addr(v), _addr(a), _addr(beta), _addr(initial_state), _i32(ckpt_cu), _i32(ckpt_pos),
        _addr(o), _addr(ckpt_states), _addr(final_states), int(segment_len), _addr(workspace),
        int(workspace_bytes), _stream(stream))
    if raise_on_error:
        _check(st, "gdn_prefill_packed_split")
    return st


def prefill_buffers(q, k, v, a, beta, initial_state, o, ckpt_states, final_states):
    """A gdn_prefill_buffers record from tensors (or addresses, or None)."""
    return gdn_prefill_buffers(*(_addr(x) for x in (q, k, v, a, beta, initial_state, o,
                                                     ckpt_states, final_states)))


def gdn_prefill_host_workspace_size(cfg: gdn_config, cu_seqlens, ckpt_cu=None,
                                    group_prompts: int = 8) -> int:
    n = ctypes.c_size_t()
    _check(load().gdn_prefill_host_workspace_size(ctypes.byref(cfg), len(cu_seqlens) - 1,
                                                  _i32(cu_seqlens), _i32(ckpt_cu),
                                                  int(group_prompts), ctypes.byref(n)),
           "gdn_prefill_host_workspace_size")
    return n.value


def gdn_prefill_packed_host(handle, cfg, cu_seqlens, ckpt_cu, ckpt_pos, host, device,
                            group_prompts, workspace, workspace_bytes, stream=None, *,
                            raise_on_error=True) -> int:
    """gdn_prefill_packed for host-resident inputs and outputs, copies overlapped per group
    of prompts. `host` and `device` are gdn_prefill_buffers records."""
    st = load().gdn_prefill_packed_host(
        handle, ctypes.byref(cfg), len(cu_seqlens) - 1, _i32(cu_seqlens), _i32(ckpt_cu),
        _i32(ckpt_pos), ctypes.byref(host), ctypes.byref(device), int(group_prompts),
        _addr(workspace), int(workspace_bytes), _stream(stream))
    if raise_on_error:
        _check(st, "gdn_prefill_packed_host")
    return st


def gdn_prefill_packed_noalloc(cfg, cu_seqlens, q, k, v, a, beta, initial_state, ckpt_cu,
                               ckpt_pos, o, ckpt_states, final_states, stream=None, *,
                               raise_on_error=True) -> int:
    """gdn_prefill_packed without workspace or handle, for callers that cannot allocate at
    call time; the work list goes to the library's fixed per-GPU device array."""
    num_seqs = len(cu_seqlens) - 1
    st = load().gdn_prefill_packed_noalloc(
        ctypes.byref(cfg), num_seqs, _i32(cu_seqlens), _addr(q), _addr(k), _addr(v), _addr(a),
        _addr(beta), _addr(initial_state), _i32(ckpt_cu), _i32(ckpt_pos), _addr(o),
        _addr(ckpt_states), _addr(final_states), _stream(stream))
    if raise_on_error:
        _check(st, "gdn_prefill_packed_noalloc")
    return st


def gdn_noalloc_read_status(stream=None) -> int:
    """The status word of the last gdn_prefill_packed_noalloc call on the current device."""
    v = ctypes.c_int32()
    _check(load().gdn_noalloc_read_status(ctypes.byref(v), _stream(stream)),
           "gdn_noalloc_read_status")
    return v.value


def gdn_noalloc_set_test_hook(hook: int) -> None:
    _check(load().gdn_noalloc_set_test_hook(int(hook)), "gdn_noalloc_set_test_hook")


def gdn_prefill_packed_async(handle, cfg, cu_seqlens, q, k, v, a, beta, initial_state, ckpt_cu,
                             ckpt_pos, o, ckpt_states, final_states, workspace, workspace_bytes,
                             after_stream=None, *, raise_on_error=True) -> int:
    """Prefill on the handle's own stream after the work queued on `after_stream`."""
    num_seqs = len(cu_seqlens) - 1
    st = load().gdn_prefill_packed_async(
        handle, ctypes.byref(cfg), num_seqs, _i32(cu_seqlens), _addr(q), _addr(k), _addr(v),
        _addr(a), _addr(beta), _addr(initial_state), _i32(ckpt_cu), _i32(ckpt_pos),
        _addr(o), _addr(ckpt_states), _addr(final_states), _addr(workspace),
        int(workspace_bytes), _stream(after_stream))
    if raise_on_error:
        _check(st, "gdn_prefill_packed_async")
    return st


def gdn_prefill_async_query(handle) -> bool:
    """True when no prefill is in flight on the handle's stream."""
    st = load().gdn_prefill_async_query(handle)
    if st == GDN_ERR_DEVICE_TIMEOUT:
        return False
    _check(st, "gdn_prefill_async_query")
    return True


def gdn_prefill_async_wait(handle) -> None:
    _check(load().gdn_prefill_async_wait(handle), "gdn_prefill_async_wait")


def gdn_prefill_async_join(handle, stream=None) -> None:
    _check(load().gdn_prefill_async_join(handle, _stream(stream)), "gdn_prefill_async_join")


def prefill_split(handle, buf: "DeviceBuffers", segment_len: int, stream=None) -> int:
    """gdn_prefill_packed_split on a DeviceBuffers bundle (allocates its own workspace)."""
    import torch
    ckpt_pos = buf.ckpt_pos if len(buf.ckpt_pos) else None
    nbytes = gdn_prefill_split_workspace_size(buf.cfg, buf.cu, buf.ckpt_cu, ckpt_pos,
                                              segment_len)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=buf.o.device)
    st = gdn_prefill_packed_split(handle, buf.cfg, buf.cu, buf.q, buf.k, buf.v, buf.a, buf.beta,
                                  buf.init, buf.ckpt_cu, ckpt_pos, buf.o,
                                  buf.ckpt if buf.ckpt.numel() else None, buf.final,
                                  segment_len, ws, nbytes, stream)
    buf.split_workspace = ws  # keep alive until the work on the stream is done
    return st


def prefill_async(handle, buf: "DeviceBuffers", after_stream=None, *, raise_on_error=True) -> int:
    """gdn_prefill_packed_async on a DeviceBuffers bundle."""
    return gdn_prefill_packed_async(handle, buf.cfg, buf.cu, buf.q, buf.k, buf.v, buf.a,
                                    buf.beta, buf.init, buf.ckpt_cu, buf.ckpt_pos, buf.o,
                                    buf.ckpt if buf.ckpt.numel() else None, buf.final,
                                    buf.workspace, buf.workspace_bytes, after_stream,
                                    raise_on_error=raise_on_error)


def gdn_prefill_worklist_host(handle, cfg, cu_seqlens, ckpt_cu=None, ckpt_pos=None) -> dict:
    """The work list gdn_prefill_packed would upload, decoded into NumPy arrays."""
    lib = load()
    num_seqs = len(cu_seqlens) - 1
    cu, cc, cp = _i32(cu_seqlens), _i32(ckpt_cu), _i32(ckpt_pos)
    need = ctypes.c_size_t()
    _check(lib.gdn_prefill_worklist_host(handle, ctypes.byref(cfg), num_seqs, cu, cc, cp, None,
                                         0, ctypes.byref(need)), "gdn_prefill_worklist_host")
    buf = (ctypes.c_uint8 * need.value)()
    _check(lib.gdn_prefill_worklist_host(handle, ctypes.byref(cfg), num_seqs, cu, cc, cp, buf,
                                         need.value, ctypes.byref(need)),
           "gdn_prefill_worklist_host")
    raw = np.frombuffer(bytes(buf), dtype=np.int32)
    nu = int(raw[1])
    units_off = 256 // 4
    seqs_off = ((256 + 16 * nu + 255) // 256 * 256) // 4
    pos_off = ((seqs_off * 4 + 24 * num_seqs + 255) // 256 * 256) // 4  # GdnSeq: 6 int32
    nck = 0 if ckpt_cu is None else int(np.asarray(ckpt_cu)[-1])
    ready_off = ((pos_off * 4 + 4 * max(nck, 1) + 255) // 256 * 256) // 4
    return dict(status=int(raw[0]), num_units=nu,
                units=raw[units_off:units_off + 4 * nu].reshape(nu, 4).copy(),
                seqs=raw[seqs_off:seqs_off + 6 * num_seqs].reshape(num_seqs, 6).copy(),
                ckpt_pos=raw[pos_off:pos_off + nck].copy(),
                ready=raw[ready_off:ready_off + num_seqs].copy(), nbytes=need.value)


def gdn_read_device_status(workspace, stream=None) -> int:
    v = ctypes.c_int32()
    _check(load().gdn_read_device_status(_addr(workspace), ctypes.byref(v), _stream(stream)),
           "gdn_read_device_status")
    return v.value


def gdn_checkpoint_copy(handle, ckpt_states, nbytes: int, pool_offset: int = 0,
                        stream=None) -> None:
    _check(load().gdn_checkpoint_copy(handle, _addr(ckpt_states), int(nbytes),
                                      int(pool_offset), _stream(stream)),
           "gdn_checkpoint_copy")


def gdn_prefill_packed_snapshot(handle, cfg, cu_seqlens, q, k, v, a, beta, initial_state,
                                ckpt_cu, ckpt_pos, o, ckpt_states, final_states, pool_offset,
                                workspace, workspace_bytes, stream=None, *,
                                raise_on_error=True) -> int:
    """gdn_prefill_packed whose checkpoints are copied into the handle's pinned pool (at
    pool_offset) while the scan still runs."""
    st = load().gdn_prefill_packed_snapshot(
        handle, ctypes.byref(cfg), len(cu_seqlens) - 1, _i32(cu_seqlens), _addr(q), _addr(k),
        _addr(v), _addr(a), _addr(beta), _addr(initial_state), _i32(ckpt_cu), _i32(ckpt_pos),
        _addr(o), _addr(ckpt_states), _addr(final_states), int(pool_offset), _addr(workspace),
        int(workspace_bytes), _stream(stream))
    if raise_on_error:
        _check(st, "gdn_prefill_packed_snapshot")
    return st


def prefill_snapshot(handle, buf: "DeviceBuffers", pool_offset: int = 0, stream=None) -> int:
    """gdn_prefill_packed_snapshot on a DeviceBuffers bundle."""
    return gdn_prefill_packed_snapshot(handle, buf.cfg, buf.cu, buf.q, buf.k, buf.v, buf.a,
                                       buf.beta, buf.init, buf.ckpt_cu,
                                       buf.ckpt_pos if len(buf.ckpt_pos) else None, buf.o,
                                       buf.ckpt if buf.ckpt.numel() else None, buf.final,
                                       pool_offset, buf.workspace, buf.workspace_bytes, stream)


def gdn_checkpoint_copy_event(handle) -> int:
    """The handle's copy-completion event (a cudaEvent_t as an integer)."""
    ev = ctypes.c_void_p()
    _check(load().gdn_checkpoint_copy_event(handle, ctypes.byref(ev)), "gdn_checkpoint_copy_event")
    return ev.value or 0


def gdn_checkpoint_copy_join(handle, stream=None) -> None:
    _check(load().gdn_checkpoint_copy_join(handle, _stream(stream)), "gdn_checkpoint_copy_join")


def gdn_checkpoint_copy_query(handle) -> bool:
    st = load().gdn_checkpoint_copy_query(handle)
    if st == GDN_ERR_DEVICE_TIMEOUT:
        return False
    _check(st, "gdn_checkpoint_copy_query")
    return True


def gdn_checkpoint_copy_wait(handle) -> None:
    _check(load().gdn_checkpoint_copy_wait(handle), "gdn_checkpoint_copy_wait")


def gdn_decode_step(handle, cfg, batch, q, k, v, a, beta, state_pool, num_slots, slot_idx, o,
                    stream=None, *, raise_on_error=True) -> int:
    st = load().gdn_decode_step(handle, ctypes.byref(cfg), int(batch), _addr(q), _addr(k),
                                _addr(v), _addr(a), _addr(beta), _addr(state_pool),
                                int(num_slots), _addr(slot_idx), _addr(o), _stream(stream))
    if raise_on_error:
        _check(st, "gdn_decode_step")
    return st


def gdn_ckpt_position(length: int, block: int, tail: int) -> int:
    return int(load().gdn_ckpt_position(int(length), int(block), int(tail)))


def gdn_mixed_budget(remaining, budget: int, max_prompts: int) -> tuple[int, list[int]]:
    rem = np.ascontiguousarray(remaining, dtype=np.int32)
    take = (ctypes.c_int32 * max(1, rem.size))()
    served = load().gdn_mixed_budget(int(rem.size), _i32(rem), int(budget), int(max_prompts),
                                     take)
    if served < 0:
        raise GdnError(GDN_ERR_INVALID_ARGUMENT, "gdn_mixed_budget")
    return int(served), [int(take[i]) for i in range(rem.size)]


# ---- convenience: one prefill call on device tensors ---------------------------------------

@dataclass
class DeviceBuffers:
    """Device copies of a packed workload plus output and workspace buffers."""

    cfg: gdn_config
    cu: np.ndarray
    ckpt_cu: np.ndarray
    ckpt_pos: np.ndarray
    q: object
    k: object
    v: object
    a: object
    beta: object
    init: object
    o: object
    ckpt: object
    final: object
    workspace: object
    workspace_bytes: int
    a_log: object = None       # device tensors kept alive for the config's pointers
    dt_bias: object = None
    split_workspace: object = None  # workspace of the last prefill_split call


def to_device(pack, device="cuda", cfg: gdn_config | None = None) -> DeviceBuffers:
    """Upload a ``Pack`` (from ``packed_linear_attention_gb300.inputs``) and allocate outputs."""
    import torch

    bf16 = pack.io_dtype == "bf16"
    a_log = dt_bias = None
    if getattr(pack, "a_log", None) is not None:
        a_log = torch.from_numpy(np.ascontiguousarray(pack.a_log, np.float32)).to(device)
        dt_bias = torch.from_numpy(np.ascontiguousarray(pack.dt_bias, np.float32)).to(device)
    if cfg is None:
        cfg = make_config(pack.num_k_heads, pack.num_v_heads, pack.head_dim, scale=pack.scale,
                          io_dtype=GDN_BF16 if bf16 else GDN_F32, chunk_size=pack.chunk_size,
                          qk_l2norm=pack.qk_l2norm, a_log=a_log, dt_bias=dt_bias)

    def up(x):
        if bf16 and x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)

    T, Hv, D = pack.total_tokens, pack.num_v_heads, pack.head_dim
    io_t = torch.bfloat16 if bf16 else torch.float32
    C = pack.num_ckpts
    ws_bytes = gdn_prefill_workspace_size(cfg, pack.cu_seqlens, pack.ckpt_cu)
    return DeviceBuffers(
        cfg=cfg, cu=pack.cu_seqlens, ckpt_cu=pack.ckpt_cu, ckpt_pos=pack.ckpt_pos,
        q=up(pack.q), k=up(pack.k), v=up(pack.v), a=up(pack.a), beta=up(pack.beta),
        init=None if pack.init is None else up(pack.init),
        o=torch.empty((T, Hv, D), dtype=io_t, device=device),
        ckpt=torch.empty((max(C, 0), Hv, D, D), dtype=torch.float32, device=device),
        final=torch.empty((pack.num_seqs, Hv, D, D), dtype=torch.float32, device=device),
        workspace=torch.empty(ws_bytes, dtype=torch.uint8, device=device),
        workspace_bytes=ws_bytes, a_log=a_log, dt_bias=dt_bias,
    )


def prefill(handle, buf: DeviceBuffers, stream=None) -> int:
    """gdn_prefill_packed on a DeviceBuffers bundle."""
    return gdn_prefill_packed(handle, buf.cfg, buf.cu, buf.q, buf.k, buf.v, buf.a, buf.beta,
                              buf.init, buf.ckpt_cu, buf.ckpt_pos, buf.o,
                              buf.ckpt if buf.ckpt.numel() else None, buf.final,
                              buf.workspace, buf.workspace_bytes, stream)
