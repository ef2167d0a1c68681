"""ctypes binding of libmk's C ABI (include/mk.h): same names, marshalling only.

Loading fails loudly when the library has not been built; there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_uint16, c_uint32, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmk.so")

MK_ABI_VERSION = 1
MK_OK = 0
MK_ERR_ARG, MK_ERR_STATE, MK_ERR_LIMIT, MK_ERR_ABI, MK_ERR_CUDA, MK_ERR_NOMEM = -1, -2, -3, -4, -5, -6
MK_DEV_OK = 0
MK_DEV_DEP_TIMEOUT, MK_DEV_BAD_OP, MK_DEV_RING_TIMEOUT = -10, -11, -12
MK_DEV_CAPACITY, MK_DEV_ABORTED, MK_DEV_BAD_INDEX = -13, -14, -15
MK_OP_NOP, MK_OP_MEMCPY, MK_OP_GEMV, MK_OP_RMSNORM, MK_OP_ATTENTION, MK_OP_MLP, MK_OP_SAMPLE = range(7)
MK_OP_ATTENTION_APPEND, MK_OP_ATTENTION_PARTIAL, MK_OP_ATTENTION_COMBINE = 7, 8, 9
MK_F_SILU_MUL, MK_F_ADD_RESIDUAL, MK_F_RMS_NORM_INPUT, MK_F_ARGMAX_EPI = 1, 2, 4, 8
MK_BF16, MK_F32, MK_I32, MK_PAIR = 1, 2, 3, 4
MK_MODE_MEGA, MK_MODE_PER_OP, MK_MODE_PER_OP_GRAPH, MK_MODE_LEVELS, MK_MODE_PER_OP_PDL = 0, 1, 2, 3, 4
MK_NO_BUF = 0xFFFF

EXPORTS = [
    "mk_graph_create", "mk_set_state", "mk_add_buffer", "mk_add_embed", "mk_add_rmsnorm", "mk_fuse_rmsnorm",
    "mk_add_matmul",
    "mk_add_attention", "mk_add_sample", "mk_attention_scratch_rows", "mk_gemv_tiles", "mk_scratch_size",
    "mk_lower", "mk_get_tasks", "mk_get_edges", "mk_get_sync_plan", "mk_get_ll_plan", "mk_get_queues",
    "mk_upload",
    "mk_decode_step", "mk_decode_step_ex", "mk_decode_step_host", "mk_status",
    "mk_get_trace", "mk_kernel_info", "mk_destroy", "mk_last_error", "mk_debug_patch_task",
    "mk_attention_decode_noalloc", "mk_gemv_tensor_core_tiles", "mk_debug_set_epoch", "mk_set_chunk",
]


class MkConfig(ctypes.Structure):
    _fields_ = [("abi_version", c_uint32), ("num_ctas", c_int32), ("tiles_target", c_int32),
                ("col_align", c_int32), ("wait_timeout_us", c_uint32)]


class MkError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} returned {code}: {msg}")
        self.code = code


_lib = None


def lib():
    """The loaded libmk.  Raises if it is missing (build it first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmk.so not built ({LIB_PATH}); run task_graph_interpreter_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    G = c_void_p
    sig = {
        "mk_graph_create": (c_int, [POINTER(MkConfig), POINTER(c_void_p)]),
        "mk_set_state": (c_int, [G, c_void_p, c_int]),
        "mk_set_chunk": (c_int, [G, c_int, c_uint16]),
        "mk_add_buffer": (c_int, [G, c_void_p, c_int, c_int64, c_int64, POINTER(c_uint16)]),
        "mk_add_embed": (c_int, [G, c_uint16, c_uint16, c_int, c_int]),
        "mk_add_matmul": (c_int, [G, c_uint16, c_uint16, c_uint16, c_uint16, c_uint16, c_uint32,
                                  c_int, c_int, c_int, c_float]),
        "mk_add_attention": (c_int, [G, c_uint16, c_uint16, c_uint16, c_uint16, c_uint16, c_int, c_int,
                                     c_int, c_int, c_int, POINTER(c_int32), c_int, c_double]),
        "mk_add_sample": (c_int, [G, c_uint16, c_uint16, c_int, c_int, c_int]),
        "mk_attention_scratch_rows": (c_int, [G, c_int, c_int, POINTER(c_int32), c_int, POINTER(c_int64)]),
        "mk_gemv_tiles": (c_int, [G, c_int, POINTER(c_int32)]),
        "mk_scratch_size": (c_int, [G, c_uint16, POINTER(c_size_t)]),
        "mk_lower": (c_int, [G]),
        "mk_get_tasks": (c_int, [G, POINTER(c_void_p), POINTER(c_size_t)]),
        "mk_get_edges": (c_int, [G, POINTER(c_void_p), POINTER(c_size_t)]),
        "mk_get_queues": (c_int, [G, POINTER(c_void_p), POINTER(c_void_p), POINTER(c_int)]),
        "mk_get_sync_plan": (c_int, [G, POINTER(c_void_p), POINTER(c_void_p), POINTER(c_void_p),
                                     POINTER(c_void_p), POINTER(c_uint32)]),
        "mk_get_ll_plan": (c_int, [G, POINTER(c_void_p), POINTER(c_void_p)]),
        "mk_upload": (c_int, [G, c_void_p]),
        "mk_decode_step": (c_int, [G, c_void_p]),
        "mk_decode_step_ex": (c_int, [G, c_void_p, c_int, c_uint32]),
        "mk_decode_step_host": (c_int, [G, c_void_p, c_void_p, c_void_p]),
        "mk_status": (c_int, [G, c_void_p, POINTER(c_int), POINTER(c_int32)]),
        "mk_get_trace": (c_int, [G, POINTER(c_void_p), POINTER(c_size_t)]),
        "mk_kernel_info": (c_int, [G, POINTER(c_int), POINTER(c_int), POINTER(c_int)]),
        "mk_destroy": (None, [G]),
        "mk_debug_patch_task": (c_int, [G, c_int, c_void_p]),
        "mk_debug_set_epoch": (c_int, [G, c_void_p, c_uint32, c_uint32]),
        "mk_add_rmsnorm": (c_int, [G, c_uint16, c_uint16, c_uint16, c_uint16, c_int, c_int, c_float]),
        "mk_fuse_rmsnorm": (c_int, [G, POINTER(c_int)]),
        "mk_gemv_tensor_core_tiles": (c_int, [G, POINTER(c_int)]),
        "mk_attention_decode_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                                c_int, c_int, c_int, POINTER(c_int32), POINTER(c_int32), c_int,
                                                c_double]),
        "mk_last_error": (c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def check(rc: int, fn: str):
    if rc != MK_OK:
        raise MkError(fn, rc, lib().mk_last_error().decode(errors="replace"))


# --------------------------------------------------------------- same-name wrappers
def mk_graph_create(num_ctas=0, tiles_target=0, col_align=16, wait_timeout_us=0,
                    abi_version=MK_ABI_VERSION):
    cfg = MkConfig(abi_version, num_ctas, tiles_target, col_align, wait_timeout_us)
    h = c_void_p()
    check(lib().mk_graph_create(ctypes.byref(cfg), ctypes.byref(h)), "mk_graph_create")
    return h


def mk_set_state(g, dptr: int, B: int):
    check(lib().mk_set_state(g, c_void_p(dptr), B), "mk_set_state")


def mk_set_chunk(g, T: int, tokens: int):
    check(lib().mk_set_chunk(g, T, tokens), "mk_set_chunk")


def mk_add_buffer(g, dptr: int, dtype: int, rows: int, cols: int) -> int:
    idx = c_uint16()
    check(lib().mk_add_buffer(g, c_void_p(dptr), dtype, rows, cols, ctypes.byref(idx)), "mk_add_buffer")
    return idx.value


def mk_add_embed(g, table: int, out: int, B: int, H: int):
    check(lib().mk_add_embed(g, table, out, B, H), "mk_add_embed")


def mk_add_rmsnorm(g, x, gamma, residual, out, B, H, eps):
    check(lib().mk_add_rmsnorm(g, x, gamma, residual, out, B, H, eps), "mk_add_rmsnorm")


def mk_fuse_rmsnorm(g) -> int:
    n = c_int()
    check(lib().mk_fuse_rmsnorm(g, ctypes.byref(n)), "mk_fuse_rmsnorm")
    return n.value


def mk_add_matmul(g, x, w, out, aux, pairs, flags, m, n, k, eps):
    check(lib().mk_add_matmul(g, x, w, out, aux, pairs, flags, m, n, k, eps), "mk_add_matmul")


def mk_add_attention(g, qkv, kc, vc, out, scratch, B, Hq, Hkv, D, capacity, len0, chunk, theta):
    arr = (c_int32 * B)(*[int(v) for v in len0])
    check(lib().mk_add_attention(g, qkv, kc, vc, out, scratch, B, Hq, Hkv, D, capacity, arr, chunk,
                                 float(theta)), "mk_add_attention")


def mk_add_sample(g, pairs, history, B, V, capacity):
    check(lib().mk_add_sample(g, pairs, history, B, V, capacity), "mk_add_sample")


def mk_attention_scratch_rows(g, B, Hkv, len0, chunk) -> int:
    arr = (c_int32 * B)(*[int(v) for v in len0])
    r = c_int64()
    check(lib().mk_attention_scratch_rows(g, B, Hkv, arr, chunk, ctypes.byref(r)), "mk_attention_scratch_rows")
    return r.value


def mk_gemv_tiles(g, n) -> int:
    t = c_int32()
    check(lib().mk_gemv_tiles(g, n, ctypes.byref(t)), "mk_gemv_tiles")
    return t.value


def mk_scratch_size(g, buf) -> int:
    n = c_size_t()
    check(lib().mk_scratch_size(g, buf, ctypes.byref(n)), "mk_scratch_size")
    return n.value


def mk_lower(g):
    check(lib().mk_lower(g), "mk_lower")


def mk_get_tasks(g) -> bytes:
    p, n = c_void_p(), c_size_t()
    check(lib().mk_get_tasks(g, ctypes.byref(p), ctypes.byref(n)), "mk_get_tasks")
    return ctypes.string_at(p, n.value)


def mk_get_edges(g):
    import numpy as np
    p, n = c_void_p(), c_size_t()
    check(lib().mk_get_edges(g, ctypes.byref(p), ctypes.byref(n)), "mk_get_edges")
    return np.frombuffer(ctypes.string_at(p, n.value * 4), dtype=np.uint32).copy()


def mk_get_sync_plan(g, num_tasks: int):
    """(wait_off, wait[:, 2], sig_off, sig, counter_words) as numpy arrays."""
    import numpy as np
    wo, w, so, sg, cw = c_void_p(), c_void_p(), c_void_p(), c_void_p(), c_uint32()
    check(lib().mk_get_sync_plan(g, ctypes.byref(wo), ctypes.byref(w), ctypes.byref(so), ctypes.byref(sg),
                                 ctypes.byref(cw)), "mk_get_sync_plan")
    u32 = lambda ptr, n: np.frombuffer(ctypes.string_at(ptr, n * 4), dtype=np.uint32).copy() if n else \
        np.zeros(0, np.uint32)
    wait_off = u32(wo, num_tasks + 1)
    sig_off = u32(so, num_tasks + 1)
    wait = u32(w, 2 * int(wait_off[-1])).reshape(-1, 2)
    sig = u32(sg, int(sig_off[-1]))
    return wait_off, wait, sig_off, sig, int(cw.value)


def mk_get_ll_plan(g, num_tasks: int, num_bufs: int):
    """(task_ll, buf_ll) as numpy uint8 arrays: the GEMV tasks that read
    tagged pairs, and the buffers whose producers write them."""
    import numpy as np
    tl, bl = c_void_p(), c_void_p()
    check(lib().mk_get_ll_plan(g, ctypes.byref(tl), ctypes.byref(bl)), "mk_get_ll_plan")
    u8 = lambda ptr, n: np.frombuffer(ctypes.string_at(ptr, n), dtype=np.uint8).copy() if n else np.zeros(0, np.uint8)
    return u8(tl, num_tasks), u8(bl, num_bufs)


def mk_get_queues(g):
    import numpy as np
    po, pt, nc = c_void_p(), c_void_p(), c_int()
    check(lib().mk_get_queues(g, ctypes.byref(po), ctypes.byref(pt), ctypes.byref(nc)), "mk_get_queues")
    off = np.frombuffer(ctypes.string_at(po, (nc.value + 1) * 4), dtype=np.int32).copy()
    tasks = np.frombuffer(ctypes.string_at(pt, int(off[-1]) * 4), dtype=np.int32).copy()
    return off, tasks


def mk_upload(g, stream: int):
    check(lib().mk_upload(g, c_void_p(stream)), "mk_upload")


def mk_decode_step(g, stream: int):
    check(lib().mk_decode_step(g, c_void_p(stream)), "mk_decode_step")


def mk_decode_step_ex(g, stream: int, mode: int, trace: int = 0):
    check(lib().mk_decode_step_ex(g, c_void_p(stream), mode, trace), "mk_decode_step_ex")


def mk_decode_step_host(g, stream: int, state_in_ptr: int, tokens_out_ptr: int):
    check(lib().mk_decode_step_host(g, c_void_p(stream), c_void_p(state_in_ptr or None),
                                    c_void_p(tokens_out_ptr or None)), "mk_decode_step_host")


def mk_status(g, stream: int):
    code, task = c_int(), c_int32()
    check(lib().mk_status(g, c_void_p(stream), ctypes.byref(code), ctypes.byref(task)), "mk_status")
    return code.value, task.value


def mk_get_trace(g):
    import numpy as np
    p, n = c_void_p(), c_size_t()
    check(lib().mk_get_trace(g, ctypes.byref(p), ctypes.byref(n)), "mk_get_trace")
    return np.frombuffer(ctypes.string_at(p, n.value * 64), dtype=np.uint64).reshape(-1, 8).copy()


def mk_kernel_info(g):
    s, t, st = c_int(), c_int(), c_int()
    check(lib().mk_kernel_info(g, ctypes.byref(s), ctypes.byref(t), ctypes.byref(st)), "mk_kernel_info")
    return s.value, t.value, st.value


def mk_destroy(g):
    lib().mk_destroy(g)


def mk_gemv_tensor_core_tiles(g) -> int:
    n = c_int()
    check(lib().mk_gemv_tensor_core_tiles(g, ctypes.byref(n)), "mk_gemv_tensor_core_tiles")
    return n.value


def mk_debug_patch_task(g, task: int, desc: bytes):
    assert len(desc) == 64
    buf = ctypes.create_string_buffer(desc, 64)
    check(lib().mk_debug_patch_task(g, task, buf), "mk_debug_patch_task")


def mk_debug_set_epoch(g, stream: int, epoch: int, tag: int):
    check(lib().mk_debug_set_epoch(g, c_void_p(stream), epoch & 0xFFFFFFFF, tag & 0xFFFFFFFF),
          "mk_debug_set_epoch")


def mk_attention_decode_noalloc(stream: int, qkv: int, kcache: int, vcache: int, out: int, B: int, Hq: int,
                                Hkv: int, D: int, capacity: int, pos, len0, chunk: int, theta: float):
    """Device pointers as ints; pos and len0 are sequences of B ints (host)."""
    pa = (c_int32 * B)(*[int(v) for v in pos])
    la = (c_int32 * B)(*[int(v) for v in len0])
    check(lib().mk_attention_decode_noalloc(c_void_p(stream), c_void_p(qkv), c_void_p(kcache), c_void_p(vcache),
                                            c_void_p(out), B, Hq, Hkv, D, capacity, pa, la, chunk, float(theta)),
          "mk_attention_decode_noalloc")


def mk_last_error() -> str:
    return lib().mk_last_error().decode(errors="replace")
