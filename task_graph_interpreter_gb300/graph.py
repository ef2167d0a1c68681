"""Graph builder over libmk: a model is composed by calling ops on a graph
object ("mega kernel initial", 1y33.com, the graph-building part).  matmul
takes the fusions as keywords -- gamma (RMSNorm of its input), residual
(added to its output), silu_mul (SiLU of the gate half times the up half) --
and attention takes the fused qkv activations and the two caches.

Each call registers its output tensor (allocated with PyTorch on the graph's
device) in libmk's append-only buffer table and adds the op; every step of
the computation runs in libmk's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib as L


@dataclass
class Buf:
    """A tensor registered in the buffer table."""
    idx: int
    tensor: torch.Tensor


_DT = {torch.bfloat16: L.MK_BF16, torch.float32: L.MK_F32, torch.int32: L.MK_I32}


class Graph:
    def __init__(self, B: int, device="cuda", num_ctas: int = 0, tiles_target: int = 0,
                 col_align: int = 16, wait_timeout_us: int = 0):
        self.device = torch.device(device)
        self.B = B
        self.h = L.mk_graph_create(num_ctas, tiles_target, col_align, wait_timeout_us)
        self.state = torch.zeros(B, 2, dtype=torch.int32, device=self.device)
        L.mk_set_state(self.h, self.state.data_ptr(), B)
        self.T = 1             # tokens per sequence per step (set_chunk)
        self.tokens = None     # int32 [B, T] input tokens of a chunk step
        self.bufs = []
        self.ops = []        # op records (kind, fields) in call order, for inspection
        self.uploaded = False

    # ------------------------------------------------------------ buffers
    def register(self, t: torch.Tensor, rows: int = None, cols: int = None, dtype: int = None) -> Buf:
        assert t.is_contiguous()
        dt = dtype if dtype is not None else _DT[t.dtype]
        if rows is None:
            rows, cols = (1, t.numel()) if t.dim() == 1 else (t.shape[0], t.numel() // t.shape[0])
        idx = L.mk_add_buffer(self.h, t.data_ptr(), dt, rows, cols)
        b = Buf(idx, t)
        self.bufs.append(b)
        return b

    def _fresh(self, rows, cols, dtype=torch.float32) -> Buf:
        return self.register(torch.empty(rows, cols, dtype=dtype, device=self.device))

    @property
    def rows(self) -> int:
        """Activation rows: B * T (row s * T + t)."""
        return self.B * self.T

    def set_chunk(self, T: int) -> Buf:
        """Make every step a chunk step of T tokens per sequence (a prefill
        chunk or draft tokens to verify).  Returns the int32 [B, T] tokens
        buffer the caller fills before each step with tokens 1..T-1 of each
        sequence (column 0 is the pending token in the state)."""
        self.tokens = self.register(torch.zeros(self.B, T, dtype=torch.int32, device=self.device))
        L.mk_set_chunk(self.h, T, self.tokens.idx)
        self.T = T
        return self.tokens

    # ------------------------------------------------------------ ops
    def embed(self, table: Buf) -> Buf:
        H = table.tensor.shape[-1]
        out = self._fresh(self.rows, H)
        L.mk_add_embed(self.h, table.idx, out.idx, self.B, H)
        self.ops.append(("embed", table.idx, out.idx))
        return out

    def rmsnorm(self, x: Buf, gamma: Buf, residual: Buf = None, eps: float = 1e-5) -> Buf:
        """Standalone RMS norm (one task per sequence): RMSNorm(x [+ residual]) * gamma."""
        M, H = x.tensor.shape
        out = self._fresh(M, H)
        L.mk_add_rmsnorm(self.h, x.idx, gamma.idx, residual.idx if residual is not None else L.MK_NO_BUF,
                         out.idx, self.B, H, eps)
        self.ops.append(("rmsnorm", x.idx, gamma.idx, out.idx))
        return out

    def fuse_rmsnorm(self) -> int:
        """Fold standalone norms into the GEMVs that consume them (before lower)."""
        return L.mk_fuse_rmsnorm(self.h)

    def matmul(self, x: Buf, w: Buf, gamma: Buf = None, residual: Buf = None, silu_mul: bool = False,
               eps: float = 1e-5, argmax: bool = False, out: Buf = None):
        """y = epilogue(W x) tiled over output columns; with argmax=True also
        returns the per-tile (max, index) pairs buffer."""
        B, K = x.tensor.shape
        rows = w.tensor.shape[0]
        n = rows // 2 if silu_mul else rows
        flags = 0
        aux = L.MK_NO_BUF
        if gamma is not None:
            flags |= L.MK_F_RMS_NORM_INPUT
            aux = gamma.idx
        if residual is not None:
            flags |= L.MK_F_ADD_RESIDUAL
            aux = residual.idx
        if silu_mul:
            flags |= L.MK_F_SILU_MUL
        out = out or self._fresh(B, n)
        pairs = None
        if argmax:
            flags |= L.MK_F_ARGMAX_EPI
            T = L.mk_gemv_tiles(self.h, n)
            pairs = self.register(torch.empty(T, B, 2, dtype=torch.int32, device=self.device),
                                  rows=T, cols=B, dtype=L.MK_PAIR)
        L.mk_add_matmul(self.h, x.idx, w.idx, out.idx, aux, pairs.idx if pairs else L.MK_NO_BUF,
                        flags, B, n, K, eps)
        self.ops.append(("matmul", x.idx, w.idx, out.idx, aux, flags))
        return (out, pairs) if argmax else out

    def attention(self, qkv: Buf, kcache: Buf, vcache: Buf, Hq: int, Hkv: int, D: int, capacity: int,
                  len0, chunk: int = 0, rope_theta: float = 5e5) -> Buf:
        G = Hq // Hkv
        rows = L.mk_attention_scratch_rows(self.h, self.B, Hkv, len0, chunk)
        scratch = self._fresh(rows, self.T * G * (D + 2))
        out = self._fresh(self.rows, Hq * D)
        L.mk_add_attention(self.h, qkv.idx, kcache.idx, vcache.idx, out.idx, scratch.idx, self.B, Hq, Hkv, D,
                           capacity, len0, chunk, rope_theta)
        self.ops.append(("attention", qkv.idx, kcache.idx, vcache.idx, out.idx, scratch.idx))
        return out

    def sample(self, pairs: Buf, history: Buf, V: int, capacity: int):
        L.mk_add_sample(self.h, pairs.idx, history.idx, self.B, V, capacity)
        self.ops.append(("sample", pairs.idx, history.idx))

    # ------------------------------------------------------------ lifecycle
    def lower(self):
        L.mk_lower(self.h)

    def tasks_bytes(self) -> bytes:
        return L.mk_get_tasks(self.h)

    def edges(self):
        return L.mk_get_edges(self.h)

    def queues(self):
        return L.mk_get_queues(self.h)

    def upload(self, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        L.mk_upload(self.h, s.cuda_stream)
        self.uploaded = True

    def step(self, mode: int = L.MK_MODE_MEGA, trace: bool = False, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        L.mk_decode_step_ex(self.h, s.cuda_stream, mode, 1 if trace else 0)

    def step_host(self, state_in: torch.Tensor = None, tokens_out: torch.Tensor = None, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        L.mk_decode_step_host(self.h, s.cuda_stream, state_in.data_ptr() if state_in is not None else 0,
                              tokens_out.data_ptr() if tokens_out is not None else 0)

    def status(self, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return L.mk_status(self.h, s.cuda_stream)

    def trace(self):
        return L.mk_get_trace(self.h)

    def chrome_trace(self, path: str = None) -> dict:
        """The last traced step as Chrome trace-event JSON (see trace.py)."""
        from .trace import chrome_trace
        return chrome_trace(self.trace(), self.tasks_bytes(), path)

    def tensor_core_tiles(self) -> int:
        """GEMV tiles that run on the tensor-core path (batch-8 ops)."""
        return L.mk_gemv_tensor_core_tiles(self.h)

    def kernel_info(self):
        return L.mk_kernel_info(self.h)

    def close(self):
        if self.h:
            L.mk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
