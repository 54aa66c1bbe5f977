"""Ring attention on one GB300: Python face of the C ABI in include/ringattn.h.

The functions below carry the C names and only marshal arguments (torch
tensors -> device pointers, the current torch stream -> cudaStream_t);
every step runs in libringattn.so.  PyTorch provides device memory and
streams.

    ra = RingAttention(B, H, N, d, P, causal=True, layout="striped")
    out, lse = ra.fwd(q, k, v)          # q, k, v: cuda bf16 [B, H, N, d]

Layouts: "contiguous" (shard r holds tokens r*n .. r*n+n-1), "striped"
(token t goes to shard t mod P) or "zigzag" (2P chunks; shard r holds chunk r
and chunk 2P-1-r).
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import (RING_BLOCK_DIAG, RING_BLOCK_FULL, RING_BLOCK_PARTIAL, RING_BLOCK_SKIP,  # noqa: F401
                   RING_LAYOUT_CONTIGUOUS, RING_LAYOUT_STRIPED, RING_LAYOUT_ZIGZAG, RING_OPT_DEBUG_DROP_V_LOADS,
                   RING_OPT_WINDOW, RING_OPT_ROTATION, RING_OPT_TIMING, RING_OPT_BWD_LAP, RING_OPT_FWD_LAP,
                   RING_OPT_WAIT_LIMIT_NS,
                   RingAttnError, RingState)

LAYOUTS = {"contiguous": RING_LAYOUT_CONTIGUOUS, "striped": RING_LAYOUT_STRIPED, "zigzag": RING_LAYOUT_ZIGZAG}


def _layout_id(layout) -> int:
    return LAYOUTS[layout] if isinstance(layout, str) else int(layout)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _state(st) -> RingState:
    m, l, o = st
    return RingState(_ptr(m), _ptr(l), _ptr(o))


# ------------------------------------------------------- C-named wrappers
def ring_attn_create(B: int, H: int, N: int, d: int, P: int, causal: bool, layout) -> int:
    lib = _lib.load()
    h = ctypes.c_void_p()
    _lib.check(lib.ring_attn_create(ctypes.byref(h), B, H, N, d, P, int(bool(causal)), _layout_id(layout)))
    return h.value


def ring_attn_create_gqa(B: int, H: int, Hkv: int, N: int, d: int, P: int, causal: bool, layout) -> int:
    lib = _lib.load()
    h = ctypes.c_void_p()
    _lib.check(lib.ring_attn_create_gqa(ctypes.byref(h), B, H, Hkv, N, d, P, int(bool(causal)), _layout_id(layout)))
    return h.value


def ring_attn_destroy(h: int) -> None:
    _lib.check(_lib.load().ring_attn_destroy(h))


def ring_attn_block_partial(h, r, step, q_shard, k_block, v_block, state, accumulate, stream=None):
    _lib.check(_lib.load().ring_attn_block_partial(h, r, step, _ptr(q_shard), _ptr(k_block), _ptr(v_block),
                                                   _state(state), int(accumulate), _stream(stream)))


def ring_attn_merge(h, state_a, state_b, stream=None):
    _lib.check(_lib.load().ring_attn_merge(h, _state(state_a), _state(state_b), _stream(stream)))


def ring_attn_finalize(h, r, state, out, lse, stream=None):
    _lib.check(_lib.load().ring_attn_finalize(h, r, _state(state), _ptr(out), _ptr(lse), _stream(stream)))


def ring_attn_state_init(h, state, stream=None):
    _lib.check(_lib.load().ring_attn_state_init(h, _state(state), _stream(stream)))


def ring_attn_fwd(h, q, k, v, out, lse, workspace, stream=None):
    _lib.check(_lib.load().ring_attn_fwd(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace),
                                         _stream(stream)))


def ring_attn_bwd(h, q, k, v, out, lse, dout, dq, dk, dv, workspace, stream=None):
    _lib.check(_lib.load().ring_attn_bwd(h, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                                         _ptr(dk), _ptr(dv), _ptr(workspace), _stream(stream)))


def ring_attn_check(h, stream=None):
    _lib.check(_lib.load().ring_attn_check(h, _stream(stream)))


# ------------------------------------------------------------ the object
class RingAttention:
    """One problem shape: plan, workspace and the calls of the C ABI."""

    def __init__(self, B: int, H: int, N: int, d: int, P: int, causal: bool = True, layout="striped",
                 kv_heads: int | None = None):
        """kv_heads: K/V heads for grouped-query attention (H a multiple of it); None = H."""
        self.B, self.H, self.N, self.d, self.P = B, H, N, d, P
        self.Hkv = H if kv_heads is None else int(kv_heads)
        self.causal = bool(causal)
        self.layout = _layout_id(layout)
        self.n = N // P
        if self.Hkv == H:
            self.handle = ring_attn_create(B, H, N, d, P, causal, self.layout)
        else:
            self.handle = ring_attn_create_gqa(B, H, self.Hkv, N, d, P, causal, self.layout)
        self._lib = _lib.load()
        self._workspace = None

    def close(self):
        if self.handle:
            ring_attn_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- planner (host only) -------------------------------------------
    def plan_block(self, r: int, step: int):
        j, cls, delta = ctypes.c_int(), ctypes.c_int(), ctypes.c_longlong()
        _lib.check(self._lib.ring_attn_plan_block(self.handle, r, step, ctypes.byref(j), ctypes.byref(cls),
                                                  ctypes.byref(delta)))
        return j.value, cls.value, delta.value

    def plan_mask(self, r: int, step: int, row: int):
        """(key_limit, delta) of local row `row`: key k allowed iff k < key_limit and k - row <= delta."""
        klim, delta = ctypes.c_longlong(), ctypes.c_longlong()
        _lib.check(self._lib.ring_attn_plan_mask(self.handle, r, step, row, ctypes.byref(klim), ctypes.byref(delta)))
        return klim.value, delta.value

    def plan_key_range(self, r: int, step: int, row: int):
        """(first, last): the block-local keys row `row` of shard r sees at step s (first > last: none)."""
        first, last = ctypes.c_longlong(), ctypes.c_longlong()
        _lib.check(self._lib.ring_attn_plan_key_range(self.handle, r, step, row, ctypes.byref(first),
                                                      ctypes.byref(last)))
        return first.value, last.value

    def shard_work(self):
        pairs = (ctypes.c_longlong * self.P)()
        tiles = (ctypes.c_longlong * self.P)()
        _lib.check(self._lib.ring_attn_shard_work(self.handle, pairs, tiles))
        return list(pairs), list(tiles)

    def step_work(self, step: int):
        pairs, tiles = ctypes.c_longlong(), ctypes.c_longlong()
        _lib.check(self._lib.ring_attn_step_work(self.handle, step, ctypes.byref(pairs), ctypes.byref(tiles)))
        return pairs.value, tiles.value

    def workspace_size(self) -> int:
        n = ctypes.c_size_t()
        _lib.check(self._lib.ring_attn_workspace_size(self.handle, ctypes.byref(n)))
        return n.value

    def set_option(self, option: int, value: int):
        _lib.check(self._lib.ring_attn_set_option(self.handle, option, int(value)))

    def set_segments(self, bounds):
        """Sequence packing: document boundaries [0, b1, .., N] (None or []
        removes them).  A valid length L is [0, L, N]."""
        b = [] if bounds is None else [int(x) for x in bounds]
        arr = (ctypes.c_longlong * max(len(b), 1))(*b)
        _lib.check(self._lib.ring_attn_set_segments(self.handle, arr, max(len(b) - 1, 0)))

    # -- device calls ---------------------------------------------------
    def workspace(self, device=None):
        import torch

        need = self.workspace_size()
        if self._workspace is None or self._workspace.numel() < need:
            self._workspace = torch.empty(need, dtype=torch.uint8, device=device or "cuda")
        return self._workspace

    def bwd_workspace_size(self) -> int:
        n = ctypes.c_size_t()
        _lib.check(self._lib.ring_attn_bwd_workspace_size(self.handle, ctypes.byref(n)))
        return n.value

    def bwd(self, q, k, v, out, lse, dout, dq=None, dk=None, dv=None, stream=None):
        """Gradients of the forward's loss with respect to q, k, v given dout
        (the gradient at out), from the forward's out and lse.  Returns fp32
        dq [B, H, N, d] and dk, dv [B, Hkv, N, d] in natural order."""
        import torch

        shape = (self.B, self.H, self.N, self.d)
        kv_shape = (self.B, self.Hkv, self.N, self.d)
        for t, want in ((q, shape), (k, kv_shape), (v, kv_shape), (dout, shape)):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != want:
                raise ValueError(f"q, dout must be contiguous CUDA bfloat16 tensors {shape}, k, v {kv_shape}")
        if out.dtype != torch.float32 or tuple(out.shape) != shape or not out.is_contiguous():
            raise ValueError(f"out must be a contiguous float32 tensor {shape}")
        if lse.dtype != torch.float32 or tuple(lse.shape) != shape[:3] or not lse.is_contiguous():
            raise ValueError(f"lse must be a contiguous float32 tensor {shape[:3]}")
        dq = torch.empty(shape, dtype=torch.float32, device=q.device) if dq is None else dq
        dk = torch.empty(kv_shape, dtype=torch.float32, device=q.device) if dk is None else dk
        dv = torch.empty(kv_shape, dtype=torch.float32, device=q.device) if dv is None else dv
        need = self.bwd_workspace_size()
        if getattr(self, "_bwd_ws", None) is None or self._bwd_ws.numel() < need:
            self._bwd_ws = torch.empty(need, dtype=torch.uint8, device=q.device)
        ring_attn_bwd(self.handle, q, k, v, out, lse, dout, dq, dk, dv, self._bwd_ws, stream)
        return dq, dk, dv

    def bwd_timing(self):
        """Per-step dK/dV and dQ kernel times (ms) of the last timed backward."""
        dkdv = (ctypes.c_float * self.P)()
        dq = (ctypes.c_float * self.P)()
        prep = ctypes.c_float()
        _lib.check(self._lib.ring_attn_get_bwd_timing(self.handle, dkdv, dq, ctypes.byref(prep)))
        return {"dkdv_ms": list(dkdv), "dq_ms": list(dq), "prep_ms": prep.value}

    def new_state(self, device=None):
        import torch

        dev = device or "cuda"
        rows = (self.B, self.H, self.n)
        return (torch.empty(rows, dtype=torch.float32, device=dev), torch.empty(rows, dtype=torch.float32, device=dev),
                torch.empty(rows + (self.d,), dtype=torch.float32, device=dev))

    def state_init(self, state, stream=None):
        ring_attn_state_init(self.handle, state, stream)

    def block_partial(self, r, step, q_shard, k_block, v_block, state, accumulate, stream=None):
        ring_attn_block_partial(self.handle, r, step, q_shard, k_block, v_block, state, accumulate, stream)

    def merge(self, state_a, state_b, stream=None):
        ring_attn_merge(self.handle, state_a, state_b, stream)

    def finalize(self, r, state, out, lse, stream=None):
        ring_attn_finalize(self.handle, r, state, out, lse, stream)

    def fwd(self, q, k, v, out=None, lse=None, stream=None):
        import torch

        for t, heads in ((q, self.H), (k, self.Hkv), (v, self.Hkv)):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError("q, k, v must be contiguous CUDA bfloat16 tensors [B, H (K/V: Hkv), N, d]")
            if tuple(t.shape) != (self.B, heads, self.N, self.d):
                raise ValueError(f"expected shape {(self.B, heads, self.N, self.d)}, got {tuple(t.shape)}")
        if out is None:
            out = torch.empty((self.B, self.H, self.N, self.d), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((self.B, self.H, self.N), dtype=torch.float32, device=q.device)
        ring_attn_fwd(self.handle, q, k, v, out, lse, self.workspace(q.device), stream)
        return out, lse

    def fwd_host(self, q_host, k_host, v_host, out_host=None, lse_host=None, stream=None):
        """End-to-end call from host memory (ring_attn_fwd_host): pinned CPU
        q, k, v in, pinned CPU out and lse back, the copies overlapped with
        the computation over head groups.  The results are ready once the
        stream (default: the current one) is synchronised."""
        import torch

        shape = (self.B, self.H, self.N, self.d)
        kv_shape = (self.B, self.Hkv, self.N, self.d)
        for t, want in ((q_host, shape), (k_host, kv_shape), (v_host, kv_shape)):
            if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous() or tuple(t.shape) != want:
                raise ValueError(f"q must be a contiguous CPU bfloat16 tensor {shape}, k, v {kv_shape}")
        for t, want in ((out_host, shape), (lse_host, shape[:3])):
            if t is not None and (t.dtype != torch.float32 or t.is_cuda or not t.is_contiguous() or
                                  tuple(t.shape) != want):
                raise ValueError(f"out, lse must be contiguous CPU float32 tensors {shape}, {shape[:3]}")
        if out_host is None:
            out_host = torch.empty(shape, dtype=torch.float32, pin_memory=True)
        if lse_host is None:
            lse_host = torch.empty(shape[:3], dtype=torch.float32, pin_memory=True)
        if stream is None:
            stream = torch.cuda.current_stream()
        _lib.check(self._lib.ring_attn_fwd_host(self.handle, _ptr(q_host), _ptr(k_host), _ptr(v_host),
                                                _ptr(out_host), _ptr(lse_host), _stream(stream)))
        return out_host, lse_host

    def decode(self, q, k, v, out=None, lse=None, stream=None):
        """Split-K/V decode / short-query prefill: q [B, H, Lq, d] bf16 at
        global positions N-Lq .. N-1 over the cache k, v [B, Hkv, N, d]
        (natural order); returns out [B, H, Lq, d] fp32 and lse [B, H, Lq]."""
        import torch

        Lq = int(q.shape[2])
        if q.dtype != torch.bfloat16 or not q.is_cuda or not q.is_contiguous() or \
                tuple(q.shape) != (self.B, self.H, Lq, self.d):
            raise ValueError(f"q must be a contiguous CUDA bfloat16 tensor {(self.B, self.H, 'Lq', self.d)}")
        for t in (k, v):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or \
                    tuple(t.shape) != (self.B, self.Hkv, self.N, self.d):
                raise ValueError(f"k, v must be contiguous CUDA bfloat16 tensors {(self.B, self.Hkv, self.N, self.d)}")
        if out is None:
            out = torch.empty((self.B, self.H, Lq, self.d), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((self.B, self.H, Lq), dtype=torch.float32, device=q.device)
        need = ctypes.c_size_t()
        _lib.check(self._lib.ring_attn_decode_workspace_size(self.handle, Lq, ctypes.byref(need)))
        ws = torch.empty(max(need.value, 256), dtype=torch.uint8, device=q.device)
        _lib.check(self._lib.ring_attn_decode(self.handle, _ptr(q), _ptr(k), _ptr(v), Lq, _ptr(out), _ptr(lse),
                                              _ptr(ws), _stream(stream)))
        return out, lse

    def timing(self):
        """Per-step means over the forwards timed since the previous read
        (RING_OPT_TIMING); reading does not clear them."""
        P = self.P
        k, c, w = (ctypes.c_float * P)(), (ctypes.c_float * P)(), (ctypes.c_float * P)()
        pk = ctypes.c_float()
        _lib.check(self._lib.ring_attn_get_timing(self.handle, k, c, w, ctypes.byref(pk)))
        rw = (ctypes.c_float * P)()
        _lib.check(self._lib.ring_attn_get_release_wait(self.handle, rw))
        return {"kernel_ms": list(k), "copy_ms": list(c), "wait_ms": list(w), "pack_ms": pk.value,
                "release_wait_ms": list(rw)}

    def check(self, stream=None):
        ring_attn_check(self.handle, stream)
