"""float64 CPU oracle for ring attention (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product path never does: the CUDA
library fails loudly when its extension is missing instead of falling back
here.  The arithmetic lives in ``ringattn_oracle.c`` (plain C, OpenMP); this
module only compiles it with gcc and marshals arrays through ctypes.

Functions mirror the C entry points; every array is numpy:
  dense(q, k, v, causal, rows=None)          -> out [BH,R,d], lse [BH,R]
  ring(q, k, v, P, causal, layout, rows=None, visits=False)
  block_partial(q_shard, k_block, v_block, P, causal, layout, r, j)
  merge_states(a, b)  (fp32 states in, float64 out)
  merge_inplace(a, b) (float64)
  finalize(m, l, o)
  naive_block_sum(q, k, v, P, causal, layout)
  dense_bwd(q, k, v, dout, causal)          -> dq, dk, dv [BH,N,d]
  dense_bwd_rows(q, k, v, dout, causal, qrows, krows)
  dense_bwd_keys(q, k, v, dout, out, lse, causal, krows) (from the forward's statistics)
  ring_bwd(q, k, v, dout, out, lse, P, causal, layout, visits=False)
q, k, v are bf16 bit patterns (uint16) shaped [BH, N, d] in natural order,
or torch bf16 tensors (converted with ``bf16_bits``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "ringattn_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

LAYOUT_CONTIGUOUS = 0
LAYOUT_STRIPED = 1
LAYOUT_ZIGZAG = 2


def build(source: str = SOURCE, output: str = LIBRARY, force: bool = False) -> str:
    """Compile the C oracle into a shared library with gcc (OpenMP on)."""
    if not force and os.path.exists(output) and os.path.getmtime(output) >= os.path.getmtime(source):
        return output
    tmp = output + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


def _segment_ids(segments, N: int):
    """Document boundaries [0, b1, .., N] (sequence packing) -> the document
    of every position as int64 [N]; None -> None (one document)."""
    if segments is None:
        return None
    b = np.asarray(segments, dtype=np.int64)
    assert b.ndim == 1 and b.size >= 2 and b[0] == 0 and b[-1] == N and np.all(np.diff(b) > 0), "bad boundaries"
    return np.ascontiguousarray(np.repeat(np.arange(b.size - 1, dtype=np.int64), np.diff(b)))


def bf16_bits(t) -> np.ndarray:
    """torch bf16 tensor (any device) or uint16 array -> contiguous uint16 numpy."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch

    assert t.dtype == torch.bfloat16, t.dtype
    return np.ascontiguousarray(t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16))


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64 (for tests)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


_P = ctypes.c_void_p
_L = ctypes.c_long
_I = ctypes.c_int


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes handle on one build of the C oracle."""

    def __init__(self, path: str | None = None, nthreads: int = 0):
        self.path = path or build()
        self.lib = ctypes.CDLL(self.path)
        self.nthreads = nthreads
        L = self.lib
        L.oracle_max_threads.argtypes = [_I]
        L.oracle_max_threads.restype = _I
        L.oracle_position.argtypes = [_I, _L, _I, _I, _L]
        L.oracle_position.restype = _L
        L.oracle_owner.argtypes = [_I, _L, _I, _L, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_long)]
        L.oracle_owner.restype = None
        L.oracle_block_at.argtypes = [_I, _I, _I]
        L.oracle_block_at.restype = _I
        L.oracle_dense_rows.argtypes = [_I, _L, _I, _I, _L, _P, _P, _P, _P, _L, _P, _P, _P, _I]
        L.oracle_dense_rows.restype = _I
        L.oracle_ring_rows.argtypes = [_I, _L, _I, _I, _I, _L, _P, _I, _P, _P, _P, _L, _P, _P, _P, _P, _I]
        L.oracle_ring_rows.restype = _I
        L.oracle_block_partial.argtypes = [_I, _L, _I, _I, _I, _L, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I]
        L.oracle_block_partial.restype = _I
        L.oracle_merge_states.argtypes = [_L, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]
        L.oracle_merge_states.restype = _I
        L.oracle_merge_inplace.argtypes = [_L, _I, _P, _P, _P, _P, _P, _P]
        L.oracle_merge_inplace.restype = _I
        L.oracle_finalize.argtypes = [_L, _I, _P, _P, _P, _P, _P]
        L.oracle_finalize.restype = _I
        L.oracle_naive_block_sum.argtypes = [_I, _L, _I, _I, _I, _L, _P, _I, _P, _P, _P, _P]
        L.oracle_naive_block_sum.restype = _I
        L.oracle_dense_bwd.argtypes = [_I, _L, _I, _I, _L, _P, _P, _P, _P, _P, _P, _P, _P, _I]
        L.oracle_dense_bwd.restype = _I
        L.oracle_dense_bwd_rows.argtypes = [_I, _L, _I, _I, _L, _P, _P, _P, _P, _P, _L, _P, _L, _P, _P, _P, _P, _I]
        L.oracle_dense_bwd_rows.restype = _I
        L.oracle_dense_bwd_keys.argtypes = [_I, _L, _I, _I, _L, _P, _P, _P, _P, _P, _P, _P, _L, _P, _P, _P, _I]
        L.oracle_dense_bwd_keys.restype = _I
        L.oracle_ring_bwd.argtypes = [_I, _L, _I, _I, _I, _L, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I]
        L.oracle_ring_bwd.restype = _I

    # -- small helpers -------------------------------------------------
    def threads(self) -> int:
        return self.lib.oracle_max_threads(self.nthreads)

    def position(self, layout: int, n: int, P: int, r: int, i: int) -> int:
        return self.lib.oracle_position(layout, n, P, r, i)

    def owner(self, layout: int, n: int, P: int, t: int):
        """(shard, local row) holding global position t."""
        r, i = ctypes.c_int(), ctypes.c_long()
        self.lib.oracle_owner(layout, n, P, t, ctypes.byref(r), ctypes.byref(i))
        return r.value, i.value

    def block_at(self, P: int, r: int, s: int) -> int:
        return self.lib.oracle_block_at(P, r, s)

    @staticmethod
    def _qkv(q, k, v):
        q, k, v = bf16_bits(q), bf16_bits(k), bf16_bits(v)
        assert q.ndim == 3 and q.shape == k.shape == v.shape
        return q, k, v

    @staticmethod
    def _rows(rows, N):
        if rows is None:
            return None, N
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < N))
        return r, r.size

    # -- the method ------------------------------------------------------
    def dense(self, q, k, v, causal: bool, rows=None, window: int = 0, segments=None):
        q, k, v = self._qkv(q, k, v)
        BH, N, d = q.shape
        r, R = self._rows(rows, N)
        out = np.empty((BH, R, d), np.float64)
        lse = np.empty((BH, R), np.float64)
        seg = _segment_ids(segments, N)
        rc = self.lib.oracle_dense_rows(BH, N, d, int(causal), int(window), _ptr(seg), _ptr(q), _ptr(k), _ptr(v), R, _ptr(r),
                                        _ptr(out), _ptr(lse), self.nthreads)
        if rc != 0:
            raise RuntimeError(f"oracle_dense_rows failed: {rc}")
        return out, lse

    def ring(self, q, k, v, P: int, causal: bool, layout: int, rows=None, visits: bool = False, window: int = 0, segments=None):
        q, k, v = self._qkv(q, k, v)
        BH, N, d = q.shape
        r, R = self._rows(rows, N)
        out = np.empty((BH, R, d), np.float64)
        lse = np.empty((BH, R), np.float64)
        cnt = np.zeros((BH, N, N), np.int64) if visits else None
        seg = _segment_ids(segments, N)
        rc = self.lib.oracle_ring_rows(BH, N, d, P, int(causal), int(window), _ptr(seg), layout, _ptr(q), _ptr(k), _ptr(v), R,
                                       _ptr(r), _ptr(out), _ptr(lse), _ptr(cnt), self.nthreads)
        if rc != 0:
            raise RuntimeError(f"oracle_ring_rows failed: {rc}")
        return (out, lse, cnt) if visits else (out, lse)

    def block_partial(self, q_shard, k_block, v_block, P: int, causal: bool, layout: int, r: int, j: int,
                      window: int = 0, segments=None):
        q, k, v = self._qkv(q_shard, k_block, v_block)
        BH, n, d = q.shape
        m = np.empty((BH, n), np.float64)
        l = np.empty((BH, n), np.float64)
        o = np.empty((BH, n, d), np.float64)
        seg = _segment_ids(segments, n * P)
        rc = self.lib.oracle_block_partial(BH, n, d, P, int(causal), int(window), _ptr(seg), layout, r, j, _ptr(q), _ptr(k), _ptr(v),
                                           _ptr(m), _ptr(l), _ptr(o), self.nthreads)
        if rc != 0:
            raise RuntimeError(f"oracle_block_partial failed: {rc}")
        return m, l, o

    def merge_states(self, a, b):
        """a, b: (m, l, o) float32 arrays, m/l [rows], o [rows, d]."""
        ma, la, oa = (np.ascontiguousarray(x, np.float32) for x in a)
        mb, lb, ob = (np.ascontiguousarray(x, np.float32) for x in b)
        rows = ma.size
        d = oa.size // max(rows, 1) if rows else 1
        m = np.empty(rows, np.float64)
        l = np.empty(rows, np.float64)
        o = np.empty((rows, d), np.float64)
        rc = self.lib.oracle_merge_states(rows, d, _ptr(ma), _ptr(la), _ptr(oa), _ptr(mb), _ptr(lb), _ptr(ob),
                                          _ptr(m), _ptr(l), _ptr(o))
        if rc != 0:
            raise RuntimeError(f"oracle_merge_states failed: {rc}")
        return m, l, o

    def merge_inplace(self, a, b):
        """a <- merge(a, b) on float64 states (m [rows], l [rows], o [rows, d])."""
        ma, la, oa = a
        mb, lb, ob = (np.ascontiguousarray(x, np.float64) for x in b)
        for x in (ma, la, oa):
            assert x.dtype == np.float64 and x.flags.c_contiguous
        rows = ma.size
        d = oa.size // max(rows, 1) if rows else 1
        rc = self.lib.oracle_merge_inplace(rows, d, _ptr(ma), _ptr(la), _ptr(oa), _ptr(mb), _ptr(lb), _ptr(ob))
        if rc != 0:
            raise RuntimeError(f"oracle_merge_inplace failed: {rc}")

    def finalize(self, m, l, o):
        m = np.ascontiguousarray(m, np.float64)
        l = np.ascontiguousarray(l, np.float64)
        o = np.ascontiguousarray(o, np.float64)
        rows = m.size
        d = o.size // max(rows, 1) if rows else 1
        out = np.empty(o.shape, np.float64)
        lse = np.empty(m.shape, np.float64)
        rc = self.lib.oracle_finalize(rows, d, _ptr(m), _ptr(l), _ptr(o), _ptr(out), _ptr(lse))
        if rc != 0:
            raise RuntimeError(f"oracle_finalize failed: {rc}")
        return out, lse

    def naive_block_sum(self, q, k, v, P: int, causal: bool, layout: int, window: int = 0, segments=None):
        q, k, v = self._qkv(q, k, v)
        BH, N, d = q.shape
        out = np.empty((BH, N, d), np.float64)
        seg = _segment_ids(segments, N)
        rc = self.lib.oracle_naive_block_sum(BH, N, d, P, int(causal), int(window), _ptr(seg), layout, _ptr(q), _ptr(k), _ptr(v),
                                             _ptr(out))
        if rc != 0:
            raise RuntimeError(f"oracle_naive_block_sum failed: {rc}")
        return out

    # -- the backward ------------------------------------------------------
    def dense_bwd(self, q, k, v, dout, causal: bool, window: int = 0, segments=None):
        """dq, dk, dv (float64, [BH][N][d]) by the plain definition."""
        q, k, v = self._qkv(q, k, v)
        do = bf16_bits(dout)
        assert do.shape == q.shape
        BH, N, d = q.shape
        dq, dk, dv = (np.empty((BH, N, d), np.float64) for _ in range(3))
        seg = _segment_ids(segments, N)
        rc = self.lib.oracle_dense_bwd(BH, N, d, int(causal), int(window), _ptr(seg), _ptr(q), _ptr(k), _ptr(v), _ptr(do),
                                       _ptr(dq), _ptr(dk), _ptr(dv), self.nthreads)
        if rc != 0:
            raise RuntimeError(f"oracle_dense_bwd failed: {rc}")
        return dq, dk, dv

    def dense_bwd_rows(self, q, k, v, dout, causal: bool, qrows, krows, window: int = 0, segments=None):
        """dq at query positions qrows ([BH][len(qrows)][d]) and dk, dv at key
        positions krows ([BH][len(krows)][d])."""
        q, k, v = self._qkv(q, k, v)
        do = bf16_bits(dout)
        BH, N, d = q.shape
        qr, nq = self._rows(qrows, N)
        kr, nk = self._rows(krows, N)
        dq = np.empty((BH, nq, d), np.float64)
        dk = np.empty((BH, nk, d), np.float64)
        dv = np.empty((BH, nk, d), np.float64)
        seg = _segment_ids(segments, N)
        rc = self.lib.oracle_dense_bwd_rows(BH, N, d, int(causal), int(window), _ptr(seg), _ptr(q), _ptr(k), _ptr(v), _ptr(do),
                                            nq, _ptr(qr), nk, _ptr(kr), _ptr(dq), _ptr(dk), _ptr(dv), self.nthreads)
        if rc != 0:
            raise RuntimeError(f"oracle_dense_bwd_rows failed: {rc}")
        return dq, dk, dv

    def dense_bwd_keys(self, q, k, v, dout, out, lse, causal: bool, krows, window: int = 0, segments=None):
        """dk, dv at key positions krows ([BH][len(krows)][d]) from the
        forward's out and lse (float64, natural order, e.g. from ``dense``)."""
        q, k, v = self._qkv(q, k, v)
        do = bf16_bits(dout)
        BH, N, d = q.shape
        out = np.ascontiguousarray(out, np.float64).reshape(BH, N, d)
        lse = np.ascontiguousarray(lse, np.float64).reshape(BH, N)
        kr, nk = self._rows(krows, N)
        dk = np.empty((BH, nk, d), np.float64)
        dv = np.empty((BH, nk, d), np.float64)
        seg = _segment_ids(segments, N)
        rc = self.lib.oracle_dense_bwd_keys(BH, N, d, int(causal), int(window), _ptr(seg), _ptr(q), _ptr(k), _ptr(v),
                                            _ptr(do), _ptr(out), _ptr(lse), nk, _ptr(kr), _ptr(dk), _ptr(dv),
                                            self.nthreads)
        if rc != 0:
            raise RuntimeError(f"oracle_dense_bwd_keys failed: {rc}")
        return dk, dv

    def ring_bwd(self, q, k, v, dout, out, lse, P: int, causal: bool, layout: int, visits: bool = False,
                 window: int = 0, segments=None):
        """The ring backward simulation from the forward's out and lse
        (float64, natural order).  Returns dq, dk, dv (and the visit counts)."""
        q, k, v = self._qkv(q, k, v)
        do = bf16_bits(dout)
        BH, N, d = q.shape
        out = np.ascontiguousarray(out, np.float64).reshape(BH, N, d)
        lse = np.ascontiguousarray(lse, np.float64).reshape(BH, N)
        dq, dk, dv = (np.empty((BH, N, d), np.float64) for _ in range(3))
        cnt = np.zeros((BH, N, N), np.int64) if visits else None
        seg = _segment_ids(segments, N)
        rc = self.lib.oracle_ring_bwd(BH, N, d, P, int(causal), int(window), _ptr(seg), layout, _ptr(q), _ptr(k), _ptr(v),
                                      _ptr(do), _ptr(out), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cnt),
                                      self.nthreads)
        if rc != 0:
            raise RuntimeError(f"oracle_ring_bwd failed: {rc}")
        return (dq, dk, dv, cnt) if visits else (dq, dk, dv)


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
