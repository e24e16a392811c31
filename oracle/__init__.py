"""Python access to the plain C oracle (oracle.c).

TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import this module.  The product (the CUDA
library and its binding) never does; the two share no code.

All functions take numpy arrays; indices and offsets are widened to int64 here
(the oracle reads int64 only).  See oracle.c for the definitions and the pages
each follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

INDEX_OOB = 2
BAD_OFFSETS = 4
MODES = {"sum": 0, "mean": 1}
DTYPES = {"f32": 0, "bf16": 1}
RULES = {"adagrad": 0, "sgd": 1}


def build(src: str = SRC, out: str = LIB, extra_flags=()) -> str:
    """Compile oracle.c with gcc into a shared library (skipped when up to date)."""
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src) and not extra_flags:
        return out
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", out, src, "-lm", *extra_flags]
    subprocess.run(cmd, check=True)
    return out


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int


class Oracle:
    """One loaded copy of the oracle library (tests may load altered copies)."""

    def __init__(self, path: str | None = None):
        self.path = path or build()
        lib = ctypes.CDLL(self.path)
        lib.oracle_embbag.argtypes = [_I, _I, _I, _P, _P, _I64, _I64, _P, _P, _I, _P, _P]
        lib.oracle_embbag.restype = _I
        lib.oracle_interact.argtypes = [_I64, _I, _I, _P, _P, _P, _P]
        lib.oracle_interact.restype = None
        lib.oracle_sparse_fwd.argtypes = [_I, _I, _I, _P, _P, _I64, _I64, _P, _P, _I, _P, _P, _P, _P]
        lib.oracle_sparse_fwd.restype = _I
        lib.oracle_interact_bwd.argtypes = [_I64, _I, _I, _P, _P, _P, _P, _P, _P]
        lib.oracle_interact_bwd.restype = None
        lib.oracle_sparse_bwd_adagrad.argtypes = [_I, _I, _P, _P, _I64, _I64, _P, _P, _I, _P, _P, _P, _P,
                                                  _P, ctypes.c_float, ctypes.c_float]
        lib.oracle_sparse_bwd_adagrad.restype = _I
        lib.oracle_sparse_bwd_update.argtypes = [_I, _I, _P, _P, _I64, _I64, _P, _P, _I, _P, _P, _P, _P, _I,
                                                 _P, ctypes.c_float, ctypes.c_float]
        lib.oracle_sparse_bwd_update.restype = _I
        lib.oracle_embbag_bwd_update.argtypes = [_I, _I, _P, _P, _I64, _I64, _P, _P, _I, _P, _I, _P,
                                                 ctypes.c_float, ctypes.c_float]
        lib.oracle_embbag_bwd_update.restype = _I
        lib.oracle_hash_indices.argtypes = [_I, _I64, _I64, _P, _P, _P, _P]
        lib.oracle_hash_indices.restype = _I
        lib.oracle_set_threads.argtypes = [_I]
        lib.oracle_set_threads.restype = _I
        self.lib = lib

    def set_threads(self, n: int) -> int:
        """Threads of the oracle's OpenMP loops (arithmetic unchanged); returns the count in effect."""
        return self.lib.oracle_set_threads(int(n))

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _tables(tables, dtype):
        want = np.uint16 if dtype == "bf16" else np.float32
        tabs = [np.ascontiguousarray(t, dtype=want) for t in tables]
        ptrs = (ctypes.c_void_p * len(tabs))(*[t.ctypes.data for t in tabs])
        return tabs, ptrs

    @staticmethod
    def _csr(num_rows, indices, offsets):
        nr = np.ascontiguousarray(num_rows, dtype=np.int64)
        idx = np.ascontiguousarray(indices, dtype=np.int64)
        off = np.ascontiguousarray(offsets, dtype=np.int64)
        return nr, idx, off

    # -- the method ------------------------------------------------------
    def embbag(self, tables, num_rows, indices, offsets, B, D, mode="sum", dtype="f32", with_abs=False):
        T = len(tables)
        tabs, ptrs = self._tables(tables, dtype)
        nr, idx, off = self._csr(num_rows, indices, offsets)
        pooled = np.empty((B, T, D), dtype=np.float32)
        pabs = np.empty((B, T, D), dtype=np.float64) if with_abs else None
        st = self.lib.oracle_embbag(T, D, DTYPES[dtype], ptrs, nr.ctypes.data, B, idx.size,
                                    idx.ctypes.data, off.ctypes.data, MODES[mode], pooled.ctypes.data,
                                    pabs.ctypes.data if with_abs else None)
        return (pooled, pabs, st) if with_abs else (pooled, st)

    def interact(self, dense, pooled, with_abs=False):
        dense = np.ascontiguousarray(dense, dtype=np.float32)
        pooled = np.ascontiguousarray(pooled, dtype=np.float32)
        B, T, D = pooled.shape
        N = T + 1
        W = D + N * (N - 1) // 2
        out = np.empty((B, W), dtype=np.float32)
        oabs = np.empty((B, W), dtype=np.float64) if with_abs else None
        self.lib.oracle_interact(B, T, D, dense.ctypes.data, pooled.ctypes.data, out.ctypes.data,
                                 oabs.ctypes.data if with_abs else None)
        return (out, oabs) if with_abs else out

    def sparse_fwd(self, tables, num_rows, indices, offsets, dense, mode="sum", dtype="f32",
                   with_abs=False, with_pooled=False):
        dense = np.ascontiguousarray(dense, dtype=np.float32)
        B, D = dense.shape
        T = len(tables)
        N = T + 1
        W = D + N * (N - 1) // 2
        tabs, ptrs = self._tables(tables, dtype)
        nr, idx, off = self._csr(num_rows, indices, offsets)
        out = np.empty((B, W), dtype=np.float32)
        oabs = np.empty((B, W), dtype=np.float64) if with_abs else None
        pooled = np.empty((B, T, D), dtype=np.float32) if with_pooled else None
        st = self.lib.oracle_sparse_fwd(T, D, DTYPES[dtype], ptrs, nr.ctypes.data, B, idx.size,
                                        idx.ctypes.data, off.ctypes.data, MODES[mode], dense.ctypes.data,
                                        out.ctypes.data, oabs.ctypes.data if with_abs else None,
                                        pooled.ctypes.data if with_pooled else None)
        res = {"out": out, "status": st}
        if with_abs:
            res["out_abs"] = oabs
        if with_pooled:
            res["pooled"] = pooled
        return res

    def interact_bwd(self, dense, pooled, grad_out, with_dV=False):
        dense = np.ascontiguousarray(dense, dtype=np.float32)
        pooled = np.ascontiguousarray(pooled, dtype=np.float32)
        grad_out = np.ascontiguousarray(grad_out, dtype=np.float32)
        B, T, D = pooled.shape
        gd = np.empty((B, D), dtype=np.float32)
        gp = np.empty((B, T, D), dtype=np.float32)
        dV = np.empty((B, T + 1, D), dtype=np.float64) if with_dV else None
        self.lib.oracle_interact_bwd(B, T, D, dense.ctypes.data, pooled.ctypes.data, grad_out.ctypes.data,
                                     gd.ctypes.data, gp.ctypes.data, dV.ctypes.data if with_dV else None)
        return (gd, gp, dV) if with_dV else (gd, gp)

    def sparse_bwd_adagrad(self, tables, num_rows, indices, offsets, dense, pooled, grad_out, accum,
                           lr, eps, mode="sum"):
        """Updates `tables` and `accum` (lists of float32 arrays) in place; returns (grad_dense, status)."""
        dense = np.ascontiguousarray(dense, dtype=np.float32)
        pooled = np.ascontiguousarray(pooled, dtype=np.float32)
        grad_out = np.ascontiguousarray(grad_out, dtype=np.float32)
        B, T, D = pooled.shape
        for a in list(tables) + list(accum):
            assert a.dtype == np.float32 and a.flags.c_contiguous
        tptr = (ctypes.c_void_p * T)(*[t.ctypes.data for t in tables])
        aptr = (ctypes.c_void_p * T)(*[a.ctypes.data for a in accum])
        nr, idx, off = self._csr(num_rows, indices, offsets)
        gd = np.empty((B, D), dtype=np.float32)
        st = self.lib.oracle_sparse_bwd_adagrad(T, D, tptr, nr.ctypes.data, B, idx.size, idx.ctypes.data,
                                                off.ctypes.data, MODES[mode], dense.ctypes.data,
                                                pooled.ctypes.data, grad_out.ctypes.data, gd.ctypes.data,
                                                aptr, ctypes.c_float(lr), ctypes.c_float(eps))
        return gd, st


    def sparse_bwd_update(self, tables, num_rows, indices, offsets, dense, pooled, grad_out, rule, lr, eps=0.0,
                          accum=None, mode="sum"):
        """The training step with update rule "adagrad" (needs accum) or "sgd"; tables (and accum) are
        updated in place; returns (grad_dense, status)."""
        dense = np.ascontiguousarray(dense, dtype=np.float32)
        pooled = np.ascontiguousarray(pooled, dtype=np.float32)
        grad_out = np.ascontiguousarray(grad_out, dtype=np.float32)
        B, T, D = pooled.shape
        tptr, aptr = self._rows_and_accum(tables, accum, rule, T)
        nr, idx, off = self._csr(num_rows, indices, offsets)
        gd = np.empty((B, D), dtype=np.float32)
        st = self.lib.oracle_sparse_bwd_update(T, D, tptr, nr.ctypes.data, B, idx.size, idx.ctypes.data,
                                               off.ctypes.data, MODES[mode], dense.ctypes.data, pooled.ctypes.data,
                                               grad_out.ctypes.data, gd.ctypes.data, RULES[rule], aptr,
                                               ctypes.c_float(lr), ctypes.c_float(eps))
        return gd, st

    def embbag_bwd_update(self, tables, num_rows, indices, offsets, grad_pooled, rule, lr, eps=0.0, accum=None,
                          mode="sum"):
        """Per-row gradient sums from grad_pooled [B, T, D] and one update of each touched row (in place);
        returns the status."""
        grad_pooled = np.ascontiguousarray(grad_pooled, dtype=np.float32)
        B, T, D = grad_pooled.shape
        tptr, aptr = self._rows_and_accum(tables, accum, rule, T)
        nr, idx, off = self._csr(num_rows, indices, offsets)
        return self.lib.oracle_embbag_bwd_update(T, D, tptr, nr.ctypes.data, B, idx.size, idx.ctypes.data,
                                                 off.ctypes.data, MODES[mode], grad_pooled.ctypes.data,
                                                 RULES[rule], aptr, ctypes.c_float(lr), ctypes.c_float(eps))

    def hash_indices(self, num_rows, raw_ids, offsets, B):
        """rows[p] = raw_ids[p] (unsigned 64-bit) mod V_t of the table holding position p; (rows, status)."""
        raw = np.ascontiguousarray(raw_ids).view(np.uint64) if np.asarray(raw_ids).dtype in (np.int64, np.uint64) \
            else np.ascontiguousarray(raw_ids, dtype=np.uint64)
        nr = np.ascontiguousarray(num_rows, dtype=np.int64)
        off = np.ascontiguousarray(offsets, dtype=np.int64)
        rows = np.empty(raw.size, dtype=np.int64)
        st = self.lib.oracle_hash_indices(nr.size, B, raw.size, nr.ctypes.data, raw.ctypes.data, off.ctypes.data,
                                          rows.ctypes.data)
        return rows, st

    @staticmethod
    def _rows_and_accum(tables, accum, rule, T):
        for a in list(tables) + list(accum or []):
            assert a.dtype == np.float32 and a.flags.c_contiguous
        if rule == "adagrad":
            assert accum is not None and len(accum) == T
        tptr = (ctypes.c_void_p * T)(*[t.ctypes.data for t in tables])
        aptr = (ctypes.c_void_p * T)(*[a.ctypes.data for a in accum]) if accum is not None else None
        return tptr, aptr


_default = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default

