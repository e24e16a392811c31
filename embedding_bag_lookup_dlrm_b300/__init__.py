"""Python binding of the DLRM sparse-path C ABI (libdlrm_sparse.so, sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  torch tensors provide device memory and streams.
The functions carry the names of the C entry points declared in
include/dlrm_sparse.h; see that header for layouts and semantics.

There is no fallback: if the CUDA library is missing or was not built, every
call raises RuntimeError.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdlrm_sparse.so")

DLRM_OK = 0
DLRM_ERR_INVALID_ARG = 1
DLRM_ERR_INDEX_OOB = 2
DLRM_ERR_BAD_OFFSETS = 4
DLRM_ERR_TIMEOUT = 8
DLRM_ERR_CUDA = 16
DLRM_ERR_UNSUPPORTED = 32
DLRM_ERR_CAPACITY = 64
MAX_TABLES = 128
STATIC_SCRATCH_BYTES = 32 << 20  # DLRM_STATIC_SCRATCH_BYTES

_MODES = {"sum": 0, "mean": 1}
_DTYPES = {torch.float32: 0, torch.bfloat16: 1}
_ITYPES = {torch.int32: 0, torch.int64: 1}

C_SYMBOLS = ("dlrm_embbag_fwd", "dlrm_interact_fwd", "dlrm_sparse_fwd", "dlrm_sparse_fwd_host",
             "dlrm_sparse_bwd_workspace_size", "dlrm_sparse_bwd_adagrad", "dlrm_sparse_bwd_update",
             "dlrm_sparse_bwd_sort", "dlrm_sparse_bwd_update_sorted",
             "dlrm_interact_bwd", "dlrm_embbag_bwd_workspace_size", "dlrm_embbag_bwd_update", "dlrm_hash_indices",
             "dlrm_pooled_exchange", "dlrm_tier_init", "dlrm_tier_cache_fill", "dlrm_tier_stage",
             "dlrm_fc_fwd_workspace_size", "dlrm_fc_fwd", "dlrm_fc_bwd_workspace_size", "dlrm_fc_bwd_sgd",
             "dlrm_head_bce_workspace_size",
             "dlrm_head_bce_sgd",
             "dlrm_sparse_bwd_adagrad_static", "dlrm_status_string", "dlrm_abi_version")
_RULES = {"adagrad": 0, "sgd": 1}


class DlrmTables(ctypes.Structure):
    _fields_ = [("num_tables", ctypes.c_int32), ("dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("data", ctypes.POINTER(ctypes.c_void_p)), ("num_rows", ctypes.POINTER(ctypes.c_int64))]


class DlrmBags(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("nnz", ctypes.c_int64), ("index_type", ctypes.c_int32),
                ("indices", ctypes.c_void_p), ("offsets", ctypes.c_void_p)]


class DlrmTieredTables(ctypes.Structure):
    _fields_ = [("num_tables", ctypes.c_int32), ("dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("host_data", ctypes.POINTER(ctypes.c_void_p)), ("num_rows", ctypes.POINTER(ctypes.c_int64)),
                ("slot_of", ctypes.POINTER(ctypes.c_void_p)), ("slot_row", ctypes.POINTER(ctypes.c_void_p)),
                ("cache", ctypes.POINTER(ctypes.c_void_p)), ("cache_rows", ctypes.POINTER(ctypes.c_int64)),
                ("stage_rows", ctypes.POINTER(ctypes.c_int64))]


class DlrmUpdate(ctypes.Structure):
    _fields_ = [("rule", ctypes.c_int32), ("lr", ctypes.c_float), ("eps", ctypes.c_float),
                ("accum", ctypes.POINTER(ctypes.c_void_p))]


class DlrmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdlrm_sparse.so (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} not found: build it with embedding_bag_lookup_dlrm_b300/build.py "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    P, T, B = ctypes.c_void_p, ctypes.POINTER(DlrmTables), ctypes.POINTER(DlrmBags)
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    sig = {
        "dlrm_embbag_fwd": ([T, B, i32, P, P, P], i32),
        "dlrm_interact_fwd": ([P, P, i64, i32, i32, P, P], i32),
        "dlrm_sparse_fwd": ([T, B, i32, P, P, P, P, P], i32),
        "dlrm_sparse_fwd_host": ([T, B, i32, P, P, P, P, P, P, P, P], i32),
        "dlrm_sparse_bwd_workspace_size": ([T, B, ctypes.POINTER(ctypes.c_size_t)], i32),
        "dlrm_sparse_bwd_adagrad": ([T, B, i32, P, P, P, P, ctypes.POINTER(ctypes.c_void_p), ctypes.c_float,
                                     ctypes.c_float, P, ctypes.c_size_t, P, P, P], i32),
        "dlrm_sparse_bwd_update": ([T, B, i32, P, P, P, P, ctypes.POINTER(DlrmUpdate), P, ctypes.c_size_t, P, P,
                                    P], i32),
        "dlrm_sparse_bwd_sort": ([T, B, P, ctypes.c_size_t, P, P], i32),
        "dlrm_sparse_bwd_update_sorted": ([T, B, i32, P, P, P, P, ctypes.POINTER(DlrmUpdate), P, ctypes.c_size_t,
                                           P, P, P, P], i32),
        "dlrm_interact_bwd": ([P, P, P, i64, i32, i32, P, P, P], i32),
        "dlrm_embbag_bwd_workspace_size": ([T, B, i32, ctypes.POINTER(ctypes.c_size_t)], i32),
        "dlrm_embbag_bwd_update": ([T, B, i32, P, ctypes.POINTER(DlrmUpdate), P, ctypes.c_size_t, P, P, P], i32),
        "dlrm_hash_indices": ([ctypes.POINTER(ctypes.c_int64), i32, i64, i64, P, P, i32, P, P, P], i32),
        "dlrm_pooled_exchange": ([P, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), i32, P], i32),
        "dlrm_fc_fwd_workspace_size": ([i64, i32, i32, ctypes.POINTER(ctypes.c_size_t)], i32),
        "dlrm_fc_fwd": ([P, P, P, i64, i32, i32, i32, P, P, ctypes.c_size_t, P, P], i32),
        "dlrm_fc_bwd_workspace_size": ([i64, i32, i32, ctypes.POINTER(ctypes.c_size_t)], i32),
        "dlrm_fc_bwd_sgd": ([P, P, P, P, P, i64, i32, i32, i32, ctypes.c_float, P, P, ctypes.c_size_t, P, P], i32),
        "dlrm_head_bce_workspace_size": ([i64, i32, ctypes.POINTER(ctypes.c_size_t)], i32),
        "dlrm_head_bce_sgd": ([P, P, P, P, i64, i32, ctypes.c_float, P, P, P, P, ctypes.c_size_t, P], i32),
        "dlrm_tier_init": ([ctypes.POINTER(DlrmTieredTables), P], i32),
        "dlrm_tier_cache_fill": ([ctypes.POINTER(DlrmTieredTables), i32, P, i64, P, P], i32),
        "dlrm_tier_stage": ([ctypes.POINTER(DlrmTieredTables), B, P, P, P, P], i32),
        "dlrm_sparse_bwd_adagrad_static": ([T, B, i32, P, P, P, P, ctypes.POINTER(ctypes.c_void_p),
                                            ctypes.c_float, ctypes.c_float, P, P], i32),
        "dlrm_status_string": ([i32], ctypes.c_char_p),
        "dlrm_abi_version": ([], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().dlrm_status_string(status).decode()
    except RuntimeError:
        return f"status {status}"


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _stream_ptr(stream, device) -> int:
    """The stream to queue on: the given one, else the current stream of `device`."""
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _device(*tensors) -> torch.device:
    """The one CUDA device all given tensors live on (the C library runs on the current device, so every
    call is made with this device current)."""
    devs = {t.device for t in tensors if isinstance(t, torch.Tensor) and t.is_cuda}
    if len(devs) != 1:
        raise ValueError(f"tensors must live on one CUDA device, got {sorted(map(str, devs))}")
    return devs.pop()


def _check_cuda(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


class Tables:
    """A C view (dlrm_tables) of a list of 2-D CUDA tensors of equal width and dtype."""

    def __init__(self, tables):
        tables = list(tables)
        if not tables:
            raise ValueError("need at least one table")
        D, dt = tables[0].shape[1], tables[0].dtype
        for i, t in enumerate(tables):
            _check_cuda(t, f"tables[{i}]")
            if t.dim() != 2 or t.shape[1] != D or t.dtype != dt:
                raise ValueError("tables must be 2-D with equal width and dtype")
        if dt not in _DTYPES:
            raise ValueError(f"unsupported table dtype {dt}")
        self.tensors = tables
        self._ptrs = (ctypes.c_void_p * len(tables))(*[t.data_ptr() for t in tables])
        self._rows = (ctypes.c_int64 * len(tables))(*[t.shape[0] for t in tables])
        self.c = DlrmTables(len(tables), D, _DTYPES[dt], self._ptrs, self._rows)
        self.T, self.D = len(tables), D


def _bags(indices, offsets, B, device=True) -> DlrmBags:
    if indices.dtype != offsets.dtype or indices.dtype not in _ITYPES:
        raise ValueError("indices and offsets must share dtype int32 or int64")
    if device:
        _check_cuda(indices, "indices")
        _check_cuda(offsets, "offsets")
    return DlrmBags(B, indices.numel(), _ITYPES[indices.dtype], indices.data_ptr() if indices.numel() else None,
                    offsets.data_ptr())


def _batch(offsets, T):
    n = offsets.numel() - 1
    if n < T or n % T:
        raise ValueError(f"offsets must hold T*B+1 entries (T={T}), got {offsets.numel()}")
    return n // T


def _raise(st, where):
    if st != DLRM_OK:
        raise DlrmError(st, where)


def _tables(tables):
    return tables if isinstance(tables, Tables) else Tables(tables)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def dlrm_embbag_fwd(tables, indices, offsets, mode="sum", pooled=None, status=None, stream=None):
    """Pooled embeddings [B, T, D] fp32 of CSR bags (table-major offsets of T*B+1 entries)."""
    lib = load_library()
    tb = _tables(tables)
    B = _batch(offsets, tb.T)
    if pooled is None:
        pooled = torch.empty((B, tb.T, tb.D), dtype=torch.float32, device=indices.device)
    _check_cuda(pooled, "pooled", torch.float32)
    bags = _bags(indices, offsets, B)
    dev = _device(*tb.tensors, indices, offsets, pooled, status)
    with torch.cuda.device(dev):
        st = lib.dlrm_embbag_fwd(ctypes.byref(tb.c), ctypes.byref(bags), _MODES[mode], pooled.data_ptr(),
                                 status.data_ptr() if status is not None else None, _stream_ptr(stream, dev))
    _raise(st, "dlrm_embbag_fwd")
    return pooled


def dlrm_interact_fwd(dense, pooled, out=None, stream=None):
    """[x, strict upper triangle of V V^T] per sample, V = [x; pooled]."""
    lib = load_library()
    _check_cuda(dense, "dense", torch.float32)
    _check_cuda(pooled, "pooled", torch.float32)
    B, T, D = pooled.shape
    N = T + 1
    if out is None:
        out = torch.empty((B, D + N * (N - 1) // 2), dtype=torch.float32, device=dense.device)
    _check_cuda(out, "out", torch.float32)
    dev = _device(dense, pooled, out)
    with torch.cuda.device(dev):
        st = lib.dlrm_interact_fwd(dense.data_ptr(), pooled.data_ptr(), B, T, D, out.data_ptr(),
                                   _stream_ptr(stream, dev))
    _raise(st, "dlrm_interact_fwd")
    return out


def dlrm_sparse_fwd(tables, indices, offsets, dense, mode="sum", out=None, pooled_save=None, status=None,
                    stream=None):
    """Fused lookup + pooling + interaction: out [B, D + N(N-1)/2] fp32."""
    lib = load_library()
    tb = _tables(tables)
    B = _batch(offsets, tb.T)
    _check_cuda(dense, "dense", torch.float32)
    N = tb.T + 1
    if out is None:
        out = torch.empty((B, tb.D + N * (N - 1) // 2), dtype=torch.float32, device=dense.device)
    _check_cuda(out, "out", torch.float32)
    if pooled_save is not None:
        _check_cuda(pooled_save, "pooled_save", torch.float32)
    bags = _bags(indices, offsets, B)
    dev = _device(*tb.tensors, indices, offsets, dense, out, pooled_save, status)
    with torch.cuda.device(dev):
        st = lib.dlrm_sparse_fwd(ctypes.byref(tb.c), ctypes.byref(bags), _MODES[mode], dense.data_ptr(),
                                 out.data_ptr(), pooled_save.data_ptr() if pooled_save is not None else None,
                                 status.data_ptr() if status is not None else None, _stream_ptr(stream, dev))
    _raise(st, "dlrm_sparse_fwd")
    return out


class HostStaging:
    """Device staging buffers for dlrm_sparse_fwd_host (allocated once by the caller)."""

    def __init__(self, B, T, D, nnz, index_dtype=torch.int32, device="cuda"):
        N = T + 1
        self.indices = torch.empty(max(nnz, 1), dtype=index_dtype, device=device)
        self.offsets = torch.empty(T * B + 1, dtype=index_dtype, device=device)
        self.dense = torch.empty((B, D), dtype=torch.float32, device=device)
        self.out = torch.empty((B, D + N * (N - 1) // 2), dtype=torch.float32, device=device)


def dlrm_sparse_fwd_host(tables, indices_host, offsets_host, dense_host, out_host, staging: HostStaging,
                         mode="sum", status=None, stream=None):
    """The fused forward fed from host (ideally pinned) tensors; the copies and the
    kernel are queued on `stream`; out_host is valid after the stream syncs."""
    lib = load_library()
    tb = _tables(tables)
    B = _batch(offsets_host, tb.T)
    for name, t in (("indices_host", indices_host), ("offsets_host", offsets_host), ("dense_host", dense_host),
                    ("out_host", out_host)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    if staging.indices.numel() < indices_host.numel() or staging.offsets.numel() < offsets_host.numel():
        raise ValueError("staging buffers too small")
    bags = _bags(indices_host, offsets_host, B, device=False)
    dev = _device(*tb.tensors, staging.indices, staging.offsets, staging.dense, staging.out, status)
    with torch.cuda.device(dev):
        st = lib.dlrm_sparse_fwd_host(ctypes.byref(tb.c), ctypes.byref(bags), _MODES[mode], dense_host.data_ptr(),
                                      out_host.data_ptr(), staging.indices.data_ptr(), staging.offsets.data_ptr(),
                                      staging.dense.data_ptr(), staging.out.data_ptr(),
                                      status.data_ptr() if status is not None else None, _stream_ptr(stream, dev))
    _raise(st, "dlrm_sparse_fwd_host")
    return out_host


def dlrm_sparse_bwd_workspace_size(tables, indices, offsets) -> int:
    lib = load_library()
    tb = _tables(tables)
    B = _batch(offsets, tb.T)
    bags = _bags(indices, offsets, B, device=False)
    n = ctypes.c_size_t(0)
    _raise(lib.dlrm_sparse_bwd_workspace_size(ctypes.byref(tb.c), ctypes.byref(bags), ctypes.byref(n)),
           "dlrm_sparse_bwd_workspace_size")
    return int(n.value)


def dlrm_sparse_bwd_adagrad(tables, accum, indices, offsets, dense, pooled_saved, grad_out, lr, eps, mode="sum",
                            grad_dense=None, workspace=None, status=None, stream=None, side_stream=None):
    """One training step of the sparse path; tables and accum are updated in place.
    side_stream (optional, same device): runs the lookup-key build and sort beside the
    interaction backward.  Returns grad_dense [B, D]."""
    lib = load_library()
    tb = _tables(tables)
    B = _batch(offsets, tb.T)
    if len(accum) != tb.T:
        raise ValueError("one accumulator per table")
    for i, a in enumerate(accum):
        _check_cuda(a, f"accum[{i}]", torch.float32)
        if a.numel() != tb.tensors[i].shape[0]:
            raise ValueError(f"accum[{i}] must hold one value per row")
    for name, t in (("dense", dense), ("pooled_saved", pooled_saved), ("grad_out", grad_out)):
        _check_cuda(t, name, torch.float32)
    if grad_dense is None:
        grad_dense = torch.empty((B, tb.D), dtype=torch.float32, device=dense.device)
    _check_cuda(grad_dense, "grad_dense", torch.float32)
    need = dlrm_sparse_bwd_workspace_size(tb, indices, offsets)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dense.device)
    _check_cuda(workspace, "workspace")
    acc_ptrs = (ctypes.c_void_p * tb.T)(*[a.data_ptr() for a in accum])
    bags = _bags(indices, offsets, B)
    dev = _device(*tb.tensors, *accum, indices, offsets, dense, pooled_saved, grad_out, grad_dense, workspace,
                  status)
    with torch.cuda.device(dev):
        st = lib.dlrm_sparse_bwd_adagrad(ctypes.byref(tb.c), ctypes.byref(bags), _MODES[mode], dense.data_ptr(),
                                         pooled_saved.data_ptr(), grad_out.data_ptr(), grad_dense.data_ptr(),
                                         acc_ptrs, float(lr), float(eps), workspace.data_ptr(), workspace.numel(),
                                         status.data_ptr() if status is not None else None,
                                         _stream_ptr(stream, dev),
                                         side_stream.cuda_stream if side_stream is not None else None)
    _raise(st, "dlrm_sparse_bwd_adagrad")
    return grad_dense


def dlrm_sparse_bwd_adagrad_static(tables, accum, indices, offsets, dense, pooled_saved, grad_out, lr, eps,
                                   mode="sum", grad_dense=None, status=None, stream=None):
    """dlrm_sparse_bwd_adagrad without a workspace: the C library uses its own
    fixed scratch of STATIC_SCRATCH_BYTES per device, for callers that cannot
    allocate device memory.  Pass grad_dense to keep this call free of
    allocations on the Python side too.  Calls that overlap on the GPU share
    the scratch and race.  Raises ValueError when the batch needs more
    scratch than the fixed array holds."""
    lib = load_library()
    tb = _tables(tables)
    B = _batch(offsets, tb.T)
    if len(accum) != tb.T:
        raise ValueError("one accumulator per table")
    for i, a in enumerate(accum):
        _check_cuda(a, f"accum[{i}]", torch.float32)
        if a.numel() != tb.tensors[i].shape[0]:
            raise ValueError(f"accum[{i}] must hold one value per row")
    for name, t in (("dense", dense), ("pooled_saved", pooled_saved), ("grad_out", grad_out)):
        _check_cuda(t, name, torch.float32)
    need = dlrm_sparse_bwd_workspace_size(tb, indices, offsets)
    if need > STATIC_SCRATCH_BYTES:
        raise ValueError(f"batch needs {need} bytes of scratch; the fixed scratch holds {STATIC_SCRATCH_BYTES}")
    if grad_dense is None:
        grad_dense = torch.empty((B, tb.D), dtype=torch.float32, device=dense.device)
    _check_cuda(grad_dense, "grad_dense", torch.float32)
    acc_ptrs = (ctypes.c_void_p * tb.T)(*[a.data_ptr() for a in accum])
    bags = _bags(indices, offsets, B)
    dev = _device(*tb.tensors, *accum, indices, offsets, dense, pooled_saved, grad_out, grad_dense, status)
    with torch.cuda.device(dev):
        st = lib.dlrm_sparse_bwd_adagrad_static(ctypes.byref(tb.c), ctypes.byref(bags), _MODES[mode],
                                                dense.data_ptr(), pooled_saved.data_ptr(), grad_out.data_ptr(),
                                                grad_dense.data_ptr(), acc_ptrs, float(lr), float(eps),
                                                status.data_ptr() if status is not None else None,
                                                _stream_ptr(stream, dev))
    _raise(st, "dlrm_sparse_bwd_adagrad_static")
    return grad_dense


def _update(tb, rule, lr, eps, accum):
    """The C update block (and the pointer array it refers to, kept alive by the caller)."""
    if rule not in _RULES:
        raise ValueError(f"unknown update rule {rule!r}")
    ptrs = None
    if rule == "adagrad":
        if accum is None or len(accum) != tb.T:
            raise ValueError("Adagrad needs one accumulator per table")
        for i, a in enumerate(accum):
            _check_cuda(a, f"accum[{i}]", torch.float32)
            if a.numel() != tb.tensors[i].shape[0]:
                raise ValueError(f"accum[{i}] must hold one value per row")
        ptrs = (ctypes.c_void_p * tb.T)(*[a.data_ptr() for a in accum])
    return DlrmUpdate(_RULES[rule], float(lr), float(eps), ptrs), ptrs


def dlrm_sparse_bwd_update(tables, indices, offsets, dense, pooled_saved, grad_out, rule, lr, eps=0.0, accum=None,
                           mode="sum", grad_dense=None, workspace=None, status=None, stream=None, side_stream=None):
    """The training step with update rule "adagrad" (accum required) or "sgd"; tables (and accum)
    are updated in place.  Returns grad_dense [B, D]."""
    lib = load_library()
    tb = _tables(tables)
    B = _batch(offsets, tb.T)
    for name, t in (("dense", dense), ("pooled_saved", pooled_saved), ("grad_out", grad_out)):
        _check_cuda(t, name, torch.float32)
    upd, _keep = _update(tb, rule, lr, eps, accum)
    if grad_dense is None:
        grad_dense = torch.empty((B, tb.D), dtype=torch.float32, device=dense.device)
    _check_cuda(grad_dense, "grad_dense", torch.float32)
    if workspace is None:
        workspace = torch.empty(max(dlrm_sparse_bwd_workspace_size(tb, indices, offsets), 16), dtype=torch.uint8,
                                device=dense.device)
    _check_cuda(workspace, "workspace")
    bags = _bags(indices, offsets, B)
    dev = _device(*tb.tensors, *(accum or []), indices, offsets, dense, pooled_saved, grad_out, grad_dense,
                  workspace, status)
    with torch.cuda.device(dev):
        st = lib.dlrm_sparse_bwd_update(ctypes.byref(tb.c), ctypes.byref(bags), _MODES[mode], dense.data_ptr(),
                                        pooled_saved.data_ptr(), grad_out.data_ptr(), grad_dense.data_ptr(),
                                        ctypes.byref(upd), workspace.data_ptr(), workspace.numel(),
                                        status.data_ptr() if status is not None else None, _stream_ptr(stream, dev),
                                        side_stream.cuda_stream if side_stream is not None else None)
    _raise(st, "dlrm_sparse_bwd_update")
    return grad_dense


def dlrm_sparse_bwd_sort(tables, indices, offsets, workspace, status=None, stream=None):
    """The lookup keys of the bags sorted by row into `workspace` (a training-step workspace of at least
    dlrm_sparse_bwd_workspace_size bytes), for a later dlrm_sparse_bwd_update_sorted on the same bags."""
    lib = load_library()
    tb = _tables(tables)
    B = _batch(offsets, tb.T)
    _check_cuda(workspace, "workspace")
    bags = _bags(indices, offsets, B)
    dev = _device(*tb.tensors, indices, offsets, workspace, status)
    with torch.cuda.device(dev):
        st = lib.dlrm_sparse_bwd_sort(ctypes.byref(tb.c), ctypes.byref(bags), workspace.data_ptr(), workspace.numel(),
                                      status.data_ptr() if status is not None else None, _stream_ptr(stream, dev))
    _raise(st, "dlrm_sparse_bwd_sort")
    return workspace


def dlrm_sparse_bwd_update_sorted(tables, indices, offsets, dense, pooled_saved, grad_out, rule, lr, eps=0.0,
                                  accum=None, mode="sum", grad_dense=None, workspace=None, status=None, sorted=None,
                                  grad_ready=None, stream=None):
    """dlrm_sparse_bwd_update on a workspace that dlrm_sparse_bwd_sort filled for the same bags (queued
    before this call).  sorted: a torch.cuda.Event recorded after the sort on its stream, waited for before
    the per-row sums only (None: the caller ordered the sort before this call).  grad_ready: a
    torch.cuda.Event the call records once grad_dense is queued, before the per-row sums.  Returns
    grad_dense [B, D]."""
    lib = load_library()
    tb = _tables(tables)
    B = _batch(offsets, tb.T)
    for name, t in (("dense", dense), ("pooled_saved", pooled_saved), ("grad_out", grad_out)):
        _check_cuda(t, name, torch.float32)
    upd, _keep = _update(tb, rule, lr, eps, accum)
    if grad_dense is None:
        grad_dense = torch.empty((B, tb.D), dtype=torch.float32, device=dense.device)
    _check_cuda(grad_dense, "grad_dense", torch.float32)
    _check_cuda(workspace, "workspace")
    bags = _bags(indices, offsets, B)
    dev = _device(*tb.tensors, *(accum or []), indices, offsets, dense, pooled_saved, grad_out, grad_dense,
                  workspace, status)
    with torch.cuda.device(dev):
        st = lib.dlrm_sparse_bwd_update_sorted(ctypes.byref(tb.c), ctypes.byref(bags), _MODES[mode],
                                               dense.data_ptr(), pooled_saved.data_ptr(), grad_out.data_ptr(),
                                               grad_dense.data_ptr(), ctypes.byref(upd), workspace.data_ptr(),
                                               workspace.numel(), status.data_ptr() if status is not None else None,
                                               sorted.cuda_event if sorted is not None else None,
                                               grad_ready.cuda_event if grad_ready is not None else None,
                                               _stream_ptr(stream, dev))
    _raise(st, "dlrm_sparse_bwd_update_sorted")
    return grad_dense


def dlrm_interact_bwd(dense, pooled, grad_out, grad_dense=None, grad_pooled=None, stream=None):
    """The interaction backward alone: (grad_dense [B, D], grad_pooled [B, T, D]); no bag lengths applied."""
    lib = load_library()
    for name, t in (("dense", dense), ("pooled", pooled), ("grad_out", grad_out)):
        _check_cuda(t, name, torch.float32)
    B, T, D = pooled.shape
    if grad_dense is None:
        grad_dense = torch.empty((B, D), dtype=torch.float32, device=dense.device)
    if grad_pooled is None:
        grad_pooled = torch.empty((B, T, D), dtype=torch.float32, device=dense.device)
    _check_cuda(grad_dense, "grad_dense", torch.float32)
    _check_cuda(grad_pooled, "grad_pooled", torch.float32)
    dev = _device(dense, pooled, grad_out, grad_dense, grad_pooled)
    with torch.cuda.device(dev):
        st = lib.dlrm_interact_bwd(dense.data_ptr(), pooled.data_ptr(), grad_out.data_ptr(), B, T, D,
                                   grad_dense.data_ptr(), grad_pooled.data_ptr(), _stream_ptr(stream, dev))
    _raise(st, "dlrm_interact_bwd")
    return grad_dense, grad_pooled


def dlrm_embbag_bwd_workspace_size(tables, indices, offsets, mode="sum") -> int:
    lib = load_library()
    tb = _tables(tables)
    B = _batch(offsets, tb.T)
    bags = _bags(indices, offsets, B, device=False)
    n = ctypes.c_size_t(0)
    _raise(lib.dlrm_embbag_bwd_workspace_size(ctypes.byref(tb.c), ctypes.byref(bags), _MODES[mode], ctypes.byref(n)),
           "dlrm_embbag_bwd_workspace_size")
    return int(n.value)


def dlrm_embbag_bwd_update(tables, indices, offsets, grad_pooled, rule, lr, eps=0.0, accum=None, mode="sum",
                           workspace=None, status=None, stream=None, side_stream=None):
    """Per-row gradient sums from grad_pooled [B, T, D] and one update of every touched row, in place."""
    lib = load_library()
    tb = _tables(tables)
    B = _batch(offsets, tb.T)
    _check_cuda(grad_pooled, "grad_pooled", torch.float32)
    if tuple(grad_pooled.shape) != (B, tb.T, tb.D):
        raise ValueError(f"grad_pooled must be [{B}, {tb.T}, {tb.D}]")
    upd, _keep = _update(tb, rule, lr, eps, accum)
    if workspace is None:
        workspace = torch.empty(max(dlrm_embbag_bwd_workspace_size(tb, indices, offsets, mode), 16),
                                dtype=torch.uint8, device=grad_pooled.device)
    _check_cuda(workspace, "workspace")
    bags = _bags(indices, offsets, B)
    dev = _device(*tb.tensors, *(accum or []), indices, offsets, grad_pooled, workspace, status)
    with torch.cuda.device(dev):
        st = lib.dlrm_embbag_bwd_update(ctypes.byref(tb.c), ctypes.byref(bags), _MODES[mode], grad_pooled.data_ptr(),
                                        ctypes.byref(upd), workspace.data_ptr(), workspace.numel(),
                                        status.data_ptr() if status is not None else None, _stream_ptr(stream, dev),
                                        side_stream.cuda_stream if side_stream is not None else None)
    _raise(st, "dlrm_embbag_bwd_update")


def dlrm_hash_indices(num_rows, raw_ids, offsets, rows=None, index_dtype=None, status=None, stream=None):
    """Raw 64-bit IDs (an int64 CUDA tensor, read as unsigned) to table rows, raw mod V_t; rows has the
    offsets' dtype unless index_dtype says otherwise."""
    lib = load_library()
    T = len(num_rows)
    B = _batch(offsets, T)
    _check_cuda(raw_ids, "raw_ids", torch.int64)
    _check_cuda(offsets, "offsets")
    dt = index_dtype or offsets.dtype
    if dt not in _ITYPES or offsets.dtype not in _ITYPES:
        raise ValueError("rows and offsets must be int32 or int64")
    if dt != offsets.dtype:
        raise ValueError("rows and offsets share the index type")
    if rows is None:
        rows = torch.empty(raw_ids.numel(), dtype=dt, device=raw_ids.device)
    _check_cuda(rows, "rows", dt)
    nr = (ctypes.c_int64 * T)(*[int(v) for v in num_rows])
    dev = _device(raw_ids, offsets, rows, status)
    with torch.cuda.device(dev):
        st = lib.dlrm_hash_indices(nr, T, B, raw_ids.numel(), raw_ids.data_ptr() if raw_ids.numel() else None,
                                   offsets.data_ptr(), _ITYPES[dt], rows.data_ptr() if rows.numel() else None,
                                   status.data_ptr() if status is not None else None, _stream_ptr(stream, dev))
    _raise(st, "dlrm_hash_indices")
    return rows


class TieredTables:
    """Tables kept in pinned host memory with a device cache of hot rows (dlrm_tiered_tables).

    host_tables: 2-D CPU tensors in pinned memory (tensor.pin_memory()), equal width and dtype; on a system
    with unified addressing their addresses are readable by the device.  cache_rows / stage_rows: per table
    (or one value for all) the device cache slots C_t and the staging rows M_t for a batch's misses.
    Device memory: (C_t + M_t) rows, V_t int32 map entries and C_t int64 slot entries per table."""

    def __init__(self, host_tables, cache_rows, stage_rows, device="cuda", stream=None):
        host_tables = list(host_tables)
        if not host_tables:
            raise ValueError("need at least one table")
        D, dt = host_tables[0].shape[1], host_tables[0].dtype
        for i, t in enumerate(host_tables):
            if t.is_cuda or not t.is_pinned() or not t.is_contiguous() or t.dim() != 2 or t.shape[1] != D or \
                    t.dtype != dt:
                raise ValueError(f"host table {i} must be a contiguous 2-D pinned CPU tensor of the common shape")
        if dt not in _DTYPES:
            raise ValueError(f"unsupported table dtype {dt}")
        T = len(host_tables)
        C = [int(cache_rows)] * T if isinstance(cache_rows, int) else [int(c) for c in cache_rows]
        M = [int(stage_rows)] * T if isinstance(stage_rows, int) else [int(m) for m in stage_rows]
        V = [t.shape[0] for t in host_tables]
        self.host, self.T, self.D, self.dtype = host_tables, T, D, dt
        self.C, self.M, self.V = C, M, V
        self.device = torch.device(device)
        self.slot_of = [torch.empty(v, dtype=torch.int32, device=self.device) for v in V]
        self.slot_row = [torch.empty(max(c, 1), dtype=torch.int64, device=self.device) for c in C]
        self.cache = [torch.empty((c + m, D), dtype=dt, device=self.device) for c, m in zip(C, M)]
        self.counters = torch.empty(T, dtype=torch.int32, device=self.device)
        self._arr = dict(
            host=(ctypes.c_void_p * T)(*[t.data_ptr() for t in host_tables]),
            rows=(ctypes.c_int64 * T)(*V),
            slot_of=(ctypes.c_void_p * T)(*[x.data_ptr() for x in self.slot_of]),
            slot_row=(ctypes.c_void_p * T)(*[x.data_ptr() for x in self.slot_row]),
            cache=(ctypes.c_void_p * T)(*[x.data_ptr() if x.numel() else None for x in self.cache]),
            C=(ctypes.c_int64 * T)(*C), M=(ctypes.c_int64 * T)(*M))
        a = self._arr
        self.c = DlrmTieredTables(T, D, _DTYPES[dt], a["host"], a["rows"], a["slot_of"], a["slot_row"], a["cache"],
                                  a["C"], a["M"])
        lib = load_library()
        with torch.cuda.device(self.device):
            _raise(lib.dlrm_tier_init(ctypes.byref(self.c), _stream_ptr(stream, self.device)), "dlrm_tier_init")
        # the forward's view: table t = its device buffer of C_t + M_t rows
        self.device_tables = Tables(self.cache)

    def fill(self, table: int, rows, status=None, stream=None):
        """Make `rows` (int64 device tensor of distinct row ids, at most C_t) the cache of `table`."""
        lib = load_library()
        _check_cuda(rows, "rows", torch.int64)
        with torch.cuda.device(self.device):
            st = lib.dlrm_tier_cache_fill(ctypes.byref(self.c), int(table), rows.data_ptr() if rows.numel() else None,
                                          rows.numel(), status.data_ptr() if status is not None else None,
                                          _stream_ptr(stream, self.device))
        _raise(st, "dlrm_tier_cache_fill")

    def stage(self, indices, offsets, out=None, status=None, stream=None):
        """Rewrite a batch's indices into rows of the device buffers (misses copied in from host memory).
        Returns the rewritten indices (dtype of `indices`), to pass with the same offsets and
        self.device_tables to the forward entry points."""
        lib = load_library()
        B = _batch(offsets, self.T)
        if out is None:
            out = torch.empty_like(indices)
        _check_cuda(out, "out", indices.dtype)
        bags = _bags(indices, offsets, B)
        dev = _device(indices, offsets, out, status, self.counters)
        with torch.cuda.device(dev):
            st = lib.dlrm_tier_stage(ctypes.byref(self.c), ctypes.byref(bags), out.data_ptr() if out.numel() else None,
                                     self.counters.data_ptr(), status.data_ptr() if status is not None else None,
                                     _stream_ptr(stream, dev))
        _raise(st, "dlrm_tier_stage")
        return out


def hot_rows(indices, offsets, B: int, T: int, capacity, num_rows=None):
    """Host-side cache policy: per table, the `capacity` rows looked up most often in the given batches
    (numpy arrays of one batch, or lists of them), ties broken by the lower row id.  Returns a list of
    int64 numpy arrays."""
    import numpy as np
    idx_list = indices if isinstance(indices, (list, tuple)) else [indices]
    off_list = offsets if isinstance(offsets, (list, tuple)) else [offsets]
    caps = [capacity] * T if isinstance(capacity, int) else list(capacity)
    out = []
    for t in range(T):
        seg = np.concatenate([np.asarray(i)[np.asarray(o)[t * B]:np.asarray(o)[(t + 1) * B]]
                              for i, o in zip(idx_list, off_list)]).astype(np.int64)
        if num_rows is not None:
            seg = seg[(seg >= 0) & (seg < num_rows[t])]
        rows, counts = np.unique(seg, return_counts=True)
        order = np.lexsort((rows, -counts))
        out.append(rows[order][:caps[t]])
    return out


# ---------------------------------------------------------------------------
# the dense layers around the sparse path
# ---------------------------------------------------------------------------
def _ptr(t):
    return t.data_ptr() if t is not None else None


def fc_fwd_workspace_size(M, K, N) -> int:
    n = ctypes.c_size_t(0)
    _raise(load_library().dlrm_fc_fwd_workspace_size(M, K, N, ctypes.byref(n)), "dlrm_fc_fwd_workspace_size")
    return int(n.value)


def dlrm_fc_fwd(x, w, b=None, relu=True, y=None, workspace=None, status=None, stream=None):
    """y = act(x W^T + b) on the tensor cores; x [M, in], w [out, in], b [out] or None."""
    lib = load_library()
    for name, t in (("x", x), ("w", w)):
        _check_cuda(t, name, torch.float32)
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("w must be [out_dim, in_dim]")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(fc_fwd_workspace_size(M, K, N), 16), dtype=torch.uint8, device=x.device)
    dev = _device(x, w, b, y, workspace, status)
    with torch.cuda.device(dev):
        st = lib.dlrm_fc_fwd(x.data_ptr(), w.data_ptr(), _ptr(b), M, K, N, 1 if relu else 0, y.data_ptr(),
                             workspace.data_ptr(), workspace.numel(), _ptr(status), _stream_ptr(stream, dev))
    _raise(st, "dlrm_fc_fwd")
    return y


def dlrm_fc_bwd_sgd(x, w, b, y, dy, lr, relu=True, dx=None, want_dx=True, workspace=None, status=None, stream=None):
    """The layer's backward with plain SGD on w (and b): returns dx [M, in] (None when not wanted)."""
    lib = load_library()
    M, K = x.shape
    N = w.shape[0]
    if want_dx and dx is None:
        dx = torch.empty((M, K), dtype=torch.float32, device=x.device)
    if workspace is None:
        n = ctypes.c_size_t(0)
        _raise(lib.dlrm_fc_bwd_workspace_size(M, K, N, ctypes.byref(n)), "dlrm_fc_bwd_workspace_size")
        workspace = torch.empty(max(n.value, 16), dtype=torch.uint8, device=x.device)
    dev = _device(x, w, b, y, dy, dx, workspace, status)
    with torch.cuda.device(dev):
        st = lib.dlrm_fc_bwd_sgd(x.data_ptr(), w.data_ptr(), _ptr(b), _ptr(y), dy.data_ptr(), M, K, N,
                                 1 if relu else 0, float(lr), _ptr(dx) if want_dx else None, workspace.data_ptr(),
                                 workspace.numel(), _ptr(status), _stream_ptr(stream, dev))
    _raise(st, "dlrm_fc_bwd_sgd")
    return dx if want_dx else None


def fc_bwd_workspace_size(M, K, N) -> int:
    n = ctypes.c_size_t(0)
    _raise(load_library().dlrm_fc_bwd_workspace_size(M, K, N, ctypes.byref(n)), "dlrm_fc_bwd_workspace_size")
    return int(n.value)


def dlrm_head_bce_sgd(h, w, b, label, lr, prob=None, loss=None, dh=None, workspace=None, stream=None):
    """Logit, sigmoid, mean BCE, its gradient dh, and SGD on w [in] and b [1]; returns (prob, loss, dh)."""
    lib = load_library()
    M, K = h.shape
    if prob is None:
        prob = torch.empty(M, dtype=torch.float32, device=h.device)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=h.device)
    if dh is None:
        dh = torch.empty((M, K), dtype=torch.float32, device=h.device)
    if workspace is None:
        n = ctypes.c_size_t(0)
        _raise(lib.dlrm_head_bce_workspace_size(M, K, ctypes.byref(n)), "dlrm_head_bce_workspace_size")
        workspace = torch.empty(max(n.value, 16), dtype=torch.uint8, device=h.device)
    dev = _device(h, w, b, label, prob, loss, dh, workspace)
    with torch.cuda.device(dev):
        st = lib.dlrm_head_bce_sgd(h.data_ptr(), w.data_ptr(), b.data_ptr(), label.data_ptr(), M, K, float(lr),
                                   prob.data_ptr(), loss.data_ptr(), dh.data_ptr(), workspace.data_ptr(),
                                   workspace.numel(), _stream_ptr(stream, dev))
    _raise(st, "dlrm_head_bce_sgd")
    return prob, loss, dh


class DLRMModel:
    """A whole DLRM around the sparse path, every step in the C library: the bottom MLP (FC + ReLU layers
    ending at width D), the fused sparse forward, the top MLP (FC + ReLU layers) and a 1-wide sigmoid head
    with the mean BCE loss; the backward with plain SGD on the MLP weights and row-wise Adagrad (or SGD) on
    the embedding rows.

    bottom: [(W, b), ...] fp32 CUDA tensors, W [out, in], the last out = D; top: the same, the first
    in = D + N(N-1)/2; head: (w [in], b [1])."""

    def __init__(self, tables, bottom, top, head):
        self.tables = _tables(tables)
        self.bottom, self.top, self.head = bottom, top, head
        self._buf = {}

    def _get(self, key, shape, dtype=torch.float32):
        t = self._buf.get(key)
        dev = self.head[0].device
        if t is None or tuple(t.shape) != tuple(shape):
            t = torch.empty(shape, dtype=dtype, device=dev)
            self._buf[key] = t
        return t

    def _ws(self, key, nbytes):
        t = self._buf.get(key)
        if t is None or t.numel() < nbytes:
            t = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=self.head[0].device)
            self._buf[key] = t
        return t

    def forward(self, dense_in, indices, offsets, mode="sum", stream=None, after=None, lookup_stream=None,
                after_lookup=None):
        """Bottom MLP, sparse forward (pooled vectors saved), top MLP; returns the top MLP's output.
        lookup_stream: forked from the caller's stream at the start; bags of more than 1.25 lookups on average
        are pooled there (dlrm_embbag_fwd) beside the bottom MLP, since the lookup needs only the bags, and the
        interaction (dlrm_interact_fwd) follows the bottom MLP; after_lookup() is called once that is queued,
        to queue more work on lookup_stream.  Otherwise the fused forward (dlrm_sparse_fwd) follows the bottom
        MLP.  Both give the same values: dlrm_sparse_fwd with pooled vectors saved runs those two kernels for
        such bags."""
        B = dense_in.shape[0]
        N = self.tables.T + 1
        out = self._get("out", (B, self.tables.D + N * (N - 1) // 2))
        pooled = self._get("pooled", (B, self.tables.T, self.tables.D))
        main = stream if stream is not None else torch.cuda.current_stream(dense_in.device)
        split = lookup_stream is not None and 4 * indices.numel() > 5 * self.tables.T * B
        lookup_ev = None
        if lookup_stream is not None:
            fork = torch.cuda.Event()
            fork.record(main)
            lookup_stream.wait_event(fork)
            if split:
                dlrm_embbag_fwd(self.tables, indices, offsets, mode, pooled=pooled, stream=lookup_stream)
                lookup_ev = torch.cuda.Event()
                lookup_ev.record(lookup_stream)
            if after_lookup:
                after_lookup()
        h = dense_in
        self.bot_in = [h]
        for i, (w, b) in enumerate(self.bottom):
            h = dlrm_fc_fwd(h, w, b, True, y=self._get(("bot", i), (B, w.shape[0])),
                            workspace=self._ws("ws_fwd", fc_fwd_workspace_size(B, w.shape[1], w.shape[0])),
                            stream=stream)
            self.bot_in.append(h)
        if after:
            after("bottom_fwd")
        x = h
        if split:
            main.wait_event(lookup_ev)
            dlrm_interact_fwd(x, pooled, out=out, stream=stream)
        else:
            dlrm_sparse_fwd(self.tables, indices, offsets, x, mode, out=out, pooled_save=pooled, stream=stream)
        if after:
            after("sparse_fwd")
        g = out
        self.top_in = [g]
        for i, (w, b) in enumerate(self.top):
            g = dlrm_fc_fwd(g, w, b, True, y=self._get(("top", i), (B, w.shape[0])),
                            workspace=self._ws("ws_fwd", fc_fwd_workspace_size(B, w.shape[1], w.shape[0])),
                            stream=stream)
            self.top_in.append(g)
        if after:
            after("top_fwd")
        return g

    def train_step(self, dense_in, indices, offsets, label, lr_mlp, lr_emb, eps=1e-8, accum=None, rule="adagrad",
                   mode="sum", stream=None, side_stream=None, after=None):
        """One training step; returns (loss [1], prob [B]) as device tensors.

        With side_stream, the work that depends only on the bags runs there from the step's start: the lookup of
        multi-lookup bags beside the bottom MLP, then the lookup-key build and sort of the sparse backward beside
        the rest of the forward; and the bottom MLP's backward, which needs only grad_x, runs on a stream of the
        model's own beside the sparse backward's per-row sums.  Without it every step runs on the caller's stream
        (the sort inside the sparse backward)."""
        B = dense_in.shape[0]
        ws = self._ws("ws_sparse", dlrm_sparse_bwd_workspace_size(self.tables, indices, offsets))
        main = stream if stream is not None else torch.cuda.current_stream(dense_in.device)
        sorted_ev = torch.cuda.Event() if side_stream is not None else None

        def sort_beside():
            dlrm_sparse_bwd_sort(self.tables, indices, offsets, ws, stream=side_stream)
            sorted_ev.record(side_stream)

        g = self.forward(dense_in, indices, offsets, mode, stream, after, lookup_stream=side_stream,
                         after_lookup=sort_beside if side_stream is not None else None)
        w, b = self.head
        prob, loss, dh = dlrm_head_bce_sgd(g, w, b, label, lr_mlp, prob=self._get("prob", (B,)),
                                           loss=self._get("loss", (1,)), dh=self._get("dh", (B, w.shape[0])),
                                           workspace=self._ws("ws_head", _head_ws(B, w.shape[0])), stream=stream)
        if after:
            after("head")
        dy = dh
        for i in range(len(self.top) - 1, -1, -1):
            W, bb = self.top[i]
            xin, yout = self.top_in[i], self.top_in[i + 1]
            dy = dlrm_fc_bwd_sgd(xin, W, bb, yout, dy, lr_mlp, True, dx=self._get(("dtop", i), tuple(xin.shape)),
                                 workspace=self._ws(("ws_top", i), fc_bwd_workspace_size(B, W.shape[1], W.shape[0])),
                                 stream=stream)
        if after:
            after("top_bwd")
        x = self.bot_in[-1]
        gx = self._get("grad_x", (B, self.tables.D))
        bottom_stream = main
        if sorted_ev is not None:
            gx_ready = torch.cuda.Event()
            dlrm_sparse_bwd_update_sorted(self.tables, indices, offsets, x, self._buf["pooled"], dy, rule, lr_emb,
                                          eps, accum, mode, grad_dense=gx, workspace=ws, sorted=sorted_ev,
                                          grad_ready=gx_ready, stream=stream)
            if "bwd_stream" not in self._buf:
                self._buf["bwd_stream"] = torch.cuda.Stream(device=dense_in.device)
            bottom_stream = self._buf["bwd_stream"]
            bottom_stream.wait_event(gx_ready)
        else:
            dlrm_sparse_bwd_update(self.tables, indices, offsets, x, self._buf["pooled"], dy, rule, lr_emb, eps,
                                   accum, mode, grad_dense=gx, workspace=ws, stream=stream)
        if after:
            after("sparse_bwd")
        dy = gx
        for i in range(len(self.bottom) - 1, -1, -1):
            W, bb = self.bottom[i]
            xin, yout = self.bot_in[i], self.bot_in[i + 1]
            dy = dlrm_fc_bwd_sgd(xin, W, bb, yout, dy, lr_mlp, True,
                                 dx=self._get(("dbot", i), tuple(xin.shape)) if i > 0 else None, want_dx=i > 0,
                                 workspace=self._ws(("ws_bot", i), fc_bwd_workspace_size(B, W.shape[1], W.shape[0])),
                                 stream=bottom_stream)
        if bottom_stream is not main:
            done = torch.cuda.Event()
            done.record(bottom_stream)
            main.wait_event(done)
        if after:
            after("bottom_bwd")
        return loss, prob


def _head_ws(M, K) -> int:
    n = ctypes.c_size_t(0)
    _raise(load_library().dlrm_head_bce_workspace_size(M, K, ctypes.byref(n)), "dlrm_head_bce_workspace_size")
    return int(n.value)
