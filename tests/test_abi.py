"""The C-ABI library builds for sm_103a, loads on a machine without a GPU, and
exports every entry point include/*.h declares.  Host-side argument checks are
exercised too: they run before any CUDA call."""
import ctypes
import glob
import os
import re

import pytest

import embedding_bag_lookup_dlrm_b300 as dl
from embedding_bag_lookup_dlrm_b300 import build as dlbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dlbuild.build()
    return dl.load_library()


def declared_entry_points():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w \*]*?\b(dlrm_\w+)\s*\(", text, flags=re.M))
    return names


def test_exports_every_declared_symbol(lib):
    declared = declared_entry_points()
    assert {"dlrm_embbag_fwd", "dlrm_interact_fwd", "dlrm_sparse_fwd", "dlrm_sparse_bwd_adagrad"} <= declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert set(dl.C_SYMBOLS) == declared


def test_built_for_sm103a():
    # the fatbinary section names the target; read only the ELF section table
    import subprocess
    out = subprocess.run(["readelf", "-S", dlbuild.LIB], capture_output=True, text=True).stdout
    assert ".nv_fatbin" in out


def test_abi_version_and_status_strings(lib):
    assert lib.dlrm_abi_version() == 2
    assert lib.dlrm_status_string(0) == b"ok"
    assert lib.dlrm_status_string(dl.DLRM_ERR_INDEX_OOB) == b"index out of range"
    assert lib.dlrm_status_string(dl.DLRM_ERR_INVALID_ARG | dl.DLRM_ERR_TIMEOUT) == b"invalid argument"


def _tables(T=2, D=128, dtype=0, rows=10, ptr=0x1000):
    ptrs = (ctypes.c_void_p * T)(*[ptr] * T)
    nr = (ctypes.c_int64 * T)(*[rows] * T)
    return dl.DlrmTables(T, D, dtype, ptrs, nr), ptrs, nr


def test_host_argument_checks(lib):
    tb, _p, _r = _tables()
    bags = dl.DlrmBags(4, 8, 0, 0x2000, 0x3000)
    st = lib.dlrm_sparse_fwd(None, ctypes.byref(bags), 0, 0x4000, 0x5000, None, None, None)
    assert st == dl.DLRM_ERR_INVALID_ARG
    bad_T, _a, _b = _tables(T=0)
    assert lib.dlrm_sparse_fwd(ctypes.byref(bad_T), ctypes.byref(bags), 0, 0x4000, 0x5000, None, None, None) == 1
    bad_D, _a, _b = _tables(D=130)
    assert lib.dlrm_embbag_fwd(ctypes.byref(bad_D), ctypes.byref(bags), 0, 0x4000, None, None) == 1
    odd_D, _a, _b = _tables(D=48)   # a multiple of 4 the library has no kernel for
    assert lib.dlrm_embbag_fwd(ctypes.byref(odd_D), ctypes.byref(bags), 0, 0x4000, None, None) == \
        dl.DLRM_ERR_UNSUPPORTED
    misaligned, _a, _b = _tables(ptr=0x1004)
    assert lib.dlrm_embbag_fwd(ctypes.byref(misaligned), ctypes.byref(bags), 0, 0x4000, None, None) == 1
    assert lib.dlrm_embbag_fwd(ctypes.byref(tb), ctypes.byref(bags), 7, 0x4000, None, None) == 1  # mode
    neg = dl.DlrmBags(0, 8, 0, 0x2000, 0x3000)
    assert lib.dlrm_embbag_fwd(ctypes.byref(tb), ctypes.byref(neg), 0, 0x4000, None, None) == 1
    assert lib.dlrm_interact_fwd(0x1000, 0x2000, 4, 0, 128, 0x3000, None) == 1
    bf, _a, _b = _tables(dtype=1)
    st = lib.dlrm_sparse_bwd_adagrad(ctypes.byref(bf), ctypes.byref(bags), 0, 0x10, 0x10, 0x10, 0x10,
                                     (ctypes.c_void_p * 2)(0x10, 0x10), 0.01, 1e-8, 0x10, 1 << 30, None, None, None)
    assert st == dl.DLRM_ERR_UNSUPPORTED


def _bwd_status(lib, T, B, nnz, itype=1, rows=10):
    tb, _p, _r = _tables(T=T, D=16, rows=rows)
    bags = dl.DlrmBags(B, nnz, itype, 0x2000, 0x3000)
    acc = (ctypes.c_void_p * T)(*[0x10] * T)
    return lib.dlrm_sparse_bwd_adagrad(ctypes.byref(tb), ctypes.byref(bags), 0, 0x10, 0x10, 0x10, 0x10, acc, 0.01,
                                       1e-8, 0x10, 1 << 62, None, None, None)


def test_backward_rejects_batches_past_32_bit_sort_fields(lib):
    """The backward sorts 32-bit keys (global rows), values (b*T + t) and positions: T*B >= 2^32 or
    nnz >= 2^32 is refused on the host, before any launch (int64 indices, so the forward accepts both)."""
    assert _bwd_status(lib, T=2, B=1 << 31, nnz=8) == dl.DLRM_ERR_UNSUPPORTED      # T*B = 2^32
    assert _bwd_status(lib, T=2, B=4, nnz=1 << 32) == dl.DLRM_ERR_UNSUPPORTED      # nnz = 2^32
    assert _bwd_status(lib, T=1, B=4, nnz=8, rows=(1 << 32) - 1) == dl.DLRM_ERR_UNSUPPORTED  # rows
    # just inside every limit the host checks pass and only the (huge) workspace need remains
    n = ctypes.c_size_t(0)
    tb, _p, _r = _tables(T=2, D=16)
    bags = dl.DlrmBags((1 << 31) - 1, (1 << 32) - 1, 1, 0x2000, 0x3000)
    assert lib.dlrm_sparse_bwd_workspace_size(ctypes.byref(tb), ctypes.byref(bags), ctypes.byref(n)) == 0
    assert n.value > 1 << 36


def test_split_step_host_checks(lib):
    """dlrm_sparse_bwd_sort and dlrm_sparse_bwd_update_sorted refuse on the host what the one-call step
    refuses: past the 32-bit sort fields, bf16 tables, no or misaligned workspace, a workspace too small."""
    def sort_status(T, B, nnz, rows=10, dtype=0, ws=0x10, ws_bytes=1 << 62):
        tb, _p, _r = _tables(T=T, D=16, rows=rows, dtype=dtype)
        bags = dl.DlrmBags(B, nnz, 1, 0x2000, 0x3000)
        return lib.dlrm_sparse_bwd_sort(ctypes.byref(tb), ctypes.byref(bags), ws, ws_bytes, None, None)

    assert sort_status(T=2, B=1 << 31, nnz=8) == dl.DLRM_ERR_UNSUPPORTED       # T*B = 2^32
    assert sort_status(T=2, B=4, nnz=1 << 32) == dl.DLRM_ERR_UNSUPPORTED       # nnz = 2^32
    assert sort_status(T=1, B=4, nnz=8, rows=(1 << 32) - 1) == dl.DLRM_ERR_UNSUPPORTED
    assert sort_status(T=2, B=4, nnz=8, dtype=1) == dl.DLRM_ERR_UNSUPPORTED     # bf16 tables
    assert sort_status(T=2, B=4, nnz=8, ws=None) == dl.DLRM_ERR_INVALID_ARG
    assert sort_status(T=2, B=4, nnz=8, ws=0x18) == dl.DLRM_ERR_INVALID_ARG     # not 16-byte aligned
    assert sort_status(T=2, B=4, nnz=8, ws_bytes=64) == dl.DLRM_ERR_INVALID_ARG  # too small

    tb, _p, _r = _tables(T=2, D=16)
    bags = dl.DlrmBags(4, 1 << 32, 1, 0x2000, 0x3000)
    acc = (ctypes.c_void_p * 2)(0x10, 0x10)
    upd = dl.DlrmUpdate(0, 0.01, 1e-8, ctypes.cast(acc, ctypes.POINTER(ctypes.c_void_p)))
    args = (ctypes.byref(tb), ctypes.byref(bags), 0, 0x10, 0x10, 0x10, 0x10, ctypes.byref(upd), 0x10, 1 << 62,
            None, None, None, None)
    assert lib.dlrm_sparse_bwd_update_sorted(*args) == dl.DLRM_ERR_UNSUPPORTED  # nnz = 2^32
    bags.nnz = 8
    upd.rule = 9
    assert lib.dlrm_sparse_bwd_update_sorted(*args) == dl.DLRM_ERR_INVALID_ARG  # unknown rule


def test_static_scratch_size_matches_header(lib):
    """The binding's copy of DLRM_STATIC_SCRATCH_BYTES is the header's."""
    text = open(os.path.join(ROOT, "include", "dlrm_sparse.h")).read()
    m = re.search(r"#define\s+DLRM_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "DLRM_STATIC_SCRATCH_BYTES not found in the header"
    assert int(m.group(1)) << int(m.group(2)) == dl.STATIC_SCRATCH_BYTES


def test_workspace_size_grows_with_batch(lib):
    tb, _p, _r = _tables(T=26)
    sizes = []
    for B, nnz in ((128, 512), (32768, 3_800_000)):
        bags = dl.DlrmBags(B, nnz, 0, 0x2000, 0x3000)
        n = ctypes.c_size_t(0)
        assert lib.dlrm_sparse_bwd_workspace_size(ctypes.byref(tb), ctypes.byref(bags), ctypes.byref(n)) == 0
        sizes.append(n.value)
        assert n.value >= B * 26 * 128 * 4 + 16 * nnz
    assert sizes[1] > sizes[0]


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _load_missing(tmp_path)


def _load_missing(tmp_path):
    saved = dl._lib
    try:
        dl._lib = None
        return dl.load_library(str(tmp_path / "missing.so"))
    finally:
        dl._lib = saved


def _build_c_smoke(tmp_path):
    import subprocess
    exe = str(tmp_path / "c_abi_smoke")
    libdir = os.path.dirname(dlbuild.LIB)
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-o", exe, os.path.join(ROOT, "tests", "c_abi_smoke.c"),
           "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include", "-L", libdir, "-ldlrm_sparse",
           f"-Wl,-rpath,{libdir}", "-L", "/usr/local/cuda/lib64", "-lcudart", "-Wl,-rpath,/usr/local/cuda/lib64"]
    subprocess.run(cmd, check=True)
    return exe


def test_plain_c_consumer_host_checks(lib, tmp_path):
    """The header compiles as C99 with warnings as errors and a C program linked against the library
    (no Python) gets the declared host-side behaviour."""
    import subprocess
    r = subprocess.run([_build_c_smoke(tmp_path)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert "c abi smoke ok" in r.stdout


@pytest.mark.gpu
def test_plain_c_consumer_device_forwards(lib, tmp_path):
    """The C program's identity-table forwards on the device: exact closed-form outputs."""
    import subprocess
    r = subprocess.run([_build_c_smoke(tmp_path), "--gpu"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert "with device forwards" in r.stdout
