"""The C-ABI library without a GPU: it builds, loads, exports every function
include/bsgemm.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os

import pytest

import verifiable_quantize_rows_gb300 as bsg
from verifiable_quantize_rows_gb300 import build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return bsg.load()


def test_header_declares_the_boundary():
    names = bsg.exported_symbols()
    for required in ("bsg_quantize_rows", "bsg_quantize_cols", "bsg_gemm_s32", "bsg_epilogue",
                     "bsgemm_i8", "bsgemm_i8_ex", "bsgemm_i8_host", "bsgemm_i8_host_batch", "bsg_hash_f32",
                     "bsg_probe_hash", "bsg_probe_hash_async", "bsg_status_str", "bsg_audit",
                     "bsg_selftest", "bsgemm_i8_requant", "bsgemm_i8_chain", "bsgemm_i8_noalloc",
                     "bsg_mma_ceiling"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in bsg.exported_symbols() if not hasattr(lib, n)]
    assert not missing


def test_status_strings_and_version(lib):
    assert lib.bsg_version() >= 100
    for code in range(9):
        assert lib.bsg_status_str(code).startswith(b"BSG_")


def test_workspace_sizes(lib):
    for M, N, K in ((1, 1, 1), (8192, 2304, 768), (4097, 12289, 8191)):
        ws = lib.bsgemm_i8_workspace_size(M, N, K)
        ldk = (K + 63) // 64 * 64
        assert ws >= 2 * ldk * (M + N) + 4 * (M + N)
        assert lib.bsgemm_i8_host_workspace_size(M, N, K) > ws
        assert lib.bsg_probe_workspace_size(M, N, K) > ws
    assert lib.bsgemm_i8_workspace_size(0, 5, 5) == 0


def test_argument_errors_without_gpu(lib):
    vp = ctypes.c_void_p
    dummy = vp(256)
    # null pointers, bad sizes, K over the limit, too-small workspace
    assert lib.bsgemm_i8(None, dummy, 4, 4, 4, 0, dummy, dummy, 1 << 20, None, None) == 1
    assert lib.bsgemm_i8(dummy, dummy, 0, 4, 4, 0, dummy, dummy, 1 << 20, None, None) == 1
    # C beyond 2^40 elements (each side under 2^31): rejected, not overflowed
    assert lib.bsgemm_i8(dummy, dummy, 1 << 30, 1 << 11, 4, 0, dummy, dummy, 1 << 20, None,
                         None) == 1
    assert lib.bsgemm_i8_workspace_size(1 << 30, (1 << 10) + 1, 4) == 0
    assert lib.bsgemm_i8(dummy, dummy, 4, 4, bsg.MAX_K + 1, 0, dummy, dummy, 1 << 30, None,
                         None) == 2
    assert lib.bsgemm_i8(dummy, dummy, 4, 4, 4, 0, dummy, dummy, 16, None, None) == 3
    assert lib.bsgemm_i8(dummy, dummy, 4, 4, 4, 0, dummy, vp(257), 1 << 20, None, None) == 3
    assert lib.bsgemm_i8_ex(dummy, 3, 0, dummy, 4, 0, 4, 4, 4, 0, dummy, 4, dummy, 1 << 20,
                            None, None) == 1   # lda < K
    assert lib.bsgemm_i8_ex(dummy, 4, 2, dummy, 4, 0, 4, 4, 4, 0, dummy, 4, dummy, 1 << 20,
                            None, None) == 1   # transA not 0/1
    assert lib.bsg_quantize_rows(dummy, 4, 8, 7, dummy, 8, dummy, None, None, None) == 1
    assert lib.bsg_quantize_cols(dummy, 4, 8, 8, dummy, 8, dummy, None, None, 0, None, None) == 3
    assert lib.bsg_epilogue(dummy, 3, dummy, dummy, 4, 4, 0, dummy, 4, None) == 1
    assert lib.bsg_gemm_s32(dummy, 4, dummy, 4, 4, 4, 4, dummy, 3, dummy, 1 << 20, None,
                            None) == 1
    assert lib.bsg_hash_f32(dummy, 2, 2, 2, None, dummy, 1 << 20, None) == 1
    assert lib.bsg_probe_hash(0, 4, 4, 4, None, dummy, 1 << 20, None) == 1
    # audit: null mismatch counter, ldc < N, no samples, K over the limit
    assert lib.bsg_audit(dummy, 4, dummy, 4, dummy, 4, 4, 4, 4, 0, 0, 8, None, None, None) == 1
    assert lib.bsg_audit(dummy, 4, dummy, 4, dummy, 3, 4, 4, 4, 0, 0, 8, dummy, None, None) == 1
    assert lib.bsg_audit(dummy, 4, dummy, 4, dummy, 4, 4, 4, 4, 0, 0, 0, dummy, None, None) == 1
    assert lib.bsg_audit(dummy, bsg.MAX_K + 1, dummy, 4, dummy, 4, 4, 4, bsg.MAX_K + 1, 0, 0, 8,
                         dummy, None, None) == 2
    # weight storage: bits other than 8/4, ldq too small for the packed int4 rows
    assert lib.bsg_wquant_cols(dummy, 4, 4, 4, 6, 0, dummy, 4, dummy, dummy, 1 << 20, None,
                               None) == 1
    assert lib.bsg_wquant_cols(dummy, 4, 5, 5, 4, 0, dummy, 2, dummy, dummy, 1 << 20, None,
                               None) == 1
    # weight storage without its workspace, or with too little of it
    assert lib.bsg_wquant_cols(dummy, 4, 5, 5, 8, 0, dummy, 5, dummy, None, 0, None, None) == 3
    assert lib.bsg_wquant_cols(dummy, 5000, 300, 300, 8, 0, dummy, 300, dummy, dummy, 256, None,
                               None) == 3
    assert lib.bsg_wquant_cols_workspace_size(5000, 300) >= (1 + 3 + 300) * 4
    assert lib.bsg_wquant_cols_workspace_size(0, 300) == 0
    assert lib.bsg_wdequant_cols(dummy, 4, 4, 4, 8, dummy, dummy, 3, None) == 1
    # grouped call: no items, too many items
    assert lib.bsgemm_i8_group(None, 1, None, None) == 1
    items = (bsg.GemmItem * 4)()
    assert lib.bsgemm_i8_group(items, 4, None, None) == 1
    assert lib.bsgemm_i8_group(items, 0, None, None) == 1
    # host batch: no items, too many, a null buffer, shared workspace or C,
    # a too-small workspace
    assert lib.bsgemm_i8_host_batch(None, 1, None, None) == 1
    hitems = (bsg.HostItem * 17)()
    assert lib.bsgemm_i8_host_batch(hitems, 0, None, None) == 1
    assert lib.bsgemm_i8_host_batch(hitems, 17, None, None) == 1
    big = 1 << 30
    for i in range(2):
        hitems[i] = bsg.HostItem(256, 256, 4, 4, 4, 0, 4096 + 1024 * i, (1 << 20) + i * big, big)
    hitems[1].workspace = (1 << 20) + big - 256          # overlaps item 0's workspace
    assert lib.bsgemm_i8_host_batch(hitems, 2, None, None) == 1
    hitems[1].workspace = (1 << 20) + big
    hitems[1].C_host = 4096 + 32                            # overlaps item 0's C (64 bytes)
    assert lib.bsgemm_i8_host_batch(hitems, 2, None, None) == 1
    hitems[1].C_host = 4096 + 64
    hitems[1].A_host = None
    assert lib.bsgemm_i8_host_batch(hitems, 2, None, None) == 1
    hitems[1].A_host = 256
    hitems[1].ws_bytes = 64
    assert lib.bsgemm_i8_host_batch(hitems, 2, None, None) == 3
    # chained units: null outputs, bad sizes, a too-small workspace
    assert lib.bsgemm_i8_requant(dummy, dummy, 4, 4, 4, 0, None, dummy, dummy, None, dummy,
                                 1 << 20, None, None) == 1
    assert lib.bsgemm_i8_requant(dummy, dummy, 4, 4, 4, 0, dummy, dummy, None, None, dummy,
                                 1 << 20, None, None) == 1
    assert lib.bsgemm_i8_requant(dummy, dummy, 4, 4, 4, 0, dummy, dummy, dummy, None, dummy,
                                 16, None, None) == 3
    assert lib.bsgemm_i8_chain(dummy, dummy, None, 4, 4, 4, 4, 0, 0, dummy, dummy, dummy,
                               1 << 20, None, None) == 1
    assert lib.bsgemm_i8_chain(dummy, dummy, dummy, 4, 4, 0, 4, 0, 0, dummy, dummy, dummy,
                               1 << 20, None, None) == 1
    assert lib.bsgemm_i8_chain(dummy, dummy, dummy, 4, 4, 4, 4, 0, 0, dummy, dummy, dummy,
                               16, None, None) == 3
    need = lib.bsgemm_i8_chain_workspace_size(8192, 768, 3072, 768)
    assert need > lib.bsgemm_i8_requant_workspace_size(8192, 3072, 768)
    assert lib.bsgemm_i8_requant_workspace_size(8192, 3072, 768) > 8192 * 4
    assert lib.bsgemm_i8_chain_workspace_size(0, 4, 4, 4) == 0
    # the tensor-pipe ceiling: iterations out of range
    assert lib.bsg_mma_ceiling(0, None, None, None) == 1
    assert lib.bsg_mma_ceiling((1 << 18) + 1, None, None, None) == 1
    # self-test: missing or small workspace
    assert lib.bsg_selftest(None, 0, None, None) == 3
    assert lib.bsg_selftest(dummy, 16, None, None) == 3


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        bsg.load(str(tmp_path / "missing.so"))


def test_selftest_known_answer_is_the_oracle_golden():
    """The self-test's compiled-in probe hash equals the value the oracle
    wrote to tests/golden/probe_hash.txt for seed 0 at 1024^3."""
    import re
    here = os.path.dirname(os.path.abspath(__file__))
    src = open(os.path.join(here, "..", "verifiable_quantize_rows_gb300", "csrc",
                            "bsgemm_api.cu")).read()
    body = re.search(r"kProbeKnownAnswer\[32\] = \{(.*?)\};", src, re.S).group(1)
    compiled = bytes(int(x, 16) for x in re.findall(r"0x([0-9a-f]{2})", body)).hex()
    golden = None
    for line in open(os.path.join(here, "golden", "probe_hash.txt")):
        p = line.split()
        if len(p) == 5 and p[:4] == ["0", "1024", "1024", "1024"]:
            golden = p[4]
    assert golden is not None and compiled == golden


def test_binding_refuses_host_tensors():
    """No CPU fallback: host tensors, wrong dtypes and non-contiguous views
    are refused before anything runs."""
    import torch
    A = torch.ones(4, 8)
    B = torch.ones(8, 3)
    with pytest.raises(TypeError, match="CUDA tensor"):
        bsg.bsgemm_i8(A, B)
    with pytest.raises(TypeError, match="CUDA tensor"):
        bsg.quantize_rows(A)
    with pytest.raises(TypeError, match="CUDA tensor"):
        bsg.quantize_cols(A)
    with pytest.raises(TypeError, match="CUDA tensor"):
        bsg.wquant_cols(A)
    with pytest.raises(TypeError, match="CUDA tensor"):
        bsg.bsgemm_i8(A.double(), B.double())


def test_product_path_never_touches_the_oracle():
    """Static check: the package, its CUDA sources and the header never
    import, load or link the oracle's module or library; bench.py imports it
    only inside its two CPU legs (cpu_baseline and the reference arm); the
    oracle never imports the package."""
    import ast
    import re
    ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(ROOT, "verifiable_quantize_rows_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath or "__pycache__" in dirpath:
            continue
        for f in files:
            if not f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                continue
            text = open(os.path.join(dirpath, f)).read()
            if f.endswith(".py"):
                tree = ast.parse(text)
                for node in ast.walk(tree):
                    if isinstance(node, ast.Import):
                        assert all(not a.name.startswith("oracle") for a in node.names), f
                    if isinstance(node, ast.ImportFrom):
                        assert not (node.module or "").startswith("oracle"), f
            assert "bsg_oracle" not in text, f
            assert not re.search(r"dlopen|CDLL\([^)]*oracle", text), f
    header = open(os.path.join(ROOT, "include", "bsgemm.h")).read()
    assert "bsg_oracle" not in header and "orc_" not in header
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    users = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, ast.Import) and any(a.name == "oracle" for a in node.names):
                    users.add(fn.name)
    top = [n for n in tree.body if isinstance(n, (ast.Import, ast.ImportFrom))]
    assert all("oracle" not in ast.dump(n) for n in top)
    assert users <= {"cpu_baseline", "run_reference", "oracle_inputs"}, users
    orc_src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert "verifiable_quantize_rows_gb300" not in orc_src
    # the oracle's C source includes system headers only: no shared header
    c_src = open(os.path.join(ROOT, "oracle", "bsg_oracle.c")).read()
    includes = re.findall(r"#\s*include\s*(\S+)", c_src)
    assert includes and all(i.startswith("<") for i in includes), includes
