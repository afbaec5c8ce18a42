"""C ABI checks that need no GPU: the library loads, exports every declared entry point,
validates arguments exactly as documented, and its tile scheduler map is a bijection."""
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "gemm.h")


@pytest.fixture(scope="module")
def lib():
    from dense_tiled_gemm_04_gb300 import build, native

    build.build()
    return native


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(gemm_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_core_entry_points():
    names = declared_functions()
    for core in ("gemm_create", "gemm_run", "gemm_destroy", "gemm_status_string", "gemm_sync_status"):
        assert core in names


def test_every_declared_symbol_is_exported(lib):
    so = lib.load()
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    so = lib.load()
    assert so.gemm_api_version() == 3 == lib.API_VERSION
    for s in range(6):
        assert lib.status_string(s).startswith("GEMM_")
    assert "unknown" in lib.status_string(99)


def test_null_handle_is_rejected_without_a_gpu(lib):
    so = lib.load()
    assert so.gemm_run(None, None, None, None, 1, 1, 1, 8, 8, 8, 0, 0, None) == lib.ERR_INVALID_ARG
    assert so.gemm_sync_status(None, None) == lib.ERR_INVALID_ARG
    assert so.gemm_set_option(None, 0, 0) == lib.ERR_INVALID_ARG
    assert so.gemm_destroy(None) == lib.OK
    assert so.gemm_create(None, 0) == lib.ERR_INVALID_ARG
    assert so.gemm_run_ex(None, None, None) == lib.ERR_INVALID_ARG
    args = lib.gemm_args_t(None, None, None, 8, 8, 8, 8, 8, 8, 0, 0, 1.0, 0.0, 0, 0, 1.0, 1.0)
    assert so.gemm_run_ex(None, args, None) == lib.ERR_INVALID_ARG


def test_args_struct_matches_the_header(lib):
    # Field order and size of gemm_args_t as declared in the header (x86-64 and aarch64 ABI).
    text = open(HEADER).read()
    end = text.index("} gemm_args_t;")
    body = text[text.rindex("typedef struct {", 0, end) + len("typedef struct {"):end]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = []
    for decl in body.split(";"):
        m = re.match(r"\s*(?:const\s+)?\w+\s*\*?\s*(.*)$", decl, flags=re.S)
        if decl.strip():
            names += [n.strip() for n in m.group(1).split(",")]
    assert names == [f for f, _ in lib.gemm_args_t._fields_]
    import ctypes
    assert ctypes.sizeof(lib.gemm_args_t) == 3 * 8 + 6 * 8 + 2 * 4 + 2 * 4 + 4 + 4 + 2 * 4


def test_create_without_a_gpu_reports_an_error(lib):
    import ctypes
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = lib.load().gemm_create(ctypes.byref(h), 0)
    assert st in (lib.ERR_CUDA, lib.ERR_INVALID_ARG)
    assert not h.value


P = 1 << 20  # a 16-byte-aligned fake address: gemm_check_args never dereferences


@pytest.mark.parametrize("case,expected", [
    # (A, B, C, M, N, K, lda, ldb, ldc, layout, dtype)
    ((P, P, P, 128, 256, 192, 192, 256, 256, 0, 0), 0),
    ((P, P, P, 1000, 1000, 1000, 1000, 1000, 1000, 1, 0), 0),
    ((P, P, P, 0, 5, 7, 0, 0, 0, 0, 0), 0),            # M == 0: no-op, nothing else checked
    ((P, P, P, 5, 0, 7, 0, 0, 0, 0, 0), 0),            # N == 0
    ((0, 0, P, 5, 8, 0, 0, 0, 8, 0, 0), 0),            # K == 0: A, B unused
    ((P, P, P, -1, 8, 8, 8, 8, 8, 0, 0), 1),           # negative size
    ((P, P, P, 8, 8, 8, 8, 8, 8, 2, 0), 1),            # bad layout
    ((P, P, P, 8, 8, 8, 8, 8, 8, 0, 7), 1),            # bad dtype
    ((P, P, P, 16, 16, 16, 16, 16, 16, 0, 2), 1),      # 8-bit operands: gemm_run_ex only
    ((0, P, P, 8, 8, 8, 8, 8, 8, 0, 0), 1),            # null A
    ((P, P, 0, 8, 8, 8, 8, 8, 8, 0, 0), 1),            # null C
    ((P, P, P, 8, 16, 16, 8, 16, 16, 0, 0), 1),        # lda < K
    ((P, P, P, 8, 16, 8, 8, 8, 16, 0, 0), 1),          # NN: ldb < N
    ((P, P, P, 8, 16, 24, 24, 16, 16, 1, 0), 1),       # TN: ldb < K
    ((P, P, P, 8, 16, 8, 8, 16, 8, 0, 0), 1),          # ldc < N
    ((P + 2, P, P, 8, 8, 8, 8, 8, 8, 0, 0), 2),        # A not 16-byte aligned
    ((P, P + 8, P, 8, 8, 8, 8, 8, 8, 0, 1), 2),        # B not 16-byte aligned
    ((P, P, P + 4, 8, 8, 8, 8, 8, 8, 0, 0), 2),        # C not 16-byte aligned
    ((P, P, P, 8, 8, 12, 12, 8, 8, 0, 0), 2),          # lda not a multiple of 8
    ((P, P, P, 65, 97, 130, 136, 104, 104, 0, 0), 0),  # the page's tail case with padded ld
    ((P, P, P, 65, 97, 130, 130, 97, 97, 0, 0), 2),    # ... and without padding
    ((P, P, P, 1 << 31, 8, 8, 8, 8, 8, 0, 0), 2),      # dimension beyond int32
])
def test_check_args(lib, case, expected):
    assert lib.check_args(*case) == expected


@pytest.mark.parametrize("tiles_m,tiles_n,group", [(1, 1, 1), (2, 4, 16), (64, 32, 16), (8, 4, 3),
                                                   (17, 5, 4), (7, 9, 7), (5, 3, 100), (33, 1, 8)])
def test_tile_coord_is_a_bijection(lib, tiles_m, tiles_n, group):
    seen = set()
    for t in range(tiles_m * tiles_n):
        tm, tn = lib.tile_coord(t, tiles_m, tiles_n, group)
        assert 0 <= tm < tiles_m and 0 <= tn < tiles_n
        seen.add((tm, tn))
    assert len(seen) == tiles_m * tiles_n


def test_tile_coord_groups_rows(lib):
    # With a group of 4 tile rows, consecutive tiles walk down the rows of one column
    # before moving to the next column.
    coords = [lib.tile_coord(t, 8, 3, 4) for t in range(6)]
    assert coords == [(0, 0), (1, 0), (2, 0), (3, 0), (0, 1), (1, 1)]
    with pytest.raises(Exception):
        lib.tile_coord(24, 8, 3, 4)


def test_mx_scale_bytes_without_a_gpu(lib):
    assert lib.mx_scale_bytes(0, 64) == 0 and lib.mx_scale_bytes(5, 0) == 0
    assert lib.mx_scale_bytes(1, 1) == 512 and lib.mx_scale_bytes(128, 128) == 512
    assert lib.mx_scale_bytes(129, 129) == 2 * 2 * 512
    assert lib.mx_scale_bytes(8192, 8192) == 64 * 64 * 512
    so = lib.load()
    assert so.gemm_mx_pack_scales(None, None, 1, 1, 1, None, None) == lib.ERR_INVALID_ARG
    assert so.gemm_run_mx(None, None, None, None, None) == lib.ERR_INVALID_ARG


def test_sparse_entry_points_without_a_gpu(lib):
    assert lib.sp_meta_bytes(0, 64) == 0 and lib.sp_meta_bytes(5, 0) == 0
    assert lib.sp_meta_bytes(1, 4) == 4096 and lib.sp_meta_bytes(128, 64) == 4096
    assert lib.sp_meta_bytes(129, 65) == 2 * 2 * 4096
    so = lib.load()
    assert so.gemm_run_sp(None, None, None, None) == lib.ERR_INVALID_ARG
    assert so.gemm_sp_compress(None, None, 1, 4, 4, 0, None, 2, None, None, None) == lib.ERR_INVALID_ARG


def header_enum_values():
    """Every `NAME = value` inside the header's enum blocks (values are integer literals)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    values = {}
    for body in re.findall(r"enum\s*\{(.*?)\}", text, flags=re.S):
        for name, value in re.findall(r"(GEMM_\w+)\s*=\s*(\d+)", body):
            values[name] = int(value)
    return values


def test_binding_constants_match_the_header(lib):
    values = header_enum_values()
    pairs = {
        "GEMM_LAYOUT_NN": lib.LAYOUT_NN, "GEMM_LAYOUT_TN": lib.LAYOUT_TN,
        "GEMM_DTYPE_F16": lib.DTYPE_F16, "GEMM_DTYPE_BF16": lib.DTYPE_BF16,
        "GEMM_DTYPE_E4M3": lib.DTYPE_E4M3, "GEMM_DTYPE_E5M2": lib.DTYPE_E5M2,
        "GEMM_OK": lib.OK, "GEMM_ERR_INVALID_ARG": lib.ERR_INVALID_ARG, "GEMM_ERR_UNSUPPORTED": lib.ERR_UNSUPPORTED,
        "GEMM_ERR_ARCH": lib.ERR_ARCH, "GEMM_ERR_CUDA": lib.ERR_CUDA, "GEMM_ERR_TIMEOUT": lib.ERR_TIMEOUT,
        "GEMM_OPT_CONFIG": lib.OPT_CONFIG, "GEMM_OPT_TIMEOUT_NS": lib.OPT_TIMEOUT_NS,
        "GEMM_OPT_MAX_CTAS": lib.OPT_MAX_CTAS, "GEMM_OPT_RASTER_GROUP": lib.OPT_RASTER_GROUP,
        "GEMM_OPT_FAULT_INJECT": lib.OPT_FAULT_INJECT, "GEMM_OPT_STREAM_K": lib.OPT_STREAM_K,
        "GEMM_OPT_HOST_ROW_CHUNKS": lib.OPT_HOST_ROW_CHUNKS, "GEMM_OPT_HOST_COL_CHUNKS": lib.OPT_HOST_COL_CHUNKS,
        "GEMM_OPT_SK_MIN_BLOCKS": lib.OPT_SK_MIN_BLOCKS, "GEMM_OPT_SPLIT_MIN_BLOCKS": lib.OPT_SPLIT_MIN_BLOCKS,
        "GEMM_OPT_K_SNAKE": lib.OPT_K_SNAKE,
        "GEMM_CONFIG_AUTO": lib.CONFIG_AUTO, "GEMM_CONFIG_128x256": lib.CONFIG_128x256,
        "GEMM_CONFIG_128x128": lib.CONFIG_128x128, "GEMM_CONFIG_256x256": lib.CONFIG_256x256,
        "GEMM_CONFIG_128x64": lib.CONFIG_128x64,
        "GEMM_KIND_DENSE": lib.KINDS["dense"], "GEMM_KIND_BLOCK_SCALED": lib.KINDS["block_scaled"],
        "GEMM_KIND_SPARSE24": lib.KINDS["sparse24"],
    }
    assert set(pairs) <= set(values), sorted(set(pairs) - set(values))
    assert {k: values[k] for k in pairs} == pairs


def test_package_exports_every_option_and_configuration():
    import dense_tiled_gemm_04_gb300 as pkg

    values = header_enum_values()
    for name, value in values.items():
        if name.startswith(("GEMM_OPT_", "GEMM_CONFIG_")):
            short = name[len("GEMM_"):]
            assert short in pkg.__all__, f"{short} missing from the package's exports"
            assert getattr(pkg, short) == value
