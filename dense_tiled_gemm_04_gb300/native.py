"""ctypes binding of the C ABI in ``include/gemm.h`` (``libdtgemm.so``).

Argument marshalling only: every step of C = A·B runs in the library's CUDA kernels.
The binding never falls back to another implementation -- if the library is missing
or the device is not an sm_103 GPU, the call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

API_VERSION = 3  # GEMM_API_VERSION the structures below are laid out for
LAYOUT_NN, LAYOUT_TN = 0, 1
DTYPE_F16, DTYPE_BF16, DTYPE_E4M3, DTYPE_E5M2 = 0, 1, 2, 3
LAYOUTS = {"NN": LAYOUT_NN, "TN": LAYOUT_TN}
DTYPES = {"f16": DTYPE_F16, "bf16": DTYPE_BF16, "e4m3": DTYPE_E4M3, "e5m2": DTYPE_E5M2}
KINDS = {"dense": 0, "block_scaled": 1, "sparse24": 2}  # gemm_kind_t
TORCH_TO_DTYPE = {torch.float16: DTYPE_F16, torch.bfloat16: DTYPE_BF16}
# 8-bit operand types (gemm_run_ex only).
TORCH_TO_DTYPE_EX = {**TORCH_TO_DTYPE, torch.float8_e4m3fn: DTYPE_E4M3, torch.float8_e5m2: DTYPE_E5M2}

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ARCH, ERR_CUDA, ERR_TIMEOUT = range(6)
OPT_CONFIG, OPT_TIMEOUT_NS, OPT_MAX_CTAS, OPT_RASTER_GROUP, OPT_FAULT_INJECT, OPT_STREAM_K, \
    OPT_HOST_ROW_CHUNKS, OPT_HOST_COL_CHUNKS, OPT_SK_MIN_BLOCKS, OPT_SPLIT_MIN_BLOCKS, OPT_K_SNAKE = range(11)
CONFIG_AUTO, CONFIG_128x256, CONFIG_128x128, CONFIG_256x256, CONFIG_128x64 = range(5)


class gemm_plan_t(ctypes.Structure):
    _fields_ = [("config", ctypes.c_int32), ("bm", ctypes.c_int32), ("bn", ctypes.c_int32),
                ("bk", ctypes.c_int32), ("stages", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("tiles_m", ctypes.c_int64), ("tiles_n", ctypes.c_int64), ("k_blocks", ctypes.c_int64),
                ("grid", ctypes.c_int64), ("threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("dp_tiles", ctypes.c_int64), ("sk_base", ctypes.c_int64), ("sk_extra", ctypes.c_int64),
                ("raster_group", ctypes.c_int64), ("k_snake", ctypes.c_int64)]


class gemm_args_t(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldc", ctypes.c_int64),
                ("layout", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("c_col_major", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("scale_a", ctypes.c_float), ("scale_b", ctypes.c_float)]


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}" if what else status_string(status))


_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load ``libdtgemm.so``; raises if it has not been built (no silent fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise ImportError(f"{_build.LIB} is missing: build it with dense_tiled_gemm_04_gb300.build.build()")
    lib = ctypes.CDLL(_build.LIB)
    i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    sig = {
        "gemm_create": ([ctypes.POINTER(p), ctypes.c_int], i32),
        "gemm_destroy": ([p], i32),
        "gemm_run": ([p, p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, p], i32),
        "gemm_run_host": ([p, p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, p], i32),
        "gemm_run_ex": ([p, ctypes.POINTER(gemm_args_t), p], i32),
        "gemm_run_mx": ([p, ctypes.POINTER(gemm_args_t), p, p, p], i32),
        "gemm_mx_scale_bytes": ([i64, i64], i64),
        "gemm_run_sp": ([p, ctypes.POINTER(gemm_args_t), p, p], i32),
        "gemm_sp_meta_bytes": ([i64, i64], i64),
        "gemm_sp_compress": ([p, p, i64, i64, i64, i32, p, i64, p, p, p], i32),
        "gemm_mx_pack_scales": ([p, p, i64, i64, i64, p, p], i32),
        "gemm_sync_status": ([p, p], i32),
        "gemm_error_info": ([p, ctypes.POINTER(i32)], i32),
        "gemm_set_option": ([p, i32, i64], i32),
        "gemm_get_option": ([p, i32, ctypes.POINTER(i64)], i32),
        "gemm_query_plan": ([p, i64, i64, i64, i32, i32, ctypes.POINTER(gemm_plan_t)], i32),
        "gemm_query_plan_kind": ([p, i64, i64, i64, i32, i32, i32, ctypes.POINTER(gemm_plan_t)], i32),
        "gemm_check_args": ([p, p, p, i64, i64, i64, i64, i64, i64, i32, i32], i32),
        "gemm_tile_coord": ([i64, i64, i64, i64, ctypes.POINTER(i64), ctypes.POINTER(i64)], i32),
        "gemm_run_noalloc": ([p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, p, ctypes.POINTER(i32)], i32),
        "gemm_status_string": ([i32], ctypes.c_char_p),
        "gemm_api_version": ([], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    if lib.gemm_api_version() != API_VERSION:
        raise ImportError(f"{_build.LIB} implements API version {lib.gemm_api_version()}, this binding "
                          f"version {API_VERSION}: rebuild it with dense_tiled_gemm_04_gb300.build.build()")
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


def check_args(A: int, B: int, C: int, M, N, K, lda, ldb, ldc, layout: int, dtype: int) -> int:
    """gemm_check_args on raw addresses (no GPU needed)."""
    return int(load().gemm_check_args(A or None, B or None, C or None, M, N, K, lda, ldb, ldc, layout, dtype))


def mx_scale_bytes(rows: int, K: int) -> int:
    """Bytes of the chunked block-scale layout for `rows` rows and K elements of K."""
    return int(load().gemm_mx_scale_bytes(rows, K))


def sp_meta_bytes(M: int, K: int) -> int:
    """Bytes of the chunked 2:4 sparsity metadata for M rows and K."""
    return int(load().gemm_sp_meta_bytes(M, K))


def tile_coord(tile: int, tiles_m: int, tiles_n: int, group_m: int):
    tm, tn = ctypes.c_int64(), ctypes.c_int64()
    st = load().gemm_tile_coord(tile, tiles_m, tiles_n, group_m, ctypes.byref(tm), ctypes.byref(tn))
    if st != OK:
        raise GemmError(st, "gemm_tile_coord")
    return tm.value, tn.value


def _ld(t: torch.Tensor) -> int:
    """Leading dimension of a 2-D row-major tensor (one-row tensors: the padded row length)."""
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.size(1) > 1 and t.stride(1) != 1:
        raise ValueError("expected unit stride along the last dimension (row-major)")
    if t.size(0) <= 1:
        align = 16 // t.element_size()  # a TMA row pitch is a multiple of 16 bytes
        return max(-(-t.size(1) // align) * align, align)
    return t.stride(0)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def empty_output(M: int, N: int, dtype: torch.dtype, device) -> torch.Tensor:
    """An M x N output whose row pitch is a multiple of 8 elements (TMA alignment)."""
    ldc = max(-(-N // 8) * 8, 8)
    return torch.empty((M, ldc), dtype=dtype, device=device)[:, :N]


class Gemm:
    """A library handle bound to one CUDA device."""

    def __init__(self, device=None):
        lib = load()
        if device is None:
            device = torch.cuda.current_device()
        self.device = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        h = ctypes.c_void_p()
        st = lib.gemm_create(ctypes.byref(h), self.device.index or 0)
        if st != OK:
            raise GemmError(st, "gemm_create")
        self._h = h
        self._lib = lib

    # -------------------------------------------------------------- lifecycle
    def close(self):
        if getattr(self, "_h", None):
            st = self._lib.gemm_destroy(self._h)
            self._h = None
            if st != OK:
                raise GemmError(st, "gemm_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -------------------------------------------------------------- options
    def set_option(self, opt: int, value: int):
        st = self._lib.gemm_set_option(self._h, opt, int(value))
        if st != OK:
            raise GemmError(st, "gemm_set_option")

    def get_option(self, opt: int) -> int:
        v = ctypes.c_int64()
        st = self._lib.gemm_get_option(self._h, opt, ctypes.byref(v))
        if st != OK:
            raise GemmError(st, "gemm_get_option")
        return v.value

    def plan(self, M, N, K, layout="NN", dtype="f16", kind: str = "dense") -> dict:
        """The launch the entry point for `kind` ("dense", "block_scaled", "sparse24") would make."""
        pl = gemm_plan_t()
        st = self._lib.gemm_query_plan_kind(self._h, M, N, K, LAYOUTS[layout], DTYPES[dtype], KINDS[kind],
                                            ctypes.byref(pl))
        if st != OK:
            raise GemmError(st, "gemm_query_plan_kind")
        return {f: getattr(pl, f) for f, _ in gemm_plan_t._fields_}

    def error_info(self):
        arr = (ctypes.c_int32 * 4)()
        self._lib.gemm_error_info(self._h, arr)
        return list(arr)

    # -------------------------------------------------------------- compute
    def run_raw(self, A: int, B: int, C: int, M, N, K, lda, ldb, ldc, layout: int, dtype: int, stream: int) -> int:
        """gemm_run on raw device addresses; returns the status code."""
        return int(self._lib.gemm_run(self._h, A or None, B or None, C or None, M, N, K, lda, ldb, ldc,
                                      layout, dtype, stream or None))

    def run(self, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, layout: str = "NN",
            stream=None) -> torch.Tensor:
        """C = A·B (NN: B is K x N) or A·B^T (TN: B is N x K) on device tensors; async on `stream`."""
        M, K = A.shape
        N = B.shape[1] if layout == "NN" else B.shape[0]
        if (B.shape[0] if layout == "NN" else B.shape[1]) != K:
            raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, layout {layout}")
        if A.dtype != B.dtype or A.dtype not in TORCH_TO_DTYPE:
            raise TypeError("A and B must both be float16 or both bfloat16")
        if C is None:
            C = empty_output(M, N, A.dtype, A.device)
        if C.shape != (M, N) or C.dtype != A.dtype:
            raise ValueError("C has the wrong shape or dtype")
        st = self.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, _ld(A), _ld(B), _ld(C),
                          LAYOUTS[layout], TORCH_TO_DTYPE[A.dtype], _stream_ptr(stream))
        if st != OK:
            raise GemmError(st, "gemm_run")
        return C

    def run_ex_raw(self, A: int, B: int, C: int, M, N, K, lda, ldb, ldc, layout: int, dtype: int, alpha: float,
                   beta: float, c_col_major: int, stream: int, out_dtype: int | None = None, scale_a: float = 1.0,
                   scale_b: float = 1.0) -> int:
        """gemm_run_ex on raw device addresses:
        C = alpha * scale_a * scale_b * A·B + beta * C (row- or column-major C)."""
        a = gemm_args_t(A or None, B or None, C or None, M, N, K, lda, ldb, ldc, layout, dtype, alpha, beta,
                        c_col_major, dtype if out_dtype is None else out_dtype, scale_a, scale_b)
        return int(self._lib.gemm_run_ex(self._h, ctypes.byref(a), stream or None))

    def run_ex(self, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, layout: str = "NN",
               out_dtype: torch.dtype | None = None, alpha: float = 1.0, beta: float = 0.0, scale_a: float = 1.0,
               scale_b: float = 1.0, c_col_major: bool = False, stream=None) -> torch.Tensor:
        """C = alpha * scale_a * scale_b * A·B + beta * C on device tensors; A, B 16-bit or 8-bit
        (float8_e4m3fn / float8_e5m2), C float16 or bfloat16.  With c_col_major, ``C`` is the
        N x M row-major tensor holding C transposed.  Async on `stream`."""
        M, K = A.shape
        N = B.shape[1] if layout == "NN" else B.shape[0]
        if (B.shape[0] if layout == "NN" else B.shape[1]) != K:
            raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, layout {layout}")
        if A.dtype != B.dtype or A.dtype not in TORCH_TO_DTYPE_EX:
            raise TypeError("A and B must have the same 16-bit or 8-bit float type")
        if out_dtype is None:
            out_dtype = C.dtype if C is not None else (A.dtype if A.dtype in TORCH_TO_DTYPE else torch.bfloat16)
        if out_dtype not in TORCH_TO_DTYPE:
            raise TypeError("C must be float16 or bfloat16")
        shape = (N, M) if c_col_major else (M, N)
        if C is None:
            C = empty_output(*shape, out_dtype, A.device)
        if tuple(C.shape) != shape or C.dtype != out_dtype:
            raise ValueError("C has the wrong shape or dtype")
        st = self.run_ex_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, _ld(A), _ld(B), _ld(C),
                             LAYOUTS[layout], TORCH_TO_DTYPE_EX[A.dtype], alpha, beta, int(c_col_major),
                             _stream_ptr(stream), TORCH_TO_DTYPE[out_dtype], scale_a, scale_b)
        if st != OK:
            raise GemmError(st, "gemm_run_ex")
        return C

    def pack_scales(self, sf: torch.Tensor, K: int | None = None, stream=None) -> torch.Tensor:
        """Row-major E8M0 exponents (rows x ceil(K/32), uint8, on the device) -> the chunked
        layout gemm_run_mx reads, in a new uint8 tensor (gemm_mx_pack_scales, async)."""
        if sf.dtype != torch.uint8 or sf.dim() != 2 or (sf.size(1) > 1 and sf.stride(1) != 1):
            raise ValueError("expected a 2-D row-major uint8 tensor")
        rows, kblocks = sf.shape
        K = 32 * kblocks if K is None else K
        if -(-K // 32) != kblocks:
            raise ValueError(f"{kblocks} K blocks do not cover K = {K}")
        out = torch.empty(max(mx_scale_bytes(rows, K), 16), dtype=torch.uint8, device=sf.device)
        ld = sf.stride(0) if rows > 1 else max(kblocks, 1)
        st = self._lib.gemm_mx_pack_scales(self._h, sf.data_ptr() or None, rows, kblocks, ld, out.data_ptr(),
                                           _stream_ptr(stream))
        if st != OK:
            raise GemmError(st, "gemm_mx_pack_scales")
        return out

    def run_mx_raw(self, A: int, B: int, C: int, sfa: int, sfb: int, M, N, K, lda, ldb, ldc, layout: int, dtype: int,
                   out_dtype: int, alpha: float = 1.0, beta: float = 0.0, c_col_major: int = 0, scale_a: float = 1.0,
                   scale_b: float = 1.0, stream: int = 0) -> int:
        """gemm_run_mx on raw device addresses; returns the status code."""
        a = gemm_args_t(A or None, B or None, C or None, M, N, K, lda, ldb, ldc, layout, dtype, alpha, beta,
                        c_col_major, out_dtype, scale_a, scale_b)
        return int(self._lib.gemm_run_mx(self._h, ctypes.byref(a), sfa or None, sfb or None, stream or None))

    def run_mx(self, A: torch.Tensor, B: torch.Tensor, sfa: torch.Tensor, sfb: torch.Tensor,
               C: torch.Tensor | None = None, layout: str = "NN", out_dtype: torch.dtype = torch.bfloat16,
               alpha: float = 1.0, beta: float = 0.0, scale_a: float = 1.0, scale_b: float = 1.0,
               c_col_major: bool = False, stream=None) -> torch.Tensor:
        """C = alpha * scale_a * scale_b * (A·B with per-tile E8M0 scales) + beta * C on device
        tensors: A, B float8_e4m3fn / float8_e5m2; sfa, sfb the chunked scales (pack_scales).
        Async on `stream`."""
        M, K = A.shape
        N = B.shape[1] if layout == "NN" else B.shape[0]
        if (B.shape[0] if layout == "NN" else B.shape[1]) != K:
            raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, layout {layout}")
        if A.dtype != B.dtype or A.dtype not in (torch.float8_e4m3fn, torch.float8_e5m2):
            raise TypeError("A and B must have the same 8-bit float type")
        if out_dtype not in TORCH_TO_DTYPE:
            raise TypeError("C must be float16 or bfloat16")
        for t, rows, what in ((sfa, M, "sfa"), (sfb, N, "sfb")):
            if t.dtype != torch.uint8 or t.numel() < mx_scale_bytes(rows, K):
                raise ValueError(f"{what} must hold {mx_scale_bytes(rows, K)} bytes of packed scales")
        shape = (N, M) if c_col_major else (M, N)
        if C is None:
            C = empty_output(*shape, out_dtype, A.device)
        if tuple(C.shape) != shape or C.dtype != out_dtype:
            raise ValueError("C has the wrong shape or dtype")
        st = self.run_mx_raw(A.data_ptr(), B.data_ptr(), C.data_ptr(), sfa.data_ptr(), sfb.data_ptr(), M, N, K, _ld(A),
                             _ld(B), _ld(C), LAYOUTS[layout], TORCH_TO_DTYPE_EX[A.dtype], TORCH_TO_DTYPE[out_dtype],
                             alpha, beta, int(c_col_major), scale_a, scale_b, _stream_ptr(stream))
        if st != OK:
            raise GemmError(st, "gemm_run_mx")
        return C

    def sp_compress(self, A: torch.Tensor, stream=None):
        """2:4 compression of a dense fp16/bf16 device matrix (gemm_sp_compress, async):
        returns (Ac: M x K/2 kept values, meta: chunked metadata bytes, bad: 1-element int32
        device tensor counting groups with more than two non-zeros)."""
        if A.dtype not in TORCH_TO_DTYPE or A.dim() != 2:
            raise TypeError("A must be a 2-D float16 or bfloat16 tensor")
        M, K = A.shape
        if K % 4:
            raise ValueError("K must be a multiple of 4")
        Ac = empty_output(M, K // 2, A.dtype, A.device)
        meta = torch.empty(max(sp_meta_bytes(M, K), 16), dtype=torch.uint8, device=A.device)
        bad = torch.zeros(1, dtype=torch.int32, device=A.device)
        st = self._lib.gemm_sp_compress(self._h, A.data_ptr() or None, M, K, _ld(A), TORCH_TO_DTYPE[A.dtype],
                                        Ac.data_ptr() or None, _ld(Ac), meta.data_ptr(), bad.data_ptr(),
                                        _stream_ptr(stream))
        if st != OK:
            raise GemmError(st, "gemm_sp_compress")
        return Ac, meta, bad

    def run_sp_raw(self, Ac: int, B: int, C: int, meta: int, M, N, K, lda, ldb, ldc, layout: int, dtype: int,
                   alpha: float = 1.0, beta: float = 0.0, c_col_major: int = 0, stream: int = 0) -> int:
        """gemm_run_sp on raw device addresses (Ac: the compressed A, lda its pitch; K logical)."""
        a = gemm_args_t(Ac or None, B or None, C or None, M, N, K, lda, ldb, ldc, layout, dtype, alpha, beta,
                        c_col_major, dtype, 1.0, 1.0)
        return int(self._lib.gemm_run_sp(self._h, ctypes.byref(a), meta or None, stream or None))

    def run_sp(self, Ac: torch.Tensor, B: torch.Tensor, meta: torch.Tensor, C: torch.Tensor | None = None,
               layout: str = "NN", alpha: float = 1.0, beta: float = 0.0, c_col_major: bool = False,
               stream=None) -> torch.Tensor:
        """C = alpha * A·B + beta * C with A 2:4-sparse, given as (Ac, meta) from sp_compress.
        K = 2 * Ac's columns.  Async on `stream`."""
        M, K = Ac.shape[0], 2 * Ac.shape[1]
        N = B.shape[1] if layout == "NN" else B.shape[0]
        if (B.shape[0] if layout == "NN" else B.shape[1]) != K:
            raise ValueError(f"shape mismatch: Ac {tuple(Ac.shape)}, B {tuple(B.shape)}, layout {layout}")
        if Ac.dtype != B.dtype or Ac.dtype not in TORCH_TO_DTYPE:
            raise TypeError("Ac and B must both be float16 or both bfloat16")
        if meta.dtype != torch.uint8 or meta.numel() < sp_meta_bytes(M, K):
            raise ValueError(f"meta must hold {sp_meta_bytes(M, K)} bytes")
        shape = (N, M) if c_col_major else (M, N)
        if C is None:
            C = empty_output(*shape, Ac.dtype, Ac.device)
        if tuple(C.shape) != shape or C.dtype != Ac.dtype:
            raise ValueError("C has the wrong shape or dtype")
        st = self.run_sp_raw(Ac.data_ptr(), B.data_ptr(), C.data_ptr(), meta.data_ptr(), M, N, K, _ld(Ac), _ld(B),
                             _ld(C), LAYOUTS[layout], TORCH_TO_DTYPE[Ac.dtype], alpha, beta, int(c_col_major),
                             _stream_ptr(stream))
        if st != OK:
            raise GemmError(st, "gemm_run_sp")
        return C

    def run_host(self, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, layout: str = "NN", stream=None) -> int:
        """gemm_run_host on CPU tensors (pin them for DMA copies); synchronous; returns the status."""
        M, K = A.shape
        N = C.shape[1]
        return int(self._lib.gemm_run_host(self._h, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                           _ld(A), _ld(B), _ld(C), LAYOUTS[layout], TORCH_TO_DTYPE[A.dtype],
                                           _stream_ptr(stream) or None))

    def sync_status(self, stream=None) -> int:
        return int(self._lib.gemm_sync_status(self._h, _stream_ptr(stream) or None))


_default: dict = {}


def matmul(A: torch.Tensor, B: torch.Tensor, layout: str = "NN", out: torch.Tensor | None = None,
           stream=None) -> torch.Tensor:
    """C = A·B with the library's kernel, on a per-device default handle."""
    dev = A.device.index if A.device.index is not None else torch.cuda.current_device()
    if dev not in _default:
        _default[dev] = Gemm(dev)
    return _default[dev].run(A, B, out, layout, stream)
