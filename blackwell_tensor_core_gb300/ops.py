"""Thin Python binding over libbwgemm.so (ctypes).

Argument marshalling only: every function here converts torch tensors to
device pointers, sizes and leading dimensions, calls the C ABI entry point of
the same name and raises on a non-zero status.  All arithmetic runs in the
library's CUDA kernels; if the library is missing or fails to load, every call
raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbwgemm.so")

OUT_BF16 = 0
OUT_FP32 = 1
OUT_FP16 = 2
_OUT_CODES = {torch.bfloat16: OUT_BF16, torch.float32: OUT_FP32, torch.float16: OUT_FP16}

KERNEL_NONE, KERNEL_ZERO, KERNEL_1CTA, KERNEL_2CTA, KERNEL_SMALL_M, KERNEL_2CTA_MC, KERNEL_2CTA_2C = range(7)

STATUS_NAMES = {0: "BWG_OK", 1: "BWG_ERR_INVALID_ARG", 2: "BWG_ERR_ALIGNMENT",
                3: "BWG_ERR_UNSUPPORTED", 4: "BWG_ERR_CUDA", 5: "BWG_ERR_TIMEOUT",
                6: "BWG_ERR_SCRATCH_LIMIT"}

_lock = threading.Lock()
_lib = None


class BwgError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed: %s (%s)" % (what, STATUS_NAMES.get(status, status), status_string(status)))
        self.status = status


class PlanInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("tile_k", ctypes.c_int), ("mma_m", ctypes.c_int), ("mma_n", ctypes.c_int),
                ("stages", ctypes.c_int), ("tiles", ctypes.c_int), ("k_blocks", ctypes.c_int),
                ("coverage", ctypes.c_double), ("smem_input_per_cta", ctypes.c_int),
                ("smem_total", ctypes.c_int), ("grid", ctypes.c_int), ("tx_bytes", ctypes.c_uint32),
                ("idesc", ctypes.c_uint32), ("units", ctypes.c_int), ("streamk", ctypes.c_int),
                ("workers", ctypes.c_int), ("dynamic", ctypes.c_int), ("sk_tiles", ctypes.c_int),
                ("sk_segs", ctypes.c_int), ("split", ctypes.c_int), ("staging_in_ring", ctypes.c_int),
                ("bt_loads", ctypes.c_int), ("pair_loads", ctypes.c_int)]


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libbwgemm.so is not built (%s); run __graft_entry__.build(). "
                                   "There is no fallback implementation." % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            vp, i, u32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64
            for name in ("gemm_bf16", "gemm_fp16", "gemm_bf16_nt", "gemm_fp16_nt"):
                f = getattr(L, name)
                f.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, vp]
                f.restype = i
            for name in ("grouped_gemm_bf16", "grouped_gemm_fp16", "grouped_gemm_swiglu_bf16",
                         "grouped_gemm_swiglu_fp16", "grouped_gemm_bf16_nt", "grouped_gemm_fp16_nt",
                         "grouped_gemm_swiglu_bf16_nt", "grouped_gemm_swiglu_fp16_nt"):
                f = getattr(L, name)
                f.argtypes = [vp, ctypes.POINTER(vp), vp, vp, i, i, i, i, vp]
                f.restype = i
            L.gemm_bf16_host.argtypes = [vp, vp, vp, i, i, i, i, vp, vp, vp, vp]
            L.gemm_bf16_host.restype = i
            L.bwg_status_string.argtypes = [i]
            L.bwg_status_string.restype = ctypes.c_char_p
            L.bwg_last_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_ulonglong)]
            L.bwg_last_device_error.restype = i
            for name, args in (("bwg_probe_cluster_pair", [vp, vp, vp, i, vp]),
                               ("bwg_probe_tma_swizzle", [vp, vp, vp]),
                               ("bwg_probe_mma", [vp, vp, vp, i, i, vp]),
                               ("bwg_probe_grouped_tables", [vp, i, i, i, i, i, i, vp, vp])):
                f = getattr(L, name)
                f.argtypes = args
                f.restype = i
            L.bwg_debug_set_trace.argtypes = [vp]
            L.bwg_debug_set_trace.restype = None
            L.bwg_set_watchdog_ns.argtypes = [ctypes.c_ulonglong]
            L.bwg_set_watchdog_ns.restype = None
            L.bwg_debug_set_tx_extra.argtypes = [ctypes.c_uint]
            L.bwg_debug_set_tx_extra.restype = None
            L.bwg_plan.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(PlanInfo)]
            L.bwg_plan.restype = i
            L.bwg_check_gemm_args.argtypes = [vp, vp, vp, i, i, i, i, i, i, i]
            L.bwg_check_gemm_args.restype = i
            L.bwg_idesc_f16.argtypes = [i, i, i, i, i]
            L.bwg_idesc_f16.restype = u32
            L.bwg_smem_desc.argtypes = [u32, u32, u32, i]
            L.bwg_smem_desc.restype = u64
            L.bwg_swizzle128_offset.argtypes = [u32, u32]
            L.bwg_swizzle128_offset.restype = u32
            L.bwg_raster_tile.argtypes = [i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
            L.bwg_raster_tile.restype = None
            ip = ctypes.POINTER(i)
            L.bwg_grouped_schedule.argtypes = [ip, i, i, i, i, ip, ip, ip]
            L.bwg_grouped_schedule.restype = i
            L.bwg_grouped_tile.argtypes = [i, i, ip, ip, ip, i, ip, ip, ip, ip]
            L.bwg_grouped_tile.restype = None
            L.bwg_tail_split.argtypes = [i, i]
            L.bwg_tail_split.restype = i
            L.bwg_unit_tile.argtypes = [i, i, i, i, ip, ip, ip]
            L.bwg_unit_tile.restype = None
            L.bwg_streamk_begin.argtypes = [i, ctypes.c_longlong, i]
            L.bwg_streamk_begin.restype = ctypes.c_longlong
            L.bwg_streamk_tile_workers.argtypes = [i, i, ctypes.c_longlong, i, ip, ip]
            L.bwg_streamk_tile_workers.restype = None
            L.bwg_grouped_swap_rows.argtypes = [i, i, i]
            L.bwg_grouped_swap_rows.restype = i
            L.bwg_tail_split_f.argtypes = [i, i, i, ip]
            L.bwg_tail_split_f.restype = i
            L.bwg_streamk_tiles.argtypes = [i, i, i, i, ip]
            L.bwg_streamk_tiles.restype = i
            L.bwg_unit_part.argtypes = [i, i, i, i, ip, ip, ip]
            L.bwg_unit_part.restype = None
            L.bwg_version.argtypes = []
            L.bwg_version.restype = ctypes.c_char_p
            _lib = L
    return _lib


def version() -> str:
    """bwg_version(): library version and the hash of the sources it was built from."""
    return lib().bwg_version().decode()


def status_string(status: int) -> str:
    try:
        return lib().bwg_status_string(int(status)).decode()
    except Exception:  # noqa: BLE001 - only used to format an error
        return "?"


def _check(status: int, what: str) -> None:
    if status != 0:
        raise BwgError(status, what)


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _matrix(t: torch.Tensor, name: str) -> int:
    if t.dim() != 2:
        raise ValueError("%s must be 2-D" % name)
    if t.stride(1) != 1:
        raise ValueError("%s must be row-major with unit column stride" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    return t.stride(0)


def gemm(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor | None = None,
         out_dtype: torch.dtype = torch.bfloat16, stream=None, b_transposed: bool = False) -> torch.Tensor:
    """D = A @ B through gemm_bf16 / gemm_fp16 (chosen by A's dtype); with
    ``b_transposed`` B is given as [N, K] and D = A @ B.T (gemm_*_nt)."""
    if A.dtype != B.dtype or A.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("A and B must both be bfloat16 or both float16")
    M, K = A.shape
    N, K2 = B.shape if b_transposed else (B.shape[1], B.shape[0])
    if K2 != K:
        raise ValueError("inner dimensions differ: %s x %s" % (tuple(A.shape), tuple(B.shape)))
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    if out.dtype not in _OUT_CODES:
        raise TypeError("output dtype must be bfloat16, float16 or float32")
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be [%d, %d], got %s" % (M, N, tuple(out.shape)))
    if not (A.device == B.device == out.device):
        raise ValueError("A, B and out must be on the same device")
    lda, ldb, ldd = _matrix(A, "A"), _matrix(B, "B"), _matrix(out, "out")
    if b_transposed:
        fn = gemm_bf16_nt if A.dtype == torch.bfloat16 else gemm_fp16_nt
    else:
        fn = gemm_bf16 if A.dtype == torch.bfloat16 else gemm_fp16
    fn(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K, lda, ldb, ldd, _OUT_CODES[out.dtype],
       _stream_handle(stream, A.device))
    return out


def gemm_bf16(A_ptr: int, B_ptr: int, D_ptr: int, M: int, N: int, K: int, lda: int, ldb: int,
              ldd: int, out_dtype: int, stream: int) -> None:
    _check(lib().gemm_bf16(A_ptr, B_ptr, D_ptr, M, N, K, lda, ldb, ldd, out_dtype, stream), "gemm_bf16")


def gemm_fp16(A_ptr: int, B_ptr: int, D_ptr: int, M: int, N: int, K: int, lda: int, ldb: int,
              ldd: int, out_dtype: int, stream: int) -> None:
    _check(lib().gemm_fp16(A_ptr, B_ptr, D_ptr, M, N, K, lda, ldb, ldd, out_dtype, stream), "gemm_fp16")


def gemm_bf16_nt(A_ptr: int, B_ptr: int, D_ptr: int, M: int, N: int, K: int, lda: int, ldb: int,
                 ldd: int, out_dtype: int, stream: int) -> None:
    """D = A x B^T with B stored [N, K] (ldb >= K)."""
    _check(lib().gemm_bf16_nt(A_ptr, B_ptr, D_ptr, M, N, K, lda, ldb, ldd, out_dtype, stream),
           "gemm_bf16_nt")


def gemm_fp16_nt(A_ptr: int, B_ptr: int, D_ptr: int, M: int, N: int, K: int, lda: int, ldb: int,
                 ldd: int, out_dtype: int, stream: int) -> None:
    _check(lib().gemm_fp16_nt(A_ptr, B_ptr, D_ptr, M, N, K, lda, ldb, ldd, out_dtype, stream),
           "gemm_fp16_nt")


def grouped_gemm(A: torch.Tensor, Bs: list, group_offsets: torch.Tensor,
                 out: torch.Tensor | None = None, stream=None, swiglu: bool = False,
                 b_transposed: bool = False) -> torch.Tensor:
    """Grouped expert product through grouped_gemm_bf16 / grouped_gemm_fp16.

    With ``swiglu`` each weight is [gate | up] ([K, N]) and the result is
    silu(gate) * up, [M_total, N/2], through grouped_gemm_swiglu_bf16/_fp16.
    With ``b_transposed`` every weight is given as [N, K] (the *_nt entry points)."""
    if A.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("A must be bfloat16 or float16")
    M_total, K = A.shape
    G = len(Bs)
    N = (Bs[0].shape[0] if b_transposed else Bs[0].shape[1]) if G else 0
    want = (N, K) if b_transposed else (K, N)
    for b in Bs:
        if b.shape != want or b.dtype != A.dtype or not b.is_contiguous():
            raise ValueError("every weight matrix must be a contiguous %s tensor of A's dtype"
                             % ("[N, K]" if b_transposed else "[K, N]"))
    if group_offsets.dtype != torch.int32 or group_offsets.numel() != G + 1 or not group_offsets.is_cuda:
        raise ValueError("group_offsets must be a CUDA int32 tensor with G+1 entries")
    if not A.is_contiguous():
        raise ValueError("A must be dense [M_total, K]")
    n_out = N // 2 if swiglu else N
    if out is None:
        out = torch.empty((M_total, n_out), dtype=A.dtype, device=A.device)
    elif out.shape != (M_total, n_out) or out.dtype != A.dtype or not out.is_contiguous():
        raise ValueError("out must be a dense [M_total, %d] tensor of A's dtype" % n_out)
    bf = A.dtype == torch.bfloat16
    if swiglu and b_transposed:
        fn = grouped_gemm_swiglu_bf16_nt if bf else grouped_gemm_swiglu_fp16_nt
    elif swiglu:
        fn = grouped_gemm_swiglu_bf16 if bf else grouped_gemm_swiglu_fp16
    elif b_transposed:
        fn = grouped_gemm_bf16_nt if bf else grouped_gemm_fp16_nt
    else:
        fn = grouped_gemm_bf16 if bf else grouped_gemm_fp16
    fn(A.data_ptr(), [b.data_ptr() for b in Bs], out.data_ptr(), group_offsets.data_ptr(), G, M_total,
       N, K, _stream_handle(stream, A.device))
    return out


def _ptr_array(ptrs):
    arr = (ctypes.c_void_p * max(len(ptrs), 1))(*[ctypes.c_void_p(p) for p in ptrs])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def grouped_gemm_bf16(A_ptr: int, B_ptrs: list, D_ptr: int, offsets_ptr: int, G: int, M_total: int,
                      N: int, K: int, stream: int) -> None:
    p, keep = _ptr_array(B_ptrs)
    _check(lib().grouped_gemm_bf16(A_ptr, p, D_ptr, offsets_ptr, G, M_total, N, K, stream),
           "grouped_gemm_bf16")
    del keep


def grouped_gemm_fp16(A_ptr: int, B_ptrs: list, D_ptr: int, offsets_ptr: int, G: int, M_total: int,
                      N: int, K: int, stream: int) -> None:
    p, keep = _ptr_array(B_ptrs)
    _check(lib().grouped_gemm_fp16(A_ptr, p, D_ptr, offsets_ptr, G, M_total, N, K, stream),
           "grouped_gemm_fp16")
    del keep


def gemm_bf16_host(A_host: torch.Tensor, B_host: torch.Tensor, D_host: torch.Tensor,
                   dA: torch.Tensor, dB: torch.Tensor, dD: torch.Tensor, stream=None) -> None:
    """Host-buffer form: copies in, multiplies, copies out; `stream` completes
    after the last copy back (the library pipelines over row chunks)."""
    M, K = A_host.shape
    N = B_host.shape[1]
    if D_host.dtype not in _OUT_CODES:
        raise TypeError("output dtype must be bfloat16, float16 or float32")
    if A_host.dtype != torch.bfloat16 or B_host.dtype != torch.bfloat16:
        raise TypeError("A_host and B_host must be bfloat16")
    if B_host.shape[0] != K or tuple(D_host.shape) != (M, N):
        raise ValueError("shapes must be A [M, K], B [K, N], D [M, N]; got %s, %s, %s"
                         % (tuple(A_host.shape), tuple(B_host.shape), tuple(D_host.shape)))
    for name, t in (("A_host", A_host), ("B_host", B_host), ("D_host", D_host)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a dense host tensor" % name)
    need = {"dA": M * K * 2, "dB": K * N * 2, "dD": M * N * D_host.element_size()}
    for name, t in (("dA", dA), ("dB", dB), ("dD", dD)):
        if not t.is_cuda or not t.is_contiguous() or t.numel() * t.element_size() < need[name]:
            raise ValueError("%s must be a dense CUDA buffer of at least %d bytes" % (name, need[name]))
    _check(lib().gemm_bf16_host(A_host.data_ptr(), B_host.data_ptr(), D_host.data_ptr(), M, N, K,
                                _OUT_CODES[D_host.dtype], dA.data_ptr(), dB.data_ptr(), dD.data_ptr(),
                                _stream_handle(stream, dA.device)), "gemm_bf16_host")


def last_device_error(stream=None) -> tuple[int, int]:
    """(status, raw error word) of the current device; clears the word."""
    info = ctypes.c_ulonglong(0)
    handle = _stream_handle(stream, torch.cuda.current_device()) if torch.cuda.is_available() else 0
    st = lib().bwg_last_device_error(handle, ctypes.byref(info))
    return st, info.value


def set_watchdog_ns(ns: int) -> None:
    lib().bwg_set_watchdog_ns(int(ns))


def debug_set_trace(buffer: "torch.Tensor | None") -> None:
    """Profiling hook: per-CTA unit timestamps into `buffer` (int64 CUDA
    tensor of at least grid * 64 * 3 entries), or None to switch off."""
    lib().bwg_debug_set_trace(None if buffer is None else buffer.data_ptr())


def debug_set_tx_extra(nbytes: int) -> None:
    lib().bwg_debug_set_tx_extra(int(nbytes))


def plan(M: int, N: int, K: int, out_dtype: int = OUT_BF16, sm_count: int = 152,
         force_kernel: int = 0, force_stages: int = 0) -> PlanInfo:
    info = PlanInfo()
    _check(lib().bwg_plan(M, N, K, out_dtype, sm_count, force_kernel, force_stages, ctypes.byref(info)),
           "bwg_plan")
    return info


def check_gemm_args(A: int, B: int, D: int, M: int, N: int, K: int, lda: int, ldb: int, ldd: int,
                    out_dtype: int) -> int:
    return int(lib().bwg_check_gemm_args(A, B, D, M, N, K, lda, ldb, ldd, out_dtype))


def grouped_gemm_swiglu_bf16(A_ptr: int, B_ptrs: list, H_ptr: int, offsets_ptr: int, G: int,
                             M_total: int, N: int, K: int, stream: int) -> None:
    p, keep = _ptr_array(B_ptrs)
    _check(lib().grouped_gemm_swiglu_bf16(A_ptr, p, H_ptr, offsets_ptr, G, M_total, N, K, stream),
           "grouped_gemm_swiglu_bf16")
    del keep


def grouped_gemm_swiglu_fp16(A_ptr: int, B_ptrs: list, H_ptr: int, offsets_ptr: int, G: int,
                             M_total: int, N: int, K: int, stream: int) -> None:
    p, keep = _ptr_array(B_ptrs)
    _check(lib().grouped_gemm_swiglu_fp16(A_ptr, p, H_ptr, offsets_ptr, G, M_total, N, K, stream),
           "grouped_gemm_swiglu_fp16")
    del keep


def _grouped_call(name: str, A_ptr: int, B_ptrs: list, D_ptr: int, offsets_ptr: int, G: int,
                  M_total: int, N: int, K: int, stream: int) -> None:
    p, keep = _ptr_array(B_ptrs)
    _check(getattr(lib(), name)(A_ptr, p, D_ptr, offsets_ptr, G, M_total, N, K, stream), name)
    del keep


def grouped_gemm_bf16_nt(A_ptr, B_ptrs, D_ptr, offsets_ptr, G, M_total, N, K, stream) -> None:
    """Grouped product with every B[g] stored [N, K]."""
    _grouped_call("grouped_gemm_bf16_nt", A_ptr, B_ptrs, D_ptr, offsets_ptr, G, M_total, N, K, stream)


def grouped_gemm_fp16_nt(A_ptr, B_ptrs, D_ptr, offsets_ptr, G, M_total, N, K, stream) -> None:
    _grouped_call("grouped_gemm_fp16_nt", A_ptr, B_ptrs, D_ptr, offsets_ptr, G, M_total, N, K, stream)


def grouped_gemm_swiglu_bf16_nt(A_ptr, B_ptrs, H_ptr, offsets_ptr, G, M_total, N, K, stream) -> None:
    _grouped_call("grouped_gemm_swiglu_bf16_nt", A_ptr, B_ptrs, H_ptr, offsets_ptr, G, M_total, N, K,
                  stream)


def grouped_gemm_swiglu_fp16_nt(A_ptr, B_ptrs, H_ptr, offsets_ptr, G, M_total, N, K, stream) -> None:
    _grouped_call("grouped_gemm_swiglu_fp16_nt", A_ptr, B_ptrs, H_ptr, offsets_ptr, G, M_total, N, K,
                  stream)
