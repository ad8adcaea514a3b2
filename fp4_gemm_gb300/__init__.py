"""Block-scaled FP8 / MXFP4 GEMM for GB300 (sm_103a): Python binding.

A thin ctypes layer over libbsg.so (include/bsg.h).  The functions carry the
C entry points' names and only marshal arguments: torch allocates device
memory and supplies the current stream; every step of the computation runs in
the library's CUDA kernels.  There is no fallback: if libbsg.so has not been
built, or no GPU is present, calls raise.

    q, s   = bsg_quantize_fp8(x, "e4m3", "row")          # x: (rows, K) fp32/bf16 CUDA
    qb, sf = bsg_quantize_mxfp4(w, layout="tcgen05")      # packed E2M1 + E8M0 scales
    D      = bsg_gemm(qa, "e4m3", sa, "row", qw, "e4m3", sw, "tile", out="bf16")

Operand B is K x N column-major, i.e. a (N, K) row-major tensor; D = A B.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbsg.so")

# enum values of include/bsg.h
STATUS = {0: "BSG_OK", 1: "BSG_ERR_INVALID_ARG", 2: "BSG_ERR_UNSUPPORTED", 3: "BSG_ERR_ALIGNMENT",
          4: "BSG_ERR_CUDA", 5: "BSG_ERR_TIMEOUT", 6: "BSG_ERR_WORKSPACE"}
FORMAT = {"e4m3": 0, "e5m2": 1, "e2m1": 2}
DTYPE = {"f32": 0, "bf16": 1}
GRAN = {"tile": 0, "row": 1, "mx": 2, "nv": 3, "bf16": 4, "f16": 5}
LAYOUT = {"rowmajor": 0, "tcgen05": 1}

EXPORTS = ("bsg_quantize_fp8", "bsg_quantize_mxfp4", "bsg_gemm", "bsg_gemm_workspace_size",
           "bsg_scale_bytes", "bsg_sf_to_tcgen05", "bsg_status_string", "bsg_device_error",
           "bsg_num_sms", "bsg_gemm_decode_noalloc", "bsg_mma_peak", "bsg_quantize_mx",
           "bsg_mma_probe", "bsg_gemm_quantized", "bsg_quantize_nvfp4", "bsg_gemm_nvfp4",
           "bsg_check_wait_timeout", "bsg_quantize_fp4_bs16", "bsg_mma_probe_mx",
           "bsg_gemm_mxfp4_act", "bsg_gemm_mxfp4_act_workspace_size", "bsg_gemm_nvfp4_ws")


class BsgError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libbsg.so and declare the C signatures.  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run fp4_gemm_gb300.build.build() "
                          "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    c = ctypes
    i64, vp, f32, i32, sz = c.c_int64, c.c_void_p, c.c_float, c.c_int, c.c_size_t
    lib.bsg_quantize_fp8.argtypes = [vp, i32, i64, i64, i64, i32, i32, f32, vp, vp, vp]
    lib.bsg_quantize_fp8.restype = i32
    lib.bsg_quantize_mxfp4.argtypes = [vp, i32, i64, i64, i64, vp, vp, i32, vp]
    lib.bsg_quantize_mxfp4.restype = i32
    lib.bsg_gemm.argtypes = [i64, i64, i64, vp, i32, vp, i32, vp, i32, vp, i32, vp, vp, i32, vp, sz, vp]
    lib.bsg_gemm.restype = i32
    lib.bsg_gemm_quantized.argtypes = [i64, i64, i64, vp, i32, vp, i32, vp, i32, vp, i32, vp, i32,
                                       f32, vp, vp, vp]
    lib.bsg_gemm_quantized.restype = i32
    lib.bsg_gemm_workspace_size.argtypes = [i64, i64, i64, i32, i32]
    lib.bsg_gemm_workspace_size.restype = sz
    lib.bsg_gemm_mxfp4_act.argtypes = [i64, i64, i64, vp, i32, i64, vp, vp, vp, vp, i32, vp, sz, vp]
    lib.bsg_gemm_mxfp4_act.restype = i32
    lib.bsg_gemm_mxfp4_act_workspace_size.argtypes = [i64, i64, i64]
    lib.bsg_gemm_mxfp4_act_workspace_size.restype = sz
    lib.bsg_scale_bytes.argtypes = [i64, i64, i32, i32]
    lib.bsg_scale_bytes.restype = sz
    lib.bsg_sf_to_tcgen05.argtypes = [vp, i64, i64, vp, vp]
    lib.bsg_sf_to_tcgen05.restype = i32
    lib.bsg_status_string.argtypes = [i32]
    lib.bsg_status_string.restype = c.c_char_p
    lib.bsg_device_error.argtypes = [vp]
    lib.bsg_device_error.restype = i32
    lib.bsg_num_sms.argtypes = []
    lib.bsg_num_sms.restype = i32
    lib.bsg_gemm_decode_noalloc.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp, vp, i32, vp]
    lib.bsg_gemm_decode_noalloc.restype = i32
    lib.bsg_quantize_mx.argtypes = [vp, i32, i64, i64, i64, i32, f32, vp, vp, i32, vp]
    lib.bsg_quantize_mx.restype = i32
    lib.bsg_quantize_nvfp4.argtypes = [vp, i32, i64, i64, i64, f32, vp, vp, i32, vp]
    lib.bsg_quantize_nvfp4.restype = i32
    lib.bsg_quantize_fp4_bs16.argtypes = [vp, i32, i64, i64, i64, i32, vp, vp, vp]
    lib.bsg_quantize_fp4_bs16.restype = i32
    lib.bsg_gemm_nvfp4.argtypes = [i64, i64, i64, vp, vp, vp, vp, f32, vp, vp, i32, vp]
    lib.bsg_gemm_nvfp4.restype = i32
    lib.bsg_gemm_nvfp4_ws.argtypes = [i64, i64, i64, vp, vp, vp, vp, f32, vp, vp, i32, vp, sz, vp]
    lib.bsg_gemm_nvfp4_ws.restype = i32
    lib.bsg_check_wait_timeout.argtypes = [vp]
    lib.bsg_check_wait_timeout.restype = i32
    lib.bsg_mma_peak.argtypes = [i32, i32, i32, i64, c.POINTER(i64), vp]
    lib.bsg_mma_probe.argtypes = [vp, i32, vp, i32, vp, vp, vp]
    lib.bsg_mma_probe.restype = i32
    lib.bsg_mma_probe_mx.argtypes = [i32, vp, vp, vp, vp, vp, vp, i32, i32, vp]
    lib.bsg_mma_probe_mx.restype = i32
    lib.bsg_mma_peak.restype = i32
    _lib = lib
    return lib


def _check(status: int, where: str):
    if status != 0:
        raise BsgError(status, where)


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("bsg: every tensor must live on the GPU")


# ----------------------------------------------------------------- sizes
def bsg_scale_bytes(rows: int, cols: int, gran: str, layout: str = "rowmajor") -> int:
    return int(load_library().bsg_scale_bytes(rows, cols, GRAN[gran], LAYOUT[layout]))


def bsg_gemm_workspace_size(M: int, N: int, K: int, fa: str, fb: str) -> int:
    return int(load_library().bsg_gemm_workspace_size(M, N, K, FORMAT[fa], FORMAT[fb]))


def bsg_num_sms() -> int:
    return int(load_library().bsg_num_sms())


def bsg_mma_peak(fmt: str = "e4m3", pair: bool = False, iters: int = 1 << 16,
                 block_scaled: bool = False, stream=None) -> int:
    """Launch the tensor-core throughput microbenchmark on `stream` (or the
    current stream) and return the FLOPs the launch performs; the caller
    times it with CUDA events.  fmt "e4m3" (kind::f8f6f4, or with
    block_scaled kind::mxf8f6f4) or "e2m1" (block-scaled kind::mxf4)."""
    flops = ctypes.c_int64(0)
    bs = 1 if (block_scaled or fmt == "e2m1") else 0
    _check(load_library().bsg_mma_peak(FORMAT[fmt], bs, 1 if pair else 0, int(iters),
                                       ctypes.byref(flops), _stream(stream)), "bsg_mma_peak")
    return int(flops.value)


def bsg_mma_probe(A: torch.Tensor, fa: str, B: torch.Tensor, fb: str, C: torch.Tensor,
                  stream=None) -> torch.Tensor:
    """One tcgen05.mma kind::f8f6f4: returns D (128, 16) float32 =
    A (128, 32) . B (16, 32)^T + C (128, 16); A, B uint8 FP8 codes."""
    if A.shape != (128, 32) or B.shape != (16, 32) or C.shape != (128, 16):
        raise ValueError("bsg_mma_probe takes A (128, 32), B (16, 32), C (128, 16)")
    A, B, C = A.contiguous(), B.contiguous(), C.contiguous().float()
    D = torch.empty((128, 16), dtype=torch.float32, device=A.device)
    _need_cuda(A, B, C, D)
    _check(load_library().bsg_mma_probe(_ptr(A), FORMAT[fa], _ptr(B), FORMAT[fb], _ptr(C), _ptr(D),
                                        _stream(stream)), "bsg_mma_probe")
    return D


def bsg_mma_probe_mx(kind: int, A: torch.Tensor, sfA: torch.Tensor, B: torch.Tensor,
                     sfB: torch.Tensor, C: torch.Tensor, fa: str = "e4m3", fb: str = "e4m3",
                     stream=None) -> torch.Tensor:
    """One block-scaled MMA (kind 0 MXFP8, 1 MXFP4, 2 NVFP4): returns D
    (128, 256) float32 from operand bytes A (128, 32), B (256, 32), scale
    cells sfA (128, 4), sfB (256, 4) (uint8) and C (128, 256)."""
    if (A.shape != (128, 32) or B.shape != (256, 32) or sfA.shape != (128, 4) or
            sfB.shape != (256, 4) or C.shape != (128, 256)):
        raise ValueError("bsg_mma_probe_mx takes A (128,32), B (256,32), sfA (128,4), sfB (256,4), C (128,256)")
    A, B, sfA, sfB = A.contiguous(), B.contiguous(), sfA.contiguous(), sfB.contiguous()
    C = C.contiguous().float()
    D = torch.empty((128, 256), dtype=torch.float32, device=A.device)
    _need_cuda(A, B, sfA, sfB, C, D)
    _check(load_library().bsg_mma_probe_mx(kind, _ptr(A), _ptr(sfA), _ptr(B), _ptr(sfB), _ptr(C),
                                           _ptr(D), FORMAT[fa], FORMAT[fb], _stream(stream)),
           "bsg_mma_probe_mx")
    return D


def bsg_status_string(status: int) -> str:
    return load_library().bsg_status_string(status).decode()


def bsg_check_wait_timeout(stream=None) -> None:
    """Launch the failure-detection self-check: a kernel whose only wait runs
    out after the library's limit.  The next bsg_device_error() returns
    BSG_ERR_TIMEOUT (5)."""
    _check(load_library().bsg_check_wait_timeout(_stream(stream)), "bsg_check_wait_timeout")


def bsg_device_error(stream=None) -> int:
    """Synchronise and return (and clear) the device error status (0 = OK)."""
    return int(load_library().bsg_device_error(_stream(stream)))


# ------------------------------------------------------------ quantisers
def bsg_quantize_fp8(x: torch.Tensor, fmt: str = "e4m3", gran: str = "tile",
                     fmt_max: float = 0.0, q: torch.Tensor | None = None,
                     scales: torch.Tensor | None = None, stream=None):
    """x: (rows, K) FP32 or BF16 CUDA tensor (row stride = leading dimension).
    Returns (codes uint8 (rows, K), scales float32): "tile" scales are
    (ceil(rows/128), ceil(K/128)); "row" scales are (ceil(K/128), rows)."""
    lib = load_library()
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit column stride")
    rows, cols = x.shape
    src = {torch.float32: 0, torch.bfloat16: 1}[x.dtype]
    kt = -(-cols // 128)
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scales is None:
        shape = (-(-rows // 128), kt) if gran == "tile" else (kt, rows)
        scales = torch.empty(shape, dtype=torch.float32, device=x.device)
    _need_cuda(x, q, scales)
    _check(lib.bsg_quantize_fp8(_ptr(x), src, rows, cols, x.stride(0), FORMAT[fmt], GRAN[gran],
                                float(fmt_max), _ptr(q), _ptr(scales), _stream(stream)),
           "bsg_quantize_fp8")
    return q, scales


def bsg_quantize_mxfp4(x: torch.Tensor, layout: str = "tcgen05", q: torch.Tensor | None = None,
                       sf: torch.Tensor | None = None, stream=None):
    """x: (rows, K) FP32 or BF16 CUDA tensor, K % 32 == 0.  Returns
    (packed uint8 (rows, K/2), E8M0 scales uint8): "rowmajor" scales are
    (rows, K/32); "tcgen05" scales are a flat buffer in the MMA's atom order."""
    lib = load_library()
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit column stride")
    rows, cols = x.shape
    src = {torch.float32: 0, torch.bfloat16: 1}[x.dtype]
    if q is None:
        q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=x.device)
    if sf is None:
        if layout == "rowmajor":
            sf = torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device)
        else:
            n = lib.bsg_scale_bytes(rows, cols, GRAN["mx"], LAYOUT["tcgen05"])
            sf = torch.empty((max(int(n), 1),), dtype=torch.uint8, device=x.device)
    _need_cuda(x, q, sf)
    _check(lib.bsg_quantize_mxfp4(_ptr(x), src, rows, cols, x.stride(0), _ptr(q), _ptr(sf),
                                  LAYOUT[layout], _stream(stream)), "bsg_quantize_mxfp4")
    return q, sf


def bsg_quantize_mx(x: torch.Tensor, fmt: str = "e4m3", layout: str = "tcgen05",
                    fmt_max: float = 0.0, q: torch.Tensor | None = None,
                    sf: torch.Tensor | None = None, stream=None):
    """MX quantisation, x: (rows, K) FP32 or BF16 CUDA tensor, K % 32 == 0.
    fmt "e4m3" / "e5m2" (MXFP8: codes uint8 (rows, K)) or "e2m1" (MXFP4:
    packed uint8 (rows, K/2)).  Returns (codes, E8M0 scales); "rowmajor"
    scales are (rows, K/32), "tcgen05" scales a flat buffer in the MMA's
    atom order."""
    lib = load_library()
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit column stride")
    rows, cols = x.shape
    src = {torch.float32: 0, torch.bfloat16: 1}[x.dtype]
    if q is None:
        q = torch.empty((rows, cols // 2 if fmt == "e2m1" else cols), dtype=torch.uint8,
                        device=x.device)
    if sf is None:
        if layout == "rowmajor":
            sf = torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device)
        else:
            n = lib.bsg_scale_bytes(rows, cols, GRAN["mx"], LAYOUT["tcgen05"])
            sf = torch.empty((max(int(n), 1),), dtype=torch.uint8, device=x.device)
    _need_cuda(x, q, sf)
    _check(lib.bsg_quantize_mx(_ptr(x), src, rows, cols, x.stride(0), FORMAT[fmt], float(fmt_max),
                               _ptr(q), _ptr(sf), LAYOUT[layout], _stream(stream)),
           "bsg_quantize_mx")
    return q, sf


def bsg_quantize_nvfp4(x: torch.Tensor, layout: str = "tcgen05", tensor_scale: float = 1.0,
                       q: torch.Tensor | None = None, sf: torch.Tensor | None = None, stream=None):
    """NVFP4 quantisation, x: (rows, K) FP32 or BF16 CUDA tensor, K % 16 == 0.
    Returns (packed E2M1 uint8 (rows, K/2), E4M3 scales): "rowmajor" scales
    are (rows, K/16), "tcgen05" scales a flat buffer in the MMA's atom order."""
    lib = load_library()
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit column stride")
    rows, cols = x.shape
    src = {torch.float32: 0, torch.bfloat16: 1}[x.dtype]
    if q is None:
        q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=x.device)
    if sf is None:
        if layout == "rowmajor":
            sf = torch.empty((rows, cols // 16), dtype=torch.uint8, device=x.device)
        else:
            n = lib.bsg_scale_bytes(rows, cols, GRAN["nv"], LAYOUT["tcgen05"])
            sf = torch.empty((max(int(n), 1),), dtype=torch.uint8, device=x.device)
    _need_cuda(x, q, sf)
    _check(lib.bsg_quantize_nvfp4(_ptr(x), src, rows, cols, x.stride(0), float(tensor_scale),
                                  _ptr(q), _ptr(sf), LAYOUT[layout], _stream(stream)),
           "bsg_quantize_nvfp4")
    return q, sf


def bsg_quantize_fp4_bs16(x: torch.Tensor, scale: str = "bf16", q: torch.Tensor | None = None,
                          sf: torch.Tensor | None = None, stream=None):
    """E2M1 quantisation with one 16-bit scale ("bf16" or "f16") per 32 along K,
    x: (rows, K) FP32 or BF16 CUDA tensor, K % 32 == 0.  Returns (packed uint8
    (rows, K/2), scale codes int16 (K/32, rows)); pass scale as the
    granularity of both operands to bsg_gemm."""
    lib = load_library()
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D tensor with unit column stride")
    rows, cols = x.shape
    src = {torch.float32: 0, torch.bfloat16: 1}[x.dtype]
    if q is None:
        q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty((cols // 32, rows), dtype=torch.int16, device=x.device)
    _need_cuda(x, q, sf)
    _check(lib.bsg_quantize_fp4_bs16(_ptr(x), src, rows, cols, x.stride(0), GRAN[scale], _ptr(q),
                                     _ptr(sf), _stream(stream)), "bsg_quantize_fp4_bs16")
    return q, sf


def bsg_gemm_nvfp4(A: torch.Tensor, sA: torch.Tensor, B: torch.Tensor, sB: torch.Tensor,
                   alpha: float = 1.0, C: torch.Tensor | None = None, out: str = "f32",
                   D: torch.Tensor | None = None, K: int | None = None,
                   workspace: torch.Tensor | None = None, stream=None):
    """D = alpha * sum_k (s_A a_k)(s_B b_k) + C for NVFP4 operands: A (M, K/2)
    and B (N, K/2) packed, sA / sB E4M3 scales in the tcgen05 layout.  Calls
    bsg_gemm_nvfp4_ws with the workspace bsg_gemm would use (cached per
    device), so that up to 32 rows take the decode-shaped kernel."""
    lib = load_library()
    M, N = A.shape[0], B.shape[0]
    if K is None:
        K = A.shape[1] * 2
    if D is None:
        D = torch.empty((M, N), dtype=torch.float32 if out == "f32" else torch.bfloat16,
                        device=A.device)
    if workspace is None:
        workspace = workspace_for(M, N, K, "e2m1", "e2m1", A.device)
    _need_cuda(A, sA, B, sB, C, D, workspace)
    _check(lib.bsg_gemm_nvfp4_ws(M, N, K, _ptr(A), _ptr(sA), _ptr(B), _ptr(sB), float(alpha), _ptr(C),
                                 _ptr(D), DTYPE[out], _ptr(workspace),
                                 0 if workspace is None else workspace.numel(), _stream(stream)),
           "bsg_gemm_nvfp4_ws")
    return D


def bsg_sf_to_tcgen05(sf_rowmajor: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    lib = load_library()
    rows, kb = sf_rowmajor.shape
    if out is None:
        n = lib.bsg_scale_bytes(rows, kb * 32, GRAN["mx"], LAYOUT["tcgen05"])
        out = torch.empty((int(n),), dtype=torch.uint8, device=sf_rowmajor.device)
    _need_cuda(sf_rowmajor, out)
    _check(lib.bsg_sf_to_tcgen05(_ptr(sf_rowmajor), rows, kb, _ptr(out), _stream(stream)),
           "bsg_sf_to_tcgen05")
    return out


# ------------------------------------------------------------------ GEMM
_workspaces: dict = {}


def workspace_for(M: int, N: int, K: int, fa: str, fb: str, device) -> torch.Tensor | None:
    """A zero-filled workspace of the size bsg_gemm needs, cached per device
    (the library leaves it zero-filled after each call, so it is reused)."""
    n = bsg_gemm_workspace_size(M, N, K, fa, fb)
    if n == 0:
        return None
    dev = torch.device(device)
    key = (dev.type, dev.index)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < n:
        ws = torch.zeros((n,), dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def bsg_gemm(A: torch.Tensor, fa: str, sA: torch.Tensor, ga: str,
             B: torch.Tensor, fb: str, sB: torch.Tensor, gb: str,
             C: torch.Tensor | None = None, out: str = "f32", D: torch.Tensor | None = None,
             workspace: torch.Tensor | None = None, K: int | None = None, stream=None):
    """D = sum_k (s_A a_k)(s_B b_k) + C.  A: (M, K) codes (E2M1: (M, K/2)
    packed); B: (N, K) codes (K x N column-major).  Returns D (M, N)."""
    lib = load_library()
    M = A.shape[0]
    N = B.shape[0]
    if K is None:
        K = A.shape[1] * (2 if fa == "e2m1" else 1)
    if D is None:
        D = torch.empty((M, N), dtype=torch.float32 if out == "f32" else torch.bfloat16,
                        device=A.device)
    if workspace is None:
        workspace = workspace_for(M, N, K, fa, fb, A.device)
    _need_cuda(A, sA, B, sB, C, D, workspace)
    _check(lib.bsg_gemm(M, N, K, _ptr(A), FORMAT[fa], _ptr(sA), GRAN[ga], _ptr(B), FORMAT[fb],
                        _ptr(sB), GRAN[gb], _ptr(C), _ptr(D), DTYPE[out], _ptr(workspace),
                        0 if workspace is None else workspace.numel(), _stream(stream)),
           "bsg_gemm")
    return D


_act_workspaces: dict = {}


def bsg_gemm_mxfp4_act_workspace_size(M: int, N: int, K: int) -> int:
    return int(load_library().bsg_gemm_mxfp4_act_workspace_size(M, N, K))


def bsg_gemm_mxfp4_act(x: torch.Tensor, B: torch.Tensor, sB: torch.Tensor,
                       C: torch.Tensor | None = None, out: str = "bf16", D: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """D = sum_k (s_A a_k)(s_B b_k) + C with the activations x (M, K; FP32 or
    BF16, rows may be padded) quantised to MXFP4 inside the call, exactly as
    bsg_quantize_mxfp4 would.  B: (N, K/2) packed E2M1, sB: tcgen05-layout
    E8M0 scales.  The workspace (zero-filled once) is cached per device and
    problem shape: after a call only its counters and partial sums are zero,
    its activation area is scratch, so another shape gets its own."""
    lib = load_library()
    M, K = x.shape
    N = B.shape[0]
    if x.dtype not in (torch.float32, torch.bfloat16) or x.stride(1) != 1:
        raise ValueError("x must be FP32 or BF16 with unit column stride")
    if D is None:
        D = torch.empty((M, N), dtype=torch.float32 if out == "f32" else torch.bfloat16, device=x.device)
    if workspace is None:
        n = max(bsg_gemm_mxfp4_act_workspace_size(M, N, K), 16)
        dev = torch.device(x.device)
        key = (dev.type, dev.index, M, N, K)
        ws = _act_workspaces.get(key)
        if ws is None or ws.numel() < n:
            ws = torch.zeros((n,), dtype=torch.uint8, device=dev)
            _act_workspaces[key] = ws
        workspace = ws
    _need_cuda(x, B, sB, C, D, workspace)
    _check(lib.bsg_gemm_mxfp4_act(M, N, K, _ptr(x), DTYPE["bf16" if x.dtype == torch.bfloat16 else "f32"],
                                  x.stride(0), _ptr(B), _ptr(sB), _ptr(C), _ptr(D), DTYPE[out],
                                  _ptr(workspace), workspace.numel(), _stream(stream)),
           "bsg_gemm_mxfp4_act")
    return D


def bsg_gemm_quantized(A: torch.Tensor, fa: str, sA: torch.Tensor, ga: str,
                       B: torch.Tensor, fb: str, sB: torch.Tensor, gb: str,
                       C: torch.Tensor | None = None, qfmt: str = "e4m3", fmt_max: float = 0.0,
                       Dq: torch.Tensor | None = None, sD: torch.Tensor | None = None,
                       stream=None):
    """The FP8 GEMM with its result quantised per 1x128 run of a row in the
    epilogue.  Returns (Dq (M, N) uint8 codes, sD (ceil(N/128), M) float32),
    ready to be the activation operand of the next bsg_gemm with "row" scales."""
    lib = load_library()
    M, N, K = A.shape[0], B.shape[0], A.shape[1]
    if Dq is None:
        Dq = torch.empty((M, N), dtype=torch.uint8, device=A.device)
    if sD is None:
        sD = torch.empty(((N + 127) // 128, M), dtype=torch.float32, device=A.device)
    _need_cuda(A, sA, B, sB, C, Dq, sD)
    _check(lib.bsg_gemm_quantized(M, N, K, _ptr(A), FORMAT[fa], _ptr(sA), GRAN[ga], _ptr(B),
                                  FORMAT[fb], _ptr(sB), GRAN[gb], _ptr(C), FORMAT[qfmt],
                                  float(fmt_max), _ptr(Dq), _ptr(sD), _stream(stream)),
           "bsg_gemm_quantized")
    return Dq, sD


def bsg_gemm_decode_noalloc(A: torch.Tensor, sA: torch.Tensor, B: torch.Tensor, sB: torch.Tensor,
                            C: torch.Tensor | None = None, out: str = "bf16",
                            D: torch.Tensor | None = None, K: int | None = None, stream=None):
    """The decode-shaped MXFP4 GEMM (M <= 32) using the library's built-in
    scratch instead of a workspace: for callers that cannot allocate.  Calls
    that overlap on the GPU race on that shared scratch."""
    lib = load_library()
    M, N = A.shape[0], B.shape[0]
    if K is None:
        K = A.shape[1] * 2
    if D is None:
        D = torch.empty((M, N), dtype=torch.float32 if out == "f32" else torch.bfloat16,
                        device=A.device)
    _need_cuda(A, sA, B, sB, C, D)
    _check(lib.bsg_gemm_decode_noalloc(M, N, K, _ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(C),
                                       _ptr(D), DTYPE[out], _stream(stream)),
           "bsg_gemm_decode_noalloc")
    return D
