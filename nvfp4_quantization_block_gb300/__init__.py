"""Python binding of the GB300 MXFP8 / per-token NVFP4 quantizer + block-scaled grouped GEMM library.

Argument marshalling only: every function here allocates its outputs with PyTorch (device memory),
passes raw pointers and the current CUDA stream to the C-ABI in ``libnvq.so`` (include/nvq.h) and
raises ``NvqError`` on a non-zero status. All arithmetic runs in the library's sm_103a kernels;
there is no CPU or PyTorch fallback, and importing this package fails loudly when the library has
not been built (``python nvfp4_quantization_block_gb300/build.py``).

Function names follow the C-ABI: ``mxfp8_quantize``, ``nvfp4_quantize_per_token``,
``nvfp4_quantize_weights``, ``dequantize_bf16``, ``block_scaled_grouped_gemm``.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python nvfp4_quantization_block_gb300/build.py)")

_lib = ctypes.CDLL(LIB_PATH)

NVQ_OK, NVQ_ERR_INVALID_ARG, NVQ_ERR_MISALIGNED, NVQ_ERR_UNSUPPORTED, NVQ_ERR_CUDA, NVQ_ERR_TIMEOUT = range(6)
SF_CANONICAL, SF_MMA = 0, 1
MXFP8, NVFP4, BF16 = 0, 1, 2
SCOPE_ROW, SCOPE_MATRIX = 0, 1
GEMM_GROUP_M, GEMM_GROUP_K = 0, 1
OUT_BF16, OUT_F32 = 0, 1
DEV_OK, DEV_TIMEOUT, DEV_BAD_OFFSETS, DEV_BAD_INDEX = 0, 1, 2, 3

_vp, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32


def _sig(name, args, res=ctypes.c_int):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = res
    return f


_status_string = _sig("nvq_status_string", [ctypes.c_int], ctypes.c_char_p)
_sf_bytes = _sig("nvq_sf_bytes", [_i64, _i64, _i32, ctypes.c_int], _i64)
_launch_count = _sig("nvq_launch_count", [], ctypes.c_uint64)
_mxfp8_quantize = _sig("mxfp8_quantize", [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, ctypes.c_int, _vp])
_nvfp4_quantize_per_token = _sig("nvfp4_quantize_per_token", [_vp, _i64, _i64, _i64, _vp, _vp, _vp, ctypes.c_int, _vp])
_nvfp4_quantize_dispatch = _sig("nvfp4_quantize_dispatch", [_vp, _i64, _i64, _i64, _vp, _i32, _i64, _vp, _vp, _vp,
                                                             ctypes.c_int, _vp, _vp])
_nvfp4_swiglu_quantize = _sig("nvfp4_swiglu_quantize_per_token", [_vp, _i64, _i64, _i64, _vp, _vp, _vp,
                                                                  ctypes.c_int, _vp])
_nvfp4_quantize_weights = _sig("nvfp4_quantize_weights", [_vp, _i64, _i64, _i64, _vp, _vp, _vp, ctypes.c_int, _vp])
_sf_layout_convert = _sig("sf_layout_convert", [_vp, ctypes.c_int, _i64, _i64, _vp, ctypes.c_int, _vp])
_quantized_gather_rows = _sig("quantized_gather_rows", [ctypes.c_int, _vp, _vp, _vp, _i64, _i64, ctypes.c_int, _vp,
                                                        _i64, _vp, _vp, _vp, ctypes.c_int, _vp, _vp])
_dequantize_bf16 = _sig("dequantize_bf16", [ctypes.c_int, _vp, _vp, _vp, ctypes.c_int, _i64, _i64, _i64,
                                            ctypes.c_int, _vp, _vp])


class GemmArgs(ctypes.Structure):
    """Mirror of ``nvq_gemm_args`` (include/nvq.h)."""
    _fields_ = [
        ("fmt", ctypes.c_int), ("mode", ctypes.c_int), ("out_type", ctypes.c_int),
        ("groups", _i64), ("m", _i64), ("n", _i64), ("k", _i64),
        ("a", _vp), ("sfa", _vp), ("s_a", _vp),
        ("b", _vp), ("sfb", _vp), ("s_b", _vp),
        ("offsets", _vp), ("d", _vp), ("ldd", _i64), ("status", _vp),
        ("wait_limit_ns", _i64), ("inject_timeout_stage", ctypes.c_int32),
    ]


_gemm = None
if hasattr(_lib, "block_scaled_grouped_gemm"):
    _gemm = _sig("block_scaled_grouped_gemm", [ctypes.POINTER(GemmArgs), _vp])


class NvqError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def status_string(status):
    return _status_string(int(status)).decode()


def _check(status, where):
    if status != NVQ_OK:
        raise NvqError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _layout(sf_layout):
    if sf_layout in ("mma", SF_MMA):
        return SF_MMA
    if sf_layout in ("canonical", SF_CANONICAL):
        return SF_CANONICAL
    raise ValueError(sf_layout)


def launch_count():
    """Kernels enqueued by the library so far (host-side counter)."""
    return int(_launch_count())


def sf_bytes(rows, cols, block, sf_layout="mma"):
    n = _sf_bytes(int(rows), int(cols), int(block), _layout(sf_layout))
    if n < 0:
        raise ValueError("invalid scale-matrix shape")
    return n


def _check_input(x, ndim):
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != ndim:
        raise ValueError(f"expected a {ndim}-D bf16 CUDA tensor")
    if x.numel() and x.stride(-1) != 1:
        raise ValueError("innermost dimension must be contiguous")


def mxfp8_quantize(x, rowwise=True, colwise=True, sf_layout="mma", out=None):
    """MXFP8 rowwise (1x32) and/or columnwise (32x1, stored transposed) copies of bf16 X [M, K].

    Returns a dict with q_row [M,K] u8, sf_row, q_colT [K,M] u8, sf_colT (as requested). ``out``
    may supply preallocated tensors under the same keys.
    """
    _check_input(x, 2)
    M, K = x.shape
    lay = _layout(sf_layout)
    o = dict(out or {})
    dev = x.device
    if rowwise:
        o.setdefault("q_row", torch.empty((M, K), dtype=torch.uint8, device=dev))
        o.setdefault("sf_row", torch.empty(sf_bytes(M, K, 32, lay), dtype=torch.uint8, device=dev))
    if colwise:
        o.setdefault("q_colT", torch.empty((K, M), dtype=torch.uint8, device=dev))
        o.setdefault("sf_colT", torch.empty(sf_bytes(K, M, 32, lay), dtype=torch.uint8, device=dev))
    st = _mxfp8_quantize(_ptr(x), M, K, x.stride(0) if M else K, _ptr(o.get("q_row")), _ptr(o.get("sf_row")),
                         _ptr(o.get("q_colT")), _ptr(o.get("sf_colT")), lay, _stream(dev))
    _check(st, "mxfp8_quantize")
    return o


def nvfp4_quantize_per_token(x, sf_layout="mma", out=None):
    """Per-token NVFP4 of bf16 X [T, K] -> (q [T, K/2] u8, sf u8, s_tok [T] f32)."""
    _check_input(x, 2)
    T, K = x.shape
    lay = _layout(sf_layout)
    dev = x.device
    if out is None:
        out = (torch.empty((T, K // 2), dtype=torch.uint8, device=dev),
               torch.empty(sf_bytes(T, K, 16, lay), dtype=torch.uint8, device=dev),
               torch.empty(T, dtype=torch.float32, device=dev))
    q, sf, s = out
    st = _nvfp4_quantize_per_token(_ptr(x), T, K, x.stride(0) if T else K, _ptr(q), _ptr(sf), _ptr(s), lay, _stream(dev))
    _check(st, "nvfp4_quantize_per_token")
    return q, sf, s


def nvfp4_swiglu_quantize_per_token(gate_up, sf_layout="mma", out=None):
    """SwiGLU of a fused gate||up activation [T, 2I] (bf16) quantized per token to NVFP4 ->
    (q [T, I/2] u8, sf u8, s_tok [T] f32), without writing the bf16 activation."""
    _check_input(gate_up, 2)
    T, I2 = gate_up.shape
    if I2 % 2:
        raise ValueError("gate_up needs an even number of columns")
    I = I2 // 2
    lay = _layout(sf_layout)
    dev = gate_up.device
    if out is None:
        out = (torch.empty((T, I // 2), dtype=torch.uint8, device=dev),
               torch.empty(sf_bytes(T, I, 16, lay), dtype=torch.uint8, device=dev),
               torch.empty(T, dtype=torch.float32, device=dev))
    q, sf, s = out
    st = _nvfp4_swiglu_quantize(_ptr(gate_up), T, I, gate_up.stride(0) if T else I2, _ptr(q), _ptr(sf), _ptr(s),
                                lay, _stream(dev))
    _check(st, "nvfp4_swiglu_quantize_per_token")
    return q, sf, s


def nvfp4_quantize_dispatch(x, dest, rows, sf_layout="mma", out=None, status=None):
    """Quantize-once dispatch: per-token NVFP4 of the tokens x [T, K] (bf16 CUDA), written to the
    routed rows dest [T, topk] (int32 CUDA, -1 = not dispatched) of (q [rows, K/2], sf, s [rows]).
    Routed rows named by no entry are left as they are (fresh outputs: undefined there)."""
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or (x.shape[0] and x.stride(1) != 1):
        raise ValueError("expected a 2-D bf16 CUDA tensor with unit column stride")
    if dest.dtype != torch.int32 or dest.dim() != 2 or not dest.is_contiguous() or dest.shape[0] != x.shape[0]:
        raise ValueError("dest must be a contiguous int32 [tokens, topk] tensor")
    T, K = x.shape
    lay = _layout(sf_layout)
    dev = x.device
    if out is None:
        out = (torch.empty((rows, K // 2), dtype=torch.uint8, device=dev),
               torch.empty(sf_bytes(rows, K, 16, lay), dtype=torch.uint8, device=dev),
               torch.empty(rows, dtype=torch.float32, device=dev))
    q, sf, s = out
    ldx = x.stride(0) if T else K                        # an empty tensor may report stride 0
    st = _nvfp4_quantize_dispatch(_ptr(x), T, K, ldx, _ptr(dest), int(dest.shape[1]), int(rows), _ptr(q),
                                  _ptr(sf), _ptr(s), lay, _ptr(status), _stream(dev))
    _check(st, "nvfp4_quantize_dispatch")
    return q, sf, s


def nvfp4_quantize_weights(w, sf_layout="mma", out=None):
    """NVFP4 expert weights W [E, K, N] (bf16, contiguous) -> (qT [E, N, K/2], sfT, s_w [E])."""
    if not w.is_cuda or w.dtype != torch.bfloat16 or w.dim() != 3 or not w.is_contiguous():
        raise ValueError("expected a contiguous 3-D bf16 CUDA tensor")
    E, K, N = w.shape
    lay = _layout(sf_layout)
    dev = w.device
    if out is None:
        out = (torch.empty((E, N, K // 2), dtype=torch.uint8, device=dev),
               torch.empty(sf_bytes(E * N, K, 16, lay), dtype=torch.uint8, device=dev),
               torch.empty(E, dtype=torch.float32, device=dev))
    q, sf, s = out
    st = _nvfp4_quantize_weights(_ptr(w), E, K, N, _ptr(q), _ptr(sf), _ptr(s), lay, _stream(dev))
    _check(st, "nvfp4_quantize_weights")
    return q, sf, s


def sf_layout_convert(sf, rows, kb, src_layout, dst_layout, out=None):
    """Permute block scales [rows, kb] between the canonical and the MMA tile layout."""
    src, dst = _layout(src_layout), _layout(dst_layout)
    if out is None:
        n = rows * kb if dst == SF_CANONICAL else sf_bytes(rows, kb * 16, 16, SF_MMA)
        out = torch.empty(n, dtype=torch.uint8, device=sf.device)
    st = _sf_layout_convert(_ptr(sf), src, int(rows), int(kb), _ptr(out), dst, _stream(sf.device))
    _check(st, "sf_layout_convert")
    return out


def quantized_gather_rows(fmt, q, sf, s, index, cols, src_layout="mma", dst_layout="mma", out=None, status=None):
    """Rows ``index`` (int32 CUDA tensor, -1 = zero row) of quantized rows (q, sf[, s]) -> new
    (q, sf, s) in ``dst_layout`` (s is None for MXFP8)."""
    src_rows = q.shape[0]
    rows = index.numel()
    dev = index.device
    block = 16 if fmt == NVFP4 else 32
    qb = cols // 2 if fmt == NVFP4 else cols
    dst = _layout(dst_layout)
    if out is None:
        out = (torch.empty((rows, qb), dtype=torch.uint8, device=dev),
               torch.empty(sf_bytes(rows, cols, block, dst), dtype=torch.uint8, device=dev),
               torch.empty(rows, dtype=torch.float32, device=dev) if fmt == NVFP4 else None)
    qo, sfo, so = out
    st = _quantized_gather_rows(int(fmt), _ptr(q), _ptr(sf), _ptr(s), int(src_rows), int(cols), _layout(src_layout),
                                _ptr(index), int(rows), _ptr(qo), _ptr(sfo), _ptr(so), dst, _ptr(status), _stream(dev))
    _check(st, "quantized_gather_rows")
    return qo, sfo, so


def dequantize_bf16(fmt, q, sf, s=None, scope=SCOPE_ROW, groups=1, rows=None, cols=None,
                    sf_layout="mma", out=None):
    """BF16 reconstruction [groups*rows, cols] of MXFP8 (fmt=MXFP8) or NVFP4 (fmt=NVFP4) data."""
    dev = q.device
    total = q.shape[0] if q.dim() == 2 else q.shape[0] * q.shape[1]
    if cols is None:
        cols = q.shape[-1] * (2 if fmt == NVFP4 else 1)
    if rows is None:
        rows = total // groups
    if out is None:
        out = torch.empty((groups * rows, cols), dtype=torch.bfloat16, device=dev)
    st = _dequantize_bf16(int(fmt), _ptr(q), _ptr(sf), _ptr(s), int(scope), int(groups), int(rows), int(cols),
                          _layout(sf_layout), _ptr(out), _stream(dev))
    _check(st, "dequantize_bf16")
    return out


def block_scaled_grouped_gemm(fmt, mode, a, sfa, b, sfb, offsets, m, n, k, groups, s_a=None, s_b=None,
                              out=None, out_type=OUT_BF16, status=None, wait_limit_ns=0, inject_timeout_stage=0):
    """Block-scaled grouped GEMM (include/nvq.h). ``offsets`` is a device int64 tensor [groups+1].

    mode GEMM_GROUP_M: D [m, n]; mode GEMM_GROUP_K: D [groups, m, n]. Returns D. ``wait_limit_ns``
    bounds each pipeline wait (0 = 2 s); ``inject_timeout_stage`` > 0 is the watchdog-test hook.
    """
    if _gemm is None:
        raise NvqError(NVQ_ERR_UNSUPPORTED, "block_scaled_grouped_gemm (not built)")
    dev = a.device
    dt = torch.bfloat16 if out_type == OUT_BF16 else torch.float32
    if out is None:
        shape = (m, n) if mode == GEMM_GROUP_M else (groups, m, n)
        out = torch.empty(shape, dtype=dt, device=dev)
    if offsets.dtype != torch.int64 or not offsets.is_cuda:
        raise ValueError("offsets must be a CUDA int64 tensor")
    args = GemmArgs(fmt=int(fmt), mode=int(mode), out_type=int(out_type), groups=int(groups), m=int(m),
                    n=int(n), k=int(k), a=_ptr(a), sfa=_ptr(sfa), s_a=_ptr(s_a), b=_ptr(b), sfb=_ptr(sfb),
                    s_b=_ptr(s_b), offsets=_ptr(offsets), d=_ptr(out), ldd=int(out.stride(-2)),
                    status=_ptr(status), wait_limit_ns=int(wait_limit_ns),
                    inject_timeout_stage=int(inject_timeout_stage))
    st = _gemm(ctypes.byref(args), _stream(dev))
    _check(st, "block_scaled_grouped_gemm")
    return out
