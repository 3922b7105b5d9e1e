"""The C-ABI library builds for sm_103a, loads, exports every entry point include/nvq.h declares,
and rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvq.h")
LIB = os.path.join(ROOT, "nvfp4_quantization_block_gb300", "libnvq.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    return ctypes.CDLL(LIB)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for required in ["mxfp8_quantize", "nvfp4_quantize_per_token", "nvfp4_quantize_weights",
                     "dequantize_bf16", "block_scaled_grouped_gemm", "nvq_status_string", "nvq_sf_bytes"]:
        assert required in names, required


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libnvq.so does not export {name}"


def test_sf_bytes_and_status_strings(lib):
    f = lib.nvq_sf_bytes
    f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int]
    f.restype = ctypes.c_int64
    assert f(256, 512, 32, 0) == 256 * 16
    assert f(256, 512, 32, 1) == 256 * 16
    assert f(300, 512, 16, 1) == 384 * 32
    assert f(300, 48, 16, 1) == 384 * 4          # 3 scale columns pad to 4
    assert f(10, 33, 32, 0) == -1
    s = lib.nvq_status_string
    s.argtypes = [ctypes.c_int]
    s.restype = ctypes.c_char_p
    assert s(0) == b"NVQ_OK" and s(2) == b"NVQ_ERR_MISALIGNED"


def test_host_validation_rejects_before_launch(lib):
    q = lib.mxfp8_quantize
    vp = ctypes.c_void_p
    q.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vp, vp, vp, ctypes.c_int, vp]
    q.restype = ctypes.c_int
    fake = vp(0x10000)          # never dereferenced: every call below fails validation first
    odd = vp(0x10008)
    assert q(fake, -1, 64, 64, fake, fake, None, None, 1, None) == 1          # negative rows
    assert q(fake, 64, 48, 64, fake, fake, None, None, 1, None) == 1          # cols % 32
    assert q(fake, 48, 64, 64, None, None, fake, fake, 1, None) == 1          # colwise needs rows % 32
    assert q(fake, 64, 64, 64, fake, None, None, None, 1, None) == 1          # q without sf
    assert q(odd, 64, 64, 64, fake, fake, None, None, 1, None) == 2           # misaligned input
    assert q(fake, 64, 64, 60, fake, fake, None, None, 1, None) == 1          # ld < cols
    assert q(fake, 64, 64, 68, fake, fake, None, None, 1, None) == 2          # ld % 8
    assert q(fake, 64, 64, 64, fake, fake, None, None, 7, None) == 1          # bad layout enum
    assert q(fake, 0, 64, 64, fake, fake, None, None, 1, None) == 0           # empty is a no-op
    t = lib.nvfp4_quantize_per_token
    t.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vp, vp, ctypes.c_int, vp]
    t.restype = ctypes.c_int
    assert t(fake, 4, 40, 40, fake, fake, fake, 0, None) == 1                 # cols % 16
    assert t(fake, 4, 64, 64, fake, fake, None, 0, None) == 1                 # missing s_tok
    assert t(fake, 0, 64, 64, None, None, None, 0, None) == 0
    assert t(fake, 4, (1 << 30) + 16, (1 << 30) + 16, fake, fake, fake, 0, None) == 1   # cols > 2^30
    assert t(fake, (1 << 32) + 1, 64, 64, fake, fake, fake, 0, None) == 1               # rows > 2^32
    sw = lib.nvfp4_swiglu_quantize_per_token
    sw.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vp, vp, ctypes.c_int, vp]
    sw.restype = ctypes.c_int
    assert sw(fake, 4, 40, 80, fake, fake, fake, 0, None) == 1     # cols % 16
    assert sw(fake, 4, 64, 100, fake, fake, fake, 0, None) == 1    # ld < 2 cols
    assert sw(fake, 4, 64, 132, fake, fake, fake, 0, None) == 2    # ld % 8
    assert sw(fake, 0, 64, 128, None, None, None, 0, None) == 0    # empty is a no-op
    assert sw(fake, 4, (1 << 30) + 16, (1 << 31) + 32, fake, fake, fake, 0, None) == 1   # cols > 2^30
    nw = lib.nvfp4_quantize_weights
    nw.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vp, vp, ctypes.c_int, vp]
    nw.restype = ctypes.c_int
    assert nw(fake, 2, 40, 64, fake, fake, fake, 1, None) == 1        # K % 16
    assert nw(fake, 2, 64, 60, fake, fake, fake, 1, None) == 1        # N % 8
    assert nw(fake, 65536, 64, 64, fake, fake, fake, 1, None) == 1    # more experts than the grid allows
    assert nw(fake, 2, 64, 64, fake, fake, None, 1, None) == 1        # missing s_w
    assert nw(fake, 2, 64, 64, fake, fake, fake, 3, None) == 1        # bad layout enum
    assert nw(odd, 2, 64, 64, fake, fake, fake, 1, None) == 2         # misaligned weights
    assert nw(fake, 2, 64, 64, fake, fake, odd, 1, None) == 2         # misaligned s_w
    assert nw(fake, 0, 64, 64, None, None, None, 1, None) == 0        # no experts is a no-op
    dq = lib.nvfp4_quantize_dispatch
    dq.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, ctypes.c_int32, ctypes.c_int64, vp, vp,
                   vp, ctypes.c_int, vp, vp]
    dq.restype = ctypes.c_int
    assert dq(fake, 4, 40, 64, fake, 2, 8, fake, fake, fake, 1, None, None) == 1       # cols % 16
    assert dq(fake, 4, 64, 64, fake, 0, 8, fake, fake, fake, 1, None, None) == 1       # topk < 1
    assert dq(fake, 4, 64, 64, fake, 33, 8, fake, fake, fake, 1, None, None) == 1      # topk > 32
    assert dq(fake, 4, 16400, 16400, fake, 2, 8, fake, fake, fake, 1, None, None) == 1  # cols > 16384
    assert dq(fake, 4, 64, 48, fake, 2, 8, fake, fake, fake, 1, None, None) == 1       # ldx < cols
    assert dq(fake, 4, 64, 64, None, 2, 8, fake, fake, fake, 1, None, None) == 1       # missing dest
    assert dq(fake, 4, 64, 64, fake, 2, 8, fake, fake, fake, 2, None, None) == 1       # bad layout enum
    assert dq(odd, 4, 64, 64, fake, 2, 8, fake, fake, fake, 1, None, None) == 2        # misaligned x
    assert dq(fake, 4, 64, 68, fake, 2, 8, fake, fake, fake, 1, None, None) == 2       # ldx % 8
    assert dq(fake, 4, 64, 64, fake, 2, 8, fake, fake, vp(0x10002), 1, None, None) == 2  # s_tok not 4-aligned
    assert dq(fake, 4, 64, 64, vp(0x10002), 2, 8, fake, fake, fake, 1, None, None) == 2  # dest not 4-aligned
    assert dq(fake, 0, 64, 64, None, 2, 0, None, None, None, 1, None, None) == 0       # empty is a no-op
    cv = lib.sf_layout_convert
    cv.argtypes = [vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, vp, ctypes.c_int, vp]
    cv.restype = ctypes.c_int
    assert cv(fake, 0, 8, 4, fake, 0, None) == 1                 # same layout both sides
    assert cv(fake, 0, 8, 4, odd, 1, None) == 2                  # misaligned destination
    assert cv(fake, 0, 0, 4, fake, 1, None) == 0                 # empty is a no-op
    g = lib.quantized_gather_rows
    g.argtypes = [ctypes.c_int, vp, vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, vp, ctypes.c_int64,
                  vp, vp, vp, ctypes.c_int, vp, vp]
    g.restype = ctypes.c_int
    assert g(1, fake, fake, fake, 4, 40, 1, fake, 8, fake, fake, fake, 1, None, None) == 1   # cols % 16
    assert g(1, fake, fake, None, 4, 64, 1, fake, 8, fake, fake, fake, 1, None, None) == 1   # NVFP4 needs s
    assert g(0, fake, fake, None, 4, 48, 1, fake, 8, fake, fake, None, 1, None, None) == 1   # MXFP8 cols % 32
    assert g(1, fake, fake, fake, 4, 64, 1, None, 8, fake, fake, fake, 1, None, None) == 1   # no index
    assert g(1, odd, fake, fake, 4, 64, 1, fake, 8, fake, fake, fake, 1, None, None) == 2    # misaligned q
    assert g(1, fake, fake, fake, 4, 64, 1, fake, 0, None, None, None, 1, None, None) == 0   # no rows
    odd4 = vp(0x10002)                                                                       # not 4-byte aligned
    assert g(1, fake, fake, fake, 4, 64, 1, odd4, 8, fake, fake, fake, 1, None, None) == 2   # index
    assert g(1, fake, fake, odd4, 4, 64, 1, fake, 8, fake, fake, fake, 1, None, None) == 2   # s
    assert g(1, fake, fake, fake, 4, 64, 1, fake, 8, fake, fake, odd4, 1, None, None) == 2   # s_out
    assert g(1, fake, fake, fake, 4, 64, 1, fake, 8, fake, fake, fake, 1, odd4, None) == 2   # status
    d = lib.dequantize_bf16
    d.argtypes = [ctypes.c_int, vp, vp, vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int, vp, vp]
    d.restype = ctypes.c_int
    assert d(1, fake, fake, None, 0, 1, 4, 32, 0, fake, None) == 1            # NVFP4 needs s
    assert d(5, fake, fake, None, 0, 1, 4, 32, 0, fake, None) == 1            # bad format


class _GemmArgs(ctypes.Structure):
    # field order and types of nvq_gemm_args in include/nvq.h
    _fields_ = [("fmt", ctypes.c_int), ("mode", ctypes.c_int), ("out_type", ctypes.c_int),
                ("groups", ctypes.c_int64), ("m", ctypes.c_int64), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
                ("a", ctypes.c_void_p), ("sfa", ctypes.c_void_p), ("s_a", ctypes.c_void_p),
                ("b", ctypes.c_void_p), ("sfb", ctypes.c_void_p), ("s_b", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("d", ctypes.c_void_p), ("ldd", ctypes.c_int64),
                ("status", ctypes.c_void_p), ("wait_limit_ns", ctypes.c_int64),
                ("inject_timeout_stage", ctypes.c_int32)]


def test_gemm_host_validation_rejects_before_launch(lib):
    g = lib.block_scaled_grouped_gemm
    g.argtypes = [ctypes.POINTER(_GemmArgs), ctypes.c_void_p]
    g.restype = ctypes.c_int
    fake, odd = 0x10000, 0x10008                    # never dereferenced: each call fails on the host

    def call(**over):
        a = _GemmArgs(fmt=1, mode=0, out_type=0, groups=2, m=256, n=256, k=256, a=fake, sfa=fake, s_a=None,
                      b=fake, sfb=fake, s_b=None, offsets=fake, d=fake, ldd=256, status=None)
        for key, v in over.items():
            setattr(a, key, v)
        return g(ctypes.byref(a), None)

    assert g(None, None) == 1                       # no argument block
    assert call(fmt=3) == 1                         # bad format
    assert call(mode=2) == 1                        # bad grouping mode
    assert call(out_type=2) == 1                    # bad output type
    assert call(k=-128) == 1                        # negative size
    assert call(groups=0) == 0                      # nothing to do
    assert call(m=0) == 0
    assert call(groups=1025) == 3                   # above the 1024-group maximum
    assert call(sfa=None) == 1                      # block-scaled operands need their scales
    assert call(fmt=2, sfa=None, sfb=None, n=200) == 1   # N % 128 (BF16 operands need no scales)
    assert call(k=96) == 1                          # row-grouped block-scaled K % 128
    assert call(ldd=200) == 1                       # ldd < n
    assert call(ldd=260) == 1                       # ldd % 8
    assert call(mode=1) == 3                        # NVFP4 weight gradient: not built
    assert call(fmt=0, mode=1, m=200) == 1          # weight gradient: M % 128
    assert call(a=odd) == 2                         # misaligned operand
    assert call(offsets=fake + 4) == 2              # offsets not 8-byte aligned
    assert call(wait_limit_ns=-1) == 1              # negative wait limit
    assert call(inject_timeout_stage=-1) == 1       # negative injection stage
