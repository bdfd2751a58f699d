"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4k.h")


@pytest.fixture(scope="module")
def q4k():
    from quantized_prefill_gemm_gb300 import build

    build.build()
    from quantized_prefill_gemm_gb300 import q4k as mod

    return mod


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(q\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = header_functions()
    for required in ("q8_quantize_rows", "q4k_gemm", "q4k_pack_weights", "q4k_packed_bytes",
                     "q4k_gemm_workspace_bytes", "q4k_status_string"):
        assert required in names


def test_library_exports_every_header_symbol(q4k):
    lib = ctypes.CDLL(q4k.LIB_PATH)
    for name in header_functions():
        assert hasattr(lib, name), name
    # the binding declares exactly the header's functions
    assert set(q4k.SIGNATURES) == set(header_functions())


def test_status_strings_and_version(q4k):
    assert q4k.q4k_abi_version() == 1
    assert q4k.q4k_status_string(0) == "ok"
    assert "timed out" in q4k.q4k_status_string(7)
    assert q4k.q4k_status_string(99) == "unknown status"


def test_size_queries(q4k):
    assert q4k.q4k_packed_bytes(100, 256) == 0       # n % 128
    assert q4k.q4k_packed_bytes(128, 100) == 0       # k % 256
    n, k = 256, 512
    nb = q4k.q4k_packed_bytes(n, k)
    # quants n*k/2, sc n*k/32, d n*k/256*4, two bf16 planes n*k/32*2 each, 1 KiB-aligned sections
    assert nb >= n * k // 2 + n * k // 32 + n * k // 64 + 4 * n * k // 32
    assert nb % 1024 == 0
    m = 70
    ws = q4k.q4k_act_workspace_bytes(m, k)
    assert ws >= m * k * 2 + 128 * (k // 32) * 4 + 4 * m * (k // 32)
    assert q4k.q4k_gemm_workspace_bytes(m, n, k, 0) == ws
    assert q4k.q4k_gemm_workspace_bytes(m, n, k, 5) == 0


def test_host_validation_rejects_before_any_cuda_call(q4k):
    L = q4k.LIB
    null = None
    # q8_quantize_rows: k not a multiple of 32, ldx < k, null x, m == 0 no-op
    assert L.q8_quantize_rows(null, 4, 33, 33, null, null, null, null) == 2
    assert L.q8_quantize_rows(null, 4, 64, 32, null, null, null, null) == 2
    assert L.q8_quantize_rows(null, 4, 64, 64, null, null, null, null) == 1
    assert L.q8_quantize_rows(null, 0, 64, 64, null, null, null, null) == 0
    assert L.q8_quantize_rows(ctypes.c_void_p(8), 4, 64, 64, null, null, null, null) == 3   # misaligned x
    # q4k_pack_weights: shapes and nulls
    assert L.q4k_pack_weights(null, 100, 256, null, 0, null) == 2
    assert L.q4k_pack_weights(null, 128, 256, null, 0, null) == 1
    assert L.q4k_pack_weights(ctypes.c_void_p(256), 128, 256, ctypes.c_void_p(4096), 16, null) == 4
    # q4k_gemm: bad n / k / act / out / ld / workspace
    args = dict(w=ctypes.c_void_p(4096), x=ctypes.c_void_p(4096), y=ctypes.c_void_p(4096), ws=ctypes.c_void_p(4096))

    def gemm(n=256, k=512, act=0, m=8, ldx=512, out=0, ldy=256, ws_bytes=1 << 30):
        return L.q4k_gemm(args["w"], n, k, act, args["x"], null, null, m, ldx, args["y"], out, ldy,
                          args["ws"], ws_bytes, null)

    assert gemm(n=200) == 2
    assert gemm(k=300) == 2
    assert gemm(act=3) == 1
    assert gemm(out=4) == 1
    assert gemm(ldy=100) == 2
    assert gemm(ldy=258) == 3            # fp32 rows must stay 16-byte aligned
    assert gemm(ldx=500) == 2
    assert gemm(m=32, ws_bytes=16) == 4   # general path (m > 16); the small-M fp32 path takes no workspace
    assert gemm(m=32, act=1, ws_bytes=16) == 1
    assert gemm(act=1) == 1              # q8 input without da / ssum
    assert gemm(m=0) == 0                # empty batch is a no-op
    # q4k_gemm_inkernel_quant: shapes, output, activation stride, workspace size, empty batch
    def inkernel(n=256, k=512, m=8, ldx=512, out=0, ldy=256, ws_bytes=1 << 30, x=args["x"]):
        return L.q4k_gemm_inkernel_quant(args["w"], n, k, x, m, ldx, args["y"], out, ldy, args["ws"], ws_bytes, null)

    assert inkernel(n=200) == 2
    assert inkernel(k=300) == 2
    assert inkernel(out=4) == 1
    assert inkernel(ldx=500) == 2
    assert inkernel(x=null) == 1
    assert inkernel(x=ctypes.c_void_p(4100)) == 3
    assert inkernel(ws_bytes=16) == 4
    assert inkernel(m=0) == 0
    # debug hook size limit
    assert L.q4k_gemm_debug_chunk_acc(args["w"], 128 * 64, 4096, args["ws"], 1 << 30, 4096, args["y"], 8192,
                                      ctypes.c_void_p(4096), null) == 2
