"""Python binding of the C ABI in include/q4k.h (ctypes; argument marshalling only).

Every function here forwards to the entry point of the same name in
``libq4k.so``; all arithmetic runs in the library's CUDA kernels.  PyTorch
only supplies device memory (outputs and workspaces are allocated with
``torch.empty`` when the caller does not pass them) and the current CUDA
stream.  There is no CPU fallback: if the library is missing, importing this
module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

Q4K_OK = 0
Q4K_ERR_TIMEOUT = 7
ACT_F32, ACT_Q8 = 0, 1
OUT_F32, OUT_BF16 = 0, 1
_OUT = {"f32": OUT_F32, "float32": OUT_F32, torch.float32: OUT_F32,
        "bf16": OUT_BF16, "bfloat16": OUT_BF16, torch.bfloat16: OUT_BF16}

_c_i64, _c_int, _c_size, _c_ptr, _c_uint = ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_uint

# name -> (restype, argtypes); must match include/q4k.h
SIGNATURES = {
    "q4k_status_string": (ctypes.c_char_p, [_c_int]),
    "q4k_abi_version": (_c_int, []),
    "q8_quantize_rows": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_i64, _c_ptr, _c_ptr, _c_ptr, _c_ptr]),
    "q4k_packed_bytes": (_c_size, [_c_i64, _c_i64]),
    "q4k_pack_weights": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_ptr, _c_size, _c_ptr]),
    "q4k_gemm_workspace_bytes": (_c_size, [_c_i64, _c_i64, _c_i64, _c_int]),
    "q4k_gemm": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64,
                          _c_ptr, _c_int, _c_i64, _c_ptr, _c_size, _c_ptr]),
    "q4k_act_workspace_bytes": (_c_size, [_c_i64, _c_i64]),
    "q4k_act_quantize": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_i64, _c_ptr, _c_size, _c_ptr]),
    "q4k_act_from_q8": (_c_int, [_c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_i64, _c_ptr, _c_size, _c_ptr]),
    "q4k_gemm_quantized": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_ptr, _c_size, _c_i64, _c_ptr, _c_int, _c_i64,
                                    _c_ptr]),
    "q4k_gemm_inkernel_quant": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_ptr, _c_i64, _c_i64, _c_ptr, _c_int, _c_i64,
                                         _c_ptr, _c_size, _c_ptr]),
    "q4k_device_error_word": (_c_uint, [_c_int]),
    "q4k_device_status": (_c_int, [_c_int]),
    "q4k_selftest_wait_timeout": (_c_int, [_c_i64, _c_ptr]),
    "q4k_peak_mma_s8": (_c_int, [_c_i64, _c_i64, _c_ptr, _c_ptr]),
    "q4k_gemm_debug_chunk_acc": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_ptr, _c_size, _c_i64, _c_ptr, _c_i64,
                                          _c_ptr, _c_ptr]),
    "q4k_swiglu_packed_bytes": (_c_size, [_c_i64, _c_i64]),
    "q4k_pack_swiglu_weights": (_c_int, [_c_ptr, _c_ptr, _c_i64, _c_i64, _c_ptr, _c_size, _c_ptr]),
    "q4k_gemm_swiglu": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64,
                                 _c_ptr, _c_size, _c_ptr, _c_size, _c_ptr]),
    "q4k_gemm_swiglu_quantized": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_ptr, _c_size, _c_i64, _c_ptr, _c_size,
                                           _c_ptr]),
    "q6k_packed_bytes": (_c_size, [_c_i64, _c_i64]),
    "q6k_pack_weights": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_ptr, _c_size, _c_ptr]),
    "q6k_gemm": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64,
                          _c_ptr, _c_int, _c_i64, _c_ptr, _c_size, _c_ptr]),
    "q6k_gemm_debug_chunk_acc": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_ptr, _c_size, _c_i64, _c_ptr, _c_i64,
                                          _c_ptr, _c_ptr]),
    "q4k_static_workspace_bytes": (_c_size, []),
    "q4k_gemm_static_workspace": (_c_int, [_c_ptr, _c_i64, _c_i64, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64,
                                           _c_ptr, _c_int, _c_i64, _c_ptr]),
}


def load_library(path: str | None = None) -> ctypes.CDLL:
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"libq4k.so not found at {path}: build it first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = load_library()
LIB_PATH = _build.LIB_PATH


class Q4KError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {LIB.q4k_status_string(status).decode()} (status {status})")


def _check(fn: str, status: int):
    if status != Q4K_OK:
        raise Q4KError(fn, status)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _row_major(t: torch.Tensor, name: str):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D row-major tensor")
    return t.shape[0], t.shape[1], t.stride(0)


# ------------------------------------------------------------------ API --

def q8_quantize_rows(x: torch.Tensor, q8=None, da=None, ssum=None, stream=None):
    """fp32 [m][k] -> (q8 int8 [m][k], d_a float16 [m][k/32], ssum int16 [m][k/32])."""
    m, k, ldx = _row_major(x, "x")
    q8 = torch.empty((m, k), dtype=torch.int8, device=x.device) if q8 is None else q8
    da = torch.empty((m, k // 32), dtype=torch.float16, device=x.device) if da is None else da
    ssum = torch.empty((m, k // 32), dtype=torch.int16, device=x.device) if ssum is None else ssum
    _check("q8_quantize_rows", LIB.q8_quantize_rows(
        _dev(x, "x", torch.float32), m, k, ldx, _dev(q8, "q8", torch.int8), _dev(da, "da", torch.float16),
        _dev(ssum, "ssum", torch.int16), _stream(stream)))
    return q8, da, ssum


def q4k_packed_bytes(n: int, k: int) -> int:
    return int(LIB.q4k_packed_bytes(n, k))


def q4k_pack_weights(blocks: torch.Tensor, n: int, k: int, packed=None, stream=None) -> torch.Tensor:
    """Canonical Q4_K blocks (uint8 [n][k/256][144] on the GPU) -> packed uint8 buffer."""
    size = q4k_packed_bytes(n, k)
    if size == 0:
        raise ValueError("unsupported weight shape (n % 128, k % 256)")
    if blocks.numel() != n * (k // 256) * 144 or not blocks.is_contiguous():
        raise ValueError("blocks must be contiguous [n][k/256][144] uint8")
    packed = torch.empty(size, dtype=torch.uint8, device=blocks.device) if packed is None else packed
    _check("q4k_pack_weights", LIB.q4k_pack_weights(
        _dev(blocks, "blocks", torch.uint8), n, k, _dev(packed, "packed", torch.uint8), packed.numel(),
        _stream(stream)))
    return packed


def q4k_act_workspace_bytes(m: int, k: int) -> int:
    return int(LIB.q4k_act_workspace_bytes(m, k))


def q4k_gemm_workspace_bytes(m: int, n: int, k: int, act: int = ACT_F32) -> int:
    return int(LIB.q4k_gemm_workspace_bytes(m, n, k, act))


def _workspace(nbytes: int, device, ws):
    if ws is None:
        return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
    if ws.numel() * ws.element_size() < nbytes:
        raise ValueError("workspace too small")
    return ws


def _out(m, n, out_dtype, y, device):
    code = _OUT[out_dtype]
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32 if code == OUT_F32 else torch.bfloat16, device=device)
    _, _, ldy = _row_major(y, "y")
    return code, y, ldy


def q4k_act_quantize(x: torch.Tensor, workspace=None, stream=None) -> torch.Tensor:
    m, k, ldx = _row_major(x, "x")
    nb = q4k_act_workspace_bytes(m, k)
    workspace = _workspace(nb, x.device, workspace)
    _check("q4k_act_quantize", LIB.q4k_act_quantize(
        _dev(x, "x", torch.float32), m, k, ldx, _dev(workspace, "workspace"), workspace.numel(), _stream(stream)))
    return workspace


def q4k_act_from_q8(q8: torch.Tensor, da: torch.Tensor, ssum: torch.Tensor, workspace=None, stream=None):
    m, k, ldq = _row_major(q8, "q8")
    nb = q4k_act_workspace_bytes(m, k)
    workspace = _workspace(nb, q8.device, workspace)
    _check("q4k_act_from_q8", LIB.q4k_act_from_q8(
        _dev(q8, "q8", torch.int8), _dev(da, "da", torch.float16), _dev(ssum, "ssum", torch.int16), m, k, ldq,
        _dev(workspace, "workspace"), workspace.numel(), _stream(stream)))
    return workspace


def q4k_gemm_quantized(packed: torch.Tensor, n: int, k: int, workspace: torch.Tensor, m: int,
                       out_dtype="f32", y=None, stream=None) -> torch.Tensor:
    code, y, ldy = _out(m, n, out_dtype, y, packed.device)
    _check("q4k_gemm_quantized", LIB.q4k_gemm_quantized(
        _dev(packed, "packed"), n, k, _dev(workspace, "workspace"), workspace.numel(), m, _dev(y, "y"), code, ldy,
        _stream(stream)))
    return y


def q4k_gemm(packed: torch.Tensor, n: int, k: int, x: torch.Tensor, out_dtype="f32", da=None, ssum=None,
             y=None, workspace=None, stream=None) -> torch.Tensor:
    """Y[m][n] = x @ W^T.  x: fp32 [m][k] (fused quantization) or int8 q8 [m][k] with da/ssum."""
    m, kx, ldx = _row_major(x, "x")
    if kx != k:
        raise ValueError("x has the wrong number of columns")
    act = ACT_Q8 if x.dtype == torch.int8 else ACT_F32
    if act == ACT_Q8 and (da is None or ssum is None):
        raise ValueError("q8 input needs da and ssum")
    code, y, ldy = _out(m, n, out_dtype, y, x.device)
    nb = q4k_gemm_workspace_bytes(m, n, k, act)
    workspace = _workspace(nb, x.device, workspace)
    _check("q4k_gemm", LIB.q4k_gemm(
        _dev(packed, "packed"), n, k, act, _dev(x, "x"),
        _dev(da, "da", torch.float16) if act == ACT_Q8 else None,
        _dev(ssum, "ssum", torch.int16) if act == ACT_Q8 else None,
        m, ldx, _dev(y, "y"), code, ldy, _dev(workspace, "workspace"), workspace.numel(), _stream(stream)))
    return y


def q4k_gemm_inkernel_quant(packed: torch.Tensor, n: int, k: int, x: torch.Tensor, out_dtype="f32", y=None,
                            workspace=None, stream=None) -> torch.Tensor:
    """q4k_gemm for fp32 x in one launch: the GEMM kernel quantizes x itself."""
    m, kx, ldx = _row_major(x, "x")
    if kx != k:
        raise ValueError("x has the wrong number of columns")
    code, y, ldy = _out(m, n, out_dtype, y, x.device)
    workspace = _workspace(q4k_act_workspace_bytes(m, k), x.device, workspace)
    _check("q4k_gemm_inkernel_quant", LIB.q4k_gemm_inkernel_quant(
        _dev(packed, "packed"), n, k, _dev(x, "x", torch.float32), m, ldx, _dev(y, "y"), code, ldy,
        _dev(workspace, "workspace"), workspace.numel(), _stream(stream)))
    return y


def q4k_swiglu_packed_bytes(n: int, k: int) -> int:
    return int(LIB.q4k_swiglu_packed_bytes(n, k))


def q4k_pack_swiglu_weights(gate_blocks: torch.Tensor, up_blocks: torch.Tensor, n: int, k: int, packed=None,
                            stream=None) -> torch.Tensor:
    """gate and up Q4_K blocks (uint8 [n][k/256*144] each, on the device) -> packed pair."""
    nb = q4k_swiglu_packed_bytes(n, k)
    if nb == 0:
        raise ValueError(f"unsupported gate/up shape n={n} k={k}")
    packed = _workspace(nb, gate_blocks.device, packed)
    _check("q4k_pack_swiglu_weights", LIB.q4k_pack_swiglu_weights(
        _dev(gate_blocks, "gate_blocks", torch.uint8), _dev(up_blocks, "up_blocks", torch.uint8), n, k,
        _dev(packed, "packed"), packed.numel(), _stream(stream)))
    return packed


def q4k_gemm_swiglu(packed: torch.Tensor, n: int, k: int, x: torch.Tensor, da=None, ssum=None, h_ws=None,
                    workspace=None, stream=None) -> torch.Tensor:
    """SiLU(x W_gate^T) * (x W_up^T), quantized for the down projection: returns the
    operand workspace (uint8) to pass to q4k_gemm_quantized(down, n_down, n, h_ws, m)."""
    m, kx, ldx = _row_major(x, "x")
    if kx != k:
        raise ValueError("x has the wrong number of columns")
    act = ACT_Q8 if x.dtype == torch.int8 else ACT_F32
    if act == ACT_Q8 and (da is None or ssum is None):
        raise ValueError("q8 input needs da and ssum")
    h_ws = _workspace(q4k_act_workspace_bytes(m, n), x.device, h_ws)
    workspace = _workspace(q4k_gemm_workspace_bytes(m, 2 * n, k, act), x.device, workspace)
    _check("q4k_gemm_swiglu", LIB.q4k_gemm_swiglu(
        _dev(packed, "packed"), n, k, act, _dev(x, "x"),
        _dev(da, "da", torch.float16) if act == ACT_Q8 else None,
        _dev(ssum, "ssum", torch.int16) if act == ACT_Q8 else None,
        m, ldx, _dev(h_ws, "h_ws"), h_ws.numel(), _dev(workspace, "workspace"), workspace.numel(), _stream(stream)))
    return h_ws


def q4k_gemm_swiglu_quantized(packed: torch.Tensor, n: int, k: int, workspace: torch.Tensor, m: int, h_ws=None,
                              stream=None) -> torch.Tensor:
    """q4k_gemm_swiglu for x already in operand form (q4k_act_quantize / q4k_act_from_q8)."""
    h_ws = _workspace(q4k_act_workspace_bytes(m, n), workspace.device, h_ws)
    _check("q4k_gemm_swiglu_quantized", LIB.q4k_gemm_swiglu_quantized(
        _dev(packed, "packed"), n, k, _dev(workspace, "workspace"), workspace.numel(), m, _dev(h_ws, "h_ws"),
        h_ws.numel(), _stream(stream)))
    return h_ws


def q6k_packed_bytes(n: int, k: int) -> int:
    return int(LIB.q6k_packed_bytes(n, k))


def q6k_pack_weights(blocks: torch.Tensor, n: int, k: int, packed=None, stream=None) -> torch.Tensor:
    """Q6_K blocks (uint8 [n][k/256][210] on the GPU) -> packed uint8 buffer."""
    size = q6k_packed_bytes(n, k)
    if size == 0:
        raise ValueError("unsupported weight shape (n % 128, k % 256)")
    if blocks.numel() != n * (k // 256) * 210 or not blocks.is_contiguous():
        raise ValueError("blocks must be contiguous [n][k/256][210] uint8")
    packed = torch.empty(size, dtype=torch.uint8, device=blocks.device) if packed is None else packed
    _check("q6k_pack_weights", LIB.q6k_pack_weights(
        _dev(blocks, "blocks", torch.uint8), n, k, _dev(packed, "packed", torch.uint8), packed.numel(),
        _stream(stream)))
    return packed


def q6k_gemm(packed: torch.Tensor, n: int, k: int, x: torch.Tensor, out_dtype="f32", da=None, ssum=None,
             y=None, workspace=None, stream=None) -> torch.Tensor:
    """Y[m][n] = x @ W^T for Q6_K weights (q6k_pack_weights), any m >= 1.

    Up to 16 tokens whose activations fit the small-M kernel's shared memory
    take the CUDA-core product; larger batches take the tensor-core GEMM."""
    m, kx, ldx = _row_major(x, "x")
    if kx != k:
        raise ValueError("x has the wrong number of columns")
    act = ACT_Q8 if x.dtype == torch.int8 else ACT_F32
    if act == ACT_Q8 and (da is None or ssum is None):
        raise ValueError("q8 input needs da and ssum")
    code, y, ldy = _out(m, n, out_dtype, y, x.device)
    workspace = _workspace(q4k_gemm_workspace_bytes(m, n, k, act), x.device, workspace)
    _check("q6k_gemm", LIB.q6k_gemm(
        _dev(packed, "packed"), n, k, act, _dev(x, "x"),
        _dev(da, "da", torch.float16) if act == ACT_Q8 else None,
        _dev(ssum, "ssum", torch.int16) if act == ACT_Q8 else None,
        m, ldx, _dev(y, "y"), code, ldy, _dev(workspace, "workspace"), workspace.numel(), _stream(stream)))
    return y


def q4k_static_workspace_bytes() -> int:
    return int(LIB.q4k_static_workspace_bytes())


def q4k_gemm_static_workspace(packed: torch.Tensor, n: int, k: int, x: torch.Tensor, y: torch.Tensor,
                              da=None, ssum=None, stream=None) -> torch.Tensor:
    """q4k_gemm into the caller's y (fp32 or bf16 [m][n..]) with the library's own fixed
    workspace: nothing is allocated, here or in the library."""
    m, kx, ldx = _row_major(x, "x")
    if kx != k:
        raise ValueError("x has the wrong number of columns")
    act = ACT_Q8 if x.dtype == torch.int8 else ACT_F32
    if act == ACT_Q8 and (da is None or ssum is None):
        raise ValueError("q8 input needs da and ssum")
    code, y, ldy = _out(m, n, y.dtype, y, x.device)
    _check("q4k_gemm_static_workspace", LIB.q4k_gemm_static_workspace(
        _dev(packed, "packed"), n, k, act, _dev(x, "x"),
        _dev(da, "da", torch.float16) if act == ACT_Q8 else None,
        _dev(ssum, "ssum", torch.int16) if act == ACT_Q8 else None,
        m, ldx, _dev(y, "y"), code, ldy, _stream(stream)))
    return y


def q4k_gemm_debug_chunk_acc(packed, n, k, workspace, m, stream=None):
    """Test hook: (y fp32 [m][n], J fp32 [m][n][k/32]) with J the exact per-chunk dot products."""
    y = torch.empty((m, n), dtype=torch.float32, device=packed.device)
    acc = torch.zeros((m, n, k // 32), dtype=torch.float32, device=packed.device)
    _check("q4k_gemm_debug_chunk_acc", LIB.q4k_gemm_debug_chunk_acc(
        _dev(packed, "packed"), n, k, _dev(workspace, "workspace"), workspace.numel(), m, _dev(y, "y"), n,
        _dev(acc, "acc"), _stream(stream)))
    return y, acc


def q6k_gemm_debug_chunk_acc(packed, n, k, workspace, m, stream=None):
    """Test hook for Q6_K (workspace: the operand form a q6k_gemm call with m > 16 left in it):
    (y fp32 [m][n], J fp32 [m][n][k/32]) with J the exact per-chunk integers."""
    y = torch.empty((m, n), dtype=torch.float32, device=packed.device)
    acc = torch.zeros((m, n, k // 32), dtype=torch.float32, device=packed.device)
    _check("q6k_gemm_debug_chunk_acc", LIB.q6k_gemm_debug_chunk_acc(
        _dev(packed, "packed"), n, k, _dev(workspace, "workspace"), workspace.numel(), m, _dev(y, "y"), n,
        _dev(acc, "acc"), _stream(stream)))
    return y, acc


def q4k_peak_mma_s8(blocks: int, iters: int, sink: torch.Tensor, stream=None) -> None:
    """Launch the INT8 tensor-peak kernel (diagnostics): blocks x 8 warps x iters x 8
    mma.sync m16n8k32 s8, 8192 integer ops each; the caller times it."""
    _check("q4k_peak_mma_s8", LIB.q4k_peak_mma_s8(blocks, iters, _dev(sink, "sink", torch.int32), _stream(stream)))


def q4k_device_error_word(reset: bool = False) -> int:
    return int(LIB.q4k_device_error_word(1 if reset else 0))


def q4k_device_status(reset: bool = False) -> int:
    return int(LIB.q4k_device_status(1 if reset else 0))


def q4k_selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    return int(LIB.q4k_selftest_wait_timeout(int(timeout_ns), _stream(stream)))


def q4k_status_string(status: int) -> str:
    return LIB.q4k_status_string(status).decode()


def q4k_abi_version() -> int:
    return int(LIB.q4k_abi_version())
