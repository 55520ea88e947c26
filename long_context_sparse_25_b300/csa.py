"""ctypes binding of libcsa_b300.so (argument marshalling only).

Every function here turns torch tensors into the C ABI's plain pointers and
sizes and calls the library on the current CUDA stream; every step of the
computation runs in the library's kernels.  There is no fallback: if the
shared library is missing or fails to load, importing this module raises.
"""

from __future__ import annotations

import ctypes as C
import re
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libcsa_b300.so"
HEADER = _PKG.parent / "include" / "csa.h"

F32, BF16, E4M3, E2M1 = 0, 1, 2, 3
WS_TOPK, WS_ATTEND, WS_HCA, WS_FORWARD, WS_ATTEND_RAW = 0, 1, 2, 3, 4
STALL_INDEX, STALL_ATTEND = 1, 2
STATUS = {0: "CSA_OK", -1: "CSA_ERR_INVALID_ARG", -2: "CSA_ERR_UNSUPPORTED", -3: "CSA_ERR_ALIGNMENT",
          -4: "CSA_ERR_WORKSPACE", -5: "CSA_ERR_CUDA", -6: "CSA_ERR_TIMEOUT"}


class CsaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


def _load():
    if not LIB_PATH.exists():
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m long_context_sparse_25_b300.build`")
    return C.CDLL(str(LIB_PATH))


lib = _load()


class Rows(C.Structure):
    _fields_ = [("dtype", C.c_int), ("data", C.c_void_p), ("rope", C.c_void_p),
                ("scale", C.c_void_p), ("n_rows", C.c_int64), ("width", C.c_int),
                ("nope", C.c_int)]


class Params(C.Structure):
    _fields_ = [("B", C.c_int), ("m", C.c_int), ("H", C.c_int), ("D_qk", C.c_int),
                ("D_v", C.c_int), ("H_I", C.c_int), ("d_I", C.c_int), ("k", C.c_int),
                ("window", C.c_int), ("scale", C.c_float)]


class ForwardArgs(C.Structure):
    _fields_ = [("x", C.c_void_p), ("gate", C.c_void_p), ("bias", C.c_void_p),
                ("xi", C.c_void_p), ("gate_i", C.c_void_p), ("bias_i", C.c_void_p),
                ("raw_dtype", C.c_int), ("R", C.c_int64), ("raw_pos0", C.c_int64),
                ("q", C.c_void_p), ("q_dtype", C.c_int), ("q_idx", C.c_void_p),
                ("q_idx_dtype", C.c_int), ("q_idx_scale", C.c_void_p), ("w", C.c_void_p),
                ("q_pos0", C.c_int64), ("Q", C.c_int), ("kv", Rows), ("keys", Rows),
                ("n_cached", C.c_int64), ("out", C.c_void_p), ("out_dtype", C.c_int),
                ("raw_all", C.c_void_p), ("raw_all_rows", C.c_int64), ("score_dtype", C.c_int)]


_P, _I, _I64, _SZ = C.c_void_p, C.c_int, C.c_int64, C.c_size_t
_SIGS = {
    "csa_compress": [_P, _P, _I, _P, _I, _I64, _I64, _I, _I, _I64, _I64, C.POINTER(Rows), _P],
    "csa_index": [C.POINTER(Params), _P, _I, _P, _P, C.POINTER(Rows), _I64, _I, _I64, _P, _P],
    "csa_topk": [C.POINTER(Params), _P, _I64, _I, _I64, _P, _P, _SZ, _P],
    "csa_attend": [C.POINTER(Params), _P, _I, C.POINTER(Rows), C.POINTER(Rows), _I64, _P, _I64,
                   _I, _I64, _P, _I, _P, _SZ, _P],
    "hca_attend": [C.POINTER(Params), _P, _I, C.POINTER(Rows), C.POINTER(Rows), _I64, _I64, _I,
                   _I64, _P, _I, _P, _SZ, _P],
    "csa_attend_raw": [C.POINTER(Params), _P, _I, C.POINTER(Rows), _I64, _P, _I64, _I, _I64, _P,
                       _I, _P, _SZ, _P],
    "csa_forward": [C.POINTER(Params), C.POINTER(ForwardArgs), _P, _SZ, _P],
    "csa_topk_noalloc": [C.POINTER(Params), _P, _I64, _I, _I64, _P, _P],
    "csa_group_proj": [_P, _I64, _I, _I, _P, _I, _I, _P, _I, _P],
    "csa_index_ex": [C.POINTER(Params), _P, _I, _P, _P, C.POINTER(Rows), _I64, _I, _I64, _P, _I,
                     _P],
    "csa_topk_ex": [C.POINTER(Params), _P, _I, _I64, _I, _I64, _P, _P, _SZ, _P],
}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = C.c_int
lib.csa_workspace_size.argtypes = [C.POINTER(Params), _I, _I, _I64]
lib.csa_workspace_size.restype = C.c_size_t
lib.csa_device_status.argtypes = [_P]
lib.csa_device_status.restype = C.c_int
lib.csa_debug_stall_next.argtypes = [_I]
lib.csa_debug_stall_next.restype = C.c_int
lib.csa_last_error.argtypes = []
lib.csa_last_error.restype = C.c_char_p


def header_functions() -> list[str]:
    """Names of the functions declared in include/csa.h."""
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:int|size_t|const char\*)\s+(\w+)\s*\(", text, flags=re.M)


def _check(code: int):
    if code != 0:
        raise CsaError(code, lib.csa_last_error().decode())


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float8_e4m3fn:
        return E4M3
    if t.dtype == torch.float4_e2m1fn_x2:  # two FP4 codes per byte
        return E2M1
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def rows(data: torch.Tensor, rope: torch.Tensor | None = None, scale: torch.Tensor | None = None,
         width: int | None = None) -> Rows:
    """Describe [B, n_rows, *] rows.  For e4m3 data the rope plane (bf16) and
    the per-row fp32 scale are given separately; width = nope + rope width.
    FP4 keys (torch.float4_e2m1fn_x2, two codes per byte) hold 2 * shape[-1]
    channels, with their per-row scale."""
    dt = dtype_code(data)
    nope = data.shape[-1] * (2 if dt == E2M1 else 1)
    if width is None:
        width = nope + (rope.shape[-1] if rope is not None else 0)
    return Rows(dt, _ptr(data), _ptr(rope), _ptr(scale), data.shape[-2], width, nope)


def params(B, m, H=0, D_qk=0, D_v=0, H_I=0, d_I=0, k=0, window=0, scale=1.0) -> Params:
    return Params(B, m, H, D_qk, D_v, H_I, d_I, k, window, scale)


def workspace_size(p: Params, which: int, Q: int, N: int) -> int:
    return int(lib.csa_workspace_size(C.byref(p), which, Q, N))


def topk_launches(p: Params, Q: int, N: int) -> int:
    """Kernels one csa_topk call launches for these sizes: three (sample,
    filter, final) for a few long rows, one otherwise."""
    return 3 if (N > 16384 and p.k <= 4096 and p.B * Q < 256) else 1


def _workspace(nbytes: int, device) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def compress(x, gate, bias, m, s_begin, s_end, out: Rows, x_pos0=0, stream=None):
    B, T, Cc = x.shape
    _check(lib.csa_compress(_ptr(x), _ptr(gate), dtype_code(x), _ptr(bias), B, x_pos0, T, m, Cc,
                            s_begin, s_end, C.byref(out), _stream(stream)))


def index(p: Params, q_idx, w, keys: Rows, q_pos0, N, scores, q_scale=None, stream=None):
    """csa_index (fp32 scores) or csa_index_ex (bf16 scores), by scores' dtype."""
    Q = q_idx.shape[1]
    if scores.dtype == torch.bfloat16:
        _check(lib.csa_index_ex(C.byref(p), _ptr(q_idx), dtype_code(q_idx), _ptr(q_scale),
                                _ptr(w), C.byref(keys), q_pos0, Q, N, _ptr(scores), BF16,
                                _stream(stream)))
        return
    _check(lib.csa_index(C.byref(p), _ptr(q_idx), dtype_code(q_idx), _ptr(q_scale), _ptr(w),
                         C.byref(keys), q_pos0, Q, N, _ptr(scores), _stream(stream)))


def topk(p: Params, scores, q_pos0, idx, ws=None, stream=None):
    B, Q, N = scores.shape
    nbytes = workspace_size(p, WS_TOPK, Q, N)
    if ws is None:
        ws = _workspace(nbytes, scores.device)
    _check(lib.csa_topk_ex(C.byref(p), _ptr(scores), dtype_code(scores), q_pos0, Q, N, _ptr(idx),
                           _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


TOPK_NOALLOC_MAX_BYTES = 16 << 20  # CSA_TOPK_NOALLOC_MAX_BYTES of include/csa.h


def topk_noalloc(p: Params, scores, q_pos0, idx, stream=None):
    """csa_topk_noalloc: top-k with the library's static scratch (no workspace)."""
    B, Q, N = scores.shape
    _check(lib.csa_topk_noalloc(C.byref(p), _ptr(scores), q_pos0, Q, N, _ptr(idx),
                                _stream(stream)))


def attend(p: Params, q, kv: Rows, raw: Rows | None, raw_pos0, idx, q_pos0, N, out, ws=None,
           stream=None):
    Q = q.shape[1]
    if ws is None:
        ws = _workspace(workspace_size(p, WS_ATTEND, Q, N), q.device)
    _check(lib.csa_attend(C.byref(p), _ptr(q), dtype_code(q), C.byref(kv),
                          C.byref(raw) if raw is not None else None, raw_pos0, _ptr(idx), q_pos0, Q,
                          N, _ptr(out), dtype_code(out), _ptr(ws),
                          0 if ws is None else ws.numel(), _stream(stream)))


def attend_raw(p: Params, q, raw: Rows, raw_pos0, idx, q_pos0, N, out, ws=None, stream=None):
    """csa_attend_raw: attention over the m raw tokens of every selected block
    plus the window."""
    Q = q.shape[1]
    if ws is None:
        ws = _workspace(workspace_size(p, WS_ATTEND_RAW, Q, N), q.device)
    _check(lib.csa_attend_raw(C.byref(p), _ptr(q), dtype_code(q), C.byref(raw), raw_pos0,
                              _ptr(idx), q_pos0, Q, N, _ptr(out), dtype_code(out), _ptr(ws),
                              0 if ws is None else ws.numel(), _stream(stream)))


def hca(p: Params, q, kv: Rows, raw: Rows | None, raw_pos0, q_pos0, N, out, ws=None, stream=None):
    Q = q.shape[1]
    if ws is None:
        ws = _workspace(workspace_size(p, WS_HCA, Q, N), q.device)
    _check(lib.hca_attend(C.byref(p), _ptr(q), dtype_code(q), C.byref(kv),
                          C.byref(raw) if raw is not None else None, raw_pos0, q_pos0, Q, N,
                          _ptr(out), dtype_code(out), _ptr(ws), 0 if ws is None else ws.numel(),
                          _stream(stream)))


def forward_args(*, x, gate, bias, xi, gate_i, bias_i, raw_pos0, q, q_idx, w, q_pos0, kv: Rows,
                 keys: Rows, n_cached, out, q_idx_scale=None, raw_all=None,
                 score_dtype=F32) -> ForwardArgs:
    """Arguments of csa_forward.  raw_all (raw rows of every position from 0)
    selects the raw-token attention; score_dtype BF16 stores the indexer
    scores in bf16."""
    return ForwardArgs(_ptr(x), _ptr(gate), _ptr(bias), _ptr(xi), _ptr(gate_i), _ptr(bias_i),
                       dtype_code(x), x.shape[1], raw_pos0, _ptr(q), dtype_code(q), _ptr(q_idx),
                       dtype_code(q_idx), _ptr(q_idx_scale), _ptr(w), q_pos0, q.shape[1], kv, keys,
                       n_cached, _ptr(out), dtype_code(out), _ptr(raw_all),
                       0 if raw_all is None else raw_all.shape[1], score_dtype)


def group_proj(o, w, y, stream=None):
    """csa_group_proj: y [.., G*d_g] = the grouped projection of the attention
    output o [.., H, D_v] with w [G, d_g, (H/G)*D_v]."""
    H, D_v = o.shape[-2], o.shape[-1]
    T = o.numel() // (H * D_v) if o.numel() else 0
    G, d_g = w.shape[0], w.shape[1]
    _check(lib.csa_group_proj(_ptr(o), T, H, D_v, _ptr(w), G, d_g, _ptr(y), dtype_code(y),
                              _stream(stream)))


def debug_stall_next(kernel: int):
    """csa_debug_stall_next: arm the one-shot test aid that makes the next
    launch of the named tensor-core kernel give up on a wait (0 disarms)."""
    _check(lib.csa_debug_stall_next(kernel))


def device_status(stream=None):
    """Synchronise the stream; raise CsaError(CSA_ERR_TIMEOUT) if a bounded
    device-side wait gave up since the previous check."""
    _check(lib.csa_device_status(_stream(stream)))


def forward(p: Params, a: ForwardArgs, ws: torch.Tensor, stream=None):
    _check(lib.csa_forward(C.byref(p), C.byref(a), _ptr(ws), ws.numel(), _stream(stream)))
