"""Sub-bit (binary / ternary) weight products on NVIDIA B300 (sm_103a).

Thin ctypes binding of libbonsai (include/bonsai.h): the functions below have
the C names and only marshal arguments; every step runs in the CUDA kernels
of libbonsai.so. PyTorch supplies device memory and streams. If the library
is missing the calls raise: there is no CPU path.

Build the library with ``python -m sub_bit_weight_binary_b300.build``.

Typical use (all tensors on the GPU, FP16 activations)::

    import torch, sub_bit_weight_binary_b300 as sb
    rb = sb.bonsai_packed_row_bytes(sb.BONSAI_FMT_TERNARY, k)
    packed = torch.empty((n, rb), dtype=torch.uint8, device="cuda")
    sb.bonsai_pack_ternary(codes_int8_n_by_k, packed)          # codes in {-1, 0, +1}
    w = sb.Weights(sb.BONSAI_FMT_TERNARY, n, k, packed, scales_fp16_n_by_k128)
    sb.bonsai_gemv(w, x_k, y_n)                                # one token
    sb.bonsai_gemm(w, x_m_by_k, y_m_by_n)                      # m tokens
    sb.check()                                                 # sync, raise on a device status
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libbonsai.so")

BONSAI_FMT_BINARY = 1
BONSAI_FMT_TERNARY = 2
BONSAI_WEIGHTS_PREFETCH = 1

STATUS = {
    0: "BONSAI_OK", 1: "BONSAI_ERR_INVALID_ARG", 2: "BONSAI_ERR_SHAPE",
    3: "BONSAI_ERR_ALIGN", 4: "BONSAI_ERR_FORMAT", 5: "BONSAI_ERR_CUDA",
    6: "BONSAI_ERR_UNSUPPORTED", 7: "BONSAI_ERR_TIMEOUT", 8: "BONSAI_ERR_BAD_CODE",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}


class BonsaiError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s returned %s" % (what, STATUS.get(status, status)))
        self.status = status


class bonsai_weights_t(C.Structure):
    _fields_ = [("format", C.c_int32), ("n", C.c_int64), ("k", C.c_int64),
                ("row_bytes", C.c_int64), ("packed", C.c_void_p), ("scales", C.c_void_p),
                ("flags", C.c_int32)]


class bonsai_decode_step_t(C.Structure):
    _fields_ = [("w", bonsai_weights_t), ("x", C.c_void_p), ("y", C.c_void_p),
                ("swiglu", C.c_int32), ("after", C.c_int32)]


_lib = None


def lib():
    """Load libbonsai.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libbonsai.so is not built: run "
                              "python -m sub_bit_weight_binary_b300.build")
        L = C.CDLL(LIB_PATH)
        P, I64, I32, S = C.c_void_p, C.c_int64, C.c_int32, C.c_int
        W = C.POINTER(bonsai_weights_t)
        L.bonsai_packed_row_bytes.argtypes = [I32, I64]
        L.bonsai_packed_row_bytes.restype = I64
        for f in (L.bonsai_pack_binary, L.bonsai_pack_ternary):
            f.argtypes = [P, I64, I64, P, I64, P]
            f.restype = S
        L.bonsai_gemv.argtypes = [W, P, P, P]
        L.bonsai_gemv.restype = S
        L.bonsai_gemv_host.argtypes = [W, P, P, P, P, P]
        L.bonsai_gemv_host.restype = S
        L.bonsai_gemv_splitk_static.argtypes = [W, P, P, P]
        L.bonsai_gemv_workspace_bytes.argtypes = [W]
        L.bonsai_gemv_workspace_bytes.restype = I64
        L.bonsai_gemv_ws.argtypes = [W, P, P, P, I64, P]
        L.bonsai_gemv_ws.restype = S
        L.bonsai_gemv_host_ws.argtypes = [W, P, P, P, P, P, I64, P]
        L.bonsai_gemv_host_ws.restype = S
        L.bonsai_gemv_splitk_static.restype = S
        L.bonsai_gemm.argtypes = [W, P, I64, P, P]
        L.bonsai_gemm.restype = S
        L.bonsai_gemm_swiglu.argtypes = [W, P, I64, P, P]
        L.bonsai_gemm_swiglu.restype = S
        L.bonsai_gemm_workspace_bytes.argtypes = [W, I64]
        L.bonsai_gemm_workspace_bytes.restype = I64
        L.bonsai_gemm_ws.argtypes = [W, P, I64, P, P, I64, P]
        L.bonsai_gemm_ws.restype = S
        L.bonsai_gemm_swiglu_ws.argtypes = [W, P, I64, P, P, I64, P]
        L.bonsai_gemm_swiglu_ws.restype = S
        L.bonsai_xnor_gemm.argtypes = [P, P, I64, W, P, P, P]
        L.bonsai_xnor_gemm.restype = S
        L.bonsai_xnor_gemm_popc.argtypes = [P, P, I64, W, P, P, P]
        L.bonsai_xnor_gemm_popc.restype = S
        L.bonsai_binarize_activations.argtypes = [P, I64, I64, P, P, P]
        L.bonsai_binarize_activations.restype = S
        L.bonsai_hadamard.argtypes = [P, I64, I64, C.c_int32, P, P, P]
        L.bonsai_hadamard.restype = S
        L.bonsai_selftest_wait_timeout.argtypes = [C.c_uint64, P]
        L.bonsai_selftest_wait_timeout.restype = S
        D = C.POINTER(bonsai_decode_step_t)
        L.bonsai_decode_plan_bytes.argtypes = [I64]
        L.bonsai_decode_plan_bytes.restype = I64
        L.bonsai_decode_plan_init.argtypes = [D, I64, P, I64, P]
        L.bonsai_decode_plan_init.restype = S
        L.bonsai_decode_run.argtypes = [D, I64, P, P]
        L.bonsai_decode_run.restype = S
        L.bonsai_selftest_plan_wait.argtypes = [C.c_uint64, P]
        L.bonsai_selftest_plan_wait.restype = S
        L.bonsai_check_async.argtypes = [P]
        L.bonsai_check_async.restype = S
        L.bonsai_status_string.argtypes = [S]
        L.bonsai_status_string.restype = C.c_char_p
        _lib = L
    return _lib


# ---------------------------------------------------------------------------
# marshalling helpers

def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t, dtypes, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtypes:
        raise ValueError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _ok(st: int, what: str):
    if st != 0:
        raise BonsaiError(st, what)


@dataclass
class Weights:
    """A packed weight matrix W[n][k] and its FP16 group scales (device tensors).

    packed: uint8 [n][row_bytes]; scales: float16 [n][k/128]."""
    format: int
    n: int
    k: int
    packed: "object"
    scales: "object"
    flags: int = 0

    @property
    def row_bytes(self) -> int:
        return int(self.packed.shape[-1]) if self.packed.dim() == 2 else \
            int(self.packed.numel() // self.n)

    def c_struct(self) -> bonsai_weights_t:
        """The C struct, built and checked once; assigning any field rebuilds
        it (the tensors' storage is assumed not to move while held here)."""
        cs = self.__dict__.get("_cs")
        if cs is None:
            import torch
            cs = bonsai_weights_t(
                self.format, self.n, self.k, self.row_bytes,
                _ptr(self.packed, (torch.uint8, torch.int32, torch.int8), "packed"),
                _ptr(self.scales, (torch.float16, torch.int16), "scales"), self.flags)
            self.__dict__["_cs"] = cs
        return cs

    def __setattr__(self, name, value):
        self.__dict__.pop("_cs", None)
        object.__setattr__(self, name, value)


# ---------------------------------------------------------------------------
# the C ABI, same names

def bonsai_packed_row_bytes(fmt: int, k: int) -> int:
    return int(lib().bonsai_packed_row_bytes(fmt, k))


def bonsai_pack_binary(codes, out, stream=None):
    import torch
    rows, k = codes.shape
    _ok(lib().bonsai_pack_binary(_ptr(codes, (torch.int8,), "codes"), rows, k,
                                 _ptr(out, (torch.uint8,), "out"), out.shape[-1], _stream(stream)),
        "bonsai_pack_binary")


def bonsai_pack_ternary(codes, out, stream=None):
    import torch
    rows, k = codes.shape
    _ok(lib().bonsai_pack_ternary(_ptr(codes, (torch.int8,), "codes"), rows, k,
                                  _ptr(out, (torch.uint8,), "out"), out.shape[-1], _stream(stream)),
        "bonsai_pack_ternary")


def bonsai_gemv(w: Weights, x, y, stream=None):
    import torch
    ws = w.c_struct()
    _ok(lib().bonsai_gemv(C.byref(ws), _ptr(x, (torch.float16,), "x"),
                          _ptr(y, (torch.float16,), "y"), _stream(stream)), "bonsai_gemv")


def _host_ptr(t, name):
    import torch
    if t.is_cuda:
        raise ValueError("%s must be a host (preferably pinned) tensor" % name)
    if t.dtype != torch.float16 or not t.is_contiguous():
        raise ValueError("%s must be a contiguous float16 tensor" % name)
    return t.data_ptr()


def bonsai_gemv_workspace_bytes(w: Weights) -> int:
    """Bytes of the workspace that bonsai_gemv_ws needs to run the one-token
    product on the table kernel (0: the shape does not take it)."""
    return int(lib().bonsai_gemv_workspace_bytes(C.byref(w.c_struct())))


def gemv_workspace(w: Weights, device="cuda"):
    """A zero-filled workspace for bonsai_gemv_ws / bonsai_gemv_host_ws (and
    bonsai_gemm_ws with one token), or None if the shape takes none."""
    import torch
    nbytes = bonsai_gemv_workspace_bytes(w)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device) if nbytes else None


def bonsai_gemv_ws(w: Weights, x, y, workspace, stream=None):
    """bonsai_gemv with a workspace (see gemv_workspace): the table kernel for
    ternary weights of a shape that takes it, bonsai_gemv's kernels otherwise."""
    import torch
    wp, wb = _ws_args(workspace)
    _ok(lib().bonsai_gemv_ws(C.byref(w.c_struct()), _ptr(x, (torch.float16,), "x"),
                             _ptr(y, (torch.float16,), "y"), wp, wb, _stream(stream)),
        "bonsai_gemv_ws")


def bonsai_gemv_host(w: Weights, x_host, x_dev, y_dev, y_host, stream=None, workspace=None):
    """Host x in, host y out: enqueue x_host -> x_dev, the decode product into
    y_dev and y_dev -> y_host on the stream (synchronise before reading y_host).
    With a workspace (see gemv_workspace) the product runs as bonsai_gemv_ws."""
    import torch
    if x_host.numel() != w.k or y_host.numel() != w.n:
        raise ValueError("x_host must hold k and y_host n values")
    args = (C.byref(w.c_struct()), _host_ptr(x_host, "x_host"),
            _ptr(x_dev, (torch.float16,), "x_dev"), _ptr(y_dev, (torch.float16,), "y_dev"),
            _host_ptr(y_host, "y_host"))
    if workspace is None:
        _ok(lib().bonsai_gemv_host(*args, _stream(stream)), "bonsai_gemv_host")
    else:
        wp, wb = _ws_args(workspace)
        _ok(lib().bonsai_gemv_host_ws(*args, wp, wb, _stream(stream)), "bonsai_gemv_host_ws")


class GemvHostPlan:
    """A decode step with host buffers, prepared once: the copies and the
    product of bonsai_gemv_host are captured in a CUDA graph, and each call
    replays it (one launch per token; the contents of x_host may change
    between calls, the buffers themselves may not). Synchronise before
    reading y_host. x_host and y_host must be pinned; the optional workspace
    is used as by bonsai_gemv_host."""

    def __init__(self, w: Weights, x_host, x_dev, y_dev, y_host, workspace=None):
        import torch
        if not (x_host.is_pinned() and y_host.is_pinned()):
            raise ValueError("x_host and y_host must be pinned host tensors")
        self._keep = (w, x_host, x_dev, y_dev, y_host, workspace)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):  # eager call first: one-time setup stays outside the capture
            bonsai_gemv_host(w, x_host, x_dev, y_dev, y_host, workspace=workspace)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            bonsai_gemv_host(w, x_host, x_dev, y_dev, y_host, workspace=workspace)

    def __call__(self):
        self.graph.replay()


def bonsai_gemv_splitk_static(w: Weights, x, y, stream=None):
    """bonsai_gemv with K split over thread blocks and a fixed device scratch
    array (no allocation); n <= 8192, calls on one device must not overlap."""
    import torch
    ws = w.c_struct()
    _ok(lib().bonsai_gemv_splitk_static(C.byref(ws), _ptr(x, (torch.float16,), "x"),
                                        _ptr(y, (torch.float16,), "y"), _stream(stream)),
        "bonsai_gemv_splitk_static")


def bonsai_gemm(w: Weights, x, y, stream=None):
    import torch
    ws = w.c_struct()
    m = x.shape[0] if x.dim() == 2 else 1
    _ok(lib().bonsai_gemm(C.byref(ws), _ptr(x, (torch.float16,), "x"), m,
                          _ptr(y, (torch.float16,), "y"), _stream(stream)), "bonsai_gemm")


def bonsai_gemm_swiglu(w: Weights, x, h, stream=None):
    """h [m][n/2] = silu(g) * u for the interleaved gate/up matrix w (16-row
    blocks: 8 gate rows, then the 8 up rows of the same features)."""
    import torch
    ws = w.c_struct()
    m = x.shape[0] if x.dim() == 2 else 1
    _ok(lib().bonsai_gemm_swiglu(C.byref(ws), _ptr(x, (torch.float16,), "x"), m,
                                 _ptr(h, (torch.float16,), "h"), _stream(stream)),
        "bonsai_gemm_swiglu")


def bonsai_gemm_workspace_bytes(w: Weights, m: int) -> int:
    """Bytes of the workspace that bonsai_gemm_ws needs for m tokens: the
    stream-K partial tiles for m > 8, the table kernel's partial sums for
    m = 1 (0: no workspace is used for this shape)."""
    ws = w.c_struct()
    return int(lib().bonsai_gemm_workspace_bytes(C.byref(ws), int(m)))


def gemm_workspace(w: Weights, m: int, device="cuda"):
    """A zero-filled workspace for bonsai_gemm_ws / bonsai_gemm_swiglu_ws
    (uint8 tensor, 256-byte aligned by the allocator), or None if the shape
    needs none."""
    import torch
    nbytes = bonsai_gemm_workspace_bytes(w, m)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device) if nbytes else None


def _ws_args(workspace):
    if workspace is None:
        return None, 0
    import torch
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")
    return C.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size()


def bonsai_gemm_ws(w: Weights, x, y, workspace, stream=None):
    """bonsai_gemm with a stream-K workspace (see gemm_workspace)."""
    import torch
    ws = w.c_struct()
    m = x.shape[0] if x.dim() == 2 else 1
    wp, wb = _ws_args(workspace)
    _ok(lib().bonsai_gemm_ws(C.byref(ws), _ptr(x, (torch.float16,), "x"), m,
                             _ptr(y, (torch.float16,), "y"), wp, wb, _stream(stream)),
        "bonsai_gemm_ws")


def bonsai_gemm_swiglu_ws(w: Weights, x, h, workspace, stream=None):
    """bonsai_gemm_swiglu with a stream-K workspace (see gemm_workspace)."""
    import torch
    ws = w.c_struct()
    m = x.shape[0] if x.dim() == 2 else 1
    wp, wb = _ws_args(workspace)
    _ok(lib().bonsai_gemm_swiglu_ws(C.byref(ws), _ptr(x, (torch.float16,), "x"), m,
                                    _ptr(h, (torch.float16,), "h"), wp, wb, _stream(stream)),
        "bonsai_gemm_swiglu_ws")


def interleave_gate_up(gate, up):
    """Stack gate and up rows [F][...] into the [2F][...] row order that
    bonsai_gemm_swiglu reads: 8 gate rows, then the 8 up rows of the same
    features, per 16-row block. Works on numpy arrays and torch tensors."""
    f = gate.shape[0]
    if f % 8 or up.shape != gate.shape:
        raise ValueError("gate and up must have the same shape with a multiple of 8 rows")
    rest = tuple(gate.shape[1:])
    g = gate.reshape((f // 8, 1, 8) + rest)
    u = up.reshape((f // 8, 1, 8) + rest)
    try:
        import torch
        if isinstance(gate, torch.Tensor):
            return torch.cat([g, u], dim=1).reshape((2 * f,) + rest)
    except ImportError:
        pass
    import numpy as np
    return np.concatenate([g, u], axis=1).reshape((2 * f,) + rest)


def bonsai_xnor_gemm(a_bits, a_scale, w: Weights, d_out=None, y_out=None, stream=None,
                     popc=False):
    """D = a . w^T (exact int32) and/or Y (FP16) for +-1 bits; tensor cores,
    or the literal XOR + popcount kernel with popc=True."""
    import torch
    ws = w.c_struct()
    fn = lib().bonsai_xnor_gemm_popc if popc else lib().bonsai_xnor_gemm
    _ok(fn(_ptr(a_bits, (torch.int32, torch.uint8), "a_bits"),
           _ptr(a_scale, (torch.float16,), "a_scale"), a_bits.shape[0],
           C.byref(ws), _ptr(d_out, (torch.int32,), "d_out"),
           _ptr(y_out, (torch.float16,), "y_out"), _stream(stream)),
        "bonsai_xnor_gemm_popc" if popc else "bonsai_xnor_gemm")


def bonsai_binarize_activations(x, a_bits, a_scale, stream=None):
    """Sign codes (bit 1 where x >= 0) and mean-|x| scales of FP16 rows x [m][k],
    written into a_bits (int32 [m][k/32]) and a_scale (float16 [m])."""
    import torch
    if x.dim() != 2:
        raise ValueError("x must be [m][k]")
    _ok(lib().bonsai_binarize_activations(_ptr(x, (torch.float16,), "x"), x.shape[0], x.shape[1],
                                          _ptr(a_bits, (torch.int32, torch.uint8), "a_bits"),
                                          _ptr(a_scale, (torch.float16,), "a_scale"),
                                          _stream(stream)),
        "bonsai_binarize_activations")


def bonsai_hadamard(x, out, block=128, signs=None, stream=None):
    """Block-diagonal signed Hadamard rotation of FP16 rows x [m][k] into out
    (may be x itself); signs: int32 [k/32] bits (1 = +1) or None (all +1)."""
    import torch
    if x.dim() != 2:
        raise ValueError("x must be [m][k]")
    _ok(lib().bonsai_hadamard(_ptr(x, (torch.float16,), "x"), x.shape[0], x.shape[1], block,
                              _ptr(signs, (torch.int32,), "signs"),
                              _ptr(out, (torch.float16,), "out"), _stream(stream)),
        "bonsai_hadamard")


def bonsai_selftest_wait_timeout(limit_ns: int, stream=None):
    """Launch the bounded-wait self-test (a wait that must run out)."""
    _ok(lib().bonsai_selftest_wait_timeout(int(limit_ns), _stream(stream)),
        "bonsai_selftest_wait_timeout")


def bonsai_decode_plan_bytes(count: int) -> int:
    return int(lib().bonsai_decode_plan_bytes(count))


def _steps_array(steps):
    """steps: list of (Weights, x, y, swiglu, after) -> ctypes array."""
    import torch
    arr = (bonsai_decode_step_t * len(steps))()
    for i, (w, x, y, swiglu, after) in enumerate(steps):
        arr[i].w = w.c_struct()
        arr[i].x = _ptr(x, (torch.float16,), "x")
        arr[i].y = _ptr(y, (torch.float16,), "y")
        arr[i].swiglu = int(bool(swiglu))
        arr[i].after = int(after)
    return arr


def bonsai_decode_plan_init(steps_arr, plan, stream=None):
    import torch
    _ok(lib().bonsai_decode_plan_init(steps_arr, len(steps_arr),
                                      _ptr(plan, (torch.uint8,), "plan"), plan.numel(),
                                      _stream(stream)), "bonsai_decode_plan_init")


def bonsai_decode_run(steps_arr, plan, stream=None):
    import torch
    _ok(lib().bonsai_decode_run(steps_arr, len(steps_arr), _ptr(plan, (torch.uint8,), "plan"),
                                _stream(stream)), "bonsai_decode_run")


class DecodePlan:
    """A decode plan: the one-token products of a token in one launch.

    steps: list of (Weights, x, y, swiglu, after) with device tensors; after
    is the index of an earlier step whose y this step's x is, or -1. The
    plan's device memory is a torch uint8 tensor owned here; the tensors of
    the steps must stay alive (and in place) while the plan is used."""

    def __init__(self, steps, stream=None):
        import torch
        self._keep = steps
        self.steps = _steps_array(steps)
        nbytes = bonsai_decode_plan_bytes(len(steps))
        if nbytes < 0:
            raise ValueError("bad number of steps")
        raw = torch.empty(nbytes + 128, dtype=torch.uint8, device="cuda")
        off = (-raw.data_ptr()) % 128
        self._raw = raw
        self.plan = raw[off:off + nbytes]
        bonsai_decode_plan_init(self.steps, self.plan, stream)

    def run(self, stream=None):
        bonsai_decode_run(self.steps, self.plan, stream)


def bonsai_selftest_plan_wait(limit_ns: int, stream=None):
    """Launch the plan dependency-wait self-test (a wait that must run out)."""
    _ok(lib().bonsai_selftest_plan_wait(int(limit_ns), _stream(stream)),
        "bonsai_selftest_plan_wait")


def bonsai_check_async(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(lib().bonsai_check_async(_stream(stream)))


def bonsai_status_string(status: int) -> str:
    return lib().bonsai_status_string(status).decode()


def check(stream=None):
    """bonsai_check_async that raises BonsaiError on a non-OK status."""
    _ok(bonsai_check_async(stream), "bonsai_check_async")
