"""Python binding of the fused-chain library (libfusechain.so).

Argument marshalling only: every step of every operation runs in the
library's generated CUDA kernels.  The functions carry the C ABI's names
(see include/fuse.h); tensor arguments may be torch tensors (their data
pointers are passed) or raw integer device addresses.  A nonzero status
raises FuseError with the library's message.

If the shared library has not been built this module raises ImportError: there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfusechain.so")

F32, F16, BF16 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", F16: "f16", BF16: "bf16"}

STATUS = {0: "FUSE_OK", -1: "FUSE_E_SPEC", -2: "FUSE_E_SHAPE", -3: "FUSE_E_DTYPE",
          -4: "FUSE_E_NULL", -5: "FUSE_E_ARCH", -6: "FUSE_E_COMPILE", -7: "FUSE_E_CUDA",
          -8: "FUSE_E_ARG"}

# every symbol include/fuse.h declares
EXPORTS = ["fuse_compile", "fuse_num_inputs", "fuse_input_dtypes", "fuse_launch", "fuse_release",
           "fuse_source", "fuse_compile_bucket", "fuse_launch_rows", "fuse_source_bucket",
           "fuse_bucket", "fuse_warmup", "rmsnorm_linear", "rmsnorm_linear_fold", "fuse_device_error", "rmsnorm_residual", "layernorm_residual", "rope_qkv_split", "rope_qkv_split_noalloc",
           "detect_decode", "channel_shuffle", "fuse_graph_begin", "fuse_graph_end",
           "fuse_graph_launch", "fuse_graph_nodes", "fuse_graph_release", "fuse_last_error",
           "fuse_stats", "fuse_device_sms", "fuse_selftest_bounded_wait"]


class FuseError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: run python elementwise_chain_jit_gb300/buildlib.py "
                      "(or __graft_entry__.build()) first")

_lib = ctypes.CDLL(LIB_PATH)
_P, _I, _I64, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
_lib.fuse_compile.argtypes = [ctypes.c_char_p, ctypes.POINTER(_I64), _I, _I, ctypes.POINTER(_P)]
_lib.fuse_num_inputs.argtypes = [_P, ctypes.POINTER(_I), ctypes.POINTER(_I)]
_lib.fuse_input_dtypes.argtypes = [_P, ctypes.POINTER(_I), _I]
_lib.fuse_launch.argtypes = [_P, ctypes.POINTER(_P), _I, _P, _P]
_lib.fuse_release.argtypes = [_P]
_lib.fuse_source.argtypes = [ctypes.c_char_p, ctypes.POINTER(_I64), _I, _I, ctypes.c_char_p,
                             ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]
_lib.fuse_compile_bucket.argtypes = [ctypes.c_char_p, ctypes.POINTER(_I64), _I, _I,
                                     ctypes.POINTER(_P)]
_lib.fuse_launch_rows.argtypes = [_P, ctypes.POINTER(_P), _I, _P, _I64, _P]
_lib.fuse_source_bucket.argtypes = [ctypes.c_char_p, ctypes.POINTER(_I64), _I, _I, ctypes.c_char_p,
                                    ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]
_lib.fuse_bucket.argtypes = [_I64, ctypes.POINTER(_I64)]
_lib.fuse_warmup.argtypes = [ctypes.c_char_p, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]
_lib.rmsnorm_residual.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _F, _I, _P]
_lib.rmsnorm_linear.argtypes = [_P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _F, _I, _P]
_lib.fuse_device_error.argtypes = [ctypes.POINTER(_I)]
_lib.rmsnorm_linear_fold.argtypes = [_P, _P, _P, _I64, _I64, _I, _P]
_lib.layernorm_residual.argtypes = [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I, _P]
_lib.rope_qkv_split.argtypes = [_P, _P, _P, _P, _I64, _I, _I, _I64, _F, _I, _P]
_lib.rope_qkv_split_noalloc.argtypes = [_P, _P, _P, _P, _I64, _I, _I, _I64, _F, _I, _P]
_lib.detect_decode.argtypes = [ctypes.POINTER(_P), ctypes.POINTER(_I), ctypes.POINTER(_F),
                               ctypes.POINTER(_F), _I, _I, _I, _I, _P, _P]
_lib.channel_shuffle.argtypes = [_P, _P, _I64, _I64, _I64, _I64, _I, _I, _P]
_lib.fuse_graph_begin.argtypes = [_P]
_lib.fuse_graph_end.argtypes = [_P, ctypes.POINTER(_P)]
_lib.fuse_graph_launch.argtypes = [_P, _P]
_lib.fuse_graph_nodes.argtypes = [_P, ctypes.POINTER(_I64)]
_lib.fuse_graph_release.argtypes = [_P]
_lib.fuse_last_error.restype = ctypes.c_char_p
_lib.fuse_stats.argtypes = [ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                            ctypes.POINTER(ctypes.c_double)]
_lib.fuse_device_sms.argtypes = [ctypes.POINTER(_I)]
_lib.fuse_selftest_bounded_wait.argtypes = [_I64, _P]


def _check(rc: int) -> None:
    if rc != 0:
        raise FuseError(rc, (_lib.fuse_last_error() or b"").decode(errors="replace"))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


_raw_stream = None  # torch's current-stream query, looked up once


def _stream(stream) -> int | None:
    """The CUstream to launch on: the given one, else torch's current stream
    (None, the legacy default stream, before torch has touched the GPU).  The
    raw query costs ~0.4 us (measured on GB300) where building torch's Stream
    object costs ~3 us, which matters next to a kernel of a few microseconds."""
    global _raw_stream
    if stream is None:
        torch = sys.modules.get("torch")
        if torch is None or not torch.cuda.is_initialized():
            return None
        if _raw_stream is None:
            raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
            # torch's raw device query; torch.cuda.current_device() would check
            # the lazy initialisation again, which is known to be done here
            dev = getattr(torch._C, "_cuda_getDevice", None) or torch.cuda.current_device
            _raw_stream = ((lambda: raw(dev())) if raw is not None
                           else (lambda: torch.cuda.current_stream().cuda_stream))
        return _raw_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


_torch_dtypes = None


def _dtype(dt) -> int:
    global _torch_dtypes
    if isinstance(dt, int):
        return dt
    if _torch_dtypes is None:
        import torch
        _torch_dtypes = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
    return _torch_dtypes[dt]


def _shape(shape):
    arr = (_I64 * len(shape))(*[int(s) for s in shape])
    return arr, len(shape)


# ---------------------------------------------------------------- chains

class Chain:
    """A compiled chain (wraps a fuse_handle)."""

    def __init__(self, handle: int, spec: str, shape):
        self.handle = handle
        self.spec = spec
        self.shape = tuple(int(s) for s in shape)
        n, o = _I(), _I()
        _check(_lib.fuse_num_inputs(handle, ctypes.byref(n), ctypes.byref(o)))
        self.n_in, self.out_dtype = n.value, o.value
        dts = (_I * max(1, self.n_in))()
        _check(_lib.fuse_input_dtypes(handle, dts, self.n_in))
        self.in_dtypes = [dts[i] for i in range(self.n_in)]

    def __call__(self, inputs, output, stream=None):
        fuse_launch(self, inputs, output, stream)
        return output

    def bind(self, inputs, output) -> "BoundLaunch":
        """This chain on these tensors, for launching again and again."""
        return BoundLaunch(self, inputs, output)

    def release(self):
        if self.handle:
            fuse_release(self)
            self.handle = None


def fuse_compile(spec: str, shape, in_dtype) -> Chain:
    h = _P()
    arr, nd = _shape(shape)
    _check(_lib.fuse_compile(spec.encode(), arr, nd, _dtype(in_dtype), ctypes.byref(h)))
    return Chain(h.value, spec, shape)


def fuse_launch(chain: Chain, inputs, output, stream=None) -> None:
    ptrs = (_P * max(1, len(inputs)))(*[_ptr(t) for t in inputs])
    _check(_lib.fuse_launch(chain.handle, ptrs, len(inputs), _ptr(output), _stream(stream)))


class BoundLaunch:
    """A chain bound to fixed input and output tensors: the pointer array is
    built once, so each call only hands it to fuse_launch (for serving loops
    that launch the same chain on the same buffers step after step).  It holds
    references to the tensors, so they stay allocated while it lives."""

    __slots__ = ("_fn", "_h", "_ptrs", "_n", "_out", "_keep")

    def __init__(self, chain: Chain, inputs, output):
        self._fn = _lib.fuse_launch
        self._h = chain.handle
        self._n = len(inputs)
        self._ptrs = (_P * max(1, self._n))(*[_ptr(t) for t in inputs])
        self._out = _ptr(output)
        self._keep = (chain, list(inputs), output)

    def __call__(self, stream=None) -> None:
        rc = self._fn(self._h, self._ptrs, self._n, self._out, _stream(stream))
        if rc:
            _check(rc)


def fuse_release(chain: Chain) -> None:
    _check(_lib.fuse_release(chain.handle))


def fuse_source(spec: str, shape, in_dtype, bucket: bool = False) -> str:
    fn = _lib.fuse_source_bucket if bucket else _lib.fuse_source
    arr, nd = _shape(shape)
    n = ctypes.c_size_t()
    _check(fn(spec.encode(), arr, nd, _dtype(in_dtype), None, 0, ctypes.byref(n)))
    buf = ctypes.create_string_buffer(n.value + 1)
    _check(fn(spec.encode(), arr, nd, _dtype(in_dtype), buf, n.value + 1, ctypes.byref(n)))
    return buf.value.decode()


def fuse_source_bucket(spec: str, shape, in_dtype) -> str:
    return fuse_source(spec, shape, in_dtype, bucket=True)


def fuse_compile_bucket(spec: str, shape, in_dtype) -> Chain:
    """A chain whose leading dimension shape[0] is an upper bound (see
    fuse_launch_rows)."""
    h = _P()
    arr, nd = _shape(shape)
    _check(_lib.fuse_compile_bucket(spec.encode(), arr, nd, _dtype(in_dtype), ctypes.byref(h)))
    return Chain(h.value, spec, shape)


def fuse_launch_rows(chain: Chain, inputs, output, rows: int, stream=None) -> None:
    ptrs = (_P * max(1, len(inputs)))(*[_ptr(t) for t in inputs])
    _check(_lib.fuse_launch_rows(chain.handle, ptrs, len(inputs), _ptr(output), int(rows),
                                 _stream(stream)))


def fuse_bucket(n: int) -> int:
    b = _I64()
    _check(_lib.fuse_bucket(int(n), ctypes.byref(b)))
    return b.value


_DT_NAMES = {F32: "f32", F16: "f16", BF16: "bf16"}


def fuse_warmup(entries, threads: int = 0) -> tuple[int, int]:
    """Compiles a warm-up list into the library's cache (see fuse.h).  Each
    entry is a line 'spec | d0,d1,... | dtype [| bucket]' or a tuple
    (spec, shape, dtype[, bucket]).  Returns (compiled, already cached)."""
    lines = []
    for e in entries:
        if isinstance(e, str):
            lines.append(e)
        else:
            dims = ",".join(str(int(d)) for d in e[1])
            line = f"{e[0]} | {dims} | {_DT_NAMES[_dtype(e[2])]}"
            lines.append(line + (" | bucket" if len(e) > 3 and e[3] else ""))
    c, h = _I(), _I()
    _check(_lib.fuse_warmup("\n".join(lines).encode(), int(threads), ctypes.byref(c),
                            ctypes.byref(h)))
    return c.value, h.value


# ---------------------------------------------------------------- fixed entry points

def rmsnorm_residual(x, residual, weight, out, residual_out, eps: float = 1e-6, dt=None,
                     rows: int | None = None, hidden: int | None = None, stream=None) -> None:
    if rows is None:
        rows, hidden = x.shape[0], x.shape[-1]
    if dt is None:
        dt = x.dtype
    _check(_lib.rmsnorm_residual(_ptr(x), _ptr(residual), _ptr(weight), _ptr(out),
                                 _ptr(residual_out), rows, hidden, eps, _dtype(dt),
                                 _stream(stream)))


def rmsnorm_linear(x, gamma, w, bias, out, eps: float = 1e-6, scale: float = 1.0, dt=None,
                   M: int | None = None, N: int | None = None, K: int | None = None,
                   stream=None) -> None:
    """out = scale * (RMSNorm(x) * gamma @ w.T + bias) on the tensor cores;
    x [M, K], w [N, K], bias may be None."""
    if M is None:
        M, K = x.shape
        N = w.shape[0]
    if dt is None:
        dt = x.dtype
    _check(_lib.rmsnorm_linear(_ptr(x), _ptr(gamma), _ptr(w), _ptr(bias), _ptr(out), M, N, K, eps,
                               scale, _dtype(dt), _stream(stream)))


def rmsnorm_linear_fold(w, gamma, w_out, dt=None, N: int | None = None, K: int | None = None,
                        stream=None) -> None:
    """w_out = w * gamma (per column k): gamma folded into the weight for the
    fast path of rmsnorm_linear (call it with gamma=None)."""
    if N is None:
        N, K = w.shape
    if dt is None:
        dt = w.dtype
    _check(_lib.rmsnorm_linear_fold(_ptr(w), _ptr(gamma), _ptr(w_out), N, K, _dtype(dt),
                                    _stream(stream)))


def fuse_device_error() -> int:
    c = _I()
    _check(_lib.fuse_device_error(ctypes.byref(c)))
    return c.value


def layernorm_residual(x, residual, gamma, beta, out, residual_out, eps: float = 1e-5, dt=None,
                       rows: int | None = None, hidden: int | None = None, stream=None) -> None:
    """residual/residual_out, gamma, beta may be None."""
    if rows is None:
        rows, hidden = x.shape[0], x.shape[-1]
    if dt is None:
        dt = x.dtype
    _check(_lib.layernorm_residual(_ptr(x), _ptr(residual), _ptr(gamma), _ptr(beta), _ptr(out),
                                   _ptr(residual_out), rows, hidden, eps, _dtype(dt),
                                   _stream(stream)))


def rope_qkv_split(qkv, q, k, v, heads: int, head_dim: int, pos0: int = 0,
                   base: float = 10000.0, dt=None, tokens: int | None = None, stream=None) -> None:
    if tokens is None:
        tokens = qkv.shape[0]
    if dt is None:
        dt = qkv.dtype
    _check(_lib.rope_qkv_split(_ptr(qkv), _ptr(q), _ptr(k), _ptr(v), tokens, heads, head_dim,
                               pos0, base, _dtype(dt), _stream(stream)))


def rope_qkv_split_noalloc(qkv, q, k, v, heads: int, head_dim: int, pos0: int = 0,
                           base: float = 10000.0, dt=None, tokens: int | None = None,
                           stream=None) -> None:
    """rope_qkv_split for callers that cannot let the library allocate device
    memory or compile at run time (see include/fuse.h): the cos/sin rows live
    in a fixed 4 MB array inside the library; tokens * head_dim <= 2^20."""
    if tokens is None:
        tokens = qkv.shape[0]
    if dt is None:
        dt = qkv.dtype
    _check(_lib.rope_qkv_split_noalloc(_ptr(qkv), _ptr(q), _ptr(k), _ptr(v), tokens, heads,
                                       head_dim, pos0, base, _dtype(dt), _stream(stream)))


def detect_decode(feats, hw, strides, anchors, na: int, no: int, out, in_dt=None,
                  stream=None) -> None:
    ns = len(feats)
    fp = (_P * ns)(*[_ptr(f) for f in feats])
    hwa = (_I * (2 * ns))(*[int(d) for pair in hw for d in pair])
    st = (_F * ns)(*[float(s) for s in strides])
    flat = [float(a) for a in _flatten(anchors)]
    an = (_F * len(flat))(*flat)
    if in_dt is None:
        in_dt = feats[0].dtype
    _check(_lib.detect_decode(fp, hwa, st, an, ns, na, no, _dtype(in_dt), _ptr(out),
                              _stream(stream)))


class DetectDecoder:
    """detect_decode with its fixed arguments -- per-scale shapes, strides,
    anchors, anchors per cell, outputs per anchor, input dtype -- converted
    once; a call passes only the feature maps, the output and the stream
    (about half the host time of a detect_decode call)."""

    def __init__(self, hw, strides, anchors, na: int, no: int, in_dt):
        self.ns, self.na, self.no, self.dt = len(hw), int(na), int(no), _dtype(in_dt)
        self._hw = (_I * (2 * self.ns))(*[int(d) for pair in hw for d in pair])
        self._st = (_F * self.ns)(*[float(v) for v in strides])
        flat = [float(a) for a in _flatten(anchors)]
        self._an = (_F * len(flat))(*flat)
        self._feats = _P * self.ns

    def __call__(self, feats, out, stream=None) -> None:
        if len(feats) != self.ns:
            raise ValueError(f"{self.ns} feature maps expected, got {len(feats)}")
        _check(_lib.detect_decode(self._feats(*[_ptr(f) for f in feats]), self._hw, self._st,
                                  self._an, self.ns, self.na, self.no, self.dt, _ptr(out),
                                  _stream(stream)))


def channel_shuffle(x, out, groups: int, dt=None, shape=None, stream=None) -> None:
    n, c, h, w = shape if shape is not None else x.shape
    if dt is None:
        dt = x.dtype
    _check(_lib.channel_shuffle(_ptr(x), _ptr(out), n, c, h, w, groups, _dtype(dt),
                                _stream(stream)))


def _flatten(a):
    try:
        import numpy as np
        return np.asarray(a, dtype=float).reshape(-1).tolist()
    except Exception:  # pragma: no cover
        return [x for row in a for pair in row for x in pair]


# ---------------------------------------------------------------- graphs

class Graph:
    """A recorded sequence of library launches (wraps a fuse_graph_handle)."""

    def __init__(self, handle: int):
        self.handle = handle
        n = _I64()
        _check(_lib.fuse_graph_nodes(handle, ctypes.byref(n)))
        self.nodes = n.value

    def launch(self, stream=None) -> None:
        fuse_graph_launch(self, stream)

    def release(self) -> None:
        if self.handle:
            fuse_graph_release(self)
            self.handle = None


def fuse_graph_begin(stream=None) -> None:
    _check(_lib.fuse_graph_begin(_stream(stream)))


def fuse_graph_end(stream=None) -> Graph:
    h = _P()
    _check(_lib.fuse_graph_end(_stream(stream), ctypes.byref(h)))
    return Graph(h.value)


def fuse_graph_launch(graph: Graph, stream=None) -> None:
    _check(_lib.fuse_graph_launch(graph.handle, _stream(stream)))


def fuse_graph_nodes(graph: Graph) -> int:
    return graph.nodes


def fuse_graph_release(graph: Graph) -> None:
    _check(_lib.fuse_graph_release(graph.handle))


# ---------------------------------------------------------------- diagnostics

def fuse_last_error() -> str:
    return (_lib.fuse_last_error() or b"").decode(errors="replace")


def fuse_stats() -> dict:
    c, h, l = _I64(), _I64(), _I64()
    ms = ctypes.c_double()
    _check(_lib.fuse_stats(ctypes.byref(c), ctypes.byref(h), ctypes.byref(l), ctypes.byref(ms)))
    return {"compiles": c.value, "cache_hits": h.value, "launches": l.value,
            "compile_ms": ms.value}


def fuse_device_sms() -> int:
    s = _I()
    _check(_lib.fuse_device_sms(ctypes.byref(s)))
    return s.value


def fuse_selftest_bounded_wait(spins: int, stream=None) -> None:
    """Launch the bounded-wait self test (see include/fuse.h); afterwards
    fuse_device_error() returns 1."""
    _check(_lib.fuse_selftest_bounded_wait(int(spins), _stream(stream)))
