"""Python binding of the B300 MiTA forward library (``libmita.so``).

Argument marshalling only: every step of the operator runs in the CUDA
kernels behind the C ABI declared in ``include/mita.h``.  PyTorch supplies
device memory and streams.  There is no CPU fallback: if the library is
missing or no CUDA device is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmita.so")

MITA_F32, MITA_BF16 = 0, 1
MITA_OK, MITA_ERR_INVALID_ARG, MITA_ERR_UNSUPPORTED, MITA_ERR_CUDA = 0, 1, 2, 3
MITA_ERR_TIMEOUT, MITA_ERR_OOM, MITA_ERR_DEVICE = 4, 5, 6
STATUS = {0: "MITA_OK", 1: "MITA_ERR_INVALID_ARG", 2: "MITA_ERR_UNSUPPORTED", 3: "MITA_ERR_CUDA",
          4: "MITA_ERR_TIMEOUT", 5: "MITA_ERR_OOM", 6: "MITA_ERR_DEVICE"}
OPT_PATH, OPT_KEEP_LANDMARKS, OPT_ROUTING_ONLY, OPT_ROUTES = 0, 1, 2, 3
PATH_AUTO, PATH_STAGED, PATH_FUSED, PATH_TILED = 0, 1, 2, 3
PATH_NAMES = {PATH_STAGED: "staged", PATH_FUSED: "fused", PATH_TILED: "tiled"}

# Every entry point declared in include/mita.h.
EXPORTS = ("mita_plan", "mita_forward", "mita_forward_host", "mita_backward", "mita_get_status", "mita_destroy", "mita_strerror",
           "mita_set_option", "mita_get_path", "mita_get_landmarks", "mita_workspace_bytes",
           "mita_launch_count", "mita_forward_noalloc", "mita_noalloc_scratch_bytes",
           "mita_testing_bucket", "mita_testing_wait")


class MitaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({strerror(code)})")


class Grid(ctypes.Structure):
    _fields_ = [("gh", ctypes.c_int), ("gw", ctypes.c_int), ("ph", ctypes.c_int), ("pw", ctypes.c_int)]


_lib = None


def load(path: str | None = None):
    """Load libmita.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} (run __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    vp, i, ip = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int32)
    lib.mita_plan.argtypes = [ctypes.POINTER(vp), i, i, i, i, Grid, i, i, i]
    lib.mita_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    lib.mita_forward_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    lib.mita_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.mita_get_status.argtypes = [vp]
    lib.mita_destroy.argtypes = [vp]
    lib.mita_destroy.restype = None
    lib.mita_strerror.argtypes = [i]
    lib.mita_strerror.restype = ctypes.c_char_p
    lib.mita_set_option.argtypes = [vp, i, i]
    lib.mita_get_path.argtypes = [vp]
    lib.mita_get_landmarks.argtypes = [vp, vp, vp, vp]
    lib.mita_workspace_bytes.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64)]
    lib.mita_launch_count.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64)]
    lib.mita_forward_noalloc.argtypes = [i, i, i, i, Grid, i, i, i, vp, vp, vp, vp, vp, vp, vp]
    lib.mita_noalloc_scratch_bytes.argtypes = []
    lib.mita_testing_bucket.argtypes = [vp, vp, vp]
    lib.mita_testing_wait.argtypes = [vp, ctypes.c_longlong, vp]
    for name in EXPORTS:
        if name not in ("mita_destroy", "mita_strerror", "mita_noalloc_scratch_bytes"):
            getattr(lib, name).restype = i
    lib.mita_noalloc_scratch_bytes.restype = ctypes.c_uint64
    if path is None:
        _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().mita_strerror(int(code)).decode()
    except RuntimeError:
        return "library not loaded"


def _check(rc: int, where: str):
    if rc != MITA_OK:
        raise MitaError(rc, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """A MiTA forward plan: shapes, dtype and the device workspace
    (``mita_plan`` / ``mita_destroy``)."""

    def __init__(self, B, H, N, d, grid, m, k, dtype="bf16"):
        self.lib = load()
        self.B, self.H, self.N, self.d, self.m, self.k = B, H, N, d, m, k
        self.grid = tuple(grid)
        self.dtype = dtype
        h = ctypes.c_void_p()
        code = MITA_BF16 if dtype == "bf16" else MITA_F32
        _check(self.lib.mita_plan(ctypes.byref(h), B, H, N, d, Grid(*grid), m, k, code), "mita_plan")
        self.handle = h

    @classmethod
    def for_workload(cls, w):
        return cls(w.B, w.H, w.N, w.d, w.grid, w.m, w.k, w.dtype)

    def set_option(self, option: int, value: int):
        _check(self.lib.mita_set_option(self.handle, option, value), "mita_set_option")

    def set_path(self, path: str):
        self.set_option(OPT_PATH, {"auto": PATH_AUTO, "staged": PATH_STAGED, "fused": PATH_FUSED,
                                  "tiled": PATH_TILED}[path])

    @property
    def path(self) -> str:
        r = self.lib.mita_get_path(self.handle)
        if r < 0:
            raise MitaError(-r, "mita_get_path")
        return PATH_NAMES[r]

    def forward(self, Q, K, V, out, expert_idx=None, route=None, stream=None):
        """Enqueue ``mita_forward`` on ``stream`` (default: torch's current
        stream).  All tensors are CUDA tensors in the layouts of mita.h."""
        rc = self.lib.mita_forward(self.handle, _ptr(Q), _ptr(K), _ptr(V), _ptr(out), _ptr(expert_idx),
                                   _ptr(route), _stream_ptr(stream))
        _check(rc, "mita_forward")

    def forward_host(self, Q, K, V, out, expert_idx=None, route=None, stream=None):
        """Enqueue ``mita_forward_host`` on ``stream`` (default: torch's
        current stream): the same forward on CPU tensors (page-locked for the
        copies to overlap), streamed through the device in chunks of heads.
        The results are in ``out``, ``expert_idx`` and ``route`` once the
        stream has passed the call."""
        for t in (Q, K, V, out, expert_idx, route):
            if t is not None and (t.is_cuda or not t.is_contiguous()):
                raise ValueError("forward_host takes contiguous CPU tensors")
        rc = self.lib.mita_forward_host(self.handle, _ptr(Q), _ptr(K), _ptr(V), _ptr(out), _ptr(expert_idx),
                                        _ptr(route), _stream_ptr(stream))
        _check(rc, "mita_forward_host")

    def backward(self, Q, K, V, dOut, dQ, dK, dV, stream=None):
        """Enqueue ``mita_backward``: input gradients dQ, dK, dV (fp32 CUDA
        tensors [B, H, N, d], overwritten) for the output gradient dOut."""
        rc = self.lib.mita_backward(self.handle, _ptr(Q), _ptr(K), _ptr(V), _ptr(dOut), _ptr(dQ), _ptr(dK),
                                    _ptr(dV), _stream_ptr(stream))
        _check(rc, "mita_backward")

    def status(self) -> int:
        return self.lib.mita_get_status(self.handle)

    def landmarks(self, Ql, Vl, stream=None):
        _check(self.lib.mita_get_landmarks(self.handle, _ptr(Ql), _ptr(Vl), _stream_ptr(stream)),
               "mita_get_landmarks")

    def workspace_bytes(self) -> int:
        b = ctypes.c_uint64()
        _check(self.lib.mita_workspace_bytes(self.handle, ctypes.byref(b)), "mita_workspace_bytes")
        return b.value

    def launch_count(self) -> int:
        n = ctypes.c_uint64()
        _check(self.lib.mita_launch_count(self.handle, ctypes.byref(n)), "mita_launch_count")
        return n.value

    def close(self):
        if getattr(self, "handle", None):
            self.lib.mita_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def forward_noalloc(Q, K, V, out, grid, m, k, expert_idx=None, route=None, stream=None):
    """``mita_forward_noalloc``: the forward without a plan and without any
    device allocation (scratch in the library's fixed device array)."""
    import torch
    B, H, N, d = Q.shape
    code = MITA_BF16 if Q.dtype == torch.bfloat16 else MITA_F32
    rc = load().mita_forward_noalloc(B, H, N, d, Grid(*grid), m, k, code, _ptr(Q), _ptr(K), _ptr(V),
                                     _ptr(out), _ptr(expert_idx), _ptr(route), _stream_ptr(stream))
    _check(rc, "mita_forward_noalloc")


def mita_forward(Q, K, V, grid, m, k, path="auto", return_all=True):
    """Allocate outputs and run one forward on CUDA tensors [B, H, N, d].
    Returns (out, expert_idx, route)."""
    import torch
    B, H, N, d = Q.shape
    dtype = "bf16" if Q.dtype == torch.bfloat16 else "f32"
    plan = Plan(B, H, N, d, grid, m, k, dtype)
    plan.set_path(path)
    out = torch.empty_like(Q)
    idx = torch.empty(B, H, m, k, dtype=torch.int32, device=Q.device)
    route = torch.empty(B, H, N, dtype=torch.int32, device=Q.device)
    plan.forward(Q, K, V, out, idx, route)
    st = plan.status()
    plan.close()
    _check(st, "device status")
    return out, idx, route
