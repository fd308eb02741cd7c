"""Python binding of libmoe_w4.so: the routed W4A16 MoE layer on GB300.

Argument marshalling only.  Every step of the layer runs in the library's
CUDA kernels; this module passes device pointers (torch tensors on a CUDA
device), sizes and the current CUDA stream through ctypes and raises on any
non-OK status.  There is no fallback: if the library is missing, importing
the binding's functions raises.

Entry points (same names as the C ABI in include/moe_w4.h):
    route_topk, permute, expert_ffn_w4a16, combine, layer_forward,
    layer_workspace_size, permute_workspace_size, expert_ffn_workspace_size,
    get_device_error, status_str, version
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_w4.so")

MOE_OK = 0
STATUS = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_MISALIGNED", 3: "MOE_ERR_UNSUPPORTED",
    4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_DEVICE_RANGE", 7: "MOE_ERR_TIMEOUT",
    8: "MOE_ERR_F16_RANGE", 9: "MOE_ERR_SCRATCH_LIMIT", 10: "MOE_ERR_CAPTURE",
}


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class moe_w4_layer(ctypes.Structure):
    _fields_ = [
        ("E", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("w13_q", ctypes.c_void_p), ("w13_s", ctypes.c_void_p), ("w13_z", ctypes.c_void_p),
        ("w2_q", ctypes.c_void_p), ("w2_s", ctypes.c_void_p), ("w2_z", ctypes.c_void_p),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m bit_quantized_expert_moe_gb300.build` (no CPU fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        V, I32, SZ, P = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.POINTER(moe_w4_layer)
        sig = {
            "moe_route_topk": (I32, [V, I32, I32, I32, V, V, V]),
            "moe_permute": (I32, [V, I32, I32, I32, V, I32, V, V, V, V, V, V, SZ, V]),
            "moe_permute_workspace_size": (SZ, [I32, I32, I32]),
            "moe_expert_ffn_w4a16": (I32, [P, V, V, I32, V, V, V, SZ, V]),
            "moe_expert_ffn_workspace_size": (SZ, [P, I32]),
            "moe_combine": (I32, [V, V, V, I32, I32, I32, V, V]),
            "moe_layer_forward": (I32, [P, V, V, I32, I32, V, V, V, SZ, V]),
            "moe_layer_workspace_size": (SZ, [P, I32, I32]),
            "moe_get_device_error": (I32, [V, V]),
            "moe_profile_stages": (I32, [V, I32, V]),
            "moe_kernel_launches": (ctypes.c_uint64, []),
            "moe_status_str": (ctypes.c_char_p, [I32]),
            "moe_version": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, what)


def status_str(status: int) -> str:
    return lib().moe_status_str(status).decode()


def version() -> str:
    return lib().moe_version().decode()


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zeroed device workspace (its first 256 bytes hold the error word)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------
@dataclass
class Layer:
    """One layer's quantised expert weights resident on a device."""
    E: int
    d_model: int
    d_ff: int
    w13_q: torch.Tensor  # int32 view of uint32 [E, 2f, d/8]
    w13_s: torch.Tensor  # float16 [E, 2f, d/128]
    w13_z: torch.Tensor
    w2_q: torch.Tensor   # int32 view of uint32 [E, d, f/8]
    w2_s: torch.Tensor   # float16 [E, d, f/128]
    w2_z: torch.Tensor

    @classmethod
    def from_numpy(cls, w: dict, device="cuda") -> "Layer":
        def q(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(device)

        def h(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).to(device)

        E, f2, d8 = w["w13_q"].shape
        return cls(E=E, d_model=d8 * 8, d_ff=f2 // 2, w13_q=q(w["w13_q"]), w13_s=h(w["w13_s"]),
                   w13_z=h(w["w13_z"]), w2_q=q(w["w2_q"]), w2_s=h(w["w2_s"]), w2_z=h(w["w2_z"]))

    def c_struct(self) -> moe_w4_layer:
        return moe_w4_layer(self.E, self.d_model, self.d_ff, 128, _ptr(self.w13_q), _ptr(self.w13_s),
                            _ptr(self.w13_z), _ptr(self.w2_q), _ptr(self.w2_s), _ptr(self.w2_z))

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in
                   (self.w13_q, self.w13_s, self.w13_z, self.w2_q, self.w2_s, self.w2_z))


# ---------------------------------------------------------------------------
def route_topk(logits: torch.Tensor, k: int, ids: torch.Tensor | None = None, w: torch.Tensor | None = None,
               stream=None):
    T, E = logits.shape
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if w is None:
        w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(lib().moe_route_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _stream(stream)), "moe_route_topk")
    return ids, w


def permute_workspace_size(T: int, k: int, E: int) -> int:
    return lib().moe_permute_workspace_size(T, k, E)


def permute(topk_ids: torch.Tensor, E: int, x: torch.Tensor | None = None, want_x_perm: bool = False,
            ws: torch.Tensor | None = None, stream=None) -> dict:
    T, k = topk_ids.shape
    R = T * k
    dev = topk_ids.device
    out = {
        "counts": torch.empty(E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "sorted": torch.empty(max(R, 1), dtype=torch.int32, device=dev),
        "inv": torch.empty(max(R, 1), dtype=torch.int32, device=dev),
    }
    d = 0
    x_perm = None
    if want_x_perm:
        d = x.shape[1]
        x_perm = torch.empty((max(R, 1), d), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = workspace(permute_workspace_size(T, k, E), dev)
    st = lib().moe_permute(_ptr(topk_ids), T, k, E, _ptr(x) if want_x_perm else None, d,
                           _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["sorted"]), _ptr(out["inv"]),
                           _ptr(x_perm), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "moe_permute")
    out["sorted"] = out["sorted"][:R]
    out["inv"] = out["inv"][:R]
    if want_x_perm:
        out["x_perm"] = x_perm[:R]
    out["ws"] = ws
    return out


def expert_ffn_workspace_size(layer: Layer, R: int) -> int:
    return lib().moe_expert_ffn_workspace_size(ctypes.byref(layer.c_struct()), R)


def expert_ffn_w4a16(layer: Layer, x_perm: torch.Tensor, offsets: torch.Tensor, row_w: torch.Tensor | None = None,
                     y_perm: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    R = x_perm.shape[0]
    if y_perm is None:
        y_perm = torch.empty((R, layer.d_model), dtype=torch.bfloat16, device=x_perm.device)
    if ws is None:
        ws = workspace(expert_ffn_workspace_size(layer, R), x_perm.device)
    L = layer.c_struct()
    st = lib().moe_expert_ffn_w4a16(ctypes.byref(L), _ptr(x_perm), _ptr(offsets), R, _ptr(row_w), _ptr(y_perm),
                                    _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "moe_expert_ffn_w4a16")
    return y_perm


def combine(y_perm: torch.Tensor, inv: torch.Tensor, topk_w: torch.Tensor, out: torch.Tensor | None = None,
            stream=None):
    T, k = topk_w.shape
    d = y_perm.shape[1]
    if out is None:
        out = torch.empty((T, d), dtype=torch.bfloat16, device=y_perm.device)
    _check(lib().moe_combine(_ptr(y_perm), _ptr(inv), _ptr(topk_w), T, k, d, _ptr(out), _stream(stream)),
           "moe_combine")
    return out


def layer_workspace_size(layer: Layer, T: int, k: int) -> int:
    return lib().moe_layer_workspace_size(ctypes.byref(layer.c_struct()), T, k)


class LayerCall:
    """A prepared moe_layer_forward call: the C struct is built once, so the
    per-call cost is one ctypes call (used for timing loops and graphs)."""

    def __init__(self, layer: Layer, T: int, k: int, ws: torch.Tensor | None = None, device="cuda"):
        self.layer, self.T, self.k = layer, T, k
        self.L = layer.c_struct()
        self.ws = ws if ws is not None else workspace(layer_workspace_size(layer, T, k), device)
        self._fn = lib().moe_layer_forward

    def __call__(self, x: torch.Tensor, logits: torch.Tensor, out: torch.Tensor,
                 topk_ids_out: torch.Tensor | None = None, stream=None):
        st = self._fn(ctypes.byref(self.L), _ptr(x), _ptr(logits), self.T, self.k, _ptr(out), _ptr(topk_ids_out),
                      _ptr(self.ws), self.ws.numel(), _stream(stream))
        _check(st, "moe_layer_forward")
        return out


def layer_forward(layer: Layer, x: torch.Tensor, logits: torch.Tensor, k: int, out: torch.Tensor | None = None,
                  topk_ids_out: torch.Tensor | None = None, ws: torch.Tensor | None = None, stream=None):
    T = x.shape[0]
    if out is None:
        out = torch.empty((T, layer.d_model), dtype=torch.bfloat16, device=x.device)
    call = LayerCall(layer, T, k, ws=ws, device=x.device)
    return call(x, logits, out, topk_ids_out, stream)


def kernel_launches() -> int:
    """CUDA kernels launched by the library so far in this process."""
    return int(lib().moe_kernel_launches())


class StageProfiler:
    """Records the six stage events of every moe_layer_forward call made from
    this thread while active (see moe_profile_stages in the header)."""

    def __init__(self, calls: int):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(6 * calls)]
        for ev in self.events:  # materialise the CUDA events
            ev.record()
        torch.cuda.synchronize()
        self._arr = (ctypes.c_void_p * len(self.events))(*[ev.cuda_event for ev in self.events])
        self._cursor = ctypes.c_int32(0)

    def __enter__(self):
        self._cursor.value = 0
        _check(lib().moe_profile_stages(self._arr, len(self.events), ctypes.byref(self._cursor)), "moe_profile_stages")
        return self

    def __exit__(self, *exc):
        lib().moe_profile_stages(None, 0, None)

    def stage_ms(self):
        """Per recorded call: durations of the five stages in ms (after a sync)."""
        torch.cuda.synchronize()
        n = self._cursor.value // 6
        out = []
        for c in range(n):
            ev = self.events[6 * c:6 * c + 6]
            out.append([ev[i].elapsed_time(ev[i + 1]) for i in range(5)])
        return out


def get_device_error(ws: torch.Tensor, stream=None) -> int:
    """Reads and clears the workspace error word (synchronises the stream)."""
    return lib().moe_get_device_error(_ptr(ws), _stream(stream))
