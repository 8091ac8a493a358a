"""Python binding of the GB300 NVFP4 library (``libnvfp4.so``, C ABI in
``include/nvfp4.h``).

Argument marshalling only: every step runs in the library's sm_103a kernels.
PyTorch provides device memory and the current CUDA stream.  If the library
has not been built (``nvfp4_block_scaled_act_gb300.build.build()``) every call
raises ``RuntimeError``: there is no fallback.

The functions keep the C names; tensors are CUDA tensors, allocated here when
the caller passes none:

* ``nvfp4_compute_global(x)`` -> fp32 [1] on the device: 2688 / amax(x)
* ``nvfp4_quantize_act(x, g)`` -> (codes uint8 [M, K/2], scales uint8 [sw])
* ``nvfp4_linear_w4a4(a_codes, a_sf, w_codes, w_sf, alpha, N, K)`` -> bf16 [M, N]
* ``nvfp4_linear_w4a16(x, w_codes, w_sf, alpha, N, K)`` -> bf16 [T, N]
* ``nvfp4_moe_w4a4(...)`` -> bf16 [T, H]
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4.so")

NVFP4_OK = 0
STATUS_NAMES = {
    0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_UNSUPPORTED_SHAPE",
    3: "NVFP4_ERR_MISALIGNED", 4: "NVFP4_ERR_WORKSPACE_TOO_SMALL", 5: "NVFP4_ERR_CUDA",
    6: "NVFP4_ERR_DEVICE_TIMEOUT", 7: "NVFP4_ERR_BAD_EXPERT_ID", 8: "NVFP4_ERR_NO_DEVICE",
}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_I = ctypes.c_int
_ST = ctypes.c_int  # nvfp4_status


class MoELayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "counts", "offsets", "n_tiles", "row_map", "tile_expert", "pos", "a1_codes", "a1_sf",
        "h_codes", "h_sf", "y", "hist", "total")] + [("p_max", ctypes.c_int64), ("row_block", ctypes.c_int64)]


# name -> (restype, argtypes); the exported symbols of include/nvfp4.h
SIGNATURES = {
    "nvfp4_status_string": (ctypes.c_char_p, [_I]),
    "nvfp4_version": (_I, []),
    "nvfp4_scale_bytes": (_SZ, [_I64, _I64]),
    "nvfp4_compute_global": (_ST, [_P, _I64, _I64, _I64, _P, _P]),
    "nvfp4_make_alpha": (_ST, [_P, _P, _I64, _P, _P]),
    "nvfp4_reduce_max": (_ST, [_P, _I64, _P, _P]),
    "nvfp4_quantize_act": (_ST, [_P, _I64, _I64, _I64, _P, _P, _P, _P]),
    "nvfp4_linear_w4a4": (_ST, [_P, _P, _I64, _P, _P, _I64, _I64, _P, _P, _I64, _P]),
    "nvfp4_linear_w4a16_workspace": (_SZ, [_I64, _I64, _I64]),
    "nvfp4_linear_w4a16": (_ST, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _P, _I64, _P, _SZ, _P]),
    "nvfp4_linear_w4a16_noalloc": (_ST, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _P, _I64, _P]),
    "nvfp4_moe_workspace": (_SZ, [_I64, _I64, _I64, _I64, _I]),
    "nvfp4_moe_workspace_layout": (_ST, [_I64, _I64, _I64, _I64, _I, ctypes.POINTER(MoELayout)]),
    "nvfp4_moe_w4a4": (_ST, [_P, _I64, _I64, _I64, _I64, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                             _P, _P, _P, _SZ, _P]),
    "nvfp4_moe_calibrate": (_ST, [_P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "nvfp4_moe_w4a16_workspace": (_SZ, [_I64, _I64, _I64, _I64, _I]),
    "nvfp4_moe_w4a16": (_ST, [_P, _I64, _I64, _I64, _I64, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                              _P]),
    "nvfp4_device_status": (_ST, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "nvfp4_selftest_wait_timeout": (_ST, [_P]),
}

_lock = threading.Lock()
_lib = None


class NVFP4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}")
        self.status = status


def load_library(path: str = LIB_PATH):
    """Load ``libnvfp4.so`` (raises if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"NVFP4 CUDA library not built: {path} is missing "
                                   "(run nvfp4_block_scaled_act_gb300.build.build())")
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != NVFP4_OK:
        raise NVFP4Error(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t


# ---------------------------------------------------------------------------
# entry points (C names)
# ---------------------------------------------------------------------------

def nvfp4_scale_bytes(rows: int, k: int) -> int:
    return int(load_library().nvfp4_scale_bytes(rows, k))


def nvfp4_compute_global(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per-tensor global 2688 / amax(x) of a bf16 [rows, cols] tensor (fp32 [1])."""
    _cuda(x, "x")
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    out = out if out is not None else torch.empty(1, dtype=torch.float32, device=x.device)
    _check("nvfp4_compute_global", load_library().nvfp4_compute_global(
        _ptr(x), x.shape[0], x.shape[1], x.stride(0), _ptr(out), _stream(stream)))
    return out


def nvfp4_make_alpha(g_a: torch.Tensor | None, g_w: torch.Tensor, out: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """alpha[i] = 1 / (g_a * g_w[i]) (g_a None: 1 / g_w[i])."""
    out = out if out is not None else torch.empty_like(g_w)
    _check("nvfp4_make_alpha", load_library().nvfp4_make_alpha(
        _ptr(g_a), _ptr(g_w), g_w.numel(), _ptr(out), _stream(stream)))
    return out


def nvfp4_reduce_max(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    out = out if out is not None else torch.empty(1, dtype=torch.float32, device=x.device)
    _check("nvfp4_reduce_max", load_library().nvfp4_reduce_max(_ptr(x), x.numel(), _ptr(out),
                                                                _stream(stream)))
    return out


def nvfp4_quantize_act(x: torch.Tensor, g: torch.Tensor, codes: torch.Tensor | None = None,
                       scales: torch.Tensor | None = None, stream=None):
    """bf16 [M, K] (row stride allowed) -> (codes [M, K/2], swizzled scales)."""
    _cuda(x, "x")
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if codes is None:
        codes = torch.empty(M, K // 2, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(nvfp4_scale_bytes(max(M, 1), K), dtype=torch.uint8, device=x.device)
    _check("nvfp4_quantize_act", load_library().nvfp4_quantize_act(
        _ptr(x), M, K, x.stride(0), _ptr(g), _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


def nvfp4_linear_w4a4(a_codes, a_sf, w_codes, w_sf, alpha, N: int, K: int, out=None, stream=None):
    """bf16 [M, N] = alpha * dequant(a) @ dequant(w).T (NVFP4 x NVFP4, tcgen05)."""
    M = a_codes.shape[0]
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=a_codes.device)
    _check("nvfp4_linear_w4a4", load_library().nvfp4_linear_w4a4(
        _ptr(a_codes), _ptr(a_sf), M, _ptr(w_codes), _ptr(w_sf), N, K, _ptr(alpha), _ptr(out),
        out.stride(0), _stream(stream)))
    return out


def nvfp4_linear_w4a16_workspace(T: int, N: int, K: int) -> int:
    return int(load_library().nvfp4_linear_w4a16_workspace(T, N, K))


def nvfp4_linear_w4a16(x, w_codes, w_sf, alpha, N: int, K: int, out=None, workspace=None, stream=None):
    """bf16 [T, N] = alpha * x @ dequant(w).T for T <= 16 (decode)."""
    _cuda(x, "x")
    T = x.shape[0]
    if out is None:
        out = torch.empty(T, N, dtype=torch.bfloat16, device=x.device)
    need = nvfp4_linear_w4a16_workspace(T, N, K)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("nvfp4_linear_w4a16", load_library().nvfp4_linear_w4a16(
        _ptr(x), T, x.stride(0), _ptr(w_codes), _ptr(w_sf), N, K, _ptr(alpha), _ptr(out),
        out.stride(0), _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def nvfp4_moe_workspace(T: int, H: int, I: int, E: int, topk: int) -> int:
    return int(load_library().nvfp4_moe_workspace(T, H, I, E, topk))


def nvfp4_moe_workspace_layout(T: int, H: int, I: int, E: int, topk: int) -> MoELayout:
    lay = MoELayout()
    _check("nvfp4_moe_workspace_layout",
           load_library().nvfp4_moe_workspace_layout(T, H, I, E, topk, ctypes.byref(lay)))
    return lay


def nvfp4_moe_w4a4(x, topk_ids, topk_w, g_a1, w13_codes, w13_sf, alpha13, g_a2, w2_codes, w2_sf,
                   alpha2, E: int, I: int, out=None, workspace=None, stream=None):
    """W4A4 MoE layer: bf16 [T, H] -> bf16 [T, H]."""
    _cuda(x, "x")
    T, H = x.shape
    topk = topk_ids.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(nvfp4_moe_workspace(T, H, I, E, topk), 1), dtype=torch.uint8,
                                device=x.device)
    _check("nvfp4_moe_w4a4", load_library().nvfp4_moe_w4a4(
        _ptr(x), T, H, I, E, topk, _ptr(topk_ids), _ptr(topk_w), _ptr(g_a1), _ptr(w13_codes),
        _ptr(w13_sf), _ptr(alpha13), _ptr(g_a2), _ptr(w2_codes), _ptr(w2_sf), _ptr(alpha2),
        _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def nvfp4_moe_w4a16_workspace(T: int, H: int, I: int, E: int, topk: int) -> int:
    return int(load_library().nvfp4_moe_w4a16_workspace(T, H, I, E, topk))


def nvfp4_moe_w4a16(x, topk_ids, topk_w, w13_codes, w13_sf, alpha13, w2_codes, w2_sf, alpha2, E: int, I: int,
                    out=None, workspace=None, stream=None):
    """W4A16 MoE layer for small batches (T <= 64): bf16 [T, H] -> bf16 [T, H];
    alpha13 = 1 / g_w13 and alpha2 = 1 / g_w2 per expert."""
    _cuda(x, "x")
    T, H = x.shape
    topk = topk_ids.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(nvfp4_moe_w4a16_workspace(T, H, I, E, topk), 1), dtype=torch.uint8,
                                device=x.device)
    _check("nvfp4_moe_w4a16", load_library().nvfp4_moe_w4a16(
        _ptr(x), T, H, I, E, topk, _ptr(topk_ids), _ptr(topk_w), _ptr(w13_codes), _ptr(w13_sf),
        _ptr(alpha13), _ptr(w2_codes), _ptr(w2_sf), _ptr(alpha2), _ptr(out), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return out


def nvfp4_moe_calibrate(x_calib, g_a1, w13_codes, w13_sf, alpha13, E: int, I: int, amax=None,
                        g_a2=None, workspace=None, stream=None):
    """Input global of the second MoE GEMM from a calibration batch: returns
    (g_a2 fp32 [1], amax fp32 [E])."""
    Tc, H = x_calib.shape
    dev = x_calib.device
    amax = amax if amax is not None else torch.empty(E, dtype=torch.float32, device=dev)
    g_a2 = g_a2 if g_a2 is not None else torch.empty(1, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(nvfp4_moe_workspace(Tc, H, I, E, E), dtype=torch.uint8, device=dev)
    _check("nvfp4_moe_calibrate", load_library().nvfp4_moe_calibrate(
        _ptr(x_calib), Tc, H, I, E, _ptr(g_a1), _ptr(w13_codes), _ptr(w13_sf), _ptr(alpha13),
        _ptr(amax), _ptr(g_a2), _ptr(workspace), workspace.numel(), _stream(stream)))
    return g_a2, amax


def nvfp4_selftest_wait_timeout(stream=None) -> None:
    """Launch the timeout self-test: one CTA's bounded pipeline wait runs out
    (about a second) and the device status word reads NVFP4_ERR_DEVICE_TIMEOUT."""
    _check("nvfp4_selftest_wait_timeout", load_library().nvfp4_selftest_wait_timeout(_stream(stream)))


def nvfp4_device_status(stream=None) -> int:
    """Synchronise, read and clear the device status word."""
    v = ctypes.c_int32(0)
    _check("nvfp4_device_status", load_library().nvfp4_device_status(_stream(stream), ctypes.byref(v)))
    return int(v.value)


# ---------------------------------------------------------------------------
# weight preparation (sequences of the calls above)
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class NVFP4Weight:
    """A row-major NVFP4 tensor on the device: codes [N, K/2], swizzled scales,
    per-tensor global (fp32 [1]) and the per-part globals of a fused weight."""
    codes: torch.Tensor
    scales: torch.Tensor
    g: torch.Tensor
    part_g: list
    N: int
    K: int


def quantize_weight(parts, stream=None) -> NVFP4Weight:
    """Quantise a weight given as one bf16 [N, K] tensor or a list of parts
    (a fused weight): each part with its own global, block scales unchanged,
    and the fused tensor taking the largest per-part global."""
    if isinstance(parts, torch.Tensor):
        parts = [parts]
    K = parts[0].shape[1]
    N = sum(p.shape[0] for p in parts)
    dev = parts[0].device
    codes = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
    scales = torch.zeros(nvfp4_scale_bytes(N, K), dtype=torch.uint8, device=dev)
    gs = torch.empty(len(parts), dtype=torch.float32, device=dev)
    row = 0
    for i, p in enumerate(parts):
        if len(parts) > 1 and i < len(parts) - 1 and p.shape[0] % 128:
            raise ValueError("fused weight parts must be multiples of 128 rows")
        nvfp4_compute_global(p, gs[i:i + 1], stream)
        sb = nvfp4_scale_bytes(p.shape[0], K)
        off = (row // 128) * 128 * ((K // 16 + 3) // 4 * 4)
        nvfp4_quantize_act(p, gs[i:i + 1], codes[row:row + p.shape[0]], scales[off:off + sb], stream)
        row += p.shape[0]
    g = nvfp4_reduce_max(gs, stream=stream) if len(parts) > 1 else gs[0:1].clone()
    return NVFP4Weight(codes, scales, g, [gs[i:i + 1] for i in range(len(parts))], N, K)


def fused_global_warning(w: NVFP4Weight, ratio: float = 0.05) -> str | None:
    """The load-time warning of a fused weight whose per-part globals differ by
    more than 5%, or None."""
    gs = [float(g.item()) for g in w.part_g]
    if len(gs) > 1 and (max(gs) - min(gs)) > ratio * max(gs):
        return f"fused NVFP4 weight: per-part globals differ by more than {ratio:.0%}: {gs}"
    return None


@dataclasses.dataclass
class MoEWeights:
    """NVFP4 expert banks of one MoE layer and their per-expert globals."""
    w13_codes: torch.Tensor
    w13_sf: torch.Tensor
    g13: torch.Tensor  # [E]
    w2_codes: torch.Tensor
    w2_sf: torch.Tensor
    g2: torch.Tensor   # [E]
    E: int
    H: int
    I: int


def quantize_moe_weights(w13_of, w2_of, E: int, H: int, I: int, device, stream=None) -> MoEWeights:
    """Quantise E experts; ``w13_of(e)`` / ``w2_of(e)`` return bf16 [2I, H] / [H, I]
    on the device.  One global per expert and tensor."""
    sb13 = nvfp4_scale_bytes(2 * I, H)
    sb2 = nvfp4_scale_bytes(H, I)
    w13c = torch.empty(E * 2 * I, H // 2, dtype=torch.uint8, device=device)
    w13s = torch.empty(E * sb13, dtype=torch.uint8, device=device)
    w2c = torch.empty(E * H, I // 2, dtype=torch.uint8, device=device)
    w2s = torch.empty(E * sb2, dtype=torch.uint8, device=device)
    g13 = torch.empty(E, dtype=torch.float32, device=device)
    g2 = torch.empty(E, dtype=torch.float32, device=device)
    for e in range(E):
        a = w13_of(e)
        nvfp4_compute_global(a, g13[e:e + 1], stream)
        nvfp4_quantize_act(a, g13[e:e + 1], w13c[e * 2 * I:(e + 1) * 2 * I],
                           w13s[e * sb13:(e + 1) * sb13], stream)
        b = w2_of(e)
        nvfp4_compute_global(b, g2[e:e + 1], stream)
        nvfp4_quantize_act(b, g2[e:e + 1], w2c[e * H:(e + 1) * H], w2s[e * sb2:(e + 1) * sb2], stream)
    return MoEWeights(w13c, w13s, g13, w2c, w2s, g2, E, H, I)
