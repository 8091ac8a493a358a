"""CPU oracle for the NVFP4 path: build and Python wrappers.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
CUDA library never imports, links or runs it, and it shares no code with it.

The arithmetic lives in ``nvfp4_oracle.c`` (plain C, IEEE fp32, built with
``-ffp-contract=off``).  This module compiles it with gcc into
``oracle/_build/libnvfp4_oracle.so`` and wraps it with ctypes.  Inputs and
outputs are CPU ``torch`` tensors (bf16 is passed as its raw 16-bit pattern).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libnvfp4_oracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float

_SIGS = {
    "nvo_set_threads": (None, [ctypes.c_int]),
    "nvo_get_threads": (ctypes.c_int, []),
    "nvo_bf16_to_f32": (_F, [ctypes.c_uint16]),
    "nvo_f32_to_bf16": (ctypes.c_uint16, [_F]),
    "nvo_e4m3_to_f32": (_F, [ctypes.c_uint8]),
    "nvo_f32_to_e4m3_satfinite": (ctypes.c_uint8, [_F]),
    "nvo_e2m1_to_f32": (_F, [ctypes.c_uint8]),
    "nvo_f32_to_e2m1_satfinite": (ctypes.c_uint8, [_F]),
    "nvo_scale_cols_padded": (_I64, [_I64]),
    "nvo_scale_bytes": (ctypes.c_size_t, [_I64, _I64]),
    "nvo_scale_offset": (_I64, [_I64, _I64, _I64]),
    "nvo_amax_bf16": (_F, [_P, _I64, _I64, _I64]),
    "nvo_global_from_amax": (_F, [_F]),
    "nvo_global_bf16": (_F, [_P, _I64, _I64, _I64]),
    "nvo_quantize_bf16": (None, [_P, _I64, _I64, _I64, _F, _P, _P]),
    "nvo_quantize_f32": (None, [_P, _I64, _I64, _I64, _F, _P, _P]),
    "nvo_dequant": (None, [_P, _P, _I64, _I64, _P]),
    "nvo_linear_w4a4": (None, [_P, _P, _I64, _P, _P, _I64, _I64, _F, _P, _I64]),
    "nvo_linear_w4a16": (None, [_P, _I64, _I64, _P, _P, _I64, _I64, _F, _P, _I64]),
    "nvo_moe_align": (_I64, [_P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _I64]),
    "nvo_moe_w4a4": (None, [_P, _I64, _I64, _I64, _I64, _I64, _P, _P, _F, _P, _P, _P,
                             _F, _P, _P, _P, _P, _P, _P]),
    "nvo_moe_h_amax": (None, [_P, _I64, _I64, _I64, _I64, _F, _P, _P, _P, _P]),
    "nvo_moe_down": (None, [_P, _P, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P]),
    "nvo_moe_w4a16": (None, [_P, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P,
                              _P, _P]),
}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FMA contraction)."""
    with _lock:
        if not force and os.path.exists(_LIB_PATH) and \
                os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
            return _LIB_PATH
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(t: torch.Tensor):
    assert t.device.type == "cpu" and t.is_contiguous()
    return ctypes.c_void_p(t.data_ptr())


def _u16(t: torch.Tensor) -> torch.Tensor:
    """bf16 tensor -> contiguous CPU int16 view of its bit patterns."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16)


def set_threads(n: int) -> None:
    lib().nvo_set_threads(int(n))


def threads() -> int:
    return int(lib().nvo_get_threads())


# --- scalar rules -----------------------------------------------------------

def e4m3_to_f32(b: int) -> float:
    return float(lib().nvo_e4m3_to_f32(b))


def f32_to_e4m3(v: float) -> int:
    return int(lib().nvo_f32_to_e4m3_satfinite(v))


def e2m1_to_f32(c: int) -> float:
    return float(lib().nvo_e2m1_to_f32(c))


def f32_to_e2m1(v: float) -> int:
    return int(lib().nvo_f32_to_e2m1_satfinite(v))


def f32_to_bf16_bits(v: float) -> int:
    return int(lib().nvo_f32_to_bf16(v))


def scale_bytes(rows: int, k: int) -> int:
    return int(lib().nvo_scale_bytes(rows, k))


def scale_offset(r: int, c: int, C: int) -> int:
    return int(lib().nvo_scale_offset(r, c, C))


# --- tensor operations ------------------------------------------------------

def amax(x: torch.Tensor) -> float:
    u = _u16(x)
    return float(lib().nvo_amax_bf16(_ptr(u), u.shape[0], u.shape[1], u.shape[1]))


def global_scale(x: torch.Tensor) -> float:
    """g = 2688 / amax(x) in fp32 (1.0 for an all-zero tensor)."""
    u = _u16(x)
    return float(lib().nvo_global_bf16(_ptr(u), u.shape[0], u.shape[1], u.shape[1]))


def global_from_amax(a: float) -> float:
    return float(lib().nvo_global_from_amax(a))


def quantize(x: torch.Tensor, g: float):
    """bf16 or fp32 [M, K] -> (uint8 codes [M, K/2], uint8 scales [sw(M, K/16)])."""
    M, K = x.shape
    codes = torch.zeros(M, K // 2, dtype=torch.uint8)
    scales = torch.zeros(scale_bytes(M, K), dtype=torch.uint8)
    if x.dtype == torch.bfloat16:
        u = _u16(x)
        lib().nvo_quantize_bf16(_ptr(u), M, K, K, g, _ptr(codes), _ptr(scales))
    else:
        f = x.detach().cpu().to(torch.float32).contiguous()
        lib().nvo_quantize_f32(_ptr(f), M, K, K, g, _ptr(codes), _ptr(scales))
    return codes, scales


def dequant(codes: torch.Tensor, scales: torch.Tensor, R: int, K: int) -> torch.Tensor:
    """codes/scales -> fp32 [R, K] = e2m1 * S (no global)."""
    out = torch.empty(R, K, dtype=torch.float32)
    c = codes.contiguous()
    s = scales.contiguous()
    lib().nvo_dequant(_ptr(c), _ptr(s), R, K, _ptr(out))
    return out


def _bf16_out(shape) -> torch.Tensor:
    return torch.empty(shape, dtype=torch.int16)


def linear_w4a4(a_codes, a_sf, M, w_codes, w_sf, N, K, alpha: float) -> torch.Tensor:
    out = _bf16_out((M, N))
    lib().nvo_linear_w4a4(_ptr(a_codes.contiguous()), _ptr(a_sf.contiguous()), M,
                          _ptr(w_codes.contiguous()), _ptr(w_sf.contiguous()), N, K,
                          alpha, _ptr(out), N)
    return out.view(torch.bfloat16)


def linear_w4a16(x: torch.Tensor, w_codes, w_sf, N, K, alpha: float) -> torch.Tensor:
    T = x.shape[0]
    u = _u16(x)
    out = _bf16_out((T, N))
    lib().nvo_linear_w4a16(_ptr(u), T, u.shape[1], _ptr(w_codes.contiguous()),
                           _ptr(w_sf.contiguous()), N, K, alpha, _ptr(out), N)
    return out.view(torch.bfloat16)


def moe_align(ids: torch.Tensor, E: int, BM: int):
    """Stable expert alignment -> dict(counts, offsets, row_map, tile_expert, P)."""
    ids = ids.to(torch.int32).contiguous()
    T, topk = ids.shape
    cap = T * topk + E * (BM - 1) + BM
    counts = torch.zeros(E, dtype=torch.int32)
    offsets = torch.zeros(E + 1, dtype=torch.int32)
    row_map = torch.full((cap,), -1, dtype=torch.int32)
    tile_expert = torch.full((cap // BM + 1,), -1, dtype=torch.int32)
    P = int(lib().nvo_moe_align(_ptr(ids), T, topk, E, BM, _ptr(counts), _ptr(offsets),
                                _ptr(row_map), _ptr(tile_expert), cap))
    assert P >= 0
    return dict(counts=counts, offsets=offsets, row_map=row_map[:P].clone(),
                tile_expert=tile_expert[:P // BM].clone(), P=P)


def moe_w4a4(x, topk_ids, topk_w, g_a1, w13_codes, w13_sf, alpha13, g_a2, w2_codes, w2_sf,
             alpha2, E, H, I, want_h: bool = False):
    """MoE layer: bf16 [T, H] -> bf16 [T, H]; optionally the NVFP4 codes and
    scales of the intermediate h for row t * topk + slot."""
    T, topk = topk_ids.shape
    u = _u16(x)
    ids = topk_ids.to(torch.int32).contiguous()
    w = topk_w.to(torch.float32).contiguous()
    a13 = torch.as_tensor(alpha13, dtype=torch.float32).contiguous()
    a2 = torch.as_tensor(alpha2, dtype=torch.float32).contiguous()
    out = _bf16_out((T, H))
    R = T * topk
    hc = torch.zeros(R, I // 2, dtype=torch.uint8) if want_h else None
    hs = torch.zeros(scale_bytes(R, I), dtype=torch.uint8) if want_h else None
    lib().nvo_moe_w4a4(_ptr(u), T, H, I, E, topk, _ptr(ids), _ptr(w), g_a1,
                       _ptr(w13_codes.contiguous()), _ptr(w13_sf.contiguous()), _ptr(a13),
                       g_a2, _ptr(w2_codes.contiguous()), _ptr(w2_sf.contiguous()), _ptr(a2),
                       _ptr(out), _ptr(hc) if want_h else None, _ptr(hs) if want_h else None)
    out = out.view(torch.bfloat16)
    return (out, hc, hs) if want_h else out


def moe_down(h_codes, h_sf, topk_ids, topk_w, w2_codes, w2_sf, alpha2, E, H, I) -> torch.Tensor:
    """The MoE down projection on a given NVFP4 intermediate: h_codes
    [T * topk, I/2] and h_sf (swizzled over T * topk rows) hold route
    t * topk + slot; returns bf16 [T, H] (the layer's last two steps)."""
    T, topk = topk_ids.shape
    ids = topk_ids.to(torch.int32).contiguous()
    w = topk_w.to(torch.float32).contiguous()
    a2 = torch.as_tensor(alpha2, dtype=torch.float32).contiguous()
    assert h_codes.shape == (T * topk, I // 2) and h_sf.numel() >= scale_bytes(T * topk, I)
    out = _bf16_out((T, H))
    lib().nvo_moe_down(_ptr(h_codes.contiguous()), _ptr(h_sf.contiguous()), T, H, I, E, topk, _ptr(ids),
                       _ptr(w), _ptr(w2_codes.contiguous()), _ptr(w2_sf.contiguous()), _ptr(a2), _ptr(out))
    return out.view(torch.bfloat16)


def moe_w4a16(x, topk_ids, topk_w, w13_codes, w13_sf, alpha13, w2_codes, w2_sf, alpha2, E, H, I,
              want_h: bool = False):
    """W4A16 MoE layer (bf16 activations throughout): bf16 [T, H] -> bf16 [T, H];
    optionally the bf16 intermediate h [T * topk, I] (row t * topk + slot)."""
    T, topk = topk_ids.shape
    u = _u16(x)
    ids = topk_ids.to(torch.int32).contiguous()
    w = topk_w.to(torch.float32).contiguous()
    a13 = torch.as_tensor(alpha13, dtype=torch.float32).contiguous()
    a2 = torch.as_tensor(alpha2, dtype=torch.float32).contiguous()
    out = _bf16_out((T, H))
    h = _bf16_out((T * topk, I)) if want_h else None
    lib().nvo_moe_w4a16(_ptr(u), T, H, I, E, topk, _ptr(ids), _ptr(w), _ptr(w13_codes.contiguous()),
                        _ptr(w13_sf.contiguous()), _ptr(a13), _ptr(w2_codes.contiguous()),
                        _ptr(w2_sf.contiguous()), _ptr(a2), _ptr(out), _ptr(h) if want_h else None)
    out = out.view(torch.bfloat16)
    return (out, h.view(torch.bfloat16)) if want_h else out


def moe_h_amax(x_calib, g_a1, w13_codes, w13_sf, alpha13, E, H, I) -> torch.Tensor:
    """Per-expert amax of h over the calibration rows (every row through every expert)."""
    u = _u16(x_calib)
    a13 = torch.as_tensor(alpha13, dtype=torch.float32).contiguous()
    out = torch.zeros(E, dtype=torch.float32)
    lib().nvo_moe_h_amax(_ptr(u), u.shape[0], H, I, E, g_a1, _ptr(w13_codes.contiguous()),
                         _ptr(w13_sf.contiguous()), _ptr(a13), _ptr(out))
    return out


# --- whole-workload helpers (oracle side of a parity case) -----------------

def f32(v) -> float:
    """Round a Python float to fp32."""
    return float(np.float32(v))


def alpha_w4a4(g_a: float, g_w: float) -> float:
    """alpha = 1 / (g_a * g_w), both operations in fp32."""
    return float(np.float32(1.0) / (np.float32(g_a) * np.float32(g_w)))


def alpha_w4a16(g_w: float) -> float:
    return float(np.float32(1.0) / np.float32(g_w))


def quantize_weight_parts(parts):
    """Fused weight: each part quantised with its own global; the fused tensor
    keeps the block scales and takes the largest per-part global ([linear],
    "Changes").  Returns (codes, scales, g_fused, per-part globals)."""
    gs = [global_scale(p) for p in parts]
    cs, ss = [], []
    for p, g in zip(parts, gs):
        c, s = quantize(p, g)
        cs.append(c)
        ss.append(s)
    rows = [int(p.shape[0]) for p in parts]
    K = int(parts[0].shape[1])
    if len(parts) == 1:
        return cs[0], ss[0], gs[0], gs
    assert all(r % 128 == 0 for r in rows[:-1]), "fused parts must be 128-row aligned"
    codes = torch.cat(cs, 0)
    scales = torch.zeros(scale_bytes(sum(rows), K), dtype=torch.uint8)
    off = 0
    for s in ss:
        scales[off:off + s.numel()] = s
        off += s.numel()
    return codes, scales, max(gs), gs
