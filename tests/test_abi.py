"""The C-ABI library loads on a machine without a GPU, exports every function
include/nvfp4.h declares, and refuses bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

import nvfp4_block_scaled_act_gb300 as nv
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_scaled_act_gb300 import build
    build.build()
    return nv.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 14
    raw = ctypes.CDLL(nv.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in nvfp4.h but not exported"
        assert n in nv.SIGNATURES, f"{n} has no Python binding"


def test_status_strings(lib):
    for s in range(9):
        assert lib.nvfp4_status_string(s)
    assert lib.nvfp4_version() >= 100


@pytest.mark.parametrize("rows,k", [(1, 16), (8, 512), (130, 64), (7168, 5120), (300, 112)])
def test_scale_bytes_matches_oracle(lib, rows, k):
    assert lib.nvfp4_scale_bytes(rows, k) == oracle.scale_bytes(rows, k)


P = ctypes.c_void_p(256)  # an aligned, never dereferenced address


def test_w4a4_argument_errors(lib):
    f = lib.nvfp4_linear_w4a4
    assert f(P, P, 8, P, P, 12, 512, P, P, 12, None) == 2        # N % 8 (N = 12 refused)
    assert f(P, P, 8, P, P, 16, 96, P, P, 16, None) == 2         # K % 64
    assert f(P, P, 8, P, P, 16, 512, P, P, 8, None) == 1         # ldo < N
    assert f(P, P, -1, P, P, 16, 512, P, P, 16, None) == 1       # negative M
    assert f(P, P, 0, P, P, 16, 512, P, P, 16, None) == 0        # M = 0: nothing to do
    assert f(ctypes.c_void_p(257), P, 8, P, P, 16, 512, P, P, 16, None) == 3
    assert f(None, P, 8, P, P, 16, 512, P, P, 16, None) == 1


def test_quant_and_w4a16_argument_errors(lib):
    q = lib.nvfp4_quantize_act
    assert q(P, 4, 24, 24, P, P, P, None) == 2                    # K % 16
    assert q(P, 4, 32, 16, P, P, P, None) == 1                    # ldx < K
    assert q(P, 4, 32, 36, P, P, P, None) == 3                    # ldx % 8
    assert q(P, 0, 32, 32, P, P, P, None) == 0
    g = lib.nvfp4_linear_w4a16
    assert g(P, 17, 512, P, P, 64, 512, P, P, 64, None, 0, None) == 2   # T > 16
    assert g(P, 4, 512, P, P, 64, 192, P, P, 64, None, 0, None) == 2    # K % 128
    assert g(P, 0, 512, P, P, 64, 512, P, P, 64, None, 0, None) == 0
    na = lib.nvfp4_linear_w4a16_noalloc
    assert na(None, 0, 512, None, None, 64, 512, None, None, 64, None) == 0   # T = 0
    assert na(P, 17, 512, P, P, 64, 512, P, P, 64, None) == 2                # T > 16


def test_helper_and_layer_argument_errors(lib):
    """The documented status of every argument error that is refused before a
    device is looked for (1 invalid argument, 2 unsupported shape, 3
    misaligned, 4 workspace too small; 0 for nothing to do)."""
    Q = ctypes.c_void_p(264)        # 8-byte aligned only
    big, small = ctypes.c_size_t(1 << 40), ctypes.c_size_t(16)
    g = lib.nvfp4_compute_global
    assert g(None, 4, 64, 64, P, None) == 1                       # null x
    assert g(P, 4, 64, 32, P, None) == 1                          # ldx < cols
    assert g(Q, 4, 64, 64, P, None) == 3                          # x not 16-byte aligned
    assert g(P, 4, 64, 68, P, None) == 3                          # ldx % 8
    a = lib.nvfp4_make_alpha
    assert a(P, None, 4, P, None) == 1 and a(P, P, -1, P, None) == 1
    assert a(None, P, 0, P, None) == 0                            # n = 0: nothing to do
    r = lib.nvfp4_reduce_max
    assert r(P, 0, P, None) == 1 and r(None, 4, P, None) == 1
    w = lib.nvfp4_linear_w4a16
    assert w(P, 4, 256, P, P, 64, 512, P, P, 64, None, 0, None) == 1     # ldx < K
    assert w(P, 4, 512, P, P, 64, 512, P, P, 32, None, 0, None) == 1     # ldo < N
    assert w(P, 4, 512, P, P, 60, 512, P, P, 64, None, 0, None) == 2     # N % 8
    assert w(Q, 4, 512, P, P, 64, 512, P, P, 64, None, 0, None) == 3     # x misaligned
    assert w(P, 4, 512, P, P, 64, 512, P, P, 65, None, 0, None) == 3     # odd ldo
    assert w(P, 4, 512, P, P, 64, 512, P, ctypes.c_void_p(258), 64, None, 0, None) == 3   # out not 4-byte aligned
    assert w(P, 4, 512, None, P, 64, 512, P, P, 64, None, 0, None) == 1  # null codes
    l4 = lib.nvfp4_linear_w4a4
    assert l4(P, Q, 8, P, P, 16, 512, P, P, 16, None) == 3              # scales misaligned
    m = lib.nvfp4_moe_w4a4
    args = [P, 16, 2048, 768, 128, 8] + [P] * 12 + [big, None]
    import torch
    if not torch.cuda.is_available():
        assert m(*args) == 8                                     # valid arguments, no device
    args[4] = 1025
    assert m(*args) == 2                                         # E > 1024
    args[4] = 128
    args[6] = ctypes.c_void_p(258)
    assert m(*args) == 3                                         # ids not 4-byte aligned
    args[6] = P
    args[-2] = small
    assert m(*args) == 4                                         # workspace too small
    args[-2] = big
    args[16] = None
    assert m(*args) == 1                                         # null out
    c = lib.nvfp4_moe_calibrate
    cargs = [P, 16, 2048, 768, 128, P, P, P, P, None, P, P, big, None]
    assert c(*cargs[:1], 0, *cargs[2:]) == 1                     # no calibration rows
    assert c(*cargs[:4], 1025, *cargs[5:]) == 2                  # E > 1024
    assert c(Q, *cargs[1:]) == 3                                 # x misaligned
    assert c(*cargs[:12], small, None) == 4                      # workspace too small
    assert c(*cargs[:10], None, *cargs[11:]) == 1                # null g_a2 (amax is optional)
    assert lib.nvfp4_device_status(None, None) == 1


def test_w4a16_workspace_only_for_long_k_at_large_t(lib):
    """The decode sums its k-split partials on chip unless the activations of
    one k-split leave too little shared memory for the weight ring; the
    boundary (host planning, 152 SMs when no device is present) does not
    depend on N."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("the boundary is stated for 152 SMs")
    q = lib.nvfp4_linear_w4a16_workspace
    for N in (1024, 8704):
        assert q(1, N, 131072) == 0 and q(4, N, 131072) == 0
        assert q(8, N, 91136) == 0 and q(8, N, 91264) > 0
        assert q(16, N, 44032) == 0 and q(16, N, 44160) > 0
        assert q(16, N, 5120) == 0 and q(16, N, 4352) == 0     # the decode workloads


def test_no_device_is_reported_without_a_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.nvfp4_linear_w4a4(P, P, 8, P, P, 16, 512, P, P, 16, None) == 8


def test_moe_workspace_layout(lib):
    T, H, I, E, topk = 4096, 2048, 768, 128, 8
    lay = nv.nvfp4_moe_workspace_layout(T, H, I, E, topk)
    assert lay.row_block == 128   # 256 routes per expert on average: 128-row segments
    assert lay.p_max == (T * topk + E * 127 + 127) // 128 * 128
    big = nv.nvfp4_moe_workspace_layout(4 * T, H, I, E, topk)   # 1024 routes per expert: CTA pairs
    assert big.row_block == 256 and big.p_max == (4 * T * topk + E * 255 + 255) // 256 * 256
    assert nv.nvfp4_moe_workspace_layout(4 * T, 1920, I, E, topk).row_block == 128   # H % 256 != 0
    assert lay.total == lib.nvfp4_moe_workspace(T, H, I, E, topk)
    offs = [lay.counts, lay.offsets, lay.n_tiles, lay.row_map, lay.tile_expert, lay.pos, lay.a1_codes,
            lay.a1_sf, lay.h_codes, lay.h_sf, lay.y, lay.hist]
    assert all(o % 256 == 0 for o in offs)
    assert lay.y + 4 * T * H <= lay.total
    assert lay.h_codes + lay.p_max * I // 2 <= lay.h_sf
    f = lib.nvfp4_moe_w4a4
    # T = 0: nothing to do, before any pointer is looked at or a device touched
    assert f(*([None, 0, 2048, 768, 128, 8] + [None] * 12 + [ctypes.c_size_t(0), None])) == 0
    args = [P, 16, 2048, 768, 128, 33] + [P] * 12 + [ctypes.c_size_t(1 << 40), None]
    assert f(*args) == 2   # topk > 32
    args[5] = 8
    args[2] = 2000
    assert f(*args) == 2   # H % 128


@pytest.mark.parametrize("T,H,I,E,topk", [
    (1, 128, 128, 1, 1), (16, 2048, 768, 128, 8), (4096, 2048, 768, 128, 8), (16384, 2048, 768, 128, 8),
    (32768, 7168, 2048, 256, 8), (175001, 256, 128, 3, 3), (3001, 128, 256, 1024, 3), (8, 7168, 2048, 256, 256)])
def test_moe_layout_regions_are_aligned_disjoint_and_large_enough(lib, T, H, I, E, topk):
    """Every region of the workspace layout starts on a 256-byte boundary,
    holds at least what the header says it holds, overlaps no other region
    and ends inside the total the workspace query reports (the last case is
    the calibration layout, every row routed to every expert)."""
    lay = nv.nvfp4_moe_workspace_layout(T, H, I, E, topk)
    R = T * topk
    bm = 256 if R >= 1024 * E and H % 256 == 0 else 128
    assert lay.row_block == bm
    P = lay.p_max
    assert P == -(-(R + E * (bm - 1)) // bm) * bm and P % 128 == 0
    need = {"counts": 4 * E, "offsets": 4 * (E + 1), "n_tiles": 4, "row_map": 4 * P, "tile_expert": 4 * (P // 128),
            "pos": 4 * R, "hist": 4 * E, "a1_codes": P * H // 2, "a1_sf": oracle.scale_bytes(P, H),
            "h_codes": P * I // 2, "h_sf": oracle.scale_bytes(P, I), "y": 4 * T * H}
    regions = sorted((getattr(lay, n), n) for n in need)
    for (off, n), nxt in zip(regions, regions[1:] + [(lay.total, "total")]):
        assert off % 256 == 0, n
        assert off + need[n] <= nxt[0], f"{n} overlaps {nxt[1]}"
    assert lay.total == lib.nvfp4_moe_workspace(T, H, I, E, topk)


def test_moe_w4a16_argument_errors(lib):
    ws = lib.nvfp4_moe_w4a16_workspace
    R = 4 * 8
    assert ws(4, 2048, 768, 128, 8) == R * 768 * 2 + R * 2048 * 4   # bf16 h, fp32 per-route down rows
    assert ws(65, 2048, 768, 128, 8) == 0      # T > 64: the W4A4 path's regime
    assert ws(4, 2048, 768, 128, 9) == 0       # topk > 8
    assert ws(4, 2000, 768, 128, 8) == 0       # H % 128
    assert ws(4, 2048, 768, 1025, 8) == 0      # E > 1024
    f = lib.nvfp4_moe_w4a16
    big = ctypes.c_size_t(1 << 40)
    args = [P, 4, 2048, 768, 128, 8] + [P] * 10 + [big, None]
    args[2] = 2000
    assert f(*args) == 2                       # H % 128
    args[2] = 2048
    args[1] = 0
    assert f(*args) == 0                       # T = 0: nothing to do
    args[1] = 4
    args[6] = None
    assert f(*args) == 1                       # null ids
    args[6] = P
    args[8] = ctypes.c_void_p(260)
    assert f(*args) == 3                       # misaligned W13 codes
    args[8] = P
    args[-2] = ctypes.c_size_t(16)
    assert f(*args) == 4                       # workspace too small
    import torch
    if not torch.cuda.is_available():
        args[-2] = big
        assert f(*args) == 8                   # valid arguments, no device


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        nv.load_library.__wrapped__ if hasattr(nv.load_library, "__wrapped__") else None
        saved = nv._lib
        nv._lib = None
        try:
            nv.load_library(str(tmp_path / "libnvfp4.so"))
        finally:
            nv._lib = saved
