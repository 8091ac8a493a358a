"""The allocation-free decode entry point, nvfp4_linear_w4a16_noalloc.

It exists for callers that cannot allocate device memory when they run a
decode GEMM (a runtime that owns the whole GPU through its own pool, code
already inside CUDA stream capture, a plugin host that hands out only inputs
and outputs): it keeps its split-K partials in a 6 MiB array compiled into the
library instead of a workspace.  Here it is called through the C ABI, twice in
a row, and each result is compared element by element with the oracle within
the tolerance of the other GEMM tests (and, as a second check, with the
workspace entry point).  Shapes whose partials exceed the array are refused.
This file is collected last so that a stop at the first failure has already
run every other test; it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

import oracle
import synthdata
from parity import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_block_scaled_act_gb300 import build
    build.build()
    import nvfp4_block_scaled_act_gb300 as m
    m.load_library()
    return m


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_noalloc(lib, x, W, alpha, N, K, out):
    return lib.nvfp4_linear_w4a16_noalloc(_p(x), x.shape[0], x.stride(0), _p(W.codes), _p(W.scales), N, K,
                                          _p(alpha), _p(out), out.stride(0),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("T,N,K", [(16, 8704, 5120), (1, 5120, 4352), (5, 1032, 256), (16, 5120, 4352)])
def test_noalloc_matches_oracle(nv, T, N, K):
    case = synthdata.decode_case(T, N, K, seed=T + N)
    w = case.w_parts[0]
    W = nv.quantize_weight(w.to(DEV))
    wc, ws = oracle.quantize(w, oracle.global_scale(w))
    assert torch.equal(W.codes.cpu(), wc) and torch.equal(W.scales.cpu(), ws)
    alpha = nv.nvfp4_make_alpha(None, W.g)
    ref = oracle.linear_w4a16(case.x, wc, ws, N, K, oracle.alpha_w4a16(oracle.global_scale(w)))
    x = case.x.to(DEV)
    lib = nv.load_library()
    for _ in range(2):  # two calls in a row share the static array
        out = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        assert _call_noalloc(lib, x, W, alpha, N, K, out) == 0
        torch.cuda.synchronize()
        check_close(out, ref, f"no-alloc W4A16 {T}x{N}x{K} against the oracle")
        check_close(out, nv.nvfp4_linear_w4a16(x, W.codes, W.scales, alpha, N, K),
                    f"no-alloc W4A16 {T}x{N}x{K} against the workspace entry point")
    assert nv.nvfp4_device_status() == 0


def test_noalloc_refuses_shapes_beyond_its_array(nv):
    """2 * SMs - 1 blocks of 256 rows split K in two: 2 * 16 * N fp32 partials,
    about SMs * 64 KB, more than the 6 MiB array on any GPU with 100 or more
    SMs (the shape follows the SM count torch reports)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sms >= 100
    T, N, K = 16, (2 * sms - 1) * 256, 256
    assert 2 * T * N * 4 > 6 * 1024 * 1024
    x = torch.zeros(T, K, dtype=torch.bfloat16, device=DEV)
    codes = torch.zeros(N, K // 2, dtype=torch.uint8, device=DEV)
    scales = torch.zeros(nv.nvfp4_scale_bytes(N, K), dtype=torch.uint8, device=DEV)
    alpha = torch.ones(1, dtype=torch.float32, device=DEV)
    out = torch.empty(T, N, dtype=torch.bfloat16, device=DEV)
    lib = nv.load_library()
    st = lib.nvfp4_linear_w4a16_noalloc(_p(x), T, K, _p(codes), _p(scales), N, K, _p(alpha), _p(out), N,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 4  # NVFP4_ERR_WORKSPACE_TOO_SMALL
