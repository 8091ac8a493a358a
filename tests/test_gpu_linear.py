"""GPU parity of the W4A4 block-scaled GEMM (tcgen05) and the W4A16 decode GEMM
against the oracle: both sides quantise the same bf16 inputs on their own (the
codes are checked bit-exact first), then the outputs must meet rel-L2 <= 1e-3
and max |err| <= 2 bf16 ulp of the row's largest output."""
import numpy as np
import pytest
import torch

import oracle
import synthdata
from parity import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def nv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_block_scaled_act_gb300 import build
    build.build()
    import nvfp4_block_scaled_act_gb300 as m
    m.load_library()
    return m


class Linear:
    """Both sides of one linear: GPU tensors and oracle tensors."""

    def __init__(self, nv, case: synthdata.LinearCase, quant_act: bool = True):
        self.N, self.K, self.M = case.N, case.K, case.x.shape[0]
        self.W = nv.quantize_weight([p.to(DEV) for p in case.w_parts])
        self.wc, self.ws, self.g_w, _ = oracle.quantize_weight_parts(case.w_parts)
        assert torch.equal(self.W.codes.cpu(), self.wc) and torch.equal(self.W.scales.cpu(), self.ws)
        self.x = case.x
        self.x_dev = case.x.to(DEV)
        if quant_act:
            self.g_a_dev = nv.nvfp4_compute_global(case.x_calib.to(DEV))
            self.g_a = oracle.global_scale(case.x_calib)
            self.ac_dev, self.as_dev = nv.nvfp4_quantize_act(self.x_dev, self.g_a_dev)
            self.ac, self.as_ = oracle.quantize(case.x, self.g_a)
            assert torch.equal(self.ac_dev.cpu(), self.ac) and torch.equal(self.as_dev.cpu(), self.as_)
            self.alpha_dev = nv.nvfp4_make_alpha(self.g_a_dev, self.W.g)
            self.alpha = oracle.alpha_w4a4(self.g_a, self.g_w)
            assert np.float32(self.alpha_dev.item()) == np.float32(self.alpha)
        self.alpha16_dev = nv.nvfp4_make_alpha(None, self.W.g)
        self.alpha16 = oracle.alpha_w4a16(self.g_w)

    def w4a4(self, nv, out=None):
        return nv.nvfp4_linear_w4a4(self.ac_dev, self.as_dev, self.W.codes, self.W.scales, self.alpha_dev,
                                    self.N, self.K, out=out)

    def w4a4_oracle(self, rows=None):
        if rows is None:
            return oracle.linear_w4a4(self.ac, self.as_, self.M, self.wc, self.ws, self.N, self.K, self.alpha)
        # rows are independent: quantise the sampled rows again (bit-identical) and multiply
        xs = self.x[rows].contiguous()
        ac, as_ = oracle.quantize(xs, self.g_a)
        return oracle.linear_w4a4(ac, as_, len(rows), self.wc, self.ws, self.N, self.K, self.alpha)


# ---------------------------------------------------------------------------
# W4A4
# ---------------------------------------------------------------------------

def test_w4a4_tiny_linear(nv):
    L = Linear(nv, synthdata.tiny_linear(seed=0))
    out = L.w4a4(nv)
    check_close(out, L.w4a4_oracle(), "tiny W4A4 8x256x512")


@pytest.mark.parametrize("M,N,K", [
    (1, 8, 64), (7, 136, 192), (130, 264, 320), (257, 128, 256), (300, 392, 576),
    (129, 1024, 1024), (64, 256, 5120), (255, 7168, 512),
])
def test_w4a4_ragged_shapes(nv, M, N, K):
    L = Linear(nv, synthdata.linear_case(M, N, K, seed=M * 7 + N))
    check_close(L.w4a4(nv), L.w4a4_oracle(), f"W4A4 {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 8, 17, 48, 100, 128, 129, 256])
def test_w4a4_small_m_fused_qkv(nv, M):
    """Small batches on the fused qkv weight (N = 7168, K = 5120): up to 128 rows
    run on 128 x 128 single-CTA tiles, above that on CTA pairs; every row is
    compared with the oracle, and a repeated call gives the same bits."""
    L = Linear(nv, synthdata.prefill_case(M, seed=M))
    out = L.w4a4(nv)
    check_close(out, L.w4a4_oracle(), f"small-M W4A4 M={M}")
    assert torch.equal(L.w4a4(nv), out), f"small-M W4A4 M={M} is not repeatable"
    assert nv.nvfp4_device_status() == 0


def test_w4a4_row_strided_output_and_repeatability(nv):
    L = Linear(nv, synthdata.linear_case(200, 256, 512, seed=3))
    big = torch.full((200, 264), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = L.w4a4(nv, out=big[:, :256])
    torch.cuda.synchronize()
    assert torch.isnan(big[:, 256:].float()).all(), "wrote past N"
    check_close(out, L.w4a4_oracle(), "row-strided out")
    again = L.w4a4(nv)
    assert torch.equal(again, out.contiguous()), "W4A4 is not repeatable"
    assert nv.nvfp4_device_status() == 0


@pytest.mark.parametrize("M", synthdata.PREFILL_M)
def test_w4a4_prefill_fused_qkv(nv, M):
    """The fused qkv-style prefill (N = 5120 + 1024 + 1024, K = 5120) at full
    size; the oracle computes a sample of rows (first, last, spread)."""
    L = Linear(nv, synthdata.prefill_case(M, seed=0))
    out = L.w4a4(nv).cpu()
    rows = sorted(set([0, 1, 127, 128, M // 2, M - 129, M - 1] + list(range(5, M, max(1, M // 9)))))
    check_close(out[rows], L.w4a4_oracle(rows), f"prefill M={M}")
    warn = nv.fused_global_warning(L.W)
    assert warn is None or "5%" in warn


def test_w4a4_zero_rows_stay_zero(nv):
    case = synthdata.linear_case(130, 256, 512, seed=4)
    case.x[5] = 0
    case.x[129] = 0
    L = Linear(nv, case)
    out = L.w4a4(nv).cpu()
    assert torch.all(out[5] == 0) and torch.all(out[129] == 0)
    check_close(out, L.w4a4_oracle(), "zero rows")


# ---------------------------------------------------------------------------
# W4A16
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,K", synthdata.DECODE_SHAPES)
@pytest.mark.parametrize("T", synthdata.DECODE_TOKENS)
def test_w4a16_decode_shapes(nv, T, N, K):
    L = Linear(nv, synthdata.decode_case(T, N, K, seed=T), quant_act=False)
    out = nv.nvfp4_linear_w4a16(L.x_dev, L.W.codes, L.W.scales, L.alpha16_dev, N, K)
    ref = oracle.linear_w4a16(L.x, L.wc, L.ws, N, K, L.alpha16)
    check_close(out, ref, f"W4A16 T={T} {N}x{K}")


@pytest.mark.parametrize("T,N,K", [(1, 8, 128), (3, 136, 384), (5, 1032, 256), (7, 264, 640),
                                   (9, 520, 128), (15, 2056, 1152), (16, 16, 4096), (2, 3584, 5120),
                                   (1, 256, 32768), (16, 128, 16384), (16, 128, 44032),
                                   (16, 256, 45056), (8, 136, 91264)])
def test_w4a16_ragged(nv, T, N, K):
    """Ragged N (partial 128-row blocks), T across both token layouts, and long
    K: (1, 256, 32768) and (16, 128, 16384) stream more 128-k blocks than the
    shared-memory ring holds; (16, 128, 44032) is the longest K at T = 16 whose
    k-split activations still fit beside the ring, so its partials are summed
    on chip; (16, 256, 45056) and (8, 136, 91264) are past that boundary and run
    the split-K kernel with its workspace."""
    need = nv.nvfp4_linear_w4a16_workspace(T, N, K)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert (need > 0) == (K > 44032 if T > 8 else K > 91136), (T, N, K, need)
    L = Linear(nv, synthdata.decode_case(T, N, K, seed=N + T), quant_act=False)
    out = nv.nvfp4_linear_w4a16(L.x_dev, L.W.codes, L.W.scales, L.alpha16_dev, N, K)
    check_close(out, oracle.linear_w4a16(L.x, L.wc, L.ws, N, K, L.alpha16), f"W4A16 {T}x{N}x{K}")
    for _ in range(4):  # refilled ring slots never hand stale weights to the MMAs
        again = nv.nvfp4_linear_w4a16(L.x_dev, L.W.codes, L.W.scales, L.alpha16_dev, N, K)
        assert torch.equal(again, out), f"W4A16 {T}x{N}x{K} is not repeatable"


@pytest.mark.parametrize("T,N,K", [(1, 8704, 5120), (8, 1024, 2048), (16, 640, 4352)])
def test_w4a16_blocks_of_distant_magnitudes(nv, T, N, K):
    """Activations whose 128-k blocks differ in magnitude by up to 2^120, with
    all-zero blocks and blocks holding one nonzero value: the decode kernel
    rescales each (token, 128-k block) on its own, and the result must still
    meet the tolerance against the oracle."""
    case = synthdata.decode_case(T, N, K, seed=77 + T)
    g = torch.Generator().manual_seed(1234 + T)
    nb = K // 128
    exps = torch.randint(-60, 61, (T, nb), generator=g).double()
    scale = torch.pow(2.0, exps).repeat_interleave(128, dim=1)
    x = (case.x.double() * scale)
    zero = torch.rand(T, nb, generator=g) < 0.15
    x = x.view(T, nb, 128)
    x[zero] = 0.0
    lone = torch.rand(T, nb, generator=g) < 0.1
    x[lone, 1:] = 0.0
    case.x = x.view(T, K).to(torch.bfloat16)
    L = Linear(nv, case, quant_act=False)
    out = nv.nvfp4_linear_w4a16(L.x_dev, L.W.codes, L.W.scales, L.alpha16_dev, N, K)
    check_close(out, oracle.linear_w4a16(L.x, L.wc, L.ws, N, K, L.alpha16), f"W4A16 distant blocks {T}x{N}x{K}")


def test_w4a16_row_strided_and_deterministic(nv):
    T, N, K = 8, 1024, 2048
    L = Linear(nv, synthdata.decode_case(T, N, K, seed=9), quant_act=False)
    big = torch.zeros(T, K + 64, dtype=torch.bfloat16, device=DEV)
    big[:, :K] = L.x_dev
    a = nv.nvfp4_linear_w4a16(big[:, :K], L.W.codes, L.W.scales, L.alpha16_dev, N, K)
    b = nv.nvfp4_linear_w4a16(big[:, :K], L.W.codes, L.W.scales, L.alpha16_dev, N, K)
    assert torch.equal(a, b), "split-K reduce is not deterministic"
    check_close(a, oracle.linear_w4a16(L.x, L.wc, L.ws, N, K, L.alpha16), "row-strided W4A16")


def test_w4a16_refcheck_against_unquantised(nv):
    """The pages' check: rel_l2 < 0.15 and cos > 0.99 against the bf16 matmul
    with the unquantised weight."""
    case = synthdata.decode_case(16, 4096, 4096, seed=5)
    L = Linear(nv, case, quant_act=False)
    out = nv.nvfp4_linear_w4a16(L.x_dev, L.W.codes, L.W.scales, L.alpha16_dev, 4096, 4096).double().cpu()
    ref = (case.x.float() @ case.w_parts[0].float().T).double()
    rel = ((out - ref).norm() / ref.norm()).item()
    cos = torch.nn.functional.cosine_similarity(out.flatten(), ref.flatten(), dim=0).item()
    assert rel < 0.15 and cos > 0.99, (rel, cos)


def test_w4a16_refuses_more_than_16_tokens(nv):
    L = Linear(nv, synthdata.decode_case(17, 64, 128, seed=1), quant_act=False)
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_linear_w4a16(L.x_dev, L.W.codes, L.W.scales, L.alpha16_dev, 64, 128)


@pytest.mark.parametrize("M", [8, 300, 2048])
def test_w4a4_agrees_with_library_nvfp4_gemm(nv, M):
    """Cross-check against cuBLASLt's NVFP4 GEMM (torch._scaled_mm on e2m1 codes
    with E4M3 block scales in the 128x4 layout), when this torch has it: it
    reads the same codes and scale buffers, so agreement pins the nibble order
    and the scale layout against outside code.  The library rounds its fp32
    sum to bf16 before alpha is applied, so the tolerance allows one more
    bf16 rounding."""
    L = Linear(nv, synthdata.linear_case(M, [512, 256], 1024, seed=M))
    out = L.w4a4(nv).float()
    try:
        ref = torch._scaled_mm(L.ac_dev.view(torch.float4_e2m1fn_x2),
                               L.W.codes.view(torch.float4_e2m1fn_x2).t(),
                               L.as_dev.view(torch.float8_e4m3fn), L.W.scales.view(torch.float8_e4m3fn),
                               out_dtype=torch.bfloat16)
    except Exception as e:  # noqa: BLE001
        pytest.skip(f"no NVFP4 _scaled_mm in this torch: {type(e).__name__}")
    ref = ref.float() * L.alpha_dev.item()
    check_close(out, ref, f"vs library NVFP4 GEMM M={M}", ulps=3.0, rel_l2=5e-3)
