"""GPU parity of the NVFP4 quantiser and the global: codes and scale bytes
bit-exact against the oracle, on the workloads' shapes, ragged and row-strided
inputs, and crafted inputs that put the e2m1 and E4M3 roundings on their ties."""
import numpy as np
import pytest
import torch

import oracle
import synthdata

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_block_scaled_act_gb300 import build
    build.build()
    import nvfp4_block_scaled_act_gb300 as nv
    nv.load_library()
    return nv


def gpu_quant(nv, x_cpu, g_value, ldx=None):
    """Quantise on the GPU with a given fp32 global; scale buffer pre-filled
    with 0xAB so that every byte the kernel must write is checked."""
    M, K = x_cpu.shape
    if ldx is not None and ldx > K:
        big = torch.zeros(M, ldx, dtype=torch.bfloat16)
        big[:, :K] = x_cpu
        x = big.to(DEV)[:, :K]
    else:
        x = x_cpu.to(DEV)
    g = torch.tensor([g_value], dtype=torch.float32, device=DEV)
    codes = torch.full((M, K // 2), 0xCD, dtype=torch.uint8, device=DEV)
    scales = torch.full((nv.nvfp4_scale_bytes(M, K),), 0xAB, dtype=torch.uint8, device=DEV)
    nv.nvfp4_quantize_act(x, g, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu(), scales.cpu()


def assert_same_quant(nv, x, g, ldx=None):
    c, s = gpu_quant(nv, x, g, ldx)
    oc, os_ = oracle.quantize(x, g)
    if not torch.equal(c, oc):
        bad = (c != oc).nonzero()[:5].tolist()
        raise AssertionError(f"codes differ at {bad}: gpu {[int(c[i][j]) for i, j in bad]} "
                             f"oracle {[int(oc[i][j]) for i, j in bad]}")
    if not torch.equal(s, os_):
        bad = (s != os_).nonzero()[:5].flatten().tolist()
        raise AssertionError(f"scales differ at {bad}: gpu {[int(s[i]) for i in bad]} "
                             f"oracle {[int(os_[i]) for i in bad]}")


@pytest.mark.parametrize("K", [512, 5120, 4352, 2048, 7168])
def test_global_bit_exact(lib, K):
    xc = synthdata.calibration_batch(K, seed=0)
    g = lib.nvfp4_compute_global(xc.to(DEV)).item()
    assert np.float32(g) == np.float32(oracle.global_scale(xc))
    w = synthdata.weights(300, K, seed=1)
    assert np.float32(lib.nvfp4_compute_global(w.to(DEV)).item()) == np.float32(oracle.global_scale(w))
    z = torch.zeros(4, K, dtype=torch.bfloat16)
    assert lib.nvfp4_compute_global(z.to(DEV)).item() == 1.0


@pytest.mark.parametrize("M,K,ldx", [
    (8, 512, None), (1, 16, None), (7, 48, None), (130, 5120, None), (257, 2048, 2056),
    (64, 7168, None), (33, 4352, 4360), (3, 80, 96),
] + [(m, 512, None) for m in (1, 2, 4, 5, 7, 8, 9, 15, 16, 17, 32)])
def test_quant_bit_exact(lib, M, K, ldx):
    x = synthdata.activations(M, K, seed=M + K)
    g = oracle.global_scale(synthdata.calibration_batch(K, seed=0))
    assert_same_quant(lib, x, g, ldx)


def test_quant_full_size_activation(lib):
    """The prefill activation of the fused qkv linear at M = 8192, K = 5120."""
    case = synthdata.prefill_case(8192, seed=0)
    g = oracle.global_scale(case.x_calib)
    assert_same_quant(lib, case.x, g)


def _bf(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)


def test_e2m1_ties_and_signs(lib):
    # block max 6 and g = 1 make S = 1 and r = 1: every element is converted as is
    vals = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.0, -0.25, -0.1, -5.0, -3.5, 0.26, 7.0, -0.0, 6.0]
    rows = [vals, [-v for v in vals], [v * 0.5 for v in vals[:15]] + [6.0]]
    x = _bf(rows)
    assert_same_quant(lib, x, 1.0)


def test_e4m3_ties(lib):
    # block amax = 6 * m with g = 1 gives s_f = m exactly: m on every E4M3 midpoint
    pos = sorted({oracle.e4m3_to_f32(b) for b in range(0x7F)})
    mids = [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    ms = [m for m in mids if float(_bf([6 * m])[0]) == 6 * m]
    assert len(ms) > 100
    rows = []
    for m in ms:
        r = [6 * m] + [m * 0.37 * (i % 5 - 2) for i in range(15)]
        rows.append(r)
    rows.append([480.0 * 6] + [1.0] * 15)  # saturation: s_f > 448
    while len(rows) % 4:
        rows.append([0.0] * 16)
    x = _bf(rows)
    assert_same_quant(lib, x, 1.0)


@pytest.mark.parametrize("g", [1.0, 2688.0 / 3.0, 1e-3, 7.7e4, 1.0e30])
def test_every_bf16_block_maximum(lib, g):
    """One block per non-negative finite bf16 value v (subnormals included) with
    v as its largest magnitude: the scale step amax / 6 is exact against the
    oracle's IEEE division for every input the quantiser can see.  With the
    large globals, x * r overflows fp32 for the largest blocks and satfinite
    clamps the codes to 6 on both sides."""
    bits = torch.arange(0, 0x7F80, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).float()
    frac = torch.tensor([1.0, -0.9, 0.75, -0.6, 0.5, -0.41, 0.33, -0.25, 0.2, -0.17, 0.12, -0.08, 0.05, -0.03,
                         0.01, -1.0])
    rows = (v[:, None] * frac[None, :]).to(torch.bfloat16)
    rows[:, 0] = v.to(torch.bfloat16)
    assert_same_quant(lib, rows, g)


def test_random_exponent_sweep(lib):
    rng = np.random.default_rng(11)
    M, K = 256, 256
    mant = rng.uniform(1, 2, size=(M, K))
    ex = rng.integers(-40, 40, size=(M, 1)) + rng.integers(-6, 7, size=(M, K))
    sign = rng.choice([-1.0, 1.0], size=(M, K))
    x = torch.from_numpy(sign * mant * np.exp2(ex)).to(torch.float32).to(torch.bfloat16)
    for g in [1.0, 2688.0 / 3.0, 1e-3, 7.7e4]:
        assert_same_quant(lib, x, g)


def test_quantize_fused_weight_matches_oracle(lib):
    """Config 2's fused weight: per-part globals, block scales unchanged, the
    fused tensor takes the largest global."""
    parts = [synthdata.weights(n, 512, seed=0, stream=100 + i) for i, n in enumerate([512, 128, 128])]
    W = lib.quantize_weight([p.to(DEV) for p in parts])
    codes, scales, g, gs = oracle.quantize_weight_parts(parts)
    assert torch.equal(W.codes.cpu(), codes) and torch.equal(W.scales.cpu(), scales)
    assert np.float32(W.g.item()) == np.float32(g)
    assert [np.float32(x.item()) for x in W.part_g] == [np.float32(x) for x in gs]
