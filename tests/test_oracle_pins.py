"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks one oracle function against a library routine (torch's
bfloat16 and float8_e4m3fn conversions), a constant the pages state
(tests/golden/pages_constants.json), the format definitions, an fp64 brute
force written here independently, or an invariant.  A dropped term, a wrong
sign, a wrong index or a transposed operand in the oracle fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synthdata

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")))


# ---------------------------------------------------------------------------
# independent decoders used by the brute-force pins (numpy / torch, not the oracle)
# ---------------------------------------------------------------------------

def e2m1_grid_from_definition():
    """e2m1 = 1 sign, 2 exponent bits (bias 1), 1 mantissa bit."""
    vals = []
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = (m * 0.5) if e == 0 else (2.0 ** (e - 1)) * (1 + m / 2)
        vals.append(-mag if s else mag)
    return np.array(vals, dtype=np.float64)


def unpack_codes_np(codes: torch.Tensor, K: int) -> np.ndarray:
    """[R, K/2] bytes -> [R, K] nibbles; element 2j in the low nibble."""
    b = codes.numpy().astype(np.uint8)
    lo = b & 0xF
    hi = b >> 4
    out = np.empty((b.shape[0], K), dtype=np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def unswizzle_np(scales: torch.Tensor, R: int, C: int) -> np.ndarray:
    """Swizzled scale bytes -> [R, C] via the atom shape [rb][cb][r%32][r%128/32][c%4]."""
    Rp = (R + 127) // 128 * 128
    Cp = (C + 3) // 4 * 4
    a = scales.numpy()[: Rp * Cp].reshape(Rp // 128, Cp // 4, 32, 4, 4)
    # -> [rb][rq][r32][cb][c4] -> rows rb*128 + rq*32 + r32, cols cb*4 + c4
    m = a.transpose(0, 3, 2, 1, 4).reshape(Rp, Cp)
    return m[:R, :C]


def e4m3_decode_torch(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(b.astype(np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy().astype(np.float64)


def dequant_np(codes, scales, R, K) -> np.ndarray:
    grid = e2m1_grid_from_definition()
    nib = unpack_codes_np(codes, K)
    S = e4m3_decode_torch(unswizzle_np(scales, R, K // 16))
    return grid[nib] * np.repeat(S, 16, axis=1)


def bf16_ulp(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, 1e-300)))
    return np.where(x > 0, 2.0 ** (e - 7), 2.0 ** -133)


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float32).numpy().astype(np.float64)


# ---------------------------------------------------------------------------
# scalar rules
# ---------------------------------------------------------------------------

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    base = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    # exact ties: a bf16 value plus half its ulp
    bf = torch.from_numpy(base).to(torch.bfloat16).to(torch.float32).numpy()
    ties = (bf.view(np.uint32) + np.uint32(0x8000)).view(np.float32)
    vals = np.concatenate([base, ties, np.float32([0.0, -0.0, 1e-40, 3.3e38, -3.3e38])])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.f32_to_bf16_bits(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_e4m3_decode_all_bytes_matches_torch():
    ref = e4m3_decode_torch(np.arange(256))
    got = np.array([oracle.e4m3_to_f32(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3_to_f32(0x7E) == GOLDEN["e4m3_max"]["value"]


def test_e4m3_encode_matches_torch_and_round_trips():
    finite = [b for b in range(256) if b not in (0x7F, 0xFF)]
    for b in finite:  # decode -> encode is the identity (negative zero included)
        assert oracle.f32_to_e4m3(oracle.e4m3_to_f32(b)) == b
    pos = np.array(sorted({oracle.e4m3_to_f32(b) for b in range(0x7F)}), dtype=np.float64)
    mids = (pos[1:] + pos[:-1]) / 2  # every tie, including the subnormal/normal seam
    rng = np.random.default_rng(2)
    rnd = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(464.0), 20000))
    vals = np.concatenate([pos, mids, rnd, [2.0 ** -10, 2.0 ** -11, 456.0, 464.0]]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.f32_to_e4m3(float(v)) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_saturates_to_448():
    for v in [448.0, 464.01, 480.0, 1e4, 3e38]:
        assert oracle.f32_to_e4m3(v) == 0x7E


def test_e2m1_table_from_definition_and_pages():
    grid = e2m1_grid_from_definition()
    got = np.array([oracle.e2m1_to_f32(c) for c in range(16)], dtype=np.float64)
    assert np.array_equal(got, grid)
    # low 3 bits magnitude, bit 3 sign (the pages' nibble table)
    nib = GOLDEN["e2m1_nibble"]
    for c in range(16):
        mag = oracle.e2m1_to_f32(c & ((1 << nib["magnitude_bits"]) - 1))
        sgn = -1.0 if (c >> nib["sign_bit"]) & 1 else 1.0
        assert oracle.e2m1_to_f32(c) == sgn * mag
    assert max(abs(grid)) == GOLDEN["e2m1_max"]["value"]
    for c in range(16):  # round trip (negative zero keeps its code)
        assert oracle.f32_to_e2m1(float(grid[c]) if c != 8 else -0.0) == c


@pytest.mark.parametrize("y,code", [
    (0.25, 0x0), (0.26, 0x1), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4),
    (3.5, 0x6), (5.0, 0x6), (5.01, 0x7), (7.0, 0x7), (1e9, 0x7),
    (-0.25, 0x8), (-0.1, 0x8), (-0.75, 0xA), (-5.0, 0xE), (-1e9, 0xF), (0.0, 0x0),
])
def test_e2m1_ties_to_even_and_saturation(y, code):
    assert oracle.f32_to_e2m1(y) == code


def test_satfinite_conversions_clamp_an_overflowed_product():
    """A product x * r far above the format's range (an activation far above the
    calibration amax, or an fp32 overflow to +-inf) is clamped by satfinite to
    the largest finite value: 6 for e2m1, 448 for E4M3."""
    inf = float("inf")
    for v in (6.0, 6.5, 7.0, 1.0e17, 3.0e38, inf):
        assert oracle.f32_to_e2m1(v) == 0x7 and oracle.f32_to_e2m1(-v) == 0xF, v
    for v in (448.0, 460.0, 470.0, 1.0e20, 3.0e38, inf):
        assert oracle.f32_to_e4m3(v) == 0x7E and oracle.f32_to_e4m3(-v) == 0xFE, v


def test_e2m1_nearest_brute_force():
    grid = e2m1_grid_from_definition()[:8]
    rng = np.random.default_rng(3)
    for v in rng.uniform(-8, 8, 3000).astype(np.float32):
        c = oracle.f32_to_e2m1(float(v))
        d = np.abs(grid - min(abs(float(v)), 6.0))
        assert d[c & 7] == d.min()
        assert (c >> 3) == (1 if v < 0 else 0)


# ---------------------------------------------------------------------------
# layout
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("R,C", [(1, 1), (8, 32), (130, 5), (256, 320), (300, 7)])
def test_swizzle_is_a_bijection_and_matches_atom_shape(R, C):
    Rp, Cp = (R + 127) // 128 * 128, (C + 3) // 4 * 4
    assert oracle.scale_bytes(R, 16 * C) == Rp * Cp
    offs = np.array([[oracle.scale_offset(r, c, C) for c in range(Cp)] for r in range(Rp)])
    assert np.array_equal(np.sort(offs.ravel()), np.arange(Rp * Cp))
    # the same layout built by reshaping: write (r, c) ids, read them back
    buf = np.zeros(Rp * Cp, dtype=np.int64)
    buf[offs.ravel()] = np.arange(Rp * Cp)
    ids = unswizzle_np(torch.from_numpy(buf), Rp, Cp)
    assert np.array_equal(ids, np.arange(Rp * Cp).reshape(Rp, Cp))


# ---------------------------------------------------------------------------
# quantisation
# ---------------------------------------------------------------------------

def test_global_scale_definition():
    x = synthdata.calibration_batch(512, seed=0)
    a = float(np.abs(bf16_np(x)).max())
    g = oracle.global_scale(x)
    assert g == float(np.float32(GOLDEN["global_numerator"]["value"]) / np.float32(a))
    assert oracle.global_scale(torch.zeros(4, 32, dtype=torch.bfloat16)) == 1.0


def _blocks(x):
    return x.reshape(x.shape[0], -1, 16)


@pytest.mark.parametrize("seed", [0, 1])
def test_quant_invariants(seed):
    K = 512
    x = synthdata.activations(37, K, seed)
    g = oracle.global_scale(synthdata.calibration_batch(K, seed))
    codes, scales = oracle.quantize(x, g)
    xv = bf16_np(x)
    grid = e2m1_grid_from_definition()
    nib = unpack_codes_np(codes, K)
    S = e4m3_decode_torch(unswizzle_np(scales, 37, K // 16))
    amax_b = np.abs(_blocks(xv)).max(axis=2)
    sat = S == 448.0
    # the block scale covers the block amax up to E4M3 rounding, unless saturated
    assert np.all((S * 6 / g >= amax_b * (1 - 2.0 ** -4)) | sat)
    # every code is the nearest grid point of x * g / S (within fp32 rounding of r)
    y = _blocks(xv) * (np.float32(g) / S.astype(np.float32))[:, :, None]
    v = _blocks(grid[nib])
    gaps = np.array([0.5, 0.5, 0.5, 0.5, 1, 1, 2, 2])  # distance to the next grid point
    idx = np.clip(np.searchsorted(grid[:8], np.minimum(np.abs(y), 6.0)), 0, 7)
    assert np.all(np.abs(np.abs(v) - np.minimum(np.abs(y), 6)) <= gaps[idx] / 2 * (1 + 1e-6))
    assert np.all((np.sign(v) == np.sign(y)) | (v == 0))
    # padding of the scale array is zero
    pad = np.ones(scales.numel(), bool)
    pad[[oracle.scale_offset(r, c, K // 16) for r in range(37) for c in range(K // 16)]] = False
    assert np.all(scales.numpy()[pad] == 0)


def test_quant_zero_rows_and_blocks():
    x = synthdata.activations(4, 64, 5)
    x[1] = 0
    x[2, 16:32] = 0
    codes, scales = oracle.quantize(x, 3.0)
    assert np.all(codes[1].numpy() == 0)
    assert np.all(codes[2, 8:16].numpy() == 0)
    S = unswizzle_np(scales, 4, 4)
    assert np.all(S[1] == 0) and S[2, 1] == 0 and np.all(S[0] > 0)
    # negative zeros in an all-zero block still give +0 codes
    xn = torch.full((1, 16), -0.0, dtype=torch.bfloat16)
    c, _ = oracle.quantize(xn, 2.0)
    assert np.all(c.numpy() == 0)


@pytest.mark.parametrize("p", [-6, -3, 0, 3, 7])
def test_quant_constant_power_of_two_blocks(p):
    # g = 6: s_f = amax exactly, S = amax, r = 6 / amax, y = +-6 -> codes 0x7 / 0xF
    x = torch.full((2, 32), 2.0 ** p, dtype=torch.bfloat16)
    x[1] = -x[1]
    codes, scales = oracle.quantize(x, 6.0)
    assert np.all(codes[0].numpy() == 0x77) and np.all(codes[1].numpy() == 0xFF)
    S = e4m3_decode_torch(unswizzle_np(scales, 2, 2))
    assert np.all(S == 2.0 ** p)
    # halving the global: S = amax / 2 exactly, y = 6 again
    c2, s2 = oracle.quantize(x, 3.0)
    assert np.all(c2[0].numpy() == 0x77)
    # the value 4 appears when the block max is 1.5x larger than the element
    x3 = torch.full((1, 16), 2.0 ** p, dtype=torch.bfloat16)
    x3[0, 0] = 1.5 * 2.0 ** p
    c3, _ = oracle.quantize(x3, 6.0)
    nib = unpack_codes_np(c3, 16)[0]
    assert nib[0] == 0x7 and np.all(nib[1:] == 0x6)


def test_quant_saturates_above_calibration():
    # a runtime block far above the calibration amax: scale 448, codes +-6
    x = torch.zeros(1, 16, dtype=torch.bfloat16)
    x[0, :8] = 1000.0
    x[0, 8:] = -1000.0
    codes, scales = oracle.quantize(x, 2688.0 / 10.0)
    assert e4m3_decode_torch(unswizzle_np(scales, 1, 1))[0, 0] == 448.0
    nib = unpack_codes_np(codes, 16)[0]
    assert np.all(nib[:8] == 0x7) and np.all(nib[8:] == 0xF)


def test_quant_round_trip_error():
    K = 256
    x = synthdata.activations(16, K, 7)
    g = oracle.global_scale(x)
    codes, scales = oracle.quantize(x, g)
    back = dequant_np(codes, scales, 16, K) / g
    xv = bf16_np(x)
    amax_b = np.repeat(np.abs(_blocks(xv)).max(axis=2), 16, axis=1)
    # half the largest e2m1 gap (1 of 6) of the block, plus E4M3 rounding of S
    assert np.all(np.abs(back - xv) <= amax_b * (1.0 / 6 + 1.0 / 8) + 1e-30)
    rel = np.linalg.norm(back - xv) / np.linalg.norm(xv)
    assert rel < 0.12


# ---------------------------------------------------------------------------
# GEMMs against an fp64 brute force
# ---------------------------------------------------------------------------

def _random_nvfp4(R, K, rng, sf_lo=0x20, sf_hi=0x48):
    codes = torch.from_numpy(rng.integers(0, 256, size=(R, K // 2), dtype=np.uint8))
    sw = oracle.scale_bytes(R, K)
    scales = torch.zeros(sw, dtype=torch.uint8)
    C = K // 16
    for r in range(R):
        for c in range(C):
            scales[oracle.scale_offset(r, c, C)] = int(rng.integers(sf_lo, sf_hi))
    return codes, scales


def _fp32_sum_bound(a, b):
    # |fp32 sum - exact| <= K * 2^-24 * sum |a_k b_k|
    return a.shape[1] * 2.0 ** -24 * (np.abs(a) @ np.abs(b).T)


@pytest.mark.parametrize("M,N,K", [(3, 5, 32), (9, 16, 64), (17, 24, 128)])
def test_w4a4_matches_fp64_brute_force(M, N, K):
    rng = np.random.default_rng(M * 100 + N)
    ac, asf = _random_nvfp4(M, K, rng)
    wc, wsf = _random_nvfp4(N, K, rng)
    alpha = 0.37
    got = bf16_np(oracle.linear_w4a4(ac, asf, M, wc, wsf, N, K, alpha))
    A = dequant_np(ac, asf, M, K)
    W = dequant_np(wc, wsf, N, K)
    ref = (A @ W.T) * np.float64(np.float32(alpha))
    tol = bf16_ulp(ref) * 0.5 + _fp32_sum_bound(A, W) * alpha * 1.01 + 1e-30
    assert np.all(np.abs(got - ref) <= tol + bf16_ulp(ref) * 1e-3)


@pytest.mark.parametrize("T,N,K", [(1, 7, 32), (4, 16, 64), (16, 9, 96)])
def test_w4a16_matches_fp64_brute_force(T, N, K):
    rng = np.random.default_rng(T * 10 + K)
    x = torch.from_numpy(rng.standard_normal((T, K)).astype(np.float32)).to(torch.bfloat16)
    wc, wsf = _random_nvfp4(N, K, rng)
    alpha = 0.011
    got = bf16_np(oracle.linear_w4a16(x, wc, wsf, N, K, alpha))
    X = bf16_np(x)
    W = dequant_np(wc, wsf, N, K)
    ref = (X @ W.T) * np.float64(np.float32(alpha))
    tol = bf16_ulp(ref) * 0.5 + _fp32_sum_bound(X, W) * alpha * 1.01
    assert np.all(np.abs(got - ref) <= tol + 1e-30)


def _refcheck(out, ref):
    o = out.double().flatten()
    r = ref.double().flatten()
    rel = ((o - r).norm() / r.norm()).item()
    cos = torch.nn.functional.cosine_similarity(o, r, dim=0).item()
    return rel, cos


def test_w4a16_refcheck_against_unquantised_weight():
    """The pages' acceptance check: rel_l2 < 0.15 and cos > 0.99 against the
    bf16 matmul with the unquantised weight."""
    case = synthdata.tiny_linear(seed=0)
    w = case.w_parts[0]
    g_w = oracle.global_scale(w)
    wc, wsf = oracle.quantize(w, g_w)
    out = oracle.linear_w4a16(case.x, wc, wsf, 256, 512, oracle.alpha_w4a16(g_w))
    ref = (case.x.float() @ w.float().T).to(torch.bfloat16)
    rel, cos = _refcheck(out, ref)
    bounds = GOLDEN["refcheck_w4a16_vs_unquantised"]
    assert rel < bounds["rel_l2_max"] and cos > bounds["cos_min"]


def test_w4a4_refcheck_against_unquantised():
    case = synthdata.tiny_linear(seed=0)
    w = case.w_parts[0]
    g_w = oracle.global_scale(w)
    g_a = oracle.global_scale(case.x_calib)
    wc, wsf = oracle.quantize(w, g_w)
    ac, asf = oracle.quantize(case.x, g_a)
    out = oracle.linear_w4a4(ac, asf, 8, wc, wsf, 256, 512, oracle.alpha_w4a4(g_a, g_w))
    ref = (case.x.float() @ w.float().T).to(torch.bfloat16)
    rel, cos = _refcheck(out, ref)
    assert rel < 0.2 and cos > 0.98


def test_fused_parts_use_largest_global():
    parts = [synthdata.weights(128, 64, 0, 100), synthdata.weights(128, 64, 0, 101) * 3]
    codes, scales, g, gs = oracle.quantize_weight_parts(parts)
    assert g == max(gs) and gs[0] > gs[1]
    c1, s1 = oracle.quantize(parts[1], gs[1])
    assert torch.equal(codes[128:], c1)
    assert torch.equal(scales[oracle.scale_bytes(128, 64):], s1)


# ---------------------------------------------------------------------------
# MoE
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,topk,E,BM", [(50, 4, 9, 16), (300, 8, 5, 128), (700, 4, 3, 256), (90, 2, 64, 256)])
def test_moe_align_matches_numpy(T, topk, E, BM):
    """The stable counting sort with BM-row segments (the 128- and 256-row
    paddings the GEMM tiles use among them) against numpy's stable argsort."""
    rng = np.random.default_rng(4 + BM)
    ids = rng.integers(0, E, size=(T, topk)).astype(np.int32)
    ids[3, 1] = -1
    ids[7, topk - 1] = E  # invalid ids are dropped
    res = oracle.moe_align(torch.from_numpy(ids), E, BM)
    flat = ids.ravel()
    valid = (flat >= 0) & (flat < E)
    counts = np.bincount(flat[valid], minlength=E)
    assert np.array_equal(res["counts"].numpy(), counts)
    padded = -(-counts // BM) * BM
    offs = np.concatenate([[0], np.cumsum(padded)])
    assert np.array_equal(res["offsets"].numpy(), offs)
    order = np.argsort(np.where(valid, flat, E), kind="stable")[: valid.sum()]
    rm = res["row_map"].numpy()
    for e in range(E):
        seg = rm[offs[e]:offs[e + 1]]
        want = order[np.where(valid, flat, E)[order] == e]
        assert np.array_equal(seg[: counts[e]], want)
        assert np.all(seg[counts[e]:] == -1)
        assert np.all(res["tile_expert"].numpy()[offs[e] // BM: offs[e + 1] // BM] == e)


def _tiny_moe(E=3, H=64, I=32, T=6, topk=2, seed=0, same_experts=False):
    case = synthdata.moe_case(T, E, H, I, topk, seed=seed)
    w13 = [case.w13(0 if same_experts else e) for e in range(E)]
    w2 = [case.w2(0 if same_experts else e) for e in range(E)]
    g13 = [oracle.global_scale(w) for w in w13]
    g2 = [oracle.global_scale(w) for w in w2]
    q13 = [oracle.quantize(w, g) for w, g in zip(w13, g13)]
    q2 = [oracle.quantize(w, g) for w, g in zip(w2, g2)]
    w13c = torch.cat([q[0] for q in q13]); w13s = torch.cat([q[1] for q in q13])
    w2c = torch.cat([q[0] for q in q2]); w2s = torch.cat([q[1] for q in q2])
    g_a1 = oracle.global_scale(case.x_calib)
    a13 = [oracle.alpha_w4a4(g_a1, g) for g in g13]
    amax = oracle.moe_h_amax(case.x_calib, g_a1, w13c, w13s, a13, E, H, I)
    g_a2 = max(oracle.global_from_amax(float(a)) for a in amax)
    a2 = [oracle.alpha_w4a4(g_a2, g) for g in g2]
    return dict(case=case, w13=w13, w2=w2, w13c=w13c, w13s=w13s, w2c=w2c, w2s=w2s,
                g_a1=g_a1, g_a2=g_a2, a13=a13, a2=a2, amax=amax, E=E, H=H, I=I)


def _silu64(v):
    return v / (1.0 + np.exp(-v))


def test_moe_reduces_to_quantised_mlp():
    """topk = 1 with weight 1: the layer is down(quant(silu(gate) * up)) of one
    expert, recomputed here with an fp64 brute force (gate = rows [0, I))."""
    d = _tiny_moe(E=2, T=5, topk=1, seed=3)
    case, E, H, I = d["case"], d["E"], d["H"], d["I"]
    ids = torch.tensor([[1], [0], [1], [1], [0]], dtype=torch.int32)
    w = torch.ones(5, 1)
    out = bf16_np(oracle.moe_w4a4(case.x, ids, w, d["g_a1"], d["w13c"], d["w13s"], d["a13"],
                                  d["g_a2"], d["w2c"], d["w2s"], d["a2"], E, H, I))
    xc, xs = oracle.quantize(case.x, d["g_a1"])
    X = dequant_np(xc, xs, 5, H)
    for t in range(5):
        e = int(ids[t, 0])
        W13 = dequant_np(*oracle.quantize(d["w13"][e], oracle.global_scale(d["w13"][e])), 2 * I, H)
        W2 = dequant_np(*oracle.quantize(d["w2"][e], oracle.global_scale(d["w2"][e])), H, I)
        G = X[t] @ W13[:I].T
        U = X[t] @ W13[I:].T
        a13 = np.float64(np.float32(d["a13"][e]))
        h = _silu64(a13 * G) * (a13 * U)
        hc, hs = oracle.quantize(torch.from_numpy(h.astype(np.float32))[None], d["g_a2"])
        Hq = dequant_np(hc, hs, 1, I)[0]
        ref = np.float64(np.float32(d["a2"][e])) * (Hq @ W2.T)
        err = np.abs(out[t] - ref)
        assert np.all(err <= 2 * bf16_ulp(np.abs(ref).max()))


@pytest.mark.parametrize("topk,seed", [(1, 21), (3, 22)])
def test_moe_down_matches_fp64_brute_force(topk, seed):
    """The down stage on an arbitrary NVFP4 intermediate (random codes and
    scales, as another implementation's h would be): per route
    d = alpha2[e] * h^ @ W2^[e].T, then the routing-weighted sum over the slots,
    against an fp64 brute force with independent decoders; a route with an id
    outside [0, E) contributes nothing."""
    E, H, I, T = 3, 48, 64, 5
    d = _tiny_moe(E=E, T=T, topk=topk, seed=seed, H=H, I=I)
    case = d["case"]
    rng = np.random.default_rng(seed)
    R = T * topk
    hc, hs = _random_nvfp4(R, I, rng)
    ids = case.topk_ids.clone()
    ids[2, topk - 1] = -1
    ids[4, 0] = E
    got = bf16_np(oracle.moe_down(hc, hs, ids, case.topk_w, d["w2c"], d["w2s"], d["a2"], E, H, I))
    Hq = dequant_np(hc, hs, R, I)
    sb = oracle.scale_bytes(H, I)
    ref = np.zeros((T, H))
    bound = np.zeros((T, H))
    for t in range(T):
        for s in range(topk):
            e = int(ids[t, s])
            if e < 0 or e >= E:
                continue
            W2 = dequant_np(d["w2c"][e * H:(e + 1) * H], d["w2s"][e * sb:(e + 1) * sb], H, I)
            i = t * topk + s
            w = np.float64(np.float32(case.topk_w[t, s]))
            a2 = np.float64(np.float32(d["a2"][e]))
            ref[t] += w * a2 * (Hq[i] @ W2.T)
            # fp32 dot (I terms), times alpha2 and w, then a sum of up to topk terms
            bound[t] += w * a2 * (I + 3 + topk) * 2.0 ** -24 * (np.abs(Hq[i]) @ np.abs(W2).T)
    tol = bf16_ulp(ref) * 0.5 + bound * 1.01 + 1e-30
    assert np.all(np.abs(got - ref) <= tol + bf16_ulp(ref) * 1e-3)


def test_moe_down_reproduces_the_layer_on_its_own_intermediate():
    """Fed the oracle layer's own NVFP4 h, the down stage gives the layer's output
    bit for bit (the two are the same steps on the same values)."""
    d = _tiny_moe(E=4, T=7, topk=3, seed=23, H=64, I=32)
    case, E, H, I = d["case"], d["E"], d["H"], d["I"]
    out, hc, hs = oracle.moe_w4a4(case.x, case.topk_ids, case.topk_w, d["g_a1"], d["w13c"], d["w13s"], d["a13"],
                                  d["g_a2"], d["w2c"], d["w2s"], d["a2"], E, H, I, want_h=True)
    again = oracle.moe_down(hc, hs, case.topk_ids, case.topk_w, d["w2c"], d["w2s"], d["a2"], E, H, I)
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


def test_moe_identical_experts_ignore_routing():
    d = _tiny_moe(E=4, T=6, topk=3, seed=5, same_experts=True)
    case, E, H, I = d["case"], d["E"], d["H"], d["I"]
    args = (d["g_a1"], d["w13c"], d["w13s"], d["a13"], d["g_a2"], d["w2c"], d["w2s"], d["a2"], E, H, I)
    out = bf16_np(oracle.moe_w4a4(case.x, case.topk_ids, case.topk_w, *args))
    one = bf16_np(oracle.moe_w4a4(case.x, torch.zeros(6, 1, dtype=torch.int32), torch.ones(6, 1), *args))
    assert np.all(np.abs(out - one) <= 2 * bf16_ulp(np.abs(one).max(axis=1, keepdims=True)))


def test_moe_invalid_ids_contribute_nothing():
    d = _tiny_moe(E=3, T=4, topk=2, seed=6)
    case, E, H, I = d["case"], d["E"], d["H"], d["I"]
    args = (d["g_a1"], d["w13c"], d["w13s"], d["a13"], d["g_a2"], d["w2c"], d["w2s"], d["a2"], E, H, I)
    ids = case.topk_ids.clone()
    ids[:, 1] = -1
    a = oracle.moe_w4a4(case.x, ids, case.topk_w, *args)
    b = oracle.moe_w4a4(case.x, case.topk_ids[:, :1].contiguous(), case.topk_w[:, :1].contiguous(), *args)
    assert torch.equal(a, b)


def test_moe_against_unquantised_fp64():
    d = _tiny_moe(E=3, T=8, topk=2, seed=7, H=128, I=64)
    case, E, H, I = d["case"], d["E"], d["H"], d["I"]
    out = oracle.moe_w4a4(case.x, case.topk_ids, case.topk_w, d["g_a1"], d["w13c"], d["w13s"],
                          d["a13"], d["g_a2"], d["w2c"], d["w2s"], d["a2"], E, H, I)
    X = bf16_np(case.x)
    ref = np.zeros((8, H))
    for t in range(8):
        for s in range(2):
            e = int(case.topk_ids[t, s])
            W13 = bf16_np(d["w13"][e]); W2 = bf16_np(d["w2"][e])
            h = _silu64(X[t] @ W13[:I].T) * (X[t] @ W13[I:].T)
            ref[t] += float(case.topk_w[t, s]) * (h @ W2.T)
    rel, cos = _refcheck(out, torch.from_numpy(ref))
    assert cos > 0.97 and rel < 0.3


def test_moe_h_amax_is_max_over_rows_and_columns():
    d = _tiny_moe(E=2, T=3, topk=1, seed=8)
    case, E, H, I = d["case"], d["E"], d["H"], d["I"]
    xc, xs = oracle.quantize(case.x_calib, d["g_a1"])
    X = dequant_np(xc, xs, case.x_calib.shape[0], H)
    for e in range(E):
        W13 = dequant_np(*oracle.quantize(d["w13"][e], oracle.global_scale(d["w13"][e])), 2 * I, H)
        a13 = np.float64(np.float32(d["a13"][e]))
        h = _silu64(a13 * (X @ W13[:I].T)) * (a13 * (X @ W13[I:].T))
        assert math.isclose(float(d["amax"][e]), float(np.abs(h).max()), rel_tol=1e-5)


# ---------------------------------------------------------------------------
# W4A16 MoE (bf16 activations, bf16 intermediate)
# ---------------------------------------------------------------------------

def _tiny_moe_w4a16(E=3, H=64, I=32, T=6, topk=2, seed=0, same_experts=False):
    case = synthdata.moe_case(T, E, H, I, topk, seed=seed)
    w13 = [case.w13(0 if same_experts else e) for e in range(E)]
    w2 = [case.w2(0 if same_experts else e) for e in range(E)]
    g13 = [oracle.global_scale(w) for w in w13]
    g2 = [oracle.global_scale(w) for w in w2]
    q13 = [oracle.quantize(w, g) for w, g in zip(w13, g13)]
    q2 = [oracle.quantize(w, g) for w, g in zip(w2, g2)]
    return dict(case=case, w13c=torch.cat([q[0] for q in q13]), w13s=torch.cat([q[1] for q in q13]),
                w2c=torch.cat([q[0] for q in q2]), w2s=torch.cat([q[1] for q in q2]),
                q13=q13, q2=q2, a13=[oracle.alpha_w4a16(g) for g in g13], a2=[oracle.alpha_w4a16(g) for g in g2],
                E=E, H=H, I=I)


def _w4a16_moe_fp64(d, x, ids, w):
    """Brute force: fp64 sums of bf16 x against dequantised weights; h rounded
    to bf16 with torch's conversion; gate = rows [0, I) of W13."""
    E, H, I = d["E"], d["H"], d["I"]
    X = x.to(torch.float64).numpy()
    T, topk = ids.shape
    y = np.zeros((T, H))
    hs = np.zeros((T * topk, I))
    for t in range(T):
        for s in range(topk):
            e = int(ids[t, s])
            if e < 0 or e >= E:
                continue
            W13 = dequant_np(*d["q13"][e], 2 * I, H)
            W2 = dequant_np(*d["q2"][e], H, I)
            a13 = np.float64(np.float32(d["a13"][e]))
            G = X[t] @ W13[:I].T
            U = X[t] @ W13[I:].T
            h = torch.from_numpy(_silu64(a13 * G) * (a13 * U)).to(torch.bfloat16).to(torch.float64).numpy()
            hs[t * topk + s] = h
            y[t] += float(w[t, s]) * np.float64(np.float32(d["a2"][e])) * (h @ W2.T)
    return y, hs


def test_moe_w4a16_reduces_to_gated_mlp():
    """topk = 1 with weight 1: down(bf16(silu(gate) * up)) of one expert."""
    d = _tiny_moe_w4a16(E=2, T=5, topk=1, seed=3)
    case, E, H, I = d["case"], d["E"], d["H"], d["I"]
    ids = torch.tensor([[1], [0], [1], [1], [0]], dtype=torch.int32)
    w = torch.ones(5, 1)
    out, h = oracle.moe_w4a16(case.x, ids, w, d["w13c"], d["w13s"], d["a13"], d["w2c"], d["w2s"], d["a2"],
                              E, H, I, want_h=True)
    ref, href = _w4a16_moe_fp64(d, case.x, ids, w)
    out, h = bf16_np(out), bf16_np(h)
    # h: the fp32 sums may round to the other side of a bf16 tie at most
    assert np.all(np.abs(h - href) <= bf16_ulp(np.abs(href)) + 1e-30)
    assert np.all(np.abs(out - ref) <= 2 * bf16_ulp(np.abs(ref).max(axis=1, keepdims=True)))


def test_moe_w4a16_topk_weighted_sum():
    d = _tiny_moe_w4a16(E=4, T=6, topk=3, seed=8, H=128, I=64)
    case, E, H, I = d["case"], d["E"], d["H"], d["I"]
    out = bf16_np(oracle.moe_w4a16(case.x, case.topk_ids, case.topk_w, d["w13c"], d["w13s"], d["a13"],
                                   d["w2c"], d["w2s"], d["a2"], E, H, I))
    ref, _ = _w4a16_moe_fp64(d, case.x, case.topk_ids, case.topk_w)
    assert np.all(np.abs(out - ref) <= 2 * bf16_ulp(np.abs(ref).max(axis=1, keepdims=True)))


def test_moe_w4a16_invalid_ids_contribute_nothing():
    d = _tiny_moe_w4a16(E=3, T=4, topk=2, seed=6)
    case, E, H, I = d["case"], d["E"], d["H"], d["I"]
    args = (d["w13c"], d["w13s"], d["a13"], d["w2c"], d["w2s"], d["a2"], E, H, I)
    ids = case.topk_ids.clone()
    ids[:, 1] = -1
    a = oracle.moe_w4a16(case.x, ids, case.topk_w, *args)
    b = oracle.moe_w4a16(case.x, case.topk_ids[:, :1].contiguous(), case.topk_w[:, :1].contiguous(), *args)
    assert torch.equal(a, b)


def test_moe_w4a16_identical_experts_ignore_routing():
    d = _tiny_moe_w4a16(E=4, T=6, topk=3, seed=5, same_experts=True)
    case, E, H, I = d["case"], d["E"], d["H"], d["I"]
    args = (d["w13c"], d["w13s"], d["a13"], d["w2c"], d["w2s"], d["a2"], E, H, I)
    w = case.topk_w
    out = bf16_np(oracle.moe_w4a16(case.x, case.topk_ids, w, *args))
    one = bf16_np(oracle.moe_w4a16(case.x, torch.zeros(6, 1, dtype=torch.int32), w.sum(1, keepdim=True), *args))
    assert np.all(np.abs(out - one) <= 2 * bf16_ulp(np.abs(one).max(axis=1, keepdims=True)))
