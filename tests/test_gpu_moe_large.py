"""The large W4A4 MoE workload: E = 256 experts, top-8, hidden 7168, intermediate
2048, a skewed router (a per-expert logit bias), T = 1024, 8192 and 32768.

The layer runs in full on the GPU at every T; the oracle computes a seeded subset
of 256 tokens of each T, drawn with no regard to the experts they use (tokens
are independent, so a subset is checked exactly like the whole).  Both sides
start from the same bf16 bytes: every expert's weights are drawn on the GPU by
the seeded generator and quantised there by the library; the oracle quantises
all 256 experts from host copies of the same bytes, and the codes and scales
must agree bit for bit.

Static globals: g_a1 = 2688 / amax of the 64-row calibration batch (the same
for every expert, since every calibration row goes through every expert); g_a2
= the largest over all 256 experts of 2688 / amax_e, amax_e being the oracle's
largest |h| of expert e over the first 16 calibration rows.  The 16-row batch
is a reading that keeps the oracle's dense pass through 256 experts within a
minute; a static global only has to be the same on both sides (values above it
saturate the same way on both).  The library's own calibration of those rows
must give the same per-expert amax.

Checks, stage by stage:
  (i)   the NVFP4 intermediate h of the subset's routes, codes and scales,
        against the oracle's: a mismatch rate, since the tensor cores add the
        fp32 products in another order and a code flips where h sits on a
        rounding boundary;
  (ii)  down alone: the oracle's down stage fed the GPU's own h codes and
        scales must match the GPU layer output at the plain tolerance;
  (iii) the layer output against the oracle's whole layer: rel-L2 <= 1e-3, and
        an element beyond 2 bf16 ulp of its row max only in a token with an h
        code or scale that differs in (i).
The three subsets go through the oracle in one call (the oracle's cost is in
its per-expert weight decode, which one call pays once)."""
import numpy as np
import pytest
import torch

import oracle
import synthdata
from parity import REL_L2, ULPS, bf16_ulp_of_rowmax, check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
CFG = synthdata.MOE_LARGE
E, H, I, TOPK = CFG["E"], CFG["H"], CFG["I"], CFG["topk"]
SUBSET = 256
CALIB_ROWS = 16
H_MISMATCH_MAX = 2e-3


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_block_scaled_act_gb300 import build
    build.build()
    import nvfp4_block_scaled_act_gb300 as m
    m.load_library()
    return m


def _unswizzle(sf: torch.Tensor, R: int, C: int) -> np.ndarray:
    """Swizzled scale bytes over R rows -> [R, C] (atoms of 128 rows x 4 columns)."""
    Rp, Cp = (R + 127) // 128 * 128, (C + 3) // 4 * 4
    a = sf.numpy()[: Rp * Cp].reshape(Rp // 128, Cp // 4, 32, 4, 4)
    return a.transpose(0, 3, 2, 1, 4).reshape(Rp, Cp)[:R, :C]


def _swizzle(m: np.ndarray) -> torch.Tensor:
    """[R, C] scale bytes -> the swizzled buffer over R rows (inverse of _unswizzle)."""
    R, C = m.shape
    Rp, Cp = (R + 127) // 128 * 128, (C + 3) // 4 * 4
    full = np.zeros((Rp, Cp), dtype=np.uint8)
    full[:R, :C] = m
    a = full.reshape(Rp // 128, 4, 32, Cp // 4, 4).transpose(0, 3, 2, 1, 4)
    return torch.from_numpy(np.ascontiguousarray(a).reshape(-1))


def test_swizzle_helpers_round_trip():
    rng = np.random.default_rng(0)
    m = rng.integers(0, 256, size=(300, 12), dtype=np.uint8)
    sw = _swizzle(m)
    assert sw.numel() == oracle.scale_bytes(300, 12 * 16)
    assert np.array_equal(_unswizzle(sw, 300, 12), m)
    for r, c in ((0, 0), (37, 5), (299, 11), (130, 7)):
        assert int(sw[oracle.scale_offset(r, c, 12)]) == m[r, c]


@pytest.fixture(scope="module")
def weights(nv):
    """Both sides' quantisation of all 256 experts, and the static globals."""
    case = synthdata.moe_case(16, E, H, I, TOPK, CFG["skewed"], seed=0, device=DEV)
    W = nv.quantize_moe_weights(lambda e: case.w13(e, DEV), lambda e: case.w2(e, DEV), E, H, I, DEV)
    s13, s2 = oracle.scale_bytes(2 * I, H), oracle.scale_bytes(H, I)
    w13c = torch.empty(E * 2 * I, H // 2, dtype=torch.uint8)
    w13s = torch.empty(E * s13, dtype=torch.uint8)
    w2c = torch.empty(E * H, I // 2, dtype=torch.uint8)
    w2s = torch.empty(E * s2, dtype=torch.uint8)
    g13, g2 = [0.0] * E, [0.0] * E
    for e in range(E):
        a = case.w13(e, DEV).cpu()
        b = case.w2(e, DEV).cpu()
        g13[e], g2[e] = oracle.global_scale(a), oracle.global_scale(b)
        ca, sa = oracle.quantize(a, g13[e])
        cb, sb = oracle.quantize(b, g2[e])
        w13c[e * 2 * I:(e + 1) * 2 * I] = ca
        w13s[e * s13:(e + 1) * s13] = sa
        w2c[e * H:(e + 1) * H] = cb
        w2s[e * s2:(e + 1) * s2] = sb
    assert torch.equal(W.w13_codes.cpu(), w13c) and torch.equal(W.w13_sf.cpu(), w13s)
    assert torch.equal(W.w2_codes.cpu(), w2c) and torch.equal(W.w2_sf.cpu(), w2s)
    assert np.array_equal(W.g13.cpu().numpy(), np.float32(g13)) and np.array_equal(W.g2.cpu().numpy(), np.float32(g2))
    x_calib = case.x_calib.cpu()
    g_a1 = oracle.global_scale(x_calib)
    a13 = [oracle.alpha_w4a4(g_a1, g) for g in g13]
    x16 = x_calib[:CALIB_ROWS].contiguous()
    amax = oracle.moe_h_amax(x16, g_a1, w13c, w13s, a13, E, H, I)
    g_a2 = max(oracle.global_from_amax(float(v)) for v in amax)
    a2 = [oracle.alpha_w4a4(g_a2, g) for g in g2]
    g_a1_dev = nv.nvfp4_compute_global(case.x_calib)
    assert np.float32(g_a1_dev.item()) == np.float32(g_a1)
    a13_dev = nv.nvfp4_make_alpha(g_a1_dev, W.g13)
    assert np.array_equal(a13_dev.cpu().numpy(), np.float32(a13))
    g_a2_dev = torch.tensor([g_a2], dtype=torch.float32, device=DEV)
    a2_dev = nv.nvfp4_make_alpha(g_a2_dev, W.g2)
    assert np.array_equal(a2_dev.cpu().numpy(), np.float32(a2))
    return dict(W=W, w13c=w13c, w13s=w13s, w2c=w2c, w2s=w2s, g_a1=g_a1, g_a2=g_a2, a13=a13, a2=a2, amax=amax,
                x16=x16, g_a1_dev=g_a1_dev, a13_dev=a13_dev, g_a2_dev=g_a2_dev, a2_dev=a2_dev)


def test_moe_large_calibration_matches_oracle(nv, weights):
    """The library's calibration of the same 16 rows through all 256 experts."""
    L = weights
    g_a2, amax = nv.nvfp4_moe_calibrate(L["x16"].to(DEV), L["g_a1_dev"], L["W"].w13_codes, L["W"].w13_sf,
                                        L["a13_dev"], E, I)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status() == 0
    assert torch.allclose(amax.cpu(), L["amax"], rtol=1e-5, atol=0)
    assert abs(g_a2.item() - L["g_a2"]) <= 1e-5 * L["g_a2"]


@pytest.fixture(scope="module")
def runs(nv, weights):
    """The GPU layer at every T, reduced to each T's seeded 256-token subset:
    its output rows and the NVFP4 h of its routes (from the workspace), then the
    oracle's layer (with its h) and its down stage on the GPU's h, all three
    subsets in one call each."""
    L = weights
    per_t = []
    for T in CFG["tokens"]:
        case = synthdata.moe_case(T, E, H, I, TOPK, CFG["skewed"], seed=0, device=DEV)
        ws = torch.empty(nv.nvfp4_moe_workspace(T, H, I, E, TOPK), dtype=torch.uint8, device=DEV)
        out = nv.nvfp4_moe_w4a4(case.x, case.topk_ids, case.topk_w, L["g_a1_dev"], L["W"].w13_codes,
                                L["W"].w13_sf, L["a13_dev"], L["g_a2_dev"], L["W"].w2_codes, L["W"].w2_sf,
                                L["a2_dev"], E, I, workspace=ws)
        torch.cuda.synchronize()
        assert nv.nvfp4_device_status() == 0
        tokens = np.sort(np.random.default_rng(T).choice(T, SUBSET, replace=False))
        tok_t = torch.from_numpy(tokens)
        lay = nv.nvfp4_moe_workspace_layout(T, H, I, E, TOPK)
        n_tiles = int(ws[lay.n_tiles:lay.n_tiles + 4].view(torch.int32).item())
        P = n_tiles * 128
        row_map = ws[lay.row_map:lay.row_map + 4 * P].view(torch.int32).cpu()
        # permuted row of every route of the subset
        inv = torch.full((T * TOPK,), -1, dtype=torch.int64)
        real = (row_map >= 0).nonzero().flatten()
        inv[row_map[real].long()] = real
        routes = (tok_t[:, None] * TOPK + torch.arange(TOPK)[None, :]).flatten()
        rows = inv[routes]
        assert bool((rows >= 0).all()), "a route of the subset has no permuted row"
        hc_all = ws[lay.h_codes:lay.h_codes + lay.p_max * (I // 2)].view(lay.p_max, I // 2)
        hc = hc_all[rows.to(DEV)].cpu()
        hs_all = ws[lay.h_sf:lay.h_sf + oracle.scale_bytes(lay.p_max, I)].cpu()
        hs = _unswizzle(hs_all, lay.p_max, I // 16)[rows.numpy()]
        per_t.append(dict(T=T, tokens=tokens, out=out[tok_t.to(DEV)].cpu(), x=case.x[tok_t.to(DEV)].cpu(),
                          ids=case.topk_ids[tok_t.to(DEV)].cpu(), w=case.topk_w[tok_t.to(DEV)].cpu(),
                          hc=hc, hs=hs))
        del ws, out, case
        torch.cuda.empty_cache()
    x = torch.cat([r["x"] for r in per_t]).contiguous()
    ids = torch.cat([r["ids"] for r in per_t]).contiguous()
    w = torch.cat([r["w"] for r in per_t]).contiguous()
    ref, ref_hc, ref_hs = oracle.moe_w4a4(x, ids, w, L["g_a1"], L["w13c"], L["w13s"], L["a13"], L["g_a2"],
                                          L["w2c"], L["w2s"], L["a2"], E, H, I, want_h=True)
    gpu_hc = torch.cat([r["hc"] for r in per_t]).contiguous()
    gpu_hs = np.concatenate([r["hs"] for r in per_t])
    down = oracle.moe_down(gpu_hc, _swizzle(gpu_hs), ids, w, L["w2c"], L["w2s"], L["a2"], E, H, I)
    ref_hs_m = _unswizzle(ref_hs, ids.numel(), I // 16)
    n = SUBSET
    for j, r in enumerate(per_t):
        sl = slice(j * n, (j + 1) * n)
        rs = slice(j * n * TOPK, (j + 1) * n * TOPK)
        r.update(ref=ref[sl], down=down[sl], ref_hc=ref_hc[rs], ref_hs=ref_hs_m[rs])
    return {r["T"]: r for r in per_t}


@pytest.mark.parametrize("T", CFG["tokens"])
def test_moe_large_intermediate_codes(runs, T):
    r = runs[T]
    code_rate = (r["hc"] != r["ref_hc"]).float().mean().item()
    scale_rate = float((r["hs"] != r["ref_hs"]).mean())
    assert code_rate <= H_MISMATCH_MAX, f"T={T}: h code mismatch rate {code_rate:.2e}"
    assert scale_rate <= H_MISMATCH_MAX, f"T={T}: h scale mismatch rate {scale_rate:.2e}"


@pytest.mark.parametrize("T", CFG["tokens"])
def test_moe_large_down_on_the_gpu_intermediate(runs, T):
    r = runs[T]
    check_close(r["out"], r["down"], f"large MoE T={T}: down on the GPU's h ({SUBSET} tokens)")


@pytest.mark.parametrize("T", CFG["tokens"])
def test_moe_large_layer(runs, T):
    r = runs[T]
    g = r["out"].float().double()
    ref = r["ref"].float().double()
    rel = ((g - ref).norm() / ref.norm()).item()
    assert rel <= REL_L2, f"T={T}: rel-L2 {rel:.3e}"
    bad_rows = ((g - ref).abs() > ULPS * bf16_ulp_of_rowmax(ref)).any(dim=1).nonzero().flatten().tolist()
    flipped = set()
    for t in range(SUBSET):
        hs = slice(t * TOPK, (t + 1) * TOPK)
        if (r["hc"][hs] != r["ref_hc"][hs]).any() or (r["hs"][hs] != r["ref_hs"][hs]).any():
            flipped.add(t)
    unexplained = [t for t in bad_rows if t not in flipped]
    assert not unexplained, f"T={T}: tokens {unexplained[:8]} beyond {ULPS} ulp with no h flip"
