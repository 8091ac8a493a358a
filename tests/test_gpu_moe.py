"""GPU parity of the W4A4 MoE layer against the oracle, stage by stage:
  align       counts, offsets, row map and tile table bit-exact (both sides
              use a stable counting sort)
  permute     NVFP4 codes and scales of x at every permuted row bit-exact
  gate_up     NVFP4 codes of SiLU(gate) * up: the fp32 accumulation order of
              the tensor cores differs from the oracle's, so a code may flip
              where the oracle's value sits on a rounding boundary; the
              mismatch rate is bounded
  layer       output within rel-L2 <= 1e-3 and 2 bf16 ulp of the row max
The static globals (g_a1 from the calibration batch, g_a2 from the oracle's
calibration) are inputs given to both sides."""
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


class MoE:
    def __init__(self, nv, T, E, H, I, topk=8, skewed=False, seed=0):
        self.case = c = synthdata.moe_case(T, E, H, I, topk, skewed, seed=seed)
        self.T, self.E, self.H, self.I, self.topk = T, E, H, I, topk
        w13 = [c.w13(e, "cpu") for e in range(E)]
        w2 = [c.w2(e, "cpu") for e in range(E)]
        self.W = nv.quantize_moe_weights(lambda e: w13[e].to(DEV), lambda e: w2[e].to(DEV), E, H, I, DEV)
        q13 = [oracle.quantize(w, oracle.global_scale(w)) for w in w13]
        q2 = [oracle.quantize(w, oracle.global_scale(w)) for w in w2]
        self.g13 = [oracle.global_scale(w) for w in w13]
        self.g2 = [oracle.global_scale(w) for w in w2]
        self.w13c = torch.cat([q[0] for q in q13]); self.w13s = torch.cat([q[1] for q in q13])
        self.w2c = torch.cat([q[0] for q in q2]); self.w2s = torch.cat([q[1] for q in q2])
        assert torch.equal(self.W.w13_codes.cpu(), self.w13c) and torch.equal(self.W.w13_sf.cpu(), self.w13s)
        assert torch.equal(self.W.w2_codes.cpu(), self.w2c) and torch.equal(self.W.w2_sf.cpu(), self.w2s)
        # static input globals: g_a1 from the calibration batch (every row to every expert,
        # so the max over experts is the batch global); g_a2 from the oracle's calibration
        self.g_a1 = oracle.global_scale(c.x_calib)
        self.a13 = [oracle.alpha_w4a4(self.g_a1, g) for g in self.g13]
        self.amax = oracle.moe_h_amax(c.x_calib, self.g_a1, self.w13c, self.w13s, self.a13, E, H, I)
        self.g_a2 = max(oracle.global_from_amax(float(a)) for a in self.amax)
        self.a2 = [oracle.alpha_w4a4(self.g_a2, g) for g in self.g2]
        # device copies of the same scalars
        self.g_a1_dev = nv.nvfp4_compute_global(c.x_calib.to(DEV))
        assert np.float32(self.g_a1_dev.item()) == np.float32(self.g_a1)
        self.a13_dev = nv.nvfp4_make_alpha(self.g_a1_dev, self.W.g13)
        assert np.array_equal(self.a13_dev.cpu().numpy(), np.float32(self.a13))
        self.g_a2_dev = torch.tensor([self.g_a2], dtype=torch.float32, device=DEV)
        self.a2_dev = nv.nvfp4_make_alpha(self.g_a2_dev, self.W.g2)
        assert np.array_equal(self.a2_dev.cpu().numpy(), np.float32(self.a2))
        self.x_dev = c.x.to(DEV)
        self.ids_dev = c.topk_ids.to(DEV)
        self.w_dev = c.topk_w.to(DEV)

    def run_gpu(self, nv, ids=None):
        ws = torch.empty(nv.nvfp4_moe_workspace(self.T, self.H, self.I, self.E, self.topk), dtype=torch.uint8,
                         device=DEV)
        out = nv.nvfp4_moe_w4a4(self.x_dev, self.ids_dev if ids is None else ids, self.w_dev, self.g_a1_dev,
                                self.W.w13_codes, self.W.w13_sf, self.a13_dev, self.g_a2_dev, self.W.w2_codes,
                                self.W.w2_sf, self.a2_dev, self.E, self.I, workspace=ws)
        torch.cuda.synchronize()
        return out, ws

    def run_oracle(self, tokens=None, ids=None, want_h=False):
        c = self.case
        ids = c.topk_ids if ids is None else ids
        x, w = c.x, c.topk_w
        if tokens is not None:
            x, ids, w = x[tokens].contiguous(), ids[tokens].contiguous(), w[tokens].contiguous()
        return oracle.moe_w4a4(x, ids, w, self.g_a1, self.w13c, self.w13s, self.a13, self.g_a2, self.w2c,
                               self.w2s, self.a2, self.E, self.H, self.I, want_h=want_h)


def ws_view(nv, ws, m, name, dtype, count):
    lay = nv.nvfp4_moe_workspace_layout(m.T, m.H, m.I, m.E, m.topk)
    off = getattr(lay, name)
    nbytes = count * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype).cpu()


def unswizzle_row(sf: torch.Tensor, r: int, C: int) -> list:
    return [int(sf[oracle.scale_offset(r, c, C)]) for c in range(C)]


def row_block(nv, m: MoE) -> int:
    """The segment padding the layer uses: 256 (CTA-pair GEMMs) or 128."""
    return int(nv.nvfp4_moe_workspace_layout(m.T, m.H, m.I, m.E, m.topk).row_block)


def staged_check(nv, m: MoE, ws, h_mismatch_max=2e-3):
    ref_al = oracle.moe_align(m.case.topk_ids, m.E, row_block(nv, m))
    P = ref_al["P"]
    counts = ws_view(nv, ws, m, "counts", torch.int32, m.E)
    offsets = ws_view(nv, ws, m, "offsets", torch.int32, m.E + 1)
    row_map = ws_view(nv, ws, m, "row_map", torch.int32, P)
    tiles = ws_view(nv, ws, m, "tile_expert", torch.int32, P // 128)
    n_tiles = ws_view(nv, ws, m, "n_tiles", torch.int32, 1)
    assert torch.equal(counts, ref_al["counts"])
    assert torch.equal(offsets, ref_al["offsets"])
    assert torch.equal(row_map, ref_al["row_map"])
    assert torch.equal(tiles, ref_al["tile_expert"].repeat_interleave(row_block(nv, m) // 128))
    assert int(n_tiles[0]) == P // 128
    # permuted activations
    lay = nv.nvfp4_moe_workspace_layout(m.T, m.H, m.I, m.E, m.topk)
    a1 = ws[lay.a1_codes:lay.a1_codes + lay.p_max * m.H // 2].view(lay.p_max, m.H // 2).cpu()
    a1s = ws[lay.a1_sf:lay.a1_sf + lay.p_max * (m.H // 16)].cpu()
    xc, xs = oracle.quantize(m.case.x, m.g_a1)
    real = (row_map >= 0).nonzero().flatten()
    toks = row_map[real] // m.topk
    assert torch.equal(a1[real], xc[toks])
    for p in real[:: max(1, len(real) // 64)].tolist():
        t = int(row_map[p]) // m.topk
        assert unswizzle_row(a1s, p, m.H // 16) == unswizzle_row(xs, t, m.H // 16)
    # intermediate codes
    _, hc, hs = m.run_oracle(want_h=True)
    h = ws[lay.h_codes:lay.h_codes + lay.p_max * m.I // 2].view(lay.p_max, m.I // 2).cpu()
    got = h[real]
    want = hc[row_map[real].long()]
    rate = (got != want).float().mean().item()
    assert rate <= h_mismatch_max, f"intermediate code mismatch rate {rate:.2e}"
    return rate


def test_moe_small_staged(nv):
    m = MoE(nv, T=40, E=8, H=256, I=128, topk=4, seed=1)
    out, ws = m.run_gpu(nv)
    assert nv.nvfp4_device_status() == 0
    staged_check(nv, m, ws)
    check_close(out, m.run_oracle(), "MoE small")


def test_moe_repeatable_layout(nv):
    m = MoE(nv, T=64, E=16, H=256, I=256, topk=8, seed=2)
    o1, ws1 = m.run_gpu(nv)
    o2, ws2 = m.run_gpu(nv)
    P = oracle.moe_align(m.case.topk_ids, m.E, row_block(nv, m))["P"]
    for name, n in (("counts", m.E), ("offsets", m.E + 1), ("n_tiles", 1), ("row_map", P),
                    ("tile_expert", P // 128), ("pos", m.T * m.topk)):
        a = ws_view(nv, ws1, m, name, torch.int32, n)
        b = ws_view(nv, ws2, m, name, torch.int32, n)
        assert torch.equal(a, b), f"{name} differs between runs"
    check_close(o1, m.run_oracle(), "MoE 64 tokens")
    check_close(o2, o1, "run to run", ulps=1.0, rel_l2=1e-5)


@pytest.mark.parametrize("T,E,H,I,topk,skewed", [
    (1024, 4, 256, 128, 4, False),   # 1024 routes per expert: segments padded to 256
    (2048, 8, 512, 256, 4, True),    # skewed: pair tiles with few real rows
    (1100, 3, 768, 384, 3, True),    # ragged segments, three 256-column down tiles
])
def test_moe_pair_tiles_staged(nv, T, E, H, I, topk, skewed):
    """Layers whose experts average >= 1024 routes: gate_up and down run on CTA
    pairs (256-row tiles of one expert); every stage against the oracle on all
    tokens."""
    m = MoE(nv, T=T, E=E, H=H, I=I, topk=topk, skewed=skewed, seed=7)
    assert row_block(nv, m) == 256
    out, ws = m.run_gpu(nv)
    assert nv.nvfp4_device_status() == 0
    staged_check(nv, m, ws)
    check_close(out, m.run_oracle(), f"MoE pairs T={T} E={E}")


@pytest.mark.parametrize("T", [16, 128])
def test_moe_config_small_tokens(nv, T):
    """E = 128, top-8, hidden 2048, intermediate 768 at small T (oracle on all tokens)."""
    m = MoE(nv, T=T, E=128, H=2048, I=768, topk=8, seed=0)
    out, ws = m.run_gpu(nv)
    assert nv.nvfp4_device_status() == 0
    staged_check(nv, m, ws)
    check_close(out, m.run_oracle(), f"MoE E=128 T={T}")


@pytest.mark.parametrize("T", [1024, 4096, 8192])
def test_moe_config_sampled_tokens(nv, T):
    """E = 128, top-8 at the larger T: the whole layer on the GPU, the oracle on a
    seeded sample of 48 tokens (tokens are independent)."""
    m = MoE(nv, T=T, E=128, H=2048, I=768, topk=8, seed=0)
    out, _ = m.run_gpu(nv)
    rng = np.random.default_rng(T)
    tokens = sorted(set([0, T - 1] + rng.choice(T, 46, replace=False).tolist()))
    ref = m.run_oracle(tokens=tokens)
    check_close(out.cpu()[tokens], ref, f"MoE E=128 T={T} sampled")


def test_moe_invalid_expert_ids_are_dropped_and_flagged(nv):
    m = MoE(nv, T=24, E=8, H=256, I=128, topk=4, seed=3)
    ids = m.case.topk_ids.clone()
    ids[3, 1] = -1
    ids[7, 0] = 8
    out, _ = m.run_gpu(nv, ids=ids.to(DEV))
    assert nv.nvfp4_device_status() == 7
    assert nv.nvfp4_device_status() == 0  # cleared
    check_close(out, m.run_oracle(ids=ids), "MoE invalid ids")


def test_moe_calibration_matches_oracle(nv):
    m = MoE(nv, T=8, E=16, H=256, I=256, topk=4, seed=4)
    g_a2, amax = nv.nvfp4_moe_calibrate(m.case.x_calib.to(DEV), m.g_a1_dev, m.W.w13_codes, m.W.w13_sf,
                                        m.a13_dev, m.E, m.I)
    torch.cuda.synchronize()
    assert torch.allclose(amax.cpu(), m.amax, rtol=1e-5, atol=0)
    assert abs(g_a2.item() - m.g_a2) <= 1e-5 * m.g_a2


def test_moe_topk1_identity_routing_matches_linear_chain(nv):
    """One expert, top-1, weight 1: the layer is down(quant(silu(gate) * up))."""
    m = MoE(nv, T=130, E=1, H=256, I=128, topk=1, seed=5)
    out, ws = m.run_gpu(nv)
    staged_check(nv, m, ws)
    check_close(out, m.run_oracle(), "MoE E=1")
