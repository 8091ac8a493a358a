"""The large W4A4 MoE workload: E = 256 experts, top-8, hidden 7168, intermediate
2048, a skewed router (a per-expert logit bias), T = 1024, 8192 and 32768.

The layer runs in full on the GPU at every T; the oracle computes a seeded
sample of tokens (tokens are independent, so a sample is checked exactly like
the whole).  The sample is drawn in a seeded order among the tokens whose
experts keep the union of experts within a budget, because the oracle's
quantisation of one expert's weights takes about a second.  Both sides start
from the same bf16 bytes: every expert's weights are drawn on the GPU by the
seeded generator and quantised there by the library; the experts the sample
uses are also copied to the host and quantised there by the oracle on its own
(the codes and scales must agree bit for bit), and the oracle's forward pass
uses its own quantisation.  The static globals are the oracle's: g_a1 from the
calibration batch; g_a2 from the oracle's calibration of experts 0-15 on the
first two calibration rows (a static global only has to be the same on both
sides; values above it saturate the same way on both)."""
import numpy as np
import pytest
import torch

import oracle
import synthdata
from parity import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
CFG = synthdata.MOE_LARGE
E, H, I, TOPK = CFG["E"], CFG["H"], CFG["I"], CFG["topk"]
CALIB_EXPERTS = 16
CALIB_ROWS = 2
MAX_EXPERTS = 40   # union of experts of a T's token sample
MAX_TOKENS = 24


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_block_scaled_act_gb300 import build
    build.build()
    import nvfp4_block_scaled_act_gb300 as m
    m.load_library()
    return m


class OracleWeights:
    """The oracle's own quantisation of the experts it needs (full-size arrays;
    the rows of experts no sampled route uses stay zero and are never read)."""

    def __init__(self, case, W):
        self.case, self.W = case, W
        self.w13c = torch.zeros(E * 2 * I, H // 2, dtype=torch.uint8)
        self.w13s = torch.zeros(E * oracle.scale_bytes(2 * I, H), dtype=torch.uint8)
        self.w2c = torch.zeros(E * H, I // 2, dtype=torch.uint8)
        self.w2s = torch.zeros(E * oracle.scale_bytes(H, I), dtype=torch.uint8)
        self.g13 = [1.0] * E
        self.g2 = [1.0] * E
        self.done = set()

    def need(self, experts):
        s13, s2 = oracle.scale_bytes(2 * I, H), oracle.scale_bytes(H, I)
        for e in sorted(set(experts) - self.done):
            a = self.case.w13(e, DEV).cpu()
            b = self.case.w2(e, DEV).cpu()
            self.g13[e], self.g2[e] = oracle.global_scale(a), oracle.global_scale(b)
            ca, sa = oracle.quantize(a, self.g13[e])
            cb, sb = oracle.quantize(b, self.g2[e])
            self.w13c[e * 2 * I:(e + 1) * 2 * I] = ca
            self.w13s[e * s13:(e + 1) * s13] = sa
            self.w2c[e * H:(e + 1) * H] = cb
            self.w2s[e * s2:(e + 1) * s2] = sb
            # the library's quantisation of the same bytes
            assert torch.equal(self.W.w13_codes[e * 2 * I:(e + 1) * 2 * I].cpu(), ca)
            assert torch.equal(self.W.w13_sf[e * s13:(e + 1) * s13].cpu(), sa)
            assert torch.equal(self.W.w2_codes[e * H:(e + 1) * H].cpu(), cb)
            assert torch.equal(self.W.w2_sf[e * s2:(e + 1) * s2].cpu(), sb)
            self.done.add(e)


@pytest.fixture(scope="module")
def layer(nv):
    case = synthdata.moe_case(16, E, H, I, TOPK, CFG["skewed"], seed=0, device=DEV)
    W = nv.quantize_moe_weights(lambda e: case.w13(e, DEV), lambda e: case.w2(e, DEV), E, H, I, DEV)
    ow = OracleWeights(case, W)
    ow.need(range(CALIB_EXPERTS))
    x_calib = case.x_calib.cpu()
    g_a1 = oracle.global_scale(x_calib)
    a13_cal = [oracle.alpha_w4a4(g_a1, ow.g13[e]) for e in range(CALIB_EXPERTS)]
    amax = oracle.moe_h_amax(x_calib[:CALIB_ROWS].contiguous(), g_a1, ow.w13c[:CALIB_EXPERTS * 2 * I],
                             ow.w13s[:CALIB_EXPERTS * oracle.scale_bytes(2 * I, H)], a13_cal, CALIB_EXPERTS, H, I)
    g_a2 = max(oracle.global_from_amax(float(v)) for v in amax)
    g_a1_dev = nv.nvfp4_compute_global(case.x_calib)
    assert np.float32(g_a1_dev.item()) == np.float32(g_a1)
    a13_dev = nv.nvfp4_make_alpha(g_a1_dev, W.g13)
    g_a2_dev = torch.tensor([g_a2], dtype=torch.float32, device=DEV)
    a2_dev = nv.nvfp4_make_alpha(g_a2_dev, W.g2)
    return dict(W=W, ow=ow, g_a1=g_a1, g_a2=g_a2, g_a1_dev=g_a1_dev, a13_dev=a13_dev, g_a2_dev=g_a2_dev,
                a2_dev=a2_dev)


def pick_tokens(ids: torch.Tensor, seed: int):
    """Tokens in a seeded order, kept while the union of their experts stays
    within MAX_EXPERTS; always the first token of that order."""
    T = ids.shape[0]
    order = np.random.default_rng(seed).permutation(T)
    union, tokens = set(), []
    for t in order:
        ex = set(ids[t].tolist())
        if len(union | ex) <= MAX_EXPERTS or not tokens:
            union |= ex
            tokens.append(int(t))
            if len(tokens) == MAX_TOKENS:
                break
    return sorted(tokens), sorted(union)


@pytest.mark.parametrize("T", CFG["tokens"])
def test_moe_large_sampled_tokens(nv, layer, T):
    L = layer
    case = synthdata.moe_case(T, E, H, I, TOPK, CFG["skewed"], seed=0, device=DEV)
    ws = torch.empty(nv.nvfp4_moe_workspace(T, H, I, E, TOPK), dtype=torch.uint8, device=DEV)
    out = nv.nvfp4_moe_w4a4(case.x, case.topk_ids, case.topk_w, L["g_a1_dev"], L["W"].w13_codes, L["W"].w13_sf,
                            L["a13_dev"], L["g_a2_dev"], L["W"].w2_codes, L["W"].w2_sf, L["a2_dev"], E, I,
                            workspace=ws)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status() == 0
    ids_cpu = case.topk_ids.cpu()
    tokens, experts = pick_tokens(ids_cpu, T)
    assert len(tokens) >= 8, f"only {len(tokens)} tokens fit the expert budget"
    ow = L["ow"]
    ow.need(experts)
    a13 = [oracle.alpha_w4a4(L["g_a1"], g) for g in ow.g13]
    a2 = [oracle.alpha_w4a4(L["g_a2"], g) for g in ow.g2]
    ref = oracle.moe_w4a4(case.x.cpu()[tokens].contiguous(), ids_cpu[tokens].contiguous(),
                          case.topk_w.cpu()[tokens].contiguous(), L["g_a1"], ow.w13c, ow.w13s, a13, L["g_a2"],
                          ow.w2c, ow.w2s, a2, E, H, I)
    check_close(out.cpu()[tokens], ref, f"large MoE T={T} sampled ({len(tokens)} tokens, {len(experts)} experts)")
