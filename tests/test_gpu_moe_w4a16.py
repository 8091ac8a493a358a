"""GPU parity of the W4A16 MoE layer for small batches against the oracle.

The layer keeps the activations in bf16 (no activation global): gate_up in
fp32, h = bf16(silu(a13 G) * (a13 U)), down in fp32 with the routing weight,
the top-k sum in fp32 in slot order, bf16 out.  The kernels' fp32 accumulation
order differs from the oracle's, so the output is compared within rel-L2 <=
1e-3 and 2 bf16 ulp of the row max.

Cases: the MoE workload of the pages (E = 128, H = 2048, I = 768, top-8) at
T = 1, 2, 4, 8, 16 and 64; duplicate and invalid expert ids; every route of
20 tokens on one expert (more routes per expert than one pass of the kernel
holds); top-1; repeatability; and the large workload (E = 256, H = 7168,
I = 2048, skewed router) at T = 1 and 4, whose touched experts the oracle
quantises on its own (bit-exact against the library's quantisation)."""
import numpy as np
import pytest
import torch

import oracle
import synthdata
from parity import check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
S = synthdata.MOE_SMALL
L = synthdata.MOE_LARGE


@pytest.fixture(scope="module")
def nv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_block_scaled_act_gb300 import build
    build.build()
    import nvfp4_block_scaled_act_gb300 as m
    m.load_library()
    return m


class Bank:
    """Expert weights of one workload: the library's quantisation on the GPU
    and the oracle's, of the same bf16 bytes, for the experts in `need`."""

    def __init__(self, nv, E, H, I, skewed, eager):
        self.E, self.H, self.I = E, H, I
        self.case0 = synthdata.moe_case(1, E, H, I, 8, skewed, seed=0, device=DEV)
        self.W = nv.quantize_moe_weights(lambda e: self.case0.w13(e, DEV), lambda e: self.case0.w2(e, DEV),
                                         E, H, I, DEV)
        self.a13_dev = nv.nvfp4_make_alpha(None, self.W.g13)
        self.a2_dev = nv.nvfp4_make_alpha(None, self.W.g2)
        self.w13c = torch.zeros(E * 2 * I, H // 2, dtype=torch.uint8)
        self.w13s = torch.zeros(E * oracle.scale_bytes(2 * I, H), dtype=torch.uint8)
        self.w2c = torch.zeros(E * H, I // 2, dtype=torch.uint8)
        self.w2s = torch.zeros(E * oracle.scale_bytes(H, I), dtype=torch.uint8)
        self.g13 = [1.0] * E
        self.g2 = [1.0] * E
        self.done = set()
        if eager:
            self.need(range(E))

    def need(self, experts):
        E, H, I = self.E, self.H, self.I
        s13, s2 = oracle.scale_bytes(2 * I, H), oracle.scale_bytes(H, I)
        for e in sorted(set(int(v) for v in experts) - self.done):
            if e < 0 or e >= E:
                continue
            a = self.case0.w13(e, DEV).cpu()
            b = self.case0.w2(e, DEV).cpu()
            self.g13[e], self.g2[e] = oracle.global_scale(a), oracle.global_scale(b)
            ca, sa = oracle.quantize(a, self.g13[e])
            cb, sb = oracle.quantize(b, self.g2[e])
            self.w13c[e * 2 * I:(e + 1) * 2 * I] = ca
            self.w13s[e * s13:(e + 1) * s13] = sa
            self.w2c[e * H:(e + 1) * H] = cb
            self.w2s[e * s2:(e + 1) * s2] = sb
            assert torch.equal(self.W.w13_codes[e * 2 * I:(e + 1) * 2 * I].cpu(), ca)
            assert torch.equal(self.W.w13_sf[e * s13:(e + 1) * s13].cpu(), sa)
            assert torch.equal(self.W.w2_codes[e * H:(e + 1) * H].cpu(), cb)
            assert torch.equal(self.W.w2_sf[e * s2:(e + 1) * s2].cpu(), sb)
            self.done.add(e)
        a13, a2 = self.a13_dev.cpu().numpy(), self.a2_dev.cpu().numpy()
        for e in self.done:
            assert a13[e] == np.float32(oracle.alpha_w4a16(self.g13[e]))
            assert a2[e] == np.float32(oracle.alpha_w4a16(self.g2[e]))

    def gpu(self, nv, x, ids, w):
        T, topk = ids.shape
        ws = torch.empty(max(nv.nvfp4_moe_w4a16_workspace(T, self.H, self.I, self.E, topk), 1), dtype=torch.uint8,
                         device=DEV)
        out = nv.nvfp4_moe_w4a16(x.to(DEV), ids.to(DEV), w.to(DEV), self.W.w13_codes, self.W.w13_sf, self.a13_dev,
                                 self.W.w2_codes, self.W.w2_sf, self.a2_dev, self.E, self.I, workspace=ws)
        torch.cuda.synchronize()
        return out

    def ref(self, x, ids, w):
        self.need(ids.flatten().tolist())
        a13 = [oracle.alpha_w4a16(g) for g in self.g13]
        a2 = [oracle.alpha_w4a16(g) for g in self.g2]
        return oracle.moe_w4a16(x.cpu(), ids.cpu(), w.cpu(), self.w13c, self.w13s, a13, self.w2c, self.w2s, a2,
                                self.E, self.H, self.I)


@pytest.fixture(scope="module")
def small(nv):
    return Bank(nv, S["E"], S["H"], S["I"], S["skewed"], eager=True)


@pytest.mark.parametrize("T", [1, 2, 4, 8, 16, 64])
def test_moe_w4a16_small_batches(nv, small, T):
    c = synthdata.moe_case(T, S["E"], S["H"], S["I"], S["topk"], S["skewed"], seed=T, device="cpu")
    out = small.gpu(nv, c.x, c.topk_ids, c.topk_w)
    assert nv.nvfp4_device_status() == 0
    check_close(out.cpu(), small.ref(c.x, c.topk_ids, c.topk_w), f"W4A16 MoE T={T}")


def test_moe_w4a16_duplicate_and_invalid_ids(nv, small):
    c = synthdata.moe_case(6, S["E"], S["H"], S["I"], S["topk"], S["skewed"], seed=11, device="cpu")
    ids = c.topk_ids.clone()
    ids[0, 1] = ids[0, 0]     # the same expert twice for one token
    ids[1, :] = 5             # every slot of a token on one expert
    ids[2, 3] = -1            # dropped
    ids[3, 7] = S["E"]        # dropped
    out = small.gpu(nv, c.x, ids, c.topk_w)
    assert nv.nvfp4_device_status() == 7  # NVFP4_ERR_BAD_EXPERT_ID
    check_close(out.cpu(), small.ref(c.x, ids, c.topk_w), "W4A16 MoE duplicate / invalid ids")


def test_moe_w4a16_unrouted_token_and_dirty_workspace(nv, small):
    """A token whose ids are all invalid gets a zero row; the workspace needs
    no initialisation, so calls that reuse one workspace filled with 0xFF
    agree bit for bit; and every output element is written (out starts as
    NaN)."""
    c = synthdata.moe_case(6, S["E"], S["H"], S["I"], S["topk"], S["skewed"], seed=14, device="cpu")
    ids = c.topk_ids.clone()
    ids[4, :] = -1            # no valid route
    ids[5, 2:] = S["E"]       # two valid routes of eight
    T, topk = ids.shape
    ws = torch.full((nv.nvfp4_moe_w4a16_workspace(T, S["H"], S["I"], S["E"], topk),), 0xFF, dtype=torch.uint8,
                    device=DEV)
    outs = []
    for i in range(3):
        out = torch.full((T, S["H"]), float("nan"), dtype=torch.bfloat16, device=DEV)
        nv.nvfp4_moe_w4a16(c.x.to(DEV), ids.to(DEV), c.topk_w.to(DEV), small.W.w13_codes, small.W.w13_sf,
                           small.a13_dev, small.W.w2_codes, small.W.w2_sf, small.a2_dev, S["E"], S["I"], out=out,
                           workspace=ws)
        assert nv.nvfp4_device_status() == 7  # NVFP4_ERR_BAD_EXPERT_ID, raised by every call
        outs.append(out)
    assert not torch.isnan(outs[0]).any()
    assert torch.count_nonzero(outs[0][4]).item() == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0]), "W4A16 MoE calls on a reused workspace differ"
    check_close(outs[0].cpu(), small.ref(c.x, ids, c.topk_w), "W4A16 MoE unrouted token")


def test_moe_w4a16_one_expert_for_all_routes(nv, small):
    """160 routes on one expert: more than one pass of 16 input rows."""
    c = synthdata.moe_case(20, S["E"], S["H"], S["I"], S["topk"], S["skewed"], seed=12, device="cpu")
    ids = torch.full_like(c.topk_ids, 3)
    out = small.gpu(nv, c.x, ids, c.topk_w)
    assert nv.nvfp4_device_status() == 0
    check_close(out.cpu(), small.ref(c.x, ids, c.topk_w), "W4A16 MoE one expert")


@pytest.mark.parametrize("T", [4, 16, 64])
def test_moe_w4a16_bitwise_repeatable(nv, small, T):
    """The same call gives the same bits every time: every sum has a fixed
    order, and a weight-ring slot is refilled only after the reads of the
    previous block are complete (the large-workload case below too)."""
    c = synthdata.moe_case(T, S["E"], S["H"], S["I"], S["topk"], S["skewed"], seed=40 + T, device=DEV)
    runs = [small.gpu(nv, c.x, c.topk_ids, c.topk_w) for _ in range(6)]
    for r in runs[1:]:
        assert torch.equal(r, runs[0]), f"W4A16 MoE T={T} is not repeatable"


def test_moe_w4a16_top1_and_repeatable(nv, small):
    c = synthdata.moe_case(5, S["E"], S["H"], S["I"], 1, S["skewed"], seed=13, device="cpu")
    a = small.gpu(nv, c.x, c.topk_ids, c.topk_w)
    b = small.gpu(nv, c.x, c.topk_ids, c.topk_w)
    assert torch.equal(a, b), "W4A16 MoE is not repeatable"
    check_close(a.cpu(), small.ref(c.x, c.topk_ids, c.topk_w), "W4A16 MoE top-1")


def test_moe_w4a16_zero_tokens_and_bad_shapes(nv, small):
    x = torch.empty(0, S["H"], dtype=torch.bfloat16, device=DEV)
    ids = torch.empty(0, 8, dtype=torch.int32, device=DEV)
    w = torch.empty(0, 8, dtype=torch.float32, device=DEV)
    out = nv.nvfp4_moe_w4a16(x, ids, w, small.W.w13_codes, small.W.w13_sf, small.a13_dev, small.W.w2_codes,
                             small.W.w2_sf, small.a2_dev, S["E"], S["I"])
    assert out.shape == (0, S["H"])
    assert nv.nvfp4_moe_w4a16_workspace(65, S["H"], S["I"], S["E"], 8) == 0   # T > 64: the W4A4 path's regime
    assert nv.nvfp4_moe_w4a16_workspace(4, S["H"], S["I"], S["E"], 9) == 0    # topk > 8


@pytest.mark.parametrize("E,topk,T", [(1, 1, 20), (2, 2, 3), (3, 2, 64)])
def test_moe_w4a16_smallest_shapes(nv, E, topk, T):
    """H = I = 128 (one 128-k block per GEMV; gate_up items of 64 gate + 64 up
    rows are the whole expert), every route on one or two experts, and more
    routes per expert than one pass of route rows holds."""
    bank = Bank(nv, E, 128, 128, False, eager=True)
    c = synthdata.moe_case(T, E, 128, 128, topk, False, seed=50 + E, device="cpu")
    out = bank.gpu(nv, c.x, c.topk_ids, c.topk_w)
    assert nv.nvfp4_device_status() == 0
    check_close(out.cpu(), bank.ref(c.x, c.topk_ids, c.topk_w), f"W4A16 MoE E={E} top-{topk} T={T}")


@pytest.fixture(scope="module")
def large(nv):
    return Bank(nv, L["E"], L["H"], L["I"], L["skewed"], eager=False)


@pytest.mark.parametrize("T", [1, 4])
def test_moe_w4a16_large_workload(nv, large, T):
    bank = large
    c = synthdata.moe_case(T, L["E"], L["H"], L["I"], L["topk"], L["skewed"], seed=T, device="cpu")
    out = bank.gpu(nv, c.x, c.topk_ids, c.topk_w)
    assert nv.nvfp4_device_status() == 0
    check_close(out.cpu(), bank.ref(c.x, c.topk_ids, c.topk_w), f"W4A16 MoE large T={T}")
    for _ in range(5):
        assert torch.equal(bank.gpu(nv, c.x, c.topk_ids, c.topk_w), out), f"W4A16 MoE large T={T} is not repeatable"


def test_moe_w4a16_large_workload_repeatable(nv, large):
    c = synthdata.moe_case(16, L["E"], L["H"], L["I"], L["topk"], L["skewed"], seed=16, device="cpu")
    runs = [large.gpu(nv, c.x, c.topk_ids, c.topk_w) for _ in range(6)]
    assert nv.nvfp4_device_status() == 0
    for r in runs[1:]:
        assert torch.equal(r, runs[0]), "W4A16 MoE large T=16 is not repeatable"
