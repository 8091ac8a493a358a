"""GPU parity of the MoE alignment (the stable counting sort of the routes by
expert, segments padded to 128-row tiles) against the oracle, bit-exact, over
route counts that take the one-block path and the chunked path (one chunk,
many chunks, the largest chunks, a ragged last chunk), expert counts from 1 to
1024, skewed routing, and both segment paddings (128 rows, and 256 rows where
the experts average 1024 routes and the grouped GEMMs run on CTA pairs).  The layer runs on placeholder weights: only the
layout in the workspace is compared, with pos (route -> permuted row) checked
as the inverse of row_map."""
import pytest
import torch

import oracle
import synthdata

pytestmark = pytest.mark.gpu
DEV = "cuda"
I = 128


@pytest.fixture(scope="module", autouse=True)
def nv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_block_scaled_act_gb300 import build
    build.build()
    import nvfp4_block_scaled_act_gb300 as m
    m.load_library()
    return m


def placeholder_weights(nv, E, H):
    """Codes of zero and unit scales (E4M3 0x38 = 1.0): every product is 0."""
    w13c = torch.zeros(E * 2 * I, H // 2, dtype=torch.uint8, device=DEV)
    w13s = torch.full((E * nv.nvfp4_scale_bytes(2 * I, H),), 0x38, dtype=torch.uint8, device=DEV)
    w2c = torch.zeros(E * H, I // 2, dtype=torch.uint8, device=DEV)
    w2s = torch.full((E * nv.nvfp4_scale_bytes(H, I),), 0x38, dtype=torch.uint8, device=DEV)
    return w13c, w13s, w2c, w2s


def ws_field(nv, ws, lay, name, count):
    off = getattr(lay, name)
    return ws[off:off + 4 * count].view(torch.int32).cpu()


@pytest.mark.parametrize("T,topk,E,skewed,H", [
    (512, 8, 8, False, 128),      # 4096 routes: the one-block path at its limit
    (2048, 2, 2, False, 256),     # the same with 2048 routes per expert: padded to 256
    (600, 8, 8, False, 128),      # just above it: 19 chunks of 256, ragged tail
    (4097, 1, 5, True, 128),      # 17 chunks, the last holding one route
    (4097, 2, 4, True, 256),      # ... 2048 routes per expert: padded to 256
    (4096, 8, 128, False, 128),   # 128 chunks, 8 runs per expert column
    (5000, 1, 1, False, 256),     # one expert: more runs than chunks, padded to 256
    (3001, 3, 1024, True, 128),   # 1024 experts: one run per column
    (3000, 4, 1000, False, 128),  # expert count not dividing the block
    (32768, 8, 256, True, 256),   # 512 chunks of 512 routes, 1024 per expert: padded to 256
    (175001, 3, 3, True, 256),    # 2048-route chunks, 257 of them
])
def test_align_layout_exact(nv, T, topk, E, skewed, H):
    assert topk <= E
    ids, w = synthdata.routing(T, E, topk, seed=T + E, skewed=skewed)
    x = synthdata.activations(T, H, seed=1).to(torch.bfloat16)
    w13c, w13s, w2c, w2s = placeholder_weights(nv, E, H)
    one = torch.ones(1, dtype=torch.float32, device=DEV)
    alphas = torch.ones(E, dtype=torch.float32, device=DEV)
    ws = torch.empty(nv.nvfp4_moe_workspace(T, H, I, E, topk), dtype=torch.uint8, device=DEV)
    out = nv.nvfp4_moe_w4a4(x.to(DEV), ids.to(DEV), w.to(DEV), one, w13c, w13s, alphas, one, w2c, w2s, alphas,
                            E, I, workspace=ws)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status() == 0
    assert torch.count_nonzero(out).item() == 0

    lay = nv.nvfp4_moe_workspace_layout(T, H, I, E, topk)
    bm = int(lay.row_block)
    assert bm == (256 if T * topk >= 1024 * E and H % 256 == 0 else 128)
    ref = oracle.moe_align(ids, E, bm)
    P = ref["P"]
    assert torch.equal(ws_field(nv, ws, lay, "counts", E), ref["counts"])
    assert torch.equal(ws_field(nv, ws, lay, "offsets", E + 1), ref["offsets"])
    assert int(ws_field(nv, ws, lay, "n_tiles", 1)[0]) == P // 128
    row_map = ws_field(nv, ws, lay, "row_map", P)
    assert torch.equal(row_map, ref["row_map"])
    # one entry per 128-row tile on the device; the oracle has one per bm-row tile
    assert torch.equal(ws_field(nv, ws, lay, "tile_expert", P // 128),
                       ref["tile_expert"].repeat_interleave(bm // 128))
    pos = ws_field(nv, ws, lay, "pos", T * topk)
    real = (row_map >= 0).nonzero().flatten()
    assert real.numel() == T * topk
    assert torch.equal(pos[row_map[real].long()], real.to(torch.int32))
