"""Parity helpers shared by the GPU tests: the tolerance of the GEMM and MoE
outputs against the oracle (rel-L2 <= 1e-3 over the whole tensor, fp64 norms,
and max |err| <= 2 bf16 ulp of the row's largest oracle output; an all-zero
oracle row must be exactly zero)."""
import torch

REL_L2 = 1e-3
ULPS = 2.0


def bf16_ulp_of_rowmax(ref: torch.Tensor) -> torch.Tensor:
    rowmax = ref.abs().amax(dim=-1, keepdim=True)
    return torch.pow(2.0, torch.floor(torch.log2(rowmax.clamp_min(1e-300))) - 7)


def check_close(got: torch.Tensor, ref: torch.Tensor, what: str = "", ulps: float = ULPS,
                rel_l2: float = REL_L2):
    g = got.detach().float().cpu().double()
    r = ref.detach().float().cpu().double()
    assert g.shape == r.shape, (g.shape, r.shape)
    assert torch.isfinite(g).all(), f"{what}: non-finite output"
    err = (g - r).abs()
    denom = r.norm().item()
    rel = (g - r).norm().item() / denom if denom > 0 else (g.norm().item())
    ulp = bf16_ulp_of_rowmax(r)
    zero_rows = r.abs().amax(dim=-1) == 0
    bad = err > ulps * ulp
    bad[zero_rows] = err[zero_rows] > 0
    assert rel <= rel_l2, f"{what}: rel-L2 {rel:.3e} > {rel_l2}"
    assert not bool(bad.any()), (f"{what}: {int(bad.sum())} elements beyond {ulps} bf16 ulp of the row max; "
                                 f"worst err {float(err.max()):.3e}")
    return rel, float((err / ulp).max())
