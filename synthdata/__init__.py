"""Seeded synthetic inputs for the NVFP4 linear and MoE workloads.

This module only draws random tensors and routing decisions.  It holds none of
the NVFP4 arithmetic (no global scale, no block scale, no rounding to e2m1 or
E4M3): both the CPU oracle and the CUDA library receive the bf16 tensors made
here and quantise them on their own.

Recipes (the workloads of the pages "run nvfp4 linears on nvfp4 activations on
sm_120" and the W4A4 MoE prefill page, restated as synthetic inputs):

* weights: bf16 draws from N(0, 0.02);
* activations: bf16 draws from N(0, 1) where one per cent of the channels
  (``floor(0.01 * K)`` channel ids taken from a seeded permutation) are scaled
  by 20, the same channel ids in the calibration batch and the runtime batch;
* calibration batch: 64 rows from the activation distribution, own seed;
* MoE routing: logits from N(0, 1) (plus a per-expert bias from N(0, 1) for the
  skewed router), the top-k logits chosen (ties go to the lower expert id),
  softmax over the chosen k in fp32; the weights then sum to one, so the
  renormalisation the workload names changes nothing.

Every draw uses a ``torch.Generator`` seeded from ``(seed, stream)``, on the
device the caller names, so that large weights can be drawn on the GPU and
copied to the host for the oracle.  The same call on the same device returns
the same tensor.
"""
from __future__ import annotations

import dataclasses
import math

import torch

CALIB_ROWS = 64
OUTLIER_FRACTION = 0.01
OUTLIER_GAIN = 20.0
WEIGHT_STD = 0.02

# stream ids keep independent draws apart for one seed
_S_WEIGHT, _S_ACT, _S_CALIB, _S_OUTLIER, _S_LOGIT, _S_BIAS, _S_W13, _S_W2 = range(8)


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + stream * 7919 + 12345) % (2**63 - 1))
    return g


def outlier_channels(K: int, seed: int = 0) -> torch.Tensor:
    """``floor(0.01 * K)`` channel ids from a seeded permutation (int64, sorted)."""
    n = int(math.floor(OUTLIER_FRACTION * K))
    perm = torch.randperm(K, generator=_gen(seed, _S_OUTLIER, "cpu"))
    return torch.sort(perm[:n]).values


def weights(rows: int, K: int, seed: int = 0, stream: int = _S_WEIGHT,
            device="cpu", std: float = WEIGHT_STD) -> torch.Tensor:
    """bf16 ``[rows, K]`` from N(0, std)."""
    w = torch.randn(rows, K, generator=_gen(seed, stream, device), device=device,
                    dtype=torch.float32)
    return (w * std).to(torch.bfloat16)


def activations(rows: int, K: int, seed: int = 0, stream: int = _S_ACT,
                device="cpu", outliers: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 ``[rows, K]`` from N(0, 1) with the outlier channels scaled by 20."""
    x = torch.randn(rows, K, generator=_gen(seed, stream, device), device=device,
                    dtype=torch.float32)
    if outliers is None:
        outliers = outlier_channels(K, seed)
    if outliers.numel():
        x[:, outliers.to(x.device)] *= OUTLIER_GAIN
    return x.to(torch.bfloat16)


def calibration_batch(K: int, seed: int = 0, device="cpu",
                      outliers: torch.Tensor | None = None) -> torch.Tensor:
    """The 64-row calibration batch, from the activation distribution."""
    return activations(CALIB_ROWS, K, seed, _S_CALIB, device, outliers)


def routing(T: int, E: int, topk: int, seed: int = 0, skewed: bool = False,
            device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """Top-k routing: int32 ids ``[T, topk]`` and fp32 weights ``[T, topk]``.

    Logits ~ N(0, 1); with ``skewed`` a per-expert bias ~ N(0, 1) is added.
    The k largest logits are taken, ties broken towards the lower expert id,
    and the weights are a softmax over those k logits.
    """
    logits = torch.randn(T, E, generator=_gen(seed, _S_LOGIT, device), device=device,
                         dtype=torch.float32)
    if skewed:
        bias = torch.randn(E, generator=_gen(seed, _S_BIAS, device), device=device,
                           dtype=torch.float32)
        logits = logits + bias
    # stable descending sort: equal logits keep ascending expert order
    order = torch.sort(logits, dim=1, descending=True, stable=True).indices[:, :topk]
    chosen = torch.gather(logits, 1, order)
    w = torch.softmax(chosen, dim=1)
    return order.to(torch.int32).contiguous(), w.contiguous()


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class LinearCase:
    """bf16 inputs of one NVFP4 linear: weight parts, activations, calibration."""
    w_parts: list          # list of bf16 [N_p, K]
    x: torch.Tensor        # bf16 [M, K]
    x_calib: torch.Tensor  # bf16 [64, K]
    K: int

    @property
    def N(self) -> int:
        return sum(int(p.shape[0]) for p in self.w_parts)


def linear_case(M: int, N_parts, K: int, seed: int = 0, device="cpu") -> LinearCase:
    """One linear: ``N_parts`` rows per weight part (a fused weight has several)."""
    if isinstance(N_parts, int):
        N_parts = [N_parts]
    out = outlier_channels(K, seed)
    parts = [weights(n, K, seed, 100 + i, device) for i, n in enumerate(N_parts)]
    x = activations(M, K, seed, _S_ACT, device, out)
    xc = calibration_batch(K, seed, device, out)
    return LinearCase(parts, x, xc, K)


def tiny_linear(seed: int = 0, device="cpu") -> LinearCase:
    """Tiny W4A4 linear: M = 8, N = 256, K = 512."""
    return linear_case(8, 256, 512, seed, device)


DECODE_SHAPES = [(8704, 5120), (5120, 4352)]
DECODE_TOKENS = [1, 2, 4, 8, 16]


def decode_case(T: int, N: int, K: int, seed: int = 0, device="cpu") -> LinearCase:
    """W4A16 decode linear: T bf16 rows against an NVFP4 weight [N, K]."""
    return linear_case(T, N, K, seed, device)


QKV_PARTS = [5120, 1024, 1024]
QKV_K = 5120
PREFILL_M = [512, 1024, 2048, 4096, 8192]


def prefill_case(M: int, seed: int = 0, device="cpu") -> LinearCase:
    """Fused qkv-style W4A4 prefill linear (N = 5120 + 1024 + 1024, K = 5120)."""
    return linear_case(M, QKV_PARTS, QKV_K, seed, device)


@dataclasses.dataclass
class MoECase:
    """bf16 inputs of one MoE layer."""
    x: torch.Tensor         # bf16 [T, H]
    x_calib: torch.Tensor   # bf16 [64, H]
    topk_ids: torch.Tensor  # int32 [T, topk]
    topk_w: torch.Tensor    # fp32 [T, topk]
    E: int
    H: int
    I: int
    topk: int
    seed: int
    device: object

    def w13(self, e: int, device=None) -> torch.Tensor:
        """bf16 ``[2I, H]`` of expert e: rows [0, I) gate, rows [I, 2I) up."""
        return weights(2 * self.I, self.H, self.seed * 4096 + e, _S_W13,
                       device or self.device)

    def w2(self, e: int, device=None) -> torch.Tensor:
        """bf16 ``[H, I]`` of expert e (down projection)."""
        return weights(self.H, self.I, self.seed * 4096 + e, _S_W2, device or self.device)


MOE_SMALL = dict(E=128, topk=8, H=2048, I=768, skewed=False, tokens=[16, 128, 1024, 4096, 8192])
MOE_LARGE = dict(E=256, topk=8, H=7168, I=2048, skewed=True, tokens=[1024, 8192, 32768])


def moe_case(T: int, E: int, H: int, I: int, topk: int = 8, skewed: bool = False,
             seed: int = 0, device="cpu") -> MoECase:
    out = outlier_channels(H, seed)
    x = activations(T, H, seed, _S_ACT, device, out)
    xc = calibration_batch(H, seed, device, out)
    ids, w = routing(T, E, topk, seed, skewed, device)
    return MoECase(x, xc, ids, w, E, H, I, topk, seed, device)
