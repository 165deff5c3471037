"""Seeded synthetic inputs for the BitLinear forward workloads.

This module only draws random tensors with the shapes and value
distributions of the workloads below; it contains none of the method's
arithmetic, so both the CUDA path's tests and the CPU oracle can be fed from
it.  Every tensor is drawn from a ``torch.Generator`` with a fixed seed on the
requested device (CPU for oracle-sized cases, CUDA for full-size runs, where a
CPU draw of billions of values would take minutes).

Workloads (shapes of a ~2B and a ~100B ternary LLM's projections; the ~2B
model's FFN uses squared ReLU, so the down projection's input is relu(z)^2):

  tiny            W fp32 [256, 512] ~ N(0, 0.02); x fp32 [4, 512] ~ N(0, 1) with
                  channel 7 scaled x20 (an outlier channel); seed 0.
  decode_2b       M = 1; per layer QKV 2560->3840, O 2560->2560, up 2560->6912,
                  down 6912->2560; W ~ N(0, 0.02); 30 layers with distinct
                  weights (388 MB packed, far beyond the 126 MB L2);
                  x bf16 ~ N(0, 1) (down: relu(z)^2).
  decode_2b_batch same weights, M in {8, 16, 32, 64}; x bf16 ~ N(0, 1) with
                  round(0.01 K) fixed seeded channels scaled x10.
  prefill_2b      M = 2048; up 2560->6912 with x ~ N(0, 1); down 6912->2560 with
                  x = relu(z)^2 (about half zeros); W ~ N(0, 0.02).
  decode_100b     M in {1, 8}; 8192->28672 and 28672->8192, W ~ N(0, 0.01);
                  80 layers' packed weights resident (9.4 GB).

Seeds: 1000 * workload_id + 10 * layer + matrix_index (workload ids 1..5 in
the order above); activations use the same rule plus 500.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

WORKLOAD_IDS = {"tiny": 1, "decode_2b": 2, "decode_2b_batch": 3,
                "prefill_2b": 4, "decode_100b": 5}

# (name, N, K, x-kind) of the ~2B model's four projections per layer.
PROJ_2B = (("qkv", 3840, 2560, "normal"),
           ("o", 2560, 2560, "normal"),
           ("up", 6912, 2560, "normal"),
           ("down", 2560, 6912, "relu2"))
PROJ_100B = (("up", 28672, 8192, "normal"),
             ("down", 8192, 28672, "normal"))


@dataclass(frozen=True)
class Matrix:
    name: str
    layer: int
    index: int
    N: int
    K: int
    std: float
    x_kind: str
    seed: int


def weight_seed(workload: str, layer: int, index: int) -> int:
    return 1000 * WORKLOAD_IDS[workload] + 10 * layer + index


def act_seed(workload: str, layer: int, index: int) -> int:
    return weight_seed(workload, layer, index) + 500


def matrices(workload: str, layers: int | None = None) -> list[Matrix]:
    """The weight matrices of a workload, in sweep order."""
    if workload == "tiny":
        return [Matrix("tiny", 0, 0, 256, 512, 0.02, "outlier7", 0)]
    if workload in ("decode_2b", "decode_2b_batch", "prefill_2b"):
        L = 30 if layers is None else layers
        base = "decode_2b"  # one set of weights serves all ~2B workloads
        out = []
        for layer in range(L):
            for i, (nm, N, K, xk) in enumerate(PROJ_2B):
                out.append(Matrix(nm, layer, i, N, K, 0.02, xk,
                                  weight_seed(base, layer, i)))
        return out
    if workload == "decode_100b":
        L = 80 if layers is None else layers
        return [Matrix(nm, layer, i, N, K, 0.01, xk,
                       weight_seed(workload, layer, i))
                for layer in range(L) for i, (nm, N, K, xk) in enumerate(PROJ_100B)]
    raise KeyError(workload)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def weight(N: int, K: int, std: float, seed: int, device="cpu",
           dtype=torch.float32) -> torch.Tensor:
    """W ~ N(0, std^2), [N, K], drawn in fp32 then cast to ``dtype``."""
    g = _gen(seed, device)
    w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32)
    w.mul_(std)
    return w.to(dtype)


def activations(M: int, K: int, kind: str, seed: int, device="cpu",
                dtype=torch.bfloat16) -> torch.Tensor:
    """Synthetic activations [M, K].

    kind: "normal"      N(0, 1)
          "outlier7"    N(0, 1), channel 7 scaled by 20
          "outliers1pct" N(0, 1), round(0.01 K) seeded channels scaled by 10
          "relu2"       relu(z)^2 with z ~ N(0, 1) (about half exact zeros)
          "zeros"       all zero
    """
    g = _gen(seed, device)
    if kind == "zeros":
        return torch.zeros((M, K), device=device, dtype=dtype)
    z = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if kind == "normal":
        pass
    elif kind == "outlier7":
        if K > 7:
            z[:, 7] *= 20.0
    elif kind == "outliers1pct":
        n_out = max(1, round(0.01 * K))
        gc = _gen(seed + 7, "cpu")
        ch = torch.randperm(K, generator=gc)[:n_out].to(device)
        z[:, ch] *= 10.0
    elif kind == "relu2":
        z = torch.clamp_min(z, 0.0).square()
    else:
        raise KeyError(kind)
    return z.to(dtype)


def rms_gain(K: int, seed: int, device="cpu") -> torch.Tensor:
    """A positive RMSNorm gain vector around 1 (fp32 [K])."""
    g = _gen(seed, device)
    return 1.0 + 0.1 * torch.rand((K,), generator=g, device=device,
                                  dtype=torch.float32)
