"""Seeded synthetic inputs for the quantized linear layer.

Shared by the tests, the CPU oracle's callers and the benchmark: this module
only makes inputs.  It holds none of the layer's arithmetic (no weight decode,
no products, no sums); the quantizers below are input preparation -- the layer
consumes weights that are already quantized -- and use torch's own
float32 -> float8_e4m3fn cast for every E4M3 code they produce.

Recipes (all seeded; with seed s the weight uses s, the activations s + 1, the
MoE routing s + 2):

* activations: x ~ N(0, 1) rounded to bfloat16;
* FP8 weight: W ~ N(0, 0.02) in float32, per-tensor scale s = absmax(W) / 448,
  codes = e4m3(clamp(W / s, -448, 448)) with torch's round-to-nearest-even cast;
* NVFP4 weight: W ~ N(0, 0.02), per-tensor second scale s2 = absmax / (448 * 6),
  per 16-element block the E4M3 scale e4m3(blockabsmax / (6 * s2)), elements
  e2m1(W / (s2 * block_scale)) rounded to nearest with ties to the even code
  (0 when the block scale is 0), packed two per byte with the low nibble first;
* MoE routing: ``total_rows`` draws from the 9 categories (experts 0..7 and one
  inactive category) with weights [1, 1, 1, 0, 1, 1, 1, 1, 0.5] and
  replacement, sorted; group z holds the rows of category z, expert_ids are
  [0, .., 7, -1], so expert 3's group is empty and the last group writes zeros.

Generation runs on the CPU generator by default so that the same seed gives the
same bytes everywhere; ``device`` moves the results.
"""

from __future__ import annotations

import torch

FP8_MAX = 448.0
E2M1_MAX = 6.0
ROUTING_WEIGHTS = (1.0, 1.0, 1.0, 0.0, 1.0, 1.0, 1.0, 1.0, 0.5)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def gaussian(shape, std: float, seed: int) -> torch.Tensor:
    """float32 N(0, std^2) on the CPU, seeded."""
    return torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32) * std


def bf16_activations(m: int, k: int, seed: int = 1, device="cpu") -> torch.Tensor:
    """bf16 [m, k] with x ~ N(0, 1)."""
    return gaussian((m, k), 1.0, seed).to(torch.bfloat16).to(device)


def e4m3_codes(v: torch.Tensor) -> torch.Tensor:
    """float32 -> float8_e4m3fn codes (uint8), saturating at +-448, RNE."""
    return v.clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def fp8_weight(n: int, k: int, seed: int = 0, device="cpu"):
    """(codes uint8 [n, k], scale float): W ~ N(0, 0.02) quantized per tensor."""
    w = gaussian((n, k), 0.02, seed)
    amax = float(w.abs().max()) if w.numel() else 1.0
    scale = amax / FP8_MAX if amax > 0 else 1.0
    codes = e4m3_codes(w / scale)
    return codes.to(device), scale


def fp8_expert_stack(e: int, n: int, k: int, seed: int = 0, device="cpu"):
    """(codes uint8 [e, n, k], scales float32 [e]): one FP8 weight per expert,
    each with its own per-tensor scale; expert j uses seed * 1000 + j."""
    codes = torch.empty((e, n, k), dtype=torch.uint8)
    scales = torch.empty(e, dtype=torch.float32)
    for j in range(e):
        c, s = fp8_weight(n, k, seed * 1000 + j)
        codes[j] = c
        scales[j] = s
    return codes.to(device), scales.to(device)


# Midpoints between consecutive E2M1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6.
_E2M1_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """float32 -> E2M1 codes (uint8 0..15), nearest magnitude with ties to the
    even code, saturating at 6; bit 3 is the sign (negative values keep it)."""
    mag = v.abs()
    code = torch.zeros(v.shape, dtype=torch.uint8)
    for i, t in enumerate(_E2M1_MIDPOINTS):
        above = mag > t
        if i % 2 == 1:                 # tie between an odd and an even code
            above = above | (mag == t)  # goes up to the even one
        code += above.to(torch.uint8)
    return code | ((v < 0).to(torch.uint8) << 3)


def nvfp4_weight(n: int, k: int, seed: int = 0, device="cpu"):
    """(q uint8 [n, k/2], bs uint8 [n, k/16], scale2 float)."""
    if k % 16:
        raise ValueError("NVFP4 needs K % 16 == 0")
    w = gaussian((n, k), 0.02, seed)
    amax = float(w.abs().max()) if w.numel() else 1.0
    scale2 = amax / (FP8_MAX * E2M1_MAX) if amax > 0 else 1.0
    blocks = w.reshape(n, k // 16, 16)
    bamax = blocks.abs().amax(dim=2)
    bs = e4m3_codes(bamax / (E2M1_MAX * scale2))
    bs_val = bs.view(torch.float8_e4m3fn).to(torch.float32)
    denom = (scale2 * bs_val).unsqueeze(2)
    safe = torch.where(denom > 0, denom, torch.ones_like(denom))
    codes = e2m1_codes(blocks / safe)
    codes = torch.where(denom > 0, codes, torch.zeros_like(codes)).reshape(n, k)
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()
    return q.to(device), bs.contiguous().to(device), scale2


def nvfp4_expert_stack(e: int, n: int, k: int, seed: int = 0, device="cpu"):
    """(q uint8 [e, n, k/2], bs uint8 [e, n, k/16], scale2 float32 [e]): one
    NVFP4 weight per expert, expert j drawn with seed * 1000 + j."""
    q = torch.empty((e, n, k // 2), dtype=torch.uint8)
    bs = torch.empty((e, n, k // 16), dtype=torch.uint8)
    s2 = torch.empty(e, dtype=torch.float32)
    for j in range(e):
        q[j], bs[j], s2[j] = nvfp4_weight(n, k, seed * 1000 + j)
    return q.to(device), bs.to(device), s2.to(device)


def int8_weight(n: int, k: int, seed: int = 0, device="cpu"):
    """(codes int8 [n, k], scale float32 [n]): W ~ N(0, 0.02) quantized per
    output row, symmetric absmax (scale = absmax / 127, round half to even)."""
    w = gaussian((n, k), 0.02, seed)
    absmax = w.abs().amax(dim=1)
    scale = absmax / 127.0
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    codes = torch.round(w / safe.unsqueeze(1)).clamp(-127, 127).to(torch.int8)
    return codes.to(device), scale.to(device)


def int8_codes(m: int, k: int, seed: int = 0, device="cpu"):
    """(codes int8 [m, k] uniform in [-127, 127], scale float32 [m] in (0, 0.05])."""
    g = _gen(seed)
    codes = torch.randint(-127, 128, (m, k), generator=g, dtype=torch.int16).to(torch.int8)
    scale = (torch.rand(m, generator=g) * 0.05 + 1e-4).to(torch.float32)
    return codes.to(device), scale.to(device)


def moe_routing(total_rows: int, seed: int = 2):
    """(a_offsets int64 [G+1], expert_ids int64 [G], counts [G]) for the
    9-category routing described in the module docstring."""
    probs = torch.tensor(ROUTING_WEIGHTS, dtype=torch.float64)
    cats = torch.multinomial(probs, total_rows, replacement=True, generator=_gen(seed))
    counts = torch.bincount(cats, minlength=len(ROUTING_WEIGHTS))
    offsets = torch.zeros(len(ROUTING_WEIGHTS) + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(counts, 0)
    expert_ids = torch.tensor(list(range(len(ROUTING_WEIGHTS) - 1)) + [-1], dtype=torch.int64)
    return offsets, expert_ids, counts


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
