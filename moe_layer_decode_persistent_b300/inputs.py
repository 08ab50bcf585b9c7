"""Seeded synthetic inputs for the decode MoE layer (input preparation only).

This module serves both the CUDA path and the CPU oracle, so it holds none of
the layer's arithmetic: it draws random activations, routings and weights and
encodes the weights into the library's storage formats (the encoder is the
inverse of the storage format, i.e. input prep; nothing here decodes or
multiplies weights). It imports nothing else from the package.

Workloads (DeepSeek-V3 shapes H=7168, I=2048, E=256, K=8, one shared expert):
  * ``tiny``      all-bf16 T=4, H=256, I=128, E=8, K=2, shared I=128, seed 0.
  * ``uniform``   K distinct experts per row drawn uniformly.
  * ``mtp``       rows in requests of 4; each row keeps each pick of the row
                  before it with probability 0.6 (kept picks first, in their old
                  slot order) and draws the rest uniformly without repeats.
  * ``zipf``      experts ranked by a seeded permutation, p(rank r) ~ r^-1.2,
                  K picks without replacement.
Router weights are a softmax of N(0,1) over each row's K picks. Activations x
are bf16 N(0,1); weights are N(0, 0.02) before encoding.

Weight encodings (layouts as in include/moe.h):
  * NVFP4: per expert and matrix a fp32 tensor scale gs = amax / (6 * 448);
    per 16-element block along the input dimension an E4M3 scale
    s = e4m3(amax_blk / (6 gs)); codes = e2m1 nearest-even of w / (s gs),
    saturating; two codes a byte, low nibble = even element.
  * FP8 (E4M3FN) with one fp32 scale per 128x128 block: s = amax_blk / 448,
    q = e4m3(w / s).
  * bf16: round to nearest even.
"""
from __future__ import annotations

import dataclasses
import hashlib

import torch

FMT_BF16, FMT_NVFP4, FMT_FP8_B128 = 0, 1, 2
FMT_NAMES = {FMT_BF16: "bf16", FMT_NVFP4: "nvfp4", FMT_FP8_B128: "fp8_b128"}


@dataclasses.dataclass(frozen=True)
class Shape:
    T: int
    H: int
    I: int
    I_shared: int
    E: int
    K: int


TINY = Shape(T=4, H=256, I=128, I_shared=128, E=8, K=2)


def dsv3(T: int, E: int = 256) -> Shape:
    return Shape(T=T, H=7168, I=2048, I_shared=2048, E=E, K=8)


def _seed(*parts) -> int:
    h = hashlib.sha256(("/".join(str(p) for p in parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------

def routing_uniform(T: int, K: int, E: int, seed: int) -> torch.Tensor:
    g = _gen("cpu", "uniform", seed, T, K, E)
    ids = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]) if T else \
        torch.zeros((0, K), dtype=torch.int64)
    return ids.to(torch.int32)


def routing_mtp(T: int, K: int, E: int, seed: int, rows_per_request: int = 4,
                keep: float = 0.6) -> torch.Tensor:
    g = _gen("cpu", "mtp", seed, T, K, E, rows_per_request, keep)
    rows = []
    for t in range(T):
        if t % rows_per_request == 0:
            row = torch.randperm(E, generator=g)[:K].tolist()
        else:
            prev = rows[-1]
            coins = torch.rand(K, generator=g).tolist()
            kept = [e for e, c in zip(prev, coins) if c < keep]
            pool = [e for e in torch.randperm(E, generator=g).tolist() if e not in kept]
            row = kept + pool[:K - len(kept)]
        rows.append(row)
    return torch.tensor(rows, dtype=torch.int32).reshape(T, K)


def routing_zipf(T: int, K: int, E: int, seed: int, s: float = 1.2) -> torch.Tensor:
    g = _gen("cpu", "zipf", seed, T, K, E, s)
    perm = torch.randperm(E, generator=g)
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    p = ranks ** (-s)
    p = p / p.sum()
    if T == 0:
        return torch.zeros((0, K), dtype=torch.int32)
    picks = torch.multinomial(p.expand(T, E).contiguous(), K, replacement=False, generator=g)
    return perm[picks].to(torch.int32)


ROUTINGS = {"uniform": routing_uniform, "mtp": routing_mtp, "zipf": routing_zipf}


def router_weights(T: int, K: int, seed: int) -> torch.Tensor:
    g = _gen("cpu", "router_w", seed, T, K)
    return torch.softmax(torch.randn(T, K, generator=g, dtype=torch.float32), dim=-1)


def activations(T: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(device, "x", seed, T, H)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


# --------------------------------------------------------------------------
# weight encoders (input prep)
# --------------------------------------------------------------------------

_E2M1_MAGS = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
# midpoints between neighbouring magnitudes; a tie goes to the even code
_E2M1_MIDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)
_E2M1_TIE_UP = (0.75, 1.75, 3.5)


def encode_e2m1(v: torch.Tensor) -> torch.Tensor:
    """Nearest-even E2M1 code (uint8 in 0..15) of each value, saturating at 6."""
    mag = v.abs().float()
    mids = torch.tensor(_E2M1_MIDS, device=v.device)
    idx = torch.bucketize(mag, mids, right=False)  # a tie goes to the lower code
    for m in _E2M1_TIE_UP:
        idx = torch.where(mag == m, idx + 1, idx)
    sign = (v < 0) & (idx > 0)
    return (idx + sign.to(idx.dtype) * 8).to(torch.uint8)


def encode_nvfp4(w: torch.Tensor):
    """w: fp32 [..., rows, cols] for ONE expert matrix -> (codes, scales, gscale).

    codes uint8 [rows, cols/2] (low nibble = even column), scales uint8 (E4M3
    bits) [rows, cols/16], gscale fp32 scalar tensor."""
    rows, cols = w.shape
    w = w.float()
    amax = w.abs().max()
    gs = (amax / (6.0 * 448.0)).clamp_min(1e-30)
    blk = w.reshape(rows, cols // 16, 16)
    bmax = blk.abs().amax(dim=-1)
    s = (bmax / (6.0 * gs)).clamp(max=448.0).to(torch.float8_e4m3fn)
    sf = s.float()
    denom = torch.where(sf > 0, sf * gs, torch.ones_like(sf))
    q = (blk / denom.unsqueeze(-1)).clamp(-6.0, 6.0)
    codes = encode_e2m1(q).reshape(rows, cols)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()
    return packed, s.view(torch.uint8).contiguous(), gs.reshape(()).float()


def encode_fp8_b128(w: torch.Tensor):
    """w: fp32 [rows, cols] -> (q uint8 E4M3 bits [rows, cols], scales fp32 [rows/128, cols/128])."""
    rows, cols = w.shape
    w = w.float()
    blk = w.reshape(rows // 128, 128, cols // 128, 128)
    bmax = blk.abs().amax(dim=(1, 3))
    s = torch.where(bmax > 0, bmax / 448.0, torch.ones_like(bmax))
    q = (blk / s[:, None, :, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.reshape(rows, cols).view(torch.uint8).contiguous(), s.contiguous()


# --------------------------------------------------------------------------
# expert sets
# --------------------------------------------------------------------------

@dataclasses.dataclass
class ExpertSet:
    """One expert set in the library's layout (tensors on one device).

    fmt: FMT_*; w13 [E][2I][H] (NVFP4 bytes [E][2I][H/2], FP8 bytes, bf16);
    w2 [E][H][I] likewise; scales / gscales as the format needs (else None)."""
    fmt: int
    E: int
    H: int
    I: int
    w13: torch.Tensor
    w2: torch.Tensor
    w13_scale: torch.Tensor | None = None
    w2_scale: torch.Tensor | None = None
    w13_gscale: torch.Tensor | None = None
    w2_gscale: torch.Tensor | None = None

    def tensors(self):
        return [t for t in (self.w13, self.w2, self.w13_scale, self.w2_scale,
                            self.w13_gscale, self.w2_gscale) if t is not None]

    def nbytes_expert(self) -> int:
        """Weight + scale bytes of one expert (what streaming it once costs)."""
        return sum(t.numel() * t.element_size() for t in self.tensors()) // self.E

    def to(self, device) -> "ExpertSet":
        f = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
             for k, v in dataclasses.asdict(self).items()}
        return ExpertSet(**f)

    def select(self, experts) -> "ExpertSet":
        """A new set holding only the listed experts (renumbered 0..n-1), on CPU."""
        idx = torch.as_tensor(list(experts), dtype=torch.long)
        f = {}
        for k, v in dataclasses.asdict(self).items():
            f[k] = v.index_select(0, idx.to(v.device)).cpu() if isinstance(v, torch.Tensor) else v
        f["E"] = len(idx)
        return ExpertSet(**f)


def _draw_expert(fmt: int, H: int, I: int, seed, e: int, device, std: float, tag: str):
    """Expert e of a set, drawn from its own seed and encoded: a dict of
    per-expert tensors (w13, w2 and the format's scales)."""
    g = _gen(device, tag, seed, e, "w13")
    w13 = torch.randn(2 * I, H, generator=g, device=device) * std
    g = _gen(device, tag, seed, e, "w2")
    w2 = torch.randn(H, I, generator=g, device=device) * std
    if fmt == FMT_BF16:
        return {"w13": w13.to(torch.bfloat16), "w2": w2.to(torch.bfloat16)}
    if fmt == FMT_NVFP4:
        q13, s13, g13 = encode_nvfp4(w13)
        q2, s2, g2 = encode_nvfp4(w2)
        return {"w13": q13, "w13_scale": s13, "w13_gscale": g13, "w2": q2, "w2_scale": s2, "w2_gscale": g2}
    if fmt == FMT_FP8_B128:
        q13, s13 = encode_fp8_b128(w13)
        q2, s2 = encode_fp8_b128(w2)
        return {"w13": q13, "w13_scale": s13, "w2": q2, "w2_scale": s2}
    raise ValueError(f"unknown weight format {fmt}")


def _empty_set(fmt: int, E: int, H: int, I: int, device) -> ExpertSet:
    if fmt == FMT_BF16:
        return ExpertSet(fmt, E, H, I, torch.zeros(E, 2 * I, H, dtype=torch.bfloat16, device=device),
                         torch.zeros(E, H, I, dtype=torch.bfloat16, device=device))
    if fmt == FMT_NVFP4:
        return ExpertSet(fmt, E, H, I,
                         torch.zeros(E, 2 * I, H // 2, dtype=torch.uint8, device=device),
                         torch.zeros(E, H, I // 2, dtype=torch.uint8, device=device),
                         torch.zeros(E, 2 * I, H // 16, dtype=torch.uint8, device=device),
                         torch.zeros(E, H, I // 16, dtype=torch.uint8, device=device),
                         torch.zeros(E, dtype=torch.float32, device=device),
                         torch.zeros(E, dtype=torch.float32, device=device))
    if fmt == FMT_FP8_B128:
        return ExpertSet(fmt, E, H, I,
                         torch.zeros(E, 2 * I, H, dtype=torch.uint8, device=device),
                         torch.zeros(E, H, I, dtype=torch.uint8, device=device),
                         torch.ones(E, 2 * I // 128, H // 128, dtype=torch.float32, device=device),
                         torch.ones(E, H // 128, I // 128, dtype=torch.float32, device=device))
    raise ValueError(f"unknown weight format {fmt}")


def make_experts(fmt: int, E: int, H: int, I: int, seed, device="cpu", std: float = 0.02,
                 tag: str = "routed", only=None) -> ExpertSet:
    """E SwiGLU experts, each drawn from its own seed (so a subset regenerates alike).

    only: if given, just those experts are drawn and the rest stay zero (tests
    that touch a few experts of a large set use it to save time)."""
    es = _empty_set(fmt, E, H, I, device)
    todo = range(E) if only is None else sorted(set(int(e) for e in only))
    for e in todo:
        for k, v in _draw_expert(fmt, H, I, seed, e, device, std, tag).items():
            getattr(es, k)[e] = v
    return es


def make_expert_subset(fmt: int, experts, H: int, I: int, seed, device="cpu", std: float = 0.02,
                       tag: str = "routed") -> ExpertSet:
    """The listed experts of a set, each drawn from the same seed as in
    make_experts, stored compactly: position i holds expert experts[i]."""
    experts = [int(e) for e in experts]
    es = _empty_set(fmt, len(experts), H, I, device)
    for i, e in enumerate(experts):
        for k, v in _draw_expert(fmt, H, I, seed, e, device, std, tag).items():
            getattr(es, k)[i] = v
    return es


@dataclasses.dataclass
class Layer:
    shape: Shape
    x: torch.Tensor          # bf16 [T][H]
    topk_ids: torch.Tensor   # int32 [T][K]
    topk_w: torch.Tensor     # fp32 [T][K]
    routed: ExpertSet
    shared: ExpertSet


def make_layer(shape: Shape, routing: str = "uniform", seed: int = 0, device="cpu",
               fmt_routed: int = FMT_NVFP4, fmt_shared: int = FMT_FP8_B128,
               layer: int = 0, used_only: bool = False) -> Layer:
    """One layer's weights and one batch of inputs. `layer` varies the weights only.

    used_only: draw only the routed experts this batch picks (others zero)."""
    s = shape
    ids = ROUTINGS[routing](s.T, s.K, s.E, seed)
    w = router_weights(s.T, s.K, seed)
    x = activations(s.T, s.H, seed, device)
    only = ids.reshape(-1).tolist() if used_only else None
    routed = make_experts(fmt_routed, s.E, s.H, s.I, ("L", layer, seed), device, tag="routed",
                          only=only)
    shared = make_experts(fmt_shared, 1, s.H, s.I_shared, ("L", layer, seed), device, tag="shared")
    return Layer(s, x, ids.to(device), w.to(device), routed, shared)


def make_tiny(seed: int = 0, device="cpu") -> Layer:
    """The all-bf16 tiny layer: T=4, H=256, I=128, E=8 top-2, shared I=128."""
    return make_layer(TINY, "uniform", seed, device, FMT_BF16, FMT_BF16)
