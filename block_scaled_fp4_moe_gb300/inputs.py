"""Seeded synthetic inputs for the small-T MXFP4 MoE layer.

This module is shared by the tests, the benchmark and the oracle checks.  It
only draws random numbers and packs them into the storage formats the layer
consumes; it holds none of the layer's arithmetic (no decoding, no routing,
no GEMMs).

Workloads (all seed 0) follow the problem statement of the small-T MoE FFN
layer that the pages keep returning to:

* ``tiny``            T=1, H=256, 8 routed + 1 shared, top-2, I=128, router
                      offset b_i = 0.01*i so that no two logits nearly tie.
* ``glm_t1``          GLM shape: H=5120, 160 routed + 1 shared (top-8, the
                      shared expert fused as the 9th slot), I=1536, T=1.
                      (GLM4-MoE: 160 routed experts, top-8, one shared expert,
                      "Optimizing GLM4-MoE for production", section 1 "Shared
                      experts fusion"; top-8 per token also on the GLM-5.2 B300
                      page, section "What it solves".)
* ``glm_verify_t4`` / ``glm_verify_t16``
                      speculative-verify batches on the GLM shape: token 0 is
                      N(0,1), draft tokens are token 0 plus N(0,0.1).
* ``1t_t1`` / ``1t_t4`` / ``1t_t8``
                      1T-class shape: H=7168, 384 routed + 1 shared, top-8,
                      I=2048.
* ``glm_zipf_t64`` / ``glm_zipf_t256``
                      batched decode with a Zipf(s=1.2) per-expert router bias
                      b_e = ln p(e), p(e) proportional to (e+1)^-1.2.

Storage formats (the layer's input contract):

* x: bf16 bit patterns, uint16 [T, H], round-to-nearest-even from float32.
* router weight: float32 [H, E] row-major; bias float32 [E] or None.
* expert bank (expert index E is the shared expert when present):
  - w13 uint8 [E+S, 2I, H/2]: rows 0..I-1 gate, rows I..2I-1 up; two E2M1
    codes per byte, element 2j in the low nibble, 2j+1 in the high nibble;
  - s13 uint8 [E+S, 2I, H/32]: one E8M0 exponent per 32 consecutive
    elements of a row;
  - w2 uint8 [E+S, H, I/2], s2 uint8 [E+S, H, I/32]: the down projection,
    same packing along I.
* codes are uniform over all 16 E2M1 codes (uniform bytes), exponents uniform
  in [118, 124].

Random streams: every array is drawn from ``numpy.random.default_rng([seed,
stream, index])``, so one expert can be regenerated on its own (the oracle
only needs the experts a token touches).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# stream ids of the counter-style seed keys
_S_X, _S_ROUTER, _S_W13, _S_S13, _S_W2, _S_S2, _S_PERTURB = 1, 2, 3, 4, 5, 6, 7

SCALE_LO, SCALE_HI = 118, 124  # E8M0 exponents are drawn uniformly in [lo, hi]


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    E: int          # routed experts
    top_k: int
    I: int
    has_shared: int = 1
    x_kind: str = "normal"      # "normal" | "draft"
    bias_kind: str = "none"     # "none" | "offset" | "zipf"
    seed: int = 0

    @property
    def n_experts_total(self) -> int:
        return self.E + self.has_shared

    @property
    def slots(self) -> int:
        return self.top_k + self.has_shared

    def with_T(self, T: int, name: str | None = None) -> "MoEConfig":
        return dataclasses.replace(self, T=T, name=name or self.name)


_GLM = dict(H=5120, E=160, top_k=8, I=1536)
_ONE_T = dict(H=7168, E=384, top_k=8, I=2048)

CONFIGS: dict[str, MoEConfig] = {
    "tiny": MoEConfig("tiny", T=1, H=256, E=8, top_k=2, I=128, bias_kind="offset"),
    "glm_t1": MoEConfig("glm_t1", T=1, **_GLM),
    "glm_verify_t4": MoEConfig("glm_verify_t4", T=4, x_kind="draft", **_GLM),
    "glm_verify_t16": MoEConfig("glm_verify_t16", T=16, x_kind="draft", **_GLM),
    "1t_t1": MoEConfig("1t_t1", T=1, **_ONE_T),
    "1t_t4": MoEConfig("1t_t4", T=4, **_ONE_T),
    "1t_t8": MoEConfig("1t_t8", T=8, **_ONE_T),
    "glm_zipf_t64": MoEConfig("glm_zipf_t64", T=64, bias_kind="zipf", **_GLM),
    "glm_zipf_t256": MoEConfig("glm_zipf_t256", T=256, bias_kind="zipf", **_GLM),
}


def _rng(cfg: MoEConfig, stream: int, index: int = 0) -> np.random.Generator:
    return np.random.default_rng([cfg.seed, stream, index])


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def make_x(cfg: MoEConfig) -> np.ndarray:
    """Hidden states x as bf16 bits, uint16 [T, H]."""
    rng = _rng(cfg, _S_X)
    if cfg.x_kind == "normal":
        return f32_to_bf16_bits(rng.standard_normal((cfg.T, cfg.H)).astype(np.float32))
    if cfg.x_kind == "draft":
        x0 = f32_to_bf16_bits(rng.standard_normal((1, cfg.H)).astype(np.float32))
        x0f = bf16_bits_to_f32(x0)
        noise = _rng(cfg, _S_PERTURB).standard_normal((cfg.T - 1, cfg.H))
        drafts = f32_to_bf16_bits(x0f + (0.1 * noise).astype(np.float32))
        return np.concatenate([x0, drafts], axis=0)
    raise ValueError(cfg.x_kind)


def make_router(cfg: MoEConfig) -> tuple[np.ndarray, np.ndarray | None]:
    """Router weight float32 [H, E] ~ N(0, 0.02) and the per-expert logit bias."""
    wr = (0.02 * _rng(cfg, _S_ROUTER).standard_normal((cfg.H, cfg.E))).astype(np.float32)
    if cfg.bias_kind == "none":
        bias = None
    elif cfg.bias_kind == "offset":
        bias = (0.01 * np.arange(cfg.E)).astype(np.float32)
    elif cfg.bias_kind == "zipf":
        ranks = np.arange(1, cfg.E + 1, dtype=np.float64)
        p = ranks ** -1.2
        bias = np.log(p / p.sum()).astype(np.float32)
    else:
        raise ValueError(cfg.bias_kind)
    return wr, bias


def expert_shapes(cfg: MoEConfig) -> dict[str, tuple[int, int]]:
    H, I = cfg.H, cfg.I
    return {"w13": (2 * I, H // 2), "s13": (2 * I, H // 32),
            "w2": (H, I // 2), "s2": (H, I // 32)}


def make_expert(cfg: MoEConfig, e: int, out: dict[str, np.ndarray] | None = None) -> dict[str, np.ndarray]:
    """Packed MXFP4 weights of expert e (e == E is the shared expert)."""
    shp = expert_shapes(cfg)
    arrs = {}
    for key, stream, lo, hi in (("w13", _S_W13, 0, 255), ("s13", _S_S13, SCALE_LO, SCALE_HI),
                                ("w2", _S_W2, 0, 255), ("s2", _S_S2, SCALE_LO, SCALE_HI)):
        rng = _rng(cfg, stream, e)
        n = math.prod(shp[key])
        if lo == 0 and hi == 255 and n % 4 == 0:
            # uniform bytes: numpy draws full-range uint8 four to a 32-bit word,
            # so these are the bytes integers(0, 256, dtype=uint8) gives, ten
            # times faster (checked by the input tests)
            a = rng.integers(0, 1 << 32, size=n // 4, dtype=np.uint32).view(np.uint8).reshape(shp[key])
        else:
            a = rng.integers(lo, hi + 1, size=shp[key], dtype=np.uint8)
        if out is not None:
            out[key][...] = a
            arrs[key] = out[key]
        else:
            arrs[key] = a
    return arrs


def bank_nbytes(cfg: MoEConfig) -> int:
    return sum(math.prod(s) for s in expert_shapes(cfg).values()) * cfg.n_experts_total


def alloc_bank(cfg: MoEConfig) -> dict[str, np.ndarray]:
    n = cfg.n_experts_total
    return {k: np.empty((n,) + s, dtype=np.uint8) for k, s in expert_shapes(cfg).items()}


def make_bank(cfg: MoEConfig, out: dict[str, np.ndarray] | None = None) -> dict[str, np.ndarray]:
    """Full expert bank, arrays [E+S, ...]; fills ``out`` in place when given."""
    bank = out if out is not None else alloc_bank(cfg)
    for e in range(cfg.n_experts_total):
        make_expert(cfg, e, out={k: v[e] for k, v in bank.items()})
    return bank
