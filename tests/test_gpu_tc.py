"""The tensor-memory expert FFN (T >= 9, H and I multiples of 512): the
decoded weight is code x 2^(s - b) in f16 with b an exponent base per weight
row, so its edge cases are about the exponent range of a row's blocks and
about the MMA width a pass selects (16 or 32 columns).  Each case is checked
element by element against the FP64 oracle with the tolerance of the other
parity tests."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_moe_gb300 import _build, inputs, moe
from gpu_support import Problem, bf16_to_f64, check_grouping, check_output

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    torch.cuda.init()


def problem(T, H, E, k, I, seed, s13, s2, has_shared=1, wr_scale=0.02):
    rng = np.random.default_rng(seed)
    x = inputs.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = (wr_scale * rng.standard_normal((H, E))).astype(np.float32)
    b = (0.05 * rng.standard_normal(E)).astype(np.float32)
    n = E + has_shared
    bank = {"w13": rng.integers(0, 256, (n, 2 * I, H // 2), dtype=np.uint8),
            "s13": s13(rng, (n, 2 * I, H // 32)),
            "w2": rng.integers(0, 256, (n, H, I // 2), dtype=np.uint8),
            "s2": s2(rng, (n, H, I // 32))}
    return Problem(x, wr, b, bank, E, k, has_shared)


def narrow(rng, shape):
    return rng.integers(118, 125, shape, dtype=np.uint8)


def layer_and_oracle(p):
    got = p.forward()
    r = p.oracle_route()
    np.testing.assert_array_equal(got["ids"], r["ids"])
    check_grouping(p.grouping(got["ws"]), r["ids"], p.E + p.has_shared, "tc")
    return got, p.oracle_tokens(r, np.arange(p.T))["y"]


@pytest.mark.parametrize("T", [16, 40])
def test_block_exponents_spanning_27_binades_are_exact(T):
    # every row's block exponents lie in [100, 127]: 27 binades, all exact in f16
    def wide(rng, shape):
        s = rng.integers(100, 128, shape, dtype=np.uint8)
        s[..., 0] = 127                     # the largest and the smallest exponent in every row
        s[..., 1] = 100
        return s
    p = problem(T, 1024, 16, 4, 512, seed=30 + T, s13=wide, s2=wide)
    got, ref = layer_and_oracle(p)
    check_output(got["y"], ref, f"27-binade rows T={T}")


def test_blocks_beyond_the_row_range_flush_within_tolerance():
    # rows with a block 40 binades below the row's largest: that block is
    # below f16 once the row is rebased, contributes zero, and the outputs
    # stay within the tolerance (its products are < 2^-40 of the largest's)
    def far(rng, shape):
        s = rng.integers(118, 125, shape, dtype=np.uint8)
        s[..., 2] = 84
        return s
    p = problem(16, 1024, 16, 4, 512, seed=41, s13=far, s2=far)
    got, ref = layer_and_oracle(p)
    check_output(got["y"], ref, "rows beyond 27 binades")


def test_nan_exponent_row_gives_nan_where_the_oracle_does():
    # output row 5 of the shared expert's down projection holds the NaN
    # exponent: that output column is NaN for every token, nothing else is
    def nan_row(rng, shape):
        s = rng.integers(118, 125, shape, dtype=np.uint8)
        s[-1, 5, 3] = 255
        return s
    p = problem(12, 1024, 16, 4, 512, seed=42, s13=narrow, s2=nan_row)
    got, ref = layer_and_oracle(p)
    y = bf16_to_f64(got["y"])
    np.testing.assert_array_equal(np.isnan(y), np.isnan(ref))
    assert np.isnan(ref[:, 5]).all() and not np.isnan(np.delete(ref, 5, axis=1)).any()
    keep = np.ones(p.H, bool)
    keep[5] = False
    check_output(got["y"][:, keep], ref[:, keep], "NaN row excluded")


@pytest.mark.parametrize("T,E,k", [(16, 2, 1), (17, 2, 1), (32, 2, 1), (24, 3, 1), (40, 3, 2)])
def test_pass_widths_select_16_and_32_column_mmas(T, E, k):
    # few experts: gate/up passes of up to 32 tokens (16 or 32 MMA columns),
    # down passes of up to 16 entries (hi + lo: 16 or 32 columns); the shared
    # expert holds all T tokens, so T = 16 / 17 / 32 put its passes on both
    # sides of the 16-row boundary
    p = problem(T, 1024, E, k, 512, seed=50 + T + E, s13=narrow, s2=narrow)
    got, ref = layer_and_oracle(p)
    check_output(got["y"], ref, f"pass widths T={T} E={E} k={k}")


def k_split(n_items, G, nraw, max_pieces=256, min_saving=4):
    """Pieces P and raw stages per piece S of the items left after every CTA
    of the G has taken the same number of whole ones (P = 1: not split)."""
    q, r = divmod(n_items, G)
    if r == 0:
        return 1, nraw
    p0 = max(min(nraw, min(G, max_pieces) // r), 1)
    S = -(-nraw // p0)
    P = -(-nraw // S)
    return (1, nraw) if nraw - S < min_saving else (P, S)


@pytest.mark.parametrize("H", [4096, 2560])
def test_last_items_split_along_k_match_the_oracle(H):
    """The gate/up items left over after every CTA has taken the same number
    of whole ones are cut along K into pieces whose sums the CTA of the last
    piece adds in piece order.  The shape is chosen from the GPU's SM count
    so that a few items are left over: 16 tiles per pass (I = 1024) and one
    more pass than fill the SMs, with H / 512 = 8 or 5 raw stages per item."""
    G = torch.cuda.get_device_properties(0).multi_processor_count
    I, tiles = 1024, 2 * 1024 // 128
    passes = G // tiles + 1                          # one pass per expert at T = 16
    E = passes - 1
    p = problem(16, H, E, min(4, E), I, seed=H, s13=narrow, s2=narrow)
    r = p.oracle_route()
    n_items = len(np.unique(r["ids"])) * tiles       # every expert active: one pass each
    P, S = k_split(n_items, G, H // 512)
    assert P > 1, (n_items, G, P, S)                  # the shape exercises the split
    out, ref = layer_and_oracle(p)
    check_output(out["y"], ref, f"split H={H} P={P} S={S}")
