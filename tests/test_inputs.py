"""The seeded input generators: recipe facts that do not depend on the layer."""
import numpy as np

from block_scaled_fp4_moe_gb300 import inputs


def test_fast_uniform_bytes_are_the_plain_draw():
    """make_expert draws the E2M1 code bytes as 32-bit words; they must be the
    bytes of the plain uniform uint8 draw from the same seed key."""
    cfg = inputs.CONFIGS["tiny"]
    for e in (0, 3, cfg.E):
        got = inputs.make_expert(cfg, e)
        for key, stream in (("w13", inputs._S_W13), ("w2", inputs._S_W2)):
            plain = inputs._rng(cfg, stream, e).integers(0, 256, size=got[key].shape, dtype=np.uint8)
            np.testing.assert_array_equal(got[key], plain)
        for key in ("s13", "s2"):
            assert got[key].min() >= inputs.SCALE_LO and got[key].max() <= inputs.SCALE_HI


def test_recipe_shapes_and_distributions():
    cfg = inputs.CONFIGS["glm_verify_t4"]
    x = inputs.bf16_bits_to_f32(inputs.make_x(cfg)).astype(np.float64)
    assert x.shape == (4, 5120)
    assert abs(x[0].std() - 1.0) < 0.05                        # token 0 ~ N(0, 1)
    d = x[1:] - x[0]
    assert abs(d.std() - 0.1) < 0.01                           # drafts = token 0 + N(0, 0.1)
    wr, bias = inputs.make_router(cfg)
    assert bias is None and abs(wr.std() - 0.02) < 1e-3
    z = inputs.CONFIGS["glm_zipf_t64"]
    _, b = inputs.make_router(z)
    p = np.exp(b.astype(np.float64))
    np.testing.assert_allclose(p.sum(), 1.0, rtol=1e-5)
    np.testing.assert_allclose(p[1] / p[0], 2.0 ** -1.2, rtol=1e-5)     # Zipf(s = 1.2) over ranks e + 1
