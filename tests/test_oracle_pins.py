"""Pins of the FP64 oracle against facts that do not come from the oracle.

Each test here checks the oracle against an independent formulation: a
format's bit-field definition, a printed table, brute-force enumeration, a
closed form, a dense numpy matmul, or an invariant of the method.  Together
they are chosen so that a dropped term, a wrong sign, a swapped nibble, a
transposed operand or a wrong block index fails at least one of them.
"""
import itertools
import math
import os
import struct

import numpy as np
import pytest

import oracle
from block_scaled_fp4_moe_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = float(v)
    return out


# ----------------------------------------------------------- independent decode

def bitfield_e2m1(code):
    """E2M1 from its bit fields: sign, 2-bit exponent (bias 1), 1-bit mantissa."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if s else mag


def ieee_e8m0(s):
    """2^(s-127) built as the float32 with that biased exponent field."""
    if s == 0:
        return struct.unpack("<f", struct.pack("<I", 0x00400000))[0]  # 2^-127, subnormal
    return struct.unpack("<f", struct.pack("<I", s << 23))[0]


def dense_decode(codes, scales):
    """numpy decode of packed rows [R, K/2] + [R, K/32] into float64 [R, K]."""
    codes = np.asarray(codes, dtype=np.uint8)
    lo = (codes & 0x0F).astype(np.int64)
    hi = (codes >> 4).astype(np.int64)
    nib = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)   # even element in the low nibble
    sign = np.where(nib & 8, -1.0, 1.0)
    e = (nib >> 1) & 3
    m = nib & 1
    mag = np.where(e == 0, 0.5 * m, np.exp2(e - 1.0) * (1.0 + 0.5 * m))
    sc = np.exp2(np.asarray(scales, dtype=np.float64) - 127.0)
    return sign * mag * np.repeat(sc, 32, axis=1)


def silu(z):
    return z / (1.0 + np.exp(-z))


def bf16_f64(bits):
    return inputs.bf16_bits_to_f32(bits).astype(np.float64)


def random_layer(T, H, E, k, I, has_shared=1, bias=True, seed=1):
    rng = np.random.default_rng(seed)
    x = inputs.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = (0.05 * rng.standard_normal((H, E))).astype(np.float32)
    b = (0.1 * rng.standard_normal(E)).astype(np.float32) if bias else None
    n = E + has_shared
    bank = {
        "w13": rng.integers(0, 256, (n, 2 * I, H // 2), dtype=np.uint8),
        "s13": rng.integers(118, 125, (n, 2 * I, H // 32), dtype=np.uint8),
        "w2": rng.integers(0, 256, (n, H, I // 2), dtype=np.uint8),
        "s2": rng.integers(118, 125, (n, H, I // 32), dtype=np.uint8),
    }
    return x, wr, b, bank


def expert_of(bank):
    return lambda e: {k: v[e] for k, v in bank.items()}


# ------------------------------------------------------------------- formats

def test_e2m1_matches_ocp_table_and_bitfields():
    table = _read_pairs("e2m1_ocp_table.txt")
    assert len(table) == 16
    for code in range(16):
        v = oracle.e2m1_value(code)
        assert v == table[str(code)], code
        assert v == bitfield_e2m1(code), code
        assert math.copysign(1.0, v) == math.copysign(1.0, bitfield_e2m1(code))
    assert math.copysign(1.0, oracle.e2m1_value(8)) == -1.0   # -0 decodes to -0.0


def test_e8m0_is_ieee_biased_exponent():
    for s in range(255):
        assert oracle.e8m0_value(s) == ieee_e8m0(s), s
    assert math.isnan(oracle.e8m0_value(255))


def test_bf16_value_and_rounding_brute_force():
    rng = np.random.default_rng(5)
    # bf16 -> double is the float32 with the same upper 16 bits
    for b in rng.integers(0, 0x7F80, 200):
        f = struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]
        assert oracle.bf16_value(int(b)) == f
    vals = np.concatenate([rng.standard_normal(300) * 10.0 ** rng.integers(-40, 38, 300),
                           [46.78774903232031, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1e-39, -3.0e-40]])
    for v in vals:
        got = oracle.bf16_round(float(v))
        # brute force over the neighbouring bf16 patterns of the float32 truncation
        base = struct.unpack("<I", struct.pack("<f", abs(float(v))))[0] >> 16
        best = None
        for cand in (base - 1, base, base + 1, base + 2):
            if cand < 0 or cand >= 0x7F80:
                continue
            cv = struct.unpack("<f", struct.pack("<I", cand << 16))[0]
            key = (abs(cv - abs(float(v))), cand & 1)        # nearest, then even
            if best is None or key < best[0]:
                best = (key, cand)
        want = best[1] | (0x8000 if v < 0 else 0)
        assert got == want, (v, hex(got), hex(want))


def test_decode_row_independent():
    rng = np.random.default_rng(7)
    K = 128
    codes = rng.integers(0, 256, K // 2, dtype=np.uint8)
    scales = rng.integers(100, 140, K // 32, dtype=np.uint8)
    got = oracle.decode_row(codes, scales, K)
    want = dense_decode(codes[None], scales[None])[0]
    np.testing.assert_array_equal(got, want)


# --------------------------------------------------------- brute-force layer

def brute_force_topk(l, k):
    """Top-k by enumerating every k-subset: the chosen set is the one whose every
    member ranks before every non-member (larger logit, ties to lower index)."""
    E = len(l)
    before = lambda a, b: l[a] > l[b] or (l[a] == l[b] and a < b)
    for sub in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in sub]
        if all(before(a, b) for a in sub for b in rest):
            return sorted(sub, key=lambda e: (-l[e], e))
    raise AssertionError("no top-k subset")


def brute_force_layer(x, wr, b, bank, k, has_shared=1, shared_weight=1.0):
    xd = bf16_f64(x)
    T, H = xd.shape
    E = wr.shape[1]
    I = bank["w13"].shape[1] // 2
    logits = xd @ wr.astype(np.float64) + (0.0 if b is None else b.astype(np.float64))
    ids, ws, ys = [], [], []
    for t in range(T):
        sel = brute_force_topk(list(logits[t]), k)
        z = np.exp(logits[t, sel] - logits[t, sel].max())
        w = list(z / z.sum())
        if has_shared:
            sel = sel + [E]
            w = w + [shared_weight]
        y = np.zeros(H)
        for e, we in zip(sel, w):
            W13 = dense_decode(bank["w13"][e], bank["s13"][e])
            W2 = dense_decode(bank["w2"][e], bank["s2"][e])
            g, u = W13[:I] @ xd[t], W13[I:] @ xd[t]
            y += we * (W2 @ (silu(g) * u))
        ids.append(sel)
        ws.append(w)
        ys.append(y)
    return np.array(ids), np.array(ws), np.array(ys)


@pytest.mark.parametrize("has_shared", [1, 0])
def test_layer_matches_brute_force(has_shared):
    x, wr, b, bank = random_layer(T=3, H=64, E=6, k=2, I=32, has_shared=has_shared)
    got = oracle.layer_forward(x, wr, b, 2, expert_of(bank), has_shared=has_shared)
    ids, w, y = brute_force_layer(x, wr, b, bank, 2, has_shared)
    np.testing.assert_array_equal(got["ids"], ids)
    np.testing.assert_allclose(got["w"], w, rtol=1e-13, atol=0)
    np.testing.assert_allclose(got["y"], y, rtol=1e-11, atol=1e-11 * np.abs(y).max())


def test_router_logits_match_dense_matmul_with_bias():
    x, wr, b, _ = random_layer(T=5, H=96, E=7, k=3, I=32)
    r = oracle.route(x, wr, b, 3)
    want = bf16_f64(x) @ wr.astype(np.float64) + b.astype(np.float64)
    np.testing.assert_allclose(r["logits"], want, rtol=1e-13, atol=1e-13)


# -------------------------------------------------------------- closed forms

def test_closed_form_all_ones():
    gold = _read_pairs("closed_form.txt")
    H = I = 32
    E, k = 4, 2
    n = E + 1
    bank = {"w13": np.full((n, 2 * I, H // 2), 0x22, np.uint8), "s13": np.full((n, 2 * I, 1), 127, np.uint8),
            "w2": np.full((n, H, I // 2), 0x22, np.uint8), "s2": np.full((n, H, 1), 127, np.uint8)}
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x3F80                                         # bf16 1.0
    wr = np.random.default_rng(0).standard_normal((H, E)).astype(np.float32)
    out = oracle.layer_forward(x, wr, None, k, expert_of(bank))
    np.testing.assert_allclose(out["y"], gold["y_double"], rtol=1e-15, atol=0)
    assert np.all(oracle.bf16_round_array(out["y"]) == oracle.bf16_round(gold["y_bf16"]))
    assert oracle.bf16_value(int(out["y_bf16"][0, 0])) == gold["y_bf16"]


@pytest.mark.parametrize("zero_code", [0x00, 0x88])
def test_zero_weights_give_zero(zero_code):
    x, wr, b, bank = random_layer(T=2, H=64, E=4, k=2, I=32)
    bank["w2"][:] = zero_code
    out = oracle.layer_forward(x, wr, b, 2, expert_of(bank))
    assert np.all(out["y"] == 0.0)


def test_single_expert_is_dense_swiglu():
    x, wr, _, bank = random_layer(T=2, H=64, E=1, k=1, I=64, has_shared=0)
    out = oracle.layer_forward(x, wr, None, 1, expert_of(bank), has_shared=0)
    W13 = dense_decode(bank["w13"][0], bank["s13"][0])
    W2 = dense_decode(bank["w2"][0], bank["s2"][0])
    xd = bf16_f64(x)
    want = (silu(xd @ W13[:64].T) * (xd @ W13[64:].T)) @ W2.T
    assert np.all(out["w"] == 1.0)
    np.testing.assert_allclose(out["y"], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


# ----------------------------------------------------------------- invariants

@pytest.fixture(scope="module")
def glm_route():
    cfg = inputs.CONFIGS["glm_zipf_t64"]
    x = inputs.make_x(cfg)
    wr, bias = inputs.make_router(cfg)
    return cfg, x, wr, bias, oracle.route(x, wr, bias, cfg.top_k)


def test_weights_sum_to_one_and_shared_slot(glm_route):
    cfg, _, _, _, r = glm_route
    assert r["ids"].shape == (cfg.T, cfg.top_k + 1)
    np.testing.assert_allclose(r["w"][:, :cfg.top_k].sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(r["ids"][:, cfg.top_k] == cfg.E)
    assert np.all(r["w"][:, cfg.top_k] == 1.0)
    routed = r["ids"][:, :cfg.top_k]
    assert all(len(set(row)) == cfg.top_k for row in routed)
    assert routed.min() >= 0 and routed.max() < cfg.E
    # ordered by descending logit
    lsel = np.take_along_axis(r["logits"], routed, axis=1)
    assert np.all(np.diff(lsel, axis=1) <= 0)


def test_softmax_shift_invariance(glm_route):
    cfg, x, wr, bias, r = glm_route
    shifted = oracle.route(x, wr, (bias.astype(np.float64) + 0.0).astype(np.float32) + np.float32(3.0), cfg.top_k)
    np.testing.assert_array_equal(shifted["ids"], r["ids"])
    np.testing.assert_allclose(shifted["w"], r["w"], rtol=0, atol=1e-12)


def test_tie_goes_to_lower_index():
    rng = np.random.default_rng(3)
    H, E = 64, 6
    x = inputs.f32_to_bf16_bits(rng.standard_normal((4, H)).astype(np.float32))
    wr = rng.standard_normal((H, E)).astype(np.float32)
    best = oracle.route(x, wr, None, 1, has_shared=0)["ids"][:, 0]
    for t in range(4):
        e = int(best[t])
        for dup in range(E):
            if dup == e:
                continue
            w2 = wr.copy()
            w2[:, dup] = wr[:, e]                       # an exact tie with the winner
            r = oracle.route(x[t:t + 1], w2, None, 2, has_shared=0)
            assert list(r["ids"][0]) == [min(e, dup), max(e, dup)]
            assert r["w"][0, 0] == r["w"][0, 1] == 0.5


def test_grouping_against_python_sort():
    rng = np.random.default_rng(11)
    T, k, E = 37, 4, 20
    ids = np.stack([np.concatenate([rng.permutation(E)[:k], [E]]) for _ in range(T)]).astype(np.int32)
    g = oracle.group(ids, E + 1)
    pairs = sorted((int(ids[t, s]), t, s) for t in range(T) for s in range(k + 1))
    assert list(g["sorted_tok"]) == [p[1] for p in pairs]
    assert list(g["sorted_slot"]) == [p[2] for p in pairs]
    counts = np.bincount(ids.ravel(), minlength=E + 1)
    np.testing.assert_array_equal(g["offsets"], np.concatenate([[0], np.cumsum(counts)]))
    np.testing.assert_array_equal(g["active"], np.nonzero(counts)[0])
    assert g["num_active"] == int((counts > 0).sum())
    assert g["offsets"][-1] == T * (k + 1)
    with pytest.raises(ValueError):
        oracle.group(np.array([[E + 1]], np.int32), E + 1)


def test_linearity_over_slots():
    x, wr, b, bank = random_layer(T=2, H=64, E=5, k=3, I=32)
    out = oracle.layer_forward(x, wr, b, 3, expert_of(bank), want_slots=True, want_h=True)
    comb = np.einsum("ts,tsh->th", out["w"], out["y_slots"])
    np.testing.assert_allclose(out["y"], comb, rtol=1e-14, atol=1e-14 * np.abs(comb).max())
    # each slot alone is the expert evaluated densely
    for t in range(2):
        for s in range(4):
            e = out["ids"][t, s]
            W2 = dense_decode(bank["w2"][e], bank["s2"][e])
            np.testing.assert_allclose(out["y_slots"][t, s], W2 @ out["h"][t, s], rtol=1e-12,
                                       atol=1e-12 * np.abs(out["y_slots"][t, s]).max())


# ------------------------------------------------- near-tie diagnostic

@pytest.mark.parametrize("T,H,E,k,bias", [(64, 96, 24, 4, True), (48, 64, 9, 3, False), (16, 32, 6, 6, True)])
def test_near_tie_diagnostic_against_numpy(T, H, E, k, bias):
    """The margin that makes bit-exact routing a fair demand: abs_sum is the
    dense |x|.|Wr| product and gap the smallest difference between
    neighbours among each token's k+1 largest logits (all k when k = E),
    both recomputed with numpy from the inputs alone.  The cases are chosen
    so that the last pair (ranks k, k+1) decides the minimum for some
    tokens and an earlier pair for others, so a range cut short by one or
    an unsigned magnitude sum both fail."""
    x, wr, b, _ = random_layer(T=T, H=H, E=E, k=k, I=32, bias=bias, seed=5 + E)
    r = oracle.route(x, wr, b, k)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    w64 = wr.astype(np.float64)
    abs_np = np.abs(xf) @ np.abs(w64)
    np.testing.assert_allclose(r["abs_sum"], abs_np, rtol=1e-13, atol=0)
    logits = xf @ w64 + (0.0 if b is None else b.astype(np.float64))
    nsel = k + 1 if k < E else k
    order = np.lexsort((np.broadcast_to(np.arange(E), logits.shape), -logits), axis=-1)[:, :nsel]
    top = np.take_along_axis(logits, order, axis=1)
    diffs = top[:, :-1] - top[:, 1:]
    gap_np = diffs.min(axis=1)
    tol = 1e-12 * abs_np.max(axis=1)
    assert np.all(np.abs(r["gap"] - gap_np) <= tol), (r["gap"], gap_np)
    np.testing.assert_allclose(r["rel_gap"], r["gap"] / r["abs_sum"].max(axis=1), rtol=1e-15)
    if k < E:
        # discriminating: the (k, k+1) pair is the minimum for some token, and
        # not for every token
        last_decides = diffs[:, -1] < diffs[:, :-1].min(axis=1) if k > 1 else np.ones(T, bool)
        assert last_decides.any() and (k == 1 or not last_decides.all())
    # without the bias, the magnitude sum bounds |logit| (an unsigned sum would not)
    if b is None:
        assert np.all(np.abs(r["logits"]) <= r["abs_sum"] * (1 + 1e-12))


# ---------------------------------------------------- workloads are well posed

@pytest.mark.parametrize("name", list(inputs.CONFIGS))
def test_workload_routing_is_not_near_tied(name):
    """The order of each token's k+1 best logits is fixed far above the
    accumulation error of any reasonable evaluation (FP64 or compensated fp32)."""
    cfg = inputs.CONFIGS[name]
    x = inputs.make_x(cfg)
    wr, bias = inputs.make_router(cfg)
    r = oracle.route(x, wr, bias, cfg.top_k)
    assert r["rel_gap"].min() > 1e-9, r["rel_gap"].min()


def test_tiny_workload_regression_fixture():
    """tests/golden/tiny_oracle.txt was written by tests/golden/make_golden.py,
    which calls only the oracle; this guards the oracle against silent change."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(GOLDEN, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    out = mg.compute()
    rows = {}
    with open(os.path.join(GOLDEN, "tiny_oracle.txt")) as f:
        for line in f:
            if not line.startswith("#"):
                k, *vals = line.split()
                rows[k] = vals
    assert [int(v) for v in rows["ids"]] == list(out["ids"].ravel())
    np.testing.assert_array_equal(np.array([float(v) for v in rows["w"]]), out["w"].ravel())
    assert [int(v, 16) for v in rows["y_bf16"]] == list(out["y_bf16"].ravel())
    np.testing.assert_array_equal(np.array([float(v) for v in rows["y"]]), out["y"].ravel())
