"""Parity of the MXFP8 live-activation-quantisation variant
(moe_layer_forward_mxfp8) with the oracle's MXFP8 mode, stage by stage.

* routing: ids bit-exact, weights to 2e-6 (the exact path's routing kernels);
* x codes and scales: bit-exact with oracle.mxfp8_quantize of every token's x;
* h (fp32, before its quantisation): within the fp32 accumulation bound of
  the oracle's h, which is computed from the same quantised x;
* h codes and scales: bit-exact with oracle.mxfp8_quantize of the kernel's own
  h -- the E4M3 rounding decision is taken on the kernel's fp32 h on both
  sides, since an fp32 h and the oracle's fp64 h may straddle a rounding
  boundary;
* per-entry outputs Y: within the fp32 accumulation bound of the dense FP64
  down projection of the kernel's dequantised h (weights decoded by the
  oracle);
* y: the bf16 of the weighted slot sum of those Y, and within max|err| <=
  2e-2 max|ref|, mean|err|/mean|ref| <= 5e-3 of the oracle's MXFP8 layer.

Accumulation bound: the tensor core's products of E2M1 x E4M3 values with
their power-of-two scales are exact; the sums run in fp32 over at most K/32
block partials, so |error| <= 2^-24 * (K/32 + 32) * sum |terms| (taken here as
K * 2^-24 * sum |terms|, with K the reduction length), plus the fp32
evaluation of silu(g) * u (a few ulps of |h|).
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_moe_gb300 import _build, inputs, moe
from gpu_support import bf16_to_f64, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    moe.lib()
    torch.cuda.init()


def dense(codes, scales):
    """Decoded weight rows [R, K] through the oracle's row decoder."""
    K = codes.shape[1] * 2
    return np.stack([oracle.decode_row(codes[r], scales[r], K) for r in range(codes.shape[0])])


class MxProblem:
    def __init__(self, T, H, E, k, I, has_shared=1, seed=0, bank_np=None, x=None, wr=None, bias=None):
        rng = np.random.default_rng(seed)
        self.T, self.H, self.E, self.k, self.I, self.S = T, H, E, k, I, has_shared
        self.kps = k + has_shared
        self.x = x if x is not None else inputs.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
        self.wr = wr if wr is not None else (0.02 * rng.standard_normal((H, E))).astype(np.float32)
        self.bias = bias if bias is not None or wr is not None else (0.05 * rng.standard_normal(E)).astype(np.float32)
        n = E + has_shared
        self.bank_np = bank_np if bank_np is not None else {
            "w13": rng.integers(0, 256, (n, 2 * I, H // 2), dtype=np.uint8),
            "s13": rng.integers(118, 125, (n, 2 * I, H // 32), dtype=np.uint8),
            "w2": rng.integers(0, 256, (n, H, I // 2), dtype=np.uint8),
            "s2": rng.integers(118, 125, (n, H, I // 32), dtype=np.uint8)}
        self.bank = moe.MXFP4Bank.from_host(self.bank_np, E, has_shared, with_mx=True)

    def expert(self, e):
        return {kk: v[e] for kk, v in self.bank_np.items()}

    def region(self, ws, name, dtype, shape):
        off = moe.moe_workspace_offset(self.T, self.H, self.I, self.E, self.k, self.S, name)
        n = int(np.prod(shape)) * np.dtype(dtype).itemsize
        return ws[off:off + n].cpu().numpy().view(dtype).reshape(shape)

    def forward(self):
        ws = moe.alloc_workspace(self.T, self.bank, self.k)
        y = torch.full((self.T, self.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        ids = torch.full((self.T, self.kps), -1, dtype=torch.int32, device="cuda")
        w = torch.full((self.T, self.kps), float("nan"), dtype=torch.float32, device="cuda")
        bd = None if self.bias is None else torch.from_numpy(self.bias).cuda()
        moe.moe_layer_forward_mxfp8(dev_bf16(self.x), torch.from_numpy(self.wr).cuda(), bd, self.k, self.bank, 1.0,
                                    y, ids, w, ws)
        torch.cuda.synchronize()
        st = moe.moe_check_device_status(ws)
        assert st == 0, moe.moe_status_string(st)
        n = self.T * self.kps
        return {"y": host_bits(y), "ids": ids.cpu().numpy(), "w": w.cpu().numpy(),
                "xq": self.region(ws, "mx_xq", np.uint8, (self.T, self.H)),
                "xs": self.region(ws, "mx_xs", np.uint8, (self.T, self.H // 32)),
                "h": self.region(ws, "mx_h32", np.float32, (n, self.I)),
                "hq": self.region(ws, "mx_hq", np.uint8, (n, self.I)),
                "hs": self.region(ws, "mx_hs", np.uint8, (n, self.I // 32)),
                "Y": self.region(ws, "mx_y", np.float32, (n, self.H)),
                "inv_pos": self.region(ws, "inv_pos", np.int32, (self.T, self.kps))}


def check_mx(p: MxProblem, out, tokens, label):
    r = oracle.route(p.x, p.wr, p.bias, p.k, p.S)
    np.testing.assert_array_equal(out["ids"], r["ids"], err_msg=label)
    np.testing.assert_allclose(out["w"], r["w"], rtol=2e-6, atol=1e-7, err_msg=label)
    ref = oracle.moe_tokens(p.x, r["ids"], r["w"], p.expert, tokens, want_h=True, act="mxfp8")
    xd = bf16_to_f64(p.x)
    H, I = p.H, p.I
    decoded = {}

    def dense_of(e):
        if e not in decoded:
            ex = p.expert(e)
            decoded[e] = (dense(ex["w13"], ex["s13"]), dense(ex["w2"], ex["s2"]))
        return decoded[e]
    for i, t in enumerate(tokens):
        codes, scales, xq = oracle.mxfp8_quantize(xd[t])
        np.testing.assert_array_equal(out["xq"][t], codes, err_msg=f"{label} x codes t={t}")
        np.testing.assert_array_equal(out["xs"][t], scales, err_msg=f"{label} x scales t={t}")
        ysum = np.zeros(H)
        yabs = np.zeros(H)
        for s in range(p.kps):
            e = int(out["ids"][t, s])
            pos = int(out["inv_pos"][t, s])
            W13, W2 = dense_of(e)
            G, U = W13[:I] @ xq, W13[I:] @ xq
            Sg, Su = np.abs(W13[:I]) @ np.abs(xq), np.abs(W13[I:]) @ np.abs(xq)
            hk = out["h"][pos].astype(np.float64)
            ho = ref["h"][i, s]
            sig = 1 / (1 + np.exp(-G))
            dsilu = np.abs(sig * (1 + G * (1 - sig)))
            eps = H * 2.0 ** -24
            hb = dsilu * eps * Sg * np.abs(U) + np.abs(G * sig) * eps * Su + 8 * 2.0 ** -24 * np.abs(ho) + 1e-30
            assert np.all(np.abs(hk - ho) <= hb), (label, t, s, float((np.abs(hk - ho) / hb).max()))
            c2, s2, hdq = oracle.mxfp8_quantize(hk)
            np.testing.assert_array_equal(out["hq"][pos], c2, err_msg=f"{label} h codes t={t} s={s}")
            np.testing.assert_array_equal(out["hs"][pos], s2, err_msg=f"{label} h scales t={t} s={s}")
            Yd = W2 @ hdq
            Yb = I * 2.0 ** -24 * (np.abs(W2) @ np.abs(hdq)) + 1e-30
            Yk = out["Y"][pos].astype(np.float64)
            assert np.all(np.abs(Yk - Yd) <= Yb), (label, t, s, float((np.abs(Yk - Yd) / Yb).max()))
            ysum += out["w"][t, s] * Yk
            yabs += np.abs(out["w"][t, s] * Yk)
        yk = bf16_to_f64(out["y"][t])
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ysum), 1e-30))) - 7)
        assert np.all(np.abs(yk - ysum) <= 0.5 * ulp * (1 + 1e-6) + p.kps * 2.0 ** -24 * yabs), (label, t)
    y = bf16_to_f64(out["y"][tokens])
    err = np.abs(y - ref["y"])
    aref = np.abs(ref["y"])
    assert err.max() <= 2e-2 * aref.max(), (label, float(err.max() / aref.max()))
    assert err.mean() / aref.mean() <= 5e-3, (label, float(err.mean() / aref.mean()))


SMALL = [
    dict(T=1, H=1024, E=16, k=4, I=512),
    dict(T=3, H=1024, E=16, k=4, I=512),
    dict(T=8, H=1024, E=16, k=4, I=512),
    dict(T=40, H=1024, E=6, k=3, I=512),           # experts hold up to 40 tokens: several passes of 16
    dict(T=5, H=2048, E=24, k=6, I=1024, has_shared=0),
    dict(T=2, H=768, E=8, k=2, I=384),             # K of 3 and 6 stages
    dict(T=160, H=1024, E=4, k=2, I=512),          # T > 128: MMA N = 32, passes of up to 32 entries
]


@pytest.mark.parametrize("case", SMALL, ids=[str(i) for i in range(len(SMALL))])
def test_mxfp8_layer_small_shapes(case):
    p = MxProblem(seed=zlib.crc32(str(case).encode()) % 1000, **case)
    out = p.forward()
    check_mx(p, out, np.arange(p.T), str(case))


def test_mxfp8_layer_glm_t1():
    cfg = inputs.CONFIGS["glm_t1"]
    wr, bias = inputs.make_router(cfg)
    p = MxProblem(cfg.T, cfg.H, cfg.E, cfg.top_k, cfg.I, cfg.has_shared, bank_np=inputs.make_bank(cfg),
                  x=inputs.make_x(cfg), wr=wr, bias=bias)
    out = p.forward()
    check_mx(p, out, np.arange(p.T), "glm_t1")
    del p
    torch.cuda.empty_cache()


def test_mxfp8_routing_matches_exact_entry_point():
    p = MxProblem(T=4, H=1024, E=16, k=4, I=512, seed=5)
    out = p.forward()
    ws = moe.alloc_workspace(p.T, p.bank, p.k)
    y = torch.empty((p.T, p.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((p.T, p.kps), dtype=torch.int32, device="cuda")
    w = torch.empty((p.T, p.kps), dtype=torch.float32, device="cuda")
    moe.moe_layer_forward(dev_bf16(p.x), torch.from_numpy(p.wr).cuda(), torch.from_numpy(p.bias).cuda(), p.k,
                          p.bank, 1.0, y, ids, w, ws)
    np.testing.assert_array_equal(ids.cpu().numpy(), out["ids"])
    np.testing.assert_array_equal(w.cpu().numpy(), out["w"])


def mx_layout_reference(bank_np, H, I):
    """The MXFP8 variant's bank as documented in moe_fp4.h, built with numpy:
    per section, per expert, per chunk of 128 K elements, every row's bytes of
    the chunk (codes 64, scales 4); sections at 256-byte aligned offsets."""
    out = np.zeros(0, dtype=np.uint8)
    for key, per in (("w13", 64), ("w2", 64), ("s13", 4), ("s2", 4)):
        a = bank_np[key]                                   # [n][rows][K bytes]
        n, rows, kb = a.shape
        sec = a.reshape(n, rows, kb // per, per).transpose(0, 2, 1, 3).ravel()
        out = np.concatenate([out, np.zeros((-out.size) % 256, np.uint8), sec])
    return np.concatenate([out, np.zeros((-out.size) % 256, np.uint8)])


def test_pack_mx_matches_documented_layout():
    H, I, E = 384, 256, 2
    rng = np.random.default_rng(11)
    n = E + 1
    bank_np = {"w13": rng.integers(0, 256, (n, 2 * I, H // 2), dtype=np.uint8),
               "s13": rng.integers(0, 256, (n, 2 * I, H // 32), dtype=np.uint8),
               "w2": rng.integers(0, 256, (n, H, I // 2), dtype=np.uint8),
               "s2": rng.integers(0, 256, (n, H, I // 32), dtype=np.uint8)}
    bank = moe.MXFP4Bank.from_host(bank_np, E, 1, with_mx=True)
    torch.cuda.synchronize()
    want = mx_layout_reference(bank_np, H, I)
    got = bank.packed_mx.cpu().numpy()
    assert got.size == want.size == moe.lib().moe_packed_mx_bank_size(H, I, E, 1)
    sections = np.zeros(want.size, bool)           # the padding between sections is not written
    o = 0
    for key in ("w13", "w2", "s13", "s2"):
        o += (-o) % 256
        sections[o:o + bank_np[key].size] = True
        o += bank_np[key].size
    np.testing.assert_array_equal(got[sections], want[sections])


def test_mxfp8_zero_tokens_is_a_noop():
    p = MxProblem(T=1, H=1024, E=16, k=4, I=512, seed=3)
    y = torch.empty((0, p.H), dtype=torch.bfloat16, device="cuda")
    x = torch.empty((0, p.H), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(moe.moe_workspace_size(0, p.H, p.I, p.E, p.k, 1) + 256, dtype=torch.uint8, device="cuda")
    moe.moe_layer_forward_mxfp8(x, torch.from_numpy(p.wr).cuda(), torch.from_numpy(p.bias).cuda(), p.k, p.bank,
                                1.0, y, ws=ws)
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["1t_t1", "glm_verify_t4"])
def test_mxfp8_layer_full_size(name):
    """Full-size shapes: every stage checked on sampled tokens (1T: split K
    in four chunks; GLM T = 4: one chunk, experts shared by tokens)."""
    cfg = inputs.CONFIGS[name]
    wr, bias = inputs.make_router(cfg)
    p = MxProblem(cfg.T, cfg.H, cfg.E, cfg.top_k, cfg.I, cfg.has_shared, bank_np=inputs.make_bank(cfg),
                  x=inputs.make_x(cfg), wr=wr, bias=bias)
    out = p.forward()
    check_mx(p, out, np.array([0, cfg.T - 1]) if cfg.T > 1 else np.arange(1), name)
    del p
    torch.cuda.empty_cache()


def test_mxfp8_is_deterministic_across_calls():
    p = MxProblem(T=6, H=1024, E=16, k=4, I=512, seed=8)
    a = p.forward()
    b = p.forward()
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["hq"], b["hq"])
